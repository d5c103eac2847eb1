// extern "C" entry points of libthd: host-side argument checks, then one or
// two kernel launches on the caller's stream.  See include/thd.h for the
// contract of every call.
#include <climits>

#include "thd_internal.cuh"

namespace thd {

namespace {
thread_local int32_t g_last_cuda_error = 0;

constexpr int64_t kMaxRows = INT32_MAX;           // row indices are int32
constexpr int64_t kMaxRowBytes = int64_t(1) << 30;
constexpr int32_t kMaxRawRows = 65535;

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

bool route_args_ok(int64_t T, int32_t cp) {
  return cp >= 1 && cp <= THD_MAX_CP && T >= 0 && T <= kMaxRows && T % (2 * cp) == 0;
}

bool route_ok(const thd_route_t* r) {
  if (!r || !route_args_ok(r->total_rows, r->cp_size)) return false;
  if (r->dir != THD_ZIGZAG_TO_CONTIGUOUS && r->dir != THD_CONTIGUOUS_TO_ZIGZAG) return false;
  return r->send_rows && r->recv_rows && r->input_split_sizes && r->output_split_sizes &&
         r->send_offsets && r->recv_offsets && r->send_identity && r->recv_identity && r->src_of_dst;
}

bool ranges_overlap(const void* a, const void* b, int64_t bytes) {
  uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return bytes > 0 && x < y + static_cast<uintptr_t>(bytes) && y < x + static_cast<uintptr_t>(bytes);
}

thd_status_t copy_entry(CopyKind kind, const void* src, void* dst, int64_t row_bytes,
                        const thd_route_t* route, int32_t* d_status, cudaStream_t stream) {
  if (!route_ok(route) || row_bytes <= 0 || row_bytes > kMaxRowBytes) return THD_ERR_INVALID_ARG;
  const int64_t bytes = route->total_rows * row_bytes;
  if (bytes > 0 && (!src || !dst)) return THD_ERR_INVALID_ARG;
  if (ranges_overlap(src, dst, bytes)) return THD_ERR_INVALID_ARG;
  return launch_copy(kind, src, dst, row_bytes, route, d_status, stream);
}

thd_status_t rank_copy_entry(bool scatter, const void* src, void* dst, int32_t cp_rank, int64_t row_bytes,
                             const thd_route_t* route, int32_t* d_status, cudaStream_t stream) {
  if (!route_ok(route) || row_bytes <= 0 || row_bytes > kMaxRowBytes) return THD_ERR_INVALID_ARG;
  if (cp_rank < 0 || cp_rank >= route->cp_size) return THD_ERR_INVALID_ARG;
  const int64_t bytes = route->total_rows / route->cp_size * row_bytes;
  if (bytes > 0 && (!src || !dst)) return THD_ERR_INVALID_ARG;
  if (ranges_overlap(src, dst, bytes)) return THD_ERR_INVALID_ARG;
  return launch_rank_copy(scatter, src, dst, cp_rank, row_bytes, route, d_status, stream);
}
}  // namespace

void record_cuda_error(cudaError_t e) { g_last_cuda_error = static_cast<int32_t>(e); }

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) return 1;
  return n;
}

}  // namespace thd

using namespace thd;

extern "C" {

size_t thd_route_bytes(int64_t T, int32_t cp) {
  if (!route_args_ok(T, cp)) return 0;
  const size_t rows = static_cast<size_t>(T) * sizeof(int32_t);
  const size_t sq = static_cast<size_t>(cp) * cp * sizeof(int32_t);
  const size_t off = static_cast<size_t>(cp) * (cp + 1) * sizeof(int32_t);
  const size_t flag = static_cast<size_t>(cp);
  return 3 * align256(rows) + 2 * align256(sq) + 2 * align256(off) + 2 * align256(flag);
}

thd_status_t thd_route_bind(thd_route_t* route, void* d_base, size_t bytes, int64_t T, int32_t cp,
                            thd_dir_t dir) {
  if (!route) return THD_ERR_INVALID_ARG;
  if (dir != THD_ZIGZAG_TO_CONTIGUOUS && dir != THD_CONTIGUOUS_TO_ZIGZAG) return THD_ERR_BAD_DIRECTION;
  const size_t need = thd_route_bytes(T, cp);
  if (need == 0 || !d_base || bytes < need || reinterpret_cast<uintptr_t>(d_base) % 256 != 0)
    return THD_ERR_INVALID_ARG;
  char* p = static_cast<char*>(d_base);
  auto take = [&p](size_t n) {
    char* q = p;
    p += align256(n);
    return q;
  };
  const size_t rows = static_cast<size_t>(T) * sizeof(int32_t);
  route->cp_size = cp;
  route->dir = dir;
  route->total_rows = T;
  route->send_rows = reinterpret_cast<int32_t*>(take(rows));
  route->recv_rows = reinterpret_cast<int32_t*>(take(rows));
  route->src_of_dst = reinterpret_cast<int32_t*>(take(rows));
  route->input_split_sizes = reinterpret_cast<int32_t*>(take(static_cast<size_t>(cp) * cp * 4));
  route->output_split_sizes = reinterpret_cast<int32_t*>(take(static_cast<size_t>(cp) * cp * 4));
  route->send_offsets = reinterpret_cast<int32_t*>(take(static_cast<size_t>(cp) * (cp + 1) * 4));
  route->recv_offsets = reinterpret_cast<int32_t*>(take(static_cast<size_t>(cp) * (cp + 1) * 4));
  route->send_identity = reinterpret_cast<uint8_t*>(take(static_cast<size_t>(cp)));
  route->recv_identity = reinterpret_cast<uint8_t*>(take(static_cast<size_t>(cp)));
  return THD_OK;
}

size_t thd_route_pair_bytes(int64_t T, int32_t cp) {
  if (!route_args_ok(T, cp)) return 0;
  const size_t rows = static_cast<size_t>(T) * sizeof(int32_t);
  const size_t sq = static_cast<size_t>(cp) * cp * sizeof(int32_t);
  const size_t off = static_cast<size_t>(cp) * (cp + 1) * sizeof(int32_t);
  const size_t flag = static_cast<size_t>(cp);
  return 4 * align256(rows) + 2 * (2 * align256(sq) + 2 * align256(off) + 2 * align256(flag));
}

thd_status_t thd_route_bind_pair(thd_route_t* route_z2c, thd_route_t* route_c2z, void* d_base, size_t bytes,
                                 int64_t T, int32_t cp) {
  if (!route_z2c || !route_c2z || route_z2c == route_c2z) return THD_ERR_INVALID_ARG;
  const size_t need = thd_route_pair_bytes(T, cp);
  if (need == 0 || !d_base || bytes < need || reinterpret_cast<uintptr_t>(d_base) % 256 != 0)
    return THD_ERR_INVALID_ARG;
  char* p = static_cast<char*>(d_base);
  auto take = [&p](size_t n) {
    char* q = p;
    p += align256(n);
    return q;
  };
  const size_t rows = static_cast<size_t>(T) * sizeof(int32_t);
  int32_t* zc_src = reinterpret_cast<int32_t*>(take(rows));
  int32_t* cz_src = reinterpret_cast<int32_t*>(take(rows));
  // z->c receive rows == c->z send rows; z->c send rows == c->z receive rows
  // == 0..S-1 on every rank
  int32_t* shared_rows = reinterpret_cast<int32_t*>(take(rows));
  int32_t* in_order = reinterpret_cast<int32_t*>(take(rows));
  thd_route_t* rt[2] = {route_z2c, route_c2z};
  for (int k = 0; k < 2; ++k) {
    thd_route_t* r = rt[k];
    r->cp_size = cp;
    r->dir = k == 0 ? THD_ZIGZAG_TO_CONTIGUOUS : THD_CONTIGUOUS_TO_ZIGZAG;
    r->total_rows = T;
    r->src_of_dst = k == 0 ? zc_src : cz_src;
    r->send_rows = k == 0 ? in_order : shared_rows;
    r->recv_rows = k == 0 ? shared_rows : in_order;
    r->input_split_sizes = reinterpret_cast<int32_t*>(take(static_cast<size_t>(cp) * cp * 4));
    r->output_split_sizes = reinterpret_cast<int32_t*>(take(static_cast<size_t>(cp) * cp * 4));
    r->send_offsets = reinterpret_cast<int32_t*>(take(static_cast<size_t>(cp) * (cp + 1) * 4));
    r->recv_offsets = reinterpret_cast<int32_t*>(take(static_cast<size_t>(cp) * (cp + 1) * 4));
    r->send_identity = reinterpret_cast<uint8_t*>(take(static_cast<size_t>(cp)));
    r->recv_identity = reinterpret_cast<uint8_t*>(take(static_cast<size_t>(cp)));
  }
  return THD_OK;
}

thd_status_t thd_route_build(const int32_t* cu_seqlens_padded, int32_t num_docs, int64_t T, int32_t cp_size,
                             thd_dir_t dir, const thd_route_t* route, int32_t* d_status,
                             cudaStream_t stream) {
  if (dir != THD_ZIGZAG_TO_CONTIGUOUS && dir != THD_CONTIGUOUS_TO_ZIGZAG) return THD_ERR_BAD_DIRECTION;
  if (!route_args_ok(T, cp_size) || !cu_seqlens_padded || !d_status || num_docs < 0 ||
      num_docs > kMaxRows - 1 || !route_ok(route))
    return THD_ERR_INVALID_ARG;
  if (route->total_rows != T || route->cp_size != cp_size || route->dir != dir) return THD_ERR_INVALID_ARG;
  const bool z2c = dir == THD_ZIGZAG_TO_CONTIGUOUS;
  return launch_route_build(cu_seqlens_padded, num_docs, static_cast<int32_t>(T), cp_size, z2c ? 1 : 2,
                            z2c ? route : nullptr, z2c ? nullptr : route, d_status, stream);
}

thd_status_t thd_route_build_pair(const int32_t* cu_seqlens_padded, int32_t num_docs, int64_t T, int32_t cp_size,
                                  const thd_route_t* route_z2c, const thd_route_t* route_c2z, int32_t* d_status,
                                  cudaStream_t stream) {
  if (!route_args_ok(T, cp_size) || !cu_seqlens_padded || !d_status || num_docs < 0 ||
      num_docs > kMaxRows - 1 || !route_ok(route_z2c) || !route_ok(route_c2z))
    return THD_ERR_INVALID_ARG;
  if (route_z2c->dir != THD_ZIGZAG_TO_CONTIGUOUS || route_c2z->dir != THD_CONTIGUOUS_TO_ZIGZAG)
    return THD_ERR_BAD_DIRECTION;
  if (route_z2c->total_rows != T || route_c2z->total_rows != T || route_z2c->cp_size != cp_size ||
      route_c2z->cp_size != cp_size)
    return THD_ERR_INVALID_ARG;
  return launch_route_build(cu_seqlens_padded, num_docs, static_cast<int32_t>(T), cp_size, 3, route_z2c,
                            route_c2z, d_status, stream);
}

thd_status_t thd_partition_indices(const int32_t* cu_seqlens_padded, int32_t num_docs, int64_t T,
                                   int32_t cp_size, int32_t cp_rank, int32_t* out, int32_t* d_status,
                                   cudaStream_t stream) {
  if (!route_args_ok(T, cp_size) || !cu_seqlens_padded || !d_status || num_docs < 0 ||
      num_docs > kMaxRows - 1 || cp_rank < -1 || cp_rank >= cp_size || (T > 0 && !out))
    return THD_ERR_INVALID_ARG;
  return launch_partition(cu_seqlens_padded, num_docs, static_cast<int32_t>(T), cp_size, cp_rank, out,
                          d_status, stream);
}

thd_status_t thd_swap(const void* src, void* dst, int64_t row_bytes, const thd_route_t* route,
                      int32_t* d_status, cudaStream_t stream) {
  return copy_entry(COPY_SWAP, src, dst, row_bytes, route, d_status, stream);
}

thd_status_t thd_swap_batched(const void* src, void* dst, int64_t outer, int64_t row_bytes,
                              const thd_route_t* route, int32_t* d_status, cudaStream_t stream) {
  if (!route_ok(route) || row_bytes <= 0 || row_bytes > kMaxRowBytes || outer < 0) return THD_ERR_INVALID_ARG;
  if (outer * route->total_rows > kMaxRows) return THD_ERR_INVALID_ARG;
  const int64_t bytes = outer * route->total_rows * row_bytes;
  if (bytes > 0 && (!src || !dst)) return THD_ERR_INVALID_ARG;
  if (ranges_overlap(src, dst, bytes)) return THD_ERR_INVALID_ARG;
  return launch_swap_batched(src, dst, static_cast<int32_t>(outer), row_bytes, route, d_status, stream);
}

thd_status_t thd_pack_rank(const void* src_shard, void* send_buf, int32_t cp_rank, int64_t row_bytes,
                           const thd_route_t* route, int32_t* d_status, cudaStream_t stream) {
  return rank_copy_entry(false, src_shard, send_buf, cp_rank, row_bytes, route, d_status, stream);
}

thd_status_t thd_scatter_rank(const void* recv_buf, void* dst_shard, int32_t cp_rank, int64_t row_bytes,
                              const thd_route_t* route, int32_t* d_status, cudaStream_t stream) {
  return rank_copy_entry(true, recv_buf, dst_shard, cp_rank, row_bytes, route, d_status, stream);
}

thd_status_t thd_pack(const void* src, void* send_buf, int64_t row_bytes, const thd_route_t* route,
                      int32_t* d_status, cudaStream_t stream) {
  return copy_entry(COPY_PACK, src, send_buf, row_bytes, route, d_status, stream);
}

thd_status_t thd_a2a_local(const void* send_buf, void* recv_buf, int64_t row_bytes, const thd_route_t* route,
                           int32_t* d_status, cudaStream_t stream) {
  return copy_entry(COPY_A2A, send_buf, recv_buf, row_bytes, route, d_status, stream);
}

thd_status_t thd_scatter(const void* recv_buf, void* dst, int64_t row_bytes, const thd_route_t* route,
                         int32_t* d_status, cudaStream_t stream) {
  return copy_entry(COPY_SCATTER, recv_buf, dst, row_bytes, route, d_status, stream);
}

thd_status_t thd_ulysses_swap(const void* src, void* dst, int64_t T, int32_t cp_size, int64_t row_bytes,
                              thd_ulysses_dir_t dir, int32_t* d_status, cudaStream_t stream) {
  if (dir != THD_SEQ_TO_HEAD && dir != THD_HEAD_TO_SEQ) return THD_ERR_BAD_DIRECTION;
  if (cp_size < 1 || cp_size > THD_MAX_CP || T < 0 || T % cp_size != 0 || T * cp_size > kMaxRows ||
      row_bytes <= 0 || row_bytes > kMaxRowBytes || row_bytes % cp_size != 0)
    return THD_ERR_INVALID_ARG;
  const int64_t bytes = T * row_bytes;
  if (bytes > 0 && (!src || !dst)) return THD_ERR_INVALID_ARG;
  if (ranges_overlap(src, dst, bytes)) return THD_ERR_INVALID_ARG;
  return launch_ulysses(src, dst, static_cast<int32_t>(T), cp_size, row_bytes, dir == THD_SEQ_TO_HEAD, d_status,
                        stream);
}

thd_status_t thd_roll_labels(const int32_t* tokens, const int32_t* cu_seqlens, const int32_t* cu_seqlens_padded,
                             int32_t num_docs, int64_t T, int32_t mtp_depth, int32_t fill,
                             const int32_t* next_token, const uint8_t* has_next, int32_t* labels,
                             uint8_t* loss_mask, uint8_t* valid_mask, int32_t* d_status, cudaStream_t stream) {
  if ((next_token == nullptr) != (has_next == nullptr)) return THD_ERR_INVALID_ARG;
  if (T < 0 || T > kMaxRows || num_docs < 0 || num_docs > kMaxRows - 1 || mtp_depth < 0 || mtp_depth > 64 ||
      !cu_seqlens || !cu_seqlens_padded || !d_status)
    return THD_ERR_INVALID_ARG;
  if (T > 0 && (!tokens || !labels || !loss_mask || !valid_mask)) return THD_ERR_INVALID_ARG;
  return launch_roll_labels(tokens, cu_seqlens, cu_seqlens_padded, num_docs, static_cast<int32_t>(T), mtp_depth,
                            fill, next_token, has_next, labels, loss_mask, valid_mask, d_status, stream);
}

thd_status_t thd_roll_labels_zigzag(const int32_t* tokens, const int32_t* cu_seqlens,
                                    const int32_t* cu_seqlens_padded, int32_t num_docs, int64_t T, int32_t cp_size,
                                    int32_t mtp_depth, int32_t fill, const int32_t* next_token,
                                    const uint8_t* has_next, int32_t* labels, uint8_t* loss_mask,
                                    uint8_t* valid_mask, int32_t* d_status, cudaStream_t stream) {
  if ((next_token == nullptr) != (has_next == nullptr)) return THD_ERR_INVALID_ARG;
  if (!route_args_ok(T, cp_size) || num_docs < 0 || num_docs > kMaxRows - 1 || mtp_depth < 0 || mtp_depth > 64 ||
      !cu_seqlens || !cu_seqlens_padded || !d_status)
    return THD_ERR_INVALID_ARG;
  if (T > 0 && (!tokens || !labels || !loss_mask || !valid_mask)) return THD_ERR_INVALID_ARG;
  return launch_roll_labels_zigzag(tokens, cu_seqlens, cu_seqlens_padded, num_docs, static_cast<int32_t>(T),
                                   cp_size, mtp_depth, fill, next_token, has_next, labels, loss_mask, valid_mask,
                                   d_status, stream);
}

size_t thd_pack_docs_workspace_bytes(int32_t B, int64_t S) {
  return (B < 0 || S < 0) ? 0 : pack_docs_chunked_workspace(B, S);
}

thd_status_t thd_pack_docs(const int32_t* raw, int32_t B, int64_t S, int32_t eod_id, int32_t trim_raw_pad,
                           int32_t raw_pad_id, int32_t align, int32_t pad_id, const int32_t* row_next,
                           int32_t* tokens_out, int64_t tokens_capacity, int32_t* cu_seqlens,
                           int32_t* cu_seqlens_padded, int32_t* next_token, uint8_t* has_next,
                           int64_t docs_capacity, int64_t* counts, void* workspace, size_t workspace_bytes,
                           int32_t* d_status, cudaStream_t stream) {
  if ((next_token == nullptr) != (has_next == nullptr) || (row_next && !has_next)) return THD_ERR_INVALID_ARG;
  if (B < 0 || B > kMaxRawRows || S < 0 || S > kMaxRows || align < 1 || tokens_capacity < 0 ||
      docs_capacity < 1 || !cu_seqlens || !cu_seqlens_padded || !counts || !d_status)
    return THD_ERR_INVALID_ARG;
  if (B > 0 && S > 0 && (!raw || !tokens_out)) return THD_ERR_INVALID_ARG;
  if (B > 0 && (!workspace || workspace_bytes < thd_pack_docs_workspace_bytes(B, S) ||
                reinterpret_cast<uintptr_t>(workspace) % 8 != 0))
    return THD_ERR_INVALID_ARG;
  return launch_pack_docs(raw, B, S, eod_id, trim_raw_pad ? 1 : 0, raw_pad_id, align, pad_id, row_next, tokens_out,
                          tokens_capacity, cu_seqlens, cu_seqlens_padded, next_token, has_next, docs_capacity,
                          counts, static_cast<int64_t*>(workspace), d_status, stream);
}

thd_status_t thd_status_clear(int32_t* d_status, cudaStream_t stream) {
  if (!d_status) return THD_ERR_INVALID_ARG;
  cudaError_t e = cudaMemsetAsync(d_status, 0, sizeof(int32_t), stream);
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return THD_ERR_CUDA;
  }
  return THD_OK;
}

thd_status_t thd_status_read(const int32_t* d_status, int32_t* host_code, cudaStream_t stream) {
  if (!d_status || !host_code) return THD_ERR_INVALID_ARG;
  cudaError_t e = cudaMemcpyAsync(host_code, d_status, sizeof(int32_t), cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return THD_ERR_CUDA;
  }
  return THD_OK;
}

const char* thd_status_string(int32_t code) {
  switch (code) {
    case THD_OK: return "ok";
    case THD_ERR_INVALID_ARG: return "invalid argument";
    case THD_ERR_BAD_DIRECTION: return "invalid THD layout direction";
    case THD_ERR_CU_NONZERO_START: return "cu_seqlens must start at 0";
    case THD_ERR_CU_NON_MONOTONE: return "cu_seqlens must be monotone non-decreasing";
    case THD_ERR_LEN_NOT_DIVISIBLE:
      return "sequence length not divisible by 2*cp for zigzag/contiguous THD partitioning";
    case THD_ERR_TOTAL_MISMATCH: return "cu_seqlens[-1] does not equal the number of rows";
    case THD_ERR_TIMEOUT: return "timeout";
    case THD_ERR_CUDA: return "CUDA error";
    case THD_ERR_INDEX_RANGE: return "route index out of range";
    case THD_ERR_VALID_EXCEEDS_PADDED: return "unpadded sequence length exceeds padded length";
    case THD_ERR_CAPACITY: return "output capacity exceeded";
    case THD_ERR_SCRATCH_LIMIT: return "request exceeds the fixed scratch of the no-allocation entry point";
    default: return "unknown status";
  }
}

int32_t thd_last_cuda_error(void) { return g_last_cuda_error; }

int32_t thd_version(void) { return 100; }

}  // extern "C"
