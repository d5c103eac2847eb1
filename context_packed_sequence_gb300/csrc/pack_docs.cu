// Pack raw [B, S] rows into one padded THD sequence on the device.
//
// "Packed Sequence 与上下文并行", section 2.2 (pack: split rows at EOD, pad
// every document to the alignment, flatten with document i starting at
// cu_seqlens_padded[i]) and the worked example of section 3.  The pages do it
// with bincount/cumsum and a per-document copy loop on the host side of the
// framework; here two kernels, one block per raw row:
//
//  1. stats: the row's valid end, its document count and its padded length
//     (a block-wide max-scan of document ends gives each document's start);
//  2. emit: every block derives its row's output offset from the stats of the
//     rows before it, rescans its row and writes tokens, padding and both
//     boundary arrays.
//
// The only scratch is 4 int64 per row between the two kernels.
#include "thd_internal.cuh"

namespace thd {
namespace {

constexpr int kPackThreads = 1024;
constexpr int kItems = 8;  // consecutive tokens per thread per tile
constexpr int64_t kTile = static_cast<int64_t>(kPackThreads) * kItems;

__device__ __forceinline__ int64_t pad_of(int64_t L, int32_t align) {
  int64_t r = L % align;
  return r == 0 ? 0 : align - r;
}

__device__ __forceinline__ bool is_end(const int32_t* row, int64_t t, int64_t ve, int32_t eod) {
  return row[t] == eod || t == ve - 1;
}

__device__ __forceinline__ int64_t block_sum(int64_t v, int64_t* tmp) {
  int64_t total;
  block_exclusive_scan(v, OpSum(), static_cast<int64_t>(0), tmp, &total);
  return total;
}

__device__ int64_t row_valid_end(const int32_t* row, int64_t S, int32_t trim, int32_t raw_pad,
                                 int64_t* tmp) {
  if (!trim) return S;
  int64_t m = 0;
  for (int64_t t = threadIdx.x; t < S; t += blockDim.x)
    if (row[t] != raw_pad) m = t + 1;
  int64_t total;
  block_exclusive_scan(m, OpMax(), static_cast<int64_t>(0), tmp, &total);
  return total;
}

__global__ void __launch_bounds__(kPackThreads)
pack_stats_kernel(const int32_t* raw, int64_t S, int32_t eod, int32_t trim, int32_t raw_pad,
                  int32_t align, int64_t* ws, int32_t* status) {
  __shared__ int64_t tmp[32];
  if (block_status_set(status)) return;
  const int64_t b = blockIdx.x;
  const int32_t* row = raw + b * S;
  const int64_t ve = row_valid_end(row, S, trim, raw_pad, tmp);
  int64_t carry_end = -1, docs = 0, padded = 0;
  for (int64_t base = 0; base < ve; base += kTile) {
    const int64_t t0 = base + static_cast<int64_t>(threadIdx.x) * kItems;
    int64_t my_last = -1;
    for (int it = 0; it < kItems; ++it) {
      int64_t t = t0 + it;
      if (t < ve && is_end(row, t, ve, eod)) my_last = t;
    }
    int64_t tile_last;
    int64_t prev = block_exclusive_scan(my_last, OpMax(), static_cast<int64_t>(-1), tmp, &tile_last);
    prev = max(prev, carry_end);
    int64_t cnt = 0, psum = 0;
    for (int it = 0; it < kItems; ++it) {
      int64_t t = t0 + it;
      if (t < ve && is_end(row, t, ve, eod)) {
        int64_t L = t - prev;
        psum += L + pad_of(L, align);
        ++cnt;
        prev = t;
      }
    }
    docs += block_sum(cnt, tmp);
    padded += block_sum(psum, tmp);
    carry_end = max(carry_end, tile_last);
  }
  if (threadIdx.x == 0) {
    ws[b * 4 + 0] = ve;
    ws[b * 4 + 1] = docs;
    ws[b * 4 + 2] = padded;
    ws[b * 4 + 3] = 0;
  }
}

__global__ void __launch_bounds__(kPackThreads)
pack_emit_kernel(const int32_t* raw, int32_t B, int64_t S, int32_t eod, int32_t align, int32_t pad_id,
                 int32_t* tokens, int64_t tok_cap, int32_t* cu_v, int32_t* cu, int64_t docs_cap,
                 int64_t* counts, const int64_t* ws, int32_t* status) {
  __shared__ int64_t tmp[32];
  if (block_status_set(status)) return;
  const int64_t b = blockIdx.x;
  // where this row starts: sums over the rows before it, and the grand totals
  int64_t d_before = 0, t_before = 0, v_before = 0, d_all = 0, t_all = 0;
  for (int64_t r = threadIdx.x; r < B; r += blockDim.x) {
    int64_t ve = ws[r * 4 + 0], nd = ws[r * 4 + 1], np = ws[r * 4 + 2];
    if (r < b) {
      d_before += nd;
      t_before += np;
      v_before += ve;
    }
    d_all += nd;
    t_all += np;
  }
  d_before = block_sum(d_before, tmp);
  t_before = block_sum(t_before, tmp);
  v_before = block_sum(v_before, tmp);
  d_all = block_sum(d_all, tmp);
  t_all = block_sum(t_all, tmp);
  const bool over = d_all + 1 > docs_cap || t_all > tok_cap || t_all > INT32_MAX;
  if (b == 0 && threadIdx.x == 0) {
    counts[0] = d_all;
    counts[1] = t_all;
    if (over) {
      status_set(status, THD_ERR_CAPACITY);
    } else {
      cu[0] = 0;
      cu_v[0] = 0;
    }
  }
  if (over) return;

  const int32_t* row = raw + b * S;
  const int64_t ve = ws[b * 4 + 0];
  int64_t carry_end = -1, row_docs = 0, row_pad = 0;
  for (int64_t base = 0; base < ve; base += kTile) {
    const int64_t t0 = base + static_cast<int64_t>(threadIdx.x) * kItems;
    int64_t my_last = -1;
    for (int it = 0; it < kItems; ++it) {
      int64_t t = t0 + it;
      if (t < ve && is_end(row, t, ve, eod)) my_last = t;
    }
    int64_t tile_last;
    int64_t first_prev = block_exclusive_scan(my_last, OpMax(), static_cast<int64_t>(-1), tmp, &tile_last);
    first_prev = max(first_prev, carry_end);
    int64_t cnt = 0, psum = 0;
    {
      int64_t prev = first_prev;
      for (int it = 0; it < kItems; ++it) {
        int64_t t = t0 + it;
        if (t < ve && is_end(row, t, ve, eod)) {
          int64_t L = t - prev;
          psum += L + pad_of(L, align);
          ++cnt;
          prev = t;
        }
      }
    }
    int64_t tile_cnt, tile_psum;
    int64_t cnt_before = block_exclusive_scan(cnt, OpSum(), static_cast<int64_t>(0), tmp, &tile_cnt);
    int64_t psum_before = block_exclusive_scan(psum, OpSum(), static_cast<int64_t>(0), tmp, &tile_psum);
    {
      int64_t prev = first_prev;
      int64_t doc = d_before + row_docs + cnt_before;     // document the next token belongs to
      int64_t out = t_before + row_pad + psum_before;     // that document's first output row
      for (int it = 0; it < kItems; ++it) {
        int64_t t = t0 + it;
        if (t >= ve) break;
        int32_t v = row[t];
        tokens[out + (t - prev - 1)] = v;
        if (v == eod || t == ve - 1) {
          int64_t L = t - prev;
          int64_t P = L + pad_of(L, align);
          for (int64_t z = L; z < P; ++z) tokens[out + z] = pad_id;
          cu_v[doc + 1] = static_cast<int32_t>(v_before + t + 1);
          cu[doc + 1] = static_cast<int32_t>(out + P);
          ++doc;
          out += P;
          prev = t;
        }
      }
    }
    row_docs += tile_cnt;
    row_pad += tile_psum;
    carry_end = max(carry_end, tile_last);
  }
}

}  // namespace

thd_status_t launch_pack_docs(const int32_t* raw, int32_t B, int64_t S, int32_t eod, int32_t trim,
                              int32_t raw_pad, int32_t align, int32_t pad_id, int32_t* tokens,
                              int64_t tok_cap, int32_t* cu_v, int32_t* cu, int64_t docs_cap,
                              int64_t* counts, int64_t* ws, int32_t* status, cudaStream_t s) {
  cudaError_t e;
  if (B == 0) {
    // no rows: no documents, T = 0
    if ((e = cudaMemsetAsync(counts, 0, 2 * sizeof(int64_t), s)) != cudaSuccess ||
        (e = cudaMemsetAsync(cu, 0, sizeof(int32_t), s)) != cudaSuccess ||
        (e = cudaMemsetAsync(cu_v, 0, sizeof(int32_t), s)) != cudaSuccess) {
      record_cuda_error(e);
      return THD_ERR_CUDA;
    }
    return THD_OK;
  }
  pack_stats_kernel<<<B, kPackThreads, 0, s>>>(raw, S, eod, trim, raw_pad, align, ws, status);
  if ((e = cudaGetLastError()) != cudaSuccess) {
    record_cuda_error(e);
    return THD_ERR_CUDA;
  }
  pack_emit_kernel<<<B, kPackThreads, 0, s>>>(raw, B, S, eod, align, pad_id, tokens, tok_cap, cu_v, cu,
                                              docs_cap, counts, ws, status);
  if ((e = cudaGetLastError()) != cudaSuccess) {
    record_cuda_error(e);
    return THD_ERR_CUDA;
  }
  return THD_OK;
}

}  // namespace thd
