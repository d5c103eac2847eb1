// Row-permutation copies: the fused swap and the pages' three steps
// (pack -> all-to-all -> scatter, "[Task32] feat: fla mcore chunkwise cp
// stage 3", Relax PR #273, section 2.1) with every virtual rank in one buffer.
//
// Pure data movement, bound by HBM bandwidth.  One engine serves all four:
// the "linear" side (the destination of a gather, the source of a scatter) is
// walked as one flat array of copy units (16, 4 or 1 bytes); each warp takes
// 32*U consecutive units per step, so linear-side accesses are 512-byte
// coalesced runs for 16-byte units, and the mapped side reads or writes
// contiguous pieces of whole rows.  Each lane keeps (row, column) of its units
// incrementally -- no division inside the loop -- and resolves a row's partner
// once per row change.  Every partner row is range-checked; a bad one is
// skipped and reported through the status word.
#include "thd_internal.cuh"

namespace thd {
namespace {

constexpr int kCopyThreads = 256;
constexpr int kUnroll = 8;
constexpr int kCopyBlocksPerSm = 3;

// ---- memory access flavours ------------------------------------------------

__device__ __forceinline__ uint4 load_unit(const uint4* p) {
  uint4 v;
  // streamed once: read-only path, do not keep in L1
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}
__device__ __forceinline__ void store_unit(uint4* p, uint4 v) {
  // streaming store: written once, not re-read by this kernel
  asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}
__device__ __forceinline__ uint32_t load_unit(const uint32_t* p) { return __ldg(p); }
__device__ __forceinline__ void store_unit(uint32_t* p, uint32_t v) { *p = v; }
__device__ __forceinline__ uint8_t load_unit(const uint8_t* p) { return __ldg(p); }
__device__ __forceinline__ void store_unit(uint8_t* p, uint8_t v) { *p = v; }

// ---- row maps: linear-side row -> mapped-side row, or -1 when out of range --

// fused swap: target row q takes source row src_of_dst[q]
struct SwapMap {
  const int32_t* idx;
  int32_t rows;
  __device__ __forceinline__ int32_t operator()(int32_t q) const {
    int32_t v = __ldg(idx + q);
    return (v >= 0 && v < rows) ? v : -1;
  }
};

// pack (gather) and scatter: row list local to each rank of S rows
struct RankLocalMap {
  const int32_t* idx;
  int32_t S;
  __device__ __forceinline__ int32_t operator()(int32_t q) const {
    int32_t rank = q / S;
    int32_t v = __ldg(idx + q);
    return (v >= 0 && v < S) ? rank * S + v : -1;
  }
};

// all-to-all: receive row j of rank d comes from the send buffer of the rank
// s whose receive block holds j, at that block's offset in s's send buffer.
struct A2AMap {
  const int32_t* send_off;  // [s][cp+1]
  const int32_t* recv_off;  // [d][cp+1]
  const int32_t* in_split;  // [s][cp]
  int32_t cp, S;
  __device__ __forceinline__ int32_t operator()(int32_t q) const {
    int32_t d = q / S;
    int32_t j = q - d * S;
    const int32_t* ro = recv_off + d * (cp + 1);
    int32_t s = 0, len = cp;  // largest s in [0, cp) with ro[s] <= j
    while (len > 1) {
      int32_t half = len >> 1;
      s = (__ldg(ro + s + half) <= j) ? s + half : s;
      len -= half;
    }
    int32_t m = j - __ldg(ro + s);
    int32_t n = __ldg(in_split + s * cp + d);
    int32_t off = __ldg(send_off + s * (cp + 1) + d);
    if (m < 0 || m >= n || off < 0 || off + m >= S) return -1;
    return s * S + off + m;
  }
};

// ---- the engine ------------------------------------------------------------

struct Walk {
  int32_t rows;    // rows on the linear side
  int32_t upr;     // units per row
  int32_t dq32, dc32;    // 32 units expressed as (rows, units)
  int64_t step_q;        // one grid-wide step expressed as rows ...
  int32_t step_c;        // ... and units
};

__device__ __forceinline__ void advance(int64_t& q, int32_t& c, int64_t dq, int32_t dc, int32_t upr) {
  c += dc;
  q += dq;
  if (c >= upr) {
    c -= upr;
    ++q;
  }
}

template <typename Unit, class Map, bool SCATTER>
__global__ void __launch_bounds__(kCopyThreads, kCopyBlocksPerSm)
copy_rows_kernel(const Unit* __restrict__ src, Unit* __restrict__ dst, Walk w, Map map, int32_t* status) {
  if (status_load(status) != 0) return;
  const int lane = threadIdx.x & 31;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t lin0 = warp * (32 * kUnroll) + lane;
  const int64_t total = static_cast<int64_t>(w.rows) * w.upr;
  if (lin0 >= total) return;
  int64_t q = lin0 / w.upr;
  int32_t c = static_cast<int32_t>(lin0 - q * w.upr);
  bool bad = false;
  int64_t last_q = -1;
  int32_t last_o = -1;

  while (q < w.rows) {
    Unit v[kUnroll];
    int32_t o[kUnroll];
    {
      int64_t qq = q;
      int32_t cc = c;
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        o[u] = -1;
        if (qq < w.rows) {
          if (qq != last_q) {
            last_o = map(static_cast<int32_t>(qq));
            last_q = qq;
          }
          o[u] = last_o;
          if (last_o >= 0) {
            int64_t row = SCATTER ? qq : last_o;
            v[u] = load_unit(src + row * w.upr + cc);
          }
        }
        advance(qq, cc, w.dq32, w.dc32, w.upr);
      }
    }
    {
      int64_t qq = q;
      int32_t cc = c;
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        if (qq < w.rows) {
          if (o[u] >= 0) {
            int64_t row = SCATTER ? o[u] : qq;
            store_unit(dst + row * w.upr + cc, v[u]);
          } else {
            bad = true;
          }
        }
        advance(qq, cc, w.dq32, w.dc32, w.upr);
      }
    }
    advance(q, c, w.step_q, w.step_c, w.upr);
  }
  if (bad) status_set(status, THD_ERR_INDEX_RANGE);
}

template <typename Unit, class Map, bool SCATTER>
thd_status_t run(const void* src, void* dst, int32_t rows, int64_t row_bytes, Map map, int32_t* status,
                 cudaStream_t s) {
  Walk w;
  w.rows = rows;
  w.upr = static_cast<int32_t>(row_bytes / static_cast<int64_t>(sizeof(Unit)));
  w.dq32 = 32 / w.upr;
  w.dc32 = 32 % w.upr;
  const int64_t total = static_cast<int64_t>(rows) * w.upr;
  const int64_t per_block = static_cast<int64_t>(kCopyThreads) * kUnroll;
  int64_t grid = (total + per_block - 1) / per_block;
  const int64_t cap = static_cast<int64_t>(sm_count()) * kCopyBlocksPerSm;
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  const int64_t step = grid * per_block;  // units all warps advance per step
  w.step_q = step / w.upr;
  w.step_c = static_cast<int32_t>(step % w.upr);
  copy_rows_kernel<Unit, Map, SCATTER><<<static_cast<unsigned>(grid), kCopyThreads, 0, s>>>(
      static_cast<const Unit*>(src), static_cast<Unit*>(dst), w, map, status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return THD_ERR_CUDA;
  }
  return THD_OK;
}

template <class Map, bool SCATTER>
thd_status_t dispatch_unit(const void* src, void* dst, int32_t rows, int64_t row_bytes, Map map,
                           int32_t* status, cudaStream_t s) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst);
  if (row_bytes % 16 == 0 && a % 16 == 0)
    return run<uint4, Map, SCATTER>(src, dst, rows, row_bytes, map, status, s);
  if (row_bytes % 4 == 0 && a % 4 == 0)
    return run<uint32_t, Map, SCATTER>(src, dst, rows, row_bytes, map, status, s);
  return run<uint8_t, Map, SCATTER>(src, dst, rows, row_bytes, map, status, s);
}

}  // namespace

thd_status_t launch_copy(CopyKind kind, const void* src, void* dst, int64_t row_bytes,
                         const thd_route_t* r, int32_t* status, cudaStream_t s) {
  const int32_t T = static_cast<int32_t>(r->total_rows);
  const int32_t cp = r->cp_size;
  const int32_t S = T / cp;
  if (T == 0) return THD_OK;
  switch (kind) {
    case COPY_SWAP:
      return dispatch_unit<SwapMap, false>(src, dst, T, row_bytes, SwapMap{r->src_of_dst, T}, status, s);
    case COPY_PACK:
      return dispatch_unit<RankLocalMap, false>(src, dst, T, row_bytes, RankLocalMap{r->send_rows, S},
                                                status, s);
    case COPY_A2A:
      return dispatch_unit<A2AMap, false>(
          src, dst, T, row_bytes,
          A2AMap{r->send_offsets, r->recv_offsets, r->input_split_sizes, cp, S}, status, s);
    case COPY_SCATTER:
      return dispatch_unit<RankLocalMap, true>(src, dst, T, row_bytes, RankLocalMap{r->recv_rows, S},
                                               status, s);
  }
  return THD_ERR_INVALID_ARG;
}

}  // namespace thd
