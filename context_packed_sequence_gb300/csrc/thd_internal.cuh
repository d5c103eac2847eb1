// Internal helpers shared by the libthd translation units (not installed).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "thd.h"

namespace thd {

constexpr unsigned kFullMask = 0xffffffffu;

// ---------------------------------------------------------------------------
// status word
// ---------------------------------------------------------------------------

__device__ __forceinline__ int32_t status_load(const int32_t* st) {
  return st ? *reinterpret_cast<const volatile int32_t*>(st) : 0;
}

// Block-uniform "is the status word already set?": one thread reads, the
// whole block sees the same answer, so kernels with barriers may return on it.
__device__ __forceinline__ bool block_status_set(const int32_t* st) {
  __shared__ int32_t flag;
  if (threadIdx.x == 0) flag = status_load(st);
  __syncthreads();
  return flag != 0;
}

// First error wins: only a zero word is replaced.
__device__ __forceinline__ void status_set(int32_t* st, int32_t code) {
  if (st) atomicCAS(st, 0, code);
}

// ---------------------------------------------------------------------------
// boundary search: largest i in [0, n] with cu[i] <= x, for cu[0] <= x.
// For x < cu[n] the answer is a non-empty document (cu[i+1] > x), so empty
// documents (repeated boundaries) are skipped by construction.
// ---------------------------------------------------------------------------

__device__ __forceinline__ int32_t doc_of(const int32_t* cu, int32_t n, int32_t x) {
  int32_t lo = 0, len = n + 1;
  // branch-light lower search over [0, n]: keep lo with cu[lo] <= x
  while (len > 1) {
    int32_t half = len >> 1;
    int32_t mid = lo + half;
    lo = (cu[mid] <= x) ? mid : lo;
    len -= half;
  }
  return lo;
}

// Boundary checks shared by the route, partition and label kernels.  Every
// thread of the block gets the same code; the order of precedence is
// cu[0] != 0, then non-monotone, then (mult > 0) a length not divisible by
// mult, then (check_total) cu[n] != T.
__device__ __forceinline__ int32_t block_check_cu(const int32_t* cu, int32_t n, int64_t T, int32_t mult,
                                                  bool check_total) {
  int mono_bad = 0, div_bad = 0;
  for (int32_t i = threadIdx.x; i < n; i += blockDim.x) {
    int32_t a = cu[i], b = cu[i + 1];
    if (b < a) mono_bad = 1;
    else if (mult > 0 && ((b - a) % mult) != 0) div_bad = 1;
  }
  int any_mono = __syncthreads_or(mono_bad);
  int any_div = __syncthreads_or(div_bad);
  if (cu[0] != 0) return THD_ERR_CU_NONZERO_START;
  if (any_mono) return THD_ERR_CU_NON_MONOTONE;
  if (any_div) return THD_ERR_LEN_NOT_DIVISIBLE;
  if (check_total && static_cast<int64_t>(cu[n]) != T) return THD_ERR_TOTAL_MISMATCH;
  return THD_OK;
}

// Copy n+1 boundaries into shared memory (when they fit) and return the view
// the kernel should search.
__device__ __forceinline__ const int32_t* stage_cu(const int32_t* cu, int32_t n, int32_t* smem, bool to_smem) {
  if (!to_smem) return cu;
  for (int32_t i = threadIdx.x; i <= n; i += blockDim.x) smem[i] = cu[i];
  __syncthreads();
  return smem;
}

// ---------------------------------------------------------------------------
// zigzag geometry ("Packed Sequence 与上下文并行", section 2.4)
// ---------------------------------------------------------------------------

// Global row held by rank r at zigzag slot `slot`.  Rank-local document i
// starts at slot cu[i]/cp (every padded length is a multiple of 2*cp), so the
// document is found by searching cu for slot*cp.
__device__ __forceinline__ int32_t zigzag_row(const int32_t* cu, int32_t n, int32_t cp, int32_t r,
                                              int32_t slot) {
  int32_t i = doc_of(cu, n, slot * cp);
  int32_t c0 = cu[i];
  int32_t c = (cu[i + 1] - c0) / (2 * cp);
  int32_t loc = slot - c0 / cp;
  return loc < c ? c0 + r * c + loc : c0 + (2 * cp - 1 - r) * c + (loc - c);
}

// Zigzag buffer position (r*S + slot) of global row g.
__device__ __forceinline__ int32_t zigzag_pos(const int32_t* cu, int32_t n, int32_t cp, int32_t S,
                                              int32_t g) {
  int32_t i = doc_of(cu, n, g);
  int32_t c0 = cu[i];
  int32_t c = (cu[i + 1] - c0) / (2 * cp);
  int32_t off = g - c0;
  int32_t k = off / c;
  int32_t j = off - k * c;
  int32_t r = k < cp ? k : 2 * cp - 1 - k;
  return r * S + c0 / cp + (k < cp ? j : c + j);
}

// Number of zigzag rows of rank r with global index < X (0 <= X <= T):
// earlier documents give cu[i]/cp rows, document i the clipped overlap of its
// front chunk [r*c, (r+1)*c) and back chunk [(2cp-1-r)*c, (2cp-r)*c) with
// [0, X - cu[i]).
__device__ __forceinline__ int32_t zigzag_count_below(const int32_t* cu, int32_t n, int32_t cp,
                                                      int32_t S, int32_t T, int32_t r, int32_t X) {
  if (X >= T) return S;
  int32_t i = doc_of(cu, n, X);
  int32_t c0 = cu[i];
  int32_t c = (cu[i + 1] - c0) / (2 * cp);
  int32_t off = X - c0;
  int32_t a = min(max(off - r * c, 0), c);
  int32_t b = min(max(off - (2 * cp - 1 - r) * c, 0), c);
  return c0 / cp + a + b;
}

// ---------------------------------------------------------------------------
// block-wide scans (warp shuffles, then one warp over the warp totals)
// ---------------------------------------------------------------------------

template <typename V, class Op>
__device__ __forceinline__ V block_exclusive_scan(V v, Op op, V identity, V* warp_tmp, V* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  V x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    V y = __shfl_up_sync(kFullMask, x, o);
    if (lane >= o) x = op(y, x);
  }
  if (lane == 31) warp_tmp[wid] = x;
  __syncthreads();
  if (wid == 0) {
    V w = lane < nw ? warp_tmp[lane] : identity;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      V y = __shfl_up_sync(kFullMask, w, o);
      if (lane >= o) w = op(y, w);
    }
    warp_tmp[lane] = w;
  }
  __syncthreads();
  V before_warp = wid > 0 ? warp_tmp[wid - 1] : identity;
  V before_lane = __shfl_up_sync(kFullMask, x, 1);
  if (lane == 0) before_lane = identity;
  V result = op(before_warp, before_lane);
  *total = warp_tmp[nw - 1];
  __syncthreads();
  return result;
}

struct OpSum {
  template <typename V>
  __device__ __forceinline__ V operator()(V a, V b) const { return a + b; }
};
struct OpMax {
  template <typename V>
  __device__ __forceinline__ V operator()(V a, V b) const { return a > b ? a : b; }
};

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

void record_cuda_error(cudaError_t e);
int sm_count();

// launchers (one per translation unit); return THD_OK or THD_ERR_CUDA
thd_status_t launch_route_build(const int32_t* cu, int32_t n, int32_t T, int32_t cp, int32_t dir,
                                const thd_route_t* route, int32_t* status, cudaStream_t s);
thd_status_t launch_partition(const int32_t* cu, int32_t n, int32_t T, int32_t cp, int32_t rank,
                              int32_t* out, int32_t* status, cudaStream_t s);
enum CopyKind { COPY_SWAP = 0, COPY_PACK = 1, COPY_A2A = 2, COPY_SCATTER = 3 };
thd_status_t launch_copy(CopyKind kind, const void* src, void* dst, int64_t row_bytes,
                         const thd_route_t* route, int32_t* status, cudaStream_t s);
thd_status_t launch_roll_labels(const int32_t* tokens, const int32_t* cu_v, const int32_t* cu,
                                int32_t n, int32_t T, int32_t depth, int32_t fill, int32_t* labels,
                                uint8_t* lmask, uint8_t* valid, int32_t* status, cudaStream_t s);
thd_status_t launch_pack_docs(const int32_t* raw, int32_t B, int64_t S, int32_t eod, int32_t trim,
                              int32_t raw_pad, int32_t align, int32_t pad_id, int32_t* tokens,
                              int64_t tok_cap, int32_t* cu_v, int32_t* cu, int64_t docs_cap,
                              int64_t* counts, int64_t* ws, int32_t* status, cudaStream_t s);

}  // namespace thd
