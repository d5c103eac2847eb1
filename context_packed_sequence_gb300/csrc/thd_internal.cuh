// Internal helpers shared by the libthd translation units (not installed).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "thd.h"
#include "tma.cuh"

namespace thd {

constexpr unsigned kFullMask = 0xffffffffu;

// ---------------------------------------------------------------------------
// status word
// ---------------------------------------------------------------------------

__device__ __forceinline__ int32_t status_load(const int32_t* st) {
  return st ? *reinterpret_cast<const volatile int32_t*>(st) : 0;
}

// Debug build (compiled with THD_CHECKED=1, loaded with THD_CHECKED=1 in the
// environment): every row index a kernel computes in closed form is checked
// against its range before it is used; a miss records THD_ERR_INDEX_RANGE and
// the access is skipped.  The default build compiles the checks away: the
// closed forms stay in range by construction on validated input.
#if defined(THD_CHECKED) && THD_CHECKED
constexpr bool kChecked = true;
#else
constexpr bool kChecked = false;
#endif

__device__ __forceinline__ bool in_range(int64_t v, int64_t lo, int64_t hi, int32_t* st) {
  if (!kChecked || (v >= lo && v < hi)) return true;
  if (st) atomicCAS(st, 0, static_cast<int32_t>(THD_ERR_INDEX_RANGE));
  return false;
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
  // a power-of-two multiple is tested with a mask (the usual 2*cp)
  const bool pow2 = mult > 0 && (mult & (mult - 1)) == 0;
  const uint32_t um = static_cast<uint32_t>(mult);
  // unsigned counter and length: n may be close to INT32_MAX, and b - a of
  // b >= a always fits 32 unsigned bits whatever the (unchecked) values are
  for (uint32_t i = threadIdx.x; i < static_cast<uint32_t>(n); i += blockDim.x) {
    const int32_t a = cu[i], b = cu[i + 1];
    const uint32_t len = static_cast<uint32_t>(b) - static_cast<uint32_t>(a);
    if (b < a) mono_bad = 1;
    else if (mult > 0 && (pow2 ? (len & (um - 1)) : (len % um)) != 0) div_bad = 1;
  }
  int any_mono = __syncthreads_or(mono_bad);
  int any_div = __syncthreads_or(div_bad);
  if (cu[0] != 0) return THD_ERR_CU_NONZERO_START;
  if (any_mono) return THD_ERR_CU_NON_MONOTONE;
  if (any_div) return THD_ERR_LEN_NOT_DIVISIBLE;
  if (check_total && static_cast<int64_t>(cu[n]) != T) return THD_ERR_TOTAL_MISMATCH;
  return THD_OK;
}

// Read the status word (one thread) while the block copies the n+1
// boundaries into shared memory (when they fit), under one barrier.  Returns
// true when the status word was already set; *view is the array to search.
__device__ __forceinline__ bool stage_cu_check_status(const int32_t* cu, int32_t n, int32_t* smem,
                                                      bool to_smem, const int32_t* st,
                                                      const int32_t** view) {
  __shared__ int32_t flag;
  if (threadIdx.x == 0) flag = status_load(st);
  if (to_smem) {
    // four independent loads in flight per thread before the stores
    for (int32_t base = threadIdx.x; base <= n; base += 4 * blockDim.x) {
      int32_t v[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int32_t i = base + k * static_cast<int32_t>(blockDim.x);
        v[k] = i <= n ? cu[i] : 0;
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int32_t i = base + k * static_cast<int32_t>(blockDim.x);
        if (i <= n) smem[i] = v[k];
      }
    }
  }
  __syncthreads();
  *view = to_smem ? smem : cu;
  return flag != 0;
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

// Division by cp and by 2*cp: a shift when cp is a power of two (the usual
// case), a division otherwise.  Operands are never negative.
struct CpMath {
  int32_t cp;
  int32_t shift;  // log2(cp) when cp is a power of two, else -1
  __device__ __forceinline__ int32_t div(int32_t x) const { return shift >= 0 ? x >> shift : x / cp; }
  __device__ __forceinline__ int32_t div2(int32_t x) const {
    return shift >= 0 ? x >> (shift + 1) : x / (2 * cp);
  }
};

inline CpMath make_cp_math(int32_t cp) {
  CpMath m;
  m.cp = cp;
  m.shift = -1;
  for (int b = 0; b < 31; ++b)
    if ((1 << b) == cp) m.shift = b;
  return m;
}

// floor(n / d) for 0 <= n < 2^31 and 1 <= d < 2^31 by one 64-bit multiply and
// a shift (Granlund and Montgomery, "Division by invariant integers using
// multiplication", 1994, theorem 4.2 with N = 31): l = ceil(log2 d),
// m = ceil(2^(31+l) / d) < 2^33, q = (n * m) >> (31 + l).
struct FastDiv {
  uint64_t m;
  int32_t shift;
  __device__ __forceinline__ int32_t div(int32_t n) const {
    return static_cast<int32_t>((static_cast<uint64_t>(n) * m) >> shift);
  }
};

inline FastDiv make_fast_div(int32_t d) {
  FastDiv f;
  int l = 0;
  while ((int64_t(1) << l) < d) ++l;
  f.shift = 31 + l;
  f.m = ((uint64_t(1) << f.shift) + static_cast<uint64_t>(d) - 1) / static_cast<uint64_t>(d);
  return f;
}

// Largest i in [lo, hi] with cu[i] <= x, given cu[lo] <= x.  The length is
// the same for all lanes of a warp when lo and hi are, so the loop is too.
__device__ __forceinline__ int32_t doc_in(const int32_t* cu, int32_t lo, int32_t hi, int32_t x) {
  int32_t len = hi - lo + 1;
  while (len > 1) {
    const int32_t half = len >> 1;
    lo = (cu[lo + half] <= x) ? lo + half : lo;
    len -= half;
  }
  return lo;
}

// Largest k >= i with cu[k] <= x, given cu[i] <= x: gallop forward from i
// (1, 2, 4, ... documents), then search the last bracket.  Costs O(log of the
// distance), so following a position that only moves forward is cheap.
__device__ __forceinline__ int32_t doc_from(const int32_t* cu, int32_t n, int32_t i, int32_t x) {
  int32_t step = 1;
  // written so that nothing overflows for n up to INT32_MAX - 1: the step
  // stops doubling at 2^30 and is compared with the distance left
  while (step <= n - i && cu[i + step] <= x) {
    i += step;
    if (step < (1 << 30)) step <<= 1;
  }
  return doc_in(cu, i, i + min(step - 1, n - i), x);
}

// The documents of a warp's 32 consecutive positions: one full search for
// the lowest and the highest position (lanes 0 and 1 search, everyone gets
// both answers), then a window search per lane, usually 0-2 steps.  lo_x and
// hi_x must be the same in every lane, and every lane's x in [lo_x, hi_x].
__device__ __forceinline__ int32_t warp_doc_of(const int32_t* cu, int32_t n, int32_t lo_x, int32_t hi_x,
                                               int32_t x) {
  const int lane = threadIdx.x & 31;
  const int32_t found = doc_of(cu, n, lane == 0 ? lo_x : hi_x);
  const int32_t i_lo = __shfl_sync(kFullMask, found, 0);
  const int32_t i_hi = __shfl_sync(kFullMask, found, 1);
  return doc_in(cu, i_lo, i_hi, x);
}

// Global row held by rank r at zigzag slot `slot`.  Rank-local document i
// starts at slot cu[i]/cp (every padded length is a multiple of 2*cp), so the
// document is found by searching cu for slot*cp.
__device__ __forceinline__ int32_t zigzag_row(const int32_t* cu, int32_t n, CpMath m, int32_t r,
                                              int32_t slot) {
  int32_t i = doc_of(cu, n, slot * m.cp);
  int32_t c0 = cu[i];
  int32_t c = m.div2(cu[i + 1] - c0);
  int32_t loc = slot - m.div(c0);
  return loc < c ? c0 + r * c + loc : c0 + (2 * m.cp - 1 - r) * c + (loc - c);
}

// Zigzag buffer position (r*S + slot) of global row g.
__device__ __forceinline__ int32_t zigzag_pos(const int32_t* cu, int32_t n, CpMath m, int32_t S,
                                              int32_t g) {
  int32_t i = doc_of(cu, n, g);
  int32_t c0 = cu[i];
  int32_t c = m.div2(cu[i + 1] - c0);
  int32_t off = g - c0;
  int32_t k = off / c;
  int32_t j = off - k * c;
  int32_t r = k < m.cp ? k : 2 * m.cp - 1 - k;
  return r * S + m.div(c0) + (k < m.cp ? j : c + j);
}

// Number of zigzag rows of rank r with global index < X (0 <= X <= T):
// earlier documents give cu[i]/cp rows, document i the clipped overlap of its
// front chunk [r*c, (r+1)*c) and back chunk [(2cp-1-r)*c, (2cp-r)*c) with
// [0, X - cu[i]).
__device__ __forceinline__ int32_t zigzag_count_below(const int32_t* cu, int32_t n, CpMath m,
                                                      int32_t S, int32_t T, int32_t r, int32_t X) {
  if (X >= T) return S;
  int32_t i = doc_of(cu, n, X);
  int32_t c0 = cu[i];
  int32_t c = m.div2(cu[i + 1] - c0);
  int32_t off = X - c0;
  int32_t a = min(max(off - r * c, 0), c);
  int32_t b = min(max(off - (2 * m.cp - 1 - r) * c, 0), c);
  return m.div(c0) + a + b;
}

// ---------------------------------------------------------------------------
// walking the zigzag buffer in warp tiles
// ---------------------------------------------------------------------------

// A warp walks a contiguous range of zigzag positions u = r*S + j, 32 per
// step, and keeps the document index of its lowest slot.  Within one rank
// the slots only grow, so the next tile's documents are found by galloping
// forward from there; a full search happens only at the start and where the
// walk enters another rank.
struct TileWalker {
  int32_t doc;      // document of the lowest slot of the previous tile
  int32_t rank;     // its rank (-1 before the first tile)
};

struct TileRow {
  int32_t u, r, j, g;
  int32_t doc;  // the document holding g
};

// Lanes hold positions u (clamped to last, the walk's final position, for
// the slot arithmetic; such lanes must not store).
__device__ __forceinline__ TileRow tile_row(const int32_t* cu, int32_t n, CpMath m, int32_t S, FastDiv divS,
                                            int32_t u, int32_t last, TileWalker& w) {
  TileRow t;
  t.u = u;
  const int32_t uc = min(u, last);
  t.r = divS.div(uc);
  t.j = uc - t.r * S;
  const int32_t r_first = __shfl_sync(kFullMask, t.r, 0), r_last = __shfl_sync(kFullMask, t.r, 31);
  const int32_t x_lo = __shfl_sync(kFullMask, t.j, 0) * m.cp;
  const int32_t x_hi = __shfl_sync(kFullMask, t.j, 31) * m.cp;
  const int32_t x = t.j * m.cp;
  int32_t i;
  if (r_first == r_last) {
    const int32_t i_lo = (w.rank == r_first) ? doc_from(cu, n, w.doc, x_lo) : doc_of(cu, n, x_lo);
    const int32_t i_hi = doc_from(cu, n, i_lo, x_hi);
    i = doc_in(cu, i_lo, i_hi, x);
    w.doc = i_lo;
    w.rank = r_first;
  } else {  // the tile crosses into the next rank
    i = doc_of(cu, n, x);
    w.rank = -1;
  }
  const int32_t c0 = cu[i];
  const int32_t c = m.div2(cu[i + 1] - c0);
  const int32_t loc = t.j - m.div(c0);
  t.g = loc < c ? c0 + t.r * c + loc : c0 + (2 * m.cp - 1 - t.r) * c + (loc - c);
  t.doc = i;
  return t;
}

// The warp's range of positions [begin, end) out of [0, total): equal shares,
// whole tiles of 32.
__device__ __forceinline__ void warp_range(int64_t total, int64_t* begin, int64_t* end) {
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int64_t tiles = (total + 31) / 32;
  const int64_t per = (tiles + nwarps - 1) / nwarps;
  *begin = min(total, warp * per * 32);
  *end = min(total, (warp + 1) * per * 32);
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

// Every kernel of this library is launched with programmatic stream
// serialization: it may be scheduled while the previous kernel on the stream
// is still finishing, which hides the launch gap between back-to-back
// kernels.  Each kernel's first statement is pdl_wait_then_release()
// (tma.cuh), so it touches memory only after its predecessor has completed.
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
  return e == cudaSuccess ? cudaGetLastError() : e;
}

// launchers (one per translation unit); return THD_OK or THD_ERR_CUDA
// dirs: bit 0 = zigzag->contiguous into zc, bit 1 = contiguous->zigzag into cz
thd_status_t launch_route_build(const int32_t* cu, int32_t n, int32_t T, int32_t cp, int32_t dirs,
                                const thd_route_t* zc, const thd_route_t* cz, int32_t* status,
                                cudaStream_t s);
thd_status_t launch_partition(const int32_t* cu, int32_t n, int32_t T, int32_t cp, int32_t rank,
                              int32_t* out, int32_t* status, cudaStream_t s);
enum CopyKind { COPY_SWAP = 0, COPY_PACK = 1, COPY_A2A = 2, COPY_SCATTER = 3 };
thd_status_t launch_copy(CopyKind kind, const void* src, void* dst, int64_t row_bytes,
                         const thd_route_t* route, int32_t* status, cudaStream_t s);
thd_status_t launch_ulysses(const void* src, void* dst, int32_t T, int32_t cp, int64_t row_bytes, bool seq_to_head,
                            int32_t* status, cudaStream_t s);
// tile transpose for head-group pieces below 1 KiB (multiples of 16 bytes,
// 16-byte aligned buffers); ulysses_tiles_apply says whether it takes the call
bool ulysses_tiles_apply(const void* src, const void* dst, int32_t T, int32_t cp, int64_t row_bytes,
                         bool seq_to_head);
thd_status_t launch_ulysses_tiles(const void* src, void* dst, int32_t T, int32_t cp, int64_t row_bytes,
                                  bool seq_to_head, int32_t* status, cudaStream_t s);
thd_status_t launch_roll_labels(const int32_t* tokens, const int32_t* cu_v, const int32_t* cu,
                                int32_t n, int32_t T, int32_t depth, int32_t fill, const int32_t* next_tok,
                                const uint8_t* has_next, int32_t* labels, uint8_t* lmask, uint8_t* valid,
                                int32_t* status, cudaStream_t s);
thd_status_t launch_roll_labels_zigzag(const int32_t* tokens, const int32_t* cu_v, const int32_t* cu, int32_t n,
                                       int32_t T, int32_t cp, int32_t depth, int32_t fill, const int32_t* next_tok,
                                       const uint8_t* has_next, int32_t* labels, uint8_t* lmask, uint8_t* valid,
                                       int32_t* status, cudaStream_t s);
// chunked packing (workspace: pack_docs_chunked_workspace bytes, 8-byte aligned); row_next, next_tok
// and has_next are optional (all null: no extra tokens)
size_t pack_docs_chunked_workspace(int32_t B, int64_t S);
thd_status_t launch_pack_docs(const int32_t* raw, int32_t B, int64_t S, int32_t eod, int32_t trim,
                              int32_t raw_pad, int32_t align, int32_t pad_id, const int32_t* row_next,
                              int32_t* tokens, int64_t tok_cap, int32_t* cu_v, int32_t* cu, int32_t* next_tok,
                              uint8_t* has_next, int64_t docs_cap, int64_t* counts, int64_t* ws, int32_t* status,
                              cudaStream_t s);
// one block per raw row (workspace: 4 int64 per row)
thd_status_t launch_pack_docs_rows(const int32_t* raw, int32_t B, int64_t S, int32_t eod, int32_t trim,
                                   int32_t raw_pad, int32_t align, int32_t pad_id, int32_t* tokens,
                                   int64_t tok_cap, int32_t* cu_v, int32_t* cu, int64_t docs_cap,
                                   int64_t* counts, int64_t* ws, int32_t* status, cudaStream_t s);

}  // namespace thd
