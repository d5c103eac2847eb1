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

// Loads each thread keeps in flight while staging an array in shared memory.
// Stores to shared memory cannot move above later global loads (a generic
// pointer might alias shared memory), so a loop of one load and one store
// per step would pay one memory round trip per step.
constexpr int kStageBatch = 8;

// Copy src[0, count) into shared memory, kStageBatch loads in flight per
// thread before their stores (no barrier).
__device__ __forceinline__ void stage_rows(const int32_t* src, int32_t count, int32_t* smem) {
  const uint32_t uc = static_cast<uint32_t>(count), bd = blockDim.x;
  for (uint32_t base = threadIdx.x; base < uc; base += kStageBatch * bd) {
    int32_t v[kStageBatch];
#pragma unroll
    for (int k = 0; k < kStageBatch; ++k) {
      const uint32_t i = base + k * bd;
      v[k] = i < uc ? src[i] : 0;
    }
#pragma unroll
    for (int k = 0; k < kStageBatch; ++k) {
      const uint32_t i = base + k * bd;
      if (i < uc) smem[i] = v[k];
    }
  }
}

// Read the status word (one thread) while the block copies the n+1
// boundaries into shared memory (when they fit), under one barrier.  Returns
// true when the status word was already set; *view is the array to search.
__device__ __forceinline__ bool stage_cu_check_status(const int32_t* cu, int32_t n, int32_t* smem,
                                                      bool to_smem, const int32_t* st,
                                                      const int32_t** view) {
  __shared__ int32_t flag;
  if (threadIdx.x == 0) flag = status_load(st);
  if (to_smem) stage_rows(cu, n + 1, smem);
  __syncthreads();
  *view = to_smem ? smem : cu;
  return flag != 0;
}

// Copy n+1 boundaries into shared memory (when they fit) and return the view
// the kernel should search.
__device__ __forceinline__ const int32_t* stage_cu(const int32_t* cu, int32_t n, int32_t* smem, bool to_smem) {
  if (!to_smem) return cu;
  stage_rows(cu, n + 1, smem);
  __syncthreads();
  return smem;
}

// Returned by stage_check_cu when the status word was already set.
constexpr int32_t kStatusWasSet = -1;

// Stage the n+1 boundaries in shared memory (when to_smem), validate them and
// read the status word under a single barrier when nothing is wrong: every
// thread loads a batch of boundary pairs (cu[i], cu[i+1]) at once, checks them
// in registers (monotone, length divisible by mult >= 1) and keeps cu[i].
// Returns kStatusWasSet when the status word was already non-zero, else the
// first failing check in block_check_cu's order (cu[0] != 0, non-monotone,
// not divisible, cu[n] != T), THD_OK when none.  Block-uniform.
__device__ __forceinline__ int32_t stage_check_cu(const int32_t* cu, int32_t n, int32_t* smem, bool to_smem,
                                                  const int32_t* st, int64_t T, int32_t mult) {
  __shared__ int32_t flag;
  if (threadIdx.x == 0) flag = status_load(st);
  const bool pow2 = (mult & (mult - 1)) == 0;
  const uint32_t um = static_cast<uint32_t>(mult), un = static_cast<uint32_t>(n), bd = blockDim.x;
  int mono_bad = 0, div_bad = 0;
  // the last boundary is loaded up front: a load after the loop's shared
  // stores would cost one more round trip before the barrier
  const int32_t last = (to_smem && threadIdx.x == 0) ? cu[n] : 0;
  for (uint32_t base = threadIdx.x; base < un; base += kStageBatch * bd) {
    int32_t lo[kStageBatch], hi[kStageBatch];
#pragma unroll
    for (int k = 0; k < kStageBatch; ++k) {
      const uint32_t i = base + k * bd;
      lo[k] = i < un ? cu[i] : 0;
      hi[k] = i < un ? cu[i + 1] : 0;
    }
#pragma unroll
    for (int k = 0; k < kStageBatch; ++k) {
      const uint32_t i = base + k * bd;
      if (i < un) {
        // b - a of b >= a fits 32 unsigned bits whatever the values are
        const uint32_t len = static_cast<uint32_t>(hi[k]) - static_cast<uint32_t>(lo[k]);
        if (hi[k] < lo[k]) mono_bad = 1;
        else if ((pow2 ? (len & (um - 1)) : (len % um)) != 0) div_bad = 1;
        if (to_smem) smem[i] = lo[k];
      }
    }
  }
  if (to_smem && threadIdx.x == 0) smem[n] = last;
  const int any_bad = __syncthreads_or(mono_bad | div_bad);
  if (flag != 0) return kStatusWasSet;
  const int32_t* v = to_smem ? smem : cu;
  if (v[0] != 0) return THD_ERR_CU_NONZERO_START;
  if (any_bad) return __syncthreads_or(mono_bad) ? THD_ERR_CU_NON_MONOTONE : THD_ERR_LEN_NOT_DIVISIBLE;
  if (static_cast<int64_t>(v[n]) != T) return THD_ERR_TOTAL_MISMATCH;
  return THD_OK;
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

// Largest i in [0, n] with cu[i] <= x, given cu[0] <= x, by the whole warp
// (every lane calls it with the same x): each round the lanes test 32
// evenly spaced candidates of the bracket and the last one that passes
// narrows it, so n + 1 = 4097 boundaries take 3 rounds instead of 12 halvings.
// cu non-decreasing makes the passing candidates a prefix of the lanes.
__device__ __forceinline__ int32_t warp_doc_of(const int32_t* cu, int32_t n, int32_t x) {
  const int32_t lane = threadIdx.x & 31;
  int32_t lo = 0, len = n + 1;  // the answer lies in [lo, lo + len)
  while (len > 1) {
    const int32_t stride = (len + 31) >> 5;
    const int32_t off = lane * stride;
    const bool ok = off < len && cu[lo + off] <= x;
    const uint32_t b = __ballot_sync(kFullMask, ok);  // bit 0 set: cu[lo] <= x
    const int32_t k = 31 - __clz(b);
    lo += k * stride;
    len = min(stride, len - k * stride);
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

// ---------------------------------------------------------------------------
// walking the zigzag layout in slot tiles
// ---------------------------------------------------------------------------

// Every rank's zigzag shard has the same shape: document i fills local slots
// [cu[i]/cp, cu[i+1]/cp) of each rank, its front chunk first, then its back
// chunk.  Only the chunk indices depend on the rank, so the global row of
// rank r at slot j is base_j + r*step_j with
//   front (loc = j - cu[i]/cp < c):  base = cu[i] + loc,            step = +c
//   back:                            base = cu[i] + (2cp-2)*c + loc, step = -c
// (chunk r at offset loc, or chunk 2cp-1-r at offset loc-c).  A warp finds
// the documents of 32 consecutive slots (a slot tile) once and serves every
// rank from them.  Work items are (tile, rank) pairs, q = tile*cp + r; a warp
// takes an equal contiguous share of them, so it visits few tiles and all or
// most ranks of each.
struct SlotTile {
  int32_t j;           // this lane's slot, clamped to S-1 in the last tile
  bool valid;          // the lane's slot is below S (clamped lanes must not store)
  int32_t doc;         // document holding slot j
  int32_t base, step;  // rank r's global row: base + r*step
  int32_t c0, c1;      // the document's rows [c0, c1)
};

// Documents of the slots of tile `tile` (every lane of the warp calls it
// with the same tile).  `wdoc` carries the document of the previous tile's
// lowest slot (-1 before the first): tiles only move forward, so the next
// one is found by galloping from there.  Slots are kept below S without
// forming tile*32 + 31, which could pass INT32_MAX when S is near 2^31.
__device__ __forceinline__ SlotTile slot_tile(const int32_t* cu, int32_t n, CpMath m, int32_t S,
                                              int32_t tile, int32_t& wdoc) {
  const int32_t lane = threadIdx.x & 31;
  const int32_t j0 = tile * 32;  // tile < ceil(S/32), so j0 <= S - 1
  const int32_t left = S - 1 - j0;
  SlotTile t;
  t.valid = lane <= left;
  t.j = j0 + min(lane, left);
  const int32_t x_lo = j0 * m.cp, x_hi = (j0 + min(31, left)) * m.cp;
  const int32_t i_lo = wdoc < 0 ? warp_doc_of(cu, n, x_lo) : doc_from(cu, n, wdoc, x_lo);
  const int32_t i_hi = doc_from(cu, n, i_lo, x_hi);
  wdoc = i_lo;
  const int32_t i = doc_in(cu, i_lo, i_hi, t.j * m.cp);
  const int32_t c0 = cu[i], c1 = cu[i + 1];
  const int32_t c = m.div2(c1 - c0);
  const int32_t loc = t.j - m.div(c0);
  const bool front = loc < c;
  t.doc = i;
  t.c0 = c0;
  t.c1 = c1;
  t.base = front ? c0 + loc : c0 + (2 * m.cp - 2) * c + loc;
  t.step = front ? c : -c;
  return t;
}

// The warp's share [begin, end) of `total` work items: equal contiguous
// shares, at least `min_per_warp` items each (later warps may get none).
__device__ __forceinline__ void warp_items(int64_t total, int64_t min_per_warp, int64_t* begin, int64_t* end) {
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  int64_t per = (total + nwarps - 1) / nwarps;
  if (per < min_per_warp) per = min_per_warp;
  *begin = min(total, warp * per);
  *end = min(total, *begin + per);
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
// outer independent [T][row] blocks through one route (outer * T < 2^31)
thd_status_t launch_swap_batched(const void* src, void* dst, int32_t outer, int64_t row_bytes,
                                 const thd_route_t* route, int32_t* status, cudaStream_t s);
// one rank's pack (scatter = false) or scatter on [S][row] shards
thd_status_t launch_rank_copy(bool scatter, const void* src, void* dst, int32_t rank, int64_t row_bytes,
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
