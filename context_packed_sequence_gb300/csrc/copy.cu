// Row-permutation copies: the fused swap and the pages' three steps
// (pack -> all-to-all -> scatter, "[Task32] feat: fla mcore chunkwise cp
// stage 3", Relax PR #273, section 2.1) with every virtual rank in one buffer.
//
// Pure data movement, bound by HBM bandwidth.  Two engines, one row map each
// call (linear-side row -> mapped-side row, range-checked):
//
//  * bulk engine (rows of >= 208 bytes, multiples of 16, 16-byte aligned
//    buffers): one warp per block drives a ring of shared-memory stages with
//    TMA bulk copies.  The linear side is cut into chunks of up to 32 rows
//    (or row pieces); each chunk is gathered with one cp.async.bulk
//    global->shared copy per run of consecutive mapped rows, completion
//    tracked by an mbarrier, and written back with one bulk store per run.
//    The SM issues a handful of instructions per 8-16 KB moved, so the copy
//    runs at the HBM copy rate.  Every wait is bounded: a wait that runs out
//    records THD_ERR_TIMEOUT, drains its own copies and returns.  Launches use
//    programmatic dependent launch, so consecutive copies on a stream overlap
//    launch and tail.
//  * run engine (rows of 16 - 192 bytes, multiples of 16, aligned): chunks
//    of up to 512 rows; runs of rows whose mapped rows are consecutive move
//    as single bulk copies through the same kind of ring.
//  * unit engine (everything else: rows that are not multiples of 16 bytes,
//    or unaligned buffers): the linear side is walked as a flat array of 4-
//    or 1-byte units, 32*U consecutive units per warp step, (row, column)
//    kept incrementally.
//
// The Ulysses exchange takes the tile transpose of ulysses_tile.cu when its
// head-group pieces are multiples of 16 bytes below 1 KiB, these engines
// otherwise.
#include "thd_internal.cuh"
#include "tma.cuh"
#include "thd_debug.h"

namespace thd {
namespace {

constexpr int kCopyThreads = 256;
constexpr int kUnroll = 8;
constexpr int kCopyBlocksPerSm = 3;
// narrower rows: the run engine.  On GB300 the run engine leads at 160-192 B
// rows (0.88-0.93 of the copy bandwidth against 0.82-0.87 row by row), the
// bulk engine from 208 B (0.89-0.95 against 0.86-0.88).
constexpr int64_t kBulkMinRowBytes = 208;

// ---- memory access flavours ------------------------------------------------

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

// fused swap of `outer` independent [T][row] blocks through one route (a
// tensor whose sequence dim is not the first, [outer][T][row] in memory):
// target row o*T + q takes source row o*T + src_of_dst[q]
struct BatchedSwapMap {
  const int32_t* idx;
  int32_t T;
  FastDiv divT;
  __device__ __forceinline__ int32_t operator()(int32_t q) const {
    const int32_t o = divT.div(q), qq = q - o * T;
    const int32_t v = __ldg(idx + qq);
    return (v >= 0 && v < T) ? o * T + v : -1;
  }
};

// one rank's shard: linear row j <-> local row rows[j] of the same rank (the
// per-rank pack and scatter of a caller that holds only its own shard)
struct OneRankMap {
  const int32_t* idx;  // the rank's S entries
  int32_t S;
  __device__ __forceinline__ int32_t operator()(int32_t j) const {
    const int32_t v = __ldg(idx + j);
    return (v >= 0 && v < S) ? v : -1;
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
    // the route's entries are checked, not trusted: 64-bit so that corrupted
    // values cannot wrap around the checks
    const int64_t m = static_cast<int64_t>(j) - __ldg(ro + s);
    const int32_t n = __ldg(in_split + s * cp + d);
    const int32_t off = __ldg(send_off + s * (cp + 1) + d);
    if (m < 0 || m >= n || off < 0 || off + m >= S) return -1;
    return s * S + off + static_cast<int32_t>(m);
  }
};

// Ulysses head <-> sequence exchange ("Packed Sequence 与上下文并行", sections
// 2.5 and 2.7): each token row is cp pieces (head groups) of P bytes.  The
// sequence-sharded buffer is [T][cp] pieces (token-major), the head-sharded
// one [cp][T] (rank r holds every token's group r).  The linear side is the
// destination's pieces.
struct UlyssesMap {
  int32_t T, cp;
  bool seq_to_head;
  FastDiv div;  // by T (seq -> head) or by cp (head -> seq)
  __device__ __forceinline__ int32_t operator()(int32_t q) const {
    int32_t v;
    if (seq_to_head) {  // destination piece (r, g) <- source piece (g, r)
      const int32_t r = div.div(q), g = q - r * T;
      v = g * cp + r;
    } else {
      const int32_t g = div.div(q), r = q - g * cp;  // destination (g, r) <- source (r, g)
      v = r * T + g;
    }
    // checked build: -1 makes the engines skip the piece and report it
    return in_range(v, 0, static_cast<int64_t>(T) * cp, nullptr) ? v : -1;
  }
};

// ---- the unit engine -------------------------------------------------------

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
  pdl_wait_then_release();
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
  const cudaError_t e = launch_pdl(copy_rows_kernel<Unit, Map, SCATTER>, dim3(static_cast<unsigned>(grid)),
                                   kCopyThreads, 0, s, static_cast<const Unit*>(src), static_cast<Unit*>(dst), w,
                                   map, status);
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return THD_ERR_CUDA;
  }
  return THD_OK;
}


// ---- the bulk (TMA) engine -------------------------------------------------

constexpr uint32_t kFull = 0xffffffffu;

// Checked build only: a one-shot request (thd_debug_stall_next_bulk_copy)
// that block 0 of the next bulk copy arms 16 bytes no copy delivers, so its
// first wait runs out and the timeout path runs for real.
__device__ int g_stall_request;

__device__ __forceinline__ void maybe_stall(int64_t i, uint64_t* bar) {
  if (kChecked && i == 0 && blockIdx.x == 0 && atomicExch(&g_stall_request, 0) != 0) mbar_expect_tx(bar, 16);
}

// Lane `lane` starts a run in `starts`; the run ends before the next lane that
// starts another run or is not in `members`.
__device__ __forceinline__ int run_end(int lane, uint32_t starts, uint32_t members) {
  const uint32_t above = lane == 31 ? 0u : ~((2u << lane) - 1u);
  const uint32_t stop = (starts | ~members) & above;
  return stop ? __ffs(stop) - 1 : 32;
}

struct BulkGeom {
  int32_t rows;       // rows on either side
  int32_t row_bytes;
  int32_t stage;      // bytes per stage
  int32_t R;          // rows per chunk (row mode) or 1
  int32_t P;          // pieces per row (piece mode) or 1
  int64_t chunks;
};

// Shared memory: NST stages, then NST mbarriers, NST valid masks, NST x 32 mapped rows.
template <int NST, class Map, bool SCATTER>
__global__ void __launch_bounds__(32)
bulk_copy_kernel(const char* __restrict__ src, char* __restrict__ dst, BulkGeom g, Map map, int32_t* status) {
  extern __shared__ __align__(128) char smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(NST) * g.stage);
  uint32_t* masks = reinterpret_cast<uint32_t*>(bars + NST);
  int32_t* mrows = reinterpret_cast<int32_t*>(masks + NST);
  const int lane = threadIdx.x;
  pdl_wait_then_release();  // launched with programmatic dependent launch
  // one read, broadcast: the warp must take this exit together
  if (__shfl_sync(kFull, lane == 0 ? status_load(status) : 0, 0) != 0) return;
  const int64_t b = blockIdx.x, G = gridDim.x;
  const int64_t n_my = g.chunks > b ? (g.chunks - b + G - 1) / G : 0;
  if (n_my == 0) return;
  const bool row_mode = g.P == 1;
  const int64_t rb = g.row_bytes;
  if (lane == 0) {
    for (int s = 0; s < NST; ++s) mbar_init(&bars[s], 1);
    mbar_init_fence();
  }
  __syncwarp();
  bool bad = false;

  // mapped row of this lane's row of chunk i (-1: out of range, -2: no row)
  auto fetch = [&](int64_t i) -> int32_t {
    const int64_t k = b + i * G;
    const int64_t q = row_mode ? k * g.R + lane : k / g.P;
    if (row_mode && (lane >= g.R || q >= g.rows)) return -2;
    return map(static_cast<int32_t>(q));
  };

  auto issue_load = [&](int64_t i, int32_t m) {
    const int s = static_cast<int>(i % NST);
    char* st = smem + static_cast<size_t>(s) * g.stage;
    const int64_t k = b + i * G;
    bad |= (m == -1);
    if (row_mode) {
      const int64_t q0 = k * g.R;
      const bool valid = m >= 0;
      const uint32_t vmask = __ballot_sync(kFull, valid);
      bool start;
      if (SCATTER) {  // contiguous linear source: runs of valid rows
        start = valid && (lane == 0 || !((vmask >> (lane - 1)) & 1u));
      } else {        // gather: runs of consecutive mapped rows
        const int32_t pm = __shfl_up_sync(kFull, m, 1);
        start = valid && (lane == 0 || pm < 0 || m != pm + 1);
      }
      const uint32_t smask = __ballot_sync(kFull, start);
      mrows[s * 32 + lane] = m;
      if (lane == 0) {
        masks[s] = vmask;
        mbar_arrive_expect_tx(&bars[s], static_cast<uint32_t>(__popc(vmask)) * static_cast<uint32_t>(rb));
        maybe_stall(i, &bars[s]);
      }
      __syncwarp();
      if (start) {
        const int end = run_end(lane, smask, vmask);
        const char* from = SCATTER ? src + (q0 + lane) * rb : src + static_cast<int64_t>(m) * rb;
        bulk_load(st + lane * rb, from, static_cast<uint32_t>((end - lane) * rb), &bars[s]);
      }
    } else if (lane == 0) {
      const int64_t q = k / g.P;
      const int64_t off = (k % g.P) * g.stage;
      const uint32_t bytes = static_cast<uint32_t>(min(static_cast<int64_t>(g.stage), rb - off));
      masks[s] = m >= 0 ? 1u : 0u;
      mrows[s * 32] = m;
      if (m >= 0) {
        mbar_arrive_expect_tx(&bars[s], bytes);
        maybe_stall(i, &bars[s]);
        const char* from = SCATTER ? src + q * rb + off : src + static_cast<int64_t>(m) * rb + off;
        bulk_load(st, from, bytes, &bars[s]);
      } else {
        mbar_arrive_expect_tx(&bars[s], 0);
      }
    }
    __syncwarp();
  };

  auto issue_store = [&](int64_t i) {
    const int s = static_cast<int>(i % NST);
    const char* st = smem + static_cast<size_t>(s) * g.stage;
    const int64_t k = b + i * G;
    const uint32_t vmask = masks[s];
    if (row_mode) {
      const int64_t q0 = k * g.R;
      const int32_t m = mrows[s * 32 + lane];
      const bool valid = (vmask >> lane) & 1u;
      bool start;
      if (SCATTER) {  // runs of consecutive mapped rows
        const int32_t pm = __shfl_up_sync(kFull, m, 1);
        start = valid && (lane == 0 || pm < 0 || m != pm + 1);
      } else {        // contiguous linear destination: runs of valid rows
        start = valid && (lane == 0 || !((vmask >> (lane - 1)) & 1u));
      }
      const uint32_t smask = __ballot_sync(kFull, start);
      if (start) {
        const int end = run_end(lane, smask, vmask);
        char* to = SCATTER ? dst + static_cast<int64_t>(m) * rb : dst + (q0 + lane) * rb;
        bulk_store(to, st + lane * rb, static_cast<uint32_t>((end - lane) * rb));
      }
    } else if (lane == 0 && vmask) {
      const int64_t q = k / g.P;
      const int64_t off = (k % g.P) * g.stage;
      const uint32_t bytes = static_cast<uint32_t>(min(static_cast<int64_t>(g.stage), rb - off));
      const int32_t m = mrows[s * 32];
      char* to = SCATTER ? dst + static_cast<int64_t>(m) * rb + off : dst + q * rb + off;
      bulk_store(to, st, bytes);
    }
    bulk_commit();
  };

  // Loads run NST-1 chunks ahead of stores.  The mapped rows of the chunk to
  // be loaded next are fetched before waiting, so their latency overlaps.
  int64_t issued = 0;
  for (; issued < NST - 1 && issued < n_my; ++issued) issue_load(issued, fetch(issued));
  bool timed_out = false;
  int64_t i = 0;
  for (; i < n_my; ++i) {
    const int64_t j = i + NST - 1;
    const int32_t mj = j < n_my ? fetch(j) : -2;
    const bool landed = mbar_wait(&bars[i % NST], static_cast<uint32_t>((i / NST) & 1));
    if (!__all_sync(kFull, landed)) {  // give up together, never with part of the warp
      timed_out = true;
      break;
    }
    issue_store(i);
    if (j < n_my) {
      bulk_wait_read_all_but_one();  // the store that used stage j % NST is done reading it
      __syncwarp();
      issue_load(j, mj);
      issued = j + 1;
    }
  }
  if (timed_out) {
    // let this block's copies in flight land before shared memory goes away
    for (int64_t r = i; r < issued; ++r) mbar_wait(&bars[r % NST], static_cast<uint32_t>((r / NST) & 1));
    if (lane == 0) status_set(status, THD_ERR_TIMEOUT);
  }
  bulk_wait_all();
  if (bad) status_set(status, THD_ERR_INDEX_RANGE);
}

// ---- the run engine (rows of 16 - 192 bytes) --------------------------------
//
// Narrow rows move as runs: a chunk holds 32*K rows (K consecutive rows per
// lane, about 8 KiB), every lane reads its K mapped rows, the warp finds the
// maximal runs of rows whose mapped rows are consecutive (bit masks per lane,
// one ballot and one shuffle for the run ends across lanes), and each run
// moves with one bulk copy in and one out through the same ring of stages as
// the bulk engine.  Row by row such rows reach 0.58-0.87 of the copy
// bandwidth on GB300, as runs 0.63-0.93.
struct RunGeom {
  int32_t rows;
  int32_t row_bytes;
  int32_t stage;   // bytes per stage: 32 * K rows
  int64_t chunks;
};

template <int K, int NST, class Map, bool SCATTER>
__global__ void __launch_bounds__(32)
run_copy_kernel(const char* __restrict__ src, char* __restrict__ dst, RunGeom g, Map map, int32_t* status) {
  constexpr int CR = 32 * K;  // rows per chunk
  extern __shared__ __align__(128) char smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(NST) * g.stage);
  int32_t* mrows = reinterpret_cast<int32_t*>(bars + NST);  // NST x CR mapped rows
  const int lane = threadIdx.x;
  pdl_wait_then_release();  // launched with programmatic dependent launch
  // one read, broadcast: the warp must take this exit together
  if (__shfl_sync(kFull, lane == 0 ? status_load(status) : 0, 0) != 0) return;
  const int64_t b = blockIdx.x, G = gridDim.x;
  const int64_t n_my = g.chunks > b ? (g.chunks - b + G - 1) / G : 0;
  if (n_my == 0) return;
  const int64_t rb = g.row_bytes;
  if (lane == 0) {
    for (int s = 0; s < NST; ++s) mbar_init(&bars[s], 1);
    mbar_init_fence();
  }
  __syncwarp();
  bool bad = false;

  // mapped rows of this lane's K rows of chunk i (-1: out of range, -2: no row)
  auto fetch = [&](int64_t i, int32_t (&m)[K]) {
    const int64_t q0 = (b + i * G) * CR + lane * K;
#pragma unroll
    for (int k = 0; k < K; ++k) m[k] = (q0 + k < g.rows) ? map(static_cast<int32_t>(q0 + k)) : -2;
  };
  // Bit k of the result: row k of this lane starts no run continuing the row
  // before it (the row is not valid, or -- on the mapped side -- its mapped
  // row does not follow the one before, or -- on the linear side -- the row
  // before is not valid).  *tail_end: the chunk position of the first such
  // break after this lane's rows.
  auto breaks = [&](const int32_t (&m)[K], bool mapped_side, uint32_t* valid_mask, int* tail_end) -> uint32_t {
    const int32_t prev_last = __shfl_up_sync(kFull, m[K - 1], 1);
    uint32_t brk = 0, vm = 0;
#pragma unroll
    for (int k = 0; k < K; ++k) {
      const int32_t pm = k == 0 ? (lane == 0 ? -2 : prev_last) : m[k - 1];
      const bool v = m[k] >= 0;
      if (v) vm |= 1u << k;
      if (!(v && pm >= 0 && (!mapped_side || m[k] == pm + 1))) brk |= 1u << k;
    }
    const int first = brk ? __ffs(brk) - 1 : K;
    const uint32_t has = __ballot_sync(kFull, brk != 0);
    const uint32_t above = lane == 31 ? 0u : (has & ~((2u << lane) - 1u));
    const int next_lane = above ? __ffs(above) - 1 : 32;
    const int next_first = __shfl_sync(kFull, first, next_lane < 32 ? next_lane : 0);
    *tail_end = next_lane < 32 ? next_lane * K + next_first : CR;
    *valid_mask = vm;
    return brk;
  };
  // calls fn(position, rows) for every run that starts in this lane's rows
  auto each_run = [&](uint32_t brk, uint32_t vm, int tail_end, auto&& fn) {
    uint32_t starts = brk & vm;
    while (starts) {
      const int k = __ffs(starts) - 1;
      starts &= starts - 1;
      const uint32_t later = brk & ~((2u << k) - 1u);
      const int pos = lane * K + k;
      fn(pos, (later ? lane * K + (__ffs(later) - 1) : tail_end) - pos);
    }
  };

  auto issue_load = [&](int64_t i, const int32_t (&m)[K]) {
    const int s = static_cast<int>(i % NST);
    char* st = smem + static_cast<size_t>(s) * g.stage;
    int32_t* mr = mrows + s * CR;
    const int64_t q0 = (b + i * G) * CR;
#pragma unroll
    for (int k = 0; k < K; ++k) {
      mr[lane * K + k] = m[k];
      bad |= (m[k] == -1);
    }
    uint32_t vm;
    int tail_end;
    // gather: runs of consecutive source rows; scatter: the source is linear
    const uint32_t brk = breaks(m, !SCATTER, &vm, &tail_end);
    const int valid_rows = __reduce_add_sync(kFull, __popc(vm));
    if (lane == 0) {
      mbar_arrive_expect_tx(&bars[s], static_cast<uint32_t>(valid_rows * rb));
      maybe_stall(i, &bars[s]);
    }
    __syncwarp();
    each_run(brk, vm, tail_end, [&](int pos, int n) {
      const char* from = SCATTER ? src + (q0 + pos) * rb : src + static_cast<int64_t>(mr[pos]) * rb;
      bulk_load(st + pos * rb, from, static_cast<uint32_t>(n * rb), &bars[s]);
    });
    __syncwarp();
  };
  auto issue_store = [&](int64_t i) {
    const int s = static_cast<int>(i % NST);
    const char* st = smem + static_cast<size_t>(s) * g.stage;
    const int32_t* mr = mrows + s * CR;
    const int64_t q0 = (b + i * G) * CR;
    int32_t m[K];
#pragma unroll
    for (int k = 0; k < K; ++k) m[k] = mr[lane * K + k];
    uint32_t vm;
    int tail_end;
    // gather: the destination is linear; scatter: runs of consecutive destination rows
    const uint32_t brk = breaks(m, SCATTER, &vm, &tail_end);
    each_run(brk, vm, tail_end, [&](int pos, int n) {
      char* to = SCATTER ? dst + static_cast<int64_t>(mr[pos]) * rb : dst + (q0 + pos) * rb;
      bulk_store(to, st + pos * rb, static_cast<uint32_t>(n * rb));
    });
    bulk_commit();
  };

  // Loads run NST-1 chunks ahead of stores, as in the bulk engine.
  int32_t m_next[K];
  int64_t issued = 0;
  for (; issued < NST - 1 && issued < n_my; ++issued) {
    fetch(issued, m_next);
    issue_load(issued, m_next);
  }
  bool timed_out = false;
  int64_t i = 0;
  for (; i < n_my; ++i) {
    const int64_t j = i + NST - 1;
    if (j < n_my) fetch(j, m_next);
    const bool landed = mbar_wait(&bars[i % NST], static_cast<uint32_t>((i / NST) & 1));
    if (!__all_sync(kFull, landed)) {  // give up together, never with part of the warp
      timed_out = true;
      break;
    }
    issue_store(i);
    if (j < n_my) {
      bulk_wait_read_all_but_one();  // the store that used stage j % NST is done reading it
      __syncwarp();
      issue_load(j, m_next);
      issued = j + 1;
    }
  }
  if (timed_out) {
    // let this block's copies in flight land before shared memory goes away
    for (int64_t r = i; r < issued; ++r) mbar_wait(&bars[r % NST], static_cast<uint32_t>((r / NST) & 1));
    if (lane == 0) status_set(status, THD_ERR_TIMEOUT);
  }
  bulk_wait_all();
  if (bad) status_set(status, THD_ERR_INDEX_RANGE);
}

constexpr int kRunBlocksPerSm = 6;
constexpr int64_t kRunStage = 8192;  // target bytes per chunk

template <int K, int NST, class Map, bool SCATTER>
thd_status_t launch_runs(const void* src, void* dst, int32_t rows, int64_t row_bytes, Map map, int32_t* status,
                         cudaStream_t s) {
  RunGeom g;
  g.rows = rows;
  g.row_bytes = static_cast<int32_t>(row_bytes);
  g.stage = static_cast<int32_t>(32 * K * row_bytes);
  g.chunks = (static_cast<int64_t>(rows) + 32 * K - 1) / (32 * K);
  const size_t smem = static_cast<size_t>(NST) * g.stage + NST * (8 + 32 * K * 4);
  cudaError_t e = cudaSuccess;
  if (smem > 48 * 1024)
    e = cudaFuncSetAttribute(run_copy_kernel<K, NST, Map, SCATTER>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
  if (e == cudaSuccess) {
    int64_t grid = static_cast<int64_t>(sm_count()) * kRunBlocksPerSm;
    if (grid > g.chunks) grid = g.chunks;
    if (grid < 1) grid = 1;
    e = launch_pdl(run_copy_kernel<K, NST, Map, SCATTER>, dim3(static_cast<unsigned>(grid)), 32, smem, s,
                   static_cast<const char*>(src), static_cast<char*>(dst), g, map, status);
  }
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return THD_ERR_CUDA;
  }
  return THD_OK;
}

// K = the largest power of two (<= 16) with 32*K rows in 8 KiB; two stages
// when a chunk fills 8 KiB, three when it is smaller (a sweep on GB300: each
// width's best of 2 or 3 stages follows this rule).
template <class Map, bool SCATTER>
thd_status_t run_runs(const void* src, void* dst, int32_t rows, int64_t row_bytes, Map map, int32_t* status,
                      cudaStream_t s) {
  const int64_t fit = kRunStage / (32 * row_bytes);
  const int K = fit >= 16 ? 16 : fit >= 8 ? 8 : fit >= 4 ? 4 : fit >= 2 ? 2 : 1;
  const bool full = 32 * K * row_bytes >= kRunStage;
  switch (K) {
    case 16: return full ? launch_runs<16, 2, Map, SCATTER>(src, dst, rows, row_bytes, map, status, s)
                         : launch_runs<16, 3, Map, SCATTER>(src, dst, rows, row_bytes, map, status, s);
    case 8: return full ? launch_runs<8, 2, Map, SCATTER>(src, dst, rows, row_bytes, map, status, s)
                        : launch_runs<8, 3, Map, SCATTER>(src, dst, rows, row_bytes, map, status, s);
    case 4: return full ? launch_runs<4, 2, Map, SCATTER>(src, dst, rows, row_bytes, map, status, s)
                        : launch_runs<4, 3, Map, SCATTER>(src, dst, rows, row_bytes, map, status, s);
    case 2: return full ? launch_runs<2, 2, Map, SCATTER>(src, dst, rows, row_bytes, map, status, s)
                        : launch_runs<2, 3, Map, SCATTER>(src, dst, rows, row_bytes, map, status, s);
    default: return launch_runs<1, 3, Map, SCATTER>(src, dst, rows, row_bytes, map, status, s);
  }
}

// Stage size, ring depth and blocks per SM by row size (chosen by a sweep on
// GB300 over 4 KiB - 48 KiB stages, 2-8 stages, 1-8 blocks per SM):
//   rows <= 8 KiB : chunks of up to 8 KiB (R rows), 2 stages, 6 blocks per SM
//   rows <= 16 KiB: one row per chunk, 4 stages, 3 blocks per SM
//   rows <= 32 KiB: one row per chunk, 3 stages, 2 blocks per SM
//   larger rows   : 16 KiB pieces, 4 stages, 3 blocks per SM
struct BulkPlan {
  int nst, cps;
  BulkGeom g;
};

BulkPlan bulk_plan(int32_t rows, int64_t row_bytes) {
  BulkPlan p;
  p.g.rows = rows;
  p.g.row_bytes = static_cast<int32_t>(row_bytes);
  if (row_bytes <= 8192) {
    p.g.R = static_cast<int32_t>(8192 / row_bytes < 32 ? 8192 / row_bytes : 32);
    p.g.P = 1;
    p.g.stage = static_cast<int32_t>(p.g.R * row_bytes);
    p.nst = 2;
    p.cps = 6;
  } else if (row_bytes <= 32768) {
    p.g.R = 1;
    p.g.P = 1;
    p.g.stage = static_cast<int32_t>(row_bytes);
    p.nst = row_bytes <= 16384 ? 4 : 3;
    p.cps = row_bytes <= 16384 ? 3 : 2;
  } else {
    p.g.R = 1;
    p.g.stage = 16384;
    p.g.P = static_cast<int32_t>((row_bytes + p.g.stage - 1) / p.g.stage);
    p.nst = 4;
    p.cps = 3;
  }
  p.g.chunks = p.g.P == 1 ? (static_cast<int64_t>(rows) + p.g.R - 1) / p.g.R : static_cast<int64_t>(rows) * p.g.P;
  return p;
}

template <int NST, class Map, bool SCATTER>
thd_status_t launch_bulk(const BulkPlan& p, const void* src, void* dst, Map map, int32_t* status, cudaStream_t s) {
  const size_t smem = static_cast<size_t>(NST) * p.g.stage + NST * (8 + 4 + 32 * 4);
  cudaError_t e = cudaSuccess;
  if (smem > 48 * 1024)
    e = cudaFuncSetAttribute(bulk_copy_kernel<NST, Map, SCATTER>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
  if (e == cudaSuccess) {
    int64_t grid = static_cast<int64_t>(sm_count()) * p.cps;
    if (grid > p.g.chunks) grid = p.g.chunks;
    if (grid < 1) grid = 1;
    // programmatic dependent launch: back-to-back copies overlap one's
    // launch and ramp-up with the previous one's tail (about 2.3 us per
    // launch on GB300); the kernel waits for its predecessor before any access
    e = launch_pdl(bulk_copy_kernel<NST, Map, SCATTER>, dim3(static_cast<unsigned>(grid)), 32, smem, s,
                   static_cast<const char*>(src), static_cast<char*>(dst), p.g, map, status);
  }
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return THD_ERR_CUDA;
  }
  return THD_OK;
}

template <class Map, bool SCATTER>
thd_status_t run_bulk(const void* src, void* dst, int32_t rows, int64_t row_bytes, Map map, int32_t* status,
                      cudaStream_t s) {
  const BulkPlan p = bulk_plan(rows, row_bytes);
  switch (p.nst) {
    case 2: return launch_bulk<2, Map, SCATTER>(p, src, dst, map, status, s);
    case 3: return launch_bulk<3, Map, SCATTER>(p, src, dst, map, status, s);
    default: return launch_bulk<4, Map, SCATTER>(p, src, dst, map, status, s);
  }
}

template <class Map, bool SCATTER>
thd_status_t dispatch_unit(const void* src, void* dst, int32_t rows, int64_t row_bytes, Map map,
                           int32_t* status, cudaStream_t s) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst);
  if (row_bytes % 16 == 0 && a % 16 == 0 && row_bytes >= kBulkMinRowBytes)
    return run_bulk<Map, SCATTER>(src, dst, rows, row_bytes, map, status, s);
  if (row_bytes % 16 == 0 && a % 16 == 0)
    return run_runs<Map, SCATTER>(src, dst, rows, row_bytes, map, status, s);
  if (row_bytes % 4 == 0 && a % 4 == 0)
    return run<uint32_t, Map, SCATTER>(src, dst, rows, row_bytes, map, status, s);
  return run<uint8_t, Map, SCATTER>(src, dst, rows, row_bytes, map, status, s);
}

}  // namespace

thd_status_t launch_ulysses(const void* src, void* dst, int32_t T, int32_t cp, int64_t row_bytes, bool seq_to_head,
                            int32_t* status, cudaStream_t s) {
  if (T == 0) return THD_OK;
  if (ulysses_tiles_apply(src, dst, T, cp, row_bytes, seq_to_head))  // small head groups: tile transpose
    return launch_ulysses_tiles(src, dst, T, cp, row_bytes, seq_to_head, status, s);
  const UlyssesMap map{T, cp, seq_to_head, make_fast_div(seq_to_head ? T : cp)};
  return dispatch_unit<UlyssesMap, false>(src, dst, T * cp, row_bytes / cp, map, status, s);
}

thd_status_t launch_swap_batched(const void* src, void* dst, int32_t outer, int64_t row_bytes,
                                 const thd_route_t* r, int32_t* status, cudaStream_t s) {
  const int32_t T = static_cast<int32_t>(r->total_rows);
  if (T == 0 || outer == 0) return THD_OK;
  // outer * T < 2^31 (checked by the caller): the engines index rows with int32
  return dispatch_unit<BatchedSwapMap, false>(src, dst, outer * T, row_bytes,
                                              BatchedSwapMap{r->src_of_dst, T, make_fast_div(T)}, status, s);
}

thd_status_t launch_rank_copy(bool scatter, const void* src, void* dst, int32_t rank, int64_t row_bytes,
                              const thd_route_t* r, int32_t* status, cudaStream_t s) {
  const int32_t T = static_cast<int32_t>(r->total_rows);
  const int32_t S = T / r->cp_size;
  if (S == 0) return THD_OK;
  const int64_t off = static_cast<int64_t>(rank) * S;
  if (scatter)  // dst_shard[recv_rows[rank][j]] = recv[j]
    return dispatch_unit<OneRankMap, true>(src, dst, S, row_bytes, OneRankMap{r->recv_rows + off, S}, status, s);
  // send[j] = src_shard[send_rows[rank][j]]
  return dispatch_unit<OneRankMap, false>(src, dst, S, row_bytes, OneRankMap{r->send_rows + off, S}, status, s);
}

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

#if defined(THD_CHECKED) && THD_CHECKED
// Declared in include/thd_debug.h; exported by the checked build only.
extern "C" thd_status_t thd_debug_stall_next_bulk_copy(cudaStream_t stream) {
  const int one = 1;
  const cudaError_t e =
      cudaMemcpyToSymbolAsync(thd::g_stall_request, &one, sizeof(one), 0, cudaMemcpyHostToDevice, stream);
  if (e != cudaSuccess) {
    thd::record_cuda_error(e);
    return THD_ERR_CUDA;
  }
  return THD_OK;
}
#endif
