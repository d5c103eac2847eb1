// Ulysses sequence <-> head exchange for head-group pieces below 1 KiB
// ("Packed Sequence 与上下文并行", sections 2.5 and 2.7): a tile transpose
// through shared memory.
//
// Token row g of the sequence-sharded buffer is cp pieces of P bytes, one per
// head group; the head-sharded buffer holds, for each group h, every token's
// piece h contiguously ([cp][T][P]).  Gathering pieces one by one (the row
// engines in copy.cu) moves P bytes per copy, so small pieces leave HBM idle
// between requests.  Here a tile of R consecutive tokens (24-44 KiB, chosen
// by cp and direction in tile_target) moves as a few large bulk copies instead:
//
//   sequence -> head (ulysses_to_heads_kernel): one bulk load of the tile's R
//     token rows (R*cp*P contiguous bytes), a shared-memory transpose into cp
//     runs of R*P bytes, one bulk store per run to [h][g0 .. g0+R);
//   head -> sequence (ulysses_to_sequence_kernel): one bulk load per run, the
//     transpose back, one bulk store of the R token rows.
//
// The runs sit in shared memory at a padded stride of H16 16-byte units with
// H16 = upr (mod 8), upr = P/16, so the eight 16-byte accesses of a
// quarter-warp that walk one token row reach eight different bank groups.
// Both kernels keep three load buffers and two store buffers per block, one
// block per SM.  Sequence -> head runs as one block of 256 threads in step
// (warp 0 issues the copies, one lane per run).  Head -> sequence, whose loads
// are cp separate runs per tile, adds a warp that only loads: it refills a
// buffer as soon as the eight transposing warps release it (an mbarrier with
// eight arrivals), without waiting for their block barrier.  Measured on GB300
// (of the copy bandwidth, pieces of 32 B - 768 B, 0.5 GiB buffers): sequence ->
// head 0.89-0.95, head -> sequence 0.90-0.97 (0.85 for 32 B pieces with a
// block in step), against 0.45-0.93 for the piece-by-piece engines; 1 GiB
// buffers of 16-128 B pieces: 0.97-0.995.  Every wait is bounded: a
// wait that runs out records THD_ERR_TIMEOUT, lets the block's copies in
// flight land and returns.
#include "thd_internal.cuh"
#include "tma.cuh"
#include "thd_debug.h"

namespace thd {
namespace {

constexpr int kTileStages = 3;           // load buffers; two more for stores
constexpr int64_t kTileMaxPiece = 1024;  // larger pieces: the bulk row engine
constexpr size_t kTileSmemLimit = 227 * 1024;
constexpr int kTransposers = 256;                      // threads that transpose a tile
constexpr int kToSequenceThreads = 32 + kTransposers;  // + the loading warp

// Checked build only: a one-shot request (thd_debug_stall_next_ulysses_tile)
// that block 0 of the next tile kernel arms 16 bytes no copy delivers on its
// first buffer, so the timeout path runs for real.
__device__ int g_tile_stall_request;

__device__ __forceinline__ void maybe_stall(int i, uint64_t* bar) {
  if (kChecked && i == 0 && blockIdx.x == 0 && atomicExch(&g_tile_stall_request, 0) != 0) mbar_expect_tx(bar, 16);
}

struct TileGeom {
  int32_t T, cp;
  int32_t upr;        // 16-byte units per piece
  int32_t R;          // tokens per tile
  int32_t H16;        // stride of the padded runs, in 16-byte units
  int32_t stage;      // bytes per shared-memory buffer
  int32_t tiles;
  FastDiv div_row;    // by cp * upr, the units of one token row
  FastDiv div_piece;  // by upr
};

// Bytes of token rows per tile.  Swept on GB300 over cp = 2-64 and tiles of
// 16-44 KiB (pieces of 32 and 64 B, 0.5 GiB buffers; the throughput depends
// on cp and the tile, hardly on the piece): 24 KiB is best for cp <= 12 in
// both directions (0.93-0.96 of the copy bandwidth, 0.87-0.91 at 28-44 KiB);
// above that each direction has its own best tile, which grows with cp:
// sequence -> head 28 KiB at cp = 16 (0.94 against 0.90 at 24 KiB), 32 KiB at
// cp = 24 (0.93 against 0.77), 40 KiB at cp = 32 (0.92 against 0.67); head ->
// sequence 28 KiB at cp = 24 (0.94 against 0.91), 32 KiB at cp = 32 (0.95
// against 0.81).  At cp = 64 the largest tile that fits does best (0.66-0.75).
int64_t tile_target(int32_t cp, bool seq_to_head) {
  constexpr int64_t K = 1024;
  if (seq_to_head) return cp <= 12 ? 24 * K : cp <= 16 ? 28 * K : cp <= 24 ? 32 * K : cp <= 32 ? 40 * K : 44 * K;
  return cp <= 16 ? 24 * K : cp <= 24 ? 28 * K : cp <= 32 ? 32 * K : 44 * K;
}

TileGeom tile_geom(int32_t T, int32_t cp, int64_t row_bytes, int64_t target) {
  TileGeom g;
  g.T = T;
  g.cp = cp;
  g.upr = static_cast<int32_t>(row_bytes / cp / 16);
  int64_t R = target / row_bytes;
  if (R < 1) R = 1;
  g.R = static_cast<int32_t>(R);
  const int64_t pad = ((g.upr - R * g.upr) % 8 + 8) % 8;  // makes H16 = upr (mod 8)
  g.H16 = static_cast<int32_t>(R * g.upr + pad);
  g.stage = static_cast<int32_t>((static_cast<int64_t>(cp) * g.H16 * 16 + 127) / 128 * 128);
  g.tiles = static_cast<int32_t>((T + R - 1) / R);
  g.div_row = make_fast_div(cp * g.upr);
  g.div_piece = make_fast_div(g.upr);
  return g;
}

// buffers, then one "loaded" and one "released" mbarrier per load buffer
size_t tile_smem(const TileGeom& g) {
  return static_cast<size_t>(kTileStages + 2) * g.stage + 2 * kTileStages * sizeof(uint64_t);
}

// The geometry for (cp, direction): the tile of tile_target, 4 KiB smaller
// at a time while its buffers do not fit in shared memory.  False when not
// even one token row per tile fits.
bool pick_geom(int32_t T, int32_t cp, int64_t row_bytes, bool seq_to_head, TileGeom* g) {
  for (int64_t target = tile_target(cp, seq_to_head);; target -= 4096) {
    *g = tile_geom(T, cp, row_bytes, target);
    if (tile_smem(*g) <= kTileSmemLimit) return true;
    if (g->R == 1) return false;
  }
}

// The tiles of block b: tile b + i*G covers tokens [start(i), start(i) + rows(i)).
struct TileSeq {
  int32_t b, G, R, T;
  __device__ __forceinline__ int64_t start(int i) const { return static_cast<int64_t>(b + i * G) * R; }
  __device__ __forceinline__ int64_t rows(int i) const { return min(static_cast<int64_t>(R), T - start(i)); }
};

// Checked build: does every tile of this block lie inside [0, T)?  A block-
// uniform answer; the default build compiles it to true.
__device__ __forceinline__ bool tiles_in_range(const TileSeq& ts, int n_my, int32_t* status) {
  if (!kChecked) return true;
  bool bad = false;
  if (threadIdx.x == 0)
    for (int i = 0; i < n_my; ++i) bad |= !in_range(ts.start(i), 0, ts.T, status);
  return !__syncthreads_or(bad);
}

// Unit k of a tile's token-major layout is (token ii, head h, unit v); its
// place in the head-major runs is h*H16 + ii*upr + v.  Transposer `first` of
// `stride` moves units first, first + stride, ...
template <bool TO_HEAD>
__device__ __forceinline__ void transpose_tile(const uint4* from, uint4* to, int rt, const TileGeom& g, int first,
                                               int stride) {
  const int units_per_row = g.cp * g.upr;
  const int units = rt * units_per_row;
#pragma unroll 4
  for (int k = first; k < units; k += stride) {
    const int ii = g.div_row.div(k);
    const int rem = k - ii * units_per_row;
    const int h = g.div_piece.div(rem);
    const int run = h * g.H16 + ii * g.upr + (rem - h * g.upr);
    if (TO_HEAD)
      to[run] = from[k];
    else
      to[k] = from[run];
  }
}

// ---- sequence -> head: one block of 256 threads in step ---------------------

__global__ void __launch_bounds__(kTransposers)
ulysses_to_heads_kernel(const char* __restrict__ src, char* __restrict__ dst, TileGeom g, int32_t* status) {
  extern __shared__ __align__(128) char smem[];
  char* const loads = smem;                           // kTileStages buffers
  char* const stores = smem + kTileStages * g.stage;  // 2 buffers
  uint64_t* const bars = reinterpret_cast<uint64_t*>(smem + (kTileStages + 2) * g.stage);
  const int tid = threadIdx.x, lane = tid & 31;
  const bool issuer = tid < 32;  // warp 0 issues the bulk copies
  pdl_wait_then_release();       // launched with programmatic dependent launch
  if (__syncthreads_or(tid == 0 && status_load(status) != 0)) return;
  const TileSeq ts{static_cast<int32_t>(blockIdx.x), static_cast<int32_t>(gridDim.x), g.R, g.T};
  const int n_my = g.tiles > ts.b ? (g.tiles - ts.b + ts.G - 1) / ts.G : 0;
  if (n_my == 0 || !tiles_in_range(ts, n_my, status)) return;
  const int64_t P = static_cast<int64_t>(g.upr) * 16, row = P * g.cp;
  if (tid == 0) {
    for (int s = 0; s < kTileStages; ++s) mbar_init(&bars[s], 1);
    mbar_init_fence();
  }
  __syncthreads();

  // warp 0 only: lane 0 loads the tile's token rows in one copy
  auto issue_load = [&](int i) {
    const int s = i % kTileStages;
    if (lane == 0) {
      const uint32_t bytes = static_cast<uint32_t>(ts.rows(i) * row);
      mbar_arrive_expect_tx(&bars[s], bytes);
      maybe_stall(i, &bars[s]);
      bulk_load(loads + s * g.stage, src + ts.start(i) * row, bytes, &bars[s]);
    }
  };
  // warp 0 only: one lane per head-group run
  auto issue_store = [&](int i) {
    const char* buf = stores + (i & 1) * g.stage;
    for (int h = lane; h < g.cp; h += 32)
      bulk_store(dst + (static_cast<int64_t>(h) * g.T + ts.start(i)) * P, buf + static_cast<int64_t>(h) * g.H16 * 16,
                 static_cast<uint32_t>(ts.rows(i) * P));
    bulk_commit();
  };

  int issued = 0;  // tiles whose loads are in flight or landed (warp 0's count)
  if (issuer)
    for (; issued < kTileStages && issued < n_my; ++issued) issue_load(issued);
  bool timed_out = false;
  int i = 0;
  for (; i < n_my; ++i) {
    const int s = i % kTileStages;
    // the stores of tile i-2 have finished reading store buffer i & 1
    if (issuer) bulk_wait_read_all_but_one();
    const bool landed = mbar_wait(&bars[s], static_cast<uint32_t>((i / kTileStages) & 1));
    if (!__syncthreads_and(landed)) {  // give up together
      timed_out = true;
      break;
    }
    transpose_tile<true>(reinterpret_cast<const uint4*>(loads + s * g.stage),
                         reinterpret_cast<uint4*>(stores + (i & 1) * g.stage), static_cast<int>(ts.rows(i)), g, tid,
                         kTransposers);
    fence_proxy_async_shared();  // the bulk stores read what this thread wrote
    __syncthreads();             // ... and load buffer s is free again
    if (issuer) {
      issue_store(i);
      if (issued < n_my) {
        issue_load(issued);
        ++issued;
      }
    }
  }
  if (timed_out && issuer) {
    // let this block's loads in flight land before shared memory goes away
    if (lane == 0)
      for (int r = i; r < issued; ++r) mbar_wait(&bars[r % kTileStages], static_cast<uint32_t>((r / kTileStages) & 1));
    if (lane == 0) status_set(status, THD_ERR_TIMEOUT);
  }
  if (issuer) bulk_wait_all();
}

// ---- head -> sequence: a loading warp and eight transposing warps -----------

// the transposing threads (warps 1-8) among themselves: named barriers 1 and 2
__device__ __forceinline__ void transposers_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kTransposers) : "memory");
}
__device__ __forceinline__ bool transposers_all(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, 2, %2, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "n"(kTransposers)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__global__ void __launch_bounds__(kToSequenceThreads)
ulysses_to_sequence_kernel(const char* __restrict__ src, char* __restrict__ dst, TileGeom g, int32_t* status) {
  extern __shared__ __align__(128) char smem[];
  char* const loads = smem;                           // kTileStages buffers
  char* const stores = smem + kTileStages * g.stage;  // 2 buffers
  uint64_t* const loaded = reinterpret_cast<uint64_t*>(smem + (kTileStages + 2) * g.stage);
  uint64_t* const released = loaded + kTileStages;    // 8 arrivals: every transposing warp is done
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  pdl_wait_then_release();  // launched with programmatic dependent launch
  if (__syncthreads_or(tid == 0 && status_load(status) != 0)) return;
  const TileSeq ts{static_cast<int32_t>(blockIdx.x), static_cast<int32_t>(gridDim.x), g.R, g.T};
  const int n_my = g.tiles > ts.b ? (g.tiles - ts.b + ts.G - 1) / ts.G : 0;
  if (n_my == 0 || !tiles_in_range(ts, n_my, status)) return;
  const int64_t P = static_cast<int64_t>(g.upr) * 16, row = P * g.cp;
  if (tid == 0) {
    for (int s = 0; s < kTileStages; ++s) {
      mbar_init(&loaded[s], 1);
      mbar_init(&released[s], kTransposers / 32);
    }
    mbar_init_fence();
  }
  __syncthreads();

  if (warp == 0) {
    // the loading warp: tile i goes into buffer i % stages once the tile
    // before it there is released; one lane per head-group run
    int issued = 0;
    for (int i = 0; i < n_my; ++i) {
      const int s = i % kTileStages;
      if (i >= kTileStages &&
          !__all_sync(kFullMask, mbar_wait(&released[s], static_cast<uint32_t>((i / kTileStages - 1) & 1))))
        break;  // the transposing warps gave up; they report it
      const uint32_t bytes = static_cast<uint32_t>(ts.rows(i) * P);
      if (lane == 0) {
        mbar_arrive_expect_tx(&loaded[s], bytes * static_cast<uint32_t>(g.cp));
        maybe_stall(i, &loaded[s]);
      }
      __syncwarp();
      char* buf = loads + s * g.stage;
      for (int h = lane; h < g.cp; h += 32)
        bulk_load(buf + static_cast<int64_t>(h) * g.H16 * 16, src + (static_cast<int64_t>(h) * g.T + ts.start(i)) * P,
                  bytes, &loaded[s]);
      issued = i + 1;
    }
    // every load this warp issued lands before it leaves (each buffer has at
    // most its last phase open, so these waits end)
    if (lane == 0)
      for (int j = max(0, issued - kTileStages); j < issued; ++j)
        mbar_wait(&loaded[j % kTileStages], static_cast<uint32_t>((j / kTileStages) & 1));
    return;
  }

  // the transposing warps; warp 1 also stores
  const bool storer = warp == 1;
  bool timed_out = false;
  for (int i = 0; i < n_my; ++i) {
    const int s = i % kTileStages;
    if (storer) bulk_wait_read_all_but_one();  // the store of tile i-2 is done reading buffer i & 1
    transposers_sync();
    if (!transposers_all(mbar_wait(&loaded[s], static_cast<uint32_t>((i / kTileStages) & 1)))) {
      timed_out = true;  // give up together
      break;
    }
    transpose_tile<false>(reinterpret_cast<const uint4*>(loads + s * g.stage),
                          reinterpret_cast<uint4*>(stores + (i & 1) * g.stage), static_cast<int>(ts.rows(i)), g,
                          tid - 32, kTransposers);
    __syncwarp();
    if (lane == 0) mbar_arrive(&released[s]);  // this warp is done reading buffer s
    fence_proxy_async_shared();                // the bulk store reads what this thread wrote
    transposers_sync();
    if (storer && lane == 0) {
      bulk_store(dst + ts.start(i) * row, stores + (i & 1) * g.stage, static_cast<uint32_t>(ts.rows(i) * row));
      bulk_commit();
    }
  }
  if (timed_out && tid == 32) status_set(status, THD_ERR_TIMEOUT);
  if (storer) bulk_wait_all();
}

template <class Kernel>
thd_status_t launch_tiles(Kernel kernel, int threads, const void* src, void* dst, const TileGeom& g, size_t smem,
                          int32_t* status, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  int per_sm = 0;
  if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem);
  if (e == cudaSuccess) {
    if (per_sm < 1) per_sm = 1;
    int64_t grid = static_cast<int64_t>(sm_count()) * per_sm;
    if (grid > g.tiles) grid = g.tiles;
    e = launch_pdl(kernel, dim3(static_cast<unsigned>(grid)), threads, smem, s, static_cast<const char*>(src),
                   static_cast<char*>(dst), g, status);
  }
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return THD_ERR_CUDA;
  }
  return THD_OK;
}

}  // namespace

bool ulysses_tiles_apply(const void* src, const void* dst, int32_t T, int32_t cp, int64_t row_bytes,
                         bool seq_to_head) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst);
  if (cp < 2 || T <= 0 || a % 16 != 0 || row_bytes % cp != 0) return false;
  const int64_t P = row_bytes / cp;
  if (P % 16 != 0 || P >= kTileMaxPiece) return false;
  TileGeom g;
  if (!pick_geom(T, cp, row_bytes, seq_to_head, &g)) return false;
  // Pieces of 256 B and more also go well piece by piece (0.83-0.91 of the
  // copy bandwidth through the bulk row engine), and a tile of them holds few
  // tokens, so its runs are short.  Measured on GB300 (cp = 16-64, pieces of
  // 256-768 B), the tile transpose wins when sequence -> head tiles hold at
  // least 4 tokens (cp = 32, 256 B: 0.93 against 0.84) and loses below (cp =
  // 32, 512 B: 0.83 against 0.90; cp = 64, 256 B: 0.54 against 0.84); head ->
  // sequence wins with 2 tokens when the runs reach 640 B (cp = 32, 512 B:
  // 0.95 against 0.90) and loses below (cp = 64, 256 B: 0.59 against 0.83).
  if (P < 256) return true;
  return seq_to_head ? g.R >= 4 : g.R >= 2 && g.R * P >= 640;
}

thd_status_t launch_ulysses_tiles(const void* src, void* dst, int32_t T, int32_t cp, int64_t row_bytes,
                                  bool seq_to_head, int32_t* status, cudaStream_t s) {
  TileGeom g;
  if (!pick_geom(T, cp, row_bytes, seq_to_head, &g)) return THD_ERR_INVALID_ARG;
  const size_t smem = tile_smem(g);
  return seq_to_head ? launch_tiles(ulysses_to_heads_kernel, kTransposers, src, dst, g, smem, status, s)
                     : launch_tiles(ulysses_to_sequence_kernel, kToSequenceThreads, src, dst, g, smem, status, s);
}

}  // namespace thd

#if defined(THD_CHECKED) && THD_CHECKED
// Declared in include/thd_debug.h; exported by the checked build only.
extern "C" thd_status_t thd_debug_stall_next_ulysses_tile(cudaStream_t stream) {
  const int one = 1;
  const cudaError_t e =
      cudaMemcpyToSymbolAsync(thd::g_tile_stall_request, &one, sizeof(one), 0, cudaMemcpyHostToDevice, stream);
  if (e != cudaSuccess) {
    thd::record_cuda_error(e);
    return THD_ERR_CUDA;
  }
  return THD_OK;
}
#endif
