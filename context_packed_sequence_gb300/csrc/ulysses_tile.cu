// Ulysses sequence <-> head exchange for head-group pieces below 1 KiB
// ("Packed Sequence 与上下文并行", sections 2.5 and 2.7): a tile transpose
// through shared memory.
//
// Token row g of the sequence-sharded buffer is cp pieces of P bytes, one per
// head group; the head-sharded buffer holds, for each group h, every token's
// piece h contiguously ([cp][T][P]).  Gathering pieces one by one (the row
// engines in copy.cu) moves P bytes per copy, so small pieces leave HBM idle
// between requests.  Here a tile of R consecutive tokens moves as a few large
// bulk copies instead:
//
//   sequence -> head: one bulk load of the tile's R token rows (R*cp*P
//     contiguous bytes), a shared-memory transpose into cp runs of R*P bytes,
//     one bulk store per run to [h][g0 .. g0+R);
//   head -> sequence: one bulk load per run, the transpose back, one bulk
//     store of the R token rows.
//
// The runs sit in shared memory at a padded stride of H16 16-byte units with
// H16 = upr (mod 8), upr = P/16, so the eight 16-byte accesses of a
// quarter-warp that walk one token row reach eight different bank groups.
// A block of 256 threads keeps a ring of three load buffers and two store
// buffers; warp 0 issues every bulk copy (one lane per run).  Tiles of about
// 24 KiB with three loads in flight per SM kept both directions at 0.85-0.96
// of the measured copy bandwidth on GB300 for pieces of 32 B - 768 B, against
// 0.45-0.93 for the piece-by-piece engines.  Every wait is bounded: a wait that
// runs out records THD_ERR_TIMEOUT, lets the block's copies in flight land and
// returns.
#include "thd_internal.cuh"
#include "tma.cuh"

namespace thd {
namespace {

constexpr int kTileThreads = 256;
constexpr int kTileStages = 3;              // load buffers; two more for stores
constexpr int64_t kTileTarget = 24 * 1024;  // bytes of token rows per tile
constexpr int64_t kTileMaxPiece = 1024;     // larger pieces: the bulk row engine
constexpr size_t kTileSmemLimit = 227 * 1024;

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

TileGeom tile_geom(int32_t T, int32_t cp, int64_t row_bytes) {
  TileGeom g;
  g.T = T;
  g.cp = cp;
  g.upr = static_cast<int32_t>(row_bytes / cp / 16);
  int64_t R = kTileTarget / row_bytes;
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

size_t tile_smem(const TileGeom& g) {
  return static_cast<size_t>(kTileStages + 2) * g.stage + kTileStages * sizeof(uint64_t);
}

template <bool TO_HEAD>
__global__ void __launch_bounds__(kTileThreads)
ulysses_tile_kernel(const char* __restrict__ src, char* __restrict__ dst, TileGeom g, int32_t* status) {
  extern __shared__ __align__(128) char smem[];
  char* const loads = smem;                               // kTileStages buffers
  char* const stores = smem + kTileStages * g.stage;      // 2 buffers
  uint64_t* const bars = reinterpret_cast<uint64_t*>(smem + (kTileStages + 2) * g.stage);
  const int tid = threadIdx.x, lane = tid & 31;
  const bool issuer = tid < 32;  // warp 0 issues the bulk copies
  pdl_wait_then_release();       // launched with programmatic dependent launch
  if (__syncthreads_or(tid == 0 && status_load(status) != 0)) return;
  const int b = blockIdx.x, G = gridDim.x;
  const int n_my = g.tiles > b ? (g.tiles - b + G - 1) / G : 0;
  if (n_my == 0) return;
  const int64_t P = static_cast<int64_t>(g.upr) * 16, row = P * g.cp;
  const int units_per_row = g.cp * g.upr;
  if (tid == 0) {
    for (int s = 0; s < kTileStages; ++s) mbar_init(&bars[s], 1);
    mbar_init_fence();
  }
  __syncthreads();

  // tile t covers tokens [t*R, t*R + rt)
  auto tile_start = [&](int i) { return static_cast<int64_t>(b + i * G) * g.R; };
  auto tile_rows = [&](int64_t g0) { return min(static_cast<int64_t>(g.R), g.T - g0); };
  // checked build: every tile of this block lies inside [0, T), else the
  // block moves nothing (no bulk copy has been issued yet)
  if (kChecked) {
    bool bad = false;
    if (tid == 0)
      for (int i = 0; i < n_my; ++i) bad |= !in_range(tile_start(i), 0, g.T, status);
    if (__syncthreads_or(bad)) return;
  }

  // warp 0 only: lane 0 arms the stage's barrier before any lane loads into it
  auto issue_load = [&](int i) {
    const int s = i % kTileStages;
    const int64_t g0 = tile_start(i), rt = tile_rows(g0);
    char* buf = loads + s * g.stage;
    if (TO_HEAD) {
      if (lane == 0) {
        const uint32_t bytes = static_cast<uint32_t>(rt * row);
        mbar_arrive_expect_tx(&bars[s], bytes);
        bulk_load(buf, src + g0 * row, bytes, &bars[s]);
      }
    } else {
      const uint32_t bytes = static_cast<uint32_t>(rt * P);
      if (lane == 0) mbar_arrive_expect_tx(&bars[s], bytes * static_cast<uint32_t>(g.cp));
      __syncwarp();
      for (int h = lane; h < g.cp; h += 32)
        bulk_load(buf + static_cast<int64_t>(h) * g.H16 * 16, src + (static_cast<int64_t>(h) * g.T + g0) * P,
                  bytes, &bars[s]);
    }
  };
  auto issue_store = [&](int i) {
    const int64_t g0 = tile_start(i), rt = tile_rows(g0);
    const char* buf = stores + (i & 1) * g.stage;
    if (TO_HEAD) {
      for (int h = lane; h < g.cp; h += 32)
        bulk_store(dst + (static_cast<int64_t>(h) * g.T + g0) * P, buf + static_cast<int64_t>(h) * g.H16 * 16,
                   static_cast<uint32_t>(rt * P));
    } else if (lane == 0) {
      bulk_store(dst + g0 * row, buf, static_cast<uint32_t>(rt * row));
    }
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
    // unit k of the token-major layout is (token ii, head h, unit v); its
    // place in the head-major runs is h*H16 + ii*upr + v
    const int rt = static_cast<int>(tile_rows(tile_start(i)));
    const uint4* from = reinterpret_cast<const uint4*>(loads + s * g.stage);
    uint4* to = reinterpret_cast<uint4*>(stores + (i & 1) * g.stage);
    const int units = rt * units_per_row;
#pragma unroll 4
    for (int k = tid; k < units; k += kTileThreads) {
      const int ii = g.div_row.div(k);
      const int rem = k - ii * units_per_row;
      const int h = g.div_piece.div(rem);
      const int run = h * g.H16 + ii * g.upr + (rem - h * g.upr);
      if (TO_HEAD)
        to[run] = from[k];
      else
        to[k] = from[run];
    }
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

template <bool TO_HEAD>
thd_status_t launch_tiles(const void* src, void* dst, const TileGeom& g, size_t smem, int32_t* status,
                          cudaStream_t s) {
  auto kernel = ulysses_tile_kernel<TO_HEAD>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  int per_sm = 0;
  if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kTileThreads, smem);
  if (e == cudaSuccess) {
    if (per_sm < 1) per_sm = 1;
    int64_t grid = static_cast<int64_t>(sm_count()) * per_sm;
    if (grid > g.tiles) grid = g.tiles;
    e = launch_pdl(kernel, dim3(static_cast<unsigned>(grid)), kTileThreads, smem, s, static_cast<const char*>(src),
                   static_cast<char*>(dst), g, status);
  }
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return THD_ERR_CUDA;
  }
  return THD_OK;
}

}  // namespace

bool ulysses_tiles_apply(const void* src, const void* dst, int32_t T, int32_t cp, int64_t row_bytes) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst);
  if (cp < 2 || T <= 0 || a % 16 != 0 || row_bytes % cp != 0) return false;
  const int64_t P = row_bytes / cp;
  if (P % 16 != 0 || P >= kTileMaxPiece) return false;
  return tile_smem(tile_geom(T, cp, row_bytes)) <= kTileSmemLimit;
}

thd_status_t launch_ulysses_tiles(const void* src, void* dst, int32_t T, int32_t cp, int64_t row_bytes,
                                  bool seq_to_head, int32_t* status, cudaStream_t s) {
  const TileGeom g = tile_geom(T, cp, row_bytes);
  const size_t smem = tile_smem(g);
  return seq_to_head ? launch_tiles<true>(src, dst, g, smem, status, s)
                     : launch_tiles<false>(src, dst, g, smem, status, s);
}

}  // namespace thd
