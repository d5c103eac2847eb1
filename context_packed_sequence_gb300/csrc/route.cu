// Device-side route build and zigzag partition indices.
//
// "[Task32] feat: fla mcore chunkwise cp stage 3" (Relax PR #273), section 2.1:
// both layouts are unions of global row intervals, so the all-to-all route
// follows from interval intersection.  The pages copy cu_seqlens to the host
// and intersect with a Python two-pointer loop.  Here one kernel per call:
//
//  1. every block stages the boundaries in shared memory and validates them
//     in one pass (all blocks reach the same verdict; block 0 writes the
//     status word), then derives the cp x (cp+1) tables "zigzag rows of rank
//     s below d*S" and the receive offsets, each entry in closed form;
//  2. warps walk the zigzag layout in slot tiles: 32 consecutive local slots
//     whose documents are found once (a galloping search forward from the
//     previous tile plus a short window search per lane) and then serve every
//     rank, since all ranks' shards share the documents' slot ranges.  The
//     global row of each (rank, slot), its contiguous rank and the entry's
//     place in every route array follow in closed form, with divisions by S
//     done by multiply-shift.
//
// No host synchronisation, no atomics on the route, deterministic.
#include "thd_internal.cuh"

namespace thd {
namespace {

// Threads per block of the walking kernels (a sweep knob).
#ifndef THD_ROUTE_THREADS
#define THD_ROUTE_THREADS 512
#endif
constexpr int kRouteThreads = THD_ROUTE_THREADS;
constexpr int kSmemBudget = 48 * 1024;
// Launch shape of the walking kernels: at most this many blocks per SM (a
// sweep on GB300 over 1-2 blocks per SM and 1-16 items per warp put one
// block per SM, one warp per item, ahead by 1-2 us on 4096 documents and
// level elsewhere).
#ifndef THD_ROUTE_BLOCKS_PER_SM
#define THD_ROUTE_BLOCKS_PER_SM 1
#endif
// Unrolling of a lane's loop over the ranks of a slot tile (1-8 timed the
// same on GB300; 1 keeps the kernels at 32 registers).
#ifndef THD_ROUTE_UNROLL
#define THD_ROUTE_UNROLL 1
#endif
constexpr int kRouteUnroll = THD_ROUTE_UNROLL;

struct RouteArgs {
  const int32_t* cu;
  int32_t n, T, S;
  CpMath m;
  FastDiv divS;
  FastDiv divCp1;  // by cp + 1
  bool cu_in_smem;
  thd_route_t zc;  // zigzag -> contiguous (used when bit 0 of DIRS is set)
  thd_route_t cz;  // contiguous -> zigzag (used when bit 1 of DIRS is set)
  // both directions: arrays that the two routes share (thd_route_bind_pair)
  // are written once -- z->c receive rows are c->z send rows, and z->c send
  // rows are c->z receive rows (0..S-1 on every rank)
  bool cz_send_shared, cz_recv_shared;
  int32_t* status;
};

constexpr int kZC = 1, kCZ = 2;

// Does rank-interval [lo, hi) of the contiguous layout contain two
// neighbouring rows whose zigzag owners decrease?  Owners along a document
// run 0,1,..,cp-1,cp-1,..,1,0 chunk by chunk, so a decrease happens exactly
// at the starts of chunks cp+1 .. 2cp-1.  No decrease <=> sorting the
// interval's rows by (owner, row) keeps them in row order <=> the receive
// rows of z->c (equally the send rows of c->z) of that rank are 0..S-1.
__device__ bool has_descent(const int32_t* cu, int32_t n, CpMath m, int32_t lo, int32_t hi) {
  const int32_t cp = m.cp;
  if (cp == 1 || hi <= lo) return false;
  int32_t ilo = doc_of(cu, n, lo), ihi = doc_of(cu, n, hi - 1);
  if (ihi > ilo && cu[ihi] > cu[ilo + 1]) return true;  // a whole non-empty document inside
  for (int pass = 0; pass < 2; ++pass) {
    int32_t i = pass == 0 ? ilo : ihi;
    if (pass == 1 && ihi == ilo) break;
    int32_t L = cu[i + 1] - cu[i];
    if (L == 0) continue;
    int32_t c = m.div2(L);
    // descents at b = cu[i] + k*c, k = cp+1 .. 2cp-1; need lo+1 <= b <= hi-1
    // (ceil(a / c) as (a - 1) / c + 1: a + c - 1 could pass INT32_MAX)
    const int32_t a = lo + 1 - cu[i];
    const int32_t klo = a <= 0 ? cp + 1 : max(cp + 1, (a - 1) / c + 1);
    const int32_t b = hi - 1 - cu[i];
    if (b < 0) continue;
    const int32_t khi = min(2 * cp - 1, b / c);
    if (klo <= khi) return true;
  }
  return false;
}

// Split sizes, offsets and identity flags of one direction (one block only).
// n_zc[s][d] = cnt[s][d+1] - cnt[s][d] rows go from zigzag rank s to
// contiguous rank d; the reverse direction transposes it.
__device__ void write_small_arrays(const thd_route_t& r, bool z2c, const int32_t* cu, int32_t n, CpMath m,
                                   int32_t S, const int32_t* cnt, const int32_t* roff) {
  const int32_t cp = m.cp;
  for (int32_t e = threadIdx.x; e < cp * cp; e += blockDim.x) {
    int32_t x = e / cp, y = e - x * cp;
    int32_t nxy = cnt[x * (cp + 1) + y + 1] - cnt[x * (cp + 1) + y];  // n_zc[x][y]
    int32_t nyx = cnt[y * (cp + 1) + x + 1] - cnt[y * (cp + 1) + x];  // n_zc[y][x]
    r.input_split_sizes[e] = z2c ? nxy : nyx;   // [s=x][d=y]
    r.output_split_sizes[e] = z2c ? nyx : nxy;  // [d=x][s=y]
  }
  for (int32_t e = threadIdx.x; e < cp * (cp + 1); e += blockDim.x) {
    r.send_offsets[e] = z2c ? cnt[e] : roff[e];
    r.recv_offsets[e] = z2c ? roff[e] : cnt[e];
  }
  for (int32_t k = threadIdx.x; k < cp; k += blockDim.x) {
    uint8_t in_order = has_descent(cu, n, m, k * S, (k + 1) * S) ? 0 : 1;
    r.send_identity[k] = z2c ? 1 : in_order;
    r.recv_identity[k] = z2c ? in_order : 1;
  }
}

template <int DIRS, bool SMEM_CU>
__global__ void __launch_bounds__(kRouteThreads) route_build_kernel(RouteArgs a) {
  extern __shared__ int32_t smem[];
  const CpMath m = a.m;
  const int32_t cp = m.cp, S = a.S, T = a.T, n = a.n;
  int32_t* cnt = smem;                        // [cp][cp+1]: zigzag rows of s below d*S
  int32_t* roff = cnt + cp * (cp + 1);        // [d][cp+1]: z->c receive offsets
  int32_t* bnd = roff + cp * (cp + 1);        // [3][cp+1]: document start, chunk, offset at d*S
  int32_t* prd = bnd + 3 * (cp + 1);          // [r][d]: d*S + roff[d][r] - cnt[r][d]
  int32_t* cu_s = prd + cp * cp;
  pdl_wait_then_release();
  const int32_t code = stage_check_cu(a.cu, n, cu_s, SMEM_CU, a.status, T, 2 * cp);
  if (code != THD_OK) {
    if (code != kStatusWasSet && blockIdx.x == 0 && threadIdx.x == 0) status_set(a.status, code);
    return;
  }
  const int32_t* cu = SMEM_CU ? cu_s : a.cu;

  // Both tables in closed form from the document holding each contiguous
  // boundary X_d = d*S (one search per boundary): its start c0, chunk length
  // c and offset off = X_d - c0 (c = -1 marks X_d = T).  Then
  //   cnt[s][d]  = zigzag rows of rank s below X_d
  //              = c0/cp + clip(off - s*c) + clip(off - (2cp-1-s)*c), clip to [0, c];
  //   roff[d][s] = rows ranks 0..s-1 send to contiguous rank d = P(s, X_{d+1}) - P(s, X_d)
  //   with P(s, X) = rows of ranks < s below X
  //              = s*c0/cp + min(off, s*c) + max(0, off - (2cp-s)*c)
  //   (ranks below s own chunks [0, s) and [2cp-s, 2cp) of every document).
  // one warp per boundary, searching together
  for (int32_t d = threadIdx.x >> 5; d <= cp; d += blockDim.x >> 5) {
    const int32_t X = d * S;
    const int32_t i = X >= T ? 0 : warp_doc_of(cu, n, X);
    if ((threadIdx.x & 31) == 0) {
      if (X >= T) {
        bnd[d] = 0, bnd[(cp + 1) + d] = -1, bnd[2 * (cp + 1) + d] = 0;
      } else {
        bnd[d] = cu[i];
        bnd[(cp + 1) + d] = m.div2(cu[i + 1] - cu[i]);
        bnd[2 * (cp + 1) + d] = X - cu[i];
      }
    }
  }
  __syncthreads();
  for (int32_t e = threadIdx.x; e < cp * (cp + 1); e += blockDim.x) {
    const int32_t x = a.divCp1.div(e), y = e - x * (cp + 1);
    {  // cnt[s = x][d = y]
      const int32_t c = bnd[(cp + 1) + y], off = bnd[2 * (cp + 1) + y];
      cnt[e] = c < 0 ? S
                     : m.div(bnd[y]) + min(max(off - x * c, 0), c) + min(max(off - (2 * cp - 1 - x) * c, 0), c);
    }
    {  // roff[d = x][s = y]
      int32_t p[2];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int32_t b = x + 1 - k;  // boundary X_{d+1}, then X_d
        const int32_t c = bnd[(cp + 1) + b], off = bnd[2 * (cp + 1) + b];
        p[k] = c < 0 ? y * S : y * m.div(bnd[b]) + min(off, y * c) + max(0, off - (2 * cp - y) * c);
      }
      roff[e] = p[0] - p[1];
    }
  }
  // where rank r's rows bound for contiguous rank d start in d's receive
  // buffer, less the zigzag rows of r below d*S: an entry's place is then
  // prd[r][d] + its slot (the same closed forms as cnt and roff)
  for (int32_t e = threadIdx.x; e < cp * cp; e += blockDim.x) {
    const int32_t r = m.div(e), d = e - r * cp;
    int32_t c = bnd[(cp + 1) + d], off = bnd[2 * (cp + 1) + d];
    const int32_t cnt_rd =
        c < 0 ? S : m.div(bnd[d]) + min(max(off - r * c, 0), c) + min(max(off - (2 * cp - 1 - r) * c, 0), c);
    int32_t p[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int32_t b = d + 1 - k;  // boundary X_{d+1}, then X_d
      c = bnd[(cp + 1) + b];
      off = bnd[2 * (cp + 1) + b];
      p[k] = c < 0 ? r * S : r * m.div(bnd[b]) + min(off, r * c) + max(0, off - (2 * cp - r) * c);
    }
    prd[e] = d * S + (p[0] - p[1]) - cnt_rd;
  }
  __syncthreads();

  // Zigzag position u = r*S + j holds global row g.  Then
  //   z->c: src_of_dst[g] = u, send_rows[u] = j;
  //   c->z: src_of_dst[u] = g, recv_rows[u] = j;
  //   with d = g / S the contiguous rank of g, the row is entry
  //   roff[d][r] + (j - cnt[r][d]) of d's z->c receive buffer and of d's c->z
  //   send buffer, with value g - d*S.
  const int64_t tiles = (static_cast<int64_t>(S) + 31) / 32;
  int64_t begin, end;
  warp_items(tiles * cp, 1, &begin, &end);
  if (begin < end) {
    const FastDiv divS = a.divS;
    // shared arrays are written once (both directions, pair-bound routes)
    const bool w_recv = !(DIRS & kZC) || !a.cz_recv_shared;
    const bool w_send = !(DIRS & kZC) || !a.cz_send_shared;
    int32_t wdoc = -1;
    const int32_t t_last = static_cast<int32_t>((end - 1) / cp);
    for (int32_t tile = static_cast<int32_t>(begin / cp); tile <= t_last; ++tile) {
      const SlotTile t = slot_tile(cu, n, m, S, tile, wdoc);
      const int64_t q0 = static_cast<int64_t>(tile) * cp;
      const int32_t r0 = static_cast<int32_t>(max(begin - q0, int64_t{0}));
      const int32_t r1 = static_cast<int32_t>(min(end - q0, static_cast<int64_t>(cp)));
      // A document inside one contiguous rank's interval (all but the few
      // that straddle a boundary d*S) sends all its rows to the same rank
      // d: then d is taken once for the lane instead of once per rank.
      const int32_t d_lo = divS.div(t.c0), d_hi = divS.div(t.c1 - 1);
      const bool one_d = __all_sync(kFullMask, !t.valid || d_lo == d_hi);
      if (!t.valid || !in_range(t.doc, 0, n, a.status)) continue;
      // rank r0's global row and zigzag position, then one rank further per step
      int32_t g = t.base + r0 * t.step;
      int32_t u = r0 * S + t.j;
      const int32_t* prow = prd + r0 * cp;
#pragma unroll kRouteUnroll
      for (int32_t r = r0; r < r1; ++r, g += t.step, u += S, prow += cp) {
        if (!in_range(g, 0, T, a.status)) continue;
        const int32_t d = one_d ? d_lo : divS.div(g);
        const int32_t pos = prow[d] + t.j;
        const int32_t gl = g - d * S;
        if (!in_range(pos, d * static_cast<int64_t>(S), (d + 1) * static_cast<int64_t>(S), a.status)) continue;
        if (DIRS & kZC) {
          a.zc.src_of_dst[g] = u;
          a.zc.send_rows[u] = t.j;
          a.zc.recv_rows[pos] = gl;
        }
        if (DIRS & kCZ) {
          a.cz.src_of_dst[u] = g;
          if (w_recv) a.cz.recv_rows[u] = t.j;
          if (w_send) a.cz.send_rows[pos] = gl;
        }
      }
    }
  }
  // split sizes, offsets and identity flags: the last block, which has the
  // fewest walk items (equal shares, remainder last), after its walk
  if (blockIdx.x == gridDim.x - 1) {
    if (DIRS & kZC) write_small_arrays(a.zc, true, cu, n, m, S, cnt, roff);
    if (DIRS & kCZ) write_small_arrays(a.cz, false, cu, n, m, S, cnt, roff);
  }
}

template <bool SMEM_CU>
__global__ void __launch_bounds__(kRouteThreads)
partition_kernel(const int32_t* cu_g, int32_t n, int32_t T, CpMath m, int32_t S, int32_t rank,
                 int32_t* out, int32_t* status) {
  extern __shared__ int32_t smem[];
  pdl_wait_then_release();
  const int32_t code = stage_check_cu(cu_g, n, smem, SMEM_CU, status, T, 2 * m.cp);
  if (code != THD_OK) {
    if (code != kStatusWasSet && blockIdx.x == 0 && threadIdx.x == 0) status_set(status, code);
    return;
  }
  const int32_t* cu = SMEM_CU ? smem : cu_g;
  // all ranks: out[r*S + j] for every (slot tile, rank) item; one rank r:
  // out[j], one item per slot tile
  const int32_t nr = rank < 0 ? m.cp : 1;
  const int32_t r_base = rank < 0 ? 0 : rank;
  const int64_t tiles = (static_cast<int64_t>(S) + 31) / 32;
  int64_t begin, end;
  warp_items(tiles * nr, 1, &begin, &end);
  if (begin >= end) return;
  int32_t wdoc = -1;
  const int32_t t_last = static_cast<int32_t>((end - 1) / nr);
  for (int32_t tile = static_cast<int32_t>(begin / nr); tile <= t_last; ++tile) {
    const SlotTile t = slot_tile(cu, n, m, S, tile, wdoc);
    const int64_t q0 = static_cast<int64_t>(tile) * nr;
    const int32_t r0 = static_cast<int32_t>(max(begin - q0, int64_t{0}));
    const int32_t r1 = static_cast<int32_t>(min(end - q0, static_cast<int64_t>(nr)));
    if (!t.valid || !in_range(t.doc, 0, n, status)) continue;
    for (int32_t rr = r0; rr < r1; ++rr) {
      const int32_t r = r_base + rr;
      const int32_t g = t.base + r * t.step;
      if (in_range(g, 0, T, status)) out[rank < 0 ? r * S + t.j : t.j] = g;
    }
  }
}

// Blocks for `items` (slot tile, rank) work items: a warp per item, at most
// THD_ROUTE_BLOCKS_PER_SM blocks per SM.
int grid_for_items(int64_t items) {
  int64_t want = (items + kRouteThreads / 32 - 1) / (kRouteThreads / 32);
  int64_t cap = static_cast<int64_t>(sm_count()) * THD_ROUTE_BLOCKS_PER_SM;
  if (want > cap) want = cap;
  if (want < 1) want = 1;
  return static_cast<int>(want);
}

}  // namespace

thd_status_t launch_route_build(const int32_t* cu, int32_t n, int32_t T, int32_t cp, int32_t dirs,
                                const thd_route_t* zc, const thd_route_t* cz, int32_t* status,
                                cudaStream_t s) {
  RouteArgs a;
  a.cu = cu;
  a.n = n;
  a.T = T;
  a.S = T / cp;
  a.m = make_cp_math(cp);
  a.divS = make_fast_div(a.S > 0 ? a.S : 1);
  a.divCp1 = make_fast_div(cp + 1);
  a.zc = zc ? *zc : thd_route_t{};
  a.cz = cz ? *cz : thd_route_t{};
  a.status = status;
  a.cz_send_shared = zc && cz && zc->recv_rows == cz->send_rows;
  a.cz_recv_shared = zc && cz && zc->send_rows == cz->recv_rows;
  const size_t tables =
      (static_cast<size_t>(2 * cp + 3) * (cp + 1) + static_cast<size_t>(cp) * cp) * sizeof(int32_t);
  const size_t cu_bytes = static_cast<size_t>(n + 1) * sizeof(int32_t);
  a.cu_in_smem = cu_bytes <= static_cast<size_t>(kSmemBudget);
  const size_t smem = tables + (a.cu_in_smem ? cu_bytes : 0);
  const int grid = grid_for_items((static_cast<int64_t>(a.S) + 31) / 32 * cp);
  auto go = [&](void (*kernel)(RouteArgs)) -> cudaError_t {
    // above 48 KB (cp near 64 with many documents) the block opts in to more
    if (smem > 48 * 1024) {
      const cudaError_t e0 =
          cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
      if (e0 != cudaSuccess) return e0;
    }
    return launch_pdl(kernel, grid, kRouteThreads, smem, s, a);
  };
  cudaError_t e;
  if (a.cu_in_smem) {
    e = go(dirs == (kZC | kCZ) ? route_build_kernel<kZC | kCZ, true>
                               : dirs == kZC ? route_build_kernel<kZC, true> : route_build_kernel<kCZ, true>);
  } else {
    e = go(dirs == (kZC | kCZ) ? route_build_kernel<kZC | kCZ, false>
                               : dirs == kZC ? route_build_kernel<kZC, false> : route_build_kernel<kCZ, false>);
  }
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return THD_ERR_CUDA;
  }
  return THD_OK;
}

thd_status_t launch_partition(const int32_t* cu, int32_t n, int32_t T, int32_t cp, int32_t rank,
                              int32_t* out, int32_t* status, cudaStream_t s) {
  size_t cu_bytes = static_cast<size_t>(n + 1) * sizeof(int32_t);
  bool in_smem = cu_bytes <= static_cast<size_t>(kSmemBudget);
  int32_t S = T / cp;
  int grid = grid_for_items((static_cast<int64_t>(S) + 31) / 32 * (rank < 0 ? cp : 1));
  const CpMath m = make_cp_math(cp);
  const cudaError_t e =
      in_smem ? launch_pdl(partition_kernel<true>, grid, kRouteThreads, cu_bytes, s, cu, n, T, m, S, rank, out,
                           status)
              : launch_pdl(partition_kernel<false>, grid, kRouteThreads, 0, s, cu, n, T, m, S, rank, out, status);
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return THD_ERR_CUDA;
  }
  return THD_OK;
}

}  // namespace thd
