// Device-side route build and zigzag partition indices.
//
// "[Task32] feat: fla mcore chunkwise cp stage 3" (Relax PR #273), section 2.1:
// both layouts are unions of global row intervals, so the all-to-all route
// follows from interval intersection.  The pages copy cu_seqlens to the host
// and intersect with a Python two-pointer loop.  Here one kernel per call:
//
//  1. every block stages the boundaries in shared memory, validates them
//     (all blocks reach the same verdict; block 0 writes the status word) and
//     derives the cp x (cp+1) table "zigzag rows of rank s below d*S" in
//     closed form, plus the receive offsets;
//  2. warps walk the zigzag buffer in tiles of 32 consecutive positions
//     (rank r, slot j).  A tile's documents come from one full search of the
//     boundaries plus a short window search per lane; the global row g, the
//     contiguous rank of g and the entry's place in every route array then
//     follow in closed form, with divisions by S done by multiply-shift.
//
// No host synchronisation, no atomics on the route, deterministic.
#include "thd_internal.cuh"

namespace thd {
namespace {

constexpr int kRouteThreads = 512;
constexpr int kSmemBudget = 48 * 1024;

struct RouteArgs {
  const int32_t* cu;
  int32_t n, T, S;
  CpMath m;
  FastDiv divS;
  bool cu_in_smem;
  thd_route_t zc;  // zigzag -> contiguous (used when bit 0 of DIRS is set)
  thd_route_t cz;  // contiguous -> zigzag (used when bit 1 of DIRS is set)
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

// Split sizes, offsets and identity flags of one direction (block 0 only).
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
  int32_t* cu_s = roff + cp * (cp + 1);
  const int32_t* unused;
  pdl_wait_then_release();
  if (stage_cu_check_status(a.cu, n, cu_s, SMEM_CU, a.status, &unused)) return;
  const int32_t* cu = SMEM_CU ? cu_s : a.cu;

  int32_t code = block_check_cu(cu, n, T, 2 * cp, true);
  if (code != THD_OK) {
    if (blockIdx.x == 0 && threadIdx.x == 0) status_set(a.status, code);
    return;
  }

  for (int32_t e = threadIdx.x; e < cp * (cp + 1); e += blockDim.x) {
    int32_t s = e / (cp + 1), d = e - s * (cp + 1);
    cnt[e] = zigzag_count_below(cu, n, m, S, T, s, d * S);
  }
  __syncthreads();
  for (int32_t d = threadIdx.x; d < cp; d += blockDim.x) {
    int32_t acc = 0;
    for (int32_t s = 0; s < cp; ++s) {
      roff[d * (cp + 1) + s] = acc;
      acc += cnt[s * (cp + 1) + d + 1] - cnt[s * (cp + 1) + d];
    }
    roff[d * (cp + 1) + cp] = acc;
  }
  __syncthreads();

  if (blockIdx.x == 0) {
    if (DIRS & kZC) write_small_arrays(a.zc, true, cu, n, m, S, cnt, roff);
    if (DIRS & kCZ) write_small_arrays(a.cz, false, cu, n, m, S, cnt, roff);
  }

  // Zigzag position u = r*S + j holds global row g.  Then
  //   z->c: src_of_dst[g] = u, send_rows[u] = j;
  //   c->z: src_of_dst[u] = g, recv_rows[u] = j;
  //   with d = g / S the contiguous rank of g, the row is entry
  //   roff[d][r] + (j - cnt[r][d]) of d's z->c receive buffer and of d's c->z
  //   send buffer, with value g - d*S.
  int64_t begin, end;
  warp_range(T, &begin, &end);
  const FastDiv divS = a.divS;
  const int32_t lane = threadIdx.x & 31;
  TileWalker w{0, -1};
  for (int64_t tile0 = begin; tile0 < end; tile0 += 32) {
    const TileRow t = tile_row(cu, n, m, S, divS, static_cast<int32_t>(tile0) + lane,
                               static_cast<int32_t>(end) - 1, w);
    if (t.u < end && in_range(t.doc, 0, n, a.status) && in_range(t.g, 0, T, a.status)) {
      const int32_t d = divS.div(t.g);
      const int32_t pos = d * S + roff[d * (cp + 1) + t.r] + (t.j - cnt[t.r * (cp + 1) + d]);
      if (!in_range(pos, d * static_cast<int64_t>(S), (d + 1) * static_cast<int64_t>(S), a.status)) continue;
      if (DIRS & kZC) {
        a.zc.src_of_dst[t.g] = t.u;
        a.zc.send_rows[t.u] = t.j;
        a.zc.recv_rows[pos] = t.g - d * S;
      }
      if (DIRS & kCZ) {
        a.cz.src_of_dst[t.u] = t.g;
        a.cz.recv_rows[t.u] = t.j;
        a.cz.send_rows[pos] = t.g - d * S;
      }
    }
  }
}

template <bool SMEM_CU>
__global__ void __launch_bounds__(kRouteThreads)
partition_kernel(const int32_t* cu_g, int32_t n, int32_t T, CpMath m, FastDiv divS, int32_t S, int32_t rank,
                 int32_t* out, int32_t* status) {
  extern __shared__ int32_t smem[];
  const int32_t* unused;
  pdl_wait_then_release();
  if (stage_cu_check_status(cu_g, n, smem, SMEM_CU, status, &unused)) return;
  const int32_t* cu = SMEM_CU ? smem : cu_g;
  int32_t code = block_check_cu(cu, n, T, 2 * m.cp, true);
  if (code != THD_OK) {
    if (blockIdx.x == 0 && threadIdx.x == 0) status_set(status, code);
    return;
  }
  // all ranks: out[u] for zigzag positions u in [0, T); one rank r: out[j]
  // for positions r*S + j, j in [0, S)
  const int32_t total = rank < 0 ? T : S;
  const int32_t base = rank < 0 ? 0 : rank * S;
  int64_t begin, end;
  warp_range(total, &begin, &end);
  const int32_t lane = threadIdx.x & 31;
  TileWalker w{0, -1};
  for (int64_t tile0 = begin; tile0 < end; tile0 += 32) {
    const int32_t k = static_cast<int32_t>(tile0) + lane;
    const TileRow t = tile_row(cu, n, m, S, divS, base + k, base + static_cast<int32_t>(end) - 1, w);
    if (k < end && in_range(t.g, 0, T, status)) out[k] = t.g;
  }
}

int grid_for(int64_t work, int threads, int per_sm) {
  int64_t want = (work + threads - 1) / threads;
  int64_t cap = static_cast<int64_t>(sm_count()) * per_sm;
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
  a.zc = zc ? *zc : thd_route_t{};
  a.cz = cz ? *cz : thd_route_t{};
  a.status = status;
  size_t tables = static_cast<size_t>(2) * cp * (cp + 1) * sizeof(int32_t);
  size_t cu_bytes = static_cast<size_t>(n + 1) * sizeof(int32_t);
  a.cu_in_smem = tables + cu_bytes <= static_cast<size_t>(kSmemBudget);
  size_t smem = tables + (a.cu_in_smem ? cu_bytes : 0);
  int grid = grid_for(T, kRouteThreads, 2);
  cudaError_t e;
  if (a.cu_in_smem) {
    if (dirs == (kZC | kCZ))
      e = launch_pdl(route_build_kernel<kZC | kCZ, true>, grid, kRouteThreads, smem, s, a);
    else if (dirs == kZC)
      e = launch_pdl(route_build_kernel<kZC, true>, grid, kRouteThreads, smem, s, a);
    else
      e = launch_pdl(route_build_kernel<kCZ, true>, grid, kRouteThreads, smem, s, a);
  } else {
    if (dirs == (kZC | kCZ))
      e = launch_pdl(route_build_kernel<kZC | kCZ, false>, grid, kRouteThreads, smem, s, a);
    else if (dirs == kZC)
      e = launch_pdl(route_build_kernel<kZC, false>, grid, kRouteThreads, smem, s, a);
    else
      e = launch_pdl(route_build_kernel<kCZ, false>, grid, kRouteThreads, smem, s, a);
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
  int grid = grid_for(rank < 0 ? T : S, kRouteThreads, 2);
  const CpMath m = make_cp_math(cp);
  const FastDiv divS = make_fast_div(S > 0 ? S : 1);
  const cudaError_t e =
      in_smem ? launch_pdl(partition_kernel<true>, grid, kRouteThreads, cu_bytes, s, cu, n, T, m, divS, S, rank, out,
                           status)
              : launch_pdl(partition_kernel<false>, grid, kRouteThreads, 0, s, cu, n, T, m, divS, S, rank, out, status);
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return THD_ERR_CUDA;
  }
  return THD_OK;
}

}  // namespace thd
