// Device-side route build and zigzag partition indices.
//
// "[Task32] feat: fla mcore chunkwise cp stage 3" (Relax PR #273), section 2.1:
// both layouts are unions of global row intervals, so the all-to-all route
// follows from interval intersection.  The pages copy cu_seqlens to the host
// and intersect with a Python two-pointer loop; here every block validates
// the boundaries itself, derives the per-(rank, rank) intersection sizes from
// a closed-form count of zigzag rows below a position, and then writes each
// route entry from its own index with a binary search of the boundaries (a
// gather, so all stores are coalesced).  No host synchronisation, no atomics
// on the route, one launch per direction.
#include "thd_internal.cuh"

namespace thd {
namespace {

constexpr int kRouteThreads = 512;
constexpr int kSmemBudget = 48 * 1024;

struct RouteArgs {
  const int32_t* cu;
  int32_t n, T, cp, S;
  bool cu_in_smem;
  thd_route_t r;
  int32_t* status;
};

// Does rank-interval [lo, lo+S) of the contiguous layout contain two
// neighbouring rows whose zigzag owners decrease?  Owners along a document
// run 0,1,..,cp-1,cp-1,..,1,0 chunk by chunk, so a decrease happens exactly
// at the starts of chunks cp+1 .. 2cp-1.  No decrease <=> sorting the
// interval's rows by (owner, row) keeps them in row order <=> the receive
// rows of z->c (equally the send rows of c->z) of that rank are 0..S-1.
__device__ bool has_descent(const int32_t* cu, int32_t n, int32_t cp, int32_t lo, int32_t hi) {
  if (cp == 1 || hi <= lo) return false;
  int32_t ilo = doc_of(cu, n, lo), ihi = doc_of(cu, n, hi - 1);
  if (ihi > ilo && cu[ihi] > cu[ilo + 1]) return true;  // a whole non-empty document inside
  for (int pass = 0; pass < 2; ++pass) {
    int32_t i = pass == 0 ? ilo : ihi;
    if (pass == 1 && ihi == ilo) break;
    int32_t L = cu[i + 1] - cu[i];
    if (L == 0) continue;
    int32_t c = L / (2 * cp);
    // descents at b = cu[i] + m*c, m = cp+1 .. 2cp-1; need lo+1 <= b <= hi-1
    int32_t a = lo + 1 - cu[i];
    int32_t mlo = a <= 0 ? cp + 1 : max(cp + 1, (a + c - 1) / c);
    int32_t b = hi - 1 - cu[i];
    if (b < 0) continue;
    int32_t mhi = min(2 * cp - 1, b / c);
    if (mlo <= mhi) return true;
  }
  return false;
}

// Receive row j of contiguous rank d under z->c (the same list is the send
// row list of contiguous rank d under c->z): the sender s is the rank whose
// block [roff[d][s], roff[d][s+1]) holds j; the row is the (j - roff[d][s])-th
// zigzag row of s inside d's interval.
__device__ __forceinline__ int32_t contiguous_side_row(const int32_t* cu, int32_t n, int32_t cp,
                                                       int32_t S, const int32_t* cnt,
                                                       const int32_t* roff, int32_t d, int32_t j) {
  const int32_t* ro = roff + d * (cp + 1);
  int32_t s = 0, len = cp;  // largest s in [0, cp) with ro[s] <= j
  while (len > 1) {
    int32_t half = len >> 1;
    s = (ro[s + half] <= j) ? s + half : s;
    len -= half;
  }
  int32_t slot = cnt[s * (cp + 1) + d] + (j - ro[s]);
  return zigzag_row(cu, n, cp, s, slot) - d * S;
}

template <int DIR>
__global__ void __launch_bounds__(kRouteThreads) route_build_kernel(RouteArgs a) {
  extern __shared__ int32_t smem[];
  if (block_status_set(a.status)) return;
  const int32_t cp = a.cp, S = a.S, T = a.T, n = a.n;
  int32_t* cnt = smem;                        // [cp][cp+1]: zigzag rows of s below d*S
  int32_t* roff = cnt + cp * (cp + 1);        // [d][cp+1]: z->c receive offsets
  int32_t* cu_s = roff + cp * (cp + 1);
  const int32_t* cu = stage_cu(a.cu, n, cu_s, a.cu_in_smem);

  int32_t code = block_check_cu(cu, n, T, 2 * cp, true);
  if (code != THD_OK) {
    if (blockIdx.x == 0 && threadIdx.x == 0) status_set(a.status, code);
    return;
  }

  for (int32_t e = threadIdx.x; e < cp * (cp + 1); e += blockDim.x) {
    int32_t s = e / (cp + 1), d = e - s * (cp + 1);
    cnt[e] = zigzag_count_below(cu, n, cp, S, T, s, d * S);
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

  const thd_route_t& r = a.r;
  if (blockIdx.x == 0) {
    for (int32_t e = threadIdx.x; e < cp * cp; e += blockDim.x) {
      int32_t x = e / cp, y = e - x * cp;
      // n_zc[s][d] = rows zigzag rank s sends to contiguous rank d
      if (DIR == THD_ZIGZAG_TO_CONTIGUOUS) {
        int32_t nxy = cnt[x * (cp + 1) + y + 1] - cnt[x * (cp + 1) + y];  // n_zc[x][y]
        r.input_split_sizes[e] = nxy;   // [s=x][d=y]
        int32_t nyx = cnt[y * (cp + 1) + x + 1] - cnt[y * (cp + 1) + x];  // n_zc[y][x]
        r.output_split_sizes[e] = nyx;  // [d=x][s=y]
      } else {
        int32_t nyx = cnt[y * (cp + 1) + x + 1] - cnt[y * (cp + 1) + x];  // n_zc[y][x]
        r.input_split_sizes[e] = nyx;   // [s=x][d=y] = n_zc[d][s]
        int32_t nxy = cnt[x * (cp + 1) + y + 1] - cnt[x * (cp + 1) + y];  // n_zc[x][y]
        r.output_split_sizes[e] = nxy;  // [d=x][s=y] = n_zc[d][s]
      }
    }
    for (int32_t e = threadIdx.x; e < cp * (cp + 1); e += blockDim.x) {
      if (DIR == THD_ZIGZAG_TO_CONTIGUOUS) {
        r.send_offsets[e] = cnt[e];   // [s][d] = zigzag rows of s below d*S
        r.recv_offsets[e] = roff[e];  // [d][s]
      } else {
        r.send_offsets[e] = roff[e];  // [s][d]
        r.recv_offsets[e] = cnt[e];   // [d][s]
      }
    }
    for (int32_t k = threadIdx.x; k < cp; k += blockDim.x) {
      uint8_t reorder = has_descent(cu, n, cp, k * S, (k + 1) * S) ? 0 : 1;
      if (DIR == THD_ZIGZAG_TO_CONTIGUOUS) {
        r.send_identity[k] = 1;
        r.recv_identity[k] = reorder;
      } else {
        r.send_identity[k] = reorder;
        r.recv_identity[k] = 1;
      }
    }
  }

  const int32_t stride = gridDim.x * blockDim.x;
  for (int32_t u = blockIdx.x * blockDim.x + threadIdx.x; u < T; u += stride) {
    int32_t rank = u / S;
    int32_t j = u - rank * S;
    if (DIR == THD_ZIGZAG_TO_CONTIGUOUS) {
      r.src_of_dst[u] = zigzag_pos(cu, n, cp, S, u);
      r.send_rows[u] = j;
      r.recv_rows[u] = contiguous_side_row(cu, n, cp, S, cnt, roff, rank, j);
    } else {
      r.src_of_dst[u] = zigzag_row(cu, n, cp, rank, j);
      r.send_rows[u] = contiguous_side_row(cu, n, cp, S, cnt, roff, rank, j);
      r.recv_rows[u] = j;
    }
  }
}

__global__ void __launch_bounds__(kRouteThreads)
partition_kernel(const int32_t* cu_g, int32_t n, int32_t T, int32_t cp, int32_t S, int32_t rank,
                 bool cu_in_smem, int32_t* out, int32_t* status) {
  extern __shared__ int32_t smem[];
  if (block_status_set(status)) return;
  const int32_t* cu = stage_cu(cu_g, n, smem, cu_in_smem);
  int32_t code = block_check_cu(cu, n, T, 2 * cp, true);
  if (code != THD_OK) {
    if (blockIdx.x == 0 && threadIdx.x == 0) status_set(status, code);
    return;
  }
  const int32_t total = rank < 0 ? T : S;
  const int32_t stride = gridDim.x * blockDim.x;
  for (int32_t u = blockIdx.x * blockDim.x + threadIdx.x; u < total; u += stride) {
    int32_t r = rank < 0 ? u / S : rank;
    int32_t slot = rank < 0 ? u - r * S : u;
    out[u] = zigzag_row(cu, n, cp, r, slot);
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

thd_status_t launch_route_build(const int32_t* cu, int32_t n, int32_t T, int32_t cp, int32_t dir,
                                const thd_route_t* route, int32_t* status, cudaStream_t s) {
  RouteArgs a;
  a.cu = cu;
  a.n = n;
  a.T = T;
  a.cp = cp;
  a.S = T / cp;
  a.r = *route;
  a.status = status;
  size_t tables = static_cast<size_t>(2) * cp * (cp + 1) * sizeof(int32_t);
  size_t cu_bytes = static_cast<size_t>(n + 1) * sizeof(int32_t);
  a.cu_in_smem = tables + cu_bytes <= static_cast<size_t>(kSmemBudget);
  size_t smem = tables + (a.cu_in_smem ? cu_bytes : 0);
  int grid = grid_for(T, kRouteThreads, 2);
  if (dir == THD_ZIGZAG_TO_CONTIGUOUS)
    route_build_kernel<THD_ZIGZAG_TO_CONTIGUOUS><<<grid, kRouteThreads, smem, s>>>(a);
  else
    route_build_kernel<THD_CONTIGUOUS_TO_ZIGZAG><<<grid, kRouteThreads, smem, s>>>(a);
  cudaError_t e = cudaGetLastError();
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
  partition_kernel<<<grid, kRouteThreads, in_smem ? cu_bytes : 0, s>>>(cu, n, T, cp, S, rank, in_smem,
                                                                      out, status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return THD_ERR_CUDA;
  }
  return THD_OK;
}

}  // namespace thd
