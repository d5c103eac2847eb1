// Document-bounded labels, MTP targets and the valid-token mask.
//
// "Packed Sequence 与上下文并行", section 1.3 (the label roll must not cross a
// sample), section 1.6 (MTP depth i must not take the next document's first
// tokens as targets), section 2.2 (valid_local_token_mask is 0 on padding)
// and section 3.8 (the EOD position's label is masked).  The pages build
// these with an O(num_docs) Python fix-up loop and a separate MTP roll; here
// one kernel writes every depth at once: position p of document i takes
// tokens[p+1+k] at depth k when p+1+k is still before the document's valid
// end e_i, else `fill` with mask 0.  Warps walk contiguous position ranges
// and follow the current document forward, so finding it costs a step or
// two per 32 positions instead of a full search per position; the zigzag
// variant walks the rows the same way and writes each to its zigzag slot.
#include "thd_internal.cuh"

namespace thd {
namespace {

constexpr int kLabelThreads = 512;
// Boundaries (padded and unpadded) staged in shared memory up to this size
// (about 20,000 documents); above 48 KB the launch opts in to the larger
// dynamic shared memory.  Searching them in global memory instead puts an L2
// round trip on every step of every warp's document search.
constexpr int kSmemBudget = 160 * 1024;

// Launch with `smem` bytes of dynamic shared memory, opting in above 48 KB.
template <typename... Params, typename... Args>
cudaError_t launch_smem(void (*kernel)(Params...), dim3 grid, size_t smem, cudaStream_t s, Args... args) {
  if (smem > 48 * 1024) {
    const cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  return launch_pdl(kernel, grid, dim3(kLabelThreads), smem, s, args...);
}
// At most this many blocks per SM for the zigzag variant.
#ifndef THD_LABEL_ZZ_BLOCKS_PER_SM
#define THD_LABEL_ZZ_BLOCKS_PER_SM 2
#endif

// Optional continuation of a document cut by the end of its sample (the
// sample's extra token, "Packed Sequence 与上下文并行" section 1.3): when
// has[i], document i's token stream is its valid tokens followed by tok[i].
struct NextTokens {
  const int32_t* tok;
  const uint8_t* has;
};

// Positions per lane: a lane writes each depth's four labels with one
// 16-byte store and its four masks with one 4-byte store (VEC: T a multiple
// of 4, labels 16-byte and masks 4-byte aligned), else one position at a time.
constexpr int kPerLane = 4;
// tokens kept per lane for four consecutive rows: four rows, depths up to 7
constexpr int kZzWindow = kPerLane + 7;

template <bool SMEM_CU, bool VEC>
__global__ void __launch_bounds__(kLabelThreads)
roll_labels_kernel(const int32_t* __restrict__ tokens, const int32_t* cu_v_g, const int32_t* cu_g,
                   int32_t n, int32_t T, int32_t depth, int32_t fill, NextTokens next, int32_t* __restrict__ labels,
                   uint8_t* __restrict__ lmask, uint8_t* __restrict__ valid, int32_t* status) {
  extern __shared__ int32_t smem[];
  const int32_t* unused;
  pdl_wait_then_release();
  if (SMEM_CU) stage_rows(cu_v_g, n + 1, smem + (n + 1));  // covered by the barrier below
  if (stage_cu_check_status(cu_g, n, smem, SMEM_CU, status, &unused)) return;
  const int32_t* cu = SMEM_CU ? smem : cu_g;
  const int32_t* cu_v = SMEM_CU ? smem + (n + 1) : cu_v_g;

  int32_t code = block_check_cu(cu, n, T, 0, true);
  if (code == THD_OK) {
    code = block_check_cu(cu_v, n, 0, 0, false);
    if (code == THD_OK) {
      int bad = 0;
      for (uint32_t i = threadIdx.x; i < static_cast<uint32_t>(n); i += blockDim.x)
        if (cu_v[i + 1] - cu_v[i] > cu[i + 1] - cu[i]) bad = 1;  // both checked monotone from 0
      if (__syncthreads_or(bad)) code = THD_ERR_VALID_EXCEEDS_PADDED;
    }
  }
  if (code != THD_OK) {
    if (blockIdx.x == 0 && threadIdx.x == 0) status_set(status, code);
    return;
  }
  if (T == 0) return;

  // Each warp walks an equal contiguous range of positions, 128 per step
  // (four consecutive ones per lane), following the document of its lowest
  // position forward (galloping search).  Steps start at multiples of 128, so
  // p + 3 stays within int32 for every T below 2^31.
  constexpr int kStep = 32 * kPerLane;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int64_t tiles = (static_cast<int64_t>(T) + kStep - 1) / kStep;
  const int64_t per = (tiles + nwarps - 1) / nwarps;
  const int64_t begin = min(static_cast<int64_t>(T), warp * per * kStep);
  const int64_t end = min(static_cast<int64_t>(T), (warp + 1) * per * kStep);
  const int32_t lane = threadIdx.x & 31;
  const int32_t last = static_cast<int32_t>(end) - 1;
  int32_t doc = -1;
  for (int64_t tile0 = begin; tile0 < end; tile0 += kStep) {
    const int32_t p0 = static_cast<int32_t>(tile0) + kPerLane * lane;
    const int32_t x_lo = static_cast<int32_t>(tile0);
    const int32_t x_hi = __shfl_sync(kFullMask, min(p0 + kPerLane - 1, last), 31);
    const int32_t i_lo = doc < 0 ? doc_of(cu, n, x_lo) : doc_from(cu, n, doc, x_lo);
    const int32_t i_hi = doc_from(cu, n, i_lo, x_hi);
    int32_t i = doc_in(cu, i_lo, i_hi, min(p0, last));
    doc = i_lo;
    if (p0 > last || !in_range(i, 0, n, status)) continue;
    // each position's document, valid end and continuation
    int32_t di[kPerLane], ei[kPerLane];
    bool full = p0 + kPerLane - 1 <= last, bad = false;
    uint32_t vbits = 0;
#pragma unroll
    for (int t = 0; t < kPerLane; ++t) {
      const int32_t q = p0 + t;
      if (q > last) {
        di[t] = i, ei[t] = 0;
        continue;
      }
      while (cu[i + 1] <= q) ++i;  // q < T = cu[n]: stops before i = n
      di[t] = i;
      ei[t] = cu[i] + (cu_v[i + 1] - cu_v[i]);  // end of the document's valid tokens
      bad |= !in_range(ei[t], 0, static_cast<int64_t>(T) + 1, status);  // token reads stay below e
      vbits |= (q < ei[t] ? 1u : 0u) << (8 * t);
    }
    if (bad) continue;
    if (VEC && full) {
      *reinterpret_cast<uint32_t*>(valid + p0) = vbits;
    } else {
      for (int t = 0; t < kPerLane && p0 + t <= last; ++t) valid[p0 + t] = static_cast<uint8_t>(vbits >> (8 * t));
    }
    // four positions of one document, depths within the window: one window
    // of tokens serves every depth (position p0 + t at depth k reads token
    // p0 + 1 + t + k while t + k < R)
    if (VEC && full && di[0] == di[kPerLane - 1] && depth <= kZzWindow - kPerLane) {
      const int32_t R = ei[0] - p0 - 1;
      int32_t w[kZzWindow];
#pragma unroll
      for (int x = 0; x < kZzWindow; ++x) w[x] = x <= depth + kPerLane - 1 && x < R ? __ldg(tokens + p0 + 1 + x) : fill;
      const bool has = next.has != nullptr && next.has[di[0]] != 0;
      const int32_t nt = has ? next.tok[di[0]] : fill;
#pragma unroll
      for (int k = 0; k <= kZzWindow - kPerLane; ++k) {
        if (k > depth) break;
        int32_t v[kPerLane];
        uint32_t mbits = 0;
#pragma unroll
        for (int t = 0; t < kPerLane; ++t) {
          const bool in = t + k < R, at_end = t + k == R && has;
          v[t] = in ? w[t + k] : (at_end ? nt : fill);
          mbits |= (in || at_end ? 1u : 0u) << (8 * t);
        }
        const int64_t o = static_cast<int64_t>(k) * T + p0;
        *reinterpret_cast<int4*>(labels + o) = make_int4(v[0], v[1], v[2], v[3]);
        *reinterpret_cast<uint32_t*>(lmask + o) = mbits;
      }
      continue;
    }
    for (int32_t k = 0; k <= depth; ++k) {
      int32_t v[kPerLane];
      uint32_t mbits = 0;
#pragma unroll
      for (int t = 0; t < kPerLane; ++t) {
        const int32_t q = p0 + t;
        v[t] = fill;
        if (q > last) continue;
        // depth k reads tokens[q+1+k] while k < room (no sum passes e)
        const int32_t room = ei[t] - q - 1;
        if (k < room) {
          v[t] = __ldg(tokens + q + 1 + k);
          mbits |= 1u << (8 * t);
        } else if (k == room && next.has != nullptr && next.has[di[t]] != 0) {
          v[t] = next.tok[di[t]];
          mbits |= 1u << (8 * t);
        }
      }
      const int64_t o = static_cast<int64_t>(k) * T + p0;
      if (VEC && full) {
        *reinterpret_cast<int4*>(labels + o) = make_int4(v[0], v[1], v[2], v[3]);
        *reinterpret_cast<uint32_t*>(lmask + o) = mbits;
      } else {
        for (int t = 0; t < kPerLane && p0 + t <= last; ++t) {
          labels[o + t] = v[t];
          lmask[o + t] = static_cast<uint8_t>(mbits >> (8 * t));
        }
      }
    }
  }
}

// The same labels written in the zigzag layout: global row g goes to zigzag
// position u = r*S + j, so out[k][u] = labels[k][g] (and the same for the
// masks) -- the label roll and the partition gather in one pass.  Warps walk
// global rows in order, following the current document forward as the
// contiguous kernel does, so every token is read once and in order; row g of document i (start c0, chunk length c) lies in chunk
// k = (g - c0) / c, which rank r = k or 2cp-1-k holds at local slot
// c0/cp + (k < cp ? 0 : c) + (g - c0 - k*c).  The writes follow the zigzag
// order in runs of one chunk.
// floor(off / c) for 0 <= off and 1 <= c: below 2^24 both are exact in
// float, the float quotient is within one of the true one, and one
// integer step on each side corrects it; larger offsets divide exactly.
__device__ __forceinline__ int32_t chunk_of(int32_t off, int32_t c) {
  if (off >= (1 << 24)) return off / c;
  int32_t k = __float2int_rz(__fdividef(static_cast<float>(off), static_cast<float>(c)));
  if (k * c > off) --k;
  else if ((k + 1) * c <= off) ++k;
  return k;
}

template <bool SMEM_CU, bool NEXT>
__global__ void __launch_bounds__(kLabelThreads)
roll_labels_zigzag_kernel(const int32_t* __restrict__ tokens, const int32_t* cu_v_g, const int32_t* cu_g,
                          int32_t n, int32_t T, CpMath m, int32_t depth, int32_t fill, NextTokens next,
                          int32_t* __restrict__ labels, uint8_t* __restrict__ lmask, uint8_t* __restrict__ valid,
                          int32_t* status) {
  extern __shared__ int32_t smem[];
  const int32_t* unused;
  pdl_wait_then_release();
  if (SMEM_CU) stage_rows(cu_v_g, n + 1, smem + (n + 1));  // covered by the barrier below
  if (stage_cu_check_status(cu_g, n, smem, SMEM_CU, status, &unused)) return;
  const int32_t* cu = SMEM_CU ? smem : cu_g;
  const int32_t* cu_v = SMEM_CU ? smem + (n + 1) : cu_v_g;

  int32_t code = block_check_cu(cu, n, T, 2 * m.cp, true);
  if (code == THD_OK) {
    code = block_check_cu(cu_v, n, 0, 0, false);
    if (code == THD_OK) {
      int bad = 0;
      for (uint32_t i = threadIdx.x; i < static_cast<uint32_t>(n); i += blockDim.x)
        if (cu_v[i + 1] - cu_v[i] > cu[i + 1] - cu[i]) bad = 1;  // both checked monotone from 0
      if (__syncthreads_or(bad)) code = THD_ERR_VALID_EXCEEDS_PADDED;
    }
  }
  if (code != THD_OK) {
    if (blockIdx.x == 0 && threadIdx.x == 0) status_set(status, code);
    return;
  }
  if (T == 0) return;
  const int32_t S = T / m.cp;
  // Each warp an equal contiguous range of rows, 128 per step: four groups of
  // 32 consecutive rows, one row of each per lane, so every depth issues four
  // independent token loads per lane.  Steps start at multiples of 128, so
  // g stays within int32 for every T below 2^31.
  constexpr int kGroups = 4;
  constexpr int kStep = 32 * kGroups;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int64_t steps = (static_cast<int64_t>(T) + kStep - 1) / kStep;
  const int64_t per = (steps + nwarps - 1) / nwarps;
  const int64_t begin = min(static_cast<int64_t>(T), warp * per * kStep);
  const int64_t end = min(static_cast<int64_t>(T), (warp + 1) * per * kStep);
  const int32_t lane = threadIdx.x & 31;
  const int32_t last = static_cast<int32_t>(end) - 1;
  int32_t doc = -1;
  for (int64_t step0 = begin; step0 < end; step0 += kStep) {
    const int32_t x_lo = static_cast<int32_t>(step0);
    const int32_t x_hi = min(x_lo + kStep - 1, last);
    const int32_t i_lo = doc < 0 ? doc_of(cu, n, x_lo) : doc_from(cu, n, doc, x_lo);
    const int32_t i_hi = doc_from(cu, n, i_lo, x_hi);
    doc = i_lo;
    int32_t gq[kGroups], uq[kGroups], room[kGroups], iq[kGroups];
    bool ok[kGroups];
    int32_t i = i_lo;
#pragma unroll
    for (int q = 0; q < kGroups; ++q) {
      const int32_t g = x_lo + 32 * q + lane;
      i = doc_in(cu, i, i_hi, min(g, last));  // rows only move forward
      const int32_t c0 = cu[i];
      const int32_t c = m.div2(cu[i + 1] - c0);  // >= 1: document i holds row min(g, last)
      const int32_t off = min(g, last) - c0;
      const int32_t k = chunk_of(off, c);        // chunk 0 .. 2cp-1
      const bool front = k < m.cp;
      const int32_t u = (front ? k : 2 * m.cp - 1 - k) * S + m.div(c0) + (front ? 0 : c) + (off - k * c);
      const int32_t e = c0 + (cu_v[i + 1] - cu_v[i]);  // end of the document's valid tokens
      ok[q] = g <= last && in_range(i, 0, n, status) && in_range(u, 0, T, status) &&
              in_range(e, 0, static_cast<int64_t>(T) + 1, status);
      gq[q] = g;
      uq[q] = u;
      iq[q] = i;
      room[q] = e - g - 1;  // depth k reads tokens[g+1+k] while k < room (no sum passes e)
      if (ok[q]) valid[u] = g < e ? 1 : 0;
    }
    // The step's tokens [x_lo + 1, x_lo + 1 + kStep + depth) in one round of
    // loads: lane l of group q holds token x_lo + 1 + 32q + l, lanes below
    // depth one past the step; depth k of row g = x_lo + 32q + l is then
    // token 32q + l + k of that window, taken from lane (l + k) mod 32 of
    // group q or q + 1 (four dependent load rounds become one).  Tokens at or
    // past T are never used (room keeps every read below the valid end).
    int32_t win[kGroups + 1];
    const bool windowed = depth < 32;
    if (windowed) {
#pragma unroll
      for (int q = 0; q < kGroups; ++q) {
        const int32_t t = x_lo + 1 + 32 * q + lane;
        win[q] = t < T ? __ldg(tokens + t) : fill;
      }
      const int32_t t = x_lo + 1 + kStep + lane;
      win[kGroups] = lane < depth && t < T ? __ldg(tokens + t) : fill;
    }
    for (int32_t k = 0; k <= depth; ++k) {
      int32_t v[kGroups];
      if (windowed) {
        const int src = (lane + k) & 31;
        const bool wraps = lane + k >= 32;
#pragma unroll
        for (int q = 0; q < kGroups; ++q) {
          const int32_t here = __shfl_sync(kFullMask, win[q], src);
          const int32_t next_group = __shfl_sync(kFullMask, win[q + 1], src);
          v[q] = ok[q] && k < room[q] ? (wraps ? next_group : here) : fill;
        }
      } else {
#pragma unroll
        for (int q = 0; q < kGroups; ++q) v[q] = ok[q] && k < room[q] ? __ldg(tokens + gq[q] + 1 + k) : fill;
      }
#pragma unroll
      for (int q = 0; q < kGroups; ++q) {
        if (!ok[q]) continue;
        uint8_t mk = k < room[q] ? 1 : 0;
        if (NEXT && k == room[q] && next.has[iq[q]] != 0) {  // the document's next token, one past its end
          v[q] = next.tok[iq[q]];
          mk = 1;
        }
        labels[static_cast<int64_t>(k) * T + uq[q]] = v[q];
        lmask[static_cast<int64_t>(k) * T + uq[q]] = mk;
      }
    }
  }
}


// The zigzag labels in slot order, for aligned outputs (T a multiple of 4,
// labels 16-byte and masks 4-byte aligned).  Warps walk zigzag positions u in
// contiguous ranges, four consecutive ones per lane, so that every depth's
// labels go out with one 16-byte store per lane and the masks with one 4-byte
// store, as in the contiguous kernel.  Position u = r*S + j is local slot j
// of rank r; slot j lies in the document i whose local slots are
// [cu[i]/cp, cu[i+1]/cp) (the same on every rank), at offset o = j -
// cu[i]/cp: in its front chunk (o < c, chunk length c = (cu[i+1] -
// cu[i])/(2cp)) global row cu[i] + r*c + o, else in its back chunk row
// cu[i] + (2cp-1-r)*c + (o - c).  A lane's four positions are four
// consecutive rows whenever they stay in one rank, one document and one
// chunk (all but a few lanes in a hundred on documents of a few hundred
// slots); the others take each position on its own.

template <bool SMEM_CU, bool NEXT>
__global__ void __launch_bounds__(kLabelThreads)
roll_labels_zigzag_slots_kernel(const int32_t* __restrict__ tokens, const int32_t* cu_v_g, const int32_t* cu_g,
                                int32_t n, int32_t T, CpMath m, FastDiv divS, int32_t depth, int32_t fill,
                                NextTokens next, int32_t* __restrict__ labels, uint8_t* __restrict__ lmask,
                                uint8_t* __restrict__ valid, int32_t* status) {
  extern __shared__ int32_t smem[];
  const int32_t* unused;
  pdl_wait_then_release();
  if (SMEM_CU) stage_rows(cu_v_g, n + 1, smem + (n + 1));  // covered by the barrier below
  if (stage_cu_check_status(cu_g, n, smem, SMEM_CU, status, &unused)) return;
  const int32_t* cu = SMEM_CU ? smem : cu_g;
  const int32_t* cu_v = SMEM_CU ? smem + (n + 1) : cu_v_g;

  int32_t code = block_check_cu(cu, n, T, 2 * m.cp, true);
  if (code == THD_OK) {
    code = block_check_cu(cu_v, n, 0, 0, false);
    if (code == THD_OK) {
      int bad = 0;
      for (uint32_t i = threadIdx.x; i < static_cast<uint32_t>(n); i += blockDim.x)
        if (cu_v[i + 1] - cu_v[i] > cu[i + 1] - cu[i]) bad = 1;  // both checked monotone from 0
      if (__syncthreads_or(bad)) code = THD_ERR_VALID_EXCEEDS_PADDED;
    }
  }
  if (code != THD_OK) {
    if (blockIdx.x == 0 && threadIdx.x == 0) status_set(status, code);
    return;
  }
  if (T == 0) return;
  const int32_t S = T / m.cp;
  constexpr int kStep = 32 * kPerLane;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int64_t tiles = (static_cast<int64_t>(T) + kStep - 1) / kStep;
  const int64_t per = (tiles + nwarps - 1) / nwarps;
  const int64_t begin = min(static_cast<int64_t>(T), warp * per * kStep);
  const int64_t end = min(static_cast<int64_t>(T), (warp + 1) * per * kStep);
  const int32_t lane = threadIdx.x & 31;
  const int32_t last = static_cast<int32_t>(end) - 1;
  // this lane's last rank and document, to search forward from
  int32_t my_rank = -1, my_doc = 0;
  // the document of local slot j of rank r (searched forward within a rank)
  auto find_doc = [&](int32_t r, int32_t j) {
    const int32_t x = j * m.cp;  // cu[i] <= j*cp < cu[i+1] exactly when slot j lies in document i
    my_doc = r == my_rank ? doc_from(cu, n, my_doc, x) : doc_of(cu, n, x);
    my_rank = r;
    return my_doc;
  };
  // one position on its own (the general case): its label, mask and valid
  // flag at every depth
  auto one_position = [&](int32_t u) {
    const int32_t r = divS.div(u), j = u - r * S;
    const int32_t i = find_doc(r, j);
    const int32_t c0 = cu[i], c = m.div2(cu[i + 1] - c0);
    const int32_t o = j - m.div(c0);
    const int32_t g = o < c ? c0 + r * c + o : c0 + (2 * m.cp - 1 - r) * c + (o - c);
    const int32_t e = c0 + (cu_v[i + 1] - cu_v[i]);  // end of the document's valid tokens
    if (!in_range(i, 0, n, status) || !in_range(g, 0, T, status) || !in_range(e, 0, static_cast<int64_t>(T) + 1, status))
      return;
    valid[u] = g < e ? 1 : 0;
    const int32_t room = e - g - 1;  // depth k reads tokens[g+1+k] while k < room
    const bool has = NEXT && next.has[i] != 0;
    for (int32_t k = 0; k <= depth; ++k) {
      int32_t v = fill;
      uint8_t mk = 0;
      if (k < room) v = __ldg(tokens + g + 1 + k), mk = 1;
      else if (k == room && has) v = next.tok[i], mk = 1;
      labels[static_cast<int64_t>(k) * T + u] = v;
      lmask[static_cast<int64_t>(k) * T + u] = mk;
    }
  };
  for (int64_t tile0 = begin; tile0 < end; tile0 += kStep) {
    const int32_t p0 = static_cast<int32_t>(tile0) + kPerLane * lane;
    if (p0 > last) continue;
    const int32_t r = divS.div(p0), j = p0 - r * S;
    const int32_t i = find_doc(r, j);
    // four positions in one rank, all in the range, depths within the window
    if (p0 + kPerLane - 1 > last || j + kPerLane - 1 >= S || depth > kZzWindow - kPerLane) {
      for (int t = 0; t < kPerLane && p0 + t <= last; ++t) one_position(p0 + t);
      continue;
    }
    // each position's row and its room R (row g at depth k reads
    // tokens[g + 1 + k] while k < R); documents only move forward
    int32_t g[kPerLane], R[kPerLane], di[kPerLane];
    uint32_t vbits = 0;
    bool bad = false;
    int32_t it = i;
#pragma unroll
    for (int t = 0; t < kPerLane; ++t) {
      const int32_t jt = j + t;
      while (cu[it + 1] <= jt * m.cp) ++it;  // jt * cp < T = cu[n]: stops before it = n
      const int32_t c0 = cu[it], c = m.div2(cu[it + 1] - c0);
      const int32_t o = jt - m.div(c0);
      g[t] = o < c ? c0 + r * c + o : c0 + (2 * m.cp - 1 - r) * c + (o - c);
      const int32_t e = c0 + (cu_v[it + 1] - cu_v[it]);  // end of the document's valid tokens
      bad |= !in_range(g[t], 0, T, status) || !in_range(e, 0, static_cast<int64_t>(T) + 1, status);
      R[t] = e - g[t] - 1;
      di[t] = it;
      vbits |= (g[t] < e ? 1u : 0u) << (8 * t);
    }
    my_doc = it;
    if (bad) continue;
    *reinterpret_cast<uint32_t*>(valid + p0) = vbits;
    // consecutive rows of one document (all but a few lanes on long
    // documents): one window of tokens serves every depth
    const bool cons = g[1] == g[0] + 1 && g[2] == g[0] + 2 && g[3] == g[0] + 3 && di[3] == di[0];
    int32_t w[kZzWindow];
    if (cons) {
#pragma unroll
      for (int x = 0; x < kZzWindow; ++x)
        w[x] = x <= depth + kPerLane - 1 && x < R[0] ? __ldg(tokens + g[0] + 1 + x) : fill;
    }
    int32_t nt[kPerLane];
    bool has[kPerLane];
#pragma unroll
    for (int t = 0; t < kPerLane; ++t) {
      has[t] = NEXT && next.has[di[t]] != 0;
      nt[t] = has[t] ? next.tok[di[t]] : fill;
    }
#pragma unroll
    for (int k = 0; k <= kZzWindow - kPerLane; ++k) {
      if (k > depth) break;
      int32_t v[kPerLane];
      uint32_t mbits = 0;
#pragma unroll
      for (int t = 0; t < kPerLane; ++t) {
        const bool in = k < R[t], at_end = k == R[t] && has[t];
        v[t] = in ? (cons ? w[t + k] : __ldg(tokens + g[t] + 1 + k)) : (at_end ? nt[t] : fill);
        mbits |= (in || at_end ? 1u : 0u) << (8 * t);
      }
      const int64_t ofs = static_cast<int64_t>(k) * T + p0;
      *reinterpret_cast<int4*>(labels + ofs) = make_int4(v[0], v[1], v[2], v[3]);
      *reinterpret_cast<uint32_t*>(lmask + ofs) = mbits;
    }
  }
}

}  // namespace

thd_status_t launch_roll_labels_zigzag(const int32_t* tokens, const int32_t* cu_v, const int32_t* cu, int32_t n,
                                       int32_t T, int32_t cp, int32_t depth, int32_t fill, const int32_t* next_tok,
                                       const uint8_t* has_next, int32_t* labels, uint8_t* lmask, uint8_t* valid,
                                       int32_t* status, cudaStream_t s) {
  const NextTokens next{next_tok, has_next};
  size_t bytes = static_cast<size_t>(2) * (n + 1) * sizeof(int32_t);
  bool in_smem = bytes <= static_cast<size_t>(kSmemBudget);
  int64_t grid = (static_cast<int64_t>(T) + 4 * kLabelThreads - 1) / (4 * kLabelThreads);  // four rows per thread
  int64_t cap = static_cast<int64_t>(sm_count()) * THD_LABEL_ZZ_BLOCKS_PER_SM;
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  const CpMath m = make_cp_math(cp);
  const dim3 blocks(static_cast<unsigned>(grid));
  const bool nx = has_next != nullptr;
  // slot order with vector stores when the outputs allow them
  const bool vec = T % kPerLane == 0 && reinterpret_cast<uintptr_t>(labels) % 16 == 0 &&
                   reinterpret_cast<uintptr_t>(lmask) % 4 == 0 && reinterpret_cast<uintptr_t>(valid) % 4 == 0;
  if (vec) {
    const FastDiv divS = make_fast_div(T >= cp && cp > 0 ? T / cp : 1);
    const cudaError_t e =
        in_smem ? (nx ? launch_smem(roll_labels_zigzag_slots_kernel<true, true>, blocks, bytes, s, tokens, cu_v, cu, n,
                                    T, m, divS, depth, fill, next, labels, lmask, valid, status)
                      : launch_smem(roll_labels_zigzag_slots_kernel<true, false>, blocks, bytes, s, tokens, cu_v, cu, n,
                                    T, m, divS, depth, fill, next, labels, lmask, valid, status))
                : (nx ? launch_smem(roll_labels_zigzag_slots_kernel<false, true>, blocks, 0, s, tokens, cu_v, cu, n,
                                    T, m, divS, depth, fill, next, labels, lmask, valid, status)
                      : launch_smem(roll_labels_zigzag_slots_kernel<false, false>, blocks, 0, s, tokens, cu_v, cu, n,
                                    T, m, divS, depth, fill, next, labels, lmask, valid, status));
    if (e != cudaSuccess) {
      record_cuda_error(e);
      return THD_ERR_CUDA;
    }
    return THD_OK;
  }
  const cudaError_t e =
      in_smem ? (nx ? launch_smem(roll_labels_zigzag_kernel<true, true>, blocks, bytes, s, tokens, cu_v, cu, n, T, m,
                                  depth, fill, next, labels, lmask, valid, status)
                    : launch_smem(roll_labels_zigzag_kernel<true, false>, blocks, bytes, s, tokens, cu_v, cu, n, T, m,
                                  depth, fill, next, labels, lmask, valid, status))
              : (nx ? launch_smem(roll_labels_zigzag_kernel<false, true>, blocks, 0, s, tokens, cu_v, cu, n, T, m,
                                  depth, fill, next, labels, lmask, valid, status)
                    : launch_smem(roll_labels_zigzag_kernel<false, false>, blocks, 0, s, tokens, cu_v, cu, n, T, m,
                                  depth, fill, next, labels, lmask, valid, status));
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return THD_ERR_CUDA;
  }
  return THD_OK;
}

thd_status_t launch_roll_labels(const int32_t* tokens, const int32_t* cu_v, const int32_t* cu,
                                int32_t n, int32_t T, int32_t depth, int32_t fill, const int32_t* next_tok,
                                const uint8_t* has_next, int32_t* labels, uint8_t* lmask, uint8_t* valid,
                                int32_t* status, cudaStream_t s) {
  const NextTokens next{next_tok, has_next};
  size_t bytes = static_cast<size_t>(2) * (n + 1) * sizeof(int32_t);
  bool in_smem = bytes <= static_cast<size_t>(kSmemBudget);
  const int64_t per_block = static_cast<int64_t>(kLabelThreads) * kPerLane;  // positions
  int64_t grid = (static_cast<int64_t>(T) + per_block - 1) / per_block;
  int64_t cap = static_cast<int64_t>(sm_count()) * 2;
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  const dim3 blocks(static_cast<unsigned>(grid));
  const bool vec = T % kPerLane == 0 && reinterpret_cast<uintptr_t>(labels) % 16 == 0 &&
                   reinterpret_cast<uintptr_t>(lmask) % 4 == 0 && reinterpret_cast<uintptr_t>(valid) % 4 == 0;
  const size_t smem = in_smem ? bytes : 0;
  const cudaError_t e =
      vec ? (in_smem ? launch_smem(roll_labels_kernel<true, true>, blocks, smem, s, tokens, cu_v, cu, n, T, depth,
                                   fill, next, labels, lmask, valid, status)
                     : launch_smem(roll_labels_kernel<false, true>, blocks, smem, s, tokens, cu_v, cu, n, T, depth,
                                   fill, next, labels, lmask, valid, status))
          : (in_smem ? launch_smem(roll_labels_kernel<true, false>, blocks, smem, s, tokens, cu_v, cu, n, T, depth,
                                   fill, next, labels, lmask, valid, status)
                     : launch_smem(roll_labels_kernel<false, false>, blocks, smem, s, tokens, cu_v, cu, n, T, depth,
                                   fill, next, labels, lmask, valid, status));
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return THD_ERR_CUDA;
  }
  return THD_OK;
}

}  // namespace thd
