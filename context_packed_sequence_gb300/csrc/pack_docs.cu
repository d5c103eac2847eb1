// Pack raw [B, S] rows into one padded THD sequence on the device.
//
// "Packed Sequence 与上下文并行", section 2.2 (pack: split rows at EOD, pad
// every document to the alignment, flatten with document i starting at
// cu_seqlens_padded[i]) and the worked example of section 3.  The pages do it
// with bincount/cumsum and a per-document copy loop on the host side of the
// framework.  Two device implementations:
//
//  * chunked (thd_pack_docs): rows are cut into chunks of 2,048 tokens (8,192
//    from 2^22 tokens per batch), one block of 512 threads each, every
//    thread holding 4 (16) consecutive tokens in registers.
//      0. (only when trimming trailing pads) one block per row finds the
//         row's valid end;
//      1. stats: per chunk, its document ends (EODs, and the row's last valid
//         token), its first and last end, and the padded lengths of the
//         documents that both start and end inside it;
//      2. scan: over the statistics of all chunks in order, a max-scan
//         carries each row's last end into the next chunk (which fixes the
//         length of the document open at a chunk boundary) and sum-scans give
//         each chunk's first document index and output offset; a sum over the
//         rows gives each row's unpadded offset; the totals go to `counts`,
//         checked against the capacities.  Up to 512 chunks every emit block
//         does this for itself; beyond that one block does it first and
//         stores every chunk's carries;
//      3. emit: every chunk writes its tokens, padding and boundaries.
//    Scratch: two int64 per row, seven per chunk and two totals.
//  * single pass (thd_pack_docs from 2^19 raw tokens, aligned rows and
//    output): one persistent kernel reads every token once; blocks take
//    6,144-token chunks in order, publish each chunk's summary, and write it
//    once a scanner block has turned the summaries before it into the
//    chunk's carries (below);
//  * per row (thd_pack_docs_noalloc, whose scratch is a fixed array of four
//    int64 per row): the same phases with one block per raw row; above 512
//    rows one block turns the rows' statistics into prefixes in place
//    between them.
#include "thd_debug.h"
#include "thd_internal.cuh"

namespace thd {
namespace {

constexpr int kPackThreads = 1024;
constexpr int kItems = 8;  // consecutive tokens per thread per tile
constexpr int64_t kTile = static_cast<int64_t>(kPackThreads) * kItems;

// (-L) mod align for L >= 0: a mask when align is a power of two (the usual
// 2 * cp), a 32-bit remainder for lengths below 2^32
__device__ __forceinline__ int64_t pad_of(int64_t L, int32_t align) {
  if ((align & (align - 1)) == 0) return (-L) & (align - 1);
  const int64_t r = (L >> 32) == 0 ? static_cast<int64_t>(static_cast<uint32_t>(L) % static_cast<uint32_t>(align))
                                   : L % align;
  return r == 0 ? 0 : align - r;
}

__device__ __forceinline__ bool is_end(const int32_t* row, int64_t t, int64_t ve, int32_t eod) {
  return row[t] == eod || t == ve - 1;
}

__device__ __forceinline__ int64_t block_sum(int64_t v, int64_t* tmp) {
  int64_t total;
  block_exclusive_scan(v, OpSum(), static_cast<int64_t>(0), tmp, &total);
  return total;
}

__device__ int64_t row_valid_end(const int32_t* row, int64_t S, int32_t trim, int32_t raw_pad,
                                 int64_t* tmp) {
  if (!trim) return S;
  int64_t m = 0;
  for (int64_t t = threadIdx.x; t < S; t += blockDim.x)
    if (row[t] != raw_pad) m = t + 1;
  int64_t total;
  block_exclusive_scan(m, OpMax(), static_cast<int64_t>(0), tmp, &total);
  return total;
}

__global__ void __launch_bounds__(kPackThreads)
pack_stats_kernel(const int32_t* raw, int64_t S, int32_t eod, int32_t trim, int32_t raw_pad,
                  int32_t align, int64_t* ws, int32_t* status) {
  __shared__ int64_t tmp[32];
  pdl_wait_then_release();
  if (block_status_set(status)) return;
  const int64_t b = blockIdx.x;
  const int32_t* row = raw + b * S;
  const int64_t ve = row_valid_end(row, S, trim, raw_pad, tmp);
  int64_t carry_end = -1, docs = 0, padded = 0;
  for (int64_t base = 0; base < ve; base += kTile) {
    const int64_t t0 = base + static_cast<int64_t>(threadIdx.x) * kItems;
    int64_t my_last = -1;
    for (int it = 0; it < kItems; ++it) {
      int64_t t = t0 + it;
      if (t < ve && is_end(row, t, ve, eod)) my_last = t;
    }
    int64_t tile_last;
    int64_t prev = block_exclusive_scan(my_last, OpMax(), static_cast<int64_t>(-1), tmp, &tile_last);
    prev = max(prev, carry_end);
    int64_t cnt = 0, psum = 0;
    for (int it = 0; it < kItems; ++it) {
      int64_t t = t0 + it;
      if (t < ve && is_end(row, t, ve, eod)) {
        int64_t L = t - prev;
        psum += L + pad_of(L, align);
        ++cnt;
        prev = t;
      }
    }
    docs += block_sum(cnt, tmp);
    padded += block_sum(psum, tmp);
    carry_end = max(carry_end, tile_last);
  }
  if (threadIdx.x == 0) {
    ws[b * 4 + 0] = ve;
    ws[b * 4 + 1] = docs;
    ws[b * 4 + 2] = padded;
    ws[b * 4 + 3] = 0;
  }
}

// Up to this many rows every emit block sums the statistics of the rows
// before it itself (two launches); beyond it one block scans them first
// (three launches), since the self-sums cost every block a pass over all rows.
#ifndef THD_PACK_SELF_SCAN_ROWS
#define THD_PACK_SELF_SCAN_ROWS 512
#endif
constexpr int32_t kSelfScanRows = THD_PACK_SELF_SCAN_ROWS;

// One block over all rows (more than kSelfScanRows): each row's exclusive
// prefixes replace its statistics in place, ws[r] = {valid end, documents
// before, padded tokens before, valid tokens before}; the totals go to
// `counts` (and THD_ERR_CAPACITY to the status word when they do not fit).
__global__ void __launch_bounds__(kPackThreads)
pack_rows_scan_kernel(int32_t B, int64_t tok_cap, int64_t docs_cap, int32_t* cu_v, int32_t* cu, int64_t* counts,
                      int64_t* ws, int32_t* status) {
  __shared__ int64_t tmp[32];
  pdl_wait_then_release();
  if (block_status_set(status)) return;
  int64_t d_carry = 0, t_carry = 0, v_carry = 0;
  for (int64_t base = 0; base < B; base += blockDim.x) {
    const int64_t r = base + threadIdx.x;
    int64_t ve = 0, nd = 0, np = 0;
    if (r < B) {
      ve = ws[r * 4 + 0];
      nd = ws[r * 4 + 1];
      np = ws[r * 4 + 2];
    }
    int64_t pass_d, pass_t, pass_v;
    const int64_t d_before = block_exclusive_scan(nd, OpSum(), static_cast<int64_t>(0), tmp, &pass_d);
    const int64_t t_before = block_exclusive_scan(np, OpSum(), static_cast<int64_t>(0), tmp, &pass_t);
    const int64_t v_before = block_exclusive_scan(ve, OpSum(), static_cast<int64_t>(0), tmp, &pass_v);
    if (r < B) {
      ws[r * 4 + 1] = d_carry + d_before;
      ws[r * 4 + 2] = t_carry + t_before;
      ws[r * 4 + 3] = v_carry + v_before;
    }
    d_carry += pass_d;
    t_carry += pass_t;
    v_carry += pass_v;
  }
  if (threadIdx.x == 0) {
    counts[0] = d_carry;
    counts[1] = t_carry;
    if (d_carry + 1 > docs_cap || t_carry > tok_cap || t_carry > INT32_MAX) {
      status_set(status, THD_ERR_CAPACITY);
    } else {
      cu[0] = 0;
      cu_v[0] = 0;
    }
  }
}

// prefixed: pack_rows_scan_kernel has run (ws holds each row's prefixes and
// counts the totals); else the block sums the rows before its own.
__global__ void __launch_bounds__(kPackThreads)
pack_emit_kernel(const int32_t* raw, int32_t B, int64_t S, int32_t eod, int32_t align, int32_t pad_id,
                 int32_t* tokens, int64_t tok_cap, int32_t* cu_v, int32_t* cu, int64_t docs_cap,
                 int64_t* counts, const int64_t* ws, bool prefixed, int32_t* status) {
  __shared__ int64_t tmp[32];
  pdl_wait_then_release();
  // (with the separate scan, that kernel has set the status word when the
  // capacities are too small)
  if (block_status_set(status)) return;
  const int64_t b = blockIdx.x;
  // where this row starts: sums over the rows before it, and the grand totals
  int64_t d_before = 0, t_before = 0, v_before = 0, d_all = 0, t_all = 0;
  if (prefixed) {
    d_before = ws[b * 4 + 1];
    t_before = ws[b * 4 + 2];
    v_before = ws[b * 4 + 3];
    d_all = counts[0];
    t_all = counts[1];
  } else {
    for (int64_t r = threadIdx.x; r < B; r += blockDim.x) {
      int64_t ve = ws[r * 4 + 0], nd = ws[r * 4 + 1], np = ws[r * 4 + 2];
      if (r < b) {
        d_before += nd;
        t_before += np;
        v_before += ve;
      }
      d_all += nd;
      t_all += np;
    }
    d_before = block_sum(d_before, tmp);
    t_before = block_sum(t_before, tmp);
    v_before = block_sum(v_before, tmp);
    d_all = block_sum(d_all, tmp);
    t_all = block_sum(t_all, tmp);
    const bool over = d_all + 1 > docs_cap || t_all > tok_cap || t_all > INT32_MAX;
    if (b == 0 && threadIdx.x == 0) {
      counts[0] = d_all;
      counts[1] = t_all;
      if (over) {
        status_set(status, THD_ERR_CAPACITY);
      } else {
        cu[0] = 0;
        cu_v[0] = 0;
      }
    }
    if (over) return;
  }

  const int32_t* row = raw + b * S;
  const int64_t ve = ws[b * 4 + 0];
  int64_t carry_end = -1, row_docs = 0, row_pad = 0;
  for (int64_t base = 0; base < ve; base += kTile) {
    const int64_t t0 = base + static_cast<int64_t>(threadIdx.x) * kItems;
    int64_t my_last = -1;
    for (int it = 0; it < kItems; ++it) {
      int64_t t = t0 + it;
      if (t < ve && is_end(row, t, ve, eod)) my_last = t;
    }
    int64_t tile_last;
    int64_t first_prev = block_exclusive_scan(my_last, OpMax(), static_cast<int64_t>(-1), tmp, &tile_last);
    first_prev = max(first_prev, carry_end);
    int64_t cnt = 0, psum = 0;
    {
      int64_t prev = first_prev;
      for (int it = 0; it < kItems; ++it) {
        int64_t t = t0 + it;
        if (t < ve && is_end(row, t, ve, eod)) {
          int64_t L = t - prev;
          psum += L + pad_of(L, align);
          ++cnt;
          prev = t;
        }
      }
    }
    int64_t tile_cnt, tile_psum;
    int64_t cnt_before = block_exclusive_scan(cnt, OpSum(), static_cast<int64_t>(0), tmp, &tile_cnt);
    int64_t psum_before = block_exclusive_scan(psum, OpSum(), static_cast<int64_t>(0), tmp, &tile_psum);
    {
      int64_t prev = first_prev;
      int64_t doc = d_before + row_docs + cnt_before;     // document the next token belongs to
      int64_t out = t_before + row_pad + psum_before;     // that document's first output row
      for (int it = 0; it < kItems; ++it) {
        int64_t t = t0 + it;
        if (t >= ve) break;
        int32_t v = row[t];
        if (in_range(out + (t - prev - 1), 0, t_all, status)) tokens[out + (t - prev - 1)] = v;
        if (v == eod || t == ve - 1) {
          int64_t L = t - prev;
          int64_t P = L + pad_of(L, align);
          for (int64_t z = L; z < P; ++z)
            if (in_range(out + z, 0, t_all, status)) tokens[out + z] = pad_id;
          if (in_range(doc + 1, 1, d_all + 1, status)) {
            cu_v[doc + 1] = static_cast<int32_t>(v_before + t + 1);
            cu[doc + 1] = static_cast<int32_t>(out + P);
          }
          ++doc;
          out += P;
          prev = t;
        }
      }
    }
    row_docs += tile_cnt;
    row_pad += tile_psum;
    carry_end = max(carry_end, tile_last);
  }
}


// ---------------------------------------------------------------------------
// chunked packing
// ---------------------------------------------------------------------------
//
// A chunk is kChunkThreads * K consecutive tokens of one row.  Thread t holds
// tokens [lo + K*t, lo + K*t + K) in registers, loaded once per kernel with
// 16-byte loads when the rows allow them (16-byte aligned rows of a multiple
// of 4 tokens).  K = 16 (8,192-token chunks) once a batch has 2^22 tokens,
// K = 4 (2,048-token chunks) below that, so small batches still spread over
// the SMs.  Per kernel a block runs one max-scan (the last document end
// before each thread) and one sum-scan (documents and padded tokens, packed
// into one 64-bit word).

constexpr int kChunkThreads = 512;
constexpr int64_t kSmallChunk = static_cast<int64_t>(kChunkThreads) * 4;
constexpr int64_t kBigChunkFrom = int64_t(1) << 22;  // tokens per batch
// The single pass from this many raw tokens per batch: measured on GB300
// against the chunked kernels, 1.3x faster at 2^20 and 1.5x at 2^21, 1.3x
// slower at 2^18 (where both are bound by launch latency)
constexpr int64_t kOnePassFrom = int64_t(1) << 19;

// documents and padded tokens of a thread or chunk in one word: the count
// fits 14 bits (at most 8,192 ends per chunk), the padded tokens the rest
constexpr int kCntBits = 14;

struct OpMin {
  template <typename V>
  __device__ __forceinline__ V operator()(V a, V b) const { return a < b ? a : b; }
};

struct ChunkGeom {
  int32_t B;
  int64_t S;
  int64_t chunk;    // tokens per chunk
  int64_t per_row;  // chunks per row
  int64_t nc;       // B * per_row
};

__global__ void __launch_bounds__(kPackThreads)
pack_row_ends_kernel(const int32_t* raw, int64_t S, int32_t raw_pad, int64_t* ve, int32_t* status) {
  __shared__ int64_t tmp[32];
  pdl_wait_then_release();
  if (block_status_set(status)) return;
  const int64_t b = blockIdx.x;
  const int64_t v = row_valid_end(raw + b * S, S, 1, raw_pad, tmp);
  if (threadIdx.x == 0) ve[b] = v;
}

// This thread's K tokens [t0, t0 + K) of `row`; tokens at or past S read 0
// (they are never used: every use is also bounded by the valid end).
template <int K, bool VEC>
__device__ __forceinline__ void load_tokens(const int32_t* row, int64_t t0, int64_t S, int32_t (&v)[K]) {
  if (VEC) {  // t0 and S multiples of 4: a group of four lies wholly below S or at or past it
#pragma unroll
    for (int q = 0; q < K / 4; ++q) {
      const int64_t t = t0 + 4 * q;
      int4 x = make_int4(0, 0, 0, 0);
      if (t < S) x = __ldg(reinterpret_cast<const int4*>(row + t));
      v[4 * q] = x.x, v[4 * q + 1] = x.y, v[4 * q + 2] = x.z, v[4 * q + 3] = x.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < K; ++i) v[i] = t0 + i < S ? __ldg(row + t0 + i) : 0;
  }
}

// The document ends among a thread's tokens: every EOD, and the row's last
// valid token.  psum = padded lengths of the documents that both start
// after this thread's first end and end at one of its later ends.
struct ThreadEnds {
  uint32_t mask;      // bit i: token t0 + i ends a document
  int32_t cnt;
  int64_t first;      // first end (INT64_MAX: none)
  int64_t last;       // last end (-1: none)
  int64_t psum;
};

template <int K>
__device__ __forceinline__ ThreadEnds thread_ends(const int32_t (&v)[K], int64_t t0, int64_t hi, int64_t ve,
                                                  int32_t eod, int32_t align) {
  ThreadEnds te;
  te.mask = 0;
#pragma unroll
  for (int i = 0; i < K; ++i)
    if (t0 + i < hi && (v[i] == eod || t0 + i == ve - 1)) te.mask |= 1u << i;
  te.cnt = __popc(te.mask);
  te.first = te.cnt ? t0 + __ffs(te.mask) - 1 : INT64_MAX;
  te.last = te.cnt ? t0 + 31 - __clz(te.mask) : -1;
  te.psum = 0;
  int64_t prev = -1;
  for (uint32_t m = te.mask; m; m &= m - 1) {
    const int64_t e = t0 + __ffs(m) - 1;
    if (prev >= 0) te.psum += (e - prev) + pad_of(e - prev, align);
    prev = e;
  }
  return te;
}

// Sum and minimum over the block, every thread gets both (tmp: 64 words).
__device__ __forceinline__ void block_sum_min(int64_t& sum, int64_t& mn, int64_t* tmp) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    sum += __shfl_xor_sync(kFullMask, sum, o);
    mn = min(mn, __shfl_xor_sync(kFullMask, mn, o));
  }
  if (lane == 0) tmp[wid] = sum, tmp[32 + wid] = mn;
  __syncthreads();
  if (wid == 0) {
    int64_t s2 = lane < nw ? tmp[lane] : 0, m2 = lane < nw ? tmp[32 + lane] : INT64_MAX;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      s2 += __shfl_xor_sync(kFullMask, s2, o);
      m2 = min(m2, __shfl_xor_sync(kFullMask, m2, o));
    }
    if (lane == 0) tmp[0] = s2, tmp[32] = m2;
  }
  __syncthreads();
  sum = tmp[0];
  mn = tmp[32];
}

// stats[z] = {ends, first end (-1: none), last end (-1: none), padded length of
// the documents after the first end}, z = b * per_row + c
template <int K, bool VEC>
__global__ void __launch_bounds__(kChunkThreads)
pack_chunk_stats_kernel(const int32_t* raw, ChunkGeom g, int32_t eod, const int64_t* ve_arr, int32_t align,
                        int64_t* stats, int32_t* status) {
  __shared__ int64_t tmp[64];
  pdl_wait_then_release();
  if (block_status_set(status)) return;
  const int64_t b = blockIdx.y, c = blockIdx.x;
  const int32_t* row = raw + b * g.S;
  const int64_t ve = ve_arr ? ve_arr[b] : g.S;
  const int64_t lo = c * g.chunk, hi = min(lo + g.chunk, ve);
  const int64_t t0 = lo + static_cast<int64_t>(threadIdx.x) * K;
  int32_t v[K];
  load_tokens<K, VEC>(row, t0, g.S, v);
  ThreadEnds te = thread_ends<K>(v, t0, hi, ve, eod, align);
  int64_t chunk_last;
  const int64_t prev = block_exclusive_scan(te.last, OpMax(), static_cast<int64_t>(-1), tmp, &chunk_last);
  if (te.cnt > 0 && prev >= 0) te.psum += (te.first - prev) + pad_of(te.first - prev, align);
  int64_t packed = (te.psum << kCntBits) | te.cnt, first = te.first;
  block_sum_min(packed, first, tmp);
  if (threadIdx.x == 0) {
    const int64_t cnt = packed & ((int64_t(1) << kCntBits) - 1);
    int64_t* st = stats + (b * g.per_row + c) * 4;
    st[0] = cnt;
    st[1] = cnt > 0 ? first : -1;
    st[2] = chunk_last;
    st[3] = packed >> kCntBits;
  }
}

// Every chunk's carries in order, by walking the statistics: a max-scan
// carries each row's last end into the next chunk, sum-scans give every
// chunk's first document index and output offset.  Chunk z's three carries
// go to carry_out[z * 3 ...] when carry_out is set, else only chunk `mine`'s
// to mine_out[0..2]; totals_out gets {documents, padded tokens}.  (The emit
// kernel's own scan when there are few chunks.)
__device__ void scan_chunks(const ChunkGeom& g, int32_t align, const int64_t* stats, int64_t* carry_out,
                            int64_t mine, int64_t* mine_out, int64_t* totals_out, int64_t* tmp) {
  const int64_t key_span = g.S + 2;  // key = row * key_span + (last end + 1)
  int64_t key_carry = -1, docs_carry = 0, pad_carry = 0;
  for (int64_t base = 0; base < g.nc; base += blockDim.x) {
    const int64_t z = base + threadIdx.x;
    int64_t n_end = 0, first = -1, last = -1, tail = 0, key = -1;
    if (z < g.nc) {
      const int64_t* st = stats + z * 4;
      n_end = st[0];
      first = st[1];
      last = st[2];
      tail = st[3];
      key = (z / g.per_row) * key_span + (last + 1);
    }
    int64_t pass_key;
    int64_t pk = block_exclusive_scan(key, OpMax(), static_cast<int64_t>(-1), tmp, &pass_key);
    pk = max(pk, key_carry);
    const int64_t zrow = z / g.per_row;
    const int64_t prev_end = (pk >= 0 && pk / key_span == zrow) ? pk % key_span - 1 : -1;
    int64_t pad_len = tail;
    if (n_end > 0) pad_len += (first - prev_end) + pad_of(first - prev_end, align);
    int64_t pass_docs, pass_pad;
    const int64_t docs_before = block_exclusive_scan(n_end, OpSum(), static_cast<int64_t>(0), tmp, &pass_docs);
    const int64_t pad_before = block_exclusive_scan(pad_len, OpSum(), static_cast<int64_t>(0), tmp, &pass_pad);
    int64_t* out = carry_out ? (z < g.nc ? carry_out + z * 3 : nullptr) : (z == mine ? mine_out : nullptr);
    if (out) {
      out[0] = prev_end;
      out[1] = docs_carry + docs_before;
      out[2] = pad_carry + pad_before;
    }
    key_carry = max(key_carry, pass_key);
    docs_carry += pass_docs;
    pad_carry += pass_pad;
  }
  if (threadIdx.x == 0) {
    totals_out[0] = docs_carry;
    totals_out[1] = pad_carry;
  }
}

// Sizes, counts and the first boundaries once the totals are known: counts
// always, then THD_ERR_CAPACITY when the outputs are too small (nothing is
// emitted), else cu[0] = cu_v[0] = 0.  One thread.
__device__ void publish_totals(int64_t d_all, int64_t t_all, int64_t tok_cap, int64_t docs_cap, int32_t* cu_v,
                               int32_t* cu, int64_t* counts, int32_t* status) {
  counts[0] = d_all;
  counts[1] = t_all;
  if (d_all + 1 > docs_cap || t_all > tok_cap || t_all > INT32_MAX) {
    status_set(status, THD_ERR_CAPACITY);
  } else {
    cu[0] = 0;
    cu_v[0] = 0;
  }
}

// Up to this many chunks every emit block scans the statistics itself (two
// launches); beyond it one block scans them first (three launches), since
// the self-scan costs every block a pass over all chunks.
constexpr int64_t kSelfScanChunks = 512;

// One block over all chunks (more than kSelfScanChunks).  Each thread takes a
// contiguous run of chunks: the largest end key of its run goes through one
// block max-scan, the run is walked to count its documents and padded
// tokens, one sum-scan of those gives each run's offsets, and a second walk
// writes every chunk's carries.  Also every row's unpadded offset (vbefore,
// when the rows are trimmed) and the totals.
constexpr int kScanThreads = 1024;

__global__ void __launch_bounds__(kScanThreads)
pack_chunk_scan_kernel(ChunkGeom g, const int64_t* ve_arr, int32_t align, const int64_t* stats, int64_t* carry,
                       int64_t* vbefore, int64_t* totals, int64_t tok_cap, int64_t docs_cap, int32_t* cu_v,
                       int32_t* cu, int64_t* counts, int32_t* status) {
  __shared__ int64_t tmp[32];
  pdl_wait_then_release();
  if (block_status_set(status)) return;
  const int64_t key_span = g.S + 2;  // key = row * key_span + (last end + 1)
  const int64_t per_thread = (g.nc + blockDim.x - 1) / blockDim.x;
  const int64_t z_lo = min(g.nc, static_cast<int64_t>(threadIdx.x) * per_thread);
  const int64_t z_hi = min(g.nc, z_lo + per_thread);
  int64_t run_key = -1;
  for (int64_t z = z_lo; z < z_hi; ++z) run_key = max(run_key, (z / g.per_row) * key_span + (stats[z * 4 + 2] + 1));
  int64_t unused;
  const int64_t key_in = block_exclusive_scan(run_key, OpMax(), static_cast<int64_t>(-1), tmp, &unused);
  // walk the run: each chunk's previous end in its row, documents and padded tokens
  auto walk = [&](bool write, int64_t docs0, int64_t pad0, int64_t* docs, int64_t* pad) {
    int64_t key = key_in, d = docs0, p = pad0;
    for (int64_t z = z_lo; z < z_hi; ++z) {
      const int64_t* st = stats + z * 4;
      const int64_t n_end = st[0], first = st[1], last = st[2], tail = st[3];
      const int64_t zrow = z / g.per_row;
      const int64_t prev_end = (key >= 0 && key / key_span == zrow) ? key % key_span - 1 : -1;
      if (write) {
        carry[z * 3 + 0] = prev_end;
        carry[z * 3 + 1] = d;
        carry[z * 3 + 2] = p;
      }
      d += n_end;
      p += tail + (n_end > 0 ? (first - prev_end) + pad_of(first - prev_end, align) : 0);
      key = max(key, zrow * key_span + (last + 1));
    }
    *docs = d;
    *pad = p;
  };
  int64_t run_docs, run_pad;
  walk(false, 0, 0, &run_docs, &run_pad);
  int64_t all_docs, all_pad;
  const int64_t docs_in = block_exclusive_scan(run_docs, OpSum(), static_cast<int64_t>(0), tmp, &all_docs);
  const int64_t pad_in = block_exclusive_scan(run_pad, OpSum(), static_cast<int64_t>(0), tmp, &all_pad);
  walk(true, docs_in, pad_in, &run_docs, &run_pad);
  if (ve_arr) {
    int64_t v_carry = 0;
    for (int64_t base = 0; base < g.B; base += blockDim.x) {
      const int64_t r = base + threadIdx.x;
      const int64_t v = r < g.B ? ve_arr[r] : 0;
      int64_t pass_v;
      const int64_t v_before = block_exclusive_scan(v, OpSum(), static_cast<int64_t>(0), tmp, &pass_v);
      if (r < g.B) vbefore[r] = v_carry + v_before;
      v_carry += pass_v;
    }
  }
  if (threadIdx.x == 0) {
    totals[0] = all_docs;
    totals[1] = all_pad;
    publish_totals(all_docs, all_pad, tok_cap, docs_cap, cu_v, cu, counts, status);
  }
}

// The emit kernel's shared-memory staging of a chunk's output: the chunk's
// tokens and padding fill one contiguous range of the packed sequence, which
// is assembled here and written out with coalesced stores (threads' own
// tokens land 4*K bytes apart otherwise; on 8,192-token chunks that took the
// L1 store sectors to 8x the bytes and the emit to 80 us for 16.8 M tokens,
// 66 us staged).  A chunk whose range is longer (many short documents, each
// padded) writes its rows directly.
constexpr int kStageWords = 11264;  // 44 KB

template <int K, bool VEC>
__global__ void __launch_bounds__(kChunkThreads)
pack_chunk_emit_kernel(const int32_t* raw, ChunkGeom g, int32_t eod, const int64_t* ve_arr, int32_t align,
                       int32_t pad_id, const int64_t* stats, const int64_t* carry, const int64_t* vbefore,
                       const int64_t* totals, const int32_t* row_next, int32_t* tokens, int64_t tok_cap,
                       int32_t* cu_v, int32_t* cu, int32_t* next_tok, uint8_t* has_next, int64_t docs_cap,
                       int64_t* counts, int32_t* status) {
  __shared__ int64_t tmp[32];
  __shared__ int64_t mine[3], tot[2];
  __shared__ int32_t stage[kStageWords];
  pdl_wait_then_release();
  // (with a separate scan, that kernel has set the status word when the
  // capacities are too small)
  if (block_status_set(status)) return;
  const int64_t b = blockIdx.y, c = blockIdx.x, me = b * g.per_row + c;
  int64_t d_all, t_all, v_before, carry_end, carry_doc, carry_out;
  if (carry) {
    d_all = totals[0];
    t_all = totals[1];
    v_before = ve_arr ? vbefore[b] : b * g.S;
    carry_end = carry[me * 3 + 0];
    carry_doc = carry[me * 3 + 1];
    carry_out = carry[me * 3 + 2];
  } else {
    // few chunks: scan them all here, and the rows before this one
    int64_t vb = 0;
    if (ve_arr) {
      for (int64_t r = threadIdx.x; r < b; r += blockDim.x) vb += ve_arr[r];
      vb = block_sum(vb, tmp);
    } else {
      vb = b * g.S;
    }
    v_before = vb;
    scan_chunks(g, align, stats, nullptr, me, mine, tot, tmp);
    __syncthreads();
    d_all = tot[0];
    t_all = tot[1];
    carry_end = mine[0];
    carry_doc = mine[1];
    carry_out = mine[2];
    if (me == 0 && threadIdx.x == 0) publish_totals(d_all, t_all, tok_cap, docs_cap, cu_v, cu, counts, status);
  }
  if (d_all + 1 > docs_cap || t_all > tok_cap || t_all > INT32_MAX) return;  // reported once, above

  const int32_t* row = raw + b * g.S;
  const int64_t ve = ve_arr ? ve_arr[b] : g.S;
  const int64_t lo = c * g.chunk, hi = min(lo + g.chunk, ve);
  const int64_t t0 = lo + static_cast<int64_t>(threadIdx.x) * K;
  int32_t v[K];
  load_tokens<K, VEC>(row, t0, g.S, v);
  const ThreadEnds te = thread_ends<K>(v, t0, hi, ve, eod, align);
  int64_t chunk_last, total;
  const int64_t prev_last = block_exclusive_scan(te.last, OpMax(), static_cast<int64_t>(-1), tmp, &chunk_last);
  int64_t pe = max(prev_last, carry_end);  // the end before this thread's first token
  const int64_t psum = te.psum + (te.cnt > 0 ? (te.first - pe) + pad_of(te.first - pe, align) : 0);
  const int64_t before =
      block_exclusive_scan((psum << kCntBits) | te.cnt, OpSum(), static_cast<int64_t>(0), tmp, &total);
  int64_t doc = carry_doc + (before & ((int64_t(1) << kCntBits) - 1));  // document the next token belongs to
  int64_t out = carry_out + (before >> kCntBits);                       // that document's first output row
  // the chunk's output rows [o_lo, o_hi): from its first token (of the
  // document open since carry_end) to its last token, or to the padding
  // after its last end when that token ends a document
  const int64_t o_lo = carry_out + (lo - carry_end - 1);
  const int64_t o_hi = chunk_last >= 0 ? carry_out + (total >> kCntBits) + (hi - 1 - chunk_last) : o_lo + (hi - lo);
  // (the large chunks only: at 2,048 tokens the staging measured slower than
  // direct stores on GB300, 10.5 against 9.0 us for 8 x 32,768 tokens)
  const bool staged = K == 16 && lo < hi && o_hi - o_lo <= kStageWords;  // block-uniform
  auto put = [&](int64_t pos, int32_t val) {
    if (!in_range(pos, 0, t_all, status)) return;
    if (staged) {
      if (in_range(pos - o_lo, 0, kStageWords, status)) stage[pos - o_lo] = val;
    } else {
      tokens[pos] = val;
    }
  };
#pragma unroll
  for (int i = 0; i < K; ++i) {
    const int64_t t = t0 + i;
    if (t >= hi) break;
    put(out + (t - pe - 1), v[i]);
    if ((te.mask >> i) & 1u) {
      const int64_t L = t - pe;
      const int64_t P = L + pad_of(L, align);
      for (int64_t zz = L; zz < P; ++zz) put(out + zz, pad_id);
      if (!in_range(doc + 1, 1, d_all + 1, status)) break;
      cu_v[doc + 1] = static_cast<int32_t>(v_before + t + 1);
      cu[doc + 1] = static_cast<int32_t>(out + P);
      if (has_next) {
        // the row's extra token continues its last document when that
        // document reaches the row's end without an EOD
        const bool cont = row_next != nullptr && v[i] != eod && ve == g.S;
        has_next[doc] = cont ? 1 : 0;
        next_tok[doc] = cont ? row_next[b] : 0;
      }
      ++doc;
      out += P;
      pe = t;
    }
  }
  if (staged) {
    __syncthreads();
    const int32_t len = static_cast<int32_t>(o_hi - o_lo);
    if (in_range(o_lo, 0, t_all, status) && in_range(o_hi, 0, t_all + 1, status))
      for (int32_t idx = threadIdx.x; idx < len; idx += blockDim.x) tokens[o_lo + idx] = stage[idx];
  }
}

// ---------------------------------------------------------------------------
// single pass (large batches of aligned rows)
// ---------------------------------------------------------------------------
//
// From 2^19 raw tokens per batch, with 16-byte aligned rows of a multiple of
// 4 tokens, a 16-byte aligned output and an alignment of at most 65,536, one
// persistent kernel packs every 6,144-token chunk reading its tokens once
// (the three kernels above read them twice and wait for each other between
// launches).  The first block to start becomes the scanner; every other
// block takes chunks in row-major order from a counter and, per chunk,
//   1. receives its tokens by one bulk copy into shared memory, requested an
//      iteration before they are needed;
//   2. summarises the chunk's document ends (a RunSummary, from one max-scan
//      and one sum-scan over its threads) and publishes the summary;
//   3. writes the chunk once the scanner has published the chunk's carries
//      (the document open at its start, the number of documents and of
//      output tokens before it): every document end writes its boundaries
//      and padding, then the block copies its tokens to their places with
//      consecutive threads on consecutive tokens.
// The scanner's warps take 32 chunks at a time: as the summaries of a
// window's first chunks arrive they scan them, combine them with the prefix
// of all earlier chunks (handed over from the warp of the previous window
// through shared memory) and publish the carries of the chunks after them;
// the one that sees the last chunk writes the totals.  A chunk's carries
// thus wait only for the summaries of the chunks before it, and a block
// holds at most one chunk without a published summary, whose number is
// larger than that of any chunk it waits for: the waits form no cycle.  A
// one-block kernel before it clears the counters and the records and, when
// rows are trimmed, sums the rows' valid lengths into per-row offsets.
// Every wait is bounded: a wait that runs out records THD_ERR_TIMEOUT and
// publishes a "poisoned" record, and nothing that depends on a poisoned
// record is written.  With too small outputs a block writes nothing past
// either capacity; the scanner reports THD_ERR_CAPACITY.

// The document ends of a run of consecutive chunks (row-major): n ends, the
// first and the last as keys (row << shift | position in the row), psum =
// the padded lengths of the documents that start after its first end and end
// at one of its later ends.  n = 0: no end (identity); n < 0: poisoned.
struct RunSummary {
  int64_t n, psum, first, last;
};

struct KeyGeom {
  int32_t shift;  // positions in a row take `shift` bits
  int64_t mask;
  int32_t align;
};

__device__ __forceinline__ RunSummary run_identity() { return RunSummary{0, 0, 0, 0}; }
__device__ __forceinline__ RunSummary run_poison() { return RunSummary{-1, 0, 0, 0}; }

// a, then b.  The document that ends at b's first end starts after a's last
// end when the two lie in one row, else at the start of b's row (every
// non-empty row ends with a document end, so no document spans rows).
__device__ __forceinline__ RunSummary run_combine(const RunSummary& a, const RunSummary& b, const KeyGeom& k) {
  if (a.n < 0 || b.n < 0) return run_poison();
  if (a.n == 0) return b;
  if (b.n == 0) return a;
  const bool same_row = (a.last >> k.shift) == (b.first >> k.shift);
  const int64_t L = (b.first & k.mask) - (same_row ? (a.last & k.mask) : -1);
  return RunSummary{a.n + b.n, a.psum + b.psum + L + pad_of(L, k.align), a.first, b.last};
}

__device__ __forceinline__ RunSummary run_shfl_up(const RunSummary& s, int o) {
  return RunSummary{__shfl_up_sync(kFullMask, s.n, o), __shfl_up_sync(kFullMask, s.psum, o),
                    __shfl_up_sync(kFullMask, s.first, o), __shfl_up_sync(kFullMask, s.last, o)};
}

// Records between blocks: two 16-byte words, each written and read with one
// 16-byte access and carrying the record's state in the top two bits of one
// of its 64-bit halves, so a reader that sees the state set in both words has
// the whole record (no fence between a flag and its payload).  The words are
// zeroed before the kernel (state 0: not yet written).
constexpr uint64_t kStateShift = 62;
constexpr uint64_t kLow62 = (uint64_t(1) << kStateShift) - 1;
constexpr uint64_t kReady = 1, kPoisoned = 2;

__device__ __forceinline__ void rec_store(int64_t* rec, uint64_t state, uint64_t x0, uint64_t y0, uint64_t x1,
                                          uint64_t y1) {
  asm volatile("st.relaxed.gpu.global.v2.u64 [%0], {%1, %2};" ::"l"(rec), "l"(x0 | (state << kStateShift)), "l"(y0)
               : "memory");
  asm volatile("st.relaxed.gpu.global.v2.u64 [%0], {%1, %2};" ::"l"(rec + 2), "l"(x1), "l"(y1 | (state << kStateShift))
               : "memory");
}

// Poll a record until both words carry a state (bounded); 0 when the wait
// gave up.  x0 and y1 come back without their state bits.
__device__ __forceinline__ uint64_t rec_wait(const int64_t* rec, uint64_t* x0, uint64_t* y0, uint64_t* x1,
                                             uint64_t* y1) {
  for (int it = 0; it < kWaitLimit; ++it) {
    uint64_t a0, b0, a1, b1;
    asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(a0), "=l"(b0) : "l"(rec) : "memory");
    asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(a1), "=l"(b1) : "l"(rec + 2) : "memory");
    const uint64_t s0 = a0 >> kStateShift, s1 = b1 >> kStateShift;
    if (s0 != 0 && s0 == s1) {
      *x0 = a0 & kLow62, *y0 = b0, *x1 = a1, *y1 = b1 & kLow62;
      return s0;
    }
  }
  return 0;
}

// a chunk's summary: {n | state, psum}, {first, last | state}
__device__ __forceinline__ void summary_publish(int64_t* rec, const RunSummary& s) {
  if (s.n < 0) rec_store(rec, kPoisoned, 0, 0, 0, 0);
  else rec_store(rec, kReady, s.n, s.psum, s.first, s.last);
}

// a chunk's carries: the documents and the output tokens before it, and the
// end before it in its row (-1: none): {docs | state, out}, {end + 1, 0 | state}
struct Carry {
  int64_t doc, out, end;
  bool ok;
};

__device__ __forceinline__ void carry_publish(int64_t* rec, const Carry& c) {
  if (!c.ok) rec_store(rec, kPoisoned, 0, 0, 0, 0);
  else rec_store(rec, kReady, c.doc, c.out, c.end + 1, 0);
}

__device__ __forceinline__ Carry carry_wait(const int64_t* rec) {
  uint64_t doc, out, end1, zero;
  const uint64_t st = rec_wait(rec, &doc, &out, &end1, &zero);
  if (st != kReady) return Carry{0, 0, -1, false};
  return Carry{static_cast<int64_t>(doc), static_cast<int64_t>(out), static_cast<int64_t>(end1) - 1, true};
}

constexpr int kOneThreads = 384;
constexpr int kOneBlocksPerSm = 2;
constexpr int kOneK = 16;
constexpr int64_t kOneChunk = static_cast<int64_t>(kOneThreads) * kOneK;
// A block's ring of chunks: kBufs buffers, a chunk written kLag iterations
// after its summary (kBufs >= kLag + 2).  A buffer holds the chunk's tokens
// and three words per thread; then the shifts from a token's place in the
// chunk to its place in the output, one per document of the chunk written.
constexpr int kBufs = 3;
constexpr int kLag = 1;
static_assert(kBufs >= kLag + 2, "a buffer is refilled one iteration after its chunk was written");
constexpr int kBufWords = static_cast<int>(kOneChunk) + 3 * kOneThreads;
constexpr size_t kOneSmem = (static_cast<size_t>(kBufs) * kBufWords + kOneChunk + 1) * sizeof(int32_t);
constexpr int kRecWords = 4;  // int64 words per record

// Checked build only: a one-shot request (thd_debug_stall_next_pack) makes
// the block that takes chunk 0 of the next single-pass packing publish no
// summary, so the scanner waits on a record that nothing writes.
__device__ int g_pack_stall_request;

struct OnePassArgs {
  int32_t eod, align, pad_id;
  KeyGeom key;
  const int64_t* ve;       // per-row valid ends (trimming), else null
  const int64_t* vbefore;  // per-row unpadded offsets (trimming)
  const int32_t* row_next;
  int32_t* tokens;
  int64_t tok_cap;
  int32_t *cu_v, *cu, *next_tok;
  uint8_t* has_next;
  int64_t docs_cap;
  int64_t* counts;
  unsigned long long* ticket;  // [0]: chunks taken, [1]: roles taken
  int64_t* sums;               // per chunk: its summary record
  int64_t* carries;            // per chunk: its carries record
  int32_t* status;
};

// Thread t's 16 tokens [16t, 16t + 16) of a chunk in shared memory.  Thread
// t reads its four 16-byte pieces starting at piece (t/2) mod 4, so the
// eight threads of a quarter warp hit eight different 16-byte bank groups,
// then puts them back in order.
__device__ __forceinline__ void read_chunk_tokens(const int32_t* buf, int32_t (&v)[kOneK]) {
  const int4* src = reinterpret_cast<const int4*>(buf) + threadIdx.x * 4;
  const int rot = (threadIdx.x >> 1) & 3;
  int4 q0 = src[rot], q1 = src[(rot + 1) & 3], q2 = src[(rot + 2) & 3], q3 = src[(rot + 3) & 3];
  if (rot & 1) {  // piece m sits in q[(m - rot) mod 4]
    const int4 t = q3;
    q3 = q2, q2 = q1, q1 = q0, q0 = t;
  }
  if (rot & 2) {
    int4 t = q0;
    q0 = q2, q2 = t;
    t = q1;
    q1 = q3, q3 = t;
  }
  const int4 q[4] = {q0, q1, q2, q3};
#pragma unroll
  for (int m = 0; m < 4; ++m) v[4 * m] = q[m].x, v[4 * m + 1] = q[m].y, v[4 * m + 2] = q[m].z, v[4 * m + 3] = q[m].w;
}

// A thread's document ends among its 16 tokens, as positions relative to
// the chunk's first token: bit i of mask is token r0 + i; first and last (-1:
// none); psum = padded lengths of the documents between its consecutive ends.
struct RelEnds {
  uint32_t mask;
  int32_t first, last;
  int64_t psum;
};

__device__ __forceinline__ RelEnds rel_ends(const int32_t (&v)[kOneK], int32_t r0, int32_t n_valid, int32_t last_valid,
                                            int32_t eod, int32_t align) {
  RelEnds e;
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < kOneK; ++i) m |= v[i] == eod ? 1u << i : 0u;
  // the row's last valid token ends a document; tokens past the valid end
  // are none
  const uint32_t lv = static_cast<uint32_t>(last_valid - r0);
  if (lv < static_cast<uint32_t>(kOneK)) m |= 1u << lv;
  if (n_valid < r0 + kOneK) m &= n_valid > r0 ? (1u << (n_valid - r0)) - 1 : 0u;
  e.mask = m;
  e.first = e.mask ? r0 + __ffs(e.mask) - 1 : -1;
  e.last = e.mask ? r0 + 31 - __clz(e.mask) : -1;
  e.psum = 0;
  int32_t prev = -1;
  for (uint32_t m = e.mask; m; m &= m - 1) {
    const int32_t r = r0 + __ffs(m) - 1;
    if (prev >= 0) e.psum += (r - prev) + pad_of(r - prev, align);
    prev = r;
  }
  return e;
}

// block_exclusive_scan without its closing barrier: the caller does not
// reuse `warp_tmp` before the next barrier
template <typename V, class Op>
__device__ __forceinline__ V block_scan_open(V v, Op op, V identity, V* warp_tmp, V* total) {
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
    warp_tmp[32 + lane] = w;
  }
  __syncthreads();
  V before_lane = __shfl_up_sync(kFullMask, x, 1);
  if (lane == 0) before_lane = identity;
  *total = warp_tmp[32 + nw - 1];
  return op(wid > 0 ? warp_tmp[32 + wid - 1] : identity, before_lane);
}

// One poll of a summary record; true (and *out) when it is there.
__device__ __forceinline__ bool summary_peek(const int64_t* rec, RunSummary* out) {
  uint64_t a0, b0, a1, b1;
  asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(a0), "=l"(b0) : "l"(rec) : "memory");
  asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(a1), "=l"(b1) : "l"(rec + 2) : "memory");
  const uint64_t s0 = a0 >> kStateShift, s1 = b1 >> kStateShift;
  if (s0 == 0 || s0 != s1) return false;
  *out = s0 == kReady ? RunSummary{static_cast<int64_t>(a0 & kLow62), static_cast<int64_t>(b0), static_cast<int64_t>(a1),
                                   static_cast<int64_t>(b1 & kLow62)}
                      : run_poison();
  return true;
}

// The scanner block.  Warp w takes the windows of 32 chunks w, w + NW, ...
// (NW warps).  The prefix of every chunk before a window comes from the warp
// of the previous window through shared memory; the window's carries wait
// only for the summaries of the chunks before them: each time the summaries
// of a longer run of the window's first chunks are there (and the prefix),
// the warp scans them and publishes the carries of the chunks after them.
// Summaries are polled while the prefix is still on its way, and a window
// whose 32 summaries are all there is scanned before its prefix arrives, so
// that the hand-over from window to window costs one combine.
__device__ void pack_scanner(const ChunkGeom& g, const OnePassArgs& a) {
  __shared__ RunSummary mail[32];     // per warp: the prefix before its next window
  __shared__ int64_t mail_window[32];  // ... and which window that is
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  if (lane == 0) mail_window[wid] = -1;
  __syncthreads();
  volatile int64_t* vwin = mail_window;
  volatile int64_t* vmail = reinterpret_cast<volatile int64_t*>(mail);
  const int64_t nwin = (g.nc + 31) / 32;
  if (threadIdx.x == 0) carry_publish(a.carries, Carry{0, 0, -1, true});  // nothing before chunk 0
  // the carries of chunk z + 1 from the summary of every chunk up to z
  auto publish = [&](int64_t z, const RunSummary& inc) {
    if (z + 1 < g.nc) {
      Carry cr{0, 0, -1, inc.n >= 0};
      if (cr.ok && inc.n > 0) {
        const int64_t L0 = (inc.first & a.key.mask) + 1;  // the first document starts at its row's start
        cr.doc = inc.n;
        cr.out = L0 + pad_of(L0, a.align) + inc.psum;
        if ((inc.last >> a.key.shift) == (z + 1) / g.per_row) cr.end = inc.last & a.key.mask;
      }
      carry_publish(a.carries + (z + 1) * kRecWords, cr);
    }
    if (z == g.nc - 1 && inc.n >= 0) {
      const int64_t L0 = (inc.first & a.key.mask) + 1;
      const int64_t t_all = inc.n > 0 ? L0 + pad_of(L0, a.align) + inc.psum : 0;
      publish_totals(inc.n, t_all, a.tok_cap, a.docs_cap, a.cu_v, a.cu, a.counts, a.status);
    }
  };
  auto scan = [&](RunSummary x) {  // inclusive, lane order
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const RunSummary w = run_shfl_up(x, o);
      if (lane >= o) x = run_combine(w, x, a.key);
    }
    return x;
  };
  for (int64_t k = wid; k < nwin; k += nw) {
    const int64_t z = k * 32 + lane;
    RunSummary before = run_identity();
    bool got_before = k == 0;
    RunSummary mine = run_identity();  // this lane's chunk (identity past the last chunk)
    bool have = z >= g.nc;
    RunSummary full = run_identity();  // the window scanned, once all its summaries are there
    bool scanned = false;
    int done = 0;  // the window's first `done` chunks have had their carries published
    for (int it = 0; done < 32; ++it) {
      if (it >= kWaitLimit) {  // gave up: whatever is missing is poisoned
        if (!got_before) before = run_poison(), got_before = true;
        if (!have) mine = run_poison(), have = true;
        status_set(a.status, THD_ERR_TIMEOUT);
      }
      if (__any_sync(kFullMask, !have)) {
        if (!have) have = summary_peek(a.sums + z * kRecWords, &mine);
        if (__ballot_sync(kFullMask, have) == 0u || !__any_sync(kFullMask, lane >= done && have)) __nanosleep(64);
      }
      if (!got_before && vwin[wid] == k) {
        __threadfence_block();
        before = RunSummary{vmail[wid * 4], vmail[wid * 4 + 1], vmail[wid * 4 + 2], vmail[wid * 4 + 3]};
        got_before = true;
      }
      const uint32_t avail = __ballot_sync(kFullMask, have);
      const int c = avail == kFullMask ? 32 : __ffs(~avail) - 1;  // leading chunks whose summaries are there
      if (c == 32 && !scanned) {
        full = scan(mine);
        scanned = true;
      }
      if (!got_before || c <= done) continue;
      const RunSummary inc = run_combine(before, c == 32 ? full : scan(lane < c ? mine : run_identity()), a.key);
      if (c == 32 && lane == 31 && k + 1 < nwin) {  // hand on the prefix through the window first
        const int nxt = wid + 1 == nw ? 0 : wid + 1;
        vmail[nxt * 4] = inc.n, vmail[nxt * 4 + 1] = inc.psum, vmail[nxt * 4 + 2] = inc.first;
        vmail[nxt * 4 + 3] = inc.last;
        __threadfence_block();
        vwin[nxt] = k + 1;
      }
      if (lane >= done && lane < c) publish(z, inc);
      done = c;
    }
  }
}

__global__ void __launch_bounds__(1024)
pack_onepass_prepare_kernel(int64_t nc, unsigned long long* ticket, int64_t* recs, const int64_t* ve, int32_t B,
                            int64_t* vbefore) {
  __shared__ int64_t tmp[32];
  pdl_wait_then_release();
  if (threadIdx.x < 2) ticket[threadIdx.x] = 0;
  // the summary and carries records of every chunk: state 0
  int4* r = reinterpret_cast<int4*>(recs);
  for (int64_t i = threadIdx.x; i < nc * 2 * kRecWords / 2; i += blockDim.x) r[i] = make_int4(0, 0, 0, 0);
  if (ve) {
    int64_t carry = 0;
    for (int64_t base = 0; base < B; base += blockDim.x) {
      const int64_t rr = base + threadIdx.x;
      const int64_t v = rr < B ? ve[rr] : 0;
      int64_t pass;
      const int64_t before = block_exclusive_scan(v, OpSum(), static_cast<int64_t>(0), tmp, &pass);
      if (rr < B) vbefore[rr] = carry + before;
      carry += pass;
    }
  }
}


// One poll of a record, without waiting: the loads stay in flight until the
// values are used.
__device__ __forceinline__ void rec_peek(const int64_t* rec, uint64_t (&w)[4]) {
  asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(w[0]), "=l"(w[1]) : "l"(rec) : "memory");
  asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(w[2]), "=l"(w[3]) : "l"(rec + 2) : "memory");
}

// The blocks that pack (every block but the scanner).  A block works on a
// ring of kBufs chunks; call the chunks it takes, in order, its chunks 0, 1,
// 2, ...  In iteration i it
//   (a) sets out to take its chunk i + 1 (the counter's answer is used after
//       (b), when thread 0 starts that chunk's bulk load into its buffer,
//       free since the chunk that held it was written);
//   (b) summarises its chunk i (whose tokens were requested one iteration
//       ago) and publishes the summary; every thread keeps its ends, the
//       last end before it and the padded tokens before it in the buffer;
//   (c) writes its chunk i - kLag, whose carries the scanner has had kLag
//       iterations to publish: every document end writes its boundaries,
//       padding and the shift of the next document's tokens, then the block
//       copies the tokens with consecutive threads on consecutive tokens.
// A chunk held between its summary and its writing delays no one (its
// summary is out); the one chunk held without a summary, i + 1, has a
// larger number than every chunk the block waits for.
__global__ void __launch_bounds__(kOneThreads, kOneBlocksPerSm)
pack_onepass_kernel(const int32_t* raw, ChunkGeom g, OnePassArgs a) {
  extern __shared__ __align__(16) int32_t one_smem[];
  __shared__ int32_t scan_a[64];
  __shared__ int64_t scan_b[64];
  __shared__ uint64_t bars[kBufs];
  // per buffer: its chunk (>= nc: none), that chunk's row's valid end, the
  // chunk's scan total, row and first token, its first and last end
  // (relative to that token) and whether its tokens failed to land
  __shared__ int64_t sh_z[kBufs], sh_ve[kBufs], sh_total[kBufs], sh_row[kBufs], sh_lo[kBufs];
  __shared__ int32_t sh_first[kBufs], sh_last[kBufs], sh_bad[kBufs];
  __shared__ Carry sh_carry;
  __shared__ int32_t sh_role;
  // buffer b: tokens [kOneChunk], then per thread its ends | ends before <<
  // 16, its last end before it, its padded tokens before it
  auto tokens_of = [&](int b) { return one_smem + b * kBufWords; };
  auto ends_of = [&](int b) { return reinterpret_cast<uint32_t*>(one_smem + b * kBufWords + kOneChunk); };
  auto prev_of = [&](int b) { return one_smem + b * kBufWords + kOneChunk + kOneThreads; };
  auto psum_of = [&](int b) { return one_smem + b * kBufWords + kOneChunk + 2 * kOneThreads; };
  int32_t* const doc_shift = one_smem + kBufs * kBufWords;
  pdl_wait_then_release();
  if (block_status_set(a.status)) return;
  if (threadIdx.x == 0) sh_role = static_cast<int32_t>(atomicAdd(a.ticket + 1, 1ull));
  __syncthreads();
  if (sh_role == 0) {
    pack_scanner(g, a);
    return;
  }
  const int32_t r0 = static_cast<int32_t>(threadIdx.x) * kOneK;
  const int64_t cnt_mask = (int64_t(1) << kCntBits) - 1;
  uint32_t phase_bits = 0;  // bit b: the parity buffer b's barrier waits for next

  // thread 0: chunk z (from the counter) into buffer b; a number >= nc
  // marks the buffer empty
  auto start_chunk = [&](int b, int64_t z) {
    sh_z[b] = z;
    if (z < g.nc) {
      const int64_t row = z / g.per_row, lo = (z - row * g.per_row) * g.chunk;
      const uint32_t bytes = static_cast<uint32_t>(min(g.chunk, g.S - lo) * sizeof(int32_t));
      sh_ve[b] = a.ve ? a.ve[row] : g.S;
      sh_row[b] = row;
      sh_lo[b] = lo;
      mbar_arrive_expect_tx(&bars[b], bytes);
      bulk_load(tokens_of(b), raw + row * g.S + lo, bytes, &bars[b]);
    }
  };
  // the chunk in buffer b: its row and first token, its valid tokens
  // [0, n_valid) relative to that token, and the row's last valid token (-1:
  // not in this chunk)
  auto chunk_span = [&](int b, int64_t ve, int64_t* row, int64_t* lo, int32_t* n_valid, int32_t* last_valid) {
    *row = sh_row[b];
    *lo = sh_lo[b];
    *n_valid = static_cast<int32_t>(max(int64_t(0), min(g.chunk, ve - *lo)));
    *last_valid = ve - *lo - 1 < g.chunk ? static_cast<int32_t>(ve - *lo - 1) : -1;
  };

  // (b): summarise the chunk in buffer b and publish its summary (a chunk
  // whose tokens did not land: poisoned)
  auto summarize = [&](int b) {
    const int64_t z = sh_z[b];
    int64_t row, lo;
    int32_t n_valid, last_valid;
    chunk_span(b, sh_ve[b], &row, &lo, &n_valid, &last_valid);
    const bool landed = mbar_wait(&bars[b], (phase_bits >> b) & 1u);
    phase_bits ^= 1u << b;
    RelEnds te;
    {
      int32_t v[kOneK];
      read_chunk_tokens(tokens_of(b), v);
      te = rel_ends(v, r0, n_valid, last_valid, a.eod, a.align);
    }
    int32_t chunk_last;
    int64_t total;
    const int32_t prev_last = block_scan_open(te.last, OpMax(), -1, scan_a, &chunk_last);
    // documents that start after the chunk's first end; the thread holding
    // that end names it (its document's length depends on the carries)
    const int32_t cnt = __popc(te.mask);
    int64_t psum = te.psum;
    if (cnt > 0) {
      if (prev_last >= 0) psum += (te.first - prev_last) + pad_of(te.first - prev_last, a.align);
      else sh_first[b] = te.first;
    }
    const int64_t before = block_scan_open((psum << kCntBits) | cnt, OpSum(), static_cast<int64_t>(0), scan_b, &total);
    ends_of(b)[threadIdx.x] = te.mask | static_cast<uint32_t>(before & cnt_mask) << 16;
    prev_of(b)[threadIdx.x] = prev_last;
    psum_of(b)[threadIdx.x] = static_cast<int32_t>(before >> kCntBits);
    const bool bad = !__syncthreads_and(landed);
    if (threadIdx.x == 0) {
      sh_total[b] = total;
      sh_last[b] = chunk_last;
      sh_bad[b] = bad;
      const bool stall = kChecked && z == 0 && atomicExch(&g_pack_stall_request, 0) != 0;
      int64_t* rec = a.sums + z * kRecWords;
      if (bad) {
        status_set(a.status, THD_ERR_TIMEOUT);
        summary_publish(rec, run_poison());
      } else if (!stall) {
        const int64_t n_end = total & cnt_mask;
        const int64_t key_row = row << a.key.shift;
        summary_publish(rec, RunSummary{n_end, total >> kCntBits, n_end ? key_row | (lo + sh_first[b]) : 0,
                                        n_end ? key_row | (lo + chunk_last) : 0});
      }
    }
  };

  bool taking = false;  // thread 0: the counter may still hand out chunks
  if (threadIdx.x == 0) {
    for (int b = 0; b < kBufs; ++b) {
      mbar_init(&bars[b], 1);
      sh_z[b] = g.nc;
    }
    mbar_init_fence();
    const int64_t z0 = static_cast<int64_t>(atomicAdd(a.ticket, 1ull));
    start_chunk(0, z0);
    taking = z0 < g.nc;
  }
  for (int64_t i = 0;; ++i) {
    __syncthreads();  // the buffers' chunk numbers are visible; the previous copy is done
    const int bs = static_cast<int>(i % kBufs), bl = static_cast<int>((i + 1) % kBufs);
    const int be = static_cast<int>((i + kBufs - kLag) % kBufs);
    // (a) the counter's answer for chunk i + 1 arrives while (b) runs
    unsigned long long tk = 0;
    if (threadIdx.x == 0 && taking) tk = atomicAdd(a.ticket, 1ull);
    const int64_t zS = sh_z[bs];
    const int64_t zE = i >= kLag ? sh_z[be] : g.nc;
    uint64_t cw[4] = {0, 0, 0, 0};
    if (threadIdx.x == 0 && zE < g.nc) rec_peek(a.carries + zE * kRecWords, cw);  // used after (b)
    if (zS >= g.nc && zE >= g.nc) break;  // (block-uniform) nothing left
    if (zS < g.nc) summarize(bs);
    if (threadIdx.x == 0) {
      // buffer bl held chunk i + 1 - kBufs, written kBufs - kLag - 1 iterations ago
      if (taking) {
        start_chunk(bl, static_cast<int64_t>(tk));
        taking = static_cast<int64_t>(tk) < g.nc;
      } else {
        sh_z[bl] = g.nc;
      }
    }
    if (zE >= g.nc) continue;

    // (c) chunk zE from buffer be
    if (threadIdx.x == 0) {
      const uint64_t s0 = cw[0] >> kStateShift, s1 = cw[3] >> kStateShift;
      Carry c;
      if (s0 == kReady && s1 == kReady)
        c = Carry{static_cast<int64_t>(cw[0] & kLow62), static_cast<int64_t>(cw[1]), static_cast<int64_t>(cw[2]) - 1,
                  true};
      else
        c = carry_wait(a.carries + zE * kRecWords);
      if (!c.ok) status_set(a.status, THD_ERR_TIMEOUT);
      sh_carry = c;
    }
    __syncthreads();
    const Carry c = sh_carry;
    int64_t row, lo;
    int32_t n_valid, last_valid;
    const int64_t ve = sh_ve[be];
    chunk_span(be, ve, &row, &lo, &n_valid, &last_valid);
    const int32_t* const tok = tokens_of(be);
    const uint32_t* const ends = ends_of(be);
    const uint32_t my_ends = ends[threadIdx.x];
    const uint32_t mask = my_ends & 0xffffu;
    const int32_t prev_last = prev_of(be)[threadIdx.x];
    const int64_t total = sh_total[be];
    const int32_t chunk_last = sh_last[be];
    const int64_t n_end = total & cnt_mask;
    // the output tokens of the chunk: [o_lo, o_hi)
    const int64_t first_len = lo + sh_first[be] - c.end;
    const int64_t first_pad = n_end > 0 ? first_len + pad_of(first_len, a.align) : 0;
    const int64_t o_lo = c.out + (lo - c.end - 1);
    const int64_t o_hi =
        n_end > 0 ? c.out + first_pad + (total >> kCntBits) + (n_valid - 1 - chunk_last) : o_lo + n_valid;
    const bool ok = c.ok && sh_bad[be] == 0 && n_valid > 0 && o_hi <= a.tok_cap && o_hi <= INT32_MAX &&
                    c.doc + n_end < a.docs_cap;
    // token r of the chunk, in the chunk's document j (the ends before r),
    // goes to o_lo + r + doc_shift[j]
    if (ok && threadIdx.x == 0) doc_shift[0] = 0;
    if (ok && mask) {
      int64_t pe = prev_last >= 0 ? lo + prev_last : c.end;  // the end before this thread's first token
      const int32_t cnt_before = static_cast<int32_t>(my_ends >> 16);
      int64_t doc = c.doc + cnt_before;
      int64_t out = c.out + (prev_last >= 0 ? first_pad : 0) + psum_of(be)[threadIdx.x];
      int32_t k = cnt_before;  // this thread's first end in the chunk
      const int64_t v_before = a.vbefore ? a.vbefore[row] : row * g.S;
      for (uint32_t m = mask; m; m &= m - 1) {
        const int32_t r = r0 + __ffs(m) - 1;
        const int64_t t = lo + r;
        const int64_t L = t - pe;
        const int64_t P = L + pad_of(L, a.align);
        for (int64_t zz = L; zz < P; ++zz)
          if (in_range(out + zz, o_lo, o_hi, a.status)) a.tokens[out + zz] = a.pad_id;
        if (in_range(doc + 1, 1, a.docs_cap, a.status) && in_range(k, 0, n_end, a.status)) {
          a.cu_v[doc + 1] = static_cast<int32_t>(v_before + t + 1);
          a.cu[doc + 1] = static_cast<int32_t>(out + P);
          if (a.has_next) {
            // the row's extra token continues its last document when that
            // document reaches the row's end without an EOD
            const bool cont = a.row_next != nullptr && tok[r] != a.eod && ve == g.S;
            a.has_next[doc] = cont ? 1 : 0;
            a.next_tok[doc] = cont ? a.row_next[row] : 0;
          }
          doc_shift[k + 1] = static_cast<int32_t>(out + P - o_lo - r - 1);
        }
        ++k;
        ++doc;
        out += P;
        pe = t;
      }
    }
    __syncthreads();
    if (ok) {
      // consecutive threads on consecutive tokens: warp w copies the groups
      // of 32 tokens [32w + q * kOneThreads, + 32); a group without a
      // document end before its last token lies in one document, whose shift
      // the warp looks up once
      int32_t* const out_base = a.tokens + o_lo;  // positions relative to o_lo (o_hi - o_lo < 2^31)
      const int32_t span = static_cast<int32_t>(o_hi - o_lo);
      const int32_t lane = static_cast<int32_t>(threadIdx.x) & 31;
#pragma unroll
      for (int q = 0; q < kOneK; ++q) {
        const int32_t rg = (static_cast<int32_t>(threadIdx.x) & ~31) + q * kOneThreads;
        if (rg < n_valid) {
          const int32_t r = rg + lane;
          const uint32_t t0 = ends[rg >> 4], t1 = ends[(rg >> 4) + 1];
          int32_t off;
          if (((t0 & 0xffffu) | (t1 & 0x7fffu)) == 0u) {
            off = r + doc_shift[t0 >> 16];
          } else {
            const uint32_t te = (r & 16) ? t1 : t0;
            off = r + doc_shift[static_cast<int32_t>(te >> 16) + __popc(te & ((1u << (r & 15)) - 1))];
          }
          if (r < n_valid && in_range(off, 0, span, a.status)) out_base[off] = tok[r];
        }
      }
    }
  }
}

}  // namespace

thd_status_t launch_pack_docs_rows(const int32_t* raw, int32_t B, int64_t S, int32_t eod, int32_t trim,
                              int32_t raw_pad, int32_t align, int32_t pad_id, int32_t* tokens,
                              int64_t tok_cap, int32_t* cu_v, int32_t* cu, int64_t docs_cap,
                              int64_t* counts, int64_t* ws, int32_t* status, cudaStream_t s) {
  cudaError_t e;
  if (B == 0) {
    // no rows: no documents, T = 0
    if ((e = cudaMemsetAsync(counts, 0, 2 * sizeof(int64_t), s)) != cudaSuccess ||
        (e = cudaMemsetAsync(cu, 0, sizeof(int32_t), s)) != cudaSuccess ||
        (e = cudaMemsetAsync(cu_v, 0, sizeof(int32_t), s)) != cudaSuccess) {
      record_cuda_error(e);
      return THD_ERR_CUDA;
    }
    return THD_OK;
  }
  if ((e = launch_pdl(pack_stats_kernel, B, kPackThreads, 0, s, raw, S, eod, trim, raw_pad, align, ws, status)) !=
      cudaSuccess) {
    record_cuda_error(e);
    return THD_ERR_CUDA;
  }
  const bool prefixed = B > kSelfScanRows;
  if (prefixed && (e = launch_pdl(pack_rows_scan_kernel, 1, kPackThreads, 0, s, B, tok_cap, docs_cap, cu_v, cu,
                                  counts, ws, status)) != cudaSuccess) {
    record_cuda_error(e);
    return THD_ERR_CUDA;
  }
  if ((e = launch_pdl(pack_emit_kernel, B, kPackThreads, 0, s, raw, B, S, eod, align, pad_id, tokens, tok_cap, cu_v,
                      cu, docs_cap, counts, static_cast<const int64_t*>(ws), prefixed, status)) != cudaSuccess) {
    record_cuda_error(e);
    return THD_ERR_CUDA;
  }
  return THD_OK;
}

}  // namespace thd

namespace thd {

// int64 words: row valid ends [B], chunk statistics [nc][4], chunk carries
// [nc][3], row offsets [B], totals [2] -- for the smaller chunks, an upper
// bound whichever chunk size the call takes; the single pass needs row valid
// ends [B], row offsets [B], two counters, one word of alignment and two
// records of four words per single-pass chunk.  The larger of the two.
size_t pack_docs_chunked_workspace(int32_t B, int64_t S) {
  const int64_t per_row = (S + kSmallChunk - 1) / kSmallChunk;
  const int64_t nc = static_cast<int64_t>(B) * per_row;
  const int64_t nc1 = static_cast<int64_t>(B) * ((S + kOneChunk - 1) / kOneChunk);
  const int64_t chunked = 2 * static_cast<int64_t>(B) + 7 * nc + 2;
  const int64_t one = 2 * static_cast<int64_t>(B) + 2 + 1 + 2 * kRecWords * nc1;
  return static_cast<size_t>(chunked > one ? chunked : one) * sizeof(int64_t);
}

namespace {
template <int K, bool VEC>
cudaError_t launch_chunked(const ChunkGeom& g, const int32_t* raw, int32_t eod, const int64_t* ve, int32_t align,
                           int32_t pad_id, int64_t* stats, int64_t* carry, int64_t* vbefore, int64_t* totals,
                           const int32_t* row_next, int32_t* tokens, int64_t tok_cap, int32_t* cu_v, int32_t* cu,
                           int32_t* next_tok, uint8_t* has_next, int64_t docs_cap, int64_t* counts, int32_t* status,
                           cudaStream_t s) {
  const dim3 grid(static_cast<unsigned>(g.per_row), static_cast<unsigned>(g.B));
  cudaError_t e = launch_pdl(pack_chunk_stats_kernel<K, VEC>, grid, kChunkThreads, 0, s, raw, g, eod, ve, align,
                             stats, status);
  if (e != cudaSuccess) return e;
  const bool self_scan = g.nc <= kSelfScanChunks;
  if (!self_scan &&
      (e = launch_pdl(pack_chunk_scan_kernel, 1, kScanThreads, 0, s, g, ve, align, static_cast<const int64_t*>(stats),
                      carry, vbefore, totals, tok_cap, docs_cap, cu_v, cu, counts, status)) != cudaSuccess)
    return e;
  return launch_pdl(pack_chunk_emit_kernel<K, VEC>, grid, kChunkThreads, 0, s, raw, g, eod, ve, align, pad_id,
                    static_cast<const int64_t*>(stats), static_cast<const int64_t*>(self_scan ? nullptr : carry),
                    static_cast<const int64_t*>(vbefore), static_cast<const int64_t*>(totals), row_next, tokens,
                    tok_cap, cu_v, cu, next_tok, has_next, docs_cap, counts, status);
}
}  // namespace

namespace {
// The single pass: [row valid ends] -> prepare -> one persistent kernel of
// two blocks per SM.
thd_status_t launch_pack_onepass(const int32_t* raw, int32_t B, int64_t S, int32_t eod, int32_t trim,
                                 int32_t raw_pad, int32_t align, int32_t pad_id, const int32_t* row_next,
                                 int32_t* tokens, int64_t tok_cap, int32_t* cu_v, int32_t* cu, int32_t* next_tok,
                                 uint8_t* has_next, int64_t docs_cap, int64_t* counts, int64_t* ws, int32_t* status,
                                 cudaStream_t s) {
  ChunkGeom g;
  g.B = B;
  g.S = S;
  g.chunk = kOneChunk;
  g.per_row = (S + kOneChunk - 1) / kOneChunk;
  g.nc = static_cast<int64_t>(B) * g.per_row;
  OnePassArgs a;
  a.eod = eod;
  a.align = align;
  a.pad_id = pad_id;
  a.key.shift = 1;
  while ((int64_t(1) << a.key.shift) < S) ++a.key.shift;
  a.key.mask = (int64_t(1) << a.key.shift) - 1;
  a.key.align = align;
  int64_t* ve = ws;
  int64_t* vbefore = ws + B;
  a.ve = trim ? ve : nullptr;
  a.vbefore = trim ? vbefore : nullptr;
  a.row_next = row_next;
  a.tokens = tokens;
  a.tok_cap = tok_cap;
  a.cu_v = cu_v;
  a.cu = cu;
  a.next_tok = next_tok;
  a.has_next = has_next;
  a.docs_cap = docs_cap;
  a.counts = counts;
  // ws: ve [B], vbefore [B], two counters, then (16-byte aligned) the summary
  // and carries records of every chunk
  a.ticket = reinterpret_cast<unsigned long long*>(ws + 2 * static_cast<int64_t>(B));
  int64_t* recs = ws + 2 * static_cast<int64_t>(B) + 2;
  if (reinterpret_cast<uintptr_t>(recs) % 16 != 0) ++recs;
  a.sums = recs;
  a.carries = recs + g.nc * kRecWords;
  a.status = status;
  cudaError_t e;
  if (trim && (e = launch_pdl(pack_row_ends_kernel, B, kPackThreads, 0, s, raw, S, raw_pad, ve, status)) !=
                  cudaSuccess) {
    record_cuda_error(e);
    return THD_ERR_CUDA;
  }
  // the kernel's shared-memory size, set when the context does not have it
  // yet (a query, so that a call made during stream capture only enqueues
  // launches, and a reset context gets it again)
  cudaFuncAttributes fa;
  if ((e = cudaFuncGetAttributes(&fa, pack_onepass_kernel)) != cudaSuccess ||
      (fa.maxDynamicSharedSizeBytes < static_cast<int>(kOneSmem) &&
       (e = cudaFuncSetAttribute(pack_onepass_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kOneSmem))) != cudaSuccess)) {
    record_cuda_error(e);
    return THD_ERR_CUDA;
  }
  if ((e = launch_pdl(pack_onepass_prepare_kernel, 1, 1024, 0, s, g.nc, a.ticket, recs,
                      static_cast<const int64_t*>(a.ve), B, vbefore)) != cudaSuccess) {
    record_cuda_error(e);
    return THD_ERR_CUDA;
  }
  // one scanner block and up to one block per chunk
  const int64_t grid = min(g.nc + 1, static_cast<int64_t>(kOneBlocksPerSm) * sm_count());
  if ((e = launch_pdl(pack_onepass_kernel, dim3(static_cast<unsigned>(grid)), kOneThreads, kOneSmem, s, raw, g, a)) !=
      cudaSuccess) {
    record_cuda_error(e);
    return THD_ERR_CUDA;
  }
  return THD_OK;
}
}  // namespace

thd_status_t launch_pack_docs(const int32_t* raw, int32_t B, int64_t S, int32_t eod, int32_t trim,
                              int32_t raw_pad, int32_t align, int32_t pad_id, const int32_t* row_next,
                              int32_t* tokens, int64_t tok_cap, int32_t* cu_v, int32_t* cu, int32_t* next_tok,
                              uint8_t* has_next, int64_t docs_cap, int64_t* counts, int64_t* ws, int32_t* status,
                              cudaStream_t s) {
  cudaError_t e;
  if (B == 0 || S == 0) {
    // no tokens: no documents, T = 0
    if ((e = cudaMemsetAsync(counts, 0, 2 * sizeof(int64_t), s)) != cudaSuccess ||
        (e = cudaMemsetAsync(cu, 0, sizeof(int32_t), s)) != cudaSuccess ||
        (e = cudaMemsetAsync(cu_v, 0, sizeof(int32_t), s)) != cudaSuccess) {
      record_cuda_error(e);
      return THD_ERR_CUDA;
    }
    return THD_OK;
  }
  const bool big = static_cast<int64_t>(B) * S >= kBigChunkFrom;
  // 16-byte loads: 16-byte aligned rows of a multiple of 4 tokens
  const bool vec = reinterpret_cast<uintptr_t>(raw) % 16 == 0 && S % 4 == 0;
  // (the single pass keys document ends as row << shift | position in 62 bits)
  int shift = 1;
  while ((int64_t(1) << shift) < S) ++shift;
  const bool keys_fit = shift < 62 && (static_cast<int64_t>(B) >> (61 - shift)) == 0;
  // (and keeps a chunk's padded tokens before a thread in 31 bits)
  if (static_cast<int64_t>(B) * S >= kOnePassFrom && vec && keys_fit && align <= 65536 &&
      reinterpret_cast<uintptr_t>(tokens) % 16 == 0)
    return launch_pack_onepass(raw, B, S, eod, trim, raw_pad, align, pad_id, row_next, tokens, tok_cap, cu_v, cu,
                               next_tok, has_next, docs_cap, counts, ws, status, s);
  ChunkGeom g;
  g.B = B;
  g.S = S;
  g.chunk = big ? 4 * kSmallChunk : kSmallChunk;
  g.per_row = (S + g.chunk - 1) / g.chunk;
  g.nc = static_cast<int64_t>(B) * g.per_row;
  int64_t* ve = trim ? ws : nullptr;
  int64_t* stats = ws + B;
  int64_t* carry = stats + 4 * g.nc;
  int64_t* vbefore = carry + 3 * g.nc;
  int64_t* totals = vbefore + B;
  if (trim) {
    if ((e = launch_pdl(pack_row_ends_kernel, B, kPackThreads, 0, s, raw, S, raw_pad, ws, status)) != cudaSuccess) {
      record_cuda_error(e);
      return THD_ERR_CUDA;
    }
  }
  const int64_t* vc = ve;
  if (big)
    e = vec ? launch_chunked<16, true>(g, raw, eod, vc, align, pad_id, stats, carry, vbefore, totals, row_next, tokens,
                                       tok_cap, cu_v, cu, next_tok, has_next, docs_cap, counts, status, s)
            : launch_chunked<16, false>(g, raw, eod, vc, align, pad_id, stats, carry, vbefore, totals, row_next,
                                        tokens, tok_cap, cu_v, cu, next_tok, has_next, docs_cap, counts, status, s);
  else
    e = vec ? launch_chunked<4, true>(g, raw, eod, vc, align, pad_id, stats, carry, vbefore, totals, row_next, tokens,
                                      tok_cap, cu_v, cu, next_tok, has_next, docs_cap, counts, status, s)
            : launch_chunked<4, false>(g, raw, eod, vc, align, pad_id, stats, carry, vbefore, totals, row_next, tokens,
                                       tok_cap, cu_v, cu, next_tok, has_next, docs_cap, counts, status, s);
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return THD_ERR_CUDA;
  }
  return THD_OK;
}

}  // namespace thd

// Declared in include/thd_debug.h; exported by the checked build only.
#if defined(THD_CHECKED) && THD_CHECKED
extern "C" thd_status_t thd_debug_stall_next_pack(cudaStream_t stream) {
  const int one = 1;
  const cudaError_t e =
      cudaMemcpyToSymbolAsync(thd::g_pack_stall_request, &one, sizeof(one), 0, cudaMemcpyHostToDevice, stream);
  if (e != cudaSuccess) {
    thd::record_cuda_error(e);
    return THD_ERR_CUDA;
  }
  return THD_OK;
}
#endif
