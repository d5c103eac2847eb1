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
//  * per row (thd_pack_docs_noalloc, whose scratch is a fixed array of four
//    int64 per row): the same phases with one block per raw row; above 512
//    rows one block turns the rows' statistics into prefixes in place
//    between them.
#include "thd_internal.cuh"

namespace thd {
namespace {

constexpr int kPackThreads = 1024;
constexpr int kItems = 8;  // consecutive tokens per thread per tile
constexpr int64_t kTile = static_cast<int64_t>(kPackThreads) * kItems;

__device__ __forceinline__ int64_t pad_of(int64_t L, int32_t align) {
  int64_t r = L % align;
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
// bound whichever chunk size the call takes
size_t pack_docs_chunked_workspace(int32_t B, int64_t S) {
  const int64_t per_row = (S + kSmallChunk - 1) / kSmallChunk;
  const int64_t nc = static_cast<int64_t>(B) * per_row;
  return static_cast<size_t>(2 * static_cast<int64_t>(B) + 7 * nc + 2) * sizeof(int64_t);
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
  // 16-byte loads: 16-byte aligned rows of a multiple of 4 tokens
  const bool vec = reinterpret_cast<uintptr_t>(raw) % 16 == 0 && S % 4 == 0;
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
