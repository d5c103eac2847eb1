// Pack raw [B, S] rows into one padded THD sequence on the device.
//
// "Packed Sequence 与上下文并行", section 2.2 (pack: split rows at EOD, pad
// every document to the alignment, flatten with document i starting at
// cu_seqlens_padded[i]) and the worked example of section 3.  The pages do it
// with bincount/cumsum and a per-document copy loop on the host side of the
// framework.  Two device implementations:
//
//  * chunked (thd_pack_docs): rows are cut into chunks of 2048 tokens, one
//    block each, so all SMs take part.
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
//         checked against the capacities.  Up to 512 chunks (about 1M raw
//         tokens) every emit block does this for itself; beyond that one
//         block does it first and stores every chunk's carries;
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

constexpr int kChunkThreads = 256;
constexpr int kChunkItems = 8;
constexpr int64_t kChunk = static_cast<int64_t>(kChunkThreads) * kChunkItems;  // tokens per chunk

struct OpMin {
  template <typename V>
  __device__ __forceinline__ V operator()(V a, V b) const { return a < b ? a : b; }
};

struct ChunkGeom {
  int32_t B;
  int64_t S;
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

// stats[z] = {ends, first end (-1: none), last end (-1: none), padded length of
// the documents after the first end}, z = b * per_row + c
__global__ void __launch_bounds__(kChunkThreads)
pack_chunk_stats_kernel(const int32_t* raw, ChunkGeom g, int32_t eod, const int64_t* ve_arr, int32_t align,
                        int64_t* stats, int32_t* status) {
  __shared__ int64_t tmp[32];
  pdl_wait_then_release();
  if (block_status_set(status)) return;
  const int64_t b = blockIdx.y, c = blockIdx.x;
  const int32_t* row = raw + b * g.S;
  const int64_t ve = ve_arr ? ve_arr[b] : g.S;
  const int64_t lo = c * kChunk, hi = min(lo + kChunk, ve);
  const int64_t t0 = lo + static_cast<int64_t>(threadIdx.x) * kChunkItems;
  int64_t my_first = INT64_MAX, my_last = -1;
  for (int it = 0; it < kChunkItems; ++it) {
    const int64_t t = t0 + it;
    if (t < hi && is_end(row, t, ve, eod)) {
      if (my_first == INT64_MAX) my_first = t;
      my_last = t;
    }
  }
  int64_t chunk_last, chunk_first;
  const int64_t prev = block_exclusive_scan(my_last, OpMax(), static_cast<int64_t>(-1), tmp, &chunk_last);
  block_exclusive_scan(my_first, OpMin(), INT64_MAX, tmp, &chunk_first);
  int64_t cnt = 0, psum = 0, pe = prev;
  for (int it = 0; it < kChunkItems; ++it) {
    const int64_t t = t0 + it;
    if (t < hi && is_end(row, t, ve, eod)) {
      if (pe >= 0) psum += (t - pe) + pad_of(t - pe, align);  // starts inside this chunk
      ++cnt;
      pe = t;
    }
  }
  cnt = block_sum(cnt, tmp);
  psum = block_sum(psum, tmp);
  if (threadIdx.x == 0) {
    int64_t* st = stats + (b * g.per_row + c) * 4;
    st[0] = cnt;
    st[1] = cnt > 0 ? chunk_first : -1;
    st[2] = chunk_last;
    st[3] = psum;
  }
}

// The block walks every chunk's statistics in order: a max-scan carries
// each row's last end into the next chunk, sum-scans give every chunk's first
// document index and output offset.  Chunk z's three carries go to
// carry_out[z * 3 ...] when carry_out is set, else only chunk `mine`'s to
// mine_out[0..2]; totals_out gets {documents, padded tokens}.
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

// One block over all chunks (more than kSelfScanChunks): every chunk's carries,
// every row's unpadded offset (vbefore, when the rows are trimmed) and the
// totals.
constexpr int kScanThreads = 1024;

__global__ void __launch_bounds__(kScanThreads)
pack_chunk_scan_kernel(ChunkGeom g, const int64_t* ve_arr, int32_t align, const int64_t* stats, int64_t* carry,
                       int64_t* vbefore, int64_t* totals, int64_t tok_cap, int64_t docs_cap, int32_t* cu_v,
                       int32_t* cu, int64_t* counts, int32_t* status) {
  __shared__ int64_t tmp[32];
  __shared__ int64_t tot[2];
  pdl_wait_then_release();
  if (block_status_set(status)) return;
  scan_chunks(g, align, stats, carry, -1, nullptr, tot, tmp);
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
  __syncthreads();
  if (threadIdx.x == 0) {
    totals[0] = tot[0];
    totals[1] = tot[1];
    publish_totals(tot[0], tot[1], tok_cap, docs_cap, cu_v, cu, counts, status);
  }
}

__global__ void __launch_bounds__(kChunkThreads)
pack_chunk_emit_kernel(const int32_t* raw, ChunkGeom g, int32_t eod, const int64_t* ve_arr, int32_t align,
                       int32_t pad_id, const int64_t* stats, const int64_t* carry, const int64_t* vbefore,
                       const int64_t* totals, const int32_t* row_next, int32_t* tokens, int64_t tok_cap,
                       int32_t* cu_v, int32_t* cu, int32_t* next_tok, uint8_t* has_next, int64_t docs_cap,
                       int64_t* counts, int32_t* status) {
  __shared__ int64_t tmp[32];
  __shared__ int64_t mine[3], tot[2];
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
  const int64_t lo = c * kChunk, hi = min(lo + kChunk, ve);
  const int64_t t0 = lo + static_cast<int64_t>(threadIdx.x) * kChunkItems;
  int64_t my_last = -1;
  for (int it = 0; it < kChunkItems; ++it) {
    const int64_t t = t0 + it;
    if (t < hi && is_end(row, t, ve, eod)) my_last = t;
  }
  int64_t unused;
  int64_t first_prev = block_exclusive_scan(my_last, OpMax(), static_cast<int64_t>(-1), tmp, &unused);
  first_prev = max(first_prev, carry_end);
  int64_t cnt = 0, psum = 0;
  {
    int64_t pe = first_prev;
    for (int it = 0; it < kChunkItems; ++it) {
      const int64_t t = t0 + it;
      if (t < hi && is_end(row, t, ve, eod)) {
        psum += (t - pe) + pad_of(t - pe, align);
        ++cnt;
        pe = t;
      }
    }
  }
  const int64_t cnt_before = block_exclusive_scan(cnt, OpSum(), static_cast<int64_t>(0), tmp, &unused);
  const int64_t psum_before = block_exclusive_scan(psum, OpSum(), static_cast<int64_t>(0), tmp, &unused);
  int64_t pe = first_prev;
  int64_t doc = carry_doc + cnt_before;  // document the next token belongs to
  int64_t out = carry_out + psum_before; // that document's first output row
  for (int it = 0; it < kChunkItems; ++it) {
    const int64_t t = t0 + it;
    if (t >= hi) break;
    const int32_t v = row[t];
    if (in_range(out + (t - pe - 1), 0, t_all, status)) tokens[out + (t - pe - 1)] = v;
    if (v == eod || t == ve - 1) {
      const int64_t L = t - pe;
      const int64_t P = L + pad_of(L, align);
      for (int64_t zz = L; zz < P; ++zz)
        if (in_range(out + zz, 0, t_all, status)) tokens[out + zz] = pad_id;
      if (!in_range(doc + 1, 1, d_all + 1, status)) break;
      cu_v[doc + 1] = static_cast<int32_t>(v_before + t + 1);
      cu[doc + 1] = static_cast<int32_t>(out + P);
      if (has_next) {
        // the row's extra token continues its last document when that
        // document reaches the row's end without an EOD
        const bool cont = row_next != nullptr && v != eod && ve == g.S;
        has_next[doc] = cont ? 1 : 0;
        next_tok[doc] = cont ? row_next[b] : 0;
      }
      ++doc;
      out += P;
      pe = t;
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
// [nc][3], row offsets [B], totals [2]
size_t pack_docs_chunked_workspace(int32_t B, int64_t S) {
  const int64_t per_row = (S + kChunk - 1) / kChunk;
  const int64_t nc = static_cast<int64_t>(B) * per_row;
  return static_cast<size_t>(2 * static_cast<int64_t>(B) + 7 * nc + 2) * sizeof(int64_t);
}

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
  ChunkGeom g;
  g.B = B;
  g.S = S;
  g.per_row = (S + kChunk - 1) / kChunk;
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
  const dim3 grid(static_cast<unsigned>(g.per_row), static_cast<unsigned>(B));
  if ((e = launch_pdl(pack_chunk_stats_kernel, grid, kChunkThreads, 0, s, raw, g, eod,
                      static_cast<const int64_t*>(ve), align, stats, status)) != cudaSuccess) {
    record_cuda_error(e);
    return THD_ERR_CUDA;
  }
  const bool self_scan = g.nc <= kSelfScanChunks;
  if (!self_scan &&
      (e = launch_pdl(pack_chunk_scan_kernel, 1, kScanThreads, 0, s, g, static_cast<const int64_t*>(ve), align,
                      static_cast<const int64_t*>(stats), carry, vbefore, totals, tok_cap, docs_cap, cu_v, cu, counts,
                      status)) != cudaSuccess) {
    record_cuda_error(e);
    return THD_ERR_CUDA;
  }
  if ((e = launch_pdl(pack_chunk_emit_kernel, grid, kChunkThreads, 0, s, raw, g, eod,
                      static_cast<const int64_t*>(ve), align, pad_id, static_cast<const int64_t*>(stats),
                      static_cast<const int64_t*>(self_scan ? nullptr : carry), static_cast<const int64_t*>(vbefore),
                      static_cast<const int64_t*>(totals), row_next, tokens, tok_cap, cu_v, cu, next_tok, has_next,
                      docs_cap, counts, status)) != cudaSuccess) {
    record_cuda_error(e);
    return THD_ERR_CUDA;
  }
  return THD_OK;
}

}  // namespace thd
