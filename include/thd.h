/*
 * thd.h -- C ABI of libthd: the packed-sequence (THD) context-parallel layout
 * conversion on one GPU.
 *
 * Terms.  A packed batch holds T rows (tokens) of num_docs documents back to
 * back; cu_seqlens_padded = [0, cu[1], ..., cu[num_docs] = T] are the padded
 * document boundaries (int32).  Every padded length cu[i+1]-cu[i] is a
 * multiple of 2*cp.  cp virtual context-parallel ranks each hold S = T/cp
 * rows; all of them live in ONE device buffer, rank-major:
 *
 *   zigzag layout      buffer[r*S + k] = global row zz[r][k], where rank r
 *                      takes, for each document in order, chunk r and then
 *                      chunk 2*cp-1-r of the document's 2*cp equal chunks
 *                      ("Packed Sequence 与上下文并行", section 2.4);
 *   contiguous layout  buffer[g] = global row g, i.e. rank r holds
 *                      [r*S, (r+1)*S) ("[Task32] feat: fla mcore chunkwise cp
 *                      stage 3", Relax PR #273, section 2.1).
 *
 * Because the ranks share one allocation, the pages' all-to-all becomes an
 * on-device row permutation.
 *
 * Conventions for every call:
 *  - Pointers marked "device" are device pointers owned by the caller; the
 *    library allocates nothing, creates no stream and keeps no state between
 *    calls (apart from a per-thread copy of the last CUDA error).
 *  - Work is enqueued asynchronously on the caller's `stream`; only
 *    thd_status_read synchronises.
 *  - Host-checkable argument errors (null pointers, sizes, direction) are
 *    returned at once; nothing is enqueued then.
 *  - Data-dependent errors (bad boundaries) are written by the GPU into the
 *    caller's status word `d_status` (device int32, clear it to 0 before
 *    first use).  The first error wins; a kernel that finds *d_status != 0
 *    on entry writes nothing, so one bad microbatch cannot scribble over
 *    memory downstream.  No kernel traps or asserts; the only waits (copy
 *    completion in the bulk copy pipeline) are bounded and report
 *    THD_ERR_TIMEOUT when they give up.
 *  - Every row index a kernel computes or reads is checked against its
 *    buffer before use; a bad one is skipped and reported as
 *    THD_ERR_INDEX_RANGE.
 */
#ifndef THD_H_
#define THD_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum thd_status {
  THD_OK = 0,
  THD_ERR_INVALID_ARG = 1,           /* host: null pointer, bad size, cp out of range */
  THD_ERR_BAD_DIRECTION = 2,         /* host: direction not one of thd_dir_t */
  THD_ERR_CU_NONZERO_START = 3,      /* device: cu[0] != 0 */
  THD_ERR_CU_NON_MONOTONE = 4,       /* device: cu[i+1] < cu[i] for some i */
  THD_ERR_LEN_NOT_DIVISIBLE = 5,     /* device: a padded length is not a multiple of 2*cp */
  THD_ERR_TOTAL_MISMATCH = 6,        /* device: cu[num_docs] != T */
  THD_ERR_TIMEOUT = 7,               /* device: a bounded wait in the bulk copy pipeline gave up */
  THD_ERR_CUDA = 8,                  /* host: a CUDA call failed, see thd_last_cuda_error() */
  THD_ERR_INDEX_RANGE = 9,           /* device: a route index was outside its buffer */
  THD_ERR_VALID_EXCEEDS_PADDED = 10, /* device: an unpadded length exceeds its padded length */
  THD_ERR_CAPACITY = 11,             /* device: pack_docs output larger than the given capacity */
  THD_ERR_SCRATCH_LIMIT = 12         /* host: request larger than thd_pack_docs_noalloc's fixed scratch */
} thd_status_t;

typedef enum thd_dir {
  THD_ZIGZAG_TO_CONTIGUOUS = 0,
  THD_CONTIGUOUS_TO_ZIGZAG = 1
} thd_dir_t;

typedef enum thd_ulysses_dir {
  THD_SEQ_TO_HEAD = 0,
  THD_HEAD_TO_SEQ = 1
} thd_ulysses_dir_t;

/* Largest supported cp_size. */
#define THD_MAX_CP 64

/*
 * The all-to-all route of one direction, every virtual rank at once
 * (Relax PR #273, sections 2.1 and 2.4: send_rows / recv_rows /
 * input_split_sizes / output_split_sizes, identity rows meaning zero-copy).
 * Source layout A and target layout B are (zigzag, contiguous) for
 * THD_ZIGZAG_TO_CONTIGUOUS and (contiguous, zigzag) for the reverse.
 *
 * All arrays are device memory owned by the caller; thd_route_bind carves
 * them out of one caller buffer of thd_route_bytes(T, cp) bytes.
 *
 *  send_rows[s*S + j]   local source row of rank s placed at slot j of its send
 *                       buffer; grouped by destination rank ascending, rows of
 *                       one group in ascending global order.
 *  recv_rows[d*S + j]   local target row of rank d that receives slot j of its
 *                       receive buffer; grouped by source rank ascending.
 *  input_split_sizes[s*cp + d]   rows rank s sends to rank d.
 *  output_split_sizes[d*cp + s]  rows rank d receives from rank s.
 *  send_offsets[s*(cp+1) + d]    exclusive prefix of input_split_sizes[s][:].
 *  recv_offsets[d*(cp+1) + s]    exclusive prefix of output_split_sizes[d][:].
 *  send_identity[s], recv_identity[d]   1 when that rank's rows are 0..S-1.
 *  src_of_dst[q]        the fused permutation over the two global buffers:
 *                       target row q is source row src_of_dst[q].  Equal, row
 *                       for row, to pack -> all-to-all -> scatter.
 */
typedef struct thd_route {
  int32_t cp_size;
  int32_t dir;                 /* thd_dir_t */
  int64_t total_rows;          /* T */
  int32_t *send_rows;          /* [cp][S] */
  int32_t *recv_rows;          /* [cp][S] */
  int32_t *input_split_sizes;  /* [cp][cp] */
  int32_t *output_split_sizes; /* [cp][cp] */
  int32_t *send_offsets;       /* [cp][cp+1] */
  int32_t *recv_offsets;       /* [cp][cp+1] */
  uint8_t *send_identity;      /* [cp] */
  uint8_t *recv_identity;      /* [cp] */
  int32_t *src_of_dst;         /* [T] */
} thd_route_t;

/* Bytes of device memory one direction's route needs (each array 256-byte
 * aligned inside it).  0 when T or cp is out of range. */
size_t thd_route_bytes(int64_t T, int32_t cp);

/* Point `route`'s arrays into the caller's device buffer `d_base`
 * (>= thd_route_bytes(T, cp) bytes, 256-byte aligned) and record T, cp and
 * dir.  Host only: enqueues nothing. */
thd_status_t thd_route_bind(thd_route_t *route, void *d_base, size_t bytes,
                            int64_t T, int32_t cp, thd_dir_t dir);

/*
 * Both directions' routes for the same T and cp in ONE caller buffer of
 * thd_route_pair_bytes(T, cp) bytes (256-byte aligned), sharing the arrays
 * whose contents the two directions have in common: route_c2z->send_rows is
 * route_z2c->recv_rows (the rows each contiguous rank receives from the
 * zigzag ranks are the rows it sends back), and route_c2z->recv_rows is
 * route_z2c->send_rows (0..S-1 on every rank: each rank's zigzag rows ascend
 * in global order).  16 bytes per row for the pair instead of 24, and
 * thd_route_build_pair writes each shared array once.  Every array of both
 * routes stays complete and valid for every other call; building one
 * direction alone into a pair-bound route writes the shared arrays with the
 * same contents.  Host only: enqueues nothing.
 */
size_t thd_route_pair_bytes(int64_t T, int32_t cp);
thd_status_t thd_route_bind_pair(thd_route_t *route_z2c, thd_route_t *route_c2z, void *d_base,
                                 size_t bytes, int64_t T, int32_t cp);

/*
 * Build the route of one direction on the device, with no host
 * synchronisation (Relax PR #273, section 2.1: route from cu_seqlens and
 * cp_size by interval intersection; section 2.3: fail-fast validation).
 * One kernel: every block validates cu (cu[0] == 0, monotone, lengths
 * multiples of 2*cp, cu[num_docs] == T; the failed check of highest priority,
 * in that order, goes to *d_status), then fills the route from closed-form
 * interval counts and a binary search of cu.  Deterministic; no atomics on
 * the route.
 *
 *  cu_seqlens_padded  device int32[num_docs+1]; empty documents (repeated
 *                     boundaries) are allowed.
 *  T                  total rows, 0 <= T < 2^31, a multiple of 2*cp.
 *  cp_size            1 .. THD_MAX_CP.
 *  route              bound with the same T, cp_size and dir.
 *  d_status           device int32[1], required.
 */
thd_status_t thd_route_build(const int32_t *cu_seqlens_padded, int32_t num_docs, int64_t T,
                             int32_t cp_size, thd_dir_t dir, const thd_route_t *route,
                             int32_t *d_status, cudaStream_t stream);

/*
 * Both directions in one launch: route_z2c (bound with THD_ZIGZAG_TO_CONTIGUOUS)
 * and route_c2z (bound with THD_CONTIGUOUS_TO_ZIGZAG) for the same T and
 * cp_size, with the same validation and d_status rules as thd_route_build.
 * The two routes share the interval counts and half of their rows (the c->z
 * send rows are the z->c receive rows), so one pass writes both -- what the
 * pages' prebuild of both directions per microbatch does (Relax PR #273,
 * section 2.4) in one kernel.  A direction mismatch returns
 * THD_ERR_BAD_DIRECTION.
 */
thd_status_t thd_route_build_pair(const int32_t *cu_seqlens_padded, int32_t num_docs, int64_t T,
                                  int32_t cp_size, const thd_route_t *route_z2c,
                                  const thd_route_t *route_c2z, int32_t *d_status,
                                  cudaStream_t stream);

/*
 * Zigzag partition indices ("Packed Sequence 与上下文并行", section 2.4, what
 * its get_slice_index returns): out[k] = global row held in local slot k.
 *  cp_rank >= 0: out is int32[T/cp] for that rank.
 *  cp_rank == -1: out is int32[cp][T/cp], all ranks rank-major.
 * Validation and d_status as for thd_route_build.
 */
thd_status_t thd_partition_indices(const int32_t *cu_seqlens_padded, int32_t num_docs, int64_t T,
                                   int32_t cp_size, int32_t cp_rank, int32_t *out,
                                   int32_t *d_status, cudaStream_t stream);

/*
 * Fused layout swap: dst[q] = src[route->src_of_dst[q]] for q < T, each row
 * `row_bytes` bytes (Relax PR #273, section 2.1: pack -> all-to-all ->
 * scatter, here one pass that reads and writes every row once).
 *  src, dst   device buffers of T*row_bytes bytes that must not overlap.
 *  row_bytes  > 0.  Rows that are a multiple of 16 bytes, with 16-byte
 *             aligned src/dst, move by TMA bulk copies through shared memory
 *             (rows of >= 208 bytes one by one, narrower rows as runs of
 *             consecutive rows); other rows by 4- or 1-byte loads/stores.
 *  d_status   device int32[1] or NULL.  When given, the swap does nothing if
 *             it is non-zero on entry, and records THD_ERR_INDEX_RANGE.
 */
thd_status_t thd_swap(const void *src, void *dst, int64_t row_bytes, const thd_route_t *route,
                      int32_t *d_status, cudaStream_t stream);

/*
 * thd_swap over `outer` independent blocks of T rows that share one route:
 * src and dst are [outer][T][row_bytes] in memory, and for every o < outer
 *   dst[o][q] = src[o][route->src_of_dst[q]].
 * This is the layout conversion of a tensor whose sequence dimension is not
 * the first one -- [outer, T, inner...] contiguous, row = the inner
 * dimensions -- done in place of the movedim + contiguous + swap + movedim
 * that the pages wrap around the conversion (Relax PR #273, section 2.6),
 * with no transposed copy.  outer * T < 2^31; outer == 0 moves nothing.
 * Buffers, row_bytes and d_status follow thd_swap's rules.
 */
thd_status_t thd_swap_batched(const void *src, void *dst, int64_t outer, int64_t row_bytes,
                              const thd_route_t *route, int32_t *d_status, cudaStream_t stream);

/* The three steps the pages run (Relax PR #273, section 2.1), for every
 * virtual rank at once; buffers are [cp][S][row_bytes], must not overlap, and
 * follow thd_swap's rules for row_bytes, alignment and d_status.
 *  thd_pack:      send[s][j] = src[s][send_rows[s][j]]
 *  thd_a2a_local: recv[d][recv_offsets[d][s] + m] = send[s][send_offsets[s][d] + m],
 *                 m < input_split_sizes[s][d]
 *  thd_scatter:   dst[d][recv_rows[d][j]] = recv[d][j]                     */
thd_status_t thd_pack(const void *src, void *send_buf, int64_t row_bytes,
                      const thd_route_t *route, int32_t *d_status, cudaStream_t stream);
thd_status_t thd_a2a_local(const void *send_buf, void *recv_buf, int64_t row_bytes,
                           const thd_route_t *route, int32_t *d_status, cudaStream_t stream);
thd_status_t thd_scatter(const void *recv_buf, void *dst, int64_t row_bytes,
                         const thd_route_t *route, int32_t *d_status, cudaStream_t stream);

/*
 * One rank's pack and scatter, for a caller that holds only its own shard
 * (one context-parallel rank per GPU; Relax PR #273, sections 2.1-2.2: each
 * rank packs its rows into a send buffer grouped by destination, exchanges
 * them with an all-to-all of input/output split sizes, and scatters what it
 * receives).  Every buffer is [S][row_bytes], S = T / cp_size, local to rank
 * cp_rank (0 <= cp_rank < cp_size):
 *  thd_pack_rank:    send_buf[j] = src_shard[send_rows[cp_rank][j]]
 *  thd_scatter_rank: dst_shard[recv_rows[cp_rank][j]] = recv_buf[j]
 * Between them, rank cp_rank sends send_buf rows [send_offsets[cp_rank][d],
 * send_offsets[cp_rank][d+1]) to rank d and receives from rank s into
 * recv_buf rows [recv_offsets[cp_rank][s], recv_offsets[cp_rank][s+1]): the
 * all-to-all's split sizes are input_split_sizes[cp_rank][:] and
 * output_split_sizes[cp_rank][:].  When send_identity[cp_rank]
 * (recv_identity[cp_rank]) is set the pack (scatter) is a plain copy, which a
 * caller that reads the flags may skip by handing over the shard itself
 * ("identity = zero-copy", section 2.2).  The route is the one thd_route_build
 * builds for all ranks from the same boundaries on every GPU.  Buffers,
 * row_bytes and d_status follow thd_swap's rules.
 */
thd_status_t thd_pack_rank(const void *src_shard, void *send_buf, int32_t cp_rank, int64_t row_bytes,
                           const thd_route_t *route, int32_t *d_status, cudaStream_t stream);
thd_status_t thd_scatter_rank(const void *recv_buf, void *dst_shard, int32_t cp_rank, int64_t row_bytes,
                              const thd_route_t *route, int32_t *d_status, cudaStream_t stream);

/*
 * Ulysses sequence <-> head exchange ("Packed Sequence 与上下文并行",
 * section 2.5: Ulysses slices the packed sequence into cp contiguous
 * shards; section 2.7: an all-to-all then gives every rank the whole
 * sequence for a subset of the heads).  Every token row of row_bytes bytes
 * is cp head groups of row_bytes/cp bytes (group r = heads
 * [r*H/cp, (r+1)*H/cp) when the row is [H][...]).
 *   THD_SEQ_TO_HEAD: src = [T][row] (rank r's shard = rows [r*T/cp, (r+1)*T/cp)),
 *                    dst = [cp][T][row/cp]: dst[r][g] = group r of src row g.
 *   THD_HEAD_TO_SEQ: the inverse.
 * With all ranks in one buffer the exchange is a block transpose.
 *  T          0 <= T, a multiple of cp_size, T*cp_size < 2^31.
 *  row_bytes  > 0, a multiple of cp_size.  With 16-byte aligned buffers and
 *             pieces (row_bytes/cp_size) that are multiples of 16 bytes, the
 *             exchange moves by TMA bulk copies: pieces below 1 KiB (cp_size
 *             >= 2) as a tile transpose through shared memory, larger pieces
 *             one by one or as runs; other shapes by 4- or 1-byte loads and stores.
 *  d_status   as for thd_swap.  A bad dir returns THD_ERR_BAD_DIRECTION.
 */
thd_status_t thd_ulysses_swap(const void *src, void *dst, int64_t T, int32_t cp_size,
                              int64_t row_bytes, thd_ulysses_dir_t dir, int32_t *d_status,
                              cudaStream_t stream);

/*
 * Document-bounded labels, MTP targets and the valid-token mask
 * ("Packed Sequence 与上下文并行", sections 1.3, 1.6, 2.2 and 3.8).  For row p
 * of document i, with valid end e_i = cu_p[i] + (cu_v[i+1] - cu_v[i]):
 *   valid_mask[p]        = p < e_i
 *   labels[k*T + p]      = tokens[p+1+k] if p+1+k < e_i else fill
 *   loss_mask[k*T + p]   = p+1+k < e_i                      (k = 0..mtp_depth)
 * so no label or MTP target ever comes from padding or from the next document.
 *  tokens             device int32[T] (packed, padded layout)
 *  cu_seqlens         device int32[num_docs+1], unpadded boundaries
 *  cu_seqlens_padded  device int32[num_docs+1], padded boundaries, last == T
 *  labels             device int32[mtp_depth+1][T]
 *  loss_mask          device uint8[mtp_depth+1][T]
 *  valid_mask         device uint8[T]
 *  next_token, has_next  device int32[num_docs], uint8[num_docs], both NULL or
 *                     both given: when has_next[i], document i continues with
 *                     next_token[i] after its last valid token (a sample's
 *                     extra token, "Packed Sequence 与上下文并行" section 1.3),
 *                     so the target exactly one past e_i is next_token[i]
 *                     (mask 1); thd_pack_docs produces both arrays.
 * Device checks, in order: padded cu (start, monotone, total), unpadded cu
 * (start, monotone), every unpadded length <= its padded length.
 */
thd_status_t thd_roll_labels(const int32_t *tokens, const int32_t *cu_seqlens,
                             const int32_t *cu_seqlens_padded, int32_t num_docs, int64_t T,
                             int32_t mtp_depth, int32_t fill, const int32_t *next_token,
                             const uint8_t *has_next, int32_t *labels, uint8_t *loss_mask,
                             uint8_t *valid_mask, int32_t *d_status, cudaStream_t stream);

/*
 * thd_roll_labels written directly in the zigzag layout of cp_size ranks:
 * position p = r*S + j of the zigzag buffer (S = T/cp_size) holds global row
 * g = the partition index of (r, j), and
 *   labels[k*T + p] = (the thd_roll_labels label of row g at depth k),
 * likewise loss_mask and valid_mask.  The label roll and the zigzag slicing
 * that "Packed Sequence 与上下文并行" section 2.4 applies to tokens, labels,
 * loss mask and valid mask alike, in one pass.  Checks: cp_size and T as for
 * thd_route_build; then the padded boundaries (start, monotone, lengths
 * multiples of 2*cp_size, total), the unpadded ones (start, monotone), and
 * valid lengths <= padded lengths.
 */
thd_status_t thd_roll_labels_zigzag(const int32_t *tokens, const int32_t *cu_seqlens,
                                    const int32_t *cu_seqlens_padded, int32_t num_docs, int64_t T,
                                    int32_t cp_size, int32_t mtp_depth, int32_t fill,
                                    const int32_t *next_token, const uint8_t *has_next,
                                    int32_t *labels, uint8_t *loss_mask, uint8_t *valid_mask,
                                    int32_t *d_status, cudaStream_t stream);

/*
 * Pack raw rows into one padded THD sequence ("Packed Sequence 与上下文并行",
 * section 2.2 and the worked example of section 3).  Row b's valid region is
 * raw[b][0 .. ve_b) where ve_b is one past its last token != raw_pad_id (the
 * whole row when trim_raw_pad == 0).  Inside it every eod_id closes a document
 * and belongs to it; a non-empty tail after the last EOD is a document too;
 * documents never span rows.  A document of length L is written to
 * tokens_out followed by ((-L) mod align) copies of pad_id.
 *
 *  raw                device int32[B][S]
 *  row_next           device int32[B] or NULL: each row's extra token (the
 *                     sample's next token, section 1.3); requires has_next
 *  tokens_out         device int32[tokens_capacity]
 *  cu_seqlens, cu_seqlens_padded   device int32[docs_capacity]
 *  next_token, has_next  device int32/uint8[docs_capacity], or both NULL: per
 *                     document, has_next = 1 and next_token = row_next[b] when
 *                     it is row b's last document, reaches the row's end and
 *                     does not end with EOD; else 0 (for thd_roll_labels)
 *  counts             device int64[2]: {num_docs, T} on completion
 *  workspace          device, >= thd_pack_docs_workspace_bytes(B, S) bytes,
 *                     8-byte aligned; scratch of the call (its contents on
 *                     entry do not matter; calls that may overlap on the GPU
 *                     need separate workspaces).
 *  d_status           device int32[1], required; THD_ERR_CAPACITY when
 *                     num_docs+1 > docs_capacity or T > tokens_capacity: then
 *                     counts holds the sizes needed, nothing is written past
 *                     either capacity and the other outputs are unspecified.
 *                     THD_ERR_TIMEOUT when a bounded wait of the single pass
 *                     (below) ran out (outputs unspecified).
 * From 2^19 raw tokens, with 16-byte aligned raw rows of a multiple of 4
 * tokens, a 16-byte aligned tokens_out and align <= 65536, the call is one
 * persistent kernel that reads every raw token once (6,144-token chunks
 * taken in order; one block turns the chunks' published summaries into each
 * chunk's offsets); otherwise three kernels (statistics, scan, emit).
 * The number of documents and T are only known on the device; a caller that
 * needs them on the host reads `counts` (one synchronisation, at data-prep
 * time).  T <= B*S*align and num_docs <= B*S always hold.
 */
size_t thd_pack_docs_workspace_bytes(int32_t B, int64_t S);
thd_status_t thd_pack_docs(const int32_t *raw, int32_t B, int64_t S, int32_t eod_id,
                           int32_t trim_raw_pad, int32_t raw_pad_id, int32_t align,
                           int32_t pad_id, const int32_t *row_next, int32_t *tokens_out,
                           int64_t tokens_capacity, int32_t *cu_seqlens,
                           int32_t *cu_seqlens_padded, int32_t *next_token, uint8_t *has_next,
                           int64_t docs_capacity, int64_t *counts, void *workspace,
                           size_t workspace_bytes, int32_t *d_status, cudaStream_t stream);

/*
 * thd_pack_docs without a workspace argument, for callers that cannot
 * allocate device memory.  The pages have no counterpart: this is a
 * convenience of this library.
 *
 * Who needs it: callers that are handed only their input and output buffers,
 * e.g. a data-loading plugin whose host framework owns all other device
 * memory through its own pool, or code that must not call cudaMalloc or
 * cudaFree because those calls can synchronise the device and stall work
 * queued on other streams.  The call itself allocates nothing and calls no
 * allocating routine.
 *
 * Arguments, results and errors are those of thd_pack_docs, minus the
 * workspace and the optional extra-token arguments (row_next, next_token,
 * has_next), which this entry point does not take.  The workspace is a fixed array compiled into the library
 * (THD_PACK_NOALLOC_MAX_ROWS rows x 32 bytes = 128 KiB), held by every GPU
 * that loads the library until the process exits:
 *  - B > THD_PACK_NOALLOC_MAX_ROWS returns THD_ERR_SCRATCH_LIMIT at once and
 *    enqueues nothing (use thd_pack_docs with your own workspace then);
 *  - every call looks up the array's device address in the current context
 *    (the address belongs to the context: after cudaDeviceReset, or in
 *    another context on the same device, it differs), which allocates
 *    nothing; the first call in a context may load the library's device
 *    code into it, so make that call before any stream capture;
 *  - above 512 rows a third kernel turns the rows' statistics into prefix
 *    sums in the array between the two packing kernels;
 *  - all calls on a device share the one array, so calls that may overlap on
 *    the GPU (different streams, no ordering between them) race and must be
 *    serialised by the caller.  Calls in order on one stream are safe: each
 *    call rewrites every scratch entry it reads.
 */
#define THD_PACK_NOALLOC_MAX_ROWS 4096
thd_status_t thd_pack_docs_noalloc(const int32_t *raw, int32_t B, int64_t S, int32_t eod_id,
                                   int32_t trim_raw_pad, int32_t raw_pad_id, int32_t align,
                                   int32_t pad_id, int32_t *tokens_out, int64_t tokens_capacity,
                                   int32_t *cu_seqlens, int32_t *cu_seqlens_padded,
                                   int64_t docs_capacity, int64_t *counts, int32_t *d_status,
                                   cudaStream_t stream);

/* Status word helpers.  thd_status_clear enqueues a zero write.
 * thd_status_read copies the word to *host_code and synchronises `stream`:
 * the one call of this library that waits for the GPU. */
thd_status_t thd_status_clear(int32_t *d_status, cudaStream_t stream);
thd_status_t thd_status_read(const int32_t *d_status, int32_t *host_code, cudaStream_t stream);

/* Name of a status code (static string). */
const char *thd_status_string(int32_t code);

/* The cudaError_t of the last failed CUDA call made by this thread inside the
 * library (0 when none). */
int32_t thd_last_cuda_error(void);

/* Library version, major*10000 + minor*100 + patch. */
int32_t thd_version(void);

#ifdef __cplusplus
}
#endif

#endif /* THD_H_ */
