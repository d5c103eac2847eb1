/*
 * Debug entry points of libthd_checked.so, the debug build of libthd
 * (compiled with THD_CHECKED=1; the default libthd.so does not export them).
 * The pages have no counterpart: these exist to test the library's own
 * failure handling without faulting the GPU.
 */
#ifndef THD_DEBUG_H
#define THD_DEBUG_H

#include "thd.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * One-shot: block 0 of the next TMA bulk copy launched by the library (a
 * thd_swap / pack / scatter of rows that are multiples of 16 bytes, or a Ulysses
 * exchange of pieces of 1 KiB or more) waits on 16 bytes that no copy
 * delivers.  Its bounded wait runs out (about 3 s), the block lets its other
 * copies land, records THD_ERR_TIMEOUT in the call's d_status and returns;
 * the rest of the copy completes normally and the context stays usable.
 *  stream   the request is written to device memory in stream order.
 * Returns THD_OK, or THD_ERR_CUDA (detail in thd_last_cuda_error()).
 */
thd_status_t thd_debug_stall_next_bulk_copy(cudaStream_t stream);

/*
 * The same one-shot request for the Ulysses tile transpose (thd_ulysses_swap
 * with head-group pieces of 16 B - 1008 B in steps of 16): block 0 of the
 * next tile kernel waits on its first buffer for 16 bytes that never come;
 * its waits give up (about 3 s each), the block lets its other copies land,
 * records THD_ERR_TIMEOUT and returns.
 */
thd_status_t thd_debug_stall_next_ulysses_tile(cudaStream_t stream);

/*
 * One-shot, for thd_pack_docs on the single-pass path (from 2^19 raw tokens,
 * 16-byte aligned rows of a multiple of 4 tokens and a 16-byte aligned
 * output): the block that takes chunk 0 of the next such call publishes no
 * summary, so the waits for it (the scanner's, and through it every block's
 * wait for its chunk's carries) run out after about a second each; the call
 * records THD_ERR_TIMEOUT, writes no output that depends on the missing
 * summary and completes, and the context stays usable.
 */
thd_status_t thd_debug_stall_next_pack(cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* THD_DEBUG_H */
