// thd_pack_docs_noalloc: document packing for callers that cannot allocate
// device memory.
//
// thd_pack_docs needs a workspace between its kernels and asks the caller
// for it.  Some callers have no way to provide
// one: a data-loading plugin, for instance, that its host framework hands only
// the input and output buffers while the framework's own pool owns every
// other byte of device memory, or code that must stay away from
// cudaMalloc/cudaFree because those calls can synchronise the device and
// stall work queued on other streams.  This entry point packs with the
// one-block-per-row kernels, whose workspace is small and fixed per row (4
// int64), taken from an array compiled into the library instead.
//
// The array: kNoAllocMaxRows rows x 4 int64 = 128 KiB, a static __device__
// variable of this translation unit.  Every GPU that loads the library holds
// its own copy until the process exits.  Host code cannot use the array's
// name as a device address (in host code it names a host-side stand-in), so
// every call looks the device address up with cudaGetSymbolAddress, with the
// caller's device current.  The address belongs to the CUDA context, not to
// the device number: a context created after cudaDeviceReset, or another
// context on the same device, has its own copy of the array at its own
// address, so nothing is cached between calls.  The lookup allocates
// nothing.  The first call in a context may load the library's device code
// into it (lazy module loading), so make that call before any stream capture.
#include "thd_internal.cuh"

namespace thd {
namespace {

constexpr int32_t kNoAllocMaxRows = THD_PACK_NOALLOC_MAX_ROWS;

// Scratch shared by every call in a context.  No entry needs to start at
// zero: each call's first kernel writes all four entries of every row the
// later kernels read, so nothing is carried over from the previous call.
static __device__ __align__(256) int64_t g_pack_scratch[kNoAllocMaxRows * 4];

// Device address of g_pack_scratch in the current context.
cudaError_t scratch_for_current_context(int64_t** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_pack_scratch);
  if (e != cudaSuccess) return e;
  *out = static_cast<int64_t*>(p);
  return cudaSuccess;
}

}  // namespace
}  // namespace thd

using namespace thd;

extern "C" thd_status_t thd_pack_docs_noalloc(const int32_t* raw, int32_t B, int64_t S, int32_t eod_id,
                                              int32_t trim_raw_pad, int32_t raw_pad_id, int32_t align,
                                              int32_t pad_id, int32_t* tokens_out, int64_t tokens_capacity,
                                              int32_t* cu_seqlens, int32_t* cu_seqlens_padded,
                                              int64_t docs_capacity, int64_t* counts, int32_t* d_status,
                                              cudaStream_t stream) {
  if (B > kNoAllocMaxRows) return THD_ERR_SCRATCH_LIMIT;
  if (B < 0 || S < 0 || S > INT32_MAX || align < 1 || tokens_capacity < 0 || docs_capacity < 1 ||
      !cu_seqlens || !cu_seqlens_padded || !counts || !d_status)
    return THD_ERR_INVALID_ARG;
  if (B > 0 && S > 0 && (!raw || !tokens_out)) return THD_ERR_INVALID_ARG;
  int64_t* scratch = nullptr;
  cudaError_t e = scratch_for_current_context(&scratch);
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return THD_ERR_CUDA;
  }
  return launch_pack_docs_rows(raw, B, S, eod_id, trim_raw_pad ? 1 : 0, raw_pad_id, align, pad_id, tokens_out,
                               tokens_capacity, cu_seqlens, cu_seqlens_padded, docs_capacity, counts, scratch,
                               d_status, stream);
}
