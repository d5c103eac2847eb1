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
// the device address is looked up once per device with cudaGetSymbolAddress,
// with that device current, on the first call made on that device.
#include <mutex>

#include "thd_internal.cuh"

namespace thd {
namespace {

constexpr int32_t kNoAllocMaxRows = THD_PACK_NOALLOC_MAX_ROWS;
constexpr int kMaxDevices = 64;

// Scratch shared by every call on a device.  No entry needs to start at
// zero: each call's first kernel writes all four entries of every row its
// second kernel reads, so nothing is carried over from the previous call.
static __device__ __align__(256) int64_t g_pack_scratch[kNoAllocMaxRows * 4];

std::mutex g_scratch_mutex;
int64_t* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_pack_scratch on the current device (looked up once).
cudaError_t scratch_for_current_device(int64_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_pack_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = static_cast<int64_t*>(p);
  }
  *out = g_scratch_ptr[dev];
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
  cudaError_t e = scratch_for_current_device(&scratch);
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return THD_ERR_CUDA;
  }
  return launch_pack_docs_rows(raw, B, S, eod_id, trim_raw_pad ? 1 : 0, raw_pad_id, align, pad_id, tokens_out,
                               tokens_capacity, cu_seqlens, cu_seqlens_padded, docs_capacity, counts, scratch,
                               d_status, stream);
}
