// noalloc.cu -- cross entropy on given logits for callers that cannot
// allocate device memory.
//
// Some callers cannot call cudaMalloc or an allocating library routine at
// the point where they need the loss: code that runs inside a caching
// allocator's own hooks (allocating there would re-enter the allocator), or
// an embedded runtime that reserves a fixed memory budget at start-up and
// hands the kernels only the input and output buffers it owns. For them
// this entry point runs the same kernels as
// lce_cross_entropy_from_logits, with the workspace (status word,
// valid-target count and one fp32 loss per row) taken from a fixed array
// that lives in this library's device image instead of a caller buffer.
//
// The array is reserved on every GPU that loads the library's device code
// and stays there until the process exits: 256 bytes plus 4 bytes per row
// for at most LCE_NOALLOC_MAX_ROWS rows (4 MiB + 256 B). CUDA loads device
// code lazily by default, so that reservation may happen at the first call
// on a device (its address look-up below); a caller with a fixed memory
// budget makes that first call outside its no-allocation region, e.g. at
// start-up. The address is cached per device for the life of the process:
// resetting a device (cudaDeviceReset, or a reset of the primary context)
// while the library is loaded is not supported by this entry point.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/lce.h"
#include "common.cuh"

namespace {

constexpr int64_t kMaxRows = LCE_NOALLOC_MAX_ROWS;
constexpr size_t kScratchBytes = 256 + static_cast<size_t>(kMaxRows) * 4;

// The scratch array. In host code its name is only a host-side stand-in;
// the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {nullptr};
std::mutex g_mu;

// Device address of the array on the current device, looked up once per
// device (with that device current) and cached. The first call on a device
// does this look-up, which may also load the module and reserve the array,
// so that first call should come before any stream capture on that device
// and before any region where the caller cannot let memory be reserved.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return LCE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return LCE_ERR_CUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return LCE_OK;
}

}  // namespace

extern "C" int lce_cross_entropy_from_logits_noalloc(void* logits_inout, const int64_t* target, int64_t N,
                                                     int64_t V, int dtype, int reduction, int64_t ignore_index,
                                                     const float* grad_out, float* loss_out, int* device_status,
                                                     void* stream) {
  if (N > kMaxRows) return LCE_ERR_SHAPE;
  void* scratch = nullptr;
  const int st = scratch_address(&scratch);
  if (st != LCE_OK) return st;
  const int rc = lce_cross_entropy_from_logits(logits_inout, target, N, V, dtype, reduction, ignore_index,
                                               grad_out, loss_out, scratch, kScratchBytes, stream);
  if (rc != LCE_OK || device_status == nullptr) return rc;
  // the status word is the first int of the scratch header
  if (cudaMemcpyAsync(device_status, scratch, sizeof(int), cudaMemcpyDeviceToDevice,
                      static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return LCE_ERR_CUDA;
  return LCE_OK;
}
