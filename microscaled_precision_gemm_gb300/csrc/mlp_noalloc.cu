// mx_mlp_noalloc: the MLP block for callers that cannot allocate device memory.
//
// mx_mlp needs scratch space for the MXFP6 activations and the MXFP6
// intermediate. Some callers cannot provide it: code hosted inside a runtime
// whose allocator owns all device memory (it must not call cudaMalloc behind the
// runtime's back), callers with a fixed device-memory budget decided at start-up,
// and paths that cannot afford cudaMalloc's implicit synchronization. For them
// this file holds the scratch in a static device array, present on every GPU
// that loads the library until the process exits, and runs the same three
// kernels as mx_mlp through it. No device memory is allocated per call.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "internal.h"
#include "mx.h"

namespace {

constexpr size_t kScratchBytes = MX_MLP_NOALLOC_WORKSPACE_BYTES;
constexpr int kMaxDevices = 64;

// The scratch itself. Host code must not pass this name to a kernel: on the host
// it is only a stand-in, so its device address is looked up once per device.
static __device__ __align__(256) uint8_t g_mlp_scratch[kScratchBytes];

std::mutex g_scratch_lock;

// The array's device address per device, with the ID of the context it was looked
// up in: after cudaDeviceReset the device's new primary context may hold the array
// elsewhere, so a changed context ID means looking it up again.
struct ScratchEntry {
  bool cached;
  unsigned long long context;
  void* addr;
};
ScratchEntry g_scratch[kMaxDevices] = {};

// Device address of g_mlp_scratch in the current device's current context.
mx_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MX_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MX_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> guard(g_scratch_lock);
  ScratchEntry& e = g_scratch[dev];
  unsigned long long ctx = 0;
  if (!(e.cached && mxk::current_context_id(&ctx) && ctx == e.context)) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_mlp_scratch) != cudaSuccess || p == nullptr) return MX_ERR_CUDA;
    // the lookup has made the device's context current; without a readable
    // context ID the address is not cached and every call looks it up
    e.cached = mxk::current_context_id(&e.context);
    e.addr = p;
  }
  *out = e.addr;
  return MX_OK;
}

}  // namespace

extern "C" mx_status mx_mlp_noalloc(const void* x, int64_t M, int64_t d, int64_t ff, const void* w1_codes,
                                    const void* w1_scales, const void* b1, const void* w2_codes,
                                    const void* w2_scales, const void* b2, void* y, cudaStream_t stream) {
  // the shape rules of mx_mlp first, so both entry points answer a bad shape alike
  mx_status st = mxk::mlp_check_shape(M, d, ff, false);
  if (st != MX_OK) return st;
  if (M == 0) return MX_OK;
  // sizes beyond the static scratch are refused before anything is launched (the
  // shape check above bounds every size, so this arithmetic cannot overflow); when
  // the scratch also holds the split-tail region, mx_mlp uses it
  if (mxk::mlp_min_workspace_bytes(M, d, ff) > kScratchBytes) return MX_ERR_WORKSPACE_TOO_SMALL;
  if (x == nullptr || w1_codes == nullptr || w1_scales == nullptr || w2_codes == nullptr || w2_scales == nullptr ||
      y == nullptr)
    return MX_ERR_INVALID_ARG;
  void* scratch = nullptr;
  st = scratch_address(&scratch);
  if (st != MX_OK) return st;
  return mx_mlp(x, M, d, ff, w1_codes, w1_scales, b1, w2_codes, w2_scales, b2, y, scratch, kScratchBytes, stream);
}
