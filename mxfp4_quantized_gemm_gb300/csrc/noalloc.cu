// mxfp4_gemm_noalloc: the W4A4 GEMM without a caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they run the
// linear layer: code executing inside CUDA stream capture (allocation there
// either breaks the capture or is forbidden by the surrounding framework),
// serving loops that must never hit cudaMalloc's implicit synchronisation,
// and host applications whose memory is owned by a foreign allocator that
// this library cannot reach.  For them, the scratch that mxfp4_gemm needs
// (quantized activation codes and scales, stream-K partial sums) lives in one
// file-scope device array of fixed size instead.
//
// The array is reserved on every GPU where this library's module is loaded
// (with eager module loading that is every device the process initialises,
// even if this entry point is never called) and stays until the process
// exits.  Its address is looked up once per device (on that device's first
// call) and handed to the existing GEMM path; nothing here allocates or
// frees memory.  The cached address belongs to the device's primary
// context: resetting the device (cudaDeviceReset) while the library is in
// use is not supported.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "internal.h"
#include "mxfp4.h"

namespace mx {

// Upper bound of the scratch a call may use.
constexpr size_t kNoAllocScratchBytes = static_cast<size_t>(48) << 20;   // 48 MiB

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

static std::atomic<void*> g_noalloc_ptr[64];   // device address of the array, per device
static std::mutex g_noalloc_mutex;

// Device address of the scratch array on the current device (looked up once
// per device, under a lock; later calls take the published address without
// it), or nullptr on failure.
static void* noalloc_scratch(int device) {
  void* p = g_noalloc_ptr[device].load(std::memory_order_acquire);
  if (p != nullptr) return p;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  p = g_noalloc_ptr[device].load(std::memory_order_relaxed);
  if (p == nullptr) {
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return nullptr;
    g_noalloc_ptr[device].store(p, std::memory_order_release);
  }
  return p;
}

}  // namespace mx

extern "C" size_t mxfp4_gemm_noalloc_max_scratch_bytes(void) { return mx::kNoAllocScratchBytes; }

extern "C" mxfp4_status mxfp4_gemm_noalloc(const void* a_bf16, int lda, const void* w_packed, const void* bias,
                                           void* out, int ldo, int M, int N, int K, void* stream) {
  if (a_bf16 == nullptr || w_packed == nullptr || out == nullptr) return MXFP4_ERR_INVALID_ARG;
  if (M <= 0 || N <= 0 || K <= 0) return MXFP4_ERR_INVALID_ARG;
  const size_t need = mxfp4_gemm_workspace_bytes(M, N, K);
  if (need == 0) return MXFP4_ERR_UNSUPPORTED_SHAPE;
  if (need > mx::kNoAllocScratchBytes) return MXFP4_ERR_WORKSPACE;   // problem too large for the static scratch
  mx::DeviceInfo dev;
  if (mx::current_device_info(&dev) != cudaSuccess || !dev.ok) return MXFP4_ERR_NO_DEVICE;
  void* scratch = mx::noalloc_scratch(dev.device);
  if (scratch == nullptr) return MXFP4_ERR_CUDA;
  return mxfp4_gemm(a_bf16, lda, nullptr, nullptr, MXFP4_LAYOUT_ROWMAJOR, w_packed, bias, out, ldo, M, N, K, scratch,
                    mx::kNoAllocScratchBytes, stream);
}
