// sgemm_f32_noalloc: the same computation as sgemm_f32 for callers that must not allocate
// device memory. Its split-K workspace is a fixed array in device global memory that this
// library owns (every GPU that loads the library holds it until the process exits),
// instead of memory from cudaMallocAsync.
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "../../include/sgemm_f32.h"

namespace {

constexpr size_t kScratchBytes = SGEMM_F32_NOALLOC_SCRATCH_BYTES;
static_assert(kScratchBytes % 256 == 0, "scratch size must keep 256-byte granularity");

// The shared scratch. Host code must not pass `g_scratch` itself to a kernel: on the host
// that name is only a stand-in for the device variable, not its device address. The device
// address is looked up once per device with cudaGetSymbolAddress below.
static __device__ __align__(256) float g_scratch[kScratchBytes / sizeof(float)];

constexpr int kMaxDevices = 64;
struct ScratchSlot {
  std::mutex mu;
  std::atomic<void *> ptr{nullptr};  // set once a lookup has succeeded
};
ScratchSlot g_slots[kMaxDevices];

// Device address of g_scratch on the current device, looked up (with that device current)
// by the first call on the device that succeeds. A failed lookup, for example one made while
// a stream capture forbids it, is not remembered: the next call tries again.
cudaError_t scratch_on_current_device(void **ptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  ScratchSlot &slot = g_slots[dev];
  void *p = slot.ptr.load(std::memory_order_acquire);
  if (p == nullptr) {
    std::lock_guard<std::mutex> lock(slot.mu);
    p = slot.ptr.load(std::memory_order_relaxed);
    if (p == nullptr) {
      e = cudaGetSymbolAddress(&p, g_scratch);
      if (e != cudaSuccess) return e;
      if (p == nullptr) return cudaErrorInvalidSymbol;
      slot.ptr.store(p, std::memory_order_release);
    }
  }
  *ptr = p;
  return cudaSuccess;
}

}  // namespace

extern "C" int sgemm_f32_noalloc(int M, int N, int K, float alpha, const float *A, int lda,
                                 const float *B, int ldb, float beta, float *C, int ldc,
                                 cudaStream_t stream) {
  void *scratch = nullptr;
  const cudaError_t e = scratch_on_current_device(&scratch);
  if (e != cudaSuccess) return (int)e;
  // The caller-workspace entry point plans exactly as sgemm_f32 does and allocates
  // nothing. It writes every partial tile in full before the reduce reads it, so nothing
  // in the scratch has to start at zero and stale contents from an earlier call are
  // harmless.
  const int rc = sgemm_f32_ws(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, scratch,
                              kScratchBytes, stream);
  // -13 here can only mean "the plan needs more scratch than the fixed array holds"
  // (the pointer is non-null and 256-byte aligned); nothing was launched.
  return rc == -13 ? SGEMM_F32_ERR_SCRATCH_TOO_SMALL : rc;
}
