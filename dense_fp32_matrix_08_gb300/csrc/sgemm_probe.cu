// FP32 pipe probe (sgemm_f32_fma_probe): the measured counterpart of the FP32 roofline.
//
// The GEMM kernels are bound by the FP32 FMA pipe. Its derived peak is SMs x 128 FP32 lanes
// x 2 FLOP x SM clock. This kernel measures what the pipe actually sustains on the GPU it
// runs on: every thread runs independent chains of packed multiply-adds (fma.rn.f32x2, the
// instruction of the GEMM inner loops) on registers only, with enough chains and warps that
// neither dependency latency nor issue limits the rate.
//
// Both multiplicands are register pairs holding one value twice ({x, x}, {y, y}). Measured
// on GB300 at 2070 MHz, that form sustains 80.3 TFLOP/s, the derived peak; with two
// different values in each multiplicand pair the same loop sustains 70.9 (about 12% less:
// the instruction then reads three full 64-bit register pairs). The GEMM inner loop reads
// one broadcast pair (A) and one pair of two B values per instruction.
#include <cmath>
#include <cstdint>
#include <vector>
#include <algorithm>
#include <cuda_runtime.h>

#include "sgemm_f32.h"
#include "sgemm_ffma.cuh"

namespace {
using sgemm::ffma2;
using sgemm::pack2;
using sgemm::unpack2;

constexpr int kProbeThreads = 256;
constexpr int kProbeBlocksPerSm = 8;  // 2048 threads, 16 warps per SM partition
constexpr int kProbeChains = 8;       // independent register pairs per thread

// Each thread: kProbeChains accumulator pairs, each advanced `iters` times by
// acc += x * y (two FP32 FMAs per instruction). x and y depend on the thread index, so
// nothing folds at compile time. The sum is stored only if it equals `never` (the host
// passes NaN, which equals nothing), which keeps every FMA observable without a store per
// thread.
__global__ void __launch_bounds__(kProbeThreads, kProbeBlocksPerSm)
    fma_probe_kernel(int iters, float never, float *sink) {
  const float t = (float)threadIdx.x * 1.0e-6f;
  const unsigned long long x = pack2(1.0e-3f + t, 1.0e-3f + t);
  const unsigned long long y = pack2(1.0f - t, 1.0f - t);
  unsigned long long acc[kProbeChains];
#pragma unroll
  for (int c = 0; c < kProbeChains; ++c) acc[c] = pack2((float)c, -(float)c);
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int c = 0; c < kProbeChains; ++c) ffma2(acc[c], x, y);
  }
  float s = 0.0f;
#pragma unroll
  for (int c = 0; c < kProbeChains; ++c) {
    const float2 v = unpack2(acc[c]);
    s += v.x + v.y;
  }
  if (s == never) *sink = s;
}

}  // namespace

int sgemm_f32_fma_probe(int iters, int reps, double *tflops, float *ms_per_launch) {
  if (tflops) *tflops = 0.0;
  if (ms_per_launch) *ms_per_launch = 0.0f;
  if (iters < 1 || iters > (1 << 24)) return -1;
  if (reps < 1 || reps > 100) return -2;
  if (tflops == nullptr) return -3;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return (int)e;
  float *sink = nullptr;
  e = cudaMalloc(reinterpret_cast<void **>(&sink), sizeof(float));
  if (e != cudaSuccess) return (int)e;
  cudaStream_t s = nullptr;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  e = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaEventCreate(&e0);
  if (e == cudaSuccess) e = cudaEventCreate(&e1);
  const int grid = sms * kProbeBlocksPerSm;
  const float never = std::nanf("");
  std::vector<float> times;
  for (int r = -1; r < reps && e == cudaSuccess; ++r) {  // r = -1: warm-up, not timed
    e = cudaEventRecord(e0, s);
    if (e == cudaSuccess) {
      fma_probe_kernel<<<grid, kProbeThreads, 0, s>>>(iters, never, sink);
      e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = cudaEventRecord(e1, s);
    if (e == cudaSuccess) e = cudaEventSynchronize(e1);
    float ms = 0.0f;
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
    if (e == cudaSuccess && r >= 0) times.push_back(ms);
  }
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  if (s) cudaStreamDestroy(s);
  cudaFree(sink);
  if (e != cudaSuccess) return (int)e;
  std::sort(times.begin(), times.end());
  const float med = times[times.size() / 2];
  // 2 FLOP per multiply-add, 2 multiply-adds per fma.rn.f32x2
  const double flops = (double)grid * kProbeThreads * iters * kProbeChains * 4.0;
  *tflops = med > 0.0f ? flops / (med * 1.0e-3) / 1.0e12 : 0.0;
  if (ms_per_launch) *ms_per_launch = med;
  return 0;
}
