// The BLAS siblings of sgemm named with it in "Lecture 4 - GPU Acceleration", section 5.2
// ("Interface": cublasSdot and cublasSgemv): single-precision matrix-vector product and dot
// product on row-major data. Both stream their operands once from HBM; every reduction is
// done in a fixed order, so results are deterministic.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "../../include/sgemm_f32.h"
#include "sgemm_internal.h"

namespace sgemm {
namespace blas2 {

// Element i of a strided BLAS vector of length n (negative increments walk backwards).
__device__ __forceinline__ long long vidx(long long i, long long n, int inc) {
  return inc > 0 ? i * inc : (n - 1 - i) * (long long)(-inc);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// y = alpha * A x + beta * y, A M x N row-major. One warp per row; lanes stride over the
// row with 16-byte loads when the row and x are contiguous and aligned (vec), else 4-byte.
__global__ void gemv_n_kernel(int M, int N, float alpha, const float *__restrict__ A,
                              long long lda, const float *__restrict__ x, int incx, float beta,
                              float *__restrict__ y, int incy, int vec) {
  const int lane = threadIdx.x & 31;
  const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long row = blockIdx.x * (long long)(blockDim.x >> 5) + (threadIdx.x >> 5);
       row < M; row += warps) {
    const float *a = A + row * lda;
    float s = 0.0f;
    if (vec) {
      const int n4 = N >> 2;
      for (int c = lane; c < n4; c += 32) {
        const float4 av = __ldcs(reinterpret_cast<const float4 *>(a) + c);
        const float4 xv = __ldg(reinterpret_cast<const float4 *>(x) + c);
        s = fmaf(av.x, xv.x, s);
        s = fmaf(av.y, xv.y, s);
        s = fmaf(av.z, xv.z, s);
        s = fmaf(av.w, xv.w, s);
      }
      for (int c = (n4 << 2) + lane; c < N; c += 32) s = fmaf(a[c], __ldg(x + c), s);
    } else {
      for (int c = lane; c < N; c += 32) s = fmaf(a[c], __ldg(x + vidx(c, N, incx)), s);
    }
    s = warp_sum(s);
    if (lane == 0) {
      float *yp = y + vidx(row, M, incy);
      *yp = (beta != 0.0f) ? fmaf(alpha, s, beta * *yp) : alpha * s;
    }
  }
}

// Partial sums of y = A^T x over the row slice [r0, r1): each thread owns 4 consecutive
// columns (16-byte loads of each row when aligned); warps of a block take rows in turn and
// are combined in shared memory in warp order. part[slice][N] (N rounded up to 4).
__global__ void gemv_t_partial_kernel(int M, int N, const float *__restrict__ A, long long lda,
                                      const float *__restrict__ x, int incx, int rows_per_slice,
                                      float *__restrict__ part, long long ldp, int vec) {
  __shared__ float4 red[8][32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = (blockIdx.x * 32 + lane) * 4;  // first of this lane's 4 columns
  const int r0 = blockIdx.y * rows_per_slice;
  const int r1 = min(M, r0 + rows_per_slice);
  float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
  if (c < N) {
    for (int r = r0 + warp; r < r1; r += 8) {
      const float xv = __ldg(x + vidx(r, M, incx));
      const float *a = A + (long long)r * lda + c;
      if (vec && c + 3 < N) {
        const float4 av = __ldcs(reinterpret_cast<const float4 *>(a));
        s.x = fmaf(av.x, xv, s.x);
        s.y = fmaf(av.y, xv, s.y);
        s.z = fmaf(av.z, xv, s.z);
        s.w = fmaf(av.w, xv, s.w);
      } else {
        s.x = fmaf(a[0], xv, s.x);
        if (c + 1 < N) s.y = fmaf(a[1], xv, s.y);
        if (c + 2 < N) s.z = fmaf(a[2], xv, s.z);
        if (c + 3 < N) s.w = fmaf(a[3], xv, s.w);
      }
    }
  }
  red[warp][lane] = s;
  __syncthreads();
  if (warp == 0 && c < N) {
    float4 t = red[0][lane];
    for (int w = 1; w < 8; ++w) {
      t.x += red[w][lane].x;
      t.y += red[w][lane].y;
      t.z += red[w][lane].z;
      t.w += red[w][lane].w;
    }
    *reinterpret_cast<float4 *>(part + blockIdx.y * ldp + c) = t;
  }
}

// y = alpha * sum_slice part[slice] + beta * y, slices in ascending order.
__global__ void gemv_t_finish_kernel(int N, int slices, const float *__restrict__ part,
                                     long long ldp, float alpha, float beta,
                                     float *__restrict__ y, int incy) {
  for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < N; j += gridDim.x * blockDim.x) {
    float s = 0.0f;
    for (int q = 0; q < slices; ++q) s += part[q * ldp + j];
    float *yp = y + vidx(j, N, incy);
    *yp = (beta != 0.0f) ? fmaf(alpha, s, beta * *yp) : alpha * s;
  }
}

// Dot product, first pass: block b reduces its grid-stride share into part[b].
__global__ void dot_partial_kernel(long long n, const float *__restrict__ x, int incx,
                                   const float *__restrict__ y, int incy,
                                   float *__restrict__ part, int vec) {
  __shared__ float red[32];
  float s = 0.0f;
  const long long tid = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  const long long stride = (long long)gridDim.x * blockDim.x;
  if (vec) {
    const long long n4 = n >> 2;
    for (long long i = tid; i < n4; i += stride) {
      const float4 a = __ldcs(reinterpret_cast<const float4 *>(x) + i);
      const float4 b = __ldcs(reinterpret_cast<const float4 *>(y) + i);
      s = fmaf(a.x, b.x, s);
      s = fmaf(a.y, b.y, s);
      s = fmaf(a.z, b.z, s);
      s = fmaf(a.w, b.w, s);
    }
    for (long long i = (n4 << 2) + tid; i < n; i += stride) s = fmaf(x[i], y[i], s);
  } else {
    for (long long i = tid; i < n; i += stride) s = fmaf(x[vidx(i, n, incx)], y[vidx(i, n, incy)], s);
  }
  s = warp_sum(s);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
  __syncthreads();
  if (threadIdx.x < 32) {
    float t = (threadIdx.x < (blockDim.x >> 5)) ? red[threadIdx.x] : 0.0f;
    t = warp_sum(t);
    if (threadIdx.x == 0) part[blockIdx.x] = t;
  }
}

// Second pass: one block adds the partials in a fixed tree order.
__global__ void dot_finish_kernel(int nparts, const float *__restrict__ part,
                                  float *__restrict__ result) {
  __shared__ float red[32];
  float s = 0.0f;
  for (int i = threadIdx.x; i < nparts; i += blockDim.x) s += part[i];
  s = warp_sum(s);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
  __syncthreads();
  if (threadIdx.x < 32) {
    float t = (threadIdx.x < (blockDim.x >> 5)) ? red[threadIdx.x] : 0.0f;
    t = warp_sum(t);
    if (threadIdx.x == 0) *result = t;
  }
}

static inline bool aligned16(const void *p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

}  // namespace blas2
}  // namespace sgemm

using namespace sgemm;

extern "C" int sgemv_f32(int trans, int M, int N, float alpha, const float *A, int lda,
                         const float *x, int incx, float beta, float *y, int incy,
                         cudaStream_t stream) {
  if (trans != 0 && trans != 1) return -1;
  if (M < 0) return -2;
  if (N < 0) return -3;
  const int ylen = trans ? N : M, xlen = trans ? M : N;
  const bool reads_ax = ylen > 0 && xlen > 0 && alpha != 0.0f;
  if (reads_ax && A == nullptr) return -5;
  if (lda < std::max(1, N)) return -6;
  if (reads_ax && x == nullptr) return -7;
  if (incx == 0) return -8;
  if (ylen > 0 && y == nullptr) return -10;
  if (incy == 0) return -11;
  if (ylen == 0) return 0;
  int num_sms = 0;
  cudaError_t e = device_setup(&num_sms);
  if (e != cudaSuccess) return (int)e;
  if (!reads_ax) {  // y = beta * y: reuse the GEMM quick return on a 1 x ylen (strided) view
    if (incy > 0) return sgemm_f32(ylen, 1, 0, 0.0f, nullptr, 1, nullptr, 1, beta, y, incy,
                                   stream);
    return sgemm_f32(ylen, 1, 0, 0.0f, nullptr, 1, nullptr, 1, beta, y, -incy, stream);
  }
  if (!trans) {
    const bool vec = incx == 1 && lda % 4 == 0 && blas2::aligned16(A) && blas2::aligned16(x);
    const long long warps_needed = M;
    const int blocks = (int)std::max<long long>(
        1, std::min<long long>((warps_needed + 7) / 8, (long long)num_sms * 16));
    blas2::gemv_n_kernel<<<blocks, 256, 0, stream>>>(M, N, alpha, A, lda, x, incx, beta, y,
                                                     incy, vec ? 1 : 0);
    return (int)cudaGetLastError();
  }
  // y = A^T x: column blocks of 128 x row slices, then a fixed-order finish
  const bool vec = lda % 4 == 0 && blas2::aligned16(A);
  const long long col_blocks = (N + 127) / 128;
  long long slices = std::max<long long>(1, (2LL * num_sms * 4 + col_blocks - 1) / col_blocks);
  slices = std::min<long long>(slices, std::max(1, M / 32));
  slices = std::min<long long>(slices, 65535);
  const int rows_per_slice = (int)((M + slices - 1) / slices);
  slices = (M + rows_per_slice - 1) / rows_per_slice;
  const long long ldp = (N + 3) / 4 * 4;
  float *part = nullptr;
  e = cudaMallocFromPoolAsync(reinterpret_cast<void **>(&part),
                              (size_t)slices * ldp * sizeof(float), workspace_pool(), stream);
  if (e != cudaSuccess) return (int)e;
  dim3 grid((unsigned)col_blocks, (unsigned)slices);
  blas2::gemv_t_partial_kernel<<<grid, 256, 0, stream>>>(M, N, A, lda, x, incx, rows_per_slice,
                                                         part, ldp, vec ? 1 : 0);
  e = cudaGetLastError();
  if (e == cudaSuccess) {
    const int blocks = (int)std::max<long long>(1, std::min<long long>((N + 255) / 256,
                                                                        (long long)num_sms * 8));
    blas2::gemv_t_finish_kernel<<<blocks, 256, 0, stream>>>(N, (int)slices, part, ldp, alpha,
                                                            beta, y, incy);
    e = cudaGetLastError();
  }
  const cudaError_t ef = cudaFreeAsync(part, stream);
  return (int)(e != cudaSuccess ? e : ef);
}

extern "C" int sdot_f32(int n, const float *x, int incx, const float *y, int incy,
                        float *result, cudaStream_t stream) {
  if (n < 0) return -1;
  if (n > 0 && x == nullptr) return -2;
  if (incx == 0) return -3;
  if (n > 0 && y == nullptr) return -4;
  if (incy == 0) return -5;
  if (result == nullptr) return -6;
  int num_sms = 0;
  cudaError_t e = device_setup(&num_sms);
  if (e != cudaSuccess) return (int)e;
  if (n == 0) return (int)cudaMemsetAsync(result, 0, sizeof(float), stream);
  const bool vec = incx == 1 && incy == 1 && blas2::aligned16(x) && blas2::aligned16(y);
  const int blocks = (int)std::max<long long>(
      1, std::min<long long>(((long long)n + 1023) / 1024, (long long)num_sms * 4));
  float *part = nullptr;
  e = cudaMallocFromPoolAsync(reinterpret_cast<void **>(&part), (size_t)blocks * sizeof(float),
                              workspace_pool(), stream);
  if (e != cudaSuccess) return (int)e;
  blas2::dot_partial_kernel<<<blocks, 256, 0, stream>>>(n, x, incx, y, incy, part, vec ? 1 : 0);
  e = cudaGetLastError();
  if (e == cudaSuccess) {
    blas2::dot_finish_kernel<<<1, 1024, 0, stream>>>(blocks, part, result);
    e = cudaGetLastError();
  }
  const cudaError_t ef = cudaFreeAsync(part, stream);
  return (int)(e != cudaSuccess ? e : ef);
}
