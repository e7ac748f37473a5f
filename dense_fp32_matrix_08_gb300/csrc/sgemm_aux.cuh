// Memory-bound helper kernels of the SGEMM path: the beta-scale quick return and the
// split-K reduction. Both stream their operands once; grids are grid-stride loops sized in
// multiples of the SM count by the host.
#pragma once

#include <cuda_runtime.h>

namespace sgemm {

// C = beta * C over an M x N view (beta == 0 writes zeros without reading C). This is the
// whole computation when alpha == 0 or K == 0 (BLAS quick return: A and B are not read).
__global__ void scale_c_kernel(float *__restrict__ C, long long ldc, int M, int N,
                               float beta, int vec) {
  const long long groups_per_row = (N + 3) / 4;
  const long long total = (long long)M * groups_per_row;
  for (long long g = blockIdx.x * (long long)blockDim.x + threadIdx.x; g < total;
       g += (long long)gridDim.x * blockDim.x) {
    const long long row = g / groups_per_row;
    const int col = (int)(g - row * groups_per_row) * 4;
    float *dst = C + row * ldc + col;
    if (vec && col + 3 < N) {
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (beta != 0.0f) {
        v = *reinterpret_cast<const float4 *>(dst);
        v.x *= beta;
        v.y *= beta;
        v.z *= beta;
        v.w *= beta;
      }
      *reinterpret_cast<float4 *>(dst) = v;
    } else {
      for (int e = 0; e < 4 && col + e < N; ++e) dst[e] = (beta != 0.0f) ? beta * dst[e] : 0.0f;
    }
  }
}

// Split-K finish: C = alpha * sum_{s < splits} ws[s] + beta * C, the slices added in
// ascending s so that results are deterministic. ws is [splits][M][ldw], ldw % 4 == 0.
__global__ void splitk_reduce_kernel(const float *__restrict__ ws, long long ldw, int splits,
                                     int M, int N, float alpha, float beta,
                                     float *__restrict__ C, long long ldc, int vec) {
  const long long groups_per_row = (N + 3) / 4;
  const long long total = (long long)M * groups_per_row;
  const long long slice = (long long)M * ldw;
  for (long long g = blockIdx.x * (long long)blockDim.x + threadIdx.x; g < total;
       g += (long long)gridDim.x * blockDim.x) {
    const long long row = g / groups_per_row;
    const int col = (int)(g - row * groups_per_row) * 4;
    const float *src = ws + row * ldw + col;
    float4 s = *reinterpret_cast<const float4 *>(src);
    for (int k = 1; k < splits; ++k) {
      const float4 t = *reinterpret_cast<const float4 *>(src + k * slice);
      s.x += t.x;
      s.y += t.y;
      s.z += t.z;
      s.w += t.w;
    }
    float *dst = C + row * ldc + col;
    if (vec && col + 3 < N) {
      float4 out;
      if (beta != 0.0f) {
        const float4 old = *reinterpret_cast<const float4 *>(dst);
        out.x = fmaf(alpha, s.x, beta * old.x);
        out.y = fmaf(alpha, s.y, beta * old.y);
        out.z = fmaf(alpha, s.z, beta * old.z);
        out.w = fmaf(alpha, s.w, beta * old.w);
      } else {
        out = make_float4(alpha * s.x, alpha * s.y, alpha * s.z, alpha * s.w);
      }
      *reinterpret_cast<float4 *>(dst) = out;
    } else {
      const float v[4] = {s.x, s.y, s.z, s.w};
      for (int e = 0; e < 4 && col + e < N; ++e)
        dst[e] = (beta != 0.0f) ? fmaf(alpha, v[e], beta * dst[e]) : alpha * v[e];
    }
  }
}

}  // namespace sgemm
