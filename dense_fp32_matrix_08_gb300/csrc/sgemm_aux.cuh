// Memory-bound helper kernels of the SGEMM path: the beta-scale quick return and the
// split-K reduction. Both stream their operands once; grids are grid-stride loops sized in
// multiples of the SM count by the host.
#pragma once

#include <cuda_runtime.h>

#include "sgemm_ffma.cuh"

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

// dst (rows x ldd floats, ldd % 4 == 0, 16-byte aligned) = src (rows x cols, row stride
// ld, any alignment): the aligned copy that lets the TMA-fed kernel read an operand whose
// leading dimension or address TMA cannot take. A thread copies 4-column groups of a row
// (scalar reads, one 128-bit write each), four groups per round with all 16 reads issued
// before the writes, so that enough bytes are in flight to run at HBM speed; a row's last
// group is zero-padded up to ldd.
__global__ void pack_rows_kernel(const float *__restrict__ src, long long ld, int rows,
                                 int cols, float *__restrict__ dst, long long ldd) {
  constexpr int U = 4;
  const long long quads = (cols + 3) / 4;
  const long long total = (long long)rows * quads;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long g0 = blockIdx.x * (long long)blockDim.x + threadIdx.x; g0 < total;
       g0 += U * stride) {
    float4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const long long g = g0 + u * stride;
      v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (g < total) {
        const long long r = g / quads;
        const int c = (int)(g - r * quads) * 4;
        const float *s = src + r * ld + c;
        v[u].x = s[0];
        v[u].y = c + 1 < cols ? s[1] : 0.0f;
        v[u].z = c + 2 < cols ? s[2] : 0.0f;
        v[u].w = c + 3 < cols ? s[3] : 0.0f;
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const long long g = g0 + u * stride;
      if (g < total) {
        const long long r = g / quads;
        const int c = (int)(g - r * quads) * 4;
        *reinterpret_cast<float4 *>(dst + r * ldd + c) = v[u];
      }
    }
  }
}

// Split-K finish for the tiles the GEMM kernel computed in K slices (CTA main_tiles + u
// wrote slice u % split of tile main_tiles + u / split to ws[u], a BM x BN row-major
// partial tile): C = alpha * sum_s partial_s + beta * C, slices added in ascending order
// so that results are deterministic. One thread handles 4 consecutive columns of a row.
__global__ void tail_reduce_kernel(const float *__restrict__ ws, int main_tiles, int tail_tiles,
                                   int split, int BM, int BN, int tiles_m, int tiles_n,
                                   int group_m, int M, int N, float alpha, float beta,
                                   float *__restrict__ C, long long ldc, int vec) {
  const int quads = BN / 4;
  const long long per_tile = (long long)BM * quads;
  const long long total = (long long)tail_tiles * per_tile;
  const long long tile_elems = (long long)BM * BN;
  for (long long g = blockIdx.x * (long long)blockDim.x + threadIdx.x; g < total;
       g += (long long)gridDim.x * blockDim.x) {
    const int t = (int)(g / per_tile);
    const int e = (int)(g - (long long)t * per_tile);
    const int r = e / quads;
    const int c4 = (e - r * quads) * 4;
    int tm, tn;
    tile_coords(main_tiles + t, tiles_m, tiles_n, group_m, tm, tn);
    const int row = tm * BM + r;
    const int col = tn * BN + c4;
    if (row >= M || col >= N) continue;
    const float *src = ws + (long long)t * split * tile_elems + (long long)r * BN + c4;
    // Slices are added in ascending order; their loads are issued four at a time, so a
    // thread waits for one memory latency per four slices instead of one per slice.
    float4 s = *reinterpret_cast<const float4 *>(src);
    int k = 1;
    for (; k + 4 <= split; k += 4) {
      float4 q[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) q[u] = *reinterpret_cast<const float4 *>(src + (k + u) * tile_elems);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        s.x += q[u].x;
        s.y += q[u].y;
        s.z += q[u].z;
        s.w += q[u].w;
      }
    }
    for (; k < split; ++k) {
      const float4 q = *reinterpret_cast<const float4 *>(src + k * tile_elems);
      s.x += q.x;
      s.y += q.y;
      s.z += q.z;
      s.w += q.w;
    }
    float *dst = C + (long long)row * ldc + col;
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
      for (int q = 0; q < 4 && col + q < N; ++q)
        dst[q] = (beta != 0.0f) ? fmaf(alpha, v[q], beta * dst[q]) : alpha * v[q];
    }
  }
}

}  // namespace sgemm
