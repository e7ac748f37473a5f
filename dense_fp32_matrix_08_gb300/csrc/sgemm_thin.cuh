// Streaming kernels for thin products, where one operand is a few rows or columns and the
// other is streamed once from HBM (the 16 x 4096 x 4096 and 4096 x 16 x 8192 shapes):
//
//  * thin-M (M <= 16 per row block): C (16 x N) = A (16 x K) * B (K x N). Each element of B
//    is used by exactly one thread, for 16 FMAs, so B is read straight from global memory
//    into registers (128-bit streaming loads, 8 k rows in flight per thread) and never
//    staged. The CTA's slice of A is staged once in shared memory as As[k][m] and read with
//    broadcast 128-bit loads. A thread owns 4 columns x 16 rows; FFMA2 pairs run along m
//    ({a_m, a_m+1} straight from the As float4) with {b, b} broadcast pairs.
//  * thin-N (N <= 16 per column block): C (M x 16) = A (M x K) * B (K x 16). Each element of
//    A is used by one thread, for 16 FMAs; A rows are streamed as two 128-bit loads (8 k,
//    one 32-byte sector) per row, double-buffered. The CTA's slice of B is staged as
//    Bs[k][16]. A thread owns 4 rows x 16 columns; FFMA2 pairs run along n ({b_n, b_n+1}
//    from the Bs float4) with {a, a} broadcast pairs; 4 rows share every B load.
//
// Both split K into slices so that the grid fills the GPU; a slice's partial tile goes to
// the workspace and tail_reduce_kernel (sgemm_aux.cuh) adds the slices in order and applies
// alpha / beta. With one slice the kernel applies alpha / beta itself. At 8 FLOP per
// streamed byte both shapes sit just below the ridge of this GPU (FP32 peak / HBM
// bandwidth is about 12 FLOP/B), so the FMA loops are written to run at the ~65% of the
// FP32 pipe that full HBM speed asks for.
#pragma once

#include <cuda_runtime.h>

#include "sgemm_ffma.cuh"

namespace sgemm {
namespace thin {

struct ThinParams {
  int M, N, K;
  float alpha, beta;
  const float *A;
  long long lda;
  const float *B;
  long long ldb;
  float *C;
  long long ldc;
  float *ws;        // partial tiles, split > 1 only
  int split;        // K slices (blockIdx.y)
  int k_per_split;  // K values per slice, a multiple of 8
  int tiles_m, tiles_n;
  int vec_c;        // C float4 stores allowed (ldc % 4 == 0, 16-byte aligned C)
};

__device__ __forceinline__ float4 ld_stream4(const float *p) {
  return __ldcs(reinterpret_cast<const float4 *>(p));
}

// Copy the rows x cols block src (row stride ld, 0 outside rows_valid) into shared memory
// transposed, dst[c * dpitch + r], with every thread of the block taking part. Loads are
// issued 16 at a time before their stores, so the staging costs a few memory latencies
// rather than one per element; consecutive threads read consecutive columns (coalesced).
template <int THREADS>
__device__ __forceinline__ void stage_transposed(const float *__restrict__ src, long long ld,
                                                 int rows, int rows_valid, int cols,
                                                 float *dst, int dpitch) {
  constexpr int U = 16;
  const int total = rows * cols;
  for (int e0 = threadIdx.x; e0 < total; e0 += THREADS * U) {
    float v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int e = e0 + u * THREADS;
      const int r = e / cols, c = e - r * cols;
      v[u] = (e < total && r < rows_valid) ? src[(long long)r * ld + c] : 0.0f;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int e = e0 + u * THREADS;
      const int r = e / cols, c = e - r * cols;
      if (e < total) dst[c * dpitch + r] = v[u];
    }
  }
}

// The same without transposing: dst[r * dpitch + c] (columns beyond cols_valid are zero).
template <int THREADS>
__device__ __forceinline__ void stage_rows(const float *__restrict__ src, long long ld, int rows,
                                           int cols, int cols_valid, float *dst, int dpitch) {
  constexpr int U = 16;
  const int total = rows * cols;
  for (int e0 = threadIdx.x; e0 < total; e0 += THREADS * U) {
    float v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int e = e0 + u * THREADS;
      const int r = e / cols, c = e - r * cols;
      v[u] = (e < total && c < cols_valid) ? src[(long long)r * ld + c] : 0.0f;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int e = e0 + u * THREADS;
      const int r = e / cols, c = e - r * cols;
      if (e < total) dst[r * dpitch + c] = v[u];
    }
  }
}

// ------------------------------------------------------------------------------------
// thin-M
namespace m {
constexpr int MT = 16;             // C rows per CTA
constexpr int TPG = 64;            // threads per k-group, 4 columns each
constexpr int KG = 4;              // k-groups per CTA (split the CTA's K slice)
constexpr int THREADS = TPG * KG;  // 256
constexpr int BNC = TPG * 4;       // C columns per CTA
constexpr int KCH = 8;             // k rows of B loaded per batch
constexpr int APITCH = MT + 4;     // As row pitch in floats (16-byte rows, 4-way store spread)
constexpr int KMAX = 512;          // largest K slice (shared memory bound)
inline size_t smem_bytes(int k_per_split) {
  return (size_t)k_per_split * APITCH * 4 + (size_t)(KG - 1) * MT * BNC * 4;
}
}  // namespace m

// VEC: 128-bit B loads allowed (ldb % 4 == 0 and B 16-byte aligned); a column quad that
// crosses N still takes the scalar path.
template <bool VEC>
__global__ void __launch_bounds__(m::THREADS, 2) thin_m_kernel(const ThinParams p) {
  using namespace m;
  extern __shared__ __align__(16) float sm[];
  const int tn = blockIdx.x, slice = blockIdx.y, tmb = blockIdx.z;
  const int n0 = tn * BNC, m0 = tmb * MT;
  const int k0 = slice * p.k_per_split;
  const int KS = min(p.K - k0, p.k_per_split);  // >= 1: the host makes no empty slice
  float *As = sm;
  float *red = sm + (size_t)p.k_per_split * APITCH;

  // Stage A[m0 .. m0+MT) x [k0, k0+KS) as As[k][m] (rows beyond M are zero).
  stage_transposed<THREADS>(p.A + (long long)m0 * p.lda + k0, p.lda, MT, min(MT, p.M - m0),
                            KS, As, APITCH);
  __syncthreads();

  const int g = threadIdx.x / TPG, j = threadIdx.x % TPG;
  const int n = n0 + 4 * j;
  const int glen = (KS + KG - 1) / KG;
  const int kb = min(KS, g * glen), ke = min(KS, kb + glen);
  const bool vec_b = VEC && n + 3 < p.N;

  unsigned long long acc[MT / 2][4];  // acc[mp][c] = {C[2mp][n+c], C[2mp+1][n+c]}
#pragma unroll
  for (int mp = 0; mp < MT / 2; ++mp)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[mp][c] = 0;

  for (int kk = kb; kk < ke; kk += KCH) {
    const int cnt = min(KCH, ke - kk);
    float4 bv[KCH];
#pragma unroll
    for (int q = 0; q < KCH; ++q) {
      bv[q] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (q < cnt) {
        const float *src = p.B + (long long)(k0 + kk + q) * p.ldb + n;
        if (vec_b) {
          bv[q] = ld_stream4(src);
        } else {
          if (n < p.N) bv[q].x = src[0];
          if (n + 1 < p.N) bv[q].y = src[1];
          if (n + 2 < p.N) bv[q].z = src[2];
          if (n + 3 < p.N) bv[q].w = src[3];
        }
      }
    }
#pragma unroll
    for (int q = 0; q < KCH; ++q) {
      if (q < cnt) {
        const float *ar = As + (kk + q) * APITCH;
        unsigned long long a2[MT / 2];
#pragma unroll
        for (int r = 0; r < MT / 4; ++r) {
          const float4 av = *reinterpret_cast<const float4 *>(ar + 4 * r);
          a2[2 * r] = pack2(av.x, av.y);
          a2[2 * r + 1] = pack2(av.z, av.w);
        }
        const unsigned long long b2[4] = {pack2(bv[q].x, bv[q].x), pack2(bv[q].y, bv[q].y),
                                          pack2(bv[q].z, bv[q].z), pack2(bv[q].w, bv[q].w)};
#pragma unroll
        for (int mp = 0; mp < MT / 2; ++mp)
#pragma unroll
          for (int c = 0; c < 4; ++c) ffma2(acc[mp][c], a2[mp], b2[c]);
      }
    }
  }

  // k-groups 1 .. KG-1 hand their sums to group 0 through shared memory ([g-1][m][col]).
  if (g > 0) {
    float *dst = red + (size_t)(g - 1) * MT * BNC + 4 * j;
#pragma unroll
    for (int mp = 0; mp < MT / 2; ++mp) {
      const float2 h0 = unpack2(acc[mp][0]), h1 = unpack2(acc[mp][1]);
      const float2 h2 = unpack2(acc[mp][2]), h3 = unpack2(acc[mp][3]);
      *reinterpret_cast<float4 *>(dst + (2 * mp) * BNC) = make_float4(h0.x, h1.x, h2.x, h3.x);
      *reinterpret_cast<float4 *>(dst + (2 * mp + 1) * BNC) =
          make_float4(h0.y, h1.y, h2.y, h3.y);
    }
  }
  __syncthreads();
  if (g != 0) return;

  float *wt = nullptr;
  if (p.split > 1)
    wt = p.ws + ((long long)(tmb * p.tiles_n + tn) * p.split + slice) * (MT * BNC) + 4 * j;
#pragma unroll
  for (int mp = 0; mp < MT / 2; ++mp) {
    const float2 h0 = unpack2(acc[mp][0]), h1 = unpack2(acc[mp][1]);
    const float2 h2 = unpack2(acc[mp][2]), h3 = unpack2(acc[mp][3]);
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int mm = 2 * mp + half;
      float4 v = half ? make_float4(h0.y, h1.y, h2.y, h3.y) : make_float4(h0.x, h1.x, h2.x, h3.x);
#pragma unroll
      for (int gg = 0; gg < KG - 1; ++gg) {  // fixed order: group 0, then 1, 2, 3
        const float4 o =
            *reinterpret_cast<const float4 *>(red + (size_t)gg * MT * BNC + mm * BNC + 4 * j);
        v.x += o.x;
        v.y += o.y;
        v.z += o.z;
        v.w += o.w;
      }
      if (wt != nullptr) {
        *reinterpret_cast<float4 *>(wt + mm * BNC) = v;
        continue;
      }
      const int row = m0 + mm;
      if (row >= p.M || n >= p.N) continue;
      float *dst = p.C + (long long)row * p.ldc + n;
      const float vv[4] = {v.x, v.y, v.z, v.w};
      if (p.vec_c && n + 3 < p.N) {
        float4 out;
        if (p.beta != 0.0f) {
          const float4 old = *reinterpret_cast<const float4 *>(dst);
          out = make_float4(fmaf(p.alpha, vv[0], p.beta * old.x), fmaf(p.alpha, vv[1], p.beta * old.y),
                            fmaf(p.alpha, vv[2], p.beta * old.z), fmaf(p.alpha, vv[3], p.beta * old.w));
        } else {
          out = make_float4(p.alpha * vv[0], p.alpha * vv[1], p.alpha * vv[2], p.alpha * vv[3]);
        }
        *reinterpret_cast<float4 *>(dst) = out;
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (n + e < p.N)
            dst[e] = (p.beta != 0.0f) ? fmaf(p.alpha, vv[e], p.beta * dst[e]) : p.alpha * vv[e];
      }
    }
  }
}

// ------------------------------------------------------------------------------------
// thin-N
namespace n {
constexpr int NC = 16;             // C columns per CTA
constexpr int R = 4;               // rows per thread
constexpr int THREADS = 256;
constexpr int ROWS = THREADS * R;  // C rows per CTA
constexpr int KCH = 8;             // k values per row and batch (one 32-byte sector)
constexpr int KMAX = 2048;         // largest K slice (shared memory bound)
inline size_t smem_bytes(int k_per_split) { return (size_t)k_per_split * NC * 4; }
}  // namespace n

// VEC: 128-bit A loads allowed (lda % 4 == 0 and A 16-byte aligned); the last, partial
// batch of a slice takes the scalar path.
template <bool VEC>
__global__ void __launch_bounds__(n::THREADS, 1) thin_n_kernel(const ThinParams p) {
  using namespace n;
  extern __shared__ __align__(16) float sm[];
  const int rb = blockIdx.x, slice = blockIdx.y, cb = blockIdx.z;
  const int m0 = rb * ROWS, c0 = cb * NC;
  const int k0 = slice * p.k_per_split;
  const int KS = min(p.K - k0, p.k_per_split);  // >= 1
  float *Bs = sm;

  // Stage B[k0 .. k0+KS) x [c0, c0+NC) as Bs[k][c] (columns beyond N are zero).
  stage_rows<THREADS>(p.B + (long long)k0 * p.ldb + c0, p.ldb, KS, NC, min(NC, p.N - c0), Bs, NC);
  __syncthreads();

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // rows of this thread: a warp owns 32 R consecutive rows, lane + 32 r of them
  const int rbase = m0 + warp * 32 * R + lane;

  unsigned long long acc[R][NC / 2];  // acc[r][jp] = {C[row_r][2jp], C[row_r][2jp+1]}
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int jp = 0; jp < NC / 2; ++jp) acc[r][jp] = 0;

  float4 av[2][R][2];
  auto load = [&](int kk, int buf) {
    const int cnt = min(KCH, KS - kk);
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int row = rbase + 32 * r;
      float4 lo = make_float4(0.f, 0.f, 0.f, 0.f), hi = lo;
      if (row < p.M) {
        const float *src = p.A + (long long)row * p.lda + (k0 + kk);
        if (VEC && cnt == KCH) {
          lo = ld_stream4(src);
          hi = ld_stream4(src + 4);
        } else {
          float t[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) t[e] = e < cnt ? src[e] : 0.0f;
          lo = make_float4(t[0], t[1], t[2], t[3]);
          hi = make_float4(t[4], t[5], t[6], t[7]);
        }
      }
      av[buf][r][0] = lo;
      av[buf][r][1] = hi;
    }
  };
  auto compute = [&](int kk, int buf) {
    const int cnt = min(KCH, KS - kk);
#pragma unroll
    for (int q = 0; q < KCH; ++q) {
      if (q < cnt) {
        const float4 *br = reinterpret_cast<const float4 *>(Bs + (kk + q) * NC);
        unsigned long long b2[NC / 2];
#pragma unroll
        for (int i = 0; i < NC / 4; ++i) {
          const float4 b = br[i];
          b2[2 * i] = pack2(b.x, b.y);
          b2[2 * i + 1] = pack2(b.z, b.w);
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const float4 &v = av[buf][r][q >> 2];
          const int e = q & 3;
          const float a = e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w;
          const unsigned long long a2 = pack2(a, a);
#pragma unroll
          for (int jp = 0; jp < NC / 2; ++jp) ffma2(acc[r][jp], a2, b2[jp]);
        }
      }
    }
  };

  // two batches in flight: batch i + 1 loads while batch i computes
  load(0, 0);
  int kk = 0;
  for (; kk + KCH < KS; kk += 2 * KCH) {
    load(kk + KCH, 1);
    compute(kk, 0);
    if (kk + 2 * KCH < KS) load(kk + 2 * KCH, 0);
    compute(kk + KCH, 1);
  }
  if (kk < KS) compute(kk, 0);

  // epilogue: a thread's row is NC contiguous floats
  const bool vec_out = p.vec_c && c0 + NC <= p.N;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int row = rbase + 32 * r;
    float v[NC];
#pragma unroll
    for (int jp = 0; jp < NC / 2; ++jp) {
      const float2 h = unpack2(acc[r][jp]);
      v[2 * jp] = h.x;
      v[2 * jp + 1] = h.y;
    }
    if (p.split > 1) {
      float *wt = p.ws + ((long long)(rb * p.tiles_n + cb) * p.split + slice) * (ROWS * NC) +
                  (long long)(row - m0) * NC;
#pragma unroll
      for (int i = 0; i < NC / 4; ++i)
        *reinterpret_cast<float4 *>(wt + 4 * i) =
            make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
      continue;
    }
    if (row >= p.M) continue;
    float *dst = p.C + (long long)row * p.ldc + c0;
    if (vec_out) {
#pragma unroll
      for (int i = 0; i < NC / 4; ++i) {
        float4 out;
        if (p.beta != 0.0f) {
          const float4 old = *reinterpret_cast<const float4 *>(dst + 4 * i);
          out = make_float4(fmaf(p.alpha, v[4 * i], p.beta * old.x),
                            fmaf(p.alpha, v[4 * i + 1], p.beta * old.y),
                            fmaf(p.alpha, v[4 * i + 2], p.beta * old.z),
                            fmaf(p.alpha, v[4 * i + 3], p.beta * old.w));
        } else {
          out = make_float4(p.alpha * v[4 * i], p.alpha * v[4 * i + 1], p.alpha * v[4 * i + 2],
                            p.alpha * v[4 * i + 3]);
        }
        *reinterpret_cast<float4 *>(dst + 4 * i) = out;
      }
    } else {
#pragma unroll
      for (int c = 0; c < NC; ++c)
        if (c0 + c < p.N)
          dst[c] = (p.beta != 0.0f) ? fmaf(p.alpha, v[c], p.beta * dst[c]) : p.alpha * v[c];
    }
  }
}

}  // namespace thin
}  // namespace sgemm
