// TMA-fed thin-M kernel for sm_103a: C (M x N) = alpha * A (M x K) * B (K x N) + beta * C
// for M <= 16 per row block, B row-major, 16-byte aligned with ldb a multiple of 4.
//
// At M = 16 every element of B is used for 16 FMAs only (8 FLOP per streamed byte, just
// below this GPU's FP32/HBM ridge of about 12), so the kernel has two jobs at once: stream B
// from HBM at full speed and keep the FP32 pipe about two-thirds busy.
//  * B streams in [8 k][256 n] chunks (8 KB) by TMA. Each of the 8 warps owns two private
//    ring stages and the chunks c = w, w + 8, w + 16, ... of the CTA's K slice: lane 0 of
//    the warp issues a chunk's copy, the warp waits on that stage's mbarrier (bounded),
//    computes, and refills the stage with its chunk two steps ahead. No barrier spans
//    warps in the main loop, and 8 to 16 chunks (64 - 128 KB) are in flight per SM.
//  * The CTA's slice of A (16 rows x its K range) is staged once as As[k][16].
//  * Lane l owns columns 4l .. 4l+3 and 128 + 4l .. 128 + 4l + 3 (two conflict-free 128-bit
//    loads per k) and all 16 rows: FFMA2 pairs run along m ({a_m, a_m+1} straight from the
//    As float4, B broadcast into {b, b}), 64 FFMA2 per k step.
//  * The 8 warps' partial tiles are added in shared memory in warp order. With several K
//    slices per column block, each slice's tile goes to the workspace and
//    tail_reduce_kernel adds the slices in order: every output is a fixed-order sum.
#pragma once

#include <cuda.h>

#include "sgemm_ffma.cuh"
#include "sgemm_ptx.cuh"
#include "sgemm_thin.cuh"

namespace sgemm {
namespace thin {
namespace mt {

constexpr int MT = 16;            // C rows per row block
constexpr int BNC = 256;          // C columns per CTA
constexpr int KC = 8;             // k rows per chunk (one TMA copy)
constexpr int WARPS = 8;
constexpr int SPW = 2;            // private stages per warp
constexpr int THREADS = WARPS * 32;
constexpr int KB = KC;            // K slice granule
constexpr int KMAX = 1024;        // largest K slice per CTA (staged A: 16 x KMAX floats)
constexpr int CHUNK_BYTES = KC * BNC * 4;
constexpr int RING_BYTES = WARPS * SPW * CHUNK_BYTES;
constexpr int RED_BYTES = WARPS * MT * BNC * 4;  // per-warp partial tiles, in the ring
static_assert(RED_BYTES <= RING_BYTES, "warp partials fit in the ring");
static_assert(BNC == 8 * 32, "eight columns per lane");
inline size_t smem_bytes(int k_per_split) {
  return 1024 + RING_BYTES + (size_t)k_per_split * MT * 4 + 8 * WARPS * SPW;
}

}  // namespace mt

// grid = (tiles_n, split, tiles_m); p.k_per_split = the K range of one CTA (a multiple of
// KC, at most KMAX). With split > 1 the slices' tiles go to p.ws for tail_reduce_kernel.
__global__ void __launch_bounds__(mt::THREADS, 1)
    thin_m_tma_kernel(const __grid_constant__ CUtensorMap map_b, const ThinParams p,
                      int *status) {
  using namespace mt;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = saddr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *sbase = smem_raw + (base - raw);
  float *ring = reinterpret_cast<float *>(sbase);
  float *As = reinterpret_cast<float *>(sbase + RING_BYTES);
  const uint32_t bars = base + RING_BYTES + (uint32_t)p.k_per_split * MT * 4;  // full[stage]

  const int tn = blockIdx.x, slice = blockIdx.y, tmb = blockIdx.z;
  const int n0 = tn * BNC, m0 = tmb * MT;
  const int k0 = slice * p.k_per_split;
  const int KS = min(p.K - k0, p.k_per_split);  // >= 1: the host makes no empty slice
  const int NCH = (KS + KC - 1) / KC;           // chunks in the slice
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int my_chunks = NCH > warp ? (NCH - warp + WARPS - 1) / WARPS : 0;

  auto stage_of = [&](int j) { return warp * SPW + (j % SPW); };
  auto issue = [&](int j) {  // lane 0: chunk warp + WARPS j into its stage
    const int st = stage_of(j);
    mbar_expect_tx(bars + 8 * st, CHUNK_BYTES);
    tma_load_2d(base + st * CHUNK_BYTES, &map_b, n0, k0 + (warp + WARPS * j) * KC, bars + 8 * st);
  };
  // B starts streaming before A is staged: each warp's lane 0 initialises its stages'
  // barriers and issues its first SPW chunks.
  if (lane == 0) {
    for (int q = 0; q < SPW; ++q) mbar_init(bars + 8 * (warp * SPW + q), 1);
    mbar_init_fence();
    if (warp == 0) tma_prefetch_map(&map_b);
    for (int j = 0; j < SPW && j < my_chunks; ++j) issue(j);
  }
  // Stage A[m0 .. m0+16) x [k0, k0+KS) as As[k][m] (rows beyond M are zero).
  stage_transposed<THREADS>(p.A + (long long)m0 * p.lda + k0, p.lda, MT, min(MT, p.M - m0),
                            KS, As, MT);
  __syncthreads();

  unsigned long long acc[MT / 2][8];  // acc[mp][c] = {C[2mp][col_c], C[2mp+1][col_c]}
#pragma unroll
  for (int mp = 0; mp < MT / 2; ++mp)
#pragma unroll
    for (int c = 0; c < 8; ++c) acc[mp][c] = 0;

  int waited = 0;  // chunks whose copy this warp has seen complete
  for (int j = 0; j < my_chunks; ++j) {
    const int st = stage_of(j);
    if (!mbar_wait(bars + 8 * st, (uint32_t)(j / SPW) & 1u)) {
      if (lane == 0) atomicCAS(status, 0, 1);
      break;
    }
    waited = j + 1;
    const float *bs = ring + st * (CHUNK_BYTES / 4);
    const int kc0 = (warp + WARPS * j) * KC;  // first k of the chunk inside the slice
    const int cnt = min(KC, KS - kc0);        // k rows of the chunk inside the slice
    // fragments double-buffered across k steps: step q + 1 loads while step q computes
    float4 fb[2][2], fa[2][MT / 4];
    auto load = [&](int q, int buf) {
      fb[buf][0] = *reinterpret_cast<const float4 *>(bs + q * BNC + 4 * lane);
      fb[buf][1] = *reinterpret_cast<const float4 *>(bs + q * BNC + 128 + 4 * lane);
#pragma unroll
      for (int r = 0; r < MT / 4; ++r)
        fa[buf][r] = *reinterpret_cast<const float4 *>(As + (kc0 + q) * MT + 4 * r);
    };
    load(0, 0);
#pragma unroll
    for (int q = 0; q < KC; ++q) {
      if (q < cnt) {  // warp-uniform
        if (q + 1 < KC && q + 1 < cnt) load(q + 1, (q + 1) & 1);
        const float4 *fac = fa[q & 1];
        const float4 b0 = fb[q & 1][0], b1 = fb[q & 1][1];
        unsigned long long a2[MT / 2];
#pragma unroll
        for (int r = 0; r < MT / 4; ++r) {
          a2[2 * r] = pack2(fac[r].x, fac[r].y);
          a2[2 * r + 1] = pack2(fac[r].z, fac[r].w);
        }
        const unsigned long long b2[8] = {pack2(b0.x, b0.x), pack2(b0.y, b0.y),
                                          pack2(b0.z, b0.z), pack2(b0.w, b0.w),
                                          pack2(b1.x, b1.x), pack2(b1.y, b1.y),
                                          pack2(b1.z, b1.z), pack2(b1.w, b1.w)};
#pragma unroll
        for (int mp = 0; mp < MT / 2; ++mp)
#pragma unroll
          for (int c = 0; c < 8; ++c) ffma2(acc[mp][c], a2[mp], b2[c]);
      }
    }
    __syncwarp();  // every lane has read the stage before it is refilled
    if (lane == 0 && j + SPW < my_chunks) issue(j + SPW);
  }
  // No copy may still be writing the ring when it is reused below: a warp that stopped
  // early waits (bounded) for the copies it issued and has not seen complete.
  if (lane == 0) {
    const int issued = min(my_chunks, waited + SPW);
    for (int j = waited; j < issued; ++j)
      if (!mbar_wait(bars + 8 * stage_of(j), (uint32_t)(j / SPW) & 1u)) atomicCAS(status, 0, 3);
  }
  __syncthreads();

  // warp partials -> ring as red[w][m][col]; then each output is their sum in warp order
  float *red = ring;
#pragma unroll
  for (int mp = 0; mp < MT / 2; ++mp) {
    float lo[8], hi[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const float2 h = unpack2(acc[mp][c]);
      lo[c] = h.x;
      hi[c] = h.y;
    }
    float *r0 = red + ((size_t)warp * MT + 2 * mp) * BNC;
    float *r1 = r0 + BNC;
    *reinterpret_cast<float4 *>(r0 + 4 * lane) = make_float4(lo[0], lo[1], lo[2], lo[3]);
    *reinterpret_cast<float4 *>(r0 + 128 + 4 * lane) = make_float4(lo[4], lo[5], lo[6], lo[7]);
    *reinterpret_cast<float4 *>(r1 + 4 * lane) = make_float4(hi[0], hi[1], hi[2], hi[3]);
    *reinterpret_cast<float4 *>(r1 + 128 + 4 * lane) = make_float4(hi[4], hi[5], hi[6], hi[7]);
  }
  __syncthreads();
  float *wt = p.split > 1
                  ? p.ws + ((long long)(tmb * p.tiles_n + tn) * p.split + slice) * (MT * BNC)
                  : nullptr;
  for (int e = tid; e < MT * BNC / 4; e += THREADS) {
    float4 sum = reinterpret_cast<const float4 *>(red)[e];
#pragma unroll
    for (int w = 1; w < WARPS; ++w) {  // warp order: a fixed summation order
      const float4 v = reinterpret_cast<const float4 *>(red + (size_t)w * MT * BNC)[e];
      sum.x += v.x;
      sum.y += v.y;
      sum.z += v.z;
      sum.w += v.w;
    }
    const int mm = e / (BNC / 4), col = (e - mm * (BNC / 4)) * 4;
    if (wt != nullptr) {
      *reinterpret_cast<float4 *>(wt + mm * BNC + col) = sum;
      continue;
    }
    const int row = m0 + mm, gcol = n0 + col;
    if (row >= p.M || gcol >= p.N) continue;
    float *dst = p.C + (long long)row * p.ldc + gcol;
    const float vv[4] = {sum.x, sum.y, sum.z, sum.w};
    if (p.vec_c && gcol + 3 < p.N) {
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
      for (int q = 0; q < 4; ++q)
        if (gcol + q < p.N)
          dst[q] = (p.beta != 0.0f) ? fmaf(p.alpha, vv[q], p.beta * dst[q]) : p.alpha * vv[q];
    }
  }
}

}  // namespace thin
}  // namespace sgemm
