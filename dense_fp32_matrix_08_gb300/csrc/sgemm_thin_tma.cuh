// TMA-fed thin-product kernel for sm_103a: C (M x N) = alpha * A (M x K) * B (K x N) + beta
// * C for M <= 16 per row block with B TMA-addressable (thin-M), or for N <= 16 per column
// block with A TMA-addressable (thin-N, computed as C^T = B^T A^T; see thin_tma_kernel).
// The description below is for thin-M.
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

// One kernel, two orientations. "Small" is the 16-wide dimension, "wide" the 256 columns a
// CTA covers, and every chunk of the streamed operand holds 8 k for the CTA's 256 wide
// indices.
//  * TN = false (thin-M): small = M, wide = N. A (16 x K) is staged as Sm[k][s], and B
//    streams as [8 k][256 n] tiles. Lane l owns wide indices 4l + c and 128 + 4l + c.
//  * TN = true (thin-N): C^T = B^T A^T, so small = N and wide = M. B (K x 16) is staged as
//    Sm[k][s] = B[k][s], and A streams as [256 m][8 k] tiles with the 32-byte swizzle
//    (16-byte chunk h of row r at h ^ ((r >> 2) & 1)). Lane l owns wide indices l + 32 c,
//    and per 4 k it loads one float4 per wide index; 8 consecutive rows land in 8 bank
//    groups. The output is written transposed, to C[wide][small].
// grid = (wide tiles, split, small tiles); p.k_per_split = the K range of one CTA (a
// multiple of KC, at most KMAX). With split > 1 the slices' tiles go to p.ws for
// tail_reduce_kernel (C-tile layout: [16][256] for thin-M, [256][16] for thin-N).
template <bool TN>
__global__ void __launch_bounds__(mt::THREADS, 1)
    thin_tma_kernel(const __grid_constant__ CUtensorMap map_s, const ThinParams p,
                    int *status) {
  using namespace mt;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = saddr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *sbase = smem_raw + (base - raw);
  float *ring = reinterpret_cast<float *>(sbase);
  float *Sm = reinterpret_cast<float *>(sbase + RING_BYTES);
  const uint32_t bars = base + RING_BYTES + (uint32_t)p.k_per_split * MT * 4;  // full[stage]

  const int wblk = blockIdx.x, slice = blockIdx.y, sblk = blockIdx.z;
  const int w0 = wblk * BNC, s0 = sblk * MT;
  const int small = TN ? p.N : p.M;
  const int k0 = slice * p.k_per_split;
  const int KS = min(p.K - k0, p.k_per_split);  // >= 1: the host makes no empty slice
  const int NCH = (KS + KC - 1) / KC;           // chunks in the slice
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int my_chunks = NCH > warp ? (NCH - warp + WARPS - 1) / WARPS : 0;

  auto stage_of = [&](int j) { return warp * SPW + (j % SPW); };
  auto issue = [&](int j) {  // lane 0: chunk warp + WARPS j into its stage
    const int st = stage_of(j);
    const int kc = k0 + (warp + WARPS * j) * KC;
    mbar_expect_tx(bars + 8 * st, CHUNK_BYTES);
    if constexpr (TN)
      tma_load_2d(base + st * CHUNK_BYTES, &map_s, kc, w0, bars + 8 * st);
    else
      tma_load_2d(base + st * CHUNK_BYTES, &map_s, w0, kc, bars + 8 * st);
  };
  // The streamed operand starts moving before the small one is staged: each warp's lane 0
  // initialises its stages' barriers and issues its first SPW chunks.
  if (lane == 0) {
    for (int q = 0; q < SPW; ++q) mbar_init(bars + 8 * (warp * SPW + q), 1);
    mbar_init_fence();
    if (warp == 0) tma_prefetch_map(&map_s);
    for (int j = 0; j < SPW && j < my_chunks; ++j) issue(j);
  }
  // Stage the small operand's slice as Sm[k][s] (s beyond the small extent is zero).
  if constexpr (TN)
    stage_rows<THREADS>(p.B + (long long)k0 * p.ldb + s0, p.ldb, KS, MT, min(MT, small - s0),
                        Sm, MT);
  else
    stage_transposed<THREADS>(p.A + (long long)s0 * p.lda + k0, p.lda, MT,
                              min(MT, small - s0), KS, Sm, MT);
  __syncthreads();

  unsigned long long acc[MT / 2][8];  // acc[sp][c] = {v(2sp, wide_c), v(2sp+1, wide_c)}
#pragma unroll
  for (int sp = 0; sp < MT / 2; ++sp)
#pragma unroll
    for (int c = 0; c < 8; ++c) acc[sp][c] = 0;

  // one k step: 16 small values (4 broadcast float4) times the lane's 8 wide values
  auto step = [&](const float4 *fs, const float (&bw)[8]) {
    unsigned long long a2[MT / 2];
#pragma unroll
    for (int r = 0; r < MT / 4; ++r) {
      a2[2 * r] = pack2(fs[r].x, fs[r].y);
      a2[2 * r + 1] = pack2(fs[r].z, fs[r].w);
    }
    unsigned long long b2[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) b2[c] = pack2(bw[c], bw[c]);
#pragma unroll
    for (int sp = 0; sp < MT / 2; ++sp)
#pragma unroll
      for (int c = 0; c < 8; ++c) ffma2(acc[sp][c], a2[sp], b2[c]);
  };

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
    if constexpr (TN) {
      const int swz = (lane >> 2) & 1;  // == ((lane + 32 c) >> 2) & 1 for every c
#pragma unroll
      for (int h = 0; h < KC / 4; ++h) {
        if (4 * h >= cnt) break;  // warp-uniform
        float4 bt[8];
#pragma unroll
        for (int c = 0; c < 8; ++c)
          bt[c] = *reinterpret_cast<const float4 *>(bs + (lane + 32 * c) * KC + ((h ^ swz) << 2));
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
          const int q = 4 * h + qq;
          if (q < cnt) {
            float4 fs[MT / 4];
#pragma unroll
            for (int r = 0; r < MT / 4; ++r)
              fs[r] = *reinterpret_cast<const float4 *>(Sm + (kc0 + q) * MT + 4 * r);
            float bw[8];
#pragma unroll
            for (int c = 0; c < 8; ++c)
              bw[c] = qq == 0 ? bt[c].x : qq == 1 ? bt[c].y : qq == 2 ? bt[c].z : bt[c].w;
            step(fs, bw);
          }
        }
      }
    } else {
      // fragments double-buffered across k steps: step q + 1 loads while step q computes
      float4 fb[2][2], fa[2][MT / 4];
      auto load = [&](int q, int buf) {
        fb[buf][0] = *reinterpret_cast<const float4 *>(bs + q * BNC + 4 * lane);
        fb[buf][1] = *reinterpret_cast<const float4 *>(bs + q * BNC + 128 + 4 * lane);
#pragma unroll
        for (int r = 0; r < MT / 4; ++r)
          fa[buf][r] = *reinterpret_cast<const float4 *>(Sm + (kc0 + q) * MT + 4 * r);
      };
      load(0, 0);
#pragma unroll
      for (int q = 0; q < KC; ++q) {
        if (q < cnt) {  // warp-uniform
          if (q + 1 < KC && q + 1 < cnt) load(q + 1, (q + 1) & 1);
          const float4 b0 = fb[q & 1][0], b1 = fb[q & 1][1];
          const float bw[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
          step(fa[q & 1], bw);
        }
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

  // warp partials -> ring as red[warp][s][wide]; then each output is their sum in warp order
  float *red = ring;
  auto wide_of = [&](int c) { return TN ? lane + 32 * c : (c < 4 ? 4 * lane + c : 124 + 4 * lane + c); };
#pragma unroll
  for (int sp = 0; sp < MT / 2; ++sp) {
    float *r0 = red + ((size_t)warp * MT + 2 * sp) * BNC;
    float *r1 = r0 + BNC;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const float2 h = unpack2(acc[sp][c]);
      r0[wide_of(c)] = h.x;
      r1[wide_of(c)] = h.y;
    }
  }
  __syncthreads();
  const long long tile = TN ? (long long)wblk * p.tiles_n + sblk : (long long)sblk * p.tiles_n + wblk;
  float *wt = p.split > 1 ? p.ws + (tile * p.split + slice) * (MT * BNC) : nullptr;
  // Output groups of 4 consecutive C columns: thin-M 4 wide indices of one small row,
  // thin-N 4 small indices of one wide row (C rows of 16 floats).
  for (int e = tid; e < MT * BNC / 4; e += THREADS) {
    int ws_, ww;  // small and wide index of the group's first element
    if constexpr (TN) {
      ww = e / (MT / 4);
      ws_ = (e - ww * (MT / 4)) * 4;
    } else {
      ws_ = e / (BNC / 4);
      ww = (e - ws_ * (BNC / 4)) * 4;
    }
    float v[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int si = TN ? ws_ + q : ws_, wi = TN ? ww : ww + q;
      float sum = red[(size_t)si * BNC + wi];
#pragma unroll
      for (int w = 1; w < WARPS; ++w) sum += red[((size_t)w * MT + si) * BNC + wi];  // in order
      v[q] = sum;
    }
    // C coordinates of the group: row, first column, and the tile-local offset
    const int row = TN ? w0 + ww : s0 + ws_;
    const int col = TN ? s0 + ws_ : w0 + ww;
    if (wt != nullptr) {
      const int off = TN ? ww * MT + ws_ : ws_ * BNC + ww;
      *reinterpret_cast<float4 *>(wt + off) = make_float4(v[0], v[1], v[2], v[3]);
      continue;
    }
    if (row >= p.M || col >= p.N) continue;
    float *dst = p.C + (long long)row * p.ldc + col;
    if (p.vec_c && col + 3 < p.N) {
      float4 out;
      if (p.beta != 0.0f) {
        const float4 old = *reinterpret_cast<const float4 *>(dst);
        out = make_float4(fmaf(p.alpha, v[0], p.beta * old.x), fmaf(p.alpha, v[1], p.beta * old.y),
                          fmaf(p.alpha, v[2], p.beta * old.z), fmaf(p.alpha, v[3], p.beta * old.w));
      } else {
        out = make_float4(p.alpha * v[0], p.alpha * v[1], p.alpha * v[2], p.alpha * v[3]);
      }
      *reinterpret_cast<float4 *>(dst) = out;
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (col + q < p.N)
          dst[q] = (p.beta != 0.0f) ? fmaf(p.alpha, v[q], p.beta * dst[q]) : p.alpha * v[q];
    }
  }
}

}  // namespace thin
}  // namespace sgemm
