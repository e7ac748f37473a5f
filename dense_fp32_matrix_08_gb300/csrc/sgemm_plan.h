// Host-side argument checks and launch planning for the SGEMM library. Plain C++ (no CUDA
// types), so the same logic is exercised by CPU-only tests through sgemm_f32_plan().
#pragma once

#include <algorithm>
#include <cstddef>
#include <cstdint>
#include <limits>

namespace sgemm {

constexpr int kErrWorkspace = -13;
constexpr int kErrBadVariant = -14;

struct Problem {
  int M, N, K, lda, ldb, ldc;
};

// Shape of one compiled tile configuration (mirrors TileConfig in sgemm_ffma.cuh).
struct VariantShape {
  int BM, BN, BK, threads, TM, TN, stages, min_blocks, smem_bytes;
  double eff;  // modelled fraction of the FP32 pipe this configuration sustains
};

constexpr int smem_of(int BM, int BN, int BK, int stages) {
  return stages * BK * (BM + BN) * 4;
}

constexpr VariantShape kVariants[] = {
    {128, 256, 16, 256, 16, 8, 3, 1, smem_of(128, 256, 16, 3), 1.00},
    {128, 128, 16, 256, 8, 8, 4, 2, smem_of(128, 128, 16, 4), 0.90},
    {64, 64, 16, 128, 8, 4, 4, 4, smem_of(64, 64, 16, 4), 0.70},
    {16, 256, 32, 128, 8, 4, 3, 2, smem_of(16, 256, 32, 3), 0.60},
    {256, 16, 32, 128, 8, 4, 3, 2, smem_of(256, 16, 32, 3), 0.60},
};
constexpr int kNumVariants = sizeof(kVariants) / sizeof(kVariants[0]);

struct Plan {
  int variant = -1;     // -1: no GEMM kernel (beta-scale only, or nothing)
  int split = 1;        // K slices
  int k_per_split = 0;  // K elements per slice (multiple of BK)
  int tiles_m = 0, tiles_n = 0;
  int group_m = 1;
  int launches = 0;
  size_t ws_bytes = 0;
};

inline long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }

// Row stride of split-K partials: N rounded up to 4 so every row starts 16-byte aligned.
inline long long workspace_ld(int N) { return ceil_div(N, 4) * 4; }

// BLAS-style check: the first illegal argument, numbered from 1 in the sgemm_f32 order
// (M, N, K, alpha, A, lda, B, ldb, beta, C, ldc). A and B only have to be present when
// they are read (alpha != 0, K > 0, non-empty C); C whenever the view is non-empty.
inline int validate(const Problem &p, float alpha, bool hasA, bool hasB, bool hasC) {
  if (p.M < 0) return -1;
  if (p.N < 0) return -2;
  if (p.K < 0) return -3;
  const bool nonempty = p.M > 0 && p.N > 0;
  const bool reads_ab = nonempty && p.K > 0 && alpha != 0.0f;
  if (reads_ab && !hasA) return -5;
  if (p.lda < std::max(1, p.K)) return -6;
  if (reads_ab && !hasB) return -7;
  if (p.ldb < std::max(1, p.N)) return -8;
  if (nonempty && !hasC) return -10;
  if (p.ldc < std::max(1, p.N)) return -11;
  return 0;
}

// Modelled cost, in SM cycles, of running variant v with `split` K slices.
// GEMM kernel: the busiest SM runs ceil(ctas / SMs) CTAs, each BM*BN*k_slice FMAs at
// 128 FMA/cycle scaled by the variant's efficiency, plus ~2500 cycles of pipeline fill and
// epilogue; it overlaps with streaming the algorithmic bytes (and the split-K partials it
// writes) at ~3400 bytes/cycle for the chip. Split-K adds a reduction kernel that runs
// after it: partials read, C read (beta != 0) and written, plus ~2000 cycles of launch.
inline double model_cycles(const Problem &p, int v, int split, int num_sms, bool beta_nz,
                           int *k_per_split_out, int *split_eff_out) {
  const VariantShape &s = kVariants[v];
  const long long tiles = ceil_div(p.M, s.BM) * ceil_div(p.N, s.BN);
  const long long kt = ceil_div(p.K, s.BK);
  const long long kt_per = ceil_div(kt, split);
  const long long split_eff = ceil_div(kt, kt_per);
  const long long ctas = tiles * split_eff;
  const double per_sm = (double)ceil_div(ctas, num_sms);
  const double fmas = (double)s.BM * s.BN * (double)(kt_per * s.BK);
  const double compute = per_sm * (fmas / (128.0 * s.eff) + 2500.0);
  const double mn = (double)p.M * (double)workspace_ld(p.N);
  double gemm_bytes = 4.0 * ((double)p.M * p.K + (double)p.K * p.N);
  double reduce = 0.0;
  if (split_eff > 1) {
    gemm_bytes += 4.0 * split_eff * mn;
    reduce = 4.0 * (split_eff + (beta_nz ? 2.0 : 1.0)) * mn / 3400.0 + 2000.0;
  } else {
    gemm_bytes += 4.0 * mn * (beta_nz ? 2.0 : 1.0);
  }
  if (k_per_split_out) *k_per_split_out = (int)(kt_per * s.BK);
  if (split_eff_out) *split_eff_out = (int)split_eff;
  return std::max(compute, gemm_bytes / 3400.0) + reduce;
}

// Choose the tile configuration and split-K factor. force_v >= 0 pins the variant;
// force_split >= 1 pins the split (clamped to the number of K tiles).
inline Plan make_plan(const Problem &p, float alpha, float beta, int num_sms, int force_v,
                      int force_split) {
  Plan pl;
  if (p.M == 0 || p.N == 0) return pl;
  if (alpha == 0.0f || p.K == 0) {
    pl.launches = (beta == 1.0f) ? 0 : 1;
    return pl;
  }
  num_sms = std::max(1, num_sms);
  const bool beta_nz = beta != 0.0f;
  double best = std::numeric_limits<double>::infinity();
  int best_v = 0, best_split = 1, best_kps = 0;
  const int v_lo = force_v >= 0 ? force_v : 0;
  const int v_hi = force_v >= 0 ? force_v : kNumVariants - 1;
  for (int v = v_lo; v <= v_hi; ++v) {
    const long long kt = ceil_div(p.K, kVariants[v].BK);
    const int max_split = (int)std::min<long long>(64, kt);
    const int s_lo = force_split >= 1 ? std::min(force_split, max_split) : 1;
    const int s_hi = force_split >= 1 ? s_lo : max_split;
    for (int sp = s_lo; sp <= s_hi; ++sp) {
      int kps = 0, seff = 0;
      const double c = model_cycles(p, v, sp, num_sms, beta_nz, &kps, &seff);
      const double ws = seff > 1 ? 4.0 * seff * (double)p.M * (double)workspace_ld(p.N) : 0;
      if (force_split < 1 && ws > 512.0 * 1024 * 1024) continue;  // workspace cap
      if (c < best * 0.999) {  // prefer fewer slices on (near) ties
        best = c;
        best_v = v;
        best_split = seff;
        best_kps = kps;
      }
    }
  }
  const VariantShape &s = kVariants[best_v];
  pl.variant = best_v;
  pl.split = best_split;
  pl.k_per_split = best_split > 1 ? best_kps : (int)(ceil_div(p.K, s.BK) * s.BK);
  pl.tiles_m = (int)ceil_div(p.M, s.BM);
  pl.tiles_n = (int)ceil_div(p.N, s.BN);
  pl.group_m = std::min(8, pl.tiles_m);
  pl.launches = best_split > 1 ? 2 : 1;
  pl.ws_bytes = best_split > 1 ? (size_t)4 * best_split * (size_t)p.M * workspace_ld(p.N) : 0;
  return pl;
}

}  // namespace sgemm
