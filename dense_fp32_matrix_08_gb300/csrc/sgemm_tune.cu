// Measured plan selection: sgemm_f32_autotune times every compiled tile configuration (and
// its split-K layouts) that can run a problem, on the caller's operands, and records the
// fastest in a per-process table that sgemm_f32 / sgemm_f32_ex / sgemm_f32_plan consult
// before the closed-form cost model. The table can be written to and read from a text file.
//
// "GPU GEMM 优化完全拆解（二）" tunes in its autotuning section by sweeping the template
// parameters that pass the kernel's static_asserts and keeping the fastest set, which
// differs from GPU to GPU. Here the compiled configurations are that legal set, and the
// sweep runs at run time, on this GPU, per problem shape.
#include <cuda_runtime.h>

#include <algorithm>
#include <cinttypes>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/sgemm_f32.h"
#include "sgemm_internal.h"
#include "sgemm_plan.h"

namespace sgemm {
namespace {

struct TuneKey {
  int num_sms, M, N, K;
  unsigned flags;  // transa, transb, tma_ok, kpair_ok, b_kmajor, beta != 0, a_tma, b_tma,
                   // at_direct
  bool operator==(const TuneKey &o) const {
    return num_sms == o.num_sms && M == o.M && N == o.N && K == o.K && flags == o.flags;
  }
};

struct TuneEntry {
  TuneKey key;
  int variant, split;
  float ms;
};

std::mutex g_mu;
std::vector<TuneEntry> g_table;

unsigned key_flags(const Problem &pr, bool beta_nz) {
  return (pr.transa ? 1u : 0u) | (pr.transb ? 2u : 0u) | (pr.tma_ok ? 4u : 0u) |
         (pr.kpair_ok ? 8u : 0u) | (pr.b_kmajor ? 16u : 0u) | (beta_nz ? 32u : 0u) |
         (pr.a_tma ? 64u : 0u) | (pr.b_tma ? 128u : 0u) | (pr.at_direct ? 256u : 0u);
}

void insert(const TuneEntry &e) {
  std::lock_guard<std::mutex> lock(g_mu);
  for (TuneEntry &x : g_table)
    if (x.key == e.key) {
      x = e;
      return;
    }
  g_table.push_back(e);
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

bool tuned_lookup(const Problem &pr, bool beta_nz, int num_sms, int *variant, int *split) {
  const TuneKey k{num_sms, pr.M, pr.N, pr.K, key_flags(pr, beta_nz)};
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_table.empty()) return false;
  for (const TuneEntry &x : g_table)
    if (x.key == k) {
      *variant = x.variant;
      *split = x.split;
      return true;
    }
  return false;
}

}  // namespace sgemm

using namespace sgemm;

extern "C" {

int sgemm_f32_autotune(int transa, int transb, int M, int N, int K, float alpha,
                       const float *A, int lda, const float *B, int ldb, float beta,
                       const float *C, int ldc, int reps, cudaStream_t stream, int *variant,
                       int *split, float *ms) {
  if (variant) *variant = -1;
  if (split) *split = 0;
  if (ms) *ms = 0.0f;
  Problem pr{M, N, K, lda, ldb, ldc, transa, transb};
  int rc = validate_ex(pr, alpha, A != nullptr, B != nullptr, C != nullptr);
  if (rc != 0) return rc;
  if (M == 0 || N == 0 || K == 0 || alpha == 0.0f) return 0;  // no GEMM kernel to choose
  pr.tma_ok = !transa && !transb && lda % 4 == 0 && ldb % 4 == 0 && aligned16(A) && aligned16(B);
  pr.kpair_ok = !transa && lda % 4 == 0 && aligned16(A);
  pr.b_kmajor = transb && ldb % 4 == 0 && aligned16(B);
  pr.a_tma = !transa && lda % 4 == 0 && aligned16(A);
  pr.b_tma = !transb && ldb % 4 == 0 && aligned16(B);
  pr.at_direct = transa && lda % 4 == 0 && aligned16(A);
  if (reps <= 0) reps = 3;
  int num_sms = 0;
  cudaError_t e = device_setup(&num_sms);
  if (e != cudaSuccess) return (int)e;
  thin_cluster_capacity(pr.cluster_ctas);
  pr.cluster_cap = cluster_capacity_table();
  const bool beta_nz = beta != 0.0f;

  // Candidates: every configuration with the model's split choice, no split, and whole
  // waves plus a split last wave; the same resulting layout is timed once. Layouts the
  // model puts at more than 4x its best are not timed.
  struct Cand {
    int v, s;
    Plan pl;
  };
  std::vector<Cand> cands;
  double best_model = std::numeric_limits<double>::infinity();
  for (int v = 0; v < kNumVariants; ++v)
    for (int s : {0, 1, -1, 2, 3, 4, 6, 8, -2, -3, -4, -6, -8}) {
      // the thin kernels take the model's split, none, whole waves plus a split tail, and
      // (the cluster thin kernels) cluster sizes 2, 4 and 8; the tile kernels every tile
      // split 2 .. 8 ways (in a cluster where it fits) and split tails of 2 .. 8 slices
      const int thin = kVariants[v].thin;
      if (thin && thin < 5 && (s > 1 || s < -1)) continue;
      if (thin >= 5 && (s < -1 || s == 3 || s == 6)) continue;
      const Plan pl = make_plan(pr, alpha, beta, num_sms, v, s);
      if (pl.variant < 0 || !(pl.cycles < std::numeric_limits<double>::infinity())) continue;
      bool dup = false;
      for (const Cand &c : cands)
        dup = dup || (c.pl.variant == pl.variant && c.pl.split == pl.split &&
                      c.pl.main_tiles == pl.main_tiles && c.pl.k_per_split == pl.k_per_split);
      if (dup) continue;
      cands.push_back({v, s, pl});
      best_model = std::min(best_model, pl.cycles);
    }

  // Scratch copy of C: tuning never modifies the caller's C.
  float *Cs = nullptr;
  const size_t c_bytes = ((size_t)(M - 1) * ldc + N) * sizeof(float);
  e = cudaMallocFromPoolAsync(reinterpret_cast<void **>(&Cs), c_bytes, workspace_pool(), stream);
  if (e != cudaSuccess) return (int)e;
  if (beta_nz)
    e = cudaMemcpy2DAsync(Cs, (size_t)ldc * 4, C, (size_t)ldc * 4, (size_t)N * 4, M,
                          cudaMemcpyDeviceToDevice, stream);
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  if (e == cudaSuccess) e = cudaEventCreate(&e0);
  if (e == cudaSuccess) e = cudaEventCreate(&e1);

  int best_v = -1, best_s = 0;
  float best_ms = 0.0f;
  for (const Cand &c : cands) {
    if (e != cudaSuccess) break;
    if (c.pl.cycles > 4.0 * best_model) continue;
    rc = sgemm_f32_ex_forced(transa, transb, M, N, K, alpha, A, lda, B, ldb, beta, Cs, ldc,
                             c.v, c.s, stream);  // warm-up (and allocation of its workspace)
    if (rc != 0) continue;  // e.g. its workspace is not available: not a candidate
    e = cudaEventRecord(e0, stream);
    for (int r = 0; r < reps && e == cudaSuccess && rc == 0; ++r)
      rc = sgemm_f32_ex_forced(transa, transb, M, N, K, alpha, A, lda, B, ldb, beta, Cs, ldc,
                               c.v, c.s, stream);
    if (e == cudaSuccess) e = cudaEventRecord(e1, stream);
    if (e == cudaSuccess) e = cudaEventSynchronize(e1);
    float t = 0.0f;
    if (e == cudaSuccess) e = cudaEventElapsedTime(&t, e0, e1);
    if (e != cudaSuccess || rc != 0) continue;
    t /= (float)reps;
    if (best_v < 0 || t < best_ms) {
      best_v = c.v;
      best_s = c.s;
      best_ms = t;
    }
  }
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  const cudaError_t fe = cudaFreeAsync(Cs, stream);
  if (e == cudaSuccess) e = fe;
  if (e != cudaSuccess) return (int)e;
  if (best_v < 0) return rc != 0 ? rc : (int)cudaErrorUnknown;
  insert({{num_sms, M, N, K, key_flags(pr, beta_nz)}, best_v, best_s, best_ms});
  if (variant) *variant = best_v;
  if (split) *split = best_s;
  if (ms) *ms = best_ms;
  return 0;
}

int sgemm_f32_tune_clear(void) {
  std::lock_guard<std::mutex> lock(g_mu);
  g_table.clear();
  return 0;
}

int sgemm_f32_tune_count(void) {
  std::lock_guard<std::mutex> lock(g_mu);
  return (int)g_table.size();
}

int sgemm_f32_tune_save(const char *path) {
  if (path == nullptr) return -1;
  std::vector<TuneEntry> copy;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    copy = g_table;
  }
  FILE *f = std::fopen(path, "w");
  if (f == nullptr) return -2;
  std::fprintf(f, "# sgemm_f32 tuned plans v1\n");
  std::fprintf(f, "# sms M N K flags variant split ms\n");
  for (const TuneEntry &x : copy)
    std::fprintf(f, "%d %d %d %d %u %d %d %.6f\n", x.key.num_sms, x.key.M, x.key.N, x.key.K,
                 x.key.flags, x.variant, x.split, (double)x.ms);
  const bool ok = std::fclose(f) == 0;
  return ok ? (int)copy.size() : -2;
}

int sgemm_f32_tune_load(const char *path) {
  if (path == nullptr) return -1;
  FILE *f = std::fopen(path, "r");
  if (f == nullptr) return -2;
  char line[256];
  int n = 0, bad = 0;
  while (std::fgets(line, sizeof line, f)) {
    if (line[0] == '#' || line[0] == '\n') continue;
    TuneEntry x{};
    double t = 0.0;
    if (std::sscanf(line, "%d %d %d %d %u %d %d %lf", &x.key.num_sms, &x.key.M, &x.key.N,
                    &x.key.K, &x.key.flags, &x.variant, &x.split, &t) != 8 ||
        x.key.num_sms <= 0 || x.key.M <= 0 || x.key.N <= 0 || x.key.K <= 0 ||
        x.key.flags > 511u || x.variant < 0 || x.variant >= kNumVariants || x.split < -64 ||
        x.split > 64) {
      ++bad;
      continue;
    }
    x.ms = (float)t;
    insert(x);
    ++n;
  }
  std::fclose(f);
  return bad ? -3 : n;
}

}  // extern "C"
