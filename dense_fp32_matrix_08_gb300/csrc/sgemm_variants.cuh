// The compiled tile configurations of the FFMA kernel, indexed like kVariants in
// sgemm_plan.h (which holds the same shapes without CUDA types, for host-side planning).
// Each configuration's two kernels (B copied with 16-byte or 4-byte copies) are
// instantiated in one of the sgemm_inst_*.cu files so that they compile in parallel.
#pragma once

#include "sgemm_ffma.cuh"
#include "sgemm_plan.h"

namespace sgemm {

using KernelFn = void (*)(const GemmParams);

struct VariantKernels {
  KernelFn k[3][3];  // [APATH][BPATH]; null where not instantiated
  int threads;
  int smem;
};

template <int V>
struct VariantCfg;

//                                   BM   BN  BK  WM  WN  TM  TN  S  MinB MODE
template <> struct VariantCfg<0> { using type = TileConfig<128, 256, 16, 64, 64, 16, 8, 3, 1, 0>; };
template <> struct VariantCfg<1> { using type = TileConfig<128, 128, 16, 32, 64, 8, 8, 4, 2, 0>; };
template <> struct VariantCfg<2> { using type = TileConfig<64, 64, 16, 32, 32, 8, 4, 4, 4, 0>; };
template <> struct VariantCfg<3> { using type = TileConfig<16, 256, 32, 16, 64, 8, 4, 3, 2, 0>; };
template <> struct VariantCfg<4> { using type = TileConfig<256, 16, 32, 64, 16, 8, 4, 3, 2, 0>; };
template <> struct VariantCfg<5> { using type = TileConfig<128, 256, 16, 64, 64, 8, 16, 3, 1, 1>; };
template <> struct VariantCfg<6> { using type = TileConfig<128, 256, 16, 64, 64, 8, 16, 3, 1, 2>; };
template <> struct VariantCfg<7> { using type = TileConfig<128, 256, 32, 64, 64, 8, 16, 3, 1, 2>; };
template <> struct VariantCfg<8> { using type = TileConfig<128, 128, 16, 32, 64, 8, 8, 4, 2, 1>; };
template <> struct VariantCfg<9> { using type = TileConfig<128, 256, 16, 64, 32, 8, 8, 3, 1, 1>; };
template <> struct VariantCfg<10> { using type = TileConfig<256, 128, 16, 64, 32, 8, 8, 3, 1, 1>; };
template <> struct VariantCfg<11> { using type = TileConfig<128, 256, 32, 64, 64, 8, 16, 3, 1, 1>; };
template <> struct VariantCfg<12> { using type = TileConfig<128, 256, 16, 32, 128, 8, 16, 3, 1, 1>; };
template <> struct VariantCfg<13> { using type = TileConfig<128, 256, 16, 64, 64, 8, 16, 4, 1, 1>; };
template <> struct VariantCfg<14> { using type = TileConfig<128, 64, 16, 64, 32, 8, 8, 3, 2, 1>; };
template <> struct VariantCfg<15> { using type = TileConfig<128, 64, 16, 64, 32, 8, 8, 4, 2, 1>; };
template <> struct VariantCfg<16> { using type = TileConfig<128, 128, 16, 64, 64, 8, 16, 3, 2, 1>; };
template <> struct VariantCfg<17> { using type = TileConfig<128, 64, 16, 64, 32, 8, 8, 3, 3, 1>; };
template <> struct VariantCfg<18> { using type = TileConfig<128, 256, 16, 32, 128, 4, 32, 4, 1, 1>; };
template <> struct VariantCfg<19> { using type = TileConfig<128, 128, 16, 32, 128, 4, 32, 3, 2, 1>; };
template <> struct VariantCfg<20> { using type = TileConfig<16, 512, 16, 16, 128, 8, 8, 3, 2, 1>; };
template <> struct VariantCfg<21> { using type = TileConfig<128, 16, 32, 32, 16, 4, 4, 4, 3, 0>; };
template <> struct VariantCfg<22> { using type = TileConfig<128, 128, 16, 64, 64, 8, 16, 4, 2, 1>; };
template <> struct VariantCfg<23> { using type = TileConfig<128, 128, 32, 64, 64, 8, 16, 3, 2, 1>; };
template <> struct VariantCfg<24> { using type = TileConfig<128, 128, 8, 64, 64, 8, 16, 6, 2, 1>; };
template <> struct VariantCfg<25> { using type = TileConfig<128, 128, 16, 64, 64, 8, 16, 3, 2, 2>; };

#define SGEMM_FOR_EACH_VARIANT(X) \
  X(0) X(1) X(2) X(3) X(4) X(5) X(6) X(7) X(8) X(9) X(10) X(11) X(12) X(13) X(14) X(15) \
  X(16) X(17) X(18) X(19) X(20) X(21) X(22) X(23) X(24) X(25)

template <class Cfg>
constexpr bool matches(const VariantShape &s) {
  return s.BM == Cfg::BM && s.BN == Cfg::BN && s.BK == Cfg::BK && s.threads == Cfg::NT &&
         s.TM == Cfg::TM && s.TN == Cfg::TN && s.stages == Cfg::STAGES &&
         s.min_blocks == Cfg::MIN_BLOCKS && s.mode == Cfg::MODE &&
         s.smem_bytes == Cfg::SMEM_BYTES;
}

#define SGEMM_CHECK_VARIANT(v)                                         \
  static_assert(matches<VariantCfg<v>::type>(kVariants[v]),            \
                "sgemm_plan.h kVariants out of step with VariantCfg"); \
  static_assert(v < kNumVariants, "variant index past kVariants");
SGEMM_FOR_EACH_VARIANT(SGEMM_CHECK_VARIANT)
#undef SGEMM_CHECK_VARIANT

// Every configuration gets the row-major paths (A as given; B with 4- or 16-byte copies);
// configurations marked trans_ok in kVariants also get the transposed-operand paths.
template <class Cfg, bool TRANS>
VariantKernels make_kernels() {
  VariantKernels vk = {};
  vk.threads = Cfg::NT;
  vk.smem = Cfg::SMEM_BYTES;
  vk.k[APATH_N][BPATH_N4] = sgemm_ffma_kernel<Cfg, APATH_N, BPATH_N4>;
  vk.k[APATH_N][BPATH_N16] = sgemm_ffma_kernel<Cfg, APATH_N, BPATH_N16>;
  if constexpr (TRANS) {
    vk.k[APATH_N][BPATH_T] = sgemm_ffma_kernel<Cfg, APATH_N, BPATH_T>;
    vk.k[APATH_T16][BPATH_N4] = sgemm_ffma_kernel<Cfg, APATH_T16, BPATH_N4>;
    vk.k[APATH_T16][BPATH_N16] = sgemm_ffma_kernel<Cfg, APATH_T16, BPATH_N16>;
    vk.k[APATH_T16][BPATH_T] = sgemm_ffma_kernel<Cfg, APATH_T16, BPATH_T>;
    vk.k[APATH_T4][BPATH_N4] = sgemm_ffma_kernel<Cfg, APATH_T4, BPATH_N4>;
    vk.k[APATH_T4][BPATH_N16] = sgemm_ffma_kernel<Cfg, APATH_T4, BPATH_N16>;
    vk.k[APATH_T4][BPATH_T] = sgemm_ffma_kernel<Cfg, APATH_T4, BPATH_T>;
  }
  return vk;
}

#define SGEMM_DEFINE_VARIANT(v)                                                        \
  template <>                                                                          \
  VariantKernels variant_kernels<v>() {                                                \
    return make_kernels<VariantCfg<v>::type, kVariants[v].trans_ok>();                 \
  }

// Defined in the sgemm_inst_*.cu files.
template <int V>
VariantKernels variant_kernels();

}  // namespace sgemm
