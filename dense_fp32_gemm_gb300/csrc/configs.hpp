// configs.hpp -- the tile configurations compiled into the library and the
// registry entry each one exports to the dispatcher.
//
// Each configuration is legal by construction: ffma_sgemm_kernel<> carries a
// static_assert(cfg_valid(S)), so an illegal tuple never becomes a kernel
// (the compile-time gate that "Autotuning: Searching the Tile-Shape Space",
// section "Mechanics" 2, builds with if constexpr).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "tile_config.hpp"

namespace sgemm_gb300 {

struct KernelParams;

// Every configuration compiled into the library, in registry order:
//   X(Name, BM, BN, BK, WM, WN, WNITER, TM, TN, NT, STAGES, MINB, KU, ORDER)
// wide:    128 x 256 CTA tile, 8 warps of 64 x 64, 16 x 8 accumulators per lane
//          (B arrives by TMA, so a wide BN costs no loader instructions);
// tall:    256 x 64, 4 warps of 64 x 64, for N <= 64;
// flat:    64 x 256, 4 warps of 64 x 64, for M <= 64;
// mini / small: 64 x 64 and 64 x 128 tiles of 2 and 4 warps (8 x 8 per lane)
//          for problems too small to fill 152 SMs with larger tiles;
// square:  128 x 128, 4 warps of 64 x 64, two CTAs per SM;
// pages:   the pages' sweep winner (128 x 64 x 16, warp 64 x 32, WNITER 2,
//          4 x 4 patches, 128 threads) on this kernel's pipeline;
// the rest vary the k-slice depth (BK), the unrolled chunk (KU) and the
// pipeline depth of the wide shape, for the tuner.
#define SGEMM_GB300_CONFIGS(X)                                     \
  X(Wide, 128, 256, 16, 64, 64, 2, 4, 4, 256, 4, 1, 4, 0)          \
  X(Tall, 256, 64, 16, 64, 64, 2, 4, 4, 128, 4, 2, 4, 0)           \
  X(Square, 128, 128, 16, 64, 64, 2, 4, 4, 128, 4, 2, 4, 0)        \
  X(Pages, 128, 64, 16, 64, 32, 2, 4, 4, 128, 3, 3, 4, 0)          \
  X(WideKu8, 128, 256, 16, 64, 64, 2, 4, 4, 256, 4, 1, 8, 0)       \
  X(WideBk32, 128, 256, 32, 64, 64, 2, 4, 4, 256, 4, 1, 4, 0)      \
  X(WideBk32Ku8, 128, 256, 32, 64, 64, 2, 4, 4, 256, 4, 1, 8, 0)   \
  X(WideBk32Ku8Zz, 128, 256, 32, 64, 64, 2, 4, 4, 256, 4, 1, 8, 1) \
  X(WideBk48Ku8, 128, 256, 48, 64, 64, 2, 4, 4, 256, 3, 1, 8, 0)   \
  X(SquareBk32, 128, 128, 32, 64, 64, 2, 4, 4, 128, 3, 2, 8, 0)    \
  X(TallBk24, 256, 64, 24, 64, 64, 2, 4, 4, 128, 3, 2, 8, 0)       \
  X(WideBk32F2, 128, 256, 32, 64, 64, 2, 4, 4, 256, 4, 1, 8, 2)    \
  X(WideBk48F2, 128, 256, 48, 64, 64, 2, 4, 4, 256, 3, 1, 8, 2)    \
  X(WideBk16F2, 128, 256, 16, 64, 64, 2, 4, 4, 256, 4, 1, 8, 2)    \
  X(SquareBk32F2, 128, 128, 32, 64, 64, 2, 4, 4, 128, 3, 2, 8, 2)  \
  X(TallBk24F2, 256, 64, 24, 64, 64, 2, 4, 4, 128, 3, 2, 8, 2)     \
  X(WideBk32F2Ku16, 128, 256, 32, 64, 64, 2, 4, 4, 256, 4, 1, 16, 2) \
  X(FlatBk24F2, 64, 256, 24, 64, 64, 2, 4, 4, 128, 3, 2, 8, 2)       \
  X(MiniF2, 64, 64, 16, 32, 64, 2, 4, 4, 64, 3, 6, 8, 2)              \
  X(SmallF2, 64, 128, 16, 32, 64, 2, 4, 4, 128, 3, 3, 8, 2)               \
  X(WideBk32F2Ku32, 128, 256, 32, 64, 64, 2, 4, 4, 256, 4, 1, 32, 2)      \
  X(FlatBk24F2Ku24, 64, 256, 24, 64, 64, 2, 4, 4, 128, 3, 2, 24, 2)       \
  X(MidBk32F2Ku32, 128, 64, 32, 64, 32, 2, 4, 4, 128, 4, 2, 32, 2)

#define SGEMM_GB300_CFG_STRUCT(NAME, BM, BN, BK, WM, WN, WNI, TM, TN, NT, ST, MINB, KU, OR)     \
  struct Cfg##NAME {                                                                            \
    static constexpr TileShape S{BM, BN, BK, WM, WN, WNI, TM, TN, NT, ST, MINB, KU, OR};        \
    static constexpr const char* name = #NAME "_" #BM "x" #BN "x" #BK "_w" #WM "x" #WN          \
                                        "_n" #WNI "_p" #TM "x" #TN "_t" #NT "_s" #ST "_u" #KU   \
                                        "_o" #OR;                                               \
  };
SGEMM_GB300_CONFIGS(SGEMM_GB300_CFG_STRUCT)
#undef SGEMM_GB300_CFG_STRUCT

// Launch of one operand-layout variant (al: ALoad, bl: BLoad, ffma_sgemm.cuh);
// map_a is used when A arrives by TMA, map_b when B does. Returns
// cudaErrorInvalidValue for a variant the configuration was not built with.
using LaunchFn = cudaError_t (*)(int al, int bl, int grid, const KernelParams& p,
                                 const CUtensorMap* map_a, const CUtensorMap* map_b,
                                 cudaStream_t stream);
using AttrFn = cudaError_t (*)();
using OccFn = cudaError_t (*)(int* blocks_per_sm);

struct ConfigEntry {
  const char* name;
  TileShape shape;
  int smem_bytes;      // dynamic shared memory per CTA, alignment slack included
  bool all_layouts;    // built for transposed operands too (else row-major A and B only)
  AttrFn set_attributes;
  OccFn occupancy;
  LaunchFn launch;
};

// Registry index of each configuration: kId<Name>.
#define SGEMM_GB300_CONFIG_ID(NAME, ...) kId##NAME,
enum ConfigId : int { SGEMM_GB300_CONFIGS(SGEMM_GB300_CONFIG_ID) kNumConfigIds };
#undef SGEMM_GB300_CONFIG_ID

// Defined in the cfg_*.cu translation units, one per configuration.
#define SGEMM_GB300_DECLARE_ENTRY(NAME, ...) extern const ConfigEntry kEntry##NAME;
SGEMM_GB300_CONFIGS(SGEMM_GB300_DECLARE_ENTRY)
#undef SGEMM_GB300_DECLARE_ENTRY

}  // namespace sgemm_gb300
