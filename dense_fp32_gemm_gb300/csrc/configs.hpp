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

// 128 x 256 CTA tile, 8 warps of 64 x 64, 16 x 8 accumulators per lane:
// the large-problem shape (B arrives by TMA, so a wide BN costs no loader
// instructions).
struct CfgWide {
  static constexpr TileShape S{128, 256, 16, 64, 64, 2, 4, 4, 256, 4, 1};
  static constexpr const char* name = "wide128x256x16_w64x64_t16x8_s4";
};
// 256 x 64 CTA tile, 4 warps of 64 x 64: for N <= 64 (skinny outputs).
struct CfgTall {
  static constexpr TileShape S{256, 64, 16, 64, 64, 2, 4, 4, 128, 4, 2};
  static constexpr const char* name = "tall256x64x16_w64x64_t16x8_s4";
};
// 128 x 128 CTA tile, 4 warps of 64 x 64, two CTAs per SM.
struct CfgSquare {
  static constexpr TileShape S{128, 128, 16, 64, 64, 2, 4, 4, 128, 4, 2};
  static constexpr const char* name = "square128x128x16_w64x64_t16x8_s4";
};
// The pages' sweep winner (128 x 64 x 16, warp 64 x 32, WNITER 2, 4 x 4
// patches, 128 threads) on this kernel's pipeline: 8 x 8 accumulators.
struct CfgPages {
  static constexpr TileShape S{128, 64, 16, 64, 32, 2, 4, 4, 128, 3, 4};
  static constexpr const char* name = "pages128x64x16_w64x32_t8x8_s3";
};

using LaunchFn = cudaError_t (*)(bool tma, int grid, const KernelParams& p, const CUtensorMap* map,
                                 cudaStream_t stream);
using AttrFn = cudaError_t (*)();
using OccFn = cudaError_t (*)(bool tma, int* blocks_per_sm);

struct ConfigEntry {
  const char* name;
  TileShape shape;
  int smem_bytes;      // dynamic shared memory per CTA, alignment slack included
  AttrFn set_attributes;
  OccFn occupancy;
  LaunchFn launch;
};

// Defined in the cfg_*.cu translation units.
extern const ConfigEntry kEntryWide;
extern const ConfigEntry kEntryTall;
extern const ConfigEntry kEntrySquare;
extern const ConfigEntry kEntryPages;

}  // namespace sgemm_gb300
