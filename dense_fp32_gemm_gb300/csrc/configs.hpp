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

// Every configuration compiled into the library, in registry order, as the
// X-macro list SGEMM_GB300_CONFIGS(X) with rows
//   X(Name, BM, BN, BK, WM, WN, WNITER, TM, TN, NT, STAGES, MINB, KU, ORDER, ALL_LAYOUTS)
// and SGEMM_GB300_FALLBACK_CONFIG (a configuration built for every operand
// layout, for transposed operands whose class winner is built for row-major
// operands only). The list is generated (configgen.py enumerates and prunes
// the legal space, tune.py keeps the measured winners); a build for the
// tuner's candidate set passes its own list as SGEMM_GB300_CONFIG_LIST.
#ifdef SGEMM_GB300_CONFIG_LIST
#include SGEMM_GB300_CONFIG_LIST
#else
#include "configs.inc"
#endif

#define SGEMM_GB300_CFG_STRUCT(NAME, BM, BN, BK, WM, WN, WNI, TM, TN, NT, ST, MINB, KU, OR, ALL) \
  struct Cfg##NAME {                                                                           \
    static constexpr TileShape S{BM, BN, BK, WM, WN, WNI, TM, TN, NT, ST, MINB, KU, OR};       \
    static constexpr bool all_layouts = (ALL) != 0;                                            \
    static constexpr const char* name = #NAME;                                                 \
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
  bool staged;         // built with the staged-A variant (ALoad kARowStg)
  OccFn occupancy_staged;  // its resident CTAs per SM (0 when not built)
};

// Registry index of each configuration: kId<Name>.
#define SGEMM_GB300_CONFIG_ID(NAME, ...) kId##NAME,
enum ConfigId : int { SGEMM_GB300_CONFIGS(SGEMM_GB300_CONFIG_ID) kNumConfigIds };
#undef SGEMM_GB300_CONFIG_ID

#define SGEMM_GB300_CAT2(a, b) a##b
#define SGEMM_GB300_CAT(a, b) SGEMM_GB300_CAT2(a, b)
// The configuration for operand layouts the class winner is not built for.
constexpr int kFallbackConfigId = SGEMM_GB300_CAT(kId, SGEMM_GB300_FALLBACK_CONFIG);

// Defined in the generated translation units, one per configuration.
#define SGEMM_GB300_DECLARE_ENTRY(NAME, ...) extern const ConfigEntry kEntry##NAME;
SGEMM_GB300_CONFIGS(SGEMM_GB300_DECLARE_ENTRY)
#undef SGEMM_GB300_DECLARE_ENTRY

}  // namespace sgemm_gb300
