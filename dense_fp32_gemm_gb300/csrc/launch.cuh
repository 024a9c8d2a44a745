// launch.cuh -- per-configuration host entry points (attribute set-up,
// occupancy query, launch) around ffma_sgemm_kernel<>.
#pragma once

#include <cuda_runtime.h>

#include "configs.hpp"
#include "ffma_sgemm.cuh"

namespace sgemm_gb300 {

// kAll: instantiate every operand-layout variant (3 x 3); otherwise only the
// row-major ones (A transposed on store; B by TMA or by copy). Configurations
// that pass stg_eligible also get the staged-A variant (kARowStg, B by TMA),
// with its own shared-memory size and one more warp.
template <class Cfg, bool kAll>
struct Launcher {
  static constexpr int kSmem = kernel_smem_bytes<Cfg>();
  static constexpr bool kStgOk = stg_eligible(Cfg::S);
  static constexpr int kSmemStg = kStgOk ? kernel_smem_bytes_stg<Cfg>() : 0;

  template <int AL>
  static constexpr int smem_of() {
    return AL == kARowStg ? kSmemStg : kSmem;
  }

  template <int AL, int BL>
  static cudaError_t attr() {
    return cudaFuncSetAttribute(ffma_sgemm_kernel<Cfg, AL, BL>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, smem_of<AL>());
  }

  static cudaError_t set_attributes() {
    cudaError_t e = attr<kARow, kBRowTma>();
    if (e == cudaSuccess) e = attr<kARow, kBRowCp>();
    if constexpr (kStgOk) {
      if (e == cudaSuccess) e = attr<kARowStg, kBRowTma>();
    }
    if constexpr (kAll) {
      if (e == cudaSuccess) e = attr<kARow, kBT>();
      if (e == cudaSuccess) e = attr<kATTma, kBRowTma>();
      if (e == cudaSuccess) e = attr<kATTma, kBRowCp>();
      if (e == cudaSuccess) e = attr<kATTma, kBT>();
      if (e == cudaSuccess) e = attr<kATCp, kBRowTma>();
      if (e == cudaSuccess) e = attr<kATCp, kBRowCp>();
      if (e == cudaSuccess) e = attr<kATCp, kBT>();
    }
    return e;
  }

  // All variants share the shared-memory size and launch bounds; the
  // row-major TMA variant stands for them.
  static cudaError_t occupancy(int* blocks) {
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        blocks, ffma_sgemm_kernel<Cfg, kARow, kBRowTma>, Cfg::S.NT, kSmem);
  }
  // the staged-A variant (its own size and thread count)
  static cudaError_t occupancy_stg(int* blocks) {
    if constexpr (kStgOk) {
      return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
          blocks, ffma_sgemm_kernel<Cfg, kARowStg, kBRowTma>, kernel_threads<Cfg, kARowStg>(),
          kSmemStg);
    } else {
      *blocks = 0;
      return cudaSuccess;
    }
  }

  // Launched with programmatic stream serialization: the grid may start while
  // the kernel before it on the stream finishes (the kernel waits for it
  // before any global memory access).
  template <int AL, int BL>
  static cudaError_t go(int grid, const KernelParams& p, const CUtensorMap* ma,
                        const CUtensorMap* mb, cudaStream_t stream) {
#if SGEMM_GB300_PDL
    cudaLaunchConfig_t lc = {};
    cudaLaunchAttribute la[1];
    la[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    la[0].val.programmaticStreamSerializationAllowed = 1;
    lc.gridDim = dim3((unsigned)grid);
    lc.blockDim = dim3((unsigned)kernel_threads<Cfg, AL>());
    lc.dynamicSmemBytes = (size_t)smem_of<AL>();
    lc.stream = stream;
    lc.attrs = la;
    lc.numAttrs = 1;
    return cudaLaunchKernelEx(&lc, ffma_sgemm_kernel<Cfg, AL, BL>, p, *ma, *mb);
#else
    ffma_sgemm_kernel<Cfg, AL, BL>
        <<<grid, kernel_threads<Cfg, AL>(), smem_of<AL>(), stream>>>(p, *ma, *mb);
    return cudaGetLastError();
#endif
  }

  static cudaError_t launch(int al, int bl, int grid, const KernelParams& p,
                            const CUtensorMap* ma, const CUtensorMap* mb, cudaStream_t stream) {
    if (al == kARow && bl == kBRowTma) return go<kARow, kBRowTma>(grid, p, ma, mb, stream);
    if (al == kARow && bl == kBRowCp) return go<kARow, kBRowCp>(grid, p, ma, mb, stream);
    if constexpr (kStgOk) {
      if (al == kARowStg && bl == kBRowTma) return go<kARowStg, kBRowTma>(grid, p, ma, mb, stream);
    }
    if constexpr (kAll) {
      if (al == kARow && bl == kBT) return go<kARow, kBT>(grid, p, ma, mb, stream);
      if (al == kATTma && bl == kBRowTma) return go<kATTma, kBRowTma>(grid, p, ma, mb, stream);
      if (al == kATTma && bl == kBRowCp) return go<kATTma, kBRowCp>(grid, p, ma, mb, stream);
      if (al == kATTma && bl == kBT) return go<kATTma, kBT>(grid, p, ma, mb, stream);
      if (al == kATCp && bl == kBRowTma) return go<kATCp, kBRowTma>(grid, p, ma, mb, stream);
      if (al == kATCp && bl == kBRowCp) return go<kATCp, kBRowCp>(grid, p, ma, mb, stream);
      if (al == kATCp && bl == kBT) return go<kATCp, kBT>(grid, p, ma, mb, stream);
    }
    return cudaErrorInvalidValue;
  }

  static ConfigEntry entry() {
    return ConfigEntry{Cfg::name, Cfg::S,      kSmem,   kAll, &set_attributes,
                       &occupancy, &launch, kStgOk, &occupancy_stg};
  }
};

}  // namespace sgemm_gb300

// The registry entry of configuration NAME (one generated translation unit
// each): every operand-layout variant when the list marks it ALL_LAYOUTS,
// else the row-major ones.
#define SGEMM_GB300_DEFINE_CONFIG(NAME)                                          \
  namespace sgemm_gb300 {                                                        \
  const ConfigEntry kEntry##NAME = Launcher<Cfg##NAME, Cfg##NAME::all_layouts>::entry(); \
  }
