// launch.cuh -- per-configuration host entry points (attribute set-up,
// occupancy query, launch) around ffma_sgemm_kernel<>.
#pragma once

#include <cuda_runtime.h>

#include "configs.hpp"
#include "ffma_sgemm.cuh"

namespace sgemm_gb300 {

// kAll: instantiate every operand-layout variant (3 x 3); otherwise only the
// row-major ones (A transposed on store; B by TMA or by copy).
template <class Cfg, bool kAll>
struct Launcher {
  static constexpr int kSmem = kernel_smem_bytes<Cfg>();

  template <int AL, int BL>
  static cudaError_t attr() {
    return cudaFuncSetAttribute(ffma_sgemm_kernel<Cfg, AL, BL>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  }

  static cudaError_t set_attributes() {
    cudaError_t e = attr<kARow, kBRowTma>();
    if (e == cudaSuccess) e = attr<kARow, kBRowCp>();
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

  template <int AL, int BL>
  static cudaError_t go(int grid, const KernelParams& p, const CUtensorMap* ma,
                        const CUtensorMap* mb, cudaStream_t stream) {
    ffma_sgemm_kernel<Cfg, AL, BL><<<grid, Cfg::S.NT, kSmem, stream>>>(p, *ma, *mb);
    return cudaGetLastError();
  }

  static cudaError_t launch(int al, int bl, int grid, const KernelParams& p,
                            const CUtensorMap* ma, const CUtensorMap* mb, cudaStream_t stream) {
    if (al == kARow && bl == kBRowTma) return go<kARow, kBRowTma>(grid, p, ma, mb, stream);
    if (al == kARow && bl == kBRowCp) return go<kARow, kBRowCp>(grid, p, ma, mb, stream);
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
    return ConfigEntry{Cfg::name, Cfg::S, kSmem, kAll, &set_attributes, &occupancy, &launch};
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
