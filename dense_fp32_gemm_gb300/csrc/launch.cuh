// launch.cuh -- per-configuration host entry points (attribute set-up,
// occupancy query, launch) around ffma_sgemm_kernel<>.
#pragma once

#include <cuda_runtime.h>

#include "configs.hpp"
#include "ffma_sgemm.cuh"

namespace sgemm_gb300 {

template <class Cfg>
struct Launcher {
  static constexpr int kSmem = kernel_smem_bytes<Cfg>();

  static cudaError_t set_attributes() {
    cudaError_t e = cudaFuncSetAttribute(ffma_sgemm_kernel<Cfg, true>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(ffma_sgemm_kernel<Cfg, false>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  }

  static cudaError_t occupancy(bool tma, int* blocks) {
    return tma ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                     blocks, ffma_sgemm_kernel<Cfg, true>, Cfg::S.NT, kSmem)
               : cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                     blocks, ffma_sgemm_kernel<Cfg, false>, Cfg::S.NT, kSmem);
  }

  static cudaError_t launch(bool tma, int grid, const KernelParams& p, const CUtensorMap* map,
                            cudaStream_t stream) {
    if (tma)
      ffma_sgemm_kernel<Cfg, true><<<grid, Cfg::S.NT, kSmem, stream>>>(p, *map);
    else
      ffma_sgemm_kernel<Cfg, false><<<grid, Cfg::S.NT, kSmem, stream>>>(p, *map);
    return cudaGetLastError();
  }

  static ConfigEntry entry() {
    return ConfigEntry{Cfg::name, Cfg::S, kSmem, &set_attributes, &occupancy, &launch};
  }
};

}  // namespace sgemm_gb300

#define SGEMM_GB300_DEFINE_ENTRY(CFG, VAR) \
  const ::sgemm_gb300::ConfigEntry VAR = ::sgemm_gb300::Launcher<::sgemm_gb300::CFG>::entry();
