// probe.cu -- sgemm_diag_tf32_mma_rate(): the TF32 tensor-core throughput of
// this GPU, measured. The 3xTF32 path is measured against it (three TF32
// products per FP32 product), so its roofline rests on this device rather
// than on a nominal figure.
//
// One CTA per SM. Each CTA fills a 128 x 32 A tile and a 256 x 32 B tile in
// shared memory (K-major, 128-byte swizzle, the layout the 3xTF32 kernel's
// MMAs read) with small nonzero values, allocates a 256-column TMEM
// accumulator, and one thread issues `iters` x 4 back-to-back
// tcgen05.mma.cta_group::1.kind::tf32 of M 128, N 256, K 8 (no loads in the
// loop). The completion wait is bounded; a CTA that gives up records status
// 1 and still frees its TMEM. The host times the launch with CUDA events.
//
// sgemm_diag_tf32_pair_mma_rate() measures the same for the pair form the
// 3xTF32 path runs by default: clusters of two CTAs, the even CTA issuing
// tcgen05.mma.cta_group::2 of M 256 (128 rows per CTA), N 256 (each CTA
// holding a 128-row half of B), K 8; per SM the same multiply-adds as above.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/sgemm_gb300.h"
#include "ptx.cuh"
#include "tcgen05.cuh"

#define SGEMM_API extern "C" __attribute__((visibility("default")))

namespace sgemm_gb300 {

int library_device_sms(int dev, int* sms);

namespace probe {

constexpr int BM = 128, BN = 256, BK = 32;
constexpr int A_BYTES = BM * BK * 4, B_BYTES = BN * BK * 4;
constexpr int SMEM_BYTES = 1024 + A_BYTES + B_BYTES + 64;
constexpr uint32_t IDESC = tc::idesc_tf32(BM, BN);

__global__ void __launch_bounds__(128, 1) tf32_mma_kernel(int iters, int* status,
                                                          long long timeout_ns) {
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = ptx::smem_addr(smem_raw);
  unsigned char* base = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  float* tiles = reinterpret_cast<float*>(base);
  uint64_t* bar = reinterpret_cast<uint64_t*>(base + A_BYTES + B_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 1);
  const int tid = threadIdx.x, warp = tid >> 5;

  // operands: small nonzero values (the data reaches the tensor cores as it
  // would in a real product)
  for (int i = tid; i < (A_BYTES + B_BYTES) / 4; i += blockDim.x)
    tiles[i] = 0.25f + 0.001f * (float)((i * 37 + blockIdx.x) & 255);
  if (tid == 0) {
    ptx::mbar_init(ptx::smem_addr(bar), 1);
    ptx::mbar_fence_init();
  }
  ptx::fence_proxy_async_shared();  // the MMAs read the tiles through the async proxy
  if (warp == 1) {
    tc::tmem_alloc(ptx::smem_addr(tmem_slot), BN);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (tid == 0) {
    const uint32_t a0 = ptx::smem_addr(base), b0 = a0 + A_BYTES;
    for (int it = 0; it < iters; ++it) {
#pragma unroll
      for (int kk = 0; kk < BK / 8; ++kk) {
        const uint32_t koff = (uint32_t)(kk * 32);
        tc::mma_tf32(tmem, tc::smem_desc_k_swizzled<128>(a0 + koff),
                     tc::smem_desc_k_swizzled<128>(b0 + koff), IDESC,
                     (it == 0 && kk == 0) ? 0u : 1u);
      }
    }
    tc::commit(ptx::smem_addr(bar));
    const uint64_t t0 = ptx::global_ns();
    while (!ptx::mbar_try_wait(ptx::smem_addr(bar), 0u)) {
      if ((long long)(ptx::global_ns() - t0) > timeout_ns) {
        atomicCAS(status, 0, 1);
        break;
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, BN);
  }
}

constexpr int B_HALF_BYTES = BN / 2 * BK * 4;
constexpr int PAIR_SMEM_BYTES = 1024 + A_BYTES + B_HALF_BYTES + 64;
constexpr uint32_t IDESC_PAIR = tc::idesc_tf32(2 * BM, BN);

__global__ void __launch_bounds__(128, 1) tf32_pair_mma_kernel(int iters, int* status,
                                                               long long timeout_ns) {
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = ptx::smem_addr(smem_raw);
  unsigned char* base = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  float* tiles = reinterpret_cast<float*>(base);
  uint64_t* bar = reinterpret_cast<uint64_t*>(base + A_BYTES + B_HALF_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 1);
  const int tid = threadIdx.x, warp = tid >> 5;
  const uint32_t rank = ptx::cluster_ctarank();

  for (int i = tid; i < (A_BYTES + B_HALF_BYTES) / 4; i += blockDim.x)
    tiles[i] = 0.25f + 0.001f * (float)((i * 37 + blockIdx.x) & 255);
  if (tid == 0) {
    ptx::mbar_init(ptx::smem_addr(bar), 1);
    ptx::mbar_fence_init();
  }
  ptx::fence_proxy_async_shared();
  if (warp == 1) {
    tc::tmem_alloc<2>(ptx::smem_addr(tmem_slot), BN);
    tc::tmem_relinquish<2>();
  }
  tc::fence_before_sync();
  __syncthreads();
  ptx::cluster_sync();  // both CTAs' tiles and barriers are ready
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (tid == 0) {
    if (rank == 0) {
      const uint32_t a0 = ptx::smem_addr(base), b0 = a0 + A_BYTES;
      for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int kk = 0; kk < BK / 8; ++kk) {
          const uint32_t koff = (uint32_t)(kk * 32);
          tc::mma_tf32_pair(tmem, tc::smem_desc_k_swizzled<128>(a0 + koff),
                            tc::smem_desc_k_swizzled<128>(b0 + koff), IDESC_PAIR,
                            (it == 0 && kk == 0) ? 0u : 1u);
        }
      }
      tc::commit_pair_multicast(ptx::smem_addr(bar), 0x3);
    }
    // both CTAs wait for the MMAs (the commit arrives on both barriers)
    const uint64_t t0 = ptx::global_ns();
    while (!ptx::mbar_try_wait(ptx::smem_addr(bar), 0u)) {
      if ((long long)(ptx::global_ns() - t0) > timeout_ns) {
        atomicCAS(status, 0, 1);
        break;
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  ptx::cluster_sync();  // the even CTA's MMAs wrote the odd CTA's TMEM
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc<2>(tmem, BN);
  }
}

}  // namespace probe
}  // namespace sgemm_gb300

using namespace sgemm_gb300;

SGEMM_API int sgemm_diag_tf32_mma_rate(int iters, double* tflops) {
  if (iters < 1 || tflops == nullptr) return SGEMM_ERR_INVALID_VALUE;
  *tflops = 0.0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return SGEMM_ERR_LAUNCH;
  }
  int sms = 0;
  int st = library_device_sms(dev, &sms);  // also rejects devices other than sm_103
  if (st != SGEMM_OK) return st;
  if (cudaFuncSetAttribute(probe::tf32_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           probe::SMEM_BYTES) != cudaSuccess) {
    cudaGetLastError();
    return SGEMM_ERR_LAUNCH;
  }
  int* status = nullptr;
  cudaStream_t stream = nullptr;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  st = SGEMM_ERR_LAUNCH;
  if (cudaMalloc(&status, sizeof(int)) == cudaSuccess &&
      cudaMemset(status, 0, sizeof(int)) == cudaSuccess &&
      cudaStreamCreateWithFlags(&stream, cudaStreamNonBlocking) == cudaSuccess &&
      cudaEventCreate(&e0) == cudaSuccess && cudaEventCreate(&e1) == cudaSuccess) {
    const long long timeout_ns = 4000000000LL;
    // one warm-up launch, then the timed one
    probe::tf32_mma_kernel<<<sms, 128, probe::SMEM_BYTES, stream>>>(1, status, timeout_ns);
    cudaEventRecord(e0, stream);
    probe::tf32_mma_kernel<<<sms, 128, probe::SMEM_BYTES, stream>>>(iters, status, timeout_ns);
    cudaEventRecord(e1, stream);
    float ms = 0.f;
    int code = 0;
    if (cudaGetLastError() == cudaSuccess && cudaEventSynchronize(e1) == cudaSuccess &&
        cudaEventElapsedTime(&ms, e0, e1) == cudaSuccess &&
        cudaMemcpy(&code, status, sizeof(int), cudaMemcpyDeviceToHost) == cudaSuccess) {
      if (code != 0) {
        st = SGEMM_ERR_DEVICE_TIMEOUT;
      } else {
        const double flop = 2.0 * probe::BM * probe::BN * probe::BK * (double)iters * sms;
        *tflops = flop / (ms * 1e-3) / 1e12;
        st = SGEMM_OK;
      }
    }
  }
  cudaGetLastError();
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  if (stream) cudaStreamDestroy(stream);
  if (status) cudaFree(status);
  return st;
}

SGEMM_API int sgemm_diag_tf32_pair_mma_rate(int iters, double* tflops) {
  if (iters < 1 || tflops == nullptr) return SGEMM_ERR_INVALID_VALUE;
  *tflops = 0.0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return SGEMM_ERR_LAUNCH;
  }
  int sms = 0;
  int st = library_device_sms(dev, &sms);
  if (st != SGEMM_OK) return st;
  if (cudaFuncSetAttribute(probe::tf32_pair_mma_kernel,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           probe::PAIR_SMEM_BYTES) != cudaSuccess) {
    cudaGetLastError();
    return SGEMM_ERR_LAUNCH;
  }
  cudaLaunchConfig_t lc = {};
  cudaLaunchAttribute la[1];
  la[0].id = cudaLaunchAttributeClusterDimension;
  la[0].val.clusterDim.x = 2;
  la[0].val.clusterDim.y = 1;
  la[0].val.clusterDim.z = 1;
  lc.blockDim = dim3(128);
  lc.dynamicSmemBytes = probe::PAIR_SMEM_BYTES;
  lc.attrs = la;
  lc.numAttrs = 1;
  // as many clusters as are resident at once, so that all run together
  lc.gridDim = dim3((unsigned)(2 * (sms / 2)));
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, probe::tf32_pair_mma_kernel, &lc) != cudaSuccess ||
      clusters < 1) {
    cudaGetLastError();
    return SGEMM_ERR_LAUNCH;
  }
  if (clusters > sms / 2) clusters = sms / 2;
  lc.gridDim = dim3((unsigned)(2 * clusters));
  int* status = nullptr;
  cudaStream_t stream = nullptr;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  st = SGEMM_ERR_LAUNCH;
  if (cudaMalloc(&status, sizeof(int)) == cudaSuccess &&
      cudaMemset(status, 0, sizeof(int)) == cudaSuccess &&
      cudaStreamCreateWithFlags(&stream, cudaStreamNonBlocking) == cudaSuccess &&
      cudaEventCreate(&e0) == cudaSuccess && cudaEventCreate(&e1) == cudaSuccess) {
    lc.stream = stream;
    const long long timeout_ns = 4000000000LL;
    // one warm-up launch, then the timed one
    bool ok = cudaLaunchKernelEx(&lc, probe::tf32_pair_mma_kernel, 1, status, timeout_ns) ==
              cudaSuccess;
    ok = ok && cudaEventRecord(e0, stream) == cudaSuccess;
    ok = ok && cudaLaunchKernelEx(&lc, probe::tf32_pair_mma_kernel, iters, status, timeout_ns) ==
                   cudaSuccess;
    ok = ok && cudaEventRecord(e1, stream) == cudaSuccess;
    float ms = 0.f;
    int code = 0;
    if (ok && cudaEventSynchronize(e1) == cudaSuccess &&
        cudaEventElapsedTime(&ms, e0, e1) == cudaSuccess &&
        cudaMemcpy(&code, status, sizeof(int), cudaMemcpyDeviceToHost) == cudaSuccess) {
      if (code != 0) {
        st = SGEMM_ERR_DEVICE_TIMEOUT;
      } else {
        // per SM (each CTA's 128 rows): 2 * 128 * 256 * 32 per iteration
        const double flop = 2.0 * probe::BM * probe::BN * probe::BK * (double)iters * 2 * clusters;
        *tflops = flop / (ms * 1e-3) / 1e12;
        st = SGEMM_OK;
      }
    }
  }
  cudaGetLastError();
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  if (stream) cudaStreamDestroy(stream);
  if (status) cudaFree(status);
  return st;
}
