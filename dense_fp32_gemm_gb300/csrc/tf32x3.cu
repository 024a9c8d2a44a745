// tf32x3.cu -- sgemm_3xtf32(): the same C = alpha * A * B + beta * C as
// sgemm(), computed on the tensor cores with three TF32 products per FP32
// product (an opt-in path; the pages stop at FP32 FFMA kernels).
//
// Method (split-operand TF32, after Ootomo and Yokota, "Recovering single
// precision accuracy from Tensor Cores while surpassing the FP32 theoretical
// peak performance", 2022): each FP32 operand x is written as
// x = x_hi + x_lo + r with x_hi = x truncated to TF32 (low 13 mantissa bits
// cleared) and x_lo = (x - x_hi) truncated to TF32, |r| < 2^-20 |x|. Then
//   a*b ~= a_hi*b_hi + a_hi*b_lo + a_lo*b_hi
// (the dropped a_lo*b_lo and the residuals are below 3 * 2^-20 |a||b|), each
// product on the TF32 tensor cores with FP32 accumulation. Integer inputs up
// to 2^11 in magnitude are exact TF32 values (x_lo = 0), so they stay exact.
//
// Data flow:
//   1. split kernels write A_hi, A_lo (M x K, K-major) and the transposed
//      B_hi, B_lo (N x K, K-major) into the per-stream workspace, with rows
//      padded to a multiple of 4 floats for TMA;
//   2. the GEMM kernel (one CTA of 6 warps per SM, persistent over 128 x 256
//      tiles): warp 0 issues TMA loads of the four operand tiles of each
//      32-wide k-slice (128-byte swizzle) into a 2-stage ring; warp 1 owns a
//      256-column TMEM accumulator and issues, per 8-wide k-step, the three
//      tcgen05.mma.kind::tf32 products; warps 2-5 read the accumulator back
//      with tcgen05.ld and apply alpha * acc + beta * C.
// Every wait is bounded (see ffma_sgemm.cuh); a CTA that gives up drains its
// copies and MMAs, frees its TMEM and returns.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/sgemm_gb300.h"
#include "ffma_sgemm.cuh"
#include "ptx.cuh"
#include "schedule.hpp"
#include "tcgen05.cuh"

#define SGEMM_API extern "C" __attribute__((visibility("default")))

namespace sgemm_gb300 {

// Provided by api.cu.
int library_workspace(int dev, cudaStream_t stream, size_t floats, float** scratch, int** status);
int library_device_sms(int dev, int* sms);
void note_last_config(const char* text);
long long library_wait_timeout_ns();

namespace x3 {

constexpr int BM = 128, BN = 256, BK = 32, ST = 2, NT = 192;
constexpr int A_BYTES = BM * BK * 4;                      // 16 KB
constexpr int B_BYTES = BN * BK * 4;                      // 32 KB
constexpr int STAGE_BYTES = 2 * A_BYTES + 2 * B_BYTES;   // 96 KB
constexpr int TMEM_COLS = 256;
constexpr uint32_t IDESC = tc::idesc_tf32(BM, BN);
static_assert(BN % 16 == 0 && BN <= 256 && BM == 128, "MMA shape");

struct Barriers {
  uint64_t full[ST];     // TMA transaction bytes of one stage
  uint64_t empty[ST];    // MMAs that read a stage have completed
  uint64_t tmem_full;    // the tile's last MMA has completed
  uint64_t tmem_empty;   // the epilogue warps have read the accumulator
  uint64_t drain;        // final MMA completion on the abort path
  uint32_t tmem_addr;
  int abort;
};
constexpr int SMEM_BYTES = 1024 + ST * STAGE_BYTES + (int)sizeof(Barriers);

struct Params {
  int M, N, K;
  float alpha, beta;
  float* C;
  long long ldc;
  Schedule sched;   // tile numbering (whole tiles only, round-robin)
  int* status;
  long long timeout_ns;
};

__device__ __forceinline__ float tf32_trunc(float x) {
  return __uint_as_float(__float_as_uint(x) & 0xFFFFE000u);
}

// A (M x K, lda) -> A_hi, A_lo (M x K, ldw).
__global__ void split_a_kernel(int M, int K, const float* __restrict__ A, long long lda,
                               float* __restrict__ hi, float* __restrict__ lo, long long ldw) {
  const long long total = (long long)M * K;
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
       e += (long long)gridDim.x * blockDim.x) {
    const long long m = e / K, k = e % K;
    const float x = A[m * lda + k];
    const float h = tf32_trunc(x);
    hi[m * ldw + k] = h;
    lo[m * ldw + k] = tf32_trunc(x - h);
  }
}

// B (K x N, ldb) -> transposed B_hi, B_lo (N x K, ldw), through 32 x 32
// shared-memory tiles so that both the reads and the writes are coalesced.
__global__ void split_bt_kernel(int K, int N, const float* __restrict__ B, long long ldb,
                                float* __restrict__ hi, float* __restrict__ lo, long long ldw) {
  __shared__ float tile[32][33];
  const int n0 = blockIdx.x * 32, k0 = blockIdx.y * 32;
  const int tx = threadIdx.x, ty = threadIdx.y;  // 32 x 8 threads
  for (int j = 0; j < 32; j += 8) {
    const int k = k0 + ty + j, n = n0 + tx;
    tile[ty + j][tx] = (k < K && n < N) ? B[(long long)k * ldb + n] : 0.f;
  }
  __syncthreads();
  for (int j = 0; j < 32; j += 8) {
    const int n = n0 + ty + j, k = k0 + tx;
    if (n < N && k < K) {
      const float x = tile[tx][ty + j];
      const float h = tf32_trunc(x);
      hi[(long long)n * ldw + k] = h;
      lo[(long long)n * ldw + k] = tf32_trunc(x - h);
    }
  }
}

__global__ void scale_c_kernel(int M, int N, float beta, float* C, long long ldc) {
  const long long total = (long long)M * N;
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
       e += (long long)gridDim.x * blockDim.x) {
    const long long i = e / N, j = e % N;
    float* c = C + i * ldc + j;
    *c = beta == 0.f ? 0.f : beta * *c;
  }
}

__global__ void __launch_bounds__(NT, 1)
    gemm_kernel(const __grid_constant__ Params p, const __grid_constant__ CUtensorMap tmA_hi,
                const __grid_constant__ CUtensorMap tmA_lo, const __grid_constant__ CUtensorMap tmB_hi,
                const __grid_constant__ CUtensorMap tmB_lo) {
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw_addr = ptx::smem_addr(smem_raw);
  unsigned char* base = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  Barriers* bar = reinterpret_cast<Barriers*>(base + ST * STAGE_BYTES);
  volatile int* abort_w = &bar->abort;
  const uint32_t base_addr = ptx::smem_addr(base);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const Schedule& sc = p.sched;
  const int kiters = sc.kiters;

  if (tid == 0) {
    for (int s = 0; s < ST; ++s) {
      ptx::mbar_init(ptx::smem_addr(&bar->full[s]), 1);
      ptx::mbar_init(ptx::smem_addr(&bar->empty[s]), 1);
    }
    ptx::mbar_init(ptx::smem_addr(&bar->tmem_full), 1);
    ptx::mbar_init(ptx::smem_addr(&bar->tmem_empty), 4);
    ptx::mbar_init(ptx::smem_addr(&bar->drain), 1);
    bar->abort = 0;
    ptx::mbar_fence_init();
    ptx::tma_prefetch_desc(&tmA_hi);
    ptx::tma_prefetch_desc(&tmA_lo);
    ptx::tma_prefetch_desc(&tmB_hi);
    ptx::tma_prefetch_desc(&tmB_lo);
  }
  if (warp == 1) {
    tc::tmem_alloc(ptx::smem_addr(&bar->tmem_addr), TMEM_COLS);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = bar->tmem_addr;

  if (warp == 0) {
    // ---- TMA producer ---------------------------------------------------------
    if (lane == 0) {
      int it = 0;
      for (int t = blockIdx.x; t < sc.tiles && !*abort_w; t += gridDim.x) {
        int tm, tn;
        tile_coords(sc, t, tm, tn);
        for (int kb = 0; kb < kiters; ++kb, ++it) {
          const int s = it % ST;
          const uint32_t par = (uint32_t)((it / ST) & 1) ^ 1u;
          if (!bounded_wait(ptx::smem_addr(&bar->empty[s]), par, abort_w, p.status,
                            kDevTimeoutEmpty, p.timeout_ns))
            break;
          const uint32_t fb = ptx::smem_addr(&bar->full[s]);
          const uint32_t st0 = base_addr + (uint32_t)(s * STAGE_BYTES);
          ptx::mbar_arrive_expect_tx(fb, (uint32_t)STAGE_BYTES);
          ptx::tma_load_2d(st0, &tmA_hi, kb * BK, tm * BM, fb);
          ptx::tma_load_2d(st0 + A_BYTES, &tmA_lo, kb * BK, tm * BM, fb);
          ptx::tma_load_2d(st0 + 2 * A_BYTES, &tmB_hi, kb * BK, tn * BN, fb);
          ptx::tma_load_2d(st0 + 2 * A_BYTES + B_BYTES, &tmB_lo, kb * BK, tn * BN, fb);
        }
      }
      // nothing may land after the CTA is gone: wait (bounded) for the last
      // stages issued
      const uint64_t t0 = ptx::global_ns();
      for (int j = it - 1; j >= 0 && j >= it - ST; --j) {
        const uint32_t fb = ptx::smem_addr(&bar->full[j % ST]);
        while (!ptx::mbar_try_wait(fb, (uint32_t)((j / ST) & 1)))
          if ((long long)(ptx::global_ns() - t0) > p.timeout_ns) break;
      }
    }
  } else if (warp == 1) {
    // ---- MMA issuer -----------------------------------------------------------
    if (lane == 0) {
      int it = 0, tcount = 0;
      bool issued_any = false;
      for (int t = blockIdx.x; t < sc.tiles && !*abort_w; t += gridDim.x, ++tcount) {
        // the epilogue must have read the previous tile's accumulator
        if (!bounded_wait(ptx::smem_addr(&bar->tmem_empty), (uint32_t)(tcount & 1) ^ 1u, abort_w,
                          p.status, kDevTimeoutSync, p.timeout_ns))
          break;
        tc::fence_after_sync();
        bool ok = true;
        for (int kb = 0; kb < kiters; ++kb, ++it) {
          const int s = it % ST;
          if (!bounded_wait(ptx::smem_addr(&bar->full[s]), (uint32_t)((it / ST) & 1), abort_w,
                            p.status, kDevTimeoutFull, p.timeout_ns)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t st0 = base_addr + (uint32_t)(s * STAGE_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / 8; ++kk) {
            const uint32_t koff = (uint32_t)(kk * 32);  // 8 TF32 values = 32 bytes
            const uint64_t a_hi = tc::smem_desc_k_sw128(st0 + koff);
            const uint64_t a_lo = tc::smem_desc_k_sw128(st0 + A_BYTES + koff);
            const uint64_t b_hi = tc::smem_desc_k_sw128(st0 + 2 * A_BYTES + koff);
            const uint64_t b_lo = tc::smem_desc_k_sw128(st0 + 2 * A_BYTES + B_BYTES + koff);
            const uint32_t first = (kb == 0 && kk == 0) ? 0u : 1u;
            tc::mma_tf32(tmem, a_hi, b_hi, IDESC, first);
            tc::mma_tf32(tmem, a_hi, b_lo, IDESC, 1u);
            tc::mma_tf32(tmem, a_lo, b_hi, IDESC, 1u);
          }
          issued_any = true;
          tc::commit(ptx::smem_addr(&bar->empty[s]));  // frees the stage when done
        }
        if (!ok) break;
        tc::commit(ptx::smem_addr(&bar->tmem_full));  // the tile's accumulator is ready
      }
      if (*abort_w && issued_any) {
        // wait (bounded) until every MMA issued has completed
        tc::commit(ptx::smem_addr(&bar->drain));
        const uint64_t t0 = ptx::global_ns();
        while (!ptx::mbar_try_wait(ptx::smem_addr(&bar->drain), 0u))
          if ((long long)(ptx::global_ns() - t0) > p.timeout_ns) break;
      }
    }
  } else {
    // ---- epilogue warps 2-5: TMEM -> registers -> C ---------------------------
    const int quarter = warp & 3;                 // TMEM lanes 32*quarter .. +31
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    int tcount = 0;
    for (int t = blockIdx.x; t < sc.tiles && !*abort_w; t += gridDim.x, ++tcount) {
      const bool ok = bounded_wait(ptx::smem_addr(&bar->tmem_full), (uint32_t)(tcount & 1),
                                   abort_w, p.status, kDevTimeoutFull, p.timeout_ns);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc::fence_after_sync();
      int tm, tn;
      tile_coords(sc, t, tm, tn);
      const int row = tm * BM + quarter * 32 + lane;
      const bool row_ok = row < p.M;
      float* crow = p.C + (long long)(row_ok ? row : 0) * p.ldc;
      const bool vec = ((reinterpret_cast<uintptr_t>(p.C) & 15u) == 0) && ((p.ldc & 3) == 0);
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 16) {
        uint32_t r[16];
        tc::tmem_ld16(tmem + lane_base + (uint32_t)c0, r);
        tc::tmem_wait_ld();
        if (!row_ok) continue;
        const int col0 = tn * BN + c0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int col = col0 + q * 4;
          float v[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) v[e] = p.alpha * __uint_as_float(r[q * 4 + e]);
          if (vec && col + 3 < p.N) {
            float4 o = make_float4(v[0], v[1], v[2], v[3]);
            if (p.beta != 0.f) {
              const float4 c = *reinterpret_cast<const float4*>(crow + col);
              o.x = fmaf(p.beta, c.x, v[0]);
              o.y = fmaf(p.beta, c.y, v[1]);
              o.z = fmaf(p.beta, c.z, v[2]);
              o.w = fmaf(p.beta, c.w, v[3]);
            }
            *reinterpret_cast<float4*>(crow + col) = o;
          } else {
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if (col + e < p.N)
                crow[col + e] = p.beta != 0.f ? fmaf(p.beta, crow[col + e], v[e]) : v[e];
          }
        }
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&bar->tmem_empty));
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, TMEM_COLS);
  }
}

// Per-device set-up (shared-memory attribute), guarded by g_mutex.
std::mutex g_mutex;
bool g_ready[64];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
bool g_encode_tried = false;

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  if (!g_encode_tried) {
    g_encode_tried = true;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return g_encode;
}

bool encode_k_major(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap* map, const float* base,
                    int rows, int K, long long ldw, int box_rows) {
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ldw * 4};
  cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace x3
}  // namespace sgemm_gb300

using namespace sgemm_gb300;

SGEMM_API int sgemm_3xtf32(int M, int N, int K, float alpha, const float* A, int lda,
                           const float* B, int ldb, float beta, float* C, int ldc, void* stream_) {
  if (M < 0 || N < 0 || K < 0) return SGEMM_ERR_INVALID_DIM;
  if (lda < (K > 1 ? K : 1) || ldb < (N > 1 ? N : 1) || ldc < (N > 1 ? N : 1))
    return SGEMM_ERR_INVALID_LD;
  if (M == 0 || N == 0) return SGEMM_OK;
  const bool reads_ab = (K > 0 && alpha != 0.f);
  if (C == nullptr || (reads_ab && (A == nullptr || B == nullptr))) return SGEMM_ERR_NULL_PTR;
  if ((reinterpret_cast<uintptr_t>(C) & 3u) ||
      (reads_ab && ((reinterpret_cast<uintptr_t>(A) & 3u) || (reinterpret_cast<uintptr_t>(B) & 3u))))
    return SGEMM_ERR_MISALIGNED;

  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return SGEMM_ERR_LAUNCH;
  }
  int sms = 0;
  int st = library_device_sms(dev, &sms);
  if (st != SGEMM_OK) return st;

  if (!reads_ab) {
    const long long total = (long long)M * N;
    int blocks = (int)((total + 255) / 256);
    if (blocks > sms * 8) blocks = sms * 8;
    x3::scale_c_kernel<<<blocks, 256, 0, stream>>>(M, N, beta, C, ldc);
    return cudaGetLastError() == cudaSuccess ? SGEMM_OK : SGEMM_ERR_LAUNCH;
  }

  {
    std::lock_guard<std::mutex> lock(x3::g_mutex);
    if (dev < 0 || dev >= 64) return SGEMM_ERR_UNSUPPORTED_DEVICE;
    if (!x3::g_ready[dev]) {
      if (cudaFuncSetAttribute(x3::gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               x3::SMEM_BYTES) != cudaSuccess) {
        cudaGetLastError();
        return SGEMM_ERR_LAUNCH;
      }
      x3::g_ready[dev] = true;
    }
  }
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  {
    std::lock_guard<std::mutex> lock(x3::g_mutex);
    enc = x3::encoder();
  }
  if (enc == nullptr) return SGEMM_ERR_LAUNCH;

  // workspace: A_hi, A_lo (M x Kp) and B_hi, B_lo transposed (N x Kp)
  const long long Kp = ((long long)K + 3) / 4 * 4;
  const size_t floats = (size_t)(2 * (long long)M * Kp + 2 * (long long)N * Kp);
  float* ws = nullptr;
  int* status = nullptr;
  st = library_workspace(dev, stream, floats, &ws, &status);
  if (st != SGEMM_OK) return st;
  float* a_hi = ws;
  float* a_lo = a_hi + (size_t)M * Kp;
  float* b_hi = a_lo + (size_t)M * Kp;
  float* b_lo = b_hi + (size_t)N * Kp;

  // 1. split (and transpose B)
  {
    const long long total = (long long)M * K;
    int blocks = (int)((total + 255) / 256);
    if (blocks > sms * 16) blocks = sms * 16;
    x3::split_a_kernel<<<blocks, 256, 0, stream>>>(M, K, A, lda, a_hi, a_lo, Kp);
    dim3 grid((N + 31) / 32, (K + 31) / 32), block(32, 8);
    x3::split_bt_kernel<<<grid, block, 0, stream>>>(K, N, B, ldb, b_hi, b_lo, Kp);
    if (cudaGetLastError() != cudaSuccess) return SGEMM_ERR_LAUNCH;
  }

  // 2. tensor-core GEMM
  CUtensorMap mA_hi, mA_lo, mB_hi, mB_lo;
  if (!x3::encode_k_major(enc, &mA_hi, a_hi, M, K, Kp, x3::BM) ||
      !x3::encode_k_major(enc, &mA_lo, a_lo, M, K, Kp, x3::BM) ||
      !x3::encode_k_major(enc, &mB_hi, b_hi, N, K, Kp, x3::BN) ||
      !x3::encode_k_major(enc, &mB_lo, b_lo, N, K, Kp, x3::BN))
    return SGEMM_ERR_LAUNCH;
  x3::Params p;
  p.M = M;
  p.N = N;
  p.K = K;
  p.alpha = alpha;
  p.beta = beta;
  p.C = C;
  p.ldc = ldc;
  const int tiles_m = (M + x3::BM - 1) / x3::BM, tiles_n = (N + x3::BN - 1) / x3::BN;
  const int kiters = (K + x3::BK - 1) / x3::BK;
  // whole tiles only (a minimum split of 2^20 k-slices disables the split)
  p.sched = make_schedule(tiles_m, tiles_n, kiters, sms, 8, 1 << 20);
  p.status = status;
  p.timeout_ns = library_wait_timeout_ns();
  x3::gemm_kernel<<<p.sched.grid, x3::NT, x3::SMEM_BYTES, stream>>>(p, mA_hi, mA_lo, mB_hi, mB_lo);
  if (cudaGetLastError() != cudaSuccess) return SGEMM_ERR_LAUNCH;
  char text[160];
  snprintf(text, sizeof(text), "3xtf32_tcgen05_%dx%dx%d_s%d grid=%d tiles=%d kiters=%d", x3::BM,
           x3::BN, x3::BK, x3::ST, p.sched.grid, p.sched.tiles, kiters);
  note_last_config(text);
  return SGEMM_OK;
}
