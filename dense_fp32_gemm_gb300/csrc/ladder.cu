// ladder.cu -- sgemm_ladder(): three kernels of the pages' series, rebuilt for
// sm_103a so that what each technique buys can be measured on this GPU:
//
//   3  shared-memory tiling ("Shared Memory Tiling"): a 32 x 32 C tile per
//      CTA of 1024 threads, one output per thread; each k-slice of 32 is
//      staged in shared memory by one load per thread and read back twice
//      per FMA;
//   7  vectorized 2-D block tiling ("Vectorized Memory Access: 128-bit Loads
//      and Stores"): a 128 x 128 C tile per CTA of 256 threads, 8 x 8 outputs
//      per thread, BK = 8; 128-bit global loads, A stored transposed in
//      shared memory (As[k][m]) so that a thread's column of A is one 128-bit
//      shared load, 128-bit epilogue;
//   8  warp tiling ("Warp Tiling: A Third Level of Tiling"): a 128 x 64 C
//      tile per CTA of 128 threads, BK = 16; each warp owns a 64 x 32 tile
//      made of 2 x 2 sub-tiles of 32 x 16, in which the 32 lanes form an
//      8 x 4 grid of 4 x 4 patches (WMITER = WNITER = 2, TM = TN = 4).
//
// They are plain SIMT kernels with one CTA per C tile, two barriers per
// k-slice and no copy pipeline: sgemm() never calls them. Unlike the pages'
// listings they take leading dimensions and any shape: loads outside the
// matrices read zero, stores outside are skipped, and the 128-bit forms are
// used only where every pointer is 16-byte aligned and every leading
// dimension a multiple of 4 (otherwise the same kernel runs with 4-byte
// accesses). beta == 0 never reads C; alpha == 0 or K == 0 never reads A or B.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>

#include "../../include/sgemm_gb300.h"

#define SGEMM_API extern "C" __attribute__((visibility("default")))

namespace sgemm_gb300 {

int library_device_sms(int dev, int* sms);
void note_last_config(const char* text);

namespace ladder {

__device__ __forceinline__ float epilogue_value(float alpha, float acc, float beta, const float* c) {
  return beta == 0.f ? alpha * acc : alpha * acc + beta * *c;
}

// ---- kernel 3: shared-memory tiling ----------------------------------------
constexpr int kT3 = 32;

__global__ void __launch_bounds__(kT3 * kT3) smem_tiling_kernel(int M, int N, int K, float alpha,
                                                                const float* __restrict__ A, int lda,
                                                                const float* __restrict__ B, int ldb,
                                                                float beta, float* C, int ldc,
                                                                int tiles_n) {
  __shared__ float As[kT3][kT3];  // As[row of the C tile][k]
  __shared__ float Bs[kT3][kT3];  // Bs[k][column of the C tile]
  const int tm = blockIdx.x / tiles_n, tn = blockIdx.x % tiles_n;
  const int tx = threadIdx.x % kT3;  // column of C (fast index: coalesced loads)
  const int ty = threadIdx.x / kT3;  // row of C
  const int row = tm * kT3 + ty, col = tn * kT3 + tx;
  float acc = 0.f;
  for (int k0 = 0; k0 < K; k0 += kT3) {
    As[ty][tx] = (row < M && k0 + tx < K) ? A[(size_t)row * lda + k0 + tx] : 0.f;
    Bs[ty][tx] = (k0 + ty < K && col < N) ? B[(size_t)(k0 + ty) * ldb + col] : 0.f;
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kT3; ++k) acc = fmaf(As[ty][k], Bs[k][tx], acc);
    __syncthreads();  // the next slice overwrites what slower warps still read
  }
  if (row < M && col < N) {
    float* c = C + (size_t)row * ldc + col;
    *c = epilogue_value(alpha, acc, beta, c);
  }
}

// Four consecutive elements p[0..3] of a row whose valid length ends at
// `limit` (elements at index >= limit read zero). VEC: p is 16-byte aligned.
template <bool VEC>
__device__ __forceinline__ float4 load_row4(const float* p, int first, int limit, bool row_ok) {
  if (VEC && row_ok && first + 3 < limit) return *reinterpret_cast<const float4*>(p);
  float4 v;
  v.x = (row_ok && first + 0 < limit) ? p[0] : 0.f;
  v.y = (row_ok && first + 1 < limit) ? p[1] : 0.f;
  v.z = (row_ok && first + 2 < limit) ? p[2] : 0.f;
  v.w = (row_ok && first + 3 < limit) ? p[3] : 0.f;
  return v;
}

// C[row][col .. col+3] = alpha * acc + beta * C for the columns below N.
template <bool VEC>
__device__ __forceinline__ void store_row4(float* c, int row, int col, int M, int N, float alpha,
                                           const float (&acc)[4], float beta) {
  if (row >= M) return;
  if (VEC && col + 3 < N) {
    float4 v;
    if (beta == 0.f) {
      v = make_float4(alpha * acc[0], alpha * acc[1], alpha * acc[2], alpha * acc[3]);
    } else {
      const float4 o = *reinterpret_cast<const float4*>(c);
      v = make_float4(alpha * acc[0] + beta * o.x, alpha * acc[1] + beta * o.y,
                      alpha * acc[2] + beta * o.z, alpha * acc[3] + beta * o.w);
    }
    *reinterpret_cast<float4*>(c) = v;
    return;
  }
#pragma unroll
  for (int j = 0; j < 4; ++j)
    if (col + j < N) c[j] = epilogue_value(alpha, acc[j], beta, c + j);
}

// ---- kernel 7: vectorized 2-D block tiling ----------------------------------
constexpr int kBM7 = 128, kBN7 = 128, kBK7 = 8, kTM7 = 8, kTN7 = 8;
constexpr int kThreads7 = (kBM7 * kBN7) / (kTM7 * kTN7);  // 256
static_assert(kBM7 * kBK7 == 4 * kThreads7, "one float4 of A per thread and slice");
static_assert(kBK7 * kBN7 == 4 * kThreads7, "one float4 of B per thread and slice");

template <bool VEC>
__global__ void __launch_bounds__(kThreads7) vectorized_kernel(int M, int N, int K, float alpha,
                                                               const float* __restrict__ A, int lda,
                                                               const float* __restrict__ B, int ldb,
                                                               float beta, float* C, int ldc,
                                                               int tiles_n) {
  __shared__ __align__(16) float As[kBK7][kBM7];  // transposed: As[k][m]
  __shared__ __align__(16) float Bs[kBK7][kBN7];  // Bs[k][n]
  const int m0 = (blockIdx.x / tiles_n) * kBM7, n0 = (blockIdx.x % tiles_n) * kBN7;
  const int t = threadIdx.x;
  const int pr = t / (kBN7 / kTN7), pc = t % (kBN7 / kTN7);  // 8 x 8 patch of C
  const int a_m = t / (kBK7 / 4), a_k = (t % (kBK7 / 4)) * 4;  // A: row, first k of the float4
  const int b_k = t / (kBN7 / 4), b_n = (t % (kBN7 / 4)) * 4;  // B: k row, first column

  float acc[kTM7][kTN7];
#pragma unroll
  for (int i = 0; i < kTM7; ++i)
#pragma unroll
    for (int j = 0; j < kTN7; ++j) acc[i][j] = 0.f;

  for (int k0 = 0; k0 < K; k0 += kBK7) {
    const int ar = m0 + a_m, ak = k0 + a_k;
    const float4 va = load_row4<VEC>(A + (size_t)(ar < M ? ar : 0) * lda + ak, ak, K, ar < M);
    As[a_k + 0][a_m] = va.x;
    As[a_k + 1][a_m] = va.y;
    As[a_k + 2][a_m] = va.z;
    As[a_k + 3][a_m] = va.w;
    const int bk = k0 + b_k, bn = n0 + b_n;
    const float4 vb = load_row4<VEC>(B + (size_t)(bk < K ? bk : 0) * ldb + bn, bn, N, bk < K);
    *reinterpret_cast<float4*>(&Bs[b_k][b_n]) = vb;
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kBK7; ++k) {
      float rm[kTM7], rn[kTN7];
      *reinterpret_cast<float4*>(&rm[0]) = *reinterpret_cast<const float4*>(&As[k][pr * kTM7]);
      *reinterpret_cast<float4*>(&rm[4]) = *reinterpret_cast<const float4*>(&As[k][pr * kTM7 + 4]);
      *reinterpret_cast<float4*>(&rn[0]) = *reinterpret_cast<const float4*>(&Bs[k][pc * kTN7]);
      *reinterpret_cast<float4*>(&rn[4]) = *reinterpret_cast<const float4*>(&Bs[k][pc * kTN7 + 4]);
#pragma unroll
      for (int i = 0; i < kTM7; ++i)
#pragma unroll
        for (int j = 0; j < kTN7; ++j) acc[i][j] = fmaf(rm[i], rn[j], acc[i][j]);
    }
    __syncthreads();
  }

#pragma unroll
  for (int i = 0; i < kTM7; ++i) {
    const int row = m0 + pr * kTM7 + i;
#pragma unroll
    for (int h = 0; h < kTN7; h += 4) {
      const int col = n0 + pc * kTN7 + h;
      const float part[4] = {acc[i][h], acc[i][h + 1], acc[i][h + 2], acc[i][h + 3]};
      store_row4<VEC>(C + (size_t)(row < M ? row : 0) * ldc + col, row, col, M, N, alpha, part,
                      beta);
    }
  }
}

// ---- kernel 8: warp tiling ---------------------------------------------------
constexpr int kBM8 = 128, kBN8 = 64, kBK8 = 16;
constexpr int kWM8 = 64, kWN8 = 32;           // warp tile
constexpr int kWMITER8 = 2, kWNITER8 = 2;     // sub-tiles per warp tile
constexpr int kTM8 = 4, kTN8 = 4;             // per-thread patch of a sub-tile
constexpr int kWSUBM8 = kWM8 / kWMITER8;      // 32
constexpr int kWSUBN8 = kWN8 / kWNITER8;      // 16
constexpr int kThreads8 = (kBM8 / kWM8) * (kBN8 / kWN8) * 32;  // 128
static_assert((kWSUBM8 / kTM8) * (kWSUBN8 / kTN8) == 32, "a sub-tile is covered by one warp");
static_assert((kBM8 * kBK8) % (4 * kThreads8) == 0 && (kBK8 * kBN8) % (4 * kThreads8) == 0,
              "whole float4 load passes");

template <bool VEC>
__global__ void __launch_bounds__(kThreads8) warptiling_kernel(int M, int N, int K, float alpha,
                                                               const float* __restrict__ A, int lda,
                                                               const float* __restrict__ B, int ldb,
                                                               float beta, float* C, int ldc,
                                                               int tiles_n) {
  __shared__ __align__(16) float As[kBK8][kBM8];  // transposed: As[k][m]
  __shared__ __align__(16) float Bs[kBK8][kBN8];
  const int m0 = (blockIdx.x / tiles_n) * kBM8, n0 = (blockIdx.x % tiles_n) * kBN8;
  const int t = threadIdx.x, warp = t / 32, lane = t % 32;
  const int wm = (warp / (kBN8 / kWN8)) * kWM8;  // warp tile origin inside the CTA tile
  const int wn = (warp % (kBN8 / kWN8)) * kWN8;
  const int lm = (lane / (kWSUBN8 / kTN8)) * kTM8;  // patch origin inside a sub-tile
  const int ln = (lane % (kWSUBN8 / kTN8)) * kTN8;

  float acc[kWMITER8 * kTM8][kWNITER8 * kTN8];
#pragma unroll
  for (int i = 0; i < kWMITER8 * kTM8; ++i)
#pragma unroll
    for (int j = 0; j < kWNITER8 * kTN8; ++j) acc[i][j] = 0.f;

  for (int k0 = 0; k0 < K; k0 += kBK8) {
#pragma unroll
    for (int pass = 0; pass < (kBM8 * kBK8) / (4 * kThreads8); ++pass) {
      const int idx = t + pass * kThreads8;
      const int r = idx / (kBK8 / 4), kq = (idx % (kBK8 / 4)) * 4;
      const int ar = m0 + r, ak = k0 + kq;
      const float4 v = load_row4<VEC>(A + (size_t)(ar < M ? ar : 0) * lda + ak, ak, K, ar < M);
      As[kq + 0][r] = v.x;
      As[kq + 1][r] = v.y;
      As[kq + 2][r] = v.z;
      As[kq + 3][r] = v.w;
    }
#pragma unroll
    for (int pass = 0; pass < (kBK8 * kBN8) / (4 * kThreads8); ++pass) {
      const int idx = t + pass * kThreads8;
      const int kr = idx / (kBN8 / 4), nq = (idx % (kBN8 / 4)) * 4;
      const int bk = k0 + kr, bn = n0 + nq;
      const float4 v = load_row4<VEC>(B + (size_t)(bk < K ? bk : 0) * ldb + bn, bn, N, bk < K);
      *reinterpret_cast<float4*>(&Bs[kr][nq]) = v;
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kBK8; ++k) {
      float rm[kWMITER8 * kTM8], rn[kWNITER8 * kTN8];
#pragma unroll
      for (int i = 0; i < kWMITER8; ++i)
        *reinterpret_cast<float4*>(&rm[i * kTM8]) =
            *reinterpret_cast<const float4*>(&As[k][wm + i * kWSUBM8 + lm]);
#pragma unroll
      for (int j = 0; j < kWNITER8; ++j)
        *reinterpret_cast<float4*>(&rn[j * kTN8]) =
            *reinterpret_cast<const float4*>(&Bs[k][wn + j * kWSUBN8 + ln]);
#pragma unroll
      for (int i = 0; i < kWMITER8 * kTM8; ++i)
#pragma unroll
        for (int j = 0; j < kWNITER8 * kTN8; ++j) acc[i][j] = fmaf(rm[i], rn[j], acc[i][j]);
    }
    __syncthreads();
  }

#pragma unroll
  for (int i = 0; i < kWMITER8; ++i)
#pragma unroll
    for (int r = 0; r < kTM8; ++r) {
      const int row = m0 + wm + i * kWSUBM8 + lm + r;
#pragma unroll
      for (int j = 0; j < kWNITER8; ++j) {
        const int col = n0 + wn + j * kWSUBN8 + ln;
        const float part[4] = {acc[i * kTM8 + r][j * kTN8 + 0], acc[i * kTM8 + r][j * kTN8 + 1],
                               acc[i * kTM8 + r][j * kTN8 + 2], acc[i * kTM8 + r][j * kTN8 + 3]};
        store_row4<VEC>(C + (size_t)(row < M ? row : 0) * ldc + col, row, col, M, N, alpha, part,
                        beta);
      }
    }
}

long long ceil_div_ll(long long a, long long b) { return (a + b - 1) / b; }

}  // namespace ladder
}  // namespace sgemm_gb300

using namespace sgemm_gb300;

SGEMM_API int sgemm_ladder(int kernel, int M, int N, int K, float alpha, const float* A, int lda,
                           const float* B, int ldb, float beta, float* C, int ldc, void* stream_) {
  if (kernel != 3 && kernel != 7 && kernel != 8) return SGEMM_ERR_INVALID_VALUE;
  if (M < 0 || N < 0 || K < 0) return SGEMM_ERR_INVALID_DIM;
  if (lda < (K > 1 ? K : 1) || ldb < (N > 1 ? N : 1) || ldc < (N > 1 ? N : 1))
    return SGEMM_ERR_INVALID_LD;
  if (M == 0 || N == 0) return SGEMM_OK;
  const bool reads_ab = (K > 0 && alpha != 0.f);
  if (C == nullptr || (reads_ab && (A == nullptr || B == nullptr))) return SGEMM_ERR_NULL_PTR;
  if ((reinterpret_cast<uintptr_t>(C) & 3u) ||
      (reads_ab && ((reinterpret_cast<uintptr_t>(A) & 3u) || (reinterpret_cast<uintptr_t>(B) & 3u))))
    return SGEMM_ERR_MISALIGNED;

  const int bm = kernel == 3 ? ladder::kT3 : (kernel == 7 ? ladder::kBM7 : ladder::kBM8);
  const int bn = kernel == 3 ? ladder::kT3 : (kernel == 7 ? ladder::kBN7 : ladder::kBN8);
  const long long tiles_m = ladder::ceil_div_ll(M, bm), tiles_n = ladder::ceil_div_ll(N, bn);
  const long long tiles = tiles_m * tiles_n;
  if (tiles > 0x7fffffffLL) return SGEMM_ERR_INVALID_DIM;  // one CTA per tile, 1-D grid

  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return SGEMM_ERR_LAUNCH;
  }
  int sms = 0;
  const int st = library_device_sms(dev, &sms);  // also rejects devices other than sm_103
  if (st != SGEMM_OK) return st;

  // alpha == 0 or K == 0: no k-slice runs, so A and B are never read
  const int k_run = reads_ab ? K : 0;
  const bool vec = ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) |
                     reinterpret_cast<uintptr_t>(C)) & 15u) == 0 &&
                   (lda % 4) == 0 && (ldb % 4) == 0 && (ldc % 4) == 0;
  const int grid = (int)tiles, tn = (int)tiles_n;
  if (kernel == 3) {
    ladder::smem_tiling_kernel<<<grid, ladder::kT3 * ladder::kT3, 0, stream>>>(
        M, N, k_run, alpha, A, lda, B, ldb, beta, C, ldc, tn);
  } else if (kernel == 7) {
    if (vec)
      ladder::vectorized_kernel<true><<<grid, ladder::kThreads7, 0, stream>>>(
          M, N, k_run, alpha, A, lda, B, ldb, beta, C, ldc, tn);
    else
      ladder::vectorized_kernel<false><<<grid, ladder::kThreads7, 0, stream>>>(
          M, N, k_run, alpha, A, lda, B, ldb, beta, C, ldc, tn);
  } else {
    if (vec)
      ladder::warptiling_kernel<true><<<grid, ladder::kThreads8, 0, stream>>>(
          M, N, k_run, alpha, A, lda, B, ldb, beta, C, ldc, tn);
    else
      ladder::warptiling_kernel<false><<<grid, ladder::kThreads8, 0, stream>>>(
          M, N, k_run, alpha, A, lda, B, ldb, beta, C, ldc, tn);
  }
  if (cudaGetLastError() != cudaSuccess) return SGEMM_ERR_LAUNCH;
  char text[96];
  snprintf(text, sizeof(text), "ladder_kernel%d %dx%d %s grid=%d", kernel, bm, bn,
           vec ? "vec128" : "scalar", grid);
  note_last_config(text);
  return SGEMM_OK;
}
