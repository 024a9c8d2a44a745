// tiny.cu -- the kernel for very small problems (M * N * K up to 2^25).
//
// There, a multiplication takes a few microseconds and its time is latency:
// the launch, the first round trip to memory, and, in the persistent kernel,
// the pipeline fill and the K-split fix-up. This kernel keeps only what such
// a problem needs: one CTA per 32 x 32 tile of C (no persistent loop, no
// split), 256 threads with 2 x 2 outputs each, and each k-chunk of up to 256
// staged in shared memory by one round of loads (all of K for K <= 256), A
// transposed on its way in so that a thread's two rows are one 64-bit load.
// Loads outside the matrices read zero, stores outside are skipped, and the
// 128-bit forms are used only where the rows allow them.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstdio>

#include "../../include/sgemm_gb300.h"

namespace sgemm_gb300 {
namespace tiny {

constexpr int kT = 32;        // C tile edge
constexpr int kKC = 256;      // k-chunk staged at once
constexpr int kThreads = 256;
constexpr int kAP = kT + 2;   // As[k][m] pitch: even (64-bit reads), not a multiple of 32
constexpr int kSmemBytes = (kKC * kAP + kKC * kT) * 4;  // 67,584 bytes

template <bool VEC>
__global__ void __launch_bounds__(kThreads) tiny_kernel(int M, int N, int K, float alpha,
                                                        const float* __restrict__ A, long long lda,
                                                        const float* __restrict__ B, long long ldb,
                                                        float beta, float* C, long long ldc,
                                                        int tiles_n) {
  extern __shared__ float smem[];
  float* As = smem;               // [kKC][kAP], As[k][m] = A[m0 + m][k0 + k]
  float* Bs = smem + kKC * kAP;   // [kKC][kT],  Bs[k][n] = B[k0 + k][n0 + n]
  const int m0 = (blockIdx.x / tiles_n) * kT, n0 = (blockIdx.x % tiles_n) * kT;
  const int t = threadIdx.x;
  const int tr = (t / 16) * 2, tc = (t % 16) * 2;  // this thread's 2 x 2 outputs
  float acc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
  // launched with programmatic dependent launch: wait for the kernel ahead of
  // this one on the stream before touching global memory, then let the next
  // one launch (it waits for this grid in turn)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  for (int k0 = 0; k0 < K; k0 += kKC) {
    const int kc = (K - k0) < kKC ? (K - k0) : kKC;
    // A: 32 rows x kc; thread -> (row, 4 consecutive k), passes over k
    for (int e = t; e < kT * (kKC / 4); e += kThreads) {
      const int m = e / (kKC / 4), kq = (e % (kKC / 4)) * 4;
      if (kq >= kc) continue;
      const int gm = m0 + m, gk = k0 + kq;
      float v[4] = {0.f, 0.f, 0.f, 0.f};
      if (gm < M) {
        const float* src = A + (long long)gm * lda + gk;
        if (VEC && gk + 3 < K) {
          const float4 q = *reinterpret_cast<const float4*>(src);
          v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j) v[j] = (gk + j < K) ? src[j] : 0.f;
        }
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) As[(kq + j) * kAP + m] = v[j];
    }
    // B: kc rows x 32; thread -> (k, 4 consecutive n)
    for (int e = t; e < kKC * (kT / 4); e += kThreads) {
      const int k = e / (kT / 4), nq = (e % (kT / 4)) * 4;
      if (k >= kc) break;
      const int gk = k0 + k, gn = n0 + nq;
      float4 q = make_float4(0.f, 0.f, 0.f, 0.f);
      const float* src = B + (long long)gk * ldb + gn;
      if (VEC && gn + 3 < N) {
        q = *reinterpret_cast<const float4*>(src);
      } else {
        if (gn + 0 < N) q.x = src[0];
        if (gn + 1 < N) q.y = src[1];
        if (gn + 2 < N) q.z = src[2];
        if (gn + 3 < N) q.w = src[3];
      }
      *reinterpret_cast<float4*>(&Bs[k * kT + nq]) = q;
    }
    __syncthreads();
#pragma unroll 8
    for (int k = 0; k < kc; ++k) {
      const float2 a = *reinterpret_cast<const float2*>(&As[k * kAP + tr]);
      const float2 b = *reinterpret_cast<const float2*>(&Bs[k * kT + tc]);
      acc[0][0] = fmaf(a.x, b.x, acc[0][0]);
      acc[0][1] = fmaf(a.x, b.y, acc[0][1]);
      acc[1][0] = fmaf(a.y, b.x, acc[1][0]);
      acc[1][1] = fmaf(a.y, b.y, acc[1][1]);
    }
    __syncthreads();  // the next chunk overwrites what slower warps still read
  }

#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int row = m0 + tr + i;
    if (row >= M) continue;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int col = n0 + tc + j;
      if (col >= N) continue;
      float* c = C + (long long)row * ldc + col;
      *c = beta == 0.f ? alpha * acc[i][j] : fmaf(alpha, acc[i][j], beta * *c);
    }
  }
}

// devices whose kernels have their shared-memory attribute set (setting it
// twice, from two threads, is harmless)
std::atomic<bool> g_attr_set[64];

}  // namespace tiny

// Whether the tiny kernel takes this problem (row-major, one matrix).
bool tiny_wanted(int M, int N, int K) {
  return (long long)M * N * K <= (1LL << 25);
}

// C = alpha * A * B + beta * C for a tiny problem (arguments checked, K > 0,
// alpha != 0). Returns a cudaError_t.
cudaError_t tiny_launch(int dev, int M, int N, int K, float alpha, const float* A, long long lda,
                        const float* B, long long ldb, float beta, float* C, long long ldc,
                        cudaStream_t stream, char* text, int text_len) {
  using namespace tiny;
  if (dev < 0 || dev >= 64 || !g_attr_set[dev].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(tiny_kernel<true>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(tiny_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kSmemBytes);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) g_attr_set[dev].store(true, std::memory_order_release);
  }
  const int tiles_m = (M + kT - 1) / kT, tiles_n = (N + kT - 1) / kT;
  const int grid = tiles_m * tiles_n;  // at most 2^25 / 32 tiles
  const bool vec = ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B)) & 15u) == 0 &&
                   (lda % 4) == 0 && (ldb % 4) == 0;
  // programmatic dependent launch: the launch overlaps the end of the kernel
  // ahead (the kernel waits for it before any global access)
  cudaLaunchConfig_t lc = {};
  cudaLaunchAttribute la[1];
  la[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  la[0].val.programmaticStreamSerializationAllowed = 1;
  lc.gridDim = dim3((unsigned)grid);
  lc.blockDim = dim3(kThreads);
  lc.dynamicSmemBytes = kSmemBytes;
  lc.stream = stream;
  lc.attrs = la;
  lc.numAttrs = 1;
  const cudaError_t e =
      vec ? cudaLaunchKernelEx(&lc, tiny_kernel<true>, M, N, K, alpha, A, lda, B, ldb, beta, C,
                               ldc, tiles_n)
          : cudaLaunchKernelEx(&lc, tiny_kernel<false>, M, N, K, alpha, A, lda, B, ldb, beta, C,
                               ldc, tiles_n);
  snprintf(text, (size_t)text_len, "tiny_32x32_k%d %s grid=%d", kKC, vec ? "vec128" : "scalar",
           grid);
  return e;
}

}  // namespace sgemm_gb300
