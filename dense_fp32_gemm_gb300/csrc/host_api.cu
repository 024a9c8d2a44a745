// host_api.cu -- sgemm_host(): C = alpha * A * B + beta * C on HOST matrices,
// with the host <-> device copies overlapped with the GEMM.
//
// K is cut into chunks. While the GPU multiplies chunk i (A[:, Ki] * B[Ki, :],
// accumulated into a device copy of C), the copy engine brings in chunk i+1.
// The chunks grow geometrically: the first is narrow so the first multiply
// starts early, and each next one is as many times wider as multiplying a
// column of K takes longer than copying it, so every copy hides under the
// previous multiply. The incoming C needed for beta * C travels on the same
// copy stream after the operand chunks, one row panel at a time. The last
// chunk is multiplied in row panels: as soon as a panel is final (beta * C
// added) it is copied back on a second copy stream while the next panel
// computes. The caller's stream waits for the last copy, so
// synchronising the caller's stream means C (host) is final. Splitting K only
// reorders the sum over k; results stay within the FP32 tolerance and integer
// inputs stay exact.
#include <cuda_runtime.h>

#include <cstdint>
#include <map>
#include <mutex>
#include <utility>

#include "../../include/sgemm_gb300.h"

#define SGEMM_API extern "C" __attribute__((visibility("default")))

namespace sgemm_gb300 {

int library_ffma(int M, int N, int K, float alpha, const float* A, int lda, const float* B,
                 int ldb, float beta, float* C, int ldc, cudaStream_t stream);
int library_device_sms(int dev, int* sms);

namespace {

constexpr int kMaxChunks = 9;
constexpr int kMaxPanels = 8;

// The copy/compute pipeline: K chunk widths and the row panels of the last
// chunk (sgemm_host_set_pipeline). Widths are rounded up to multiples of 32.
struct Pipeline {
  int first = 128;   // first chunk
  int mid = 0;       // 0: geometric growth; > 0: equal chunks of about `mid`
                     // between the first and the last
  int last = 0;      // last chunk; 0: what the growth leaves (geometric), or as
                     // wide as the middle chunks (equal)
  int panels = 4;    // row panels of the last chunk (only when M >= 512 * panels)
};
Pipeline g_pipe;

// Growth of the geometric chunk widths for an M x N result: multiplying one
// column of K costs 2 M N flops (about 68 TFLOP/s), copying it 4 (M + N)
// bytes (about 200 GB/s from pinned memory), so a chunk may be
// M N / (M + N) / 680 times wider than the previous one and still copy within
// the previous multiply; with a 10 % margin, clamped to [1.5, 4].
double chunk_growth(int M, int N) {
  const double g = (double)M * N / ((double)M + N) / 755.0;
  return g < 1.5 ? 1.5 : (g > 4.0 ? 4.0 : g);
}

// Chunk boundaries 0 = kb[0] < ... < kb[n] = K for an M x N x K problem;
// returns the chunk count n (at most kMaxChunks).
int chunk_bounds(int M, int N, int K, const Pipeline& pp, int* kb) {
  auto r32 = [](long long x) { return (int)((x + 31) / 32 * 32); };
  if (pp.mid == 0) {
    const int last = pp.last > 0 ? r32(pp.last) : 0;
    const int k_hi = (last > 0 && K > last) ? K - last : K;
    const int budget = kMaxChunks - (k_hi < K ? 1 : 0);
    const double g = chunk_growth(M, N);
    int n = 0, k = 0, w = r32(pp.first > 0 ? pp.first : 128);
    kb[0] = 0;
    while (k < k_hi) {
      int wc = w < k_hi - k ? w : k_hi - k;
      const int next = r32((long long)(wc * g));
      // a remainder narrower than half the next chunk joins this one, and so
      // does everything once the chunk budget is used up
      if (k_hi - (k + wc) < next / 2 || n + 1 >= budget) wc = k_hi - k;
      k += wc;
      kb[++n] = k;
      w = next;
    }
    if (k_hi < K) kb[++n] = K;
    return n;
  }
  const int first = r32(pp.first), last = pp.last > 0 ? r32(pp.last) : 0;
  int n = 0;
  kb[n++] = 0;
  int k_lo = 0, k_hi = K;
  if (first > 0 && K >= 2 * first + last) {
    kb[n++] = first;
    k_lo = first;
  }
  if (last > 0 && k_hi - last > k_lo) k_hi -= last;
  int parts = (k_hi - k_lo) / (pp.mid > 32 ? pp.mid : 32);
  const int room = kMaxChunks - (n - 1) - (k_hi < K ? 1 : 0);
  parts = parts < 1 ? 1 : (parts > room ? room : parts);
  const int step = r32((k_hi - k_lo + parts - 1) / parts);
  for (int k = k_lo + step; k < k_hi; k += step) kb[n++] = k;
  if (k_hi < K) kb[n++] = k_hi;
  kb[n] = K;
  return n;
}

// Row panels of the last chunk for `panels` panels of M rows: bounds
// 0 = r[0] < ... < r[n] = M, returns n. The panel copied back last is the
// only copy nothing hides, so it is short: about M / (4 panels) rows (measured
// on GB300 at 4096^3: 2.34 ms against 2.39 for four equal panels); the others
// share the rest equally (all multiples of 128 rows but the end).
int panel_bounds(int M, int panels, int* r) {
  auto r128 = [](long long x) { return (int)((x + 127) / 128 * 128); };
  int n = 0;
  r[0] = 0;
  if (panels <= 1) {
    r[++n] = M;
    return n;
  }
  int last = r128((long long)M / (4 * panels));
  if (last >= M / 2) last = 0;
  const int body = M - last, nb = last > 0 ? panels - 1 : panels;
  const int rows = r128((body + nb - 1) / nb);
  for (int r0 = 0; r0 < body; r0 += rows) r[++n] = r0 + rows < body ? r0 + rows : body;
  if (last > 0) r[++n] = M;
  return n;
}

struct HostCtx {
  bool ready = false;
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t start = nullptr, chunk[kMaxChunks] = {}, panel[kMaxPanels] = {}, c_in = nullptr,
              done = nullptr, out = nullptr, c_in_panel[kMaxPanels] = {};
  float *dA = nullptr, *dB = nullptr, *dC = nullptr, *dC0 = nullptr;
  size_t capA = 0, capB = 0, capC = 0, capC0 = 0;  // floats
};

std::mutex g_host_mutex;
std::map<std::pair<int, cudaStream_t>, HostCtx> g_host;

int grow(float** buf, size_t* cap, size_t need) {
  if (*cap >= need) return SGEMM_OK;
  if (*buf != nullptr) {
    cudaFree(*buf);  // synchronises the device: no queued work still uses it
    *buf = nullptr;
    *cap = 0;
  }
  if (cudaMalloc(buf, need * sizeof(float)) != cudaSuccess) {
    cudaGetLastError();
    *buf = nullptr;
    return SGEMM_ERR_ALLOC;
  }
  *cap = need;
  return SGEMM_OK;
}

int ctx_for(int dev, cudaStream_t user, HostCtx** out) {
  HostCtx& c = g_host[{dev, user}];
  if (!c.ready) {
    if (cudaStreamCreateWithFlags(&c.h2d, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&c.d2h, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&c.start, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&c.c_in, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&c.done, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&c.out, cudaEventDisableTiming) != cudaSuccess) {
      cudaGetLastError();
      return SGEMM_ERR_LAUNCH;
    }
    for (int i = 0; i < kMaxChunks; ++i)
      if (cudaEventCreateWithFlags(&c.chunk[i], cudaEventDisableTiming) != cudaSuccess) {
        cudaGetLastError();
        return SGEMM_ERR_LAUNCH;
      }
    for (int i = 0; i < kMaxPanels; ++i)
      if (cudaEventCreateWithFlags(&c.panel[i], cudaEventDisableTiming) != cudaSuccess ||
          cudaEventCreateWithFlags(&c.c_in_panel[i], cudaEventDisableTiming) != cudaSuccess) {
        cudaGetLastError();
        return SGEMM_ERR_LAUNCH;
      }
    c.ready = true;
  }
  *out = &c;
  return SGEMM_OK;
}

// C = C + beta * C0 (both M x N, dense). Launched with programmatic
// dependent launch after the panel's GEMM: it waits for that GEMM before
// touching memory, and lets the next panel's GEMM launch.
__global__ void add_scaled_kernel(long long n, float beta, float* __restrict__ C,
                                  const float* __restrict__ C0) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < n;
       e += (long long)gridDim.x * blockDim.x)
    C[e] = fmaf(beta, C0[e], C[e]);
}

// C = beta * C (beta == 0 writes zeros without reading C).
__global__ void host_scale_kernel(long long n, float beta, float* C) {
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < n;
       e += (long long)gridDim.x * blockDim.x)
    C[e] = beta == 0.f ? 0.f : beta * C[e];
}

}  // namespace

// Frees every buffer, stream and event of sgemm_host (called by
// sgemm_shutdown after the device work is done).
void host_api_release() {
  std::lock_guard<std::mutex> lock(g_host_mutex);
  for (auto& kv : g_host) {
    HostCtx& c = kv.second;
    cudaSetDevice(kv.first.first);
    cudaDeviceSynchronize();
    cudaFree(c.dA);
    cudaFree(c.dB);
    cudaFree(c.dC);
    cudaFree(c.dC0);
    if (c.ready) {
      cudaStreamDestroy(c.h2d);
      cudaStreamDestroy(c.d2h);
      cudaEventDestroy(c.start);
      cudaEventDestroy(c.c_in);
      cudaEventDestroy(c.done);
      cudaEventDestroy(c.out);
      for (int i = 0; i < kMaxChunks; ++i) cudaEventDestroy(c.chunk[i]);
      for (int i = 0; i < kMaxPanels; ++i) {
        cudaEventDestroy(c.panel[i]);
        cudaEventDestroy(c.c_in_panel[i]);
      }
    }
  }
  g_host.clear();
  cudaGetLastError();
}

}  // namespace sgemm_gb300

using namespace sgemm_gb300;

SGEMM_API int sgemm_host(int M, int N, int K, float alpha, const float* A, int lda,
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

  cudaStream_t user = static_cast<cudaStream_t>(stream_);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return SGEMM_ERR_LAUNCH;
  }
  int sms = 0;
  int st = library_device_sms(dev, &sms);
  if (st != SGEMM_OK) return st;

  std::lock_guard<std::mutex> lock(g_host_mutex);
  HostCtx* c = nullptr;
  st = ctx_for(dev, user, &c);
  if (st != SGEMM_OK) return st;
  const size_t mn = (size_t)M * N;
  if ((st = grow(&c->dC, &c->capC, mn)) != SGEMM_OK) return st;
  const size_t pitch_c = (size_t)ldc * 4, row_c = (size_t)N * 4;
  auto fail = [] {
    cudaGetLastError();
    return SGEMM_ERR_LAUNCH;
  };
  int blocks = (int)((mn + 255) / 256);
  if (blocks > sms * 8) blocks = sms * 8;

  // earlier work on the caller's stream (which may still read these buffers)
  // comes first
  if (cudaEventRecord(c->start, user) != cudaSuccess ||
      cudaStreamWaitEvent(c->h2d, c->start, 0) != cudaSuccess)
    return fail();

  if (!reads_ab) {
    // C = beta * C
    if (beta != 0.f &&
        cudaMemcpy2DAsync(c->dC, row_c, C, pitch_c, row_c, M, cudaMemcpyHostToDevice, c->h2d) !=
            cudaSuccess)
      return fail();
    if (cudaEventRecord(c->c_in, c->h2d) != cudaSuccess ||
        cudaStreamWaitEvent(user, c->c_in, 0) != cudaSuccess)
      return fail();
    host_scale_kernel<<<blocks, 256, 0, user>>>((long long)mn, beta, c->dC);
  } else {
    if ((st = grow(&c->dA, &c->capA, (size_t)M * K)) != SGEMM_OK ||
        (st = grow(&c->dB, &c->capB, (size_t)K * N)) != SGEMM_OK)
      return st;
    if (beta != 0.f && (st = grow(&c->dC0, &c->capC0, mn)) != SGEMM_OK) return st;
    // K chunk boundaries: a narrow first chunk, equal middle chunks, and a
    // last chunk that is computed (and copied back) in row panels
    int kb[kMaxChunks + 2];
    const int nk = chunk_bounds(M, N, K, g_pipe, kb);
    for (int i = 0; i < nk; ++i) {
      const int k0 = kb[i], k1 = kb[i + 1];
      if (cudaMemcpy2DAsync(c->dA + k0, (size_t)K * 4, A + k0, (size_t)lda * 4,
                            (size_t)(k1 - k0) * 4, M, cudaMemcpyHostToDevice, c->h2d) != cudaSuccess ||
          cudaMemcpy2DAsync(c->dB + (size_t)k0 * N, row_c, B + (size_t)k0 * ldb, (size_t)ldb * 4,
                            row_c, k1 - k0, cudaMemcpyHostToDevice, c->h2d) != cudaSuccess ||
          cudaEventRecord(c->chunk[i], c->h2d) != cudaSuccess)
        return fail();
    }
    // row panels of the last chunk: [r_0, r_1), [r_1, r_2), ...
    const int panels = M >= 512 * g_pipe.panels ? g_pipe.panels : (M >= 1024 ? M / 512 : 1);
    int pr[kMaxPanels + 1];
    const int np = panel_bounds(M, panels, pr);
    // the incoming C, one row panel at a time: panel p's add waits only for
    // its own rows
    if (beta != 0.f) {
      for (int pi = 0; pi < np; ++pi) {
        const int r0 = pr[pi], r1 = pr[pi + 1];
        if (cudaMemcpy2DAsync(c->dC0 + (size_t)r0 * N, row_c, C + (size_t)r0 * ldc, pitch_c, row_c,
                              r1 - r0, cudaMemcpyHostToDevice, c->h2d) != cudaSuccess ||
            cudaEventRecord(c->c_in_panel[pi], c->h2d) != cudaSuccess)
          return fail();
      }
    }
    for (int i = 0; i + 1 < nk; ++i) {
      if (cudaStreamWaitEvent(user, c->chunk[i], 0) != cudaSuccess) return fail();
      st = library_ffma(M, N, kb[i + 1] - kb[i], alpha, c->dA + kb[i], K, c->dB + (size_t)kb[i] * N,
                        N, i == 0 ? 0.f : 1.f, c->dC, N, user);
      if (st != SGEMM_OK) return st;
    }
    // last chunk in row panels, each copied back as soon as it is final
    const int k0 = kb[nk - 1], kl = K - k0;
    if (cudaStreamWaitEvent(user, c->chunk[nk - 1], 0) != cudaSuccess) return fail();
    for (int pi = 0; pi < np; ++pi) {
      const int r0 = pr[pi], r1 = pr[pi + 1];
      float* dCp = c->dC + (size_t)r0 * N;
      st = library_ffma(r1 - r0, N, kl, alpha, c->dA + (size_t)r0 * K + k0, K,
                        c->dB + (size_t)k0 * N, N, nk == 1 ? 0.f : 1.f, dCp, N, user);
      if (st != SGEMM_OK) return st;
      const size_t pn = (size_t)(r1 - r0) * N;
      if (beta != 0.f) {
        if (cudaStreamWaitEvent(user, c->c_in_panel[pi], 0) != cudaSuccess) return fail();
        int pb = (int)((pn + 255) / 256);
        if (pb > sms * 8) pb = sms * 8;
        cudaLaunchConfig_t lc = {};
        cudaLaunchAttribute la[1];
        la[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        la[0].val.programmaticStreamSerializationAllowed = 1;
        lc.gridDim = dim3((unsigned)pb);
        lc.blockDim = dim3(256);
        lc.stream = user;
        lc.attrs = la;
        lc.numAttrs = 1;
        if (cudaLaunchKernelEx(&lc, add_scaled_kernel, (long long)pn, beta, dCp,
                               (const float*)(c->dC0 + (size_t)r0 * N)) != cudaSuccess)
          return fail();
      }
      if (cudaEventRecord(c->panel[pi], user) != cudaSuccess ||
          cudaStreamWaitEvent(c->d2h, c->panel[pi], 0) != cudaSuccess ||
          cudaMemcpy2DAsync(C + (size_t)r0 * ldc, pitch_c, dCp, row_c, row_c, r1 - r0,
                            cudaMemcpyDeviceToHost, c->d2h) != cudaSuccess)
        return fail();
    }
    if (cudaEventRecord(c->out, c->d2h) != cudaSuccess ||
        cudaStreamWaitEvent(user, c->out, 0) != cudaSuccess)
      return fail();
    return SGEMM_OK;
  }
  // copy the result back, then let the caller's stream wait for the copy
  if (cudaEventRecord(c->done, user) != cudaSuccess ||
      cudaStreamWaitEvent(c->d2h, c->done, 0) != cudaSuccess ||
      cudaMemcpy2DAsync(C, pitch_c, c->dC, row_c, row_c, M, cudaMemcpyDeviceToHost, c->d2h) !=
          cudaSuccess ||
      cudaEventRecord(c->out, c->d2h) != cudaSuccess ||
      cudaStreamWaitEvent(user, c->out, 0) != cudaSuccess)
    return fail();
  return SGEMM_OK;
}

SGEMM_API int sgemm_host_set_pipeline(int first, int mid, int last, int panels) {
  if (first < 0 || mid < 0 || last < 0 || panels < 0 || panels > kMaxPanels)
    return SGEMM_ERR_INVALID_VALUE;
  std::lock_guard<std::mutex> lock(g_host_mutex);
  const Pipeline defaults;
  g_pipe.first = first;
  g_pipe.mid = mid;
  g_pipe.last = last;
  g_pipe.panels = panels > 0 ? panels : defaults.panels;
  if (mid == 0 && first == 0) g_pipe.first = defaults.first;
  return SGEMM_OK;
}
