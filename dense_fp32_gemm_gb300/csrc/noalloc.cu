// noalloc.cu -- sgemm_noalloc(): the same GEMM as sgemm(), for callers that
// must not allocate device memory.
//
// sgemm() allocates (once per device and stream) the scratch its kernel needs:
// a status word, one flag per persistent CTA, and the partial tiles of the
// K-split schedule. Some callers cannot let a library call cudaMalloc: code
// that runs while a stream is being captured into a graph (allocation is not
// allowed there), code inside an application whose memory pool owns every free
// byte of the device and forbids hidden allocations, and latency-critical
// loops that cannot absorb an allocation or its implicit synchronisation.
// For them, this file keeps that scratch in one fixed, file-scope device
// array. Every GPU that loads the library holds the array until the process
// exits; nothing is allocated per call.
//
// Limits and sharing:
//   * the array is kNoAllocScratchBytes (24 MiB): a 256-byte status word,
//     flags for up to kNoAllocMaxFlags CTAs, and 24 MiB - 64 KiB of partial
//     tiles. On a 152-SM GB300 every problem fits with the built-in tile
//     configurations (the largest need is about 20 MB); a call whose
//     schedule needs more returns SGEMM_ERR_NOALLOC_CAPACITY and launches
//     nothing;
//   * all calls share the one array and it keeps the last call's contents.
//     The flags are matched against a per-device call counter, so stale flags
//     are never mistaken for fresh ones (they are cleared whenever the counter
//     wraps, and by a poll that reports a timeout); partial tiles are always
//     written before they are read. Calls that overlap on the GPU (two
//     streams, or two host threads) race on the array;
//   * the first call on a device performs its set-up: it looks up the
//     array's device address (cudaGetSymbolAddress, with that device current)
//     and sets the kernels' shared-memory attributes. Make that first call
//     before any stream capture;
//   * every wait inside the kernel is bounded by the library's wait limit
//     (sgemm_set_wait_timeout_ns); a kernel that gives up records its code in
//     the array's status word, which stays set until sgemm_noalloc_poll_status
//     reads and clears it (that poll also clears the flags, which an aborted
//     call can leave published).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/sgemm_gb300.h"
#include "configs.hpp"
#include "dispatch.hpp"
#include "ffma_sgemm.cuh"
#include "schedule.hpp"
#include "tile_config.hpp"

#define SGEMM_API extern "C" __attribute__((visibility("default")))

namespace sgemm_gb300 {

// Provided by api.cu.
long long library_wait_timeout_ns();
bool library_staged_a_wanted(bool built, int occ, int occ_staged, const Schedule& s);

// The kernel for very small problems (tiny.cu); it needs no scratch.
bool tiny_wanted(int M, int N, int K);
cudaError_t tiny_launch(int dev, int M, int N, int K, float alpha, const float* A, long long lda,
                        const float* B, long long ldb, float beta, float* C, long long ldc,
                        cudaStream_t stream, char* text, int text_len);

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(24) << 20;
constexpr size_t kNoAllocHeaderBytes = size_t(64) << 10;  // status word + flags
constexpr size_t kNoAllocStatusBytes = 256;
constexpr size_t kNoAllocMaxFlags = (kNoAllocHeaderBytes - kNoAllocStatusBytes) / 4;
constexpr int kNoAllocMaxDevices = 64;

// The scratch itself. Host code must not use this name as an address: it only
// stands for the symbol; the device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

#define SGEMM_GB300_NOALLOC_PTR(NAME, ...) &kEntry##NAME,
const ConfigEntry* const kNoAllocConfigs[] = {SGEMM_GB300_CONFIGS(SGEMM_GB300_NOALLOC_PTR)};
#undef SGEMM_GB300_NOALLOC_PTR
constexpr int kNoAllocNumConfigs = sizeof(kNoAllocConfigs) / sizeof(kNoAllocConfigs[0]);

struct NoAllocDevice {
  bool ready;
  int sms;
  int occupancy[kNoAllocNumConfigs];
  int occupancy_staged[kNoAllocNumConfigs];  // staged-A variant (0: not built)
  unsigned char* base;  // device address of g_noalloc_scratch on this device
  uint32_t epoch;
};

std::mutex g_na_mutex;
NoAllocDevice g_na_devices[kNoAllocMaxDevices];  // fixed storage: no heap use

// The automatic tile configuration and schedule policy are those of sgemm()
// (dispatch.hpp), so both entry points run the same kernel and schedule.

// Once per device, with that device current: symbol address, kernel
// attributes, occupancy. Called with g_na_mutex held.
int noalloc_setup(int dev, NoAllocDevice** out) {
  if (dev < 0 || dev >= kNoAllocMaxDevices) return SGEMM_ERR_UNSUPPORTED_DEVICE;
  NoAllocDevice& d = g_na_devices[dev];
  if (!d.ready) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return SGEMM_ERR_LAUNCH;
    }
    if (!(major == 10 && minor == 3)) return SGEMM_ERR_UNSUPPORTED_DEVICE;
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
      cudaGetLastError();
      return SGEMM_ERR_LAUNCH;
    }
    for (int c = 0; c < kNoAllocNumConfigs; ++c) {
      if (kNoAllocConfigs[c]->set_attributes() != cudaSuccess) {
        cudaGetLastError();
        return SGEMM_ERR_LAUNCH;
      }
      int blocks = 0;
      if (kNoAllocConfigs[c]->occupancy(&blocks) != cudaSuccess) {
        cudaGetLastError();
        return SGEMM_ERR_LAUNCH;
      }
      d.occupancy[c] = blocks;
      blocks = 0;
      if (kNoAllocConfigs[c]->staged &&
          kNoAllocConfigs[c]->occupancy_staged(&blocks) != cudaSuccess) {
        cudaGetLastError();
        return SGEMM_ERR_LAUNCH;
      }
      d.occupancy_staged[c] = blocks;
    }
    d.base = static_cast<unsigned char*>(ptr);
    d.epoch = 0;
    d.ready = true;
  }
  *out = &d;
  return SGEMM_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 noalloc_encoder() {
  // looked up once; the initialisation of a function-local static is thread-safe
  static const PFN_cuTensorMapEncodeTiled_v12000 enc = [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    cudaGetLastError();
    return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
  }();
  return enc;
}

__global__ void noalloc_scale_c_kernel(int M, int N, float beta, float* C, long long ldc) {
  const long long total = (long long)M * N;
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
       e += (long long)gridDim.x * blockDim.x) {
    const long long i = e / N, j = e % N;
    float* c = C + i * ldc + j;
    *c = beta == 0.f ? 0.f : beta * *c;
  }
}

}  // namespace
}  // namespace sgemm_gb300

using namespace sgemm_gb300;

SGEMM_API int sgemm_noalloc(int M, int N, int K, float alpha, const float* A, int lda,
                            const float* B, int ldb, float beta, float* C, int ldc,
                            void* stream_) {
  // argument checks: identical to sgemm(), nothing launched on error
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
  std::lock_guard<std::mutex> lock(g_na_mutex);
  NoAllocDevice* d = nullptr;
  int st = noalloc_setup(dev, &d);
  if (st != SGEMM_OK) return st;

  if (!reads_ab) {
    const long long total = (long long)M * N;
    int blocks = (int)((total + 255) / 256);
    if (blocks > d->sms * 8) blocks = d->sms * 8;
    noalloc_scale_c_kernel<<<blocks, 256, 0, stream>>>(M, N, beta, C, ldc);
    return cudaGetLastError() == cudaSuccess ? SGEMM_OK : SGEMM_ERR_LAUNCH;
  }

  // very small problems: the same tiny kernel as sgemm(), so both give the
  // same bits
  if (tiny_wanted(M, N, K)) {
    char text[96];
    return tiny_launch(dev, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream, text,
                       (int)sizeof(text)) == cudaSuccess
               ? SGEMM_OK
               : SGEMM_ERR_LAUNCH;
  }

  const int id = choose_config(M, N, K);
  const ConfigEntry& cfg = *kNoAllocConfigs[id];
  const TileShape& S = cfg.shape;
  // the schedule numbers tiles with 32-bit integers (the same limit as sgemm())
  const int tiles_m = ceil_div_nn(M, S.BM), tiles_n = ceil_div_nn(N, S.BN);
  if ((long long)tiles_m * tiles_n > 0x7fffffffLL) return SGEMM_ERR_INVALID_DIM;

  bool tma = ((reinterpret_cast<uintptr_t>(B) & 15u) == 0) && ((ldb & 3) == 0);
  CUtensorMap map_a, map_b;
  std::memset(&map_a, 0, sizeof(map_a));
  std::memset(&map_b, 0, sizeof(map_b));
  PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
  if (tma) {
    enc = noalloc_encoder();
    tma = false;
    if (enc != nullptr) {
      // one matrix: a 3-D map with a batch extent of 1
      cuuint64_t dims[3] = {(cuuint64_t)N, (cuuint64_t)K, 1};
      cuuint64_t strides[2] = {(cuuint64_t)ldb * 4,
                               (cuuint64_t)(((long long)ldb * (K > 0 ? K : 1) * 4 + 15) / 16 * 16)};
      cuuint32_t box[3] = {(cuuint32_t)S.BN, (cuuint32_t)S.BK, 1};
      cuuint32_t estr[3] = {1, 1, 1};
      tma = enc(&map_b, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(B), dims, strides,
                box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    }
  }

  const int occ = d->occupancy[id];
  if (occ < 1) return SGEMM_ERR_LAUNCH;
  const Schedule sched = make_schedule(tiles_m, tiles_n, ceil_div_nn(K, S.BK), d->sms * occ,
                                       choose_policy(M, N, K));
  // row-major A through the staging ring, under the same rule as sgemm() (the
  // same kernel variant, so the same bits): a K x M box of 32 x BM, 128-byte
  // swizzled
  int al = kARow;
  if (tma && enc != nullptr &&
      library_staged_a_wanted(cfg.staged, occ, d->occupancy_staged[id], sched) &&
      ((reinterpret_cast<uintptr_t>(A) & 15u) == 0) && ((lda & 3) == 0)) {
    cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)M, 1};
    cuuint64_t strides[2] = {(cuuint64_t)lda * 4,
                             (cuuint64_t)(((long long)lda * (M > 0 ? M : 1) * 4 + 15) / 16 * 16)};
    cuuint32_t box[3] = {(cuuint32_t)S.BK, (cuuint32_t)S.BM, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    if (enc(&map_a, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(A), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS)
      al = kARowStg;
  }
  const bool split = sched.dp_tiles < sched.tiles;
  const size_t partial_bytes = split ? (size_t)sched.grid * S.BM * S.BN * 4 : 0;
  if ((size_t)sched.grid > kNoAllocMaxFlags ||
      partial_bytes > kNoAllocScratchBytes - kNoAllocHeaderBytes)
    return SGEMM_ERR_NOALLOC_CAPACITY;

  int* status = reinterpret_cast<int*>(d->base);
  uint32_t* flags = reinterpret_cast<uint32_t*>(d->base + kNoAllocStatusBytes);
  float* partials = reinterpret_cast<float*>(d->base + kNoAllocHeaderBytes);
  // the flags are cleared on a wrap of the call counter (a flag is fresh when
  // it equals this call's number); the status word keeps the first recorded
  // code until sgemm_noalloc_poll_status clears it
  if (++d->epoch == 0) {
    d->epoch = 1;
    if (cudaMemsetAsync(flags, 0, kNoAllocMaxFlags * 4, stream) != cudaSuccess)
      return SGEMM_ERR_LAUNCH;
  }

  KernelParams p;
  p.M = M;
  p.N = N;
  p.K = K;
  p.alpha = alpha;
  p.beta = beta;
  p.A = A;
  p.lda = lda;
  p.B = B;
  p.ldb = ldb;
  p.C = C;
  p.ldc = ldc;
  p.sA = 0;
  p.sB = 0;
  p.sC = 0;
  p.sched = sched;
  p.ws = partials;
  p.flags = flags;
  p.status = status;
  p.epoch = d->epoch;
  p.c_vec = ((reinterpret_cast<uintptr_t>(C) & 15u) == 0) && ((ldc & 3) == 0);
  p.timeout_ns = library_wait_timeout_ns();
  if (cfg.launch(al, tma ? kBRowTma : kBRowCp, sched.grid, p, &map_a, &map_b, stream) !=
      cudaSuccess) {
    cudaGetLastError();
    return SGEMM_ERR_LAUNCH;
  }
  return SGEMM_OK;
}

SGEMM_API int sgemm_noalloc_poll_status(void* stream_, int* detail) {
  if (detail) *detail = 0;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return SGEMM_ERR_LAUNCH;
  }
  if (cudaStreamSynchronize(stream) != cudaSuccess) {
    cudaGetLastError();
    return SGEMM_ERR_LAUNCH;
  }
  std::lock_guard<std::mutex> lock(g_na_mutex);
  if (dev < 0 || dev >= kNoAllocMaxDevices || !g_na_devices[dev].ready) return SGEMM_OK;
  NoAllocDevice& d = g_na_devices[dev];
  int code = 0;
  // plain synchronous copies to and from the array: nothing is allocated
  if (cudaMemcpy(&code, d.base, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return SGEMM_ERR_LAUNCH;
  }
  if (code == 0) return SGEMM_OK;
  // an aborted call can leave flags published that no owner consumed; a
  // replayed graph reuses its call number, so clear them
  if (cudaMemset(d.base, 0, kNoAllocHeaderBytes) != cudaSuccess) {
    cudaGetLastError();
    return SGEMM_ERR_LAUNCH;
  }
  if (detail) *detail = code;
  return SGEMM_ERR_DEVICE_TIMEOUT;
}
