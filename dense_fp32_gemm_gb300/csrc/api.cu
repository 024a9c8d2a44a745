// api.cu -- the extern "C" boundary of the library: argument validation,
// quick returns, choice of tile configuration, TMA descriptor for B, the
// per-(device, stream) workspace, and the launch.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>
#include <vector>

#include "../../include/sgemm_gb300.h"
#include "configs.hpp"
#include "dispatch.hpp"
#include "ffma_sgemm.cuh"
#include "schedule.hpp"
#include "tile_config.hpp"

#define SGEMM_API extern "C" __attribute__((visibility("default")))

namespace sgemm_gb300 {

bool library_staged_a_wanted(bool built, int occ, int occ_staged, const Schedule& s);

// The kernel for very small problems (tiny.cu).
bool tiny_wanted(int M, int N, int K);
cudaError_t tiny_launch(int dev, int M, int N, int K, float alpha, const float* A, long long lda,
                        const float* B, long long ldb, float beta, float* C, long long ldc,
                        cudaStream_t stream, char* text, int text_len);

namespace {

// ---- configuration registry -------------------------------------------------
#define SGEMM_GB300_ENTRY_PTR(NAME, ...) &kEntry##NAME,
const ConfigEntry* const kConfigs[] = {SGEMM_GB300_CONFIGS(SGEMM_GB300_ENTRY_PTR)};
#undef SGEMM_GB300_ENTRY_PTR
constexpr int kNumConfigs = sizeof(kConfigs) / sizeof(kConfigs[0]);
static_assert(kNumConfigIds == kNumConfigs, "config ids");

std::mutex g_mutex;
std::atomic<int> g_forced{-1};
// Row-major A through the staging ring and producer warp (ALoad kARowStg)
// where the configuration is built with it and A is TMA-aligned
// (sgemm_set_staged_a): 1 where each CTA also runs at least kStagedMinSteps
// k-slices, 2 whatever the size, 0 never (the transposing copy everywhere).
std::atomic<int> g_staged_a{1};
// Fewest k-slices per CTA (on average) for which the staged variant is used.
constexpr int kStagedMinSteps = 8;
// A schedule policy forced for every later call (tuner, tests); mode < 0:
// the tuned policy of the problem's shape class. Guarded by g_mutex.
SchedPolicy g_forced_policy{-1, 8, 4, 1};
std::atomic<long long> g_timeout_ns{4000000000LL};
thread_local char g_last_config[192] = "none";

struct DeviceInfo {
  bool ready = false;
  bool supported = false;
  int sms = 0;
  int occupancy[kNumConfigs] = {};  // resident CTAs per SM
  int occupancy_staged[kNumConfigs] = {};  // same, staged-A variant (0: not built)
};
std::map<int, DeviceInfo> g_devices;

struct Workspace {
  void* block = nullptr;
  size_t bytes = 0;
  int* status = nullptr;
  uint32_t* flags = nullptr;
  float* partials = nullptr;
  size_t flag_cap = 0;
  size_t partial_cap = 0;  // floats
  uint32_t epoch = 0;
};
std::map<std::pair<int, cudaStream_t>, Workspace> g_workspaces;

// Per-device set-up: compute capability check, shared-memory attributes and
// occupancy of every configuration. Called with g_mutex held.
int device_info(int dev, DeviceInfo** out) {
  DeviceInfo& d = g_devices[dev];
  if (!d.ready) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return SGEMM_ERR_LAUNCH;
    d.supported = (major == 10 && minor == 3);
    if (d.supported) {
      for (int c = 0; c < kNumConfigs; ++c) {
        if (kConfigs[c]->set_attributes() != cudaSuccess) return SGEMM_ERR_LAUNCH;
        int blocks = 0;
        if (kConfigs[c]->occupancy(&blocks) != cudaSuccess) return SGEMM_ERR_LAUNCH;
        d.occupancy[c] = blocks;
        blocks = 0;
        if (kConfigs[c]->staged && kConfigs[c]->occupancy_staged(&blocks) != cudaSuccess)
          return SGEMM_ERR_LAUNCH;
        d.occupancy_staged[c] = blocks;
      }
    }
    d.ready = true;
  }
  *out = &d;
  return d.supported ? SGEMM_OK : SGEMM_ERR_UNSUPPORTED_DEVICE;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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

// Workspace of at least `flags` flags and `partial_floats` floats for this
// (device, stream); grows by reallocation. Called with g_mutex held.
int get_workspace(int dev, cudaStream_t stream, size_t flags, size_t partial_floats,
                  Workspace** out) {
  Workspace& w = g_workspaces[{dev, stream}];
  if (w.block == nullptr || w.flag_cap < flags || w.partial_cap < partial_floats) {
    // allocation is not allowed while the stream is captured into a graph:
    // refuse instead of invalidating the capture
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
      cudaGetLastError();
      return SGEMM_ERR_CAPTURE;
    }
    if (cs != cudaStreamCaptureStatusNone) return SGEMM_ERR_CAPTURE;
    const size_t fcap = flags > w.flag_cap ? flags : w.flag_cap;
    const size_t pcap = partial_floats > w.partial_cap ? partial_floats : w.partial_cap;
    const size_t status_bytes = 256;
    const size_t flag_bytes = ((fcap * 4 + 255) / 256) * 256;
    const size_t bytes = status_bytes + flag_bytes + pcap * 4;
    if (w.block != nullptr) {
      // the old block may still be in use by queued work on this stream
      if (cudaStreamSynchronize(stream) != cudaSuccess) return SGEMM_ERR_LAUNCH;
      cudaFree(w.block);
      w.block = nullptr;
    }
    void* blk = nullptr;
    if (cudaMalloc(&blk, bytes) != cudaSuccess) {
      cudaGetLastError();
      w = Workspace{};
      return SGEMM_ERR_ALLOC;
    }
    if (cudaMemsetAsync(blk, 0, status_bytes + flag_bytes, stream) != cudaSuccess)
      return SGEMM_ERR_LAUNCH;
    w.block = blk;
    w.bytes = bytes;
    w.status = static_cast<int*>(blk);
    w.flags = reinterpret_cast<uint32_t*>(static_cast<char*>(blk) + status_bytes);
    w.partials = reinterpret_cast<float*>(static_cast<char*>(blk) + status_bytes + flag_bytes);
    w.flag_cap = fcap;
    w.partial_cap = pcap;
  }
  *out = &w;
  return SGEMM_OK;
}


int current_device(int* dev) {
  if (cudaGetDevice(dev) != cudaSuccess) {
    cudaGetLastError();
    return SGEMM_ERR_LAUNCH;
  }
  return SGEMM_OK;
}

// C = beta * C for `batch` matrices (beta == 0 writes zeros without reading C).
__global__ void scale_c_kernel(int M, int N, float beta, float* C, long long ldc, long long sC,
                               int batch) {
  const long long per = (long long)M * N;
  const long long total = per * batch;
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
       e += (long long)gridDim.x * blockDim.x) {
    const long long bi = e / per, r = e - bi * per;
    const long long i = r / N, j = r % N;
    float* c = C + bi * sC + i * ldc + j;
    *c = beta == 0.f ? 0.f : beta * *c;
  }
}

// 3-D tensor map over `batch` row-major matrices of rows x cols (row pitch ld,
// matrix pitch stride, in elements) with a box of box_cols x box_rows x 1.
bool encode_3d(PFN_cuTensorMapEncodeTiled_v12000 enc, CUtensorMap* map, const float* base,
               int cols, int rows, long long ld, long long stride, int batch, int box_cols,
               int box_rows, CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_NONE) {
  const long long pitch2 = batch > 1 ? stride : ld * (rows > 0 ? rows : 1);
  cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)batch};
  cuuint64_t strides[2] = {(cuuint64_t)ld * 4, (cuuint64_t)(((pitch2 * 4) + 15) / 16 * 16)};
  cuuint32_t box[3] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Argument checks shared by every FFMA entry point; 0 when valid.
int check_args(int opA, int opB, int M, int N, int K, float alpha, const float* A, int lda,
               long long sA, const float* B, int ldb, long long sB, float* C, int ldc,
               long long sC, int batch) {
  if ((opA != SGEMM_OP_N && opA != SGEMM_OP_T) || (opB != SGEMM_OP_N && opB != SGEMM_OP_T))
    return SGEMM_ERR_INVALID_VALUE;
  if (M < 0 || N < 0 || K < 0 || batch < 0) return SGEMM_ERR_INVALID_DIM;
  const int lda_min = opA == SGEMM_OP_N ? K : M;
  const int ldb_min = opB == SGEMM_OP_N ? N : K;
  if (lda < (lda_min > 1 ? lda_min : 1) || ldb < (ldb_min > 1 ? ldb_min : 1) ||
      ldc < (N > 1 ? N : 1))
    return SGEMM_ERR_INVALID_LD;
  if (sA < 0 || sB < 0 || sC < 0) return SGEMM_ERR_INVALID_VALUE;
  if (M == 0 || N == 0 || batch == 0) return SGEMM_OK;
  const bool reads_ab = (K > 0 && alpha != 0.f);
  if (C == nullptr || (reads_ab && (A == nullptr || B == nullptr))) return SGEMM_ERR_NULL_PTR;
  if ((reinterpret_cast<uintptr_t>(C) & 3u) ||
      (reads_ab && ((reinterpret_cast<uintptr_t>(A) & 3u) || (reinterpret_cast<uintptr_t>(B) & 3u))))
    return SGEMM_ERR_MISALIGNED;
  return SGEMM_OK;
}

// The FFMA path for every operand layout and batch count (arguments checked).
int run_ffma(int opA, int opB, int M, int N, int K, float alpha, const float* A, int lda,
             long long sA, const float* B, int ldb, long long sB, float beta, float* C, int ldc,
             long long sC, int batch, cudaStream_t stream) {
  if (M == 0 || N == 0 || batch == 0) return SGEMM_OK;
  const bool reads_ab = (K > 0 && alpha != 0.f);
  int dev = 0;
  int st = current_device(&dev);
  if (st != SGEMM_OK) return st;

  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceInfo* di = nullptr;
  st = device_info(dev, &di);
  if (st != SGEMM_OK) return st;

  if (!reads_ab) {
    const long long total = (long long)M * N * batch;
    int blocks = (int)((total + 255) / 256);
    if (blocks > di->sms * 8) blocks = di->sms * 8;
    scale_c_kernel<<<blocks, 256, 0, stream>>>(M, N, beta, C, ldc, sC, batch);
    if (cudaGetLastError() != cudaSuccess) return SGEMM_ERR_LAUNCH;
    snprintf(g_last_config, sizeof(g_last_config), "scale_c");
    return SGEMM_OK;
  }

  const bool row_major = (opA == SGEMM_OP_N && opB == SGEMM_OP_N);
  int id = g_forced.load();
  // very small row-major problems: the latency-first kernel (tiny.cu), unless
  // a tile configuration is forced
  if (id < 0 && row_major && batch == 1 && tiny_wanted(M, N, K)) {
    if (tiny_launch(dev, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream, g_last_config,
                    (int)sizeof(g_last_config)) != cudaSuccess) {
      cudaGetLastError();
      return SGEMM_ERR_LAUNCH;
    }
    return SGEMM_OK;
  }
  if (id < 0 || id >= kNumConfigs || (!row_major && !kConfigs[id]->all_layouts))
    id = choose_config(M, N, K);
  const SchedPolicy policy =
      g_forced_policy.mode >= 0 ? g_forced_policy : choose_policy(M, N, K);
  // transposed operands need a configuration built for them
  if (!row_major && !kConfigs[id]->all_layouts) id = kFallbackConfigId;
  const ConfigEntry& cfg = *kConfigs[id];
  const TileShape& S = cfg.shape;

  // operand load modes: TMA where the pointer, leading dimension and batch
  // stride are 16-byte multiples, else 4-byte copies
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  const bool single = batch == 1;
  CUtensorMap map_a, map_b;
  std::memset(&map_a, 0, sizeof(map_a));
  std::memset(&map_b, 0, sizeof(map_b));
  int al = kARow, bl = kBRowCp;
  if (opA == SGEMM_OP_T) {
    al = kATCp;
    if (enc != nullptr && ((reinterpret_cast<uintptr_t>(A) & 15u) == 0) && ((lda & 3) == 0) &&
        (single || (sA & 3) == 0) &&
        encode_3d(enc, &map_a, A, M, K, lda, sA, batch, S.BM, S.BK))
      al = kATTma;
  }
  if (opB == SGEMM_OP_T) {
    bl = kBT;
  } else if (enc != nullptr && ((reinterpret_cast<uintptr_t>(B) & 15u) == 0) && ((ldb & 3) == 0) &&
             (single || (sB & 3) == 0) &&
             encode_3d(enc, &map_b, B, N, K, ldb, sB, batch, S.BN, S.BK)) {
    bl = kBRowTma;
  }

  const int occ = di->occupancy[id];
  if (occ < 1) return SGEMM_ERR_LAUNCH;
  const int tiles_m = ceil_div_nn(M, S.BM), tiles_n = ceil_div_nn(N, S.BN);
  const int kiters = ceil_div_nn(K, S.BK);
  const long long total_tiles = (long long)tiles_m * tiles_n * batch;
  if (total_tiles > 0x7fffffffLL) return SGEMM_ERR_INVALID_DIM;
  Schedule sched = make_schedule(tiles_m, tiles_n, kiters, di->sms * occ, policy, batch);
  // row-major A with B by TMA: the staged variant where it is built, keeps
  // the configuration's residency, A is TMA-aligned (a K x M box of 32 x BM,
  // 128-byte swizzled), and each CTA runs enough k-slices to cover the extra
  // step of latency the staging adds before the first FMA (measured on
  // GB300: 4 k-slices per CTA at 512^3 lose 5 %, 13 at 1024^3 gain 4 %)
  if (al == kARow && bl == kBRowTma &&
      library_staged_a_wanted(cfg.staged, occ, di->occupancy_staged[id], sched) &&
      ((reinterpret_cast<uintptr_t>(A) & 15u) == 0) && ((lda & 3) == 0) &&
      (single || (sA & 3) == 0) &&
      encode_3d(enc, &map_a, A, K, M, lda, sA, batch, S.BK, S.BM, CU_TENSOR_MAP_SWIZZLE_128B))
    al = kARowStg;

  const bool split = sched.dp_tiles < sched.tiles;
  Workspace* ws = nullptr;
  st = get_workspace(dev, stream, (size_t)sched.grid,
                     split ? (size_t)sched.grid * S.BM * S.BN : 0, &ws);
  if (st != SGEMM_OK) return st;
  if (++ws->epoch == 0) ws->epoch = 1;

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
  p.sA = sA;
  p.sB = sB;
  p.sC = sC;
  p.sched = sched;
  p.ws = ws->partials;
  p.flags = ws->flags;
  p.status = ws->status;
  p.epoch = ws->epoch;
  p.c_vec = ((reinterpret_cast<uintptr_t>(C) & 15u) == 0) && ((ldc & 3) == 0) &&
            (single || (sC & 3) == 0);
  p.timeout_ns = g_timeout_ns.load();

  if (cfg.launch(al, bl, sched.grid, p, &map_a, &map_b, stream) != cudaSuccess) {
    cudaGetLastError();
    return SGEMM_ERR_LAUNCH;
  }
  static const char* const kAName[] = {"a=rowT", "a=tma", "a=cp", "a=stg"};
  static const char* const kBName[] = {"b=tma", "b=cp", "b=colT"};
  snprintf(g_last_config, sizeof(g_last_config),
           "%s %s %s grid=%d dp=%d split=%d kiters=%d sched=%d/g%d/u%d/s%d%s", cfg.name,
           kAName[al], kBName[bl], sched.grid, sched.dp_tiles, sched.tiles - sched.dp_tiles,
           sched.kiters, policy.mode, sched.group_m, policy.min_units, policy.splits,
           batch > 1 ? " batched" : "");
  return SGEMM_OK;
}

__global__ void diag_wait_kernel(int* status, long long timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_w;
  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_addr(&bar), 1);
    abort_w = 0;
    ptx::mbar_fence_init();
  }
  __syncthreads();
  // phase 0 of `bar` never completes: nothing arrives
  bounded_wait(ptx::smem_addr(&bar), 0u, &abort_w, status, kDevTimeoutFull, timeout_ns);
}


}  // namespace

// ---- internal hooks for the other entry points of the library -------------
// Scratch of at least `floats` floats (and the status word) in the
// per-(device, stream) workspace.
// With nflags > 0 it also returns the flag array and this call's epoch (a
// value no flag holds before this call publishes it).
int library_workspace(int dev, cudaStream_t stream, size_t floats, size_t nflags, float** scratch,
                      int** status, uint32_t** flags, uint32_t* epoch) {
  std::lock_guard<std::mutex> lock(g_mutex);
  Workspace* ws = nullptr;
  const int st = get_workspace(dev, stream, nflags > 0 ? nflags : 1, floats, &ws);
  if (st != SGEMM_OK) return st;
  *scratch = ws->partials;
  *status = ws->status;
  if (flags != nullptr) *flags = ws->flags;
  if (epoch != nullptr) {
    if (++ws->epoch == 0) ws->epoch = 1;
    *epoch = ws->epoch;
  }
  return SGEMM_OK;
}

// SM count of a supported device (and its one-time set-up).
int library_device_sms(int dev, int* sms) {
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceInfo* di = nullptr;
  const int st = device_info(dev, &di);
  if (st != SGEMM_OK) return st;
  *sms = di->sms;
  return SGEMM_OK;
}

void note_last_config(const char* text) { snprintf(g_last_config, sizeof(g_last_config), "%s", text); }

long long library_wait_timeout_ns() { return g_timeout_ns.load(); }

// Whether a row-major problem whose B arrives by TMA takes A through the
// staging ring (ALoad kARowStg), before the alignment checks: the
// configuration is built with it at the same residency, and the
// sgemm_set_staged_a mode allows it (2: always; 1: when each CTA runs at
// least kStagedMinSteps k-slices). Shared by sgemm() and sgemm_noalloc.
bool library_staged_a_wanted(bool built, int occ, int occ_staged, const Schedule& s) {
  const int mode = g_staged_a.load();
  return built && mode != 0 && occ_staged == occ &&
         (mode == 2 || (long long)s.tiles * s.kiters >= (long long)kStagedMinSteps * s.grid);
}

// The FFMA path on device matrices (row-major, arguments already checked).
int library_ffma(int M, int N, int K, float alpha, const float* A, int lda, const float* B,
                 int ldb, float beta, float* C, int ldc, cudaStream_t stream) {
  return run_ffma(SGEMM_OP_N, SGEMM_OP_N, M, N, K, alpha, A, lda, 0, B, ldb, 0, beta, C, ldc, 0, 1,
                  stream);
}

}  // namespace sgemm_gb300

using namespace sgemm_gb300;

SGEMM_API const char* sgemm_status_string(int status) {
  switch (status) {
    case SGEMM_OK: return "ok";
    case SGEMM_ERR_INVALID_DIM: return "invalid dimension (M, N or K negative)";
    case SGEMM_ERR_INVALID_LD: return "invalid leading dimension";
    case SGEMM_ERR_NULL_PTR: return "null matrix pointer";
    case SGEMM_ERR_UNSUPPORTED_DEVICE: return "current device is not sm_103 (GB300)";
    case SGEMM_ERR_LAUNCH: return "CUDA runtime error";
    case SGEMM_ERR_DEVICE_TIMEOUT: return "a kernel gave up on a bounded wait";
    case SGEMM_ERR_ALLOC: return "workspace allocation failed";
    case SGEMM_ERR_MISALIGNED: return "matrix pointer not 4-byte aligned";
    case SGEMM_ERR_INVALID_VALUE: return "invalid argument value";
    case SGEMM_ERR_NOALLOC_CAPACITY:
      return "problem needs more scratch than the fixed no-allocation buffer holds";
    case SGEMM_ERR_CAPTURE:
      return "workspace must grow while the stream is being captured (call once before capture)";
    default: return "unknown status";
  }
}

SGEMM_API int sgemm(int M, int N, int K, float alpha, const float* A, int lda, const float* B,
                    int ldb, float beta, float* C, int ldc, void* stream) {
  const int st = check_args(SGEMM_OP_N, SGEMM_OP_N, M, N, K, alpha, A, lda, 0, B, ldb, 0, C, ldc,
                            0, 1);
  if (st != SGEMM_OK || M == 0 || N == 0) return st;
  return run_ffma(SGEMM_OP_N, SGEMM_OP_N, M, N, K, alpha, A, lda, 0, B, ldb, 0, beta, C, ldc, 0,
                  1, static_cast<cudaStream_t>(stream));
}

SGEMM_API int sgemm_ex(int opA, int opB, int M, int N, int K, float alpha, const float* A,
                       int lda, const float* B, int ldb, float beta, float* C, int ldc,
                       void* stream) {
  const int st = check_args(opA, opB, M, N, K, alpha, A, lda, 0, B, ldb, 0, C, ldc, 0, 1);
  if (st != SGEMM_OK || M == 0 || N == 0) return st;
  return run_ffma(opA, opB, M, N, K, alpha, A, lda, 0, B, ldb, 0, beta, C, ldc, 0, 1,
                  static_cast<cudaStream_t>(stream));
}

SGEMM_API int sgemm_strided_batched(int opA, int opB, int M, int N, int K, float alpha,
                                    const float* A, int lda, long long strideA, const float* B,
                                    int ldb, long long strideB, float beta, float* C, int ldc,
                                    long long strideC, int batch, void* stream) {
  const int st = check_args(opA, opB, M, N, K, alpha, A, lda, strideA, B, ldb, strideB, C, ldc,
                            strideC, batch);
  if (st != SGEMM_OK || M == 0 || N == 0 || batch == 0) return st;
  return run_ffma(opA, opB, M, N, K, alpha, A, lda, strideA, B, ldb, strideB, beta, C, ldc,
                  strideC, batch, static_cast<cudaStream_t>(stream));
}

SGEMM_API int sgemm_last_config(char* buf, int len) {
  if (buf == nullptr || len < 1) return SGEMM_ERR_INVALID_VALUE;
  snprintf(buf, (size_t)len, "%s", g_last_config);
  return SGEMM_OK;
}

SGEMM_API int sgemm_poll_device_status(void* stream_, int* detail) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  if (detail) *detail = 0;
  int dev = 0;
  int st = current_device(&dev);
  if (st != SGEMM_OK) return st;
  if (cudaStreamSynchronize(stream) != cudaSuccess) {
    cudaGetLastError();
    return SGEMM_ERR_LAUNCH;
  }
  std::lock_guard<std::mutex> lock(g_mutex);
  auto it = g_workspaces.find({dev, stream});
  if (it == g_workspaces.end() || it->second.status == nullptr) return SGEMM_OK;
  int code = 0;
  if (cudaMemcpy(&code, it->second.status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return SGEMM_ERR_LAUNCH;
  if (code != 0) {
    if (cudaMemset(it->second.status, 0, sizeof(int)) != cudaSuccess) return SGEMM_ERR_LAUNCH;
    // an aborted launch can leave split-K flags set that no owner consumed
    if (it->second.flags != nullptr &&
        cudaMemset(it->second.flags, 0, it->second.flag_cap * 4) != cudaSuccess)
      return SGEMM_ERR_LAUNCH;
    if (detail) *detail = code;
    return SGEMM_ERR_DEVICE_TIMEOUT;
  }
  return SGEMM_OK;
}

namespace sgemm_gb300 {
void host_api_release();
}

SGEMM_API void sgemm_shutdown(void) {
  sgemm_gb300::host_api_release();
  std::lock_guard<std::mutex> lock(g_mutex);
  int cur = 0;
  const bool have_cur = cudaGetDevice(&cur) == cudaSuccess;
  for (auto& kv : g_workspaces) {
    if (kv.second.block) {
      cudaSetDevice(kv.first.first);
      cudaDeviceSynchronize();
      cudaFree(kv.second.block);
    }
  }
  g_workspaces.clear();
  if (have_cur) cudaSetDevice(cur);
  cudaGetLastError();
}

SGEMM_API int sgemm_config_count(void) { return kNumConfigs; }

SGEMM_API int sgemm_config_info(int id, char* name, int len, int* params) {
  if (id < 0 || id >= kNumConfigs) return SGEMM_ERR_INVALID_VALUE;
  const ConfigEntry& c = *kConfigs[id];
  if (name != nullptr && len > 0) snprintf(name, (size_t)len, "%s", c.name);
  if (params != nullptr) {
    const TileShape& s = c.shape;
    const int v[13] = {s.BM, s.BN, s.BK, s.WM, s.WN, s.WNITER, s.TM, s.TN, s.NT, s.STAGES, s.MINB,
                       s.KU, s.ORDER};
    for (int i = 0; i < 13; ++i) params[i] = v[i];
  }
  return SGEMM_OK;
}

SGEMM_API int sgemm_config_layouts(int id) {
  if (id < 0 || id >= kNumConfigs) return SGEMM_ERR_INVALID_VALUE;
  return kConfigs[id]->all_layouts ? 1 : 0;
}

SGEMM_API int sgemm_set_staged_a(int on) {
  if (on < 0 || on > 2) return SGEMM_ERR_INVALID_VALUE;
  return g_staged_a.exchange(on);
}

SGEMM_API int sgemm_force_config(int id) {
  if (id < -1 || id >= kNumConfigs) return SGEMM_ERR_INVALID_VALUE;
  g_forced.store(id);
  return SGEMM_OK;
}

SGEMM_API int sgemm_cfg_check(const int* params, int* derived) {
  if (params == nullptr) return SGEMM_ERR_INVALID_VALUE;
  const TileShape s{params[0], params[1], params[2], params[3], params[4],  params[5],
                    params[6], params[7], params[8], params[9], params[10], params[11], params[12]};
  const int rule = cfg_check(s);
  if (rule == 0 && derived != nullptr) {
    derived[0] = wmiter(s);
    derived[1] = wsubm(s);
    derived[2] = wsubn(s);
    derived[3] = acc_per_thread(s);
    derived[4] = smem_bytes(s);
  }
  return rule;
}

namespace {
int schedule_out(int M, int N, int K, int BM, int BN, int BK, int capacity,
                 const SchedPolicy& pol, int* out) {
  if ((long long)ceil_div_nn(M, BM) * ceil_div_nn(N, BN) > 0x7fffffffLL)
    return SGEMM_ERR_INVALID_DIM;
  const Schedule s = make_schedule(ceil_div_nn(M, BM), ceil_div_nn(N, BN), ceil_div_nn(K, BK),
                                   capacity, pol);
  const int v[8] = {s.tiles_m, s.tiles_n, s.kiters, s.grid, s.dp_tiles, s.sk_q, s.sk_r, s.group_m};
  for (int i = 0; i < 8; ++i) out[i] = v[i];
  return SGEMM_OK;
}
}  // namespace

SGEMM_API int sgemm_schedule_query(int M, int N, int K, int id, int capacity, int* out) {
  if (M < 0 || N < 0 || K < 0) return SGEMM_ERR_INVALID_DIM;
  if (id < 0 || id >= kNumConfigs || capacity < 1 || out == nullptr)
    return SGEMM_ERR_INVALID_VALUE;
  const TileShape& S = kConfigs[id]->shape;
  SchedPolicy pol;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    pol = g_forced_policy.mode >= 0 ? g_forced_policy : choose_policy(M, N, K);
  }
  return schedule_out(M, N, K, S.BM, S.BN, S.BK, capacity, pol, out);
}

SGEMM_API int sgemm_schedule_plan(int M, int N, int K, int BM, int BN, int BK, int capacity,
                                  const int* policy, int* out) {
  if (M < 0 || N < 0 || K < 0) return SGEMM_ERR_INVALID_DIM;
  if (BM < 1 || BN < 1 || BK < 1 || capacity < 1 || policy == nullptr || out == nullptr)
    return SGEMM_ERR_INVALID_VALUE;
  const SchedPolicy pol{policy[0], policy[1], policy[2], policy[3]};
  if (!policy_valid(pol)) return SGEMM_ERR_INVALID_VALUE;
  return schedule_out(M, N, K, BM, BN, BK, capacity, pol, out);
}

SGEMM_API int sgemm_force_schedule(const int* policy) {
  std::lock_guard<std::mutex> lock(g_mutex);
  if (policy == nullptr || policy[0] < 0) {
    g_forced_policy.mode = -1;
    return SGEMM_OK;
  }
  const SchedPolicy pol{policy[0], policy[1], policy[2], policy[3]};
  if (!policy_valid(pol)) return SGEMM_ERR_INVALID_VALUE;
  g_forced_policy = pol;
  return SGEMM_OK;
}

SGEMM_API int sgemm_choose_policy(int M, int N, int K, int* policy) {
  if (M < 0 || N < 0 || K < 0) return SGEMM_ERR_INVALID_DIM;
  if (policy == nullptr) return SGEMM_ERR_INVALID_VALUE;
  const SchedPolicy p = choose_policy(M, N, K);
  policy[0] = p.mode;
  policy[1] = p.group_m;
  policy[2] = p.min_units;
  policy[3] = p.splits;
  return SGEMM_OK;
}

SGEMM_API int sgemm_schedule_piece(const int* v, int b, int i, int* out) {
  if (v == nullptr || out == nullptr) return SGEMM_ERR_INVALID_VALUE;
  Schedule s{};
  s.tiles_m = v[0];
  s.tiles_n = v[1];
  s.tiles = v[0] * v[1];
  s.kiters = v[2];
  s.grid = v[3];
  s.dp_tiles = v[4];
  s.sk_q = v[5];
  s.sk_r = v[6];
  s.group_m = v[7];
  s.sk_units = (int64_t)(s.tiles - s.dp_tiles) * s.kiters;
  if (s.grid < 1 || s.kiters < 1 || s.group_m < 1 || b < 0 || b >= s.grid)
    return SGEMM_ERR_INVALID_VALUE;
  const int n = num_pieces(s, b);
  if (i < 0 || i >= n) return SGEMM_ERR_INVALID_VALUE;
  const Piece p = get_piece(s, b, i);
  int tm, tn;
  tile_coords(s, p.tile, tm, tn);
  const int o[7] = {p.tile, p.kb, p.ke, tm, tn, num_contributors(s, b, p),
                    is_partial_piece(s, p) ? 1 : 0};
  for (int k = 0; k < 7; ++k) out[k] = o[k];
  return n;
}

SGEMM_API int sgemm_diag_wait_timeout(long long timeout_ns, void* stream_) {
  if (timeout_ns < 1000) return SGEMM_ERR_INVALID_VALUE;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  int dev = 0;
  int st = current_device(&dev);
  if (st != SGEMM_OK) return st;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceInfo* di = nullptr;
  st = device_info(dev, &di);
  if (st != SGEMM_OK) return st;
  Workspace* ws = nullptr;
  st = get_workspace(dev, stream, 1, 0, &ws);
  if (st != SGEMM_OK) return st;
  diag_wait_kernel<<<1, 32, 0, stream>>>(ws->status, timeout_ns);
  return cudaGetLastError() == cudaSuccess ? SGEMM_OK : SGEMM_ERR_LAUNCH;
}

SGEMM_API long long sgemm_set_wait_timeout_ns(long long ns) {
  if (ns < 1000) return SGEMM_ERR_INVALID_VALUE;
  return g_timeout_ns.exchange(ns);
}

SGEMM_API int sgemm_choose_config(int M, int N, int K, int* shape_class) {
  if (M < 0 || N < 0 || K < 0) return SGEMM_ERR_INVALID_DIM;
  if (shape_class != nullptr) *shape_class = classify_shape(M, N, K);
  return choose_config(M, N, K);
}
