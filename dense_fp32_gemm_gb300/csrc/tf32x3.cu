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
// x_hi is never stored: the TF32 MMA reads an FP32 value's sign, exponent and
// top 10 mantissa bits and ignores the low 13, which is exactly x_hi. (Measured
// on GB300: results with x_hi = x and with x_hi = trunc(x) are bit-identical;
// the parity tests hold the path to the oracle either way.)
//
// Data flow:
//   1. B is transposed into the per-stream workspace (N x K, K-major, rows
//      padded to a multiple of 4 floats for TMA); A is read where it is when
//      its rows are 16-byte aligned, else copied there too;
//   2. the GEMM kernel (one CTA of 10 warps per SM, persistent over 128 x 256
//      tiles, or the narrow tiles below): warp 0 issues TMA loads of the raw
//      A and B^T tiles of each k-slice (swizzled) into a ring of stages;
//      warps 6-9 write the residual tiles A_lo, B_lo beside them in the same
//      stage; warp 1 owns two TMEM accumulators of the tile's width and
//      issues, per 8-wide k-step, the three tcgen05.mma.kind::tf32 products;
//      warps 2-5 read an accumulator back with tcgen05.ld and apply
//      alpha * acc + beta * C.
//
// Kernel forms (sgemm_3xtf32_set_kernel_form):
//   * two-SM pairs (the default where the device co-schedules CTA pairs and
//     the problem has two waves of whole tile pairs): the CTAs of a cluster
//     of two take tile rows 2i and 2i + 1 of one tile column. Each holds its
//     A tile and one half (128 columns) of the B tile, so a 32-wide stage is
//     64 KB; the even CTA issues M = 256 MMAs (cta_group::2) that read A and
//     B from both CTAs' shared memory and write each CTA's 128 accumulator
//     rows into its own TMEM. The even CTA's conv barrier completes when the
//     converters of both CTAs are done (the odd CTA's through one relayed
//     remote arrival per stage); its commits free the stage and publish the
//     accumulator in both CTAs; its MMA thread waits for both epilogues.
//   * single CTAs, each with its own A and B tiles.
//   * narrow tiles, 64 wide (N <= 64, or few tiles) or 128 wide (N <= 128,
//     or little 256-wide work): single CTAs whose converter warps store A's raw values
//     and residuals into tensor memory (tcgen05.st), where the MMAs read A;
//     shared memory holds A's raw tile and B's two parts, so a stage is 32 KB
//     (six fit) or 48 KB (four).
// Each CTA loads only its own tiles; no TMA load is multicast.
// Before exiting, a CTA of a pair waits (bounded) until its barriers have
// received the peer's last arrivals, then meets the peer at a cluster
// barrier (two-SM pairs free their TMEM together after it).
// Every wait is bounded (see ffma_sgemm.cuh); a CTA that gives up drains its
// copies and MMAs, frees its TMEM and returns.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
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
int library_workspace(int dev, cudaStream_t stream, size_t floats, size_t nflags, float** scratch,
                      int** status, uint32_t** flags, uint32_t* epoch);
int library_device_sms(int dev, int* sms);
void note_last_config(const char* text);
long long library_wait_timeout_ns();

namespace x3 {

constexpr int BM = 128, BN = 256, NT = 320;

constexpr int kStageRegion = 192 * 1024;  // the ring of stages
constexpr int kMaxStages = 6;

// The k-slice: BK values of K per stage, in swizzled rows of 4 * BK bytes,
// with as many stages as fit in the stage region. With whole B tiles, BK = 16
// (four 48 KB stages, 64-byte swizzle) lets the loads run three stages ahead
// of the MMAs and BK = 32 (two 96 KB stages, 128-byte swizzle) has half the
// per-stage hand-offs; measured on GB300, 16 is faster from K = 1024 up
// (4096^3: 251 against 226 TFLOP/s), 32 below (8191 x 1000 x 777: 99 against
// 86 TFLOP/s). B_PARTS = 2 (the two-SM form): a CTA holds half of each B
// tile, and BK = 32 gives three 64 KB stages (its hand-offs between the CTAs
// of a pair cost more, so it always takes 32; 16-wide stages measured 158
// against 265 TFLOP/s at 4096^3).
// BNT: the tile's width in N (BN, or 64 or 128: see make_plan); a narrow
// tile gets as many stages as fit, up to kMaxStages. A_TMEM (the narrow
// tiles): A's parts live in tensor memory, so a stage holds only A's raw
// tile for them.
template <int BK_, int B_PARTS = 1, int BNT = BN, bool A_TMEM = false>
struct Slice {
  static constexpr int BK = BK_;
  static_assert(BK == 32 || BK == 16, "k-slice width");
  static constexpr int ROW_BYTES = BK * 4;
  static constexpr int A_BYTES = BM * BK * 4;                      // one of A_hi, A_lo
  static constexpr int B_BYTES = BNT / B_PARTS * BK * 4;           // one of B_hi, B_lo
  // a stage: [A_hi | A_lo | B_hi | B_lo]; TMA writes the _hi tiles (the raw
  // values), the converter warps the _lo tiles. A_TMEM: [A_hi | B_hi | B_lo],
  // the converters put A's two parts in tensor memory instead
  static constexpr int B_OFF = (A_TMEM ? 1 : 2) * A_BYTES;        // B_hi in a stage
  static constexpr int STAGE_BYTES = B_OFF + 2 * B_BYTES;  // 96 / 48 KB, 64 KB pairs, 32 KB narrow
  static constexpr int ST = kStageRegion / STAGE_BYTES < kMaxStages
                                ? kStageRegion / STAGE_BYTES
                                : kMaxStages;                      // 2 / 4, or 3 / 6
};
static_assert(Slice<16>::ST * Slice<16>::STAGE_BYTES == kStageRegion &&
                  Slice<32>::ST * Slice<32>::STAGE_BYTES == kStageRegion &&
                  Slice<32, 2>::ST * Slice<32, 2>::STAGE_BYTES == kStageRegion &&
                  Slice<16>::ST <= kMaxStages,
              "every width fills the same stage region");
constexpr int NBUF = 2;                   // accumulators, so the epilogue overlaps the next MMAs
// One FP32 accumulator is 128 lanes x BNT columns; NBUF of them (all 512
// columns for BNT = BN; 128 or 256 for the narrow tiles, whose A slots take
// the rest).
constexpr int tmem_cols(int bnt) { return NBUF * bnt; }
// Kernel forms (the values sgemm_3xtf32_set_kernel_form takes): single CTAs;
// CTA pairs whose even CTA issues M = 256 MMAs over both (cta_group::2),
// each CTA holding half of every B tile.
enum Form : int { kSingle = 1, kTwoSmPair = 2 };
// Stages of a (form, k-slice width, tile width): Slice<>::ST, for the host.
constexpr int stages_of(int form, int bk, int bnt) {
  const bool a_tmem = form == kSingle && bnt != BN;  // the kernel's A_TM
  const int b_rows = bnt / (form == kTwoSmPair ? 2 : 1);
  const int stage = (a_tmem ? 1 : 2) * BM * bk * 4 + 2 * b_rows * bk * 4;
  return kStageRegion / stage < kMaxStages ? kStageRegion / stage : kMaxStages;
}
constexpr int EPI_THREADS = 128;          // warps 2-5
constexpr int CONV_WARP0 = 6;             // warps 6-9 write the residual tiles
constexpr int CONV_THREADS = 128;
constexpr uint32_t IDESC_PAIR = tc::idesc_tf32(2 * BM, BN);  // M = 256 over a CTA pair
static_assert(BN % 16 == 0 && BN <= 256 && BM == 128, "MMA shape");
// the narrow tiles: 64 wide for N <= 64 and problems of few tiles, 128 wide
// for N <= 128 and problems with little 256-wide work (make_plan)
constexpr int BN_NARROW = 64, BN_MID = 128;
// the host's stage count (plan, shared-memory layout) is the kernel's, for
// every instantiated tile
static_assert(stages_of(kSingle, 16, BN) == Slice<16>::ST &&
                  stages_of(kSingle, 32, BN) == Slice<32>::ST &&
                  stages_of(kTwoSmPair, 32, BN) == Slice<32, 2>::ST &&
                  stages_of(kSingle, 32, BN_NARROW) == Slice<32, 1, BN_NARROW, true>::ST &&
                  stages_of(kSingle, 32, BN_MID) == Slice<32, 1, BN_MID, true>::ST,
              "stage counts");

struct Barriers {
  uint64_t full[kMaxStages];   // TMA transaction bytes of one stage (the raw tiles)
  uint64_t conv[kMaxStages];   // the converter warps have written the stage's residuals
                               // (two-SM form, even CTA: also the odd CTA's, relayed)
  uint64_t empty[kMaxStages];  // MMAs that read a stage have completed
  uint64_t tmem_full[NBUF];    // a piece's last MMA into accumulator i has completed
  uint64_t tmem_empty[NBUF];   // the epilogue warps have read accumulator i (two-SM
                               // form, even CTA: those of both CTAs)
  uint64_t drain;          // final MMA completion on the abort path
  uint64_t epi_sync;       // rendezvous of the 128 epilogue threads
  uint32_t tmem_addr;
  int abort;
};
// epilogue staging: per epilogue warp 32 rows x 32 columns (pitch 36 floats:
// row-wise 128-bit writes and the transposed 128-bit reads are conflict-free)
constexpr int EPI_PITCH = 36;
constexpr int EPI_WARP_FLOATS = 32 * EPI_PITCH;
constexpr int BAR_BYTES = ((int)sizeof(Barriers) + 15) / 16 * 16;
constexpr int SMEM_BYTES = 1024 + kStageRegion + BAR_BYTES + 4 * EPI_WARP_FLOATS * 4;
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");

struct Params {
  int M, N, K;
  float alpha, beta;
  float* C;
  long long ldc;
  Schedule sched;     // whole tiles, then K-split tiles (schedule.hpp)
  float* ws;          // grid partial tiles of BM x BNT floats, column-major
  uint32_t* flags;    // flags[s] == epoch once slot s's partial is written; reset
                      // to 0 by the owner that reads it
  uint32_t epoch;
  int* status;
  long long timeout_ns;
};

__device__ __forceinline__ float tf32_trunc(float x) {
  return __uint_as_float(__float_as_uint(x) & 0xFFFFE000u);
}

// A (M x K, lda) -> a copy with rows of ldw floats (a multiple of 4), for an A
// whose rows are not 16-byte aligned (TMA needs them to be). Rows over
// blockIdx.y (strided by gridDim.y), columns over x.
__global__ void pack_a_kernel(int M, int K, const float* __restrict__ A, long long lda,
                              float* __restrict__ out, long long ldw) {
  for (int m = blockIdx.y; m < M; m += gridDim.y) {
    const float* a = A + (long long)m * lda;
    float* o = out + (long long)m * ldw;
    for (int k = blockIdx.x * blockDim.x + threadIdx.x; k < K; k += gridDim.x * blockDim.x)
      o[k] = a[k];
  }
}

// B (K x N, ldb) -> B^T (N x K, ldw), through 32 x 32 shared-memory tiles so
// that both the reads and the writes are coalesced: one tile per block, tile
// column blockIdx.x, tile row k_base / 32 + blockIdx.y (the host launches one
// grid per 65535 tile rows). Bounds are compared as remaining extents, so no
// index passes K or N even for K, N near 2^31. (A grid-stride form of this
// kernel, looping over tile rows in 64-bit indices, took 43 us instead of
// 23 us at 4096 x 4096 on GB300.)
__global__ void transpose_b_kernel(int K, int N, const float* __restrict__ B, long long ldb,
                                   float* __restrict__ bt, long long ldw, int k_base) {
  __shared__ float tile[32][33];
  // may be launched before the kernel ahead of it on the stream has finished
  // (programmatic dependent launch): wait for it before touching memory
  ptx::griddep_wait();
  const int n0 = blockIdx.x * 32, k0 = k_base + blockIdx.y * 32;
  const int kn = K - k0, nn = N - n0;             // both > 0
  const int tx = threadIdx.x, ty = threadIdx.y;  // 32 x 8 threads
#pragma unroll
  for (int j = 0; j < 32; j += 8)
    tile[ty + j][tx] =
        (ty + j < kn && tx < nn) ? B[(long long)(k0 + ty + j) * ldb + (n0 + tx)] : 0.f;
  __syncthreads();
#pragma unroll
  for (int j = 0; j < 32; j += 8)
    if (ty + j < nn && tx < kn) bt[(long long)(n0 + ty + j) * ldw + (k0 + tx)] = tile[tx][ty + j];
}

// The residual x_lo of four raw values.
__device__ __forceinline__ float4 tf32_residual4(float4 x) {
  return make_float4(tf32_trunc(x.x - tf32_trunc(x.x)), tf32_trunc(x.y - tf32_trunc(x.y)),
                     tf32_trunc(x.z - tf32_trunc(x.z)), tf32_trunc(x.w - tf32_trunc(x.w)));
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

// bounded_wait for a barrier that threads of the peer CTA arrive on: the
// polling is CTA-scoped (cheap); once the phase is seen complete, one more
// test of the same phase acquires at cluster scope. The phase cannot move on
// in between: its next completion needs work this thread has not issued yet.
__device__ __forceinline__ bool bounded_wait_cluster(uint32_t bar, uint32_t parity,
                                                     volatile int* abort_w, int* status, int code,
                                                     long long timeout_ns) {
  if (!bounded_wait(bar, parity, abort_w, status, code, timeout_ns)) return false;
  return ptx::mbar_try_wait_cluster(bar, parity);
}

template <int FORM, int BK, int BNT = BN>
__global__ void __launch_bounds__(NT, 1)
    gemm_kernel(const __grid_constant__ Params p, const __grid_constant__ CUtensorMap tmA,
                const __grid_constant__ CUtensorMap tmB) {
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw_addr = ptx::smem_addr(smem_raw);
  unsigned char* base = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  Barriers* bar = reinterpret_cast<Barriers*>(base + kStageRegion);
  float* epi = reinterpret_cast<float*>(base + kStageRegion + BAR_BYTES);
  volatile int* abort_w = &bar->abort;
  const uint32_t base_addr = ptx::smem_addr(base);

  static_assert(FORM == kSingle || FORM == kTwoSmPair, "form");
  constexpr bool TWO_SM = FORM == kTwoSmPair;
  constexpr int CL = TWO_SM ? 2 : 1;                // CTAs per cluster
  constexpr int CG = TWO_SM ? 2 : 1;                // cta_group of every tcgen05 instruction
  static_assert(BNT == BN || (!TWO_SM && BNT % 16 == 0 && BNT >= 32), "tile width");
  // narrow tiles keep A's two TF32 parts in tensor memory (the MMAs read A
  // from there, B from shared memory): a stage then holds a third less, so
  // more stages fit, and the A residual never passes through shared memory
  constexpr bool A_TM = !TWO_SM && BNT != BN;
  static_assert(!A_TM || BK == 32, "A in tensor memory: 32-wide slices");
  using S = Slice<BK, TWO_SM ? 2 : 1, BNT, A_TM>;
  constexpr int ACC_COLS = BNT;
  constexpr int A_TCOL0 = NBUF * BNT;  // A slots after the accumulators: [hi | lo] per stage
  constexpr int A_TCOLS = 2 * BK;
  constexpr int TMEM_COLS = A_TM ? 512 : tmem_cols(BNT);
  static_assert(!A_TM || A_TCOL0 + S::ST * A_TCOLS <= TMEM_COLS, "tensor memory columns");
  constexpr int B_OFF = S::B_OFF;
  constexpr uint32_t IDESC = tc::idesc_tf32(BM, BNT);
  constexpr int ST = S::ST, ROW_BYTES = S::ROW_BYTES;
  constexpr int A_BYTES = S::A_BYTES, B_BYTES = S::B_BYTES, STAGE_BYTES = S::STAGE_BYTES;
  constexpr uint16_t kPair = 0x3;  // both CTAs of a cluster of two
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const Schedule& sc = p.sched;
  // the schedule hands out work per cluster; rank r takes tile row CL * i + r
  const int rank = CL == 2 ? (int)ptx::cluster_ctarank() : 0;
  const int b = blockIdx.x / CL;
  const int slot = b * CL + rank;  // this CTA's partial tile and flag
  const int npieces = num_pieces(sc, b);

  if (tid == 0) {
    // two-SM form: the even CTA's MMA thread waits on its own conv barrier
    // (its converter warps, plus one relayed arrival for the odd CTA's) and
    // tmem_empty barriers (the epilogue warps of both CTAs), and its commits
    // arrive on the empty and tmem_full barriers of both
    for (int s = 0; s < ST; ++s) {
      ptx::mbar_init(ptx::smem_addr(&bar->full[s]), 1);
      ptx::mbar_init(ptx::smem_addr(&bar->conv[s]),
                     CONV_THREADS / 32 + ((TWO_SM && rank == 0) ? 1 : 0));
      ptx::mbar_init(ptx::smem_addr(&bar->empty[s]), 1);
    }
    for (int i = 0; i < NBUF; ++i) {
      ptx::mbar_init(ptx::smem_addr(&bar->tmem_full[i]), 1);
      ptx::mbar_init(ptx::smem_addr(&bar->tmem_empty[i]), (TWO_SM ? 2 : 1) * 4);
    }
    ptx::mbar_init(ptx::smem_addr(&bar->drain), 1);
    ptx::mbar_init(ptx::smem_addr(&bar->epi_sync), EPI_THREADS);
    bar->abort = 0;
    ptx::mbar_fence_init();
    ptx::tma_prefetch_desc(&tmA);
    ptx::tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tc::tmem_alloc<CG>(ptx::smem_addr(&bar->tmem_addr), TMEM_COLS);
    tc::tmem_relinquish<CG>();
  }
  tc::fence_before_sync();
  __syncthreads();
  // the peer's barriers must be initialised before the pair's first remote
  // arrival or commit reaches them
  if (CL == 2) ptx::cluster_sync();
  tc::fence_after_sync();
  const uint32_t tmem = bar->tmem_addr;
  if (TWO_SM && tid == 0) {
    // the MMAs of the pair write the same TMEM address in both CTAs
    const uint32_t peer = ptx::ld_shared_cluster(
        ptx::mapa(ptx::smem_addr(&bar->tmem_addr), (uint32_t)(rank ^ 1)));
    if (peer != tmem) {
      *abort_w = 1;
      atomicCAS(p.status, 0, (int)kDevTmemMismatch);
    }
  }
  if (TWO_SM) __syncthreads();  // every role sees the abort word
  // Launched with programmatic stream serialization after the B^T pre-pass:
  // the set-up above (barriers, TMEM, the cluster rendezvous) overlaps its
  // end; nothing below touches global memory before it has completed. The
  // next call's pre-pass may then launch (it waits for this grid in turn).
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();

  if (warp == 0) {
    // ---- TMA producer: the raw A and B^T tiles of every k-slice of every piece
    if (lane == 0) {
      int it = 0;
      for (int i = 0; i < npieces && !*abort_w; ++i) {
        const Piece pc = get_piece(sc, b, i);
        int tm, tn;
        tile_coords(sc, pc.tile, tm, tn);
        tm = tm * CL + rank;
        bool ok = true;
        for (int kb = pc.kb; kb < pc.ke; ++kb, ++it) {
          const int s = it % ST;
          const uint32_t par = (uint32_t)((it / ST) & 1) ^ 1u;
          if (!bounded_wait(ptx::smem_addr(&bar->empty[s]), par, abort_w, p.status,
                            kDevTimeoutEmpty, p.timeout_ns)) {
            ok = false;
            break;
          }
          const uint32_t fb = ptx::smem_addr(&bar->full[s]);
          const uint32_t st0 = base_addr + (uint32_t)(s * STAGE_BYTES);
          ptx::mbar_arrive_expect_tx(fb, (uint32_t)(A_BYTES + B_BYTES));
          ptx::tma_load_2d(st0, &tmA, kb * BK, tm * BM, fb);
          if (TWO_SM) {
            // this CTA's half of the B tile (N columns 128 * rank ..), into this CTA
            ptx::tma_load_2d(st0 + B_OFF, &tmB, kb * BK, tn * BN + rank * (BN / 2), fb);
          } else {
            ptx::tma_load_2d(st0 + B_OFF, &tmB, kb * BK, tn * BNT, fb);
          }
        }
        if (!ok) break;
      }
      // nothing may land after the CTA is gone: wait (bounded) for the last
      // stages issued
      const uint64_t t0 = ptx::global_ns();
      for (int j = it - 1; j >= 0 && j >= it - ST; --j) {
        const uint32_t fb = ptx::smem_addr(&bar->full[j % ST]);
        while (!ptx::mbar_try_wait(fb, (uint32_t)((j / ST) & 1)))
          if ((long long)(ptx::global_ns() - t0) > cleanup_bound_ns(p.timeout_ns)) break;
      }
      if (CL == 2) {
        // the even CTA's MMA commits arrive on this CTA's empty barriers: wait
        // (bounded) for its arrivals on the last use of every stage
        for (int j = it; j < it + ST; ++j) {
          const uint32_t eb = ptx::smem_addr(&bar->empty[j % ST]);
          while (!ptx::mbar_try_wait(eb, (uint32_t)((j / ST) & 1) ^ 1u))
            if ((long long)(ptx::global_ns() - t0) > cleanup_bound_ns(p.timeout_ns)) break;
        }
      }
    }
  } else if (warp == 1) {
    // ---- two-SM form, odd CTA: relays each stage's conv completion to the
    // even CTA with one remote arrival. (Measured on GB300: one relayed
    // arrival per stage runs 26 % faster at 4096^3 than an arrival from each
    // converter warp of the odd CTA.)
    if (TWO_SM && rank != 0 && lane == 0) {
      int it = 0;
      bool ok = true;
      for (int i = 0; i < npieces && ok && !*abort_w; ++i) {
        const Piece pc = get_piece(sc, b, i);
        for (int kb = pc.kb; kb < pc.ke; ++kb, ++it) {
          const int s = it % ST;
          ok = bounded_wait(ptx::smem_addr(&bar->conv[s]), (uint32_t)((it / ST) & 1), abort_w,
                            p.status, kDevTimeoutFull, p.timeout_ns);
          if (!ok) break;
          ptx::mbar_arrive_remote(ptx::mapa(ptx::smem_addr(&bar->conv[s]), 0u));
        }
      }
    }
    // ---- MMA issuer: piece i accumulates into TMEM columns (i % NBUF) * BNT.
    // In the two-SM form the even CTA issues for the pair.
    if (lane == 0 && (!TWO_SM || rank == 0)) {
      int it = 0;
      bool issued_any = false;
      for (int i = 0; i < npieces && !*abort_w; ++i) {
        const Piece pc = get_piece(sc, b, i);
        const int buf = i % NBUF;
        const uint32_t d = tmem + (uint32_t)(buf * ACC_COLS);
        // the epilogue (of both CTAs, in the two-SM form) must have read this
        // accumulator's previous piece
        const uint32_t eb = ptx::smem_addr(&bar->tmem_empty[buf]);
        const uint32_t epar = (uint32_t)((i / NBUF) & 1) ^ 1u;
        if (!(TWO_SM ? bounded_wait_cluster(eb, epar, abort_w, p.status, kDevTimeoutSync,
                                            p.timeout_ns)
                     : bounded_wait(eb, epar, abort_w, p.status, kDevTimeoutSync, p.timeout_ns)))
          break;
        tc::fence_after_sync();
        bool ok = true;
        for (int kb = pc.kb; kb < pc.ke; ++kb, ++it) {
          const int s = it % ST;
          const uint32_t par = (uint32_t)((it / ST) & 1);
          // the raw tiles (TMA) and the residual tiles (converter warps). In
          // the two-SM form this CTA's conv barrier completes once the
          // converters of both CTAs are done, each only after its own CTA's
          // raw tiles landed.
          const bool ready =
              TWO_SM ? bounded_wait_cluster(ptx::smem_addr(&bar->conv[s]), par, abort_w, p.status,
                                            kDevTimeoutFull, p.timeout_ns)
                     : (bounded_wait(ptx::smem_addr(&bar->full[s]), par, abort_w, p.status,
                                     kDevTimeoutFull, p.timeout_ns) &&
                        bounded_wait(ptx::smem_addr(&bar->conv[s]), par, abort_w, p.status,
                                     kDevTimeoutFull, p.timeout_ns));
          if (!ready) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t st0 = base_addr + (uint32_t)(s * STAGE_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / 8; ++kk) {
            const uint32_t koff = (uint32_t)(kk * 32);  // 8 TF32 values = 32 bytes
            const uint64_t b_hi = tc::smem_desc_k_swizzled<ROW_BYTES>(st0 + B_OFF + koff);
            const uint64_t b_lo = tc::smem_desc_k_swizzled<ROW_BYTES>(st0 + B_OFF + B_BYTES + koff);
            const uint32_t first = (kb == pc.kb && kk == 0) ? 0u : 1u;
            if (A_TM) {
              // A's parts in the stage's tensor-memory slot: 8 columns per 8 values of K
              const uint32_t a_hi = tmem + (uint32_t)(A_TCOL0 + s * A_TCOLS + kk * 8);
              tc::mma_tf32_ts(d, a_hi, b_hi, IDESC, first);
              tc::mma_tf32_ts(d, a_hi, b_lo, IDESC, 1u);
              tc::mma_tf32_ts(d, a_hi + (uint32_t)BK, b_hi, IDESC, 1u);
              continue;
            }
            const uint64_t a_hi = tc::smem_desc_k_swizzled<ROW_BYTES>(st0 + koff);
            const uint64_t a_lo = tc::smem_desc_k_swizzled<ROW_BYTES>(st0 + A_BYTES + koff);
            if (TWO_SM) {
              tc::mma_tf32_pair(d, a_hi, b_hi, IDESC_PAIR, first);
              tc::mma_tf32_pair(d, a_hi, b_lo, IDESC_PAIR, 1u);
              tc::mma_tf32_pair(d, a_lo, b_hi, IDESC_PAIR, 1u);
            } else {
              tc::mma_tf32(d, a_hi, b_hi, IDESC, first);
              tc::mma_tf32(d, a_hi, b_lo, IDESC, 1u);
              tc::mma_tf32(d, a_lo, b_hi, IDESC, 1u);
            }
          }
          issued_any = true;
          // frees the stage (in both CTAs of a pair) once these MMAs are done
          if (TWO_SM)
            tc::commit_pair_multicast(ptx::smem_addr(&bar->empty[s]), kPair);
          else
            tc::commit(ptx::smem_addr(&bar->empty[s]));
        }
        if (!ok) break;
        // the piece's accumulator is ready (in both CTAs, in the two-SM form)
        if (TWO_SM)
          tc::commit_pair_multicast(ptx::smem_addr(&bar->tmem_full[buf]), kPair);
        else
          tc::commit(ptx::smem_addr(&bar->tmem_full[buf]));
      }
      if (*abort_w && issued_any) {
        // wait (bounded) until every MMA issued has completed
        if (TWO_SM)
          tc::commit_pair(ptx::smem_addr(&bar->drain));
        else
          tc::commit(ptx::smem_addr(&bar->drain));
        const uint64_t t0 = ptx::global_ns();
        while (!ptx::mbar_try_wait(ptx::smem_addr(&bar->drain), 0u))
          if ((long long)(ptx::global_ns() - t0) > cleanup_bound_ns(p.timeout_ns)) break;
      }
    }
  } else if (warp >= CONV_WARP0) {
    // ---- converter warps 6-9: x_lo = trunc(x - trunc(x)) of every raw value of
    // a stage, written at the same offset in the stage's _lo tile (the tiles
    // have one shape and swizzle, so a value keeps its position) -------------
    const int ct = tid - CONV_WARP0 * 32;
    int it = 0;
    bool ok = true;
    for (int i = 0; i < npieces && ok && !*abort_w; ++i) {
      const Piece pc = get_piece(sc, b, i);
      for (int kb = pc.kb; kb < pc.ke; ++kb, ++it) {
        const int s = it % ST;
        ok = bounded_wait(ptx::smem_addr(&bar->full[s]), (uint32_t)((it / ST) & 1), abort_w,
                          p.status, kDevTimeoutFull, p.timeout_ns);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        unsigned char* st = base + s * STAGE_BYTES;
        const float4* a_raw = reinterpret_cast<const float4*>(st);
        const float4* b_raw = reinterpret_cast<const float4*>(st + B_OFF);
        float4* b_lo = reinterpret_cast<float4*>(st + B_OFF + B_BYTES);
        if (A_TM) {
          // this thread's row of the A tile (the warp may reach TMEM lanes
          // 32 * (warp % 4) ..): its 32 raw values into the stage's hi
          // columns, their residuals into the lo columns. The 16-byte chunks
          // of a row sit at the 128-byte swizzle's positions.
          const int r = (warp & 3) * 32 + lane;
          uint32_t hi[32], lo[32];
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const float4 v = a_raw[r * 8 + (c ^ (r & 7))];
            const float4 l = tf32_residual4(v);
            hi[4 * c] = __float_as_uint(v.x);
            hi[4 * c + 1] = __float_as_uint(v.y);
            hi[4 * c + 2] = __float_as_uint(v.z);
            hi[4 * c + 3] = __float_as_uint(v.w);
            lo[4 * c] = __float_as_uint(l.x);
            lo[4 * c + 1] = __float_as_uint(l.y);
            lo[4 * c + 2] = __float_as_uint(l.z);
            lo[4 * c + 3] = __float_as_uint(l.w);
          }
          // the MMAs that read this slot last have completed (they freed the
          // stage before its raw tiles were loaded again)
          tc::fence_after_sync();
          const uint32_t slot_t =
              tmem + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)(A_TCOL0 + s * A_TCOLS);
          tc::tmem_st32(slot_t, hi);
          tc::tmem_st32(slot_t + (uint32_t)BK, lo);
        } else {
          float4* a_lo = reinterpret_cast<float4*>(st + A_BYTES);
#pragma unroll
          for (int q = ct; q < A_BYTES / 16; q += CONV_THREADS) a_lo[q] = tf32_residual4(a_raw[q]);
        }
#pragma unroll
        for (int q = ct; q < B_BYTES / 16; q += CONV_THREADS) b_lo[q] = tf32_residual4(b_raw[q]);
        // the MMAs read these tiles through the async proxy
        ptx::fence_proxy_async_shared();
        if (A_TM) {
          tc::tmem_wait_st();
          tc::fence_before_sync();
        }
        __syncwarp();
        if (lane == 0) {
          ptx::mbar_arrive(ptx::smem_addr(&bar->conv[s]));
        }
      }
    }
  } else {
    // ---- epilogue warps 2-5: TMEM -> registers -> C, or -> a partial tile ----
    const int quarter = warp & 3;                 // TMEM lanes 32*quarter .. +31
    const int r = quarter * 32 + lane;            // this thread's row of the tile
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const bool vec = ((reinterpret_cast<uintptr_t>(p.C) & 15u) == 0) && ((p.ldc & 3) == 0);
    uint32_t sync_phase = 0;
    auto epi_sync = [&]() -> bool {  // bounded rendezvous of the 128 epilogue threads
      ptx::mbar_arrive(ptx::smem_addr(&bar->epi_sync));
      const bool ok = bounded_wait(ptx::smem_addr(&bar->epi_sync), sync_phase, abort_w, p.status,
                                   kDevTimeoutSync, p.timeout_ns);
      sync_phase ^= 1u;
      return __all_sync(0xffffffffu, ok);
    };
    for (int i = 0; i < npieces && !*abort_w; ++i) {
      const Piece pc = get_piece(sc, b, i);
      const int buf = i % NBUF;
      const uint32_t acc = tmem + (uint32_t)(buf * ACC_COLS) + lane_base;
      const bool ok = bounded_wait(ptx::smem_addr(&bar->tmem_full[buf]), (uint32_t)((i / NBUF) & 1),
                                   abort_w, p.status, kDevTimeoutFull, p.timeout_ns);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc::fence_after_sync();
      float* my_ws = p.ws + (long long)slot * (BM * BNT);
      if (is_partial_piece(sc, pc)) {
        // publish the partial tile (column-major: a warp writes 128 bytes
        // per column)
#pragma unroll 1
        for (int c0 = 0; c0 < BNT; c0 += 16) {
          uint32_t v[16];
          tc::tmem_ld16(acc + (uint32_t)c0, v);
          tc::tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e) __stcg(my_ws + (c0 + e) * BM + r, __uint_as_float(v[e]));
        }
        if (!epi_sync()) break;
        if (warp == 2 && lane == 0) {
          __threadfence();
          ptx::st_release(p.flags + slot, p.epoch);
        }
      } else {
        const int nc = num_contributors(sc, b, pc);
        if (nc > 0) {
          if (warp == 2 && lane == 0) {
            for (int c = 1; c <= nc && !*abort_w; ++c) {
              uint32_t* f = p.flags + (b + c) * CL + rank;
              const uint64_t t0 = ptx::global_ns();
              while (ptx::ld_acquire(f) != p.epoch) {
                if ((long long)(ptx::global_ns() - t0) > p.timeout_ns) {
                  *abort_w = 1;
                  atomicCAS(p.status, 0, (int)kDevTimeoutFlag);
                  break;
                }
                __nanosleep(200);
              }
              // consumed: a later launch (or graph replay, which reuses this
              // epoch) never mistakes it for its own
              if (!*abort_w) *f = 0u;
            }
          }
          if (!epi_sync() || *abort_w) break;
        }
        int tm, tn;
        tile_coords(sc, pc.tile, tm, tn);
        tm = tm * CL + rank;
        // 32 columns at a time: lane = row while reading TMEM and the
        // (column-major) partials, then through the warp's staging block so
        // that the C accesses are row segments of 128 bytes: 8 lanes per row,
        // 4 rows per access, 8 accesses for the warp's 32 rows
        float* stage = epi + quarter * EPI_WARP_FLOATS;
        const int sub_r = lane >> 3, sub_c = (lane & 7) * 4;
#pragma unroll 1
        for (int c0 = 0; c0 < BNT; c0 += 32) {
          uint32_t v[32];
          tc::tmem_ld16(acc + (uint32_t)c0, *reinterpret_cast<uint32_t(*)[16]>(&v[0]));
          tc::tmem_ld16(acc + (uint32_t)(c0 + 16), *reinterpret_cast<uint32_t(*)[16]>(&v[16]));
          tc::tmem_wait_ld();
          float a[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) a[e] = __uint_as_float(v[e]);
          // partials of schedule units b+1 .. b+nc (same rank), in that order
          for (int c = 1; c <= nc; ++c) {
            const float* src = p.ws + (long long)((b + c) * CL + rank) * (BM * BNT);
#pragma unroll
            for (int e = 0; e < 32; ++e) a[e] += __ldcg(src + (c0 + e) * BM + r);
          }
          __syncwarp();  // the previous block's reads of the staging are done
#pragma unroll
          for (int q = 0; q < 8; ++q)
            *reinterpret_cast<float4*>(stage + lane * EPI_PITCH + q * 4) =
                make_float4(a[q * 4], a[q * 4 + 1], a[q * 4 + 2], a[q * 4 + 3]);
          __syncwarp();
          const int col = tn * BNT + c0 + sub_c;
          const int row0 = tm * BM + quarter * 32 + sub_r;  // + 4 g for access g
          const bool full = vec && col + 3 < p.N;
          // every read of C is issued before any write, so the reads overlap
          float4 old[8];
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            old[g] = make_float4(0.f, 0.f, 0.f, 0.f);
            const int row = row0 + 4 * g;
            if (p.beta == 0.f || row >= p.M) continue;
            const float* cp = p.C + (long long)row * p.ldc + col;
            if (full) {
              old[g] = *reinterpret_cast<const float4*>(cp);
            } else {
              if (col + 0 < p.N) old[g].x = cp[0];
              if (col + 1 < p.N) old[g].y = cp[1];
              if (col + 2 < p.N) old[g].z = cp[2];
              if (col + 3 < p.N) old[g].w = cp[3];
            }
          }
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            const int row = row0 + 4 * g;
            if (row >= p.M) continue;
            const float4 t =
                *reinterpret_cast<const float4*>(stage + (sub_r + 4 * g) * EPI_PITCH + sub_c);
            float4 w4 = make_float4(p.alpha * t.x, p.alpha * t.y, p.alpha * t.z, p.alpha * t.w);
            if (p.beta != 0.f) {
              w4.x = fmaf(p.beta, old[g].x, w4.x);
              w4.y = fmaf(p.beta, old[g].y, w4.y);
              w4.z = fmaf(p.beta, old[g].z, w4.z);
              w4.w = fmaf(p.beta, old[g].w, w4.w);
            }
            float* cp = p.C + (long long)row * p.ldc + col;
            if (full) {
              *reinterpret_cast<float4*>(cp) = w4;
            } else {
              if (col + 0 < p.N) cp[0] = w4.x;
              if (col + 1 < p.N) cp[1] = w4.y;
              if (col + 2 < p.N) cp[2] = w4.z;
              if (col + 3 < p.N) cp[3] = w4.w;
            }
          }
        }
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        // the even CTA's MMA thread waits for both CTAs' epilogues
        if (TWO_SM && rank != 0)
          ptx::mbar_arrive_remote(ptx::mapa(ptx::smem_addr(&bar->tmem_empty[buf]), 0u));
        else
          ptx::mbar_arrive(ptx::smem_addr(&bar->tmem_empty[buf]));
      }
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (TWO_SM) {
    // the even CTA's MMAs write the odd CTA's TMEM and read its shared
    // memory: the pair frees its TMEM together, once both are done
    ptx::cluster_sync();
    if (warp == 1) {
      tc::fence_after_sync();
      tc::tmem_dealloc<CG>(tmem, TMEM_COLS);
    }
  } else {
    if (warp == 1) {
      tc::fence_after_sync();
      tc::tmem_dealloc(tmem, TMEM_COLS);
    }
  }
}

// Per-device set-up (shared-memory attributes, how many CTA pairs can be
// resident at once), guarded by g_mutex.
std::mutex g_mutex;
bool g_ready[64];
int g_pairs[64];          // resident clusters of two; 0 = the pair form cannot run
// the requested Form; the pair form runs where possible
std::atomic<int> g_form{kTwoSmPair};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
bool g_encode_tried = false;

// The launch plan of sgemm_3xtf32 (host arithmetic only): the kernel form
// that runs, the k-slice width and the persistent schedule. `want` is the
// requested form, `pairs` how many CTA pairs the device keeps resident (0:
// none), `sms` the SM count.
struct Plan {
  int form, bk, kiters, bn;
  Schedule sched;
};
Plan make_plan(int M, int N, int K, int want, int pairs, int sms) {
  Plan pl{};
  pl.form = (want != kSingle && pairs > 0) ? want : (int)kSingle;
  // The tile's width in N. Narrow tiles run on single CTAs with A's parts in
  // tensor memory; per stage they issue as many MMAs as the wide tile for a
  // quarter (64) or half (128) of its work, and with few tiles the schedule
  // splits each tile along K over many CTAs, whose partial tiles one CTA then
  // adds up. Measured on GB300 (us; 64 / 128 / 256 wide):
  //   * N <= 64: 64 wide, so that the MMAs compute no columns beyond N
  //     (16384 x 64 x 4096: 81 against 149 with 256-wide tiles);
  //   * few 128-wide tiles for the K they have -- (sms / tiles)^2 > kiters / 2
  //     with kiters 32-wide slices, the fix-up's partial tiles per tile
  //     (sms / tiles) against the main loop's slices per CTA (tiles x kiters
  //     / sms): 64 wide, as more, smaller tiles keep the fix-up short:
  //     512^3 17.6 / 23.9, 300 x 520 x 4096 33.0 / 40.3; but 512 x 512 x 8192
  //     53.5 / 48.9;
  //   * otherwise 128 wide for N <= 128 (16384 x 128 x 4096: 88.5 against
  //     140; 8192 x 96 x 4096: 57.3 against 90.2) and, below two waves of
  //     256-wide tiles (where the wide schedule splits most of them), while
  //     their work is at most 48 slices of 32 per CTA: 1024^3 30.4 / 26.8, 1024 x
  //     1024 x 2048 47.1 / 36.2, 1024 x 1024 x 4096 - / 55.3 / 64.1, 2048 x
  //     1024 x 1024 - / 33.3 / 41.1, 8191 x 1000 x 777 - / 98.5 / 105.7;
  //   * beyond that 256 wide: 2048^3 (54 slices per CTA) 84.9 against 79.6,
  //     1024 x 1024 x 16384 (108) 181.0 against 172.4.
  const long long kiters32 = ceil_div_nn(K, 32);
  const long long tiles_mid = (long long)ceil_div_nn(M, BM) * ceil_div_nn(N, BN_MID);
  const long long wide_tiles = (long long)ceil_div_nn(M, BM) * ceil_div_nn(N, BN);
  // (the products are formed only below these bounds, so they cannot overflow)
  const bool few_mid_tiles =
      tiles_mid < 2LL * sms && 2LL * sms * sms > kiters32 * tiles_mid * tiles_mid;
  constexpr long long kMidMaxSlicesPerCta = 48;
  const bool little_wide_work =
      wide_tiles < 2LL * sms && wide_tiles * kiters32 <= kMidMaxSlicesPerCta * sms;
  if (N <= BN_NARROW || few_mid_tiles)
    pl.bn = BN_NARROW;
  else if (N <= BN_MID || little_wide_work)
    pl.bn = BN_MID;
  else
    pl.bn = BN;
  if (pl.bn != BN) pl.form = kSingle;
  // schedule: whole tiles, then the last one to two waves split along K. In
  // the pair form a schedule unit is two vertically adjacent tiles (a tile
  // row pair), handed to one cluster.
  const int tiles_m = ceil_div_nn(M, BM), tiles_n = ceil_div_nn(N, pl.bn);
  // the k-slice width (see Slice). The two-SM form always takes 32: its
  // stages halve the per-stage hand-offs between the CTAs of a pair
  // (measured at 4096^3: 265 against 158 TFLOP/s with 16).
  // Narrow tiles also take 32: their stages carry a quarter or half of the
  // MMA work, so the per-stage hand-offs dominate (measured at 16384 x 64 x
  // 4096: 89.7 against 106.8 us with 16-wide slices)
  auto slice_width = [K, &pl](int f) {
    return (f == kTwoSmPair || K < 1024 || pl.bn != BN) ? 32 : 16;
  };
  pl.bk = slice_width(pl.form);
  pl.kiters = ceil_div_nn(K, pl.bk);
  if (pl.form != kSingle) {
    // groups of 8 tile-row pairs in the raster (measured at 8192^3: 309 against
    // 305 TFLOP/s with 4, 298 with 2; 16 the same as 8)
    // whole pair tiles, then, with at least two waves of them, a K split of
    // the last wave when it is at least a quarter full, else of the last two
    // (below two waves the two-wave split leaves no whole tiles, and single
    // CTAs run: 3072 x 2048 x 1536 190 TFLOP/s against 174 for pairs with
    // only the last wave split). Measured at 4096^3, 3.37 waves:
    // 284.8 against 273.3 TFLOP/s; 5120^3: 305.3 against 297.9; 8192^3, 13.5
    // waves: 323.3 against 319.7; 6144 x 4096 x 4096, 5.05 waves: splitting
    // only the last 0.05 of a wave lost 8 %)
    const long long units = (long long)((tiles_m + 1) / 2) * tiles_n;
    const bool full_tail = pairs > 0 && units >= 2LL * pairs && (units % pairs) * 4 >= pairs;
    pl.sched = make_schedule((tiles_m + 1) / 2, tiles_n, pl.kiters, pairs,
                             SchedPolicy{full_tail ? kSchedHybridTail : kSchedHybrid, 8,
                                         64 / pl.bk, 1});
    // every tile split along K: the pairs' lockstep costs more than they save
    // (measured at 1024^3, 1024 x 1024 x 16384 and 16384 x 64 x 4096; the
    // two-SM form gained 4 % at 2048^3 only)
    if (pl.sched.dp_tiles == 0) pl.form = kSingle;
  }
  if (pl.form == kSingle) {
    pl.bk = slice_width(pl.form);
    pl.kiters = ceil_div_nn(K, pl.bk);
    // at least 64 of K per CTA in a split
    pl.sched = make_schedule(tiles_m, tiles_n, pl.kiters, sms,
                             SchedPolicy{kSchedHybrid, 8, 64 / pl.bk, 1});
  }
  return pl;
}

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
                    int rows, int K, long long ldw, int box_rows, int bk) {
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ldw * 4};
  cuuint32_t box[2] = {(cuuint32_t)bk, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             bk == 32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
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
      (reads_ab &&
       ((reinterpret_cast<uintptr_t>(A) & 3u) || (reinterpret_cast<uintptr_t>(B) & 3u))))
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
  // the schedule numbers tiles with 32-bit integers (the same limit as sgemm())
  if ((long long)ceil_div_nn(M, x3::BM) * ceil_div_nn(N, x3::BN) > 0x7fffffffLL)
    return SGEMM_ERR_INVALID_DIM;

  int pairs = 0;
  {
    std::lock_guard<std::mutex> lock(x3::g_mutex);
    if (dev < 0 || dev >= 64) return SGEMM_ERR_UNSUPPORTED_DEVICE;
    if (!x3::g_ready[dev]) {
      const auto attr = cudaFuncAttributeMaxDynamicSharedMemorySize;
      using namespace x3;
      if (cudaFuncSetAttribute(gemm_kernel<kSingle, 16>, attr, SMEM_BYTES) != cudaSuccess ||
          cudaFuncSetAttribute(gemm_kernel<kSingle, 32>, attr, SMEM_BYTES) != cudaSuccess ||
          cudaFuncSetAttribute(gemm_kernel<kSingle, 32, BN_NARROW>, attr, SMEM_BYTES) !=
              cudaSuccess ||
          cudaFuncSetAttribute(gemm_kernel<kSingle, 32, BN_MID>, attr, SMEM_BYTES) != cudaSuccess ||
          cudaFuncSetAttribute(gemm_kernel<kTwoSmPair, 32>, attr, SMEM_BYTES) != cudaSuccess) {
        cudaGetLastError();
        return SGEMM_ERR_LAUNCH;
      }
      // how many clusters of two fit at once (SMs pair up within a GPC, so
      // this can be below sms / 2)
      cudaLaunchConfig_t qc = {};
      cudaLaunchAttribute qa[1];
      qa[0].id = cudaLaunchAttributeClusterDimension;
      qa[0].val.clusterDim.x = 2;
      qa[0].val.clusterDim.y = 1;
      qa[0].val.clusterDim.z = 1;
      qc.gridDim = dim3(2 * (unsigned)(sms / 2 > 0 ? sms / 2 : 1));
      qc.blockDim = dim3(x3::NT);
      qc.dynamicSmemBytes = x3::SMEM_BYTES;
      qc.attrs = qa;
      qc.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, gemm_kernel<kTwoSmPair, 32>, &qc) != cudaSuccess) {
        cudaGetLastError();
        n = 0;
      }
      x3::g_pairs[dev] = n;
      x3::g_ready[dev] = true;
    }
    pairs = x3::g_pairs[dev];
  }
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  {
    std::lock_guard<std::mutex> lock(x3::g_mutex);
    enc = x3::encoder();
  }
  if (enc == nullptr) return SGEMM_ERR_LAUNCH;

  const x3::Plan plan = x3::make_plan(M, N, K, x3::g_form.load(), pairs, sms);
  const int form = plan.form, bk = plan.bk, kiters = plan.kiters, bn = plan.bn;
  const Schedule& sched = plan.sched;
  const int CL = form == x3::kSingle ? 1 : 2;
  const bool split = sched.dp_tiles < sched.tiles;
  const int ctas = sched.grid * CL;

  // workspace: B^T (N x Kp), a copy of A (M x Kp) only when A's rows are not
  // 16-byte aligned, then one partial tile per CTA when the schedule splits
  const long long Kp = ((long long)K + 3) / 4 * 4;
  const bool a_direct = ((reinterpret_cast<uintptr_t>(A) & 15u) == 0) && ((lda & 3) == 0);
  const size_t bt_floats = (size_t)N * Kp;
  const size_t a_floats = a_direct ? 0 : (size_t)M * Kp;
  const size_t partial_floats = split ? (size_t)ctas * x3::BM * bn : 0;
  float* ws = nullptr;
  int* status = nullptr;
  uint32_t* flags = nullptr;
  uint32_t epoch = 0;
  st = library_workspace(dev, stream, bt_floats + a_floats + partial_floats, (size_t)ctas, &ws,
                         &status, &flags, &epoch);
  if (st != SGEMM_OK) return st;
  float* bt = ws;
  float* a_copy = bt + bt_floats;
  float* partials = a_copy + a_floats;

  // 1. B^T (and, when needed, an aligned copy of A)
  {
    constexpr long long kRowsPerGrid = 65535LL * 32;  // tile rows of one grid (gridDim.y)
    for (long long kb = 0; kb < K; kb += kRowsPerGrid) {
      const int ktiles = ceil_div_nn((int)(K - kb < kRowsPerGrid ? K - kb : kRowsPerGrid), 32);
      // programmatic dependent launch: the grid waits for the kernel ahead of
      // it (the previous call's GEMM reads this workspace) before any access
      cudaLaunchConfig_t tc = {};
      cudaLaunchAttribute ta[1];
      ta[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      ta[0].val.programmaticStreamSerializationAllowed = 1;
      tc.gridDim = dim3((unsigned)ceil_div_nn(N, 32), (unsigned)ktiles);
      tc.blockDim = dim3(32, 8);
      tc.stream = stream;
      tc.attrs = ta;
      tc.numAttrs = 1;
      if (cudaLaunchKernelEx(&tc, x3::transpose_b_kernel, K, N, B, (long long)ldb, bt, Kp,
                             (int)kb) != cudaSuccess) {
        cudaGetLastError();
        return SGEMM_ERR_LAUNCH;
      }
    }
    if (!a_direct) {
      const int bx = (K + 255) / 256 < 8 ? (K + 255) / 256 : 8;
      const int by = M < 65535 ? M : 65535;
      x3::pack_a_kernel<<<dim3(bx, by), 256, 0, stream>>>(M, K, A, lda, a_copy, Kp);
    }
    if (cudaGetLastError() != cudaSuccess) return SGEMM_ERR_LAUNCH;
  }

  // 2. tensor-core GEMM on the raw tiles
  CUtensorMap mA, mB;
  if (!x3::encode_k_major(enc, &mA, a_direct ? A : a_copy, M, K, a_direct ? (long long)lda : Kp,
                          x3::BM, bk) ||
      !x3::encode_k_major(enc, &mB, bt, N, K, Kp, bn / CL, bk))
    return SGEMM_ERR_LAUNCH;
  x3::Params p;
  p.M = M;
  p.N = N;
  p.K = K;
  p.alpha = alpha;
  p.beta = beta;
  p.C = C;
  p.ldc = ldc;
  p.sched = sched;
  p.ws = partials;
  p.flags = flags;
  p.epoch = epoch;
  p.status = status;
  p.timeout_ns = library_wait_timeout_ns();
  {
    // programmatic stream serialization (the kernel waits for the pre-pass
    // before any global access), and clusters of two for the pair form
    cudaLaunchConfig_t lc = {};
    cudaLaunchAttribute la[2];
    la[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    la[0].val.programmaticStreamSerializationAllowed = 1;
    la[1].id = cudaLaunchAttributeClusterDimension;
    la[1].val.clusterDim.x = 2;
    la[1].val.clusterDim.y = 1;
    la[1].val.clusterDim.z = 1;
    lc.gridDim = dim3((unsigned)ctas);
    lc.blockDim = dim3(x3::NT);
    lc.dynamicSmemBytes = x3::SMEM_BYTES;
    lc.stream = stream;
    lc.attrs = la;
    lc.numAttrs = CL == 2 ? 2 : 1;
    using x3::BN_MID;
    using x3::BN_NARROW;
    cudaError_t e;
    if (CL == 2)  // the two-SM form always runs 32-wide slices (make_plan)
      e = cudaLaunchKernelEx(&lc, x3::gemm_kernel<x3::kTwoSmPair, 32>, p, mA, mB);
    else if (bn == BN_NARROW)  // narrow tiles always run 32-wide slices (make_plan)
      e = cudaLaunchKernelEx(&lc, x3::gemm_kernel<x3::kSingle, 32, BN_NARROW>, p, mA, mB);
    else if (bn == BN_MID)
      e = cudaLaunchKernelEx(&lc, x3::gemm_kernel<x3::kSingle, 32, BN_MID>, p, mA, mB);
    else if (bk == 16)
      e = cudaLaunchKernelEx(&lc, x3::gemm_kernel<x3::kSingle, 16>, p, mA, mB);
    else
      e = cudaLaunchKernelEx(&lc, x3::gemm_kernel<x3::kSingle, 32>, p, mA, mB);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return SGEMM_ERR_LAUNCH;
    }
  }
  char text[160];
  snprintf(text, sizeof(text),
           "3xtf32_tcgen05_%dx%dx%d_s%d cluster=%d%s grid=%d units=%d dp=%d split=%d kiters=%d%s",
           x3::BM, bn, bk, x3::stages_of(form, bk, bn), CL,
           form == x3::kTwoSmPair ? " pair=2sm" : "",
           ctas, sched.grid, sched.dp_tiles,
           sched.tiles - sched.dp_tiles, kiters, a_direct ? "" : " a=copied");
  note_last_config(text);
  return SGEMM_OK;
}

SGEMM_API int sgemm_3xtf32_plan(int M, int N, int K, int form, int pairs, int sms, int* out) {
  if (M < 1 || N < 1 || K < 1) return SGEMM_ERR_INVALID_DIM;
  if ((form != SGEMM_X3_SINGLE && form != SGEMM_X3_PAIR) || pairs < 0 || sms < 1 ||
      out == nullptr)
    return SGEMM_ERR_INVALID_VALUE;
  if ((long long)ceil_div_nn(M, x3::BM) * ceil_div_nn(N, x3::BN) > 0x7fffffffLL)
    return SGEMM_ERR_INVALID_DIM;
  const x3::Plan pl = x3::make_plan(M, N, K, form, pairs, sms);
  out[0] = pl.form;
  out[1] = pl.bk;
  out[2] = x3::stages_of(pl.form, pl.bk, pl.bn);             // stages
  out[3] = pl.sched.grid * (pl.form == x3::kSingle ? 1 : 2);  // CTAs
  out[4] = pl.sched.grid;                                    // schedule units
  out[5] = pl.sched.dp_tiles;
  out[6] = pl.sched.tiles - pl.sched.dp_tiles;
  out[7] = pl.kiters;
  out[8] = pl.bn;
  return SGEMM_OK;
}

SGEMM_API int sgemm_3xtf32_set_kernel_form(int form) {
  if (form != SGEMM_X3_SINGLE && form != SGEMM_X3_PAIR) return SGEMM_ERR_INVALID_VALUE;
  return x3::g_form.exchange(form);
}
