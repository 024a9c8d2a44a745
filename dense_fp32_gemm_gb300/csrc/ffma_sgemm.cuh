// ffma_sgemm.cuh -- the FP32 FFMA SGEMM kernel for sm_103a:
// C = alpha * A * B + beta * C on row-major matrices with arbitrary M, N, K and
// leading dimensions.
//
// What the pages contribute, and what changed for this part:
//   * Shared-memory staging of an A and a B tile per k-slice ("Shared Memory
//     Tiling", kernel listing and "Memory Access Pattern"), here as a ring of
//     STAGES buffers filled asynchronously and handed over by mbarriers instead
//     of two __syncthreads per slice.
//   * A stored transposed, As[k][m], so that a lane's TM values of A for one k
//     are contiguous and come in with 128-bit shared loads ("Vectorized Memory
//     Access: 128-bit Loads and Stores", sections "Why As Has To Be Transposed"
//     and "Mechanics" 1). The transpose still happens on the store side, but
//     the store is a 4-byte cp.async per element (no registers, no wait) and
//     the rows are padded so the scattered stores hit 32 distinct banks -- the
//     page's own "What Could Be Improved" measures 4.2-way conflicts for the
//     unpadded store.
//   * B needs no transpose (same page, "Mechanics" 1); it is one TMA box per
//     k-slice when its pointer and leading dimension allow (16-byte aligned
//     base, ldb*4 a multiple of 16), else 4-byte cp.async.
//   * Block / warp / sub-tile / lane decomposition with WMITER x WNITER
//     interleaved sub-tiles ("Warp Tiling: A Third Level of Tiling", sections
//     "The Warp Tile Is Not Contiguous Either" and "Mechanics" 1-2). Each lane
//     keeps WMITER*TM x WNITER*TN accumulators in registers; the default
//     config uses 16 x 8 = 128 so that one k-step issues 128 FFMA against six
//     128-bit shared loads (the pages' balance argument in "Shared Memory
//     Tiling", "What Could Be Improved": at least four FMA per shared load,
//     counted here per 32-bit word).
//   * Predicated edges: out-of-range A and B elements are zero-filled by the
//     copy engines and out-of-range C elements are skipped, so any M, N, K
//     works (the pages assume divisibility).
//   * A persistent grid driven by schedule.hpp (whole tiles, then k-split
//     tiles with a fixed-order fix-up), so every SM gets the same work.
//   * Epilogue alpha * acc + beta * C with 128-bit read-modify-write where C's
//     alignment allows; C is not read when beta == 0.
//
// Every wait is bounded: a barrier, slot or flag that does not arrive within
// timeout_ns makes the CTA record a status code, drain its own copies in
// flight and return, so a fault can never leave the GPU spinning.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include <utility>

#include "ptx.cuh"
#include "schedule.hpp"
#include "tile_config.hpp"

namespace sgemm_gb300 {

// Device status codes written to KernelParams::status (first error wins).
enum DeviceStatus : int {
  kDevOk = 0,
  kDevTimeoutFull = 1,    // operand tile never landed
  kDevTimeoutEmpty = 2,   // a slot was never released by its consumers
  kDevTimeoutFlag = 3,    // a split partial was never published
  kDevTimeoutSync = 4,    // a CTA-wide rendezvous did not complete
  kDevTmemMismatch = 5,   // the two CTAs of a two-SM pair got different TMEM columns
};

struct KernelParams {
  int M, N, K;
  float alpha, beta;
  const float* A;
  long long lda;
  const float* B;
  long long ldb;
  float* C;
  long long ldc;
  long long sA, sB, sC; // elements between consecutive matrices of a batch
  Schedule sched;
  float* ws;            // grid * BM * BN floats: one partial tile per CTA
  uint32_t* flags;      // grid flags: flags[b] == epoch once slot b is written; the
                        // owner of the tile resets it to 0 after reading the slot
  int* status;          // device status word
  uint32_t epoch;       // value of a flag published by this launch
  int c_vec;            // C is 16-byte aligned and ldc % 4 == 0
  long long timeout_ns; // bound on every wait
};

// How each operand tile reaches shared memory (template parameters AL, BL):
//   A: kARow   A stored M x K (op N): transposing 4-byte cp.async into As[k][m]
//      kATTma  A stored K x M (op T): one 3-D TMA box, As[k][m] needs no transpose
//      kATCp   A stored K x M (op T): plain 4-byte cp.async (A not TMA-aligned)
//      kARowStg A stored M x K (op N), TMA-aligned: one 3-D TMA box per k-slice
//              into a staging slot as stored, transposed into As[k][m] by an
//              extra producer warp (with B by TMA only; tile_config.hpp,
//              stg_eligible); the FMA warps then issue no copies at all
//   B: kBRowTma B stored K x N (op N): one 3-D TMA box into Bs[k][n]
//      kBRowCp  B stored K x N (op N): plain 4-byte cp.async
//      kBT      B stored N x K (op T): transposing 4-byte cp.async into Bs[k][n]
enum ALoad : int { kARow = 0, kATTma = 1, kATCp = 2, kARowStg = 3 };
enum BLoad : int { kBRowTma = 0, kBRowCp = 1, kBT = 2 };

// Shared-memory layout (from a 1024-byte aligned base):
//   Bs[STAGES][BK][BP] | As[STAGES][BK][AP] | fullA[STAGES] | fullB[STAGES] |
//   empty[STAGES] | sync barrier | abort word
// and for kARowStg (with the ring depth of stg_ring_stages):
//   Bs | As | staging[kStgSlots][BM][BK] | the barrier block | staged[kStgSlots]
// with row pitches AP = BM (+ kApad when transposed on store) and likewise BP.
template <int ST>
struct BarrierBlock {
  uint64_t fullA[ST];   // NT cp.async arrivals: this thread's copies landed (kARowStg:
                        // one arrival by the producer warp once all its lanes have stored)
  uint64_t fullB[ST];   // one expect_tx arrival + the TMA transaction bytes of the stage
  uint64_t empty[ST];   // one arrival per warp: the slot may be refilled
  uint64_t sync;        // CTA-wide rendezvous with a bounded wait
  int abort;            // set by the first thread that gives up waiting
};

template <class Cfg>
constexpr int kernel_smem_bytes() {
  constexpr TileShape S = Cfg::S;
  static_assert(sizeof(BarrierBlock<S.STAGES>) <= S.STAGES * 3 * 8 + 16, "barrier block size");
  return smem_bytes(S);
}
template <class Cfg>
constexpr int kernel_smem_bytes_stg() {
  constexpr TileShape S = Cfg::S;
  constexpr int ST = stg_ring_stages(S);
  static_assert(sizeof(BarrierBlock<ST>) <= ST * 3 * 8 + 16, "barrier block size");
  return stg_smem_bytes(S, ST);
}
// Threads of one CTA: the FMA warps, plus the producer warp of kARowStg.
template <class Cfg, int AL>
constexpr int kernel_threads() {
  return Cfg::S.NT + (AL == kARowStg ? kWarp : 0);
}

// Bound of the clean-up waits of an aborting CTA (copies and MMAs it already
// issued, a peer's last arrivals): these end within microseconds, so the bound
// is at least 100 ms whatever the detection timeout, and a short timeout never
// lets a CTA free its tensor memory or exit with work still in flight.
__device__ __forceinline__ long long cleanup_bound_ns(long long timeout_ns) {
  return timeout_ns > 100000000LL ? timeout_ns : 100000000LL;
}

// Bounded wait on an mbarrier phase. Returns false (after recording `code`
// and raising the CTA's abort word) if the phase does not complete within
// timeout_ns, or if another thread has already raised the abort word.
__device__ __forceinline__ bool bounded_wait(uint32_t bar, uint32_t parity, volatile int* abort_w,
                                             int* status, int code, long long timeout_ns) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::global_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 16; ++i)
      if (ptx::mbar_try_wait(bar, parity)) return true;
    if (*abort_w) return false;
    if ((long long)(ptx::global_ns() - t0) > timeout_ns) {
      *abort_w = 1;
      atomicCAS(status, 0, code);
      return false;
    }
  }
}

// Interior transposing copies of one row group (rows of A, or of a stored
// transposed B): for each k-group KG, one 4-byte copy with both offsets
// compile-time (destination: KG*8 rows of the tile plus the group's
// MG*A_ROWS columns; source: KG*8 floats along the row).
template <int AP, int A_ROWS, int MG, int... KG>
__device__ __forceinline__ void issue_a_group(uint32_t dst, const float* src,
                                              std::integer_sequence<int, KG...>) {
  (ptx::cp_async_4_imm<(KG * kAloadK * AP + MG * A_ROWS) * 4, KG * kAloadK * 4>(dst, src), ...);
}

// All interior transposing copies of one k-slice: row group MG starts
// MG*stride floats after the first.
template <int AP, int A_ROWS, int A_KG, int... MG>
__device__ __forceinline__ void issue_a_tile(uint32_t dst, const float* src, long long stride,
                                             std::integer_sequence<int, MG...>) {
  (issue_a_group<AP, A_ROWS, MG>(dst, src + MG * stride, std::make_integer_sequence<int, A_KG>{}),
   ...);
}

template <class Cfg, int AL, int BL>
__global__ void __launch_bounds__(kernel_threads<Cfg, AL>(), Cfg::S.MINB)
    ffma_sgemm_kernel(const __grid_constant__ KernelParams p,
                      const __grid_constant__ CUtensorMap tmapA,
                      const __grid_constant__ CUtensorMap tmapB) {
  constexpr TileShape S = Cfg::S;
  static_assert(cfg_valid(S), "illegal tile configuration");
  constexpr bool kStg = (AL == kARowStg);
  static_assert(!kStg || (stg_eligible(S) && BL == kBRowTma), "staged A needs an eligible shape");
  constexpr int BM = S.BM, BN = S.BN, BK = S.BK, NT = S.NT, KU = S.KU;
  constexpr int ST = kStg ? stg_ring_stages(S) : S.STAGES;
  constexpr int ORDER = S.ORDER;
  constexpr int WM = S.WM, WN = S.WN, TM = S.TM, TN = S.TN, WNITER = S.WNITER;
  constexpr int WMITER = wmiter(S), WSUBM = wsubm(S), WSUBN = wsubn(S);
  constexpr int AP = (AL == kARow || kStg) ? BM + kApad : BM;  // As row pitch (floats)
  constexpr int BP = (BL == kBT) ? BN + kApad : BN;     // Bs row pitch (floats)
  constexpr int A_ST = a_stage_floats(S), B_ST = b_stage_floats(S);
  static_assert(BK * AP <= A_ST && BK * BP <= B_ST, "stage sizes");
  constexpr int D = ST - 2;                    // k-slices loaded ahead
  // k-step of a slice's last chunk at which the copies of a later slice are
  // issued when D >= 2 (always inside the chunk, so exactly once per slice)
  constexpr int kIssueAt = KU > 4 ? 4 : 0;
  static_assert(kIssueAt < KU, "issue point inside the last chunk");
  constexpr int LANES_N = WSUBN / TN;          // lanes along n in a sub-tile
  constexpr int RM = WMITER * TM, RN = WNITER * TN;  // a lane's rows / cols
  constexpr int A_ROWS = NT / kAloadK;         // rows per transposing-copy pass
  constexpr int A_MG = BM / A_ROWS, A_KG = BK / kAloadK;
  constexpr int B_MG = BN / A_ROWS;            // same, for a stored transposed B
  constexpr int B_PASSES = (BK * BN) / NT;
  constexpr int AT_PASSES = (BK * BM) / NT;
  constexpr int WARPS_N = BN / WN;
  constexpr bool kUsesCp = (AL != kATTma && !kStg) || (BL != kBRowTma);
  constexpr bool kUsesTma = (AL == kATTma) || (BL == kBRowTma);
  // the FMA warps wait for fullA when A arrives by copies or from the producer
  constexpr bool kWaitA = kUsesCp || kStg;
  constexpr uint32_t TMA_BYTES =
      (uint32_t)(((AL == kATTma) ? BK * BM * 4 : 0) + ((BL == kBRowTma) ? BK * BN * 4 : 0));
  constexpr uint32_t FULL = 0xffffffffu;

  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw_addr = ptx::smem_addr(smem_raw);
  unsigned char* base = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  float* Bs = reinterpret_cast<float*>(base);
  float* As = Bs + ST * B_ST;
  float* Stg = As + ST * A_ST;  // kARowStg staging slots (1024-byte aligned)
  BarrierBlock<ST>* bb =
      reinterpret_cast<BarrierBlock<ST>*>(Stg + (kStg ? kStgSlots * BM * BK : 0));
  uint64_t* staged = reinterpret_cast<uint64_t*>(bb + 1);  // kARowStg: slot landed
  volatile int* abort_w = &bb->abort;

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int b = blockIdx.x;
  const Schedule& sc = p.sched;

  if (tid == 0) {
    for (int s = 0; s < ST; ++s) {
      ptx::mbar_init(ptx::smem_addr(&bb->fullA[s]), kStg ? 1 : NT);
      ptx::mbar_init(ptx::smem_addr(&bb->fullB[s]), 1);
      ptx::mbar_init(ptx::smem_addr(&bb->empty[s]), NT / 32);
    }
    ptx::mbar_init(ptx::smem_addr(&bb->sync), NT);
    if (kStg)
      for (int j = 0; j < kStgSlots; ++j) ptx::mbar_init(ptx::smem_addr(&staged[j]), 1);
    bb->abort = 0;
    ptx::mbar_fence_init();
    if (AL == kATTma || kStg) ptx::tma_prefetch_desc(&tmapA);
    if (BL == kBRowTma) ptx::tma_prefetch_desc(&tmapB);
  }
  __syncthreads();
  // Launched with programmatic stream serialization, this grid may start
  // while the kernel before it on the stream is finishing: the set-up above
  // touches only shared memory and the parameters, and nothing below reads or
  // writes global memory before that kernel has completed. The next grid may
  // launch now (its own wait protects this grid's results).
#if SGEMM_GB300_PDL
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
#endif

  const int npieces = num_pieces(sc, b);
  const int nsteps = (int)total_steps(sc, b);

  if constexpr (kStg) {
    if (warp == NT / kWarp) {
      // ---- the producer warp of kARowStg --------------------------------------
      // Walks the same steps as the FMA warps. Step s: wait until ring slot
      // s % ST is free, start the TMA of its B tile, wait for the staged A
      // slice of step s, transpose it into the slot's As[k][m] and arrive on
      // fullA; then start the staging TMA of step s + kStgSlots into the
      // staging slot just read. A slice is thus requested kStgSlots steps
      // before it is transposed, and the B tile of a step as soon as its slot
      // is free.
      struct Cursor {
        int piece, k, ke, m0, n0, bi;
      };
      auto cur_set = [&](Cursor& c, int i) {
        const Piece lp = get_piece(sc, b, i);
        int tm, tn;
        tile_coords_batched(sc, lp.tile, c.bi, tm, tn);
        c.piece = i;
        c.k = lp.kb;
        c.ke = lp.ke;
        c.m0 = tm * BM;
        c.n0 = tn * BN;
      };
      auto cur_next = [&](Cursor& c) {
        if (++c.k == c.ke && c.piece + 1 < npieces) cur_set(c, c.piece + 1);
      };
      Cursor ca{0, 0, 0, 0, 0, 0}, cb{0, 0, 0, 0, 0, 0};
      if (npieces > 0) {
        cur_set(ca, 0);
        cur_set(cb, 0);
      }
      const uint32_t stg_addr = ptx::smem_addr(Stg);
      constexpr uint32_t kStgBytes = (uint32_t)(BM * BK * 4);
      int a_issued = 0, b_issued = 0, s = 0;
      auto issue_staging = [&]() {
        if (lane == 0) {
          const int j = a_issued % kStgSlots;
          const uint32_t fa = ptx::smem_addr(&staged[j]);
          ptx::mbar_arrive_expect_tx(fa, kStgBytes);
          ptx::tma_load_3d(stg_addr + (uint32_t)j * kStgBytes, &tmapA, ca.k * BK, ca.m0, ca.bi, fa);
        }
        ++a_issued;
        cur_next(ca);
      };
      // One staging slot (BM rows of 32 k-values, 128-byte rows; TMA's 128-byte
      // swizzle keeps 16-byte chunk c of row r at chunk c ^ (r & 7)) into
      // As[k][m]: the lane moves 4 x 4 blocks e = q * 32 + lane, rows 4 rg ..
      // 4 rg + 3 with rg = e % (BM / 4), k-chunk c = (e / (BM / 4) + rg) % 8,
      // with four 128-bit loads and four 128-bit stores. Each group of eight
      // lanes then reads eight different chunk positions and writes eight
      // different 16-byte bank groups (the row pitch BM + 4 shifts each k-row
      // by one group), so neither side has bank conflicts.
      auto transpose_slot = [&](const float* src, float* dst) {
        constexpr int R = BM / 4, NB = BM / 16, UB = NB < 4 ? NB : 4;
        static_assert(NB % UB == 0, "staging blocks per lane");
        const char* sb = reinterpret_cast<const char*>(src);
#pragma unroll
        for (int q0 = 0; q0 < NB; q0 += UB) {
          float4 v[UB][4];
#pragma unroll
          for (int u = 0; u < UB; ++u) {
            const int e = (q0 + u) * kWarp + lane;
            const int rg = e % R, c = (e / R + rg) & 7;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int r = 4 * rg + j;
              v[u][j] = *reinterpret_cast<const float4*>(sb + r * 128 + ((c ^ (r & 7)) << 4));
            }
          }
#pragma unroll
          for (int u = 0; u < UB; ++u) {
            const int e = (q0 + u) * kWarp + lane;
            const int rg = e % R, c = (e / R + rg) & 7;
            float* d = dst + (4 * c) * AP + 4 * rg;
            *reinterpret_cast<float4*>(d + 0 * AP) =
                make_float4(v[u][0].x, v[u][1].x, v[u][2].x, v[u][3].x);
            *reinterpret_cast<float4*>(d + 1 * AP) =
                make_float4(v[u][0].y, v[u][1].y, v[u][2].y, v[u][3].y);
            *reinterpret_cast<float4*>(d + 2 * AP) =
                make_float4(v[u][0].z, v[u][1].z, v[u][2].z, v[u][3].z);
            *reinterpret_cast<float4*>(d + 3 * AP) =
                make_float4(v[u][0].w, v[u][1].w, v[u][2].w, v[u][3].w);
          }
        }
      };

      bool ok = true;
      for (int j = 0; j < kStgSlots && a_issued < nsteps; ++j) issue_staging();
      for (s = 0; s < nsteps; ++s) {
        const int slot = s % ST;
        if (s >= ST) {
          const uint32_t par = (uint32_t)((s / ST) & 1) ^ 1u;
          ok = __all_sync(FULL, bounded_wait(ptx::smem_addr(&bb->empty[slot]), par, abort_w,
                                             p.status, kDevTimeoutEmpty, p.timeout_ns));
          if (!ok) break;
        }
        if (lane == 0) {
          const uint32_t fb = ptx::smem_addr(&bb->fullB[slot]);
          ptx::mbar_arrive_expect_tx(fb, TMA_BYTES);
          ptx::tma_load_3d(ptx::smem_addr(Bs + slot * B_ST), &tmapB, cb.n0, cb.k * BK, cb.bi, fb);
        }
        ++b_issued;
        const int j = s % kStgSlots;
        ok = __all_sync(FULL, bounded_wait(ptx::smem_addr(&staged[j]),
                                           (uint32_t)((s / kStgSlots) & 1), abort_w, p.status,
                                           kDevTimeoutFull, p.timeout_ns));
        if (!ok) break;
        transpose_slot(Stg + j * (BM * BK), As + slot * A_ST);
        // each lane orders its reads of staging slot j before the async-proxy
        // write that refills it; the warp sync then orders every lane's
        // stores and reads before lane 0's release on fullA and its TMA
        const bool refill = a_issued < nsteps;
        if (refill) ptx::fence_proxy_async_shared();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&bb->fullA[slot]));
        if (refill) issue_staging();
        cur_next(cb);
      }
      if (!ok && lane == 0) {
        // abandoned: wait (bounded) for this warp's TMAs still in flight --
        // the staging slices of steps s .. a_issued - 1 and the B tiles of
        // the last ST steps issued -- so nothing lands after the CTA is gone
        const uint64_t t0 = ptx::global_ns();
        const long long bound = cleanup_bound_ns(p.timeout_ns);
        for (int t = s; t < a_issued; ++t) {
          const uint32_t fa = ptx::smem_addr(&staged[t % kStgSlots]);
          while (!ptx::mbar_try_wait(fa, (uint32_t)((t / kStgSlots) & 1)))
            if ((long long)(ptx::global_ns() - t0) > bound) break;
        }
        for (int t = b_issued - 1; t >= 0 && t >= b_issued - ST; --t) {
          const uint32_t fb = ptx::smem_addr(&bb->fullB[t % ST]);
          while (!ptx::mbar_try_wait(fb, (uint32_t)((t / ST) & 1)))
            if ((long long)(ptx::global_ns() - t0) > bound) break;
        }
      }
      return;
    }
  }

  // ---- lane geometry --------------------------------------------------------
  const int warp_m = warp / WARPS_N, warp_n = warp % WARPS_N;
  const int lr = lane / LANES_N, lc = lane % LANES_N;
  // fragment read offsets inside one stage (floats)
  const int a_frag_off = warp_m * WM + lr * TM;
  const int b_frag_off = warp_n * WN + lc * TN;
  // transposing copies: this thread copies k = kg*8 + a_k of rows mg*A_ROWS + a_m
  const int a_k = tid % kAloadK, a_m = tid / kAloadK;

  const float* __restrict__ Ag = p.A;
  const float* __restrict__ Bg = p.B;
  const int M = p.M, N = p.N, K = p.K;
  const long long lda = p.lda, ldb = p.ldb;
  const long long a_group_stride = (long long)A_ROWS * lda;  // floats between row groups
  const long long b_group_stride = (long long)A_ROWS * ldb;

  const uint32_t As_addr = ptx::smem_addr(As);
  const uint32_t Bs_addr = ptx::smem_addr(Bs);

  // ---- load cursor: which (tile, k-slice) the next issued step is ---------
  int l_piece = 0, l_k = 0, l_ke = 0, l_m0 = 0, l_n0 = 0, l_bi = 0;
  bool l_m_inside = false;            // all BM rows of the tile are < M
  bool l_n_inside = false;            // all BN columns of the tile are < N
  const float* l_arow = Ag;           // row-major A: A + bi*sA + (m0 + a_m) * lda
  const float* l_brow = Bg;           // stored transposed B: B + bi*sB + (n0 + a_m) * ldb
  auto set_load_piece = [&](int i) {
    const Piece lp = get_piece(sc, b, i);
    int tm, tn;
    tile_coords_batched(sc, lp.tile, l_bi, tm, tn);
    l_k = lp.kb;
    l_ke = lp.ke;
    l_m0 = tm * BM;
    l_n0 = tn * BN;
    l_m_inside = l_m0 + BM <= M;
    l_n_inside = l_n0 + BN <= N;
    if (AL == kARow)
      l_arow = Ag + (long long)l_bi * p.sA + (l_m_inside ? (long long)(l_m0 + a_m) * lda : 0);
    if (BL == kBT)
      l_brow = Bg + (long long)l_bi * p.sB + (l_n_inside ? (long long)(l_n0 + a_m) * ldb : 0);
  };
  if (npieces > 0) set_load_piece(0);
  // steps whose copies this thread has issued (kARowStg: the producer warp
  // issues every copy, so the FMA warps start with all of them "issued")
  int issued = kStg ? nsteps : 0;

  // Issue the copies of the next step into its ring slot, then advance the
  // cursor. Returns false on abort.
  auto issue_next = [&]() -> bool {
    const int slot = issued % ST;
    if (issued >= ST) {
      const uint32_t par = (uint32_t)((issued / ST) & 1) ^ 1u;
      const bool ok = bounded_wait(ptx::smem_addr(&bb->empty[slot]), par, abort_w, p.status,
                                   kDevTimeoutEmpty, p.timeout_ns);
      if (!__all_sync(FULL, ok)) return false;
    }
    const int k0 = l_k * BK;
    const uint32_t a_slot = As_addr + (uint32_t)(slot * A_ST * 4);
    const uint32_t b_slot = Bs_addr + (uint32_t)(slot * B_ST * 4);
    const uint32_t t_dst0 = (uint32_t)((a_k * AP + a_m) * 4);  // transposing-copy offsets
    if constexpr (AL == kARow) {
      // A transposed on store, As[k][m] <- A[m0 + m][k0 + k], zero outside
      if (l_m_inside && k0 + BK <= K) {
        issue_a_tile<AP, A_ROWS, A_KG>(a_slot + t_dst0, l_arow + k0 + a_k, a_group_stride,
                                       std::make_integer_sequence<int, A_MG>{});
      } else {
        const float* Ab = Ag + (long long)l_bi * p.sA;
#pragma unroll
        for (int mg = 0; mg < A_MG; ++mg) {
          const int row = l_m0 + mg * A_ROWS + a_m;
          const bool row_ok = row < M;
          const float* src_row = Ab + (row_ok ? (long long)row * lda : 0);
#pragma unroll
          for (int kg = 0; kg < A_KG; ++kg) {
            const int k = k0 + kg * kAloadK + a_k;
            const bool ok = row_ok && (k < K);
            ptx::cp_async_4(a_slot + t_dst0 + (uint32_t)((kg * kAloadK * AP + mg * A_ROWS) * 4),
                            ok ? (const void*)(src_row + k) : (const void*)Ag, ok ? 4u : 0u);
          }
        }
      }
    } else if constexpr (AL == kATCp) {
      // stored transposed A: As[k][m] <- A[k0 + k][m0 + m], zero outside
      const float* Ab = Ag + (long long)l_bi * p.sA;
#pragma unroll
      for (int ps = 0; ps < AT_PASSES; ++ps) {
        const int e = ps * NT + tid;
        const int kk = e / BM, mm = e % BM;
        const int k = k0 + kk, m = l_m0 + mm;
        const bool ok = (k < K) && (m < M);
        ptx::cp_async_4(a_slot + (uint32_t)((kk * AP + mm) * 4),
                        ok ? (const void*)(Ab + (long long)k * lda + m) : (const void*)Ag,
                        ok ? 4u : 0u);
      }
    }
    if constexpr (BL == kBRowCp) {
      // B without TMA: Bs[k][n] <- B[k0 + k][n0 + n], zero outside
      const float* Bb = Bg + (long long)l_bi * p.sB;
#pragma unroll
      for (int ps = 0; ps < B_PASSES; ++ps) {
        const int e = ps * NT + tid;
        const int kk = e / BN, nn = e % BN;
        const int k = k0 + kk, n = l_n0 + nn;
        const bool ok = (k < K) && (n < N);
        ptx::cp_async_4(b_slot + (uint32_t)((kk * BP + nn) * 4),
                        ok ? (const void*)(Bb + (long long)k * ldb + n) : (const void*)Bg,
                        ok ? 4u : 0u);
      }
    } else if constexpr (BL == kBT) {
      // stored transposed B: Bs[k][n] <- B[n0 + n][k0 + k], transposed on store
      const uint32_t bt_dst0 = (uint32_t)((a_k * BP + a_m) * 4);
      if (l_n_inside && k0 + BK <= K) {
        issue_a_tile<BP, A_ROWS, A_KG>(b_slot + bt_dst0, l_brow + k0 + a_k, b_group_stride,
                                       std::make_integer_sequence<int, B_MG>{});
      } else {
        const float* Bb = Bg + (long long)l_bi * p.sB;
#pragma unroll
        for (int ng = 0; ng < B_MG; ++ng) {
          const int row = l_n0 + ng * A_ROWS + a_m;
          const bool row_ok = row < N;
          const float* src_row = Bb + (row_ok ? (long long)row * ldb : 0);
#pragma unroll
          for (int kg = 0; kg < A_KG; ++kg) {
            const int k = k0 + kg * kAloadK + a_k;
            const bool ok = row_ok && (k < K);
            ptx::cp_async_4(b_slot + bt_dst0 + (uint32_t)((kg * kAloadK * BP + ng * A_ROWS) * 4),
                            ok ? (const void*)(src_row + k) : (const void*)Bg, ok ? 4u : 0u);
          }
        }
      }
    }
    if (kUsesCp) ptx::cp_async_arrive_noinc(ptx::smem_addr(&bb->fullA[slot]));
    if (kUsesTma && tid == 0) {
      const uint32_t fb = ptx::smem_addr(&bb->fullB[slot]);
      ptx::mbar_arrive_expect_tx(fb, TMA_BYTES);
      if (AL == kATTma) ptx::tma_load_3d(a_slot, &tmapA, l_m0, k0, l_bi, fb);
      if (BL == kBRowTma) ptx::tma_load_3d(b_slot, &tmapB, l_n0, k0, l_bi, fb);
    }
    ++issued;
    if (++l_k == l_ke) {
      if (++l_piece < npieces) set_load_piece(l_piece);
    }
    return true;
  };

  // Non-blocking test: have the operand tiles of `step` landed? (The copy
  // and TMA barriers are polled at once so their latencies overlap.)
  auto test_full = [&](int step) -> bool {
    const int slot = step % ST;
    const uint32_t par = (uint32_t)((step / ST) & 1);
    const bool a = kWaitA ? ptx::mbar_try_wait(ptx::smem_addr(&bb->fullA[slot]), par) : true;
    const bool b2 = kUsesTma ? ptx::mbar_try_wait(ptx::smem_addr(&bb->fullB[slot]), par) : true;
    return a && b2;
  };
  // Bounded wait until the operand tiles of `step` have landed; `ready` is
  // the result of an earlier test_full(step), if one was made.
  auto wait_full = [&](int step, bool ready) -> bool {
    bool ok = true;
    if (!ready) {
      const int slot = step % ST;
      const uint32_t par = (uint32_t)((step / ST) & 1);
      if (kWaitA)
        ok = bounded_wait(ptx::smem_addr(&bb->fullA[slot]), par, abort_w, p.status,
                          kDevTimeoutFull, p.timeout_ns);
      if (kUsesTma && ok)
        ok = bounded_wait(ptx::smem_addr(&bb->fullB[slot]), par, abort_w, p.status,
                          kDevTimeoutFull, p.timeout_ns);
    }
    return __all_sync(FULL, ok);
  };

  // Accumulators, stored as pairs along m: acc2[i/2][j] holds rows i and i+1
  // of column j (the operand layout of the paired FMA; the scalar orders use
  // the two halves separately).
  static_assert(RM % 2 == 0, "paired accumulators need an even row count");
  float2 acc2[RM / 2][RN];
#pragma unroll
  for (int i = 0; i < RM / 2; ++i)
#pragma unroll
    for (int j = 0; j < RN; ++j) acc2[i][j] = make_float2(0.f, 0.f);
#define SG_ACC(i, j) (((i) & 1) ? acc2[(i) >> 1][j].y : acc2[(i) >> 1][j].x)

  // Two fragment buffers: while the FMAs of k-step k read one, the 128-bit
  // loads of k-step k+1 fill the other.
  float af[2][RM], bfr[2][RN];
  auto load_frags = [&](int buf, const float* a_row, const float* b_row) {
#pragma unroll
    for (int wm = 0; wm < WMITER; ++wm)
#pragma unroll
      for (int q = 0; q < TM / 4; ++q) {
        const float4 v = *reinterpret_cast<const float4*>(a_row + wm * WSUBM + q * 4);
        af[buf][wm * TM + q * 4 + 0] = v.x;
        af[buf][wm * TM + q * 4 + 1] = v.y;
        af[buf][wm * TM + q * 4 + 2] = v.z;
        af[buf][wm * TM + q * 4 + 3] = v.w;
      }
#pragma unroll
    for (int wn = 0; wn < WNITER; ++wn)
#pragma unroll
      for (int q = 0; q < TN / 4; ++q) {
        const float4 v = *reinterpret_cast<const float4*>(b_row + wn * WSUBN + q * 4);
        bfr[buf][wn * TN + q * 4 + 0] = v.x;
        bfr[buf][wn * TN + q * 4 + 1] = v.y;
        bfr[buf][wn * TN + q * 4 + 2] = v.z;
        bfr[buf][wn * TN + q * 4 + 3] = v.w;
      }
  };

  uint32_t sync_phase = 0;
  // CTA-wide rendezvous with a bounded wait (a plain __syncthreads could not
  // be abandoned if another warp has given up).
  auto cta_sync = [&]() -> bool {
    ptx::mbar_arrive(ptx::smem_addr(&bb->sync));
    const bool ok = bounded_wait(ptx::smem_addr(&bb->sync), sync_phase, abort_w, p.status,
                                 kDevTimeoutSync, p.timeout_ns);
    sync_phase ^= 1u;
    return __all_sync(FULL, ok);
  };

  bool aborted = false;
  for (int s = 0; s < D && issued < nsteps; ++s) {
    if (!issue_next()) {
      aborted = true;
      break;
    }
  }

  int c_piece = 0, c_k = 0;
  Piece cpc{0, 0, 0};
  if (npieces > 0) {
    cpc = get_piece(sc, b, 0);
    c_k = cpc.kb;
  }
  if (!aborted && nsteps > 0) {
    if (wait_full(0, false))
      load_frags(0, As + a_frag_off, Bs + b_frag_off);
    else
      aborted = true;
  }

  for (int step = 0; step < nsteps && !aborted; ++step) {
    // With two or more slices in flight ahead (D >= 2), the copies for a later
    // step are issued a few k-steps into this one, so that the step's FMAs
    // start without waiting behind them; with one (D == 1) that slice is the
    // next one, so its copies go out first to have the whole step to land.
    bool issue_ok = true;
    if (D < 2 && issued < nsteps) issue_ok = issue_next();
    const int slot = step % ST;
    const float* a_s = As + slot * A_ST + a_frag_off;
    const float* b_s = Bs + slot * B_ST + b_frag_off;
    bool next_ok = true;

    // ---- BK k-steps of outer-product FMA on this slot, KU per chunk ----------
    // One k-step: update the accumulators from fragment buffer `cur`.
    auto kstep = [&](int cur) {
      if constexpr (ORDER == 2) {
        // paired FMA: two rows of one column per instruction; the A pair
        // comes straight from the 128-bit fragment load, the B value is
        // duplicated into both halves
        float2 bd[RN];
#pragma unroll
        for (int j = 0; j < RN; ++j) bd[j] = make_float2(bfr[cur][j], bfr[cur][j]);
#pragma unroll
        for (int ip = 0; ip < RM / 2; ++ip) {
          const float2 a2 = make_float2(af[cur][2 * ip], af[cur][2 * ip + 1]);
#pragma unroll
          for (int j = 0; j < RN; ++j) acc2[ip][j] = __ffma2_rn(a2, bd[j], acc2[ip][j]);
        }
      } else if constexpr (ORDER == 3) {
        // paired FMA, column by column: one duplicated B pair feeds RM/2
        // consecutive instructions
#pragma unroll
        for (int j = 0; j < RN; ++j) {
          const float2 bd = make_float2(bfr[cur][j], bfr[cur][j]);
#pragma unroll
          for (int ip = 0; ip < RM / 2; ++ip)
            acc2[ip][j] = __ffma2_rn(make_float2(af[cur][2 * ip], af[cur][2 * ip + 1]), bd,
                                     acc2[ip][j]);
        }
      } else {
        // scalar outer product; ORDER 1 walks odd rows backwards so that
        // consecutive FFMAs at a row change still share their B operand
#pragma unroll
        for (int i = 0; i < RM; ++i)
#pragma unroll
          for (int jj = 0; jj < RN; ++jj) {
            const int j = (ORDER == 1 && (i & 1)) ? RN - 1 - jj : jj;
            SG_ACC(i, j) = fmaf(af[cur][i], bfr[cur][j], SG_ACC(i, j));
          }
      }
    };

    // all chunks but the last: the next fragment always comes from this slot
#pragma unroll 1
    for (int kc = 0; kc < BK - KU; kc += KU) {
#pragma unroll
      for (int kk = 0; kk < KU; ++kk) {
        const int cur = kk & 1;
        load_frags(cur ^ 1, a_s + (kc + kk + 1) * AP, b_s + (kc + kk + 1) * BP);
        kstep(cur);
      }
    }
    // last chunk: halfway through, test whether the next slot has landed;
    // in the last k-step, fetch its first fragment under this k-step's FMAs
    {
      constexpr int kc = BK - KU;
      const bool has_next = step + 1 < nsteps;
      bool ready = false;
#pragma unroll
      for (int kk = 0; kk < KU; ++kk) {
        const int cur = kk & 1;
        if (D >= 2 && kk == kIssueAt && issued < nsteps) issue_ok = issue_next();
        if (kk + 1 < KU) {
          load_frags(cur ^ 1, a_s + (kc + kk + 1) * AP, b_s + (kc + kk + 1) * BP);
          if (kk == KU / 2 - 1 && has_next) ready = test_full(step + 1);
        } else if (has_next) {
          next_ok = wait_full(step + 1, ready);
          const int ns = (step + 1) % ST;
          load_frags(cur ^ 1, As + ns * A_ST + a_frag_off, Bs + ns * B_ST + b_frag_off);
        }
        kstep(cur);
      }
    }

    // release the slot: one arrival per warp once all its lanes are done
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&bb->empty[slot]));
    if (!next_ok || !issue_ok) {
      aborted = true;
      break;
    }

    if (++c_k < cpc.ke) continue;

    // ---- the current piece is complete: publish a partial or write C --------
    float* ws_tile = p.ws + (long long)b * (BM * BN);
    if (is_partial_piece(sc, cpc)) {
      float4* dst = reinterpret_cast<float4*>(ws_tile);
#pragma unroll
      for (int i = 0; i < RM; ++i)
#pragma unroll
        for (int j4 = 0; j4 < RN / 4; ++j4)
          __stcg(dst + (i * (RN / 4) + j4) * NT + tid,
                 make_float4(SG_ACC(i, j4 * 4 + 0), SG_ACC(i, j4 * 4 + 1), SG_ACC(i, j4 * 4 + 2),
                             SG_ACC(i, j4 * 4 + 3)));
      if (!cta_sync()) {
        aborted = true;
        break;
      }
      if (tid == 0) {
        __threadfence();
        ptx::st_release(p.flags + b, p.epoch);
      }
    } else {
      const int nc = num_contributors(sc, b, cpc);
      if (nc > 0) {
        if (tid == 0) {
          for (int c = 1; c <= nc; ++c) {
            uint32_t* f = p.flags + b + c;
            if (ptx::ld_acquire(f) != p.epoch) {
              const uint64_t t0 = ptx::global_ns();
              while (ptx::ld_acquire(f) != p.epoch) {
                if ((long long)(ptx::global_ns() - t0) > p.timeout_ns) {
                  *abort_w = 1;
                  atomicCAS(p.status, 0, (int)kDevTimeoutFlag);
                  break;
                }
                __nanosleep(200);
              }
            }
            if (*abort_w) break;
            // consumed: no later launch can mistake it for its own, even one
            // that reuses this epoch (a CUDA graph replays its arguments)
            *f = 0u;
          }
        }
        if (!cta_sync() || *abort_w) {
          aborted = true;
          break;
        }
        // add the partials of CTAs b+1 .. b+nc, in that order
        for (int c = 1; c <= nc; ++c) {
          const float4* src = reinterpret_cast<const float4*>(ws_tile + (long long)c * (BM * BN));
#pragma unroll
          for (int i = 0; i < RM; ++i)
#pragma unroll
            for (int j4 = 0; j4 < RN / 4; ++j4) {
              const float4 v = __ldcg(src + (i * (RN / 4) + j4) * NT + tid);
              SG_ACC(i, j4 * 4 + 0) += v.x;
              SG_ACC(i, j4 * 4 + 1) += v.y;
              SG_ACC(i, j4 * 4 + 2) += v.z;
              SG_ACC(i, j4 * 4 + 3) += v.w;
            }
        }
      }
      // epilogue: C = alpha * acc + beta * C for this lane's RM x RN patch,
      // one row group (TM rows x RN columns) at a time: all of the group's
      // 128-bit reads of C are issued before any of its writes, so their
      // latencies overlap instead of adding up.
      int bi, tm, tn;
      tile_coords_batched(sc, cpc.tile, bi, tm, tn);
      float* Cb = p.C + (long long)bi * p.sC;
      const int row0 = tm * BM + a_frag_off;
      const int col0 = tn * BN + b_frag_off;
      const float alpha = p.alpha, beta = p.beta;
      constexpr int QN = WNITER * (TN / 4);  // float4 groups per row
#pragma unroll
      for (int wm = 0; wm < WMITER; ++wm) {
        float4 old[TM][QN];
#pragma unroll
        for (int i = 0; i < TM; ++i) {
          const int row = row0 + wm * WSUBM + i;
#pragma unroll
          for (int g = 0; g < QN; ++g) {
            const int col = col0 + (g / (TN / 4)) * WSUBN + (g % (TN / 4)) * 4;
            const float* cp = Cb + (long long)row * p.ldc + col;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (beta != 0.f && row < M) {
              if (p.c_vec && col + 3 < N) {
                v = *reinterpret_cast<const float4*>(cp);
              } else {
                if (col + 0 < N) v.x = cp[0];
                if (col + 1 < N) v.y = cp[1];
                if (col + 2 < N) v.z = cp[2];
                if (col + 3 < N) v.w = cp[3];
              }
            }
            old[i][g] = v;
          }
        }
#pragma unroll
        for (int i = 0; i < TM; ++i) {
          const int row = row0 + wm * WSUBM + i;
          if (row >= M) continue;
          float* crow = Cb + (long long)row * p.ldc;
          const int ai = wm * TM + i;
#pragma unroll
          for (int g = 0; g < QN; ++g) {
            const int col = col0 + (g / (TN / 4)) * WSUBN + (g % (TN / 4)) * 4;
            const int cj = (g / (TN / 4)) * TN + (g % (TN / 4)) * 4;
            float4 v;
            if (beta != 0.f) {
              v.x = fmaf(alpha, SG_ACC(ai, cj + 0), beta * old[i][g].x);
              v.y = fmaf(alpha, SG_ACC(ai, cj + 1), beta * old[i][g].y);
              v.z = fmaf(alpha, SG_ACC(ai, cj + 2), beta * old[i][g].z);
              v.w = fmaf(alpha, SG_ACC(ai, cj + 3), beta * old[i][g].w);
            } else {
              v = make_float4(alpha * SG_ACC(ai, cj + 0), alpha * SG_ACC(ai, cj + 1),
                              alpha * SG_ACC(ai, cj + 2), alpha * SG_ACC(ai, cj + 3));
            }
            if (p.c_vec && col + 3 < N) {
              *reinterpret_cast<float4*>(crow + col) = v;
            } else {
              if (col + 0 < N) crow[col + 0] = v.x;
              if (col + 1 < N) crow[col + 1] = v.y;
              if (col + 2 < N) crow[col + 2] = v.z;
              if (col + 3 < N) crow[col + 3] = v.w;
            }
          }
        }
      }
    }
#pragma unroll
    for (int i = 0; i < RM / 2; ++i)
#pragma unroll
      for (int j = 0; j < RN; ++j) acc2[i][j] = make_float2(0.f, 0.f);
    if (++c_piece < npieces) {
      cpc = get_piece(sc, b, c_piece);
      c_k = cpc.kb;
    }
  }

  if (aborted) {
    // Drain this thread's copies; the TMA issuer also waits (bounded) for
    // the tiles it issued and nobody consumed, so nothing lands in shared
    // memory after the CTA is gone.
    ptx::cp_async_wait_all();
    if (kUsesTma && !kStg && tid == 0) {
      const uint64_t t0 = ptx::global_ns();
      for (int s = issued - 1; s >= 0 && s >= issued - ST; --s) {
        const uint32_t fb = ptx::smem_addr(&bb->fullB[s % ST]);
        const uint32_t par = (uint32_t)((s / ST) & 1);
        while (!ptx::mbar_try_wait(fb, par)) {
          if ((long long)(ptx::global_ns() - t0) > cleanup_bound_ns(p.timeout_ns)) break;
        }
      }
    }
    __nanosleep(20000);
  }
#undef SG_ACC
}

}  // namespace sgemm_gb300
