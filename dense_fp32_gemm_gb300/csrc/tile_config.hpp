// tile_config.hpp -- compile-time tile parameters of the FFMA SGEMM kernel and
// the legality rules they must satisfy.
//
// Notation follows "Warp Tiling: A Third Level of Tiling" (sections "The Warp
// Tile Is Not Contiguous Either" and "The Kernel"): a CTA computes a BM x BN
// tile of C, stepping through K in slices of BK; each warp owns a WM x WN
// rectangle of the CTA tile, covered in WMITER x WNITER sub-tiles of
// WSUBM x WSUBN; inside a sub-tile each of the 32 lanes owns a TM x TN patch.
// WMITER is derived, never chosen: WMITER = WM*WN / (32*TM*TN*WNITER).
//
// "Autotuning: Searching the Tile-Shape Space" (section "Most Configurations
// Are Not Wrong By A Little") makes the point that an illegal tuple still
// compiles and silently computes garbage, so legality must be decided before
// a kernel exists. cfg_valid() below is this kernel's own list: one guard per
// assumption the kernel body makes, ordered so that no guard divides by a
// quantity an earlier guard has not checked.
#pragma once

namespace sgemm_gb300 {

constexpr int kWarp = 32;
// FFMA launches use programmatic dependent launch (launch.cuh, ffma_sgemm.cuh).
#ifndef SGEMM_GB300_PDL
#define SGEMM_GB300_PDL 1
#endif
// Shared memory a CTA may use on sm_103a (opt-in maximum per block).
constexpr int kMaxSmemPerCta = 227 * 1024;
// Padding (in floats) added to each k-row of the transposed A tile. With the
// A loader's lane map (8 consecutive k x 4 consecutive m per warp instruction)
// a row pitch of BM + 4 with BM % 32 == 0 puts the 32 scattered 4-byte stores
// of one instruction in 32 distinct banks, and keeps every row 16-byte
// aligned for the 128-bit fragment reads.
constexpr int kApad = 4;
// Lanes of one A-load instruction that walk along k (the rest walk along m).
constexpr int kAloadK = 8;
// Largest TMA box extent in one dimension.
constexpr int kTmaMaxBox = 256;

struct TileShape {
  int BM, BN, BK;        // CTA tile and k-slice
  int WM, WN, WNITER;    // warp tile and its sub-tile count along N
  int TM, TN;            // per-lane patch inside one sub-tile
  int NT;                // threads per CTA
  int STAGES;            // shared-memory pipeline depth
  int MINB;              // CTAs per SM promised to the register allocator
  int KU;                // k-steps per unrolled chunk of the inner loop
  int ORDER;             // k-step update: 0 FFMA row by row, 1 FFMA zig-zag,
                         // 2 paired FMA (two rows of a column per instruction),
                         // 3 paired FMA column by column
};

// Derived quantities; valid only for shapes that pass cfg_valid().
constexpr int wmiter(const TileShape& s) { return (s.WM * s.WN) / (kWarp * s.TM * s.TN * s.WNITER); }
constexpr int wsubm(const TileShape& s) { return s.WM / wmiter(s); }
constexpr int wsubn(const TileShape& s) { return s.WN / s.WNITER; }
constexpr int acc_per_thread(const TileShape& s) { return wmiter(s) * s.TM * s.WNITER * s.TN; }
constexpr int est_registers(const TileShape& s) {
  return acc_per_thread(s) + 2 * (wmiter(s) * s.TM + s.WNITER * s.TN) + 24;
}
// Floats reserved per stage for each operand tile: BK rows of the tile's width
// plus the padding a transposing copy needs, rounded up to 1024 bytes so that
// every stage of either operand can be a TMA destination. One size serves all
// operand layouts (the padding is unused when a tile arrives by TMA).
constexpr int round_1k_floats(int floats) { return (floats + 255) / 256 * 256; }
constexpr int a_stage_floats(const TileShape& s) { return round_1k_floats(s.BK * (s.BM + kApad)); }
constexpr int b_stage_floats(const TileShape& s) { return round_1k_floats(s.BK * (s.BN + kApad)); }
// Dynamic shared memory of one CTA: 1024 bytes of alignment slack, the stage
// buffers, then 3 mbarriers per stage (A landed, B landed, slot free), one
// rendezvous barrier and an abort word.
constexpr int smem_bytes(const TileShape& s) {
  return 1024 + s.STAGES * (a_stage_floats(s) + b_stage_floats(s)) * 4 + s.STAGES * 3 * 8 + 16;
}

// Row-major A through a staging ring (ALoad kARowStg in ffma_sgemm.cuh): one
// TMA box of BM rows x 32 k per k-slice lands, 128-byte swizzled, in one of
// kStgSlots staging slots, and one extra producer warp transposes it into the
// padded As[k][m] of the ring. The slots (and one mbarrier each) come on top
// of the ring, which keeps the configuration's depth or gives up stages until
// everything fits.
constexpr int kStgSlots = 2;
constexpr int stg_smem_bytes(const TileShape& s, int stages) {
  return 1024 + stages * (a_stage_floats(s) + b_stage_floats(s)) * 4 +
         kStgSlots * s.BM * s.BK * 4 + stages * 3 * 8 + 16 + kStgSlots * 8;
}
constexpr bool stg_fits(const TileShape& s, int stages) {
  return stg_smem_bytes(s, stages) <= kMaxSmemPerCta &&
         s.MINB * (stg_smem_bytes(s, stages) + 1024) <= 228 * 1024;
}
constexpr int stg_ring_stages(const TileShape& s) {
  int st = s.STAGES;
  while (st > 3 && !stg_fits(s, st)) --st;
  return st;
}
// A configuration is built with the staged variant when its slices are 32
// wide (one 128-byte swizzle span per row), its tile rows fit one TMA box, the
// ring keeps at least three stages beside the staging slots, and a lane of at
// most 64 accumulators leaves room for the extra warp: the register cap
// 65536 / ((NT + 32) * MINB) stays at 200 or more (the 64-accumulator kernels
// use about 190).
constexpr bool stg_eligible(const TileShape& s) {
  return s.BK == 32 && s.BM % 32 == 0 && s.BM <= kTmaMaxBox && stg_fits(s, stg_ring_stages(s)) &&
         acc_per_thread(s) <= 64 && (s.NT + kWarp) * s.MINB * 200 <= 65536;
}

// Every assumption of the kernel in ffma_sgemm.cuh, in the order the kernel
// relies on them. Returns 0 when legal, else the number of the first failed
// rule (so a test can tell which rule rejected a tuple).
constexpr int cfg_check(const TileShape& s) {
  // 1. positive extents
  if (s.BM <= 0 || s.BN <= 0 || s.BK <= 0 || s.WM <= 0 || s.WN <= 0 || s.WNITER <= 0 ||
      s.TM <= 0 || s.TN <= 0 || s.NT <= 0 || s.STAGES <= 0 || s.MINB <= 0 || s.KU <= 0 ||
      s.ORDER < 0 || s.ORDER > 3)
    return 1;
  // 2. whole warps, and warp tiles that tile the CTA tile one warp each
  if (s.NT % kWarp != 0) return 2;
  if (s.BM % s.WM != 0 || s.BN % s.WN != 0) return 3;
  if ((s.BM / s.WM) * (s.BN / s.WN) != s.NT / kWarp) return 4;
  // 3. the warp tile splits into a whole number of sub-tile passes
  if ((s.WM * s.WN) % (kWarp * s.TM * s.TN * s.WNITER) != 0) return 5;
  if (wmiter(s) < 1) return 6;
  if (s.WM % wmiter(s) != 0 || s.WN % s.WNITER != 0) return 7;
  // 4. each sub-tile is covered by exactly the 32 lanes of the warp
  if (wsubm(s) % s.TM != 0 || wsubn(s) % s.TN != 0) return 8;
  if ((wsubm(s) / s.TM) * (wsubn(s) / s.TN) != kWarp) return 9;
  // 5. 128-bit fragment reads from both operand tiles and 128-bit C updates
  if (s.TM % 4 != 0 || s.TN % 4 != 0) return 10;
  // 6. A loader: per instruction 8 lanes along k x (NT/8) rows along m; the
  //    transposed-store bank argument needs BM to be a multiple of 32
  if (s.BK % kAloadK != 0) return 11;
  if (s.BM % (s.NT / kAloadK) != 0 || s.BM % 32 != 0) return 12;
  // 7. B tile: one TMA box of BK rows x BN columns; the cp.async fallback
  //    covers the tile in whole passes of NT consecutive elements; a stored
  //    transposed B goes through the same transposing copy as A (rule 6 with
  //    BN for BM); a stored transposed A arrives as one TMA box of BK x BM or
  //    in whole passes of NT elements
  if (s.BN > kTmaMaxBox || s.BK > kTmaMaxBox || (s.BN * 4) % 16 != 0) return 13;
  if ((s.BK * s.BN) % s.NT != 0) return 14;
  if (s.BN % (s.NT / kAloadK) != 0 || s.BN % 32 != 0) return 23;
  if (s.BM > kTmaMaxBox || (s.BK * s.BM) % s.NT != 0) return 24;
  // 8. every C element owned by exactly one lane
  if (static_cast<long>(s.NT) * acc_per_thread(s) != static_cast<long>(s.BM) * s.BN) return 15;
  // 9. pipeline: at least one stage of slack between producer and consumer
  if (s.STAGES < 3) return 16;
  // 10. hard limits: shared memory per CTA (and per SM at MINB CTAs), and an
  //     accumulator count above which the register file cannot hold a lane
  if (smem_bytes(s) > kMaxSmemPerCta) return 17;
  if (s.MINB * (smem_bytes(s) + 1024) > 228 * 1024) return 18;
  if (acc_per_thread(s) > 128) return 19;
  // 11. registers: a lane holds its accumulators, two buffers of operand
  //     fragments and about 24 scalars; that estimate must fit the 255
  //     registers a thread can address and, for MINB resident CTAs, the
  //     64K-entry register file of an SM
  if (est_registers(s) > 255) return 20;
  if (s.NT * s.MINB * est_registers(s) > 65536) return 21;
  // 12. the inner loop runs BK/KU chunks of KU fully unrolled k-steps; the
  //     two fragment buffers alternate inside a chunk, so KU must be even
  if (s.KU % 2 != 0 || s.BK % s.KU != 0) return 22;
  return 0;
}

constexpr bool cfg_valid(const TileShape& s) { return cfg_check(s) == 0; }

}  // namespace sgemm_gb300
