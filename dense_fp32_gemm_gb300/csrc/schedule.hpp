// schedule.hpp -- persistent tile scheduler: which (tile, k-slice) units each
// CTA of the persistent grid computes, and who finishes a tile that was split.
//
// The pages launch one CTA per C tile (grid = ceil(N/BN) x ceil(M/BM)) and
// note that residency decides speed ("Autotuning: Searching the Tile-Shape
// Space", section "What The Sweep Found": a config that fits one block per SM
// finishes last). On a 152-SM part a plain one-CTA-per-tile grid also wastes
// the tail wave: 512 tiles over 152 SMs run in 4 waves with the last one 37%
// full. The scheduler here instead launches one persistent CTA per resident
// slot and balances the work exactly:
//
//   * the tile space is numbered in grouped raster order (GROUP_M tile rows at
//     a time, column by column inside a group) so that concurrently running
//     CTAs share A row-panels and B column-panels in L2;
//   * "whole" tiles [0, dp_tiles) are dealt round-robin: CTA b takes tiles
//     b, b + grid, b + 2*grid, ...;
//   * the remaining sk_tiles tiles (between one and two waves' worth, or all
//     tiles when there are fewer tiles than CTAs) are cut into k-slice units,
//     kiters per tile, and every CTA takes one contiguous run of
//     sk_units / grid units (the first sk_units % grid CTAs take one more);
//   * a run that starts inside a tile (not at its first k-slice) produces a
//     partial sum and stores it in workspace slot b; the CTA whose run holds
//     the tile's first k-slice owns the tile: it adds the partials of the
//     following CTAs in CTA order (a fixed order, so the result does not
//     depend on timing) and writes C.
//
// Everything here is plain integer arithmetic usable on host and device.
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define SG_HD __host__ __device__ __forceinline__
#else
#define SG_HD inline
#endif

namespace sgemm_gb300 {

struct Schedule {
  int tiles_m, tiles_n;   // tile grid over one C
  int tiles;              // batch * tiles_m * tiles_n (the batch index is outermost)
  int kiters;             // k-slices per tile: ceil(K / BK)
  int grid;               // persistent CTAs
  int group_m;            // raster group height in tiles
  int dp_tiles;           // tiles computed whole
  int sk_q, sk_r;         // units per split CTA: sk_q, +1 for CTAs < sk_r
  int64_t sk_units;       // (tiles - dp_tiles) * kiters
};

// One contiguous piece of a CTA's work: k-slices [kb, ke) of tile `tile`.
struct Piece {
  int tile;
  int kb, ke;
};

SG_HD int ceil_div_i(int a, int b) { return (a + b - 1) / b; }
// ceil(a / b) for 0 <= a <= INT_MAX and b >= 1, without overflow near INT_MAX.
SG_HD int ceil_div_nn(int a, int b) { return (int)(((long long)a + b - 1) / b); }

// Tile index -> (tile row, tile column) in grouped raster order.
SG_HD void tile_coords(const Schedule& s, int t, int& tm, int& tn) {
  const int per_group = s.group_m * s.tiles_n;
  const int group = t / per_group;
  const int first = group * s.group_m;
  const int rows = (s.tiles_m - first) < s.group_m ? (s.tiles_m - first) : s.group_m;
  const int r = t - group * per_group;
  tm = first + r % rows;
  tn = r / rows;
}

// Tile index -> (matrix of the batch, tile row, tile column).
SG_HD void tile_coords_batched(const Schedule& s, int t, int& bi, int& tm, int& tn) {
  const int per_matrix = s.tiles_m * s.tiles_n;
  bi = t / per_matrix;
  tile_coords(s, t - bi * per_matrix, tm, tn);
}

SG_HD int num_dp_pieces(const Schedule& s, int b) {
  return b < s.dp_tiles ? (s.dp_tiles - 1 - b) / s.grid + 1 : 0;
}

// The split units of CTA b: [u0, u1) in the k-slice numbering of the split
// tiles (unit u is k-slice u % kiters of split tile u / kiters).
SG_HD int64_t sk_begin(const Schedule& s, int b) {
  return (int64_t)b * s.sk_q + (b < s.sk_r ? b : s.sk_r);
}
SG_HD int64_t sk_end(const Schedule& s, int b) {
  return sk_begin(s, b) + s.sk_q + (b < s.sk_r ? 1 : 0);
}

SG_HD int num_sk_pieces(const Schedule& s, int b) {
  const int64_t u0 = sk_begin(s, b), u1 = sk_end(s, b);
  if (u1 <= u0) return 0;
  return (int)((u1 - 1) / s.kiters - u0 / s.kiters + 1);
}

SG_HD int num_pieces(const Schedule& s, int b) { return num_dp_pieces(s, b) + num_sk_pieces(s, b); }

// Total k-slices CTA b computes.
SG_HD int64_t total_steps(const Schedule& s, int b) {
  return (int64_t)num_dp_pieces(s, b) * s.kiters + (sk_end(s, b) - sk_begin(s, b));
}

// Piece i of CTA b (0 <= i < num_pieces(s, b)): whole tiles first, then the
// split run in ascending unit order.
SG_HD Piece get_piece(const Schedule& s, int b, int i) {
  Piece p;
  const int ndp = num_dp_pieces(s, b);
  if (i < ndp) {
    p.tile = b + i * s.grid;
    p.kb = 0;
    p.ke = s.kiters;
    return p;
  }
  const int j = i - ndp;
  const int64_t u0 = sk_begin(s, b), u1 = sk_end(s, b);
  const int64_t rel = u0 / s.kiters + j;            // split tile, relative
  const int64_t start = rel * s.kiters;
  const int64_t lo = (j == 0) ? u0 : start;
  const int64_t hi = (u1 < start + s.kiters) ? u1 : start + s.kiters;
  p.tile = s.dp_tiles + (int)rel;
  p.kb = (int)(lo - start);
  p.ke = (int)(hi - start);
  return p;
}

// For a split piece that holds the tile's first k-slice but not its last, the
// CTAs whose partial sums complete the tile are b+1, ..., b+count (in that
// order; each of them stored the partial in its own workspace slot).
SG_HD int num_contributors(const Schedule& s, int b, const Piece& p) {
  if (p.kb != 0 || p.ke == s.kiters || p.tile < s.dp_tiles) return 0;
  const int64_t tile_end = (int64_t)(p.tile - s.dp_tiles + 1) * s.kiters;
  int c = b + 1, n = 0;
  while (c < s.grid && sk_begin(s, c) < tile_end) {
    ++n;
    ++c;
  }
  return n;
}

// True for a split piece that starts inside its tile: its CTA stores a partial.
SG_HD bool is_partial_piece(const Schedule& s, const Piece& p) {
  return p.tile >= s.dp_tiles && p.kb != 0;
}

// How the tile space is decomposed (a per-shape-class choice of the tuner;
// every mode is exact and deterministic, they differ only in speed):
//   kSchedHybrid      whole tiles, then the last one to two waves' worth of
//                     tiles split into k-slice units (with fewer tiles than
//                     slots, everything is split);
//   kSchedHybridTail  whole waves of whole tiles; only the ragged last wave
//                     is split;
//   kSchedDataParallel whole tiles only, dealt round-robin;
//   kSchedStreamK     every tile split, the units spread evenly over the slots;
//   kSchedSplitK      every tile cut into `splits` equal k-ranges, one CTA each
//                     (capped at the slot count, beyond which it is stream-K).
// group_m is the raster group height; min_units the fewest k-slices worth
// giving one CTA when the hybrid and stream-K modes split.
enum SchedMode : int {
  kSchedHybrid = 0,
  kSchedHybridTail = 1,
  kSchedDataParallel = 2,
  kSchedStreamK = 3,
  kSchedSplitK = 4,
  kNumSchedModes = 5
};

struct SchedPolicy {
  int mode;       // SchedMode
  int group_m;    // raster group height in tiles (>= 1)
  int min_units;  // >= 1
  int splits;     // kSchedSplitK: k-ranges per tile (>= 1)
};

SG_HD bool policy_valid(const SchedPolicy& p) {
  return p.mode >= 0 && p.mode < kNumSchedModes && p.group_m >= 1 && p.min_units >= 1 &&
         p.splits >= 1;
}

// Host-side choice of the decomposition for a problem of batch x tiles_m x
// tiles_n tiles with kiters k-slices each on `capacity` resident CTA slots.
inline Schedule make_schedule(int tiles_m, int tiles_n, int kiters, int capacity,
                              const SchedPolicy& pol, int batch = 1) {
  Schedule s{};
  s.tiles_m = tiles_m;
  s.tiles_n = tiles_n;
  s.tiles = tiles_m * tiles_n * batch;
  s.kiters = kiters;
  s.group_m = pol.group_m < 1 ? 1 : (pol.group_m > tiles_m ? tiles_m : pol.group_m);
  if (s.group_m < 1) s.group_m = 1;
  const int T = s.tiles;
  const int P = capacity < 1 ? 1 : capacity;
  const int mu = pol.min_units < 1 ? 1 : pol.min_units;
  if (T == 0 || kiters == 0) {
    s.grid = 0;
    return s;
  }
  const int64_t units = (int64_t)T * kiters;
  auto whole = [&]() {
    s.grid = T < P ? T : P;
    s.dp_tiles = T;
  };
  // every tile split, over g CTAs (clamped to [1, P]; never more than units)
  auto split_all = [&](int64_t g) {
    g = g < 1 ? 1 : (g > P ? P : g);
    s.grid = (int)(g < units ? g : units);
    s.dp_tiles = 0;
  };
  switch (pol.mode) {
    case kSchedDataParallel:
      whole();
      break;
    case kSchedStreamK:
      split_all(units / mu);
      break;
    case kSchedSplitK: {
      const int sp = pol.splits < kiters ? pol.splits : kiters;
      split_all((int64_t)T * (sp < 1 ? 1 : sp));
      break;
    }
    case kSchedHybridTail:
    default:
      if (T % P == 0 || kiters < 2 * mu) {
        whole();  // nothing gained by splitting
      } else if (T >= P) {
        // keep whole waves (all but the last one-to-two, in the plain hybrid)
        s.grid = P;
        s.dp_tiles = (pol.mode == kSchedHybridTail ? T / P : T / P - 1) * P;
      } else {
        // fewer tiles than slots: split everything, at least mu units per CTA
        const int64_t g = units / mu;
        split_all(g < T ? T : g);
      }
      break;
  }
  s.sk_units = (int64_t)(T - s.dp_tiles) * kiters;
  s.sk_q = (int)(s.sk_units / s.grid);
  s.sk_r = (int)(s.sk_units % s.grid);
  return s;
}

}  // namespace sgemm_gb300
