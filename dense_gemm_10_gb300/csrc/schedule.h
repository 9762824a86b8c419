// schedule.h -- which output tiles and k-ranges each persistent CTA (or CTA
// pair) computes, and where split tiles keep their partial sums.  Plain C++
// shared by the kernels and the host planner.
//
// Two schedules:
//  * kSchedTiles: work units u = slot, slot + slots, ... over tiles x split_k;
//    split_k == 1 is one whole output tile per unit, split_k > 1 cuts each
//    tile's k-blocks into split_k ranges ("GPU GEMM 优化完全拆解（三）",
//    Split-K 与 Sliced-K).
//  * kSchedStreamK: the last sk_tiles tiles (those that would form an
//    incomplete last wave) are cut into sk_tiles * num_kb k-block iterations
//    that are dealt out in equal contiguous ranges, one per slot, so every
//    slot finishes at the same time; a range is cut again at tile edges.  Each
//    slot runs its share of those iterations first, then whole tiles
//    slot, slot + slots, ... of the first dp_tiles.  This removes the tail
//    effect of a last, partly filled wave ("CUDA GEMM 矩阵乘法优化指南", 12.5,
//    which names Stream-K as the cure for it).
// A strided batch of GEMMs shares one schedule: the tiles of batch b follow
// those of batch b - 1 (tile index = b * tiles_i * tiles_j + raster position),
// so whole tiles, split-K and stream-K treat the batch as one larger grid.
// Grouped GEMMs (groups > 0) do the same with a different row count per group:
// group g owns tiles [group_tile_start[g], group_tile_start[g + 1]).
// A tile split over several units is finished by whichever contribution
// arrives last: every contribution stores an fp32 partial, and the last one
// sums all partials in k order, so results do not depend on timing.
#pragma once

#include <cstdint>

#if defined(__CUDACC__)
#define G10_HD __host__ __device__ __forceinline__
#else
#define G10_HD inline
#endif

namespace g10 {

enum : int32_t { kSchedTiles = 0, kSchedStreamK = 1 };

struct Sched {
  int32_t tiles_i, tiles_j;  // output tiles along I and J (of one batch)
  int32_t batch;             // independent GEMMs sharing the schedule (>= 1)
  int32_t groups;            // > 0: grouped GEMMs, tile ranges in group_tile_start
  const int32_t* group_tile_start;  // groups + 1 prefix sums of tile_rows_g * tiles_j
  int32_t num_kb;            // k-blocks per tile
  int32_t raster_group;      // tile rows per raster group
  int32_t mode;              // kSchedTiles or kSchedStreamK
  int32_t split_k;           // kSchedTiles: k-ranges per tile
  int32_t dp_tiles;          // kSchedStreamK: tiles [0, dp_tiles) run whole
  int32_t sk_slots;          // kSchedStreamK: slots sharing the other tiles' k-blocks
  int64_t sk_iters;          // kSchedStreamK: (tiles - dp_tiles) * num_kb (>= sk_slots)
};

struct Unit {
  int32_t ti, tj, tile;  // output tile (raster position and linear index)
  int32_t tb;            // batch (or group) of the tile
  int32_t kb0, kb1;      // k-blocks [kb0, kb1) of the tile
  int32_t partial;       // 1: store an fp32 partial; the last contribution sums them
  int32_t pslot;         // partial slot of this contribution
  int32_t ctr;           // arrival counter of the tile
  int32_t ncontrib;      // contributions to the tile
  int32_t first_c;       // stream-K: slot of the tile's lowest-k contribution
  int32_t first_j;       // stream-K: which of that slot's two partial slots it used
};

// Output tiles of the whole schedule (every batch).
G10_HD int64_t sched_tiles(const Sched& s) {
  if (s.groups > 0) return s.group_tile_start[s.groups];
  return static_cast<int64_t>(s.tiles_i) * s.tiles_j * s.batch;
}

// Tile index -> (batch, ti, tj): within a batch, grouped raster order:
// raster_group tile rows at a time, walking down the rows of a group before
// moving one column right, so that tiles running together share rows of P and
// columns of Q in L2 ("GPU GEMM 优化完全拆解（三）", rasterization).
G10_HD void raster_tile(const Sched& s, int32_t tile, int32_t& ti, int32_t& tj, int32_t& tb) {
  int32_t tiles_i = s.tiles_i;
  if (s.groups > 0) {  // the group holding the tile: the last start <= tile
    int32_t lo = 0, hi = s.groups - 1;
    while (lo < hi) {
      const int32_t mid = (lo + hi + 1) / 2;
      if (s.group_tile_start[mid] <= tile) lo = mid;
      else hi = mid - 1;
    }
    tb = lo;
    tiles_i = (s.group_tile_start[lo + 1] - s.group_tile_start[lo]) / s.tiles_j;
    tile -= s.group_tile_start[lo];
  } else {
    const int32_t per_batch = s.tiles_i * s.tiles_j;
    tb = tile / per_batch;
    tile -= tb * per_batch;
  }
  const int32_t group_tiles = s.raster_group * s.tiles_j;
  const int32_t g = tile / group_tiles;
  const int32_t first_i = g * s.raster_group;
  const int32_t rows = (tiles_i - first_i) < s.raster_group ? (tiles_i - first_i) : s.raster_group;
  const int32_t r = tile - g * group_tiles;
  ti = first_i + r % rows;
  tj = r / rows;
}

// First stream-K iteration of slot c (slot c owns [sk_begin(c), sk_begin(c + 1))).
G10_HD int64_t sk_begin(const Sched& s, int32_t c) {
  return static_cast<int64_t>(c) * s.sk_iters / s.sk_slots;
}

// The slot whose range holds stream-K iteration x.
G10_HD int32_t sk_owner(const Sched& s, int64_t x) {
  return static_cast<int32_t>(((x + 1) * s.sk_slots - 1) / s.sk_iters);
}

// Number of partial slots the schedule needs.
G10_HD int64_t partial_slots(const Sched& s) {
  return s.mode == kSchedTiles ? sched_tiles(s) * s.split_k : static_cast<int64_t>(s.sk_slots) * 2;
}

// Partial slot of contribution k (k = 0 holds the lowest k-blocks) to w's tile.
G10_HD int32_t contrib_slot(const Sched& s, const Unit& w, int32_t k) {
  if (s.mode == kSchedTiles) return w.tile * s.split_k + k;
  return (w.first_c + k) * 2 + (k == 0 ? w.first_j : 0);
}

struct WorkIter {
  Sched s;            // a copy: on the device it stays in registers
  int32_t slot, slots;
  int32_t phase;      // stream-K: 0 = this slot's k-range share, 1 = whole tiles
  int64_t x, x_end;   // stream-K iteration cursor
  int32_t u;          // unit cursor
  int32_t nseg;       // stream-K segments produced so far

  G10_HD WorkIter(const Sched& sc, int32_t slot_, int32_t slots_)
      : s(sc), slot(slot_), slots(slots_), phase(0), x(0), x_end(0), u(slot_), nseg(0) {
    if (sc.mode == kSchedStreamK && slot_ < sc.sk_slots) {
      x = sk_begin(sc, slot_);
      x_end = sk_begin(sc, slot_ + 1);
    }
  }

  G10_HD bool next(Unit& w) {
    const Sched& S = s;
    if (S.mode == kSchedTiles) {
      const int32_t units = static_cast<int32_t>(sched_tiles(S)) * S.split_k;
      if (u >= units) return false;
      w.tile = u / S.split_k;
      const int32_t k = u - w.tile * S.split_k;
      w.kb0 = static_cast<int32_t>(static_cast<int64_t>(k) * S.num_kb / S.split_k);
      w.kb1 = static_cast<int32_t>(static_cast<int64_t>(k + 1) * S.num_kb / S.split_k);
      w.partial = S.split_k > 1 ? 1 : 0;
      w.pslot = u;
      w.ctr = w.tile;
      w.ncontrib = S.split_k;
      w.first_c = 0;
      w.first_j = 0;
      raster_tile(S, w.tile, w.ti, w.tj, w.tb);
      u += slots;
      return true;
    }
    if (phase == 0) {
      if (x < x_end) {
        const int64_t q = x / S.num_kb;
        const int64_t t0 = q * S.num_kb;
        const int64_t end = x_end < t0 + S.num_kb ? x_end : t0 + S.num_kb;
        w.tile = S.dp_tiles + static_cast<int32_t>(q);
        w.kb0 = static_cast<int32_t>(x - t0);
        w.kb1 = static_cast<int32_t>(end - t0);
        const int32_t c_first = sk_owner(S, t0);
        const int32_t c_last = sk_owner(S, t0 + S.num_kb - 1);
        w.partial = c_first != c_last ? 1 : 0;
        w.pslot = slot * 2 + (nseg == 0 ? 0 : 1);  // a slot's first / last range piece
        w.ctr = static_cast<int32_t>(q);
        w.ncontrib = c_last - c_first + 1;
        w.first_c = c_first;
        w.first_j = sk_begin(S, c_first) < t0 ? 1 : 0;
        raster_tile(S, w.tile, w.ti, w.tj, w.tb);
        ++nseg;
        x = end;
        return true;
      }
      phase = 1;
    }
    if (u >= S.dp_tiles) return false;
    w.tile = u;
    w.kb0 = 0;
    w.kb1 = S.num_kb;
    w.partial = 0;
    w.pslot = 0;
    w.ctr = 0;
    w.ncontrib = 1;
    w.first_c = 0;
    w.first_j = 0;
    raster_tile(S, w.tile, w.ti, w.tj, w.tb);
    u += slots;
    return true;
  }
};

}  // namespace g10
