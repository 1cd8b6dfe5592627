// Work decomposition of one GEMM call over the persistent workers (one
// worker = one CTA, or one CTA pair for pair MMAs). Compiled for host and
// device: every role of every CTA walks the same deterministic sequence of
// units, and the host tests check that the units cover every (tile, k-block)
// exactly once.
//
// Three modes (and a mix of two), following "SASS-Level Kernel Generation for Blackwell"
// (sections "The numbers" and "Inside the kernels", paragraph "Stream-K and
// split-K, added in the L2"):
//  * data parallel: one unit per output tile, tiles taken by stride in
//    grouped raster order (groups of `group` tile rows);
//  * split-K: K of every tile split `splits` ways into contiguous k-block
//    ranges whose sizes differ by at most one; the tile's CTAs zero it first
//    and then each adds its whole partial into C;
//  * stream-K: the (tile, k-block) iterations of all tiles, tile-major, are
//    cut into one contiguous, near-equal range per worker; the unit holding a
//    tile's first k-block stores it and raises the tile's flag, the others add
//    to it once the flag is up. A worker walks its range from the end, so its
//    first unit is the one that owns a tile start: no owner waits behind a
//    unit that waits;
//  * data-parallel waves with a stream-K tail: the leading `dp_tiles` tiles
//    (whole waves, one tile per worker per wave) run data parallel, and the
//    tiles left over are shared out by stream-K over the same workers, after
//    their data-parallel units. The page's stream-K spreads all tiles; this
//    mix splits only the partial last wave (or the last few waves), so that
//    the reduce-adds stay few when tiles outnumber workers;
//  * stream-K with zeroing first (`zero_first`): the same ranges as
//    stream-K, with the fix-up of split-K. The unit holding a tile's first
//    k-block zeroes the tile when its CTA starts and raises the tile's flag;
//    every unit of the tile, that one included, adds its partial into C once
//    the flag is up. No unit waits on another unit's main loop.
#pragma once
#include <stdint.h>

#if defined(__CUDACC__)
#define WG_PLAN_HD __host__ __device__ __forceinline__
#else
#define WG_PLAN_HD inline
#endif

namespace wg {

// kHybridK and kStreamKZero are host-side requests: their plans run as
// kStreamK (with dp_tiles > 0, or with zero_first = 1).
enum PlanMode : int32_t { kDataParallel = 0, kSplitK = 1, kStreamK = 2, kHybridK = 3,
                          kStreamKZero = 4 };

// What the epilogue does with a unit's accumulator.
enum UnitKind : int32_t {
  kUnitStore = 0,        // whole K of the tile: plain store
  kUnitStoreRaise = 1,   // stream-K: owns the tile's first k-block: store, then raise the flag
  kUnitAddAfterOwner = 2,// stream-K: add into C once the owner's flag is up
  kUnitAddAfterZero = 3, // split-K, and a zero-first stream-K owner: zero this unit's slice
                         // of the tile first; add into C once every slice of the tile is zeroed
  kUnitAddAfterZeroed = 4,  // zero-first stream-K: add into C once the tile is zeroed
};

struct Plan {
  int32_t M, N, K;
  int32_t tile_rows;    // C rows of one worker tile
  int32_t tile_cols;    // C columns of one worker tile
  int32_t tiles_m, tiles_n, num_tiles;
  int32_t kblocks;      // ceil(K / 64)
  int32_t mode;         // PlanMode
  int32_t splits;       // split-K ways (1 otherwise)
  int32_t group;        // raster group (tile rows per group)
  int32_t workers;      // persistent workers in the grid (clusters launched, with CLC)
  int32_t sched;        // 0: static stride; 1: cluster launch control (tiles taken at run time)
  int32_t dp_tiles;     // stream-K: leading tiles run data parallel (a multiple of workers)
  int64_t total_iters;  // stream-K: (num_tiles − dp_tiles) · kblocks
  int32_t zero_first;   // stream-K: 1 = owners zero the tile first and every unit adds
  int32_t pad_;
};

struct Unit {
  int32_t tile, tm, tn;
  int32_t kb_begin, kb_end;  // k-block range [kb_begin, kb_end)
  int32_t kind;              // UnitKind
  int32_t split;             // split index (split-K), else 0
};

// Tile t → (tm, tn): consecutive t walk down a column of `group` tile rows,
// then move one tile column right.
WG_PLAN_HD void plan_tile_coords(const Plan& p, int32_t t, int32_t& tm, int32_t& tn) {
  const int32_t per_group = p.group * p.tiles_n;
  const int32_t g = t / per_group;
  const int32_t first_m = g * p.group;
  const int32_t rows_left = p.tiles_m - first_m;
  const int32_t gm = rows_left < p.group ? rows_left : p.group;
  const int32_t local = t - g * per_group;
  tm = first_m + local % gm;
  tn = local / gm;
  // With cluster launch control the tiles of a group run in serpentine order:
  // every other column of the group walks its rows bottom-up, so consecutive
  // tiles stay adjacent (and share operand panels) across column boundaries.
  if (p.sched == 1 && (tn & 1)) tm = first_m + (gm - 1 - local % gm);
}

// The data-parallel unit of tile t (its whole K range).
WG_PLAN_HD void plan_tile_unit(const Plan& p, int32_t t, Unit& u) {
  u.tile = t;
  plan_tile_coords(p, t, u.tm, u.tn);
  u.kb_begin = 0;
  u.kb_end = p.kblocks;
  u.kind = kUnitStore;
  u.split = 0;
}

// The i-th unit of worker w; false when w has no i-th unit. With cluster
// launch control a worker's first unit is its own tile and the rest are only
// known at run time, so this lists just the first.
WG_PLAN_HD bool plan_unit(const Plan& p, int32_t w, int32_t i, Unit& u) {
  if (p.sched == 1) {
    if (i > 0 || w >= p.num_tiles) return false;
    plan_tile_unit(p, w, u);
    return true;
  }
  if (p.mode == kStreamK) {
    // Data-parallel waves first: worker w's tiles w, w + P, … below dp_tiles.
    const int32_t dp_waves = p.dp_tiles / p.workers;
    if (i < dp_waves) {
      plan_tile_unit(p, w + i * p.workers, u);
      return true;
    }
    i -= dp_waves;
    const int64_t T = p.total_iters, P = p.workers;
    const int64_t b = (T * w) / P, e = (T * (w + 1)) / P;
    if (e <= b) return false;
    const int64_t kb = p.kblocks;
    const int64_t t = (e - 1) / kb - i;  // walk tiles downwards from the range end
    if (t < 0 || (t + 1) * kb <= b) return false;
    const int64_t s0 = t * kb > b ? t * kb : b;
    const int64_t s1 = (t + 1) * kb < e ? (t + 1) * kb : e;
    u.tile = p.dp_tiles + (int32_t)t;
    plan_tile_coords(p, u.tile, u.tm, u.tn);
    u.kb_begin = (int32_t)(s0 - t * kb);
    u.kb_end = (int32_t)(s1 - t * kb);
    u.split = 0;
    if (u.kb_begin == 0 && u.kb_end == p.kblocks) u.kind = kUnitStore;
    else if (p.zero_first) u.kind = u.kb_begin == 0 ? kUnitAddAfterZero : kUnitAddAfterZeroed;
    else if (u.kb_begin == 0) u.kind = kUnitStoreRaise;
    else u.kind = kUnitAddAfterOwner;
    return true;
  }
  const int64_t idx = (int64_t)w + (int64_t)i * p.workers;
  if (p.mode == kSplitK) {
    const int64_t S = p.splits;
    if (idx >= (int64_t)p.num_tiles * S) return false;
    u.tile = (int32_t)(idx / S);
    u.split = (int32_t)(idx % S);
    plan_tile_coords(p, u.tile, u.tm, u.tn);
    u.kb_begin = (int32_t)(((int64_t)u.split * p.kblocks) / S);
    u.kb_end = (int32_t)(((int64_t)(u.split + 1) * p.kblocks) / S);
    u.kind = kUnitAddAfterZero;
    return true;
  }
  if (idx >= p.num_tiles) return false;
  plan_tile_unit(p, (int32_t)idx, u);
  return true;
}

// plan_unit for kernels that never split K (the host gives them data-parallel
// plans only): the same units without the split-K and stream-K arithmetic.
WG_PLAN_HD bool plan_unit_dp(const Plan& p, int32_t w, int32_t i, Unit& u) {
  if (p.sched == 1) {
    if (i > 0 || w >= p.num_tiles) return false;
    plan_tile_unit(p, w, u);
    return true;
  }
  const int32_t idx = w + i * p.workers;
  if (idx >= p.num_tiles) return false;
  plan_tile_unit(p, idx, u);
  return true;
}

// Rows [r0, r1) of a tile's `tile_rows` that split `s` of `S` zeroes.
WG_PLAN_HD void plan_zero_rows(int32_t tile_rows, int32_t S, int32_t s, int32_t& r0, int32_t& r1) {
  const int32_t per = (tile_rows + S - 1) / S;
  r0 = s * per < tile_rows ? s * per : tile_rows;
  r1 = (s + 1) * per < tile_rows ? (s + 1) * per : tile_rows;
}

}  // namespace wg
