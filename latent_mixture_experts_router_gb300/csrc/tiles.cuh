// tiles.cuh — the output-tile sequence of the persistent GEMMs.
#pragma once
#include "internal.h"
#include "ptx.cuh"

namespace lmoe {

// Split count of a grouped GEMM with `units` output tiles on `grid` persistent CTAs: the
// smallest divisor of num_kb (at most max_splits, and leaving every split at least
// kMinSplitKb K blocks: a short unit costs more in pipeline refill than it gains in balance)
// whose last wave is best filled, when the tiles alone fill fewer than three waves.
// Split-K pays a partial write and a reduce pass, so it is offered only where the A rows are
// few (the host bounds max_splits).
constexpr int kMinSplitKb = 8;
__host__ __device__ inline int choose_splits(int units, int num_kb, int grid, int max_splits) {
  if (max_splits <= 1 || units <= 0 || units >= 3 * grid) return 1;
  const int w1 = (units + grid - 1) / grid;
  float best_eff = static_cast<float>(units) / static_cast<float>(w1 * grid);
  int best = 1;
  for (int s = 2; s <= max_splits && s * kMinSplitKb <= num_kb; ++s) {
    if (num_kb % s) continue;
    const int u = units * s, waves = (u + grid - 1) / grid;
    const float eff = static_cast<float>(u) / static_cast<float>(waves * grid);
    if (eff > best_eff + 0.02f) {
      best = s;
      best_eff = eff;
    }
  }
  return best;
}

// Every role of a CTA walks tile ids blockIdx.x, + gridDim.x, ... over the grouped raster
// of (M tile, N tile); ids in the padding of the last raster group are skipped by all roles
// alike.  Grouped GEMMs take their M tiles from the device tile table.
struct TileWalk {
  const Tile* tiles;
  int M, N, total_m, nt, n_ids, bn, splits, num_kb, kb_per_split;
  int bm;   // rows of a dense M tile (a grouped table's tiles carry their own row counts)
  // splits > 1: every output tile is computed as `splits` partial products over disjoint K
  // ranges (split-K), consecutive ids taking the K ranges of one tile
  // adaptive (grouped only): splits_ is the upper bound, the count comes from choose_splits
  LMOE_DEV TileWalk(const Tile* tiles_, const int* n_tiles, int M_, int N_, int bn_, int splits_ = 1,
                    int num_kb_ = 1, bool adaptive = false, int bm_ = kBM)
      : TileWalk(tiles_, tiles_ != nullptr ? *n_tiles : (M_ + bm_ - 1) / bm_, M_, N_, bn_, splits_,
                 num_kb_, adaptive, bm_) {}
  // same, with the live M-tile count given
  LMOE_DEV TileWalk(const Tile* tiles_, int total_m_, int M_, int N_, int bn_, int splits_, int num_kb_,
                    bool adaptive, int bm_ = kBM)
      : tiles(tiles_), M(M_), N(N_), bn(bn_), splits(splits_ < 1 ? 1 : splits_), num_kb(num_kb_), bm(bm_) {
    total_m = total_m_;
    nt = (N + bn - 1) / bn;
    if (adaptive && tiles != nullptr)
      splits = choose_splits(total_m * nt, num_kb, static_cast<int>(gridDim.x), splits);
    n_ids = ((total_m + kRasterGroup - 1) / kRasterGroup) * kRasterGroup * nt * splits;
    kb_per_split = (num_kb + splits - 1) / splits;
  }
  // K blocks [kb0, kb1) of tile id (all of K without split-K)
  LMOE_DEV void k_range(int id, int& kb0, int& kb1) const {
    const int ks = id % splits;
    kb0 = ks * kb_per_split;
    kb1 = min(num_kb, kb0 + kb_per_split);
  }
  // (expert, first row, rows, N tile) of tile id; false if the id is padding
  LMOE_DEV bool at(int id, int& expert, int& row0, int& nrows, int& ntile) const {
    int mt;
    return at(id, mt, expert, row0, nrows, ntile);
  }
  // same, also returning the M tile index (the row block of block-layout scales)
  LMOE_DEV bool at(int id, int& mt, int& expert, int& row0, int& nrows, int& ntile) const {
    if (!grouped_tile(id / splits, total_m, nt, kRasterGroup, mt, ntile)) return false;
    int kb0, kb1;
    k_range(id, kb0, kb1);
    if (kb0 >= kb1) return false;
    if (tiles != nullptr) {
      const Tile t = tiles[mt];
      expert = t.expert;
      row0 = t.row0;
      nrows = t.nrows;
    } else {
      expert = 0;
      row0 = mt * bm;
      nrows = min(bm, M - row0);
    }
    return nrows > 0;
  }
};

// A tile id resolved to its raster position (arithmetic only; the tile-table entry is
// loaded separately, so that a producer can issue that load one tile ahead).
struct TileRef {
  int id, mt, ntile;
  bool valid;
};
LMOE_DEV TileRef find_tile(const TileWalk& w, int from) {
  for (int id = from; id < w.n_ids; id += gridDim.x) {
    int mt, nt_;
    if (!grouped_tile(id / w.splits, w.total_m, w.nt, kRasterGroup, mt, nt_)) continue;
    int kb0, kb1;
    w.k_range(id, kb0, kb1);
    if (kb0 < kb1) return TileRef{id, mt, nt_, true};
  }
  return TileRef{w.n_ids, 0, 0, false};
}
LMOE_DEV Tile tile_of(const TileWalk& w, int mt) {
  if (w.tiles != nullptr) return w.tiles[mt];
  return Tile{0, mt * w.bm, min(w.bm, w.M - mt * w.bm), 0};
}

// This CTA's first weight tile, for an L2 prefetch issued before the CTA waits on the previous
// kernel.  A grouped GEMM's tile table is written by an earlier kernel of the stream, so it
// is read here with relaxed gpu-scope loads as a hint only: every index is clamped into the
// table and the expert count, and the tiles the GEMM computes come from the walk it builds
// after the wait.  Returns false if there is nothing to prefetch.
LMOE_DEV int ld_relaxed_gpu(const int* p) {
  int v;
  asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
LMOE_DEV bool first_tile_hint(const Tile* tiles, const int* n_tiles, int max_tiles, int n_groups, int M,
                              int N, int bn, int splits, int num_kb, bool adaptive, int& brow, int& kb0,
                              int& kb1, int bm = kBM) {
  int total_m;
  if (tiles != nullptr) {
    total_m = min(max(ld_relaxed_gpu(n_tiles), 0), max_tiles);
  } else {
    total_m = (M + bm - 1) / bm;
  }
  const TileWalk w(tiles, total_m, M, N, bn, splits, num_kb, adaptive, bm);
  int mt, nt_;
  if (static_cast<int>(blockIdx.x) >= w.n_ids ||
      !grouped_tile(static_cast<int>(blockIdx.x) / w.splits, w.total_m, w.nt, kRasterGroup, mt, nt_))
    return false;
  // dense: the group's M tiles share one weight tile, which its first CTA warms; grouped: the
  // M tiles of a group mostly belong to different experts, so every CTA warms its own
  if (tiles == nullptr && mt % kRasterGroup != 0) return false;
  int expert = 0;
  if (tiles != nullptr) {
    expert = ld_relaxed_gpu(&tiles[mt].expert);
    if (expert < 0 || expert >= n_groups) return false;
  }
  w.k_range(blockIdx.x, kb0, kb1);
  brow = expert * N + nt_ * bn;
  return kb0 < kb1;
}

// Host side: whether a grouped GEMM whose live M-tile count lies in [lo, hi] can pick a split
// count above 1 (if not, it runs unsplit and no reduce pass is launched).
inline bool grouped_split_possible(int lo, int hi, int nt, int num_kb, int grid, int max_splits) {
  for (int m = lo < 1 ? 1 : lo; m <= hi; ++m)
    if (choose_splits(m * nt, num_kb, grid, max_splits) > 1) return true;
  return false;
}

// Upper bound of the tile ids of a launch (host side): m_tiles M tiles of at most kBM rows.
inline long long tile_id_bound(int m_tiles, int N, int bn, int splits = 1) {
  const long long nt = (N + bn - 1) / bn;
  return (m_tiles + kRasterGroup - 1) / kRasterGroup * kRasterGroup * nt * splits;
}

}  // namespace lmoe
