// tiles.cuh — the output-tile sequence of the persistent GEMMs.
#pragma once
#include "internal.h"
#include "ptx.cuh"

namespace lmoe {

// Every role of a CTA walks tile ids blockIdx.x, + gridDim.x, ... over the grouped raster
// of (M tile, N tile); ids in the padding of the last raster group are skipped by all roles
// alike.  Grouped GEMMs take their M tiles from the device tile table.
struct TileWalk {
  const Tile* tiles;
  int M, N, total_m, nt, n_ids, bn, splits, num_kb, kb_per_split;
  // splits > 1: every output tile is computed as `splits` partial products over disjoint K
  // ranges (split-K), consecutive ids taking the K ranges of one tile
  LMOE_DEV TileWalk(const Tile* tiles_, const int* n_tiles, int M_, int N_, int bn_, int splits_ = 1,
                    int num_kb_ = 1)
      : tiles(tiles_), M(M_), N(N_), bn(bn_), splits(splits_ < 1 ? 1 : splits_), num_kb(num_kb_) {
    total_m = tiles != nullptr ? *n_tiles : (M + kBM - 1) / kBM;
    nt = (N + bn - 1) / bn;
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
      row0 = mt * kBM;
      nrows = min(kBM, M - row0);
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
  return Tile{0, mt * kBM, min(kBM, w.M - mt * kBM), 0};
}

// Upper bound of the tile ids of a launch (host side): m_tiles M tiles of at most kBM rows.
inline long long tile_id_bound(int m_tiles, int N, int bn, int splits = 1) {
  const long long nt = (N + bn - 1) / bn;
  return (m_tiles + kRasterGroup - 1) / kRasterGroup * kRasterGroup * nt * splits;
}

}  // namespace lmoe
