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
  int M, N, total_m, nt, n_ids, bn;
  LMOE_DEV TileWalk(const Tile* tiles_, const int* n_tiles, int M_, int N_, int bn_)
      : tiles(tiles_), M(M_), N(N_), bn(bn_) {
    total_m = tiles != nullptr ? *n_tiles : (M + kBM - 1) / kBM;
    nt = (N + bn - 1) / bn;
    n_ids = ((total_m + kRasterGroup - 1) / kRasterGroup) * kRasterGroup * nt;
  }
  // (expert, first row, rows, N tile) of tile id; false if the id is padding
  LMOE_DEV bool at(int id, int& expert, int& row0, int& nrows, int& ntile) const {
    int mt;
    return at(id, mt, expert, row0, nrows, ntile);
  }
  // same, also returning the M tile index (the row block of block-layout scales)
  LMOE_DEV bool at(int id, int& mt, int& expert, int& row0, int& nrows, int& ntile) const {
    if (!grouped_tile(id, total_m, nt, kRasterGroup, mt, ntile)) return false;
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

// Upper bound of the tile ids of a launch (host side): m_tiles M tiles of at most kBM rows.
inline long long tile_id_bound(int m_tiles, int N, int bn) {
  const long long nt = (N + bn - 1) / bn;
  return (m_tiles + kRasterGroup - 1) / kRasterGroup * kRasterGroup * nt;
}

}  // namespace lmoe
