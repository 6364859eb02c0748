// Persistent tile scheduler of the tensor-core kernels: maps a linear tile
// index to (matrix, row tile, column tile).  Used by the kernels and by the
// host-side helper muon_ns_tile_coords(), so both walk the same order.
//
// Output tiles are kTileM x kTileN = 128 x 256.  A launch covers the flattened
// (matrix, tile) space of a whole stack, matrix-major, so a stack of small
// expert matrices fills every SM (the leading axis is the batch: prime-rl PR
// #3873, Summary item 2).
//
// Lower triangle (Gram and polynomial products, output m x m, symmetric):
// row tile I (128 rows) and column tile J (256 columns) are needed iff some
// (i, j) with j <= i lies in the tile, i.e. J <= floor(I / 2).  Rows 2p and
// 2p+1 each hold p + 1 tiles, so rows 0..2p-1 hold p (p + 1) tiles; when the
// number of row tiles is odd the last row (I = 2T - 1) does not exist.  The
// triangle is walked in groups of kGroupT row tiles, column-major inside a
// group, so CTAs running at the same time read a band of A-operand rows and a
// limited set of B-operand column panels (the operand of a large matrix
// would otherwise be re-streamed from DRAM by every wave).
//
// Full grid (update product): groups of kGroupM row tiles are walked
// column-major inside the group, so CTAs running at the same time share
// operand panels in L2.
//
// Paired spaces (kernels launched as clusters of two CTAs that share the
// B-operand panel of a column tile through TMA multicast): a unit of the
// space is a pair of row tiles (2p, 2p + 1) with one column tile J; CTA rank r
// of the cluster computes row tile 2p + r.  For the triangle, both row tiles
// of a pair hold the column tiles J <= p, so the pairs form the plain lower
// triangle J <= p of ceil(tiles_m / 2) pair rows.  A row tile 2p + 1 beyond
// the last row tile (odd tiles_m) is computed on zero-filled operands and
// not stored.
#pragma once

#include <cstdint>

#ifdef __CUDACC__
#define MNS_HD __host__ __device__ __forceinline__
#else
#define MNS_HD inline
#endif

namespace mns {

constexpr int kTileM = 128;
constexpr int kTileN = 256;
constexpr int kGroupM = 8;
#ifndef MNS_TRI_GROUP
#define MNS_TRI_GROUP 16
#endif
constexpr int kGroupT = MNS_TRI_GROUP;  // row tiles per group of the triangle walk

MNS_HD int ceil_div_i(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

// Number of lower-triangle tiles of one m x m output with `tiles_m` row tiles.
MNS_HD long long tri_tiles(int tiles_m) {
  const long long T = (tiles_m + 1) / 2;
  return (tiles_m & 1) ? T * T : T * (T + 1);
}

// Tiles in row tiles [0, x) of the triangle: x = 2p -> p (p + 1), x = 2p + 1 -> (p + 1)^2.
MNS_HD long long tri_rows_tiles(long long x) {
  const long long p = x / 2;
  return (x & 1) ? (p + 1) * (p + 1) : p * (p + 1);
}

// Local triangle index u -> (I, J), grouped walk (groups of kGroupT row tiles,
// column-major inside a group).
MNS_HD void tri_decode_grouped(long long u, int tiles_m, int* I, int* J) {
  long long r0 = 0;
  while (true) {
    const long long r1 = (r0 + kGroupT < tiles_m) ? r0 + kGroupT : tiles_m;
    const long long cnt = tri_rows_tiles(r1) - tri_rows_tiles(r0);
    if (u < cnt || r1 >= tiles_m) {
      for (long long j = 0;; ++j) {
        const long long first = (2 * j > r0) ? 2 * j : r0;
        const long long n = r1 - first;
        if (u < n) {
          *I = static_cast<int>(first + u);
          *J = static_cast<int>(j);
          return;
        }
        u -= n;
      }
    }
    u -= cnt;
    r0 = r1;
  }
}

// Local index u of the paired triangle (pair rows p, J <= p) -> (p, J),
// grouped walk (groups of kGroupT / 2 pair rows, column-major inside a group).
MNS_HD void ptri_decode_grouped(long long u, int pair_rows, int* p, int* J) {
  constexpr long long kG = kGroupT / 2 > 0 ? kGroupT / 2 : 1;
  long long r0 = 0;
  while (true) {
    const long long r1 = (r0 + kG < pair_rows) ? r0 + kG : pair_rows;
    const long long cnt = r1 * (r1 + 1) / 2 - r0 * (r0 + 1) / 2;
    if (u < cnt || r1 >= pair_rows) {
      for (long long j = 0;; ++j) {
        const long long first = j > r0 ? j : r0;
        const long long n = r1 - first;
        if (u < n) {
          *p = static_cast<int>(first + u);
          *J = static_cast<int>(j);
          return;
        }
        u -= n;
      }
    }
    u -= cnt;
    r0 = r1;
  }
}

// Local full-grid index u -> (I, J), grouped raster.
MNS_HD void grid_decode(long long u, int tiles_m, int tiles_n, int* I, int* J,
                        int group = kGroupM) {
  const long long per_group = static_cast<long long>(group) * tiles_n;
  const long long g = u / per_group;
  const long long r = u - g * per_group;
  const long long first = g * group;
  long long rows = tiles_m - first;
  if (rows > group) rows = group;
  *I = static_cast<int>(first + r % rows);
  *J = static_cast<int>(r / rows);
}

struct TileSpace {
  int sym;          // 1: lower triangle, 0: full grid
  int pair;         // 1: units are pairs of row tiles (clusters of two CTAs)
  int tiles_m;      // row tiles per matrix
  int tiles_n;      // column tiles per matrix
  long long per_matrix;  // units per matrix
  long long total;
};

MNS_HD TileSpace make_tile_space(int sym, int batch, int M, int N, int pair = 0) {
  TileSpace s;
  s.sym = sym;
  s.pair = pair;
  s.tiles_m = ceil_div_i(M, kTileM);
  s.tiles_n = ceil_div_i(N, kTileN);
  const long long pr = (s.tiles_m + 1) / 2;
  if (pair)
    s.per_matrix = sym ? pr * (pr + 1) / 2 : pr * s.tiles_n;
  else
    s.per_matrix = sym ? tri_tiles(s.tiles_m) : static_cast<long long>(s.tiles_m) * s.tiles_n;
  s.total = s.per_matrix * batch;
  return s;
}

// Unit t -> (matrix b, row tile I, column tile J); for a paired space I is
// the pair row p (the CTAs compute row tiles 2p and 2p + 1).
MNS_HD void tile_decode(const TileSpace& s, long long t, int* b, int* I, int* J) {
  const long long bb = t / s.per_matrix;
  const long long u = t - bb * s.per_matrix;
  *b = static_cast<int>(bb);
  if (s.pair) {
    const int pr = (s.tiles_m + 1) / 2;
    if (s.sym)
      ptri_decode_grouped(u, pr, I, J);
    else
      grid_decode(u, pr, s.tiles_n, I, J, kGroupM / 2);
  } else if (s.sym) {
    tri_decode_grouped(u, s.tiles_m, I, J);
  } else {
    grid_decode(u, s.tiles_m, s.tiles_n, I, J);
  }
}

}  // namespace mns
