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
#pragma once

#include <cmath>
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

// Local triangle index u -> (I, J).
MNS_HD void tri_decode(long long u, int* I, int* J) {
  // p = largest integer with p (p + 1) <= u.
  long long p = static_cast<long long>((sqrtf(4.0f * static_cast<float>(u) + 1.0f) - 1.0f) * 0.5f);
  if (p < 0) p = 0;
  while (p > 0 && p * (p + 1) > u) --p;
  while ((p + 1) * (p + 2) <= u) ++p;
  const long long v = u - p * (p + 1);
  if (v <= p) {
    *I = static_cast<int>(2 * p);
    *J = static_cast<int>(v);
  } else {
    *I = static_cast<int>(2 * p + 1);
    *J = static_cast<int>(v - (p + 1));
  }
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

// Local full-grid index u -> (I, J), grouped raster.
MNS_HD void grid_decode(long long u, int tiles_m, int tiles_n, int* I, int* J) {
  const long long per_group = static_cast<long long>(kGroupM) * tiles_n;
  const long long g = u / per_group;
  const long long r = u - g * per_group;
  const long long first = g * kGroupM;
  long long rows = tiles_m - first;
  if (rows > kGroupM) rows = kGroupM;
  *I = static_cast<int>(first + r % rows);
  *J = static_cast<int>(r / rows);
}

struct TileSpace {
  int sym;          // 1: lower triangle, 0: full grid
  int tiles_m;      // row tiles per matrix
  int tiles_n;      // column tiles per matrix
  long long per_matrix;
  long long total;
};

MNS_HD TileSpace make_tile_space(int sym, int batch, int M, int N) {
  TileSpace s;
  s.sym = sym;
  s.tiles_m = ceil_div_i(M, kTileM);
  s.tiles_n = ceil_div_i(N, kTileN);
  s.per_matrix = sym ? tri_tiles(s.tiles_m) : static_cast<long long>(s.tiles_m) * s.tiles_n;
  s.total = s.per_matrix * batch;
  return s;
}

MNS_HD void tile_decode(const TileSpace& s, long long t, int* b, int* I, int* J) {
  const long long bb = t / s.per_matrix;
  const long long u = t - bb * s.per_matrix;
  *b = static_cast<int>(bb);
  if (s.sym)
    tri_decode_grouped(u, s.tiles_m, I, J);
  else
    grid_decode(u, s.tiles_m, s.tiles_n, I, J);
}

}  // namespace mns
