// Work items of the chunk-parallel tensor-core kernels: one item is one head
// of one chunk, f = ((b * nc + c) * G + g) * hpg + jh, and a persistent grid
// gives CTA i the contiguous range [i * total / grid, (i + 1) * total / grid),
// so every SM gets the same number of heads and the heads of a chunk (which
// share its B, C and C B^T) follow one another.
#pragma once

namespace ssd {
namespace tc {

struct ItemGeom {
  int hpg, G, nc;
};

// Walks a CTA's items in order without divisions.
struct ItemCursor {
  int f, k, b, c, g, jh;  // item, chunk id (b * nc + c) * G + g, its batch, chunk, group and head in group
  __device__ __forceinline__ void seek(const ItemGeom& m, int f0) {
    f = f0;
    k = f0 / m.hpg;
    jh = f0 - k * m.hpg;
    g = k % m.G;
    const int bc = k / m.G;
    c = bc % m.nc;
    b = bc / m.nc;
  }
  __device__ __forceinline__ void next(const ItemGeom& m) {
    ++f;
    if (++jh == m.hpg) {
      jh = 0;
      ++k;
      if (++g == m.G) {
        g = 0;
        if (++c == m.nc) {
          c = 0;
          ++b;
        }
      }
    }
  }
  __device__ __forceinline__ int h(const ItemGeom& m) const { return g * m.hpg + jh; }
  // first / last item of this CTA's run on chunk k
  __device__ __forceinline__ bool first(int q0) const { return f == q0 || jh == 0; }
  __device__ __forceinline__ bool last(const ItemGeom& m, int q1) const { return f == q1 - 1 || jh == m.hpg - 1; }
};

// The CTA that owns item f.
__host__ __device__ __forceinline__ long long cta_of(long long f, long long total, long long grid) {
  return ((f + 1) * grid - 1) / total;
}

}  // namespace tc
}  // namespace ssd
