// kvq_split.cuh -- the decode work list shared by the decode kernels: every
// (sequence b, KV head, key tile i) in order, cut into contiguous ranges, one
// per CTA ("stream-K"), so ragged lengths cost no load imbalance.  A segment
// is one (b, KV head); the run of a segment's tiles inside one CTA's range is
// a piece.
#pragma once

#include <cstdint>

namespace kvq {
namespace split {

// Position in the flat work list: sequence b, KV head, tile index i.
struct Cursor {
  int b, kvh, i;
};

// pre[b] = number of tiles of sequences 0 .. b-1 (per KV head).
__device__ __forceinline__ void advance(Cursor& c, const int32_t* pre, int B, int Hkv) {
  const int n = pre[c.b + 1] - pre[c.b];
  if (++c.i < n) return;
  c.i = 0;
  if (++c.kvh < Hkv) return;
  c.kvh = 0;
  do {
    ++c.b;
  } while (c.b < B && pre[c.b + 1] == pre[c.b]);
}

__device__ __forceinline__ Cursor locate(int64_t f, const int32_t* pre, int B, int Hkv) {
  // largest b with Hkv * pre[b] <= f; it is a non-empty sequence because f < Hkv * pre[B]
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (static_cast<int64_t>(Hkv) * pre[mid] <= f) lo = mid; else hi = mid - 1;
  }
  const int b = lo;
  const int n = pre[b + 1] - pre[b];
  const int64_t off = f - static_cast<int64_t>(Hkv) * pre[b];
  Cursor c;
  c.b = b;
  // off < Hkv * n: a 32-bit division unless that exceeds 32 bits
  if (off <= 0xFFFFFFFFll) {
    const uint32_t o32 = static_cast<uint32_t>(off), q = o32 / static_cast<uint32_t>(n);
    c.kvh = static_cast<int>(q);
    c.i = static_cast<int>(o32 - q * static_cast<uint32_t>(n));
  } else {
    c.kvh = static_cast<int>(off / n);
    c.i = static_cast<int>(off % n);
  }
  return c;
}

// Number of pieces in a CTA's tile range [f0, f0 + ntiles).
__device__ __forceinline__ int count_pieces(int64_t f0, int ntiles, const int32_t* pre, int B, int Hkv) {
  Cursor c = locate(f0, pre, B, Hkv);
  int left = ntiles, n = 0;
  while (left > 0) {
    const int nb = pre[c.b + 1] - pre[c.b];
    const int take = min(left, nb - c.i);
    left -= take;
    ++n;
    c.i = nb - 1;
    advance(c, pre, B, Hkv);
  }
  return n;
}

// The CTAs c0 .. c1 holding the first and the last tile of segment (b, kvh)
// when N tiles are split over C CTAs (CTA c owns [N c / C, N (c+1) / C)).
__device__ __forceinline__ void segment_ctas(const int32_t* pre, int Hkv, int b, int kvh, int64_t N, int C,
                                             int* c0, int* c1) {
  const int n_b = pre[b + 1] - pre[b];
  const int64_t start = static_cast<int64_t>(Hkv) * pre[b] + static_cast<int64_t>(kvh) * n_b;
  *c0 = static_cast<int>(((start + 1) * C - 1) / N);
  *c1 = static_cast<int>(((start + n_b) * C - 1) / N);
}

}  // namespace split
}  // namespace kvq
