// The backward's query-tile walk, shared by the dK/dV kernel and the host
// build of the tests.
#pragma once

#include "ring_iter.cuh"

namespace ra {

// The query tiles that see key rows [kv_lo, kv_hi], in ring order: query
// heads [h, h_end) of the group, then ring steps t = 0..P-1 (rank src + t),
// the rank's segments in position order, tiles in order. Under the causal
// rule a tile whose last query precedes the first key sees nothing; since
// positions grow along a segment, such tiles form a prefix of it.
struct QTile {
  int h, seg, ti, lo, valid;
  bool mask;    // some (query, key) pair of the tile is masked
};

template <int kT>
struct QIterT {
  int h, h_end, t, r, which, ti, ti_end, len, src, kv_lo, kv_hi;

  __device__ __forceinline__ void start_segment(const Geometry& g) {
    const int seg = rank_seg(g, r, which);
    const int s0 = seg * g.seg_len;
    len = seg_tokens(g, seg);
    ti_end = (len + kT - 1) / kT;               // tiles holding tokens
    if (!g.causal || kv_lo <= s0) ti = 0;
    else if (s0 + len - 1 < kv_lo) ti = ti_end;
    else ti = (kv_lo - s0) / kT;
  }
  __device__ __forceinline__ void init(const Geometry& g, int src_, int kv_lo_, int kv_valid,
                                       int h_begin, int h_end_) {
    h = h_begin;
    h_end = kv_valid > 0 ? h_end_ : h_begin;   // a key tile of padding only: no visit
    src = src_; t = 0; r = src_; which = 0;
    kv_lo = kv_lo_; kv_hi = kv_lo_ + kv_valid - 1;
    start_segment(g);
  }
  __device__ __forceinline__ bool next(const Geometry& g, QTile& o) {
    while (h < h_end) {
      if (ti < ti_end) {
        const int seg = rank_seg(g, r, which);
        o.h = h;
        o.seg = seg;
        o.ti = ti;
        o.lo = seg * g.seg_len + ti * kT;
        o.valid = min(kT, len - ti * kT);
        o.mask = g.causal && kv_hi > o.lo;
        ++ti;
        return true;
      }
      if (++which >= g.segs_per_rank) {
        which = 0;
        if (++t >= g.P) { t = 0; ++h; }
        r = src + t;
        if (r >= g.P) r -= g.P;
      }
      if (h < h_end) start_segment(g);
    }
    return false;
  }
};

}  // namespace ra
