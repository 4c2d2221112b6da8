// Device-side ring bookkeeping shared by the attention kernels.
//
// Glossary "sequence parallelism transformers", §Ring Attention: at step t
// virtual rank r holds the key/value block that started on rank
// (r - t) mod P; after P steps every block has been visited once. A block is
// one segment (contiguous order) or two halves (zig-zag order: rank r owns
// halves r and 2P-1-r, §Implementation Considerations "Load Balancing").
//
// Every role of a kernel walks the same sequence with KvIter, so producer,
// MMA issuer and softmax threads agree on the visit order without talking.
#pragma once

#include "ra_internal.h"

namespace ra {

// Rank owning segment g (segments numbered in position order).
__device__ __forceinline__ int seg_owner(const Geometry& g, int seg) {
  if (g.order == RA_ORDER_CONTIGUOUS) return seg;
  return seg < g.P ? seg : 2 * g.P - 1 - seg;
}

// The `which`-th segment (ascending position) of rank r.
__device__ __forceinline__ int rank_seg(const Geometry& g, int r, int which) {
  if (g.order == RA_ORDER_CONTIGUOUS) return r;
  return which == 0 ? r : 2 * g.P - 1 - r;
}

struct KvTile {
  int step;     // ring step t
  int src;      // rank the block started on
  int id;       // global tile id = segment * nt + index in segment
  int lo;       // first token position
  int valid;    // rows in this tile (< tile only at a ragged segment end)
};

// Walks, for query rank r, the key tiles of steps [t_begin, t_end) in ring
// order: step by step, the source rank's segments in ascending position,
// each segment's tiles in order.
struct KvIter {
  int t, t_end, which, i;

  __device__ __forceinline__ void init(const Geometry& g) {
    if (g.step >= 0) { t = g.step; t_end = g.step + 1; }
    else { t = 0; t_end = g.P; }
    which = 0;
    i = 0;
  }

  __device__ __forceinline__ bool next(const Geometry& g, int r, KvTile& kv) {
    while (t < t_end) {
      if (i < g.nt) {
        const int src = ((r - t) % g.P + g.P) % g.P;
        const int seg = rank_seg(g, src, which);
        kv.step = t;
        kv.src = src;
        kv.id = seg * g.nt + i;
        kv.lo = seg * g.seg_len + i * g.tile;
        kv.valid = min(g.tile, g.seg_len - i * g.tile);
        ++i;
        return true;
      }
      i = 0;
      if (++which >= g.segs_per_rank) { which = 0; ++t; }
    }
    return false;
  }
};

// What a (query tile, key tile) pair needs.
enum TileWork { kSkip = 0, kNoMask = 1, kMask = 2 };

// q_lo/q_valid: the query tile's first position and valid rows.
__device__ __forceinline__ int tile_work(const Geometry& g, int q_lo, int q_valid,
                                         const KvTile& kv) {
  if (q_valid <= 0) return kSkip;
  if (g.causal && kv.lo > q_lo + q_valid - 1) return kSkip;   // all keys after all queries
  const bool all_allowed = !g.causal || (kv.lo + kv.valid - 1 <= q_lo);
  return (all_allowed && kv.valid == g.tile) ? kNoMask : kMask;
}

// Pair class for the visit log: FULL iff every (valid query, valid key) pair
// is allowed, PARTIAL otherwise (SKIP tiles are never visited).
__device__ __forceinline__ int tile_class(const Geometry& g, int q_lo, const KvTile& kv) {
  return (!g.causal || kv.lo + kv.valid - 1 <= q_lo) ? RA_CLASS_FULL : RA_CLASS_PARTIAL;
}

__device__ __forceinline__ void log_visit(int* entry_base, int n, const KvTile& kv, int cls) {
  int* e = entry_base + 1 + 4 * n;
  e[0] = kv.step;
  e[1] = kv.src;
  e[2] = kv.id;
  e[3] = cls;
}

}  // namespace ra
