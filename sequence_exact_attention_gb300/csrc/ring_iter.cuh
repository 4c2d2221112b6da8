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

// Tokens of segment `seg`: its seg_len positions clipped at S. When S is not
// a multiple of the split the sequence counts as padded to one, and the
// padding positions (S and beyond) hold no token: a trailing segment can be
// short or empty.
__device__ __forceinline__ int seg_tokens(const Geometry& g, int seg) {
  return max(0, min(g.seg_len, g.S - seg * g.seg_len));
}

// Rows of tile `ti` of segment `seg`; <= 0 for a tile that holds no token.
__device__ __forceinline__ int tile_tokens(const Geometry& g, int seg, int ti) {
  return min(g.tile, seg_tokens(g, seg) - ti * g.tile);
}

// Geometry of packed sequence b: the grid's geometry `gp` (sized by the
// longest sequence) with S = the sequence's own length, so its chunks are
// ceil(S_b / n_seg) positions, padded like any uneven length. `row0` is the
// sequence's first row in the packed tensors. Offsets are clamped into
// [0, total] and lengths to [0, S], so a malformed table cannot move any
// access outside the tensors. The checked build also reports such a table:
// when clamping changes an offset or a length it sets RA_ERR_RANGE in
// `status` (if given).
__device__ __forceinline__ void varlen_geometry(const Geometry& gp, int b, Geometry& gs,
                                                int& row0, int* status = nullptr) {
  const int lo_raw = __ldg(gp.cu_seqlens + b);
  const int hi_raw = __ldg(gp.cu_seqlens + b + 1);
  const int lo = min(max(lo_raw, 0), gp.total);
  const int hi = min(max(hi_raw, lo), gp.total);
#ifdef RA_DEBUG_CHECKS
  if (status && (lo != lo_raw || hi != hi_raw || hi - lo > gp.S))
    atomicExch(status, (int)RA_ERR_RANGE);
#else
  (void)status;
#endif
  gs = gp;
  gs.S = min(hi - lo, gp.S);
  gs.seg_len = (gs.S + gp.n_seg - 1) / gp.n_seg;
  gs.nt = (gs.seg_len + gp.tile - 1) / gp.tile;
  row0 = lo;
}

// Where the rows of segment `seg` of batch b live in the tensors' layout.
// Natural [B, S, H, D]: TMA batch b, positions as rows. Packed sequences:
// batch 0, rows from the sequence's first row `row0`. Sequence-sharded
// [P, B, C, H, D] (mapped as [P*B, C, H, D]; segment p is shard p): TMA
// batch p*B + b, row = position - p*C.
struct SegRows {
  int trow;       // added to a position: the TMA row coordinate
  int tbat;       // the TMA batch coordinate
  size_t grow;    // added to a position: the row index in units of H*D elements
};

__device__ __forceinline__ SegRows seg_rows(const Geometry& gp, int b, int seg, int row0,
                                            bool varlen) {
  SegRows r;
  if (varlen) {
    r.trow = row0;
    r.tbat = 0;
    r.grow = (size_t)row0;
  } else if (gp.shard_rows > 0) {
    const size_t lb = (size_t)seg * gp.B + b, c = (size_t)gp.shard_rows;
    r.trow = -seg * gp.shard_rows;
    r.tbat = (int)lb;
    r.grow = lb * c - (size_t)seg * c;
  } else {
    r.trow = 0;
    r.tbat = b;
    r.grow = (size_t)b * gp.S;
  }
  return r;
}

// Index of the lse entry of position 0 of segment `seg`, head h, batch b:
// natural [B, H, S]; packed [H, total]; sequence-sharded [P, B, H, C].
__device__ __forceinline__ size_t lse_base(const Geometry& gp, int b, int h, int seg, int row0,
                                           bool varlen) {
  if (varlen) return (size_t)h * gp.total + row0;
  if (gp.shard_rows > 0) {
    const size_t c = (size_t)gp.shard_rows;
    return (((size_t)seg * gp.B + b) * gp.H_q + h) * c - (size_t)seg * c;
  }
  return ((size_t)b * gp.H_q + h) * gp.S;
}

struct KvTile {
  int step;     // ring step t
  int src;      // rank the block started on
  int seg;      // segment (position order) the tile belongs to
  int id;       // global tile id = segment * nt + index in segment
  int lo;       // first token position
  int valid;    // rows in this tile (< tile only at a ragged segment end)
  int work;     // kNoMask or kMask (SKIP tiles are never returned)
};

// What a (query tile, key tile) pair needs.
enum TileWork { kSkip = 0, kNoMask = 1, kMask = 2 };

// Walks, for one query tile of rank r, the key tiles of steps
// [t_begin, t_end) in ring order: step by step, the source rank's segments in
// ascending position, each segment's tiles in order. Tiles that the causal
// rule masks out entirely are left out; since positions grow along a
// segment, the rest of a segment is dropped at its first such tile.
// Everything is updated incrementally (no division in the loop): every role
// of a kernel walks this sequence once per key tile.
struct KvIter {
  int t, t_end;    // current step, end step
  int src;         // source rank of step t
  int which;       // segment of src being walked (0 or 1)
  int lo;          // first position of the next tile
  int id;          // id of the next tile
  int seg;         // segment being walked
  int rem;         // tokens of the current segment from `lo` on
  int q_lo, q_hi;  // the query tile's first and last valid position

  __device__ __forceinline__ void start_segment(const Geometry& g) {
    seg = rank_seg(g, src, which);
    lo = seg * g.seg_len;
    id = seg * g.nt;
    rem = seg_tokens(g, seg);
  }

  __device__ __forceinline__ void init(const Geometry& g, int r, int q_first, int q_valid) {
    if (g.step >= 0) { t = g.step; t_end = g.step + 1; }
    else { t = 0; t_end = g.P; }
    src = r - t;
    if (src < 0) src += g.P;
    which = 0;
    q_lo = q_first;
    q_hi = q_first + q_valid - 1;
    if (q_valid <= 0) t = t_end;       // nothing to attend to
    start_segment(g);
  }

  __device__ __forceinline__ bool next(const Geometry& g, KvTile& kv) {
    while (t < t_end) {
      if (rem > 0 && !(g.causal && lo > q_hi)) {
        const int valid = min(g.tile, rem);
        kv.step = t;
        kv.src = src;
        kv.seg = seg;
        kv.id = id;
        kv.lo = lo;
        kv.valid = valid;
        const bool all_allowed = !g.causal || (lo + valid - 1 <= q_lo);
        kv.work = (all_allowed && valid == g.tile) ? kNoMask : kMask;
        lo += g.tile;
        rem -= g.tile;
        ++id;
        return true;
      }
      // next segment of this source rank, or the next ring step
      if (++which >= g.segs_per_rank) {
        which = 0;
        ++t;
        if (--src < 0) src += g.P;
      }
      start_segment(g);
    }
    return false;
  }
};

// Number of key tiles KvIter walks for the query rows [q_lo, q_lo + q_valid),
// in closed form per segment: a segment of len tokens from s0 holds
// ceil(len / tile) tiles, and under the causal rule the walk stops after the
// last tile starting at or before the last query row.
__device__ __forceinline__ int kv_walk_length(const Geometry& g, int r, int q_lo, int q_valid) {
  if (q_valid <= 0) return 0;
  const int q_hi = q_lo + q_valid - 1;
  const int t0 = g.step >= 0 ? g.step : 0;
  const int t1 = g.step >= 0 ? g.step + 1 : g.P;
  int n = 0;
  for (int t = t0; t < t1; ++t) {
    const int src = r - t < 0 ? r - t + g.P : r - t;
    for (int w = 0; w < g.segs_per_rank; ++w) {
      const int seg = rank_seg(g, src, w);
      const int s0 = seg * g.seg_len;
      int k = (seg_tokens(g, seg) + g.tile - 1) / g.tile;
      if (g.causal) k = min(k, q_hi < s0 ? 0 : (q_hi - s0) / g.tile + 1);
      n += k;
    }
  }
  return n;
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
