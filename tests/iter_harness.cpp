// Host build of the kernels' ring bookkeeping (csrc/ring_iter.cuh and the
// backward's csrc/q_iter.cuh), the checked build's range checks
// (csrc/checks.cuh) and the host planner (csrc/plan.cpp), for the CPU tests
// in test_iter_cpu.py. The functions
// below walk the key tiles of one query tile exactly as every role of the
// attention kernels does, so the walk can be compared with the oracle's
// tile_visits on many shapes without a GPU.
#include <algorithm>
namespace ra {
using std::max;
using std::min;
}  // namespace ra
#define __ldg(p) (*(p))
// the checked build's range checks, with the device atomic as a plain store
#define RA_DEBUG_CHECKS
#define atomicExch(p, v) (*(p) = (v))
#include "ring_iter.cuh"
#include "q_iter.cuh"
#include "checks.cuh"

namespace {

// The kernel's walk for query tile (seg, ti) of geometry g: entries
// (step, src, kv tile id, class), at most `cap`; returns the count (0 for a
// tile that holds no token, like the kernels' early exit).
int walk(const ra::Geometry& g, int seg, int ti, int* out, int cap) {
  const int r = ra::seg_owner(g, seg);
  const int q_lo = seg * g.seg_len + ti * g.tile;
  const int q_valid = ra::tile_tokens(g, seg, ti);
  if (q_valid <= 0) return 0;
  ra::KvIter it;
  it.init(g, r, q_lo, q_valid);
  ra::KvTile kv;
  int n = 0;
  while (it.next(g, kv)) {
    if (n < cap) {
      out[4 * n + 0] = kv.step;
      out[4 * n + 1] = kv.src;
      out[4 * n + 2] = kv.id;
      out[4 * n + 3] = ra::tile_class(g, q_lo, kv);
    }
    ++n;
  }
  // the MMA issuers count the walk in closed form: it must agree
  if (ra::kv_walk_length(g, r, q_lo, q_valid) != n) return -2;
  return n;
}

// The forward kernel's walk for a block of `rows` query rows starting at
// tile (seg, ti): (step, src, kv tile id, first position) per key tile, plus
// the closed-form length check; returns the count (-2 on a length mismatch).
int block_walk(const ra::Geometry& g, int seg, int ti, int rows, int* out, int cap) {
  const int r = ra::seg_owner(g, seg);
  const int q_lo = seg * g.seg_len + ti * g.tile;
  const int q_valid = std::min(rows, ra::seg_tokens(g, seg) - ti * g.tile);
  if (q_valid <= 0) return 0;
  ra::KvIter it;
  it.init(g, r, q_lo, q_valid);
  ra::KvTile kv;
  int n = 0;
  while (it.next(g, kv)) {
    if (n < cap) {
      out[4 * n + 0] = kv.step;
      out[4 * n + 1] = kv.src;
      out[4 * n + 2] = kv.id;
      out[4 * n + 3] = kv.lo;
    }
    ++n;
  }
  if (ra::kv_walk_length(g, r, q_lo, q_valid) != n) return -2;
  return n;
}

}  // namespace

extern "C" {

// Geometry facts: [seg_len, n_seg, nt]; returns the planner's status.
int ra_test_geometry(int S, int P, int order, int tile, int* facts) {
  ra::Geometry g;
  const int st = ra::make_geometry(1, 1, 1, S, 128, P, 1, 0.f, order, -1, tile, &g);
  if (st != RA_OK) return st;
  facts[0] = g.seg_len;
  facts[1] = g.n_seg;
  facts[2] = g.nt;
  return RA_OK;
}

// Walk of the two-tile block whose first tile is `qid` (= segment * nt +
// tile) of a fixed-length call.
int ra_test_block_walk(int S, int P, int causal, int order, int step, int qid, int* out,
                       int cap) {
  ra::Geometry g;
  if (ra::make_geometry(1, 1, 1, S, 128, P, causal, 0.f, order, step, 128, &g) != RA_OK)
    return -1;
  return block_walk(g, qid / g.nt, qid % g.nt, 2 * g.tile, out, cap);
}

// Walk of query tile `qid` (= segment * nt + tile) of a fixed-length call.
int ra_test_walk(int S, int P, int causal, int order, int tile, int step, int qid, int* out,
                 int cap) {
  ra::Geometry g;
  if (ra::make_geometry(1, 1, 1, S, 128, P, causal, 0.f, order, step, tile, &g) != RA_OK)
    return -1;
  return walk(g, qid / g.nt, qid % g.nt, out, cap);
}

// Walk of query tile (seg, ti) of packed sequence b, with the grid's
// geometry sized by max_seqlen as the launchers size it; row0 receives the
// sequence's first row and facts its [S, seg_len, nt].
int ra_test_walk_varlen(const int* cu_seqlens, int n_seq, int total, int max_seqlen, int P,
                        int causal, int order, int tile, int b, int seg, int ti, int* out,
                        int cap, int* row0, int* facts) {
  ra::Geometry gp;
  if (ra::make_geometry(n_seq, 1, 1, max_seqlen, 128, P, causal, 0.f, order, -1, tile, &gp) !=
      RA_OK)
    return -1;
  gp.cu_seqlens = cu_seqlens;
  gp.total = total;
  ra::Geometry g;
  ra::varlen_geometry(gp, b, g, *row0);
  facts[0] = g.S;
  facts[1] = g.seg_len;
  facts[2] = g.nt;
  return walk(g, seg, ti, out, cap);
}

// The checked build's report on packed sequence b's offsets: the status word
// varlen_geometry leaves (0, or RA_ERR_RANGE when it had to clamp).
int ra_test_varlen_status(const int* cu_seqlens, int n_seq, int total, int max_seqlen, int b) {
  ra::Geometry gp;
  if (ra::make_geometry(n_seq, 1, 1, max_seqlen, 128, 1, 1, 0.f, 0, -1, 128, &gp) != RA_OK)
    return -1;
  gp.cu_seqlens = cu_seqlens;
  gp.total = total;
  ra::Geometry g;
  int row0 = 0, status = 0;
  ra::varlen_geometry(gp, b, g, row0, &status);
  return status;
}

// The dK/dV kernel's walk for key tile `kid` (= segment * nt + tile) of a
// fixed-length call, one query head: entries (ring step, query segment,
// query tile, mask), at most `cap`; returns the count.
int ra_test_qwalk(int S, int P, int causal, int order, int tile, int kid, int* out, int cap) {
  ra::Geometry g;
  if (ra::make_geometry(1, 1, 1, S, 128, P, causal, 0.f, order, -1, tile, &g) != RA_OK)
    return -1;
  const int kseg = kid / g.nt, kti = kid % g.nt;
  const int src = ra::seg_owner(g, kseg);
  const int kv_lo = kseg * g.seg_len + kti * g.tile;
  const int kv_valid = ra::tile_tokens(g, kseg, kti);
  ra::QTile qt;
  int n = 0;
  auto run = [&](auto& it) {
    it.init(g, src, kv_lo, kv_valid, 0, 1);
    while (it.next(g, qt)) {
      if (n < cap) {
        out[4 * n + 0] = it.t;
        out[4 * n + 1] = qt.seg;
        out[4 * n + 2] = qt.ti;
        out[4 * n + 3] = qt.mask ? 1 : 0;
      }
      ++n;
    }
  };
  if (tile == 128) {
    ra::QIterT<128> it;
    run(it);
  } else if (tile == 64) {
    ra::QIterT<64> it;
    run(it);
  } else {
    return -1;
  }
  return n;
}

// Row addressing of the kernels' loads and stores: for batch b, head h and
// every position of segment `seg`, the tensor row (in units of H*D
// elements) and the lse index. layout 0 fixed-length, 1 packed (rows from
// row0), 2 sequence-sharded; returns the number of positions written.
int ra_test_rows(int layout, int B, int H_q, int S, int P, int order, int total, int row0,
                 int b, int h, int seg, long long* rows, long long* lse_idx, int cap) {
  ra::Geometry g;
  if (ra::make_geometry(B, H_q, 1, S, 128, P, 1, 0.f, order, -1, 128, &g) != RA_OK) return -1;
  if (layout == 1) {
    static const int kDummy[2] = {0, 0};
    g.cu_seqlens = kDummy;
    g.total = total;
  } else if (layout == 2) {
    g.shard_rows = g.seg_len;
  }
  const bool varlen = layout == 1;
  const ra::SegRows r = ra::seg_rows(g, b, seg, row0, varlen);
  const size_t l0 = ra::lse_base(g, b, h, seg, row0, varlen);
  const int n = ra::seg_tokens(g, seg);
  for (int i = 0; i < n && i < cap; ++i) {
    const int pos = seg * g.seg_len + i;
    rows[i] = (long long)(r.grow + pos);
    lse_idx[i] = (long long)(l0 + pos);
  }
  return n;
}

// The checked build's tensor extents for a geometry: layout 0 fixed-length
// [B, S, H, D], 1 packed (`total` rows), 2 sequence-sharded (P * B * C rows);
// ext = [q/out, k/v, lse] in elements.
int ra_test_extents(int layout, int B, int H_q, int H_kv, int S, int D, int P, int total,
                    long long* ext) {
  ra::Geometry g;
  if (ra::make_geometry(B, H_q, H_kv, S, D, P, 1, 0.f, RA_ORDER_CONTIGUOUS, -1, 128, &g) !=
      RA_OK)
    return -1;
  static const int kDummy[2] = {0, 0};
  if (layout == 1) {
    g.cu_seqlens = kDummy;
    g.total = total;
  } else if (layout == 2) {
    g.shard_rows = g.seg_len;
  }
  ext[0] = ra::extent_q(g);
  ext[1] = ra::extent_kv(g);
  ext[2] = ra::extent_lse(g);
  return 0;
}

// One range check as the checked kernels make it: 1 if in range; else 0 and
// *status = RA_ERR_RANGE.
int ra_test_in_range(long long first, long long count, long long extent, int* status) {
  return ra::in_range(first, count, extent, status) ? 1 : 0;
}

}  // extern "C"
