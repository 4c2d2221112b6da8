"""Ring schedule of virtual ranks on one device: who holds which chunk when.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Sources, glossary "sequence parallelism transformers":
* §Sequence Parallelism Fundamentals, "Sequence Dimension Splitting": a length
  S sequence is cut into P chunks, one per rank, S/P tokens each.
* §Ring Attention, "Ring Communication": rank i sends its block to i+1 and
  receives from i-1; P steps visit every block. So at step t rank r holds the
  key/value chunk that started on rank (r - t) mod P.
* §Implementation Considerations, "Load Balancing": uneven work must be
  balanced. Under a causal mask a contiguous split gives rank P-1 P times the
  work of rank 0; the zig-zag order is the balancing scheme used here: the
  sequence is cut into 2P equal halves and rank r owns halves r and 2P-1-r.
  Inputs and outputs stay in natural token order; only the ownership changes.

Uneven lengths (the mvp-engine "sequence-parallel" skill: seq_len divisible
by the split, else pad explicitly and mask; the nvFuser PR "Transformer
sequence parallel forward" skips the s % d != 0 case instead): the sequence
is padded to the next multiple of P (contiguous) or 2P (zig-zag), so every
chunk (half) spans L = ceil(S / P) (ceil(S / 2P)) positions starting at a
multiple of L, and the padding positions, at S and beyond, hold no tokens:
a chunk's tokens are its positions below S. Ranges are therefore clipped at
S; a trailing chunk can be shorter than L or empty. When S is a multiple,
this is the plain even split.

Classes of a (query set, key set) pair under the causal rule j <= i:
SKIP (no allowed pair), FULL (every pair allowed), PARTIAL (some allowed).
Without a causal mask every pair is FULL.
"""

import numpy as np

SKIP, FULL, PARTIAL = 0, 1, 2
ORDER_CONTIGUOUS, ORDER_ZIGZAG = 0, 1


def _check(S, P, order):
    if P <= 0 or S <= 0:
        raise ValueError("S and P must be positive")
    if order not in (ORDER_CONTIGUOUS, ORDER_ZIGZAG):
        raise ValueError("unknown order")


def segment_length(S, P, order):
    """L: positions spanned by one chunk (contiguous) or half (zig-zag) of
    the padded sequence."""
    _check(S, P, order)
    parts = P if order == ORDER_CONTIGUOUS else 2 * P
    return -(-S // parts)


def _clip(start, L, S):
    return (start, max(0, min(L, S - start)))


def rank_segments(S, P, order):
    """Per rank, the list of (start, length) token ranges it owns, ascending.
    Lengths are clipped at S (possibly 0); starts are multiples of L."""
    L = segment_length(S, P, order)
    if order == ORDER_CONTIGUOUS:
        return [[_clip(r * L, L, S)] for r in range(P)]
    return [[_clip(r * L, L, S), _clip((2 * P - 1 - r) * L, L, S)] for r in range(P)]


def classify(q_ranges, kv_ranges, causal):
    """SKIP / FULL / PARTIAL of the pair set q x kv under j <= i.

    Each argument is a list of (start, length) ranges. For one query range
    [a, a+n) and one key range [c, c+m): every pair is allowed iff the last
    key is not after the first query (c+m-1 <= a); none is iff the first key
    is after the last query (c > a+n-1). Over unions of ranges: FULL iff
    every range pair is FULL, SKIP iff every range pair is SKIP.
    """
    if not causal:
        return FULL
    all_full, all_skip = True, True
    for a, n in q_ranges:
        if n <= 0:
            continue
        for c, m in kv_ranges:
            if m <= 0:
                continue
            if not (c + m - 1 <= a):
                all_full = False
            if not (c > a + n - 1):
                all_skip = False
    if all_skip:
        return SKIP
    if all_full:
        return FULL
    return PARTIAL


def ring_schedule(S, P, causal, order):
    """List of dicts, one per (rank, step), in rank-major then step order."""
    segs = rank_segments(S, P, order)
    out = []
    for r in range(P):
        for t in range(P):
            src = (r - t) % P
            out.append(dict(rank=r, step=t, src=src, q=segs[r], kv=segs[src],
                            cls=classify(segs[r], segs[src], causal)))
    return out


def schedule_table(S, P, causal, order):
    """The schedule as an int32 table [P*P, 9]:
    rank, step, src, cls, L (the padded segment length), q_a, q_b, kv_a, kv_b
    (segment starts; -1 where a rank has a single segment). Same row order as
    ``ring_schedule``."""
    L = segment_length(S, P, order)
    rows = []
    for e in ring_schedule(S, P, causal, order):
        q = [s for s, _ in e["q"]] + [-1] * (2 - len(e["q"]))
        kv = [s for s, _ in e["kv"]] + [-1] * (2 - len(e["kv"]))
        rows.append([e["rank"], e["step"], e["src"], e["cls"], L,
                     q[0], q[1], kv[0], kv[1]])
    return np.asarray(rows, dtype=np.int32)


def segments_in_position_order(S, P, order):
    """All (start, length) segments sorted by start, with the owning rank."""
    segs = rank_segments(S, P, order)
    flat = [(s, n, r) for r, lst in enumerate(segs) for s, n in lst]
    return sorted(flat)


def tile_visits(S, P, causal, order, tile):
    """Expected key-tile visits of a tiled kernel, per query tile.

    Every segment is cut into tiles of ``tile`` rows (the last one shorter if
    the segment length is not a multiple; tiles at or past S are empty and
    visit nothing, and tiles are clipped at S). Tiles are numbered globally:
    segment index g in position order times tiles-per-segment plus the tile
    index inside the segment. For the query tile (g, i) owned by rank r, the
    visits are, in order: for t = 0..P-1, src = (r - t) mod P, for each
    segment of src in ascending position, for each of its tiles in order,
    the entry (step, src, kv_tile_id, cls) with cls classified from the
    tiles' own token ranges; SKIP tiles are left out.

    Returns a list indexed by query tile id of lists of 4-tuples.
    """
    flat = segments_in_position_order(S, P, order)
    seg_len = segment_length(S, P, order)
    nt = -(-seg_len // tile)
    seg_index = {s: g for g, (s, _, _) in enumerate(flat)}
    segs = rank_segments(S, P, order)

    def tiles_of(start):
        g = seg_index[start]
        res = []
        for i in range(nt):
            lo = start + i * tile
            n = max(0, min(tile, start + seg_len - lo, S - lo))
            res.append((g * nt + i, lo, n))
        return res

    visits = [None] * (len(flat) * nt)
    for s_start, _, r in flat:
        for qid, qlo, qn in tiles_of(s_start):
            seq = []
            for t in range(P):
                src = (r - t) % P
                for kv_start, _ in segs[src]:
                    for kid, klo, kn in tiles_of(kv_start):
                        if qn <= 0 or kn <= 0:
                            continue
                        c = classify([(qlo, qn)], [(klo, kn)], causal)
                        if c != SKIP:
                            seq.append((t, src, kid, c))
            visits[qid] = seq
    return visits
