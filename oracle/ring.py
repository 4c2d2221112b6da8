"""Ring attention restated step by step on the CPU, float64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Glossary "sequence parallelism transformers", §Ring Attention: every rank
keeps its local query block; at each of the P steps it computes attention of
its queries against the key/value block it currently holds and accumulates the
outputs; blocks move one rank forward per step. Here the ranks are virtual:
rank r owns the query positions ``rank_segments(...)[r]``; at step t it holds
the chunk of rank (r - t) mod P. The per-step partial results are folded in
step order with the exact log-sum-exp merge (``oracle.merge``).
"""

import numpy as np

from .attention import f64, partial_attention
from .merge import lse_merge
from .schedule import rank_segments


def _positions(ranges):
    return np.concatenate([np.arange(s, s + n) for s, n in ranges])


def ring_attention(q, k, v, causal, scale, P, order, return_partials=False):
    """(out [B,S,H_q,D], lse [B,H_q,S]) float64, computed as a ring of P ranks.

    With ``return_partials`` also returns, per step t, the partial results
    (o_t [B,S,H_q,D], lse_t [B,H_q,S]) that every rank computes at step t,
    written at that rank's query positions.
    """
    q, k, v = f64(q), f64(k), f64(v)
    B, S, H_q, D = q.shape
    segs = rank_segments(S, P, order)
    out = np.zeros((B, S, H_q, D))
    lse = np.full((B, H_q, S), -np.inf)
    parts = [(np.zeros((B, S, H_q, D)), np.full((B, H_q, S), -np.inf))
             for _ in range(P)]
    for r in range(P):
        qp = _positions(segs[r])
        acc_o, acc_l = None, None
        for t in range(P):
            src = (r - t) % P
            kp = _positions(segs[src])
            o_t, l_t = partial_attention(q, k, v, causal, scale, qp, kp)
            parts[t][0][:, qp] = o_t
            parts[t][1][:, :, qp] = l_t
            if acc_o is None:
                acc_o, acc_l = o_t, l_t
            else:
                # merge works on [B, S', H, D] / [B, H, S'] slices alike
                acc_o, acc_l = lse_merge(acc_o, acc_l, o_t, l_t)
        out[:, qp] = acc_o
        lse[:, :, qp] = acc_l
    if return_partials:
        return out, lse, parts
    return out, lse
