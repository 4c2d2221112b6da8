"""Exact log-sum-exp merge of partial attention results, float64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Source: glossary "sequence parallelism transformers", §Ring Attention (each
device "accumulates attention outputs" over the received blocks and the result
is mathematically equivalent to full attention) and §Implementation
Considerations, "Numerical Stability" (softmax normalisation across devices
must be handled with care). The pages give no formula; the only combination
that makes the block-wise accumulation equal full attention is the one that
follows from splitting the key set A(i) into disjoint parts A_1, ..., A_n:

    lse   = log sum_t exp(lse_t)
    o     = sum_t exp(lse_t - lse) * o_t

where (o_t, lse_t) is softmax attention over A_t alone. It is evaluated with
the largest lse_t factored out (M = max_t lse_t), which is the same number.
A part with no allowed key has lse_t = -inf and weight 0. If every part is
empty the merged row is o = 0, lse = -inf.

Layouts: o_t [B, S, H, D], lse_t [B, H, S].
"""

import numpy as np

from .attention import f64


def lse_merge_n(os, lses):
    """N-way merge; ``os`` and ``lses`` are sequences of equal-shaped parts."""
    if len(os) != len(lses) or len(os) == 0:
        raise ValueError("need the same positive number of outputs and lse")
    L = np.stack([f64(x) for x in lses])               # [n, B, H, S]
    O = np.stack([f64(x) for x in os])                 # [n, B, S, H, D]
    M = L.max(axis=0)                                  # [B, H, S]
    finite = np.isfinite(M)
    M_safe = np.where(finite, M, 0.0)
    W = np.exp(L - M_safe[None])                       # exp(-inf) = 0
    Z = W.sum(axis=0)
    with np.errstate(divide="ignore", invalid="ignore"):
        lse = np.where(Z > 0, M_safe + np.log(Z), -np.inf)
        C = np.where(Z[None] > 0, W / Z[None], 0.0)    # = exp(lse_t - lse)
    # weights [n, B, H, S] -> [n, B, S, H, 1] to scale the rows of o_t
    C = np.transpose(C, (0, 1, 3, 2))[..., None]
    out = (C * O).sum(axis=0)
    return out, lse


def lse_merge(o_a, lse_a, o_b, lse_b):
    """Pairwise merge of two partial results (the N-way rule with n = 2)."""
    return lse_merge_n([o_a, o_b], [lse_a, lse_b])
