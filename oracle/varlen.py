"""Packed variable-length batches in float64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Sequence b occupies rows [cu[b], cu[b+1]) of packed tensors q, out
[total, H_q, D] and k, v [total, H_kv, D]; lse is [H_q, total]. Every
sequence is its own attention problem (glossary "sequence parallelism
transformers", §Ring Attention: each sequence's result equals its full
attention, whatever its length; uneven lengths are padded per sequence,
mvp-engine "sequence-parallel" skill), so the packed result is the
definition applied to each sequence alone.
"""

import numpy as np

from .attention import attention_naive, f64
from .backward import attention_backward


def _bounds(cu):
    cu = np.asarray(cu, dtype=np.int64)
    return [(int(cu[b]), int(cu[b + 1])) for b in range(len(cu) - 1)]


def attention_varlen(q, k, v, cu, causal, scale):
    """(out [total, H_q, D], lse [H_q, total]) float64."""
    q, k, v = f64(q), f64(k), f64(v)
    total, H_q, D = q.shape
    out = np.zeros((total, H_q, D))
    lse = np.full((H_q, total), -np.inf)
    for lo, hi in _bounds(cu):
        if hi <= lo:
            continue
        o, l = attention_naive(q[None, lo:hi], k[None, lo:hi], v[None, lo:hi], causal, scale)
        out[lo:hi] = o[0]
        lse[:, lo:hi] = l[0]
    return out, lse


def attention_backward_varlen(q, k, v, dout, cu, causal, scale):
    """(dq, dk, dv) float64 of the packed problem, sequence by sequence."""
    q, k, v, dout = f64(q), f64(k), f64(v), f64(dout)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for lo, hi in _bounds(cu):
        if hi <= lo:
            continue
        a, b_, c = attention_backward(q[None, lo:hi], k[None, lo:hi], v[None, lo:hi],
                                      dout[None, lo:hi], causal, scale)
        dq[lo:hi], dk[lo:hi], dv[lo:hi] = a[0], b_[0], c[0]
    return dq, dk, dv
