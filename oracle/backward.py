"""Gradients of softmax attention in float64, from the chain rule.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Glossary "sequence parallelism transformers", §Implementation Considerations:
the backward pass of ring attention runs over the same ring as the forward
pass. The pages give no formula for it, so the quantity every kernel must
reproduce is the plain derivative of the forward definition
(``oracle.attention``) with respect to q, k and v, for an upstream gradient
dO = dL/d(out). The log-sum-exp output is auxiliary: it carries no upstream
gradient of its own.

With p_ij = exp(s_ij - lse_i) on the allowed pairs (0 elsewhere), the chain
rule through o_i = sum_j p_ij v_j and the row softmax gives

    dV_j    = sum_i p_ij dO_i
    dp_ij   = <dO_i, v_j>
    delta_i = sum_j p_ij dp_ij                   (= <dO_i, o_i>)
    ds_ij   = p_ij (dp_ij - delta_i)
    dQ_i    = scale * sum_j ds_ij k_j
    dK_j    = scale * sum_i ds_ij q_i

Grouped heads: a key/value head's dK and dV add up the contributions of every
query head that reads it (query head h reads head h // (H_q / H_kv)).
Layouts as in the forward: dq [B, S, H_q, D], dk and dv [B, S, H_kv, D].
"""

import numpy as np

from .attention import f64, _group, _rows_softmax, attention_naive
from .schedule import rank_segments


def attention_backward(q, k, v, dout, causal, scale, row_block=512):
    """(dq, dk, dv) in float64 from the definition, every row.

    ``delta_i`` is formed as sum_j p_ij dp_ij, straight from the chain rule.
    Query rows are processed in blocks only to bound memory; each block
    computes its full softmax rows over every allowed key.
    """
    q, k, v, dout = f64(q), f64(k), f64(v), f64(dout)
    B, S, H_q, D = q.shape
    H_kv = k.shape[2]
    g = _group(H_q, H_kv)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        for h in range(H_q):
            hk = h // g
            K = k[b, :, hk, :]
            V = v[b, :, hk, :]
            for i0 in range(0, S, row_block):
                i1 = min(S, i0 + row_block)
                nk = i1 if causal else S          # later keys are masked for the block
                s = scale * (q[b, i0:i1, h, :] @ K[:nk].T)
                if causal:
                    ii = np.arange(i0, i1)[:, None]
                    jj = np.arange(nk)[None, :]
                    s = np.where(jj <= ii, s, -np.inf)
                _, p = _rows_softmax(s)             # p_ij, zero where masked
                dO = dout[b, i0:i1, h, :]
                dp = dO @ V[:nk].T
                delta = (p * dp).sum(axis=1)
                ds = p * (dp - delta[:, None])
                dq[b, i0:i1, h, :] = scale * (ds @ K[:nk])
                dk[b, :nk, hk, :] += scale * (ds.T @ q[b, i0:i1, h, :])
                dv[b, :nk, hk, :] += p.T @ dO
    return dq, dk, dv


def _positions(ranges):
    return np.concatenate([np.arange(s, s + n) for s, n in ranges])


def ring_attention_backward(q, k, v, dout, causal, scale, P, order):
    """(dq, dk, dv) in float64, computed as a ring of P virtual ranks.

    Rank r owns the query positions ``rank_segments(S, P, order)[r]``; at step
    t it holds the key/value chunk of rank src = (r - t) mod P (the forward's
    ring). It adds its queries' contributions for that chunk: dq of its own
    rows, and dk, dv of the chunk's rows, which travel with the chunk and
    reach its owner after P steps. Every contribution uses the full-row
    statistics lse_i and delta_i = <dO_i, o_i> of the finished forward pass,
    so the per-step pieces add up to the definition exactly.
    """
    q, k, v, dout = f64(q), f64(k), f64(v), f64(dout)
    B, S, H_q, D = q.shape
    H_kv = k.shape[2]
    g = _group(H_q, H_kv)
    out, lse = attention_naive(q, k, v, causal, scale)
    delta = np.einsum("bshd,bshd->bhs", dout, out)
    segs = rank_segments(S, P, order)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for r in range(P):
        qp = _positions(segs[r])
        for t in range(P):
            kp = _positions(segs[(r - t) % P])
            allowed = (kp[None, :] <= qp[:, None]) if causal else None
            for b in range(B):
                for h in range(H_q):
                    hk = h // g
                    s = scale * (q[b, qp, h, :] @ k[b, kp, hk, :].T)
                    p = np.exp(s - lse[b, h, qp][:, None])
                    if allowed is not None:
                        p = np.where(allowed, p, 0.0)
                    dO = dout[b, qp, h, :]
                    dp = dO @ v[b, kp, hk, :].T
                    ds = p * (dp - delta[b, h, qp][:, None])
                    dq[b, qp, h, :] += scale * (ds @ k[b, kp, hk, :])
                    dk[b, kp, hk, :] += scale * (ds.T @ q[b, qp, h, :])
                    dv[b, kp, hk, :] += p.T @ dO
    return dq, dk, dv


def backward_rows(q, k, v, dout, causal, scale, h, q_rows, k_rows):
    """Gradients of one query head ``h`` at sampled positions, float64.

    Returns (dq [B, len(q_rows), D], dk_h [B, len(k_rows), D],
    dv_h [B, len(k_rows), D]) where dk_h, dv_h are the contributions of query
    head h alone (the full dk, dv of a key/value head sum these over the
    query heads of its group). Every quantity comes from the definition; the
    key-row gradients need lse and delta of every query row, which are
    computed here for head h (row blocks, full rows).
    """
    q, k, v, dout = f64(q), f64(k), f64(v), f64(dout)
    B, S, H_q, D = q.shape
    g = _group(H_q, k.shape[2])
    hk = h // g
    q_rows = np.asarray(q_rows, dtype=np.int64)
    k_rows = np.asarray(k_rows, dtype=np.int64)
    dq = np.zeros((B, len(q_rows), D))
    dk = np.zeros((B, len(k_rows), D))
    dv = np.zeros((B, len(k_rows), D))
    for b in range(B):
        K = k[b, :, hk, :]
        V = v[b, :, hk, :]
        # sampled query rows: full rows of p, dp
        s = scale * (q[b, q_rows, h, :] @ K.T)
        if causal:
            s = np.where(np.arange(S)[None, :] <= q_rows[:, None], s, -np.inf)
        _, p = _rows_softmax(s)
        dO = dout[b, q_rows, h, :]
        dp = dO @ V.T
        delta = (p * dp).sum(axis=1)
        dq[b] = scale * ((p * (dp - delta[:, None])) @ K)
        # sampled key rows: every query row's p_ij, ds_ij for those keys
        for i0 in range(0, S, 2048):
            i1 = min(S, i0 + 2048)
            s = scale * (q[b, i0:i1, h, :] @ K.T)
            if causal:
                s = np.where(np.arange(S)[None, :] <= np.arange(i0, i1)[:, None], s, -np.inf)
            _, p = _rows_softmax(s)
            dO = dout[b, i0:i1, h, :]
            dp = dO @ V.T
            delta = (p * dp).sum(axis=1)
            ps = p[:, k_rows]
            ds = ps * (dp[:, k_rows] - delta[:, None])
            dk[b] += scale * (ds.T @ q[b, i0:i1, h, :])
            dv[b] += ps.T @ dO
    return dq, dk, dv
