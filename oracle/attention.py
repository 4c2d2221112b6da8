"""Full softmax attention in float64, from its definition.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Source: glossary "sequence parallelism transformers", §Ring Attention: the
block-wise ring computation "accumulates attention outputs" and is exactly
equal to full attention. So the quantity every kernel must reproduce is plain
softmax attention over the allowed keys:

    s_ij   = scale * <q_i, k_j>                 for j in A(i)
    lse_i  = log sum_{j in A(i)} exp(s_ij)      (natural log)
    o_i    = sum_{j in A(i)} exp(s_ij - lse_i) * v_j

with A(i) = all key positions (non-causal) or {j : j <= i} (causal, global
positions, diagonal included). Grouped heads: query head h reads key/value head
h // (H_q / H_kv) (consecutive grouping). Layouts: q, out are [B, S, H_q, D];
k, v are [B, S, H_kv, D]; lse is [B, H_q, S]. Sequence is dimension 1, as in
the nvFuser PR "Transformer sequence parallel forward" (the input is sharded on
dim 1) and the mvp-engine "sequence-parallel" skill (sequence dim 1 for
[batch, seq, hidden]).

The evaluation subtracts the row maximum before exponentiating. That is the
usual overflow guard and changes nothing mathematically: exp(s - m) / sum
exp(s - m) equals exp(s) / sum exp(s), and lse = m + log(sum exp(s - m)).
Rows are processed in blocks only to bound memory; every row is independent.
"""

import numpy as np


def f64(x):
    """Exact upcast of a NumPy array or a (CPU or GPU) torch tensor to float64."""
    if hasattr(x, "detach"):
        return x.detach().to("cpu").double().numpy()
    return np.asarray(x, dtype=np.float64)


def _group(H_q, H_kv):
    if H_q % H_kv != 0:
        raise ValueError("H_q must be a multiple of H_kv")
    return H_q // H_kv


def _rows_softmax(scores):
    """Row-wise (lse, weights) of a score block whose masked entries are -inf.

    Rows with no allowed key get lse = -inf and all-zero weights.
    """
    m = scores.max(axis=1)
    finite = np.isfinite(m)
    m_safe = np.where(finite, m, 0.0)
    e = np.exp(scores - m_safe[:, None])          # exp(-inf) = 0 for masked keys
    z = e.sum(axis=1)
    with np.errstate(divide="ignore", invalid="ignore"):
        lse = np.where(z > 0, m_safe + np.log(z), -np.inf)
        w = np.where(z[:, None] > 0, e / z[:, None], 0.0)
    return lse, w


def _attend(q_rows, k, v, causal, scale, q_pos, kv_pos):
    """Attention of the query rows ``q_rows`` [B, n, H_q, D] (at global
    positions ``q_pos``) over the keys at ``kv_pos`` only."""
    q_rows, k, v = f64(q_rows), f64(k), f64(v)
    B, n, H_q, D = q_rows.shape
    H_kv = k.shape[2]
    g = _group(H_q, H_kv)
    q_pos = np.asarray(q_pos, dtype=np.int64)
    kv_pos = np.asarray(kv_pos, dtype=np.int64)
    out = np.zeros((B, n, H_q, D))
    lse = np.full((B, H_q, n), -np.inf)
    if n == 0 or len(kv_pos) == 0:
        return out, lse
    allowed = None
    if causal:
        allowed = kv_pos[None, :] <= q_pos[:, None]
    for b in range(B):
        for h in range(H_q):
            hk = h // g
            s = scale * (q_rows[b, :, h, :] @ k[b, kv_pos, hk, :].T)
            if allowed is not None:
                s = np.where(allowed, s, -np.inf)
            l_row, w = _rows_softmax(s)
            lse[b, h, :] = l_row
            out[b, :, h, :] = w @ v[b, kv_pos, hk, :]
    return out, lse


def partial_attention(q, k, v, causal, scale, q_pos, kv_pos):
    """Attention of the queries at ``q_pos`` over the keys at ``kv_pos`` only.

    This is one ring step (glossary "sequence parallelism transformers",
    §Ring Attention, "Computation": attention between the local queries and
    the received keys/values). Positions are global token indices, so the
    causal rule j <= i is applied in global coordinates. Returns
    o [B, len(q_pos), H_q, D] and lse [B, H_q, len(q_pos)], float64; a query
    row with no allowed key in this set gets o = 0 and lse = -inf.
    """
    q_pos = np.asarray(q_pos, dtype=np.int64)
    return _attend(q[:, q_pos], k, v, causal, scale, q_pos, kv_pos)


def attention_rows(q, k, v, causal, scale, rows):
    """Full attention for a subset of query positions ``rows`` (all heads).

    Used to check large problems on sampled outputs: each row is computed on
    its own from the definition, over all S keys. Only the sampled rows of q
    are converted to float64.
    """
    rows = np.asarray(rows, dtype=np.int64)
    S = k.shape[1]
    return _attend(q[:, rows], k, v, causal, scale, rows, np.arange(S))


def attention_naive(q, k, v, causal, scale, row_block=1024):
    """Full softmax attention for every query row; returns (out, lse) in f64.

    out [B, S, H_q, D], lse [B, H_q, S]. For the causal case the key range of
    a row block is cut at the block's last row: every key beyond it is masked
    for every row of the block, so nothing is lost.
    """
    q, k, v = f64(q), f64(k), f64(v)
    B, S, H_q, D = q.shape
    H_kv = k.shape[2]
    g = _group(H_q, H_kv)
    out = np.zeros((B, S, H_q, D))
    lse = np.zeros((B, H_q, S))
    for b in range(B):
        for h in range(H_q):
            hk = h // g
            K = k[b, :, hk, :]
            V = v[b, :, hk, :]
            for i0 in range(0, S, row_block):
                i1 = min(S, i0 + row_block)
                nk = i1 if causal else S
                s = scale * (q[b, i0:i1, h, :] @ K[:nk].T)
                if causal:
                    ii = np.arange(i0, i1)[:, None]
                    jj = np.arange(nk)[None, :]
                    s = np.where(jj <= ii, s, -np.inf)
                l_row, w = _rows_softmax(s)
                lse[b, h, i0:i1] = l_row
                out[b, i0:i1, h, :] = w @ V[:nk]
    return out, lse
