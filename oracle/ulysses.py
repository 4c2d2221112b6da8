"""Ulysses-style sequence parallelism on P virtual ranks, float64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Glossary "sequence parallelism transformers", §Ulysses Sequence Parallelism:
tokens start in a sequence-parallel layout (rank p holds a contiguous shard
of the sequence, all heads); an all-to-all redistributes them into a
head-parallel layout (rank r holds every token of its subset of heads); each
rank computes full attention for its heads; a second all-to-all restores the
sequence-parallel layout. The steps below follow that order.

Layouts: the sequence-parallel tensors are the ranks' local tensors stacked,
[P, B, C, H, D] with C = ceil(S/P); rank p's shard is positions
[p*C, min((p+1)*C, S)), and rows of a last, partly filled shard past S are
padding (zero here, never read). lse: [P, B, H, C]. Heads split into P
consecutive groups of H/P (rank r: heads [r*H/P, (r+1)*H/P)).
"""

import numpy as np

from .attention import attention_naive, f64


def shard_rows(S, P):
    return -(-S // P)


def to_sequence_shards(x, P):
    """[B, S, H, D] -> [P, B, C, H, D] (padding rows zero)."""
    x = f64(x)
    B, S, H, D = x.shape
    C = shard_rows(S, P)
    xs = np.zeros((P, B, C, H, D))
    for p in range(P):
        lo, hi = p * C, min((p + 1) * C, S)
        if hi > lo:
            xs[p, :, :hi - lo] = x[:, lo:hi]
    return xs


def from_sequence_shards(xs, S):
    """[P, B, C, H, D] -> [B, S, H, D] (padding rows dropped)."""
    P, B, C, H, D = xs.shape
    x = np.zeros((B, S, H, D))
    for p in range(P):
        lo, hi = p * C, min((p + 1) * C, S)
        if hi > lo:
            x[:, lo:hi] = xs[p, :, :hi - lo]
    return x


def all_to_all_seq_to_head(xs, S):
    """Sequence-parallel [P, B, C, H, D] -> per rank r, [B, S, H/P, D]: every
    rank's shard rows of head group r, concatenated in position order."""
    P, B, C, H, D = xs.shape
    Hr = H // P
    parts = []
    for r in range(P):
        y = np.zeros((B, S, Hr, D))
        for p in range(P):                      # the piece rank p sends to rank r
            lo, hi = p * C, min((p + 1) * C, S)
            if hi > lo:
                y[:, lo:hi] = xs[p, :, :hi - lo, r * Hr:(r + 1) * Hr]
        parts.append(y)
    return parts


def all_to_all_head_to_seq(parts, P, S):
    """Inverse: per rank r [B, S, H/P, D] -> sequence-parallel [P, B, C, H, D]."""
    B, _, Hr, D = parts[0].shape
    C = shard_rows(S, P)
    xs = np.zeros((P, B, C, Hr * P, D))
    for r in range(P):
        for p in range(P):                      # the piece rank r sends back to rank p
            lo, hi = p * C, min((p + 1) * C, S)
            if hi > lo:
                xs[p, :, :hi - lo, r * Hr:(r + 1) * Hr] = parts[r][:, lo:hi]
    return xs


def ulysses_attention(q_sh, k_sh, v_sh, S, causal, scale):
    """(out [P, B, C, H_q, D], lse [P, B, H_q, C]) from sequence-parallel
    inputs, through the head-parallel phase."""
    q_sh, k_sh, v_sh = f64(q_sh), f64(k_sh), f64(v_sh)
    P, B, C, H_q, D = q_sh.shape
    H_kv = k_sh.shape[3]
    if H_q % P or H_kv % P:
        raise ValueError("the heads must split evenly over the P ranks")
    qh = all_to_all_seq_to_head(q_sh, S)
    kh = all_to_all_seq_to_head(k_sh, S)
    vh = all_to_all_seq_to_head(v_sh, S)
    outs, lse_sh = [], np.full((P, B, H_q, C), -np.inf)
    Hr = H_q // P
    for r in range(P):                          # full attention for rank r's heads
        o, l = attention_naive(qh[r], kh[r], vh[r], causal, scale)
        outs.append(o)
        for p in range(P):
            lo, hi = p * C, min((p + 1) * C, S)
            if hi > lo:
                lse_sh[p, :, r * Hr:(r + 1) * Hr, :hi - lo] = l[:, :, lo:hi]
    return all_to_all_head_to_seq(outs, P, S), lse_sh
