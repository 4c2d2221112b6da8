"""Pins of the Ulysses oracle.

* the sharded layout element by element: shard p, row c holds position
  p*C + c (scalar loops);
* the two all-to-alls are inverse to each other, and the head-parallel piece
  of rank r holds exactly heads r*H/P.. of every position;
* the whole method equals full attention (its exactness is the point of the
  method), causal or not, GQA, uneven S.
"""

import numpy as np
import pytest

from oracle import attention_naive
from oracle.ulysses import (all_to_all_head_to_seq, all_to_all_seq_to_head,
                            from_sequence_shards, shard_rows, to_sequence_shards,
                            ulysses_attention)


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


@pytest.mark.parametrize("S,P", [(12, 3), (10, 4), (5, 2)])
def test_shard_layout_elementwise(S, P):
    B, H, D = 2, 3, 2
    x = _rand((B, S, H, D), 1)
    xs = to_sequence_shards(x, P)
    C = shard_rows(S, P)
    assert xs.shape == (P, B, C, H, D)
    for p in range(P):
        for b in range(B):
            for c in range(C):
                pos = p * C + c
                for h in range(H):
                    for d in range(D):
                        want = x[b, pos, h, d] if pos < S else 0.0
                        assert xs[p, b, c, h, d] == want
    np.testing.assert_array_equal(from_sequence_shards(xs, S), x)


def test_all_to_alls_are_inverse():
    S, P, B, H, D = 10, 4, 1, 8, 3
    x = _rand((B, S, H, D), 2)
    xs = to_sequence_shards(x, P)
    parts = all_to_all_seq_to_head(xs, S)
    for r, part in enumerate(parts):
        np.testing.assert_array_equal(part, x[:, :, r * 2:(r + 1) * 2])
    np.testing.assert_array_equal(all_to_all_head_to_seq(parts, P, S), xs)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("S,P,Hq,Hkv", [(24, 4, 8, 4), (23, 4, 4, 4), (9, 2, 4, 2)])
def test_equals_full_attention(S, P, Hq, Hkv, causal):
    B, D = 2, 5
    q, k, v = _rand((B, S, Hq, D), 3), _rand((B, S, Hkv, D), 4), _rand((B, S, Hkv, D), 5)
    out_sh, lse_sh = ulysses_attention(to_sequence_shards(q, P), to_sequence_shards(k, P),
                                       to_sequence_shards(v, P), S, causal, 0.45)
    want_o, want_l = attention_naive(q, k, v, causal, 0.45)
    np.testing.assert_allclose(from_sequence_shards(out_sh, S), want_o, atol=1e-12)
    C = shard_rows(S, P)
    for p in range(P):
        for c in range(C):
            pos = p * C + c
            if pos < S:
                np.testing.assert_allclose(lse_sh[p, :, :, c], want_l[:, :, pos], atol=1e-12)
