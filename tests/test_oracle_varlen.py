"""Pins of the packed variable-length oracle.

* one masked softmax over the whole packed tensor, with a block-diagonal
  (same sequence, and causal) mask written out element by element, equals
  the per-sequence result -- a different formulation of the same definition;
* the gradients match central finite differences of the (pinned) packed
  forward;
* a sequence's result does not move when another sequence changes.
"""

import math

import numpy as np
import pytest

from oracle.varlen import attention_backward_varlen, attention_varlen

CU = [0, 5, 5, 6, 13]          # lengths 5, 0, 1, 7


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _seq_of(cu, total):
    seq = np.full(total, -1)
    for b in range(len(cu) - 1):
        seq[cu[b]:cu[b + 1]] = b
    return seq


@pytest.mark.parametrize("causal", [False, True])
def test_block_diagonal_softmax(causal):
    total, H_q, H_kv, D = CU[-1], 4, 2, 3
    q, k, v = _rand((total, H_q, D), 1), _rand((total, H_kv, D), 2), _rand((total, H_kv, D), 3)
    scale = 0.6
    out, lse = attention_varlen(q, k, v, CU, causal, scale)
    seq = _seq_of(CU, total)
    for h in range(H_q):
        hk = h // (H_q // H_kv)
        for i in range(total):
            allowed = [j for j in range(total)
                       if seq[j] == seq[i] and (not causal or j <= i)]
            s = [scale * math.fsum(q[i, h, d] * k[j, hk, d] for d in range(D)) for j in allowed]
            m = max(s)
            z = math.fsum(math.exp(x - m) for x in s)
            assert lse[h, i] == pytest.approx(m + math.log(z), abs=1e-12)
            for d in range(D):
                o = math.fsum(math.exp(x - m) / z * v[j, hk, d] for x, j in zip(s, allowed))
                assert out[i, h, d] == pytest.approx(o, abs=1e-12)


def test_sequences_are_independent():
    total, H, D = CU[-1], 2, 4
    q, k, v = _rand((total, H, D), 4), _rand((total, H, D), 5), _rand((total, H, D), 6)
    out, lse = attention_varlen(q, k, v, CU, True, 0.5)
    k2, v2 = k.copy(), v.copy()
    k2[6:13] += 5.0                      # change the last sequence only
    v2[6:13] -= 2.0
    out2, lse2 = attention_varlen(q, k2, v2, CU, True, 0.5)
    np.testing.assert_array_equal(out[:6], out2[:6])
    np.testing.assert_array_equal(lse[:, :6], lse2[:, :6])
    assert not np.allclose(out[6:], out2[6:])


@pytest.mark.parametrize("causal", [False, True])
def test_backward_finite_differences(causal):
    cu = [0, 3, 3, 7]
    total, H_q, H_kv, D = cu[-1], 2, 1, 2
    q, k, v = _rand((total, H_q, D), 7), _rand((total, H_kv, D), 8), _rand((total, H_kv, D), 9)
    dout = _rand((total, H_q, D), 10)
    scale = 0.8
    dq, dk, dv = attention_backward_varlen(q, k, v, dout, cu, causal, scale)

    def loss():
        o, _ = attention_varlen(q, k, v, cu, causal, scale)
        return float((o * dout).sum())

    hstep = 1e-5
    for x, gx in ((q, dq), (k, dk), (v, dv)):
        num = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = x[idx]
            x[idx] = old + hstep
            lp = loss()
            x[idx] = old - hstep
            lm = loss()
            x[idx] = old
            num[idx] = (lp - lm) / (2 * hstep)
        np.testing.assert_allclose(gx, num, atol=1e-8, rtol=1e-7)
