"""Pins of the float64 backward oracle against facts that do not come from it.

* central finite differences of the forward oracle (itself pinned in
  test_oracle.py): any dropped term, wrong sign, index or transposed operand
  in the gradient formulas shows up here;
* a two-token causal closed form derived by hand;
* invariants of the softmax gradient (shift invariance: dK sums to zero over
  the keys; rows of p sum to one: dV sums to the summed dO);
* special cases: causal row 0, identical values, zero scale, grouped heads;
* the ring restatement and the sampled-row evaluator against the full one.
"""

import math

import numpy as np
import pytest

from oracle import ORDER_CONTIGUOUS, ORDER_ZIGZAG, attention_naive
from oracle.backward import attention_backward, backward_rows, ring_attention_backward


def _rand(shape, seed, std=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * std


def _loss(q, k, v, dout, causal, scale):
    out, _ = attention_naive(q, k, v, causal, scale)
    return float((out * dout).sum())


@pytest.mark.parametrize("causal", [False, True])
def test_finite_differences(causal):
    B, S, H_q, H_kv, D = 1, 5, 2, 1, 3
    q = _rand((B, S, H_q, D), 1)
    k = _rand((B, S, H_kv, D), 2)
    v = _rand((B, S, H_kv, D), 3)
    dout = _rand((B, S, H_q, D), 4)
    scale = 0.7
    dq, dk, dv = attention_backward(q, k, v, dout, causal, scale)
    h = 1e-5
    for x, gx in ((q, dq), (k, dk), (v, dv)):
        num = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = x[idx]
            x[idx] = old + h
            lp = _loss(q, k, v, dout, causal, scale)
            x[idx] = old - h
            lm = _loss(q, k, v, dout, causal, scale)
            x[idx] = old
            num[idx] = (lp - lm) / (2 * h)
        np.testing.assert_allclose(gx, num, atol=1e-8, rtol=1e-7)


def test_two_token_causal_closed_form():
    # positions 0, 1; D = 1; row 0 sees key 0 only, row 1 sees keys 0 and 1.
    q0, q1, k0, k1, v0, v1, do0, do1, c = 0.3, -1.2, 0.8, -0.5, 1.5, -0.7, 0.9, -1.1, 0.6
    q = np.array([q0, q1]).reshape(1, 2, 1, 1)
    k = np.array([k0, k1]).reshape(1, 2, 1, 1)
    v = np.array([v0, v1]).reshape(1, 2, 1, 1)
    dout = np.array([do0, do1]).reshape(1, 2, 1, 1)
    dq, dk, dv = attention_backward(q, k, v, dout, True, c)
    a0, a1 = c * q1 * k0, c * q1 * k1
    p10 = math.exp(a0) / (math.exp(a0) + math.exp(a1))
    p11 = 1.0 - p10
    g = do1 * p10 * p11 * (v0 - v1)            # dL/da0 = -dL/da1
    assert dq[0, 0, 0, 0] == 0.0
    assert dq[0, 1, 0, 0] == pytest.approx(c * g * (k0 - k1), abs=1e-14)
    assert dk[0, 0, 0, 0] == pytest.approx(c * g * q1, abs=1e-14)
    assert dk[0, 1, 0, 0] == pytest.approx(-c * g * q1, abs=1e-14)
    assert dv[0, 0, 0, 0] == pytest.approx(do0 + p10 * do1, abs=1e-14)
    assert dv[0, 1, 0, 0] == pytest.approx(p11 * do1, abs=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_invariants(causal):
    B, S, H_q, H_kv, D = 2, 37, 4, 2, 8
    q, k, v = _rand((B, S, H_q, D), 5), _rand((B, S, H_kv, D), 6), _rand((B, S, H_kv, D), 7)
    dout = _rand((B, S, H_q, D), 8)
    dq, dk, dv = attention_backward(q, k, v, dout, causal, 0.35, row_block=16)
    # softmax is invariant to adding one constant to a row's scores, so the
    # key gradients of every (batch, kv head, component) sum to zero
    np.testing.assert_allclose(dk.sum(axis=1), 0.0, atol=1e-12)
    # rows of p sum to one: sum_j dV_j = sum over the group's query heads of sum_i dO_i
    want = dout.reshape(B, S, H_kv, H_q // H_kv, D).sum(axis=(1, 3))
    np.testing.assert_allclose(dv.sum(axis=1), want, atol=1e-12)
    if causal:
        np.testing.assert_array_equal(dq[:, 0], 0.0)       # a single key: no query gradient


def test_identical_values_give_no_score_gradient():
    B, S, H, D = 1, 19, 2, 4
    q, k = _rand((B, S, H, D), 9), _rand((B, S, H, D), 10)
    v = np.broadcast_to(_rand((1, 1, H, D), 11), (B, S, H, D)).copy()
    dout = _rand((B, S, H, D), 12)
    for causal in (False, True):
        dq, dk, _ = attention_backward(q, k, v, dout, causal, 0.5)
        np.testing.assert_allclose(dq, 0.0, atol=1e-13)
        np.testing.assert_allclose(dk, 0.0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_zero_scale_is_uniform(causal):
    B, S, H, D = 1, 11, 1, 3
    q, k, v = _rand((B, S, H, D), 13), _rand((B, S, H, D), 14), _rand((B, S, H, D), 15)
    dout = _rand((B, S, H, D), 16)
    dq, dk, dv = attention_backward(q, k, v, dout, causal, 0.0)
    np.testing.assert_array_equal(dq, 0.0)
    np.testing.assert_array_equal(dk, 0.0)
    want = np.zeros_like(dv)
    for i in range(S):
        keys = range(i + 1) if causal else range(S)
        for j in keys:
            want[0, j, 0] += dout[0, i, 0] / len(keys)
    np.testing.assert_allclose(dv, want, atol=1e-14)


def test_grouped_heads_equal_repeated_heads():
    B, S, H_q, H_kv, D = 1, 23, 6, 2, 5
    q = _rand((B, S, H_q, D), 17)
    k, v = _rand((B, S, H_kv, D), 18), _rand((B, S, H_kv, D), 19)
    dout = _rand((B, S, H_q, D), 20)
    g = H_q // H_kv
    k_rep, v_rep = np.repeat(k, g, axis=2), np.repeat(v, g, axis=2)
    for causal in (False, True):
        dq, dk, dv = attention_backward(q, k, v, dout, causal, 0.4)
        dq_m, dk_m, dv_m = attention_backward(q, k_rep, v_rep, dout, causal, 0.4)
        np.testing.assert_allclose(dq, dq_m, atol=1e-12)
        np.testing.assert_allclose(dk, dk_m.reshape(B, S, H_kv, g, D).sum(axis=3), atol=1e-12)
        np.testing.assert_allclose(dv, dv_m.reshape(B, S, H_kv, g, D).sum(axis=3), atol=1e-12)


@pytest.mark.parametrize("P,order", [(1, ORDER_CONTIGUOUS), (2, ORDER_ZIGZAG),
                                     (4, ORDER_CONTIGUOUS), (4, ORDER_ZIGZAG)])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("S", [48, 45])          # 45: uneven chunks, padded
def test_ring_restatement_equals_definition(P, order, causal, S):
    B, H_q, H_kv, D = 1, 2, 1, 6
    q = _rand((B, S, H_q, D), 21)
    k, v = _rand((B, S, H_kv, D), 22), _rand((B, S, H_kv, D), 23)
    dout = _rand((B, S, H_q, D), 24)
    ref = attention_backward(q, k, v, dout, causal, 0.4)
    got = ring_attention_backward(q, k, v, dout, causal, 0.4, P, order)
    for a, b in zip(got, ref):
        np.testing.assert_allclose(a, b, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_sampled_rows_equal_definition(causal):
    B, S, H_q, H_kv, D = 2, 40, 4, 2, 6
    q = _rand((B, S, H_q, D), 25)
    k, v = _rand((B, S, H_kv, D), 26), _rand((B, S, H_kv, D), 27)
    dout = _rand((B, S, H_q, D), 28)
    dq, _, _ = attention_backward(q, k, v, dout, causal, 0.3)
    rows = np.array([0, 7, 39])
    keys = np.array([0, 13, 39])
    for h_kv in range(H_kv):
        dk_sum = np.zeros((B, len(keys), D))
        dv_sum = np.zeros((B, len(keys), D))
        for h in range(h_kv * 2, h_kv * 2 + 2):
            dq_r, dk_r, dv_r = backward_rows(q, k, v, dout, causal, 0.3, h, rows, keys)
            np.testing.assert_allclose(dq_r, dq[:, rows, h], atol=1e-12)
            dk_sum += dk_r
            dv_sum += dv_r
        _, dk, dv = attention_backward(q, k, v, dout, causal, 0.3)
        np.testing.assert_allclose(dk_sum, dk[:, keys, h_kv], atol=1e-12)
        np.testing.assert_allclose(dv_sum, dv[:, keys, h_kv], atol=1e-12)
