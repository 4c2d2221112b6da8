"""Pins of the CPU oracle against facts fixed outside the oracle itself.

Each test checks the oracle against a hand-derived fixture, a closed form, an
invariant that full softmax attention must satisfy, or a brute-force scalar
evaluation on tiny inputs. No GPU is needed.
"""

import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import (attention_naive, attention_rows, partial_attention,
                    lse_merge, lse_merge_n, ring_attention, ring_schedule,
                    schedule_table, tile_visits, rank_segments,
                    SKIP, FULL, PARTIAL)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
TOL = 1e-12


def _num(x):
    if isinstance(x, (int, float)):
        return float(x)
    if x == "-inf":
        return -math.inf
    if x.startswith("ln"):
        return math.log(float(x[2:]))
    return float(x)


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)["cases"]


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


# --------------------------------------------------------------------------
# hand-derived fixtures
# --------------------------------------------------------------------------

@pytest.mark.parametrize("case", _golden("attention_hand.json"),
                         ids=lambda c: c["name"])
def test_golden_attention(case):
    S = len(case["q"])
    q = np.array([_num(x) for x in case["q"]]).reshape(1, S, 1, 1)
    k = np.array([_num(x) for x in case["k"]]).reshape(1, S, 1, 1)
    v = np.array([_num(x) for x in case["v"]]).reshape(1, S, 1, 1)
    out, lse = attention_naive(q, k, v, case["causal"], case["scale"])
    np.testing.assert_allclose(out.reshape(S), case["out"], rtol=0, atol=TOL)
    np.testing.assert_allclose(lse.reshape(S), [_num(x) for x in case["lse"]],
                               rtol=0, atol=TOL)
    for P in (1, S):
        if S % P == 0:
            o2, l2 = ring_attention(q, k, v, case["causal"], case["scale"], P, 0)
            np.testing.assert_allclose(o2.reshape(S), case["out"], atol=TOL)


@pytest.mark.parametrize("case", _golden("merge_hand.json"),
                         ids=lambda c: c["name"])
def test_golden_merge(case):
    def o(x):
        return np.array(x, dtype=np.float64).reshape(1, 1, 1, -1)

    def l(x):
        return np.array([_num(x)]).reshape(1, 1, 1)

    out, lse = lse_merge(o(case["o_a"]), l(case["lse_a"]),
                         o(case["o_b"]), l(case["lse_b"]))
    np.testing.assert_allclose(out.reshape(-1), case["out"], rtol=0, atol=TOL)
    want = _num(case["lse"])
    if math.isinf(want):
        assert lse.reshape(-1)[0] == want
    else:
        assert abs(lse.reshape(-1)[0] - want) < TOL


@pytest.mark.parametrize("case", _golden("schedule_hand.json"),
                         ids=lambda c: c["name"])
def test_golden_schedule(case):
    got = schedule_table(case["S"], case["P"], case["causal"], case["order"])
    np.testing.assert_array_equal(got, np.array(case["table"], dtype=np.int32))


# --------------------------------------------------------------------------
# brute force on tiny inputs: scalar loops with exactly rounded sums
# --------------------------------------------------------------------------

def _brute(q, k, v, causal, scale):
    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    g = Hq // Hkv
    out = np.zeros_like(q)
    lse = np.zeros((B, Hq, S))
    for b in range(B):
        for h in range(Hq):
            hk = h // g
            for i in range(S):
                keys = range(i + 1) if causal else range(S)
                s = [scale * math.fsum(q[b, i, h, d] * k[b, j, hk, d]
                                       for d in range(D)) for j in keys]
                z = math.fsum(math.exp(x) for x in s)
                lse[b, h, i] = math.log(z)
                for d in range(D):
                    out[b, i, h, d] = math.fsum(
                        math.exp(x) / z * v[b, j, hk, d]
                        for x, j in zip(s, keys))
    return out, lse


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [(1, 5, 1, 1, 3), (2, 8, 4, 2, 4),
                                   (1, 7, 3, 1, 2)])
def test_bruteforce_tiny(causal, shape):
    B, S, Hq, Hkv, D = shape
    q = _rand((B, S, Hq, D), 1)
    k = _rand((B, S, Hkv, D), 2)
    v = _rand((B, S, Hkv, D), 3)
    scale = 0.7
    o1, l1 = attention_naive(q, k, v, causal, scale, row_block=3)
    o2, l2 = _brute(q, k, v, causal, scale)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=TOL)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=TOL)


# --------------------------------------------------------------------------
# invariants and closed forms
# --------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
def test_weights_sum_to_one(causal):
    """V = 1 everywhere gives out = 1; and sum_j exp(s_ij - lse_i) = 1."""
    B, S, H, D = 1, 33, 2, 8
    q, k = _rand((B, S, H, D), 4), _rand((B, S, H, D), 5)
    ones = np.ones((B, S, H, D))
    out, lse = attention_naive(q, k, ones, causal, 0.4)
    np.testing.assert_allclose(out, 1.0, rtol=0, atol=TOL)
    s = 0.4 * np.einsum("bihd,bjhd->bhij", q, k)
    if causal:
        s = np.where(np.tril(np.ones((S, S), bool)), s, -np.inf)
    tot = np.exp(s - lse[..., None]).sum(-1)
    np.testing.assert_allclose(tot, 1.0, rtol=0, atol=TOL)


@pytest.mark.parametrize("causal", [False, True])
def test_identical_keys_give_mean_of_values(causal):
    B, S, H, D = 2, 20, 2, 4
    q = _rand((B, S, H, D), 6)
    kk = _rand((D,), 7)
    k = np.broadcast_to(kk, (B, S, H, D)).copy()
    v = _rand((B, S, H, D), 8)
    scale = 0.9
    out, lse = attention_naive(q, k, v, causal, scale)
    for i in range(S):
        n = i + 1 if causal else S
        np.testing.assert_allclose(out[:, i], v[:, :n].mean(axis=1), atol=TOL)
        want = scale * (q[:, i] @ kk) + math.log(n)          # [B, H]
        np.testing.assert_allclose(lse[:, :, i], want, atol=TOL)


def test_causal_first_row_is_first_value():
    B, S, H, D = 2, 16, 3, 5
    q, k, v = (_rand((B, S, H, D), s) for s in (9, 10, 11))
    out, lse = attention_naive(q, k, v, True, 0.3)
    np.testing.assert_array_equal(out[:, 0], v[:, 0])
    np.testing.assert_allclose(lse[:, :, 0],
                               0.3 * np.einsum("bhd,bhd->bh", q[:, 0], k[:, 0]),
                               atol=TOL)


@pytest.mark.parametrize("causal", [False, True])
def test_zero_scale_is_uniform_mean(causal):
    B, S, H, D = 1, 12, 2, 3
    q, k, v = (_rand((B, S, H, D), s) for s in (12, 13, 14))
    out, lse = attention_naive(q, k, v, causal, 0.0)
    for i in range(S):
        n = i + 1 if causal else S
        np.testing.assert_allclose(out[:, i], v[:, :n].mean(axis=1), atol=TOL)
        np.testing.assert_allclose(lse[:, :, i], math.log(n), atol=TOL)


def test_noncausal_permutation_invariance():
    B, S, H, D = 1, 24, 2, 6
    q, k, v = (_rand((B, S, H, D), s) for s in (15, 16, 17))
    perm = np.random.default_rng(18).permutation(S)
    o1, l1 = attention_naive(q, k, v, False, 0.5)
    o2, l2 = attention_naive(q, k[:, perm], v[:, perm], False, 0.5)
    np.testing.assert_allclose(o1, o2, atol=TOL)
    np.testing.assert_allclose(l1, l2, atol=TOL)


def test_causal_rows_ignore_future_keys():
    B, S, H, D = 1, 24, 2, 6
    q, k, v = (_rand((B, S, H, D), s) for s in (19, 20, 21))
    cut = 10
    k2, v2 = k.copy(), v.copy()
    k2[:, cut + 1:] = _rand(k2[:, cut + 1:].shape, 22)
    v2[:, cut + 1:] = _rand(v2[:, cut + 1:].shape, 23)
    o1, l1 = attention_naive(q, k, v, True, 0.5)
    o2, l2 = attention_naive(q, k2, v2, True, 0.5)
    np.testing.assert_array_equal(o1[:, :cut + 1], o2[:, :cut + 1])
    np.testing.assert_array_equal(l1[:, :, :cut + 1], l2[:, :, :cut + 1])
    assert np.abs(o1[:, cut + 1:] - o2[:, cut + 1:]).max() > 1e-3


@pytest.mark.parametrize("causal", [False, True])
def test_gqa_equals_mha_with_repeated_heads(causal):
    B, S, Hq, Hkv, D = 1, 17, 8, 2, 4
    q = _rand((B, S, Hq, D), 24)
    k, v = _rand((B, S, Hkv, D), 25), _rand((B, S, Hkv, D), 26)
    o1, l1 = attention_naive(q, k, v, causal, 0.5)
    rep = Hq // Hkv
    k_rep = np.repeat(k, rep, axis=2)          # head h reads kv head h // rep
    v_rep = np.repeat(v, rep, axis=2)
    o2, l2 = attention_naive(q, k_rep, v_rep, causal, 0.5)
    np.testing.assert_allclose(o1, o2, atol=TOL)
    np.testing.assert_allclose(l1, l2, atol=TOL)
    # and it is not the "h mod H_kv" grouping
    k_mod = np.concatenate([k] * rep, axis=2)
    v_mod = np.concatenate([v] * rep, axis=2)
    o3, _ = attention_naive(q, k_mod, v_mod, causal, 0.5)
    assert np.abs(o1 - o3).max() > 1e-3


def test_rows_and_partial_match_full():
    B, S, H, D = 2, 40, 2, 4
    q, k, v = (_rand((B, S, H, D), s) for s in (27, 28, 29))
    o, l = attention_naive(q, k, v, True, 0.6)
    rows = [0, 5, 39, 17]
    o2, l2 = attention_rows(q, k, v, True, 0.6, rows)
    np.testing.assert_allclose(o2, o[:, rows], atol=TOL)
    np.testing.assert_allclose(l2, l[:, :, rows], atol=TOL)
    # keys strictly after the query: no allowed key -> o = 0, lse = -inf
    o3, l3 = partial_attention(q, k, v, True, 0.6, [3], [10, 11])
    assert np.all(o3 == 0) and np.all(np.isneginf(l3))


# --------------------------------------------------------------------------
# ring restatement: the result does not depend on P or on the chunk order
# --------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("order", [0, 1])
@pytest.mark.parametrize("P", [1, 2, 4, 8])
@pytest.mark.parametrize("S", [48, 45])          # 45: uneven chunks, padded
def test_ring_equals_full_attention(causal, order, P, S):
    B, Hq, Hkv, D = 1, 4, 2, 8
    q = _rand((B, S, Hq, D), 30)
    k, v = _rand((B, S, Hkv, D), 31), _rand((B, S, Hkv, D), 32)
    o1, l1 = attention_naive(q, k, v, causal, 0.35)
    o2, l2 = ring_attention(q, k, v, causal, 0.35, P, order)
    np.testing.assert_allclose(o2, o1, rtol=0, atol=TOL)
    np.testing.assert_allclose(l2, l1, rtol=0, atol=TOL)


def test_ring_partials_merge_to_full():
    B, S, H, D = 1, 32, 2, 4
    q, k, v = (_rand((B, S, H, D), s) for s in (33, 34, 35))
    o, l, parts = ring_attention(q, k, v, True, 0.5, 4, 1, return_partials=True)
    o2, l2 = lse_merge_n([p[0] for p in parts], [p[1] for p in parts])
    np.testing.assert_allclose(o2, o, atol=TOL)
    np.testing.assert_allclose(l2, l, atol=TOL)
    o1, l1 = attention_naive(q, k, v, True, 0.5)
    np.testing.assert_allclose(o, o1, atol=TOL)


# --------------------------------------------------------------------------
# merge algebra
# --------------------------------------------------------------------------

def _parts(n, seed, with_empty=True):
    rng = np.random.default_rng(seed)
    B, S, H, D = 1, 9, 3, 4
    os_ = [rng.standard_normal((B, S, H, D)) for _ in range(n)]
    ls = [rng.uniform(-20, 20, (B, H, S)) for _ in range(n)]
    if with_empty:
        ls[0][0, 1, 2] = -np.inf
        for t in range(n):
            ls[t][0, 2, 5] = -np.inf
            os_[t][0, 5, 2] = 0.0
    return os_, ls


def test_merge_commutes_and_folds_like_a_tree():
    os_, ls = _parts(4, 40)
    ab = lse_merge(os_[0], ls[0], os_[1], ls[1])
    ba = lse_merge(os_[1], ls[1], os_[0], ls[0])
    np.testing.assert_allclose(ab[0], ba[0], atol=TOL)
    np.testing.assert_allclose(ab[1], ba[1], atol=TOL)
    seq = (os_[0], ls[0])
    for t in range(1, 4):
        seq = lse_merge(seq[0], seq[1], os_[t], ls[t])
    cd = lse_merge(os_[2], ls[2], os_[3], ls[3])
    tree = lse_merge(ab[0], ab[1], cd[0], cd[1])
    nway = lse_merge_n(os_, ls)
    for got in (tree, nway):
        np.testing.assert_allclose(got[0], seq[0], atol=TOL)
        np.testing.assert_allclose(got[1], seq[1], atol=TOL)
    # the all-empty row merges to (0, -inf)
    assert np.isneginf(nway[1][0, 2, 5]) and np.all(nway[0][0, 5, 2] == 0)


def test_merge_closed_form_two_sets():
    """Splitting the keys of one row into two sets and merging the two
    partial attentions gives attention over all the keys."""
    B, S, H, D = 1, 30, 2, 5
    q, k, v = (_rand((B, S, H, D), s) for s in (41, 42, 43))
    rows = np.arange(S)
    ka = np.arange(0, S, 3)
    kb = np.setdiff1d(np.arange(S), ka)
    oa, la = partial_attention(q, k, v, False, 0.5, rows, ka)
    ob, lb = partial_attention(q, k, v, False, 0.5, rows, kb)
    o, l = lse_merge(oa, la, ob, lb)
    o1, l1 = attention_naive(q, k, v, False, 0.5)
    np.testing.assert_allclose(o, o1, atol=TOL)
    np.testing.assert_allclose(l, l1, atol=TOL)


# --------------------------------------------------------------------------
# schedule: every allowed pair exactly once, classes by brute force
# --------------------------------------------------------------------------

def _pairs(ranges_q, ranges_k):
    qs = np.concatenate([np.arange(s, s + n) for s, n in ranges_q])
    ks = np.concatenate([np.arange(s, s + n) for s, n in ranges_k])
    return qs, ks


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("order", [0, 1])
@pytest.mark.parametrize("S,P", [(16, 2), (48, 4), (64, 8), (24, 3), (10, 4), (7, 3),
                                 (5, 4), (3, 8)])
def test_schedule_covers_every_pair_once(S, P, causal, order):
    segs = rank_segments(S, P, order)
    parts = P if order == 0 else 2 * P
    L = -(-S // parts)                       # padded to a multiple of the split
    owner = np.full(S, -1)
    starts = []
    for r, lst in enumerate(segs):
        for s, n in lst:
            assert s % L == 0 and n == max(0, min(L, S - s))
            starts.append(s)
            assert np.all(owner[s:s + n] == -1)
            owner[s:s + n] = r
    assert sorted(starts) == [i * L for i in range(parts)]
    assert np.all(owner >= 0)
    count = np.zeros((S, S), int)
    for e in ring_schedule(S, P, causal, order):
        assert e["src"] == (e["rank"] - e["step"]) % P
        qs, ks = _pairs(e["q"], e["kv"])
        allowed = (ks[None, :] <= qs[:, None]) if causal else np.ones(
            (len(qs), len(ks)), bool)
        if e["cls"] == SKIP:
            assert not allowed.any()
        elif e["cls"] == FULL:
            assert allowed.all()
        else:
            assert allowed.any() and not allowed.all()
        count[np.ix_(qs, ks)] += 1
    assert np.all(count == 1)     # every (query, key) pair visited exactly once


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("order", [0, 1])
@pytest.mark.parametrize("S,P,T", [(64, 2, 8), (96, 4, 5), (40, 2, 16),
                                   (128, 8, 4), (50, 4, 4), (37, 2, 5), (9, 4, 2)])
def test_tile_visits_by_brute_force(S, P, T, causal, order):
    visits = tile_visits(S, P, causal, order, T)
    segs = sorted((s, n, r) for r, lst in enumerate(rank_segments(S, P, order))
                  for s, n in lst)
    L = -(-S // (P if order == 0 else 2 * P))
    nt = -(-L // T)

    def tile_range(tid):
        g, i = divmod(tid, nt)
        lo = segs[g][0] + i * T
        return lo, max(0, min(T, segs[g][0] + L - lo, S - lo)), segs[g][2]

    covered = np.zeros((S, S), int)
    for qid, seq in enumerate(visits):
        qlo, qn, r = tile_range(qid)
        steps = [e[0] for e in seq]
        assert steps == sorted(steps)                 # ring order
        for t, src, kid, cls in seq:
            klo, kn, kr = tile_range(kid)
            assert kr == src == (r - t) % P
            qs, ks = np.arange(qlo, qlo + qn), np.arange(klo, klo + kn)
            allowed = (ks[None, :] <= qs[:, None]) if causal else np.ones(
                (qn, kn), bool)
            assert allowed.any()
            assert (cls == FULL) == bool(allowed.all())
            covered[np.ix_(qs, ks)] += allowed
    want = np.tril(np.ones((S, S), int)) if causal else np.ones((S, S), int)
    np.testing.assert_array_equal(covered, want)
