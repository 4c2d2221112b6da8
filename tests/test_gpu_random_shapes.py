"""Parity with the float64 oracle on seeded random shapes, through the C ABI.

The hand-picked cases elsewhere cover the boundaries one at a time; here the
shapes are drawn at random (a fixed seed per case, so every run checks the
same ones): batch, grouped heads, head size, any length from a single token
up to several tiles per chunk, 1-8 virtual ranks, both chunk orders, with and
without the causal mask. Every output element is compared: the forward's out
and lse (bf16 tensor-core path and float32 CUDA-core path), the backward's dq,
dk and dv, and packed batches of sequences of random lengths (empty ones
included), forward and backward.
"""

import numpy as np
import pytest
import torch

import oracle
from oracle.backward import attention_backward
from sequence_exact_attention_gb300 import binding
from sequence_exact_attention_gb300.workloads import AttnWorkload, make_dout, make_qkv

from helpers import assert_close
from test_gpu_backward import check as check_grad

pytestmark = pytest.mark.gpu

ORDERS = ("contiguous", "zigzag")


def _draw(seed, s_max):
    rng = np.random.default_rng(seed)
    H_kv = int(rng.integers(1, 3))
    grp = int(rng.choice([1, 2, 4]))
    return (int(rng.integers(1, 3)), H_kv * grp, H_kv, int(rng.integers(1, s_max)),
            int(rng.choice([64, 128])), int(rng.integers(1, 9)), bool(rng.integers(0, 2)),
            ORDERS[int(rng.integers(0, 2))])


def _ids(cases):
    return ["B{}-H{}-{}-S{}-D{}-P{}-{}-{}".format(b, hq, hk, s, d, p, "c" if c else "n", o[0])
            for b, hq, hk, s, d, p, c, o in cases]


FWD = [_draw(7000 + i, 1400) for i in range(96)]
BWD = [_draw(8000 + i, 700) for i in range(24)]
F32 = [_draw(6000 + i, 400) for i in range(12)]


def _forward_case(case, seed):
    B, H_q, H_kv, S, D, P, causal, order = case
    w = AttnWorkload("rand", "bf16", B, H_q, H_kv, S, D, P, causal, order, seed=seed)
    q, k, v = make_qkv(w)
    dev = torch.device("cuda")
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out, lse = binding.ring_attn_fwd(q.to(dev), k.to(dev), v.to(dev), P, causal, w.scale, order,
                                     dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    want_o, want_l = oracle.attention_naive(q, k, v, causal, w.scale)
    assert_close(out, want_o, "bf16", "out")
    assert_close(lse, want_l, "bf16", "lse")


@pytest.mark.parametrize("case", FWD, ids=_ids(FWD))
def test_random_forward_matches_oracle(case):
    _forward_case(case, 7500 + FWD.index(case))


@pytest.mark.parametrize("case", F32, ids=_ids(F32))
def test_random_f32_forward_matches_oracle(case):
    B, H_q, H_kv, S, D, P, causal, order = case
    w = AttnWorkload("rand", "f32", B, H_q, H_kv, S, D, P, causal, order,
                     seed=6500 + F32.index(case))
    q, k, v = make_qkv(w)
    dev = torch.device("cuda")
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out, lse = binding.ring_attn_fwd(q.to(dev), k.to(dev), v.to(dev), P, causal, w.scale, order,
                                     dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    want_o, want_l = oracle.attention_naive(q, k, v, causal, w.scale)
    assert_close(out, want_o, "f32", "out")
    assert_close(lse, want_l, "f32", "lse")


@pytest.mark.parametrize("case", BWD, ids=_ids(BWD))
def test_random_backward_matches_oracle(case):
    B, H_q, H_kv, S, D, P, causal, order = case
    w = AttnWorkload("rand", "bf16", B, H_q, H_kv, S, D, P, causal, order,
                     seed=8500 + BWD.index(case))
    q, k, v = make_qkv(w)
    dout = make_dout(w)
    dev = torch.device("cuda")
    qd, kd, vd, dd = (t.to(dev) for t in (q, k, v, dout))
    out, lse = binding.ring_attn_fwd(qd, kd, vd, P, causal, w.scale, order)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    dq, dk, dv = binding.ring_attn_bwd(qd, kd, vd, out, lse, dd, P, causal, w.scale, order,
                                       dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rq, rk, rv = attention_backward(q, k, v, dout, causal, w.scale)
    check_grad("dq", dq, rq)
    check_grad("dk", dk, rk)
    check_grad("dv", dv, rv)


def _draw_pack(seed):
    rng = np.random.default_rng(seed)
    lengths = [int(n) for n in rng.integers(0, 900, int(rng.integers(2, 7)))]
    if max(lengths) == 0:
        lengths[0] = 1
    H_kv = int(rng.integers(1, 3))
    return (lengths, H_kv * int(rng.choice([1, 2])), H_kv, int(rng.choice([64, 128])),
            int(rng.integers(1, 9)), bool(rng.integers(0, 2)), ORDERS[int(rng.integers(0, 2))])


PACKS = [_draw_pack(9000 + i) for i in range(16)]
BWD_PACKS = [_draw_pack(9800 + i) for i in range(6)]


def _pack_inputs(case, seed):
    lengths, H_q, H_kv, D, P, causal, order = case
    g = torch.Generator().manual_seed(seed)
    total = sum(lengths)
    q = torch.randn(total, H_q, D, generator=g).to(torch.bfloat16)
    k = torch.randn(total, H_kv, D, generator=g).to(torch.bfloat16)
    v = torch.randn(total, H_kv, D, generator=g).to(torch.bfloat16)
    dout = torch.randn(total, H_q, D, generator=g).to(torch.bfloat16)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    return q, k, v, dout, cu


@pytest.mark.parametrize("case", PACKS, ids=[f"pack{i}" for i in range(len(PACKS))])
def test_random_packed_forward_matches_oracle(case):
    lengths, H_q, H_kv, D, P, causal, order = case
    q, k, v, _, cu = _pack_inputs(case, 9500 + PACKS.index(case))
    dev = torch.device("cuda")
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out, lse = binding.ring_attn_fwd_varlen(q.to(dev), k.to(dev), v.to(dev),
                                            torch.from_numpy(cu).to(dev), max(lengths), P,
                                            causal, order=order, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    want_o, want_l = oracle.attention_varlen(q, k, v, cu, causal, 1.0 / np.sqrt(D))
    assert_close(out, want_o, "bf16", "out")
    assert_close(lse, want_l, "bf16", "lse")


@pytest.mark.parametrize("case", BWD_PACKS, ids=[f"pack{i}" for i in range(len(BWD_PACKS))])
def test_random_packed_backward_matches_oracle(case):
    lengths, H_q, H_kv, D, P, causal, order = case
    q, k, v, dout, cu = _pack_inputs(case, 9900 + BWD_PACKS.index(case))
    dev = torch.device("cuda")
    qd, kd, vd, dd = (t.to(dev) for t in (q, k, v, dout))
    cud = torch.from_numpy(cu).to(dev)
    out, lse = binding.ring_attn_fwd_varlen(qd, kd, vd, cud, max(lengths), P, causal, order=order)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    dq, dk, dv = binding.ring_attn_bwd_varlen(qd, kd, vd, out, lse, dd, cud, max(lengths), P,
                                              causal, order=order, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rq, rk, rv = oracle.attention_backward_varlen(q, k, v, dout, cu, causal, 1.0 / np.sqrt(D))
    check_grad("dq", dq, rq)
    check_grad("dk", dk, rk)
    check_grad("dv", dv, rv)


MEDIUM = [(b, hq, hk, 2000 + s, d, p, c, o)
          for b, hq, hk, s, d, p, c, o in (_draw(7700 + i, 2500) for i in range(6))]


@pytest.mark.parametrize("case", MEDIUM, ids=_ids(MEDIUM))
def test_random_medium_forward_matches_oracle(case):
    """Lengths of 2000-4500: walks of up to 36 key tiles a block, so every
    K/V slot is refilled many times over."""
    _forward_case(case, 7800 + MEDIUM.index(case))


CHECKED = [_draw(7900 + i, 900) for i in range(16)]


@pytest.fixture
def release_after():
    prev = binding.use_library("release")
    yield
    binding.use_library(prev)


@pytest.mark.parametrize("case", CHECKED, ids=_ids(CHECKED))
def test_random_shapes_in_range_in_the_checked_build(release_after, case):
    """The bounds-checked build (every index-computed global access tested
    against its tensor's extent) leaves the status word at 0 on random shapes,
    forward and backward, and gives the release build's results bit for bit."""
    B, H_q, H_kv, S, D, P, causal, order = case
    w = AttnWorkload("rand", "bf16", B, H_q, H_kv, S, D, P, causal, order,
                     seed=7950 + CHECKED.index(case))
    q, k, v = (t.cuda() for t in make_qkv(w))
    dout = make_dout(w).cuda()

    def run():
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        out, lse = binding.ring_attn_fwd(q, k, v, P, causal, w.scale, order, dev_status=status)
        grads = binding.ring_attn_bwd(q, k, v, out, lse, dout, P, causal, w.scale, order,
                                      dev_status=status)
        torch.cuda.synchronize()
        return int(status.item()), [out, lse, *grads]

    binding.use_library("release")
    st, want = run()
    assert st == 0
    binding.use_library("debug")
    st, got = run()
    assert st == 0, binding.strerror(st)
    for a, b in zip(got, want):
        assert torch.equal(a, b)
