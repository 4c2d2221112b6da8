"""Parity of packed variable-length batches (ring_attn_fwd_varlen,
ring_attn_bwd_varlen) with the float64 oracle, through the C ABI.

Sequences of very different lengths share one launch: empty and one-token
sequences, lengths that are not multiples of the tile or of the split, and
the longest sequence sizing the grid. Every sequence is its own ring problem.
"""

import numpy as np
import pytest
import torch

import oracle
from sequence_exact_attention_gb300 import binding

from helpers import assert_close

pytestmark = pytest.mark.gpu

LENGTHS = [300, 0, 1, 777, 128, 1000]


def _packed(lengths, H_q, H_kv, D, dtype, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    total = int(sum(lengths))
    q = (torch.randn(total, H_q, D, generator=g) * std).to(dtype)
    k = (torch.randn(total, H_kv, D, generator=g) * std).to(dtype)
    v = (torch.randn(total, H_kv, D, generator=g) * std).to(dtype)
    dout = (torch.randn(total, H_q, D, generator=g) * std).to(dtype)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    return q, k, v, dout, cu


def _lse_close(got, want, kind):
    # rows of empty sequences do not exist; every other lse entry is finite
    assert_close(got, want, kind, "lse")


@pytest.mark.parametrize("dtype,D,P,causal,order", [
    ("bf16", 128, 4, True, "zigzag"),
    ("bf16", 64, 3, False, "contiguous"),
    ("bf16", 128, 1, True, "contiguous"),
    ("f32", 64, 2, True, "zigzag"),
])
def test_varlen_forward_matches_oracle(dtype, D, P, causal, order):
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    q, k, v, _, cu = _packed(LENGTHS, 4, 2, D, tdt, seed=4000 + D + P)
    dev = torch.device("cuda")
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out, lse = binding.ring_attn_fwd_varlen(q.to(dev), k.to(dev), v.to(dev),
                                            torch.from_numpy(cu).to(dev), max(LENGTHS), P,
                                            causal, order=order, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    scale = 1.0 / np.sqrt(D)
    want_o, want_l = oracle.attention_varlen(q, k, v, cu, causal, scale)
    assert_close(out, want_o, dtype, "out")
    _lse_close(lse, want_l, dtype)


def test_varlen_single_sequence_equals_fixed_length_call():
    """One packed sequence is the same computation as the BSHD entry point."""
    S, H, D, P = 1000, 4, 128, 4
    q, k, v, _, cu = _packed([S], H, H, D, torch.bfloat16, seed=4100)
    dev = torch.device("cuda")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o1, l1 = binding.ring_attn_fwd_varlen(qd, kd, vd, torch.from_numpy(cu).to(dev), S, P, True,
                                          order="zigzag")
    o2, l2 = binding.ring_attn_fwd(qd[None], kd[None], vd[None], P, True, order="zigzag")
    torch.cuda.synchronize()
    assert torch.equal(o1, o2[0])
    assert torch.equal(l1, l2[0])


@pytest.mark.parametrize("P,order,causal", [(4, "zigzag", True), (3, "contiguous", False)])
def test_varlen_backward_matches_oracle(P, order, causal):
    D = 128
    q, k, v, dout, cu = _packed(LENGTHS, 4, 2, D, torch.bfloat16, seed=4200 + P)
    dev = torch.device("cuda")
    qd, kd, vd, dd = (t.to(dev) for t in (q, k, v, dout))
    cud = torch.from_numpy(cu).to(dev)
    out, lse = binding.ring_attn_fwd_varlen(qd, kd, vd, cud, max(LENGTHS), P, causal, order=order)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    dq, dk, dv = binding.ring_attn_bwd_varlen(qd, kd, vd, out, lse, dd, cud, max(LENGTHS), P,
                                              causal, order=order, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rq, rk, rv = oracle.attention_backward_varlen(q, k, v, dout, cu, causal, 1.0 / np.sqrt(D))
    for name, got, want in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        g = got.double().cpu().numpy()
        err = np.abs(g - want)
        rel_max = err.max() / np.abs(want).max()
        rel_mean = err.mean() / np.abs(want).mean()
        print(f"{name}: {rel_max:.2e} {rel_mean:.2e}")
        # the backward's tolerance (tests/test_gpu_backward.py)
        assert rel_max <= 2e-2 and rel_mean <= 1e-2, (name, rel_max, rel_mean)
