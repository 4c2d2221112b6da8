"""Parity of the Ulysses-layout entry point (ring_attn_fwd_ulysses) with the
float64 oracle's Ulysses steps, through the C ABI.

Inputs and outputs stay in the sequence-parallel layout [P, B, C, H, D]; the
two all-to-alls of the method are an index map inside the kernel's loads and
stores.
"""

import numpy as np
import pytest
import torch

import oracle
from sequence_exact_attention_gb300 import binding
from sequence_exact_attention_gb300.workloads import AttnWorkload, make_qkv

from helpers import assert_close

pytestmark = pytest.mark.gpu


def _sharded(t, P):
    # [B, S, H, D] -> [P, B, C, H, D] (zero padding rows), on the device
    return torch.from_numpy(oracle.to_sequence_shards(t.float(), P)).to(t.dtype).cuda()


@pytest.mark.parametrize("dtype,B,Hq,Hkv,S,D,P,causal", [
    ("bf16", 2, 8, 4, 1000, 128, 4, True),      # uneven S: shards of 250 (128 + 122)
    ("bf16", 1, 4, 4, 2048, 128, 2, True),
    ("bf16", 3, 4, 2, 700, 64, 2, False),
    ("f32", 2, 4, 2, 301, 64, 2, True),         # shards of 151, the last holds 150
])
def test_ulysses_matches_oracle(dtype, B, Hq, Hkv, S, D, P, causal):
    w = AttnWorkload("u", dtype, B, Hq, Hkv, S, D, P, causal, "contiguous", seed=5000 + S + B)
    q, k, v = make_qkv(w)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = binding.ring_attn_fwd_ulysses(_sharded(q, P), _sharded(k, P), _sharded(v, P), S,
                                             causal, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    qs, ks, vs = (oracle.to_sequence_shards(t, P) for t in (q, k, v))
    want_o, want_l = oracle.ulysses_attention(qs, ks, vs, S, causal, w.scale)
    C = -(-S // P)
    valid = np.zeros((P, C), bool)                 # rows that hold tokens
    for p in range(P):
        valid[p, :max(0, min(C, S - p * C))] = True
    got_o = out.double().cpu().numpy()[valid.nonzero()[0], :, valid.nonzero()[1]]
    got_l = lse.double().cpu().numpy().transpose(0, 3, 1, 2)[valid]
    assert_close(torch.from_numpy(got_o), want_o[valid.nonzero()[0], :, valid.nonzero()[1]],
                 dtype, "out")
    assert_close(torch.from_numpy(got_l), want_l.transpose(0, 3, 1, 2)[valid], dtype, "lse")


def test_ulysses_one_batch_equals_ring_call():
    """With B = 1 and S a multiple of P the sharded layout is the natural one;
    the results are the contiguous-order ring call's, bit for bit."""
    S, P, H, D = 2048, 4, 4, 128
    w = AttnWorkload("u1", "bf16", 1, H, H, S, D, P, True, "contiguous", seed=5100)
    q, k, v = (t.cuda() for t in make_qkv(w))
    C = S // P
    o1, l1 = binding.ring_attn_fwd_ulysses(q.view(P, 1, C, H, D), k.view(P, 1, C, H, D),
                                           v.view(P, 1, C, H, D), S, True)
    o2, l2 = binding.ring_attn_fwd(q, k, v, P, True, order="contiguous")
    torch.cuda.synchronize()
    assert torch.equal(o1.view(1, S, H, D), o2)
    assert torch.equal(l1.view(P, H, C).permute(1, 0, 2).reshape(1, H, S), l2)


def test_ulysses_backward_one_batch_equals_ring_call():
    S, P, H, D = 2048, 4, 4, 128
    w = AttnWorkload("ub1", "bf16", 1, H, H, S, D, P, True, "contiguous", seed=5200)
    q, k, v = (t.cuda() for t in make_qkv(w))
    dout = torch.randn(1, S, H, D, generator=torch.Generator().manual_seed(5201)).to(
        torch.bfloat16).cuda()
    C = S // P
    sh = lambda t: t.view(P, 1, C, t.shape[2], D)
    o1, l1 = binding.ring_attn_fwd_ulysses(sh(q), sh(k), sh(v), S, True)
    g1 = binding.ring_attn_bwd_ulysses(sh(q), sh(k), sh(v), o1, l1, sh(dout), S, True)
    o2, l2 = binding.ring_attn_fwd(q, k, v, P, True, order="contiguous")
    g2 = binding.ring_attn_bwd(q, k, v, o2, l2, dout, P, True, order="contiguous")
    torch.cuda.synchronize()
    for a, b in zip(g1, g2):
        assert torch.equal(a.view(b.shape), b)


@pytest.mark.parametrize("B,Hq,Hkv,S,D,P", [(2, 8, 4, 1000, 128, 4), (3, 4, 2, 301, 64, 2)])
def test_ulysses_backward_matches_oracle(B, Hq, Hkv, S, D, P):
    w = AttnWorkload("ub", "bf16", B, Hq, Hkv, S, D, P, True, "contiguous", seed=5300 + S)
    q, k, v = make_qkv(w)
    dout = (torch.randn(B, S, Hq, D, generator=torch.Generator().manual_seed(5301)) * 1.0).to(
        torch.bfloat16)
    qs, ks, vs, ds = (_sharded(t, P) for t in (q, k, v, dout))
    out, lse = binding.ring_attn_fwd_ulysses(qs, ks, vs, S, True)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dq, dk, dv = binding.ring_attn_bwd_ulysses(qs, ks, vs, out, lse, ds, S, True,
                                               dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = oracle.attention_backward(q, k, v, dout, True, w.scale)
    for name, got, want in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        g = oracle.from_sequence_shards(got.double().cpu().numpy(), S)
        err = np.abs(g - want)
        rel_max, rel_mean = err.max() / np.abs(want).max(), err.mean() / np.abs(want).mean()
        # the backward's tolerance (tests/test_gpu_backward.py)
        assert rel_max <= 2e-2 and rel_mean <= 1e-2, (name, rel_max, rel_mean)
