"""Parity of the CUDA ring-attention kernels with the float64 oracle.

Small and medium shapes that span several tiles, ragged tile tails, both
chunk orders, grouped heads, both head sizes, one-token chunks, every single
ring step and the bookkeeping of visited key tiles (compared bit for bit with
the oracle's schedule). Every call goes through the C ABI.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from sequence_exact_attention_gb300 import binding
from sequence_exact_attention_gb300.workloads import AttnWorkload, make_qkv

from helpers import assert_close, decode_visit_log

pytestmark = pytest.mark.gpu

ORDER = {"contiguous": oracle.ORDER_CONTIGUOUS, "zigzag": oracle.ORDER_ZIGZAG}


def _inputs(dtype, B, Hq, Hkv, S, D, P, causal, order, seed, std=1.0, shift=0.0):
    w = AttnWorkload("case", dtype, B, Hq, Hkv, S, D, P, causal, order, std=std,
                     k_shift_odd=shift, seed=seed)
    q, k, v = make_qkv(w)
    return w, q, k, v


def _run(w, q, k, v, step=-1, log=False):
    dev = torch.device("cuda")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    vlog = None
    lay = None
    if log:
        lay = binding.visit_log_layout(w.B, w.H_q, w.S, w.D, w.P, w.dtype, w.order)
        vlog = torch.full((lay["len"],), -7, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out, lse = binding.ring_attn_fwd(qd, kd, vd, w.P, w.causal, w.scale, w.order,
                                     step=step, visit_log=vlog, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, "device-side wait expired"
    return out, lse, vlog, lay


BF16_CASES = [
    # B, Hq, Hkv, S,    D,   P,  causal, order
    (1, 2, 2, 512, 128, 2, True, "contiguous"),
    (1, 2, 2, 512, 128, 2, True, "zigzag"),
    (2, 4, 2, 768, 128, 4, True, "zigzag"),        # GQA; halves of 96 rows (ragged)
    (1, 2, 1, 960, 64, 3, False, "contiguous"),    # D=64, chunks of 320 (128+128+64)
    (1, 3, 3, 1000, 128, 5, True, "contiguous"),   # chunks of 200 (128+72)
    (1, 2, 2, 384, 128, 1, True, "contiguous"),    # P = 1: plain attention
    (1, 2, 2, 16, 128, 16, True, "contiguous"),    # one-token chunks
    (1, 2, 2, 64, 64, 32, True, "zigzag"),         # one-token halves
    (1, 4, 4, 2048, 128, 8, True, "zigzag"),       # halves of exactly 128
    (2, 4, 1, 1024, 64, 4, True, "zigzag"),        # MQA, D=64
    (1, 2, 2, 1536, 128, 4, False, "zigzag"),      # non-causal zig-zag
    (1, 2, 2, 130, 128, 2, True, "contiguous"),    # S not a multiple of 128
    # uneven lengths: S padded to a multiple of the split, padding masked
    (1, 3, 3, 1000, 128, 3, True, "contiguous"),   # chunks of 334 (last 332 tokens)
    (1, 2, 2, 1001, 128, 4, True, "zigzag"),       # halves of 126 (last 119)
    (2, 4, 2, 300, 64, 8, True, "zigzag"),         # halves of 19 (last 15)
    (1, 2, 2, 5, 128, 4, True, "contiguous"),      # chunks of 2: the last is empty
    (1, 2, 1, 700, 128, 3, False, "zigzag"),       # non-causal, halves of 117
    (1, 2, 2, 1, 128, 1, True, "contiguous"),      # a single token
    (2, 2, 1, 3, 64, 4, True, "zigzag"),           # 3 tokens over 8 halves: most empty
]


@pytest.mark.parametrize("case", BF16_CASES, ids=lambda c: "-".join(map(str, c)))
def test_bf16_matches_oracle(case):
    B, Hq, Hkv, S, D, P, causal, order = case
    w, q, k, v = _inputs("bf16", B, Hq, Hkv, S, D, P, causal, order,
                         seed=2000 + BF16_CASES.index(case))
    out, lse, vlog, lay = _run(w, q, k, v, log=True)
    want_o, want_l = oracle.attention_naive(q, k, v, causal, w.scale)
    assert_close(out, want_o, "bf16", "out")
    assert_close(lse, want_l, "bf16", "lse")
    # bookkeeping: the visited key tiles, in order, per query tile
    got = decode_visit_log(vlog, B, Hq, lay["n_query_tiles"], lay["stride"])
    want = oracle.tile_visits(S, P, causal, ORDER[order], lay["tile_rows"])
    for b in range(B):
        for h in range(Hq):
            assert got[b][h] == want, f"visit log differs at b={b} h={h}"


F32_CASES = [
    (1, 2, 2, 256, 64, 4, False, "contiguous"),    # the float32 workload's shape
    (1, 2, 2, 256, 64, 4, True, "contiguous"),
    (2, 4, 2, 384, 128, 3, True, "zigzag"),        # halves of 64
    (1, 2, 1, 200, 64, 2, True, "contiguous"),     # chunks of 100 (64+36)
    (1, 2, 2, 24, 128, 12, True, "zigzag"),        # one-token halves
    (1, 2, 2, 250, 64, 4, True, "contiguous"),     # uneven: chunks of 63 (last 61)
    (1, 2, 2, 99, 128, 4, True, "zigzag"),         # uneven: halves of 13 (last 8)
    (1, 2, 2, 1, 64, 1, False, "contiguous"),      # a single token
    (1, 2, 2, 3, 64, 4, True, "contiguous"),       # 3 tokens over 4 chunks: one empty
]


@pytest.mark.parametrize("case", F32_CASES, ids=lambda c: "-".join(map(str, c)))
def test_f32_matches_oracle(case):
    B, Hq, Hkv, S, D, P, causal, order = case
    w, q, k, v = _inputs("f32", B, Hq, Hkv, S, D, P, causal, order,
                         seed=3000 + F32_CASES.index(case))
    out, lse, vlog, lay = _run(w, q, k, v, log=True)
    want_o, want_l = oracle.attention_naive(q, k, v, causal, w.scale)
    assert_close(out, want_o, "f32", "out")
    assert_close(lse, want_l, "f32", "lse")
    got = decode_visit_log(vlog, B, Hq, lay["n_query_tiles"], lay["stride"])
    want = oracle.tile_visits(S, P, causal, ORDER[order], lay["tile_rows"])
    for b in range(B):
        for h in range(Hq):
            assert got[b][h] == want


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_result_does_not_depend_on_P(dtype):
    """The sequence-parallel result equals the P = 1 result (same inputs)."""
    S = 1024
    w1, q, k, v = _inputs(dtype, 1, 4, 2, S, 128, 1, True, "contiguous", seed=77)
    want_o, want_l = oracle.attention_naive(q, k, v, True, w1.scale)
    outs = []
    for P in (1, 2, 4, 8):
        for order in ("contiguous", "zigzag"):
            w = w1.scaled(P=P, order=order)
            out, lse, _, _ = _run(w, q, k, v)
            assert_close(out, want_o, dtype, f"out P={P} {order}")
            assert_close(lse, want_l, dtype, f"lse P={P} {order}")
            outs.append(out.float().cpu())
    ref = outs[0]
    for o in outs[1:]:
        assert (o - ref).abs().max().item() <= (1e-2 if dtype == "bf16" else 1e-5)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("order", ["contiguous", "zigzag"])
@pytest.mark.parametrize("S", [768, 700])      # 700: uneven chunks
def test_single_steps_merge_to_full(dtype, order, S):
    """Each ring step alone gives the oracle's per-step partial; folding the
    partials with the merge kernel gives full attention."""
    P = 3
    w, q, k, v = _inputs(dtype, 1, 4, 2, S, 64, P, True, order, seed=91)
    want_o, want_l, parts = oracle.ring_attention(q, k, v, True, w.scale, P,
                                                  ORDER[order], return_partials=True)
    got_o, got_l = [], []
    for t in range(P):
        o_t, l_t, _, _ = _run(w, q, k, v, step=t)
        assert o_t.dtype == torch.float32
        assert_close(o_t, parts[t][0], dtype, f"partial out step {t}")
        assert_close(l_t, parts[t][1], dtype, f"partial lse step {t}")
        got_o.append(o_t)
        got_l.append(l_t)
    out, lse = binding.attn_lse_merge_n(got_o, got_l)
    assert_close(out, want_o, dtype, "merged out")
    assert_close(lse, want_l, dtype, "merged lse")
    # pairwise fold in ring order gives the same
    acc_o, acc_l = got_o[0], got_l[0]
    for t in range(1, P):
        acc_o, acc_l = binding.attn_lse_merge(acc_o, acc_l, got_o[t], got_l[t])
    assert_close(acc_o, want_o, dtype, "folded out")


def test_running_max_stress_bf16():
    """Every other key row shifted by +3 (the GQA workload's stress) on a
    small shape: the running maximum moves a lot between tiles."""
    w, q, k, v = _inputs("bf16", 1, 4, 1, 2048, 128, 4, True, "contiguous",
                         seed=5, shift=3.0)
    out, lse, _, _ = _run(w, q, k, v)
    want_o, want_l = oracle.attention_naive(q, k, v, True, w.scale)
    assert_close(out, want_o, "bf16", "out")
    assert_close(lse, want_l, "bf16", "lse")


def test_large_scores_trigger_rescale_bf16():
    """Scores growing along the sequence force many lazy rescales."""
    S = 1024
    w, q, k, v = _inputs("bf16", 1, 2, 2, S, 64, 2, True, "zigzag", seed=6)
    ramp = torch.linspace(0, 6, S).view(1, S, 1, 1)
    k = (k.float() + ramp).to(torch.bfloat16)
    q = (q.float().abs() + 1).to(torch.bfloat16)
    out, lse, _, _ = _run(w, q, k, v)
    want_o, want_l = oracle.attention_naive(q, k, v, True, w.scale)
    assert_close(out, want_o, "bf16", "out")
    assert_close(lse, want_l, "bf16", "lse")


def test_plain_entry_point_bf16():
    w, q, k, v = _inputs("bf16", 1, 2, 2, 512, 128, 4, True, "contiguous", seed=8)
    dev = torch.device("cuda")
    out = torch.empty(1, 512, 2, 128, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(1, 2, 512, dtype=torch.float32, device=dev)
    binding.ring_attn_fwd_plain(q.to(dev), k.to(dev), v.to(dev), out, lse, 4, True, w.scale)
    torch.cuda.synchronize()
    want_o, want_l = oracle.attention_naive(q, k, v, True, w.scale)
    assert_close(out, want_o, "bf16", "out")
    assert_close(lse, want_l, "bf16", "lse")


def test_errors_raise_and_launch_nothing():
    dev = torch.device("cuda")
    q = torch.zeros(1, 100, 2, 128, dtype=torch.bfloat16, device=dev)
    with pytest.raises(binding.RingAttnError) as e:
        binding.ring_attn_fwd(q[:, :, :1].contiguous(), q, q, 2, True)   # H_q % H_kv
    assert e.value.status == 2
    with pytest.raises(binding.RingAttnError) as e:
        binding.ring_attn_fwd(q, q, q, 2, True, order="zigzag", step=5)
    assert e.value.status == 10
    q96 = torch.zeros(1, 64, 2, 96, dtype=torch.bfloat16, device=dev)
    with pytest.raises(binding.RingAttnError) as e:
        binding.ring_attn_fwd(q96, q96, q96, 2, True)
    assert e.value.status == 3
    with pytest.raises(ValueError):
        binding.ring_attn_fwd(q.cpu(), q, q, 2, True)
