"""Parity of the tensor-core backward pass (ring_attn_bwd) with the float64
oracle, through the C ABI.

The GPU side gets the seeded bf16 q, k, v and dout, runs the library's own
forward for out and lse, then the backward. The oracle differentiates the
forward definition in float64 from the same bf16 inputs.

Tolerance, from the arithmetic: the kernels round three things to bf16
(unit roundoff u = 2^-9): P before dV += P^T dO, dS before dK and dQ, and
each gradient on output; out (bf16, from the forward) enters delta. Products
are exact and sums are float32. A gradient entry is a weighted sum of many
terms whose rounding errors have random signs, so its error stays within a
few u of the gradient's own scale: max-abs error <= 2e-2 * max|ref| (about
10 u) and mean-abs error <= 1e-2 * mean|ref| (5 u) for each of dq, dk, dv.
The scales have a floor of 1e-2 (far below the gradients' typical size), so
a gradient that is exactly zero -- dq and dk of a single causal token --
is held to an absolute 2e-4 rather than to a division by zero.
"""

import numpy as np
import pytest
import torch

from oracle.backward import attention_backward, backward_rows
from sequence_exact_attention_gb300 import binding
from sequence_exact_attention_gb300.workloads import (AttnWorkload, BWD_WORKLOADS, make_dout,
                                                      make_qkv)

pytestmark = pytest.mark.gpu

REL_MAX, REL_MEAN = 2e-2, 1e-2


def rel_errors(got, want):
    g = got.detach().to("cpu").double().numpy()
    w = np.asarray(want, dtype=np.float64)
    assert g.shape == w.shape
    d = np.abs(g - w)
    assert np.all(np.isfinite(d)), "non-finite gradient"
    return (float(d.max() / max(np.abs(w).max(), 1e-2)),
            float(d.mean() / max(np.abs(w).mean(), 1e-2)))


def check(name, got, want):
    mx, mean = rel_errors(got, want)
    print(f"{name}: max-abs/max|ref| {mx:.2e}, mean-abs/mean|ref| {mean:.2e}")
    assert mx <= REL_MAX and mean <= REL_MEAN, (
        f"{name}: relative max {mx:.3e} (tol {REL_MAX}), mean {mean:.3e} (tol {REL_MEAN})")


def run_gpu(w, q, k, v, dout):
    dev = torch.device("cuda")
    qd, kd, vd, dd = (t.to(dev) for t in (q, k, v, dout))
    out, lse = binding.ring_attn_fwd(qd, kd, vd, w.P, w.causal, w.scale, w.order)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    dq, dk, dv = binding.ring_attn_bwd(qd, kd, vd, out, lse, dd, w.P, w.causal, w.scale, w.order,
                                       dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return dq, dk, dv


CASES = [
    # name, B, H_q, H_kv, S, D, P, causal, order
    ("s512_causal", 1, 2, 2, 512, 128, 2, True, "contiguous"),
    ("s1024_zigzag_gqa", 1, 4, 2, 1024, 128, 4, True, "zigzag"),
    ("s384_noncausal_d64", 1, 2, 1, 384, 64, 3, False, "contiguous"),
    ("s600_ragged_zigzag", 1, 2, 2, 600, 128, 4, True, "zigzag"),     # halves of 75 rows
    ("s1000_ragged_d64", 2, 2, 2, 1000, 64, 2, True, "contiguous"),   # 500 = 3 x 128 + 116
    ("s256_p1_noncausal", 1, 3, 3, 256, 128, 1, False, "contiguous"),
    ("s1001_uneven_zigzag", 1, 2, 2, 1001, 128, 4, True, "zigzag"),   # halves of 126
    ("s5_uneven_empty_chunk", 1, 2, 1, 5, 64, 4, True, "contiguous"),  # last chunk empty
    ("s700_uneven_noncausal", 1, 2, 2, 700, 128, 3, False, "zigzag"),
    ("s1_single_token", 1, 2, 2, 1, 128, 1, True, "contiguous"),
    ("s3_mostly_empty", 2, 2, 1, 3, 64, 4, True, "zigzag"),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_backward_matches_oracle(case):
    name, B, H_q, H_kv, S, D, P, causal, order = case
    w = AttnWorkload(name, "bf16", B, H_q, H_kv, S, D, P, causal, order, std=1.0,
                     seed=2000 + CASES.index(case))
    q, k, v = make_qkv(w)
    dout = make_dout(w)
    dq, dk, dv = run_gpu(w, q, k, v, dout)
    rq, rk, rv = attention_backward(q, k, v, dout, causal, w.scale)
    check(f"{name} dq", dq, rq)
    check(f"{name} dk", dk, rk)
    check(f"{name} dv", dv, rv)


def test_backward_is_independent_of_P_and_order():
    base = AttnWorkload("p_indep", "bf16", 1, 2, 2, 1024, 128, 1, True, "contiguous", std=1.0,
                        seed=2100)
    q, k, v = make_qkv(base)
    dout = make_dout(base)
    rq, rk, rv = attention_backward(q, k, v, dout, True, base.scale)
    for P, order in ((1, "contiguous"), (2, "zigzag"), (4, "contiguous"), (8, "zigzag")):
        w = base.scaled(P=P, order=order)
        dq, dk, dv = run_gpu(w, q, k, v, dout)
        check(f"P={P} {order} dq", dq, rq)
        check(f"P={P} {order} dk", dk, rk)
        check(f"P={P} {order} dv", dv, rv)


def test_backward_phases_split_equal_whole_call():
    """Prep, then dK/dV and dQ on two streams at once, equals the single call."""
    w = AttnWorkload("phases", "bf16", 1, 4, 2, 1024, 128, 4, True, "zigzag", std=1.0, seed=2150)
    dev = torch.device("cuda")
    q, k, v = (t.to(dev) for t in make_qkv(w))
    dout = make_dout(w).to(dev)
    out, lse = binding.ring_attn_fwd(q, k, v, w.P, True, w.scale, w.order)
    dq, dk, dv = binding.ring_attn_bwd(q, k, v, out, lse, dout, w.P, True, w.scale, w.order)
    ws = torch.empty(binding.bwd_workspace_bytes(w.B, w.H_q, w.S, w.D, w.P, w.order),
                     dtype=torch.uint8, device=dev)
    dq2, dk2, dv2 = torch.empty_like(dq), torch.empty_like(dk), torch.empty_like(dv)
    kw = dict(dq=dq2, dk=dk2, dv=dv2, workspace=ws)
    main = torch.cuda.current_stream()
    binding.ring_attn_bwd(q, k, v, out, lse, dout, w.P, True, w.scale, w.order,
                          phases=binding.BWD_PREP, stream=main, **kw)
    side = torch.cuda.Stream()
    side.wait_stream(main)
    binding.ring_attn_bwd(q, k, v, out, lse, dout, w.P, True, w.scale, w.order,
                          phases=binding.BWD_DKDV, stream=main, **kw)
    binding.ring_attn_bwd(q, k, v, out, lse, dout, w.P, True, w.scale, w.order,
                          phases=binding.BWD_DQ, stream=side, **kw)
    main.wait_stream(side)
    torch.cuda.synchronize()
    assert torch.equal(dq, dq2) and torch.equal(dk, dk2) and torch.equal(dv, dv2)


def test_backward_headline_shape_sampled():
    """The 32K causal zig-zag shape in the launch configuration the bench
    times, checked on sampled query rows and key rows of two heads."""
    w = BWD_WORKLOADS["bf16_s32k_causal_zigzag_bwd"]
    q, k, v = make_qkv(w)
    dout = make_dout(w)
    dq, dk, dv = run_gpu(w, q, k, v, dout)
    rng = np.random.default_rng(77)
    seg = w.S // (2 * w.P)
    rows = np.unique(np.concatenate([np.arange(0, w.S, seg), np.arange(seg - 1, w.S, seg),
                                     rng.integers(0, w.S, 48)]))
    for h in (0, w.H_q - 1):
        rq, rk, rv = backward_rows(q, k, v, dout, True, w.scale, h, rows, rows)
        hk = h // (w.H_q // w.H_kv)
        check(f"h={h} dq rows", dq[:, rows, h], rq)
        check(f"h={h} dk rows", dk[:, rows, hk], rk)
        check(f"h={h} dv rows", dv[:, rows, hk], rv)


def test_backward_argument_errors():
    w = AttnWorkload("err", "bf16", 1, 2, 2, 256, 64, 2, True, "contiguous", seed=2200)
    q, k, v = (t.cuda() for t in make_qkv(w))
    out, lse = binding.ring_attn_fwd(q, k, v, w.P, True)
    with pytest.raises(binding.RingAttnError):
        binding.ring_attn_bwd(q.float(), k.float(), v.float(), out.float(), lse, out.float(),
                              w.P, True)
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(binding.RingAttnError):
        binding.ring_attn_bwd(q, k, v, out, lse, out, w.P, True, workspace=small)
