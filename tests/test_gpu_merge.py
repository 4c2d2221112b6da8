"""Parity of the standalone log-sum-exp merge kernel with the oracle."""

import numpy as np
import pytest
import torch

import oracle
from sequence_exact_attention_gb300 import binding
from sequence_exact_attention_gb300.workloads import MergeWorkload, make_merge_parts

from helpers import assert_close

pytestmark = pytest.mark.gpu


def _parts(dtype, n, B, H, S, D, seed, empty=True):
    w = MergeWorkload("m", dtype, n, B, H, S, D, seed=seed)
    os_, ls = make_merge_parts(w)
    if empty:
        # rows where some or all partials saw no key
        ls[0][0, 0, 1] = -float("inf")
        for t in range(n):
            ls[t][0, H - 1, S - 1] = -float("inf")
    return os_, ls


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("n", [1, 2, 3, 8, 16])
@pytest.mark.parametrize("D", [64, 128])
def test_merge_n_matches_oracle(dtype, n, D):
    os_, ls = _parts(dtype, n, 2, 3, 100, D, seed=n * 10 + D)
    dev = torch.device("cuda")
    od = [o.to(dev) for o in os_]
    ld = [l.to(dev) for l in ls]
    out, lse = binding.attn_lse_merge_n(od, ld)
    torch.cuda.synchronize()
    want_o, want_l = oracle.lse_merge_n(os_, ls)
    assert_close(out, want_o, dtype, "out")
    assert_close(lse, want_l, "f32" if dtype == "f32" else "bf16", "lse")
    if n > 1:
        assert np.isneginf(lse[0, 2, 99].item())
        assert out[0, 99, 2].abs().max().item() == 0.0


@pytest.mark.parametrize("D", [32, 256])
def test_merge_other_head_dims(D):
    os_, ls = _parts("f32", 4, 1, 2, 70, D, seed=D)
    dev = torch.device("cuda")
    out, lse = binding.attn_lse_merge_n([o.to(dev) for o in os_], [l.to(dev) for l in ls])
    torch.cuda.synchronize()
    want_o, want_l = oracle.lse_merge_n(os_, ls)
    assert_close(out, want_o, "f32", "out")
    assert_close(lse, want_l, "f32", "lse")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_pairwise_merge_in_place(dtype):
    """out and lse may alias the first input."""
    os_, ls = _parts(dtype, 2, 1, 4, 257, 128, seed=3)
    want_o, want_l = oracle.lse_merge(os_[0], ls[0], os_[1], ls[1])
    dev = torch.device("cuda")
    a, la = os_[0].to(dev), ls[0].to(dev)
    out, lse = binding.attn_lse_merge(a, la, os_[1].to(dev), ls[1].to(dev), out=a, lse=la)
    torch.cuda.synchronize()
    assert out.data_ptr() == a.data_ptr()
    assert_close(a, want_o, dtype, "out")
    assert_close(la, want_l, "f32" if dtype == "f32" else "bf16", "lse")


def test_merge_special_rows_exact():
    """Equal lse -> weights 1/2; one side -inf -> the other side."""
    dev = torch.device("cuda")
    o_a = torch.tensor([2.0, -6.0] * 16, device=dev).view(1, 1, 1, 32)
    o_b = torch.tensor([4.0, 10.0] * 16, device=dev).view(1, 1, 1, 32)
    l = torch.full((1, 1, 1), 1.5, device=dev)
    out, lse = binding.attn_lse_merge(o_a, l, o_b, l.clone())
    torch.cuda.synchronize()
    assert torch.allclose(out, torch.tensor([3.0, 2.0] * 16, device=dev).view(1, 1, 1, 32))
    assert abs(lse.item() - (1.5 + np.log(2))) < 1e-6
    ninf = torch.full((1, 1, 1), -float("inf"), device=dev)
    out, lse = binding.attn_lse_merge(o_a, ninf, o_b, l)
    torch.cuda.synchronize()
    assert torch.equal(out, o_b) and lse.item() == 1.5
    out, lse = binding.attn_lse_merge(o_a, ninf, o_b, ninf.clone())
    torch.cuda.synchronize()
    assert torch.all(out == 0) and np.isneginf(lse.item())
