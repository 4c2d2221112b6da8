"""The bounds-checked build (``libringattn_debug.so``) against the release one.

The checked build tests every global-memory access a kernel computes from
indices against its tensor's extent (TMA copies are bounds-checked by the
hardware); a violation sets RA_ERR_RANGE in the status word and skips the
access. Each call below goes through every entry point family on small
shapes that reach the edge cases (ragged tiles, uneven and empty chunks,
packed sequences of length 0 and 1, grouped heads, the sequence-sharded
layout, the visit log) and must

* leave the status word at 0 in the checked build: no access out of range;
* give bit-identical results in both builds: the checks change no arithmetic.
"""

import numpy as np
import pytest
import torch

from sequence_exact_attention_gb300 import binding
from sequence_exact_attention_gb300.workloads import AttnWorkload, make_dout, make_qkv

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda")


def _status():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


def _fwd_bwd(w, with_log=False):
    def run(status):
        q, k, v = (t.to(DEV) for t in make_qkv(w))
        dout = make_dout(w).to(DEV) if w.dtype == "bf16" else None
        log = None
        if with_log:
            lay = binding.visit_log_layout(w.B, w.H_q, w.S, w.D, w.P, w.dtype, w.order)
            log = torch.full((lay["len"],), -7, dtype=torch.int32, device=DEV)
        out, lse = binding.ring_attn_fwd(q, k, v, w.P, w.causal, w.scale, w.order,
                                         visit_log=log, dev_status=status)
        res = [out, lse] + ([log] if log is not None else [])
        if dout is not None:
            res += list(binding.ring_attn_bwd(q, k, v, out, lse, dout, w.P, w.causal, w.scale,
                                              w.order, dev_status=status))
        return res
    return run


def _varlen(lengths, dtype, P, causal, order):
    def run(status):
        tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
        g = torch.Generator().manual_seed(77)
        total = int(sum(lengths))
        q, k, v, dout = (torch.randn(total, h, 64, generator=g).to(tdt).to(DEV)
                         for h in (4, 2, 2, 4))
        cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32,
                          device=DEV)
        out, lse = binding.ring_attn_fwd_varlen(q, k, v, cu, max(lengths), P, causal,
                                                order=order, dev_status=status)
        res = [out, lse]
        if dtype == "bf16":
            res += list(binding.ring_attn_bwd_varlen(q, k, v, out, lse, dout, cu, max(lengths),
                                                     P, causal, order=order,
                                                     dev_status=status))
        return res
    return run


def _ulysses(B, H, S, D, P, dtype):
    def run(status):
        tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
        C = -(-S // P)
        g = torch.Generator().manual_seed(78)
        q, k, v, dout = (torch.randn(P, B, C, H, D, generator=g).to(tdt).to(DEV)
                         for _ in range(4))
        out, lse = binding.ring_attn_fwd_ulysses(q, k, v, S, True, dev_status=status)
        res = [out, lse]
        if dtype == "bf16":
            res += list(binding.ring_attn_bwd_ulysses(q, k, v, out, lse, dout, S, True,
                                                      dev_status=status))
        return res
    return run


def _w(name, dtype, B, H_q, H_kv, S, D, P, causal, order):
    return AttnWorkload(name, dtype, B, H_q, H_kv, S, D, P, causal, order, std=1.0, seed=3300)


CASES = {
    "bf16_s1001_zigzag_gqa_log": _fwd_bwd(_w("a", "bf16", 1, 4, 2, 1001, 128, 4, True, "zigzag"),
                                          with_log=True),
    "bf16_s5_empty_chunk": _fwd_bwd(_w("b", "bf16", 2, 2, 1, 5, 64, 4, True, "contiguous")),
    "bf16_s700_noncausal": _fwd_bwd(_w("c", "bf16", 1, 2, 2, 700, 128, 3, False, "zigzag")),
    "f32_s600_zigzag_log": _fwd_bwd(_w("d", "f32", 1, 2, 1, 600, 64, 4, True, "zigzag"),
                                    with_log=True),
    "bf16_varlen": _varlen([300, 0, 1, 777, 128], "bf16", 4, True, "zigzag"),
    "f32_varlen": _varlen([65, 0, 1, 200], "f32", 2, False, "contiguous"),
    "bf16_ulysses": _ulysses(2, 4, 1000, 128, 4, "bf16"),
    "f32_ulysses": _ulysses(1, 2, 300, 64, 2, "f32"),
}


@pytest.fixture
def library():
    prev = binding.use_library("release")
    yield binding
    binding.use_library(prev)


@pytest.mark.parametrize("name", list(CASES))
def test_checked_build_is_in_range_and_identical(library, name):
    run = CASES[name]
    binding.use_library("release")
    st = _status()
    want = run(st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    binding.use_library("debug")
    st = _status()
    got = run(st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, binding.strerror(int(st.item()))
    assert len(got) == len(want)
    for i, (a, b) in enumerate(zip(got, want)):
        assert torch.equal(a, b), f"{name}: result {i} differs between the builds"


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_checked_build_reports_a_sequence_longer_than_max_seqlen(library, dtype):
    """A packed batch whose offsets describe a sequence longer than the
    max_seqlen the call passes: the kernels clamp it (every access stays
    inside the tensors), and the checked build reports the malformed table
    as RA_ERR_RANGE in the status word instead of leaving it at 0. The
    backward reports it the same way."""
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    g = torch.Generator().manual_seed(79)
    total = 400
    q, k, v, dout = (torch.randn(total, h, 64, generator=g).to(tdt).to(DEV) for h in (2, 1, 1, 2))
    cu = torch.tensor([0, 100, 400], dtype=torch.int32, device=DEV)   # second sequence: 300 rows
    binding.use_library("debug")
    st = _status()
    out, lse = binding.ring_attn_fwd_varlen(q, k, v, cu, 256, 2, True, order="zigzag",
                                            dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 10, binding.strerror(int(st.item()))      # RA_ERR_RANGE
    if dtype == "bf16":
        st = _status()
        binding.ring_attn_bwd_varlen(q, k, v, out, lse, dout, cu, 256, 2, True, order="zigzag",
                                     dev_status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 10
    # the same table with a max_seqlen that covers it is clean
    st = _status()
    binding.ring_attn_fwd_varlen(q, k, v, cu, 300, 2, True, order="zigzag", dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
