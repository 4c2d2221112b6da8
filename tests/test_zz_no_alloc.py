"""The backward entry point that allocates nothing (ring_attn_bwd_noalloc).

Some callers cannot call cudaMalloc: a plugin whose host framework owns the
device memory through its own pool and hands it no workspace, or a
latency-critical path on which cudaMalloc / cudaFree may synchronise the
device. For them the library keeps the backward's workspace in a built-in
8 MiB device array. These tests check, through the C ABI, that this entry
point gives the same gradients as ring_attn_bwd with a caller workspace, on
two calls in a row (the second call finds the first call's statistics in the
shared array and must not depend on them), and that a problem too large for
the array is refused before anything runs.

The file is named so that pytest collects it last.
"""

import ctypes

import pytest
import torch

from sequence_exact_attention_gb300 import binding
from sequence_exact_attention_gb300.workloads import AttnWorkload, make_dout, make_qkv

# the backward parity tolerance of tests/test_gpu_backward.py: per gradient,
# max-abs error <= 2e-2 * max|ref| and mean-abs error <= 1e-2 * mean|ref|
REL_MAX, REL_MEAN = 2e-2, 1e-2

A = 0x10000          # a 16-byte aligned fake address, never dereferenced


def _noalloc_status(lib, B, H, S, D, P, order):
    vp = ctypes.c_void_p
    return lib.ring_attn_bwd_noalloc(*([vp(A)] * 9), B, H, H, S, D, P, 1, 0.0, 0, order,
                                     None, None)


def test_noalloc_refuses_problems_beyond_its_scratch(lib):
    """Host-side size check: 2^20 tile-padded query rows fit, one tile more
    does not (RA_ERR_SCRATCH, nothing launched, no GPU needed)."""
    n = ctypes.c_size_t()
    assert lib.ring_attn_bwd_workspace(1, 32, 32768, 128, 8, 1, ctypes.byref(n)) == 0
    assert n.value == binding.BWD_NOALLOC_MAX_BYTES
    assert lib.ring_attn_bwd_workspace(1, 33, 32768, 128, 8, 1, ctypes.byref(n)) == 0
    assert n.value > binding.BWD_NOALLOC_MAX_BYTES
    assert _noalloc_status(lib, 1, 33, 32768, 128, 8, 1) == binding.RA_ERR_SCRATCH
    assert _noalloc_status(lib, 2, 16, 32769, 64, 4, 0) == binding.RA_ERR_SCRATCH
    msg = binding.strerror(binding.RA_ERR_SCRATCH)
    assert "scratch" in msg and msg != "unknown status"


def _rel(got, want):
    d = (got.float() - want.float()).abs()
    w = want.float().abs()
    return (float(d.max()) / max(float(w.max()), 1e-2),
            float(d.mean()) / max(float(w.mean()), 1e-2))


def _one_call(w):
    dev = torch.device("cuda")
    q, k, v = (t.to(dev) for t in make_qkv(w))
    dout = make_dout(w).to(dev)
    out, lse = binding.ring_attn_fwd(q, k, v, w.P, w.causal, w.scale, w.order)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    want = binding.ring_attn_bwd(q, k, v, out, lse, dout, w.P, w.causal, w.scale, w.order,
                                 dev_status=status)
    # outputs allocated up front, so the call under test allocates nothing
    got = tuple(torch.empty_like(t) for t in want)
    torch.cuda.synchronize()
    before = torch.cuda.memory_allocated()
    binding.ring_attn_bwd_noalloc(q, k, v, out, lse, dout, w.P, w.causal, w.scale, w.order,
                                  dq=got[0], dk=got[1], dv=got[2], dev_status=status)
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == before
    assert int(status.item()) == 0, "a device-side wait expired"
    for name, g, r in zip(("dq", "dk", "dv"), got, want):
        mx, mean = _rel(g, r)
        assert mx <= REL_MAX and mean <= REL_MEAN, (w.name, name, mx, mean)


@pytest.mark.gpu
def test_noalloc_matches_workspace_backward_twice_in_a_row():
    torch.cuda.set_device(0)
    # two different problems back to back through the one shared array: the
    # second is larger and uses D = 64, the first a GQA zig-zag ring
    first = AttnWorkload("noalloc_s1024_zigzag_gqa", "bf16", 1, 4, 2, 1024, 128, 4, True,
                         "zigzag", seed=2101)
    second = AttnWorkload("noalloc_s1000_ragged_d64", "bf16", 2, 4, 4, 1000, 64, 2, True,
                          "contiguous", seed=2102)
    _one_call(first)
    _one_call(second)
