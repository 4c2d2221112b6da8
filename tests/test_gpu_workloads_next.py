"""The named workloads of the next rows (backward, packed variable-length
batch, Ulysses layout) at full size, in the launch configuration the bench
times: in full where the oracle finishes in seconds, else on sampled rows
(segment boundary rows plus seeded random rows), each computed on its own
from the definition.
"""

import numpy as np
import pytest
import torch

import oracle
from sequence_exact_attention_gb300 import binding
from sequence_exact_attention_gb300.workloads import (BWD_WORKLOADS, ULYSSES_WORKLOADS,
                                                      VARLEN_WORKLOADS, make_dout, make_qkv,
                                                      make_sharded_qkv, make_varlen)

from helpers import assert_close, sample_rows

pytestmark = pytest.mark.gpu


def _rel(got, want):
    g = got.double().cpu().numpy() if hasattr(got, "cpu") else np.asarray(got)
    err = np.abs(g - want)
    return err.max() / np.abs(want).max(), err.mean() / np.abs(want).mean()


def test_backward_s4k_full():
    """The 4K backward workload against the oracle on every element (the
    backward's tolerance, tests/test_gpu_backward.py)."""
    w = BWD_WORKLOADS["bf16_s4k_causal_bwd"]
    q, k, v = make_qkv(w)
    dout = make_dout(w)
    dev = torch.device("cuda")
    qd, kd, vd, dd = (t.to(dev) for t in (q, k, v, dout))
    out, lse = binding.ring_attn_fwd(qd, kd, vd, w.P, w.causal, w.scale, w.order)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    dq, dk, dv = binding.ring_attn_bwd(qd, kd, vd, out, lse, dd, w.P, w.causal, w.scale,
                                       w.order, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = oracle.attention_backward(q, k, v, dout, w.causal, w.scale)
    for name, got, want in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        mx, mean = _rel(got, want)
        assert mx <= 2e-2 and mean <= 1e-2, (name, mx, mean)


def test_varlen_workload_sampled():
    w = VARLEN_WORKLOADS["bf16_varlen_32k_causal_zigzag"]
    q, k, v, cu = make_varlen(w)
    dev = torch.device("cuda")
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out, lse = binding.ring_attn_fwd_varlen(q.to(dev), k.to(dev), v.to(dev),
                                            torch.tensor(cu, dtype=torch.int32, device=dev),
                                            w.max_seqlen, w.P, w.causal, w.scale, w.order,
                                            dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for b, n in enumerate(w.lengths):
        lo = cu[b]
        seg = -(-n // (2 * w.P))
        rows = sample_rows(n, seg, 24, seed=600 + b)
        want_o, want_l = oracle.attention_rows(q[None, lo:lo + n], k[None, lo:lo + n],
                                               v[None, lo:lo + n], w.causal, w.scale, rows)
        assert_close(out[lo + rows][None], want_o, "bf16", f"out seq {b}")
        assert_close(lse[:, lo + rows][None], want_l, "bf16", f"lse seq {b}")


def test_ulysses_workload_sampled():
    w = ULYSSES_WORKLOADS["bf16_ulysses_s16k_b2_causal"]
    q_sh, k_sh, v_sh = make_sharded_qkv(w)
    dev = torch.device("cuda")
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out, lse = binding.ring_attn_fwd_ulysses(q_sh.to(dev), k_sh.to(dev), v_sh.to(dev), w.S,
                                             w.causal, w.scale, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    # the oracle reads the natural layout: undo the sharding, then the definition
    q, k, v = (torch.from_numpy(oracle.from_sequence_shards(t.float(), w.S)).to(torch.bfloat16)
               for t in (q_sh, k_sh, v_sh))
    C = q_sh.shape[2]
    rows = sample_rows(w.S, C, 32, seed=700)
    want_o, want_l = oracle.attention_rows(q, k, v, w.causal, w.scale, rows)
    p, c = rows // C, rows % C
    got_o = out.permute(1, 0, 2, 3, 4)[:, p, c]               # [B, n, H, D]
    got_l = lse.permute(1, 2, 0, 3)[:, :, p, c]               # [B, H, n]
    assert_close(got_o, want_o, "bf16", "out")
    assert_close(got_l, want_l, "bf16", "lse")
