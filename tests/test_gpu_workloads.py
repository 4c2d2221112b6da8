"""The named workloads at full size, in the launch configuration the bench
times, checked against the oracle: in full where the oracle finishes in
seconds, else on sampled rows (every chunk/half boundary row plus seeded
random rows, all heads), each computed on its own from the definition.
"""

import numpy as np
import pytest
import torch

import oracle
from sequence_exact_attention_gb300 import binding
from sequence_exact_attention_gb300.workloads import (WORKLOADS, MERGE_WORKLOADS,
                                                      make_qkv, make_merge_parts)

from helpers import assert_close, decode_visit_log, sample_rows

pytestmark = pytest.mark.gpu

ORDER = {"contiguous": oracle.ORDER_CONTIGUOUS, "zigzag": oracle.ORDER_ZIGZAG}


def _run(w, log=False):
    q, k, v = make_qkv(w)
    dev = torch.device("cuda")
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    vlog, lay = None, None
    if log:
        lay = binding.visit_log_layout(w.B, w.H_q, w.S, w.D, w.P, w.dtype, w.order)
        vlog = torch.full((lay["len"],), -7, dtype=torch.int32, device=dev)
    out, lse = binding.ring_attn_fwd(q.to(dev), k.to(dev), v.to(dev), w.P, w.causal,
                                     w.scale, w.order, visit_log=vlog, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.isfinite(out.float()).all()
    return q, k, v, out, lse, vlog, lay


def _check_visits(w, vlog, lay, heads):
    got = decode_visit_log(vlog, w.B, w.H_q, lay["n_query_tiles"], lay["stride"])
    want = oracle.tile_visits(w.S, w.P, w.causal, ORDER[w.order], lay["tile_rows"])
    for b in range(w.B):
        for h in heads:
            assert got[b][h] == want, f"visit log differs at b={b} h={h}"


@pytest.mark.parametrize("name", ["fp32_s256", "bf16_s4k_causal"])
def test_workload_full(name):
    w = WORKLOADS[name]
    q, k, v, out, lse, vlog, lay = _run(w, log=True)
    want_o, want_l = oracle.attention_naive(q, k, v, w.causal, w.scale)
    assert_close(out, want_o, w.dtype, "out")
    assert_close(lse, want_l, w.dtype, "lse")
    _check_visits(w, vlog, lay, range(w.H_q))


@pytest.mark.parametrize("name", ["bf16_s32k_causal_zigzag", "bf16_s128k_gqa_causal",
                                  "bf16_s16k_d64", "bf16_s32760_uneven_causal_zigzag"])
def test_workload_sampled(name):
    w = WORKLOADS[name]
    log = name in ("bf16_s32k_causal_zigzag", "bf16_s32760_uneven_causal_zigzag")
    q, k, v, out, lse, vlog, lay = _run(w, log=log)
    # segment length: S / parts, rounded up when the parts do not divide S
    seg = -(-w.S // (2 * w.P if w.order == "zigzag" else w.P))
    rows = sample_rows(w.S, seg, 48, seed=w.seed)
    want_o, want_l = oracle.attention_rows(q, k, v, w.causal, w.scale, rows)
    assert_close(out[:, rows], want_o, w.dtype, "out")
    assert_close(lse[:, :, rows], want_l, w.dtype, "lse")
    if log:
        _check_visits(w, vlog, lay, [0, w.H_q - 1])


def test_merge_workload_sampled():
    w = MERGE_WORKLOADS["merge_p8_s64k"]
    os_, ls = make_merge_parts(w)
    dev = torch.device("cuda")
    od = [o.to(dev) for o in os_]
    ld = [l.to(dev) for l in ls]
    out, lse = binding.attn_lse_merge_n(od, ld)
    torch.cuda.synchronize()
    rows = sample_rows(w.S, 8192, 2048, seed=w.seed)
    want_o, want_l = oracle.lse_merge_n([o[:, rows] for o in os_],
                                        [l[:, :, rows] for l in ls])
    assert_close(out[:, rows], want_o, w.dtype, "out")
    assert_close(lse[:, :, rows], want_l, w.dtype, "lse")
