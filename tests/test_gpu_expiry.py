"""Failure detection without a GPU fault: one load of the tensor-core kernel
is withheld, so a bounded wait expires; the kernel must give up in every
role, free its resources, report RA_ERR_TIMEOUT through the status word, and
leave the CUDA context usable."""

import time

import numpy as np
import pytest
import torch

import oracle
from sequence_exact_attention_gb300 import binding
from sequence_exact_attention_gb300.workloads import AttnWorkload, make_qkv

from helpers import assert_close

pytestmark = pytest.mark.gpu

RA_ERR_TIMEOUT = 8


def test_withheld_load_expires_and_context_survives():
    w = AttnWorkload("expiry", "bf16", 1, 1, 1, 512, 128, 1, False, "contiguous", seed=77)
    q, k, v = make_qkv(w)
    dev = torch.device("cuda")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    out = torch.zeros(1, 512, 1, 128, dtype=torch.bfloat16, device=dev)
    lse = torch.zeros(1, 1, 512, dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    t0 = time.time()
    binding.expiry_test(qd, kd, vd, out, lse, status)
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    assert int(status.item()) == RA_ERR_TIMEOUT
    assert elapsed < 30.0
    # the context is intact: a normal call right after is exact
    st2 = torch.zeros(1, dtype=torch.int32, device=dev)
    o2, l2 = binding.ring_attn_fwd(qd, kd, vd, 1, False, w.scale, dev_status=st2)
    torch.cuda.synchronize()
    assert int(st2.item()) == 0
    want_o, want_l = oracle.attention_naive(q, k, v, False, w.scale)
    assert_close(o2, want_o, "bf16", "out after expiry")
    assert_close(l2, want_l, "bf16", "lse after expiry")
