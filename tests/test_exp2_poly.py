"""The FMA-pipe exp2 used for part of the softmax exponentials, checked on the
CPU: the kernel's constants (read from its source) and its range reduction,
replayed step by step in float32, against the exact 2^x over the range the
softmax feeds it (x <= 8 after the lazy-rescale threshold)."""

import os
import re

import numpy as np

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "sequence_exact_attention_gb300", "csrc", "fastmath.cuh")


def _constants():
    text = open(SRC).read()
    vals = {}
    for name in ("kExp2C1", "kExp2C2", "kExp2C3"):
        m = re.search(name + r"\s*=\s*([0-9.eE+-]+)f", text)
        vals[name] = np.float32(float(m.group(1)))
    return vals["kExp2C1"], vals["kExp2C2"], vals["kExp2C3"]


def _exp2_poly(x):
    c1, c2, c3 = _constants()
    x = np.maximum(x.astype(np.float32), np.float32(-127.0))
    magic = np.float32(12582912.0)
    t = (x + magic).astype(np.float32)
    f = (x - (t - magic)).astype(np.float32)
    p = np.float32(1.0) + f * (c1 + f * (c2 + f * c3))          # Horner, float32
    p = np.asarray(p, dtype=np.float32)
    bits = p.view(np.uint32) + (t.view(np.uint32) << np.uint32(23))
    return bits.astype(np.uint32).view(np.float32)


def test_relative_error_bound():
    x = np.linspace(-120.0, 8.0, 2_000_001, dtype=np.float64).astype(np.float32)
    got = _exp2_poly(x).astype(np.float64)
    want = np.exp2(x.astype(np.float64))
    rel = np.abs(got / want - 1.0)
    assert rel.max() < 1.1e-4          # bf16 rounding of P is 2^-9 = 2e-3


def test_integers_and_masked_values_exact():
    n = np.arange(-126, 9, dtype=np.float32)
    np.testing.assert_array_equal(_exp2_poly(n), np.exp2(n.astype(np.float64)).astype(np.float32))
    masked = np.array([-np.inf, -1e30, -127.0, -200.0], dtype=np.float32)
    assert np.all(_exp2_poly(masked) == 0.0)
    tiny = _exp2_poly(np.linspace(-127.0, -126.0, 1001, dtype=np.float32))
    assert np.all(np.isfinite(tiny)) and np.all(tiny >= 0) and tiny.max() < 2.0 ** -125
