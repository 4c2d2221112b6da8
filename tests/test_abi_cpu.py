"""Host-side checks of the C-ABI library; no GPU work is launched.

The library must load and export every entry point of include/ring_attn.h,
its host-only planner must equal the oracle's schedule bit for bit, and every
invalid argument must be rejected before the library touches the GPU.
"""

import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from sequence_exact_attention_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ring_attn.h")

RA_OK, RA_ERR_NULL, RA_ERR_SHAPE, RA_ERR_HEADDIM, RA_ERR_ALIGN = 0, 1, 2, 3, 4
RA_ERR_DTYPE, RA_ERR_DEVICE, RA_ERR_BUFFER, RA_ERR_RANGE = 5, 6, 9, 10


def _header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:ra_status|const char\*|int)\s+(\w+)\s*\(",
                                 text, flags=re.M)))


def test_library_exports_every_declared_symbol(lib):
    names = _header_functions()
    assert len(names) >= 8
    assert set(names) == set(binding.EXPORTS)
    for n in names:
        assert hasattr(lib, n), f"{n} not exported"
    assert lib.ring_attn_version() >= 103


def test_checked_build_exports_the_same_symbols(lib):
    """The bounds-checked build loads without a GPU and has the same ABI."""
    path = binding.LIBRARIES["debug"]
    assert os.path.exists(path), "the build makes both libraries"
    dbg = ctypes.CDLL(path)
    for n in _header_functions():
        assert hasattr(dbg, n), f"{n} not exported by the checked build"
    dbg.ring_attn_version.restype = ctypes.c_int
    assert dbg.ring_attn_version() == lib.ring_attn_version()


def test_use_library_switches_and_restores():
    prev = binding.use_library("debug")
    try:
        assert binding._lib_path == binding.LIBRARIES["debug"]
    finally:
        binding.use_library(prev)
    assert binding._lib_path == binding.LIBRARIES[prev]


def test_strerror_covers_every_status(lib):
    seen = set()
    for st in range(0, 11):
        msg = binding.strerror(st)
        assert msg and msg != "unknown status"
        seen.add(msg)
    assert len(seen) == 11
    assert binding.strerror(99) == "unknown status"


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("order", ["contiguous", "zigzag"])
@pytest.mark.parametrize("S,P", [(8, 2), (256, 4), (4096, 8), (32768, 8),
                                 (131072, 16), (96, 3), (16, 16), (7, 7),
                                 (1001, 4), (5, 4), (3, 8), (700, 3)])   # last four uneven
def test_plan_matches_oracle_schedule(S, P, causal, order):
    o = oracle.ORDER_ZIGZAG if order == "zigzag" else oracle.ORDER_CONTIGUOUS
    got = binding.ring_attn_plan(S, P, causal, order)
    want = oracle.schedule_table(S, P, causal, o)
    np.testing.assert_array_equal(got, want)


def test_plan_rejects_small_buffer_and_bad_args(lib):
    buf = (ctypes.c_int * 10)()
    assert lib.ring_attn_plan(8, 2, 1, 0, buf, 10) == RA_ERR_BUFFER
    assert lib.ring_attn_plan(8, 2, 1, 0, None, 100) == RA_ERR_NULL
    assert lib.ring_attn_plan(0, 2, 1, 0, buf, 10) == RA_ERR_SHAPE
    assert lib.ring_attn_plan(8, 0, 1, 0, buf, 10) == RA_ERR_SHAPE
    assert lib.ring_attn_plan(8, 2, 1, 7, buf, 10) == RA_ERR_DTYPE


@pytest.mark.parametrize("dtype,tile", [("bf16", 128), ("f32", 64)])
def test_visit_log_layout(dtype, tile):
    lay = binding.visit_log_layout(2, 4, 4096, 128, 8, dtype, "zigzag")
    seg = 4096 // 16
    nt = -(-seg // tile)
    assert lay["tile_rows"] == tile
    assert lay["tiles_per_segment"] == nt
    assert lay["n_query_tiles"] == 16 * nt
    assert lay["stride"] == 1 + 4 * 16 * nt
    assert lay["len"] == 2 * 4 * 16 * nt * lay["stride"]


# ---- argument checks: every call below fails before the GPU is touched.
# Pointer values are never dereferenced; the checks are on the host.
A = 0x10000          # a 16-byte aligned fake address


def _fwd(lib, q=A, k=A, v=A, out=A, lse=A, B=1, Hq=2, Hkv=2, S=256, D=64, P=4,
         causal=1, scale=0.0, dtype=0, order=0, step=-1, log=None, status=None):
    vp = ctypes.c_void_p
    return lib.ring_attn_fwd_ex(vp(q), vp(k), vp(v), vp(out), vp(lse), B, Hq, Hkv,
                                S, D, P, causal, scale, dtype, order, step,
                                vp(log), vp(status), None)


def test_fwd_argument_errors(lib):
    assert _fwd(lib, q=0) == RA_ERR_NULL
    assert _fwd(lib, out=0) == RA_ERR_NULL
    assert _fwd(lib, lse=0, step=1) == RA_ERR_NULL        # partials need lse
    assert _fwd(lib, B=0) == RA_ERR_SHAPE
    assert _fwd(lib, S=0) == RA_ERR_SHAPE
    assert _fwd(lib, S=-5) == RA_ERR_SHAPE
    assert _fwd(lib, S=250, Hq=3) == RA_ERR_SHAPE         # uneven S is valid; H_q % H_kv is not
    assert _fwd(lib, Hq=3, Hkv=2) == RA_ERR_SHAPE
    assert _fwd(lib, P=0) == RA_ERR_SHAPE
    assert _fwd(lib, D=96) == RA_ERR_HEADDIM
    assert _fwd(lib, D=256) == RA_ERR_HEADDIM
    assert _fwd(lib, q=A + 8) == RA_ERR_ALIGN
    assert _fwd(lib, out=A + 4) == RA_ERR_ALIGN
    assert _fwd(lib, lse=A + 2) == RA_ERR_ALIGN
    assert _fwd(lib, dtype=2) == RA_ERR_DTYPE
    assert _fwd(lib, order=2) == RA_ERR_DTYPE
    assert _fwd(lib, step=4) == RA_ERR_RANGE
    assert _fwd(lib, step=-2) == RA_ERR_RANGE
    assert _fwd(lib, B=1, Hq=64, Hkv=64, S=1 << 20, D=128, P=8) == RA_ERR_RANGE
    vp = ctypes.c_void_p
    assert lib.ring_attn_fwd(vp(0), vp(A), vp(A), vp(A), vp(A), 1, 2, 2, 256, 64,
                             4, 1, 0.0, None) == RA_ERR_NULL


def test_merge_argument_errors(lib):
    vp = ctypes.c_void_p
    assert lib.attn_lse_merge(vp(0), vp(A), vp(A), vp(A), vp(A), vp(A), 1, 2, 8, 64,
                              1, None) == RA_ERR_NULL
    assert lib.attn_lse_merge(vp(A), vp(A), vp(A), vp(A), vp(A), vp(A), 1, 2, 8, 48,
                              1, None) == RA_ERR_HEADDIM
    assert lib.attn_lse_merge(vp(A + 4), vp(A), vp(A), vp(A), vp(A), vp(A), 1, 2, 8,
                              64, 1, None) == RA_ERR_ALIGN
    assert lib.attn_lse_merge(vp(A), vp(A), vp(A), vp(A), vp(A), vp(A), 1, 2, 0, 64,
                              1, None) == RA_ERR_SHAPE
    assert lib.attn_lse_merge(vp(A), vp(A), vp(A), vp(A), vp(A), vp(A), 1, 2, 8, 64,
                              3, None) == RA_ERR_DTYPE
    arr = (ctypes.c_void_p * 17)(*([A] * 17))
    assert lib.attn_lse_merge_n(arr, arr, 17, vp(A), vp(A), 1, 2, 8, 64, 1,
                                None) == RA_ERR_SHAPE
    assert lib.attn_lse_merge_n(arr, arr, 0, vp(A), vp(A), 1, 2, 8, 64, 1,
                                None) == RA_ERR_SHAPE


def _ws_bytes(lib, B=1, Hq=2, S=256, D=64, P=4, order=0):
    n = ctypes.c_size_t()
    st = lib.ring_attn_bwd_workspace(B, Hq, S, D, P, order, ctypes.byref(n))
    return st, n.value


def test_bwd_workspace_size(lib):
    # per (b, h, query tile): 128 negated base-2 lse values and 128 negated deltas, float32;
    # tiles are 128 rows, cut per segment (the last tile of a segment padded)
    st, n = _ws_bytes(lib, B=2, Hq=3, S=1000, D=128, P=4)        # segments of 250: 2 tiles
    assert st == RA_OK and n == 2 * (2 * 3 * 4 * 2 * 128) * 4
    st, n = _ws_bytes(lib, B=1, Hq=1, S=512, D=64, P=2, order=1)  # 4 halves of 128: 1 tile
    assert st == RA_OK and n == 2 * (4 * 1 * 128) * 4
    assert _ws_bytes(lib, D=96)[0] == RA_ERR_HEADDIM
    st, n = _ws_bytes(lib, S=250, P=4)                            # uneven: chunks of 63, 1 tile
    assert st == RA_OK and n == 2 * (2 * 4 * 1 * 128) * 4
    assert _ws_bytes(lib, S=0)[0] == RA_ERR_SHAPE
    assert _ws_bytes(lib, order=3)[0] == RA_ERR_DTYPE
    assert lib.ring_attn_bwd_workspace(1, 2, 256, 64, 4, 0, None) == RA_ERR_NULL


def _bwd(lib, q=A, k=A, v=A, out=A, lse=A, dout=A, dq=A, dk=A, dv=A, B=1, Hq=2, Hkv=2,
         S=256, D=64, P=4, causal=1, scale=0.0, dtype=0, order=0, ws=A, ws_bytes=1 << 20,
         status=None):
    vp = ctypes.c_void_p
    return lib.ring_attn_bwd(vp(q), vp(k), vp(v), vp(out), vp(lse), vp(dout), vp(dq), vp(dk),
                             vp(dv), B, Hq, Hkv, S, D, P, causal, scale, dtype, order, vp(ws),
                             ws_bytes, vp(status), None)


def test_bwd_argument_errors(lib):
    for name in ("q", "out", "lse", "dout", "dq", "dk", "dv", "ws"):
        assert _bwd(lib, **{name: 0}) == RA_ERR_NULL, name
    assert _bwd(lib, S=0) == RA_ERR_SHAPE
    assert _bwd(lib, Hq=3, Hkv=2) == RA_ERR_SHAPE
    assert _bwd(lib, D=96) == RA_ERR_HEADDIM
    assert _bwd(lib, dtype=1) == RA_ERR_DTYPE              # bf16 only
    assert _bwd(lib, order=2) == RA_ERR_DTYPE
    assert _bwd(lib, dout=A + 8) == RA_ERR_ALIGN
    assert _bwd(lib, dk=A + 2) == RA_ERR_ALIGN
    assert _bwd(lib, ws=A + 4) == RA_ERR_ALIGN
    need = _ws_bytes(lib)[1]
    assert _bwd(lib, ws_bytes=need - 1) == RA_ERR_BUFFER
    vp = ctypes.c_void_p
    for bad in (0, 8, -1):
        assert lib.ring_attn_bwd_ex(vp(A), vp(A), vp(A), vp(A), vp(A), vp(A), vp(A), vp(A),
                                    vp(A), 1, 2, 2, 256, 64, 4, 1, 0.0, 0, 0, vp(A), 1 << 20,
                                    bad, None, None) == RA_ERR_RANGE


def _fwd_varlen(lib, q=A, k=A, v=A, out=A, lse=A, cu=A, n=3, total=600, mx=300, Hq=2,
                Hkv=2, D=128, P=4, causal=1, dtype=0, order=1):
    vp = ctypes.c_void_p
    return lib.ring_attn_fwd_varlen(vp(q), vp(k), vp(v), vp(out), vp(lse), vp(cu), n, total,
                                    mx, Hq, Hkv, D, P, causal, 0.0, dtype, order, None, None)


def test_varlen_argument_errors(lib):
    assert _fwd_varlen(lib, cu=0) == RA_ERR_NULL
    assert _fwd_varlen(lib, q=0) == RA_ERR_NULL
    assert _fwd_varlen(lib, n=0) == RA_ERR_SHAPE
    assert _fwd_varlen(lib, total=0) == RA_ERR_SHAPE
    assert _fwd_varlen(lib, mx=0) == RA_ERR_SHAPE
    assert _fwd_varlen(lib, Hq=3) == RA_ERR_SHAPE
    assert _fwd_varlen(lib, D=96) == RA_ERR_HEADDIM
    assert _fwd_varlen(lib, cu=A + 2) == RA_ERR_ALIGN
    assert _fwd_varlen(lib, q=A + 8) == RA_ERR_ALIGN
    assert _fwd_varlen(lib, dtype=4) == RA_ERR_DTYPE
    assert _fwd_varlen(lib, order=5) == RA_ERR_DTYPE
    assert _fwd_varlen(lib, total=1 << 24, Hq=64, Hkv=64) == RA_ERR_RANGE
    vp = ctypes.c_void_p
    args = [vp(A)] * 10

    def bwd(**kw):
        a = dict(n=3, total=600, mx=300, Hq=2, Hkv=2, D=128, P=4, causal=1, dtype=0, order=0,
                 ws_bytes=1 << 24)
        a.update(kw)
        return lib.ring_attn_bwd_varlen(*args, a["n"], a["total"], a["mx"], a["Hq"], a["Hkv"],
                                        a["D"], a["P"], a["causal"], 0.0, a["dtype"], a["order"],
                                        vp(A), a["ws_bytes"], None, None)

    assert bwd(dtype=1) == RA_ERR_DTYPE
    assert bwd(n=0) == RA_ERR_SHAPE
    need = _ws_bytes(lib, B=3, Hq=2, S=300, D=128, P=4)[1]
    assert bwd(ws_bytes=need - 1) == RA_ERR_BUFFER


def test_ulysses_argument_errors(lib):
    vp = ctypes.c_void_p

    def call(q=A, B=1, Hq=4, Hkv=4, S=1000, D=128, P=4, dtype=0):
        return lib.ring_attn_fwd_ulysses(vp(q), vp(A), vp(A), vp(A), vp(A), B, Hq, Hkv, S, D, P,
                                         1, 0.0, dtype, None, None)

    assert call(q=0) == RA_ERR_NULL
    assert call(Hq=6, Hkv=6) == RA_ERR_SHAPE          # heads do not split over 4 ranks
    assert call(Hkv=2) == RA_ERR_SHAPE
    assert call(P=0) == RA_ERR_SHAPE
    assert call(D=96) == RA_ERR_HEADDIM
    assert call(dtype=3) == RA_ERR_DTYPE
    assert call(q=A + 4) == RA_ERR_ALIGN

    def bwd(Hq=4, Hkv=4, dtype=0, ws_bytes=1 << 24, ws=A):
        return lib.ring_attn_bwd_ulysses(*([vp(A)] * 9), 1, Hq, Hkv, 1000, 128, 4, 1, 0.0, dtype,
                                         vp(ws), ws_bytes, None, None)

    assert bwd(Hq=6, Hkv=6) == RA_ERR_SHAPE
    assert bwd(dtype=1) == RA_ERR_DTYPE
    assert bwd(ws=0) == RA_ERR_NULL
    need = _ws_bytes(lib, B=1, Hq=4, S=1000, D=128, P=4)[1]
    assert bwd(ws_bytes=need - 1) == RA_ERR_BUFFER


def test_valid_call_without_gpu_reports_device_error(lib):
    """With every argument valid the only thing missing here is the GPU."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present: this case would launch on fake pointers")
    assert _fwd(lib) == RA_ERR_DEVICE
    assert _bwd(lib) == RA_ERR_DEVICE
    assert _fwd_varlen(lib) == RA_ERR_DEVICE


def test_binding_refuses_host_tensors():
    """No CPU fallback: every compute entry of the binding refuses tensors
    that are not on a CUDA device before it calls the library."""
    import torch
    q = torch.zeros(1, 128, 2, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        binding.ring_attn_fwd(q, q, q, 2, True)
    with pytest.raises(ValueError):
        binding.ring_attn_bwd(q, q, q, q, torch.zeros(1, 2, 128), q, 2, True)
    with pytest.raises(ValueError):
        binding.attn_lse_merge(q.float(), torch.zeros(1, 2, 128), q.float(),
                               torch.zeros(1, 2, 128))
    cu = torch.tensor([0, 128], dtype=torch.int32)
    with pytest.raises(ValueError):
        binding.ring_attn_fwd_varlen(q[0], q[0], q[0], cu, 128, 2, True)
    s = q.view(2, 1, 64, 2, 64)
    with pytest.raises(ValueError):
        binding.ring_attn_fwd_ulysses(s, s, s, 128, True)


def test_missing_library_raises(monkeypatch, tmp_path):
    """A missing shared library is an error at the first call, not a
    fallback."""
    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setattr(binding, "_lib_path", str(tmp_path / "absent.so"))
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        binding.load()


def test_binding_checks_caller_buffers_before_anything_else():
    """The library writes through bare pointers, so every caller-supplied
    buffer must have exactly the shape and dtype the call implies; the
    binding refuses a wrong one (before it looks at devices)."""
    import torch
    bf, f32, i32 = torch.bfloat16, torch.float32, torch.int32
    B, S, H, Hk, D, P = 1, 256, 4, 2, 64, 2
    q = torch.zeros(B, S, H, D, dtype=bf)
    k = torch.zeros(B, S, Hk, D, dtype=bf)
    lse = torch.zeros(B, H, S, dtype=f32)
    cases = [
        (lambda: binding.ring_attn_fwd(q, k, k, P, True, out=torch.zeros(B, S, H, D)), "out"),
        (lambda: binding.ring_attn_fwd(q, k, k, P, True, out=q[:, :128].contiguous()), "out"),
        (lambda: binding.ring_attn_fwd(q, k, k, P, True, lse=torch.zeros(B, S, H)), "lse"),
        (lambda: binding.ring_attn_fwd(q, k, k, P, True, dev_status=torch.zeros(1)),
         "dev_status"),
        (lambda: binding.ring_attn_fwd(q, k, k, P, True, step=0, out=q), "out"),
        (lambda: binding.ring_attn_fwd(q, k, k[:, :, :1].contiguous(), P, True), "k and v"),
        (lambda: binding.ring_attn_bwd(q, k, k, q, lse, q[:, :128].contiguous(), P, True),
         "dout"),
        (lambda: binding.ring_attn_bwd(q, k, k, q, lse, q, P, True, dk=q), "dk"),
        (lambda: binding.ring_attn_bwd(q, k, k, q, lse, q, P, True,
                                       workspace=torch.zeros(64, dtype=f32)), "workspace"),
        (lambda: binding.attn_lse_merge(q.float(), lse, q.float()[:, :, :2].contiguous(), lse),
         "o_b"),
        (lambda: binding.attn_lse_merge_n([q.float(), q.float()], [lse]), "as many"),
        (lambda: binding.attn_lse_merge_n([q.float(), q.float()], [lse, lse[:, :2]]), "lse 1"),
    ]
    total = 300
    qv = torch.zeros(total, H, D, dtype=bf)
    kv = torch.zeros(total, Hk, D, dtype=bf)
    cu = torch.tensor([0, 100, 300], dtype=i32)
    cases += [
        (lambda: binding.ring_attn_fwd_varlen(qv, kv, kv, cu, 200, P, True,
                                              lse=torch.zeros(total, H)), "lse"),
        (lambda: binding.ring_attn_bwd_varlen(qv, kv, kv, qv, torch.zeros(H, total), qv[:10],
                                              cu, 200, P, True), "dout"),
    ]
    C = S // P
    qs = torch.zeros(P, B, C, H, D, dtype=bf)
    ks = torch.zeros(P, B, C, Hk, D, dtype=bf)
    cases += [
        (lambda: binding.ring_attn_fwd_ulysses(qs, ks, ks, S, True,
                                               lse=torch.zeros(P, B, C, H)), "lse"),
        (lambda: binding.ring_attn_bwd_ulysses(qs, ks, qs, qs, torch.zeros(P, B, H, C), qs, S,
                                               True), "v"),
    ]
    for call, name in cases:
        with pytest.raises(ValueError, match=name):
            call()
