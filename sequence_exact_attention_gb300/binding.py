"""ctypes binding of the C-ABI library (``include/ring_attn.h``).

Argument marshalling only: tensors become device pointers and sizes, the
current torch stream becomes the ``stream`` argument, a non-zero status
becomes ``RingAttnError``. Because the library reads and writes through bare
pointers, every tensor a call passes must have exactly the shape and dtype
the call implies, be contiguous and live on the current CUDA device; the
binding checks that first and raises ``ValueError`` otherwise. Every step of the computation runs in the CUDA
kernels of ``_lib/libringattn.so``; there is no fallback of any kind, and a
missing library raises at the first call.
"""

import ctypes
import math
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libringattn.so")
LIBRARIES = {"release": LIB_PATH,
             "debug": os.path.join(_HERE, "_lib", "libringattn_debug.so")}

RA_BF16, RA_F32 = 0, 1
ORDERS = {"contiguous": 0, "zigzag": 1}
PLAN_COLS = 9
MERGE_MAX_N = 16

# every entry point declared in include/ring_attn.h
EXPORTS = ("ring_attn_fwd", "ring_attn_fwd_ex", "ring_attn_visit_log_len",
           "ring_attn_fwd_varlen", "ring_attn_bwd_varlen", "ring_attn_fwd_ulysses",
           "ring_attn_bwd_ulysses",
           "ring_attn_bwd_workspace", "ring_attn_bwd", "ring_attn_bwd_ex",
           "ring_attn_bwd_noalloc",
           "attn_lse_merge", "attn_lse_merge_n", "ring_attn_plan",
           "ring_attn_expiry_test", "ring_attn_strerror", "ring_attn_version")

_lib = None
_lib_path = LIB_PATH


class RingAttnError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__(f"{where}: {strerror(status)} (status {status})")


def use_library(variant):
    """Select the library the next calls go through: "release" (the default)
    or "debug" (the bounds-checked build, same entry points). Returns the
    variant that was in use."""
    global _lib, _lib_path
    prev = next(k for k, p in LIBRARIES.items() if p == _lib_path)
    if LIBRARIES[variant] != _lib_path:
        _lib_path = LIBRARIES[variant]
        _lib = None
    return prev


def load():
    """Load the selected shared library once; raises if it was not built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_lib_path):
        raise RuntimeError(
            f"{_lib_path} is missing: build it with "
            "`python -m sequence_exact_attention_gb300.build` (no CPU fallback)")
    lib = ctypes.CDLL(_lib_path)
    c_int, c_float, vp = ctypes.c_int, ctypes.c_float, ctypes.c_void_p
    ip = ctypes.POINTER(ctypes.c_int)
    lib.ring_attn_fwd.restype = c_int
    lib.ring_attn_fwd.argtypes = [vp, vp, vp, vp, vp] + [c_int] * 7 + [c_float, vp]
    lib.ring_attn_fwd_ex.restype = c_int
    lib.ring_attn_fwd_ex.argtypes = ([vp, vp, vp, vp, vp] + [c_int] * 7 + [c_float]
                                     + [c_int] * 3 + [vp, vp, vp])
    lib.ring_attn_visit_log_len.restype = c_int
    lib.ring_attn_visit_log_len.argtypes = [c_int] * 7 + [ip, ip, ip, ip,
                                                          ctypes.POINTER(ctypes.c_longlong)]
    lib.ring_attn_bwd_workspace.restype = c_int
    lib.ring_attn_bwd_workspace.argtypes = [c_int] * 6 + [ctypes.POINTER(ctypes.c_size_t)]
    lib.ring_attn_bwd.restype = c_int
    lib.ring_attn_bwd.argtypes = ([vp] * 9 + [c_int] * 7 + [c_float, c_int, c_int, vp,
                                                             ctypes.c_size_t, vp, vp])
    lib.ring_attn_bwd_ex.restype = c_int
    lib.ring_attn_bwd_ex.argtypes = ([vp] * 9 + [c_int] * 7 + [c_float, c_int, c_int, vp,
                                                                ctypes.c_size_t, c_int, vp, vp])
    lib.ring_attn_bwd_noalloc.restype = c_int
    lib.ring_attn_bwd_noalloc.argtypes = [vp] * 9 + [c_int] * 7 + [c_float, c_int, c_int, vp, vp]
    lib.ring_attn_fwd_ulysses.restype = c_int
    lib.ring_attn_fwd_ulysses.argtypes = [vp] * 5 + [c_int] * 7 + [c_float, c_int, vp, vp]
    lib.ring_attn_bwd_ulysses.restype = c_int
    lib.ring_attn_bwd_ulysses.argtypes = ([vp] * 9 + [c_int] * 7 + [c_float, c_int, vp,
                                                                    ctypes.c_size_t, vp, vp])
    lib.ring_attn_fwd_varlen.restype = c_int
    lib.ring_attn_fwd_varlen.argtypes = ([vp] * 6 + [c_int] * 8 + [c_float, c_int, c_int,
                                                                   vp, vp])
    lib.ring_attn_bwd_varlen.restype = c_int
    lib.ring_attn_bwd_varlen.argtypes = ([vp] * 10 + [c_int] * 8 + [c_float, c_int, c_int, vp,
                                                                    ctypes.c_size_t, vp, vp])
    lib.attn_lse_merge.restype = c_int
    lib.attn_lse_merge.argtypes = [vp] * 6 + [c_int] * 5 + [vp]
    lib.attn_lse_merge_n.restype = c_int
    lib.attn_lse_merge_n.argtypes = [vp, vp, c_int, vp, vp] + [c_int] * 5 + [vp]
    lib.ring_attn_plan.restype = c_int
    lib.ring_attn_plan.argtypes = [c_int, c_int, c_int, c_int, ip, ctypes.c_size_t]
    lib.ring_attn_expiry_test.restype = c_int
    lib.ring_attn_expiry_test.argtypes = [vp, vp, vp, vp, vp, c_int, vp, vp]
    lib.ring_attn_strerror.restype = ctypes.c_char_p
    lib.ring_attn_strerror.argtypes = [c_int]
    lib.ring_attn_version.restype = c_int
    lib.ring_attn_version.argtypes = []
    _lib = lib
    return lib


def strerror(status):
    return load().ring_attn_strerror(int(status)).decode()


def _check(status, where):
    if status != 0:
        raise RingAttnError(status, where)


# ------------------------------------------------------------------ host-only

def ring_attn_plan(S, P, causal, order="contiguous"):
    """The ring schedule table, int32 [P*P, 9] (see ring_attn_plan in the header)."""
    lib = load()
    n = P * P * PLAN_COLS
    buf = (ctypes.c_int * n)()
    _check(lib.ring_attn_plan(S, P, int(bool(causal)), ORDERS[order], buf, n),
           "ring_attn_plan")
    return np.frombuffer(buf, dtype=np.int32).reshape(P * P, PLAN_COLS).copy()


def visit_log_layout(B, H_q, S, D, P, dtype, order="contiguous"):
    """dict(tile_rows, tiles_per_segment, n_query_tiles, stride, len)."""
    lib = load()
    vals = [ctypes.c_int() for _ in range(4)]
    ln = ctypes.c_longlong()
    _check(lib.ring_attn_visit_log_len(B, H_q, S, D, P, _dtype_code(dtype),
                                       ORDERS[order], *[ctypes.byref(x) for x in vals],
                                       ctypes.byref(ln)), "ring_attn_visit_log_len")
    keys = ("tile_rows", "tiles_per_segment", "n_query_tiles", "stride")
    out = {k: v.value for k, v in zip(keys, vals)}
    out["len"] = ln.value
    return out


# ------------------------------------------------------------------ tensors

def _dtype_code(dt):
    import torch
    if dt in (torch.bfloat16, "bf16"):
        return RA_BF16
    if dt in (torch.float32, "f32"):
        return RA_F32
    raise ValueError(f"unsupported dtype {dt}")


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dev(t, name):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _like(t, name, shape, dtype):
    """A tensor the library reads or writes through a bare pointer must have
    exactly the shape and dtype the call implies (None: not given)."""
    if t is None:
        return
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


def _int_buffer(t, name, n):
    """An int32 buffer of at least n elements (None: not given)."""
    import torch
    if t is None:
        return
    if t.dtype != torch.int32 or t.numel() < n:
        raise ValueError(f"{name} must be int32 with at least {n} elements")


def _on_device(named):
    """Every tensor on one CUDA device, contiguous, and that device current
    (the library launches on the current device)."""
    import torch
    devs = set()
    for t, n in named:
        if t is not None:
            _dev(t, n)
            devs.add(t.device)
    if len(devs) > 1:
        raise ValueError(f"the call's tensors are on several devices: {sorted(map(str, devs))}")
    if devs and next(iter(devs)).index != torch.cuda.current_device():
        raise ValueError("the call's tensors must be on the current CUDA device")


def ring_attn_fwd(q, k, v, P, causal, scale=None, order="contiguous", step=-1,
                  out=None, lse=None, want_lse=True, visit_log=None,
                  dev_status=None, stream=None):
    """Ring attention of q [B,S,H_q,D], k/v [B,S,H_kv,D] (CUDA tensors).

    Returns (out, lse). bf16 inputs run on the tensor-core kernel, float32 on
    the exact CUDA-core kernel. With ``step`` = t >= 0 only ring step t runs
    and (out, lse) are that step's float32 partial result.
    """
    import torch
    lib = load()
    B, S, H_q, D = q.shape
    H_kv = k.shape[2]
    if k.shape != (B, S, H_kv, D) or v.shape != k.shape:
        raise ValueError("k and v must be [B, S, H_kv, D] matching q")
    if not (q.dtype == k.dtype == v.dtype):
        raise ValueError("q, k, v must share a dtype")
    code = _dtype_code(q.dtype)
    out_dtype = torch.float32 if step >= 0 else q.dtype
    _like(out, "out", (B, S, H_q, D), out_dtype)
    _like(lse, "lse", (B, H_q, S), torch.float32)
    _int_buffer(dev_status, "dev_status", 1)
    if visit_log is not None:
        _int_buffer(visit_log, "visit_log",
                    visit_log_layout(B, H_q, S, D, P, q.dtype, order)["len"])
    _on_device(((q, "q"), (k, "k"), (v, "v"), (out, "out"), (lse, "lse"),
                (visit_log, "visit_log"), (dev_status, "dev_status")))
    if out is None:
        out = torch.empty(B, S, H_q, D, device=q.device, dtype=out_dtype)
    if lse is None and (want_lse or step >= 0):
        lse = torch.empty(B, H_q, S, device=q.device, dtype=torch.float32)
    sc = float(scale) if scale is not None else 1.0 / math.sqrt(D)
    st = lib.ring_attn_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse),
                              B, H_q, H_kv, S, D, P, int(bool(causal)), sc,
                              code, ORDERS[order], int(step), _ptr(visit_log),
                              _ptr(dev_status), _stream(stream))
    _check(st, "ring_attn_fwd_ex")
    return out, lse


def ring_attn_fwd_plain(q, k, v, out, lse, P, causal, scale=None, stream=None):
    """The plain ``ring_attn_fwd`` entry point (bf16, contiguous order)."""
    import torch
    lib = load()
    B, S, H_q, D = q.shape
    H_kv = k.shape[2]
    _like(k, "k", (B, S, H_kv, D), q.dtype)
    _like(v, "v", (B, S, H_kv, D), q.dtype)
    _like(out, "out", (B, S, H_q, D), q.dtype)
    _like(lse, "lse", (B, H_q, S), torch.float32)
    _on_device(((q, "q"), (k, "k"), (v, "v"), (out, "out"), (lse, "lse")))
    sc = float(scale) if scale is not None else 1.0 / math.sqrt(D)
    st = lib.ring_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse),
                           B, H_q, H_kv, S, D, P, int(bool(causal)), sc,
                           _stream(stream))
    _check(st, "ring_attn_fwd")
    return out, lse


def bwd_workspace_bytes(B, H_q, S, D, P, order="contiguous"):
    """Bytes of device workspace ``ring_attn_bwd`` needs for this shape."""
    lib = load()
    n = ctypes.c_size_t()
    _check(lib.ring_attn_bwd_workspace(B, H_q, S, D, P, ORDERS[order], ctypes.byref(n)),
           "ring_attn_bwd_workspace")
    return n.value


BWD_PREP, BWD_DKDV, BWD_DQ, BWD_ALL = 1, 2, 4, 7


def ring_attn_bwd(q, k, v, out, lse, dout, P, causal, scale=None, order="contiguous",
                  dq=None, dk=None, dv=None, workspace=None, dev_status=None, stream=None,
                  phases=BWD_ALL):
    """Gradients (dq, dk, dv) of ring attention for the upstream gradient dout.

    ``out`` and ``lse`` are the forward's results for the same arguments. All
    tensors are bf16 CUDA tensors (lse float32 [B, H_q, S]). ``workspace``
    (a uint8 CUDA tensor of at least ``bwd_workspace_bytes`` bytes) is
    allocated here when not given; the library itself allocates nothing.
    ``phases`` other than BWD_ALL selects kernels (ring_attn_bwd_ex); a split
    call must reuse the workspace the prep phase filled.
    """
    import torch
    lib = load()
    B, S, H_q, D = q.shape
    H_kv = k.shape[2]
    for t, n in ((k, "k"), (v, "v"), (dk, "dk"), (dv, "dv")):
        _like(t, n, (B, S, H_kv, D), q.dtype)
    for t, n in ((out, "out"), (dout, "dout"), (dq, "dq")):
        _like(t, n, q.shape, q.dtype)
    _like(lse, "lse", (B, H_q, S), torch.float32)
    _int_buffer(dev_status, "dev_status", 1)
    if workspace is not None and workspace.dtype != torch.uint8:
        raise ValueError("workspace must be a uint8 tensor")
    _on_device(((q, "q"), (k, "k"), (v, "v"), (out, "out"), (lse, "lse"), (dout, "dout"),
                (dq, "dq"), (dk, "dk"), (dv, "dv"), (workspace, "workspace"),
                (dev_status, "dev_status")))
    code = _dtype_code(q.dtype)
    if dq is None:
        dq = torch.empty_like(q)
    if dk is None:
        dk = torch.empty_like(k)
    if dv is None:
        dv = torch.empty_like(v)
    need = bwd_workspace_bytes(B, H_q, S, D, P, order)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    sc = float(scale) if scale is not None else 1.0 / math.sqrt(D)
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk),
            _ptr(dv), B, H_q, H_kv, S, D, P, int(bool(causal)), sc, code, ORDERS[order],
            _ptr(workspace), workspace.numel() * workspace.element_size())
    if phases == BWD_ALL:
        st = lib.ring_attn_bwd(*args, _ptr(dev_status), _stream(stream))
    else:
        st = lib.ring_attn_bwd_ex(*args, int(phases), _ptr(dev_status), _stream(stream))
    _check(st, "ring_attn_bwd")
    return dq, dk, dv


BWD_NOALLOC_MAX_BYTES = 8 << 20
RA_ERR_SCRATCH = 11


def ring_attn_bwd_noalloc(q, k, v, out, lse, dout, P, causal, scale=None, order="contiguous",
                          dq=None, dk=None, dv=None, dev_status=None, stream=None):
    """``ring_attn_bwd`` through the entry point that allocates nothing.

    For callers that cannot allocate device memory (a plugin whose host
    framework owns the memory pool, a path where cudaMalloc may synchronise):
    the library keeps the backward's workspace in its own built-in 8 MiB
    device array. Pass dq, dk, dv to make the whole call allocation-free; when
    omitted they are allocated here, by torch, as for ``ring_attn_bwd``.
    Calls that overlap on the GPU share that array and race: serialise them.
    A problem needing more than ``BWD_NOALLOC_MAX_BYTES`` of workspace raises
    ``RingAttnError`` with status ``RA_ERR_SCRATCH``.
    """
    import torch
    lib = load()
    B, S, H_q, D = q.shape
    H_kv = k.shape[2]
    for t, n in ((k, "k"), (v, "v"), (dk, "dk"), (dv, "dv")):
        _like(t, n, (B, S, H_kv, D), q.dtype)
    for t, n in ((out, "out"), (dout, "dout"), (dq, "dq")):
        _like(t, n, q.shape, q.dtype)
    _like(lse, "lse", (B, H_q, S), torch.float32)
    _int_buffer(dev_status, "dev_status", 1)
    _on_device(((q, "q"), (k, "k"), (v, "v"), (out, "out"), (lse, "lse"), (dout, "dout"),
                (dq, "dq"), (dk, "dk"), (dv, "dv"), (dev_status, "dev_status")))
    code = _dtype_code(q.dtype)
    if dq is None:
        dq = torch.empty_like(q)
    if dk is None:
        dk = torch.empty_like(k)
    if dv is None:
        dv = torch.empty_like(v)
    sc = float(scale) if scale is not None else 1.0 / math.sqrt(D)
    st = lib.ring_attn_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout),
                                   _ptr(dq), _ptr(dk), _ptr(dv), B, H_q, H_kv, S, D, P,
                                   int(bool(causal)), sc, code, ORDERS[order],
                                   _ptr(dev_status), _stream(stream))
    _check(st, "ring_attn_bwd_noalloc")
    return dq, dk, dv


def _varlen_args(q, k, v, cu_seqlens, max_seqlen):
    import torch
    if cu_seqlens.dtype != torch.int32 or cu_seqlens.dim() != 1:
        raise ValueError("cu_seqlens must be a 1-D int32 CUDA tensor")
    total, H_q, D = q.shape
    H_kv = k.shape[1]
    _like(k, "k", (total, H_kv, D), q.dtype)
    _like(v, "v", (total, H_kv, D), q.dtype)
    return total, H_q, H_kv, D, cu_seqlens.numel() - 1, int(max_seqlen)


def ring_attn_fwd_varlen(q, k, v, cu_seqlens, max_seqlen, P, causal, scale=None,
                         order="contiguous", out=None, lse=None, dev_status=None,
                         stream=None):
    """Ring attention of packed sequences: q [total,H_q,D], k/v [total,H_kv,D],
    cu_seqlens int32 [n+1] (CUDA). Returns (out [total,H_q,D], lse [H_q,total])."""
    import torch
    lib = load()
    total, H_q, H_kv, D, n, mx = _varlen_args(q, k, v, cu_seqlens, max_seqlen)
    _like(out, "out", q.shape, q.dtype)
    _like(lse, "lse", (H_q, total), torch.float32)
    _int_buffer(dev_status, "dev_status", 1)
    _on_device(((q, "q"), (k, "k"), (v, "v"), (cu_seqlens, "cu_seqlens"), (out, "out"),
                (lse, "lse"), (dev_status, "dev_status")))
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(H_q, total, device=q.device, dtype=torch.float32)
    sc = float(scale) if scale is not None else 1.0 / math.sqrt(D)
    st = lib.ring_attn_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse),
                                  _ptr(cu_seqlens), n, total, mx, H_q, H_kv, D, P,
                                  int(bool(causal)), sc, _dtype_code(q.dtype), ORDERS[order],
                                  _ptr(dev_status), _stream(stream))
    _check(st, "ring_attn_fwd_varlen")
    return out, lse


def ring_attn_bwd_varlen(q, k, v, out, lse, dout, cu_seqlens, max_seqlen, P, causal,
                         scale=None, order="contiguous", workspace=None, dev_status=None,
                         stream=None):
    """Gradients (dq, dk, dv) of ``ring_attn_fwd_varlen`` for the upstream dout."""
    import torch
    lib = load()
    total, H_q, H_kv, D, n, mx = _varlen_args(q, k, v, cu_seqlens, max_seqlen)
    _like(out, "out", q.shape, q.dtype)
    _like(dout, "dout", q.shape, q.dtype)
    _like(lse, "lse", (H_q, total), torch.float32)
    _int_buffer(dev_status, "dev_status", 1)
    if workspace is not None and workspace.dtype != torch.uint8:
        raise ValueError("workspace must be a uint8 tensor")
    _on_device(((q, "q"), (k, "k"), (v, "v"), (cu_seqlens, "cu_seqlens"), (out, "out"),
                (lse, "lse"), (dout, "dout"), (workspace, "workspace"),
                (dev_status, "dev_status")))
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    need = bwd_workspace_bytes(n, H_q, mx, D, P, order)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    sc = float(scale) if scale is not None else 1.0 / math.sqrt(D)
    st = lib.ring_attn_bwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout),
                                  _ptr(dq), _ptr(dk), _ptr(dv), _ptr(cu_seqlens), n, total, mx,
                                  H_q, H_kv, D, P, int(bool(causal)), sc, _dtype_code(q.dtype),
                                  ORDERS[order], _ptr(workspace),
                                  workspace.numel() * workspace.element_size(),
                                  _ptr(dev_status), _stream(stream))
    _check(st, "ring_attn_bwd_varlen")
    return dq, dk, dv


def ring_attn_fwd_ulysses(q, k, v, S, causal, scale=None, out=None, lse=None,
                          dev_status=None, stream=None):
    """Attention of sequence-sharded tensors q [P,B,C,H_q,D], k/v [P,B,C,H_kv,D]
    (C = ceil(S/P)). Returns (out [P,B,C,H_q,D], lse [P,B,H_q,C])."""
    import torch
    lib = load()
    P, B, C, H_q, D = q.shape
    H_kv = k.shape[3]
    _like(k, "k", (P, B, C, H_kv, D), q.dtype)
    _like(v, "v", (P, B, C, H_kv, D), q.dtype)
    if C != -(-S // P):
        raise ValueError("shard length must be ceil(S / P)")
    _like(out, "out", q.shape, q.dtype)
    _like(lse, "lse", (P, B, H_q, C), torch.float32)
    _int_buffer(dev_status, "dev_status", 1)
    _on_device(((q, "q"), (k, "k"), (v, "v"), (out, "out"), (lse, "lse"),
                (dev_status, "dev_status")))
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(P, B, H_q, C, device=q.device, dtype=torch.float32)
    sc = float(scale) if scale is not None else 1.0 / math.sqrt(D)
    st = lib.ring_attn_fwd_ulysses(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H_q, H_kv,
                                   S, D, P, int(bool(causal)), sc, _dtype_code(q.dtype),
                                   _ptr(dev_status), _stream(stream))
    _check(st, "ring_attn_fwd_ulysses")
    return out, lse


def ring_attn_bwd_ulysses(q, k, v, out, lse, dout, S, causal, scale=None, workspace=None,
                          dev_status=None, stream=None):
    """Gradients (dq, dk, dv) of ``ring_attn_fwd_ulysses``, all in the
    sequence-parallel layout [P, B, C, H, D]."""
    import torch
    lib = load()
    P, B, C, H_q, D = q.shape
    H_kv = k.shape[3]
    _like(k, "k", (P, B, C, H_kv, D), q.dtype)
    _like(v, "v", (P, B, C, H_kv, D), q.dtype)
    if C != -(-S // P):
        raise ValueError("shard length must be ceil(S / P)")
    _like(out, "out", q.shape, q.dtype)
    _like(dout, "dout", q.shape, q.dtype)
    _like(lse, "lse", (P, B, H_q, C), torch.float32)
    _int_buffer(dev_status, "dev_status", 1)
    if workspace is not None and workspace.dtype != torch.uint8:
        raise ValueError("workspace must be a uint8 tensor")
    _on_device(((q, "q"), (k, "k"), (v, "v"), (out, "out"), (lse, "lse"), (dout, "dout"),
                (workspace, "workspace"), (dev_status, "dev_status")))
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    need = bwd_workspace_bytes(B, H_q, S, D, P, "contiguous")
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    sc = float(scale) if scale is not None else 1.0 / math.sqrt(D)
    st = lib.ring_attn_bwd_ulysses(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout),
                                   _ptr(dq), _ptr(dk), _ptr(dv), B, H_q, H_kv, S, D, P,
                                   int(bool(causal)), sc, _dtype_code(q.dtype), _ptr(workspace),
                                   workspace.numel() * workspace.element_size(),
                                   _ptr(dev_status), _stream(stream))
    _check(st, "ring_attn_bwd_ulysses")
    return dq, dk, dv


def attn_lse_merge(o_a, lse_a, o_b, lse_b, out=None, lse=None, stream=None):
    """Pairwise merge; o_* [B,S,H,D], lse_* [B,H,S] float32."""
    import torch
    lib = load()
    B, S, H, D = o_a.shape
    for t, n in ((o_b, "o_b"), (out, "out")):
        _like(t, n, o_a.shape, o_a.dtype)
    for t, n in ((lse_a, "lse_a"), (lse_b, "lse_b"), (lse, "lse")):
        _like(t, n, (B, H, S), torch.float32)
    _on_device(((o_a, "o_a"), (o_b, "o_b"), (lse_a, "lse_a"), (lse_b, "lse_b"), (out, "out"),
                (lse, "lse")))
    if out is None:
        out = torch.empty_like(o_a)
    if lse is None:
        lse = torch.empty_like(lse_a)
    st = lib.attn_lse_merge(_ptr(o_a), _ptr(lse_a), _ptr(o_b), _ptr(lse_b),
                            _ptr(out), _ptr(lse), B, H, S, D,
                            _dtype_code(o_a.dtype), _stream(stream))
    _check(st, "attn_lse_merge")
    return out, lse


def attn_lse_merge_n(os_, lses, out=None, lse=None, stream=None):
    """N-way merge of lists of partials (one pass)."""
    import torch
    lib = load()
    n = len(os_)
    if n < 1 or len(lses) != n:
        raise ValueError("need as many lse tensors as partial outputs, at least one")
    B, S, H, D = os_[0].shape
    for i, t in enumerate(os_):
        _like(t, f"partial {i}", os_[0].shape, os_[0].dtype)
    for i, t in enumerate(lses):
        _like(t, f"lse {i}", (B, H, S), torch.float32)
    _like(out, "out", os_[0].shape, os_[0].dtype)
    _like(lse, "lse", (B, H, S), torch.float32)
    _on_device([(t, "partial") for t in os_] + [(t, "lse") for t in lses] +
               [(out, "out"), (lse, "lse")])
    if out is None:
        out = torch.empty_like(os_[0])
    if lse is None:
        lse = torch.empty_like(lses[0])
    o_arr = (ctypes.c_void_p * max(n, 1))(*[t.data_ptr() for t in os_])
    l_arr = (ctypes.c_void_p * max(n, 1))(*[t.data_ptr() for t in lses])
    st = lib.attn_lse_merge_n(o_arr, l_arr, n, _ptr(out), _ptr(lse), B, H, S, D,
                              _dtype_code(os_[0].dtype), _stream(stream))
    _check(st, "attn_lse_merge_n")
    return out, lse


def expiry_test(q, k, v, out, lse, dev_status, stream=None):
    """Launch the kernel with one load withheld (see ring_attn_expiry_test)."""
    lib = load()
    _int_buffer(dev_status, "dev_status", 1)
    _on_device(((q, "q"), (k, "k"), (v, "v"), (out, "out"), (lse, "lse"),
                (dev_status, "dev_status")))
    S = q.shape[1]
    st = lib.ring_attn_expiry_test(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), S,
                                   _ptr(dev_status), _stream(stream))
    _check(st, "ring_attn_expiry_test")
