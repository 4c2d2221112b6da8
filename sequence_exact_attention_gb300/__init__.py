"""Exact ring (blockwise) attention on one GB300 (sm_103a).

The compute path is a C-ABI shared library of hand-written CUDA kernels
(``csrc/``, declared in ``include/ring_attn.h``). ``binding`` is a thin ctypes
layer over it that only marshals torch tensors into pointers and sizes;
``workloads`` draws the seeded synthetic inputs. There is no CPU fallback: if
the library is missing, every call raises.
"""

__all__ = ["binding", "workloads"]
