"""Seeded synthetic inputs shared by the tests, the bench and the smoke check.

This module holds none of the attention arithmetic: it only draws random
tensors. The CUDA path and the CPU oracle both receive exactly the tensors it
returns, so neither side generates its own inputs.

The pages name no dataset; their long-context workloads (books of 100K+
tokens, hidden size 4096 in the glossary "sequence parallelism transformers",
§Sequence Parallelism Fundamentals and §Use Cases) are stood in for by the
named shapes below, with Gaussian queries/keys/values.

Recipe (every tensor drawn on the CPU with ``torch.Generator().manual_seed``):
draw q, then k, then v, each float32 N(0, std^2) in [B, S, H, D] order; for
the GQA workload add +3.0 to every odd sequence row of k (all heads, all
components) before the cast; cast to the target dtype with round-to-nearest-
even (``Tensor.to``). Backward workloads add the upstream gradient dout,
float32 N(0, std^2) [B, S, H_q, D] from its own generator seeded with
seed + 500000, cast the same way. Merge partials: n float32 N(0, 1) outputs [B, S, H, D],
then n lse tensors U(-20, 20) [B, H, S].
"""

from dataclasses import dataclass, replace
import math

import torch


@dataclass(frozen=True)
class AttnWorkload:
    name: str
    dtype: str          # "bf16" or "f32"
    B: int
    H_q: int
    H_kv: int
    S: int
    D: int
    P: int
    causal: bool
    order: str          # "contiguous" or "zigzag"
    std: float = 1.0
    k_shift_odd: float = 0.0
    seed: int = 0

    @property
    def scale(self):
        return 1.0 / math.sqrt(self.D)

    @property
    def flop(self):
        """Algorithmic FLOP: 4*B*H_q*S^2*D, halved under the causal mask."""
        f = 4.0 * self.B * self.H_q * self.S * self.S * self.D
        return f / 2 if self.causal else f

    def scaled(self, **kw):
        return replace(self, **kw)


@dataclass(frozen=True)
class MergeWorkload:
    name: str
    dtype: str
    n: int
    B: int
    H: int
    S: int
    D: int
    lse_range: float = 20.0
    seed: int = 0

    @property
    def bytes(self):
        """Algorithmic bytes of one N-way merge: read n partials, write one."""
        esz = 4 if self.dtype == "f32" else 2
        rows = self.B * self.H * self.S
        return rows * (self.n + 1) * (self.D * esz + 4)


WORKLOADS = {
    "fp32_s256": AttnWorkload("fp32_s256", "f32", 1, 2, 2, 256, 64, 4, False,
                              "contiguous", seed=1001),
    "bf16_s4k_causal": AttnWorkload("bf16_s4k_causal", "bf16", 2, 16, 16, 4096,
                                    128, 8, True, "contiguous", seed=1002),
    "bf16_s32k_causal_zigzag": AttnWorkload(
        "bf16_s32k_causal_zigzag", "bf16", 1, 32, 32, 32768, 128, 8, True,
        "zigzag", std=0.5, seed=1003),
    "bf16_s128k_gqa_causal": AttnWorkload(
        "bf16_s128k_gqa_causal", "bf16", 1, 32, 8, 131072, 128, 16, True,
        "contiguous", k_shift_odd=3.0, seed=1004),
    "bf16_s16k_d64": AttnWorkload("bf16_s16k_d64", "bf16", 4, 16, 16, 16384,
                                  64, 4, False, "contiguous", seed=1006),
    # Uneven chunks: S = 32760 is not a multiple of 2P = 16, so every zig-zag
    # half spans ceil(S / 2P) = 2048 positions and the last one holds 2040.
    "bf16_s32760_uneven_causal_zigzag": AttnWorkload(
        "bf16_s32760_uneven_causal_zigzag", "bf16", 1, 32, 32, 32760, 128, 8, True,
        "zigzag", std=0.5, seed=1009),
}

MERGE_WORKLOADS = {
    "merge_p8_s64k": MergeWorkload("merge_p8_s64k", "f32", 8, 1, 32, 65536, 128,
                                   seed=1005),
}

@dataclass(frozen=True)
class VarlenWorkload:
    """A packed batch of sequences of different lengths."""
    name: str
    dtype: str
    lengths: tuple
    H_q: int
    H_kv: int
    D: int
    P: int
    causal: bool
    order: str
    std: float = 1.0
    seed: int = 0

    @property
    def total(self):
        return int(sum(self.lengths))

    @property
    def max_seqlen(self):
        return int(max(self.lengths))

    @property
    def scale(self):
        return 1.0 / math.sqrt(self.D)

    @property
    def flop(self):
        """4*H_q*S_b^2*D per sequence, halved under the causal mask."""
        f = sum(4.0 * self.H_q * n * n * self.D for n in self.lengths)
        return f / 2 if self.causal else f


def make_varlen(w: VarlenWorkload):
    """(q [total,H_q,D], k, v [total,H_kv,D], cu_seqlens int32 list) CPU tensors."""
    g = torch.Generator().manual_seed(w.seed)
    dt = _TORCH_DTYPE[w.dtype]
    q = (torch.randn(w.total, w.H_q, w.D, generator=g) * w.std).to(dt)
    k = (torch.randn(w.total, w.H_kv, w.D, generator=g) * w.std).to(dt)
    v = (torch.randn(w.total, w.H_kv, w.D, generator=g) * w.std).to(dt)
    cu = [0]
    for n in w.lengths:
        cu.append(cu[-1] + int(n))
    return q, k, v, cu


def make_sharded_qkv(w: AttnWorkload):
    """(q [P,B,C,H_q,D], k, v [P,B,C,H_kv,D]) drawn directly in the
    sequence-parallel layout of P ranks (C = ceil(S/P)); CPU tensors."""
    g = torch.Generator().manual_seed(w.seed)
    C = -(-w.S // w.P)
    dt = _TORCH_DTYPE[w.dtype]
    q = (torch.randn(w.P, w.B, C, w.H_q, w.D, generator=g) * w.std).to(dt)
    k = (torch.randn(w.P, w.B, C, w.H_kv, w.D, generator=g) * w.std).to(dt)
    v = (torch.randn(w.P, w.B, C, w.H_kv, w.D, generator=g) * w.std).to(dt)
    return q, k, v


# A packed batch of the headline's total length (32768 tokens) in six
# sequences of mixed lengths, zig-zag order per sequence.
VARLEN_WORKLOADS = {
    "bf16_varlen_32k_causal_zigzag": VarlenWorkload(
        "bf16_varlen_32k_causal_zigzag", "bf16", (8192, 4096, 11000, 1000, 3000, 5480),
        32, 32, 128, 8, True, "zigzag", std=0.5, seed=1007),
}

# Ulysses layout: two sequences of 16K in the sequence-parallel layout of 8 ranks.
ULYSSES_WORKLOADS = {
    "bf16_ulysses_s16k_b2_causal": AttnWorkload(
        "bf16_ulysses_s16k_b2_causal", "bf16", 2, 32, 32, 16384, 128, 8, True, "contiguous",
        std=0.5, seed=1008),
}

# Backward workloads: the forward shapes of the causal bf16 workloads.
BWD_WORKLOADS = {
    "bf16_s4k_causal_bwd": WORKLOADS["bf16_s4k_causal"].scaled(name="bf16_s4k_causal_bwd"),
    "bf16_s32k_causal_zigzag_bwd": WORKLOADS["bf16_s32k_causal_zigzag"].scaled(
        name="bf16_s32k_causal_zigzag_bwd"),
}

HEADLINE = "bf16_s32k_causal_zigzag"

_TORCH_DTYPE = {"bf16": torch.bfloat16, "f32": torch.float32}


def torch_dtype(name):
    return _TORCH_DTYPE[name]


def make_qkv(w: AttnWorkload):
    """(q, k, v) CPU tensors of ``w``'s dtype, drawn with ``w.seed``."""
    g = torch.Generator().manual_seed(w.seed)
    q = torch.randn(w.B, w.S, w.H_q, w.D, generator=g) * w.std
    k = torch.randn(w.B, w.S, w.H_kv, w.D, generator=g) * w.std
    v = torch.randn(w.B, w.S, w.H_kv, w.D, generator=g) * w.std
    if w.k_shift_odd:
        k[:, 1::2] += w.k_shift_odd
    dt = _TORCH_DTYPE[w.dtype]
    return q.to(dt), k.to(dt), v.to(dt)


def make_dout(w: AttnWorkload):
    """Upstream gradient dout [B,S,H_q,D] for the backward pass, CPU tensor."""
    g = torch.Generator().manual_seed(w.seed + 500000)
    d = torch.randn(w.B, w.S, w.H_q, w.D, generator=g) * w.std
    return d.to(_TORCH_DTYPE[w.dtype])


def bwd_flop(w: AttnWorkload):
    """Algorithmic FLOP of the backward pass: 2.5x the forward's (five
    products of the forward's size: S and dP recomputed, dV, dK, dQ)."""
    return 2.5 * w.flop


def make_merge_parts(w: MergeWorkload):
    """(list of n outputs [B,S,H,D], list of n lse [B,H,S]) CPU tensors."""
    g = torch.Generator().manual_seed(w.seed)
    dt = _TORCH_DTYPE[w.dtype]
    os_ = [torch.randn(w.B, w.S, w.H, w.D, generator=g).to(dt)
           for _ in range(w.n)]
    lses = [(torch.rand(w.B, w.H, w.S, generator=g) * 2 - 1) * w.lse_range
            for _ in range(w.n)]
    return os_, lses
