"""Seeded synthetic workloads for the attention forward pass.

This module only draws random inputs and describes shapes; it holds none of
the attention arithmetic, so both the CUDA path's tests/benchmark and the CPU
oracle can take their inputs from here.

Recipe (the pages fix no data; these readings are stated once here):
  * Q, K, V are i.i.d. N(0, 1): drawn in float32 with a CPU
    ``torch.Generator`` seeded with 0, in the order q, k, v, then rounded to
    the workload's storage dtype (FP16 or BF16).
  * The large-logit variant multiplies the float32 Q draw by 30 before
    rounding, so that logits have a standard deviation near 30 and the running
    maximum changes across key tiles.
  * The packed variable-length batch has 16 sequences whose lengths come from
    ``torch.randint(1, 16385, (16,))`` with a generator seeded with 7; tokens
    are concatenated in sequence order and located by ``cu_seqlens``.
  * The transposed layout stores the same logical [B, H, N, D] values
    contiguously as [B, N, H, D] and is addressed through strides.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

# Lengths drawn by torch.randint(1, 16385, (16,), generator=Generator().manual_seed(7)).
VARLEN_LENGTHS_SEED7 = [12464, 9413, 538, 10743, 5700, 4308, 920, 13928,
                        1373, 11450, 7567, 2584, 11849, 4442, 12655, 14891]


@dataclass(frozen=True)
class Workload:
    name: str
    description: str
    B: int
    Hq: int
    Hkv: int
    N: int            # tokens per sequence (batched) or max_seqlen (varlen)
    D: int
    dtype: torch.dtype
    causal: bool
    layout: str = "bhnd"          # "bhnd" | "bnhd" | "varlen"
    q_scale: float = 1.0          # multiplier on the float32 Q draw
    seqlens: tuple = field(default_factory=tuple)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def total_tokens(self) -> int:
        return sum(self.seqlens) if self.layout == "varlen" else self.B * self.N

    def flops_convention(self) -> float:
        """4 * N^2 * D per (sequence, query head), halved when causal."""
        lens = self.seqlens if self.layout == "varlen" else [self.N] * self.B
        f = sum(4.0 * L * L * self.D for L in lens) * self.Hq
        return f / 2 if self.causal else f

    def flops_exact(self) -> float:
        """Multiply-adds actually required: causal rows see i+1 keys."""
        lens = self.seqlens if self.layout == "varlen" else [self.N] * self.B
        if self.causal:
            return sum(4.0 * self.D * L * (L + 1) / 2 for L in lens) * self.Hq
        return self.flops_convention()

    def io_bytes(self) -> int:
        """Algorithmic HBM bytes of one call: read Q, K, V once, write O and
        the FP32 logsumexp once."""
        esz = torch.tensor([], dtype=self.dtype).element_size()
        tq = self.total_tokens
        return (2 * tq * self.Hq * self.D + 2 * tq * self.Hkv * self.D) * esz + tq * self.Hq * 4


WORKLOADS = {
    "c1": Workload("c1", "single head, causal, N=129, D=32, FP16", 1, 1, 1, 129, 32, torch.float16, True),
    "c2_causal": Workload("c2_causal", "single head, causal, N=512, D=64, FP16", 1, 1, 1, 512, 64,
                          torch.float16, True),
    "c2_noncausal": Workload("c2_noncausal", "single head, non-causal, N=512, D=64, FP16", 1, 1, 1, 512, 64,
                             torch.float16, False),
    "c2_large_logit": Workload("c2_large_logit", "single head, causal, N=512, D=64, FP16, Q x30", 1, 1, 1,
                               512, 64, torch.float16, True, q_scale=30.0),
    "c3": Workload("c3", "B=4, H=16, N=4096, D=128, BF16, causal, [B,H,N,D]", 4, 16, 16, 4096, 128,
                   torch.bfloat16, True),
    "c3_bnhd": Workload("c3_bnhd", "B=4, H=16, N=4096, D=128, BF16, causal, [B,N,H,D] strides", 4, 16, 16,
                        4096, 128, torch.bfloat16, True, layout="bnhd"),
    "c4": Workload("c4", "GQA B=2, Hq=32, Hkv=8, N=8192, D=128, BF16, causal", 2, 32, 8, 8192, 128,
                   torch.bfloat16, True),
    "c5": Workload("c5", "packed varlen, 16 sequences (seed 7), H=16, D=128, BF16, causal", 1, 16, 16,
                   max(VARLEN_LENGTHS_SEED7), 128, torch.bfloat16, True, layout="varlen",
                   seqlens=tuple(VARLEN_LENGTHS_SEED7)),
}


def varlen_lengths_from_seed(seed: int = 7, count: int = 16, max_len: int = 16384):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(1, max_len + 1, (count,), generator=g).tolist()


def cu_seqlens_of(lengths) -> torch.Tensor:
    cu = [0]
    for L in lengths:
        cu.append(cu[-1] + int(L))
    return torch.tensor(cu, dtype=torch.int32)


def _draw(shape, g, dtype, scale=1.0):
    x = torch.randn(shape, generator=g, dtype=torch.float32)
    if scale != 1.0:
        x.mul_(scale)
    return x.to(dtype)


def make_inputs(w: Workload | str, seed: int = 0):
    """Storage tensors on the CPU for a workload.

    Returns a dict with ``q``, ``k``, ``v`` as *logical* views:
      bhnd / bnhd: [B, H, N, D] (bnhd is a strided view of [B, N, H, D] storage)
      varlen:      [T, H, D] plus ``cu_seqlens`` (int32, [S+1])
    """
    if isinstance(w, str):
        w = WORKLOADS[w]
    g = torch.Generator().manual_seed(seed)
    if w.layout == "varlen":
        T = sum(w.seqlens)
        q = _draw((T, w.Hq, w.D), g, w.dtype, w.q_scale)
        k = _draw((T, w.Hkv, w.D), g, w.dtype)
        v = _draw((T, w.Hkv, w.D), g, w.dtype)
        return {"q": q, "k": k, "v": v, "cu_seqlens": cu_seqlens_of(w.seqlens)}
    q = _draw((w.B, w.Hq, w.N, w.D), g, w.dtype, w.q_scale)
    k = _draw((w.B, w.Hkv, w.N, w.D), g, w.dtype)
    v = _draw((w.B, w.Hkv, w.N, w.D), g, w.dtype)
    if w.layout == "bnhd":
        q, k, v = (t.permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3) for t in (q, k, v))
    return {"q": q, "k": k, "v": v}


def random_qkv(B, Hq, Hkv, N, D, dtype, seed=0, layout="bhnd", q_scale=1.0):
    """Small seeded inputs of arbitrary shape (same recipe as make_inputs)."""
    w = Workload("adhoc", "adhoc", B, Hq, Hkv, N, D, dtype, True, layout=layout, q_scale=q_scale)
    return make_inputs(w, seed)


def random_varlen(lengths, Hq, Hkv, D, dtype, seed=0, q_scale=1.0):
    w = Workload("adhoc_varlen", "adhoc", 1, Hq, Hkv, max(lengths) if lengths else 0, D, dtype, True,
                 layout="varlen", q_scale=q_scale, seqlens=tuple(int(x) for x in lengths))
    return make_inputs(w, seed)
