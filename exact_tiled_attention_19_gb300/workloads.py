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
  * Workloads with Nk != Nq (a chunk of new queries over a longer key
    cache) draw K and V with Nk tokens; packed batches with separate key
    lengths draw Tk = sum of key lengths.  The draw order stays q, k, v.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
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
    Nk: int | None = None         # key tokens per sequence (batched); None = N
    seqlens_k: tuple = field(default_factory=tuple)  # packed key lengths; empty = seqlens
    window_left: int = -1         # local window (keys before the row's key position); -1 = none
    window_right: int = -1
    num_global: int = 0           # global tokens beside the window (the first positions of each sequence)
    splitkv: bool = False         # run through the split-KV entry point (few queries, many keys)
    backward: bool = False        # the backward pass (dQ, dK, dV for a seeded upstream gradient)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def keys(self) -> int:
        return self.N if self.Nk is None else self.Nk

    def lengths(self):
        """(query length, key length) of every sequence."""
        if self.layout == "varlen":
            lk = self.seqlens_k or self.seqlens
            return list(zip(self.seqlens, lk))
        return [(self.N, self.keys)] * self.B

    @property
    def total_tokens(self) -> int:
        return sum(lq for lq, _ in self.lengths())

    @property
    def total_keys(self) -> int:
        return sum(lk for _, lk in self.lengths())

    @property
    def square(self) -> bool:
        """Equal query and key lengths and no window."""
        return (all(lq == lk for lq, lk in self.lengths()) and self.window_left < 0 and self.window_right < 0
                and self.num_global == 0)

    def flops_convention(self) -> float:
        """4 * N^2 * D per (sequence, query head), halved when causal.  For
        unequal lengths or a window, the exact count."""
        if not self.square:
            return self.flops_exact()
        f = sum(4.0 * lq * lk * self.D for lq, lk in self.lengths()) * self.Hq
        return f / 2 if self.causal else f

    def flops(self) -> float:
        """The FLOPs a call is credited with: the forward convention, times
        2.5 for the backward pass (five products of the forward's size
        instead of two: S, dP, dV, dK, dQ)."""
        return self.flops_convention() * (2.5 if self.backward else 1.0)

    def eligible_pairs(self) -> int:
        """(query row, key) pairs that enter the softmax, per query head,
        summed over sequences.  Query row r of Lq sits at key position
        r + Lk - Lq; the causal mask and a window bound the keys it reads.
        With G global tokens a row also reads the keys below G and a global
        row (position < G) every key, under the causal mask: the union is
        counted by inclusion-exclusion, each pair once."""
        total = 0
        for lq, lk in self.lengths():
            if lq == 0 or lk == 0:
                continue
            c = np.arange(lq, dtype=np.int64) + (lk - lq)
            hi = np.full(lq, lk - 1, dtype=np.int64)
            if self.causal:
                hi = np.minimum(hi, c)
            if self.window_right >= 0:
                hi = np.minimum(hi, c + self.window_right)
            lo = np.zeros(lq, dtype=np.int64)
            if self.window_left >= 0:
                lo = np.maximum(lo, c - self.window_left)
            n = np.maximum(hi - lo + 1, 0)
            G = self.num_global
            if G > 0:
                hc = np.minimum(c, lk - 1) if self.causal else np.full(lq, lk - 1, dtype=np.int64)
                bhi = np.minimum(G - 1, hc)                     # global keys [0, bhi]
                n_b = np.maximum(bhi + 1, 0)
                n_both = np.maximum(np.minimum(hi, bhi) - lo + 1, 0)
                n = np.where(c < G, np.maximum(hc + 1, 0), n + n_b - n_both)
            total += int(n.sum())
        return total

    def flops_exact(self) -> float:
        """Multiply-adds actually required: 4 * D per eligible pair (QK^T and
        PV, two flops per multiply-add each)."""
        return 4.0 * self.D * self.eligible_pairs() * self.Hq

    @property
    def memory_bound(self) -> bool:
        """Below about 64 FLOP per algorithmic byte the HBM, not the tensor
        core, bounds the call (the GB300 ridge point is near 280)."""
        return self.flops() < 64 * self.io_bytes()

    def io_bytes(self) -> int:
        """Algorithmic HBM bytes of one call.  Forward: read Q, K, V once,
        write O and the FP32 logsumexp once.  Backward: read Q, K, V, O, dO
        and lse once, write dQ, dK, dV once."""
        esz = torch.tensor([], dtype=self.dtype).element_size()
        tq, tk = self.total_tokens, self.total_keys
        if self.backward:
            return (4 * tq * self.Hq * self.D + 4 * tk * self.Hkv * self.D) * esz + tq * self.Hq * 4
        return (2 * tq * self.Hq * self.D + 2 * tk * self.Hkv * self.D) * esz + tq * self.Hq * 4


def _named(name, description, *args, **kw):
    return name, Workload(name, description, *args, **kw)


F16, BF16 = torch.float16, torch.bfloat16

# Workloads by what they are: sizes, layout, dtype and mask.
WORKLOADS = dict([
    _named("n129_d32_f16_causal", "single head, causal, N=129, D=32, FP16", 1, 1, 1, 129, 32, F16, True),
    _named("n512_d64_f16_causal", "single head, causal, N=512, D=64, FP16", 1, 1, 1, 512, 64, F16, True),
    _named("n512_d64_f16_noncausal", "single head, non-causal, N=512, D=64, FP16", 1, 1, 1, 512, 64, F16, False),
    _named("n512_d64_f16_causal_qx30", "single head, causal, N=512, D=64, FP16, Q x30", 1, 1, 1, 512, 64, F16, True,
           q_scale=30.0),
    _named("b4_h16_n4096_d128_bf16", "B=4, H=16, N=4096, D=128, BF16, causal, [B,H,N,D]", 4, 16, 16, 4096, 128,
           BF16, True),
    _named("b4_h16_n4096_d128_bf16_bnhd", "B=4, H=16, N=4096, D=128, BF16, causal, [B,N,H,D] strides", 4, 16, 16,
           4096, 128, BF16, True, layout="bnhd"),
    _named("gqa_b2_h32x8_n8192_d128_bf16", "GQA B=2, Hq=32, Hkv=8, N=8192, D=128, BF16, causal", 2, 32, 8, 8192,
           128, BF16, True),
    _named("varlen16_h16_d128_bf16", "packed varlen, 16 sequences (seed 7), H=16, D=128, BF16, causal", 1, 16, 16,
           max(VARLEN_LENGTHS_SEED7), 128, BF16, True, layout="varlen", seqlens=tuple(VARLEN_LENGTHS_SEED7)),
    # Unequal lengths and local windows.
    _named("chunk2048_cache16384_gqa", "GQA B=2, Hq=32, Hkv=8, 2048 new queries over 16384 keys (bottom-right "
           "causal), D=128, BF16", 2, 32, 8, 2048, 128, BF16, True, Nk=16384),
    _named("window4096_n16384", "B=2, H=16, N=16384, causal local window of 4096 keys (diagonal included), D=128, "
           "BF16", 2, 16, 16, 16384, 128, BF16, True, window_left=4095),
    _named("global64_window4096_n16384", "B=2, H=16, N=16384, causal local window of 4096 keys plus 64 global "
           "tokens, D=128, BF16", 2, 16, 16, 16384, 128, BF16, True, window_left=4095, num_global=64),
    # The backward pass of two forward workloads.
    _named("bwd_b4_h16_n4096_d128_bf16", "backward: B=4, H=16, N=4096, D=128, BF16, causal, [B,H,N,D]", 4, 16, 16,
           4096, 128, BF16, True, backward=True),
    _named("bwd_gqa_b2_h32x8_n8192_d128_bf16", "backward: GQA B=2, Hq=32, Hkv=8, N=8192, D=128, BF16, causal", 2,
           32, 8, 8192, 128, BF16, True, backward=True),
    # Few queries over many keys: split-KV.
    _named("decode_b8_h32x8_k32768", "decode step: GQA B=8, Hq=32, Hkv=8, 1 query over 32768 keys, D=128, BF16, "
           "split-KV", 8, 32, 8, 1, 128, BF16, True, Nk=32768, splitkv=True),
])


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
        T, Tk = w.total_tokens, w.total_keys
        q = _draw((T, w.Hq, w.D), g, w.dtype, w.q_scale)
        k = _draw((Tk, w.Hkv, w.D), g, w.dtype)
        v = _draw((Tk, w.Hkv, w.D), g, w.dtype)
        out = {"q": q, "k": k, "v": v, "cu_seqlens": cu_seqlens_of(w.seqlens)}
        if w.seqlens_k:
            out["cu_seqlens_k"] = cu_seqlens_of(w.seqlens_k)
        return out
    q = _draw((w.B, w.Hq, w.N, w.D), g, w.dtype, w.q_scale)
    k = _draw((w.B, w.Hkv, w.keys, w.D), g, w.dtype)
    v = _draw((w.B, w.Hkv, w.keys, w.D), g, w.dtype)
    if w.layout == "bnhd":
        q, k, v = (t.permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3) for t in (q, k, v))
    return {"q": q, "k": k, "v": v}


def random_qkv(B, Hq, Hkv, N, D, dtype, seed=0, layout="bhnd", q_scale=1.0, Nk=None):
    """Small seeded inputs of arbitrary shape (same recipe as make_inputs)."""
    w = Workload("adhoc", "adhoc", B, Hq, Hkv, N, D, dtype, True, layout=layout, q_scale=q_scale, Nk=Nk)
    return make_inputs(w, seed)


def random_varlen(lengths, Hq, Hkv, D, dtype, seed=0, q_scale=1.0, lengths_k=None):
    w = Workload("adhoc_varlen", "adhoc", 1, Hq, Hkv, max(lengths) if lengths else 0, D, dtype, True,
                 layout="varlen", q_scale=q_scale, seqlens=tuple(int(x) for x in lengths),
                 seqlens_k=tuple(int(x) for x in lengths_k) if lengths_k is not None else ())
    return make_inputs(w, seed)
