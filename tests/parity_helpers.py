"""Shared helpers for the GPU parity tests: run the CUDA path through the C
ABI and the FP64 oracle on the same stored inputs and compare."""

import math

import numpy as np
import torch

import oracle
from exact_tiled_attention_19_gb300 import binding

# Tolerances fixed for this path: max |dO| <= 2e-3 (FP16) / 1e-2 (BF16),
# max |d lse| <= 1e-3 (absolute, natural-log units).
O_TOL = {torch.float16: 2e-3, torch.bfloat16: 1e-2}
LSE_TOL = 1e-3


def to64(t):
    """Exact float64 copy of stored FP16/BF16/FP32 values."""
    return t.detach().to("cpu", torch.float32).double().numpy()


def run_gpu(inputs, causal, scale=None, stream=None):
    q, k, v = (inputs[n].cuda() if not inputs[n].is_cuda else inputs[n] for n in ("q", "k", "v"))
    if "cu_seqlens" in inputs:
        cu = inputs["cu_seqlens"]
        lens = (cu[1:] - cu[:-1]).tolist()
        o, lse = binding.attention_varlen(q, k, v, cu.cuda(), max(lens) if lens else 0, causal=causal,
                                          scale=scale, cu_seqlens_host=cu, stream=stream)
    else:
        o, lse = binding.attention(q, k, v, causal=causal, scale=scale, stream=stream)
    torch.cuda.synchronize()
    return o, lse


def rebuild_strided(t):
    """Bring a logical view to the CUDA device keeping its memory layout."""
    if t.is_contiguous():
        return t.cuda()
    # [B,H,N,D] view of [B,N,H,D] storage
    return t.permute(0, 2, 1, 3).contiguous().cuda().permute(0, 2, 1, 3)


def compare_full(inputs, o, lse, causal, scale, dtype):
    """Compare every output element with the dense oracle."""
    if "cu_seqlens" in inputs:
        ro, rl = oracle.attention_varlen(to64(inputs["q"]), to64(inputs["k"]), to64(inputs["v"]),
                                         inputs["cu_seqlens"].numpy(), causal=causal, scale=scale)
    else:
        ro, rl = oracle.attention_dense(to64(inputs["q"]), to64(inputs["k"]), to64(inputs["v"]),
                                        causal=causal, scale=scale)
    go, gl = to64(o), to64(lse)
    do = float(np.max(np.abs(go - ro))) if go.size else 0.0
    finite = np.isfinite(rl)
    dl = float(np.max(np.abs(gl[finite] - rl[finite]))) if finite.any() else 0.0
    assert np.all(np.isfinite(go)), "non-finite output"
    assert do <= O_TOL[dtype], f"max|dO|={do} > {O_TOL[dtype]}"
    assert dl <= LSE_TOL, f"max|dlse|={dl} > {LSE_TOL}"
    return do, dl


def sample_rows(N, rng, extra=8):
    base = {0, 1, 2, 63, 64, 127, 128, 129, 255, 256, N // 2, N - 129, N - 128, N - 2, N - 1}
    base |= set(int(x) for x in rng.integers(0, N, size=extra))
    return sorted(r for r in base if 0 <= r < N)


def compare_sampled_batched(inputs, o, lse, causal, scale, dtype, heads, rng):
    """Compare sampled rows of selected (batch, head) pairs with the oracle
    computed row by row."""
    q, k, v = inputs["q"], inputs["k"], inputs["v"]
    Hq, Hkv, N = q.shape[1], k.shape[1], q.shape[2]
    group = Hq // Hkv
    worst_o = worst_l = 0.0
    for b, h in heads:
        rows = sample_rows(N, rng)
        hk = h // group
        ro, rl = oracle.attention_rows(to64(q[b, h]), to64(k[b, hk]), to64(v[b, hk]), rows, causal=causal,
                                       scale=scale)
        go = to64(o[b, h][rows])
        gl = to64(lse[b, h][rows])
        worst_o = max(worst_o, float(np.max(np.abs(go - ro))))
        worst_l = max(worst_l, float(np.max(np.abs(gl - rl))))
    assert worst_o <= O_TOL[dtype], f"max|dO|={worst_o}"
    assert worst_l <= LSE_TOL, f"max|dlse|={worst_l}"
    return worst_o, worst_l


def compare_sampled_varlen(inputs, o, lse, causal, scale, dtype, seq_heads, rng):
    q, k, v, cu = inputs["q"], inputs["k"], inputs["v"], inputs["cu_seqlens"].numpy()
    group = q.shape[1] // k.shape[1]
    worst_o = worst_l = 0.0
    for s, h in seq_heads:
        L = int(cu[s + 1] - cu[s])
        if L == 0:
            continue
        rows = sample_rows(L, rng)
        t0 = int(cu[s])
        ro, rl = oracle.attention_varlen_rows(to64(q[t0:t0 + L]), to64(k[t0:t0 + L]), to64(v[t0:t0 + L]),
                                              np.array([0, L]), 0, h, rows, causal=causal, scale=scale,
                                              group=group)
        go = to64(o[t0:t0 + L, h][rows])
        gl = to64(lse[h, t0:t0 + L][rows])
        worst_o = max(worst_o, float(np.max(np.abs(go - ro))))
        worst_l = max(worst_l, float(np.max(np.abs(gl - rl))))
    assert worst_o <= O_TOL[dtype], f"max|dO|={worst_o}"
    assert worst_l <= LSE_TOL, f"max|dlse|={worst_l}"
    return worst_o, worst_l


def default_scale(D):
    return 1.0 / math.sqrt(D)
