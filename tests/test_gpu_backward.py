"""GPU parity of the attention backward pass (attn_bwd) against the FP64
oracle ("Attention algorithms and data movement", lesson 03): dQ, dK, dV of
sum(dO * O) on the same seeded inputs, element by element, under the bound
derived in tests/parity_helpers.compare_backward.  O and lse come from the
GPU forward pass, as in training."""

import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_19_gb300 import binding
from exact_tiled_attention_19_gb300 import workloads as W
from tests.parity_helpers import HALF_ULP, compare_backward, default_scale, rebuild_strided, to64

pytestmark = pytest.mark.gpu

DT = {"f16": torch.float16, "bf16": torch.bfloat16}


@pytest.fixture(autouse=True)
def _device_status_clean():
    yield
    assert binding.etattn_read_device_status(clear=True) == 0


def dout_like(q, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(q.shape, generator=g, dtype=torch.float32).to(q.dtype)


def fwd_bwd(inp, dout, causal, window_left=-1, window_right=-1, scale=None):
    dev = {n: (inp[n] if inp[n].is_cuda else rebuild_strided(inp[n])) for n in ("q", "k", "v")}
    win = dict(window_left=window_left, window_right=window_right)
    o, lse = binding.attention(dev["q"], dev["k"], dev["v"], causal=causal, scale=scale, **win)
    grads = binding.attention_backward(dev["q"], dev["k"], dev["v"], o, lse, dout.cuda(), causal=causal, scale=scale,
                                       **win)
    torch.cuda.synchronize()
    return grads


@pytest.mark.parametrize("N", [1, 129, 300])
@pytest.mark.parametrize("D,dt", [(128, "bf16"), (64, "f16"), (32, "bf16")])
@pytest.mark.parametrize("causal", [True, False])
def test_single_head(N, D, dt, causal):
    inp = W.random_qkv(1, 1, 1, N, D, DT[dt], seed=N + D)
    dout = dout_like(inp["q"], N)
    grads = fwd_bwd(inp, dout, causal)
    compare_backward(inp, dout, grads, causal, default_scale(D), DT[dt])


@pytest.mark.parametrize("layout", ["bhnd", "bnhd"])
def test_gqa_multihead(layout):
    inp = W.random_qkv(2, 8, 2, 333, 128, torch.bfloat16, seed=5, layout=layout)
    dout = dout_like(inp["q"], 6)
    grads = fwd_bwd(inp, dout, True)
    compare_backward(inp, dout, grads, True, default_scale(128), torch.bfloat16)


def test_uneven_dispatch_groups():
    """41 (KV head, batch) pairs of 8 key blocks: the grouped longest-first
    launch cuts them into groups of 21 and 20 pairs (the remainder path of
    the 1-D order); every gradient element against the oracle."""
    inp = W.random_qkv(1, 41, 41, 1024, 64, torch.float16, seed=71)
    dout = dout_like(inp["q"], 72)
    grads = fwd_bwd(inp, dout, True)
    compare_backward(inp, dout, grads, True, default_scale(64), torch.float16)


@pytest.mark.parametrize("Nq,Nk", [(100, 700), (700, 100), (1, 300), (300, 1)])
def test_unequal_lengths(Nq, Nk):
    inp = W.random_qkv(1, 4, 2, Nq, 64, torch.bfloat16, seed=Nq + Nk, Nk=Nk)
    dout = dout_like(inp["q"], 7)
    grads = fwd_bwd(inp, dout, True)
    compare_backward(inp, dout, grads, True, default_scale(64), torch.bfloat16)


@pytest.mark.parametrize("wl,wr,causal", [(50, -1, True), (20, 30, False), (0, 0, True)])
def test_windows(wl, wr, causal):
    inp = W.random_qkv(1, 2, 1, 400, 128, torch.bfloat16, seed=wl + 11)
    dout = dout_like(inp["q"], 8)
    grads = fwd_bwd(inp, dout, causal, window_left=wl, window_right=wr)
    compare_backward(inp, dout, grads, causal, default_scale(128), torch.bfloat16, window_left=wl, window_right=wr)


def test_no_queries_and_no_keys():
    inp = W.random_qkv(1, 2, 2, 0, 64, torch.bfloat16, seed=1, Nk=200)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    o = torch.empty_like(q)
    lse = torch.empty((1, 2, 0), dtype=torch.float32, device="cuda")
    dq, dk, dv = binding.attention_backward(q, k, v, o, lse, torch.empty_like(q), causal=True)
    torch.cuda.synchronize()
    assert bool((dk == 0).all()) and bool((dv == 0).all())
    inp = W.random_qkv(1, 2, 2, 50, 64, torch.bfloat16, seed=2, Nk=0)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    o, lse = binding.attention(q, k, v, causal=True)
    dq, dk, dv = binding.attention_backward(q, k, v, o, lse, torch.ones_like(q), causal=True)
    torch.cuda.synchronize()
    assert bool((dq == 0).all())


def test_oracle_forward_outputs_as_inputs():
    """The backward on its own: O (rounded to the input type) and lse from
    the FP64 forward oracle instead of the GPU forward."""
    inp = W.random_qkv(2, 4, 4, 200, 64, torch.float16, seed=13)
    dout = dout_like(inp["q"], 9)
    ro, rl = oracle.attention_dense(to64(inp["q"]), to64(inp["k"]), to64(inp["v"]), causal=True,
                                    scale=default_scale(64))
    o = torch.tensor(ro, dtype=torch.float32).to(torch.float16).cuda()
    lse = torch.tensor(rl, dtype=torch.float32).cuda()
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    grads = binding.attention_backward(q, k, v, o, lse, dout.cuda(), causal=True)
    torch.cuda.synchronize()
    compare_backward(inp, dout, grads, True, default_scale(64), torch.float16)


def test_key_and_value_gradients_are_deterministic():
    inp = W.random_qkv(1, 8, 2, 500, 128, torch.bfloat16, seed=14)
    dout = dout_like(inp["q"], 10)
    g1 = fwd_bwd(inp, dout, True)
    g2 = fwd_bwd(inp, dout, True)
    assert torch.equal(g1[1], g2[1]) and torch.equal(g1[2], g2[2])  # dQ sums atomically: order may vary


def test_named_workload_sampled():
    w = W.WORKLOADS["b4_h16_n4096_d128_bf16"]
    inp = W.make_inputs(w)
    dout = dout_like(inp["q"], 15)
    dq, dk, dv = fwd_bwd(inp, dout, True)
    u = HALF_ULP[w.dtype]
    rng = np.random.default_rng(4)
    rows = sorted({0, 1, 127, 128, 2047, 4095} | set(int(x) for x in rng.integers(0, 4096, 4)))
    worst = 0.0
    for b, hk in ((0, 0), (w.B - 1, w.Hkv - 1), (1, 7)):
        out = oracle.attention_backward_sampled(to64(inp["q"][b, hk:hk + 1]), to64(inp["k"][b, hk]),
                                                to64(inp["v"][b, hk]), to64(dout[b, hk:hk + 1]), rows, rows,
                                                causal=True, scale=w.scale, group=1, magnitudes=True)
        gpu = (to64(dq[b, hk:hk + 1])[:, rows], to64(dk[b, hk])[rows], to64(dv[b, hk])[rows])
        for g, r, m in zip(gpu, out[:3], out[3:]):
            bound = u * np.abs(r) + 8 * u * m + 1e-6 * max(float(m.max()), 1e-30)  # as in compare_backward
            worst = max(worst, float((np.abs(g - r) / bound).max()))
    assert worst <= 1.0, worst
