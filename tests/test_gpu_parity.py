"""GPU parity: the CUDA path (through the C ABI) against the FP64 oracle on
the same seeded inputs.  Small shapes are compared element by element (several
tiles plus ragged tails); the full-size workloads are compared on sampled rows
the oracle computes one by one, in the launch configuration the benchmark
times."""

import numpy as np
import pytest
import torch

from exact_tiled_attention_19_gb300 import binding
from exact_tiled_attention_19_gb300 import workloads as W
from tests.parity_helpers import (compare_full, compare_sampled_batched, compare_sampled_varlen,
                                  default_scale, rebuild_strided, run_gpu)

pytestmark = pytest.mark.gpu

DT = {"f16": torch.float16, "bf16": torch.bfloat16}


@pytest.fixture(autouse=True)
def _device_status_clean():
    yield
    assert binding.etattn_read_device_status(clear=True) == 0


@pytest.mark.parametrize("dt", ["f16", "bf16"])
@pytest.mark.parametrize("D", [32, 64, 128])
@pytest.mark.parametrize("N", [1, 2, 127, 128, 129, 255, 300])
@pytest.mark.parametrize("causal", [True, False])
def test_single_head_ragged(dt, D, N, causal):
    inp = W.random_qkv(1, 1, 1, N, D, DT[dt], seed=N + D)
    o, lse = run_gpu(inp, causal)
    compare_full(inp, o, lse, causal, default_scale(D), DT[dt])


@pytest.mark.parametrize("layout", ["bhnd", "bnhd"])
@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_multihead_gqa_small(layout, dt):
    inp = W.random_qkv(2, 8, 2, 333, 128, DT[dt], seed=5, layout=layout)
    inp = {k_: rebuild_strided(t) for k_, t in inp.items()}
    o, lse = run_gpu(inp, True)
    compare_full({k_: t.cpu() for k_, t in inp.items()}, o, lse, True, default_scale(128), DT[dt])


@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_varlen_small(dt):
    inp = W.random_varlen([1, 130, 0, 257, 64, 128], 4, 2, 128, DT[dt], seed=3)
    o, lse = run_gpu(inp, True)
    compare_full(inp, o, lse, True, default_scale(128), DT[dt])


def test_varlen_small_noncausal():
    inp = W.random_varlen([77, 300, 5], 2, 1, 64, torch.float16, seed=4)
    o, lse = run_gpu(inp, False)
    compare_full(inp, o, lse, False, default_scale(64), torch.float16)


@pytest.mark.parametrize("q_scale", [30.0, 100.0])
@pytest.mark.parametrize("causal", [True, False])
def test_large_logits(q_scale, causal):
    inp = W.random_qkv(1, 2, 2, 640, 64, torch.float16, seed=1, q_scale=q_scale)
    o, lse = run_gpu(inp, causal)
    compare_full(inp, o, lse, causal, default_scale(64), torch.float16)


def test_nondefault_scale():
    inp = W.random_qkv(1, 2, 1, 200, 64, torch.bfloat16, seed=2)
    o, lse = run_gpu(inp, True, scale=0.37)
    compare_full(inp, o, lse, True, 0.37, torch.bfloat16)


# ---------------------------------------------------------------- the named workloads

@pytest.mark.parametrize("name", ["n129_d32_f16_causal", "n512_d64_f16_causal", "n512_d64_f16_noncausal",
                                  "n512_d64_f16_causal_qx30"])
def test_small_workloads_full(name):
    w = W.WORKLOADS[name]
    inp = W.make_inputs(w)
    o, lse = run_gpu(inp, w.causal)
    compare_full(inp, o, lse, w.causal, w.scale, w.dtype, derived_ok=False)


@pytest.mark.parametrize("name", ["b4_h16_n4096_d128_bf16", "b4_h16_n4096_d128_bf16_bnhd",
                                  "gqa_b2_h32x8_n8192_d128_bf16"])
def test_large_batched_workloads_sampled(name):
    w = W.WORKLOADS[name]
    inp = W.make_inputs(w)
    dev = {k_: rebuild_strided(t) for k_, t in inp.items()}
    o, lse = run_gpu(dev, w.causal)
    assert bool(torch.isfinite(o).all()) and bool(torch.isfinite(lse).all())
    rng = np.random.default_rng(0)
    heads = [(0, 0), (w.B - 1, w.Hq - 1), (1 % w.B, w.Hq // 2), (0, 3 % w.Hq), (w.B - 1, 5 % w.Hq)]
    compare_sampled_batched(inp, o.cpu(), lse.cpu(), w.causal, w.scale, w.dtype, heads, rng)


def test_varlen_workload_sampled():
    w = W.WORKLOADS["varlen16_h16_d128_bf16"]
    inp = W.make_inputs(w)
    o, lse = run_gpu(inp, w.causal)
    assert bool(torch.isfinite(o).all()) and bool(torch.isfinite(lse).all())
    rng = np.random.default_rng(1)
    pairs = [(s, (3 * s) % w.Hq) for s in range(len(w.seqlens))] + [(15, 0), (2, 15)]
    compare_sampled_varlen(inp, o.cpu(), lse.cpu(), w.causal, w.scale, w.dtype, pairs, rng)


# The launch uses two 128-row sub-tiles per CTA when that still gives at least
# one CTA per SM, and one sub-tile otherwise.  Many heads with short sequences
# put ragged shapes on the two-sub-tile path (the small cases above take the
# one-sub-tile path).
@pytest.mark.parametrize("N", [129, 300, 511])
@pytest.mark.parametrize("D,dt", [(64, "f16"), (128, "bf16"), (32, "bf16")])
@pytest.mark.parametrize("causal", [True, False])
def test_two_subtile_path_ragged(N, D, dt, causal):
    inp = W.random_qkv(1, 152, 38, N, D, DT[dt], seed=N + 3 * D)
    o, lse = run_gpu(inp, causal)
    compare_full(inp, o, lse, causal, default_scale(D), DT[dt])


def test_two_subtile_path_varlen():
    lengths = [1, 200, 0, 257, 129, 700]
    inp = W.random_varlen(lengths, 64, 16, 128, torch.bfloat16, seed=21)
    o, lse = run_gpu(inp, True)
    compare_full(inp, o, lse, True, default_scale(128), torch.bfloat16)
