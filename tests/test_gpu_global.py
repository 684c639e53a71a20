"""GPU parity of global tokens beside a local window (attn_fwd_global;
"Attention algorithms and data movement", lesson 07, global-token unions).
Every row also reads the first num_global keys and every global row reads
all keys, both under the causal mask only; the kernel streams each query
tile's global keys and then the rest of its rows' keys, so each connection is
counted once.  The result must match the FP64 oracle on
the same seeded inputs."""

import numpy as np
import pytest
import torch

from exact_tiled_attention_19_gb300 import binding
from exact_tiled_attention_19_gb300 import workloads as W
from tests.parity_helpers import compare_full, compare_sampled_batched, default_scale, rebuild_strided

pytestmark = pytest.mark.gpu

DT = {"f16": torch.float16, "bf16": torch.bfloat16}


@pytest.fixture(autouse=True)
def _device_status_clean():
    yield
    assert binding.etattn_read_device_status(clear=True) == 0


def run_global(inp, G, causal, wl, wr):
    q, k, v = (inp[n] if inp[n].is_cuda else rebuild_strided(inp[n]) for n in ("q", "k", "v"))
    o, lse = binding.attention_global(q, k, v, num_global=G, causal=causal, window_left=wl, window_right=wr)
    torch.cuda.synchronize()
    return o, lse


@pytest.mark.parametrize("N", [1, 64, 129, 300, 700])
@pytest.mark.parametrize("G,wl,wr,causal", [(1, 16, 0, True), (7, 100, 0, True), (64, 200, 0, True),
                                            (130, 50, 0, True), (5, 30, 40, False), (200, 0, 0, False)])
def test_global_matches_oracle(N, G, wl, wr, causal):
    inp = W.random_qkv(1, 4, 2, N, 64, torch.bfloat16, seed=N + G + wl)
    o, lse = run_global(inp, G, causal, wl, wr)
    compare_full(inp, o, lse, causal, default_scale(64), torch.bfloat16, window_left=wl, window_right=wr,
                 num_global=G)


@pytest.mark.parametrize("D,dt", [(32, "f16"), (64, "f16"), (128, "bf16"), (128, "f16")])
def test_global_head_dims_and_types(D, dt):
    inp = W.random_qkv(2, 2, 2, 333, D, DT[dt], seed=D)
    o, lse = run_global(inp, 40, True, 96, 0)
    compare_full(inp, o, lse, True, default_scale(D), DT[dt], window_left=96, window_right=0, num_global=40)


@pytest.mark.parametrize("Nq,Nk", [(37, 500), (128, 900), (500, 200)])
def test_global_unequal_lengths(Nq, Nk):
    """Bottom-right alignment: query row r sits at key position r + Nk - Nq;
    it is a global row when that position is below num_global."""
    inp = W.random_qkv(1, 8, 2, Nq, 128, torch.bfloat16, seed=Nq + Nk, Nk=Nk)
    for G, wl in ((20, 64), (300, 10)):
        o, lse = run_global(inp, G, True, wl, 0)
        compare_full(inp, o, lse, True, default_scale(128), torch.bfloat16, window_left=wl, window_right=0,
                     num_global=G)


def test_global_decode_rows_pack_query_heads():
    """Few query tokens of a grouped-query problem share a tile across the
    group's query heads (the decode packing) in the global launch too."""
    inp = W.random_qkv(2, 32, 8, 1, 128, torch.bfloat16, seed=3, Nk=5000)
    o, lse = run_global(inp, 64, True, 1024, 0)
    compare_full(inp, o, lse, True, default_scale(128), torch.bfloat16, window_left=1024, window_right=0,
                 num_global=64)


def test_global_strided_layout():
    inp = W.random_qkv(2, 4, 4, 300, 64, torch.float16, seed=9, layout="bnhd")
    o, lse = run_global(inp, 33, True, 70, 0)
    compare_full(inp, o, lse, True, default_scale(64), torch.float16, window_left=70, window_right=0, num_global=33)


def test_global_zero_and_window_covering_everything_equal_plain_calls_bitwise():
    inp = W.random_qkv(1, 4, 4, 400, 64, torch.bfloat16, seed=11)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    o0, l0 = binding.attention_global(q, k, v, num_global=0, causal=True, window_left=50, window_right=0)
    p0, m0 = binding.attention(q, k, v, causal=True, window_left=50, window_right=0)
    assert torch.equal(o0, p0) and torch.equal(l0, m0)
    o1, l1 = binding.attention_global(q, k, v, num_global=32, causal=True, window_left=-1)
    p1, m1 = binding.attention(q, k, v, causal=True)
    assert torch.equal(o1, p1) and torch.equal(l1, m1)


def test_global_more_than_every_key_is_causal_attention():
    inp = W.random_qkv(1, 4, 4, 300, 64, torch.bfloat16, seed=12)
    o, lse = run_global(inp, 10_000, True, 5, 0)
    compare_full(inp, o, lse, True, default_scale(64), torch.bfloat16)


def test_global_repeated_calls_are_bitwise_stable():
    inp = W.random_qkv(2, 4, 2, 600, 128, torch.bfloat16, seed=13)
    o1, l1 = run_global(inp, 48, True, 128, 0)
    o2, l2 = run_global(inp, 48, True, 128, 0)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_global_window_workload_sampled():
    """The benchmarked shape: sampled rows (every global row boundary, window
    edges, the ends) of selected heads against the oracle row by row."""
    w = W.WORKLOADS["global64_window4096_n16384"]
    inp = W.make_inputs(w)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    o, lse = binding.attention_global(q, k, v, num_global=w.num_global, causal=True, window_left=w.window_left,
                                      window_right=w.window_right)
    torch.cuda.synchronize()
    inp_dev = {"q": q, "k": k, "v": v}
    rng = np.random.default_rng(0)
    rows = sorted({0, 1, 62, 63, 64, 65, 127, 128, 4095, 4096, 4159, 4160, 4161, 8191, 12000, w.N - 2, w.N - 1}
                  | set(int(x) for x in rng.integers(0, w.N, size=8)))
    compare_sampled_batched(inp_dev, o, lse, True, default_scale(w.D), w.dtype, [(0, 0), (0, w.Hq - 1)], rng,
                            window_left=w.window_left, window_right=w.window_right, num_global=w.num_global,
                            rows=rows)


@pytest.mark.parametrize("causal,wl,wr", [(True, 48, 0), (False, 20, 30)])
def test_varlen_global_tokens_are_per_sequence(causal, wl, wr):
    """Packed batches: the first G positions of every sequence are global."""
    inp = W.random_varlen([1, 0, 129, 700, 40, 333], 4, 2, 128, torch.bfloat16, seed=14)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    cu = inp["cu_seqlens"]
    lens = (cu[1:] - cu[:-1]).tolist()
    o, lse = binding.attention_varlen(q, k, v, cu.cuda(), max(lens), causal=causal, cu_seqlens_host=cu,
                                      num_global=17, window_left=wl, window_right=wr)
    torch.cuda.synchronize()
    compare_full(inp, o, lse, causal, default_scale(128), torch.bfloat16, window_left=wl, window_right=wr,
                 num_global=17)


def test_varlen_global_with_separate_key_offsets():
    inp = W.random_varlen([20, 5, 128], 8, 2, 64, torch.float16, seed=15, lengths_k=[400, 60, 128])
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    cu, cuk = inp["cu_seqlens"], inp["cu_seqlens_k"]
    o, lse = binding.attention_varlen(q, k, v, cu.cuda(), 128, causal=True, cu_seqlens_host=cu,
                                      cu_seqlens_k=cuk.cuda(), max_seqlen_k=400, cu_seqlens_k_host=cuk,
                                      num_global=10, window_left=32)
    torch.cuda.synchronize()
    compare_full(inp, o, lse, True, default_scale(64), torch.float16, window_left=32, num_global=10)
