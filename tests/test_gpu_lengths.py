"""GPU parity for unequal query/key lengths, local windows and rows with no
eligible key ("Attention algorithms and data movement", lessons 04 and 07),
through attn_fwd_ex / attn_fwd_varlen_ex, against the FP64 oracle on the same
seeded inputs.  Query row r of Lq sits at key position r + Lk - Lq; rows with
no eligible key must come out exactly as O = 0, lse = -inf."""

import numpy as np
import pytest
import torch

from exact_tiled_attention_19_gb300 import binding
from exact_tiled_attention_19_gb300 import workloads as W
from tests.parity_helpers import compare_full, compare_sampled_batched, default_scale, rebuild_strided, run_gpu

pytestmark = pytest.mark.gpu

DT = {"f16": torch.float16, "bf16": torch.bfloat16}


@pytest.fixture(autouse=True)
def _device_status_clean():
    yield
    assert binding.etattn_read_device_status(clear=True) == 0


# ---------------------------------------------------------------- unequal lengths

@pytest.mark.parametrize("Nq,Nk", [(1, 1), (1, 300), (7, 1000), (128, 129), (129, 128), (200, 70), (255, 513),
                                   (300, 77), (5, 3), (129, 1)])
@pytest.mark.parametrize("causal", [True, False])
def test_unequal_lengths_single_head(Nq, Nk, causal):
    inp = W.random_qkv(1, 2, 1, Nq, 64, torch.float16, seed=Nq + 7 * Nk, Nk=Nk)
    o, lse = run_gpu(inp, causal)
    compare_full(inp, o, lse, causal, default_scale(64), torch.float16)


@pytest.mark.parametrize("Nq,Nk", [(129, 700), (511, 129), (300, 300), (1, 2000)])
@pytest.mark.parametrize("D,dt", [(128, "bf16"), (32, "f16")])
def test_unequal_lengths_two_subtile_path(Nq, Nk, D, dt):
    # 152 query heads keep the launch on two 128-row sub-tiles per CTA.
    inp = W.random_qkv(1, 152, 38, Nq, D, DT[dt], seed=Nq + Nk + D, Nk=Nk)
    o, lse = run_gpu(inp, True)
    compare_full(inp, o, lse, True, default_scale(D), DT[dt])


@pytest.mark.parametrize("causal", [True, False])
def test_no_keys_gives_empty_rows(causal):
    inp = W.random_qkv(2, 4, 2, 300, 128, torch.bfloat16, seed=3, Nk=0)
    o, lse = run_gpu(inp, causal)
    assert bool((o == 0).all()) and bool((lse == float("-inf")).all())


def test_square_ex_call_matches_square_entry_point_bitwise():
    inp = W.random_qkv(2, 8, 2, 700, 128, torch.bfloat16, seed=9)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    o1, l1 = binding.attention(q, k, v, causal=True)
    o2, l2 = binding.attention(q, k, v, causal=True, window_left=1 << 20)  # a window wider than the keys
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_decode_gqa_full():
    # One new query per sequence over a 16384-key cache, GQA 32/8.
    inp = W.random_qkv(4, 32, 8, 1, 128, torch.bfloat16, seed=11, Nk=16384)
    o, lse = run_gpu(inp, True)
    compare_full(inp, o, lse, True, default_scale(128), torch.bfloat16)


# ---------------------------------------------------------------- local windows

WINDOWS = [(0, 0, True), (5, -1, True), (127, -1, True), (128, -1, True), (200, 0, True), (3, 7, False),
           (-1, 10, False), (100, 100, False), (0, -1, False)]


@pytest.mark.parametrize("wl,wr,causal", WINDOWS)
@pytest.mark.parametrize("Nq,Nk", [(300, 300), (100, 700), (700, 100)])
def test_windows_single_head(wl, wr, causal, Nq, Nk):
    inp = W.random_qkv(1, 1, 1, Nq, 64, torch.float16, seed=wl + 3 * wr + Nq, Nk=Nk)
    o, lse = run_gpu(inp, causal, window_left=wl, window_right=wr)
    compare_full(inp, o, lse, causal, default_scale(64), torch.float16, window_left=wl, window_right=wr)


@pytest.mark.parametrize("wl,wr,causal", [(200, -1, True), (64, 64, False), (0, 0, True)])
@pytest.mark.parametrize("N", [513, 1000])
def test_windows_two_subtile_path(wl, wr, causal, N):
    inp = W.random_qkv(1, 152, 38, N, 128, torch.bfloat16, seed=N + wl, layout="bnhd")
    dev = {k_: rebuild_strided(t) for k_, t in inp.items()}
    o, lse = run_gpu(dev, causal, window_left=wl, window_right=wr)
    compare_full(inp, o, lse, causal, default_scale(128), torch.bfloat16, window_left=wl, window_right=wr)


def test_window_mask_is_exact_under_perturbation():
    """Changing a key/value outside a row's window leaves that row's output
    bit-identical; rows whose window holds the key change."""
    N, wl, j0 = 600, 50, 300
    inp = W.random_qkv(1, 1, 1, N, 128, torch.bfloat16, seed=5)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    o1, l1 = binding.attention(q, k, v, causal=True, window_left=wl)
    k2, v2 = k.clone(), v.clone()
    k2[0, 0, j0] = 0.0    # a logit of 0 against ~N(0, 1) others: weight about 1/50 in every window holding it
    v2[0, 0, j0] = 100.0
    o2, l2 = binding.attention(q, k2, v2, causal=True, window_left=wl)
    torch.cuda.synchronize()
    sees = np.zeros(N, dtype=bool)
    sees[j0:j0 + wl + 1] = True  # rows i with i - wl <= j0 <= i
    same_o = (o1[0, 0] == o2[0, 0]).all(dim=1).cpu().numpy()
    same_l = (l1[0, 0] == l2[0, 0]).cpu().numpy()
    assert same_o[~sees].all() and same_l[~sees].all()
    assert not same_o[sees].any()


# ---------------------------------------------------------------- packed batches with separate key offsets

@pytest.mark.parametrize("wl,wr,causal", [(-1, -1, True), (-1, -1, False), (40, -1, True), (20, 30, False)])
def test_varlen_separate_key_lengths(wl, wr, causal):
    lq = [1, 130, 0, 257, 64, 5, 300]
    lk = [300, 130, 10, 0, 64, 700, 100]
    inp = W.random_varlen(lq, 4, 2, 128, torch.bfloat16, seed=17, lengths_k=lk)
    o, lse = run_gpu(inp, causal, window_left=wl, window_right=wr)
    compare_full(inp, o, lse, causal, default_scale(128), torch.bfloat16, window_left=wl, window_right=wr)


def test_varlen_separate_keys_two_subtile_path():
    lq = [700, 1, 129, 0, 512]
    lk = [900, 4000, 129, 50, 256]
    inp = W.random_varlen(lq, 64, 16, 128, torch.bfloat16, seed=23, lengths_k=lk)
    o, lse = run_gpu(inp, True, window_left=300)
    compare_full(inp, o, lse, True, default_scale(128), torch.bfloat16, window_left=300)


def test_varlen_no_keys_at_all():
    inp = W.random_varlen([3, 200, 0], 2, 2, 64, torch.float16, seed=2, lengths_k=[0, 0, 0])
    o, lse = run_gpu(inp, False)
    assert bool((o == 0).all()) and bool((lse == float("-inf")).all())


def test_varlen_bad_key_offsets_reported_by_the_device():
    inp = W.random_varlen([64, 64], 2, 2, 64, torch.float16, seed=2, lengths_k=[64, 64])
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    cu = inp["cu_seqlens"].cuda()
    bad_k = torch.tensor([0, 100, 90], dtype=torch.int32, device="cuda")  # decreasing
    binding.attention_varlen(q, k, v, cu, 64, cu_seqlens_k=bad_k, max_seqlen_k=100)
    assert binding.etattn_read_device_status(clear=True) == 9


# ---------------------------------------------------------------- the named workloads (sampled)

@pytest.mark.parametrize("name", ["chunk2048_cache16384_gqa", "window4096_n16384"])
def test_named_length_and_window_workloads_sampled(name):
    w = W.WORKLOADS[name]
    inp = W.make_inputs(w)
    o, lse = run_gpu(inp, w.causal, window_left=w.window_left, window_right=w.window_right)
    assert bool(torch.isfinite(o).all()) and bool(torch.isfinite(lse).all())
    rng = np.random.default_rng(2)
    heads = [(0, 0), (w.B - 1, w.Hq - 1), (1 % w.B, w.Hq // 2), (0, 5 % w.Hq)]
    compare_sampled_batched(inp, o.cpu(), lse.cpu(), w.causal, w.scale, w.dtype, heads, rng,
                            window_left=w.window_left, window_right=w.window_right)


# ---------------------------------------------------------------- grouped-query packing
# Fewer than 128 query tokens of a grouped-query problem share a 128-row tile
# among P query heads of one KV group (P = the largest power of two dividing
# Hq / Hkv): 128 / P tokens of each head.

@pytest.mark.parametrize("Hq,Hkv", [(12, 2), (16, 1), (64, 1), (128, 1)])
@pytest.mark.parametrize("Nq", [1, 3, 40])
@pytest.mark.parametrize("layout", ["bhnd", "bnhd"])
def test_gqa_packing_group_sizes(Hq, Hkv, Nq, layout):
    inp = W.random_qkv(2, Hq, Hkv, Nq, 64, torch.float16, seed=Hq + Nq, layout=layout, Nk=700)
    dev = {k_: rebuild_strided(t) for k_, t in inp.items()}
    o, lse = run_gpu(dev, True)
    compare_full(inp, o, lse, True, default_scale(64), torch.float16)


def test_gqa_packing_with_window_and_empty_rows():
    inp = W.random_qkv(1, 8, 2, 100, 128, torch.bfloat16, seed=31, Nk=60)  # first 40 causal rows empty
    o, lse = run_gpu(inp, True, window_left=20)
    compare_full(inp, o, lse, True, default_scale(128), torch.bfloat16, window_left=20)


def test_gqa_packing_packed_batch():
    lq = [1, 5, 0, 64, 2]
    lk = [300, 700, 10, 64, 0]
    inp = W.random_varlen(lq, 8, 2, 128, torch.bfloat16, seed=29, lengths_k=lk)
    o, lse = run_gpu(inp, True)
    compare_full(inp, o, lse, True, default_scale(128), torch.bfloat16)


@pytest.mark.parametrize("causal", [True, False])
def test_key_split_wave_model_launch_full(causal):
    """A general (Lq != Lk) launch whose 192 equal two-sub-tile CTAs would
    leave its second wave mostly empty on a 148- or 152-SM GPU, with 32 key
    tiles per query block: the launcher takes the key split (384 CTAs of half
    the keys each).  Every element against the oracle, at the stated bounds."""
    inp = W.random_qkv(1, 24, 6, 2048, 128, torch.bfloat16, seed=61, Nk=4096)
    o, lse = run_gpu(inp, causal)
    compare_full(inp, o, lse, causal, default_scale(128), torch.bfloat16)
