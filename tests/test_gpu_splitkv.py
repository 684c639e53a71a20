"""GPU parity of the split-KV forward pass (attn_fwd_splitkv): the keys are
cut into slices computed by separate CTAs, and a second launch merges the
slices' partial states ("Intermediate and advanced extension", workshop row
"Split softmax").  The result must match the FP64 oracle of plain attention
on the same seeded inputs, with rows that have no eligible key exactly
O = 0, lse = -inf."""

import numpy as np
import pytest
import torch

from exact_tiled_attention_19_gb300 import binding
from exact_tiled_attention_19_gb300 import workloads as W
from tests.parity_helpers import (LSE_TOL, O_TOL, compare_full, compare_sampled_batched, default_scale,
                                  rebuild_strided)

pytestmark = pytest.mark.gpu

DT = {"f16": torch.float16, "bf16": torch.bfloat16}


@pytest.fixture(autouse=True)
def _device_status_clean():
    yield
    assert binding.etattn_read_device_status(clear=True) == 0


def run_split(inp, causal, num_splits, window_left=-1, window_right=-1, workspace=None):
    q, k, v = (inp[n] if inp[n].is_cuda else inp[n].cuda() for n in ("q", "k", "v"))
    o, lse = binding.attention_splitkv(q, k, v, causal=causal, num_splits=num_splits, workspace=workspace,
                                       window_left=window_left, window_right=window_right)
    torch.cuda.synchronize()
    return o, lse


@pytest.mark.parametrize("Nq,Nk", [(1, 1), (1, 127), (1, 1000), (3, 5000), (128, 700), (129, 900), (300, 300)])
@pytest.mark.parametrize("splits", [2, 3, 16])
@pytest.mark.parametrize("causal", [True, False])
def test_splitkv_matches_oracle(Nq, Nk, splits, causal):
    inp = W.random_qkv(2, 8, 2, Nq, 128, torch.bfloat16, seed=Nq + Nk + splits, Nk=Nk)
    o, lse = run_split(inp, causal, splits)
    compare_full(inp, o, lse, causal, default_scale(128), torch.bfloat16)


@pytest.mark.parametrize("D,dt", [(32, "f16"), (64, "f16"), (64, "bf16")])
def test_splitkv_head_dims(D, dt):
    inp = W.random_qkv(1, 4, 4, 5, D, DT[dt], seed=D, Nk=3000)
    o, lse = run_split(inp, True, 6)
    compare_full(inp, o, lse, True, default_scale(D), DT[dt])


@pytest.mark.parametrize("wl,wr,causal", [(300, -1, True), (0, 0, True), (50, 50, False)])
def test_splitkv_windows(wl, wr, causal):
    # Slices wholly outside a row's window leave lse_s = -inf for it.
    inp = W.random_qkv(1, 4, 1, 64, 64, torch.float16, seed=wl + 5, Nk=2000)
    o, lse = run_split(inp, causal, 8, window_left=wl, window_right=wr)
    compare_full(inp, o, lse, causal, default_scale(64), torch.float16, window_left=wl, window_right=wr)


def test_splitkv_empty_rows_and_no_keys():
    inp = W.random_qkv(1, 2, 2, 200, 64, torch.float16, seed=8, Nk=70)  # the first 130 causal rows are empty
    o, lse = run_split(inp, True, 2)
    compare_full(inp, o, lse, True, default_scale(64), torch.float16)
    inp0 = W.random_qkv(1, 2, 2, 10, 64, torch.float16, seed=8, Nk=0)
    o0, l0 = run_split(inp0, True, 4)
    assert bool((o0 == 0).all()) and bool((l0 == float("-inf")).all())


def test_splitkv_strided_output_layout():
    inp = W.random_qkv(2, 8, 2, 4, 128, torch.bfloat16, seed=3, layout="bnhd", Nk=2048)
    dev = {k_: rebuild_strided(t) for k_, t in inp.items()}
    q, k, v = dev["q"], dev["k"], dev["v"]
    out = torch.empty((2, 4, 8, 128), dtype=torch.bfloat16, device="cuda").permute(0, 2, 1, 3)  # [B,N,H,D] storage
    o, lse = binding.attention_splitkv(q, k, v, causal=True, num_splits=5, out=out)
    torch.cuda.synchronize()
    assert o.data_ptr() == out.data_ptr()
    compare_full(inp, o, lse, True, default_scale(128), torch.bfloat16)


def test_one_slice_is_the_plain_call_bitwise():
    inp = W.random_qkv(2, 8, 2, 7, 128, torch.bfloat16, seed=4, Nk=3000)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    o1, l1 = binding.attention(q, k, v, causal=True)
    o2, l2 = binding.attention_splitkv(q, k, v, causal=True, num_splits=1)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_workspace_contents_do_not_matter():
    inp = W.random_qkv(2, 8, 2, 2, 128, torch.bfloat16, seed=6, Nk=4096)
    need = binding.attn_fwd_splitkv_workspace_size(2, 8, 2, 128, 7)
    ws = torch.full((need // 4,), float("nan"), dtype=torch.float32, device="cuda").view(torch.uint8)
    o1, l1 = run_split(inp, True, 7, workspace=ws)
    ws.fill_(0xff)
    o2, l2 = run_split(inp, True, 7, workspace=ws)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    compare_full(inp, o1, l1, True, default_scale(128), torch.bfloat16)


def test_split_and_plain_results_agree_within_rounding():
    inp = W.random_qkv(4, 16, 4, 1, 128, torch.bfloat16, seed=12, Nk=16384)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    o1, l1 = binding.attention(q, k, v, causal=True)
    o2, l2 = binding.attention_splitkv(q, k, v, causal=True, num_splits=32)
    torch.cuda.synchronize()
    assert float((o1.float() - o2.float()).abs().max()) <= O_TOL[torch.bfloat16]
    assert float((l1 - l2).abs().max()) <= LSE_TOL


def test_plan_is_sane():
    rc, n = binding.attn_fwd_splitkv_plan(8, 32, 8, 1, 32768)
    assert rc == 0 and 2 <= n <= 64
    rc, n = binding.attn_fwd_splitkv_plan(4, 16, 16, 4096, 4096)
    assert rc == 0 and n == 1  # enough query blocks to fill the GPU
    rc, n = binding.attn_fwd_splitkv_plan(1, 1, 1, 1, 500)
    assert rc == 0 and n == 1  # too few key tiles to cut
    assert binding.attn_fwd_splitkv_plan(1, 6, 4, 1, 500)[0] == 4  # Hq not a multiple of Hkv


def test_named_decode_workload():
    w = W.WORKLOADS["decode_b8_h32x8_k32768"]
    inp = W.make_inputs(w)
    rc, n = binding.attn_fwd_splitkv_plan(w.B, w.Hq, w.Hkv, w.N, w.keys)
    assert rc == 0 and n > 1
    o, lse = run_split(inp, w.causal, n)
    rng = np.random.default_rng(3)
    heads = [(b, h) for b in (0, w.B - 1) for h in (0, 5, w.Hq - 1)]
    compare_sampled_batched(inp, o.cpu(), lse.cpu(), w.causal, w.scale, w.dtype, heads, rng)


# ---------------------------------------------------------------- packed batches (attn_fwd_varlen_splitkv)

def run_varlen_split(inp, causal, num_splits, window_left=-1, window_right=-1):
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    cu = inp["cu_seqlens"]
    cuk = inp.get("cu_seqlens_k", cu)
    lq, lk = (cu[1:] - cu[:-1]).tolist(), (cuk[1:] - cuk[:-1]).tolist()
    kw = dict(cu_seqlens_k=cuk.cuda(), max_seqlen_k=max(lk), cu_seqlens_k_host=cuk) if "cu_seqlens_k" in inp else {}
    o, lse = binding.attention_varlen(q, k, v, cu.cuda(), max(lq), causal=causal, cu_seqlens_host=cu,
                                      num_splits=num_splits, window_left=window_left, window_right=window_right,
                                      **kw)
    torch.cuda.synchronize()
    return o, lse


@pytest.mark.parametrize("splits", [2, 5])
@pytest.mark.parametrize("causal", [True, False])
def test_varlen_splitkv_self_attention_matches_oracle(splits, causal):
    inp = W.random_varlen([1, 0, 129, 700, 33, 1500], 4, 2, 128, torch.bfloat16, seed=splits)
    o, lse = run_varlen_split(inp, causal, splits)
    compare_full(inp, o, lse, causal, default_scale(128), torch.bfloat16)


@pytest.mark.parametrize("splits", [3, 8])
def test_varlen_splitkv_decode_rows_over_long_keys(splits):
    """A few query rows per sequence over long key histories (packed
    decode): bottom-right causal, grouped-query heads packed per tile, a
    sequence without keys and one without queries."""
    inp = W.random_varlen([1, 4, 0, 2, 1], 16, 4, 128, torch.bfloat16, seed=10 + splits,
                          lengths_k=[3000, 257, 900, 0, 1])
    o, lse = run_varlen_split(inp, True, splits)
    compare_full(inp, o, lse, True, default_scale(128), torch.bfloat16)


def test_varlen_splitkv_with_window_equals_oracle():
    inp = W.random_varlen([300, 1000, 64], 4, 4, 64, torch.float16, seed=21)
    o, lse = run_varlen_split(inp, True, 4, window_left=200)
    compare_full(inp, o, lse, True, default_scale(64), torch.float16, window_left=200)
