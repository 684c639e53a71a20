"""CPU checks of the seeded workload generators (shapes, seeds, lengths)."""

import torch

from exact_tiled_attention_19_gb300 import workloads as W


def test_varlen_lengths_seed7():
    assert W.varlen_lengths_from_seed(7) == W.VARLEN_LENGTHS_SEED7
    assert sum(W.VARLEN_LENGTHS_SEED7) == 124825 and max(W.VARLEN_LENGTHS_SEED7) == 14891


def test_cu_seqlens():
    cu = W.cu_seqlens_of([3, 0, 5])
    assert cu.tolist() == [0, 3, 3, 8] and cu.dtype == torch.int32


def test_small_workload_shapes_and_determinism():
    a = W.make_inputs("n129_d32_f16_causal")
    b = W.make_inputs("n129_d32_f16_causal")
    assert a["q"].shape == (1, 1, 129, 32) and a["q"].dtype == torch.float16
    assert torch.equal(a["q"], b["q"]) and torch.equal(a["v"], b["v"])
    big = W.make_inputs("n512_d64_f16_causal_qx30")
    base = W.make_inputs("n512_d64_f16_causal")
    assert torch.equal(big["k"], base["k"])
    assert float(big["q"].float().abs().max()) > 20 * float(base["q"].float().abs().max()) * 0.9


def test_transposed_layout_is_same_logical_values():
    w = W.Workload("t", "t", 2, 3, 3, 17, 32, torch.bfloat16, True)
    wt = W.Workload("t", "t", 2, 3, 3, 17, 32, torch.bfloat16, True, layout="bnhd")
    a, b = W.make_inputs(w), W.make_inputs(wt)
    assert torch.equal(a["q"], b["q"])
    assert b["q"].stride() == (17 * 3 * 32, 32, 3 * 32, 1)


def test_flop_and_byte_conventions():
    packed = W.WORKLOADS["varlen16_h16_d128_bf16"]
    assert abs(packed.flops_convention() - 5.507e12) / 5.507e12 < 1e-3
    batched = W.WORKLOADS["b4_h16_n4096_d128_bf16"]
    assert batched.flops_convention() == 4 * 4096 ** 2 * 128 * 64 / 2
    assert batched.io_bytes() == 4 * 4 * 16 * 4096 * 128 * 2 + 4 * 16 * 4096 * 4


def test_eligible_pair_counts_match_the_oracle_masks():
    """The exact FLOP counts of windowed, chunked and global-token workloads
    come from Workload.eligible_pairs (interval arithmetic); they must equal
    the number of eligible (row, key) pairs of the oracle's own mask."""
    import random

    import numpy as np

    from oracle import dense
    rng = random.Random(5)
    for _ in range(60):
        Nq, Nk = rng.randint(1, 400), rng.randint(1, 400)
        causal = rng.random() < 0.6
        wl = rng.choice([-1, 0, 3, 50, 600])
        wr = rng.choice([-1, 0, 7, 90])
        G = rng.choice([0, 0, 1, 16, 130, 500])
        w = W.Workload("t", "t", 1, 1, 1, Nq, 32, W.BF16, causal, Nk=Nk, window_left=wl, window_right=wr,
                       num_global=G)
        e = dense.eligible_keys(np.arange(Nq), Nk, causal, Nq, wl, wr, G)
        assert w.eligible_pairs() == int(e.sum()), (Nq, Nk, causal, wl, wr, G)
    # the named windowed / chunked / global workloads at their real sizes (one sequence, one head),
    # counted from the oracle's mask in row chunks
    for name in ("window4096_n16384", "chunk2048_cache16384_gqa", "global64_window4096_n16384"):
        w = W.WORKLOADS[name]
        total = 0
        for r0 in range(0, w.N, 2048):
            rows = np.arange(r0, min(w.N, r0 + 2048))
            total += int(dense.eligible_keys(rows, w.keys, w.causal, w.N, w.window_left, w.window_right,
                                             w.num_global).sum())
        assert w.eligible_pairs() == total * w.B, name
        assert w.flops_exact() == 4.0 * w.D * total * w.B * w.Hq
