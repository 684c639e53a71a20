"""Pins for the oracle's unequal query/key lengths, sliding windows and empty
rows (CPU only).  Reading fixed here: query row i of Lq sits at key position
c_i = i + Lk - Lq (bottom-right alignment); causal keeps j <= c_i; a window
keeps c_i - window_left <= j <= c_i + window_right; a row with no eligible
key gives O = 0 and lse = -inf."""

import math

import numpy as np
import pytest

from oracle import dense


def close(a, b, tol=1e-13):
    """Equal up to FP64 rounding order (a BLAS product over a different
    number of rows may sum in another order); -inf must match exactly."""
    a, b = np.asarray(a), np.asarray(b)
    fa, fb = np.isfinite(a), np.isfinite(b)
    return np.array_equal(fa, fb) and np.array_equal(a[~fa], b[~fb]) and (
        not fa.any() or float(np.max(np.abs(a[fa] - b[fb]))) <= tol)


def rnd(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def window_count(c, Lk, wl, wr, causal):
    hi = Lk - 1
    if causal:
        hi = min(hi, c)
    if wr >= 0:
        hi = min(hi, c + wr)
    lo = 0 if wl < 0 else max(0, c - wl)
    return max(0, hi - lo + 1), lo, hi


@pytest.mark.parametrize("Lq,Lk", [(1, 300), (7, 300), (128, 300), (300, 300)])
def test_decode_rows_equal_the_suffix_of_the_square_problem(Lq, Lk):
    """Bottom-right causal attention of Lq queries equals the last Lq rows of
    the square causal problem over the same keys (a decode step over a
    cache)."""
    q, k, v = rnd((1, 2, Lk, 16), 1), rnd((1, 1, Lk, 16), 2), rnd((1, 1, Lk, 16), 3)
    o_sq, l_sq = dense.attention_dense(q, k, v, causal=True, scale=0.25)
    o, l = dense.attention_dense(q[:, :, Lk - Lq:], k, v, causal=True, scale=0.25)
    assert close(o, o_sq[:, :, Lk - Lq:]) and close(l, l_sq[:, :, Lk - Lq:])


@pytest.mark.parametrize("Lq,Lk", [(200, 70), (129, 1), (5, 3)])
def test_more_queries_than_keys_gives_empty_leading_rows(Lq, Lk):
    q, k, v = rnd((1, 1, Lq, 8), 4), rnd((1, 1, Lk, 8), 5), rnd((1, 1, Lk, 8), 6)
    o, l = dense.attention_dense(q, k, v, causal=True, scale=0.3)
    e = Lq - Lk
    assert np.all(o[:, :, :e] == 0.0) and np.all(l[:, :, :e] == -np.inf)
    o_sq, l_sq = dense.attention_dense(q[:, :, e:], k, v, causal=True, scale=0.3)
    assert close(o[:, :, e:], o_sq) and close(l[:, :, e:], l_sq)


@pytest.mark.parametrize("wl,wr,causal", [(0, 0, True), (5, 0, True), (40, -1, True), (3, 7, False),
                                          (-1, 10, False), (100, 100, False)])
@pytest.mark.parametrize("Lq,Lk", [(90, 90), (30, 90), (90, 30)])
def test_window_row_equals_attention_over_the_key_slice(wl, wr, causal, Lq, Lk):
    q, k, v = rnd((Lq, 12), 7), rnd((Lk, 12), 8), rnd((Lk, 12), 9)
    o, l = dense.attention_rows(q, k, v, np.arange(Lq), causal=causal, scale=0.2, window_left=wl, window_right=wr)
    for i in range(Lq):
        n, lo, hi = window_count(i + Lk - Lq, Lk, wl, wr, causal)
        if n == 0:
            assert np.all(o[i] == 0) and l[i] == -np.inf
            continue
        o_s, l_s = dense.attention_rows(q[i:i + 1], k[lo:hi + 1], v[lo:hi + 1], [0], causal=False, scale=0.2)
        assert np.max(np.abs(o[i] - o_s[0])) < 1e-13 and abs(l[i] - l_s[0]) < 1e-13


@pytest.mark.parametrize("wl,wr,causal", [(3, 2, False), (10, 0, True), (-1, 0, True)])
def test_window_q_zero_closed_form(wl, wr, causal):
    """Q = 0: O_i is the mean of the values in the window, lse_i = ln(count)."""
    Lq, Lk = 20, 50
    k, v = rnd((Lk, 4), 10), rnd((Lk, 4), 11)
    o, l = dense.attention_rows(np.zeros((Lq, 4)), k, v, np.arange(Lq), causal=causal, scale=1.0,
                                window_left=wl, window_right=wr)
    for i in range(Lq):
        n, lo, hi = window_count(i + Lk - Lq, Lk, wl, wr, causal)
        assert np.max(np.abs(o[i] - v[lo:hi + 1].mean(axis=0))) < 1e-14
        assert abs(l[i] - math.log(n)) < 1e-14


def test_varlen_separate_key_offsets_match_per_sequence_dense():
    lq, lk = [3, 0, 40, 17], [10, 5, 40, 0]
    cuq, cuk = np.concatenate([[0], np.cumsum(lq)]), np.concatenate([[0], np.cumsum(lk)])
    q, k, v = rnd((cuq[-1], 4, 8), 12), rnd((cuk[-1], 2, 8), 13), rnd((cuk[-1], 2, 8), 14)
    o, l = dense.attention_varlen(q, k, v, cuq, cu_seqlens_k=cuk, causal=True, scale=0.35, window_left=6)
    for s in range(len(lq)):
        if lq[s] == 0:
            continue
        qs = q[cuq[s]:cuq[s + 1]].transpose(1, 0, 2)[None]
        ks = k[cuk[s]:cuk[s + 1]].transpose(1, 0, 2)[None]
        vs = v[cuk[s]:cuk[s + 1]].transpose(1, 0, 2)[None]
        o_d, l_d = dense.attention_dense(qs, ks, vs, causal=True, scale=0.35, window_left=6)
        assert close(o[cuq[s]:cuq[s + 1]], o_d[0].transpose(1, 0, 2))
        assert close(l[:, cuq[s]:cuq[s + 1]], l_d[0])
    assert np.all(o[cuq[3]:] == 0) and np.all(l[:, cuq[3]:] == -np.inf)  # sequence with no keys


def test_mutation_top_left_alignment_is_caught(monkeypatch):
    orig = dense.eligible_keys
    monkeypatch.setattr(dense, "eligible_keys",
                        lambda pos, L, causal, Lq=None, wl=-1, wr=-1, g=0: orig(pos, L, causal, L, wl, wr, g))
    with pytest.raises(AssertionError):
        test_decode_rows_equal_the_suffix_of_the_square_problem(7, 300)
