"""Pins for the oracle's global tokens (CPU only).

Reading fixed here ("Attention algorithms and data movement", lesson 07,
global-token unions): the first G positions are global.  Every row may also
read the global keys j < G, and a global row (key position c < G) may read
every key; both obey the causal mask and ignore the window.  A key that is
both global and inside the window is one connection, not two.

The pins derive the eligible set a second way, by interval arithmetic:
E = C for a global row, else (W ∩ C) ∪ ([0, G-1] ∩ C), counted by
inclusion-exclusion and, for the outputs, as two explicit key slices fed to
the unmasked definition."""

import math

import numpy as np
import pytest

from oracle import dense


def rnd(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def intervals(c, Lk, G, wl, wr, causal):
    """The eligible keys of the row at key position c as at most two disjoint
    inclusive intervals, and their count by inclusion-exclusion."""
    hc = min(Lk - 1, c) if causal else Lk - 1          # the causal set C = [0, hc]
    if hc < 0:
        return [], 0
    if c < G:                                           # a global row reads all of C
        return [(0, hc)], hc + 1
    wlo = 0 if wl < 0 else max(0, c - wl)
    whi = Lk - 1 if wr < 0 else min(Lk - 1, c + wr)
    whi = min(whi, hc)                                  # W ∩ C
    bhi = min(G - 1, hc)                                # [0, G-1] ∩ C
    n_w = max(0, whi - wlo + 1)
    n_b = max(0, bhi + 1)
    n_both = max(0, min(whi, bhi) - wlo + 1)            # W ∩ B: B starts at 0 <= wlo
    count = n_w + n_b - n_both
    parts = []
    if n_b:
        parts.append((0, bhi))
    lo2 = max(wlo, bhi + 1)                             # the window keys past the global ones
    if whi >= lo2:
        parts.append((lo2, whi))
    return parts, count


CASES = [  # (Lq, Lk, G, wl, wr, causal)
    (60, 60, 5, 8, 0, True),
    (60, 60, 5, 8, -1, True),      # causal, left window only (the right bound is the diagonal)
    (60, 60, 16, 3, 0, True),      # window inside the global prefix for early rows
    (60, 60, 7, 4, 6, False),      # two-sided window, non-causal
    (60, 60, 1, 0, 0, False),
    (30, 80, 9, 10, 0, True),      # fewer queries than keys (decode-like chunk)
    (80, 30, 9, 5, 0, True),       # more queries than keys: empty leading rows
    (50, 50, 50, 2, 0, True),      # every position global
    (50, 50, 70, 2, 3, False),     # G beyond the sequence
    (40, 40, 0, 5, 0, True),       # no global token
]


@pytest.mark.parametrize("Lq,Lk,G,wl,wr,causal", CASES)
def test_eligible_counts_by_inclusion_exclusion(Lq, Lk, G, wl, wr, causal):
    e = dense.eligible_keys(np.arange(Lq), Lk, causal, Lq, wl, wr, G)
    for i in range(Lq):
        parts, count = intervals(i + Lk - Lq, Lk, G, wl, wr, causal)
        assert int(e[i].sum()) == count
        assert count == sum(hi - lo + 1 for lo, hi in parts)  # the slices are disjoint
        want = np.zeros(Lk, dtype=bool)
        for lo, hi in parts:
            want[lo:hi + 1] = True
        assert np.array_equal(e[i], want)


def test_total_connections_causal_window_closed_form():
    """Causal square, left window w (right bound the diagonal), G global
    tokens: a row c < G reads c + 1 keys; a row c >= G reads its window
    [start, c] with start = max(0, c - w) (min(c, w) + 1 keys) plus the global
    keys below the window's start, min(G, start) of them.  Summed in closed
    form over the three row ranges."""
    for N, w, G in ((200, 20, 8), (200, 5, 30), (64, 63, 10), (100, 0, 1)):
        # rows c < G: sum of c + 1
        t1 = G * (G + 1) // 2
        # rows G <= c: window keys min(c, w) + 1
        t2 = sum(min(c, w) + 1 for c in range(G, N))
        # global keys below start = c - w (only rows with c > w have start > 0)
        t3 = sum(min(G, c - w) for c in range(max(G, w + 1), N))
        e = dense.eligible_keys(np.arange(N), N, True, N, w, 0, G)
        assert int(e.sum()) == t1 + t2 + t3


@pytest.mark.parametrize("Lq,Lk,G,wl,wr,causal", CASES)
def test_rows_equal_unmasked_attention_over_the_key_slices(Lq, Lk, G, wl, wr, causal):
    q, k, v = rnd((Lq, 12), 1), rnd((Lk, 12), 2), rnd((Lk, 12), 3)
    o, l = dense.attention_rows(q, k, v, np.arange(Lq), causal=causal, scale=0.3, window_left=wl, window_right=wr,
                                num_global=G)
    for i in range(Lq):
        parts, count = intervals(i + Lk - Lq, Lk, G, wl, wr, causal)
        if count == 0:
            assert np.all(o[i] == 0) and l[i] == -np.inf
            continue
        idx = np.concatenate([np.arange(lo, hi + 1) for lo, hi in parts])
        o_s, l_s = dense.attention_rows(q[i:i + 1], k[idx], v[idx], [0], causal=False, scale=0.3)
        assert np.max(np.abs(o[i] - o_s[0])) < 1e-13 and abs(l[i] - l_s[0]) < 1e-13


@pytest.mark.parametrize("G,wl,wr,causal", [(6, 4, 0, True), (10, 2, 3, False), (3, 0, 0, True)])
def test_q_zero_closed_form(G, wl, wr, causal):
    """Q = 0: every eligible key has the same score, so O_i is the mean of the
    values over the two key intervals and lse_i = ln(count)."""
    Lq = Lk = 40
    k, v = rnd((Lk, 4), 4), rnd((Lk, 4), 5)
    o, l = dense.attention_rows(np.zeros((Lq, 4)), k, v, np.arange(Lq), causal=causal, scale=1.0, window_left=wl,
                                window_right=wr, num_global=G)
    for i in range(Lq):
        parts, count = intervals(i, Lk, G, wl, wr, causal)
        total = sum(v[lo:hi + 1].sum(axis=0) for lo, hi in parts)
        assert np.max(np.abs(o[i] - total / count)) < 1e-14
        assert abs(l[i] - math.log(count)) < 1e-14


def test_global_rows_equal_plain_causal_rows_and_large_g_is_causal():
    q, k, v = rnd((1, 2, 70, 8), 6), rnd((1, 1, 70, 8), 7), rnd((1, 1, 70, 8), 8)
    G = 12
    o, l = dense.attention_dense(q, k, v, causal=True, scale=0.4, window_left=5, num_global=G)
    o_c, l_c = dense.attention_dense(q, k, v, causal=True, scale=0.4)
    assert np.max(np.abs(o[:, :, :G] - o_c[:, :, :G])) < 1e-13
    assert np.max(np.abs(l[:, :, :G] - l_c[:, :, :G])) < 1e-13
    o_all, l_all = dense.attention_dense(q, k, v, causal=True, scale=0.4, window_left=5, num_global=70)
    assert np.max(np.abs(o_all - o_c)) < 1e-13 and np.max(np.abs(l_all - l_c)) < 1e-13
    # non-global rows differ from plain causal (the window drops keys)
    assert np.max(np.abs(o[:, :, G + 10:] - o_c[:, :, G + 10:])) > 1e-3
    # without the causal mask a global row reads every key, the future ones too
    o_n, l_n = dense.attention_dense(q, k, v, causal=False, scale=0.4, window_left=5, window_right=2, num_global=G)
    o_f, l_f = dense.attention_dense(q, k, v, causal=False, scale=0.4)
    assert np.max(np.abs(o_n[:, :, :G] - o_f[:, :, :G])) < 1e-13
    assert np.max(np.abs(l_n[:, :, :G] - l_f[:, :, :G])) < 1e-13


def test_varlen_global_tokens_are_per_sequence():
    lq = [25, 0, 40, 9]
    cu = np.concatenate([[0], np.cumsum(lq)])
    q, k, v = rnd((cu[-1], 4, 8), 9), rnd((cu[-1], 2, 8), 10), rnd((cu[-1], 2, 8), 11)
    o, l = dense.attention_varlen(q, k, v, cu, causal=True, scale=0.35, window_left=4, num_global=3)
    for s in range(len(lq)):
        if lq[s] == 0:
            continue
        qs = q[cu[s]:cu[s + 1]].transpose(1, 0, 2)[None]
        ks = k[cu[s]:cu[s + 1]].transpose(1, 0, 2)[None]
        vs = v[cu[s]:cu[s + 1]].transpose(1, 0, 2)[None]
        o_d, l_d = dense.attention_dense(qs, ks, vs, causal=True, scale=0.35, window_left=4, num_global=3)
        assert np.max(np.abs(o[cu[s]:cu[s + 1]] - o_d[0].transpose(1, 0, 2))) < 1e-13
        assert np.max(np.abs(l[:, cu[s]:cu[s + 1]] - l_d[0])) < 1e-13


# ---------------------------------------------------------------- planted mistakes

def _patch(monkeypatch, fn):
    orig = dense.eligible_keys
    monkeypatch.setattr(dense, "eligible_keys",
                        lambda pos, L, causal, Lq=None, wl=-1, wr=-1, g=0: fn(orig, pos, L, causal, Lq, wl, wr, g))


def test_mutation_global_rows_keep_their_window_is_caught(monkeypatch):
    """Forgetting that a global row reads every key (visible without the
    causal mask: under it a global row's keys are all global keys)."""
    def bad(orig, pos, L, causal, Lq, wl, wr, g):
        Lq = L if Lq is None else Lq
        c = np.asarray(pos)[:, None] + (L - Lq)
        j = np.arange(L)[None, :]
        return orig(pos, L, causal, Lq, wl, wr, 0) | ((j < g) & ((j <= c) if causal else True))
    _patch(monkeypatch, bad)
    with pytest.raises(AssertionError):
        test_global_rows_equal_plain_causal_rows_and_large_g_is_causal()


def test_mutation_global_keys_past_the_diagonal_is_caught(monkeypatch):
    """Letting every row read all global keys even past its causal limit."""
    def bad(orig, pos, L, causal, Lq, wl, wr, g):
        j = np.arange(L)[None, :]
        return orig(pos, L, causal, Lq, wl, wr, g) | (j < g)
    _patch(monkeypatch, bad)
    with pytest.raises(AssertionError):
        test_eligible_counts_by_inclusion_exclusion(60, 60, 16, 3, 0, True)


def test_mutation_double_counted_overlap_is_caught(monkeypatch):
    """Counting a global key inside the window twice (weight 2 in the sum)
    changes the softmax: the Q = 0 closed form catches it."""
    orig_rows = dense._rows_attention

    def bad_rows(q_rows, pos_rows, k, v, causal, scale, Lq=None, wl=-1, wr=-1, g=0):
        o, l = orig_rows(q_rows, pos_rows, k, v, causal, scale, Lq, wl, wr, g)
        if g <= 0:
            return o, l
        # duplicate the keys that are both global and in the window
        L = k.shape[0]
        w = dense.eligible_keys(pos_rows, L, causal, Lq, wl, wr, 0)
        j = np.arange(L)[None, :]
        dup = w & (j < g)
        for r in range(len(pos_rows)):
            if dup[r].any():
                kk = np.concatenate([k, k[dup[r]]])
                vv = np.concatenate([v, v[dup[r]]])
                e = np.concatenate([dense.eligible_keys(pos_rows[r:r + 1], L, causal, Lq, wl, wr, g)[0],
                                    np.ones(int(dup[r].sum()), dtype=bool)])
                s = scale * (q_rows[r] @ kk.T)
                p = np.where(e, np.exp(s - s[e].max()), 0.0)
                o[r] = p @ vv / p.sum()
                l[r] = s[e].max() + math.log(p.sum())
        return o, l
    monkeypatch.setattr(dense, "_rows_attention", bad_rows)
    with pytest.raises(AssertionError):
        test_q_zero_closed_form(6, 4, 0, True)
