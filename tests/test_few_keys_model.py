"""CPU check of the rule that decides which calls launch the forward kernel's
split-P build (no GPU).

A Python statement of the launcher's keys_of_row and has_few_key_rows
(attn_api.cu): the number of keys a query row reads, and whether any row of a
sequence reads at least one and fewer than 128 keys, found by evaluating the
count only at the first and last rows and next to the breakpoints of its
piecewise-linear form.  Checked here: keys_of_row equals the oracle's
eligibility count row by row (windows, unequal lengths, global tokens), and
the breakpoint search agrees with a brute-force scan of every row."""

import itertools

import numpy as np
import pytest

from oracle import dense

UNB = (1 << 30) - 1
FEW = 128


def keys_of_row(c, Lk, wl, wr, wrc, G):
    lo, hi = max(0, c - wl), min(Lk - 1, c + wr)
    if G <= 0:
        return max(0, hi - lo + 1)
    h = min(Lk - 1, c + wrc)
    glob = max(0, min(G - 1, h) + 1)
    rest = max(0, h - G + 1) if c < G else max(0, hi - max(lo, G) + 1)
    return glob + rest


def has_few_key_rows(Lq, Lk, wl, wr, wrc, G):
    if Lq <= 0 or Lk <= 0:
        return False
    delta = Lk - Lq
    cs = [0, wl, Lk - 1 - wr, Lk - 1 + wl, -wr, G - 1, G, G + wl, Lk - 1 - wrc, Lk - 1, G - wr]
    rows = [0, Lq - 1] + [c + d - delta for c in cs for d in (-1, 0, 1)]
    for r in rows:
        if 0 <= r < Lq:
            n = keys_of_row(r + delta, Lk, wl, wr, wrc, G)
            if 0 < n < FEW:
                return True
    return False


def eff(causal, wl, wr):
    wl_e = UNB if wl < 0 else wl
    wr_e = 0 if causal else (UNB if wr < 0 else wr)
    return wl_e, wr_e, (0 if causal else UNB)


CASES = list(itertools.product([1, 5, 127, 128, 129, 300, 700], [1, 64, 128, 129, 300, 1000],
                               [(True, -1, -1), (False, -1, -1), (True, 40, -1), (True, 200, -1), (False, 60, 60),
                                (False, -1, 10), (True, 126, -1), (True, 127, -1)],
                               [0, 1, 20, 150]))


@pytest.mark.parametrize("Lq,Lk,win,G", CASES[::7])
def test_keys_of_row_matches_the_oracle_eligibility(Lq, Lk, win, G):
    causal, wl, wr = win
    wl_e, wr_e, wrc = eff(causal, wl, wr)
    elig = dense.eligible_keys(np.arange(Lq), Lk, causal, Lq, wl, wr, G)
    want = elig.sum(axis=1)
    got = [keys_of_row(r + Lk - Lq, Lk, wl_e, wr_e, wrc, G) for r in range(Lq)]
    assert list(want) == got


@pytest.mark.parametrize("Lq,Lk,win,G", CASES)
def test_breakpoint_search_equals_a_scan_of_every_row(Lq, Lk, win, G):
    causal, wl, wr = win
    wl_e, wr_e, wrc = eff(causal, wl, wr)
    counts = [keys_of_row(r + Lk - Lq, Lk, wl_e, wr_e, wrc, G) for r in range(Lq)]
    brute = any(0 < n < FEW for n in counts)
    assert has_few_key_rows(Lq, Lk, wl_e, wr_e, wrc, G) == brute


def test_the_benchmarked_shapes():
    # causal self-attention always starts with a one-key row; a decode step
    # over a long history and a chunk of new rows over a long cache never
    # read fewer than 128 keys
    assert has_few_key_rows(4096, 4096, *eff(True, -1, -1), 0)
    assert not has_few_key_rows(1, 32768, *eff(True, -1, -1), 0)
    assert not has_few_key_rows(2048, 16384, *eff(True, -1, -1), 0)
    assert has_few_key_rows(16384, 16384, *eff(True, 4095, -1), 0)
    assert not has_few_key_rows(512, 512, *eff(False, -1, -1), 0)
