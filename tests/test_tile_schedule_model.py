"""CPU check of the forward kernel's tile schedule (no GPU).

A Python statement of the integer arithmetic in attn_fwd_kernel.cuh that
decides which key tiles a CTA streams and which keys each query row keeps:
the per-row key ranges (row_key_range), the per-sub-tile tile ranges
(sub_tile_key_tiles: the first and last rows' ranges bound every row's), the
CTA's streamed tile sequence and each sub-tile's reads of it, the global-token
build's two phases (global keys' tiles, then window tiles), and each row's two
mask limits moving down one 128-key tile per step.  It is checked against the
oracle's eligibility: every eligible (row, key) pair is read exactly once and
no other key is read.  This guards the schedule's design; the GPU parity
tests check the kernel itself."""

import numpy as np
import pytest

from oracle import dense

UNB = (1 << 30) - 1
BN = BM = 128


def wl_of(wl):
    return UNB if wl < 0 or wl > UNB else wl


def wr_of(wr, causal):
    return 0 if causal else (UNB if wr < 0 or wr > UNB else wr)


def row_key_range(c, Lk, wl, wr, G, wrc, part):
    lo, hi = max(0, c - wl), min(Lk - 1, c + wr)
    if G > 0:
        h = min(Lk - 1, c + wrc)
        if part == 1:
            lo, hi = 0, min(G - 1, h)
        elif c < G:
            lo, hi = G, h
        else:
            lo = max(lo, G)
    return lo, hi


def sub_tile_key_tiles(r0, Lq, Lk, delta, wl, wr, G, wrc, part):
    if r0 >= Lq:
        return 0, 0
    cf, cl = r0 + delta, min(r0 + BM - 1, Lq - 1) + delta
    a = row_key_range(cf, Lk, wl, wr, G, wrc, part)
    b = row_key_range(cl, Lk, wl, wr, G, wrc, part)
    lo, hi = min(a[0], b[0]), max(a[1], b[1])
    return (0, 0) if hi < lo else (lo // BN, hi // BN + 1)


def reads_per_row(Lq, Lk, causal, wl_in, wr_in, G, nsub):
    """[Lq, Lk] count of how many times the schedule lets each row read each key."""
    wl, wr, wrc = wl_of(wl_in), wr_of(wr_in, causal), 0 if causal else UNB
    got = np.zeros((Lq, Lk), dtype=np.int64)
    delta = Lk - Lq
    for blk in range((Lq + nsub * BM - 1) // (nsub * BM)):
        row0 = blk * nsub * BM
        rows = [row0 + s * BM for s in range(nsub)]
        if G > 0:   # the global-token build: two phases per sub-tile
            g = [sub_tile_key_tiles(r, Lq, Lk, delta, wl, wr, G, wrc, 1) for r in rows]
            w = [sub_tile_key_tiles(r, Lq, Lk, delta, wl, wr, G, wrc, 0) for r in rows]
            assert all(x[0] == 0 for x in g)
            ga = [x[1] for x in g]
            ng = max(ga)
            act = [x[1] > x[0] for x in w]
            wt0 = min(x[0] for x, a in zip(w, act) if a) if any(act) else 0
            n_tot = ng + ((max(x[1] for x, a in zip(w, act) if a) - wt0) if any(act) else 0)
            f = [ng + w[s][0] - wt0 if act[s] else ng for s in range(nsub)]
            n = [ga[s] + (w[s][1] - w[s][0] if act[s] else 0) for s in range(nsub)]

            def key_tile(j):
                return j if j < ng else wt0 + (j - ng)

            def reads(s, j):
                return j < ga[s] if j < ng else 0 <= j - f[s] < n[s] - ga[s]
        else:       # one contiguous tile range per sub-tile
            r_ = [sub_tile_key_tiles(r, Lq, Lk, delta, wl, wr, 0, wrc, 0) for r in rows]
            act = [x[1] > x[0] for x in r_]
            kt0 = min(x[0] for x, a in zip(r_, act) if a) if any(act) else 0
            n_tot = (max(x[1] for x, a in zip(r_, act) if a) - kt0) if any(act) else 0
            f = [x[0] - kt0 for x in r_]
            n = [x[1] - x[0] if a else 0 for x, a in zip(r_, act)]
            ga = [0] * nsub

            def key_tile(j):
                return kt0 + j

            def reads(s, j):
                return 0 <= j - f[s] < n[s]
        for s in range(nsub):
            own = [j for j in range(n_tot) if reads(s, j)]
            assert len(own) == n[s]
            for t in range(BM):
                r = rows[s] + t
                if r >= Lq:
                    continue
                c = r + delta
                kw = row_key_range(c, Lk, wl, wr, G, wrc, 0)
                first_w = key_tile(own[ga[s]]) * BN if n[s] > ga[s] else 0
                win = (kw[1] - first_w, kw[0] - first_w)
                if ga[s] > 0:
                    kg = row_key_range(c, Lk, wl, wr, G, wrc, 1)
                    hi, lo = kg[1], kg[0]
                else:
                    hi, lo = win
                for li, j in enumerate(own):
                    kb = key_tile(j) * BN
                    for i in range(max(0, lo), min(BN - 1, hi) + 1):
                        if kb + i < Lk:
                            got[r, kb + i] += 1
                    hi, lo = hi - BN, lo - BN
                    if li + 1 == ga[s]:
                        hi, lo = win
    return got


CASES = [(Lq, Lk) for Lq in (1, 129, 300) for Lk in (3, 128, 300, 700)]


@pytest.mark.parametrize("Lq,Lk", CASES)
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("wl,wr,G", [(-1, -1, 0), (5, -1, 0), (200, 0, 0), (130, 130, 0), (-1, 3, 0),
                                     (16, 0, 1), (64, -1, 130), (3, 2, 7), (0, 0, 400)])
def test_schedule_reads_every_eligible_key_exactly_once(Lq, Lk, causal, wl, wr, G):
    want = dense.eligible_keys(np.arange(Lq), Lk, causal, Lq, wl, wr, G).astype(np.int64)
    for nsub in (1, 2):
        got = reads_per_row(Lq, Lk, causal, wl, wr, G, nsub)
        assert np.array_equal(got, want), (Lq, Lk, causal, wl, wr, G, nsub)
