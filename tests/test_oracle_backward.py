"""Pins for the backward oracle (CPU only): PyTorch float64 autograd through
scaled_dot_product_attention (a library routine), central finite differences
of sum(dO * O) through the forward oracle, the key-shift invariant, a closed
form, empty rows, and planted mistakes that a pin must catch.

Masks handed to PyTorch are built here by brute force from the reading
(query row i of Lq sits at key position i + Lk - Lq; causal keeps keys at or
before it; a window keeps c - left <= j <= c + right), not by the oracle."""

import numpy as np
import pytest
import torch

from oracle import backward, dense


def rnd(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def brute_mask(Lq, Lk, causal, wl=-1, wr=-1):
    m = np.zeros((Lq, Lk), dtype=bool)
    for i in range(Lq):
        c = i + Lk - Lq
        for j in range(Lk):
            ok = True
            if causal and j > c:
                ok = False
            if wr >= 0 and j > c + wr:
                ok = False
            if wl >= 0 and j < c - wl:
                ok = False
            m[i, j] = ok
    return m


def torch_grads(q, k, v, do, mask, scale):
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=torch.tensor(mask), scale=scale,
                                                         enable_gqa=q.shape[1] != k.shape[1])
    o.backward(torch.tensor(do, dtype=torch.float64))
    return tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy()


CASES = [  # (B, Hq, Hkv, Nq, Nk, causal, wl, wr)
    (1, 1, 1, 17, 17, True, -1, -1),
    (2, 4, 2, 23, 23, False, -1, -1),
    (1, 4, 1, 9, 30, True, -1, -1),       # decode-like chunk over a longer cache
    (2, 2, 2, 20, 20, True, 5, -1),       # causal window
    (1, 2, 1, 25, 25, False, 3, 4),       # two-sided window
]


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,causal,wl,wr", CASES)
def test_backward_matches_torch_autograd(B, Hq, Hkv, Nq, Nk, causal, wl, wr):
    D = 8
    q, do = rnd((B, Hq, Nq, D), 1), rnd((B, Hq, Nq, D), 2)
    k, v = rnd((B, Hkv, Nk, D), 3), rnd((B, Hkv, Nk, D), 4)
    scale = 0.4
    dq, dk, dv = backward.attention_backward_dense(q, k, v, do, causal=causal, scale=scale, window_left=wl,
                                                   window_right=wr)
    tq, tk, tv = torch_grads(q, k, v, do, brute_mask(Nq, Nk, causal, wl, wr), scale)
    for a, b in ((dq, tq), (dk, tk), (dv, tv)):
        assert np.max(np.abs(a - b)) < 1e-12


def test_backward_matches_central_finite_differences():
    B, H, N, D, scale = 1, 1, 5, 3, 0.7
    q, k, v, do = rnd((B, H, N, D), 5), rnd((B, H, N, D), 6), rnd((B, H, N, D), 7), rnd((B, H, N, D), 8)

    def loss(q_, k_, v_):
        o, _ = dense.attention_dense(q_, k_, v_, causal=True, scale=scale)
        return float(np.sum(o * do))

    grads = backward.attention_backward_dense(q, k, v, do, causal=True, scale=scale)
    eps = 1e-6
    for which, g in enumerate(grads):
        for idx in np.ndindex(q.shape):
            args = [q.copy(), k.copy(), v.copy()]
            args[which][idx] += eps
            up = loss(*args)
            args[which][idx] -= 2 * eps
            down = loss(*args)
            assert abs((up - down) / (2 * eps) - g[idx]) < 1e-7


@pytest.mark.parametrize("causal,wl", [(True, -1), (False, -1), (True, 4)])
def test_key_gradients_sum_to_zero(causal, wl):
    """Adding one vector to every key leaves each row's softmax unchanged, so
    the key gradients of every (batch, KV head) sum to zero."""
    q, do = rnd((2, 4, 30, 8), 9), rnd((2, 4, 30, 8), 10)
    k, v = rnd((2, 2, 30, 8), 11), rnd((2, 2, 30, 8), 12)
    _, dk, _ = backward.attention_backward_dense(q, k, v, do, causal=causal, scale=0.3, window_left=wl)
    assert np.max(np.abs(dk.sum(axis=2))) < 1e-12


def test_single_key_closed_form():
    """One key: every row's P is 1, so dV = sum of dO rows, dQ = dK = 0."""
    q, do = rnd((1, 2, 6, 4), 13), rnd((1, 2, 6, 4), 14)
    k, v = rnd((1, 1, 1, 4), 15), rnd((1, 1, 1, 4), 16)
    dq, dk, dv = backward.attention_backward_dense(q, k, v, do, causal=False, scale=0.5)
    assert np.max(np.abs(dq)) < 1e-15 and np.max(np.abs(dk)) < 1e-15
    assert np.max(np.abs(dv[0, 0, 0] - do[0].sum(axis=(0, 1)))) < 1e-13


def test_empty_rows_contribute_nothing():
    """Lq > Lk under the causal mask: the first Lq - Lk rows read no key;
    their dQ is 0 and the key gradients equal those of the remaining rows."""
    q, do = rnd((1, 1, 12, 4), 17), rnd((1, 1, 12, 4), 18)
    k, v = rnd((1, 1, 5, 4), 19), rnd((1, 1, 5, 4), 20)
    dq, dk, dv = backward.attention_backward_dense(q, k, v, do, causal=True, scale=0.6)
    assert np.all(dq[:, :, :7] == 0)
    dq2, dk2, dv2 = backward.attention_backward_dense(q[:, :, 7:], k, v, do[:, :, 7:], causal=True, scale=0.6)
    assert np.max(np.abs(dq[:, :, 7:] - dq2)) < 1e-13
    assert np.max(np.abs(dk - dk2)) < 1e-13 and np.max(np.abs(dv - dv2)) < 1e-13


@pytest.mark.parametrize("causal,wl", [(True, -1), (False, 6)])
def test_sampled_rows_equal_dense(causal, wl):
    q, do = rnd((1, 4, 40, 8), 21), rnd((1, 4, 40, 8), 22)
    k, v = rnd((1, 2, 50, 8), 23), rnd((1, 2, 50, 8), 24)
    dq, dk, dv = backward.attention_backward_dense(q, k, v, do, causal=causal, scale=0.3, window_left=wl)
    qr, kr = [0, 7, 39], [0, 11, 49]
    for hk in range(2):
        sq, sk, sv = backward.attention_backward_sampled(q[0, 2 * hk:2 * hk + 2], k[0, hk], v[0, hk],
                                                         do[0, 2 * hk:2 * hk + 2], qr, kr, causal=causal,
                                                         scale=0.3, group=2, window_left=wl)
        assert np.max(np.abs(sq - dq[0, 2 * hk:2 * hk + 2][:, qr])) < 1e-12
        assert np.max(np.abs(sk - dk[0, hk, kr])) < 1e-12 and np.max(np.abs(sv - dv[0, hk, kr])) < 1e-12
    mq, mk, mv = backward.backward_magnitudes(q, k, v, do, causal=causal, scale=0.3, window_left=wl)
    for hk in range(2):
        out = backward.attention_backward_sampled(q[0, 2 * hk:2 * hk + 2], k[0, hk], v[0, hk], do[0, 2 * hk:2 * hk + 2],
                                                  qr, kr, causal=causal, scale=0.3, group=2, window_left=wl,
                                                  magnitudes=True)
        assert np.max(np.abs(out[3] - mq[0, 2 * hk:2 * hk + 2][:, qr])) < 1e-12
        assert np.max(np.abs(out[4] - mk[0, hk, kr])) < 1e-12 and np.max(np.abs(out[5] - mv[0, hk, kr])) < 1e-12


# ---------------------------------------------------------------- planted mistakes

def _torch_error(monkeypatch_fn=None):
    q, do = rnd((1, 2, 12, 8), 25), rnd((1, 2, 12, 8), 26)
    k, v = rnd((1, 1, 12, 8), 27), rnd((1, 1, 12, 8), 28)
    dq, dk, dv = backward.attention_backward_dense(q, k, v, do, causal=True, scale=0.5)
    tq, tk, tv = torch_grads(q, k, v, do, brute_mask(12, 12, True), 0.5)
    return max(np.max(np.abs(dq - tq)), np.max(np.abs(dk - tk)), np.max(np.abs(dv - tv)))


def test_mutation_dropped_row_term_is_caught(monkeypatch):
    def bad(q, k, v, do, causal, scale, wl, wr):
        Nq = q.shape[0]
        p = backward._probabilities(q, np.arange(Nq), k, causal, scale, Nq, wl, wr)
        ds = p * (do @ v.T)  # missing the - Dr_i term
        return scale * (ds @ k), scale * (ds.T @ q), p.T @ do
    monkeypatch.setattr(backward, "_head_backward", bad)
    assert _torch_error() > 1e-3


def test_mutation_unscaled_key_gradient_is_caught(monkeypatch):
    orig = backward._head_backward

    def bad(*a):
        dq, dk, dv = orig(*a)
        return dq, dk / a[5], dv  # forgot the scale on dK
    monkeypatch.setattr(backward, "_head_backward", bad)
    assert _torch_error() > 1e-3


def test_mutation_untransposed_value_gradient_is_caught(monkeypatch):
    def bad(q, k, v, do, causal, scale, wl, wr):
        Nq = q.shape[0]
        p = backward._probabilities(q, np.arange(Nq), k, causal, scale, Nq, wl, wr)
        dp = do @ v.T
        ds = p * (dp - np.sum(p * dp, axis=1)[:, None])
        return scale * (ds @ k), scale * (ds.T @ q), p @ do  # P dO instead of P^T dO
    monkeypatch.setattr(backward, "_head_backward", bad)
    assert _torch_error() > 1e-3


def test_mutation_group_overwrite_is_caught(monkeypatch):
    """Keeping only the last query head's dK/dV for a KV head (no sum over
    the group) must fail the GQA autograd pin."""
    orig = backward.attention_backward_dense

    def bad(q, k, v, do, **kw):
        dq, dk, dv = orig(q, k, v, do, **kw)
        last = orig(q[:, 1:2], k, v, do[:, 1:2], **kw)
        return dq, last[1], last[2]
    monkeypatch.setattr(backward, "attention_backward_dense", bad)
    assert _torch_error() > 1e-3


def _bf16_round(x):
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = ((b + 0x7FFF + ((b >> 16) & 1)) & 0xFFFF0000).astype(np.uint32)
    return b.view(np.float32).astype(np.float64)


@pytest.mark.parametrize("kw", [dict(causal=True), dict(causal=False, window_left=5, window_right=2)])
def test_d_rounding_bounds_the_effect_of_a_16_bit_output(kw):
    """D taken as <dO, O> from O rounded to FP16 or BF16 moves dQ and dK by
    at most u E (backward_d_rounding); the bound is attained to within a
    small factor, so it is not vacuous.  The change is computed directly:
    dS moves by -P_ij (D~_i - D_i), dQ and dK by its products with K and Q."""
    q, do = rnd((1, 2, 30, 8), 51), rnd((1, 2, 30, 8), 52)
    k, v = rnd((1, 1, 40, 8), 53), rnd((1, 1, 40, 8), 54)
    eq, ek = backward.backward_d_rounding(q, k, v, do, scale=0.3, **kw)
    rows = np.arange(30)
    wl, wr = kw.get("window_left", -1), kw.get("window_right", -1)
    for rnd16, u in ((lambda x: x.astype(np.float16).astype(np.float64), 2.0 ** -11), (_bf16_round, 2.0 ** -8)):
        dk_move = np.zeros_like(k[0, 0])
        worst = 0.0
        for h in range(2):
            p = backward._probabilities(q[0, h], rows, k[0, 0], kw["causal"], 0.3, 30, wl, wr)
            o = p @ v[0, 0]
            delta = np.sum(do[0, h] * rnd16(o), axis=1) - np.sum(do[0, h] * o, axis=1)
            ds_move = -p * delta[:, None]
            dq_move = 0.3 * (ds_move @ k[0, 0])
            assert np.all(np.abs(dq_move) <= u * eq[0, h] + 1e-15)
            worst = max(worst, float(np.max(np.abs(dq_move) / (u * eq[0, h] + 1e-300))))
            dk_move += 0.3 * (ds_move.T @ q[0, h])
        assert np.all(np.abs(dk_move) <= u * ek[0, 0] + 1e-15)
        assert worst > 0.1  # measured 0.14-0.20 on these inputs


def test_magnitudes_bound_the_gradients():
    """Each magnitude is a sum of absolute values of the terms its gradient
    element sums, so it bounds the element (triangle inequality); with
    dO >= 0 the value-gradient terms are nonnegative and M_dV equals dV."""
    q, do = rnd((1, 4, 30, 8), 29), rnd((1, 4, 30, 8), 30)
    k, v = rnd((1, 2, 40, 8), 31), rnd((1, 2, 40, 8), 32)
    for kw in (dict(causal=True), dict(causal=False, window_left=5, window_right=2)):
        g = backward.attention_backward_dense(q, k, v, do, scale=0.3, **kw)
        m = backward.backward_magnitudes(q, k, v, do, scale=0.3, **kw)
        for gi, mi in zip(g, m):
            assert np.all(mi >= np.abs(gi) - 1e-12)
    dop = np.abs(do)
    _, _, dv = backward.attention_backward_dense(q, k, v, dop, causal=True, scale=0.3)
    _, _, mv = backward.backward_magnitudes(q, k, v, dop, causal=True, scale=0.3)
    assert np.max(np.abs(mv - dv)) < 1e-12
