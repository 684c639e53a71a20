"""Pins for the CPU FP64 oracle (CPU only; no CUDA import).

Each test checks the oracle against something other than itself: a
hand-worked example, closed forms, special cases, library routines (PyTorch's
CPU scaled_dot_product_attention in float64, SciPy's logsumexp), invariants the
pages name (partition / merge-order invariance, the explicit empty identity,
future-value perturbation, large logits) and metamorphic relations.  The
``test_mutation_*`` tests plant plausible mistakes in the oracle and check that
a pin catches each one.
"""

import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import dense, online_state
from oracle.online_state import empty_state, finalize, merge, state_of_block
from tests.conftest import read_golden

RNG = np.random.default_rng(20260923)


def rand_inputs(B, Hq, Hkv, N, D, seed=0, qscale=1.0):
    r = np.random.default_rng(seed)
    q = r.standard_normal((B, Hq, N, D)) * qscale
    k = r.standard_normal((B, Hkv, N, D))
    v = r.standard_normal((B, Hkv, N, D))
    return q, k, v


# ---------------------------------------------------------------- pin functions
# Each returns an error measure so that the mutation tests can show a planted
# mistake makes it large.

def worked_example_error(golden):
    """Two one-key tiles s = (1, 3), v = (10, 20): merged state and the dense
    oracle against the hand-derived closed form."""
    s = golden["scores"]
    vals = golden["values"]
    st = merge(state_of_block([s[0]], [[vals[0]]]), state_of_block([s[1]], [[vals[1]]]))
    o, lse = finalize(st)
    err = max(abs(o[0] - golden["O"][0]), abs(lse - golden["lse"][0]))
    # dense oracle: D = 1, q = 1, k = (1, 3), scale = 1, non-causal
    q = np.array([[[[1.0]]]])
    k = np.array([[[[s[0]], [s[1]]]]])
    v = np.array([[[[vals[0]], [vals[1]]]]])
    q2 = np.concatenate([q, q], axis=2)  # two identical queries so N matches keys
    o_d, lse_d = dense.attention_dense(q2, k, v, causal=False, scale=1.0)
    err = max(err, abs(o_d[0, 0, 0, 0] - golden["O"][0]), abs(lse_d[0, 0, 0] - golden["lse"][0]))
    return err


def sdpa_error(B, Hq, Hkv, N, D, causal, seed=0):
    """Oracle O against torch's CPU float64 scaled_dot_product_attention."""
    q, k, v = rand_inputs(B, Hq, Hkv, N, D, seed)
    scale = 1.0 / math.sqrt(D)
    o, _ = dense.attention_dense(q, k, v, causal=causal, scale=scale)
    tq, tk, tv = (torch.from_numpy(x) for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(
        tq, tk, tv, is_causal=causal, scale=scale, enable_gqa=(Hq != Hkv)).numpy()
    return float(np.max(np.abs(o - ref)))


def lse_scipy_error(N, D, causal, seed=0, qscale=1.0):
    """Oracle lse against SciPy's logsumexp of the masked scaled scores."""
    from scipy.special import logsumexp
    q, k, v = rand_inputs(1, 1, 1, N, D, seed, qscale)
    scale = 1.0 / math.sqrt(D)
    _, lse = dense.attention_dense(q, k, v, causal=causal, scale=scale)
    s = scale * (q[0, 0] @ k[0, 0].T)
    err = 0.0
    for i in range(N):
        row = s[i, : i + 1] if causal else s[i]
        err = max(err, abs(lse[0, 0, i] - logsumexp(row)))
    return err


def q_zero_error(N, D, causal, Hq=2, Hkv=1):
    """Q = 0: every eligible score is 0, so O_i is the mean of the eligible
    values and lse_i = ln |E(i)|."""
    _, k, v = rand_inputs(1, Hq, Hkv, N, D, seed=3)
    q = np.zeros((1, Hq, N, D))
    o, lse = dense.attention_dense(q, k, v, causal=causal, scale=0.125)
    err = 0.0
    for h in range(Hq):
        hk = h // (Hq // Hkv)
        for i in range(N):
            n_elig = i + 1 if causal else N
            mean = v[0, hk, :n_elig].mean(axis=0)
            err = max(err, np.max(np.abs(o[0, h, i] - mean)), abs(lse[0, h, i] - math.log(n_elig)))
    return err


def single_key_error(D=16, seed=5):
    """N = 1: O = v_0 and lse = scale * <q_0, k_0>."""
    q, k, v = rand_inputs(1, 1, 1, 1, D, seed)
    scale = 0.3
    err = 0.0
    for causal in (False, True):
        o, lse = dense.attention_dense(q, k, v, causal=causal, scale=scale)
        err = max(err, np.max(np.abs(o[0, 0, 0] - v[0, 0, 0])),
                  abs(lse[0, 0, 0] - scale * float(q[0, 0, 0] @ k[0, 0, 0])))
    return err


# ---------------------------------------------------------------- worked example

def test_worked_example_rescale(golden_dir):
    g = read_golden(os.path.join(golden_dir, "rescale_worked_example.txt"))
    assert abs(math.exp(g["scores"][0] - g["scores"][1]) - g["alpha"][0]) < 1e-16
    assert worked_example_error(g) < 1e-14


def test_mutation_no_numerator_rescale_fails(golden_dir, monkeypatch):
    """A merge that rescales only the denominator must fail the worked example."""
    g = read_golden(os.path.join(golden_dir, "rescale_worked_example.txt"))

    def bad_merge(a, b):
        if a.m == -math.inf:
            return b
        if b.m == -math.inf:
            return a
        m = max(a.m, b.m)
        return online_state.State(m, a.l * math.exp(a.m - m) + b.l * math.exp(b.m - m), a.acc + b.acc)

    st = bad_merge(state_of_block([g["scores"][0]], [[g["values"][0]]]),
                   state_of_block([g["scores"][1]], [[g["values"][1]]]))
    o, _ = finalize(st)
    assert abs(o[0] - g["O_without_numerator_rescale"][0]) < 1e-12
    assert abs(o[0] - g["O"][0]) > 1.0


# ---------------------------------------------------------------- empty identity

def test_empty_identity():
    d = 4
    e = empty_state(d)
    ee = merge(e, empty_state(d))
    assert ee.m == -math.inf and ee.l == 0.0 and np.all(ee.acc == 0.0)
    assert not np.any(np.isnan(ee.acc))
    x = state_of_block(RNG.standard_normal(5), RNG.standard_normal((5, d)))
    for y in (merge(e, x), merge(x, e)):
        assert y.m == x.m and y.l == x.l and np.array_equal(y.acc, x.acc)
    o, lse = finalize(e)
    assert lse == -math.inf and np.all(o == 0.0)
    assert state_of_block([], np.zeros((0, d))).m == -math.inf


def test_empty_row_contract_dense():
    """A row with no eligible key (non-causal with zero keys) gives O = 0, lse = -inf."""
    o, lse = dense._rows_attention(np.ones((3, 4)), np.arange(3), np.zeros((0, 4)), np.zeros((0, 4)), False, 1.0)
    assert np.all(o == 0) and np.all(lse == -np.inf)


# ---------------------------------------------------------------- partition / merge order

def _random_partition(n, rng, max_parts=6):
    cuts = sorted(rng.integers(0, n + 1, size=rng.integers(1, max_parts)))
    bounds = [0] + list(cuts) + [n]
    return [(bounds[i], bounds[i + 1]) for i in range(len(bounds) - 1)]  # may contain empty parts


def _tree_merge(states, rng):
    states = list(states)
    while len(states) > 1:
        i = int(rng.integers(0, len(states) - 1))
        states[i:i + 2] = [merge(states[i], states[i + 1])]
    return states[0]


@pytest.mark.parametrize("trial", range(8))
def test_partition_and_merge_order_invariance(trial):
    rng = np.random.default_rng(100 + trial)
    n, d = int(rng.integers(1, 40)), 5
    scores = rng.standard_normal(n) * (1 + 10 * (trial % 3))
    values = rng.standard_normal((n, d))
    o_ref, lse_ref = dense._rows_attention(scores[None, :], np.array([0]), np.eye(n), values, False, 1.0)
    parts = _random_partition(n, rng)
    states = [state_of_block(scores[a:b], values[a:b]) for a, b in parts]
    left = states[0]
    for st in states[1:]:
        left = merge(left, st)
    right = states[-1]
    for st in reversed(states[:-1]):
        right = merge(st, right)
    one_by_one = empty_state(d)
    for j in rng.permutation(n):  # one key at a time, random order
        one_by_one = merge(one_by_one, state_of_block(scores[j:j + 1], values[j:j + 1]))
    for st in (left, right, _tree_merge(states, rng), one_by_one):
        o, lse = finalize(st)
        assert np.max(np.abs(o - o_ref[0])) < 1e-12
        assert abs(lse - lse_ref[0]) < 1e-12


# ---------------------------------------------------------------- library cross-checks

@pytest.mark.parametrize("B,Hq,Hkv,N,D,causal", [
    (1, 1, 1, 129, 32, True), (1, 1, 1, 129, 32, False), (2, 3, 3, 70, 16, True),
    (2, 4, 1, 65, 8, True), (1, 8, 2, 33, 64, False), (1, 2, 2, 1, 4, True),
])
def test_matches_torch_sdpa_fp64(B, Hq, Hkv, N, D, causal):
    assert sdpa_error(B, Hq, Hkv, N, D, causal) < 1e-12


@pytest.mark.parametrize("causal,qscale", [(True, 1.0), (False, 1.0), (True, 30.0)])
def test_lse_matches_scipy_logsumexp(causal, qscale):
    assert lse_scipy_error(97, 16, causal, qscale=qscale) < 1e-10


# ---------------------------------------------------------------- closed forms / special cases

@pytest.mark.parametrize("causal", [True, False])
def test_q_zero_closed_form(causal):
    assert q_zero_error(37, 8, causal) < 1e-13


def test_single_key_closed_form():
    assert single_key_error() < 1e-14


def test_causal_row0_is_v0():
    q, k, v = rand_inputs(1, 1, 1, 50, 16, seed=9, qscale=5.0)
    o, _ = dense.attention_dense(q, k, v, causal=True, scale=0.25)
    assert np.array_equal(o[0, 0, 0], v[0, 0, 0])


def test_convex_combination():
    """Each output is a convex combination of the eligible value rows."""
    q, k, v = rand_inputs(1, 1, 1, 60, 8, seed=11, qscale=3.0)
    o, _ = dense.attention_dense(q, k, v, causal=True, scale=0.35)
    for i in range(60):
        lo, hi = v[0, 0, : i + 1].min(axis=0), v[0, 0, : i + 1].max(axis=0)
        assert np.all(o[0, 0, i] >= lo - 1e-12) and np.all(o[0, 0, i] <= hi + 1e-12)


# ---------------------------------------------------------------- invariants the pages name

def test_future_value_perturbation():
    """Changing keys/values after position i0 must not change causal rows <= i0."""
    q, k, v = rand_inputs(1, 2, 2, 90, 16, seed=4)
    o1, l1 = dense.attention_dense(q, k, v, causal=True, scale=0.25)
    i0 = 41
    k2, v2 = k.copy(), v.copy()
    k2[:, :, i0 + 1:] = RNG.standard_normal(k2[:, :, i0 + 1:].shape) * 50
    v2[:, :, i0 + 1:] = RNG.standard_normal(v2[:, :, i0 + 1:].shape) * 50
    o2, l2 = dense.attention_dense(q, k2, v2, causal=True, scale=0.25)
    assert np.array_equal(o1[:, :, : i0 + 1], o2[:, :, : i0 + 1])
    assert np.array_equal(l1[:, :, : i0 + 1], l2[:, :, : i0 + 1])
    assert not np.allclose(o1[:, :, i0 + 1:], o2[:, :, i0 + 1:])


def test_large_logits_no_overflow_and_near_argmax():
    """Q x30 drives logits past ln(FLT_MAX); the result stays finite and is
    within the exact softmax bound of the arg-max value row:
    |O_i - v_*| <= max_j |v_j - v_*| * sum_{j != *} exp(s_j - s_*)."""
    q, k, v = rand_inputs(1, 1, 1, 128, 64, seed=0, qscale=30.0)
    scale = 1 / 8
    o, lse = dense.attention_dense(q, k, v, causal=True, scale=scale)
    s = scale * (q[0, 0] @ k[0, 0].T)
    assert np.max(s) > 88.8 and np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    for i in range(128):
        row = s[i, : i + 1]
        j = int(np.argmax(row))
        tail = np.exp(row - row[j]).sum() - 1.0
        bound = np.max(np.abs(v[0, 0, : i + 1] - v[0, 0, j])) * tail
        assert np.max(np.abs(o[0, 0, i] - v[0, 0, j])) <= bound + 1e-12


def test_noncausal_key_permutation_invariance():
    q, k, v = rand_inputs(1, 1, 1, 64, 16, seed=6)
    perm = RNG.permutation(64)
    o1, l1 = dense.attention_dense(q, k, v, causal=False, scale=0.25)
    o2, l2 = dense.attention_dense(q, k[:, :, perm], v[:, :, perm], causal=False, scale=0.25)
    assert np.max(np.abs(o1 - o2)) < 1e-13 and np.max(np.abs(l1 - l2)) < 1e-13


def test_gqa_equals_repeated_kv():
    q, k, v = rand_inputs(2, 8, 2, 40, 16, seed=8)
    o1, l1 = dense.attention_dense(q, k, v, causal=True, scale=0.25)
    rep = lambda x: np.repeat(x, 4, axis=1)
    o2, l2 = dense.attention_dense(q, rep(k), rep(v), causal=True, scale=0.25)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_varlen_matches_sdpa_per_sequence():
    """Packed batch: each sequence against torch SDPA on its own slice, causal
    by logical position; lengths include 1 and a zero-length sequence."""
    lengths = [5, 1, 0, 37, 129]
    cu = np.concatenate([[0], np.cumsum(lengths)])
    T, Hq, Hkv, D = int(cu[-1]), 4, 2, 16
    r = np.random.default_rng(2)
    q, k, v = r.standard_normal((T, Hq, D)), r.standard_normal((T, Hkv, D)), r.standard_normal((T, Hkv, D))
    o, lse = dense.attention_varlen(q, k, v, cu, causal=True, scale=0.25)
    for s in range(len(lengths)):
        t0, t1 = int(cu[s]), int(cu[s + 1])
        if t1 == t0:
            continue
        tq = torch.from_numpy(q[t0:t1]).transpose(0, 1)[None]
        tk = torch.from_numpy(k[t0:t1]).transpose(0, 1)[None]
        tv = torch.from_numpy(v[t0:t1]).transpose(0, 1)[None]
        ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=True, scale=0.25,
                                                               enable_gqa=True)[0].transpose(0, 1).numpy()
        assert np.max(np.abs(o[t0:t1] - ref)) < 1e-12
        rows = np.arange(t1 - t0)
        o_r, l_r = dense.attention_varlen_rows(q, k, v, cu, s, 3, rows, causal=True, scale=0.25, group=2)
        assert np.array_equal(o_r, o[t0:t1, 3]) and np.array_equal(l_r, lse[3, t0:t1])


def test_rows_api_matches_dense():
    q, k, v = rand_inputs(1, 1, 1, 300, 32, seed=12)
    o, lse = dense.attention_dense(q, k, v, causal=True, scale=0.2)
    rows = [0, 1, 127, 128, 129, 299]
    o_r, l_r = dense.attention_rows(q[0, 0], k[0, 0], v[0, 0], rows, causal=True, scale=0.2)
    assert np.array_equal(o_r, o[0, 0, rows]) and np.array_equal(l_r, lse[0, 0, rows])


# ---------------------------------------------------------------- planted mistakes

def test_mutation_causal_mask_without_diagonal_is_caught(monkeypatch):
    monkeypatch.setattr(dense, "eligible_keys",
                        lambda pos, L, causal, *rest: (np.arange(L)[None, :] < np.asarray(pos)[:, None]) if causal
                        else np.ones((len(pos), L), dtype=bool))
    assert sdpa_error(1, 1, 1, 20, 8, True) > 1e-3
    assert not single_key_error() < 1e-3  # causal row 0 becomes empty (inf/nan error)
    assert not q_zero_error(10, 4, True) < 1e-3  # ln |E(i)| closed form violated


def test_mutation_wrong_gqa_mapping_is_caught(monkeypatch):
    monkeypatch.setattr(dense, "kv_head_of", lambda h, group: h % max(1, 8 // group) if group > 1 else h)
    assert sdpa_error(1, 8, 2, 16, 8, True) > 1e-3


def test_mutation_dropped_scale_is_caught(monkeypatch):
    orig = dense._rows_attention
    monkeypatch.setattr(dense, "_rows_attention",
                        lambda q, pos, k, v, causal, scale, *rest: orig(q, pos, k, v, causal, 1.0, *rest))
    assert single_key_error() > 1e-3
    assert sdpa_error(1, 1, 1, 16, 16, True) > 1e-3


def test_mutation_lse_log2_is_caught(monkeypatch):
    orig = dense._rows_attention

    def bad(q, pos, k, v, causal, scale, *rest):
        o, lse = orig(q, pos, k, v, causal, scale, *rest)
        return o, lse / math.log(2.0)
    monkeypatch.setattr(dense, "_rows_attention", bad)
    assert lse_scipy_error(33, 8, True) > 1e-3


def test_mutation_transposed_value_operand_is_caught(monkeypatch):
    orig = dense._rows_attention
    monkeypatch.setattr(dense, "_rows_attention",
                        lambda q, pos, k, v, causal, scale, *rest: orig(q, pos, k, k, causal, scale, *rest))
    assert sdpa_error(1, 2, 2, 24, 8, False) > 1e-3


def test_package_exports():
    for name in oracle.__all__:
        assert hasattr(oracle, name)
