"""Dense float64 gradients of softmax attention: the plain definition of what
the backward kernel computes.  TEST INFRASTRUCTURE ONLY (see the package
docstring).

Definition followed ("Attention algorithms and data movement", lesson 03,
recompute probabilities and differentiate the normalised row, saved
normalisation state; "Intermediate and advanced workshop validation",
"Correctness and review", which checks backward against FP64 autograd and a
central finite difference).  With the forward of ``dense`` (same masks, GQA
map and empty-row contract) and an upstream gradient dO of O:

  P_ij  = exp(s_ij - lse_i) on eligible keys, 0 elsewhere (0 for empty rows)
  dV_j  = sum_i P_ij dO_i
  dP_ij = <dO_i, v_j>
  Dr_i  = sum_j P_ij dP_ij            (= <dO_i, O_i>)
  dS_ij = P_ij (dP_ij - Dr_i)
  dQ_i  = scale * sum_j dS_ij k_j
  dK_j  = scale * sum_i dS_ij q_i

Under grouped-query attention a key/value head's dK and dV sum the
contributions of every query head that reads it.  The scores and lse are
recomputed here from the definition, not taken from the forward kernel.
"""

from __future__ import annotations

import numpy as np

from .dense import eligible_keys, kv_head_of

_ROW_CHUNK = 1024


def _probabilities(q_rows, pos_rows, k, causal, scale, Lq, window_left, window_right):
    """P [R, L] for query rows at positions pos_rows (of Lq), from the
    definition: a masked row-wise softmax of scale * q k^T."""
    L = k.shape[0]
    R = q_rows.shape[0]
    if R == 0 or L == 0:
        return np.zeros((R, L))
    s = scale * (q_rows @ k.T)
    eligible = eligible_keys(pos_rows, L, causal, Lq, window_left, window_right)
    nonempty = eligible.any(axis=1)
    s = np.where(eligible, s, -np.inf)
    m = np.where(nonempty, np.max(s, axis=1), 0.0)
    p = np.where(eligible, np.exp(s - m[:, None]), 0.0)
    l = p.sum(axis=1)
    p[nonempty] /= l[nonempty, None]
    return p


def _head_backward(q, k, v, do, causal, scale, window_left, window_right):
    """dq [Nq, D], dk [Nk, D], dv [Nk, D] of one (batch, query head)."""
    Nq, Nk = q.shape[0], k.shape[0]
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for r0 in range(0, Nq, _ROW_CHUNK):
        rows = np.arange(r0, min(Nq, r0 + _ROW_CHUNK))
        p = _probabilities(q[rows], rows, k, causal, scale, Nq, window_left, window_right)
        dv += p.T @ do[rows]
        dp = do[rows] @ v.T
        dr = np.sum(p * dp, axis=1)
        ds = p * (dp - dr[:, None])
        dq[rows] = scale * (ds @ k)
        dk += scale * (ds.T @ q[rows])
    return dq, dk, dv


def attention_backward_dense(q, k, v, do, *, causal, scale, window_left=-1, window_right=-1):
    """Gradients of sum(dO * O) for batched multi-head attention.

    q, do: [B, Hq, Nq, D]; k, v: [B, Hkv, Nk, D] with Hq % Hkv == 0.
    Returns dq [B, Hq, Nq, D], dk and dv [B, Hkv, Nk, D] (float64)."""
    q, k, v, do = (np.asarray(t, dtype=np.float64) for t in (q, k, v, do))
    B, Hq, Nq, D = q.shape
    Hkv = k.shape[1]
    if Hkv <= 0 or Hq % Hkv != 0:
        raise ValueError("Hq must be a multiple of Hkv")
    group = Hq // Hkv
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        for h in range(Hq):
            hk = kv_head_of(h, group)
            gq, gk, gv = _head_backward(q[b, h], k[b, hk], v[b, hk], do[b, h], causal, scale, window_left,
                                        window_right)
            dq[b, h] = gq
            dk[b, hk] += gk
            dv[b, hk] += gv
    return dq, dk, dv


def attention_backward_sampled(q, k, v, do, q_rows, k_rows, *, causal, scale, group=1, window_left=-1,
                               window_right=-1, magnitudes=False):
    """Selected gradient rows of one (batch, KV head) of a large problem.

    q, do: [G, Nq, D] for the ``group`` query heads that read the KV head;
    k, v: [Nk, D].  Returns dq [G, len(q_rows), D] and dk, dv
    [len(k_rows), D].  Every query row's probabilities are recomputed (in
    chunks), so dK and dV hold the full sums over queries and heads.  With
    ``magnitudes`` the same rows of backward_magnitudes follow."""
    q, k, v, do = (np.asarray(t, dtype=np.float64) for t in (q, k, v, do))
    G, Nq = q.shape[0], q.shape[1]
    if G != group:
        raise ValueError("q must hold the group's query heads")
    q_rows = np.asarray(q_rows, dtype=np.int64)
    k_rows = np.asarray(k_rows, dtype=np.int64)
    dq = np.zeros((G, len(q_rows), q.shape[2]))
    dk = np.zeros((len(k_rows), k.shape[1]))
    dv = np.zeros((len(k_rows), v.shape[1]))
    mq, mk, mv = np.zeros_like(dq), np.zeros_like(dk), np.zeros_like(dv)
    for g in range(G):
        for r0 in range(0, Nq, _ROW_CHUNK):
            rows = np.arange(r0, min(Nq, r0 + _ROW_CHUNK))
            p = _probabilities(q[g, rows], rows, k, causal, scale, Nq, window_left, window_right)
            dp = do[g, rows] @ v.T
            dr = np.sum(p * dp, axis=1)
            ds = p * (dp - dr[:, None])
            dv += p[:, k_rows].T @ do[g, rows]
            dk += scale * (ds[:, k_rows].T @ q[g, rows])
            sel = np.nonzero((q_rows >= r0) & (q_rows < r0 + len(rows)))[0]
            if len(sel):
                dq[g, sel] = scale * (ds[q_rows[sel] - r0] @ k)
            if magnitudes:
                adp = np.abs(dp)
                a = p * (adp + np.sum(p * adp, axis=1)[:, None])
                mv += p[:, k_rows].T @ np.abs(do[g, rows])
                mk += scale * (a[:, k_rows].T @ np.abs(q[g, rows]))
                if len(sel):
                    mq[g, sel] = scale * (a[q_rows[sel] - r0] @ np.abs(k))
    if magnitudes:
        return dq, dk, dv, mq, mk, mv
    return dq, dk, dv


def _d_magnitude(p, do_rows, v):
    """|D|_i = sum_d |dO_id| sum_l P_il |v_ld|: the absolute terms of
    D_i = <dO_i, O_i> with O_i = sum_l P_il v_l."""
    return np.sum(p * (np.abs(do_rows) @ np.abs(v).T), axis=1)


def backward_d_rounding(q, k, v, do, *, causal, scale, window_left=-1, window_right=-1):
    """How far an error of relative size 1 in each O element moves the
    gradients when D is taken as D_i = <dO_i, O_i> from the stored output
    (lesson 03's saved normalisation state), not a result the kernel computes.
    Rounding every O element to a 16-bit type (relative error at most u)
    moves D_i by at most u |D|_i, |D|_i = sum_d |dO_id| sum_l P_il |v_ld|;
    through dS_ij = P_ij (dP_ij - D_i) that moves
      dQ_i by at most u E_dQ_i,  E_dQ_i = scale * |D|_i sum_j P_ij |k_j|
      dK_j by at most u E_dK_j,  E_dK_j = scale * sum_i P_ij |D|_i |q_i|
    and dV not at all.  Returns (E_dQ, E_dK), shaped as dQ and dK (dK terms
    summed over the group)."""
    q, k, v, do = (np.asarray(t, dtype=np.float64) for t in (q, k, v, do))
    B, Hq, Nq, D = q.shape
    group = Hq // k.shape[1]
    eq = np.zeros_like(q)
    ek = np.zeros_like(k)
    for b in range(B):
        for h in range(Hq):
            hk = kv_head_of(h, group)
            for r0 in range(0, Nq, _ROW_CHUNK):
                rows = np.arange(r0, min(Nq, r0 + _ROW_CHUNK))
                p = _probabilities(q[b, h, rows], rows, k[b, hk], causal, scale, Nq, window_left, window_right)
                pd = p * _d_magnitude(p, do[b, h, rows], v[b, hk])[:, None]
                eq[b, h, rows] = scale * (pd @ np.abs(k[b, hk]))
                ek[b, hk] += scale * (pd.T @ np.abs(q[b, h, rows]))
    return eq, ek


def backward_magnitudes(q, k, v, do, *, causal, scale, window_left=-1, window_right=-1):
    """Sums of the absolute values of the terms of each gradient element, the
    scale against which rounding errors in a 16-bit implementation are
    measured (not a result the kernel computes):
      M_dV_j = sum_i P_ij |dO_i|
      A_ij   = P_ij (|dP_ij| + sum_l P_il |dP_il|)
      M_dQ_i = scale * sum_j A_ij |k_j|,   M_dK_j = scale * sum_i A_ij |q_i|
    Shapes as in attention_backward_dense (dK, dV terms summed over the group)."""
    q, k, v, do = (np.asarray(t, dtype=np.float64) for t in (q, k, v, do))
    B, Hq, Nq, D = q.shape
    group = Hq // k.shape[1]
    mq = np.zeros_like(q)
    mk = np.zeros_like(k)
    mv = np.zeros_like(v)
    for b in range(B):
        for h in range(Hq):
            hk = kv_head_of(h, group)
            for r0 in range(0, Nq, _ROW_CHUNK):
                rows = np.arange(r0, min(Nq, r0 + _ROW_CHUNK))
                p = _probabilities(q[b, h, rows], rows, k[b, hk], causal, scale, Nq, window_left, window_right)
                adp = np.abs(do[b, h, rows] @ v[b, hk].T)
                a = p * (adp + np.sum(p * adp, axis=1)[:, None])
                mv[b, hk] += p.T @ np.abs(do[b, h, rows])
                mq[b, h, rows] = scale * (a @ np.abs(k[b, hk]))
                mk[b, hk] += scale * (a.T @ np.abs(q[b, h, rows]))
    return mq, mk, mv
