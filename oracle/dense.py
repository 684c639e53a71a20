"""Dense float64 softmax attention: the plain definition of what the streaming
kernel computes.  TEST INFRASTRUCTURE ONLY (see the package docstring).

Definition followed ("Intermediate and advanced extension", workshop table row
"Streaming attention" and "Logic review before implementation";
"Intermediate and advanced workshop validation", "Correctness and review",
which checks attention against dense FP64 math):

  s_ij   = scale * <q_i, k_j>
  E(i)   = eligible keys: {j <= i} under the causal mask (the diagonal is
           included, so no causal row is empty), else every key
  M_i    = max_{j in E(i)} s_ij
  O_i    = sum_{j in E(i)} exp(s_ij - M_i) v_j / sum_{j in E(i)} exp(s_ij - M_i)
  lse_i  = M_i + ln sum_{j in E(i)} exp(s_ij - M_i)          (natural log)

Grouped-query attention ("Attention algorithms and data movement", lesson 05,
GQA head mapping): query head h reads key/value head h // (Hq / Hkv).

Packed variable-length batches (same page, lesson 04, packed causal
eligibility): positions i, j are logical positions 0..L_s-1 inside sequence s;
no key is eligible across sequences.

Unequal lengths (same page, lesson 04, unequal-length alignment; the pages
fix no convention, the reading taken here is bottom-right): with Lq queries
and Lk keys, query row i sits at key position c_i = i + (Lk - Lq), so a short
block of queries attends as the LAST Lq rows of a square problem would.
Causal: j <= c_i.  An optional window keeps keys with
c_i - window_left <= j <= c_i + window_right (-1 = unbounded on that side);
causal is window_right = 0.

Global tokens (same page, lesson 07, "global-token unions"; the pages give only
the lesson's title, the reading taken here is the usual one): the first
num_global positions of a sequence are global tokens.  Every row may also read
the global keys, and a global row (c_i < num_global) may read every key; both
still obey the causal mask, neither obeys the window.  So
E(i) = C(i) ∩ (W(i) ∪ {j < num_global} ∪ [every key if c_i < num_global]),
with C(i) the causal set and W(i) the window: a union of sets, in which a key
that is both global and inside the window counts once.

Empty rows (same page, lesson 01, explicit empty-row contract): a row with no
eligible key (e.g. c_i < 0 under the causal mask when Lq > Lk) gets O = 0 and
lse = -inf.

Inputs are float64 arrays holding the exact stored FP16/BF16 values.  Query
rows are processed in chunks only to bound memory; each row's arithmetic is
the definition above, unchanged.
"""

from __future__ import annotations

import numpy as np

_ROW_CHUNK = 1024


def kv_head_of(h, group):
    """GQA head mapping: query head h reads key/value head h // group, where
    group = Hq / Hkv ("Attention algorithms and data movement", lesson 05)."""
    return h // group


def eligible_keys(pos_rows, L, causal, Lq=None, window_left=-1, window_right=-1, num_global=0):
    """[R, L] boolean eligibility of L keys for query rows at positions
    pos_rows (in 0..Lq-1; Lq defaults to L).  The row sits at key position
    c = pos + L - Lq.  Causal: key j is eligible iff j <= c (the diagonal is
    included, "Logic review before implementation"); a window further keeps
    c - window_left <= j <= c + window_right (negative = unbounded).  With
    num_global = G > 0 the global keys j < G, and every key for a global row
    (c < G), are added to the window's keys, under the causal mask only."""
    Lq = L if Lq is None else Lq
    c = np.asarray(pos_rows, dtype=np.int64)[:, None] + (L - Lq)
    j = np.arange(L)[None, :]
    causal_ok = (j <= c) if causal else np.ones((len(pos_rows), L), dtype=bool)
    window_ok = np.ones((len(pos_rows), L), dtype=bool)
    if window_right >= 0:
        window_ok &= j <= c + window_right
    if window_left >= 0:
        window_ok &= j >= c - window_left
    if num_global > 0:
        window_ok = window_ok | (j < num_global) | (c < num_global)
    return causal_ok & window_ok


def _rows_attention(q_rows, pos_rows, k, v, causal, scale, Lq=None, window_left=-1, window_right=-1, num_global=0):
    """O and lse for query rows ``q_rows`` [R, D] at logical positions
    ``pos_rows`` [R] (of Lq query rows, default Lq = L) against keys ``k``
    [L, D] / values ``v`` [L, D] at positions 0..L-1."""
    q_rows = np.asarray(q_rows, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    R, L = q_rows.shape[0], k.shape[0]
    o = np.zeros((R, v.shape[1]), dtype=np.float64)
    lse = np.full((R,), -np.inf, dtype=np.float64)
    if R == 0 or L == 0:
        return o, lse
    s = scale * (q_rows @ k.T)  # [R, L]
    eligible = eligible_keys(pos_rows, L, causal, Lq, window_left, window_right, num_global)
    nonempty = eligible.any(axis=1)
    s_masked = np.where(eligible, s, -np.inf)
    m = np.max(s_masked, axis=1)
    m_safe = np.where(nonempty, m, 0.0)
    p = np.where(eligible, np.exp(s_masked - m_safe[:, None]), 0.0)
    l = p.sum(axis=1)
    o[nonempty] = (p[nonempty] @ v) / l[nonempty, None]
    lse[nonempty] = m[nonempty] + np.log(l[nonempty])
    return o, lse


def attention_rows(q, k, v, rows, *, causal, scale, window_left=-1, window_right=-1, num_global=0):
    """Attention for selected query positions of one (batch, head).

    q: [Nq, D], k, v: [Nk, D]; rows: int indices into 0..Nq-1.
    Returns (O [len(rows), D], lse [len(rows)])."""
    rows = np.asarray(rows, dtype=np.int64)
    return _rows_attention(np.asarray(q, dtype=np.float64)[rows], rows, k, v, causal, scale, len(q),
                           window_left, window_right, num_global)


def attention_dense(q, k, v, *, causal, scale, window_left=-1, window_right=-1, num_global=0):
    """Batched multi-head attention.

    q: [B, Hq, Nq, D]; k, v: [B, Hkv, Nk, D] with Hq % Hkv == 0.
    Returns O [B, Hq, Nq, D] (float64) and lse [B, Hq, Nq] (float64)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, Hq, N, D = q.shape
    Hkv = k.shape[1]
    if Hkv <= 0 or Hq % Hkv != 0:
        raise ValueError("Hq must be a multiple of Hkv")
    group = Hq // Hkv
    o = np.zeros((B, Hq, N, v.shape[3]), dtype=np.float64)
    lse = np.full((B, Hq, N), -np.inf, dtype=np.float64)
    for b in range(B):
        for h in range(Hq):
            hk = kv_head_of(h, group)
            for r0 in range(0, N, _ROW_CHUNK):
                rows = np.arange(r0, min(N, r0 + _ROW_CHUNK))
                o[b, h, rows], lse[b, h, rows] = _rows_attention(
                    q[b, h, rows], rows, k[b, hk], v[b, hk], causal, scale, N, window_left, window_right,
                    num_global)
    return o, lse


def attention_varlen(q, k, v, cu_seqlens, *, causal, scale, cu_seqlens_k=None, window_left=-1, window_right=-1,
                     num_global=0):
    """Packed variable-length attention.

    q: [Tq, Hq, D]; k, v: [Tk, Hkv, D]; cu_seqlens: [S+1] non-decreasing
    query-token offsets from 0 to Tq; cu_seqlens_k: the same for the keys
    (default: cu_seqlens, i.e. self-attention).
    Returns O [Tq, Hq, D] and lse [Hq, Tq] (float64)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    cuk = cu if cu_seqlens_k is None else np.asarray(cu_seqlens_k, dtype=np.int64)
    T, Hq, D = q.shape
    Hkv = k.shape[1]
    if Hkv <= 0 or Hq % Hkv != 0:
        raise ValueError("Hq must be a multiple of Hkv")
    group = Hq // Hkv
    o = np.zeros((T, Hq, v.shape[2]), dtype=np.float64)
    lse = np.full((Hq, T), -np.inf, dtype=np.float64)
    for s in range(len(cu) - 1):
        t0, t1 = int(cu[s]), int(cu[s + 1])
        k0, k1 = int(cuk[s]), int(cuk[s + 1])
        for h in range(Hq):
            hk = kv_head_of(h, group)
            for r0 in range(0, t1 - t0, _ROW_CHUNK):
                rows = np.arange(r0, min(t1 - t0, r0 + _ROW_CHUNK))
                o[t0 + rows, h], lse[h, t0 + rows] = _rows_attention(
                    q[t0 + rows, h], rows, k[k0:k1, hk], v[k0:k1, hk], causal, scale, t1 - t0,
                    window_left, window_right, num_global)
    return o, lse


def attention_varlen_rows(q, k, v, cu_seqlens, seq, head, rows, *, causal, scale, group=1, cu_seqlens_k=None,
                          window_left=-1, window_right=-1, num_global=0):
    """Attention for selected logical positions ``rows`` of sequence ``seq``
    and query head ``head`` of a packed batch (layout as in attention_varlen).
    Returns (O [len(rows), D], lse [len(rows)])."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    cuk = cu if cu_seqlens_k is None else np.asarray(cu_seqlens_k, dtype=np.int64)
    t0, t1 = int(cu[seq]), int(cu[seq + 1])
    k0, k1 = int(cuk[seq]), int(cuk[seq + 1])
    rows = np.asarray(rows, dtype=np.int64)
    hk = kv_head_of(head, group)
    return _rows_attention(np.asarray(q[t0 + rows, head], dtype=np.float64), rows,
                           k[k0:k1, hk], v[k0:k1, hk], causal, scale, t1 - t0, window_left, window_right,
                           num_global)
