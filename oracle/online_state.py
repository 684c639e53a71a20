"""Mergeable online-normaliser state for one query row.  TEST INFRASTRUCTURE
ONLY (see the package docstring).

Follows "Intermediate and advanced extension": the workshop table rows
"Online normalization" (a mergeable (maximum, exponential sum) state whose
result must not depend on how the keys are partitioned or in which order the
parts are merged) and "Streaming attention" (online rescaling), and "Logic
review before implementation" (a -inf empty maximum needs an explicit identity;
attention rescales the numerator accumulator as well as its denominator).
"Attention algorithms and data movement", lesson 01, names the same rescaling
law and the explicit empty-row contract.

A state summarises a set P of (score s_j, value v_j) pairs:
  m   = max_{j in P} s_j                     (-inf for the empty set)
  l   = sum_{j in P} exp(s_j - m)            (0 for the empty set)
  acc = sum_{j in P} exp(s_j - m) v_j        (0 for the empty set)
Merging two states of disjoint sets moves both onto the larger maximum: each
side's l and acc are multiplied by exp(m_side - m_new).  finalize gives
O = acc / l and lse = m + ln l; the empty state finalizes to O = 0, lse = -inf.
Scores are the already-scaled logits.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class State:
    m: float
    l: float
    acc: np.ndarray  # float64 [D]


def empty_state(d: int) -> State:
    """The identity of merge: (m, l, acc) = (-inf, 0, 0)."""
    return State(-math.inf, 0.0, np.zeros(d, dtype=np.float64))


def state_of_block(scores, values) -> State:
    """State of one block of keys: scores [n] (scaled logits), values [n, D]."""
    scores = np.asarray(scores, dtype=np.float64)
    values = np.asarray(values, dtype=np.float64)
    d = values.shape[1] if values.ndim == 2 else 0
    if scores.size == 0:
        return empty_state(d)
    m = float(np.max(scores))
    p = np.exp(scores - m)
    return State(m, float(p.sum()), p @ values)


def merge(a: State, b: State) -> State:
    """Combine the states of two disjoint key sets.  The empty state is an
    explicit identity, so empty+empty stays empty and never forms
    exp(-inf - (-inf)) = NaN."""
    if a.m == -math.inf:
        return b
    if b.m == -math.inf:
        return a
    m = max(a.m, b.m)
    alpha = math.exp(a.m - m)  # rescale factor of side a
    beta = math.exp(b.m - m)   # rescale factor of side b
    return State(m, a.l * alpha + b.l * beta, a.acc * alpha + b.acc * beta)


def finalize(st: State):
    """(O, lse) of a state; the empty state gives (0, -inf)."""
    if st.m == -math.inf:
        return np.zeros_like(st.acc), -math.inf
    return st.acc / st.l, st.m + math.log(st.l)
