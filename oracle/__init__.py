"""CPU FP64 oracle for exact softmax self-attention.

TEST INFRASTRUCTURE ONLY. Nothing in the product path may import this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` use it. The CUDA path shares no code
with it (no kernels, headers, helpers, constants or pre/post-processing).

Modules
-------
``dense``        the plain definition of the result: O = softmax(scale*Q K^T +
                 mask) V and the per-row logsumexp, computed densely in float64
                 per (batch, head) or per packed sequence.
``online_state`` the mergeable (running max m, rescaled exp-sum l, numerator
                 acc) state with its explicit empty identity, the algebra the
                 streaming method is built on.
``backward``     the gradients dQ, dK, dV of sum(dO * O), from probabilities
                 recomputed by the definition (dense, or sampled rows of a
                 large problem).

Sources (web pages, cited by title and section):
  * "Intermediate and advanced extension" (triton-cuda-lab), workshop table row
    "Streaming attention" and "Logic review before implementation".
  * "Intermediate and advanced workshop validation" (triton-cuda-lab),
    "Correctness and review".
  * "Attention algorithms and data movement" (study.greatitself.com), lessons
    01 (merging normalised attention), 03 (differentiating the normalised
    row), 04 (packed causal eligibility, unequal lengths), 05 (GQA head
    mapping) and 07 (local windows, global-token unions).

Parity status: every function here is pinned by CPU tests in
``tests/test_oracle.py``, ``tests/test_oracle_lengths.py``,
``tests/test_oracle_global.py`` and ``tests/test_oracle_backward.py`` against
closed forms (interval inclusion-exclusion counts among them), a hand-worked example, library
routines (PyTorch's CPU scaled_dot_product_attention and its float64
autograd, SciPy's logsumexp), finite differences, invariants and brute
force; none is "parity unpinned".
"""

from .dense import attention_dense, attention_varlen, attention_rows, attention_varlen_rows
from .online_state import State, empty_state, state_of_block, merge, finalize
from .backward import attention_backward_dense, attention_backward_sampled, backward_d_rounding, backward_magnitudes

__all__ = [
    "attention_dense",
    "attention_varlen",
    "attention_rows",
    "attention_varlen_rows",
    "State",
    "empty_state",
    "state_of_block",
    "merge",
    "finalize",
    "attention_backward_dense",
    "attention_backward_sampled",
    "backward_d_rounding",
    "backward_magnitudes",
]
