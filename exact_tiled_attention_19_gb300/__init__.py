"""Exact streaming self-attention forward for NVIDIA GB300 (sm_103a).

O = softmax(scale * Q K^T + causal mask) V is computed tile by tile with an
online (running max, rescaled exp-sum) normaliser in hand-written tcgen05 /
TMA / tensor-memory CUDA kernels behind a C ABI (``include/etattn.h``); this
package holds the kernels' sources, the ctypes binding and the seeded
synthetic workloads.
"""
