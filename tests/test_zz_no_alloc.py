"""GPU check of attn_fwd_splitkv_noalloc, the split-KV entry point that uses
the library's fixed scratch instead of a caller workspace.  Two calls in a
row must each equal the workspace entry point (attn_fwd_splitkv) bit for
bit.  The file name keeps it last in collection; it also passes on its own,
when its call is the first on the device."""

import pytest
import torch

from exact_tiled_attention_19_gb300 import binding
from exact_tiled_attention_19_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def call_noalloc(q, k, v, num_splits, causal=True):
    B, Hq, Nq, D = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    o = torch.empty((B, Hq, Nq, D), dtype=q.dtype, device=q.device)
    lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=q.device)
    strides = [*q.stride(), *k.stride(), *v.stride(), *o.stride()]
    dtype = binding.ETATTN_BF16 if q.dtype == torch.bfloat16 else binding.ETATTN_F16
    rc = binding.attn_fwd_splitkv_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                          B, Hq, Hkv, Nq, Nk, D, dtype, strides, 1 if causal else 0, -1, -1,
                                          D ** -0.5, num_splits, torch.cuda.current_stream().cuda_stream)
    assert rc == 0, binding.etattn_status_string(rc)
    return o, lse


@pytest.mark.parametrize("Nq,Nk,splits", [(1, 8192, 6), (4, 3000, 3)])
def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row(Nq, Nk, splits):
    inp = W.random_qkv(4, 16, 4, Nq, 128, torch.bfloat16, seed=Nq + splits, Nk=Nk)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    o_ref, l_ref = binding.attention_splitkv(q, k, v, causal=True, num_splits=splits)
    o1, l1 = call_noalloc(q, k, v, splits)
    o2, l2 = call_noalloc(q, k, v, splits)
    torch.cuda.synchronize()
    assert torch.equal(o1, o_ref) and torch.equal(l1, l_ref)
    assert torch.equal(o2, o_ref) and torch.equal(l2, l_ref)
    assert binding.etattn_read_device_status(clear=True) == 0
