"""GPU check of the failure-detection path: every pipeline wait of the
attention kernels is bounded, and a wait that runs out must be reported
through the device status word instead of hanging the GPU.  The self-test
kernel waits, with a 1 ms limit, on an mbarrier that nothing arrives at,
through the same bounded wait the pipelines use; it holds no tensor memory
and starts no copy or MMA, so the early return leaves nothing in flight."""

import pytest
import torch

from exact_tiled_attention_19_gb300 import binding
from exact_tiled_attention_19_gb300 import workloads as W
from tests.parity_helpers import compare_full, default_scale, run_gpu

pytestmark = pytest.mark.gpu


def test_a_wait_that_runs_out_is_reported_and_cleared():
    assert binding.etattn_read_device_status(clear=True) == binding.ETATTN_OK
    stream = torch.cuda.Stream()
    assert binding.etattn_selftest_wait_timeout(1000, stream.cuda_stream) == binding.ETATTN_OK
    assert binding.etattn_read_device_status(clear=True, stream=stream.cuda_stream) == binding.ETATTN_ERR_DEVICE
    assert binding.etattn_read_device_status(clear=True) == binding.ETATTN_OK


def test_the_device_stays_usable_after_a_timeout():
    assert binding.etattn_selftest_wait_timeout(500) == binding.ETATTN_OK
    assert binding.etattn_read_device_status(clear=True) == binding.ETATTN_ERR_DEVICE
    inp = W.random_qkv(1, 2, 2, 300, 64, torch.float16, seed=11)
    o, lse = run_gpu(inp, True)
    compare_full(inp, o, lse, True, default_scale(64), torch.float16)
    assert binding.etattn_read_device_status(clear=True) == binding.ETATTN_OK
