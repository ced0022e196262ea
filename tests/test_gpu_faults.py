"""Bounded waits on the GPU: the TMA pipelines poll their barriers a bounded number of
times and report through a device fault word instead of hanging. The self-test makes one
wait run out on a barrier that nothing completes (no copy is in flight), then checks that
the word reports it and that the context stays usable."""
import numpy as np
import pytest
import torch

import oracle
import fp4_communication_compression_gb300 as fq
from fp4_communication_compression_gb300 import _lib, inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fq.build()
    return torch.device("cuda:0")


def test_normal_runs_leave_no_fault(dev):
    fq.fault_flags(clear=True)
    x = inputs.bits_to_torch(inputs.sweep(1 << 20).ravel(), dev)
    p = fq.compress(x)
    d = torch.zeros_like(x)
    fq.decompress_accumulate(p, x.numel(), d, beta=1)
    fq.roundtrip(x)
    assert fq.fault_flags() == 0


def test_selftest_wait_runs_out_and_is_reported(dev):
    fq.fault_flags(clear=True)
    st = _lib.lib().fp4q_selftest_wait_timeout(1000, None)
    assert st == _lib.OK
    torch.cuda.synchronize()
    assert fq.fault_flags(clear=True) == 4
    assert fq.fault_flags() == 0
    # the context is still usable and exact
    xb = inputs.toy(0).ravel()
    p = fq.compress(inputs.bits_to_torch(xb, dev))
    assert np.array_equal(p.cpu().numpy(), oracle.compress(xb))
