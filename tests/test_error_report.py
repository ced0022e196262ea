"""Directional error claims, checked on the oracle (CPU only).

The pages state two qualitative effects without numbers: micro-groups keep the local
distribution of the tensor ("FP4Quant", shd-paper.top summary, key design: dual-scale
micro-grouping), and the fast transform keeps the quantisation error low (zot.news, lead
paragraph). Neither is a parity pin; these tests compute the round-trip relative L2 error
of the oracle on reduced copies of the gradient-payload and TP-activation workloads and
check the directions this reading reproduces:

* groups of 16 are never worse than groups of 32 (dual scales, transform on and off);
* with power-of-two (E8M0) scales the transform lowers the error;
* with dual scales at G = 16 the transform raises the error on these workloads: the pages'
  claim is not reproduced for this format (an outlier only spoils its own 16-element
  group, while the transform spreads it over 256 elements). This is recorded as a finding,
  so that a change to the oracle that flips it is noticed.
"""
import numpy as np
import pytest

import oracle
from fp4_communication_compression_gb300 import inputs

f32 = inputs.bf16_bits_to_f32


@pytest.fixture(scope="module")
def workloads():
    return {
        "gradient [512, 4096]": inputs.gradient(rows=512).ravel(),
        "TP activation [512, 4096]": inputs.tp_activation(tokens=512).ravel(),
    }


def rel_err(x, group, fwht, scales="dual"):
    xf = f32(x).astype(np.float64)
    y = f32(oracle.roundtrip(x, group=group, fwht=fwht, scales=scales)).astype(np.float64)
    return float(np.linalg.norm(y - xf) / np.linalg.norm(xf))


@pytest.mark.parametrize("fwht", [0, 1])
def test_group16_error_not_above_group32(workloads, fwht):
    for name, x in workloads.items():
        e16, e32 = rel_err(x, 16, fwht), rel_err(x, 32, fwht)
        assert e16 <= e32, (name, e16, e32)


def test_transform_lowers_microscaled_error(workloads):
    for name, x in workloads.items():
        off, on = rel_err(x, 32, 0, "e8m0"), rel_err(x, 32, 1, "e8m0")
        assert on < off, (name, off, on)


def test_transform_raises_dual_scale_error_at_group16(workloads):
    for name, x in workloads.items():
        off, on = rel_err(x, 16, 0), rel_err(x, 16, 1)
        assert off < on, (name, off, on)
        # sanity bound: these round-trip errors are 0.07-0.11
        assert on < 0.15 and off < 0.15, (name, off, on)
