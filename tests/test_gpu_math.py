"""The codec's branch-free reciprocal and division (csrc/fp4q_math.cuh) against CUDA's IEEE
__frcp_rn and __fdiv_rn: every significand of every exponent the codec's scales can take,
plus 2^30 random and midpoint-steered quotient pairs and the codec's whole scale chain for
every block maximum. Any mismatch would break bit parity
of the scales and codes."""
import os
import re
import subprocess

import pytest
import torch

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "fp4_communication_compression_gb300", "csrc")


def test_reciprocal_and_division_match_ieee(tmp_path):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    exe = str(tmp_path / "math_check")
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-fmad=false",
                    "-std=c++17", "-I", CSRC, os.path.join(HERE, "gpu_checks", "math_check.cu"),
                    "-o", exe], check=True)
    out = subprocess.run([exe], check=True, capture_output=True, text=True, timeout=300).stdout
    found = dict(re.findall(r"(\w+) bad=(\d+) tested=\d+", out))
    assert set(found) == {"rcp_rn", "div_rn_2688", "divider", "scale_chain"}, out
    assert all(v == "0" for v in found.values()), out
