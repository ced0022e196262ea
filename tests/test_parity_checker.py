"""The GPU parity checker itself, on the CPU: planted mismatches in an oracle payload must be
accepted or rejected exactly as the contract's criterion says (a code may differ only when
its q lies within 2 float32 ulp of the E2M1 midpoint nearest to it, at most 1e-6 of all
codes, and the strict mode used by the GPU tests accepts no mismatch at all)."""
import numpy as np
import pytest

import oracle
from fp4_communication_compression_gb300 import inputs
from parity_check import check_payload, ulps_to_nearest_midpoint

N = 1 << 20


@pytest.fixture(scope="module")
def payload():
    x = inputs.sweep(N, seed=3).ravel()
    want, q = oracle.compress(x, group=16, fwht=1, want_q=True)
    return want, q


def _step(v, k):
    """The float32 k representable values above (k > 0) or below (k < 0) the positive v."""
    return np.array([np.float32(v)]).view(np.int32)[0] + np.int32(k)


def _plant(want, q, elem, qv):
    """A copy of the payload whose code `elem` differs, with q[elem] set to qv."""
    got = want.copy()
    byte, hi = elem // 2, elem % 2
    shift = 4 * hi
    c = (got[byte] >> shift) & 15
    got[byte] = (got[byte] & ~np.uint8(15 << shift)) | np.uint8(((c ^ 1) & 15) << shift)
    q2 = q.copy()
    q2[elem] = qv
    return got, q2


def _f32(bits):
    return np.array([bits], np.int32).view(np.float32)[0]


def test_identical_payload_passes(payload):
    want, q = payload
    assert check_payload(want.copy(), want, q, N, 16, "identity") == 0


@pytest.mark.parametrize("mid", [0.25, 0.75, 1.25, 5.0])
@pytest.mark.parametrize("k", [-2, -1, 1, 2])
def test_within_two_ulp_is_exempt_but_not_strict(payload, mid, k):
    want, q = payload
    got, q2 = _plant(want, q, 1234, _f32(_step(mid, k)))
    assert ulps_to_nearest_midpoint(q2[[1234]])[0] == abs(k)
    assert check_payload(got, want, q2, N, 16, "planted", strict=False) == 1
    with pytest.raises(AssertionError, match="code mismatches"):
        check_payload(got, want, q2, N, 16, "planted")


@pytest.mark.parametrize("mid", [0.25, 0.75, 1.75, 3.5])
@pytest.mark.parametrize("k", [-3, 3, 16])
def test_three_ulp_off_a_midpoint_is_rejected(payload, mid, k):
    """The former checker took 2 ulp of the largest midpoint (5.0) as the window for every
    midpoint, which at 0.25 is 32 ulp; 3 ulp off any midpoint must now fail."""
    want, q = payload
    got, q2 = _plant(want, q, 777, _f32(_step(mid, k)))
    with pytest.raises(AssertionError, match="from an E2M1 midpoint"):
        check_payload(got, want, q2, N, 16, "planted", strict=False)


def test_negative_q_uses_its_magnitude(payload):
    want, q = payload
    got, q2 = _plant(want, q, 99, -_f32(_step(0.75, 2)))
    assert check_payload(got, want, q2, N, 16, "planted", strict=False) == 1
    got, q2 = _plant(want, q, 99, -_f32(_step(0.75, -3)))
    with pytest.raises(AssertionError):
        check_payload(got, want, q2, N, 16, "planted", strict=False)


def test_more_than_one_per_million_is_rejected(payload):
    want, q = payload
    got, q2 = want.copy(), q.copy()
    for e in (10, 5000, 90001):          # three mismatches in 2^20 codes > 1e-6 * n
        got, q2 = _plant(got, q2, e, _f32(_step(1.25, 1)))
    with pytest.raises(AssertionError, match="midpoint mismatches"):
        check_payload(got, want, q2, N, 16, "planted", strict=False)


def test_scale_difference_is_rejected(payload):
    want, q = payload
    got = want.copy()
    got[oracle.gscale_offset(N, 16) + 17] ^= 1
    with pytest.raises(AssertionError, match="scales differ"):
        check_payload(got, want, q, N, 16, "planted", strict=False)
    got = want.copy()
    got[-1] ^= 0x80                      # a block scale's sign bit
    with pytest.raises(AssertionError, match="scales differ"):
        check_payload(got, want, q, N, 16, "planted", strict=False)
