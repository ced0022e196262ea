"""Payload and value comparison of the CUDA path against the CPU oracle (no GPU needed).

Criterion of the codec contract (include/fp4q.h): group and block scales bit-exact; codes
bit-exact except codes whose pre-rounding q lies within 2 float32 ulp of the E2M1 decision
midpoint nearest to it, at most 1e-6 of all codes; decoded / accumulated outputs within
1e-5 relative L2. Both sides compute q with the same correctly rounded steps, so the number
of such exempted codes is expected to be zero, and ``check_payload`` asserts that unless the
caller passes ``strict=False``.
"""
from __future__ import annotations

import numpy as np

import oracle
from fp4_communication_compression_gb300 import inputs

# E2M1 decision midpoints (between consecutive grid values 0, 0.5, 1, 1.5, 2, 3, 4, 6)
MIDS = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32)
MAX_ULPS = 2
MAX_FRACTION = 1e-6


def nibbles(codes: np.ndarray) -> np.ndarray:
    c = np.empty(codes.size * 2, np.uint8)
    c[0::2], c[1::2] = codes & 15, codes >> 4
    return c


def ulps_to_nearest_midpoint(q: np.ndarray) -> np.ndarray:
    """Distance in float32 ulps between |q| and the E2M1 midpoint nearest to it: the
    difference of the bit patterns (for non-negative floats the bit pattern is monotone in
    the value, so this counts the representable floats between them)."""
    qa = np.abs(np.asarray(q, np.float32))
    m = MIDS[np.argmin(np.abs(qa[:, None].astype(np.float64) - MIDS[None, :].astype(np.float64)), axis=1)]
    return np.abs(qa.view(np.int32).astype(np.int64) - m.view(np.int32).astype(np.int64))


def check_payload(got, want, q, n, G, what="", strict=True):
    """Compare a payload with the oracle's. Returns the number of code mismatches (each
    within MAX_ULPS of its nearest midpoint, at most MAX_FRACTION of n); with strict, any
    mismatch at all fails, since the contract expects none."""
    got = np.asarray(got, np.uint8)
    assert got.shape == want.shape, what
    g0 = oracle.gscale_offset(n, G)
    assert np.array_equal(got[g0:], want[g0:]), f"{what}: scales differ"
    cg, cw = nibbles(got[:g0]), nibbles(want[:g0])
    bad = np.nonzero(cg != cw)[0]
    if bad.size:
        d = ulps_to_nearest_midpoint(q[bad])
        far = d > MAX_ULPS
        assert not far.any(), (f"{what}: {int(far.sum())} code mismatches more than {MAX_ULPS} ulp from "
                               f"an E2M1 midpoint (first at element {int(bad[far][0])})")
        assert bad.size <= MAX_FRACTION * n, f"{what}: {bad.size} midpoint mismatches > {MAX_FRACTION} of {n}"
        assert not strict, f"{what}: {bad.size} code mismatches (all within {MAX_ULPS} ulp of a midpoint)"
    return int(bad.size)


def check_values(got, want, exact, what=""):
    """Decoded outputs: bit-identical when exact, and within 1e-5 relative L2 always."""
    if exact:
        assert np.array_equal(got.view(np.uint32 if got.dtype == np.float32 else np.uint16),
                              want.view(np.uint32 if want.dtype == np.float32 else np.uint16)), what
    a = got.astype(np.float64) if got.dtype == np.float32 else inputs.bf16_bits_to_f32(got).astype(np.float64)
    b = want.astype(np.float64) if want.dtype == np.float32 else inputs.bf16_bits_to_f32(want).astype(np.float64)
    den = np.linalg.norm(b)
    assert np.linalg.norm(a - b) <= 1e-5 * (den if den > 0 else 1.0), what
