"""Pins of the oracle's microscaled variant (scales="e8m0": a power-of-two E8M0 scale per
group of 32 E2M1 codes, no block scale; the MXFP4 format the pages mention, scaled blocks
of 32 E2M1 elements). Each check ties the oracle to something other than its own code: a
hand-worked block, the defining property of the scale, brute-force optimality of every code
in exact rational arithmetic, exact decoding, and the exact idempotence of requantising a
decoded payload."""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from fp4_communication_compression_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "hand_worked_mx_block.json")
GRID = [Fraction(0), Fraction(1, 2), Fraction(1), Fraction(3, 2), Fraction(2), Fraction(3), Fraction(4), Fraction(6)]


def f32(bits16):
    return inputs.bf16_bits_to_f32(bits16)


def test_hand_worked_mx_block():
    g = json.load(open(GOLDEN))
    x = np.zeros(256, np.float32)
    for off, vals in g["values"].items():
        x[int(off):int(off) + len(vals)] = vals
    xb = inputs.to_bf16_bits(x)
    assert np.array_equal(f32(xb), x), "fixture values must be bfloat16-exact"
    p = oracle.compress(xb, fwht=0, scales="e8m0")
    codes, gsc, bsc = oracle.split_payload(p, 256, scales="e8m0")
    assert bsc.size == 0 and p.size == 128 + 16
    for off, hexes in g["expected_code_bytes"].items():
        want = np.array([int(h, 16) for h in hexes], np.uint8)
        assert np.array_equal(codes[int(off):int(off) + len(want)], want), off
    assert gsc.tolist() == g["expected_scale_codes"]
    d = np.zeros(256, np.float32)
    oracle.decompress_accumulate(p, 256, d, beta=0, fwht=0, scales="e8m0")
    for off, vals in g["expected_decoded"].items():
        got = d[int(off):int(off) + len(vals)]
        assert np.array_equal(got, np.array(vals, np.float32)), off
        assert np.array_equal(np.signbit(got), np.signbit(np.array(vals, np.float32))), off
    assert not d[64:].any()


def test_e8m0_scale_defining_property():
    """X = 2^(code - 127) is the power of two with amax / X in [4, 8); below 2^-125 the
    exponent is clamped at -127 (code 0), and amax = 0 gives code 0."""
    rng = np.random.default_rng(1)
    mant = rng.uniform(1.0, 2.0, 20000)
    exps = rng.integers(-125, 126, 20000)
    a = np.ldexp(mant, exps).astype(np.float32)
    a = np.concatenate([a, np.ldexp(1.0, np.arange(-125, 126)).astype(np.float32),
                        np.nextafter(np.ldexp(1.0, np.arange(-124, 126)), 0).astype(np.float32)])
    codes = oracle.e8m0_scale(a)
    for v, c in zip(a.tolist(), codes.tolist()):
        X = math.ldexp(1.0, int(c) - 127)
        assert 4.0 <= v / X < 8.0, (v, c)
    tiny = np.array([0.0, 2.0 ** -126, 2.0 ** -127, 2.0 ** -140, 2.0 ** -149, 2.0 ** -125 * 1.5], np.float32)
    assert oracle.e8m0_scale(tiny).tolist() == [0, 0, 0, 0, 0, 0]
    assert oracle.e8m0_decode([0, 127, 254]).tolist() == [2.0 ** -127, 1.0, 2.0 ** 127]


def _nearest_code(q: Fraction) -> int:
    """Exhaustive nearest E2M1 magnitude to |q| (ties to the even index), saturating at 6."""
    a = abs(q)
    best = min(range(8), key=lambda i: (abs(a - GRID[i]), i % 2, i))
    return best


@pytest.mark.parametrize("fwht", [0, 1])
def test_every_code_is_the_nearest_grid_point(fwht):
    rng = np.random.default_rng(7 + fwht)
    n = 256 * 12
    x = rng.standard_normal(n) * np.exp(rng.uniform(-12, 12, n // 32).repeat(32))
    x[rng.choice(n, 20, replace=False)] *= 300.0
    x[512:544] = 0.0
    x[544:576] = 1e-38
    xb = inputs.to_bf16_bits(x.astype(np.float32))
    p, q = oracle.compress(xb, fwht=fwht, scales="e8m0", want_q=True)
    codes, gsc, _ = oracle.split_payload(p, n, scales="e8m0")
    c = np.empty(n, np.uint8)
    c[0::2], c[1::2] = codes & 0xF, codes >> 4
    y = f32(xb).astype(np.float32)
    if fwht:
        y = oracle.fwht256(y.copy())
    for g in range(n // 32):
        yg = y[32 * g:32 * g + 32]
        X = Fraction(2) ** (int(gsc[g]) - 127)
        amax = max(abs(Fraction(float(v))) for v in yg)
        if amax >= Fraction(2) ** -125:
            assert 4 <= amax / X < 8
            assert max(int(k) & 7 for k in c[32 * g:32 * g + 32]) >= 6
        for i in range(32):
            qi = Fraction(float(q[32 * g + i]))
            assert qi == Fraction(float(yg[i])) / X or abs(qi) < Fraction(2) ** -126
            ci = int(c[32 * g + i])
            assert (ci & 7) == _nearest_code(Fraction(float(yg[i])) / X), (g, i)
            assert (ci >> 3) == int(np.signbit(yg[i]))


def test_decode_is_exact_grid_times_power_of_two():
    xb = inputs.sweep(1 << 14, seed=3).ravel()
    n = xb.size
    p = oracle.compress(xb, fwht=0, scales="e8m0")
    codes, gsc, _ = oracle.split_payload(p, n, scales="e8m0")
    d = np.zeros(n, np.float32)
    oracle.decompress_accumulate(p, n, d, beta=0, fwht=0, scales="e8m0")
    c = np.empty(n, np.uint8)
    c[0::2], c[1::2] = codes & 0xF, codes >> 4
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float64)
    want = grid[c & 7] * np.ldexp(1.0, gsc.astype(np.int64).repeat(32) - 127) * np.where(c >> 3, -1.0, 1.0)
    assert np.array_equal(d.astype(np.float64), want)


@pytest.mark.parametrize("fwht", [0, 1])
def test_requantising_a_decoded_payload_is_the_identity(fwht):
    """Reduce with R = 1 decodes in the transform domain and quantises again: with a
    power-of-two scale the decoded group maximum is 4X or 6X, so the same X comes back and
    every code is reproduced exactly (the dual-scale format has no such identity)."""
    xb = inputs.sweep(1 << 15, seed=9).ravel()
    p = oracle.compress(xb, fwht=fwht, scales="e8m0")
    assert np.array_equal(oracle.reduce_requantize([p], xb.size, scales="e8m0"), p)


def test_mx_roundtrip_matches_compress_then_decompress():
    xb = inputs.toy(0).ravel()
    for fwht in (0, 1):
        p = oracle.compress(xb, fwht=fwht, scales="e8m0")
        y = np.zeros(xb.size, np.uint16)
        oracle.decompress_accumulate(p, xb.size, y, beta=0, fwht=fwht, scales="e8m0")
        assert np.array_equal(oracle.roundtrip(xb, fwht=fwht, scales="e8m0"), y)


def test_mx_rejects_group_16():
    with pytest.raises(ValueError):
        oracle.compress(inputs.toy(0).ravel(), group=16, scales="e8m0")
    assert oracle.payload_bytes(4096, 16, "e8m0") == 0
    assert oracle.payload_bytes(4096, scales="e8m0") == 2048 + 128
