"""Pins of the CPU oracle against things fixed outside it (no GPU needed).

Each test checks the oracle against a closed form, a library routine, an exhaustive sweep
or a value worked out by hand, so that a plausible slip anywhere in the oracle (a dropped
term, a wrong sign, a swapped nibble, a transposed index, a different tie rule) fails one
of them. The codec contract being pinned: micro-grouped dual-scale FP4 (E2M1) quantisation
after a two-level FWHT, two codes per byte ("FP4Quant: Efficient 4-Bit Communication
Compression for Model-Parallel LLM Training", abstract; "4-bit compression speeds up LLM
training by 56 percent", lead paragraph).
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.linalg
import torch

import oracle
from fp4_communication_compression_gb300 import inputs

HERE = os.path.dirname(os.path.abspath(__file__))
U = 2.0 ** -24
GRID = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float64)
H256 = scipy.linalg.hadamard(256).astype(np.float64)      # Sylvester order, library routine


def _f32(x):
    return np.asarray(x, np.float32)


# ---------------------------------------------------------------------------- FWHT

def _blocks(seed, k):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((k, 256)).astype(np.float32)
    x[0] *= 1e-30
    x[1] *= 1e30
    x[2, ::17] *= 1000.0
    x[3] = rng.laplace(0, 1e-3, 256)
    return x


@pytest.mark.parametrize("inverse", [False, True])
def test_fwht_matches_dense_fp64_hadamard(inverse):
    """Butterfly FWHT in FP32 (forward order, and the decode's mirror order) vs the dense
    product H256 x / 16 in FP64 (scipy's Hadamard). Error bound of 8 stages of RN
    butterflies on an orthogonal transform: 8 u ||x||."""
    x = _blocks(1, 64)
    y = oracle.fwht256(x, inverse).reshape(x.shape).astype(np.float64)
    exact = x.astype(np.float64) @ H256.T / 16.0
    for i in range(x.shape[0]):
        nx = np.linalg.norm(x[i].astype(np.float64))
        assert np.linalg.norm(y[i] - exact[i]) <= 8 * U * nx * (1 + 1e-9)


def test_forward_and_mirror_orders_round_differently():
    """The two stage orders agree in exact arithmetic but not bit for bit, which is why the
    decode's order is part of the contract."""
    x = _blocks(9, 64)
    a, b = oracle.fwht256(x), oracle.fwht256(x, inverse=True)
    assert not np.array_equal(a, b)
    assert np.max(np.abs(a - b)) <= 1e-5 * np.max(np.abs(a))


@pytest.mark.parametrize("inverse", [False, True])
def test_fwht_special_cases_exact(inverse):
    e0 = np.zeros(256, np.float32); e0[0] = 1
    assert np.array_equal(oracle.fwht256(e0, inverse), np.full(256, 0.0625, np.float32))
    for k in (1, 2, 17, 128, 255):
        ek = np.zeros(256, np.float32); ek[k] = 1
        expect = np.array([(-1) ** bin(i & k).count("1") / 16 for i in range(256)], np.float32)
        assert np.array_equal(oracle.fwht256(ek, inverse), expect)
    ones = np.ones(256, np.float32)
    expect = np.zeros(256, np.float32); expect[0] = 16
    assert np.array_equal(oracle.fwht256(ones, inverse), expect)


def test_fwht_is_an_involution_and_preserves_energy():
    x = _blocks(2, 32)
    y = oracle.fwht256(x).reshape(x.shape)
    z = oracle.fwht256(y, inverse=True).reshape(x.shape)
    for i in range(x.shape[0]):
        nx = np.linalg.norm(x[i].astype(np.float64))
        assert np.linalg.norm(z[i].astype(np.float64) - x[i]) <= 16 * U * nx
        assert abs(np.linalg.norm(y[i].astype(np.float64)) - nx) <= 8 * U * nx * (1 + 1e-9)


def test_fwht_levels_act_on_groups_then_across_groups():
    """H256 = H16 (x) H16: a block that is constant inside each 16-group only excites the
    first position of each group (level 1), and a block equal across groups at a fixed
    position only excites group 0 (level 2)."""
    rng = np.random.default_rng(3)
    g = np.repeat(rng.integers(-8, 8, 16).astype(np.float32), 16)       # const per group
    for inv in (False, True):
        y = oracle.fwht256(g, inv)
        assert np.all(y.reshape(16, 16)[:, 1:] == 0)
    p = np.tile(rng.integers(-8, 8, 16).astype(np.float32), 16)          # same in every group
    for inv in (False, True):
        y = oracle.fwht256(p, inv)
        assert np.all(y.reshape(16, 16)[1:, :] == 0)


# ---------------------------------------------------------------------------- rounding

def _nonneg_patterns(lo_bits, hi_bits, chunk=1 << 26):
    for s in range(lo_bits, hi_bits, chunk):
        yield np.arange(s, min(s + chunk, hi_bits), dtype=np.uint32)


def test_e2m1_exhaustive_nonnegative():
    """Every non-negative float32 up to 8 (1.09e9 patterns). Expected code from the grid's
    decision boundaries: non-negative floats are ordered like their bit patterns, and the
    ties go to the even code, so the boundary is the midpoint itself when the upper code is
    even (0.75, 1.75, 3.5) and the next float above it when the lower code is even
    (0.25, 1.25, 2.5, 5)."""
    b = lambda v: int(np.float32(v).view(np.uint32))
    bounds = np.array(sorted([b(0.25) + 1, b(0.75), b(1.25) + 1, b(1.75), b(2.5) + 1,
                              b(3.5), b(5.0) + 1]), np.uint32)
    for pat in _nonneg_patterns(0, b(8.0) + 1):
        expect = np.searchsorted(bounds, pat, side="right").astype(np.uint8)
        got = oracle.e2m1_encode(pat.view(np.float32))
        assert np.array_equal(got, expect)


def test_e2m1_negative_and_signed_zero():
    rng = np.random.default_rng(4)
    q = rng.uniform(0, 8, 1 << 20).astype(np.float32)
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32)
    q = np.concatenate([q, mids, np.nextafter(mids, 0), np.nextafter(mids, 9), [0.0, 1e-40]]).astype(np.float32)
    pos = oracle.e2m1_encode(q)
    neg = oracle.e2m1_encode(-q)
    assert np.array_equal(neg, pos | 8)                      # sign bit kept, even for -0
    assert oracle.e2m1_encode(np.float32(-0.0))[0] == 8
    assert oracle.e2m1_encode(np.float32(1e9))[0] == 7 and oracle.e2m1_encode(np.float32(-1e9))[0] == 15


def test_e2m1_matches_ml_dtypes():
    ml = pytest.importorskip("ml_dtypes")
    rng = np.random.default_rng(5)
    q = np.concatenate([rng.uniform(-6, 6, 1 << 22), rng.standard_normal(1 << 20)]).astype(np.float32)
    lib = q.astype(ml.float4_e2m1fn).view(np.uint8) & 0xF
    assert np.array_equal(oracle.e2m1_encode(q), lib)


def test_e2m1_decode_table():
    assert np.array_equal(oracle.e2m1_decode(np.arange(8)), GRID.astype(np.float32))
    d = oracle.e2m1_decode(np.arange(8, 16))
    assert np.array_equal(d, -GRID.astype(np.float32)) and np.signbit(d[0])


def test_e4m3_exhaustive_against_two_libraries():
    """Every non-negative float32 below 464 against ml_dtypes.float8_e4m3fn and
    torch.float8_e4m3fn (both round to nearest even; they give NaN from 464 on, where the
    contract saturates)."""
    ml = pytest.importorskip("ml_dtypes")
    top = int(np.float32(464.0).view(np.uint32))
    for pat in _nonneg_patterns(0, top):
        f = pat.view(np.float32)
        got = oracle.e4m3_encode(f)
        assert np.array_equal(got, f.astype(ml.float8_e4m3fn).view(np.uint8))
        assert np.array_equal(got, torch.from_numpy(f).to(torch.float8_e4m3fn).view(torch.uint8).numpy())


def test_e4m3_saturation_and_ties():
    enc = lambda v: int(oracle.e4m3_encode(np.float32(v))[0])
    assert enc(464.0) == 0x7E and enc(1e30) == 0x7E and enc(448.0) == 0x7E
    assert enc(136.0) == 0x70 and enc(152.0) == 0x72 and enc(133.33) == 0x70
    assert enc(2.0 ** -10) == 0 and enc(np.nextafter(np.float32(2.0 ** -10), 1)) == 1
    assert enc(0.0) == 0 and enc(5.1e-6) == 0
    vals = oracle.e4m3_decode(np.arange(127))
    assert vals[0x7E] == 448 and vals[1] == 2.0 ** -9 and vals[0x38] == 1.0
    assert np.all(np.diff(vals) > 0)


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(6)
    pats = rng.integers(0, 1 << 32, 1 << 24, dtype=np.uint64).astype(np.uint32)
    # all tie patterns (low half exactly 0x8000) for a spread of upper halves
    ties = (np.arange(0, 1 << 16, 7, dtype=np.uint32) << 16) | 0x8000
    f = np.concatenate([pats, ties, ties + 1, ties - 1]).view(np.float32)
    finite = np.isfinite(f)
    f = f[finite]
    lib = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.bf16_round(f), lib)


# ---------------------------------------------------------------------------- payload

def test_payload_layout_sizes():
    assert oracle.payload_bytes(4096, 16) == 2048 + 256 + 64
    assert oracle.payload_bytes(4096, 32) == 2048 + 128 + 64
    assert oracle.payload_bytes(256, 32) == 128 + 16 + 4          # 8 scale bytes padded to 16
    assert oracle.bscale_offset(256, 32) == 144
    assert oracle.payload_bytes(1 << 24, 16) * 8 / (1 << 24) == 4.625   # bits per element
    assert oracle.payload_bytes(100, 16) == 128 + 16 + 4         # one zero-padded block
    for bad in [(0, 16), (512, 8), (-256, 16)]:
        assert oracle.payload_bytes(*bad) == 0


def test_unpack_every_byte_value():
    """Decode (fwht=0, scale 1.0) of a payload whose code bytes are 0..255: element 2k is
    the low nibble of byte k, element 2k+1 the high nibble."""
    n = 512
    p = np.zeros(oracle.payload_bytes(n, 16), np.uint8)
    codes, gsc, bsc = oracle.split_payload(p, n, 16)
    codes[:] = np.arange(256, dtype=np.uint8)
    gsc[:] = 0x38                                     # e4m3 1.0
    bsc[:] = 1.0
    out = np.zeros(n, np.float32)
    oracle.decompress_accumulate(p, n, out, beta=0, group=16, fwht=0)
    table = np.concatenate([GRID, -GRID]).astype(np.float32)
    b = np.arange(256)
    assert np.array_equal(out[0::2], table[b & 15]) and np.array_equal(out[1::2], table[b >> 4])
    assert np.array_equal(np.signbit(out[0::2]), (b & 15) >= 8)


def test_pack_every_byte_value():
    """Compress (fwht=0) a tensor whose every group holds a +-6 (so the scales are exactly 1)
    and otherwise grid values: the packed bytes must be exactly the chosen nibble pairs."""
    table = np.concatenate([GRID, -GRID]).astype(np.float32)
    free = list(range(256))
    rows = []
    while free:
        row = [0x77] + free[:7]                      # first byte: two codes of 6
        free = free[7:]
        row += [0x00] * (8 - len(row))
        rows.append(row)
    while len(rows) % 16:
        rows.append([0x77] + [0] * 7)
    want = np.array(rows, np.uint8).ravel()
    n = want.size * 2
    vals = np.empty(n, np.float32)
    vals[0::2] = table[want & 15]
    vals[1::2] = table[want >> 4]
    x = inputs.to_bf16_bits(vals)
    p = oracle.compress(x, group=16, fwht=0)
    codes, gsc, bsc = oracle.split_payload(p, n, 16)
    assert np.all(gsc == 0x7E)
    S = np.float32(oracle.e4m3_decode([0x7E])[0]) * bsc[0]
    assert S == 1.0
    assert np.array_equal(codes, want)


# ---------------------------------------------------------------------------- hand-worked

def _hand_block():
    g = json.load(open(os.path.join(HERE, "golden", "hand_worked_block.json")))
    x = np.zeros(256, np.float32)
    for off, vals in g["values"].items():
        x[int(off):int(off) + len(vals)] = vals
    xb = inputs.to_bf16_bits(x)
    assert np.array_equal(inputs.bf16_bits_to_f32(xb), x)      # every value is bf16-exact
    return g, xb


def test_hand_worked_block():
    g, xb = _hand_block()
    p = oracle.compress(xb, group=16, fwht=0)
    codes, gsc, bsc = oracle.split_payload(p, 256, 16)
    want = np.zeros(128, np.uint8)
    for off, bytes_ in g["expected_code_bytes"].items():
        want[int(off):int(off) + 8] = [int(v, 16) for v in bytes_]
    assert np.array_equal(codes, want)
    assert [f"{v:02X}" for v in gsc] == g["expected_group_scales"]
    assert f"{int(bsc.view(np.uint32)[0]):08X}" == g["expected_block_scale_bits"]
    out = np.zeros(256, np.float32)
    oracle.decompress_accumulate(p, 256, out, beta=0, group=16, fwht=0)
    dec = np.array(g["expected_group2_decoded"], np.float32)
    assert np.array_equal(out[32:48], dec) and np.array_equal(np.signbit(out[32:48]), np.signbit(dec))


def test_constant_block_roundtrips_exactly_with_fwht():
    """c = 168 * 2^-12: y_0 = 16 c = 0.65625, s_b = 2^-12, S = 0.109375, q_0 = 6 exactly."""
    c = np.float32(168 * 2.0 ** -12)
    xb = inputs.to_bf16_bits(np.full(512, c, np.float32))
    p = oracle.compress(xb, group=16, fwht=1)
    codes, gsc, bsc = oracle.split_payload(p, 512, 16)
    assert np.all(bsc == np.float32(2.0 ** -12))
    assert np.array_equal(gsc.reshape(2, 16)[:, 0], [0x7E, 0x7E]) and np.all(gsc.reshape(2, 16)[:, 1:] == 0)
    cb = codes.reshape(2, 128)
    assert np.all(cb[:, 0] == 0x07) and np.all(cb[:, 1:] == 0)
    y = oracle.roundtrip(xb, group=16, fwht=1)
    assert np.array_equal(y, xb)


def test_all_zero_and_tiny_blocks_give_zero_payload():
    x = np.zeros(1024, np.float32)
    x[512:768] = 2.0 ** -100                  # A below 2688 * 2^-100 after the FWHT
    p = oracle.compress(inputs.to_bf16_bits(x), group=16, fwht=1)
    assert not p.any()
    neg = inputs.to_bf16_bits(np.full(256, -0.0, np.float32))
    assert not oracle.compress(neg, group=16, fwht=1).any()


@pytest.mark.parametrize("fwht", [0, 1])
def test_zero_block_limit_is_inclusive_at_2688_times_2_pow_minus_100(fwht):
    """A block whose maximum is exactly 2688 * 2^-100 is coded (s_b = 2^-100, the spike's
    group scale 448 = 0x7E, its code 6 = 0x7); one bfloat16 ulp below, the block is all zero.
    With the transform a lone spike x gives |y| = |x| / 16 everywhere, so the spike is 16x.
    A mistaken comparison (<= instead of <) or a zero limit off by a factor fails here."""
    k = 16.0 if fwht else 1.0
    lim = 1.3125 * 2.0 ** -89
    assert np.float32(2688.0) * np.float32(2.0 ** -100) == np.float32(lim)
    at = np.zeros(256, np.float32); at[3] = k * lim
    p = oracle.compress(inputs.to_bf16_bits(at), group=16, fwht=fwht)
    codes, gsc, bsc = oracle.split_payload(p, 256, 16)
    assert bsc[0] == np.float32(2.0 ** -100)
    if fwht:      # every element is y = +-lim (row 3 of the Hadamard matrix): scales 448, codes +-6
        assert np.all(gsc == 0x7E) and np.all(codes & 0x77 == 0x77)
    else:
        assert gsc[0] == 0x7E and not gsc[1:].any()
        assert codes[1] == 0x70 and not np.delete(codes, 1).any()
    below = np.zeros(256, np.float32); below[3] = -k * (1.3125 - 2.0 ** -7) * 2.0 ** -89
    assert not oracle.compress(inputs.to_bf16_bits(below), group=16, fwht=fwht).any()


# ---------------------------------------------------------------------------- whole codec

def _decode_scales(p, n, G):
    codes, gsc, bsc = oracle.split_payload(p, n, G)
    ml = pytest.importorskip("ml_dtypes")
    sg = gsc.view(ml.float8_e4m3fn).astype(np.float32)            # library decode of E4M3
    S = (np.repeat(sg, G).reshape(-1, 256) * bsc[:, None]).astype(np.float32)
    return codes, S.ravel(), bsc


def _codes(codes):
    c = np.empty(codes.size * 2, np.uint8)
    c[0::2], c[1::2] = codes & 15, codes >> 4
    return c


def _y32(x, fwht):
    """Transform-domain values in FP32 (the oracle's FWHT, pinned above)."""
    xf = inputs.bf16_bits_to_f32(x)
    return oracle.fwht256(xf) if fwht else xf.copy()


MIDS = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])


def _check_codes_optimal(y, q, c, S):
    """No other E2M1 code is closer to y / S in exact arithmetic, except where q lies within
    3 float32 ulp of a decision midpoint (q = fl(y * fl(1/S)) differs from y / S by less)."""
    nz = S > 0
    t = np.abs(y[nz].astype(np.float64)) / S[nz].astype(np.float64)
    mag = GRID[c[nz] & 7]
    err = np.abs(t - mag)
    best = np.min(np.abs(t[:, None] - GRID[None, :]), axis=1)
    qa = np.abs(q[nz]).astype(np.float64)
    near = np.min(np.abs(qa[:, None] - MIDS[None, :]), axis=1) <= 3 * 2.0 ** -23 * np.maximum(qa, 0.25)
    assert np.all((err <= best * (1 + 1e-12)) | near)
    # the sign bit is the sign of y (also for -0 and for values coded 0)
    assert np.array_equal(c[nz] >= 8, np.signbit(y[nz]))
    # a group with a zero scale codes only +-0
    assert np.all((c[~nz] & 7) == 0)


@pytest.mark.parametrize("G,fwht", [(16, 1), (32, 1), (16, 0), (32, 0)])
def test_codes_are_optimal_given_the_scales(G, fwht):
    x = np.concatenate([inputs.toy(0).ravel(), inputs.sweep(1 << 15)[: 1 << 14],
                        inputs.edge_blocks().ravel()])
    n = x.size
    p, q = oracle.compress(x, group=G, fwht=fwht, want_q=True)
    codes, S, bsc = _decode_scales(p, n, G)
    y = _y32(x, fwht)
    zero_blocks = np.repeat(bsc == 0, 256)
    _check_codes_optimal(y[~zero_blocks], q[~zero_blocks], _codes(codes)[~zero_blocks], S[~zero_blocks])
    assert not _codes(codes)[zero_blocks].any()


def test_group_maximum_gets_the_top_code():
    """When the group scale is an E4M3 normal (r >= 2^-6), q_max = 6 r / s_g lies in
    [5.65, 6.4], so the largest element of every group is coded +-6."""
    x = inputs.sweep(1 << 15)
    n = x.size
    for fwht in (0, 1):
        p, q = oracle.compress(x, group=16, fwht=fwht, want_q=True)
        codes, gsc, bsc = oracle.split_payload(p, n, 16)
        c = _codes(codes).reshape(-1, 16)
        qa = np.abs(q).reshape(-1, 16)
        top = np.argmax(qa, axis=1)
        normal = gsc >= 0x08
        assert normal.mean() > 0.9
        assert np.all((c[np.arange(qa.shape[0]), top] & 7)[normal] == 7)
        qm = qa.max(axis=1)[normal]
        assert np.all(qm >= 5.65) and np.all(qm <= 6.4)


def test_quantisation_error_bound():
    """In the transform domain |y - x~| <= S for every element (the widest E2M1 gap is 2,
    saturation costs at most 0.4 S). The round-trip relative L2 error is only reported: the
    pages print no error figures."""
    x = inputs.sweep(1 << 17)
    xf = inputs.bf16_bits_to_f32(x).astype(np.float64)
    for fwht in (0, 1):
        p = oracle.compress(x, group=16, fwht=fwht)
        codes, S, bsc = _decode_scales(p, x.size, 16)
        xt = GRID[_codes(codes) & 7] * np.where(_codes(codes) >= 8, -1.0, 1.0) * S
        y = _y32(x, fwht).astype(np.float64)
        assert np.all(np.abs(y - xt) <= S * (1 + 1e-6))
        out = np.zeros(x.size, np.float32)
        oracle.decompress_accumulate(p, x.size, out, beta=0, group=16, fwht=fwht)
        assert np.linalg.norm(out - xf) / np.linalg.norm(xf) < 0.15


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_decompress_accumulate_matches_torch_add(dtype):
    x = inputs.sweep(1 << 15)
    n = x.size
    p = oracle.compress(x, group=16, fwht=1)
    xhat = np.zeros(n, np.float32)
    oracle.decompress_accumulate(p, n, xhat, beta=0, group=16, fwht=1)
    rng = np.random.default_rng(7)
    base = rng.standard_normal(n).astype(np.float32)
    if dtype == "bf16":
        d = inputs.to_bf16_bits(base)
        got = oracle.decompress_accumulate(p, n, d.copy(), beta=1, group=16, fwht=1)
        ref = (torch.from_numpy(inputs.bf16_bits_to_f32(d)) + torch.from_numpy(xhat)).to(torch.bfloat16)
        assert np.array_equal(got, ref.view(torch.int16).numpy().view(np.uint16))
        got0 = oracle.decompress_accumulate(p, n, d.copy(), beta=0, group=16, fwht=1)
        assert np.array_equal(got0, torch.from_numpy(xhat).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))
    else:
        got = oracle.decompress_accumulate(p, n, base.copy(), beta=1, group=16, fwht=1)
        assert np.array_equal(got, (torch.from_numpy(base) + torch.from_numpy(xhat)).numpy())


def test_roundtrip_is_compress_then_decompress():
    x = inputs.toy(0).ravel()
    for G in (16, 32):
        for fwht in (0, 1):
            y = oracle.roundtrip(x, group=G, fwht=fwht)
            p = oracle.compress(x, group=G, fwht=fwht)
            d = np.zeros(x.size, np.uint16)
            oracle.decompress_accumulate(p, x.size, d, beta=0, group=G, fwht=fwht)
            assert np.array_equal(y, d)


# ---------------------------------------------------------------------------- reduce

def test_reduce_of_the_hand_block_is_the_hand_block():
    """The hand-worked payload decodes to values whose requantisation reproduces it exactly
    (s_b stays 2^-9, every group scale and code is recovered); two identical ranks double
    only the block scale (z = 2 x~ exactly, so r and q are unchanged)."""
    g, xb = _hand_block()
    p = oracle.compress(xb, group=16, fwht=0)
    assert np.array_equal(oracle.reduce_requantize([p], 256, 16), p)
    p2 = oracle.reduce_requantize([p, p], 256, 16)
    codes, gsc, bsc = oracle.split_payload(p2, 256, 16)
    c0, g0, b0 = oracle.split_payload(p, 256, 16)
    assert np.array_equal(codes, c0) and np.array_equal(gsc, g0) and bsc[0] == 2 * b0[0]


def test_reduce_doubling_is_exact_on_random_payloads():
    x = inputs.sweep(1 << 15)
    p = oracle.compress(x, group=16, fwht=1)
    one = oracle.reduce_requantize([p], x.size, 16)
    two = oracle.reduce_requantize([p, p], x.size, 16)
    a1, g1, b1 = oracle.split_payload(one, x.size, 16)
    a2, g2, b2 = oracle.split_payload(two, x.size, 16)
    assert np.array_equal(a1, a2) and np.array_equal(g1, g2) and np.array_equal(b2, 2 * b1)


def test_reduce_sums_in_the_transform_domain():
    """The reduce's pre-rounding q times its output scale equals the FP64 transform of the
    sum of the ranks' original-domain decodes (H is linear and H * H = I), so the sum is
    taken over all ranks in the transform domain; and its codes are optimal for its scales."""
    xs = [inputs.toy(s).ravel() for s in (0, 1, 2)]
    n = xs[0].size
    ps = [oracle.compress(x, group=16, fwht=1) for x in xs]
    red, q = oracle.reduce_requantize(ps, n, 16, want_q=True)
    codes, S, bsc = _decode_scales(red, n, 16)
    dec = np.zeros(n)
    for p in ps:
        d = np.zeros(n, np.float32)
        oracle.decompress_accumulate(p, n, d, beta=0, group=16, fwht=1)
        dec += d
    z = (dec.reshape(-1, 256) @ H256.T / 16.0).ravel()
    zq = q.astype(np.float64) * S
    for b in range(n // 256):
        sl = slice(256 * b, 256 * b + 256)
        assert np.linalg.norm(zq[sl] - z[sl]) <= 1e-5 * np.linalg.norm(z[sl])
    zt = np.zeros(n, np.float32)
    for p in ps:                                        # transform-domain FP32 sum, rank order
        c2, S2, _ = _decode_scales(p, n, 16)
        cc = _codes(c2)
        zt = zt + (GRID[cc & 7] * np.where(cc >= 8, -1.0, 1.0)).astype(np.float32) * S2
    _check_codes_optimal(zt, q, _codes(codes), S)


@pytest.mark.parametrize("scales,G", [("dual", 16), ("dual", 32), ("e8m0", 32)])
@pytest.mark.parametrize("n", [1, 17, 255, 257, 256 * 3 + 1, 4096 + 100, 256 * 37 + 255])
def test_tail_is_the_zero_padded_block(n, scales, G):
    """n not a multiple of 256: the payload is that of the input zero-padded to whole blocks
    (written out here by the caller, not by the oracle), and the decode gives the first n
    values of the padded decode, leaving everything past n untouched."""
    m = -(-n // 256) * 256
    x = inputs.sweep(4096 * 4, seed=n % 11).ravel()[:n].copy()
    xp = np.zeros(m, np.uint16)
    xp[:n] = x
    for fwht in (0, 1):
        p = oracle.compress(x, group=G, fwht=fwht, scales=scales)
        pp = oracle.compress(xp, group=G, fwht=fwht, scales=scales)
        assert p.size == oracle.payload_bytes(m, G, scales)
        assert np.array_equal(p, pp)
        d = np.full(n + 7, 3.0, np.float32)
        oracle.decompress_accumulate(p, n, d[:n], beta=0, group=G, fwht=fwht, scales=scales)
        dp = np.zeros(m, np.float32)
        oracle.decompress_accumulate(pp, m, dp, beta=0, group=G, fwht=fwht, scales=scales)
        assert np.array_equal(d[:n], dp[:n]) and (d[n:] == 3.0).all()
        y = oracle.roundtrip(x, group=G, fwht=fwht, scales=scales)
        assert np.array_equal(y, oracle.roundtrip(xp, group=G, fwht=fwht, scales=scales)[:n])
        r = oracle.reduce_requantize([p, p], n, group=G, scales=scales)
        assert np.array_equal(r, oracle.reduce_requantize([pp, pp], m, group=G, scales=scales))


@pytest.mark.parametrize("scales,G", [("dual", 16), ("dual", 32), ("e8m0", 32)])
def test_f32_input_equals_bf16_input_on_bf16_values(scales, G):
    """FP32 input holding bfloat16-exact values must give the payload of the BF16 path (the
    widening is the only difference), at a length with a partial last block."""
    x = inputs.sweep(4096 * 8, seed=4).ravel()[:4096 * 8 - 77].copy()
    xf = inputs.bf16_bits_to_f32(x).astype(np.float32)
    for fwht in (0, 1):
        p16 = oracle.compress(x, group=G, fwht=fwht, scales=scales)
        p32 = oracle.compress_f32(xf, group=G, fwht=fwht, scales=scales)
        assert np.array_equal(p16, p32)
        y32 = oracle.roundtrip_f32(xf, group=G, fwht=fwht, scales=scales)
        d = np.zeros(xf.size, np.float32)
        oracle.decompress_accumulate(p32, xf.size, d, beta=0, group=G, fwht=fwht, scales=scales)
        assert np.array_equal(y32.view(np.uint32), d.view(np.uint32))
        assert np.array_equal(oracle.bf16_round(y32), oracle.roundtrip(x, group=G, fwht=fwht, scales=scales))


def test_f32_input_codes_are_optimal():
    """General FP32 input (not BF16-representable): with the FWHT off every code is the
    nearest grid point of q, which is y times the group's reciprocal scale, and the
    low mantissa bits of the input reach the codes (they differ from the BF16-rounded input's)."""
    rng = np.random.default_rng(12)
    x = (rng.standard_normal(256 * 64) * np.exp(rng.uniform(-3, 3, 64).repeat(256))).astype(np.float32)
    p, q = oracle.compress_f32(x, fwht=0, want_q=True)
    codes, _, _ = oracle.split_payload(p, x.size)
    c = np.empty(x.size, np.uint8)
    c[0::2], c[1::2] = codes & 15, codes >> 4
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    dist = np.abs(np.abs(q.astype(np.float64))[:, None] - grid[None, :])
    best = dist.min(axis=1)
    assert np.all(dist[np.arange(x.size), c & 7] == best)
    assert np.all((c >> 3) == np.signbit(q))
    pb = oracle.compress(inputs.to_bf16_bits(x), fwht=0)
    assert not np.array_equal(p, pb)
