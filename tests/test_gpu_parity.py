"""GPU (sm_103a) vs CPU oracle parity, through the C ABI, on every workload at full size.

Criterion (the codec contract in include/fp4q.h; checker in parity_check.py): group and
block scales bit-exact; codes bit-exact except codes whose pre-rounding q lies within 2
float32 ulp of the E2M1 decision midpoint nearest to it, at most 1e-6 of all codes; decoded /
accumulated outputs within 1e-5 relative L2 (and bit-identical whenever every code matches,
since the decode is exact FP32 arithmetic in a fixed order on both sides). Both sides take
every rounding decision with the same correctly rounded steps, so every test here also
requires zero code mismatches (check_payload's strict mode) and prints the count.
"""
import numpy as np
import pytest
import torch

import oracle
import fp4_communication_compression_gb300 as fq
from fp4_communication_compression_gb300 import inputs
from parity_check import check_payload, check_values

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fq.build()
    return torch.device("cuda:0")


def _bits(t):
    return inputs.torch_to_bits(t)


def run_codec(dev, x_bits, G, fwht, dst_kinds=("bf16_0", "bf16_1", "f32_0", "f32_1"), tag=""):
    """Compress, decompress-accumulate (each dst kind) and roundtrip x on the GPU; compare
    every output with the oracle."""
    x = np.ascontiguousarray(x_bits).ravel()
    n = x.size
    xt = inputs.bits_to_torch(x, dev)
    p = fq.compress(xt, group=G, fwht=fwht)
    want, q = oracle.compress(x, group=G, fwht=fwht, want_q=True)
    torch.cuda.synchronize()
    mism = check_payload(p.cpu().numpy(), want, q, n, G, f"{tag} compress G={G} fwht={fwht}")
    print(f"{tag} compress G={G} fwht={fwht} n={n}: {mism} code mismatches")
    rng = np.random.default_rng(n + G + fwht)
    for kind in dst_kinds:
        dt, beta = kind.split("_")
        beta = int(beta)
        base = rng.standard_normal(n).astype(np.float32)
        if dt == "bf16":
            d0 = inputs.to_bf16_bits(base)
            dtt = inputs.bits_to_torch(d0, dev).clone()
        else:
            d0 = base
            dtt = torch.from_numpy(base).to(dev)
        fq.decompress_accumulate(p, n, dtt, beta=beta, group=G, fwht=fwht)
        # the oracle decodes the GPU payload: this isolates the decode from any compress flip
        ref = oracle.decompress_accumulate(p.cpu().numpy(), n, d0.copy(), beta=beta, group=G, fwht=fwht)
        got = _bits(dtt) if dt == "bf16" else dtt.cpu().numpy()
        check_values(got, ref, True, f"{tag} decompress {kind} G={G} fwht={fwht}")
    y = fq.roundtrip(xt, group=G, fwht=fwht)
    yref = oracle.roundtrip(x, group=G, fwht=fwht)
    check_values(_bits(y), yref, mism == 0, f"{tag} roundtrip G={G} fwht={fwht}")
    return p, want


# ------------------------------------------------------------------ small / ragged shapes

SMALL = [256, 512, 768, 2048, 2304, 256 * 17, 256 * 1000, 256 * 2049, 256 * 19457]


@pytest.mark.parametrize("fwht", [1, 0])
@pytest.mark.parametrize("G", [16, 32])
@pytest.mark.parametrize("n", SMALL)
def test_small_and_ragged_sizes(dev, n, G, fwht):
    run_codec(dev, inputs.sweep(n, seed=n % 97), G, fwht, tag=f"n={n}")


@pytest.mark.parametrize("fwht", [1, 0])
@pytest.mark.parametrize("G", [16, 32])
def test_edge_blocks(dev, G, fwht):
    run_codec(dev, inputs.edge_blocks(), G, fwht, tag="edge")


def test_hand_worked_block_on_gpu(dev):
    import json
    import os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "hand_worked_block.json")))
    x = np.zeros(256, np.float32)
    for off, vals in g["values"].items():
        x[int(off):int(off) + len(vals)] = vals
    p = fq.compress(inputs.bits_to_torch(inputs.to_bf16_bits(x), dev), group=16, fwht=0)
    pb = p.cpu().numpy()
    want = np.zeros(128, np.uint8)
    for off, b in g["expected_code_bytes"].items():
        want[int(off):int(off) + 8] = [int(v, 16) for v in b]
    assert np.array_equal(pb[:128], want)
    assert [f"{v:02X}" for v in pb[128:144]] == g["expected_group_scales"]
    assert f"{int(pb[144:148].view(np.uint32)[0]):08X}" == g["expected_block_scale_bits"]


# ------------------------------------------------------------------ the five workloads

def test_toy_config_with_two_rank_reduce(dev):
    """[8, 512] N(0,1) with +-40 outliers, R = 2 emulated ranks (seeds 0 and 1)."""
    xs = [inputs.toy(0), inputs.toy(1)]
    pays = [run_codec(dev, x, 16, 1, tag="toy")[0] for x in xs]
    n = xs[0].size
    red = fq.reduce_requantize(pays, n)
    want, q = oracle.reduce_requantize([p.cpu().numpy() for p in pays], n, 16, want_q=True)
    check_payload(red.cpu().numpy(), want, q, n, 16, "toy reduce")


def test_tp_activation_4096x4096(dev):
    run_codec(dev, inputs.tp_activation(), 16, 1, tag="tp_act")


@pytest.fixture(scope="module")
def four_ranks(dev):
    """Four [8192, 4096] rank buffers (seeds 1-4), compressed on the GPU and by the oracle;
    each GPU payload is checked against the oracle's."""
    xs = inputs.reduce_ranks(4)
    n = xs[0].size
    pays, refs = [], []
    for i, x in enumerate(xs):
        p = fq.compress(inputs.bits_to_torch(x.ravel(), dev))
        w, q = oracle.compress(x.ravel(), want_q=True)
        torch.cuda.synchronize()
        check_payload(p.cpu().numpy(), w, q, n, 16, f"rank {i} compress")
        pays.append(p)
        refs.append(w)
    return xs, pays, refs


@pytest.mark.parametrize("R", [4, 1, 2, 3, 8])
def test_emulated_reduce_8192x4096(dev, four_ranks, R):
    """Fused decompress-sum-requantize of R rank payloads held on one GPU (R = 4 is the
    workload; R = 1..8 reuse the four buffers cyclically)."""
    xs, pays, refs = four_ranks
    n = xs[0].size
    sel = [i % 4 for i in range(R)]
    red = fq.reduce_requantize([pays[i] for i in sel], n)
    want, q = oracle.reduce_requantize([refs[i] for i in sel], n, 16, want_q=True)
    mism = check_payload(red.cpu().numpy(), want, q, n, 16, f"reduce R={R}")
    print(f"reduce R={R} n={n}: {mism} code mismatches")
    out = torch.empty(n, dtype=torch.bfloat16, device=dev)
    fq.decompress_accumulate(red, n, out, beta=0)
    ref = oracle.decompress_accumulate(want, n, np.zeros(n, np.uint16), beta=0)
    check_values(_bits(out), ref, mism == 0, f"reduce R={R} decode")
    if R == 4:
        s = sum(inputs.bf16_bits_to_f32(x.ravel()).astype(np.float64) for x in xs)
        rel = np.linalg.norm(inputs.bf16_bits_to_f32(_bits(out)) - s) / np.linalg.norm(s)
        assert rel < 0.2


@pytest.mark.parametrize("fwht", [1, 0])
@pytest.mark.parametrize("G", [16, 32])
def test_gradient_16384x4096(dev, G, fwht):
    run_codec(dev, inputs.gradient(), G, fwht, dst_kinds=("bf16_1",), tag="grad")


@pytest.mark.parametrize("n", inputs.SWEEP_SIZES)
def test_size_sweep(dev, n):
    run_codec(dev, inputs.sweep(n), 16, 1, dst_kinds=("bf16_0", "bf16_1"), tag=f"sweep n={n}")


# ------------------------------------------------------------------ memory safety and streams

def test_guard_bands_untouched(dev):
    """Outputs placed inside larger buffers filled with a canary: nothing outside the
    declared output range may change (stand-in for a memory checker)."""
    n = 256 * 37
    G = 32                                   # odd block count: exercises the padding write
    x = inputs.bits_to_torch(inputs.sweep(n).ravel(), dev)
    nb = fq.payload_bytes(n, G)
    pad = 4096
    big = torch.full((nb + 2 * pad,), 0xA5, dtype=torch.uint8, device=dev)
    p = big[pad:pad + nb]
    fq.compress(x, payload=p, group=G)
    dbig = torch.full((n + 2 * pad,), 7.0, dtype=torch.float32, device=dev)
    fq.decompress_accumulate(p, n, dbig[pad:pad + n], beta=1, group=G)
    ybig = torch.full((n + 2 * pad,), 3.0, dtype=torch.bfloat16, device=dev)
    fq.roundtrip(x, y=ybig[pad:pad + n], group=G)
    rbig = torch.full((nb + 2 * pad,), 0x5A, dtype=torch.uint8, device=dev)
    fq.reduce_requantize([p, p, p], n, out=rbig[pad:pad + nb], group=G)
    torch.cuda.synchronize()
    b = big.cpu().numpy()
    assert np.all(b[:pad] == 0xA5) and np.all(b[pad + nb:] == 0xA5)
    d = dbig.cpu().numpy()
    assert np.all(d[:pad] == 7.0) and np.all(d[pad + n:] == 7.0)
    y = ybig.float().cpu().numpy()
    assert np.all(y[:pad] == 3.0) and np.all(y[pad + n:] == 3.0)
    r = rbig.cpu().numpy()
    assert np.all(r[:pad] == 0x5A) and np.all(r[pad + nb:] == 0x5A)
    g0 = oracle.gscale_offset(n, G)
    assert np.all(b[pad + g0 + n // G: pad + oracle.bscale_offset(n, G)] == 0)   # zeroed padding


def test_side_stream_and_determinism(dev):
    n = 1 << 20
    x = inputs.bits_to_torch(inputs.sweep(n).ravel(), dev)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        p1 = fq.compress(x)
        y1 = fq.roundtrip(x)
    s.synchronize()
    p2 = fq.compress(x)
    y2 = fq.roundtrip(x)
    torch.cuda.synchronize()
    assert torch.equal(p1, p2) and torch.equal(y1, y2)


def test_repeated_accumulate(dev):
    """Accumulating the same payload three times equals three oracle accumulations."""
    n = 1 << 16
    xb = inputs.sweep(n).ravel()
    p = fq.compress(inputs.bits_to_torch(xb, dev))
    d = torch.zeros(n, dtype=torch.float32, device=dev)
    ref = np.zeros(n, np.float32)
    pw = oracle.compress(xb)
    for _ in range(3):
        fq.decompress_accumulate(p, n, d, beta=1)
        oracle.decompress_accumulate(pw, n, ref, beta=1)
    torch.cuda.synchronize()
    assert np.array_equal(d.cpu().numpy(), ref)


def test_back_to_back_chain_keeps_stream_order(dev):
    """Kernels launched back to back with no host synchronisation, reusing buffers so that
    each kernel writes what the previous one reads (the payloads) and reads what the previous
    one wrote (the payloads and the accumulators): the kernels may start while their
    predecessor finishes, so this checks that each waits for it before touching memory."""
    n = 1 << 22
    xs = [inputs.sweep(n, seed=s).ravel() for s in (11, 12, 13)]
    xt = [inputs.bits_to_torch(x, dev) for x in xs]
    p = [torch.empty(fq.payload_bytes(n), dtype=torch.uint8, device=dev) for _ in range(2)]
    red = torch.empty_like(p[0])
    d = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    y = torch.empty_like(xt[0])
    torch.cuda.synchronize()
    ref_d = np.zeros(n, np.uint16)
    for it in range(4):
        a, b = xs[it % 3], xs[(it + 1) % 3]
        fq.compress(xt[it % 3], payload=p[0])
        fq.compress(xt[(it + 1) % 3], payload=p[1])
        fq.reduce_requantize(p, n, out=red)
        fq.decompress_accumulate(red, n, d, beta=1)
        fq.roundtrip(xt[it % 3], y=y)
        ref_red = oracle.reduce_requantize([oracle.compress(a), oracle.compress(b)], n)
        ref_d = oracle.decompress_accumulate(ref_red, n, ref_d, beta=1)
    torch.cuda.synchronize()
    assert np.array_equal(red.cpu().numpy(), ref_red)
    assert np.array_equal(_bits(d), ref_d)
    assert np.array_equal(_bits(y), oracle.roundtrip(xs[3 % 3]))
    assert fq.fault_flags() == 0


@pytest.mark.parametrize("G", [16, 32])
@pytest.mark.parametrize("nb", [1, 2, 3, 4, 5, 6, 7, 9, 13, 8 * 97 + 3, 8 * 2431 + 7])
def test_reduce_ragged_tails(dev, nb, G):
    """Block counts with every remainder modulo the 8-block tile: the last tile's codes,
    group scales and block scales are partly bulk-copied and partly loaded directly. R = 3, 4
    also cover the deferred pipeline start on warps with one tile or none."""
    n = 256 * nb
    xs = [inputs.sweep(n, seed=s).ravel() for s in (5, 6, 7, 8)]
    for R in (1, 2, 3, 4):
        pays = [fq.compress(inputs.bits_to_torch(x, dev), group=G) for x in xs[:R]]
        refs = [oracle.compress(x, group=G) for x in xs[:R]]
        torch.cuda.synchronize()
        for p, w in zip(pays, refs):
            assert np.array_equal(p.cpu().numpy(), w)
        red = fq.reduce_requantize(pays, n, group=G)
        want, q = oracle.reduce_requantize(refs, n, G, want_q=True)
        check_payload(red.cpu().numpy(), want, q, n, G, f"reduce nb={nb} R={R} G={G}")
