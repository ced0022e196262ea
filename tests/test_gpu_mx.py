"""GPU (sm_103a) vs CPU oracle parity of the microscaled variant (scales="e8m0": a
power-of-two E8M0 scale per group of 32, no block scale), through the C ABI.

With a power-of-two scale every q = y * 2^k is exact on both sides and the transform is the
same FP32 butterfly sequence, so payloads, decoded values and accumulations are required to
be bit-identical (no midpoint exemption)."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import fp4_communication_compression_gb300 as fq
from fp4_communication_compression_gb300 import inputs

pytestmark = pytest.mark.gpu
SC = "e8m0"
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "hand_worked_mx_block.json")


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fq.build()
    return torch.device("cuda:0")


def _bits(t):
    return inputs.torch_to_bits(t)


def run_mx(dev, x_bits, fwht, tag=""):
    x = np.ascontiguousarray(x_bits).ravel()
    n = x.size
    xt = inputs.bits_to_torch(x, dev)
    p = fq.compress(xt, fwht=fwht, scales=SC)
    want = oracle.compress(x, fwht=fwht, scales=SC)
    torch.cuda.synchronize()
    got = p.cpu().numpy()
    assert got.size == want.size == fq.payload_bytes(n, scales=SC), tag
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, f"{tag} fwht={fwht}: {bad.size} payload bytes differ, first at {bad[:5]}"
    rng = np.random.default_rng(n + fwht)
    for dt in ("bf16", "f32"):
        for beta in (0, 1):
            base = rng.standard_normal(n).astype(np.float32)
            if dt == "bf16":
                d0 = inputs.to_bf16_bits(base)
                dtt = inputs.bits_to_torch(d0, dev).clone()
            else:
                d0 = base
                dtt = torch.from_numpy(base).to(dev)
            fq.decompress_accumulate(p, n, dtt, beta=beta, fwht=fwht, scales=SC)
            ref = oracle.decompress_accumulate(want, n, d0.copy(), beta=beta, fwht=fwht, scales=SC)
            g = _bits(dtt) if dt == "bf16" else dtt.cpu().numpy().view(np.uint32)
            r = ref if dt == "bf16" else ref.view(np.uint32)
            assert np.array_equal(g, r), f"{tag} decompress {dt} beta={beta} fwht={fwht}"
    y = fq.roundtrip(xt, fwht=fwht, scales=SC)
    assert np.array_equal(_bits(y), oracle.roundtrip(x, fwht=fwht, scales=SC)), f"{tag} roundtrip fwht={fwht}"
    return p, want


@pytest.mark.parametrize("fwht", [1, 0])
@pytest.mark.parametrize("n", [256, 512, 768, 2048, 2304, 256 * 17, 256 * 1000, 256 * 2049, 256 * 19457])
def test_mx_small_and_ragged_sizes(dev, n, fwht):
    run_mx(dev, inputs.sweep(n, seed=n % 89), fwht, f"n={n}")


@pytest.mark.parametrize("fwht", [1, 0])
def test_mx_edge_blocks(dev, fwht):
    run_mx(dev, inputs.edge_blocks(), fwht, "edge blocks")


def test_mx_hand_worked_block_on_gpu(dev):
    g = json.load(open(GOLDEN))
    x = np.zeros(256, np.float32)
    for off, vals in g["values"].items():
        x[int(off):int(off) + len(vals)] = vals
    p, _ = run_mx(dev, inputs.to_bf16_bits(x), 0, "hand-worked")
    codes = p.cpu().numpy()
    for off, hexes in g["expected_code_bytes"].items():
        assert codes[int(off):int(off) + len(hexes)].tolist() == [int(h, 16) for h in hexes]
    assert codes[128:136].tolist() == g["expected_scale_codes"]


@pytest.mark.parametrize("fwht", [1, 0])
def test_mx_gradient_16384x4096(dev, fwht):
    run_mx(dev, inputs.gradient(), fwht, "gradient")


def test_mx_tp_activation_4096x4096(dev):
    run_mx(dev, inputs.tp_activation(), 1, "tp activation")


@pytest.mark.parametrize("R", [1, 2, 3, 4, 8])
def test_mx_reduce(dev, R):
    n = 1 << 21
    xs = [inputs.sweep(n, seed=40 + r).ravel() for r in range(R)]
    pays = [fq.compress(inputs.bits_to_torch(x, dev), scales=SC) for x in xs]
    out = fq.reduce_requantize(pays, n, scales=SC)
    refs = [oracle.compress(x, scales=SC) for x in xs]
    want = oracle.reduce_requantize(refs, n, scales=SC)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), want)


@pytest.mark.parametrize("nb", [1, 2, 3, 5, 7, 9, 13, 8 * 97 + 3])
def test_mx_reduce_ragged_tails(dev, nb):
    n = 256 * nb
    xs = [inputs.sweep(n, seed=s).ravel() for s in (5, 6, 7)]
    for R in (1, 2, 3):
        pays = [fq.compress(inputs.bits_to_torch(x, dev), scales=SC) for x in xs[:R]]
        out = fq.reduce_requantize(pays, n, scales=SC)
        want = oracle.reduce_requantize([oracle.compress(x, scales=SC) for x in xs[:R]], n, scales=SC)
        torch.cuda.synchronize()
        assert np.array_equal(out.cpu().numpy(), want), (nb, R)


def test_mx_reduce_of_one_payload_is_the_identity_at_full_size(dev):
    """A property that holds at any size: requantising a decoded E8M0 payload gives it back
    (checked here at 2^28 elements, 512 MiB of bfloat16 input, without the oracle)."""
    n = 1 << 28
    x = torch.randn(n, device=dev).to(torch.bfloat16)
    x[::997] *= 40
    for fwht in (0, 1):
        p = fq.compress(x, fwht=fwht, scales=SC)
        out = fq.reduce_requantize([p], n, scales=SC)
        assert torch.equal(out, p), fwht
    del x
    assert fq.fault_flags() == 0


@pytest.mark.parametrize("n", [1 << 24, 1 << 26])
def test_mx_size_sweep(dev, n):
    run_mx(dev, inputs.sweep(n), 1, f"sweep n={n}")
