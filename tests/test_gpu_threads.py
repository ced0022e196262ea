"""Calls from several host threads at once: each thread drives its own stream with its own
codec variant and sizes (fixed-grid and dynamic-claim), while the others run; every result
equals the same call made from one thread. The C calls run without the Python interpreter
lock (ctypes releases it), so the library's per-kernel plan cache and launch path are
exercised concurrently."""
import threading

import pytest
import torch

import fp4_communication_compression_gb300 as fq
from fp4_communication_compression_gb300 import inputs

pytestmark = pytest.mark.gpu

# (n, group, fwht, scales): one variant per thread
VARIANTS = [((1 << 22) + 3 * 256 + 5, 16, 1, "dual"), (1 << 25, 32, 0, "dual"),
            ((1 << 21) + 256, 32, 1, "e8m0"), (1 << 25, 16, 1, "dual")]
ITERS = 8


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    fq.build()
    return torch.device("cuda:0")


def _case(dev, n, G, F, sc, seed):
    """One thread's tensor and codec parameters."""
    x = inputs.bits_to_torch(inputs.sweep(n, seed=seed).ravel(), dev)
    kw = dict(group=G, fwht=F, scales=sc)
    return x, kw


def test_concurrent_threads_match_single_thread(dev):
    cases = [_case(dev, n, G, F, sc, 40 + i) for i, (n, G, F, sc) in enumerate(VARIANTS)]
    torch.cuda.synchronize()
    results, errors = [None] * len(cases), []

    def run(i):
        try:
            torch.cuda.set_device(dev)
            x, kw = cases[i]
            s = torch.cuda.Stream(dev)
            with torch.cuda.stream(s):
                d = torch.zeros_like(x)
                for _ in range(ITERS):
                    p = fq.compress(x, stream=s, **kw)
                    y = fq.roundtrip(x, stream=s, **kw)
                    fq.decompress_accumulate(p, x.numel(), d, beta=1, stream=s, **kw)
            s.synchronize()
            results[i] = (p, y, d)
        except Exception as e:      # reported below, on the main thread
            errors.append((i, repr(e)))

    threads = [threading.Thread(target=run, args=(i,)) for i in range(len(cases))]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    assert not any(t.is_alive() for t in threads), "a thread did not finish"
    assert not errors, errors
    for (x, kw), (p, y, d) in zip(cases, results):
        p1 = fq.compress(x, **kw)
        y1 = fq.roundtrip(x, **kw)
        d1 = torch.zeros_like(x)
        for _ in range(ITERS):
            fq.decompress_accumulate(p1, x.numel(), d1, beta=1, **kw)
        torch.cuda.synchronize()
        assert torch.equal(p, p1)
        assert torch.equal(y.view(torch.int16), y1.view(torch.int16))
        assert torch.equal(d.view(torch.int16), d1.view(torch.int16))
    assert fq.fault_flags() == 0
