"""Host-side buffer checks of the Python binding (CPU only, no launch).

The C ABI receives bare pointers and cannot know how long a buffer is, so the binding must
reject every wrong payload, output or data buffer before anything is launched: an undersized
or mistyped buffer would otherwise be read or written out of bounds by the kernels. The
tensors here are stand-ins that report a CUDA device, and the library's compute entry points
are replaced by functions that fail the test if they are ever reached; the size queries
(fp4q_payload_bytes and the offsets) are the real library's host functions.
"""
import ctypes

import pytest
import torch

import fp4_communication_compression_gb300 as fq
from fp4_communication_compression_gb300 import _lib

N = 4096 * 4


class FakeCuda:
    """Duck-typed stand-in for a CUDA tensor (shape, dtype, device, contiguity)."""

    def __init__(self, numel, dtype, device="cuda:0", cuda=True, contiguous=True, shape=None, strides=None):
        self._n = int(numel)
        self.dtype = dtype
        self.device = torch.device(device)
        self.is_cuda = cuda
        self._contig = contiguous
        self.shape = tuple(shape) if shape else (self._n,)
        self._strides = tuple(strides) if strides else tuple(
            int(torch.tensor(self.shape[i + 1:]).prod()) if i + 1 < len(self.shape) else 1 for i in range(len(self.shape)))

    def numel(self):
        return self._n

    def is_contiguous(self):
        return self._contig

    def data_ptr(self):
        return 1 << 20

    def dim(self):
        return len(self.shape)

    def size(self, i=None):
        return self.shape if i is None else self.shape[i]

    def stride(self, i=None):
        return self._strides if i is None else self._strides[i]


class NoLaunch:
    HOST = {"fp4q_payload_bytes", "fp4q_gscale_offset", "fp4q_bscale_offset", "fp4q_status_string"}

    def __init__(self, real):
        self.real = real

    def __getattr__(self, name):
        if name in self.HOST:
            return getattr(self.real, name)

        def reached(*args):
            raise RuntimeError(f"LAUNCH {name}")
        return reached


@pytest.fixture()
def nolaunch(monkeypatch):
    _lib.build()
    stub = NoLaunch(_lib.lib())
    monkeypatch.setattr(_lib, "lib", lambda: stub)
    monkeypatch.setattr(fq, "_stream", lambda stream, device: ctypes.c_void_p(0))   # no CUDA runtime here
    return stub


def pb(n=N, **kw):
    return fq.payload_bytes(n, **kw)


def x16(**kw):
    return FakeCuda(N, torch.bfloat16, **kw)


def u8(nbytes, **kw):
    return FakeCuda(nbytes, torch.uint8, **kw)


def test_valid_calls_reach_the_library(nolaunch):
    """The stand-ins pass every check: each call below gets as far as the launch."""
    with pytest.raises(RuntimeError, match="LAUNCH fp4q_compress"):
        fq.compress(x16(), payload=u8(pb()))
    with pytest.raises(RuntimeError, match="LAUNCH fp4q_decompress_accumulate"):
        fq.decompress_accumulate(u8(pb()), N, x16())
    with pytest.raises(RuntimeError, match="LAUNCH fp4q_roundtrip"):
        fq.roundtrip(x16(), y=x16())
    with pytest.raises(RuntimeError, match="LAUNCH fp4q_reduce_requantize"):
        fq.reduce_requantize([u8(pb()), u8(pb() + 64)], N, out=u8(pb()))


BAD_PAYLOADS = {
    "undersized": lambda: u8(pb() - 1),
    "wrong dtype": lambda: FakeCuda(pb(), torch.int8),
    "float buffer": lambda: FakeCuda(pb() // 4 + 1, torch.float32),
    "not contiguous": lambda: u8(pb(), contiguous=False),
    "host tensor": lambda: u8(pb(), cuda=False, device="cpu"),
    "other device": lambda: u8(pb(), device="cuda:1"),
}


@pytest.mark.parametrize("case", sorted(BAD_PAYLOADS))
def test_compress_rejects_bad_payload(nolaunch, case):
    with pytest.raises(ValueError):
        fq.compress(x16(), payload=BAD_PAYLOADS[case]())


@pytest.mark.parametrize("case", sorted(BAD_PAYLOADS))
def test_decompress_rejects_bad_payload(nolaunch, case):
    with pytest.raises(ValueError):
        fq.decompress_accumulate(BAD_PAYLOADS[case](), N, x16())


@pytest.mark.parametrize("case", sorted(BAD_PAYLOADS))
@pytest.mark.parametrize("where", ["first", "last", "out"])
def test_reduce_rejects_bad_payload_or_out(nolaunch, case, where):
    good = [u8(pb()) for _ in range(3)]
    out = u8(pb())
    if where == "first":
        if case in ("host tensor", "other device"):
            pytest.skip("the first payload defines the device")
        good[0] = BAD_PAYLOADS[case]()
    elif where == "last":
        good[-1] = BAD_PAYLOADS[case]()
    else:
        out = BAD_PAYLOADS[case]()
    with pytest.raises(ValueError):
        fq.reduce_requantize(good, N, out=out)


def test_reduce_rejects_empty_list(nolaunch):
    with pytest.raises(ValueError):
        fq.reduce_requantize([], N)


def test_payload_size_follows_params(nolaunch):
    """The needed size is that of the call's own format: a G = 32 payload is smaller than a
    G = 16 one, so a G = 32-sized buffer is too small for a G = 16 call."""
    assert pb(group=32) < pb(group=16)
    with pytest.raises(ValueError):
        fq.compress(x16(), payload=u8(pb(group=32)), group=16)
    with pytest.raises(RuntimeError, match="LAUNCH"):
        fq.compress(x16(), payload=u8(pb(group=32)), group=32)
    with pytest.raises(ValueError):
        fq.decompress_accumulate(u8(pb(scales="e8m0")), N, x16(), scales="dual")


def test_data_tensors_are_checked(nolaunch):
    with pytest.raises(ValueError):
        fq.compress(x16(cuda=False, device="cpu"), payload=u8(pb()))
    with pytest.raises(ValueError):
        fq.decompress_accumulate(u8(pb()), N, x16(cuda=False, device="cpu"))
    with pytest.raises(ValueError):
        fq.decompress_accumulate(u8(pb()), N + 256, x16())              # dst has N elements
    with pytest.raises(ValueError):
        fq.roundtrip(x16(), y=x16(device="cuda:1"))
    with pytest.raises(ValueError):
        fq.roundtrip(x16(), y=FakeCuda(N - 256, torch.bfloat16))
    with pytest.raises(ValueError):
        fq.roundtrip(x16(), y=FakeCuda(N, torch.bfloat16, cuda=False, device="cpu"))
    with pytest.raises(TypeError):
        fq.compress(FakeCuda(N, torch.float16), payload=u8(pb()))
    with pytest.raises(ValueError):
        fq.compress(x16(), payload=u8(pb()), group=24)                  # invalid params: size 0


def test_strided_views_are_checked_too(nolaunch):
    """A strided 2-D view takes the *_2d entry point; its payload gets the same checks."""
    x = FakeCuda(N, torch.bfloat16, shape=(4, N // 4), strides=(N // 2, 1), contiguous=False)
    with pytest.raises(RuntimeError, match="LAUNCH fp4q_compress_2d"):
        fq.compress(x, payload=u8(pb()))
    with pytest.raises(ValueError):
        fq.compress(x, payload=u8(pb() - 16))
    with pytest.raises(ValueError):
        fq.decompress_accumulate(u8(pb() - 16), N, x)
