"""C ABI checks that need no GPU: the library builds, loads and exports every function
include/fp4q.h declares; sizes and offsets follow the payload layout; and every argument
error is returned as a status before anything is launched (each call below fails a host
check, so no CUDA call is made)."""
import ctypes
import os
import re

import pytest

import oracle
from fp4_communication_compression_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp4q.h")


@pytest.fixture(scope="module")
def L():
    _lib.build()
    return _lib.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fp4q_[a-z_0-9]+)\s*\(", text)))


def test_build_flags_keep_exact_arithmetic():
    """Bit parity with the oracle needs every FP32 operation rounded on its own: the library
    must be built without FMA contraction, for sm_103a only."""
    assert "-fmad=false" in _lib.NVCC_FLAGS
    assert not any("fast-math" in f or "ftz=true" in f for f in _lib.NVCC_FLAGS)
    assert "arch=compute_103a,code=sm_103a" in _lib.NVCC_FLAGS


def test_header_declares_the_binding_exports():
    assert declared_functions() == sorted(_lib.EXPORTS)


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name
    assert L.fp4q_version() >= 100


def test_status_strings(L):
    for s in range(7):
        assert isinstance(_lib.status_string(s), str) and _lib.status_string(s)
    assert _lib.status_string(99) == "unknown status"


@pytest.mark.parametrize("n", [256, 4096, 256 * 17, 1 << 24, 256 * 1001, 1, 100, 4095, 256 * 1001 + 17])
@pytest.mark.parametrize("G", [16, 32])
def test_payload_layout_matches_oracle(L, n, G):
    p = _lib.params(G, 1)
    assert L.fp4q_payload_bytes(n, ctypes.byref(p)) == oracle.payload_bytes(n, G)
    assert L.fp4q_gscale_offset(n, ctypes.byref(p)) == oracle.gscale_offset(n, G)
    assert L.fp4q_bscale_offset(n, ctypes.byref(p)) == oracle.bscale_offset(n, G)
    assert L.fp4q_bscale_offset(n, ctypes.byref(p)) % 16 == 0


@pytest.mark.parametrize("n", [256, 4096, 256 * 17, 1 << 24, 256 * 1001])
def test_e8m0_payload_layout_matches_oracle(L, n):
    p = _lib.params(fwht=1, scales="e8m0")
    assert p.group == 32
    assert L.fp4q_payload_bytes(n, ctypes.byref(p)) == oracle.payload_bytes(n, scales="e8m0")
    assert L.fp4q_payload_bytes(n, ctypes.byref(p)) == n // 2 + (n // 32 + 15) // 16 * 16
    assert L.fp4q_gscale_offset(n, ctypes.byref(p)) == oracle.gscale_offset(n, scales="e8m0")
    assert L.fp4q_bscale_offset(n, ctypes.byref(p)) == oracle.bscale_offset(n, scales="e8m0")


def test_payload_bytes_defaults_and_invalid(L):
    assert L.fp4q_payload_bytes(4096, None) == 2368
    for n in (0, -256, 1 << 37, 1 << 40):
        assert L.fp4q_payload_bytes(n, None) == 0
    # a length that is not a multiple of 256 gets a zero-padded last block
    assert L.fp4q_payload_bytes(100, None) == 128 + 16 + 4
    assert L.fp4q_payload_bytes(4096 + 1, None) == L.fp4q_payload_bytes(4096 + 256, None)
    for g, b, f in [(8, 256, 1), (16, 128, 1), (16, 256, 3), (64, 256, 0)]:
        assert L.fp4q_payload_bytes(4096, ctypes.byref(_lib.Params(g, b, f))) == 0
    # fwht = 2 (the tensor-core encoder) writes either payload format
    assert L.fp4q_payload_bytes(4096, ctypes.byref(_lib.Params(16, 256, 2))) == 2368
    assert L.fp4q_payload_bytes(4096, ctypes.byref(_lib.Params(32, 256, 2, 1))) == 2048 + 128
    # E8M0 scales need group 32; unknown scale formats are rejected
    for g, sc in [(16, 1), (32, 2), (32, -1), (16, 7)]:
        assert L.fp4q_payload_bytes(4096, ctypes.byref(_lib.Params(g, 256, 1, sc))) == 0
    assert L.fp4q_payload_bytes(4096, ctypes.byref(_lib.Params(32, 256, 0, 1))) == 2048 + 128


# Fake, never dereferenced device addresses: every call below must fail a host check.
A = 0x7f0000000000          # 16-byte aligned
B = 0x7f0000100000
P = _lib.params(16, 1)


def test_compress_argument_errors(L):
    pp = ctypes.byref(P)
    assert L.fp4q_compress(None, 4096, B, pp, None) == _lib.ERR_NULL
    assert L.fp4q_compress(A, 4096, None, pp, None) == _lib.ERR_NULL
    for n in (0, -256, 1 << 37, 1 << 40):
        assert L.fp4q_compress(A, n, B, pp, None) == _lib.ERR_SIZE
    assert L.fp4q_compress(A + 8, 4096, B, pp, None) == _lib.ERR_ALIGN
    assert L.fp4q_compress(A, 4096, B + 2, pp, None) == _lib.ERR_ALIGN
    assert L.fp4q_compress(A, 4096, A + 16, pp, None) == _lib.ERR_OVERLAP
    assert L.fp4q_compress(A, 4096, A + 2 * 4096 - 16, pp, None) == _lib.ERR_OVERLAP
    for bad in [(8, 256, 1), (16, 512, 1), (16, 256, -1), (33, 256, 0), (16, 256, 1, 1), (32, 256, 1, 3)]:
        assert L.fp4q_compress(A, 4096, B, ctypes.byref(_lib.Params(*bad)), None) == _lib.ERR_PARAM


def test_decompress_argument_errors(L):
    pp = ctypes.byref(P)
    f = L.fp4q_decompress_accumulate
    assert f(None, 4096, B, _lib.BF16, 1, pp, None) == _lib.ERR_NULL
    assert f(A, 4096, None, _lib.BF16, 1, pp, None) == _lib.ERR_NULL
    assert f(A, 4096, B, 2, 1, pp, None) == _lib.ERR_PARAM
    assert f(A, 4096, B, _lib.BF16, 2, pp, None) == _lib.ERR_PARAM
    assert f(A, 4096, B, _lib.F32, -1, pp, None) == _lib.ERR_PARAM
    assert f(A, 0, B, _lib.BF16, 1, pp, None) == _lib.ERR_SIZE
    assert f(A + 4, 4096, B, _lib.BF16, 1, pp, None) == _lib.ERR_ALIGN
    assert f(A, 4096, B + 4, _lib.F32, 0, pp, None) == _lib.ERR_ALIGN
    assert f(A, 4096, A + 2048, _lib.BF16, 1, pp, None) == _lib.ERR_OVERLAP
    # a float32 dst is twice as long as a bfloat16 one: overlap is checked on its real size
    assert f(A + 8192 + 16, 4096, A, _lib.F32, 1, pp, None) == _lib.ERR_OVERLAP


def test_roundtrip_argument_errors(L):
    pp = ctypes.byref(P)
    f = L.fp4q_roundtrip
    assert f(None, 4096, B, pp, None) == _lib.ERR_NULL
    assert f(A, 4096, None, pp, None) == _lib.ERR_NULL
    assert f(A, -1, B, pp, None) == _lib.ERR_SIZE
    assert f(A, 4096, B + 8, pp, None) == _lib.ERR_ALIGN
    assert f(A, 4096, A, pp, None) == _lib.ERR_OVERLAP
    assert f(A, 4096, A + 8176, pp, None) == _lib.ERR_OVERLAP


def test_reduce_argument_errors(L):
    pp = ctypes.byref(P)
    f = L.fp4q_reduce_requantize

    def arr(*ptrs):
        a = (ctypes.c_void_p * len(ptrs))(*ptrs)
        return ctypes.cast(a, ctypes.c_void_p)

    two = arr(A, A + 0x10000)
    assert f(two, 0, 4096, B, pp, None) == _lib.ERR_PARAM
    assert f(two, 9, 4096, B, pp, None) == _lib.ERR_PARAM
    assert f(None, 2, 4096, B, pp, None) == _lib.ERR_NULL
    assert f(two, 2, 4096, None, pp, None) == _lib.ERR_NULL
    assert f(arr(A, None), 2, 4096, B, pp, None) == _lib.ERR_NULL
    assert f(two, 2, 0, B, pp, None) == _lib.ERR_SIZE
    assert f(arr(A, A + 0x10008), 2, 4096, B, pp, None) == _lib.ERR_ALIGN
    assert f(two, 2, 4096, B + 4, pp, None) == _lib.ERR_ALIGN
    assert f(two, 2, 4096, A + 0x10000 + 1024, pp, None) == _lib.ERR_OVERLAP
    assert f(two, 2, 4096, A, pp, None) == _lib.ERR_OVERLAP


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "absent.so"))
    monkeypatch.setattr(_lib, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        _lib.lib()


def test_fault_and_selftest_argument_errors(L):
    assert L.fp4q_fault_flags(None, 0) == _lib.ERR_NULL
    assert L.fp4q_selftest_wait_timeout(0, None) == _lib.ERR_PARAM
    assert L.fp4q_selftest_wait_timeout((1 << 20) + 1, None) == _lib.ERR_PARAM


def test_f32_entry_points_argument_errors(L):
    pp = ctypes.byref(P)
    for f in (L.fp4q_compress_f32, L.fp4q_roundtrip_f32):
        assert f(None, 4096, B, pp, None) == _lib.ERR_NULL
        assert f(A, 0, B, pp, None) == _lib.ERR_SIZE
        assert f(A + 4, 4096, B, pp, None) == _lib.ERR_ALIGN
        assert f(A, 4096, B, ctypes.byref(_lib.Params(16, 256, 1, 1)), None) == _lib.ERR_PARAM
    # FP32 input spans 4 bytes per element: an output starting inside the second half of it
    # overlaps (it would not for a BF16 input of the same n)
    assert L.fp4q_compress_f32(A, 4096, A + 2 * 4096 + 16, pp, None) == _lib.ERR_OVERLAP
    assert L.fp4q_roundtrip_f32(A, 4096, A + 4 * 4096 - 16, pp, None) == _lib.ERR_OVERLAP


def test_2d_entry_points_argument_errors(L):
    pp = ctypes.byref(P)
    c2, d2, r2 = L.fp4q_compress_2d, L.fp4q_decompress_accumulate_2d, L.fp4q_roundtrip_2d
    assert c2(None, 4, 512, 1024, B, pp, None) == _lib.ERR_NULL
    for rows, cols in [(0, 512), (4, 0), (4, 300), (4, 100), (1 << 30, 1 << 10)]:
        assert c2(A, rows, cols, 4096, B, pp, None) == _lib.ERR_SIZE, (rows, cols)
    assert c2(A, 4, 512, 256, B, pp, None) == _lib.ERR_PARAM          # ld < cols
    assert c2(A, 4, 512, 1 << 40, B, pp, None) == _lib.ERR_PARAM
    assert c2(A, 4, 512, 516, B, pp, None) == _lib.ERR_ALIGN          # 1032-byte rows
    assert c2(A, 4, 512, 520, B + 8, pp, None) == _lib.ERR_ALIGN
    # the view spans (rows - 1) * ld + cols elements: a payload inside the last row overlaps
    assert c2(A, 4, 512, 1024, A + 2 * (3 * 1024 + 128), pp, None) == _lib.ERR_OVERLAP
    assert d2(A, 4, 512, B, 514, _lib.F32, 1, pp, None) == _lib.ERR_ALIGN   # 2056-byte f32 rows
    assert d2(A, 4, 512, B, 1024, 7, 1, pp, None) == _lib.ERR_PARAM
    assert r2(A, 4, 512, 1024, B, 256, pp, None) == _lib.ERR_PARAM
    assert r2(A, 4, 512, 1024, A + 1024, 1024, pp, None) == _lib.ERR_OVERLAP


def _seg(c, g, b):
    return _lib.Segments(c, g, b)


def test_segment_bytes(L):
    c, g, b = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    for n, G, sc in [(4096, 16, "dual"), (256 * 37 + 5, 32, "dual"), (256 * 7, 32, "e8m0"), (1, 16, "dual")]:
        p = _lib.params(G, 1, scales=sc)
        assert L.fp4q_segment_bytes(n, ctypes.byref(p), ctypes.byref(c), ctypes.byref(g), ctypes.byref(b)) == _lib.OK
        total = oracle.payload_bytes(n, G, scales=sc)
        assert c.value == oracle.gscale_offset(n, G, scales=sc)
        assert g.value == oracle.bscale_offset(n, G, scales=sc) - c.value
        assert c.value + g.value + b.value == total
        assert (b.value == 0) == (sc == "e8m0")
    assert L.fp4q_segment_bytes(0, ctypes.byref(P), ctypes.byref(c), ctypes.byref(g), ctypes.byref(b)) == _lib.ERR_SIZE
    assert L.fp4q_segment_bytes(4096, ctypes.byref(P), None, ctypes.byref(g), ctypes.byref(b)) == _lib.ERR_NULL
    assert L.fp4q_segment_bytes(4096, ctypes.byref(_lib.Params(8, 256, 1)), ctypes.byref(c), ctypes.byref(g),
                                ctypes.byref(b)) == _lib.ERR_PARAM


def test_segment_entry_points_argument_errors(L):
    pp = ctypes.byref(P)
    good = _seg(B, B + 0x10000, B + 0x20000)
    cs, ds, rs = L.fp4q_compress_segments, L.fp4q_decompress_accumulate_segments, L.fp4q_reduce_requantize_segments
    assert cs(A, _lib.BF16, 4096, None, pp, None) == _lib.ERR_NULL
    assert cs(None, _lib.BF16, 4096, ctypes.byref(good), pp, None) == _lib.ERR_NULL
    assert cs(A, _lib.BF16, 4096, ctypes.byref(_seg(B, None, B + 0x20000)), pp, None) == _lib.ERR_NULL
    assert cs(A, _lib.BF16, 4096, ctypes.byref(_seg(B, B + 0x10000, None)), pp, None) == _lib.ERR_NULL
    # E8M0 scales have no block-scale segment: NULL passes the null check there (the call is
    # stopped by the misaligned input instead, before any launch)
    mx = ctypes.byref(_lib.params(32, 1, scales="e8m0"))
    assert cs(A + 8, _lib.BF16, 4096, ctypes.byref(_seg(B, B + 0x10000, None)), mx, None) == _lib.ERR_ALIGN
    assert cs(A, 5, 4096, ctypes.byref(good), pp, None) == _lib.ERR_PARAM
    assert cs(A, _lib.BF16, 0, ctypes.byref(good), pp, None) == _lib.ERR_SIZE
    assert cs(A, _lib.BF16, 4096, ctypes.byref(_seg(B, B + 0x10008, B + 0x20000)), pp, None) == _lib.ERR_ALIGN
    assert cs(A + 8, _lib.BF16, 4096, ctypes.byref(good), pp, None) == _lib.ERR_ALIGN
    # a segment inside the input, or two segments on top of each other
    assert cs(A, _lib.BF16, 4096, ctypes.byref(_seg(B, A + 4096, B + 0x20000)), pp, None) == _lib.ERR_OVERLAP
    assert cs(A, _lib.F32, 4096, ctypes.byref(_seg(B, A + 3 * 4096, B + 0x20000)), pp, None) == _lib.ERR_OVERLAP
    assert cs(A, _lib.BF16, 4096, ctypes.byref(_seg(B, B + 1024, B + 0x20000)), pp, None) == _lib.ERR_OVERLAP
    assert cs(A, _lib.BF16, 4096, ctypes.byref(_seg(B, B + 0x10000, B + 0x10000 + 128)), pp, None) == _lib.ERR_OVERLAP
    assert ds(None, 4096, A, _lib.BF16, 1, pp, None) == _lib.ERR_NULL
    assert ds(ctypes.byref(good), 4096, A, _lib.BF16, 3, pp, None) == _lib.ERR_PARAM
    assert ds(ctypes.byref(good), 4096, A + 4, _lib.BF16, 1, pp, None) == _lib.ERR_ALIGN
    assert ds(ctypes.byref(good), 4096, B + 0x20000 - 64, _lib.BF16, 1, pp, None) == _lib.ERR_OVERLAP
    two = (_lib.Segments * 2)(_seg(A, A + 0x10000, A + 0x20000), _seg(A + 0x30000, A + 0x40000, A + 0x50000))
    assert rs(two, 0, 4096, ctypes.byref(good), pp, None) == _lib.ERR_PARAM
    assert rs(two, 9, 4096, ctypes.byref(good), pp, None) == _lib.ERR_PARAM
    assert rs(None, 2, 4096, ctypes.byref(good), pp, None) == _lib.ERR_NULL
    assert rs(two, 2, 4096, None, pp, None) == _lib.ERR_NULL
    assert rs(two, 2, -5, ctypes.byref(good), pp, None) == _lib.ERR_SIZE
    assert rs(two, 2, 4096, ctypes.byref(_seg(B + 4, B + 0x10000, B + 0x20000)), pp, None) == _lib.ERR_ALIGN
    assert rs(two, 2, 4096, ctypes.byref(_seg(A + 0x30000 + 512, B + 0x10000, B + 0x20000)), pp, None) == _lib.ERR_OVERLAP
    assert rs(two, 2, 4096, ctypes.byref(_seg(B, B + 0x10000, A + 0x40000)), pp, None) == _lib.ERR_OVERLAP


def test_tensor_core_encoder_argument_errors(L):
    """fwht = 2 is an encoder option: contiguous BF16 compress only (plain or segments); the
    other producers reject it before any launch, the decoders accept it as fwht = 1."""
    p2 = ctypes.byref(_lib.Params(16, 256, 2))
    assert L.fp4q_roundtrip(A, 4096, B, p2, None) == _lib.ERR_PARAM
    assert L.fp4q_roundtrip_f32(A, 4096, B, p2, None) == _lib.ERR_PARAM
    assert L.fp4q_compress_2d(A, 4, 512, 1024, B, p2, None) == _lib.ERR_PARAM
    assert L.fp4q_roundtrip_2d(A, 4, 512, 1024, B, 1024, p2, None) == _lib.ERR_PARAM
    assert L.fp4q_compress(A, 4096, None, ctypes.byref(_lib.Params(32, 256, 2, 1)), None) == _lib.ERR_NULL
    # decoders: fwht = 2 passes the parameter check (these calls then stop at a host check)
    assert L.fp4q_decompress_accumulate(A, 4096, B + 4, _lib.BF16, 1, p2, None) == _lib.ERR_ALIGN
    assert L.fp4q_decompress_accumulate_2d(A, 4, 512, B + 4, 1024, _lib.BF16, 1, p2, None) == _lib.ERR_ALIGN
