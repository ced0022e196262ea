"""GB300-native FP4 communication compression (FP4Quant's data-parallel hot path).

Torch-facing wrappers of the C ABI in ``include/fp4q.h``; the names follow the ABI. Every
function takes CUDA tensors, runs on the current torch stream (or the ``stream`` given)
and returns without synchronising. The codec itself runs only in the sm_103a kernels of
``csrc/fp4q.cu``; there is no CPU fallback (a missing library raises ``RuntimeError``).

    payload = compress(x)                                  # x: bfloat16 or float32, any numel
    decompress_accumulate(payload, x.numel(), dst, beta=1) # dst += decode(payload)
    y = roundtrip(x)                                       # fused fake-quantisation
    out = reduce_requantize([p0, p1, p2, p3], n)           # emulated 4-rank reduce
    p = compress(x, scales="e8m0")                         # microscaled variant (group 32)

``scales="dual"`` (default) is the E4M3 group scale x FP32 block scale format (group 16 or
32); ``scales="e8m0"`` the power-of-two scale per group of 32 with no block scale. Every
call on one payload must use the same group, fwht and scales.

Every buffer a caller passes in is checked on the host before anything is launched (the C
ABI sees only pointers and cannot know how long a buffer is): payloads must be contiguous
uint8 CUDA tensors of at least ``payload_bytes(n, ...)`` bytes on the data tensor's device,
data tensors CUDA tensors of the right dtype and size; a wrong buffer raises ``ValueError``.

A return without an exception means the kernels were launched, not that they completed: a
kernel whose bounded wait on a copy gives up returns early and sets the device fault word.
``check=True`` synchronises the device after the call and raises ``Fp4qFault`` if that word
is set (the word is cleared when read this way).

Method: "FP4Quant: Efficient 4-Bit Communication Compression for Model-Parallel LLM
Training" (abstract: micro-grouped dual-scale FP4 quantization, warp-cooperative FP4
packing, hybrid two-level FWHT).
"""
from __future__ import annotations

import ctypes

from . import _lib
from ._lib import BF16, F32, Fp4qError, build  # noqa: F401

__all__ = ["payload_bytes", "gscale_offset", "bscale_offset", "compress",
           "decompress_accumulate", "roundtrip", "reduce_requantize", "segment_bytes",
           "compress_segments", "decompress_accumulate_segments", "reduce_requantize_segments",
           "build", "Fp4qError", "Fp4qFault", "library_path", "fault_flags"]


class Fp4qFault(RuntimeError):
    """The device fault word was set: a kernel gave up a bounded wait and returned early,
    so the outputs of the calls since the word was last cleared are incomplete."""

    def __init__(self, flags: int):
        super().__init__(f"fp4q device fault word 0x{flags:x}: a kernel gave up waiting for a copy "
                         "and returned early (outputs incomplete)")
        self.flags = flags


def library_path() -> str:
    return _lib.LIB_PATH


def _stream(stream, device):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _dev(t, name):
    if not getattr(t, "is_cuda", False):
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _buffer(t, name, nbytes, device):
    """A payload buffer: a contiguous uint8 CUDA tensor on `device` of at least nbytes bytes
    (the kernels read or write exactly payload_bytes(n) bytes from its start)."""
    import torch
    if not getattr(t, "is_cuda", False):
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != torch.uint8:
        raise ValueError(f"{name} must be uint8 (got {t.dtype})")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, the data tensor on {device}")
    if t.numel() < nbytes:
        raise ValueError(f"{name} holds {t.numel()} bytes, the payload needs {nbytes}")
    return ctypes.c_void_p(t.data_ptr())


def _need_bytes(n, group, fwht, scales) -> int:
    nb = payload_bytes(n, group, fwht, scales)
    if nb == 0:
        raise ValueError(f"invalid size {n} or parameters (group={group}, fwht={fwht}, scales={scales!r})")
    return nb


def _cuda_data(t, name):
    if not getattr(t, "is_cuda", False):
        raise ValueError(f"{name} must be a CUDA tensor")


def _fault_check(device, check):
    if not check:
        return
    import torch
    torch.cuda.synchronize(device)
    with torch.cuda.device(device):
        flags = fault_flags(clear=True)
    if flags:
        raise Fp4qFault(flags)


def _strided_2d(t) -> bool:
    """A 2-D CUDA view with unit column stride and a larger row stride (a slice of a wider
    matrix): handled by the *_2d entry points without a copy."""
    return t.is_cuda and t.dim() == 2 and not t.is_contiguous() and t.stride(1) == 1 and t.size(0) > 1


def payload_bytes(n: int, group: int | None = None, fwht: int = 1, scales: str = "dual") -> int:
    p = _lib.params(group, fwht, scales=scales)
    return int(_lib.lib().fp4q_payload_bytes(int(n), ctypes.byref(p)))


def gscale_offset(n: int, group: int | None = None, fwht: int = 1, scales: str = "dual") -> int:
    p = _lib.params(group, fwht, scales=scales)
    return int(_lib.lib().fp4q_gscale_offset(int(n), ctypes.byref(p)))


def bscale_offset(n: int, group: int | None = None, fwht: int = 1, scales: str = "dual") -> int:
    p = _lib.params(group, fwht, scales=scales)
    return int(_lib.lib().fp4q_bscale_offset(int(n), ctypes.byref(p)))


def compress(x, payload=None, group: int | None = None, fwht: int = 1, stream=None, scales: str = "dual",
             check: bool = False):
    """bfloat16 or float32 CUDA tensor -> uint8 payload tensor (allocated by torch if not given)."""
    import torch
    _cuda_data(x, "x")
    if x.dtype == torch.bfloat16:
        fn, name = _lib.lib().fp4q_compress, "fp4q_compress"
    elif x.dtype == torch.float32:
        fn, name = _lib.lib().fp4q_compress_f32, "fp4q_compress_f32"
    else:
        raise TypeError("x must be bfloat16 or float32")
    n = x.numel()
    if _strided_2d(x) and x.dtype != torch.bfloat16:
        raise ValueError("strided 2-D input must be bfloat16")
    nb = _need_bytes(n, group, fwht, scales)
    if payload is None:
        payload = torch.empty(nb, dtype=torch.uint8, device=x.device)
    pp = _buffer(payload, "payload", nb, x.device)
    p = _lib.params(group, fwht, scales=scales)
    if _strided_2d(x):
        st = _lib.lib().fp4q_compress_2d(ctypes.c_void_p(x.data_ptr()), x.size(0), x.size(1), x.stride(0),
                                         pp, ctypes.byref(p), _stream(stream, x.device))
        _lib.check("fp4q_compress_2d", st)
    else:
        st = fn(_dev(x, "x"), n, pp, ctypes.byref(p), _stream(stream, x.device))
        _lib.check(name, st)
    _fault_check(x.device, check)
    return payload


def decompress_accumulate(payload, n: int, dst, beta: int = 1, group: int | None = None, fwht: int = 1,
                          stream=None, scales: str = "dual", check: bool = False):
    """dst (bfloat16 or float32 CUDA tensor of n elements) = beta ? dst + x^ : x^."""
    import torch
    _cuda_data(dst, "dst")
    if dst.dtype == torch.bfloat16:
        dt = BF16
    elif dst.dtype == torch.float32:
        dt = F32
    else:
        raise TypeError("dst must be bfloat16 or float32")
    if dst.numel() != n:
        raise ValueError("dst must have n elements")
    pp = _buffer(payload, "payload", _need_bytes(n, group, fwht, scales), dst.device)
    p = _lib.params(group, fwht, scales=scales)
    if _strided_2d(dst):
        st = _lib.lib().fp4q_decompress_accumulate_2d(pp, dst.size(0), dst.size(1),
                                                      ctypes.c_void_p(dst.data_ptr()), dst.stride(0), dt,
                                                      int(beta), ctypes.byref(p), _stream(stream, dst.device))
        _lib.check("fp4q_decompress_accumulate_2d", st)
    else:
        st = _lib.lib().fp4q_decompress_accumulate(pp, int(n), _dev(dst, "dst"), dt, int(beta), ctypes.byref(p),
                                                   _stream(stream, dst.device))
        _lib.check("fp4q_decompress_accumulate", st)
    _fault_check(dst.device, check)
    return dst


def roundtrip(x, y=None, group: int | None = None, fwht: int = 1, stream=None, scales: str = "dual",
              check: bool = False):
    """y = decode(compress(x)) in one kernel, no payload written; bfloat16 in and out, or
    float32 in and out (no bfloat16 rounding)."""
    import torch
    _cuda_data(x, "x")
    if x.dtype == torch.bfloat16:
        fn, name = _lib.lib().fp4q_roundtrip, "fp4q_roundtrip"
    elif x.dtype == torch.float32:
        fn, name = _lib.lib().fp4q_roundtrip_f32, "fp4q_roundtrip_f32"
    else:
        raise TypeError("x must be bfloat16 or float32")
    if y is None:
        y = torch.empty(x.shape, dtype=x.dtype, device=x.device)
    _cuda_data(y, "y")
    if y.dtype != x.dtype or y.numel() != x.numel():
        raise ValueError("y must match x in dtype and size")
    if y.device != x.device:
        raise ValueError(f"y is on {y.device}, x on {x.device}")
    p = _lib.params(group, fwht, scales=scales)
    if _strided_2d(x) or _strided_2d(y):
        if x.dtype != torch.bfloat16 or x.dim() != 2 or y.shape != x.shape:
            raise ValueError("strided 2-D roundtrip needs bfloat16 x and y of the same 2-D shape")
        st = _lib.lib().fp4q_roundtrip_2d(ctypes.c_void_p(x.data_ptr()), x.size(0), x.size(1), x.stride(0),
                                          ctypes.c_void_p(y.data_ptr()), y.stride(0), ctypes.byref(p),
                                          _stream(stream, x.device))
        _lib.check("fp4q_roundtrip_2d", st)
    else:
        st = fn(_dev(x, "x"), x.numel(), _dev(y, "y"), ctypes.byref(p), _stream(stream, x.device))
        _lib.check(name, st)
    _fault_check(x.device, check)
    return y


def reduce_requantize(payloads, n: int, out=None, group: int | None = None, fwht: int = 1, stream=None,
                      scales: str = "dual", check: bool = False):
    """R payloads (uint8 CUDA tensors, same n and params) -> requantised sum payload."""
    import torch
    R = len(payloads)
    if R < 1:
        raise ValueError("reduce_requantize needs at least one payload")
    nb = _need_bytes(n, group, fwht, scales)
    _cuda_data(payloads[0], "payloads[0]")
    device = payloads[0].device
    ptrs = (ctypes.c_void_p * R)(*[_buffer(p, f"payloads[{i}]", nb, device).value for i, p in enumerate(payloads)])
    if out is None:
        out = torch.empty(nb, dtype=torch.uint8, device=device)
    po = _buffer(out, "out", nb, device)
    p = _lib.params(group, fwht, scales=scales)
    st = _lib.lib().fp4q_reduce_requantize(ctypes.cast(ptrs, ctypes.c_void_p), R, int(n), po, ctypes.byref(p),
                                           _stream(stream, device))
    _lib.check("fp4q_reduce_requantize", st)
    _fault_check(device, check)
    return out


# ------------------------------------------------------------------ payloads as separate segments

def segment_bytes(n: int, group: int | None = None, fwht: int = 1, scales: str = "dual"):
    """(codes, group scales, block scales) bytes of a payload of n elements placed as three
    separate segments (block scales 0 for E8M0 scales)."""
    p = _lib.params(group, fwht, scales=scales)
    c, g, b = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    _lib.check("fp4q_segment_bytes", _lib.lib().fp4q_segment_bytes(int(n), ctypes.byref(p), ctypes.byref(c),
                                                                    ctypes.byref(g), ctypes.byref(b)))
    return int(c.value), int(g.value), int(b.value)


def _segments(segs, n, group, fwht, scales, device, name):
    """fp4q_segments of a (codes, gscales, bscales) tuple of uint8 CUDA tensors, each checked
    to be large enough (bscales may be None for E8M0 scales)."""
    if len(segs) != 3:
        raise ValueError(f"{name} must be (codes, gscales, bscales)")
    sizes = segment_bytes(n, group, fwht, scales)
    ptrs = []
    for t, need, part in zip(segs, sizes, ("codes", "gscales", "bscales")):
        if need == 0 and t is None:
            ptrs.append(None)
            continue
        ptrs.append(_buffer(t, f"{name}.{part}", need, device).value)
    return _lib.Segments(*ptrs)


def compress_segments(x, segs, group: int | None = None, fwht: int = 1, stream=None, scales: str = "dual",
                      check: bool = False):
    """compress(x) writing the payload into three separate uint8 buffers (codes, gscales,
    bscales); bit-identical to the contiguous payload's segments."""
    import torch
    _cuda_data(x, "x")
    if x.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("x must be bfloat16 or float32")
    sg = _segments(segs, x.numel(), group, fwht, scales, x.device, "segs")
    p = _lib.params(group, fwht, scales=scales)
    st = _lib.lib().fp4q_compress_segments(_dev(x, "x"), BF16 if x.dtype == torch.bfloat16 else F32, x.numel(),
                                           ctypes.byref(sg), ctypes.byref(p), _stream(stream, x.device))
    _lib.check("fp4q_compress_segments", st)
    _fault_check(x.device, check)
    return segs


def decompress_accumulate_segments(segs, n: int, dst, beta: int = 1, group: int | None = None, fwht: int = 1,
                                   stream=None, scales: str = "dual", check: bool = False):
    """decompress_accumulate reading the payload from three separate segments."""
    import torch
    _cuda_data(dst, "dst")
    if dst.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("dst must be bfloat16 or float32")
    if dst.numel() != n:
        raise ValueError("dst must have n elements")
    sg = _segments(segs, n, group, fwht, scales, dst.device, "segs")
    p = _lib.params(group, fwht, scales=scales)
    st = _lib.lib().fp4q_decompress_accumulate_segments(ctypes.byref(sg), int(n), _dev(dst, "dst"),
                                                        BF16 if dst.dtype == torch.bfloat16 else F32, int(beta),
                                                        ctypes.byref(p), _stream(stream, dst.device))
    _lib.check("fp4q_decompress_accumulate_segments", st)
    _fault_check(dst.device, check)
    return dst


def reduce_requantize_segments(ins, n: int, out, group: int | None = None, fwht: int = 1, stream=None,
                               scales: str = "dual", check: bool = False):
    """reduce_requantize over R payloads given as segment tuples, into the segments of out."""
    R = len(ins)
    if R < 1:
        raise ValueError("reduce_requantize_segments needs at least one input")
    _cuda_data(out[0], "out.codes")
    device = out[0].device
    arr = (_lib.Segments * R)(*[_segments(sg, n, group, fwht, scales, device, f"ins[{i}]") for i, sg in enumerate(ins)])
    so = _segments(out, n, group, fwht, scales, device, "out")
    p = _lib.params(group, fwht, scales=scales)
    st = _lib.lib().fp4q_reduce_requantize_segments(arr, R, int(n), ctypes.byref(so), ctypes.byref(p),
                                                    _stream(stream, device))
    _lib.check("fp4q_reduce_requantize_segments", st)
    _fault_check(device, check)
    return out


def fault_flags(clear: bool = False) -> int:
    """The device fault word (0 = every bounded wait completed); synchronises the device."""
    v = ctypes.c_uint32(0)
    _lib.check("fp4q_fault_flags", _lib.lib().fp4q_fault_flags(ctypes.byref(v), int(bool(clear))))
    return int(v.value)
