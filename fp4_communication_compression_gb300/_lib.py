"""ctypes binding of the fp4q C ABI (include/fp4q.h): argument marshalling only.

Every step of the codec runs in the CUDA kernels of ``csrc/fp4q.cu``; this module only
turns torch tensors into device pointers and the current torch stream into a
``cudaStream_t``. There is no CPU path: if the library has not been built, every call
raises ``RuntimeError``.
"""
from __future__ import annotations

import ctypes
import hashlib
import os
import platform
import subprocess
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_PKG)
_SRC = os.path.join(_PKG, "csrc", "fp4q.cu")
_HDR = os.path.join(_ROOT, "include", "fp4q.h")
LIB_PATH = os.path.join(_PKG, f"libfp4q_{platform.machine()}.so")

NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-fmad=false", "-split-compile=0",
              "-std=c++17", "-Xcompiler", "-fPIC", "-shared"]

# status codes (fp4q_status)
OK, ERR_NULL, ERR_SIZE, ERR_ALIGN, ERR_PARAM, ERR_OVERLAP, ERR_CUDA = range(7)
BF16, F32 = 0, 1

# exported symbols of the library, in the order include/fp4q.h declares them
EXPORTS = ["fp4q_payload_bytes", "fp4q_gscale_offset", "fp4q_bscale_offset", "fp4q_compress",
           "fp4q_compress_f32", "fp4q_decompress_accumulate", "fp4q_roundtrip", "fp4q_roundtrip_f32",
           "fp4q_compress_2d", "fp4q_decompress_accumulate_2d", "fp4q_roundtrip_2d",
           "fp4q_reduce_requantize", "fp4q_segment_bytes", "fp4q_compress_segments",
           "fp4q_decompress_accumulate_segments", "fp4q_reduce_requantize_segments",
           "fp4q_fault_flags", "fp4q_selftest_wait_timeout",
           "fp4q_status_string", "fp4q_version"]


class Fp4qError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn} failed: status {status} ({msg})")
        self.status = status


SCALES = {"dual": 0, "e8m0": 1}   # fp4q_params.scales: FP4Q_SCALES_DUAL, FP4Q_SCALES_E8M0


class Params(ctypes.Structure):
    _fields_ = [("group", ctypes.c_int32), ("block", ctypes.c_int32), ("fwht", ctypes.c_int32),
                ("scales", ctypes.c_int32)]


class Segments(ctypes.Structure):
    """fp4q_segments: device pointers of a payload's codes, group scales and block scales."""
    _fields_ = [("codes", ctypes.c_void_p), ("gscales", ctypes.c_void_p), ("bscales", ctypes.c_void_p)]


def build(force: bool = False, nvcc: str = "nvcc") -> str:
    """Compile csrc/fp4q.cu for sm_103a into the package directory; returns the .so path."""
    # up to date when the library was built from exactly these sources and flags (a content
    # hash, not file times: a copied tree keeps neither order nor clock of the original)
    csrc = os.path.dirname(_SRC)
    deps = [_HDR] + sorted(os.path.join(csrc, f) for f in os.listdir(csrc) if f.endswith((".cu", ".cuh")))
    h = hashlib.sha256(" ".join([nvcc, *NVCC_FLAGS]).encode())
    for f in deps:
        with open(f, "rb") as fh:
            h.update(os.path.basename(f).encode() + b"\0" + fh.read())
    stamp = LIB_PATH + ".sha256"
    if not force and os.path.exists(LIB_PATH) and os.path.exists(stamp):
        with open(stamp) as fh:
            if fh.read().strip() == h.hexdigest():
                return LIB_PATH
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = [nvcc, *NVCC_FLAGS, "-I", os.path.dirname(_HDR), _SRC, "-o", tmp]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + res.stdout + res.stderr)
    os.replace(tmp, LIB_PATH)
    with open(stamp + f".tmp{os.getpid()}", "w") as fh:
        fh.write(h.hexdigest())
    os.replace(stamp + f".tmp{os.getpid()}", stamp)
    return LIB_PATH


_lock = threading.Lock()
_lib = None


def lib():
    """The loaded library (raises RuntimeError if it was never built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"fp4q CUDA library not built ({LIB_PATH} missing); "
                               "run `python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        P, I64, I32, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t
        pp = ctypes.POINTER(Params)
        ps = ctypes.POINTER(Segments)
        SZP = ctypes.POINTER(ctypes.c_size_t)
        sig = {
            "fp4q_payload_bytes": (SZ, [I64, pp]),
            "fp4q_gscale_offset": (SZ, [I64, pp]),
            "fp4q_bscale_offset": (SZ, [I64, pp]),
            "fp4q_compress": (ctypes.c_int, [P, I64, P, pp, P]),
            "fp4q_compress_f32": (ctypes.c_int, [P, I64, P, pp, P]),
            "fp4q_roundtrip_f32": (ctypes.c_int, [P, I64, P, pp, P]),
            "fp4q_compress_2d": (ctypes.c_int, [P, I64, I64, I64, P, pp, P]),
            "fp4q_decompress_accumulate_2d": (ctypes.c_int, [P, I64, I64, P, I64, ctypes.c_int, I32, pp, P]),
            "fp4q_roundtrip_2d": (ctypes.c_int, [P, I64, I64, I64, P, I64, pp, P]),
            "fp4q_decompress_accumulate": (ctypes.c_int, [P, I64, P, ctypes.c_int, I32, pp, P]),
            "fp4q_roundtrip": (ctypes.c_int, [P, I64, P, pp, P]),
            "fp4q_reduce_requantize": (ctypes.c_int, [P, I32, I64, P, pp, P]),
            "fp4q_segment_bytes": (ctypes.c_int, [I64, pp, SZP, SZP, SZP]),
            "fp4q_compress_segments": (ctypes.c_int, [P, ctypes.c_int, I64, ps, pp, P]),
            "fp4q_decompress_accumulate_segments": (ctypes.c_int, [ps, I64, P, ctypes.c_int, I32, pp, P]),
            "fp4q_reduce_requantize_segments": (ctypes.c_int, [ps, I32, I64, ps, pp, P]),
            "fp4q_fault_flags": (ctypes.c_int, [ctypes.POINTER(ctypes.c_uint32), I32]),
            "fp4q_selftest_wait_timeout": (ctypes.c_int, [ctypes.c_uint32, P]),
            "fp4q_status_string": (ctypes.c_char_p, [ctypes.c_int]),
            "fp4q_version": (I32, []),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
        return L


def params(group: int | None = None, fwht: int = 1, block: int = 256, scales: str = "dual") -> Params:
    """fp4q_params; group None means 16 for dual scales and 32 for E8M0 scales. An unknown
    scales name maps to -1, which the library rejects (FP4Q_ERR_PARAM)."""
    sc = SCALES.get(scales, -1)
    if group is None:
        group = 32 if sc == 1 else 16
    return Params(int(group), int(block), int(fwht), sc)


def status_string(status: int) -> str:
    return lib().fp4q_status_string(status).decode()


def check(fn: str, status: int) -> None:
    if status != OK:
        raise Fp4qError(fn, status, status_string(status))
