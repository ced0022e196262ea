"""CPU oracle of the FP4 communication codec (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import this package. It wraps ``fp4q_oracle.c`` (plain scalar C, built with
``-ffp-contract=off``) through ctypes; numpy arrays in, numpy arrays out. It shares no code
with the CUDA library and never imports it.
"""
from __future__ import annotations

import ctypes
import hashlib
import os
import platform
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp4q_oracle.c")
_LIB = os.path.join(_HERE, f"liboracle_{platform.machine()}.so")
_lock = threading.Lock()
_lib = None

BLOCK = 256


def build(force: bool = False) -> str:
    """Compile the oracle into a shared library next to its source and return its path."""
    base = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]
    # up to date when built from exactly this source (a content hash, not file times)
    with open(_SRC, "rb") as fh:
        digest = hashlib.sha256(" ".join(base).encode() + b"\0" + fh.read()).hexdigest()
    stamp = _LIB + ".sha256"
    if not force and os.path.exists(_LIB) and os.path.exists(stamp):
        with open(stamp) as fh:
            if fh.read().strip() == digest:
                return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    try:
        subprocess.run(base + ["-fopenmp", _SRC, "-lm", "-o", tmp], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base + [_SRC, "-lm", "-o", tmp], check=True, capture_output=True)
    os.replace(tmp, _LIB)
    with open(stamp + f".tmp{os.getpid()}", "w") as fh:
        fh.write(digest)
    os.replace(stamp + f".tmp{os.getpid()}", stamp)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        sig = {
            "oracle_bf16_to_f32": (ctypes.c_float, [ctypes.c_uint16]),
            "oracle_f32_to_bf16": (ctypes.c_uint16, [ctypes.c_float]),
            "oracle_e4m3_decode": (ctypes.c_float, [ctypes.c_uint8]),
            "oracle_e4m3_encode": (ctypes.c_uint8, [ctypes.c_float]),
            "oracle_e2m1_decode": (ctypes.c_float, [ctypes.c_uint8]),
            "oracle_e2m1_encode": (ctypes.c_uint8, [ctypes.c_float]),
            "oracle_fwht256": (None, [P]),
            "oracle_payload_bytes": (I64, [I64, I, I]),
            "oracle_gscale_offset": (I64, [I64, I, I]),
            "oracle_bscale_offset": (I64, [I64, I, I]),
            "oracle_e8m0_scale": (ctypes.c_uint8, [ctypes.c_float]),
            "oracle_e8m0_decode": (ctypes.c_float, [ctypes.c_uint8]),
            "oracle_e8m0_scale_array": (None, [P, P, I64]),
            "oracle_max_threads": (I, []),
            "oracle_set_threads": (None, [I]),
            "oracle_compress": (I, [P, I64, P, I, I, I, P]),
            "oracle_decompress_accumulate": (I, [P, I64, P, I, I, I, I, I]),
            "oracle_roundtrip": (I, [P, I64, P, I, I, I]),
            "oracle_compress_f32": (I, [P, I64, P, I, I, I, P]),
            "oracle_roundtrip_f32": (I, [P, I64, P, I, I, I]),
            "oracle_reduce_requantize": (I, [P, I, I64, P, I, I, P]),
            "oracle_e4m3_encode_array": (None, [P, P, I64]),
            "oracle_e2m1_encode_array": (None, [P, P, I64]),
            "oracle_bf16_round_array": (None, [P, P, I64]),
            "oracle_fwht256_array": (None, [P, I64, I]),
            "oracle_ifwht256": (None, [P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


# ------------------------------------------------------------------ scalar / array pins

def set_threads(t: int) -> None:
    _load().oracle_set_threads(int(t))


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def e4m3_encode(r) -> np.ndarray:
    r = _c(r, np.float32).ravel()
    out = np.empty(r.size, np.uint8)
    _load().oracle_e4m3_encode_array(_ptr(r), _ptr(out), r.size)
    return out


def e4m3_decode(codes) -> np.ndarray:
    lib = _load()
    return np.array([lib.oracle_e4m3_decode(int(c)) for c in np.asarray(codes).ravel()], np.float32)


def e2m1_encode(q) -> np.ndarray:
    q = _c(q, np.float32).ravel()
    out = np.empty(q.size, np.uint8)
    _load().oracle_e2m1_encode_array(_ptr(q), _ptr(out), q.size)
    return out


def e2m1_decode(codes) -> np.ndarray:
    lib = _load()
    return np.array([lib.oracle_e2m1_decode(int(c)) for c in np.asarray(codes).ravel()], np.float32)


def bf16_round(f) -> np.ndarray:
    """float32 -> bfloat16 bit patterns (uint16), round to nearest even."""
    f = _c(f, np.float32).ravel()
    out = np.empty(f.size, np.uint16)
    _load().oracle_bf16_round_array(_ptr(f), _ptr(out), f.size)
    return out


def bf16_to_f32(h) -> np.ndarray:
    h = _c(h, np.uint16)
    return (h.astype(np.uint32) << 16).view(np.float32)


def fwht256(v, inverse: bool = False) -> np.ndarray:
    """Orthonormal FWHT of each consecutive 256-block of v (float32); returns a copy.
    inverse=True applies the decode's mirror stage order (h = 128 ... 1)."""
    v = np.array(v, dtype=np.float32, copy=True).ravel()
    assert v.size % BLOCK == 0
    _load().oracle_fwht256_array(_ptr(v), v.size // BLOCK, int(bool(inverse)))
    return v


# ------------------------------------------------------------------ codec
#
# scales = "dual": E4M3 group scale x FP32 block scale (group 16 or 32, default 16);
# scales = "e8m0": microscaled variant, power-of-two E8M0 scale per group of 32 and no block
# scale (group 32, the default for it).

SCALES = {"dual": 0, "e8m0": 1}


def _fmt(group, scales):
    if scales not in SCALES:
        raise ValueError(f"scales must be one of {sorted(SCALES)}")
    mx = SCALES[scales]
    return (int(group) if group is not None else (32 if mx else 16)), mx


def e8m0_scale(amax) -> np.ndarray:
    a = np.ascontiguousarray(amax, dtype=np.float32).ravel()
    out = np.empty(a.size, np.uint8)
    _load().oracle_e8m0_scale_array(_ptr(a), _ptr(out), a.size)
    return out


def e8m0_decode(codes) -> np.ndarray:
    return np.array([_load().oracle_e8m0_decode(int(c)) for c in np.ravel(codes)], np.float32)


def payload_bytes(n: int, group: int | None = None, scales: str = "dual") -> int:
    G, mx = _fmt(group, scales)
    return int(_load().oracle_payload_bytes(int(n), G, mx))


def gscale_offset(n: int, group: int | None = None, scales: str = "dual") -> int:
    G, mx = _fmt(group, scales)
    return int(_load().oracle_gscale_offset(int(n), G, mx))


def bscale_offset(n: int, group: int | None = None, scales: str = "dual") -> int:
    G, mx = _fmt(group, scales)
    return int(_load().oracle_bscale_offset(int(n), G, mx))


def compress(x_bf16: np.ndarray, group: int | None = None, fwht: int = 1, want_q: bool = False,
             scales: str = "dual"):
    """x_bf16: uint16 bit patterns. Returns the payload (uint8) and, if want_q, every q."""
    G, mx = _fmt(group, scales)
    x = _c(x_bf16, np.uint16).ravel()
    n = x.size
    nbytes = payload_bytes(n, G, scales)
    if nbytes == 0:
        raise ValueError(f"invalid n={n} or group={G} for scales={scales}")
    out = np.zeros(nbytes, np.uint8)
    q = np.empty(n, np.float32) if want_q else None
    rc = _load().oracle_compress(_ptr(x), n, _ptr(out), G, fwht, mx, _ptr(q) if want_q else None)
    if rc != 0:
        raise ValueError(f"oracle_compress failed ({rc})")
    return (out, q) if want_q else out


def compress_f32(x: np.ndarray, group: int | None = None, fwht: int = 1, want_q: bool = False,
                 scales: str = "dual"):
    """FP32 input (used as it is): returns the payload (uint8) and, if want_q, every q."""
    G, mx = _fmt(group, scales)
    x = _c(x, np.float32).ravel()
    n = x.size
    nbytes = payload_bytes(n, G, scales)
    if nbytes == 0:
        raise ValueError(f"invalid n={n} or group={G} for scales={scales}")
    out = np.zeros(nbytes, np.uint8)
    q = np.empty(n, np.float32) if want_q else None
    rc = _load().oracle_compress_f32(_ptr(x), n, _ptr(out), G, fwht, mx, _ptr(q) if want_q else None)
    if rc != 0:
        raise ValueError(f"oracle_compress_f32 failed ({rc})")
    return (out, q) if want_q else out


def roundtrip_f32(x: np.ndarray, group: int | None = None, fwht: int = 1, scales: str = "dual") -> np.ndarray:
    """FP32 in, FP32 out: decode(compress_f32(x)) without a BF16 rounding of the result."""
    G, mx = _fmt(group, scales)
    x = _c(x, np.float32).ravel()
    y = np.empty_like(x)
    rc = _load().oracle_roundtrip_f32(_ptr(x), x.size, _ptr(y), G, fwht, mx)
    if rc != 0:
        raise ValueError(f"oracle_roundtrip_f32 failed ({rc})")
    return y


def decompress_accumulate(payload: np.ndarray, n: int, dst: np.ndarray, beta: int,
                          group: int | None = None, fwht: int = 1, scales: str = "dual") -> np.ndarray:
    """dst: uint16 (bfloat16 bits) or float32 array of n elements, updated in place."""
    G, mx = _fmt(group, scales)
    p = _c(payload, np.uint8)
    if dst.dtype == np.uint16:
        dtype = 0
    elif dst.dtype == np.float32:
        dtype = 1
    else:
        raise TypeError("dst must be uint16 (bfloat16 bits) or float32")
    assert dst.flags.c_contiguous and dst.size == n
    rc = _load().oracle_decompress_accumulate(_ptr(p), int(n), _ptr(dst), dtype, int(beta),
                                              G, fwht, mx)
    if rc != 0:
        raise ValueError(f"oracle_decompress_accumulate failed ({rc})")
    return dst


def roundtrip(x_bf16: np.ndarray, group: int | None = None, fwht: int = 1,
              scales: str = "dual") -> np.ndarray:
    G, mx = _fmt(group, scales)
    x = _c(x_bf16, np.uint16).ravel()
    y = np.empty_like(x)
    rc = _load().oracle_roundtrip(_ptr(x), x.size, _ptr(y), G, fwht, mx)
    if rc != 0:
        raise ValueError(f"oracle_roundtrip failed ({rc})")
    return y


def reduce_requantize(payloads, n: int, group: int | None = None, want_q: bool = False,
                      scales: str = "dual"):
    G, mx = _fmt(group, scales)
    ps = [_c(p, np.uint8) for p in payloads]
    R = len(ps)
    arr = (ctypes.c_void_p * R)(*[_ptr(p) for p in ps])
    out = np.zeros(payload_bytes(n, G, scales), np.uint8)
    q = np.empty(n, np.float32) if want_q else None
    rc = _load().oracle_reduce_requantize(ctypes.cast(arr, ctypes.c_void_p), R, int(n), _ptr(out),
                                          G, mx, _ptr(q) if want_q else None)
    if rc != 0:
        raise ValueError(f"oracle_reduce_requantize failed ({rc})")
    return (out, q) if want_q else out


def split_payload(payload: np.ndarray, n: int, group: int | None = None, scales: str = "dual"):
    """(codes, group scales, block scales) views of a payload of n elements, each covering
    ceil(n/256) blocks (the block scales are empty for scales="e8m0")."""
    G, mx = _fmt(group, scales)
    m = -(-n // BLOCK) * BLOCK          # a last partial block is zero-padded to 256 elements
    g0, b0 = gscale_offset(n, G, scales), bscale_offset(n, G, scales)
    codes = payload[:m // 2]
    gsc = payload[g0:g0 + m // G]
    bsc = payload[b0:b0 + (0 if mx else 4 * (m // BLOCK))].view(np.float32)
    return codes, gsc, bsc
