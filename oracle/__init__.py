"""CPU oracle for the symmetric-window collectives -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s cpu_baseline /
``--impl reference`` leg may import this package.  The product path (the CUDA
library and its Python binding) never imports it, and the two share no code.

The arithmetic lives in ``oracle.c`` (plain C, IEEE binary32 in source order,
built with ``-O2 -ffp-contract=off -fno-fast-math``); this module only builds
it with gcc, loads it with ctypes and marshals numpy arrays.

Parity status: every function is pinned by ``tests/test_oracle.py`` to facts
that do not come from this code.  ``rolling_le`` (the GIN reference page names a
rolling comparison without printing it) is pinned to RFC 1982 serial number
arithmetic and to the page's x <= x+1 property; the reading taken where the RFC
is undefined is documented in ``oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_CFLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-std=c11",
           "-Wall", "-Wextra", "-pthread"]
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc; host arch only)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *_CFLAGS, _SRC, "-o", tmp], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        sz = ctypes.c_size_t
        i32 = ctypes.c_int
        u64 = ctypes.c_uint64
        lib.oracle_allreduce_sum_f32.argtypes = [i32, sz, P, sz, P]
        lib.oracle_allreduce_sum_f32.restype = None
        lib.oracle_allreduce_sum_bf16.argtypes = [i32, sz, P, sz, P]
        lib.oracle_allreduce_sum_bf16.restype = None
        lib.oracle_allreduce_sum_mt.argtypes = [i32, i32, sz, P, sz, P, i32]
        lib.oracle_allreduce_sum_mt.restype = i32
        lib.oracle_f32_to_bf16_rne.argtypes = [ctypes.c_float]
        lib.oracle_f32_to_bf16_rne.restype = ctypes.c_uint16
        lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_f32.restype = ctypes.c_float
        lib.oracle_f32_to_bf16_array.argtypes = [sz, P, P]
        lib.oracle_f32_to_bf16_array.restype = None
        lib.oracle_allgather.argtypes = [i32, sz, P, sz, P]
        lib.oracle_allgather.restype = None
        lib.oracle_put_signal_allgather.argtypes = [i32, sz, sz, sz, P, sz, P, P, P]
        lib.oracle_put_signal_allgather.restype = None
        lib.oracle_prefix_mismatch.argtypes = [sz, sz, sz, u64, P, P]
        lib.oracle_prefix_mismatch.restype = u64
        lib.oracle_rolling_le.argtypes = [u64, u64, i32]
        lib.oracle_rolling_le.restype = i32
        lib.oracle_read_bits.argtypes = [u64, i32]
        lib.oracle_read_bits.restype = u64
        _lib = lib
        return lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _rows(x: np.ndarray, dtype) -> np.ndarray:
    x = np.ascontiguousarray(x)
    if x.dtype != dtype or x.ndim != 2:
        raise TypeError(f"expected a 2-D {np.dtype(dtype).name} array (ranks x elements)")
    return x


def allreduce_sum_f32(x: np.ndarray) -> np.ndarray:
    """x: (R, N) float32 -> y: (N,) float32, summed in rank order 0..R-1."""
    x = _rows(x, np.float32)
    R, n = x.shape
    y = np.empty(n, np.float32)
    if n:
        _load().oracle_allreduce_sum_f32(R, n, _ptr(x), n, _ptr(y))
    return y


def allreduce_sum_bf16(x_bits: np.ndarray) -> np.ndarray:
    """x_bits: (R, N) uint16 bf16 patterns -> (N,) uint16, fp32 accumulate, one RNE rounding."""
    x = _rows(x_bits, np.uint16)
    R, n = x.shape
    y = np.empty(n, np.uint16)
    if n:
        _load().oracle_allreduce_sum_bf16(R, n, _ptr(x), n, _ptr(y))
    return y


def allreduce_sum_mt(x: np.ndarray, nthreads: int) -> tuple[np.ndarray, int]:
    """Threaded driver of the same per-element routine (timing); returns (y, threads used)."""
    x = np.ascontiguousarray(x)
    if x.dtype == np.float32:
        is_bf16 = 0
    elif x.dtype == np.uint16:
        is_bf16 = 1
    else:
        raise TypeError("float32 or uint16 (bf16 bits) expected")
    R, n = x.shape
    y = np.empty(n, x.dtype)
    used = _load().oracle_allreduce_sum_mt(is_bf16, R, n, _ptr(x), n, _ptr(y), int(nthreads))
    return y, int(used)


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    """float32 array -> uint16 bf16 patterns, round to nearest even (NaN -> 0x7FC0)."""
    x = np.ascontiguousarray(x, dtype=np.float32).ravel()
    y = np.empty(x.size, np.uint16)
    if x.size:
        _load().oracle_f32_to_bf16_array(x.size, _ptr(x), _ptr(y))
    return y


def f32_to_bf16_scalar(v: float) -> int:
    return int(_load().oracle_f32_to_bf16_rne(ctypes.c_float(v)))


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    """uint16 bf16 patterns -> float32 (exact widening)."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def allgather(x: np.ndarray) -> np.ndarray:
    """x: (R, S) uint8 -> (R*S,) uint8: the recv buffer every rank holds."""
    x = _rows(x, np.uint8)
    R, S = x.shape
    y = np.empty(R * S, np.uint8)
    if y.size:
        _load().oracle_allgather(R, S, _ptr(x), S, _ptr(y))
    return y


def alltoall(x: np.ndarray) -> np.ndarray:
    """x: (R, R*B) uint8 -> (R, R*B) uint8 with recv[p][q*B:(q+1)*B] = send[q][p*B:(p+1)*B]."""
    x = _rows(x, np.uint8)
    R, RB = x.shape
    if RB % R:
        raise ValueError("each row must hold R equal segments")
    y = np.empty_like(x)
    lib = _load()
    lib.oracle_alltoall.argtypes = [ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_size_t,
                                    ctypes.c_void_p, ctypes.c_size_t]
    lib.oracle_alltoall.restype = None
    if x.size:
        lib.oracle_alltoall(R, RB // R, _ptr(x), RB, _ptr(y), RB)
    return y


def scale_allreduce(a: np.ndarray, alpha) -> tuple[np.ndarray, np.ndarray]:
    """a: (R, N) float32, alpha: R floats -> (s (R, N) = alpha_r * a_r, y (N,) rank-order sum)."""
    a = _rows(a, np.float32)
    R, n = a.shape
    al = np.ascontiguousarray(np.asarray(alpha, np.float32).ravel())
    if al.size != R:
        raise ValueError("one alpha per rank")
    s = np.empty_like(a)
    y = np.empty(n, np.float32)
    lib = _load()
    P, sz = ctypes.c_void_p, ctypes.c_size_t
    lib.oracle_scale_allreduce.argtypes = [ctypes.c_int, sz, P, P, sz, P, sz, P]
    lib.oracle_scale_allreduce.restype = None
    if n:
        lib.oracle_scale_allreduce(R, n, _ptr(al), _ptr(a), n, _ptr(s), n, _ptr(y))
    return s, y


def put_signal_allgather(x: np.ndarray, chunk: int, batch: int):
    """Sequential put+signal model. x: (R, S) uint8.

    Returns (recv (R*S,) uint8, sig (R, R) uint64 indexed [peer, sender], cnt (R,) uint64).
    """
    x = _rows(x, np.uint8)
    R, S = x.shape
    if chunk < 1 or batch < 1:
        raise ValueError("chunk and batch must be >= 1")
    recv = np.empty(R * S, np.uint8)
    sig = np.empty((R, R), np.uint64)
    cnt = np.empty(R, np.uint64)
    _load().oracle_put_signal_allgather(R, S, chunk, batch, _ptr(x), S, _ptr(recv),
                                        _ptr(sig), _ptr(cnt))
    return recv, sig, cnt


def prefix_mismatch(src_q: np.ndarray, seg: np.ndarray, chunk: int, batch: int, k: int) -> int:
    src_q = np.ascontiguousarray(src_q, dtype=np.uint8)
    seg = np.ascontiguousarray(seg, dtype=np.uint8)
    if src_q.size != seg.size:
        raise ValueError("segment and source sizes differ")
    return int(_load().oracle_prefix_mismatch(src_q.size, chunk, batch, k, _ptr(src_q), _ptr(seg)))


def rolling_le(a: int, b: int, bits: int = 64) -> bool:
    """Rolling a <= b on the low `bits` bits (reading and pins in oracle.c)."""
    return bool(_load().oracle_rolling_le(a & (2**64 - 1), b & (2**64 - 1), bits))


def read_bits(v: int, bits: int) -> int:
    return int(_load().oracle_read_bits(v & (2**64 - 1), bits))


# ---------------------------------------------------------------- fp16 and reduction operators

_DT = {"f32": 0, "bf16": 1, "f16": 2}
_OP = {"sum": 0, "max": 1, "min": 2}


def _load_ext():
    lib = _load()
    if not getattr(lib, "_ext_ready", False):
        P, sz, i32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
        lib.oracle_f32_to_f16_rne.argtypes = [ctypes.c_float]
        lib.oracle_f32_to_f16_rne.restype = ctypes.c_uint16
        lib.oracle_f16_to_f32.argtypes = [ctypes.c_uint16]
        lib.oracle_f16_to_f32.restype = ctypes.c_float
        lib.oracle_f32_to_f16_array.argtypes = [sz, P, P]
        lib.oracle_f32_to_f16_array.restype = None
        lib.oracle_apply_op.argtypes = [i32, ctypes.c_float, ctypes.c_float]
        lib.oracle_apply_op.restype = ctypes.c_float
        lib.oracle_allreduce.argtypes = [i32, i32, i32, sz, P, sz, P]
        lib.oracle_allreduce.restype = None
        lib._ext_ready = True
    return lib


def f32_to_f16(x: np.ndarray) -> np.ndarray:
    """float32 -> uint16 binary16 patterns, round to nearest even (NaN -> 0x7E00)."""
    x = np.ascontiguousarray(x, dtype=np.float32).ravel()
    y = np.empty(x.size, np.uint16)
    if x.size:
        _load_ext().oracle_f32_to_f16_array(x.size, _ptr(x), _ptr(y))
    return y


def f16_to_f32_scalar(h: int) -> float:
    return float(_load_ext().oracle_f16_to_f32(h))


def apply_op(op: str, a: float, b: float) -> float:
    return float(_load_ext().oracle_apply_op(_OP[op], a, b))


def allreduce(x: np.ndarray, dtype: str = "f32", op: str = "sum") -> np.ndarray:
    """x: (R, N) float32 (f32) or uint16 bit patterns (bf16, f16) -> (N,) same type.

    Widen exactly, fold in rank order 0..R-1 in fp32 with `op`, narrow once.
    """
    want = np.float32 if dtype == "f32" else np.uint16
    x = _rows(x, want)
    R, n = x.shape
    y = np.empty(n, want)
    if n:
        _load_ext().oracle_allreduce(_DT[dtype], _OP[op], R, n, _ptr(x), n, _ptr(y))
    return y
