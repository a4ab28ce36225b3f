"""ctypes binding of libsymar.so -- argument marshalling only.

Every function has the name of its C entry point (include/symar.h) and does
nothing but convert arguments, call it, and raise SymError on a non-zero
status.  All device work happens in the library's CUDA kernels; there is no
Python or CPU fallback, and loading fails loudly if the library is missing.
PyTorch is used for streams and for tensor views of window memory.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libsymar.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "symar.h")

# enums (mirror include/symar.h)
SYM_OK, SYM_ERR_INVALID_ARG, SYM_ERR_OOM, SYM_ERR_CUDA = 0, 1, 2, 3
SYM_ERR_TIMEOUT, SYM_ERR_UNSUPPORTED, SYM_ERR_DEVICE_STATUS = 4, 5, 6
SYM_F32, SYM_BF16, SYM_F16 = 0, 1, 2
SYM_SUM, SYM_MAX, SYM_MIN = 0, 1, 2
SYM_ALGO_AUTO, SYM_ALGO_ONESHOT, SYM_ALGO_TWOSHOT, SYM_ALGO_PUT_SIGNAL = 0, 1, 2, 3
SYM_ALGO_TWOSHOT_PULL, SYM_ALGO_TWOSHOT_SPLIT = 4, 5
SYM_ALGO_COPY, SYM_ALGO_CE = 6, 7
SYM_WINDOW_CUDA_MALLOC, SYM_WINDOW_REGISTERED, SYM_WINDOW_VMM_EXPORTABLE, SYM_WINDOW_VMM = 0, 1, 2, 3
NO_ID = 0xFFFFFFFF

ALGOS = {"auto": SYM_ALGO_AUTO, "oneshot": SYM_ALGO_ONESHOT, "twoshot": SYM_ALGO_TWOSHOT,
         "twoshot_pull": SYM_ALGO_TWOSHOT_PULL, "twoshot_split": SYM_ALGO_TWOSHOT_SPLIT,
         "copy": SYM_ALGO_COPY, "put_signal": SYM_ALGO_PUT_SIGNAL, "ce": SYM_ALGO_CE}
DTYPES = {"f32": SYM_F32, "bf16": SYM_BF16, "f16": SYM_F16}
OPS = {"sum": SYM_SUM, "max": SYM_MAX, "min": SYM_MIN}


class SymError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        name = _lib.sym_status_string(status).decode() if _lib else str(status)
        super().__init__(f"{where}: {name}" + (f" ({detail})" if detail else ""))


_lib = None
_lock = threading.Lock()

P, sz, i32, u32, u64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_uint32, ctypes.c_uint64
PP = ctypes.POINTER(ctypes.c_void_p)
_SIGS = {
    "sym_window_alloc": ([i32, sz, u32, u32, PP], i32),
    "sym_window_alloc_vmm": ([i32, sz, u32, u32, PP], i32),
    "sym_window_kind": ([P], i32),
    "sym_window_register": ([P, i32, sz, sz, u32, u32, PP], i32),
    "sym_window_free": ([P], i32),
    "sym_window_rank_ptr": ([P, i32, PP], i32),
    "sym_window_stride": ([P], sz),
    "sym_window_bytes": ([P], sz),
    "sym_window_nranks": ([P], i32),
    "sym_window_device": ([P], i32),
    "sym_window_write": ([P, i32, sz, P, sz, P], i32),
    "sym_window_read": ([P, i32, sz, P, sz, P], i32),
    "sym_allreduce": ([P, P, sz, i32, i32, i32, P], i32),
    "sym_allreduce_algo": ([P, sz, i32, ctypes.POINTER(i32)], i32),
    "sym_allgather": ([P, P, sz, i32, i32, sz, u32, P], i32),
    "sym_allgather_put_signal": ([P, P, sz, sz, u32, P, u64, P], i32),
    "sym_put_signal": ([P, P, i32, i32, sz, sz, sz, u32, u32, P], i32),
    "sym_get": ([P, P, i32, i32, sz, sz, sz, u32, P], i32),
    "sym_barrier": ([P, u32, u64, P], i32),
    "sym_alltoall": ([P, P, sz, i32, i32, u64, P], i32),
    "sym_scale_allreduce": ([P, P, P, P, sz, P], i32),
    "sym_allreduce_noalloc": ([P, P, sz, i32, sz, i32, i32, P], i32),
    "sym_signal": ([P, i32, u32, u64, P], i32),
    "sym_signal_wait": ([P, i32, u32, u64, i32, u64, P], i32),
    "sym_signal_read": ([P, i32, u32, i32, ctypes.POINTER(u64), P], i32),
    "sym_signal_reset": ([P, i32, u32, P], i32),
    "sym_counter_read": ([P, i32, u32, i32, ctypes.POINTER(u64), P], i32),
    "sym_counter_wait": ([P, i32, u32, u64, i32, u64, P], i32),
    "sym_counter_reset": ([P, i32, u32, P], i32),
    "sym_stream_status": ([P], i32),
    "sym_status_string": ([i32], ctypes.c_char_p),
    "sym_last_error": ([], ctypes.c_char_p),
    "sym_launch_count": ([], u64),
    "sym_abi_version": ([], i32),
}


def header_symbols() -> list[str]:
    """Every function the C header declares."""
    txt = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:sym_status_t|size_t|int|const char\*|uint64_t)\s+(sym_\w+)\(",
                                 txt, re.M)))


def load():
    """Load libsymar.so (built in-tree by build.py). Raises if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "`python -m symmetric_memory_allreduce_gb300.build` (nvcc, sm_103a)")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in _SIGS.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


def _check(status: int, where: str):
    if status != SYM_OK:
        detail = _lib.sym_last_error().decode(errors="replace")
        raise SymError(status, where, detail)


def _stream(stream) -> int | None:
    """cudaStream_t of a torch stream, an int handle, or the current torch stream."""
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream or None
    if isinstance(stream, int):
        return stream or None
    return stream.cuda_stream or None


def _handle(w):
    return w.handle if isinstance(w, Window) else w


class Window:
    """R equal rank windows (sym_window_alloc, sym_window_alloc_vmm with vmm=True, or
    sym_window_register with base=...)."""

    def __init__(self, R: int, bytes_per_rank: int, nsignals: int = 0, ncounters: int = 0,
                 base: int | None = None, stride: int | None = None, keepalive=None,
                 vmm: bool = False):
        lib = load()
        h = ctypes.c_void_p()
        if base is None and vmm:
            _check(lib.sym_window_alloc_vmm(R, bytes_per_rank, nsignals, ncounters, ctypes.byref(h)),
                   "sym_window_alloc_vmm")
        elif base is None:
            _check(lib.sym_window_alloc(R, bytes_per_rank, nsignals, ncounters, ctypes.byref(h)),
                   "sym_window_alloc")
        else:
            _check(lib.sym_window_register(base, R, bytes_per_rank, stride, nsignals, ncounters,
                                           ctypes.byref(h)), "sym_window_register")
        self.handle = h.value
        self.R = R
        self.bytes = bytes_per_rank
        self.stride = lib.sym_window_stride(self.handle)
        self.device = lib.sym_window_device(self.handle)
        self.nsignals, self.ncounters = nsignals, ncounters
        self.kind = lib.sym_window_kind(self.handle)
        self._keepalive = keepalive

    def rank_ptr(self, r: int) -> int:
        p = ctypes.c_void_p()
        _check(_lib.sym_window_rank_ptr(self.handle, r, ctypes.byref(p)), "sym_window_rank_ptr")
        return p.value

    def tensor(self, dtype=None):
        """torch view (R, stride // itemsize) of the whole window (no copy; valid until free())."""
        import torch

        dtype = dtype or torch.uint8

        class _CAI:
            pass

        o = _CAI()
        o.__cuda_array_interface__ = {"shape": (self.R * self.stride,), "typestr": "|u1",
                                      "data": (self.rank_ptr(0), False), "version": 3,
                                      "strides": None}
        t = torch.as_tensor(o, device=f"cuda:{self.device}")
        return t.view(dtype).view(self.R, -1)

    def write(self, rank: int, src, off: int = 0, nbytes: int | None = None, stream=None):
        """sym_window_write from a host pointer / numpy array / CPU tensor."""
        ptr, n = _buffer(src)
        _check(_lib.sym_window_write(self.handle, rank, off, ptr, n if nbytes is None else nbytes,
                                     _stream(stream)), "sym_window_write")

    def read(self, rank: int, dst, off: int = 0, nbytes: int | None = None, stream=None):
        ptr, n = _buffer(dst)
        _check(_lib.sym_window_read(self.handle, rank, off, ptr, n if nbytes is None else nbytes,
                                    _stream(stream)), "sym_window_read")

    def free(self):
        if self.handle:
            h, self.handle = self.handle, None
            _check(_lib.sym_window_free(h), "sym_window_free")

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.free()


def _buffer(obj):
    """(address, nbytes) of a numpy array, a torch tensor, or an (address, nbytes) pair."""
    if isinstance(obj, tuple):
        return obj
    try:
        import numpy as np

        if isinstance(obj, np.ndarray):
            if not obj.flags.c_contiguous:
                raise ValueError("numpy buffer must be C-contiguous")
            return obj.ctypes.data, obj.nbytes
    except ImportError:
        pass
    if hasattr(obj, "data_ptr"):
        if not obj.is_contiguous():
            raise ValueError("tensor must be contiguous")
        return obj.data_ptr(), obj.numel() * obj.element_size()
    raise TypeError(f"unsupported buffer {type(obj)}")


# ----------------------------------------------------------------- collectives

def sym_allreduce(send, recv, count: int, dtype="f32", op="sum", algo="auto", stream=None):
    _check(_lib.sym_allreduce(_handle(send), _handle(recv), count, DTYPES.get(dtype, dtype),
                              OPS.get(op, op), ALGOS.get(algo, algo), _stream(stream)),
           "sym_allreduce")


def sym_allreduce_algo(send, count: int, dtype="f32") -> str:
    out = ctypes.c_int()
    _check(_lib.sym_allreduce_algo(_handle(send), count, DTYPES.get(dtype, dtype), ctypes.byref(out)),
           "sym_allreduce_algo")
    return {v: k for k, v in ALGOS.items()}[out.value]


def sym_allgather(send, recv, sendcount: int, dtype="f32", algo="auto", chunk_bytes: int = 0,
                  chunks_per_signal: int = 0, stream=None):
    _check(_lib.sym_allgather(_handle(send), _handle(recv), sendcount, DTYPES.get(dtype, dtype),
                              ALGOS.get(algo, algo), chunk_bytes, chunks_per_signal, _stream(stream)),
           "sym_allgather")


def sym_allgather_put_signal(send, recv, bytes_per_rank: int, chunk_bytes: int = 0,
                             chunks_per_signal: int = 0, d_mismatch: int = 0, timeout_ns: int = 0,
                             stream=None):
    _check(_lib.sym_allgather_put_signal(_handle(send), _handle(recv), bytes_per_rank, chunk_bytes,
                                         chunks_per_signal, d_mismatch or None, timeout_ns,
                                         _stream(stream)), "sym_allgather_put_signal")


def sym_alltoall(send, recv, count: int, dtype="f32", algo="auto", timeout_ns: int = 0,
                 stream=None):
    _check(_lib.sym_alltoall(_handle(send), _handle(recv), count, DTYPES.get(dtype, dtype),
                             ALGOS.get(algo, algo), timeout_ns, _stream(stream)), "sym_alltoall")


def sym_allreduce_noalloc(send_ptr: int, recv_ptr: int, stride: int, R: int, count: int,
                          dtype="f32", op="sum", stream=None):
    """AllReduce over caller-owned buffers (rank r at ptr + r*stride) that allocates nothing.

    For callers that cannot allocate device memory (e.g. an engine that forbids
    allocations after start-up, or a plug-in whose framework owns the allocator).
    """
    _check(_lib.sym_allreduce_noalloc(send_ptr, recv_ptr, stride, R, count, DTYPES.get(dtype, dtype),
                                      OPS.get(op, op), _stream(stream)), "sym_allreduce_noalloc")


def sym_scale_allreduce(inp, send, recv, alpha, count: int, stream=None):
    """alpha: sequence of R floats (copied into the launch)."""
    al = (ctypes.c_float * len(alpha))(*[float(v) for v in alpha])
    _check(_lib.sym_scale_allreduce(_handle(inp), _handle(send), _handle(recv), al, count,
                                    _stream(stream)), "sym_scale_allreduce")


def sym_put_signal(src, dst, src_rank: int, peer: int, dst_off: int, src_off: int, nbytes: int,
                   signal_id: int = NO_ID, counter_id: int = NO_ID, stream=None):
    _check(_lib.sym_put_signal(_handle(src), _handle(dst), src_rank, peer, dst_off, src_off, nbytes,
                               signal_id, counter_id, _stream(stream)), "sym_put_signal")


def sym_get(remote, local, rank: int, peer: int, local_off: int, remote_off: int, nbytes: int,
            counter_id: int = NO_ID, stream=None):
    _check(_lib.sym_get(_handle(remote), _handle(local), rank, peer, local_off, remote_off, nbytes,
                        counter_id, _stream(stream)), "sym_get")


def sym_barrier(w, signal_id: int = 0, timeout_ns: int = 0, stream=None):
    _check(_lib.sym_barrier(_handle(w), signal_id, timeout_ns, _stream(stream)), "sym_barrier")


def sym_signal(dst, peer: int, signal_id: int, value: int = 1, stream=None):
    _check(_lib.sym_signal(_handle(dst), peer, signal_id, value, _stream(stream)), "sym_signal")


def sym_signal_wait(w, rank: int, signal_id: int, least: int, bits: int = 64, timeout_ns: int = 0,
                    stream=None):
    _check(_lib.sym_signal_wait(_handle(w), rank, signal_id, least & (2**64 - 1), bits, timeout_ns,
                                _stream(stream)), "sym_signal_wait")


def sym_signal_read(w, rank: int, signal_id: int, bits: int = 64, stream=None) -> int:
    out = ctypes.c_uint64()
    _check(_lib.sym_signal_read(_handle(w), rank, signal_id, bits, ctypes.byref(out), _stream(stream)),
           "sym_signal_read")
    return out.value


def sym_signal_reset(w, rank: int, signal_id: int, stream=None):
    _check(_lib.sym_signal_reset(_handle(w), rank, signal_id, _stream(stream)), "sym_signal_reset")


def sym_counter_read(w, rank: int, counter_id: int, bits: int = 56, stream=None) -> int:
    out = ctypes.c_uint64()
    _check(_lib.sym_counter_read(_handle(w), rank, counter_id, bits, ctypes.byref(out),
                                 _stream(stream)), "sym_counter_read")
    return out.value


def sym_counter_wait(w, rank: int, counter_id: int, least: int, bits: int = 56, timeout_ns: int = 0,
                     stream=None):
    _check(_lib.sym_counter_wait(_handle(w), rank, counter_id, least & (2**64 - 1), bits, timeout_ns,
                                 _stream(stream)), "sym_counter_wait")


def sym_counter_reset(w, rank: int, counter_id: int, stream=None):
    _check(_lib.sym_counter_reset(_handle(w), rank, counter_id, _stream(stream)), "sym_counter_reset")


def sym_stream_status(stream=None) -> int:
    """Returns the status code (does not raise), so callers can expect SYM_ERR_TIMEOUT."""
    return int(_lib.sym_stream_status(_stream(stream)))


def sym_status_string(status: int) -> str:
    return load().sym_status_string(status).decode()


def sym_last_error() -> str:
    return load().sym_last_error().decode(errors="replace")


def sym_launch_count() -> int:
    return int(load().sym_launch_count())


def sym_abi_version() -> int:
    return int(load().sym_abi_version())
