"""sym_allreduce_noalloc: the AllReduce entry point for callers that cannot
allocate device memory (engines that forbid allocations after start-up,
plug-ins whose framework owns the allocator).  Its results must equal the
oracle's (the rank-order fold of [SYMEX] Example 1) and the regular entry
point's, sym_allreduce, on two calls in a row that share its static scratch.
Collected last on purpose; it also passes on its own in a fresh process."""
import os
import subprocess
import sys

import numpy as np
import pytest

from _gpu_util import bf16_ulp_distance, download, upload

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _regular(sm, x, dtype, op="sum"):
    """Result of the regular entry point (windows, two-shot) for inputs x (R, n)."""
    R, n = x.shape
    es = x.itemsize
    send, recv = sm.Window(R, n * es), sm.Window(R, n * es)
    try:
        upload(send, x)
        sm.sym_allreduce(send, recv, n, dtype, op, "twoshot")
        assert sm.sym_stream_status() == sm.SYM_OK
        return download(recv, n * es, x.dtype)
    finally:
        send.free()
        recv.free()


def _buffers(R, stride):
    """Caller-owned buffers: torch allocations made by the test, not by the entry point."""
    import torch

    return (torch.empty(R * stride, dtype=torch.uint8, device="cuda"),
            torch.empty(R * stride, dtype=torch.uint8, device="cuda"))


def _noalloc(sm, x, dtype, send_t, recv_t, stride, op="sum"):
    import torch

    R, n = x.shape
    es = x.itemsize
    host = torch.zeros((R, stride), dtype=torch.uint8)
    host[:, : n * es] = torch.from_numpy(np.ascontiguousarray(x).view(np.uint8))
    send_t.copy_(host.view(-1))
    recv_t.fill_(0xAB)
    sm.sym_allreduce_noalloc(send_t.data_ptr(), recv_t.data_ptr(), stride, R, n, dtype, op)
    torch.cuda.synchronize()
    out = recv_t.view(R, stride)[:, : n * es].cpu().numpy()
    return np.ascontiguousarray(out).view(x.dtype)


def _equal(y, want, dtype):
    """fp32 bit-exact; 16-bit types within 1 ulp and bit-exact (NaN payloads not compared)."""
    if dtype == "f32":
        nan = np.isnan(want)
        assert np.all(np.isnan(y[:, nan]))
        assert np.array_equal(y[:, ~nan].view(np.uint32),
                              np.broadcast_to(want[~nan].view(np.uint32), y[:, ~nan].shape))
        return
    nanbits = (want & 0x7FFF) > (0x7F80 if dtype == "bf16" else 0x7C00)
    keep = ~nanbits
    if dtype == "bf16":
        assert bf16_ulp_distance(y[:, keep], np.broadcast_to(want[keep], y[:, keep].shape)).max(
            initial=0) <= 1
    assert np.array_equal(y[:, keep], np.broadcast_to(want[keep], y[:, keep].shape))


def _inputs(dtype, f):
    from symmetric_memory_allreduce_gb300 import workloads as wl

    if dtype == "f32":
        return f
    if dtype == "bf16":
        return wl.to_bf16_bits(f)
    return np.ascontiguousarray(f.astype(np.float16).view(np.uint16))


def test_noalloc_matches_oracle_and_regular_entry_two_calls(symar, oracle):
    from symmetric_memory_allreduce_gb300 import workloads as wl

    R, n = 8, 1_000_003                       # several tiles per chunk plus a ragged tail
    stride = (n * 4 + 4095) // 4096 * 4096
    send_t, recv_t = _buffers(R, stride)
    for call in range(2):                     # two calls in a row, different inputs
        x = wl.normal_f32(2, R, n) if call == 0 else wl.uniform_f32(3, R, n)
        y = _noalloc(symar, x, "f32", send_t, recv_t, stride)
        _equal(y, oracle.allreduce_sum_f32(x), "f32")
        _equal(y, _regular(symar, x, "f32")[0], "f32")


def test_noalloc_bf16_two_calls(symar, oracle):
    from symmetric_memory_allreduce_gb300 import workloads as wl

    R, n = 16, 300_007
    stride = (n * 2 + 4095) // 4096 * 4096
    send_t, recv_t = _buffers(R, stride)
    for call in range(2):
        x = wl.to_bf16_bits(wl.uniform_f32(10 + call, R, n))
        y = _noalloc(symar, x, "bf16", send_t, recv_t, stride)
        _equal(y, oracle.allreduce_sum_bf16(x), "bf16")
        _equal(y, _regular(symar, x, "bf16")[0], "bf16")


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("op", ["sum", "max", "min"])
def test_noalloc_dtypes_and_ops(symar, oracle, dtype, op):
    """Every element type and operator against the oracle, ragged sizes, signed zeros, NaNs."""
    rng = np.random.default_rng(400)
    for R, n in [(1, 9), (3, 4097), (8, 100_003)]:
        f = rng.uniform(-2, 2, size=(R, n)).astype(np.float32)
        f[:, ::97] = 0.0
        f[R // 2, ::89] = -0.0
        if op != "sum":
            f[0, ::101] = np.nan
        x = _inputs(dtype, f)
        stride = (n * x.itemsize + 4095) // 4096 * 4096
        send_t, recv_t = _buffers(R, stride)
        _equal(_noalloc(symar, x, dtype, send_t, recv_t, stride, op), oracle.allreduce(x, dtype, op),
               dtype)


_GIVE_UP_CHILD = r"""
import sys
import numpy as np
import torch
sys.path.insert(0, sys.argv[1])
import oracle
import symmetric_memory_allreduce_gb300 as sm
from symmetric_memory_allreduce_gb300 import workloads as wl

sm.load()
R, n = 8, 2_000_003
stride = (n * 4 + 4095) // 4096 * 4096
send = torch.empty(R * stride, dtype=torch.uint8, device="cuda")
recv = torch.empty(R * stride, dtype=torch.uint8, device="cuda")
for call in range(2):
    x = wl.normal_f32(20 + call, R, n)
    host = torch.zeros((R, stride), dtype=torch.uint8)
    host[:, : n * 4] = torch.from_numpy(x.view(np.uint8))
    send.copy_(host.view(-1))
    recv.fill_(0xAB)
    sm.sym_allreduce_noalloc(send.data_ptr(), recv.data_ptr(), stride, R, n, "f32", "sum")
    torch.cuda.synchronize()
    y = np.ascontiguousarray(recv.view(R, stride)[:, : n * 4].cpu().numpy()).view(np.float32)
    want = oracle.allreduce_sum_f32(x)
    assert np.array_equal(y.view(np.uint32), np.broadcast_to(want.view(np.uint32), y.shape)), call
print("GIVE_UP_OK")
"""


def test_noalloc_gives_up_waiting_and_stays_exact(symar):
    """With every flag wait bounded at 1 ns (and gathers one grid wave behind their
    reductions), gathers give up and reduce their tiles from the inputs themselves;
    the result is still bit-exact against the oracle, on two calls in a row.  Runs in a
    child process because the bound is read from the environment once per process."""
    env = dict(os.environ, SYM_TIMEOUT_NS="1", SYM_PULL_LAG_WAVES="1")
    r = subprocess.run([sys.executable, "-c", _GIVE_UP_CHILD, ROOT], env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "GIVE_UP_OK" in r.stdout


def test_noalloc_rejects_oversize_and_overlap(symar):
    import torch

    buf = torch.empty(2 * 4096, dtype=torch.uint8, device="cuda")
    p = buf.data_ptr()
    # more than 65536 tiles of 16 KiB: rejected before any device work, with a reason
    with pytest.raises(symar.SymError) as e:     # (never dereferenced: rejected on the host)
        symar.sym_allreduce_noalloc(p, p + (1 << 43), 1 << 40, 2, (1 << 40) // 4, "f32", "sum")
    assert e.value.status == symar.SYM_ERR_INVALID_ARG
    assert "static scratch" in symar.sym_last_error()
    with pytest.raises(symar.SymError):          # input and output ranges overlap
        symar.sym_allreduce_noalloc(p, p + 16, 4096, 1, 64, "f32", "sum")
