"""Windows over caller memory (sym_window_register) that alias: every collective rejects
two different windows sharing a byte of the ranges it touches, on the host, before any
launch; interleaved windows that share no byte still run and match the oracle."""
import numpy as np
import pytest

from _gpu_util import download, upload

pytestmark = pytest.mark.gpu


def _buffer(nbytes):
    import torch

    return torch.zeros(nbytes, dtype=torch.uint8, device="cuda")


def test_allreduce_rejects_partly_aliased_windows(symar):
    buf = _buffer(1 << 20)
    base = buf.data_ptr()
    R, n = 4, 1024                      # 4 KiB per rank
    send = symar.Window(R, 4096, base=base, stride=8192)
    recv = symar.Window(R, 4096, base=base + 8192, stride=8192)   # recv rank r = send rank r+1
    try:
        launches = symar.sym_launch_count()
        for algo in ("oneshot", "twoshot", "twoshot_pull", "twoshot_split", "auto"):
            with pytest.raises(symar.SymError) as e:
                symar.sym_allreduce(send, recv, n, "f32", "sum", algo)
            assert e.value.status == symar.SYM_ERR_INVALID_ARG
            assert "share memory" in symar.sym_last_error()
        # a call touching fewer bytes than the windows hold is judged on those bytes only
        with pytest.raises(symar.SymError):
            symar.sym_allreduce(send, recv, 1, "f32", "sum", "twoshot")
        assert symar.sym_launch_count() == launches            # nothing was enqueued
    finally:
        send.free()
        recv.free()


def test_allreduce_interleaved_windows_run(symar, oracle):
    """send rank r at base + r*8192, recv rank r at base + 4096 + r*8192: no shared byte."""
    buf = _buffer(1 << 20)
    base = buf.data_ptr()
    R, n = 4, 1024
    send = symar.Window(R, 4096, base=base, stride=8192)
    recv = symar.Window(R, 4096, base=base + 4096, stride=8192)
    try:
        x = np.random.default_rng(3).standard_normal((R, n)).astype(np.float32)
        upload(send, x)
        want = oracle.allreduce_sum_f32(x)
        for algo in ("oneshot", "twoshot", "twoshot_pull", "twoshot_split"):
            symar.sym_allreduce(send, recv, n, "f32", "sum", algo)
            assert symar.sym_stream_status() == symar.SYM_OK
            y = download(recv, n * 4, np.float32)
            assert all(np.array_equal(y[r].view(np.uint32), want.view(np.uint32)) for r in range(R))
    finally:
        send.free()
        recv.free()


def test_allgather_alltoall_fused_reject_aliases(symar, oracle):
    buf = _buffer(1 << 22)
    base = buf.data_ptr()
    R, S, st = 4, 4096, 1 << 16
    send = symar.Window(R, S, ncounters=1, base=base, stride=st)              # [r*st, r*st + S)
    alias = symar.Window(R, R * S, nsignals=R, base=base + 2048, stride=st)   # overlaps send rank r
    recv = symar.Window(R, R * S, nsignals=R, base=base + 8192, stride=st)    # interleaved, disjoint
    other = symar.Window(R, R * S, nsignals=R, base=base + (1 << 20), stride=st)
    try:
        launches = symar.sym_launch_count()
        for algo in ("copy", "ce", "put_signal"):
            with pytest.raises(symar.SymError) as e:
                symar.sym_allgather(send, alias, S // 4, "f32", algo)
            assert e.value.status == symar.SYM_ERR_INVALID_ARG
        with pytest.raises(symar.SymError):
            symar.sym_allgather_put_signal(send, alias, S)
        for algo in ("copy", "put_signal"):
            with pytest.raises(symar.SymError):
                symar.sym_alltoall(send, alias, S // (4 * R), "f32", algo)
        with pytest.raises(symar.SymError):
            symar.sym_scale_allreduce(other, send, alias, [1.0] * R, S // 4)
        assert symar.sym_launch_count() == launches          # rejected before any launch
        # windows over the same buffer that share no byte run
        x = np.random.default_rng(4).integers(0, 256, size=(R, S), dtype=np.uint8)
        upload(send, x)
        want = oracle.allgather(x)
        for dst in (recv, other):
            symar.sym_allgather(send, dst, S // 4, "f32", "copy")
            assert symar.sym_stream_status() == symar.SYM_OK
            out = download(dst, R * S)
            assert all(np.array_equal(out[r], want) for r in range(R))
    finally:
        for w in (send, alias, recv, other):
            w.free()
