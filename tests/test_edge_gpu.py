"""Edge cases on the GPU: the maximum rank count (R = 64) for every collective,
and zero-size calls (no-ops that launch nothing)."""
import numpy as np
import pytest

from _gpu_util import download, upload

pytestmark = pytest.mark.gpu

RMAX = 64


@pytest.mark.parametrize("algo", ["oneshot", "twoshot", "twoshot_pull", "twoshot_split"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_allreduce_max_ranks(symar, oracle, algo, dtype):
    from symmetric_memory_allreduce_gb300 import workloads as wl

    rng = np.random.default_rng(64)
    for n in (4097, 100_003):
        f = rng.standard_normal((RMAX, n)).astype(np.float32)
        x = f if dtype == "f32" else wl.to_bf16_bits(f)
        es = x.itemsize
        send, recv = symar.Window(RMAX, n * es), symar.Window(RMAX, n * es)
        try:
            upload(send, x)
            symar.sym_allreduce(send, recv, n, dtype, "sum", algo)
            assert symar.sym_stream_status() == symar.SYM_OK
            want = oracle.allreduce(x, dtype, "sum")
            got = download(recv, n * es, x.dtype, ranks=[0, 31, 63])
            assert np.array_equal(got.view(np.uint8), np.broadcast_to(want, got.shape).view(np.uint8))
        finally:
            send.free()
            recv.free()


def test_allgather_and_put_signal_max_ranks(symar, oracle):
    S = 4096 + 16
    rng = np.random.default_rng(65)
    x = rng.integers(0, 256, size=(RMAX, S), dtype=np.uint8)
    send, recv = symar.Window(RMAX, S, ncounters=1), symar.Window(RMAX, RMAX * S, nsignals=RMAX)
    try:
        upload(send, x)
        want = oracle.allgather(x)
        for algo in ("copy", "ce", "put_signal"):
            recv.tensor().zero_()
            symar.sym_allgather(send, recv, S // 4, "f32", algo, 1024, 2)
            assert symar.sym_stream_status() == symar.SYM_OK
            got = download(recv, RMAX * S, ranks=[0, 17, 63])
            assert all(np.array_equal(g, want) for g in got), algo
        assert symar.sym_signal_read(recv, 63, 63) == -(-(-(-S // 1024)) // 2)
        assert symar.sym_counter_read(send, 5, 0) == RMAX * -(-S // 1024)
    finally:
        send.free()
        recv.free()


def test_alltoall_max_ranks(symar, oracle):
    B = 256
    rng = np.random.default_rng(66)
    x = rng.integers(0, 256, size=(RMAX, RMAX * B), dtype=np.uint8)
    send, recv = symar.Window(RMAX, RMAX * B), symar.Window(RMAX, RMAX * B, nsignals=1)
    try:
        upload(send, x)
        want = oracle.alltoall(x)
        for algo in ("copy", "put_signal"):
            recv.tensor().zero_()
            symar.sym_alltoall(send, recv, B // 4, "f32", algo)
            assert symar.sym_stream_status() == symar.SYM_OK
            assert np.array_equal(download(recv, RMAX * B), want), algo
        assert symar.sym_signal_read(recv, 40, 0) == RMAX
    finally:
        send.free()
        recv.free()


def test_fused_max_ranks(symar, oracle):
    n = 70_001
    rng = np.random.default_rng(67)
    a = rng.standard_normal((RMAX, n)).astype(np.float32)
    alpha = rng.uniform(0.5, 2.0, RMAX).astype(np.float32)
    s_w, y_w = oracle.scale_allreduce(a, alpha)
    wins = [symar.Window(RMAX, n * 4) for _ in range(3)]
    try:
        upload(wins[0], a)
        symar.sym_scale_allreduce(wins[0], wins[1], wins[2], alpha, n)
        assert symar.sym_stream_status() == symar.SYM_OK
        y = download(wins[2], n * 4, np.float32, ranks=[0, 63])
        assert np.array_equal(y.view(np.uint32), np.broadcast_to(y_w.view(np.uint32), y.shape))
    finally:
        for w in wins:
            w.free()


def test_zero_size_calls_launch_nothing(symar):
    a, b = symar.Window(4, 4096, ncounters=1), symar.Window(4, 4 * 4096, nsignals=4)
    c = symar.Window(4, 4096)
    try:
        n0 = symar.sym_launch_count()
        symar.sym_allgather(a, b, 0, "f32", "copy")
        symar.sym_allgather(a, b, 0, "f32", "put_signal")
        symar.sym_allgather_put_signal(a, b, 0)
        symar.sym_alltoall(a, c, 0, "f32", "copy")
        symar.sym_scale_allreduce(a, c, b, [1.0] * 4, 0)
        symar.sym_allreduce(a, c, 0)
        assert symar.sym_launch_count() == n0
        assert symar.sym_stream_status() == symar.SYM_OK
    finally:
        for w in (a, b, c):
            w.free()
