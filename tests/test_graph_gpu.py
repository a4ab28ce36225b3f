"""The flag-synchronised collectives (pull two-shot, fused producer + AllReduce,
put + signal AllGather, signalled AlltoAll) replayed from a CUDA graph: every
replay must see a fresh flag epoch and a zeroed item ticket, so each replay with
new inputs must match the oracle."""
import numpy as np
import pytest

from _gpu_util import download, upload

pytestmark = pytest.mark.gpu


def _capture(fn):
    import torch

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()                                   # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


@pytest.mark.parametrize("algo", ["twoshot_pull", "twoshot", "twoshot_split", "oneshot"])
def test_allreduce_graph_replay(symar, oracle, algo):
    import torch

    R, n = 8, 300_007
    send, recv = symar.Window(R, n * 4), symar.Window(R, n * 4)
    try:
        g = _capture(lambda: symar.sym_allreduce(send, recv, n, "f32", "sum", algo))
        rng = np.random.default_rng(77)
        for _ in range(4):
            x = rng.standard_normal((R, n)).astype(np.float32)
            upload(send, x)
            recv.tensor().zero_()
            g.replay()
            torch.cuda.synchronize()
            assert symar.sym_stream_status() == symar.SYM_OK
            y = download(recv, n * 4, np.float32)
            want = oracle.allreduce_sum_f32(x)
            assert np.array_equal(y.view(np.uint32), np.broadcast_to(want.view(np.uint32), y.shape))
    finally:
        send.free()
        recv.free()


def test_fused_graph_replay(symar, oracle):
    import torch

    R, n = 8, 1_000_003
    win_in, send, recv = (symar.Window(R, n * 4) for _ in range(3))
    alpha = [0.5 + 0.25 * r for r in range(R)]
    try:
        g = _capture(lambda: symar.sym_scale_allreduce(win_in, send, recv, alpha, n))
        rng = np.random.default_rng(78)
        for _ in range(4):
            a = rng.standard_normal((R, n)).astype(np.float32)
            upload(win_in, a)
            recv.tensor().zero_()
            g.replay()
            torch.cuda.synchronize()
            assert symar.sym_stream_status() == symar.SYM_OK
            _, y_w = oracle.scale_allreduce(a, alpha)
            y = download(recv, n * 4, np.float32, ranks=[0, R - 1])
            assert np.array_equal(y.view(np.uint32), np.broadcast_to(y_w.view(np.uint32), y.shape))
    finally:
        for w in (win_in, send, recv):
            w.free()


def test_put_signal_allgather_graph_replay(symar, oracle):
    """The put + signal AllGather from a graph: each replay resets the slots and
    the item ticket in stream order, so every replay must give exact bytes,
    signal counts and counters, and a clean prefix check."""
    import torch

    R, S, chunk, B = 8, 3 * 65536 * 8 + 4096, 65536, 3
    send, recv = symar.Window(R, S, ncounters=1), symar.Window(R, R * S, nsignals=R)
    mism = torch.zeros(1, dtype=torch.int64, device="cuda")
    try:
        g = _capture(lambda: symar.sym_allgather_put_signal(send, recv, S, chunk, B,
                                                            d_mismatch=mism.data_ptr()))
        rng = np.random.default_rng(79)
        for _ in range(3):
            x = rng.integers(0, 256, size=(R, S), dtype=np.uint8)
            recv_o, sig_o, cnt_o = oracle.put_signal_allgather(x, chunk, B)
            upload(send, x)
            recv.tensor().zero_()
            g.replay()
            torch.cuda.synchronize()
            assert symar.sym_stream_status() == symar.SYM_OK
            assert int(mism.item()) == 0
            got = download(recv, R * S, ranks=[0, R - 1])
            for i in range(2):
                assert np.array_equal(got[i], recv_o)
            for q in range(R):
                assert symar.sym_signal_read(recv, R - 1, q) == int(sig_o[R - 1, q])
                assert symar.sym_counter_read(send, q, 0) == int(cnt_o[q])
    finally:
        send.free()
        recv.free()


def test_alltoall_put_signal_graph_replay(symar, oracle):
    import torch

    R, B = 8, 300_000                      # bytes per segment
    send, recv = symar.Window(R, R * B), symar.Window(R, R * B, nsignals=1)
    try:
        g = _capture(lambda: symar.sym_alltoall(send, recv, B // 4, "f32", "put_signal"))
        rng = np.random.default_rng(80)
        for _ in range(3):
            x = rng.integers(0, 256, size=(R, R * B), dtype=np.uint8)
            upload(send, x)
            recv.tensor().zero_()
            g.replay()
            torch.cuda.synchronize()
            assert symar.sym_stream_status() == symar.SYM_OK
            want = oracle.alltoall(x)
            got = download(recv, R * B)
            assert np.array_equal(got, want)
            for p in range(R):
                assert symar.sym_signal_read(recv, p, 0) == R
    finally:
        send.free()
        recv.free()
