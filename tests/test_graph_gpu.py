"""The flag-synchronised collectives (pull two-shot, fused producer + AllReduce)
replayed from a CUDA graph: every replay must see a fresh flag epoch, so each
replay with new inputs must match the oracle."""
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
