"""Collectives on different windows, enqueued on different streams at the same
time: each window keeps its own epoch, flags, ticket and slots, so every
result must still match the oracle (calls on the same window are the caller's
to order; see the header)."""
import numpy as np
import pytest

from _gpu_util import download, upload

pytestmark = pytest.mark.gpu


def test_concurrent_streams_independent_windows(symar, oracle):
    import torch

    R, n = 8, 2_000_003
    S_ag, chunk, B = 1 << 20, 65536, 4
    rng = np.random.default_rng(90)
    x = rng.standard_normal((R, n)).astype(np.float32)
    y = rng.standard_normal((R, n)).astype(np.float32)
    b = rng.integers(0, 256, size=(R, S_ag), dtype=np.uint8)
    a_in, a_out = symar.Window(R, n * 4), symar.Window(R, n * 4)
    c_in, c_out = symar.Window(R, n * 4), symar.Window(R, n * 4)
    p_send, p_recv = symar.Window(R, S_ag, ncounters=1), symar.Window(R, R * S_ag, nsignals=R)
    s1, s2, s3 = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    try:
        upload(a_in, x)
        upload(c_in, y)
        upload(p_send, b)
        want_x, want_y = oracle.allreduce_sum_f32(x), oracle.allreduce_sum_f32(y)
        want_b = oracle.allgather(b)
        torch.cuda.synchronize()
        for _ in range(5):
            symar.sym_allreduce(a_in, a_out, n, "f32", "sum", "twoshot_pull", stream=s1)
            symar.sym_allreduce(c_in, c_out, n, "f32", "sum", "twoshot", stream=s2)
            symar.sym_allgather_put_signal(p_send, p_recv, S_ag, chunk, B, stream=s3)
        torch.cuda.synchronize()
        assert symar.sym_stream_status() == symar.SYM_OK
        got_a = download(a_out, n * 4, np.float32, ranks=[0, R - 1])
        got_c = download(c_out, n * 4, np.float32, ranks=[0, R - 1])
        got_p = download(p_recv, R * S_ag, ranks=[0, R - 1])
        for i in range(2):
            assert np.array_equal(got_a[i].view(np.uint32), want_x.view(np.uint32))
            assert np.array_equal(got_c[i].view(np.uint32), want_y.view(np.uint32))
            assert np.array_equal(got_p[i], want_b)
        for q in range(R):
            assert symar.sym_signal_read(p_recv, R - 1, q) == -(-(S_ag // chunk) // B)
    finally:
        for w in (a_in, a_out, c_in, c_out, p_send, p_recv):
            w.free()
