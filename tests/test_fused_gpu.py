"""Producer + AllReduce (sym_scale_allreduce) against the oracle: the contributions
alpha_r * a_r and their rank-order sum, bit-exact, at ragged and full sizes."""
import numpy as np
import pytest

from _gpu_util import download, upload

pytestmark = pytest.mark.gpu


def _run(sm, a, alpha):
    R, n = a.shape
    win_in, send, recv = (sm.Window(R, n * 4) for _ in range(3))
    try:
        upload(win_in, a)
        sm.sym_scale_allreduce(win_in, send, recv, alpha, n)
        assert sm.sym_stream_status() == sm.SYM_OK, sm.sym_last_error()
        return download(send, n * 4, np.float32), download(recv, n * 4, np.float32)
    finally:
        for w in (win_in, send, recv):
            w.free()


@pytest.mark.parametrize("R", [1, 2, 3, 8, 16])
def test_scale_allreduce_ragged(symar, oracle, R):
    rng = np.random.default_rng(500 + R)
    for n in [1, 5, 1000, 4097, 65_539, 262_147]:
        a = rng.standard_normal((R, n)).astype(np.float32)
        alpha = rng.standard_normal(R).astype(np.float32)
        s_w, y_w = oracle.scale_allreduce(a, alpha)
        s, y = _run(symar, a, alpha)
        assert np.array_equal(s.view(np.uint32), s_w.view(np.uint32)), n
        assert np.array_equal(y.view(np.uint32), np.broadcast_to(y_w.view(np.uint32), y.shape)), n


def test_scale_allreduce_closed_form(symar):
    R, n = 8, 1 << 20
    a = np.repeat(np.arange(R, dtype=np.float32)[:, None], n, axis=1)
    _, y = _run(symar, a, np.arange(1, R + 1, dtype=np.float32))
    assert np.all(y == np.float32((R - 1) * R * (R + 1) // 3))


def test_scale_allreduce_full_size_repeat(symar, oracle):
    """R=8 x 16M fp32 (64 MiB per rank), three calls on the same windows (epoch flags)."""
    from symmetric_memory_allreduce_gb300 import workloads as wl

    a = wl.workload_inputs(2)
    R, n = a.shape
    alpha = np.linspace(0.5, 2.0, R).astype(np.float32)
    s_w, y_w = oracle.scale_allreduce(a, alpha)
    win_in, send, recv = (symar.Window(R, n * 4) for _ in range(3))
    try:
        upload(win_in, a)
        for _ in range(3):
            recv.tensor().zero_()
            symar.sym_scale_allreduce(win_in, send, recv, alpha, n)
            assert symar.sym_stream_status() == symar.SYM_OK
            for r in (0, R - 1):
                y = download(recv, n * 4, np.float32, ranks=[r])[0]
                assert np.array_equal(y.view(np.uint32), y_w.view(np.uint32))
        s = download(send, n * 4, np.float32, ranks=[3])[0]
        assert np.array_equal(s.view(np.uint32), s_w[3].view(np.uint32))
    finally:
        for w in (win_in, send, recv):
            w.free()


def test_scale_allreduce_validation(symar):
    a, b = symar.Window(4, 4096), symar.Window(4, 4096)
    try:
        with pytest.raises(symar.SymError):
            symar.sym_scale_allreduce(a, a, b, [1.0] * 4, 16)          # in == send
        with pytest.raises(symar.SymError):
            symar.sym_scale_allreduce(a, b, b, [1.0] * 4, 16)          # send == recv
    finally:
        a.free()
        b.free()
