"""Windows from the virtual-memory allocator (sym_window_alloc_vmm): one physical
allocation per rank mapped back to back, as the symmetric allocator on the
[SYMEX] page builds them.  Every collective must give the same bits on these
windows as on cudaMalloc ones."""
import numpy as np
import pytest

from _gpu_util import download, upload

pytestmark = pytest.mark.gpu


def test_vmm_window_layout(symar):
    w = symar.Window(8, 5_000_000, nsignals=8, ncounters=1, vmm=True)
    try:
        assert w.kind in (symar.SYM_WINDOW_VMM, symar.SYM_WINDOW_VMM_EXPORTABLE)
        assert w.stride >= 5_000_000 and w.stride % (2 << 20) == 0      # whole 2 MiB pages per rank
        base = w.rank_ptr(0)
        for r in range(8):
            assert w.rank_ptr(r) == base + r * w.stride
    finally:
        w.free()


@pytest.mark.parametrize("algo", ["oneshot", "twoshot", "twoshot_pull", "twoshot_split"])
def test_vmm_allreduce_matches_oracle(symar, oracle, algo):
    R, n = 8, 3_000_017
    x = np.random.default_rng(41).standard_normal((R, n)).astype(np.float32)
    send, recv = symar.Window(R, n * 4, vmm=True), symar.Window(R, n * 4, vmm=True)
    try:
        upload(send, x)
        symar.sym_allreduce(send, recv, n, "f32", "sum", algo)
        assert symar.sym_stream_status() == symar.SYM_OK
        want = oracle.allreduce_sum_f32(x)
        y = download(recv, n * 4, np.float32)
        assert np.array_equal(y.view(np.uint32), np.broadcast_to(want.view(np.uint32), y.shape))
    finally:
        send.free()
        recv.free()


def test_vmm_put_signal_allgather(symar, oracle):
    R, S, chunk, B = 8, 4 << 20, 65536, 8
    x = np.random.default_rng(42).integers(0, 256, size=(R, S), dtype=np.uint8)
    send = symar.Window(R, S, ncounters=1, vmm=True)
    recv = symar.Window(R, R * S, nsignals=R, vmm=True)
    try:
        upload(send, x)
        symar.sym_allgather_put_signal(send, recv, S, chunk, B)
        assert symar.sym_stream_status() == symar.SYM_OK
        recv_o, sig_o, cnt_o = oracle.put_signal_allgather(x, chunk, B)
        got = download(recv, R * S, ranks=[0, R - 1])
        for i in range(2):
            assert np.array_equal(got[i], recv_o)
        for q in range(R):
            assert symar.sym_signal_read(recv, 0, q) == int(sig_o[0, q])
            assert symar.sym_counter_read(send, q, 0) == int(cnt_o[q])
    finally:
        send.free()
        recv.free()


def test_vmm_windows_free_and_reuse(symar):
    """Allocate and free VMM windows repeatedly: the reserved ranges and
    physical allocations are returned each time."""
    for _ in range(20):
        w = symar.Window(4, 64 << 20, vmm=True)
        w.free()
