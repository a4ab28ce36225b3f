"""AllReduce parity: the CUDA path (through the C ABI) against the CPU oracle.

fp32: bit-exact (same rank order, IEEE adds).  bf16: within 1 ulp of the
oracle's fp32-accumulated, once-rounded result (expected bit-exact as well;
the exact-match count is asserted separately).
"""
import os

import numpy as np
import pytest

from _gpu_util import bf16_ulp_distance, download, sync, upload

pytestmark = pytest.mark.gpu

ALGOS = ["oneshot", "twoshot", "twoshot_pull", "twoshot_split"]


def _run(sm, x, dtype, algo, in_place=False, op="sum"):
    """x: (R, n) float32 or uint16 (16-bit patterns). Returns (R, n) results of every rank."""
    R, n = x.shape
    es = x.itemsize
    send = sm.Window(R, max(n * es, 16))
    recv = send if in_place else sm.Window(R, max(n * es, 16))
    try:
        upload(send, x)
        sm.sym_allreduce(send, recv, n, dtype, op, algo)
        assert sm.sym_stream_status() == sm.SYM_OK
        return download(recv, n * es, x.dtype)
    finally:
        send.free()
        if not in_place:
            recv.free()


def _check_f32(y, want):
    assert np.array_equal(y.view(np.uint32), np.broadcast_to(want.view(np.uint32), y.shape))


def _check_bf16(y, want):
    d = bf16_ulp_distance(y, np.broadcast_to(want, y.shape))
    assert d.max(initial=0) <= 1
    assert np.array_equal(y, np.broadcast_to(want, y.shape))     # same order, one rounding


def test_worked_example_rankfill(symar, oracle):
    """4 ranks of 1,048,576 floats filled with their rank: every element 6.0."""
    from symmetric_memory_allreduce_gb300 import workloads as wl

    x = wl.workload_inputs(1, dist="rankfill")
    for algo in ALGOS:
        y = _run(symar, x, "f32", algo)
        assert np.all(np.abs(y - 6.0) <= 0.001)
        assert np.all(y == np.float32(6.0))


@pytest.mark.parametrize("algo", ALGOS)
def test_rank4_normal(symar, oracle, algo):
    from symmetric_memory_allreduce_gb300 import workloads as wl

    x = wl.workload_inputs(1, dist="normal")
    _check_f32(_run(symar, x, "f32", algo), oracle.allreduce_sum_f32(x))


# ragged sizes that span several tiles: fp32 tile = 2048 (two-shot/one-shot)
# or 4096 (pull) elements per slot chunk; tails of 1..V-1 elements
SIZES = [1, 3, 4, 5, 7, 8, 9, 63, 1000, 4097, 65_539, 100_003, 262_147]


@pytest.mark.parametrize("R", [1, 2, 3, 4, 8, 16])
@pytest.mark.parametrize("algo", ALGOS)
def test_ragged_f32(symar, oracle, R, algo):
    rng = np.random.default_rng(100 + R)
    for n in SIZES:
        x = rng.standard_normal((R, n)).astype(np.float32)
        _check_f32(_run(symar, x, "f32", algo), oracle.allreduce_sum_f32(x))


@pytest.mark.parametrize("R", [1, 2, 3, 8, 16])
@pytest.mark.parametrize("algo", ALGOS)
def test_ragged_bf16(symar, oracle, R, algo):
    from symmetric_memory_allreduce_gb300 import workloads as wl

    rng = np.random.default_rng(200 + R)
    for n in SIZES:
        x = wl.to_bf16_bits(rng.uniform(-1, 1, size=(R, n)).astype(np.float32))
        _check_bf16(_run(symar, x, "bf16", algo), oracle.allreduce_sum_bf16(x))


@pytest.mark.parametrize("algo", ["twoshot", "twoshot_pull", "twoshot_split"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_in_place(symar, oracle, algo, dtype):
    from symmetric_memory_allreduce_gb300 import workloads as wl

    rng = np.random.default_rng(7)
    for R, n in [(8, 100_003), (3, 4097), (16, 65_539)]:
        xf = rng.standard_normal((R, n)).astype(np.float32)
        if dtype == "f32":
            _check_f32(_run(symar, xf, "f32", algo, in_place=True), oracle.allreduce_sum_f32(xf))
        else:
            xb = wl.to_bf16_bits(xf)
            _check_bf16(_run(symar, xb, "bf16", algo, in_place=True), oracle.allreduce_sum_bf16(xb))


def test_in_place_oneshot_rejected(symar):
    w = symar.Window(4, 4096)
    try:
        with pytest.raises(symar.SymError) as e:
            symar.sym_allreduce(w, w, 16, "f32", "sum", "oneshot")
        assert e.value.status == symar.SYM_ERR_UNSUPPORTED
    finally:
        w.free()


def test_order_sensitive_values(symar, oracle):
    """Values whose sum depends on the order: only rank order 0..R-1 matches."""
    n = 5000
    x = np.empty((4, n), np.float32)
    x[0], x[1], x[2], x[3] = 1e8, 1.0, -1e8, 1.0        # forward 1.0, tree 0.0
    want = oracle.allreduce_sum_f32(x)
    assert np.all(want == 1.0)
    for algo in ALGOS:
        _check_f32(_run(symar, x, "f32", algo), want)


def test_special_values(symar, oracle):
    """Subnormals are not flushed; -0.0, inf and NaN propagate like the oracle."""
    tiny = np.float32(1e-45)
    base = np.array([tiny, -0.0, 1e-40, np.inf, 3.0, -2.5, 1e38, 1e38], np.float32)
    x = np.stack([base, base, np.roll(base, 1)]).astype(np.float32)
    x = np.tile(x, (1, 1000))
    want = oracle.allreduce_sum_f32(x)
    nan = np.isnan(want)
    for algo in ALGOS:
        y = _run(symar, x, "f32", algo)
        assert np.all(np.isnan(y[:, nan]))
        assert np.array_equal(y[:, ~nan].view(np.uint32),
                              np.broadcast_to(want[~nan].view(np.uint32), y[:, ~nan].shape))


def _half_inputs(dtype, f):
    from symmetric_memory_allreduce_gb300 import workloads as wl

    if dtype == "f32":
        return f
    if dtype == "bf16":
        return wl.to_bf16_bits(f)
    return np.ascontiguousarray(f.astype(np.float16).view(np.uint16))


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("op", ["sum", "max", "min"])
@pytest.mark.parametrize("algo", ALGOS)
def test_dtypes_and_ops(symar, oracle, dtype, op, algo):
    """Every (dtype, op) through every algorithm: widen, fold in rank order in fp32, narrow once."""
    rng = np.random.default_rng(300)
    for R, n in [(1, 9), (3, 4097), (8, 100_003), (16, 65_539)]:
        f = rng.uniform(-2, 2, size=(R, n)).astype(np.float32)
        f[:, ::97] = 0.0
        f[R // 2, ::89] = -0.0
        if op != "sum":
            f[0, ::101] = np.nan
        x = _half_inputs(dtype, f)
        want = oracle.allreduce(x, dtype, op)
        y = _run(symar, x, dtype, algo, op=op)
        if dtype == "f32":
            nan = np.isnan(want)
            assert np.all(np.isnan(y[:, nan]))
            assert np.array_equal(y[:, ~nan].view(np.uint32),
                                  np.broadcast_to(want[~nan].view(np.uint32), y[:, ~nan].shape))
        else:
            nanbits = (want & 0x7FFF) > (0x7F80 if dtype == "bf16" else 0x7C00)
            assert np.array_equal(y[:, ~nanbits], np.broadcast_to(want[~nanbits], y[:, ~nanbits].shape))


def test_f16_rounding_edges(symar, oracle):
    """fp16 sums that overflow to Inf, land on subnormals, or tie in rounding."""
    R, n = 4, 4096
    rng = np.random.default_rng(301)
    f = np.empty((R, n), np.float32)
    f[:] = rng.choice([65504.0, 30000.0, 2.0 ** -24, 2.0 ** -15, 1.0, 2.0 ** -11, -65504.0],
                      size=(R, n)).astype(np.float32)
    x = _half_inputs("f16", f)
    for algo in ALGOS:
        want = oracle.allreduce(x, "f16", "sum")
        assert np.array_equal(_run(symar, x, "f16", algo), np.broadcast_to(want, (R, n)))


def test_zero_count_and_validation(symar):
    a, b = symar.Window(4, 4096), symar.Window(8, 4096)
    try:
        n0 = symar.sym_launch_count()
        symar.sym_allreduce(a, a, 0, "f32", "sum", "twoshot")            # no-op
        assert symar.sym_launch_count() == n0
        for bad in [lambda: symar.sym_allreduce(a, b, 16),               # different R
                    lambda: symar.sym_allreduce(a, a, 1025),             # too many elements
                    lambda: symar.sym_allreduce(a, a, 16, "f32", "sum", 99)]:
            with pytest.raises(symar.SymError) as e:
                bad()
            assert e.value.status == symar.SYM_ERR_INVALID_ARG
        with pytest.raises(symar.SymError) as e:
            symar.sym_allreduce(a, a, 16, "f32", 7, "twoshot")             # unknown op
        assert e.value.status == symar.SYM_ERR_INVALID_ARG
    finally:
        a.free()
        b.free()


def test_repeat_calls_reuse_windows(symar, oracle):
    """Epoch-tagged flags: repeated pull calls on the same windows need no reset."""
    rng = np.random.default_rng(3)
    R, n = 8, 300_001
    send, recv = symar.Window(R, n * 4), symar.Window(R, n * 4)
    try:
        for it in range(5):
            x = rng.standard_normal((R, n)).astype(np.float32)
            upload(send, x)
            symar.sym_allreduce(send, recv, n, "f32", "sum", "twoshot_pull")
            assert symar.sym_stream_status() == symar.SYM_OK
            _check_f32(download(recv, n * 4, np.float32), oracle.allreduce_sum_f32(x))
    finally:
        send.free()
        recv.free()


def test_registered_torch_memory(symar, oracle):
    """sym_window_register over a torch allocation (caller-owned memory)."""
    import torch

    R, n = 4, 70_000
    stride = ((n * 4 + 4095) // 4096) * 4096
    buf_s = torch.empty(R * stride, dtype=torch.uint8, device="cuda")
    buf_r = torch.empty(R * stride, dtype=torch.uint8, device="cuda")
    send = symar.Window(R, n * 4, base=buf_s.data_ptr(), stride=stride, keepalive=buf_s)
    recv = symar.Window(R, n * 4, base=buf_r.data_ptr(), stride=stride, keepalive=buf_r)
    try:
        x = np.random.default_rng(5).standard_normal((R, n)).astype(np.float32)
        upload(send, x)
        symar.sym_allreduce(send, recv, n, "f32", "sum", "twoshot")
        sync()
        y = buf_r.view(R, stride)[:, : n * 4].contiguous().view(torch.float32).cpu().numpy()
        _check_f32(y, oracle.allreduce_sum_f32(x))
        # the window's own tensor view sees the same memory
        t = recv.tensor(torch.float32)
        assert torch.equal(t[:, :n], torch.from_numpy(y).cuda())
    finally:
        send.free()
        recv.free()


# ---------------------------------------------------------------- full-size workloads

def _full(symar, oracle, x, dtype, algos):
    R, n = x.shape
    es = x.itemsize
    send, recv = symar.Window(R, n * es), symar.Window(R, n * es)
    try:
        upload(send, x)
        if dtype == "f32":
            want, _ = oracle.allreduce_sum_mt(x, 16)
        else:
            want, _ = oracle.allreduce_sum_mt(x, 16)
        for algo in algos:
            symar.sym_allreduce(send, recv, n, dtype, "sum", algo)
            assert symar.sym_stream_status() == symar.SYM_OK
            for r in range(R):
                y = download(recv, n * es, x.dtype, ranks=[r])[0]
                if dtype == "f32":
                    assert np.array_equal(y.view(np.uint32), want.view(np.uint32)), (algo, r)
                else:
                    assert bf16_ulp_distance(y, want).max() <= 1, (algo, r)
                    assert np.array_equal(y, want), (algo, r)
            recv.tensor().zero_()
            sync()
    finally:
        send.free()
        recv.free()


def test_full_R8x64MiB(symar, oracle):
    """R=8 x 16,777,216 fp32 N(0,1): one-shot and two-shot, every rank bit-exact."""
    from symmetric_memory_allreduce_gb300 import workloads as wl

    _full(symar, oracle, wl.workload_inputs(2), "f32", ALGOS)


def test_full_R8x256MiB_f32(symar, oracle):
    """R=8 x 67,108,864 fp32 U(-1,1) (256 MiB per rank), two-shot forms."""
    from symmetric_memory_allreduce_gb300 import workloads as wl

    _full(symar, oracle, wl.workload_inputs(3), "f32", ["twoshot", "twoshot_pull", "twoshot_split", "auto"])


def test_full_R8x128MiB_bf16(symar, oracle):
    """The same draws rounded to bf16 (128 MiB per rank), fp32 accumulation."""
    from symmetric_memory_allreduce_gb300 import workloads as wl

    xb = wl.to_bf16_bits(wl.workload_inputs(3))
    _full(symar, oracle, xb, "bf16", ["twoshot", "twoshot_pull", "twoshot_split"])


def test_full_R8x128MiB_f16(symar, oracle):
    """The same draws rounded to fp16 (128 MiB per rank): fp32 accumulation in rank
    order, one rounding, bit-exact on every rank for the two-shot forms."""
    from symmetric_memory_allreduce_gb300 import workloads as wl

    x = np.ascontiguousarray(wl.workload_inputs(3).astype(np.float16).view(np.uint16))
    R, n = x.shape
    want = oracle.allreduce(x, "f16", "sum")
    send, recv = symar.Window(R, n * 2), symar.Window(R, n * 2)
    try:
        upload(send, x)
        for algo in ["twoshot", "twoshot_pull", "twoshot_split"]:
            symar.sym_allreduce(send, recv, n, "f16", "sum", algo)
            assert symar.sym_stream_status() == symar.SYM_OK
            for r in (0, R // 2, R - 1):
                y = download(recv, n * 2, np.uint16, ranks=[r])[0]
                assert np.array_equal(y, want), (algo, r)
            recv.tensor().zero_()
            sync()
    finally:
        send.free()
        recv.free()


@pytest.mark.parametrize("nbytes", [1024 * 4 ** k for k in range(10)])
def test_size_sweep(symar, oracle, nbytes):
    """R=8, 1 KiB .. 256 MiB per rank, fp32 N(0,1), every algorithm and AUTO."""
    from symmetric_memory_allreduce_gb300 import workloads as wl

    x = wl.workload_inputs(4, n=nbytes // 4)
    _full(symar, oracle, x, "f32", ALGOS + ["auto"])


def test_size_sweep_1gib_full(symar, oracle):
    """The 1 GiB-per-rank point, every element of every rank against the oracle
    ([SYMEX] Example 1 step 6 checks every element), for every algorithm and AUTO.
    Host memory: the 8 GiB of inputs, the 1 GiB oracle result and one rank's output."""
    from symmetric_memory_allreduce_gb300 import workloads as wl

    R, n = 8, (1 << 30) // 4
    x = wl.workload_inputs(4, n=n)
    send, recv = symar.Window(R, n * 4), symar.Window(R, n * 4)
    try:
        upload(send, x)
        want, _ = oracle.allreduce_sum_mt(x, os.cpu_count() or 1)
        del x
        want_u = want.view(np.uint32)
        y = np.empty(n, np.float32)
        for algo in ["oneshot", "twoshot", "twoshot_pull", "twoshot_split", "auto"]:
            symar.sym_allreduce(send, recv, n, "f32", "sum", algo)
            assert symar.sym_stream_status() == symar.SYM_OK
            for r in range(R):
                recv.read(r, y)
                sync()
                assert np.array_equal(y.view(np.uint32), want_u), (algo, r)
            recv.tensor().zero_()
            sync()
    finally:
        send.free()
        recv.free()
