"""AllGather, put+signal and signal/counter parity on the GPU (through the C ABI).

Bytes and counts are bit-exact against the oracle; device waits are bounded, and
the timeout case uses a signal that nothing sets (no GPU fault, no hang).
"""
import numpy as np
import pytest

from _gpu_util import download, sync, upload

pytestmark = pytest.mark.gpu


def test_allgather_worked_example(symar, oracle):
    """4 ranks of 1,048,576 floats filled with their rank: segment q holds q.0 everywhere."""
    R, n = 4, 1 << 20
    x = np.repeat(np.arange(R, dtype=np.float32)[:, None], n, axis=1)
    send, recv = symar.Window(R, n * 4), symar.Window(R, R * n * 4)
    try:
        upload(send, x)
        symar.sym_allgather(send, recv, n, "f32", "copy")
        assert symar.sym_stream_status() == symar.SYM_OK
        y = download(recv, R * n * 4, np.float32)
        for q in range(R):
            assert np.all(y[:, q * n:(q + 1) * n] == float(q))
        assert np.array_equal(y[0].view(np.uint8), oracle.allgather(x.view(np.uint8)))
    finally:
        send.free()
        recv.free()


@pytest.mark.parametrize("R,S", [(1, 48), (3, 4096 + 16), (16, 65536), (5, 1001), (8, 6),
                                 (16, 1 << 20)])
@pytest.mark.parametrize("algo", ["copy", "put_signal", "ce"])
def test_allgather_random_bytes(symar, oracle, R, S, algo):
    rng = np.random.default_rng(R * 1000 + S)
    x = rng.integers(0, 256, size=(R, S), dtype=np.uint8)
    send, recv = symar.Window(R, S, ncounters=1), symar.Window(R, R * S, nsignals=R)
    try:
        upload(send, x)
        es = 4 if S % 4 == 0 else (2 if S % 2 == 0 else 1)
        if algo == "put_signal":
            symar.sym_allgather_put_signal(send, recv, S, 256, 3)
        elif es == 1:
            pytest.skip("a dtype must divide the bytes; odd sizes are covered by put_signal")
        else:
            symar.sym_allgather(send, recv, S // es, "f32" if es == 4 else "bf16", algo)
        assert symar.sym_stream_status() == symar.SYM_OK
        want = oracle.allgather(x)
        got = download(recv, R * S)
        for r in range(R):
            assert np.array_equal(got[r], want), r
        if algo == "put_signal":
            nchunks = -(-S // 256)
            for p in range(R):
                for q in range(R):
                    assert symar.sym_signal_read(recv, p, q) == -(-nchunks // 3)
            for q in range(R):
                assert symar.sym_counter_read(send, q, 0) == R * nchunks
    finally:
        send.free()
        recv.free()


@pytest.mark.parametrize("batch", [8, 1, 64])
def test_put_signal_full_R16x32MiB(symar, oracle, batch):
    """R=16, 32 MiB per rank, 64 KiB chunks: bytes, signal counts, counters, and the
    prefix-visibility check made by the receivers while the senders run."""
    import torch
    from symmetric_memory_allreduce_gb300 import workloads as wl

    cfg = wl.PUT_SIGNAL
    R, S, chunk = cfg["R"], cfg["nbytes"], cfg["chunk"]
    x = wl.random_bytes(5, R, S)
    recv_o, sig_o, cnt_o = oracle.put_signal_allgather(x, chunk, batch)
    send, recv = symar.Window(R, S, ncounters=1), symar.Window(R, R * S, nsignals=R)
    mism = torch.zeros(1, dtype=torch.int64, device="cuda")
    try:
        upload(send, x)
        symar.sym_allgather_put_signal(send, recv, S, chunk, batch, d_mismatch=mism.data_ptr())
        assert symar.sym_stream_status() == symar.SYM_OK
        assert int(mism.item()) == 0
        for p in range(R):
            got = download(recv, R * S, ranks=[p])[0]
            assert np.array_equal(got, recv_o), p
            for q in range(R):
                assert symar.sym_signal_read(recv, p, q) == int(sig_o[p, q])
        assert all(int(sig_o[p, q]) == -(-512 // batch) for p in range(R) for q in range(R))
        for q in range(R):
            assert symar.sym_counter_read(send, q, 0) == int(cnt_o[q]) == R * 512
        # the timed form (no check) gives the same bytes and counts
        recv.tensor().zero_()
        symar.sym_allgather(send, recv, S // 4, "f32", "put_signal", chunk, batch)
        assert symar.sym_stream_status() == symar.SYM_OK
        got = download(recv, R * S, ranks=[R - 1])[0]
        assert np.array_equal(got, recv_o)
        assert symar.sym_signal_read(recv, 3, 7) == -(-512 // batch)
    finally:
        send.free()
        recv.free()


def test_put_signal_rankfill_bytes(symar, oracle):
    """Byte fill (rank q writes the byte q): segment q of every receiver is all q."""
    R, S = 16, 3 * 65536 + 4096
    x = np.tile(np.arange(R, dtype=np.uint8)[:, None], (1, S))
    send, recv = symar.Window(R, S, ncounters=1), symar.Window(R, R * S, nsignals=R)
    try:
        upload(send, x)
        symar.sym_allgather_put_signal(send, recv, S, 65536, 2)
        assert symar.sym_stream_status() == symar.SYM_OK
        got = download(recv, R * S)
        for q in range(R):
            assert np.all(got[:, q * S:(q + 1) * S] == q)
        assert symar.sym_signal_read(recv, 0, 15) == 2     # 4 chunks in batches of 2
    finally:
        send.free()
        recv.free()


def test_single_put_signal_counter(symar):
    R = 4
    src, dst = symar.Window(R, 1 << 20, ncounters=2), symar.Window(R, 1 << 20, nsignals=3)
    try:
        data = np.random.default_rng(2).integers(0, 256, size=(R, 1 << 20), dtype=np.uint8)
        upload(src, data)
        # aligned, multi-CTA put with both actions
        symar.sym_put_signal(src, dst, 2, 1, 4096, 8192, 600_000 // 16 * 16, signal_id=2,
                             counter_id=1)
        # unaligned put, loopback (peer == src rank), no counter
        symar.sym_put_signal(src, dst, 1, 1, 700_001, 3, 1001, signal_id=2)
        symar.sym_signal_wait(dst, 1, 2, 2, timeout_ns=2_000_000_000)
        assert symar.sym_stream_status() == symar.SYM_OK
        got = download(dst, 1 << 20, ranks=[1])[0]
        n1 = 600_000 // 16 * 16
        assert np.array_equal(got[4096:4096 + n1], data[2, 8192:8192 + n1])
        assert np.array_equal(got[700_001:700_001 + 1001], data[1, 3:3 + 1001])
        assert symar.sym_signal_read(dst, 1, 2) == 2
        assert symar.sym_counter_read(src, 2, 1) == 1
        assert symar.sym_counter_read(src, 1, 1) == 0
        symar.sym_signal(dst, 3, 0, 41)
        symar.sym_signal(dst, 3, 0, 1)
        assert symar.sym_signal_read(dst, 3, 0) == 42
        symar.sym_signal_reset(dst, 3, 0)
        assert symar.sym_signal_read(dst, 3, 0) == 0
        # overlapping src/dst ranges and out-of-window ranges are rejected on the host
        with pytest.raises(symar.SymError):
            symar.sym_put_signal(src, src, 0, 0, 16, 0, 64)
        with pytest.raises(symar.SymError):
            symar.sym_put_signal(src, dst, 0, 0, (1 << 20) - 8, 0, 16)
        with pytest.raises(symar.SymError):
            symar.sym_put_signal(src, dst, 0, 0, 0, 0, 16, signal_id=3)
    finally:
        src.free()
        dst.free()


def test_many_puts_one_stream_strong_order(symar):
    """A chain of puts to one peer, each signalling; the final wait covers all of them."""
    R, n, k = 2, 1 << 16, 64
    src, dst = symar.Window(R, n * k), symar.Window(R, n * k, nsignals=1)
    try:
        data = np.random.default_rng(8).integers(0, 256, size=(R, n * k), dtype=np.uint8)
        upload(src, data)
        for i in range(k):
            symar.sym_put_signal(src, dst, 0, 1, i * n, i * n, n, signal_id=0)
        symar.sym_signal_wait(dst, 1, 0, k)
        assert symar.sym_stream_status() == symar.SYM_OK
        assert np.array_equal(download(dst, n * k, ranks=[1])[0], data[0])
    finally:
        src.free()
        dst.free()


def test_wait_timeout_reports_status(symar, oracle):
    """A wait on a signal that nothing sets returns SYM_ERR_TIMEOUT; the context stays usable."""
    import time

    w = symar.Window(2, 4096, nsignals=1, ncounters=1)
    try:
        symar.sym_signal(w, 0, 0, 5)
        t0 = time.time()
        symar.sym_signal_wait(w, 0, 0, 6, timeout_ns=50_000_000)        # 50 ms
        st = symar.sym_stream_status()
        dt = time.time() - t0
        assert st == symar.SYM_ERR_TIMEOUT, symar.sym_status_string(st)
        assert dt < 5.0
        assert "site 1" in symar.sym_last_error()
        assert symar.sym_stream_status() == symar.SYM_OK               # cleared
        symar.sym_counter_wait(w, 1, 0, 1, timeout_ns=20_000_000)
        assert symar.sym_stream_status() == symar.SYM_ERR_TIMEOUT
        # still usable afterwards
        x = np.random.default_rng(0).standard_normal((2, 1000)).astype(np.float32)
        a, b = symar.Window(2, 4000), symar.Window(2, 4000)
        upload(a, x)
        symar.sym_allreduce(a, b, 1000, "f32", "sum", "twoshot_pull")
        assert symar.sym_stream_status() == symar.SYM_OK
        y = download(b, 4000, np.float32)
        assert np.array_equal(y[0].view(np.uint32), oracle.allreduce_sum_f32(x).view(np.uint32))
        a.free()
        b.free()
    finally:
        w.free()


def test_rolling_wait_semantics(symar, oracle):
    """waitSignal's rolling comparison across 64-bit wrap and on 8 low bits."""
    w = symar.Window(1, 4096, nsignals=2)
    try:
        M = 2**64 - 1
        symar.sym_signal(w, 0, 0, M)                    # value 2^64-1
        assert symar.sym_signal_read(w, 0, 0) == M
        symar.sym_signal(w, 0, 0, 2)                    # wraps to 1
        assert symar.sym_signal_read(w, 0, 0) == 1
        assert oracle.rolling_le(M, 1)
        symar.sym_signal_wait(w, 0, 0, M, timeout_ns=50_000_000)     # M <= 1 (rolling)
        assert symar.sym_stream_status() == symar.SYM_OK
        symar.sym_signal(w, 0, 1, 0x1FF)                # low 8 bits = 0xFF
        assert symar.sym_signal_read(w, 0, 1, bits=8) == 0xFF
        symar.sym_signal_wait(w, 0, 1, 0xF0, bits=8, timeout_ns=50_000_000)
        assert symar.sym_stream_status() == symar.SYM_OK
        assert not oracle.rolling_le(0x7F, 0xFF, 8)     # half-range apart: not reached
        symar.sym_signal_wait(w, 0, 1, 0x7F, bits=8, timeout_ns=20_000_000)
        assert symar.sym_stream_status() == symar.SYM_ERR_TIMEOUT
    finally:
        w.free()


def _rolling_cases(rng):
    """(least, value, bits) around the wrap and the half-range edge, with high bits set."""
    cases = []
    for n in (1, 2, 3, 7, 8, 16, 32, 55, 56, 57, 63, 64):
        mod, half = 1 << n, 1 << (n - 1)
        anchors = sorted({0, 1, half - 1, half, mod - 1, int(rng.integers(0, mod, dtype=np.uint64))})
        for a in anchors:
            for d in sorted({0, 1, half - 1, half, half + 1, mod - 1} - {mod}):
                v = (a + d) % mod
                least = a
                if n < 64:                      # bits above the mask must not matter
                    v |= int(rng.integers(0, 1 << (64 - n), dtype=np.uint64)) << n
                    least |= int(rng.integers(0, 1 << (64 - n), dtype=np.uint64)) << n
                cases.append((least, v, n))
    return cases


def test_rolling_wait_sweep_matches_oracle(symar, oracle):
    """sym_signal_wait ends (SYM_OK) or runs out (SYM_ERR_TIMEOUT, 1 ms bound) exactly when the
    oracle's rolling_le(least, value, bits) says the value has or has not reached `least`:
    [GIN] "Signals and Counters", waitSignal(least, bits) on the rolling comparison."""
    cases = _rolling_cases(np.random.default_rng(1982))
    w = symar.Window(1, 4096, nsignals=len(cases))
    try:
        for i, (_, v, _) in enumerate(cases):
            if v:
                symar.sym_signal(w, 0, i, v)             # slots start at 0
        assert symar.sym_stream_status() == symar.SYM_OK
        reached = timed_out = 0
        for i, (least, v, n) in enumerate(cases):
            assert symar.sym_signal_read(w, 0, i) == v
            want = oracle.rolling_le(least, v, n)
            symar.sym_signal_wait(w, 0, i, least, bits=n, timeout_ns=1_000_000)
            st = symar.sym_stream_status()
            assert st == (symar.SYM_OK if want else symar.SYM_ERR_TIMEOUT), (hex(least), hex(v), n)
            reached += want
            timed_out += not want
        assert reached > 100 and timed_out > 100
    finally:
        w.free()


def test_rolling_counter_wait_matches_oracle(symar, oracle):
    """waitCounter on 1..3 low bits of a counter at 3 (three puts): the rolling outcome, not <=."""
    src, dst = symar.Window(2, 4096, ncounters=1), symar.Window(2, 4096, nsignals=1)
    try:
        for _ in range(3):
            symar.sym_put_signal(src, dst, 0, 1, 0, 16, 32, counter_id=0)
        assert symar.sym_counter_read(src, 0, 0) == 3
        for n in (1, 2, 3, 56):
            for least in range(8):
                want = oracle.rolling_le(least, 3, n)
                symar.sym_counter_wait(src, 0, 0, least, bits=n, timeout_ns=1_000_000)
                st = symar.sym_stream_status()
                assert st == (symar.SYM_OK if want else symar.SYM_ERR_TIMEOUT), (least, n)
    finally:
        src.free()
        dst.free()


def test_counter_56_bits(symar):
    src, dst = symar.Window(2, 4096, ncounters=1), symar.Window(2, 4096, nsignals=1)
    try:
        for _ in range(3):
            symar.sym_put_signal(src, dst, 0, 1, 0, 16, 32, counter_id=0)
        assert symar.sym_counter_read(src, 0, 0) == 3
        assert symar.sym_counter_read(src, 0, 0, bits=1) == 1
        symar.sym_counter_reset(src, 0, 0)
        assert symar.sym_counter_read(src, 0, 0) == 0
        with pytest.raises(symar.SymError):
            symar.sym_counter_read(src, 0, 0, bits=57)
    finally:
        src.free()
        dst.free()


@pytest.mark.parametrize("algo", ["copy", "put_signal"])
def test_alltoall_gin_pattern(symar, oracle, algo):
    """The GIN page's AlltoAll check: rank p finds my_rank*1000 + dest_rank*100 + idx from q."""
    R, count = 8, 4096 + 3
    send_h = np.empty((R, R * count), np.float32)
    for q in range(R):
        for p in range(R):
            send_h[q, p * count:(p + 1) * count] = q * 1000 + p * 100 + np.arange(count)
    send, recv = symar.Window(R, R * count * 4), symar.Window(R, R * count * 4, nsignals=1)
    try:
        upload(send, send_h)
        symar.sym_alltoall(send, recv, count, "f32", algo)
        assert symar.sym_stream_status() == symar.SYM_OK
        got = download(recv, R * count * 4, np.float32)
        for p in range(R):
            for q in range(R):
                assert np.array_equal(got[p, q * count:(q + 1) * count],
                                      q * 1000 + p * 100 + np.arange(count, dtype=np.float32))
        assert np.array_equal(got.view(np.uint8), oracle.alltoall(send_h.view(np.uint8)))
        if algo == "put_signal":
            assert all(symar.sym_signal_read(recv, p, 0) == R for p in range(R))
    finally:
        send.free()
        recv.free()


@pytest.mark.parametrize("R,B", [(1, 16), (3, 6), (16, 65536), (5, 1000)])
def test_alltoall_random(symar, oracle, R, B):
    rng = np.random.default_rng(R + B)
    x = rng.integers(0, 256, size=(R, R * B), dtype=np.uint8)
    send, recv = symar.Window(R, R * B), symar.Window(R, R * B, nsignals=2)
    try:
        upload(send, x)
        es = 4 if B % 4 == 0 else 2
        for algo in ("copy", "put_signal"):
            recv.tensor().zero_()
            symar.sym_alltoall(send, recv, B // es, "f32" if es == 4 else "bf16", algo)
            assert symar.sym_stream_status() == symar.SYM_OK
            assert np.array_equal(download(recv, R * B), oracle.alltoall(x))
    finally:
        send.free()
        recv.free()


def test_get_reads_peer_into_local(symar, oracle):
    """[GIN] get: rank `rank` reads peer's bytes into its own window; the optional
    local counter counts completed gets; loopback and argument checks."""
    R, S = 4, 300_000 + 16
    x = np.random.default_rng(61).integers(0, 256, size=(R, S), dtype=np.uint8)
    remote, local = symar.Window(R, S), symar.Window(R, 2 * S, ncounters=2)
    try:
        upload(remote, x)
        local.tensor().zero_()
        # rank 1 gets peer 3's bytes 1000.. into its window at offset 16 (vector path)
        symar.sym_get(remote, local, 1, 3, 16, 1008, 200_000, counter_id=1)
        # rank 2 gets peer 0's bytes at odd offsets (byte path)
        symar.sym_get(remote, local, 2, 0, S + 3, 5, 77_777, counter_id=1)
        # loopback: rank 0 reads its own part of `local`, non-overlapping ranges
        symar.sym_get(local, local, 0, 0, S, 0, 1000)
        assert symar.sym_stream_status() == symar.SYM_OK
        got = download(local, 2 * S)
        assert np.array_equal(got[1, 16:16 + 200_000], x[3, 1008:1008 + 200_000])
        assert np.array_equal(got[2, S + 3:S + 3 + 77_777], x[0, 5:5 + 77_777])
        assert not got[1, :16].any() and not got[1, 16 + 200_000:].any()
        assert symar.sym_counter_read(local, 1, 1) == 1
        assert symar.sym_counter_read(local, 2, 1) == 1
        assert symar.sym_counter_read(local, 0, 1) == 0
        with pytest.raises(symar.SymError):
            symar.sym_get(remote, local, 0, 4, 0, 0, 16)          # peer out of range
        with pytest.raises(symar.SymError):
            symar.sym_get(remote, local, 0, 0, 0, S - 8, 16)      # past the remote window
        with pytest.raises(symar.SymError):
            symar.sym_get(local, local, 0, 0, 0, 8, 64)           # overlapping loopback
        with pytest.raises(symar.SymError):
            symar.sym_get(remote, local, 0, 0, 0, 0, 16, counter_id=2)   # no such counter
    finally:
        remote.free()
        local.free()


@pytest.mark.parametrize("R", [1, 3, 8, 64])
def test_barrier_adds_R_per_call(symar, R):
    """[GIN] barrier session, signal form: each call adds exactly R to every
    rank's slot and returns once all R adds have arrived, also when recorded in
    a CUDA graph and replayed."""
    import torch

    w = symar.Window(R, 4096, nsignals=2)
    try:
        for k in range(1, 4):
            symar.sym_barrier(w, 1, timeout_ns=1_000_000_000)
            assert symar.sym_stream_status() == symar.SYM_OK
            for r in range(R):
                assert symar.sym_signal_read(w, r, 1) == k * R
                assert symar.sym_signal_read(w, r, 0) == 0
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            symar.sym_barrier(w, 1, timeout_ns=1_000_000_000, stream=s)
        for k in range(4, 7):
            g.replay()
            torch.cuda.synchronize()
            assert symar.sym_stream_status() == symar.SYM_OK
            assert all(symar.sym_signal_read(w, r, 1) == k * R for r in range(R))
    finally:
        w.free()
