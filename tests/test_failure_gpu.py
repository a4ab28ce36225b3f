"""Failure detection without a GPU fault: a put + signal AllGather whose (0 -> 0)
stream omits its last signal (host-side fault injection, SYM_TEST_DROP_LAST_SIGNAL)
leaves one receiver waiting on a signal that nothing will set.  The wait must
run out within its limit, the launch's other waits must not be held up, the host
must read SYM_ERR_TIMEOUT, and the context must stay usable afterwards.  Runs in
a child process because the switch is read once per process."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_SCRIPT = r"""
import sys, time
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import numpy as np
import torch
import oracle
import symmetric_memory_allreduce_gb300 as sm
from _gpu_util import upload, download
sm.load(); oracle.build()
R, S, chunk, B = 8, 1 << 20, 65536, 4
x = np.random.default_rng(9).integers(0, 256, size=(R, S), dtype=np.uint8)
send, recv = sm.Window(R, S, ncounters=1), sm.Window(R, R * S, nsignals=R)
upload(send, x)
t0 = time.time()
sm.sym_allgather_put_signal(send, recv, S, chunk, B, timeout_ns=50_000_000)
st = sm.sym_stream_status()
dt = time.time() - t0
print("STATUS", sm.sym_status_string(st), "SECONDS", round(dt, 3), "WHERE", sm.sym_last_error())
assert st == sm.SYM_ERR_TIMEOUT, st
assert dt < 10.0
# every other (p, q) stream completed; only (0 <- 0) is one short
assert sm.sym_signal_read(recv, 0, 0) == (S // chunk) // B - 1
assert sm.sym_signal_read(recv, 1, 0) == (S // chunk) // B
# the bytes all arrived (only the signal was dropped)
assert np.array_equal(download(recv, R * S, ranks=[3])[0], oracle.allgather(x))
# the context stays usable: a normal AllReduce afterwards
y = np.random.default_rng(1).standard_normal((R, 1000)).astype(np.float32)
a, b = sm.Window(R, 4000), sm.Window(R, 4000)
upload(a, y)
sm.sym_allreduce(a, b, 1000, "f32", "sum", "twoshot_pull")
assert sm.sym_stream_status() == sm.SYM_OK
got = download(b, 4000, np.float32)
assert np.array_equal(got[0].view(np.uint32), oracle.allreduce_sum_f32(y).view(np.uint32))
print("FAILURE_TEST_OK")
"""


def test_dropped_signal_times_out_cleanly():
    env = dict(os.environ, SYM_TEST_DROP_LAST_SIGNAL="1")
    out = subprocess.run([sys.executable, "-c", _SCRIPT.format(root=ROOT,
                                                               tests=os.path.join(ROOT, "tests"))],
                         env=env, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stdout[-3000:] + out.stderr[-3000:]
    assert "FAILURE_TEST_OK" in out.stdout
    assert "site 4" in out.stdout          # the put + signal receiver reported it


_SCRIPT_FIRST = r"""
import sys, time
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import numpy as np
import oracle
import symmetric_memory_allreduce_gb300 as sm
from _gpu_util import upload, download
sm.load(); oracle.build()
# enough work items (8 senders x 64 batches of 8 chunks) that the receivers,
# which come after every put, start long after the stream's second batch
# begins to wait for the missing first signal
R, S, chunk, B = 8, 32 << 20, 65536, 8
x = np.random.default_rng(10).integers(0, 256, size=(R, S), dtype=np.uint8)
send, recv = sm.Window(R, S, ncounters=1), sm.Window(R, R * S, nsignals=R)
upload(send, x)
t0 = time.time()
sm.sym_allgather_put_signal(send, recv, S, chunk, B, timeout_ns=50_000_000)
st = sm.sym_stream_status()
dt = time.time() - t0
print("STATUS", sm.sym_status_string(st), "SECONDS", round(dt, 3), "WHERE", sm.sym_last_error())
assert st == sm.SYM_ERR_TIMEOUT, st
assert dt < 10.0
# batch 0 of (0 -> 0) never signalled, so no later batch of that stream may signal
assert sm.sym_signal_read(recv, 0, 0) == 0
# the bytes all arrived (the copies do not wait; only the signals are ordered)
assert np.array_equal(download(recv, R * S, ranks=[0])[0], oracle.allgather(x))
# the context stays usable
y = np.random.default_rng(2).standard_normal((R, 1000)).astype(np.float32)
a, b = sm.Window(R, 4000), sm.Window(R, 4000)
upload(a, y)
sm.sym_allreduce(a, b, 1000, "f32", "sum", "twoshot_pull")
assert sm.sym_stream_status() == sm.SYM_OK
got = download(b, 4000, np.float32)
assert np.array_equal(got[0].view(np.uint32), oracle.allreduce_sum_f32(y).view(np.uint32))
print("FAILURE_TEST_OK")
"""


def test_dropped_first_signal_stops_the_stream_in_order():
    """The (0 -> 0) stream omits its first signal (SYM_TEST_DROP_SIGNAL=first):
    the put of its second batch waits for it to keep the signals in batch order,
    runs out (site 6), and no later signal of the stream is added."""
    env = dict(os.environ, SYM_TEST_DROP_SIGNAL="first")
    out = subprocess.run([sys.executable, "-c", _SCRIPT_FIRST.format(root=ROOT,
                                                                     tests=os.path.join(ROOT, "tests"))],
                         env=env, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stdout[-3000:] + out.stderr[-3000:]
    assert "FAILURE_TEST_OK" in out.stdout
    assert "site 6" in out.stdout          # the batch-order wait reported it


_PULL_GIVE_UP = r"""
import sys, time
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import numpy as np
import oracle
import symmetric_memory_allreduce_gb300 as sm
from _gpu_util import upload, download
sm.load(); oracle.build()
for R, n in ((8, 1 << 22), (8, 40_000)):       # the warp-specialised kernel, then the single-role one
    x = np.random.default_rng(n).standard_normal((R, n)).astype(np.float32)
    want = oracle.allreduce_sum_f32(x)
    a, b = sm.Window(R, n * 4), sm.Window(R, n * 4)
    upload(a, x)
    t0 = time.time()
    sm.sym_allreduce(a, b, n, "f32", "sum", "twoshot_pull")
    st = sm.sym_stream_status()
    dt = time.time() - t0
    print("N", n, "STATUS", sm.sym_status_string(st), "SECONDS", round(dt, 3), "WHERE", sm.sym_last_error())
    assert dt < 10.0
    y = download(b, n * 4, np.float32)
    if st == sm.SYM_OK:
        assert all(np.array_equal(y[r].view(np.uint32), want.view(np.uint32)) for r in range(R))
    else:
        assert st == sm.SYM_ERR_TIMEOUT and "site 3" in sm.sym_last_error()
        # reducers never wait: every slot's own chunk is complete even when pulls gave up
        nvec = n * 4 // 16
        cv = -(-nvec // R) * 4
        for q in range(R):
            lo, hi = q * cv, min((q + 1) * cv, nvec * 4)
            assert np.array_equal(y[q, lo:hi].view(np.uint32), want[lo:hi].view(np.uint32)), q
    # the context stays usable: the store-form two-shot (no waits) afterwards is exact
    sm.sym_allreduce(a, b, n, "f32", "sum", "twoshot")
    assert sm.sym_stream_status() == sm.SYM_OK
    y = download(b, n * 4, np.float32)
    assert all(np.array_equal(y[r].view(np.uint32), want.view(np.uint32)) for r in range(R))
    a.free(); b.free()
print("PULL_GIVE_UP_OK")
"""


def test_pull_waits_give_up_cleanly():
    """Pull two-shot with every flag wait bounded at 1 ns: pulls that find their tile's flag
    unset give up (the launch ends, SYM_ERR_TIMEOUT at the pull-flag site), the slots' own
    reduced chunks are still exact, and the context stays usable."""
    env = dict(os.environ, SYM_TIMEOUT_NS="1")
    out = subprocess.run([sys.executable, "-c", _PULL_GIVE_UP.format(root=ROOT,
                                                                     tests=os.path.join(ROOT, "tests"))],
                         env=env, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stdout[-3000:] + out.stderr[-3000:]
    assert "PULL_GIVE_UP_OK" in out.stdout
