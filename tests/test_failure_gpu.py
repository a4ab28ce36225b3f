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
