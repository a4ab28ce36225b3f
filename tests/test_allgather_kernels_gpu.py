"""Parity of both AllGather copy kernels: the one staged through shared memory
by bulk copies (TMA engine, the default) and the register load/store one
(SYM_ALLGATHER_KERNEL=ldst), each in a child process (the choice is read once
per process).  Bytes are compared bit-exactly with the oracle."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_SCRIPT = r"""
import sys
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import numpy as np
import oracle
import symmetric_memory_allreduce_gb300 as sm
from _gpu_util import upload, download
sm.load(); oracle.build()
rng = np.random.default_rng(23)
# segment sizes: one vector, ragged tails past whole 16 KiB tiles, many tiles,
# and a non-multiple of 16 (byte-granular kernel)
for R in (1, 2, 3, 8, 16):
    for S in (16, 4096 + 16, 3 * 16384 + 48, 1 << 20, (1 << 20) + 16400, 1002):
        x = rng.integers(0, 256, size=(R, S), dtype=np.uint8)
        send, recv = sm.Window(R, S), sm.Window(R, R * S)
        upload(send, x)
        es = 4 if S % 4 == 0 else 2
        sm.sym_allgather(send, recv, S // es, "f32" if es == 4 else "bf16", "copy")
        assert sm.sym_stream_status() == sm.SYM_OK, sm.sym_last_error()
        want = oracle.allgather(x)
        got = download(recv, R * S)
        for r in range(R):
            assert np.array_equal(got[r], want), (R, S, r)
        send.free(); recv.free()
# the put + signal workload's shape: 16 ranks x 32 MiB, two calls in a row
R, S = 16, 32 << 20
x = rng.integers(0, 256, size=(R, S), dtype=np.uint8)
send, recv = sm.Window(R, S), sm.Window(R, R * S)
upload(send, x)
for _ in range(2):
    sm.sym_allgather(send, recv, S // 4, "f32", "copy")
assert sm.sym_stream_status() == sm.SYM_OK
want = oracle.allgather(x)
got = download(recv, R * S, ranks=[0, R - 1])
for i in range(2):
    assert np.array_equal(got[i], want), i
print("AG_KERNEL_OK")
"""


@pytest.mark.parametrize("kernel", ["bulk", "ldst"])
def test_allgather_kernel_parity(kernel):
    env = dict(os.environ, SYM_ALLGATHER_KERNEL=kernel)
    out = subprocess.run([sys.executable, "-c", _SCRIPT.format(root=ROOT, tests=os.path.join(ROOT, "tests"))],
                         env=env, capture_output=True, text=True, timeout=900)
    assert out.returncode == 0, out.stdout[-2000:] + out.stderr[-4000:]
    assert "AG_KERNEL_OK" in out.stdout
