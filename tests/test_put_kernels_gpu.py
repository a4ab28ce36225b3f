"""Parity of both put + signal AllGather copy paths: bulk copies through shared
memory (TMA engine) and register copies, selected with SYM_PUT_KERNEL in a child
process (read once per process).  Bytes, signal counts and counters are exact;
the in-kernel prefix check (a receiver that reads k compares batch k-1 with the
source) must count no differing byte."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_SCRIPT = r"""
import sys
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import numpy as np, torch
import oracle
import symmetric_memory_allreduce_gb300 as sm
from symmetric_memory_allreduce_gb300 import workloads as wl
from _gpu_util import upload, download
sm.load(); oracle.build()
rng = np.random.default_rng(31)
cases = [(16, 32 << 20, 65536, 8), (16, 32 << 20, 65536, 1), (16, 32 << 20, 65536, 64),
         (5, 3 * 65536 + 4096, 65536, 2), (3, 1 << 20, 4096, 300), (4, 100003, 4096, 3),
         (2, 48, 16, 1)]
for R, S, chunk, B in cases:
    x = rng.integers(0, 256, size=(R, S), dtype=np.uint8)
    recv_o, sig_o, cnt_o = oracle.put_signal_allgather(x, chunk, B)
    send, recv = sm.Window(R, S, ncounters=1), sm.Window(R, R * S, nsignals=R)
    mism = torch.zeros(1, dtype=torch.int64, device="cuda")
    upload(send, x)
    for check in (True, False):
        recv.tensor().zero_()
        sm.sym_allgather_put_signal(send, recv, S, chunk, B, d_mismatch=mism.data_ptr() if check else None)
        assert sm.sym_stream_status() == sm.SYM_OK, sm.sym_last_error()
        assert int(mism.item()) == 0
        got = download(recv, R * S, ranks=[0, R - 1])
        for i in range(2):
            assert np.array_equal(got[i], recv_o), (R, S, chunk, B, check, i)
        for p in (0, R - 1):
            for q in range(R):
                assert sm.sym_signal_read(recv, p, q) == int(sig_o[p, q])
        for q in range(R):
            assert sm.sym_counter_read(send, q, 0) == int(cnt_o[q])
    send.free(); recv.free()
print("PUT_KERNEL_OK")
"""


@pytest.mark.parametrize("kernel", ["bulk", "ldst"])
def test_put_kernel_parity(kernel):
    env = dict(os.environ, SYM_PUT_KERNEL=kernel)
    out = subprocess.run([sys.executable, "-c", _SCRIPT.format(root=ROOT, tests=os.path.join(ROOT, "tests"))],
                         env=env, capture_output=True, text=True, timeout=900)
    assert out.returncode == 0, out.stdout[-2000:] + out.stderr[-4000:]
    assert "PUT_KERNEL_OK" in out.stdout
