"""Parity of the bulk-copy (TMA engine) two-shot kernel, selected with
SYM_TWOSHOT_KERNEL=bulk in a child process (the choice is read once per process)."""
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
from symmetric_memory_allreduce_gb300 import workloads as wl
from _gpu_util import upload, download
sm.load(); oracle.build()
rng = np.random.default_rng(11)
for R in (1, 2, 3, 8, 16):
    for n in (1, 5, 1000, 4097, 65539, 262147, 1 << 21):
        for dt in ("f32", "bf16"):
            xf = rng.standard_normal((R, n)).astype(np.float32)
            x = xf if dt == "f32" else wl.to_bf16_bits(xf)
            es = x.itemsize
            for in_place in (False, True):
                a = sm.Window(R, n * es)
                b = a if in_place else sm.Window(R, n * es)
                upload(a, x)
                sm.sym_allreduce(a, b, n, dt, "sum", "twoshot")
                assert sm.sym_stream_status() == sm.SYM_OK, sm.sym_last_error()
                y = download(b, n * es, x.dtype)
                want = oracle.allreduce_sum_f32(x) if dt == "f32" else oracle.allreduce_sum_bf16(x)
                assert np.array_equal(y.view(np.uint8), np.broadcast_to(want, y.shape).view(np.uint8)), (R, n, dt, in_place)
                a.free()
                if not in_place:
                    b.free()
x = wl.workload_inputs(3)
R, n = x.shape
a, b = sm.Window(R, n * 4), sm.Window(R, n * 4)
upload(a, x)
sm.sym_allreduce(a, b, n, "f32", "sum", "twoshot")
assert sm.sym_stream_status() == sm.SYM_OK
want, _ = oracle.allreduce_sum_mt(x, 16)
for r in range(R):
    assert np.array_equal(download(b, n * 4, np.float32, ranks=[r])[0].view(np.uint32), want.view(np.uint32)), r
print("BULK_OK")
"""


def test_bulk_twoshot_parity():
    env = dict(os.environ, SYM_TWOSHOT_KERNEL="bulk")
    out = subprocess.run([sys.executable, "-c", _SCRIPT.format(root=ROOT, tests=os.path.join(ROOT, "tests"))],
                         env=env, capture_output=True, text=True, timeout=900)
    assert out.returncode == 0, out.stdout[-2000:] + out.stderr[-4000:]
    assert "BULK_OK" in out.stdout
