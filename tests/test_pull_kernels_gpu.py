"""Parity of both fused pull two-shot kernels at every size: SYM_PULL_KERNEL=ws (the
warp-specialised kernel: reducer warps + a TMA copy lane per CTA) and =items (the
single-role kernel), each forced in a child process (the choice is read once per
process; by default the library picks items up to 256 KiB per rank and ws above)."""
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
rng = np.random.default_rng(12)
for R in (2, 3, 8, 16, 64):
    for n in (1, 5, 8, 1000, 4097, 65539, 262147, 1 << 21):
        if R * n > (1 << 24):
            continue
        for dt, op in (("f32", "sum"), ("bf16", "sum"), ("f16", "max"), ("f32", "min")):
            xf = rng.standard_normal((R, n)).astype(np.float32)
            x = xf if dt == "f32" else (wl.to_bf16_bits(xf) if dt == "bf16" else
                                        np.ascontiguousarray(xf.astype(np.float16).view(np.uint16)))
            es = x.itemsize
            for in_place in (False, True):
                a = sm.Window(R, n * es)
                b = a if in_place else sm.Window(R, n * es)
                upload(a, x)
                for rep in range(2):          # repeated calls: fresh epochs, reused ticket
                    sm.sym_allreduce(a, b, n, dt, op, "twoshot_pull")
                    assert sm.sym_stream_status() == sm.SYM_OK, sm.sym_last_error()
                    if in_place:
                        break
                y = download(b, n * es, x.dtype)
                want = oracle.allreduce(x, dt, op)
                assert np.array_equal(y.view(np.uint8), np.broadcast_to(want, y.shape).view(np.uint8)), (R, n, dt, op, in_place)
                a.free()
                if not in_place:
                    b.free()
x = wl.workload_inputs(3)
R, n = x.shape
a, b = sm.Window(R, n * 4), sm.Window(R, n * 4)
upload(a, x)
sm.sym_allreduce(a, b, n, "f32", "sum", "twoshot_pull")
assert sm.sym_stream_status() == sm.SYM_OK
want, _ = oracle.allreduce_sum_mt(x, 16)
for r in range(R):
    assert np.array_equal(download(b, n * 4, np.float32, ranks=[r])[0].view(np.uint32), want.view(np.uint32)), r
print("PULL_OK")
"""


@pytest.mark.parametrize("kernel", ["ws", "items"])
def test_pull_kernel_parity(kernel):
    env = dict(os.environ, SYM_PULL_KERNEL=kernel)
    out = subprocess.run([sys.executable, "-c", _SCRIPT.format(root=ROOT, tests=os.path.join(ROOT, "tests"))],
                         env=env, capture_output=True, text=True, timeout=900)
    assert out.returncode == 0, out.stdout[-2000:] + out.stderr[-4000:]
    assert "PULL_OK" in out.stdout
