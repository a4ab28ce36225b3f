"""The native benchmark of the C ABI (symar_bench, built with the library)."""
import json
import os
import subprocess

import pytest

from symmetric_memory_allreduce_gb300 import build as symar_build


def _tool():
    symar_build.build()
    assert os.access(symar_build.TOOL, os.X_OK)
    return symar_build.TOOL


def test_tool_rejects_bad_arguments():
    for args in (["--bogus"], ["--algo", "threeshot"], ["--dtype", "f64"], ["--ranks"]):
        r = subprocess.run([_tool(), *args], capture_output=True, text=True, timeout=60)
        assert r.returncode == 2, (args, r.stdout, r.stderr)


@pytest.mark.gpu
@pytest.mark.parametrize("args", [
    ["--ranks", "8", "--bytes", str(16 << 20), "--algo", "twoshot"],
    ["--ranks", "4", "--bytes", str(1 << 20), "--algo", "auto", "--dtype", "bf16"],
    ["--ranks", "8", "--bytes", str(8 << 20), "--algo", "twoshot_pull", "--dtype", "f16", "--vmm"],
])
def test_tool_runs(args):
    r = subprocess.run([_tool(), *args, "--iters", "20", "--warmup", "3"], capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    d = json.loads(r.stdout.strip().splitlines()[-1])
    assert d["ranks_agree"] is True
    assert d["us_median"] > 0 and d["iters"] == 20
    if "--vmm" in args:
        assert d["window"] == "vmm"
