"""The C ABI from plain C: tests/native/c_abi_parity.c, compiled with gcc against
include/symar.h, linked with libsymar.so and the oracle, compares every AllReduce
algorithm and the AllGather forms with the oracle byte for byte.  Building it
needs no GPU; running it does."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "native", "c_abi_parity.c")


def _build(tmp_path):
    from symmetric_memory_allreduce_gb300 import build as symar_build

    import oracle

    symar_build.build()
    oracle.build()
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lib_dir = os.path.dirname(symar_build.LIB)
    ora_dir = os.path.join(ROOT, "oracle")
    exe = str(tmp_path / "c_abi_parity")
    cmd = [cc, "-std=c11", "-O2", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
           SRC, "-o", exe, "-L", lib_dir, "-lsymar", "-L", ora_dir, "-l:liboracle.so",
           f"-Wl,-rpath,{lib_dir}:{ora_dir}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    return exe


def test_c_caller_builds(tmp_path):
    assert os.access(_build(tmp_path), os.X_OK)


@pytest.mark.gpu
def test_c_caller_matches_oracle(tmp_path):
    exe = _build(tmp_path)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "C_ABI_PARITY_OK" in r.stdout
