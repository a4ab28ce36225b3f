"""Host-side checks of the C ABI: the library loads and exports every declared
symbol, and argument validation rejects bad requests before any device work.
These run without a GPU (no compute calls)."""
import ctypes

import pytest


@pytest.fixture(scope="module")
def lib():
    from symmetric_memory_allreduce_gb300 import build

    build.build()
    from symmetric_memory_allreduce_gb300 import _binding

    return _binding.load()


def test_exports_every_declared_symbol(lib):
    from symmetric_memory_allreduce_gb300 import _binding

    names = _binding.header_symbols()
    assert len(names) >= 25
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    # the binding wraps every declared entry point
    assert set(names) <= set(_binding._SIGS), set(names) - set(_binding._SIGS)


def test_status_strings_and_version(lib):
    assert lib.sym_abi_version() == 1
    assert lib.sym_status_string(0) == b"SYM_OK"
    assert lib.sym_status_string(4) == b"SYM_ERR_TIMEOUT"
    assert lib.sym_status_string(99) == b"SYM_ERR_UNKNOWN"
    assert lib.sym_launch_count() == 0


def test_host_validation_without_device(lib):
    h = ctypes.c_void_p(1234)
    assert lib.sym_window_alloc(0, 4096, 0, 0, ctypes.byref(h)) == 1
    assert h.value is None                       # *out cleared on error
    assert lib.sym_window_alloc(65, 4096, 0, 0, ctypes.byref(h)) == 1
    assert lib.sym_window_alloc(4, 0, 0, 0, ctypes.byref(h)) == 1
    assert lib.sym_window_alloc(4, 4096, 0, 0, None) == 1
    assert lib.sym_window_register(None, 4, 4096, 4096, 0, 0, ctypes.byref(h)) == 1
    assert lib.sym_window_register(ctypes.c_void_p(4096 + 8), 4, 4096, 4096, 0, 0,
                                   ctypes.byref(h)) == 1          # misaligned base
    assert lib.sym_allreduce(None, None, 1, 0, 0, 0, None) == 1
    assert lib.sym_allgather(None, None, 1, 0, 0, 0, 0, None) == 1
    assert lib.sym_put_signal(None, None, 0, 0, 0, 0, 16, 0, 0, None) == 1
    assert lib.sym_signal_wait(None, 0, 0, 1, 64, 0, None) == 1
    assert lib.sym_window_free(None) == 0
    assert lib.sym_window_nranks(None) == 0
    assert lib.sym_window_stride(None) == 0
    assert lib.sym_window_device(None) == -1
    assert lib.sym_launch_count() == 0          # nothing was launched
