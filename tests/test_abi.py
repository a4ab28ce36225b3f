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
    assert lib.sym_abi_version() == 2
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


def _header_enum_values() -> dict:
    """NAME -> value of every enumerator the header spells out as NAME = number."""
    import re

    from symmetric_memory_allreduce_gb300 import _binding

    body = open(_binding.HEADER).read()
    return {m.group(1): int(m.group(2)) for m in re.finditer(r"\b(SYM_[A-Z0-9_]+)\s*=\s*(\d+)", body)}


def test_enum_values_are_fixed():
    """The numeric values a C caller relies on, as first published for this library:
    status codes, SYM_F32/SYM_BF16, SYM_SUM, and SYM_ALGO_AUTO/ONESHOT/TWOSHOT/PUT_SIGNAL = 0..3;
    everything added later takes a value of its own after those."""
    v = _header_enum_values()
    fixed = {"SYM_OK": 0, "SYM_ERR_INVALID_ARG": 1, "SYM_ERR_OOM": 2, "SYM_ERR_CUDA": 3,
             "SYM_ERR_TIMEOUT": 4, "SYM_ERR_UNSUPPORTED": 5, "SYM_ERR_DEVICE_STATUS": 6,
             "SYM_F32": 0, "SYM_BF16": 1, "SYM_SUM": 0,
             "SYM_ALGO_AUTO": 0, "SYM_ALGO_ONESHOT": 1, "SYM_ALGO_TWOSHOT": 2,
             "SYM_ALGO_PUT_SIGNAL": 3}
    for name, val in fixed.items():
        assert v.get(name) == val, name
    added = {"SYM_F16": 2, "SYM_MAX": 1, "SYM_MIN": 2, "SYM_ALGO_TWOSHOT_PULL": 4,
             "SYM_ALGO_TWOSHOT_SPLIT": 5, "SYM_ALGO_COPY": 6, "SYM_ALGO_CE": 7,
             "SYM_WINDOW_CUDA_MALLOC": 0, "SYM_WINDOW_REGISTERED": 1,
             "SYM_WINDOW_VMM_EXPORTABLE": 2, "SYM_WINDOW_VMM": 3}
    for name, val in added.items():
        assert v.get(name) == val, name
    algos = [k for k in v if k.startswith("SYM_ALGO_")]
    assert len({v[k] for k in algos}) == len(algos)          # no two algorithms share a value


def test_binding_mirrors_header_enums():
    from symmetric_memory_allreduce_gb300 import _binding

    v = _header_enum_values()
    for name, val in v.items():
        if hasattr(_binding, name):
            assert getattr(_binding, name) == val, name
    for key, code in _binding.ALGOS.items():
        assert v["SYM_ALGO_" + key.upper()] == code


def test_binding_signatures_match_header_arity():
    """Every declared entry point takes as many arguments as the ctypes binding passes."""
    import re

    from symmetric_memory_allreduce_gb300 import _binding

    body = open(_binding.HEADER).read()
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)          # drop comments
    decls = re.findall(r"\b(sym_\w+)\s*\(([^;{]*?)\)\s*;", body, flags=re.S)
    seen = 0
    for name, params in decls:
        if name not in _binding._SIGS:
            continue
        params = params.strip()
        arity = 0 if params in ("", "void") else params.count(",") + 1
        assert arity == len(_binding._SIGS[name][0]), name
        seen += 1
    assert seen == len(_binding.header_symbols())
