"""Symmetric-window collectives on one GB300: AllReduce(sum), AllGather and
chunked put+signal over R rank windows carved from one GPU's HBM.

The compute path is libsymar.so (hand-written CUDA for sm_103a behind the C ABI
in include/symar.h); this package is its thin ctypes binding.
"""
from ._binding import (  # noqa: F401
    ALGOS, DTYPES, NO_ID, OPS, SYM_ERR_INVALID_ARG, SYM_ERR_TIMEOUT, SYM_ERR_UNSUPPORTED, SYM_OK,
    SymError, Window, header_symbols, load, sym_abi_version, sym_allgather,
    sym_allgather_put_signal, sym_allreduce, sym_alltoall, sym_barrier, sym_scale_allreduce, sym_allreduce_algo, sym_counter_read,
    sym_counter_reset, sym_counter_wait, sym_get, sym_last_error, sym_launch_count, sym_put_signal,
    sym_allreduce_noalloc, sym_signal, sym_signal_read, sym_signal_reset, sym_signal_wait,
    sym_status_string,
    sym_stream_status,
    SYM_WINDOW_CUDA_MALLOC, SYM_WINDOW_REGISTERED, SYM_WINDOW_VMM, SYM_WINDOW_VMM_EXPORTABLE,
)
from ._binding import LIB_PATH  # noqa: F401
