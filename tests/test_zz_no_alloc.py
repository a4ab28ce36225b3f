"""sym_allreduce_noalloc: the AllReduce entry point for callers that cannot
allocate device memory (engines that forbid allocations after start-up,
plug-ins whose framework owns the allocator).  It must give the same result as
the regular entry point, sym_allreduce, on two calls in a row that share its
static scratch.  Collected last on purpose; it also passes on its own in a
fresh process."""
import numpy as np
import pytest

from _gpu_util import bf16_ulp_distance, download, upload

pytestmark = pytest.mark.gpu


def _reference(sm, x, dtype):
    """Result of the regular entry point (windows, two-shot) for inputs x (R, n)."""
    R, n = x.shape
    es = x.itemsize
    send, recv = sm.Window(R, n * es), sm.Window(R, n * es)
    try:
        upload(send, x)
        sm.sym_allreduce(send, recv, n, dtype, "sum", "twoshot")
        assert sm.sym_stream_status() == sm.SYM_OK
        return download(recv, n * es, x.dtype)
    finally:
        send.free()
        recv.free()


def _noalloc(sm, x, dtype, send_t, recv_t, stride):
    """Caller-owned buffers (torch allocations made by the test, not by the entry point)."""
    import torch

    R, n = x.shape
    es = x.itemsize
    host = torch.zeros((R, stride), dtype=torch.uint8)
    host[:, : n * es] = torch.from_numpy(np.ascontiguousarray(x).view(np.uint8))
    send_t.copy_(host.view(-1))
    recv_t.fill_(0xAB)
    sm.sym_allreduce_noalloc(send_t.data_ptr(), recv_t.data_ptr(), stride, R, n, dtype, "sum")
    torch.cuda.synchronize()
    out = recv_t.view(R, stride)[:, : n * es].cpu().numpy()
    return np.ascontiguousarray(out).view(x.dtype)


def _same(y, ref, dtype):
    if dtype == "f32":
        assert np.array_equal(y.view(np.uint32), ref.view(np.uint32))
    else:
        assert bf16_ulp_distance(y, ref).max(initial=0) <= 1
        assert np.array_equal(y, ref)


def test_noalloc_matches_regular_entry_two_calls(symar):
    import torch
    from symmetric_memory_allreduce_gb300 import workloads as wl

    R, n = 8, 1_000_003                       # several tiles per chunk plus a ragged tail
    stride = (n * 4 + 4095) // 4096 * 4096
    send_t = torch.empty(R * stride, dtype=torch.uint8, device="cuda")
    recv_t = torch.empty(R * stride, dtype=torch.uint8, device="cuda")
    for call, seed_cfg in enumerate((2, 3)):  # two calls in a row, different inputs
        x = wl.normal_f32(seed_cfg, R, n) if call == 0 else wl.uniform_f32(seed_cfg, R, n)
        ref = _reference(symar, x, "f32")
        y = _noalloc(symar, x, "f32", send_t, recv_t, stride)
        _same(y, ref, "f32")


def test_noalloc_bf16_two_calls(symar):
    import torch
    from symmetric_memory_allreduce_gb300 import workloads as wl

    R, n = 16, 300_007
    stride = (n * 2 + 4095) // 4096 * 4096
    send_t = torch.empty(R * stride, dtype=torch.uint8, device="cuda")
    recv_t = torch.empty(R * stride, dtype=torch.uint8, device="cuda")
    for call in range(2):
        x = wl.to_bf16_bits(wl.uniform_f32(10 + call, R, n))
        ref = _reference(symar, x, "bf16")
        _same(_noalloc(symar, x, "bf16", send_t, recv_t, stride), ref, "bf16")


def test_noalloc_rejects_oversize_and_overlap(symar):
    import torch

    buf = torch.empty(2 * 4096, dtype=torch.uint8, device="cuda")
    p = buf.data_ptr()
    # more than 65536 tiles of 16 KiB: rejected before any device work, with a reason
    with pytest.raises(symar.SymError) as e:     # (never dereferenced: rejected on the host)
        symar.sym_allreduce_noalloc(p, p + (1 << 43), 1 << 40, 2, (1 << 40) // 4, "f32", "sum")
    assert e.value.status == symar.SYM_ERR_INVALID_ARG
    assert "static scratch" in symar.sym_last_error()
    with pytest.raises(symar.SymError):          # input and output ranges overlap
        symar.sym_allreduce_noalloc(p, p + 16, 4096, 1, 64, "f32", "sum")
