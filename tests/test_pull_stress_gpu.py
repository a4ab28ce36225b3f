"""Ordering stress for the flag-synchronised pull two-shot: hundreds of calls on
changing inputs, each compared bit for bit with the store-form two-shot on the
device (both kernels are separately pinned to the oracle; a pull that read a
tile before its release was visible would differ).  Sizes on both sides of the
256 KiB-per-rank switch between the single-role and warp-specialised kernels."""
import numpy as np
import pytest

from _gpu_util import upload

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n", [40_000, 1_000_003])
def test_pull_matches_store_form_under_repetition(symar, oracle, n):
    import torch

    R = 8
    x = np.random.default_rng(n).standard_normal((R, n)).astype(np.float32)
    send, pull, st = symar.Window(R, n * 4), symar.Window(R, n * 4), symar.Window(R, n * 4)
    try:
        upload(send, x)
        s = send.tensor(torch.float32)[:, :n]
        p = pull.tensor(torch.float32)[:, :n]
        q = st.tensor(torch.float32)[:, :n]
        for it in range(300):
            if it:
                s.mul_(-0.5).add_(0.25)                 # new inputs each call (exact in fp32)
            symar.sym_allreduce(send, pull, n, "f32", "sum", "twoshot_pull")
            symar.sym_allreduce(send, st, n, "f32", "sum", "twoshot")
            if it % 50 == 0 or it == 299:
                assert symar.sym_stream_status() == symar.SYM_OK
            assert torch.equal(p.view(torch.int32), q.view(torch.int32)), it
        # and the last call against the oracle, host side
        xs = s.cpu().numpy()
        want = oracle.allreduce_sum_f32(np.ascontiguousarray(xs))
        got = p.cpu().numpy()
        assert all(np.array_equal(got[r].view(np.uint32), want.view(np.uint32)) for r in range(R))
    finally:
        send.free()
        pull.free()
        st.free()
