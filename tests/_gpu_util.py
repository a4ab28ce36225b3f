"""Helpers for GPU tests: move seeded host inputs into windows and results back.

Everything here is plumbing (stream-ordered host<->device copies through the
library's own sym_window_write / sym_window_read); no arithmetic of the method.
"""
import numpy as np


def sync():
    import torch

    torch.cuda.current_stream().synchronize()


def upload(win, x: np.ndarray):
    """x: (R, ...) array; row r goes to rank r at offset 0."""
    x = np.ascontiguousarray(x)
    for r in range(x.shape[0]):
        win.write(r, x[r])
    sync()


def download(win, nbytes: int, dtype=np.uint8, ranks=None) -> np.ndarray:
    ranks = range(win.R) if ranks is None else ranks
    out = np.empty((len(ranks), nbytes), np.uint8)
    for i, r in enumerate(ranks):
        win.read(r, out[i], nbytes=nbytes)
    sync()
    return out.view(dtype)


def bf16_ulp_distance(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """|ord(a) - ord(b)| for bf16 bit patterns, ord monotone with +0 == -0."""
    def ord_(x):
        x = x.astype(np.int64)
        mag = x & 0x7FFF
        return np.where(x & 0x8000, -mag, mag)
    return np.abs(ord_(a) - ord_(b))
