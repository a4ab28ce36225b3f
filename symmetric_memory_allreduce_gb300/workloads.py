"""Seeded synthetic inputs for the symmetric-window collectives.

This module only draws random numbers; it holds none of the collectives'
arithmetic.  Tests, the oracle and the CUDA path all take their inputs from
here, so both sides see identical bytes.

Recipe (host numpy, ``Generator(PCG64(seed))``):

* per-rank seed = ``20261202 + 1000 * workload + rank`` (workloads numbered 1-5 as below);
* N(0,1) values: ``standard_normal(n, dtype=float32)``;
* U(-1,1) values: ``2 * random(n, dtype=float32) - 1`` (float32 arithmetic);
* "rank fill": every element of rank ``r`` is ``float(r)``;
* bf16 inputs: the same float32 draws converted with torch's CPU
  round-to-nearest-even conversion, kept as uint16 bit patterns;
* random bytes: ``integers(0, 256, n, dtype=uint8)``.

The five workloads follow the pages' AllReduce and AllGather examples (four
ranks of 1,048,576 floats filled with their rank) and scale them up: eight
ranks of 64 MiB and 256 MiB, a message-size sweep of 1 KiB to 1 GiB per rank in
powers of four, and a sixteen-rank chunked put+signal AllGather of 32 MiB per
rank in 64 KiB chunks.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

SEED_BASE = 20261202
KiB = 1024
MiB = 1024 * KiB
GiB = 1024 * MiB


def rank_seed(workload: int, rank: int) -> int:
    return SEED_BASE + 1000 * int(workload) + int(rank)


def _gen(workload: int, rank: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(rank_seed(workload, rank)))


def normal_f32(workload: int, R: int, n: int) -> np.ndarray:
    """(R, n) float32, rank r drawn N(0,1) from its own seed."""
    out = np.empty((R, n), np.float32)
    for r in range(R):
        out[r] = _gen(workload, r).standard_normal(n, dtype=np.float32)
    return out


def uniform_f32(workload: int, R: int, n: int) -> np.ndarray:
    """(R, n) float32, rank r drawn U(-1,1) from its own seed."""
    out = np.empty((R, n), np.float32)
    for r in range(R):
        u = _gen(workload, r).random(n, dtype=np.float32)
        np.multiply(u, np.float32(2.0), out=u)
        np.subtract(u, np.float32(1.0), out=u)
        out[r] = u
    return out


def rank_fill_f32(R: int, n: int) -> np.ndarray:
    """(R, n) float32 with row r filled with float(r)."""
    return np.repeat(np.arange(R, dtype=np.float32)[:, None], n, axis=1)


def random_bytes(workload: int, R: int, nbytes: int) -> np.ndarray:
    out = np.empty((R, nbytes), np.uint8)
    for r in range(R):
        out[r] = _gen(workload, r).integers(0, 256, nbytes, dtype=np.uint8)
    return out


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 array -> uint16 bf16 patterns via torch's CPU conversion."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).reshape(x.shape)


@dataclass(frozen=True)
class AllReduceWorkload:
    index: int
    name: str
    R: int
    count: int          # elements per rank
    dist: str           # "normal" | "uniform" | "rankfill"
    algos: tuple


WORKLOADS = {
    1: AllReduceWorkload(1, "allreduce R=4 N=1048576 fp32 (rank fill, then N(0,1))", 4, 1 << 20,
                       "normal", ("oneshot",)),
    2: AllReduceWorkload(2, "allreduce R=8 N=16777216 fp32 N(0,1)", 8, 1 << 24, "normal",
                       ("oneshot", "twoshot")),
    3: AllReduceWorkload(3, "allreduce R=8 N=67108864 (256 MiB fp32 / 128 MiB bf16) U(-1,1)", 8,
                       1 << 26, "uniform", ("twoshot",)),
}

# message-size sweep: R=8, 1 KiB .. 1 GiB per rank in powers of four, fp32 N(0,1)
SWEEP_BYTES = [KiB * 4 ** k for k in range(11)]

# chunked put+signal AllGather: R=16, 32 MiB per rank, 64 KiB chunks, 8 chunks per signal
PUT_SIGNAL = dict(R=16, nbytes=32 * MiB, chunk=64 * KiB, batch=8)


def workload_inputs(index: int, n: int | None = None, dist: str | None = None) -> np.ndarray:
    """Inputs of AllReduce workload ``index`` (optionally truncated to ``n`` elements per rank)."""
    if index == 4:
        R, dist = 8, dist or "normal"
        if n is None:
            raise ValueError("the sweep needs an explicit element count")
    else:
        c = WORKLOADS[index]
        R, n, dist = c.R, (c.count if n is None else n), (dist or c.dist)
    if dist == "normal":
        return normal_f32(index, R, n)
    if dist == "uniform":
        return uniform_f32(index, R, n)
    if dist == "rankfill":
        return rank_fill_f32(R, n)
    raise ValueError(dist)
