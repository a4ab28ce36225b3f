"""Seeded synthetic inputs for the symmetric-window collectives.

This module only draws random numbers; it holds none of the collectives'
arithmetic.  Tests, the oracle and the CUDA path all take their inputs from
here, so both sides see identical bytes.

Recipe (host numpy, ``Generator(PCG64(seed))``):

* per-rank seed = ``20261202 + 1000 * config + rank``;
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


def rank_seed(config: int, rank: int) -> int:
    return SEED_BASE + 1000 * int(config) + int(rank)


def _gen(config: int, rank: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(rank_seed(config, rank)))


def normal_f32(config: int, R: int, n: int) -> np.ndarray:
    """(R, n) float32, rank r drawn N(0,1) from its own seed."""
    out = np.empty((R, n), np.float32)
    for r in range(R):
        out[r] = _gen(config, r).standard_normal(n, dtype=np.float32)
    return out


def uniform_f32(config: int, R: int, n: int) -> np.ndarray:
    """(R, n) float32, rank r drawn U(-1,1) from its own seed."""
    out = np.empty((R, n), np.float32)
    for r in range(R):
        u = _gen(config, r).random(n, dtype=np.float32)
        np.multiply(u, np.float32(2.0), out=u)
        np.subtract(u, np.float32(1.0), out=u)
        out[r] = u
    return out


def rank_fill_f32(R: int, n: int) -> np.ndarray:
    """(R, n) float32 with row r filled with float(r)."""
    return np.repeat(np.arange(R, dtype=np.float32)[:, None], n, axis=1)


def random_bytes(config: int, R: int, nbytes: int) -> np.ndarray:
    out = np.empty((R, nbytes), np.uint8)
    for r in range(R):
        out[r] = _gen(config, r).integers(0, 256, nbytes, dtype=np.uint8)
    return out


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 array -> uint16 bf16 patterns via torch's CPU conversion."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).reshape(x.shape)


@dataclass(frozen=True)
class AllReduceConfig:
    index: int
    name: str
    R: int
    count: int          # elements per rank
    dist: str           # "normal" | "uniform" | "rankfill"
    algos: tuple


CONFIGS = {
    1: AllReduceConfig(1, "allreduce R=4 N=1048576 fp32 (rank fill, then N(0,1))", 4, 1 << 20,
                       "normal", ("oneshot",)),
    2: AllReduceConfig(2, "allreduce R=8 N=16777216 fp32 N(0,1)", 8, 1 << 24, "normal",
                       ("oneshot", "twoshot")),
    3: AllReduceConfig(3, "allreduce R=8 N=67108864 (256 MiB fp32 / 128 MiB bf16) U(-1,1)", 8,
                       1 << 26, "uniform", ("twoshot",)),
}

# message-size sweep: R=8, 1 KiB .. 1 GiB per rank in powers of four, fp32 N(0,1)
SWEEP_BYTES = [KiB * 4 ** k for k in range(11)]

# chunked put+signal AllGather: R=16, 32 MiB per rank, 64 KiB chunks, 8 chunks per signal
PUT_SIGNAL = dict(R=16, nbytes=32 * MiB, chunk=64 * KiB, batch=8)


def config_inputs(index: int, n: int | None = None, dist: str | None = None) -> np.ndarray:
    """Inputs of AllReduce config ``index`` (optionally truncated to ``n`` elements per rank)."""
    if index == 4:
        R, dist = 8, dist or "normal"
        if n is None:
            raise ValueError("the sweep needs an explicit element count")
    else:
        c = CONFIGS[index]
        R, n, dist = c.R, (c.count if n is None else n), (dist or c.dist)
    if dist == "normal":
        return normal_f32(index, R, n)
    if dist == "uniform":
        return uniform_f32(index, R, n)
    if dist == "rankfill":
        return rank_fill_f32(R, n)
    raise ValueError(dist)
