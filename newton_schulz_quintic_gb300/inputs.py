"""Seeded synthetic inputs for batched Newton-Schulz workloads.

This module is shared by the CUDA path's tests and benchmark and by the CPU
oracle's tests. It holds none of the method's arithmetic: only random-number
generation, the torch.chunk-style split of a dimension over shards, and
zero padding of shards to a common size.

Recipe. Matrix ``i`` of a workload with seed ``S`` is drawn with
``torch.Generator('cpu').manual_seed(S * 1_000_003 + i)`` as
``randn(shape, float32) * std`` and then cast to the workload's dtype by
round-to-nearest-even (torch's CPU cast). Every matrix has its own seed, so a
single matrix of a large batch can be regenerated alone on the CPU.

The workloads follow the pages' shapes: 8192 x 6144 bf16 matrices (the xtuner
Muon remainder-strategy PR's timing tables), an 18 x 2304 attention-gate weight
split over 8 FSDP2 shards (the first page's "Concrete repro"), and 76 expert
matrices processed as remainder batches of 64 and 12 (GLM-5.2 in the xtuner
PR). No public dataset is involved.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


def chunk_sizes(size: int, shards: int) -> list[int]:
    """Row counts that torch.chunk gives when splitting ``size`` rows into
    ``shards`` pieces, padded with empty pieces up to ``shards`` entries (the
    ``_chunk_with_empty`` behaviour of the first page's "Concrete repro")."""
    if shards <= 0:
        raise ValueError("shards must be positive")
    if size == 0:
        return [0] * shards
    step = -(-size // shards)  # ceil
    out = []
    start = 0
    for _ in range(shards):
        n = max(0, min(step, size - start))
        out.append(n)
        start += n
    return out


def pad_shards(x: torch.Tensor, shards: int) -> torch.Tensor:
    """Split rows torch.chunk-style over ``shards`` and zero-pad every shard to
    the largest shard's row count, then concatenate the padded shards (the
    padded_local_size layout of the first page's "Fix" section)."""
    sizes = chunk_sizes(x.shape[0], shards)
    width = max(sizes)
    out = torch.zeros((width * shards,) + tuple(x.shape[1:]), dtype=x.dtype)
    start = 0
    for r, n in enumerate(sizes):
        out[r * width: r * width + n] = x[start:start + n]
        start += n
    return out


def matrix_seed(seed: int, index: int) -> int:
    return int(seed) * 1_000_003 + int(index)


def make_matrix(shape, std: float, dtype: str, seed: int, index: int) -> torch.Tensor:
    g = torch.Generator(device="cpu")
    g.manual_seed(matrix_seed(seed, index))
    x = torch.randn(tuple(shape), generator=g, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(DTYPES[dtype])


@dataclass(frozen=True)
class Workload:
    name: str
    shapes: tuple          # per matrix (M, N) as given to the library
    dtype: str             # "f32" or "bf16"
    std: float
    seed: int
    steps: int = 5
    real_rows: int = 0     # >0: draw real_rows x N, then split over `shards` and pad
    shards: int = 0
    calls: tuple = field(default_factory=tuple)  # split of the batch into library calls

    @property
    def count(self) -> int:
        return len(self.shapes)

    def matrix(self, i: int) -> torch.Tensor:
        M, N = self.shapes[i]
        if self.real_rows:
            x = make_matrix((self.real_rows, N), self.std, self.dtype, self.seed, i)
            x = pad_shards(x, self.shards)
            assert tuple(x.shape) == (M, N)
            return x
        return make_matrix((M, N), self.std, self.dtype, self.seed, i)

    def matrices(self, indices=None) -> list:
        idx = range(self.count) if indices is None else indices
        return [self.matrix(i) for i in idx]

    def call_slices(self) -> list:
        if not self.calls:
            return [slice(0, self.count)]
        out, start = [], 0
        for n in self.calls:
            out.append(slice(start, start + n))
            start += n
        assert start == self.count
        return out


def subset(wl: Workload, count: int) -> Workload:
    """The first ``count`` matrices of a workload (same seeds), one call."""
    count = max(1, min(int(count), wl.count))
    return Workload(f"{wl.name}[:{count}]", tuple(wl.shapes[:count]), wl.dtype, wl.std, wl.seed,
                    wl.steps, wl.real_rows, wl.shards, ())


def _mixed_shapes():
    return (((4096, 4096),) * 24 + ((4096, 14336),) * 24 + ((14336, 4096),) * 24
            + ((1024, 4096),) * 48)


WORKLOADS = {
    # 8 fp32 64x128 N(0,1)
    "f32-8x64x128": Workload("f32-8x64x128", ((64, 128),) * 8, "f32", 1.0, 1001),
    # 32 bf16 18x2304 N(0,0.02), rows split over 8 shards (3,3,3,3,3,3,0,0) and
    # padded to 3 rows each: 24x2304, rows 18..23 zero
    "bf16-32x24x2304-pad": Workload("bf16-32x24x2304-pad", ((24, 2304),) * 32, "bf16", 0.02,
                                    1002, real_rows=18, shards=8),
    # 8 bf16 8192x6144 N(0,0.02): worked on as its 6144x8192 transpose
    "bf16-8x8192x6144": Workload("bf16-8x8192x6144", ((8192, 6144),) * 8, "bf16", 0.02, 1003),
    # mixed-shape hybrid transformer stack, one call, sorted by cost inside
    "bf16-mixed-120": Workload("bf16-mixed-120", _mixed_shapes(), "bf16", 0.02, 1004),
    # MoE expert stack: 76 x 2048x6144 as remainder batches of 64 and 12
    "bf16-moe-76x2048x6144": Workload("bf16-moe-76x2048x6144", ((2048, 6144),) * 76, "bf16",
                                      0.02, 1005, calls=(64, 12)),
    # the expert shape in fp32 (large fp32 matrices: the fp32 tensor-core path)
    "f32-8x2048x6144": Workload("f32-8x2048x6144", ((2048, 6144),) * 8, "f32", 0.02, 1006),
}

HEADLINE = "bf16-8x8192x6144"
