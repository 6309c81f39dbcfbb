"""The five workloads (synthetic stand-ins shaped like the pages' datasets).

Each workload is one partition of a graph plus the layer widths of an L-layer
model.  Only sizes and structure come from the pages' datasets; no dataset is
read.  ``tiny=True`` variants keep the same recipe at a size the oracle runs in
well under a second (used by the CPU tests and the smoke check).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Callable, List

import synth


@dataclass
class Workload:
    name: str
    description: str
    agg: str  # "gcn" | "sage"
    dtype: str  # "f32" | "bf16"
    widths: List[int]  # f_0 (input features), hidden..., classes
    feat_dist: str  # "uniform" | "normal"
    make: Callable[[int], "synth.Partition"] = field(repr=False)

    @property
    def layers(self) -> int:
        return len(self.widths) - 1

    @property
    def bf16(self) -> bool:
        return self.dtype == "bf16"


RMAT = (0.57, 0.19, 0.19)

# expected unique (non-loop) edges of the R-MAT block partition grow with the
# number of samples; 1.125e9 samples gives ~400M unique edges at scale 24
RMAT_BLOCK_SAMPLES = 1.125e9

WORKLOADS = {
    "er5k": Workload(
        "er5k",
        "2-layer GCN, Erdos-Renyi G(5120, 16/5119), 4096 local + 1024 halo, 64 -> 64 -> 16, fp32 U[-1,1]",
        "gcn", "f32", [64, 64, 16], "uniform",
        lambda seed: synth.er_partition(5120, 4096, 16.0 / 5119.0, seed)),
    "rmat131k": Workload(
        "rmat131k",
        "2-layer GCN, R-MAT scale 17 (2,097,152 undirected edges), 10% halo, 256 -> 256 -> 32, fp32 N(0,1)",
        "gcn", "f32", [256, 256, 32], "normal",
        lambda seed: synth.rmat_sym_partition(17, 2_097_152, 131_072 - 13_107, seed, RMAT, True)),
    "powerlaw233k": Workload(
        "powerlaw233k",
        "2-layer GCN, Chung-Lu power law n=232,965, 114.6M directed edges (mean 492), partition 0 of 4, "
        "602 -> 256 -> 41, fp32 N(0,1)",
        "gcn", "f32", [602, 256, 41], "normal",
        lambda seed: synth.chunglu_partition(232_965, 57_300_000, 491.9, 4, seed)),
    "sage2m": Workload(
        "sage2m",
        "3-layer GraphSAGE-mean, Chung-Lu power law n=2,449,029, 123.7M directed edges, partition 0 of 8, "
        "100 -> 256 -> 256 -> 47, bf16 N(0,1)",
        "sage", "bf16", [100, 256, 256, 47], "normal",
        lambda seed: synth.chunglu_partition(2_449_029, 61_850_000, 50.5, 8, seed)),
    "rmat16m": Workload(
        "rmat16m",
        "3-layer GCN, one partition of an R-MAT scale-24 graph: 8,388,608 local + 4,194,304 halo vertices, "
        "~400M local edges, 128 -> 256 -> 256 -> 172, bf16 N(0,1), stale tables of 2^24 rows",
        "gcn", "bf16", [128, 256, 256, 172], "normal",
        lambda seed: synth.rmat_block_partition(24, 1 << 23, 1 << 22, RMAT_BLOCK_SAMPLES, seed, RMAT)),
}

# the same recipes at tiny sizes (CPU tests, smoke check, quick GPU parity)
TINY = {
    "er5k": Workload("er5k-tiny", "ER 600 / 480 local", "gcn", "f32", [64, 64, 16], "uniform",
                     lambda seed: synth.er_partition(600, 480, 16.0 / 599.0, seed)),
    "rmat131k": Workload("rmat131k-tiny", "R-MAT scale 11", "gcn", "f32", [256, 256, 32], "normal",
                         lambda seed: synth.rmat_sym_partition(11, 16_384, 2048 - 205, seed, RMAT, True)),
    "powerlaw233k": Workload("powerlaw233k-tiny", "Chung-Lu n=3000 mean 60", "gcn", "f32", [602, 256, 41], "normal",
                             lambda seed: synth.chunglu_partition(3000, 90_000, 60.0, 4, seed)),
    "sage2m": Workload("sage2m-tiny", "Chung-Lu n=8000 mean 20", "sage", "bf16", [100, 256, 256, 47], "normal",
                       lambda seed: synth.chunglu_partition(8000, 80_000, 20.0, 8, seed)),
    "rmat16m": Workload("rmat16m-tiny", "R-MAT block scale 14", "gcn", "bf16", [128, 256, 256, 172], "normal",
                        lambda seed: synth.rmat_block_partition(14, 1 << 13, 1 << 12, 1.2e5, seed, RMAT)),
}

# a quarter-scale instance of the R-MAT partition for detailed profiling (inputs
# still far larger than L2, a few GB on the device)
PROFILE = {
    "rmat4m": Workload(
        "rmat4m", "3-layer GCN, R-MAT scale-22 partition: 2,097,152 local + 1,048,576 halo, ~100M entries",
        "gcn", "bf16", [128, 256, 256, 172], "normal",
        lambda seed: synth.rmat_block_partition(22, 1 << 21, 1 << 20, RMAT_BLOCK_SAMPLES / 4, seed, RMAT)),
}

BENCH_WORKLOAD = "rmat16m"
