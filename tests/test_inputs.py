"""Input generator: the torch.chunk split and padding against the pages'
printed values (tests/golden/chunk_split.json), and seeding."""
import json
import os

import torch

from newton_schulz_quintic_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "chunk_split.json")


def test_chunk_sizes_match_pages():
    with open(GOLDEN) as f:
        g = json.load(f)
    for case in g["splits"]:
        assert inputs.chunk_sizes(case["size"], case["shards"]) == case["sizes"]
        # the same split torch.chunk produces, padded with empty shards
        got = [c.shape[0] for c in torch.chunk(torch.zeros(case["size"], 1), case["shards"])]
        got += [0] * (case["shards"] - len(got))
        assert got == case["sizes"]


def test_watchdog_numel_matches_padded_layout():
    # every rank's padded shard of the 18-row weight holds 3 rows; per_rank = 4
    # such matrices go to each of 8 ranks: 8 x 4 x 3 x 2304 elements
    with open(GOLDEN) as f:
        w = json.load(f)["watchdog_numel"]
    x = torch.randn(18, w["cols"])
    p = inputs.pad_shards(x, w["world_size"])
    rows_per_shard = p.shape[0] // w["world_size"]
    assert rows_per_shard == w["rows_per_shard"]
    assert w["world_size"] * w["per_rank"] * rows_per_shard * w["cols"] == w["numel"]


def test_padded_workload_layout():
    wl = inputs.WORKLOADS["bf16-32x24x2304-pad"]
    x = wl.matrix(3)
    assert x.shape == (24, 2304) and x.dtype == torch.bfloat16
    assert torch.all(x[18:] == 0) and torch.all(x[:18].abs().sum(1) > 0)


def test_seeded_and_independent_per_matrix():
    wl = inputs.WORKLOADS["f32-8x64x128"]
    a, b = wl.matrix(2), wl.matrix(2)
    assert torch.equal(a, b)
    assert not torch.equal(wl.matrix(1), a)
    assert abs(float(a.std()) - 1.0) < 0.05


def test_call_slices():
    wl = inputs.WORKLOADS["bf16-moe-76x2048x6144"]
    sl = wl.call_slices()
    assert [s.stop - s.start for s in sl] == [64, 12]
    wl3 = inputs.WORKLOADS["bf16-8x8192x6144"]
    assert wl3.call_slices() == [slice(0, 8)]


def test_mixed_workload_shapes():
    wl = inputs.WORKLOADS["bf16-mixed-120"]
    assert wl.count == 120
    assert wl.shapes.count((14336, 4096)) == 24 and wl.shapes.count((1024, 4096)) == 48
