"""Host planner ns_plan_shards (no GPU): largest-first assignment to the
least-loaded shard by Newton-Schulz cost, per the second page ("Balance
LayerWise optimizer shards by Newton-Schulz cost, not parameter size",
"Changes" items 1-3 and its "Tests" and "Notes" sections), plus a
world-size-2 gloo run of the multi-rank split."""
import json
import os

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from newton_schulz_quintic_gb300 import api, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    api.load_library()


def loads_of(shapes, assign, nshards, numels=None):
    out = [0] * nshards
    for s, a in zip(shapes, assign):
        out[a] += api.cost(*s)
    return out


def imbalance(loads):
    return max(loads) / (sum(loads) / len(loads))


def gtp_case():
    # five dense 256x256 matrices (cost 2^24, numel 65536) and three matrices
    # stored as 1/64 shards but orthogonalised at full 4096x256 (cost 2^28 =
    # 16x the largest dense matrix, numel the smallest in the set)
    shapes = [(256, 256)] * 5 + [(4096, 256)] * 3
    numels = [65536] * 5 + [4096 * 256 // 64] * 3
    return shapes, numels


def test_cost_values_of_the_pages_example():
    # 268,435,456 vs 16,777,216: the expensive matrices cost 16x the dense one
    with open(os.path.join(os.path.dirname(__file__), "golden", "ns_cost.json")) as f:
        g = json.load(f)
    for c in g["costs"]:
        assert api.cost(*c["shape"]) == c["cost"]


def test_cost_order_spreads_what_numel_order_piles_up():
    shapes, numels = gtp_case()
    a_num, _ = api.plan_shards(shapes, 3, numel_eps=-1, order="numel", numels=numels)
    a_cost, _ = api.plan_shards(shapes, 3, numel_eps=0.3, order="cost", numels=numels)
    gtp_num = {a_num[i] for i in range(5, 8)}
    gtp_cost = {a_cost[i] for i in range(5, 8)}
    assert len(gtp_num) == 1            # numel order: all three on one shard
    assert gtp_cost == {0, 1, 2}        # cost order: one per shard
    imb_num = imbalance(loads_of(shapes, a_num, 3))
    imb_cost = imbalance(loads_of(shapes, a_cost, 3))
    assert imb_num > 2.5 and imb_cost < 1.1


def test_aspect_ratio_is_weighed():
    # same byte count, different work: cost = numel * min(M, N) ("Notes")
    shapes = [(4096, 4096), (1024, 16384), (1024, 16384), (1024, 16384), (1024, 16384)]
    a, loads = api.plan_shards(shapes, 2, numel_eps=-1)
    assert a[0] != a[1] or a[0] != a[2]
    assert imbalance(loads) < imbalance(loads_of(shapes, api.plan_shards(shapes, 2, -1, "numel")[0], 2)) + 1e-9


def test_every_matrix_assigned_once_and_deterministic():
    shapes = [(64 * (i % 7 + 1), 128 * (i % 5 + 1)) for i in range(40)]
    a1, l1 = api.plan_shards(shapes, 5)
    a2, l2 = api.plan_shards(shapes, 5)
    assert a1 == a2 and l1 == l2
    assert all(0 <= x < 5 for x in a1) and len(a1) == 40
    assert sum(l1) == sum(api.cost(*s) for s in shapes)


def test_numel_cap_and_least_numel_fallback():
    # one expensive matrix with few stored elements and 100 cheap dense ones
    # on 2 shards: cost balancing alone sends 58 cheap matrices to the shard
    # without the expensive one; a 5% numel cap stops that shard at 52
    shapes = [(4096, 256)] + [(256, 256)] * 100
    numels = [1024] + [65536] * 100
    cap = -(-int(1.05 * sum(numels)) // 2)

    def placed(a):
        out = [0, 0]
        for n, x in zip(numels, a):
            out[x] += n
        return out

    a_free, _ = api.plan_shards(shapes, 2, numel_eps=-1, numels=numels)
    a_cap, _ = api.plan_shards(shapes, 2, numel_eps=0.05, numels=numels)
    assert max(placed(a_free)) > cap
    assert max(placed(a_cap)) <= cap
    # a matrix larger than any cap still gets placed (least-numel fallback)
    a2, _ = api.plan_shards([(5000, 5000), (10, 10), (10, 10)], 4, numel_eps=0.0)
    assert len(a2) == 3 and a2[1] != a2[0] and a2[2] != a2[0]


def test_loads_persist_across_buckets():
    # each bucket holds one expensive matrix and three cheap ones; with loads
    # carried over, the expensive matrices land on different shards
    bucket = [(4096, 256)] + [(256, 256)] * 3
    loads = [0, 0]
    a1, loads = api.plan_shards(bucket, 2, numel_eps=-1, loads=loads)
    a2, loads = api.plan_shards(bucket, 2, numel_eps=-1, loads=loads)
    assert a1[0] != a2[0]
    r1, _ = api.plan_shards(bucket, 2, numel_eps=-1)
    r2, _ = api.plan_shards(bucket, 2, numel_eps=-1)
    assert r1[0] == r2[0]           # reset per bucket: both on the same shard


def test_bad_arguments():
    with pytest.raises(api.NSError):
        api.plan_shards([(4, 4)], 0)
    with pytest.raises(api.NSError):
        api.plan_shards([(-1, 4)], 2)


def _rank_main(rank, world, port, result_q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from newton_schulz_quintic_gb300 import api as a
    from newton_schulz_quintic_gb300 import inputs
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_rank", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    wl = inputs.WORKLOADS["bf16-mixed-120"]
    assign, loads = a.plan_shards(wl.shapes, world)
    mine = [i for i, r in enumerate(assign) if r == rank]
    # the benchmark's split mode runs exactly the planner's share on this rank
    assert bench.rank_share(wl, world, rank) == mine
    my_cost = sum(a.cost(*wl.shapes[i]) for i in mine)
    t = torch.tensor([len(mine), my_cost], dtype=torch.float64)
    tot = t.clone()
    dist.all_reduce(tot, op=dist.ReduceOp.SUM)
    mx = t.clone()
    dist.all_reduce(mx, op=dist.ReduceOp.MAX)
    result_q.put((rank, mine, float(tot[0]), float(tot[1]), float(mx[1]), loads))
    dist.destroy_process_group()


def test_two_rank_split_with_gloo():
    import socket
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(2)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res.sort()
    from newton_schulz_quintic_gb300 import inputs
    wl = inputs.WORKLOADS["bf16-mixed-120"]
    mine0, mine1 = res[0][1], res[1][1]
    assert sorted(mine0 + mine1) == list(range(wl.count))        # disjoint and complete
    total_cost = sum(api.cost(*s) for s in wl.shapes)
    assert res[0][2] == wl.count and res[0][3] == float(total_cost)
    assert res[0][4] / (total_cost / 2) < 1.05                   # max rank within 5% of the mean
