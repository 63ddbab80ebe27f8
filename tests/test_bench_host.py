"""Host-side helpers of bench.py (no GPU): the DRAM-traffic record is taken
only for the kernel source, kernel and workload it was captured from; the
flop counts follow the definitions the bench reports (nominal 4m^2n + 2m^3
and executed 3m^2n + m^3 per step, apply 2m^2n); the GPU index honours
CUDA_VISIBLE_DEVICES; the CPU baseline reports the BLAS threads it ran with;
and the reference arm runs as two torchrun ranks on the CPU (gloo)."""
import hashlib
import importlib.util
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture()
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _fake_tree(tmp_path, source: bytes, record: str):
    src = tmp_path / "newton_schulz_quintic_gb300" / "csrc"
    src.mkdir(parents=True)
    (src / "ns_tc.cu").write_bytes(source)
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "traffic.txt").write_text(record)
    return hashlib.sha256(source).hexdigest()[:16]


def test_traffic_record_matches_source_kernel_and_workload(bench, tmp_path):
    sha = hashlib.sha256(b"kernel v1").hexdigest()[:16]
    _fake_tree(tmp_path, b"kernel v1",
               f"kernel=apply workload=w1 source_sha={sha} bytes_per_launch=123\n"
               f"kernel=gemm workload=w1 source_sha={sha} bytes_per_launch=456\n")
    bench.ROOT = str(tmp_path)
    assert bench.traffic_record("apply", "w1")["bytes_per_launch"] == "123"
    assert bench.traffic_record("gemm", "w1")["bytes_per_launch"] == "456"
    assert bench.traffic_record("apply", "w2") is None          # another workload
    assert bench.traffic_record("apply", "w1[:2]") is None      # a subset of it
    assert bench.traffic_record("square", "w1") is None         # another kernel


def test_traffic_record_is_dropped_when_the_kernel_source_changes(bench, tmp_path):
    old = hashlib.sha256(b"kernel v1").hexdigest()[:16]
    _fake_tree(tmp_path, b"kernel v2", f"kernel=apply workload=w1 source_sha={old} bytes_per_launch=123\n")
    bench.ROOT = str(tmp_path)
    assert bench.traffic_record("apply", "w1") is None


def test_workload_flops(bench):
    nominal, executed, apply = bench.workload_flops([(8192, 6144)], 5)
    m, n = 6144, 8192
    assert nominal == 5 * (4 * m * m * n + 2 * m ** 3)
    assert executed == 5 * (3 * m * m * n + m ** 3)
    assert apply == 5 * 2 * m * m * n
    # orientation does not matter: the iteration runs on the short side
    assert bench.workload_flops([(6144, 8192)], 5) == (nominal, executed, apply)


def test_physical_gpu_index(bench, monkeypatch):
    monkeypatch.setenv("CUDA_VISIBLE_DEVICES", "3,5")
    assert bench.physical_gpu_index(0) == 3
    assert bench.physical_gpu_index(1) == 5
    monkeypatch.delenv("CUDA_VISIBLE_DEVICES")
    assert bench.physical_gpu_index(2) == 2


def test_blas_threads_reports_the_thread_variables(bench, monkeypatch):
    n = bench.cores()
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        monkeypatch.delenv(var, raising=False)
    assert bench.blas_threads() == n
    monkeypatch.setenv("OMP_NUM_THREADS", "1")
    assert bench.blas_threads() == 1
    monkeypatch.setenv("OPENBLAS_NUM_THREADS", str(n + 100))   # capped at the usable cores
    assert bench.blas_threads() == n


def test_reference_arm_under_torchrun_two_ranks():
    # the reference arm as launched for N > 1: rank 0 alone times the oracle
    # (on every host core) and prints one line; the other rank exits 0
    import json
    import socket
    import subprocess
    import sys
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "2", "--warmup", "1", "--workload", "f32-8x64x128"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(x) for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1
    out = lines[0]
    assert out["impl"] == "reference" and out["n_gpus"] == 2 and out["steps"] == 2
    assert out["value"] > 0 and out["e2e"]["value"] == out["value"]
    assert out["e2e"]["h2d_bytes_per_step"] == 0 and out["e2e"]["d2h_bytes_per_step"] == 0
    cb = out["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == out["value"] and cb["cores"] == len(os.sched_getaffinity(0))
    assert cb["cpu"].startswith(os.uname().machine)


def test_input_digest_covers_every_byte(bench):
    import torch
    a = (torch.arange(12, dtype=torch.float32).reshape(3, 4) / 7).to(torch.bfloat16)
    b = torch.ones(2, 5, dtype=torch.bfloat16)
    want = hashlib.sha256(a.view(torch.int16).numpy().tobytes() + b.view(torch.int16).numpy().tobytes())
    assert bench.input_digest([a, b]) == want.hexdigest()
    c = a.clone()
    c[2, 3] = -c[2, 3]
    assert bench.input_digest([c, b]) != want.hexdigest()
    f = torch.zeros(4, 4)
    assert bench.input_digest([f]) == hashlib.sha256(bytes(64)).hexdigest()


def test_norm_pass_record(bench):
    # 768 MiB read once per step, 10 steps in 1.2 ms of kernel time
    kt = {"norm_pass": (1.2, 10), "prep": (5.0, 10)}
    r = bench.norm_pass_record(kt, 805306368, 10, 6789.3)
    assert r["achieved"] == round(805306368 * 10 / 1.2e-3 / 1e9, 1)
    assert r["frac"] == round(r["achieved"] / 6789.3, 4) and r["unit"] == "GB/s" and r["launches"] == 10
    assert bench.norm_pass_record({"norm_pass": (0.0, 0)}, 1, 1, 1.0) is None
    assert bench.norm_pass_record({}, 1, 1, 1.0) is None


def test_rank_share_is_the_planners_split(bench):
    # one batch over several GPUs: each rank's share is what the library's
    # planner assigns it, the shares are disjoint and complete, and one GPU
    # takes the whole batch
    from newton_schulz_quintic_gb300 import api, inputs
    wl = inputs.WORKLOADS["bf16-mixed-120"]
    assert bench.rank_share(wl, 1, 0) == list(range(wl.count))
    for world in (2, 4, 8):
        assign, _ = api.plan_shards(wl.shapes, world, numel_eps=0.3)
        shares = [bench.rank_share(wl, world, r) for r in range(world)]
        for r, share in enumerate(shares):
            assert share == [i for i, a in enumerate(assign) if a == r]
        assert sorted(sum(shares, [])) == list(range(wl.count))
        costs = [sum(api.cost(*wl.shapes[i]) for i in sh) for sh in shares]
        assert max(costs) / (sum(costs) / world) < 1.10


def test_rank_calls(bench):
    from newton_schulz_quintic_gb300 import inputs
    wl = inputs.WORKLOADS["bf16-moe-76x2048x6144"]
    # a replica keeps the workload's remainder batches, a split share is one call
    assert bench.rank_calls(wl, list(range(76)), split=False) == [list(range(64)), list(range(64, 76))]
    assert bench.rank_calls(wl, [3, 9], split=True) == [[3, 9]]
    assert bench.rank_calls(wl, [], split=True) == []
