"""Debug builds check every store of the library's kernels against the buffer
it belongs to: a store outside it is not made and the device status word
reports NS_EBOUNDS. It stands in for a memory checker, which is not available
on these GPUs. This file builds that variant in a child process (so the
release library of the other tests stays loaded here), exercises the check
mechanism without touching memory, and runs workloads of every path through
the checked kernels: no check fires and every result matches the oracle. The
release build reports that it has no checks."""
import os
import subprocess
import sys
import textwrap

import pytest

from newton_schulz_quintic_gb300 import api

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = textwrap.dedent("""
    import os, sys
    import numpy as np
    import torch
    sys.path.insert(0, %r)
    from newton_schulz_quintic_gb300 import build, api
    os.environ["NS_LIBRARY_PATH"] = build.build()
    api.load_library()
    import oracle

    assert api.selftest_bounds_check() == 0          # the check ran ...
    assert api.get_status() == -8                    # ... and fired (no memory touched)
    assert api.get_status() == 0

    def seeded(shape, dtype, seed, std):
        g = torch.Generator().manual_seed(seed)
        return (torch.randn(shape, generator=g) * std).to(dtype)

    def rel(a, b):
        return float(np.linalg.norm(a - b) / np.linalg.norm(b))

    def check(xs, ys, tol, steps=5):
        for x, y in zip(xs, ys):
            assert rel(oracle.to_f64(y.cpu()), oracle.orthogonalize(x, steps=steps)) <= tol, tuple(x.shape)

    cases = [
        ([(300, 520), (520, 300), (1024, 768), (129, 1031), (24, 2304), (64, 100)], torch.bfloat16, 0.02, 3e-2),
        ([(64, 128), (100, 300), (300, 100)], torch.float32, 1.0, 1e-4),
    ]
    for shapes, dtype, std, tol in cases:
        xs = [seeded(s, dtype, 40 + i, std) for i, s in enumerate(shapes)]
        for steps in (5, 0):
            ys = [x.cuda() for x in xs]
            api.orthogonalize_batched(ys, steps=steps)
            assert api.get_status() == 0, ("a bounds check fired", dtype, steps)
            check(xs, ys, tol if steps else 1e-2, steps)
        # matrices 2 bytes past a 16-byte boundary (the copying first step)
        x = xs[0]
        buf = torch.zeros(x.numel() + 8, dtype=dtype, device="cuda")
        v = buf[1:1 + x.numel()].view(x.shape)
        v.copy_(x.cuda())
        api.orthogonalize_batched([v])
        assert api.get_status() == 0
        check([x], [v], tol)
    # the single-launch schedule and the fused optimizer step
    xs = [seeded(s, torch.bfloat16, 60 + i, 0.02) for i, s in enumerate([(640, 1200), (1200, 640)])]
    api.set_gemm_schedule("single")
    ys = [x.cuda() for x in xs]
    api.orthogonalize_batched(ys)
    api.set_gemm_schedule("phase")
    assert api.get_status() == 0
    check(xs, ys, 3e-2)
    g = [x.cuda() for x in xs]
    m = [torch.zeros_like(t) for t in g]
    o = [torch.empty_like(t) for t in g]
    api.muon_update_batched(g, m, o, mu=0.9, nesterov=True, scale=1.0)
    assert api.get_status() == 0
    print("debug-bounds ok")
""") % ROOT


def test_debug_build_checks_every_store():
    env = dict(os.environ, NS_BUILD_TAG="debugbounds", NS_EXTRA_NVCC_FLAGS="-DNS_DEBUG_BOUNDS")
    env.pop("NS_LIBRARY_PATH", None)
    r = subprocess.run([sys.executable, "-c", CHILD], env=env, capture_output=True, text=True, timeout=1200,
                       cwd=ROOT)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "debug-bounds ok" in r.stdout


def test_release_build_has_no_bounds_checks():
    from newton_schulz_quintic_gb300 import build
    build.build()
    api.load_library()
    assert api.selftest_bounds_check() == -1
    assert api.get_status() == 0
