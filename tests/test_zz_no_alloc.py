"""The entry point that allocates no device memory.

Some callers cannot allocate device memory when they orthogonalize (their
framework allocator already holds nearly all of HBM, or their step cannot wait
on an allocator); ns_orthogonalize_batched_noalloc serves them from a fixed
256 MiB scratch array inside the library. This file checks, through the C ABI,
that it gives the same results as ns_orthogonalize_batched on two calls in a
row (the second call reuses the array the first one left behind), and that a
batch too large for the array is refused before anything runs. It is named to
be collected last, and builds and loads the library itself so it also passes
alone in a fresh process.
"""
import numpy as np
import pytest
import torch

import oracle
from newton_schulz_quintic_gb300 import api

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-4, torch.bfloat16: 3e-2}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from newton_schulz_quintic_gb300 import build
    build.build()
    api.load_library()


def _batch(shapes, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    return [(torch.randn(s, generator=g) * 0.02).to(dtype) for s in shapes]


def _rel(a, b):
    a, b = oracle.to_f64(a), oracle.to_f64(b)
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / nb) if nb > 0 else float(np.linalg.norm(a))


def _compare(xs):
    ref = [x.cuda() for x in xs]
    got = [x.cuda() for x in xs]
    api.orthogonalize_batched(ref)
    api.orthogonalize_batched_noalloc(got)
    torch.cuda.synchronize()
    assert api.get_status() == 0
    for x, r, g in zip(xs, ref, got):
        assert _rel(g.cpu(), r.cpu()) <= TOL[x.dtype]
        assert torch.all(torch.isfinite(g.float()))


def test_noalloc_matches_default_entry_point_two_calls_in_a_row():
    # first call: tensor-core path (two orientations) + resident kernel
    _compare(_batch([(1024, 2048), (520, 300), (24, 2304)], torch.bfloat16, seed=1))
    # second call: different shapes over the scratch the first call left behind
    _compare(_batch([(300, 520), (2048, 1024), (64, 128)], torch.bfloat16, seed=2))


def test_noalloc_fp32_path():
    _compare(_batch([(100, 300), (64, 128)], torch.float32, seed=3))


def test_noalloc_rejects_batches_beyond_its_scratch():
    x = torch.zeros((8192, 6144), dtype=torch.bfloat16, device="cuda")
    before = x.clone()
    with pytest.raises(api.NSError) as e:
        api.orthogonalize_batched_noalloc([x])
    assert e.value.code == -7
    assert torch.equal(x, before)
