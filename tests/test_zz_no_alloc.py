"""The entry point that allocates no device memory.

Some callers cannot allocate device memory at the moment they orthogonalize:
a training process whose framework allocator already holds nearly all of HBM,
an optimizer step that cannot wait on an allocator, a runtime that forbids
allocation after start-up. ns_orthogonalize_batched_noalloc serves them from a
fixed 256 MiB scratch array inside the library. Through the C ABI this file
checks that it runs the same kernels as ns_orthogonalize_batched -- the same
bits, on two calls in a row, the second over the scratch the first left
behind -- that it requests no device allocation even when the library's
workspace cache is empty, and that a batch too large for the array is refused
before anything runs. It is named to be collected last, and builds and loads
the library itself, so it also passes alone in a fresh process.
"""
import pytest
import torch

from newton_schulz_quintic_gb300 import api

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from newton_schulz_quintic_gb300 import build
    build.build()
    api.load_library()


def _batch(shapes, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    return [(torch.randn(s, generator=g) * 0.02).to(dtype) for s in shapes]


def _compare(xs):
    ref = [x.cuda() for x in xs]
    api.orthogonalize_batched(ref)
    torch.cuda.synchronize()
    # empty the library's workspace cache: a fall-back onto the allocating
    # path would now have to allocate, and the counter would show it
    api.release_workspace()
    allocs = api.num_workspace_allocations()
    got = [x.cuda() for x in xs]
    api.orthogonalize_batched_noalloc(got)      # the first call on a device also finds the array
    torch.cuda.synchronize()
    again = [x.cuda() for x in xs]
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    api.orthogonalize_batched_noalloc(again)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] >= free_before
    assert api.num_workspace_allocations() == allocs
    assert api.get_status() == 0
    for r, g, a in zip(ref, got, again):
        assert torch.equal(g, r)             # same kernels, same inputs: the same bits
        assert torch.equal(a, r)


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
