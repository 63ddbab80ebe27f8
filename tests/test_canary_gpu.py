"""Guard bands around everything the library writes (a substitute for a
memory checker, which is not available on these GPUs).

* Caller matrices embedded in one large buffer, each with sentinel bytes
  before and after it, some starting on a 16-byte boundary (step 1 reads them
  in place through TMA) and some 2 bytes past one (step 1 works on a copy):
  after bf16 and fp32 calls every sentinel byte is unchanged and every matrix
  has the same bits as the same matrix orthogonalized on its own.
* An explicit workspace larger than ns_workspace_bytes with a sentinel tail:
  the tail is unchanged after the call.
"""
import pytest
import torch

from newton_schulz_quintic_gb300 import api

pytestmark = pytest.mark.gpu

GUARD = 4096                    # sentinel elements before and after each matrix
SENTINEL = {torch.bfloat16: 0x4B4B, torch.float32: 0x4B4B4B4B}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from newton_schulz_quintic_gb300 import build
    build.build()
    api.load_library()


def seeded(shape, dtype, seed, std):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * std).to(dtype)


def bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


def embed(xs, misalign):
    """One device buffer: [guard][matrix 0][guard][matrix 1]...[guard], the
    matrices at offsets rounded to 16 bytes, plus `misalign[i]` elements."""
    dtype = xs[0].dtype
    elt = torch.tensor([], dtype=dtype).element_size()
    per16 = 16 // elt
    offs, pos = [], GUARD
    for x, mis in zip(xs, misalign):
        pos = (pos + per16 - 1) // per16 * per16 + mis
        offs.append(pos)
        pos += x.numel() + GUARD
    buf = torch.empty(pos, dtype=dtype, device="cuda")
    bits(buf).fill_(SENTINEL[dtype])
    views = []
    for x, o in zip(xs, offs):
        v = buf[o:o + x.numel()].view(x.shape)
        v.copy_(x.cuda())
        views.append(v)
    return buf, offs, views


def check_guards(buf, offs, xs):
    b = bits(buf).cpu()
    mask = torch.ones(b.numel(), dtype=torch.bool)
    for x, o in zip(xs, offs):
        mask[o:o + x.numel()] = False
    guard = b[mask]
    assert guard.numel() > 0
    assert torch.all(guard == SENTINEL[buf.dtype]), "a sentinel byte outside the matrices changed"


@pytest.mark.parametrize("dtype,shapes,std", [
    (torch.bfloat16, [(300, 520), (520, 300), (1024, 2048), (24, 2304), (129, 1031), (1000, 17)], 0.02),
    (torch.float32, [(64, 128), (100, 300), (300, 100), (130, 129)], 1.0),
])
@pytest.mark.parametrize("mis", [0, 1])
def test_matrices_in_guarded_buffer(dtype, shapes, std, mis):
    xs = [seeded(s, dtype, 500 + i, std) for i, s in enumerate(shapes)]
    # every other matrix misaligned by `mis` elements
    misalign = [mis * (i % 2) for i in range(len(xs))]
    buf, offs, views = embed(xs, misalign)
    api.orthogonalize_batched(views)
    torch.cuda.synchronize()
    assert api.get_status() == 0
    check_guards(buf, offs, xs)
    # each matrix alone, in its own allocation, gives the same bits
    alone = [x.cuda() for x in xs]
    for a in alone:
        api.orthogonalize_batched([a])
    torch.cuda.synchronize()
    for v, a in zip(views, alone):
        assert torch.equal(bits(v.contiguous()), bits(a))


@pytest.mark.parametrize("dtype,shapes,std", [
    (torch.bfloat16, [(300, 520), (520, 300), (24, 2304)], 0.02),
    (torch.float32, [(100, 300), (64, 128)], 1.0),
])
def test_workspace_tail_untouched(dtype, shapes, std):
    xs = [seeded(s, dtype, 600 + i, std) for i, s in enumerate(shapes)]
    need = api.workspace_bytes([tuple(x.shape) for x in xs], dtype)
    tail = 1 << 16
    ws = torch.empty(need + tail, dtype=torch.uint8, device="cuda")
    ws.fill_(0xA5)
    dev = [x.cuda() for x in xs]
    api.orthogonalize_batched(dev, workspace=ws)
    torch.cuda.synchronize()
    assert api.get_status() == 0
    assert torch.all(ws[need:] == 0xA5), "the call wrote past ns_workspace_bytes"
    ref = [x.cuda() for x in xs]
    api.orthogonalize_batched(ref)
    torch.cuda.synchronize()
    for d, r in zip(dev, ref):
        assert torch.equal(bits(d), bits(r))
