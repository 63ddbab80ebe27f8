"""GPU parity of ns_muon_update_batched (the momentum step, Newton-Schulz and
a scaled write of the result) against the oracle's muon_update on the same
seeded inputs: the momentum buffer within one rounding of the working type,
the update within the Newton-Schulz bars (relative Frobenius error 3e-2 for
bf16, 1e-4 for fp32), on the tensor-core, resident and fp32 paths, both
orientations, with and without Nesterov momentum, steps = 0, an output written
over the gradient, and zero rows kept exactly zero."""
import numpy as np
import pytest
import torch

import oracle
from newton_schulz_quintic_gb300 import api

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-4, torch.bfloat16: 3e-2}
MOM_TOL = {torch.float32: 1e-6, torch.bfloat16: 2.5e-3}   # one rounding of each element


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from newton_schulz_quintic_gb300 import build
    build.build()
    api.load_library()


def seeded(shape, dtype, seed, std):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * std).to(dtype)


def rel(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def run(gs, ms, mu, nesterov, scale, steps=5, alias=False):
    g = [x.cuda() for x in gs]
    m = [x.cuda() for x in ms]
    o = g if alias else [torch.empty_like(x) for x in g]
    api.muon_update_batched(g, m, o, mu=mu, nesterov=nesterov, scale=scale, steps=steps)
    torch.cuda.synchronize()
    assert api.get_status() == 0
    return [x.cpu() for x in m], [x.cpu() for x in o]


CASES = [
    (torch.bfloat16, [(300, 520), (520, 300), (1024, 768), (24, 2304), (64, 100)], 0.02),
    (torch.float32, [(64, 128), (100, 300), (300, 100)], 1.0),
]


@pytest.mark.parametrize("dtype,shapes,std", CASES)
@pytest.mark.parametrize("nesterov", [True, False])
def test_matches_oracle(dtype, shapes, std, nesterov):
    gs = [seeded(s, dtype, 900 + i, std) for i, s in enumerate(shapes)]
    ms = [seeded(s, dtype, 950 + i, std) for i, s in enumerate(shapes)]
    mu, scale = 0.95, 0.37
    mom, out = run(gs, ms, mu, nesterov, scale)
    for g, m0, m1, o in zip(gs, ms, mom, out):
        ref_m, ref_o = oracle.muon_update(g, m0, mu, nesterov, scale)
        assert rel(oracle.to_f64(m1), ref_m) <= MOM_TOL[dtype]
        got = oracle.to_f64(o)
        assert np.all(np.isfinite(got))
        assert rel(got, ref_o) <= TOL[dtype], tuple(g.shape)


@pytest.mark.parametrize("dtype,shapes,std", CASES)
def test_without_momentum_is_the_plain_call_bitwise(dtype, shapes, std):
    # mu = 0, scale = 1: the buffer becomes G exactly and the update is exactly
    # what ns_orthogonalize_batched writes for G
    gs = [seeded(s, dtype, 800 + i, std) for i, s in enumerate(shapes)]
    ms = [seeded(s, dtype, 850 + i, std) for i, s in enumerate(shapes)]
    mom, out = run(gs, ms, 0.0, True, 1.0)
    ref = [g.cuda() for g in gs]
    api.orthogonalize_batched(ref)
    torch.cuda.synchronize()
    for g, m1, o, r in zip(gs, mom, out, ref):
        assert torch.equal(m1, g)
        assert torch.equal(o, r.cpu())


def test_output_over_the_gradient_and_zero_steps():
    shapes = [(300, 520), (24, 2304)]
    gs = [seeded(s, torch.bfloat16, 700 + i, 0.02) for i, s in enumerate(shapes)]
    ms = [seeded(s, torch.bfloat16, 750 + i, 0.02) for i, s in enumerate(shapes)]
    m_sep, o_sep = run(gs, ms, 0.9, True, 0.5)
    m_al, o_al = run(gs, ms, 0.9, True, 0.5, alias=True)
    for a, b, c, d in zip(m_sep, m_al, o_sep, o_al):
        assert torch.equal(a, b) and torch.equal(c, d)
    _, o0 = run(gs, ms, 0.9, False, 0.5, steps=0)
    for g, m0, o in zip(gs, ms, o0):
        _, ref = oracle.muon_update(g, m0, 0.9, False, 0.5, steps=0)
        assert rel(oracle.to_f64(o), ref) <= 1e-2   # one normalisation, rounded to bf16


def test_zero_rows_stay_zero():
    x = seeded((18, 2304), torch.bfloat16, 60, 0.02)
    g = torch.zeros((24, 2304), dtype=torch.bfloat16)
    g[:18] = x
    m = torch.zeros_like(g)
    m[:18] = seeded((18, 2304), torch.bfloat16, 61, 0.02)
    big = torch.zeros((600, 1000), dtype=torch.bfloat16)
    big[:, :900] = seeded((600, 900), torch.bfloat16, 62, 0.02)
    mom, out = run([g, big], [m, torch.zeros_like(big)], 0.9, True, 1.0)
    assert torch.all(out[0][18:].view(torch.int16) == 0) and torch.all(mom[0][18:].view(torch.int16) == 0)
    assert torch.all(out[1][:, 900:].view(torch.int16) == 0)
