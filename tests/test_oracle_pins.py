"""Pins for the CPU fp64 oracle, independent of the oracle's own code.

Each test checks the step-by-step oracle against something fixed by the
mathematics or printed on the pages:

* the SVD closed form U f^steps(S/(||X||+eps)) V^T (a different algorithm);
* exact special cases (one row, a diagonal matrix, orthonormal rows, the zero
  matrix, zero steps) whose result is a scalar recurrence;
* the cubic iteration's limit, the polar factor U V^T;
* invariants: zero rows stay exactly zero (the first page's "Fix" section),
  zero padding leaves the real rows bit-identical, the two orientations agree,
  scale invariance and orthogonal equivariance;
* the quintic's band for the output singular values.

test_mutations plants a numbered mistake in the oracle's C source (a dropped
term, a wrong sign, a wrong index, a wrong norm, one step short) and checks
that the pins fail on it.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import svd_twin
from newton_schulz_quintic_gb300 import inputs

CO = oracle.DEFAULT_COEFFS
EPS = oracle.DEFAULT_EPS


@pytest.fixture(params=["c", "numpy"])
def ns(request):
    """Both implementations of the oracle's steps face the same pins."""
    return oracle.orthogonalize if request.param == "c" else oracle.orthogonalize_np


def rel(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def randn(shape, seed, std=1.0):
    g = np.random.default_rng(seed)
    return g.standard_normal(shape) * std


SHAPES = [(1, 7), (7, 1), (1, 1), (5, 5), (12, 40), (40, 12), (64, 128), (128, 64),
          (33, 97), (97, 33), (24, 2304), (130, 300)]


@pytest.mark.parametrize("shape", SHAPES)
def test_matches_svd_closed_form(ns, shape):
    X = randn(shape, seed=shape[0] * 1000 + shape[1], std=0.02)
    got = ns(X)
    ref = svd_twin.closed_form(X, 5, CO, EPS)
    assert rel(got, ref) < 1e-10


@pytest.mark.parametrize("steps", [0, 1, 2, 3, 7])
def test_matches_svd_closed_form_any_steps(ns, steps):
    X = randn((20, 50), seed=steps)
    assert rel(ns(X, steps=steps), svd_twin.closed_form(X, steps, CO, EPS)) < 1e-10


def test_custom_coefficients_closed_form(ns):
    X = randn((16, 30), seed=3)
    co = (2.0, -1.5, 0.5)
    assert rel(ns(X, steps=4, coeffs=co), svd_twin.closed_form(X, 4, co, EPS)) < 1e-10


def test_zero_steps_is_normalisation(ns):
    X = randn((9, 13), seed=4)
    s = np.sqrt(np.sum(X ** 2))
    got = ns(X, steps=0)
    assert rel(got, X / (s + EPS)) < 1e-15


@pytest.mark.parametrize("shape", [(1, 50), (50, 1), (1, 2304)])
def test_single_row_or_column_scalar_recurrence(ns, shape):
    # one singular value sigma = ||x||: result is f^5(sigma/(sigma+eps)) * x/sigma
    x = randn(shape, seed=11)
    s = np.linalg.norm(x)
    g = svd_twin.quintic_iterate(s / (s + EPS), 5, CO)
    assert rel(ns(x), g * x / s) < 1e-13


def test_diagonal_scalar_recurrence(ns):
    # diagonal input: every entry follows the scalar recurrence on its own
    d = np.array([0.3, -1.7, 0.02, 4.0, -0.5])
    X = np.zeros((5, 9))
    X[np.arange(5), np.arange(5)] = d
    s = np.linalg.norm(d)
    expect = np.zeros_like(X)
    expect[np.arange(5), np.arange(5)] = svd_twin.quintic_iterate(d / (s + EPS), 5, CO)
    got = ns(X)
    assert np.max(np.abs(got - expect)) < 1e-14
    assert np.array_equal(got == 0, expect == 0)


@pytest.mark.parametrize("m,n", [(1, 16), (8, 32), (24, 64), (64, 128)])
def test_orthonormal_rows_scale(ns, m, n):
    # X X^T = I: every step keeps X up to the scalar g = f^5(1/(sqrt(m)+eps))
    Q, _ = np.linalg.qr(randn((n, n), seed=m))
    X = Q[:m]
    g = svd_twin.quintic_iterate(1.0 / (np.sqrt(m) + EPS), 5, CO)
    assert rel(ns(X), g * X) < 1e-12
    assert rel(ns(X.T.copy()), g * X.T) < 1e-12


def test_orthonormal_scale_values(ns):
    # spot values of g (m=1, 8, 24, 64), recomputed from the scalar map
    want = {1: 0.6964365, 8: 1.0669680, 24: 0.7072018, 64: 0.6881399}
    for m, g in want.items():
        Q, _ = np.linalg.qr(randn((2 * m + 3, 2 * m + 3), seed=7))
        X = Q[:m]
        out = ns(X)
        ratio = np.sum(out * X) / np.sum(X * X)
        assert abs(ratio - g) < 1e-6


def test_zero_matrix(ns):
    for shape in [(4, 6), (6, 4), (1, 1)]:
        out = ns(np.zeros(shape))
        assert np.all(out == 0) and not np.any(np.signbit(out))


@pytest.mark.parametrize("shape,zero_rows", [((10, 40), [0, 4, 9]), ((40, 10), [3, 39]),
                                             ((24, 100), list(range(18, 24)))])
def test_zero_rows_stay_exactly_zero(ns, shape, zero_rows):
    X = randn(shape, seed=5)
    X[zero_rows] = 0.0
    out = ns(X)
    assert np.all(out[zero_rows] == 0)
    assert not np.any(np.signbit(out[zero_rows]))
    assert np.all(out[[i for i in range(shape[0]) if i not in zero_rows]] != 0)


def test_zero_columns_stay_exactly_zero(ns):
    X = randn((12, 30), seed=6)
    X[:, [0, 17, 29]] = 0.0
    out = ns(X)
    assert np.all(out[:, [0, 17, 29]] == 0)


@pytest.mark.parametrize("real,shards", [(18, 8), (5, 4), (2, 4), (15, 4)])
def test_padding_equivalence_bit_exact(real, shards):
    # the first page's "Fix": zero-padding shards does not change the real rows
    x = torch.from_numpy(randn((real, 64), seed=real))
    padded = inputs.pad_shards(x, shards)
    out_p = oracle.orthogonalize(padded.numpy())
    out_r = oracle.orthogonalize(x.numpy())
    sizes = inputs.chunk_sizes(real, shards)
    width = max(sizes)
    rows = [r * width + j for r, n in enumerate(sizes) for j in range(n)]
    assert np.array_equal(out_p[rows], out_r)
    pad_rows = [i for i in range(padded.shape[0]) if i not in rows]
    assert np.all(out_p[pad_rows] == 0)


@pytest.mark.parametrize("shape", [(20, 50), (50, 20), (1, 9), (30, 30)])
def test_orientations_agree(ns, shape):
    # X p(X^T X) = p(X X^T) X: the iteration on X and on X^T give one result
    X = randn(shape, seed=8)
    a = ns(X, orient=1)
    b = ns(X, orient=2)
    assert rel(a, b) < 1e-12


def test_scale_invariance(ns):
    X = randn((16, 48), seed=9)
    for alpha in (1e-3, 7.5, 1e4):
        assert rel(ns(alpha * X, eps=0.0), ns(X, eps=0.0)) < 1e-12


def test_orthogonal_equivariance(ns):
    X = randn((16, 40), seed=10)
    Q, _ = np.linalg.qr(randn((16, 16), seed=12))
    R, _ = np.linalg.qr(randn((40, 40), seed=13))
    lhs = ns(Q @ X @ R)
    rhs = Q @ ns(X) @ R
    assert rel(lhs, rhs) < 1e-11


@pytest.mark.parametrize("shape", [(8, 16), (16, 32), (16, 9), (5, 5)])
def test_cubic_iteration_converges_to_polar_factor(ns, shape):
    # (a,b,c) = (1.5, -0.5, 0) is the cubic Newton-Schulz iteration, whose fixed
    # point on full-rank inputs is the orthogonal polar factor U V^T
    X = randn(shape, seed=shape[0] + shape[1])
    out = ns(X, steps=60, coeffs=(1.5, -0.5, 0.0))
    assert np.max(np.abs(out - svd_twin.polar(X))) < 1e-8


def test_singular_value_band(ns):
    # for sigma/||X|| in [2e-3, 1], f^5 stays in [0.6818, 1.2024]; a
    # Gaussian 64x128 has all its normalised singular values in that range
    X = randn((64, 128), seed=14)
    s_in = svd_twin.singular_values(X) / np.linalg.norm(X)
    assert s_in.min() > 2e-3
    s_out = svd_twin.singular_values(ns(X))
    assert s_out.min() >= 0.6818 - 1e-9 and s_out.max() <= 1.2024 + 1e-9
    grid = np.logspace(np.log10(2e-3), 0, 20001)
    g = svd_twin.quintic_iterate(grid, 5, CO)
    assert g.min() >= 0.6818 and g.max() <= 1.2024


def test_bf16_widening_exact():
    x = (torch.randn(100) * 3).to(torch.bfloat16)
    assert np.array_equal(oracle.to_f64(x), x.to(torch.float64).numpy())


def test_cost_of_the_pages_printed_figures():
    # second page: the expensive and dense matrices' costs as printed there
    with open(os.path.join(os.path.dirname(__file__), "golden", "ns_cost.json")) as f:
        g = json.load(f)
    for c in g["costs"]:
        assert oracle.cost(*c["shape"]) == c["cost"]
    hi, dense = g["costs"][0]["cost"], g["costs"][2]["cost"]
    assert hi == g["ratio_expensive_to_dense"] * dense


def test_cost_formula():
    # second page, "Changes" item 1: max(M,N)*min(M,N)^2; and its "Notes":
    # cost = numel * min(M,N)
    for M, N in [(8192, 6144), (6144, 8192), (1, 1), (0, 5), (14336, 4096), (18, 2304)]:
        c = oracle.cost(M, N)
        assert c == M * N * min(M, N)
        assert c == oracle.cost(N, M)
    assert oracle.cost(-1, 3) == -1


MUTATIONS = [1, 2, 3, 4, 5, 6, 7]


@pytest.mark.parametrize("mutation", MUTATIONS)
def test_mutations_are_caught(mutation):
    X = randn((12, 40), seed=15, std=0.02)
    got = oracle.orthogonalize(X, mutation=mutation)
    ref = svd_twin.closed_form(X, 5, CO, EPS)
    # a planted mistake is caught if the result is far from the closed form,
    # or has diverged (some mistakes blow the iteration up to inf / nan)
    if not np.all(np.isfinite(got)):
        return
    with np.errstate(over="ignore", invalid="ignore"):
        err = rel(got, ref)
    assert not np.isfinite(err) or err > 1e-3


@pytest.mark.parametrize("shape", [(40, 12), (12, 40), (64, 64), (130, 300)])
def test_eigh_closed_form_matches_svd_closed_form(shape):
    # the large-size form used for sampled full-size parity agrees with the SVD form
    X = randn(shape, seed=21, std=0.02)
    a = svd_twin.closed_form_eigh(X, 5, CO, EPS)
    b = svd_twin.closed_form(X, 5, CO, EPS)
    assert rel(a, b) < 1e-9
    assert rel(a, oracle.orthogonalize(X)) < 1e-9


def test_eigh_closed_form_keeps_zero_rows():
    X = randn((30, 80), seed=22)
    X[25:] = 0.0
    out = svd_twin.closed_form_eigh(X, 5, CO, EPS)
    assert np.max(np.abs(out[25:])) < 1e-14


def test_round_bf16_matches_torch_cast():
    x = np.random.default_rng(30).standard_normal(10000) * np.logspace(-6, 6, 10000)
    got = oracle.round_bf16(x)
    ref = torch.from_numpy(x).to(torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(got, ref)


def test_bf16_emulation_is_the_oracle_plus_storage_rounding():
    # without rounding it is the oracle; with it, it stays within the bf16
    # error band of the oracle (~1e-2) and is not the oracle
    X = randn((96, 160), seed=31, std=0.02)
    exact = oracle.orthogonalize_np(X)
    emu = oracle.orthogonalize_np(X, emulate="bf16")
    err = rel(emu, exact)
    assert 1e-4 < err < 3e-2
    assert rel(oracle.orthogonalize_np(X, emulate=None), oracle.orthogonalize(X)) < 1e-12


SCHEDULE = [(3.4445, -4.7750, 2.0315), (3.0, -3.2, 1.2), (2.2, -1.8, 0.6), (1.5, -0.5, 0.0), (1.5, -0.5, 0.0)]


@pytest.mark.parametrize("shape", [(20, 50), (50, 20), (64, 64)])
def test_per_step_schedule_matches_closed_form(ns, shape):
    # a different (a, b, c) each step: the singular values follow f_4(...f_0(s))
    X = randn(shape, seed=40, std=0.02)
    got = ns(X, steps=5, coeffs=SCHEDULE)
    assert rel(got, svd_twin.closed_form(X, 5, SCHEDULE, EPS)) < 1e-10


def test_constant_schedule_is_the_plain_call(ns):
    X = randn((30, 70), seed=41)
    assert np.array_equal(ns(X, steps=3, coeffs=[CO] * 3), ns(X, steps=3, coeffs=CO))


def test_round_e4m3_matches_torch_float8_cast():
    # the fp8 emulation's rounding against torch's float8_e4m3fn cast (nearest,
    # ties to even, subnormals), over values spanning the format's range
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    rng = np.random.default_rng(31)
    x = rng.standard_normal(100000) * np.exp(rng.uniform(-12, 6, 100000))
    x = np.concatenate([x, [0.0, 448.0, -448.0, 2.0 ** -9, 2.0 ** -10, 3 * 2.0 ** -10, 1.0625, 1.1875]])
    x = x[np.abs(x) <= 448.0].astype(np.float32).astype(np.float64)
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(oracle.round_e4m3(x), want)
    assert oracle.round_e4m3(np.array([1e6, -1e6])).tolist() == [448.0, -448.0]   # saturates


def test_fp8_operand_quantisers():
    rng = np.random.default_rng(32)
    x = rng.standard_normal((40, 70)) * np.exp(rng.uniform(-3, 3, (40, 70)))
    x[3] = 0.0
    for q in (oracle.quantise_e4m3_tensor, lambda v: oracle.quantise_mxfp8(v, 1),
              lambda v: oracle.quantise_mxfp8(v, 0)):
        y = q(x)
        assert np.array_equal(q(y), y)                  # idempotent: already on the grid
        assert np.all(y[3] == 0)                        # zero rows stay zero
    # block scaling: within a 32-element block along the axis, the error of an
    # element is at most half an e4m3 step at its block's scale
    y = oracle.quantise_mxfp8(x, 1)
    for r in range(40):
        for b0 in range(0, 70, 32):
            blk, qb = x[r, b0:b0 + 32], y[r, b0:b0 + 32]
            amax = np.max(np.abs(blk))
            if amax == 0:
                continue
            scale = 2.0 ** np.ceil(np.log2(amax / 448.0))
            assert np.max(np.abs(qb)) <= 448.0 * scale
            assert np.all(np.abs(qb - blk) <= np.maximum(np.abs(blk) * 2.0 ** -4, scale * 2.0 ** -10) + 1e-300)


# ------------------------------------------------------------ the optimizer step around it

def _rel(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def test_muon_update_without_momentum_is_scaled_newton_schulz():
    # mu = 0: the momentum buffer becomes the gradient and the update is
    # scale times the (separately pinned) Newton-Schulz of the gradient
    g = np.random.default_rng(40).standard_normal((12, 30))
    m0 = np.random.default_rng(41).standard_normal((12, 30))
    for nesterov in (False, True):
        m1, upd = oracle.muon_update(g, m0, 0.0, nesterov, 0.7)
        assert np.array_equal(m1, g)
        assert np.allclose(upd, 0.7 * oracle.orthogonalize(g), rtol=0, atol=1e-14)


def test_muon_momentum_is_a_geometric_series():
    # a constant gradient from a zero buffer: after k steps the buffer is
    # G (1 - mu^k) / (1 - mu); every update is scale * NS(G) because
    # Newton-Schulz does not see the input's scale (up to eps)
    g = np.random.default_rng(42).standard_normal((10, 24))
    mu = 0.9
    m = np.zeros_like(g)
    ref = oracle.orthogonalize(g)
    for k in range(1, 6):
        m, upd = oracle.muon_update(g, m, mu, False, 1.5)
        assert np.allclose(m, g * (1 - mu ** k) / (1 - mu), rtol=1e-14, atol=1e-14)
        assert _rel(upd, 1.5 * ref) < 1e-6


def test_muon_nesterov_input():
    # Nesterov: X = G + mu (mu M + G) = (1 + mu) G + mu^2 M
    rng = np.random.default_rng(43)
    g, m0 = rng.standard_normal((16, 40)), rng.standard_normal((16, 40))
    mu = 0.95
    m1, upd = oracle.muon_update(g, m0, mu, True, 1.0)
    assert np.allclose(m1, mu * m0 + g, rtol=1e-15, atol=1e-15)
    x = (1 + mu) * g + mu * mu * m0
    assert _rel(upd, oracle.orthogonalize(x)) < 1e-12
    # without Nesterov the buffer itself is orthogonalized
    _, plain = oracle.muon_update(g, m0, mu, False, 1.0)
    assert _rel(plain, oracle.orthogonalize(mu * m0 + g)) < 1e-12
    assert _rel(plain, upd) > 1e-3           # the two inputs differ, so the updates do


def test_muon_update_scale_is_linear():
    rng = np.random.default_rng(44)
    g, m0 = rng.standard_normal((8, 20)), rng.standard_normal((8, 20))
    _, u1 = oracle.muon_update(g, m0, 0.5, True, 1.0)
    _, u3 = oracle.muon_update(g, m0, 0.5, True, -3.0)
    assert np.allclose(u3, -3.0 * u1, rtol=1e-15, atol=1e-15)
