"""CPU fp64 oracle for batched quintic Newton-Schulz orthogonalization.

TEST INFRASTRUCTURE ONLY. Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package. The CUDA library never
loads, links or calls anything here, and this package imports nothing from the
CUDA library: the only code the two sides share is the seeded input generator
(``newton_schulz_quintic_gb300.inputs``), which holds none of the method's
arithmetic.

Two independent computations live here:

* ``orthogonalize`` -- the iteration itself, step by step in fp64, in plain C
  (``ns_oracle.c``): s = ||X||_F, X <- X/(s+eps), work on X^T when M > N, then
  ``steps`` times A = X X^T, B = b A + c A^2, X = a X + B X.
  ``orthogonalize_np`` takes the same steps in the same order with NumPy's
  fp64 matrix product as the product primitive; it is what the CPU baseline
  times (the C loops run minutes per step on the largest matrices).
* ``svd_twin`` -- the closed form of the same map through LAPACK's SVD: every
  step is an odd matrix polynomial, so it keeps the singular vectors and maps
  each singular value through f(s) = a s + b s^3 + c s^5.
* ``muon_update`` -- the momentum step before the orthogonalization and the
  scaled update after it, with every constant a parameter.

The pages this follows ("Fix megabatch_orthogonalize_async hang on empty FSDP2
shards", "Balance LayerWise optimizer shards by Newton-Schulz cost, not
parameter size", and the xtuner Muon remainder-strategy PR) run the iteration
but never print it; the step form and coefficients are the standard quintic
Newton-Schulz of Muon. The zero-row invariant is from the first page's "Fix"
section, the cost max(M,N)*min(M,N)^2 from the second page's "Changes" item 1.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

DEFAULT_COEFFS = (3.4445, -4.7750, 2.0315)
DEFAULT_STEPS = 5
DEFAULT_EPS = 1e-7

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ns_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_lock = threading.Lock()
_libs: dict[int, ctypes.CDLL] = {}


def lib_path(mutation: int = 0) -> str:
    name = "libns_oracle.so" if mutation == 0 else f"libns_oracle_mut{mutation}.so"
    return os.path.join(_BUILD, name)


def build(mutation: int = 0, force: bool = False) -> str:
    """Compile ns_oracle.c with gcc (mutation != 0 plants a numbered mistake)."""
    out = lib_path(mutation)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
        return out
    os.makedirs(_BUILD, exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fopenmp", "-shared", "-fPIC",
           f"-DNS_ORACLE_MUTATION={int(mutation)}", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _lib(mutation: int = 0) -> ctypes.CDLL:
    with _lock:
        if mutation not in _libs:
            lib = ctypes.CDLL(build(mutation))
            lib.ns_oracle_cost.restype = ctypes.c_int64
            lib.ns_oracle_cost.argtypes = [ctypes.c_int64, ctypes.c_int64]
            lib.ns_oracle_frobenius.restype = ctypes.c_double
            lib.ns_oracle_frobenius.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64]
            lib.ns_oracle_orthogonalize.restype = ctypes.c_int
            lib.ns_oracle_orthogonalize.argtypes = [
                ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                ctypes.c_double, ctypes.c_double, ctypes.c_double, ctypes.c_double, ctypes.c_int]
            lib.ns_oracle_orthogonalize_sched.restype = ctypes.c_int
            lib.ns_oracle_orthogonalize_sched.argtypes = [
                ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                ctypes.c_void_p, ctypes.c_double, ctypes.c_int]
            _libs[mutation] = lib
        return _libs[mutation]


def cost(M: int, N: int) -> int:
    """Newton-Schulz cost max(M,N)*min(M,N)^2 (second page, "Changes" item 1)."""
    return int(_lib().ns_oracle_cost(int(M), int(N)))


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns (uint16) to float64: a bf16 is the
    top half of an IEEE binary32, so shifting left by 16 gives the same value."""
    u32 = bits.astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


def to_f64(x) -> np.ndarray:
    """Exact fp64 copy of a CPU tensor/array given in float32, float64 or bfloat16."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if x.dtype == torch.bfloat16:
                return bf16_bits_to_f64(x.view(torch.int16).numpy().view(np.uint16))
            return x.numpy().astype(np.float64)
    except ImportError:  # pragma: no cover - torch is always present in this repo
        pass
    return np.asarray(x, dtype=np.float64)


def coeff_table(coeffs, steps):
    """None for one (a, b, c) triple used by every step; else the per-step
    table as a contiguous (steps, 3) fp64 array (row s = a, b, c of step s)."""
    arr = np.asarray(coeffs, dtype=np.float64)
    if arr.ndim == 1:
        return None
    if arr.shape != (int(steps), 3):
        raise ValueError("a coefficient table must have shape (steps, 3)")
    return np.ascontiguousarray(arr)


def orthogonalize(X, steps: int = DEFAULT_STEPS, coeffs=DEFAULT_COEFFS,
                  eps: float = DEFAULT_EPS, orient: int = 0, mutation: int = 0) -> np.ndarray:
    """Newton-Schulz of one M x N matrix in fp64; returns a new array.

    orient 0 follows the rule (work on X^T when M > N); 1 never transposes and
    2 always transposes (only the tests use 1 and 2).
    """
    W = np.ascontiguousarray(to_f64(X), dtype=np.float64).copy()
    if W.ndim != 2:
        raise ValueError("oracle takes 2-D matrices")
    table = coeff_table(coeffs, steps)
    if table is None:
        a, b, c = (float(v) for v in coeffs)
        rc = _lib(mutation).ns_oracle_orthogonalize(
            W.ctypes.data, W.shape[0], W.shape[1], int(steps), a, b, c, float(eps), int(orient))
    else:
        rc = _lib(mutation).ns_oracle_orthogonalize_sched(
            W.ctypes.data, W.shape[0], W.shape[1], int(steps), table.ctypes.data, float(eps), int(orient))
    if rc != 0:
        raise RuntimeError(f"ns_oracle_orthogonalize failed with {rc}")
    return W


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round fp64 values to the nearest bfloat16 (ties to even), returned as
    fp64: first to fp32 (nearest even), then to the top 16 bits of the fp32
    pattern with round-to-nearest-even on the dropped 16 bits."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16) << np.uint64(16)
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


E4M3_MAX = 448.0  # largest finite e4m3 value (1.75 * 2^8; the format has no infinities)


def round_e4m3(x: np.ndarray) -> np.ndarray:
    """Round fp64 values to the nearest 8-bit e4m3 value (1 sign, 4 exponent
    bits with bias 7, 3 mantissa bits; ties to even; subnormals below 2^-6 in
    steps of 2^-9), saturating at +-448, returned as fp64."""
    x = np.asarray(x, dtype=np.float64)
    ax = np.abs(x)
    _, e2 = np.frexp(ax)               # ax = f * 2^e2, f in [0.5, 1)
    e = np.maximum(e2 - 1, -6)         # binade exponent; subnormals share 2^-6's spacing
    step = np.ldexp(1.0, e - 3)        # 3 mantissa bits
    q = np.rint(ax / step) * step      # np.rint rounds halves to even
    q = np.minimum(q, E4M3_MAX)
    return np.where(ax == 0.0, 0.0, np.copysign(q, x))


def quantise_e4m3_tensor(x: np.ndarray) -> np.ndarray:
    """fp8 operand with one scale per tensor: x/s rounded to e4m3, times s,
    s = max|x| / 448 (values exactly representable after scaling back)."""
    amax = float(np.max(np.abs(x))) if x.size else 0.0
    if amax == 0.0:
        return np.zeros_like(x)
    s = amax / E4M3_MAX
    return round_e4m3(x / s) * s


def quantise_mxfp8(x: np.ndarray, axis: int) -> np.ndarray:
    """fp8 operand with block scaling: blocks of 32 consecutive elements along
    `axis` (the contraction index) share the power-of-two scale
    2^ceil(log2(amax / 448)), the smallest that keeps the block's largest
    magnitude within e4m3's range, and each element is rounded to e4m3 after
    dividing by it (MX-style block scaling with e4m3 elements)."""
    x = np.moveaxis(np.asarray(x, dtype=np.float64), axis, -1)
    k = x.shape[-1]
    pad = (-k) % 32
    xp = np.concatenate([x, np.zeros(x.shape[:-1] + (pad,))], axis=-1) if pad else x
    blocks = xp.reshape(xp.shape[:-1] + (-1, 32))
    amax = np.max(np.abs(blocks), axis=-1, keepdims=True)
    scale = np.exp2(np.ceil(np.log2(np.where(amax > 0, amax, 1.0) / E4M3_MAX)))
    q = round_e4m3(blocks / scale) * scale
    q = np.where(amax > 0, q, 0.0).reshape(xp.shape)[..., :k]
    return np.moveaxis(q, -1, axis)


def orthogonalize_np(X, steps: int = DEFAULT_STEPS, coeffs=DEFAULT_COEFFS,
                     eps: float = DEFAULT_EPS, orient: int = 0, emulate: str | None = None) -> np.ndarray:
    """The same steps as ``orthogonalize`` with numpy.matmul (fp64) as the
    product: s = ||X||_F; X/(s+eps); transpose when M > N (orient as above);
    then ``steps`` times A = W W^T, B = b A + c A A, W = a W + B W.

    emulate="bf16" is a diagnostic, not the oracle: after every step it
    rounds A, B and W to bfloat16 (each product and element-wise combination
    itself stays fp64), i.e. the storage precision of a bf16 tensor-core
    implementation that keeps those three matrices in bf16 between phases and
    folds the normalisation into the first step (W_0 = Y/(s+eps) itself is
    never stored, so never rounded).

    emulate="e4m3" and emulate="mxfp8" are diagnostics of an fp8 tensor-core
    variant (not built): W, A and B are stored as bfloat16 as above, and every
    matrix product takes its two operands rounded to e4m3 -- with one scale
    per tensor ("e4m3") or one power-of-two scale per 32 elements along the
    contraction index ("mxfp8") -- while the element-wise terms a W and b A
    use the bf16 values and every sum stays fp64."""
    W = np.array(to_f64(X), dtype=np.float64, copy=True)
    if W.ndim != 2:
        raise ValueError("oracle takes 2-D matrices")
    if W.size == 0:
        return W
    if emulate not in (None, "bf16", "e4m3", "mxfp8"):
        raise ValueError("emulate must be None, 'bf16', 'e4m3' or 'mxfp8'")
    rnd = round_bf16 if emulate is not None else (lambda v: v)
    if emulate == "e4m3":
        qa = qb = lambda v, axis: quantise_e4m3_tensor(v)
    elif emulate == "mxfp8":
        qa = qb = quantise_mxfp8
    else:
        qa = qb = lambda v, axis: v
    table = coeff_table(coeffs, steps)
    rows = [tuple(float(v) for v in coeffs)] * int(steps) if table is None else [tuple(r) for r in table]
    s = np.sqrt(np.sum(W * W))
    W = W / (s + float(eps))
    M, N = W.shape
    transpose = (M > N) if orient == 0 else (orient == 2)
    if transpose:
        W = np.ascontiguousarray(W.T)
    for a, b, c in rows:
        # contraction index: columns of the first operand, rows of the second
        Wq = qa(W, 1)
        A = rnd(Wq @ Wq.T)
        Aq = qa(A, 1)
        B = rnd(b * A + c * (Aq @ Aq))
        W = rnd(a * W + qa(B, 1) @ qb(W, 0))
    return np.ascontiguousarray(W.T) if transpose else W


def orthogonalize_batched(mats, steps: int = DEFAULT_STEPS, coeffs=DEFAULT_COEFFS,
                          eps: float = DEFAULT_EPS) -> list:
    """The batched form: each matrix of the list independently."""
    return [orthogonalize(X, steps, coeffs, eps) for X in mats]


def muon_update(G, Mom, mu: float, nesterov: bool, scale: float, steps: int = DEFAULT_STEPS,
                coeffs=DEFAULT_COEFFS, eps: float = DEFAULT_EPS):
    """The optimizer step around the orthogonalization, in fp64, every constant
    a parameter (the dion page's "Summary" names Muon, NorMuon and Dion2 as the
    callers of the megabatch Newton-Schulz; the pages do not print their
    updates): the momentum buffer becomes Mom' = mu * Mom + G; the matrix
    orthogonalized is X = G + mu * Mom' with Nesterov momentum, else X = Mom';
    the update is scale * NS(X). Returns (Mom', update) as fp64 arrays."""
    g = to_f64(G)
    m_new = float(mu) * to_f64(Mom) + g
    x = g + float(mu) * m_new if nesterov else m_new
    return m_new, float(scale) * orthogonalize(x, steps, coeffs, eps)


def frobenius(X) -> float:
    W = np.ascontiguousarray(to_f64(X))
    return float(_lib().ns_oracle_frobenius(W.ctypes.data, W.shape[0], W.shape[1]))
