"""ctypes binding of libns (C ABI in include/ns.h).

Argument marshalling only: torch tensors become device pointers, shapes become
an int64 array, and the current torch CUDA stream becomes the cudaStream_t.
Every step of the computation runs in the library's CUDA kernels. There is no
fallback: if ``libns.so`` is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import itertools
import os
import threading

NS_F32 = 0
NS_BF16 = 1

_ERRORS = {0: "NS_OK", -1: "NS_EINVAL", -2: "NS_EALIGN", -3: "NS_ENOMEM", -4: "NS_ECUDA",
           -5: "NS_ETIMEOUT", -6: "NS_ENODEV", -7: "NS_ETOOBIG", -8: "NS_EBOUNDS"}

_PKG = os.path.dirname(os.path.abspath(__file__))
_lock = threading.Lock()
_lib = None


class NSError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = int(code)
        name = _ERRORS.get(self.code, str(code))
        msg = f"{what}: {name}" if what else name
        try:
            desc = load_library().ns_strerror(self.code)
            if desc:
                msg += f" ({desc.decode()})"
        except Exception:  # the library itself may be what is missing
            pass
        super().__init__(msg)


def library_path() -> str:
    return os.environ.get("NS_LIBRARY_PATH", os.path.join(_PKG, "libns.so"))


def load_library() -> ctypes.CDLL:
    """Load libns.so (built in-tree by ``newton_schulz_quintic_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(
                f"libns.so not found at {path}: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'` "
                "(no CPU fallback exists)")
        lib = ctypes.CDLL(path)
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        lib.ns_orthogonalize_batched.restype = i32
        lib.ns_orthogonalize_batched.argtypes = [vp, vp, i32, i32, vp, i32, vp]
        lib.ns_orthogonalize_batched_ex.restype = i32
        lib.ns_orthogonalize_batched_ex.argtypes = [vp, vp, i32, i32, vp, ctypes.c_float, i32, vp,
                                                    ctypes.c_size_t, vp]
        lib.ns_orthogonalize_batched_host.restype = i32
        lib.ns_orthogonalize_batched_host.argtypes = [vp, vp, i32, i32, vp, i32, vp]
        lib.ns_workspace_bytes.restype = ctypes.c_size_t
        lib.ns_workspace_bytes.argtypes = [vp, i32, i32]
        lib.ns_cost.restype = i64
        lib.ns_cost.argtypes = [i64, i64]
        lib.ns_get_status.restype = i32
        lib.ns_get_status.argtypes = [vp]
        lib.ns_strerror.restype = ctypes.c_char_p
        lib.ns_strerror.argtypes = [i32]
        lib.ns_release_workspace.restype = i32
        lib.ns_release_workspace.argtypes = []
        lib.ns_num_kernel_launches.restype = i64
        lib.ns_num_kernel_launches.argtypes = []
        lib.ns_orthogonalize_batched_sched.restype = i32
        lib.ns_orthogonalize_batched_sched.argtypes = [vp, vp, i32, i32, vp, i32, vp]
        lib.ns_orthogonalize_batched_noalloc.restype = i32
        lib.ns_orthogonalize_batched_noalloc.argtypes = [vp, vp, i32, i32, vp, i32, vp]
        lib.ns_selftest_wait_timeout.restype = i32
        lib.ns_selftest_wait_timeout.argtypes = [i32, vp]
        lib.ns_selftest_dependency_timeout.restype = i32
        lib.ns_selftest_dependency_timeout.argtypes = [i32, vp]
        lib.ns_muon_update_batched.restype = i32
        lib.ns_muon_update_batched.argtypes = [vp, vp, vp, vp, i32, i32, vp, ctypes.c_float, i32,
                                               ctypes.c_float, i32, vp]
        lib.ns_selftest_bounds_check.restype = i32
        lib.ns_selftest_bounds_check.argtypes = [vp]
        lib.ns_set_workspace_limit.restype = i32
        lib.ns_set_workspace_limit.argtypes = [ctypes.c_size_t]
        lib.ns_set_nvtx.restype = i32
        lib.ns_set_nvtx.argtypes = [i32]
        lib.ns_num_workspace_allocations.restype = i64
        lib.ns_num_workspace_allocations.argtypes = []
        lib.ns_plan_shards.restype = i32
        lib.ns_plan_shards.argtypes = [vp, vp, i32, i32, ctypes.c_double, i32, vp, vp]
        lib.ns_set_gemm_schedule.restype = i32
        lib.ns_set_gemm_schedule.argtypes = [i32]
        lib.ns_set_f32_gemm.restype = i32
        lib.ns_set_f32_gemm.argtypes = [i32]
        lib.ns_set_kernel_timing.restype = i32
        lib.ns_set_kernel_timing.argtypes = [i32]
        lib.ns_get_kernel_times.restype = i32
        lib.ns_get_kernel_times.argtypes = [vp, vp, i32]
        _lib = lib
        return lib


def _dtype_code(dtype) -> int:
    import torch
    if dtype == torch.float32:
        return NS_F32
    if dtype == torch.bfloat16:
        return NS_BF16
    raise TypeError(f"unsupported dtype {dtype}: use float32 or bfloat16")


def _marshal(mats, coeffs):
    """Device pointers and (M, N) pairs of the matrices as C arrays (numpy
    buffers, kept alive by the caller for the duration of the call)."""
    import numpy as np
    import torch
    n = len(mats)
    ptrs = np.fromiter(map(torch.Tensor.data_ptr, mats), dtype=np.uint64, count=n)
    shapes = np.fromiter(itertools.chain.from_iterable(t.shape for t in mats), dtype=np.int64, count=2 * n)
    co = None
    if coeffs is not None:
        if len(coeffs) != 3:
            raise ValueError("coeffs must be (a, b, c)")
        co = (ctypes.c_float * 3)(*[float(v) for v in coeffs])
    return ptrs, shapes, co


def _ptr(a) -> ctypes.c_void_p:
    return ctypes.c_void_p(a.ctypes.data)


def _check(mats, want_cuda: bool):
    if not mats:
        return None
    t0 = mats[0]
    dt, dev = t0.dtype, t0.device
    for t in mats:
        if t.dim() != 2:
            raise ValueError("every matrix must be 2-D")
        if t.dtype != dt or t.device != dev:
            raise ValueError("all matrices must share dtype and device")
        if not t.is_contiguous():
            raise ValueError("matrices must be contiguous (row-major)")
    if want_cuda and dev.type != "cuda":
        raise ValueError("matrices must be CUDA tensors")
    if not want_cuda and dev.type == "cuda":
        raise ValueError("host entry point takes CPU tensors")
    return _dtype_code(dt)


def orthogonalize_batched(mats, steps: int = 5, coeffs=None, eps: float | None = None,
                          stream=None, workspace=None) -> None:
    """In-place Newton-Schulz of a list of 2-D CUDA tensors (float32 or bfloat16).

    ``stream`` defaults to torch's current stream on the tensors' device.
    With ``eps`` or ``workspace`` given, the ``_ex`` entry point is used
    (``workspace`` is a CUDA uint8 tensor of at least ``workspace_bytes``).
    """
    import torch
    lib = load_library()
    mats = list(mats)
    code = _check(mats, want_cuda=True)
    if code is None:
        return
    dev = mats[0].device
    with torch.cuda.device(dev):
        s = stream if stream is not None else torch.cuda.current_stream(dev)
        sp = ctypes.c_void_p(s.cuda_stream)
        ptrs, shapes, co = _marshal(mats, coeffs)
        if eps is None and workspace is None:
            rc = lib.ns_orthogonalize_batched(_ptr(ptrs), _ptr(shapes), len(mats), int(steps), co, code, sp)
        else:
            e = 1e-7 if eps is None else float(eps)
            if workspace is None:
                need = workspace_bytes([tuple(t.shape) for t in mats], mats[0].dtype)
                workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
                # the caching allocator must not hand this block out again
                # before the work queued on `s` has finished with it
                workspace.record_stream(s)
            rc = lib.ns_orthogonalize_batched_ex(_ptr(ptrs), _ptr(shapes), len(mats), int(steps), co, e, code,
                                                 ctypes.c_void_p(workspace.data_ptr()),
                                                 workspace.numel(), sp)
    if rc != 0:
        raise NSError(rc, "ns_orthogonalize_batched")


def muon_update_batched(grads, moms, outs, mu: float = 0.95, nesterov: bool = True, scale: float = 1.0,
                        steps: int = 5, coeffs=None, stream=None) -> None:
    """One optimizer step around the orthogonalization (ns_muon_update_batched):
    for every matrix, moms[i] <- mu * moms[i] + grads[i] (in place), then
    outs[i] <- scale * NS(grads[i] + mu * moms[i]) with Nesterov momentum, else
    scale * NS(moms[i]). outs[i] may be grads[i] itself. Three lists of CUDA
    tensors of one dtype, matching shapes, contiguous."""
    import torch
    lib = load_library()
    grads, moms, outs = list(grads), list(moms), list(outs)
    if not (len(grads) == len(moms) == len(outs)):
        raise ValueError("grads, moms and outs must have the same length")
    code = _check(grads + moms + outs, want_cuda=True)
    if code is None:
        return
    for g, m, o in zip(grads, moms, outs):
        if g.shape != m.shape or g.shape != o.shape:
            raise ValueError("a matrix's gradient, momentum and output must have one shape")
    dev = grads[0].device
    with torch.cuda.device(dev):
        s = stream if stream is not None else torch.cuda.current_stream(dev)
        pg, shapes, co = _marshal(grads, coeffs)
        pm, _, _ = _marshal(moms, None)
        po, _, _ = _marshal(outs, None)
        rc = lib.ns_muon_update_batched(_ptr(pg), _ptr(pm), _ptr(po), _ptr(shapes), len(grads), int(steps), co,
                                        float(mu), 1 if nesterov else 0, float(scale), code,
                                        ctypes.c_void_p(s.cuda_stream))
    if rc != 0:
        raise NSError(rc, "ns_muon_update_batched")


class PreparedBatch:
    """A batch whose arguments are marshalled once: calling it runs
    ns_orthogonalize_batched on the same matrices with the same steps and
    coefficients, passing on the device pointers and shapes built when it was
    made. For callers that orthogonalize the same buffers every optimizer step,
    where per-call argument marshalling would otherwise be a noticeable share
    of a small batch's time. The tensors must keep their storage (the same
    data_ptr) for as long as the batch is used; it holds references to them."""

    def __init__(self, mats, steps: int = 5, coeffs=None):
        import torch
        self.mats = list(mats)
        self.code = _check(self.mats, want_cuda=True)
        self.steps = int(steps)
        self.device = self.mats[0].device if self.mats else torch.device("cuda")
        self._ptrs, self._shapes, self._co = _marshal(self.mats, coeffs)
        self._args = (_ptr(self._ptrs), _ptr(self._shapes), len(self.mats), self.steps, self._co, self.code)

    def __call__(self, stream=None) -> None:
        import torch
        if self.code is None:
            return
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        rc = load_library().ns_orthogonalize_batched(*self._args, ctypes.c_void_p(s.cuda_stream))
        if rc != 0:
            raise NSError(rc, "ns_orthogonalize_batched")


def orthogonalize_batched_schedule(mats, table, stream=None) -> None:
    """In-place Newton-Schulz with a per-step coefficient table: ``table`` is a
    sequence of (a, b, c) triples, one per step (at most 32 steps)."""
    import torch
    lib = load_library()
    mats = list(mats)
    rows = [tuple(float(v) for v in r) for r in table]
    if any(len(r) != 3 for r in rows):
        raise ValueError("every table row must be (a, b, c)")
    code = _check(mats, want_cuda=True)
    if code is None:
        return
    dev = mats[0].device
    with torch.cuda.device(dev):
        s = stream if stream is not None else torch.cuda.current_stream(dev)
        ptrs, shapes, _ = _marshal(mats, None)
        tab = (ctypes.c_float * max(3 * len(rows), 3))(*[v for r in rows for v in r])
        rc = lib.ns_orthogonalize_batched_sched(_ptr(ptrs), _ptr(shapes), len(mats), len(rows), tab, code,
                                                ctypes.c_void_p(s.cuda_stream))
    if rc != 0:
        raise NSError(rc, "ns_orthogonalize_batched_sched")


def orthogonalize_batched_noalloc(mats, steps: int = 5, coeffs=None, stream=None) -> None:
    """In-place Newton-Schulz through the entry point that allocates no device
    memory (for callers that cannot allocate: its scratch is a fixed 256 MiB
    array inside the library; larger batches raise NSError NS_ETOOBIG)."""
    import torch
    lib = load_library()
    mats = list(mats)
    code = _check(mats, want_cuda=True)
    if code is None:
        return
    dev = mats[0].device
    with torch.cuda.device(dev):
        s = stream if stream is not None else torch.cuda.current_stream(dev)
        ptrs, shapes, co = _marshal(mats, coeffs)
        rc = lib.ns_orthogonalize_batched_noalloc(_ptr(ptrs), _ptr(shapes), len(mats), int(steps), co, code,
                                                  ctypes.c_void_p(s.cuda_stream))
    if rc != 0:
        raise NSError(rc, "ns_orthogonalize_batched_noalloc")


def orthogonalize_batched_host(mats, steps: int = 5, coeffs=None, device=None, stream=None) -> None:
    """In-place Newton-Schulz of CPU tensors through the library's host entry
    point (host-to-device copies, compute, device-to-host copies, sync)."""
    import torch
    lib = load_library()
    mats = list(mats)
    code = _check(mats, want_cuda=False)
    if code is None:
        return
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        s = stream if stream is not None else torch.cuda.current_stream(dev)
        ptrs, shapes, co = _marshal(mats, coeffs)
        rc = lib.ns_orthogonalize_batched_host(_ptr(ptrs), _ptr(shapes), len(mats), int(steps), co, code,
                                               ctypes.c_void_p(s.cuda_stream))
    if rc != 0:
        raise NSError(rc, "ns_orthogonalize_batched_host")


def workspace_bytes(shapes, dtype) -> int:
    lib = load_library()
    code = dtype if isinstance(dtype, int) else _dtype_code(dtype)
    shapes = list(shapes)
    arr = (ctypes.c_int64 * max(2 * len(shapes), 1))(*[int(d) for s in shapes for d in s])
    return int(lib.ns_workspace_bytes(arr, len(shapes), code))


def cost(M: int, N: int) -> int:
    """max(M,N) * min(M,N)^2, computed by the library."""
    return int(load_library().ns_cost(int(M), int(N)))


def get_status(stream=None) -> int:
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(load_library().ns_get_status(ctypes.c_void_p(s.cuda_stream)))


def release_workspace() -> None:
    """Synchronise the current device and free the library's cached workspaces there."""
    rc = load_library().ns_release_workspace()
    if rc != 0:
        raise NSError(rc, "ns_release_workspace")


def num_kernel_launches() -> int:
    return int(load_library().ns_num_kernel_launches())


KERNEL_KINDS = ("norm_pass", "norm_finish", "gram", "square", "apply", "resident", "gemm", "prep",
                "momentum")


def set_kernel_timing(enable: bool) -> None:
    load_library().ns_set_kernel_timing(1 if enable else 0)


def kernel_times() -> dict:
    """{kind: (total_ms, launches)} recorded since set_kernel_timing(True)."""
    n = len(KERNEL_KINDS)
    ms = (ctypes.c_double * n)()
    cnt = (ctypes.c_int64 * n)()
    rc = load_library().ns_get_kernel_times(ms, cnt, n)
    if rc != 0:
        raise NSError(rc, "ns_get_kernel_times")
    return {k: (float(ms[i]), int(cnt[i])) for i, k in enumerate(KERNEL_KINDS)}


def selftest_wait_timeout(limit_us: int = 20000, stream=None) -> int:
    """Run the bounded-wait self-test (see include/ns.h); returns its status code."""
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(load_library().ns_selftest_wait_timeout(int(limit_us), ctypes.c_void_p(s.cuda_stream)))


def selftest_dependency_timeout(limit_us: int = 20000, stream=None) -> int:
    """Run the dependency-counter timeout self-test (see include/ns.h); returns
    its status code."""
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(load_library().ns_selftest_dependency_timeout(int(limit_us),
                                                             ctypes.c_void_p(s.cuda_stream)))


def selftest_bounds_check(stream=None) -> int:
    """Exercise a debug build's bounds checks (see include/ns.h); NS_OK in a
    debug build, NS_EINVAL in a release build."""
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(load_library().ns_selftest_bounds_check(ctypes.c_void_p(s.cuda_stream)))


def set_workspace_limit(nbytes: int) -> None:
    """Cap on any one workspace the library's cache allocates (0: none)."""
    load_library().ns_set_workspace_limit(int(nbytes))


def set_nvtx(enable: bool) -> None:
    """NVTX ranges around every call and launch of the library (for profilers)."""
    load_library().ns_set_nvtx(1 if enable else 0)


def num_workspace_allocations() -> int:
    """Device workspace allocations the library has requested since load."""
    return int(load_library().ns_num_workspace_allocations())


PLAN_ORDERS = {"cost": 0, "numel": 1}


def plan_shards(shapes, nshards: int, numel_eps: float = 0.3, order: str = "cost", loads=None,
                numels=None):
    """Assign matrices (list of (M, N)) to nshards shards; returns (assign, loads).

    Largest first onto the least-loaded shard, sized by ns_cost (order="cost")
    or by element count (order="numel"), with a per-call numel cap and a
    least-numel fallback; ``loads`` carries per-shard loads across calls and
    ``numels`` overrides the stored element counts. Host-only: no GPU is touched."""
    lib = load_library()
    shapes = [tuple(int(d) for d in s) for s in shapes]
    n = len(shapes)
    arr = (ctypes.c_int64 * max(2 * n, 1))(*[d for s in shapes for d in s])
    ld = (ctypes.c_int64 * nshards)(*([0] * nshards if loads is None else [int(v) for v in loads]))
    out = (ctypes.c_int * max(n, 1))()
    nm = None if numels is None else (ctypes.c_int64 * max(n, 1))(*[int(v) for v in numels])
    rc = lib.ns_plan_shards(arr, nm, n, int(nshards), float(numel_eps), PLAN_ORDERS[order], ld, out)
    if rc != 0:
        raise NSError(rc, "ns_plan_shards")
    return [int(out[i]) for i in range(n)], [int(v) for v in ld]


GEMM_SCHEDULES = {"phase": 0, "single": 1}


F32_GEMMS = {"tensor": 0, "simt": 1}


def set_f32_gemm(mode: str) -> None:
    """GEMMs of large fp32 matrices: 'tensor' (default; tcgen05 on three bf16
    slices per tensor, six slice products per GEMM) or 'simt' (CUDA-core fp32)."""
    rc = load_library().ns_set_f32_gemm(F32_GEMMS[mode])
    if rc != 0:
        raise NSError(rc, "ns_set_f32_gemm")


def set_gemm_schedule(mode: str) -> None:
    """'phase' (default): one tensor-core launch per step and phase;
    'single': one launch per call with per-matrix dependency counters."""
    rc = load_library().ns_set_gemm_schedule(GEMM_SCHEDULES[mode])
    if rc != 0:
        raise NSError(rc, "ns_set_gemm_schedule")
