"""C ABI checks that need no GPU: the library builds for sm_103a and loads,
exports every function include/ns.h declares, and rejects bad arguments
before touching a device (validation runs first and launches nothing)."""
import ctypes
import os
import re
import subprocess

import pytest

from newton_schulz_quintic_gb300 import api, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ns.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return api.load_library()


def _has_gpu():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


def declared_functions():
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ns_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ["ns_orthogonalize_batched", "ns_orthogonalize_batched_ex", "ns_workspace_bytes",
                 "ns_orthogonalize_batched_host", "ns_cost", "ns_get_status", "ns_strerror",
                 "ns_release_workspace"]:
        assert want in names


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", api.library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\sT\s(ns_\w+)", out))
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(lib, name)


def test_built_for_sm103a(lib):
    assert build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]
    assert build.up_to_date()


def test_cost_matches_formula(lib):
    # second page, "Changes" item 1: max(M,N) * min(M,N)^2
    for M, N in [(8192, 6144), (6144, 8192), (4096, 14336), (1024, 4096), (18, 2304), (0, 7), (1, 1)]:
        assert api.cost(M, N) == max(M, N) * min(M, N) ** 2
    assert api.cost(-1, 4) == -1


def test_workspace_bytes(lib):
    assert api.workspace_bytes([], 1) > 0
    small = api.workspace_bytes([(64, 128)], api.NS_F32)      # resident path: descriptors only
    big = api.workspace_bytes([(8192, 6144)], api.NS_BF16)
    # bf16: two iterates in the caller's orientation, A and B (6144 x 6144)
    need = 2 * (2 * 8192 * 6144 + 2 * 6144 * 6144)
    assert need <= big < need + (1 << 20)
    # fp32 on the tensor cores (default): iterates, A and B as three bf16 slices each
    big32 = api.workspace_bytes([(8192, 6144)], api.NS_F32)
    need32 = 3 * need
    assert need32 <= big32 < need32 + (1 << 20)
    # fp32 on the CUDA cores: W, two W^T buffers, A and B
    api.set_f32_gemm("simt")
    try:
        simt32 = api.workspace_bytes([(8192, 6144)], api.NS_F32)
        long_simt = api.workspace_bytes([(70, 20000)], api.NS_F32)
        edge_simt = api.workspace_bytes([(70, 16384)], api.NS_F32)
    finally:
        api.set_f32_gemm("tensor")
    need_simt = 4 * (3 * 6144 * 8192 + 2 * 6144 * 6144)
    assert need_simt <= simt32 < need_simt + (1 << 20)
    # a call with an fp32 matrix longer than 16384 runs on the CUDA cores in either mode
    assert api.workspace_bytes([(70, 20000)], api.NS_F32) == long_simt
    assert api.workspace_bytes([(70, 16384)], api.NS_F32) != edge_simt
    with pytest.raises(KeyError):
        api.set_f32_gemm("fp64")
    assert lib.ns_set_f32_gemm(7) == -1  # NS_EINVAL
    assert small < 1 << 20
    assert api.workspace_bytes([(-1, 5)], api.NS_BF16) == 0
    assert api.workspace_bytes([(5, 5)], 7) == 0


def _call(lib, ptrs, shapes, count, steps=5, dtype=api.NS_BF16):
    return lib.ns_orthogonalize_batched(ptrs, shapes, count, steps, None, dtype, None)


def test_validation_rejects_before_launch(lib):
    P = ctypes.c_void_p
    S = ctypes.c_int64
    good_ptrs = (P * 1)(0x100000)
    good_shape = (S * 2)(4, 8)
    assert _call(lib, good_ptrs, good_shape, 0) == 0                     # empty batch: no-op
    assert _call(lib, good_ptrs, good_shape, -1) == -1                   # negative count
    assert _call(lib, good_ptrs, good_shape, 1, steps=-2) == -1          # negative steps
    assert _call(lib, good_ptrs, good_shape, 1, dtype=5) == -1           # bad dtype
    assert _call(lib, good_ptrs, (S * 2)(-4, 8), 1) == -1                # negative dim
    assert _call(lib, None, good_shape, 1) == -1                         # null pointer array
    assert _call(lib, (P * 1)(0), good_shape, 1) == -1                   # null matrix
    assert _call(lib, (P * 1)(0x100001), good_shape, 1) == -2            # misaligned bf16
    assert _call(lib, (P * 1)(0x100002), good_shape, 1, dtype=api.NS_F32) == -2  # misaligned f32
    assert lib.ns_orthogonalize_batched_ex(good_ptrs, good_shape, 1, 5, None, 1e-7, 1, None, 0, None) == -1
    # size limits: a side above 2^30 - 1 or more than 2^40 elements is refused
    assert _call(lib, good_ptrs, (S * 2)(1 << 30, 1), 1) == -1
    assert _call(lib, good_ptrs, (S * 2)(1, 1 << 30), 1) == -1
    assert _call(lib, good_ptrs, (S * 2)(1 << 21, 1 << 20), 1) == -1
    assert lib.ns_workspace_bytes((S * 2)(1 << 21, 1 << 20), 1, 1) == 0
    assert lib.ns_workspace_bytes((S * 2)(1 << 20, 1 << 20), 1, 1) > 0


@pytest.mark.skipif(_has_gpu(), reason="uses fake device pointers: only run where nothing can launch")
def test_validation_rejects_overlapping_matrices(lib):
    # every case here must be refused by validation, before any launch
    P, S = ctypes.c_void_p, ctypes.c_int64
    shapes = (S * 4)(4, 8, 4, 8)                                        # 64 bytes each in bf16
    assert _call(lib, (P * 2)(0x100000, 0x100000), shapes, 2) == -1    # the same matrix twice
    assert _call(lib, (P * 2)(0x100000, 0x100030), shapes, 2) == -1    # overlapping by 16 bytes
    assert _call(lib, (P * 2)(0x100030, 0x100000), shapes, 2) == -1    # either order
    assert _call(lib, (P * 3)(0x200000, 0x100000, 0x10003e), (S * 6)(4, 8, 4, 8, 1, 1), 3) == -1


@pytest.mark.skipif(_has_gpu(), reason="checks the error path of a machine with no CUDA device")
def test_no_device_is_reported_as_enodev(lib):
    # valid arguments on a machine without a CUDA driver or device: every entry
    # point that needs the GPU says so with NS_ENODEV and touches nothing
    import numpy as np
    P, S = ctypes.c_void_p, ctypes.c_int64
    x = np.arange(64 * 128, dtype=np.float32).reshape(64, 128)
    before = x.copy()
    ptrs, shapes = (P * 1)(x.ctypes.data), (S * 2)(64, 128)
    f32 = api.NS_F32
    tab = (ctypes.c_float * 3)(3.4445, -4.7750, 2.0315)
    ws = np.zeros(1 << 20, dtype=np.uint8)
    assert lib.ns_orthogonalize_batched(ptrs, shapes, 1, 5, None, f32, None) == -6
    assert lib.ns_orthogonalize_batched_host(ptrs, shapes, 1, 5, None, f32, None) == -6
    assert lib.ns_orthogonalize_batched_noalloc(ptrs, shapes, 1, 5, None, f32, None) == -6
    assert lib.ns_orthogonalize_batched_sched(ptrs, shapes, 1, 1, tab, f32, None) == -6
    ws_ptr = P(ws.ctypes.data + (-ws.ctypes.data) % 256)
    assert lib.ns_orthogonalize_batched_ex(ptrs, shapes, 1, 5, None, 1e-7, f32, ws_ptr, 1 << 19, None) == -6
    assert lib.ns_get_status(None) == -6
    assert lib.ns_release_workspace() == -6
    assert lib.ns_selftest_wait_timeout(1000, None) == -6
    assert np.array_equal(x, before)
    # validation still comes first
    assert lib.ns_orthogonalize_batched(ptrs, shapes, 1, -1, None, f32, None) == -1


def test_strerror(lib):
    for code in [0, -1, -2, -3, -4, -5, -6, -7]:
        assert lib.ns_strerror(code)
    assert b"unknown" in lib.ns_strerror(-99)


def test_selftest_rejects_bad_limits_before_launch(lib):
    assert lib.ns_selftest_wait_timeout(0, None) == -1
    assert lib.ns_selftest_wait_timeout(-5, None) == -1
    assert lib.ns_selftest_wait_timeout(20000000, None) == -1
    assert lib.ns_selftest_dependency_timeout(0, None) == -1
    assert lib.ns_selftest_dependency_timeout(20000001, None) == -1


@pytest.mark.skipif(_has_gpu(), reason="uses fake device pointers: only run where nothing can launch")
def test_noalloc_checks_arguments_and_device_before_its_size_limit(lib):
    # the no-allocation entry point returns what every entry point returns for
    # bad arguments and for a missing device, even for a batch that would also
    # be too large for its scratch array; its own refusal comes last
    P, S = ctypes.c_void_p, ctypes.c_int64
    big = (S * 2)(8192, 6144)                     # beyond the 256 MiB scratch
    f = lib.ns_orthogonalize_batched_noalloc
    assert f((P * 1)(0), big, 1, 5, None, 1, None) == -1             # null matrix
    assert f((P * 1)(0x100001), big, 1, 5, None, 1, None) == -2      # misaligned
    assert f((P * 2)(0x100000, 0x100000), (S * 4)(8192, 6144, 8192, 6144), 2, 5, None, 1, None) == -1
    assert f((P * 1)(0x100000), big, 1, -1, None, 1, None) == -1     # negative steps
    assert f((P * 1)(0x100000), big, 1, 5, None, 1, None) == -6      # no device, not "too big"
    assert f(None, None, 0, 5, None, 1, None) == 0                   # empty batch: no-op
    assert lib.ns_selftest_dependency_timeout(1000, None) == -6


def test_schedule_rejects_bad_tables_before_launch(lib):
    P, S = ctypes.c_void_p, ctypes.c_int64
    ptrs, shape = (P * 1)(0x100000), (S * 2)(4, 8)
    assert lib.ns_orthogonalize_batched_sched(ptrs, shape, 1, 5, None, 1, None) == -1
    tab = (ctypes.c_float * (3 * 40))()
    assert lib.ns_orthogonalize_batched_sched(ptrs, shape, 1, 40, tab, 1, None) == -1


def test_gemm_schedule_setter(lib):
    assert lib.ns_set_gemm_schedule(5) == -1
    assert lib.ns_set_gemm_schedule(1) == 0 and lib.ns_set_gemm_schedule(0) == 0


@pytest.mark.skipif(_has_gpu(), reason="uses fake device pointers: only run where nothing can launch")
def test_muon_update_validation_before_launch(lib):
    # every refusal below happens before any launch: arguments, then the
    # overlap of the three buffers, then the device
    P, S = ctypes.c_void_p, ctypes.c_int64
    f = lib.ns_muon_update_batched
    shp = (S * 2)(4, 8)                            # 64 bytes in bf16
    g, m, o = (P * 1)(0x100000), (P * 1)(0x200000), (P * 1)(0x300000)
    c = ctypes.c_float
    assert f(g, m, o, shp, 0, 5, None, c(0.9), 1, c(1.0), 1, None) == 0          # empty batch
    assert f(None, m, o, shp, 1, 5, None, c(0.9), 1, c(1.0), 1, None) == -1      # null array
    assert f(g, (P * 1)(0x200001), o, shp, 1, 5, None, c(0.9), 1, c(1.0), 1, None) == -2  # misaligned
    assert f(g, m, o, shp, 1, 5, None, c(float("nan")), 1, c(1.0), 1, None) == -1
    assert f(g, m, o, shp, 1, 5, None, c(0.9), 1, c(float("inf")), 1, None) == -1
    assert f(g, m, o, shp, 1, 5, None, c(0.9), 2, c(1.0), 1, None) == -1         # nesterov not 0/1
    assert f(g, g, o, shp, 1, 5, None, c(0.9), 1, c(1.0), 1, None) == -1         # momentum is the gradient
    assert f(g, m, m, shp, 1, 5, None, c(0.9), 1, c(1.0), 1, None) == -1         # output is the momentum
    assert f(g, m, (P * 1)(0x200020), shp, 1, 5, None, c(0.9), 1, c(1.0), 1, None) == -1  # partial overlap
    two = (S * 4)(4, 8, 4, 8)
    assert f((P * 2)(0x100000, 0x110000), (P * 2)(0x200000, 0x210000), (P * 2)(0x110000, 0x100000), two, 2, 5,
             None, c(0.9), 1, c(1.0), 1, None) == -1                            # output is another gradient
    # the output written over the gradient is allowed: the call gets as far as the device
    assert f(g, m, g, shp, 1, 5, None, c(0.9), 1, c(1.0), 1, None) == -6
    assert f(g, m, o, shp, 1, 5, None, c(0.9), 0, c(1.0), 1, None) == -6
