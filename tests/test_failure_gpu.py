"""Failure detection on the device, without faulting anything.

Every wait inside the library's kernels is bounded, with its limit passed in
as a kernel parameter; when one gives up, the kernel records NS_ETIMEOUT in the
device status word, drains its in-flight work and returns, so the host can read
the failure and the CUDA context stays usable. Two self-tests make a wait run
out with a 20 ms limit:

* an mbarrier that nothing arrives on (one CTA);
* the tensor-core kernel's own dependency waits: a cooperative single-launch
  call whose completion counters are never advanced, so every item that needs
  an earlier phase of its matrix waits on a counter that never reaches its
  target (the hang the dion page's "Test plan" catches with a timeout).

After each, the status is read once, then cleared, and a parity call runs.
"""
import numpy as np
import pytest
import torch

import oracle
from newton_schulz_quintic_gb300 import api

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from newton_schulz_quintic_gb300 import build
    build.build()
    api.load_library()


def _parity_call_still_works():
    g = torch.Generator().manual_seed(3)
    x = (torch.randn((300, 520), generator=g) * 0.02).to(torch.bfloat16)
    d = x.cuda()
    api.orthogonalize_batched([d])
    torch.cuda.synchronize()
    assert api.get_status() == 0
    ref = oracle.orthogonalize(x)
    got = oracle.to_f64(d.cpu())
    assert np.linalg.norm(got - ref) / np.linalg.norm(ref) <= 3e-2


def test_bounded_wait_reports_timeout_and_context_survives():
    assert api.get_status() == 0
    assert api.selftest_wait_timeout(20000) == 0          # the wait gave up as designed
    assert api.get_status() == -5                         # NS_ETIMEOUT, read once ...
    assert api.get_status() == 0                          # ... then cleared
    _parity_call_still_works()


def test_dependency_counter_wait_times_out_and_context_survives():
    assert api.get_status() == 0
    assert api.selftest_dependency_timeout(20000) == 0    # the counter waits gave up
    assert api.get_status() == -5
    assert api.get_status() == 0
    _parity_call_still_works()
    # the single-launch schedule itself is unharmed
    api.set_gemm_schedule("single")
    try:
        _parity_call_still_works()
    finally:
        api.set_gemm_schedule("phase")



def test_workspace_allocation_failure_is_reported_before_launch():
    # the host refuses the workspace (as if the allocation failed): NS_ENOMEM,
    # nothing launched, the matrices untouched, and the library still works
    g = torch.Generator().manual_seed(5)
    x = (torch.randn((1024, 2048), generator=g) * 0.02).to(torch.bfloat16)
    d = x.cuda()
    api.release_workspace()                      # the cache holds nothing to reuse
    launches = api.num_kernel_launches()
    api.set_workspace_limit(1 << 20)             # far below the batch's workspace
    try:
        with pytest.raises(api.NSError) as e:
            api.orthogonalize_batched([d])
        assert e.value.code == -3                # NS_ENOMEM
    finally:
        api.set_workspace_limit(0)
    torch.cuda.synchronize()
    assert api.num_kernel_launches() == launches
    assert torch.equal(d.cpu(), x)
    assert api.get_status() == 0
    _parity_call_still_works()
