"""Failure detection on the device, without faulting anything.

Every wait inside the library's kernels is bounded; when one gives up, the
kernel records NS_ETIMEOUT in the device status word and returns, so the host
can read the failure and the CUDA context stays usable. The self-test entry
point makes one such wait run out (an mbarrier that nothing arrives on, with a
20 ms limit) and this test checks the status and that work still runs after.
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


def test_bounded_wait_reports_timeout_and_context_survives():
    assert api.get_status() == 0
    assert api.selftest_wait_timeout(20000) == 0          # the wait gave up as designed
    assert api.get_status() == -5                         # NS_ETIMEOUT, read once ...
    assert api.get_status() == 0                          # ... then cleared
    g = torch.Generator().manual_seed(3)
    x = (torch.randn((300, 520), generator=g) * 0.02).to(torch.bfloat16)
    d = x.cuda()
    api.orthogonalize_batched([d])
    torch.cuda.synchronize()
    assert api.get_status() == 0
    ref = oracle.orthogonalize(x)
    got = oracle.to_f64(d.cpu())
    assert np.linalg.norm(got - ref) / np.linalg.norm(ref) <= 3e-2
