"""Bounded waits report their expiry through a status, and the GPU stays usable.

Every mbarrier wait in the tensor-core kernels gives up after a bounded number
of SM cycles.  A wait that expires sets the device's timeout flag; the next
compute call returns GMA_ERR_TIMEOUT without launching anything, and
gma_sync_status(stream) reports it after synchronising.  The wait is made to
expire by the library's test kernel, which waits on an mbarrier that nothing
ever arrives on: no copy or tensor-core product is issued against it, so
nothing is in flight when it gives up (no fault, no hang: about 1 ms).
"""
import pytest
import torch

from gaussian_mixture_sequence_gb300 import gma, workloads
from gpu_cases import TOL, Case, normwise, shape_of

pytestmark = pytest.mark.gpu
LIMIT = 2_000_000   # SM cycles, about 1 ms


def _status(fn):
    try:
        fn()
    except gma.GMAError as e:
        return e.status
    return 0


def test_expired_wait_is_reported_once_by_sync_status():
    gma.gma_sync_status()                      # nothing pending
    gma.gma_test_wait_timeout(LIMIT)
    assert _status(gma.gma_sync_status) == gma.TIMEOUT
    assert _status(gma.gma_sync_status) == 0   # reported once, then cleared


def test_expired_wait_fails_the_next_call_then_the_library_works():
    wl = workloads.WORKLOADS["tiny"].with_(B=1, H=2, N=300, d=64, dv=64, K=128)
    c = Case(wl)
    q, k, v = c.dev["seq"]
    out = torch.full((wl.B, wl.H, wl.N, wl.dv), -1.0, device="cuda:0")
    gma.gma_test_wait_timeout(LIMIT)
    torch.cuda.synchronize()                   # the flag is visible to the host now
    call = lambda: gma.gma_forward_causal(shape_of(wl), *c.prm, q, k, v, out)
    assert _status(call) == gma.TIMEOUT       # nothing was launched
    torch.cuda.synchronize()
    assert (out == -1.0).all()
    call()                                     # the flag was cleared: this call runs
    gma.gma_sync_status()                      # and its kernels' waits did not expire
    err = normwise(c.pick(out), c.ref_causal())
    print(f"causal after a reported timeout: normwise error {err:.3e}")
    assert err <= TOL["f32"]
