"""The allocation-free decode step against the workspace decode step.

gma_decode_step_noalloc exists for callers that cannot allocate device memory
when they run a decode step (for example a plugin whose host application owns
every device allocation, or code held to a fixed memory budget).  It keeps
its scratch in a fixed device array inside the library instead of a
caller-provided workspace.  This file runs last on purpose (pytest collects
files in name order), so a run that stops at the first failure has already
run every other test.
"""
import pytest
import torch

from gaussian_mixture_sequence_gb300 import gma, workloads

pytestmark = pytest.mark.gpu
TOL = 1e-4  # the fp32 tolerance of the parity tests (normwise per slice)


def _normwise(a, b):
    a = a.reshape(a.shape[0] * a.shape[1], -1).double()
    b = b.reshape(b.shape[0] * b.shape[1], -1).double()
    return ((a - b).abs().max(1).values / b.abs().max(1).values.clamp_min(1e-300)).max().item()


def test_noalloc_decode_matches_workspace_decode_two_calls():
    wl = workloads.WORKLOADS["decode_b256"].with_(B=4, N=300)
    dev = torch.device("cuda:0")
    mu, vr, lp = (torch.from_numpy(a).to(dev) for a in workloads.params(wl))
    shape = gma.Shape.make(wl.B, wl.H, wl.N, wl.d, wl.dv, wl.K, eps=wl.eps)
    g = torch.Generator(device=dev).manual_seed(11)
    q, k, v = (torch.randn(wl.B, wl.H, wl.N, w, device=dev, generator=g) for w in (wl.d, wl.d, wl.dv))
    state = torch.empty(wl.B, wl.H, wl.K * wl.dv + wl.K, device=dev)
    gma.gma_forward_causal(shape, mu, vr, lp, q, k, v, torch.empty_like(v), state_out=state)
    st_ref, st_na = state.clone(), state.clone()
    for step in range(2):
        qx, kx = (torch.randn(wl.B, wl.H, wl.d, device=dev, generator=g) for _ in range(2))
        vx = torch.randn(wl.B, wl.H, wl.dv, device=dev, generator=g)
        o_ref = torch.empty(wl.B, wl.H, wl.dv, device=dev)
        o_na = torch.empty_like(o_ref)
        gma.gma_decode_step(shape, mu, vr, lp, qx, kx, vx, st_ref, o_ref)
        gma.gma_decode_step_noalloc(shape, mu, vr, lp, qx, kx, vx, st_na, o_na)
        torch.cuda.synchronize(dev)
        eo, es = _normwise(o_na, o_ref), _normwise(st_na, st_ref)
        print(f"step {step}: output {eo:.2e}, state {es:.2e}")
        assert eo <= TOL and es <= TOL
        # both entries launch the same kernels on the same inputs: the results are identical
        assert torch.equal(o_na, o_ref) and torch.equal(st_na, st_ref)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    dev = torch.device("cuda:0")
    H, K, d, dv = 64, 512, 128, 16          # packed parameters: 64*512*128*8 B = 32 MiB > 8 MiB
    shape = gma.Shape.make(1, H, 1, d, dv, K)
    mu = torch.zeros(H, K, d, device=dev)
    lp = torch.zeros(H, K, device=dev)
    x = torch.zeros(1, H, d, device=dev)
    v = torch.zeros(1, H, dv, device=dev)
    st = torch.zeros(1, H, K * dv + K, device=dev)
    o = torch.zeros(1, H, dv, device=dev)
    with pytest.raises(gma.GMAError) as e:
        gma.gma_decode_step_noalloc(shape, mu, mu, lp, x, x, v, st, o)
    assert e.value.status == 4
