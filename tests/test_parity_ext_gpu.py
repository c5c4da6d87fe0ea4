"""GPU parity of the extensions of the hot path: cross-attention (queries of one
sequence reading the memory of another) and the responsibility diagnostics
(soft usage, hard assignments and their entropies), through the C ABI, against
the fp64 oracle on the same seeded inputs."""
import numpy as np
import pytest
import torch

import oracle
from gaussian_mixture_sequence_gb300 import gma, workloads
from gpu_cases import DEV, TOL, normwise, shape_of

pytestmark = pytest.mark.gpu
W = workloads.WORKLOADS


def _t(a, dtype=torch.float32):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV).to(dtype)


def _tdt(name):
    return torch.bfloat16 if name == "bf16" else torch.float32


# --------------------------------------------------------- cross-attention ---

CROSS = [
    (W["tiny"].with_(mode="bidir"), 100, 256),
    (W["tiny"].with_(mode="bidir", B=2, H=3, d=32, dv=128, K=40), 257, 1000),
    (W["tiny"].with_(mode="bidir", B=2, H=2, d=64, dv=64, K=128), 300, 1000),     # tensor-core path
    (W["tiny"].with_(mode="bidir", B=2, H=2, d=64, dv=64, K=128), 1000, 130),
    (W["tiny"].with_(mode="bidir", B=1, H=2, d=64, dv=64, K=128, dist="peaked"), 700, 2049),
    (W["tiny"].with_(mode="bidir", B=1, H=2, d=32, dv=128, K=128, gemm_dtype="bf16", v_dtype="bf16"), 129, 700),
    (W["tiny"].with_(mode="bidir", B=4, H=16, d=64, dv=64, K=128), 1100, 300),   # more chunks than SMs
    (W["tiny"].with_(mode="bidir", B=2, H=2, d=64, dv=64, K=128), 1, 77),
    (W["tiny"].with_(mode="bidir", B=2, H=2, d=16, dv=16, K=8), 50, 0),           # empty memory
    (W["tiny"].with_(mode="bidir", B=2, H=2, d=64, dv=64, K=128), 50, 0),
    (W["tiny"].with_(mode="bidir", B=2, H=2, d=64, dv=64, K=256), 700, 300),  # component groups
    (W["tiny"].with_(mode="bidir", B=2, H=2, d=32, dv=64, K=48), 300, 900),   # padded components
    (W["tiny"].with_(mode="bidir", B=2, H=2, d=64, dv=64, K=256), 50, 0),
]


@pytest.mark.parametrize("wl,nq,nk", CROSS, ids=[f"K{w.K}-dv{w.dv}-q{q}-k{k}-{w.gemm_dtype}" for w, q, k in CROSS])
def test_cross(wl, nq, nk):
    mu, vr, lp = workloads.params(wl)
    S = wl.B * wl.H
    q = workloads.full_inputs(wl.with_(N=nq, seed=wl.seed + 17))[0]
    _, k, v = workloads.full_inputs(wl.with_(N=nk))
    out = torch.empty(wl.B, wl.H, nq, wl.dv, device=DEV)
    gma.gma_forward_cross(shape_of(wl, N=nq), _t(mu), _t(vr), _t(lp), _t(q, _tdt(wl.x_dtype)),
                          _t(k, _tdt(wl.x_dtype)), _t(v, _tdt(wl.v_dtype)), out)
    torch.cuda.synchronize()
    ref = oracle.cross(mu, vr, lp, q.reshape(S, nq, wl.d), k.reshape(S, nk, wl.d), v.reshape(S, nk, wl.dv),
                       wl.eps)
    o = out.reshape(S, nq, wl.dv).cpu().numpy()
    if nk == 0:
        assert np.array_equal(o, ref)   # an empty memory reads 0 / (0 + eps) = 0
        return
    err = normwise(o, ref)
    print(f"cross K={wl.K} nq={nq} nk={nk}: normwise error {err:.3e}")
    assert err <= TOL[wl.gemm_dtype]


def test_cross_equals_bidir_on_the_same_sequence():
    """With the same rows for queries and keys the cross form is the bidirectional form:
    the same kernels in the same order, so the results are identical."""
    for wl in (W["tiny"].with_(mode="bidir", B=2, H=2, N=1000, d=64, dv=64, K=128),
               W["tiny"].with_(mode="bidir", B=2, H=2, N=300)):
        mu, vr, lp = (_t(a) for a in workloads.params(wl))
        q, k, v = (_t(a) for a in workloads.full_inputs(wl))
        a = torch.empty(wl.B, wl.H, wl.N, wl.dv, device=DEV)
        b = torch.empty_like(a)
        gma.gma_forward_cross(shape_of(wl), mu, vr, lp, q, k, v, a)
        gma.gma_forward_bidir(shape_of(wl), mu, vr, lp, q, k, v, b)
        torch.cuda.synchronize()
        assert torch.equal(a, b)


# ------------------------------------------------------------- diagnostics ---

STATS = [
    W["tiny"],
    W["tiny"].with_(B=2, H=3, N=1000, K=40, d=32),
    W["tiny"].with_(B=2, H=2, N=777, K=1),
    W["tiny"].with_(B=2, H=2, N=3000, K=128, d=64),                 # bounded routing
    W["tiny"].with_(B=2, H=2, N=3000, K=128, d=64, dist="peaked"),
    W["tiny"].with_(B=1, H=2, N=600, K=512, d=128),
    W["causal_4k"],
    W["bidir_16k_peaked"].with_(B=1, H=4),
    W["causal_64k_bf16"].with_(H=2, N=8192),
]


@pytest.mark.parametrize("wl", STATS, ids=[f"{w.name}-B{w.B}-H{w.H}-N{w.N}-K{w.K}-{w.dist}" for w in STATS])
def test_responsibility_stats(wl):
    mu, vr, lp = workloads.params(wl)
    x = workloads.full_inputs(wl)[1]                     # the key routing rows
    S = wl.B * wl.H
    usage = torch.empty(wl.H, wl.K, device=DEV)
    counts = torch.empty(wl.H, wl.K, dtype=torch.int64, device=DEV)
    ent = torch.empty(wl.H, 2, device=DEV)
    assign = torch.empty(wl.B, wl.H, wl.N, dtype=torch.int32, device=DEV)
    gma.gma_responsibility_stats(shape_of(wl), _t(mu), _t(vr), _t(lp), _t(x, _tdt(wl.x_dtype)), usage, counts, ent,
                                 assign)
    torch.cuda.synchronize()
    heads = [s % wl.H for s in range(S)]
    xs = x.reshape(S, wl.N, -1)
    u, c, a, e = oracle.usage(mu, vr, lp, xs, heads=heads)
    g = oracle.responsibilities(mu, vr, lp, xs, heads=heads)
    top2 = np.sort(g, -1)[..., -2:] if wl.K > 1 else np.concatenate([np.zeros_like(g), g], -1)
    clear = (top2[..., 1] - top2[..., 0]) > 1e-5           # rows whose argmax fp32 rounding cannot flip
    ga = assign.reshape(S, wl.N).cpu().numpy()
    assert np.array_equal(ga[clear], a[clear])
    gc = counts.cpu().numpy()
    assert (gc.sum(1) == wl.B * wl.N).all()
    assert np.abs(gc - c).sum() <= 2 * int((~clear).sum())
    for h in range(wl.H):                                   # the counts are those of the returned assignments
        assert np.array_equal(gc[h], np.bincount(ga[[s for s in range(S) if heads[s] == h]].ravel(),
                                                 minlength=wl.K))
    err_u = normwise(usage.cpu().numpy(), u)
    err_e = float(np.abs(ent.cpu().numpy() - e).max())
    print(f"stats {wl.name} K={wl.K}: usage {err_u:.2e}, entropy {err_e:.2e}, ambiguous rows {(~clear).sum()}")
    assert err_u <= TOL["f32"] and err_e <= 1e-4


def test_responsibility_stats_repeatable():
    wl = W["causal_4k"].with_(B=2, H=2, N=5000)
    mu, vr, lp = (_t(a) for a in workloads.params(wl))
    x = _t(workloads.full_inputs(wl)[0])
    outs = []
    for _ in range(2):
        r = (torch.empty(wl.H, wl.K, device=DEV), torch.empty(wl.H, wl.K, dtype=torch.int64, device=DEV),
             torch.empty(wl.H, 2, device=DEV))
        gma.gma_responsibility_stats(shape_of(wl), mu, vr, lp, x, *r)
        outs.append(r)
    torch.cuda.synchronize()
    for a, b in zip(*outs):
        assert torch.equal(a, b)
