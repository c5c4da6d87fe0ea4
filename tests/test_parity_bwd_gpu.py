"""GPU parity of the gradients (end-to-end training of the GMM parameters
through the softplus and softmax reparameterisations, as the GMA explainer's
"변형 및 학습" describes): gma_backward through the C ABI against the fp64
oracle's chain rule on the same seeded inputs and the same dL/dO.

Tolerance: normwise per (batch, head) slice for dQ_X, dK_X and dV, and per
head for the parameter gradients, 1e-4: the gradient pass computes in fp32
throughout.  The denominator is max|g_ref|, floored at 1e-2 times the largest
|dV| of the case: dV = Gamma_K^T Gamma_Q dL/dO / den is always of the order of
dL/dO, while the routing gradients vanish when the posteriors saturate (peaked
inputs: every row one-hot to within e^-30, routing gradients ~1e-12 in fp64,
below what fp32 resolves; the kernels drop posteriors below e^-30 exactly)."""
import numpy as np
import pytest
import torch

import oracle
from gaussian_mixture_sequence_gb300 import gma, workloads
from gpu_cases import DEV, normwise, shape_of

pytestmark = pytest.mark.gpu
W = workloads.WORKLOADS
TOL = 1e-4


def _t(a, dtype=torch.float32):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV).to(dtype)


def _run(wl, causal):
    mu, vr, lp = workloads.params(wl)
    q, k, v = workloads.full_inputs(wl)
    S = wl.B * wl.H
    g = np.random.default_rng(wl.seed + 5).standard_normal((wl.B, wl.H, wl.N, wl.dv)).astype(np.float32)
    xdt = torch.bfloat16 if wl.x_dtype == "bf16" else torch.float32
    vdt = torch.bfloat16 if wl.v_dtype == "bf16" else torch.float32
    outs = (torch.empty(wl.B, wl.H, wl.N, wl.d, device=DEV), torch.empty(wl.B, wl.H, wl.N, wl.d, device=DEV),
            torch.empty(wl.B, wl.H, wl.N, wl.dv, device=DEV), torch.empty(wl.H, wl.K, wl.d, device=DEV),
            torch.empty(wl.H, wl.K, wl.d, device=DEV), torch.empty(wl.H, wl.K, device=DEV))
    gma.gma_backward(shape_of(wl), _t(mu), _t(vr), _t(lp), _t(q, xdt), _t(k, xdt), _t(v, vdt), _t(g), *outs,
                     causal=causal)
    torch.cuda.synchronize()
    ref = oracle.backward(mu, vr, lp, q.reshape(S, wl.N, wl.d), k.reshape(S, wl.N, wl.d),
                          v.reshape(S, wl.N, wl.dv), wl.eps, g.reshape(S, wl.N, wl.dv), causal=causal,
                          heads=[s % wl.H for s in range(S)])
    return [o.cpu().numpy() for o in outs], ref


CASES = [
    (W["tiny"], True),
    (W["tiny"], False),
    (W["tiny"].with_(B=2, H=3, N=1000, d=32, dv=128, K=40), True),
    (W["tiny"].with_(B=2, H=3, N=1000, d=32, dv=128, K=40), False),
    (W["tiny"].with_(B=2, H=2, N=777, d=64, dv=64, K=128), True),      # bounded routing in the recompute
    (W["tiny"].with_(B=1, H=2, N=300, d=64, dv=32, K=128, dist="peaked"), True),
    (W["tiny"].with_(B=1, H=2, N=513, d=64, dv=64, K=128, x_dtype="bf16", v_dtype="bf16"), True),
    # one row: with eps = 1e-6 the output is v den / (den + eps) and its routing gradient an O(eps)
    # difference of O(1) terms; a larger eps keeps the single-row case well conditioned
    (W["tiny"].with_(B=2, H=2, N=1, K=16, eps=0.1), True),
    (W["tiny"].with_(B=1, H=1, N=300, d=128, dv=16, K=512), False),
    # d = 128 in the causal form, K = 100 (a ragged last tile of 32 components), ragged row blocks
    (W["tiny"].with_(B=1, H=2, N=650, d=128, dv=64, K=100), True),
    (W["causal_4k"], True),
]


@pytest.mark.parametrize("wl,causal", CASES,
                         ids=[f"{w.name}-B{w.B}H{w.H}N{w.N}K{w.K}d{w.d}dv{w.dv}-{'c' if c else 'b'}-{w.x_dtype}"
                              for w, c in CASES])
def test_backward(wl, causal):
    got, ref = _run(wl, causal)
    S = wl.B * wl.H
    names = ("dqx", "dkx", "dv", "dmu", "dvar_raw", "dlogit_pi")
    floor = 1e-2 * np.abs(ref[2]).max()
    for name, a, b in zip(names, got, ref):
        n = S if name in ("dqx", "dkx", "dv") else wl.H
        a, b = np.asarray(a, np.float64).reshape(n, -1), b.reshape(n, -1)
        err = float((np.abs(a - b).max(1) / np.maximum(np.abs(b).max(1), floor)).max())
        print(f"backward {wl.name} K={wl.K} {'causal' if causal else 'bidir'} {name}: normwise error {err:.3e} "
              f"(max |ref| {np.abs(b).max():.2e})")
        assert err <= TOL, f"{name}: {err:.3e}"


def test_backward_repeatable_and_causal_structure():
    """Repeated calls give identical bits; in the causal form dL/dO of the last rows
    does not reach the query gradients of earlier rows."""
    wl = W["tiny"].with_(B=1, H=2, N=700, d=64, dv=64, K=128)
    mu, vr, lp = (_t(a) for a in workloads.params(wl))
    q, k, v = (_t(a) for a in workloads.full_inputs(wl))
    g = torch.randn(wl.B, wl.H, wl.N, wl.dv, device=DEV, generator=torch.Generator(device=DEV).manual_seed(3))

    def run(gg):
        outs = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v), torch.empty_like(mu),
                torch.empty_like(vr), torch.empty_like(lp))
        gma.gma_backward(shape_of(wl), mu, vr, lp, q, k, v, gg, *outs)
        return outs

    a, b = run(g), run(g)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    g2 = g.clone()
    g2[:, :, 500:] += 1.0
    c = run(g2)
    assert torch.equal(c[0][:, :, :500], a[0][:, :, :500])
