"""The error bound behind the bounded routing (K = 128, d = 64), checked on the CPU.

The routing kernel estimates every log-joint with one bf16 product per row,
  l~_k = [x^2 | x] . [-a_k / 2 | a_k mu_k] + c'_k,   c'_k = c_k - 1/2 sum_d a_kd mu_kd^2,
(a = 1/sigma^2; operands rounded to bf16, fp32 accumulation, c' in fp32), and
keeps component k exactly iff l~_k >= max_j l~_j - T - 2 delta with T = 30 and
  delta = 4e-3 (A/2 sum_d x_d^2 + M sqrt(d) sqrt(sum_d x_d^2)) + 1e-3,
A = max a, M = max |a mu| over the head.  This emulates that arithmetic and
measures |l~_k - l_k| against the fp64 log-joint l_k.
"""
import numpy as np
import pytest
import torch

from gaussian_mixture_sequence_gb300 import workloads

T = 30.0


def _bf(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16).to(torch.float32).numpy()


def _estimates(mu, var_raw, logit_pi, x):
    """(l~ [n,K] as the kernel forms it, delta [n], fp64 log-joints [n,K], c' [K]).
    The 2 pi term cancels in the posterior and is left out on both sides."""
    v64 = np.logaddexp(0.0, var_raw.astype(np.float64))
    lpi = logit_pi.astype(np.float64) - np.logaddexp.reduce(logit_pi.astype(np.float64))
    dx = x.astype(np.float64)[:, None, :] - mu.astype(np.float64)[None]
    exact = lpi[None] - 0.5 * np.log(v64).sum(1)[None] - 0.5 * (dx * dx / v64[None]).sum(-1)
    v32 = np.logaddexp(np.float32(0), var_raw.astype(np.float32)).astype(np.float32)
    s = (1.0 / np.sqrt(v32)).astype(np.float32)
    ms = (-mu.astype(np.float32) * s).astype(np.float32)
    lse = np.float32(np.logaddexp.reduce(logit_pi.astype(np.float32)))
    c = (logit_pi.astype(np.float32) - lse) - np.float32(0.5) * np.log(v32).sum(1, dtype=np.float32)
    cp = (c - np.float32(0.5) * (ms * ms).sum(1, dtype=np.float32)).astype(np.float32)
    w = np.concatenate([_bf(-0.5 * s * s), _bf(-s * ms)], 1)
    a = np.concatenate([_bf(x * x), _bf(x)], 1)
    s2 = (x.astype(np.float32) ** 2).sum(1)
    delta = 4e-3 * (0.5 * (s * s).max() * s2 + np.abs(s * ms).max() * np.sqrt(mu.shape[1]) * np.sqrt(s2)) + 1e-3
    return a @ w.T + cp[None], delta, exact, cp


def _estimate_error(mu, var_raw, logit_pi, x):
    """(max over rows and components of |l~ - l| / delta, max |l~ - l|, max |c'|)."""
    est, delta, exact, cp = _estimates(mu, var_raw, logit_pi, x)
    err = np.abs(est - exact)
    return (err / delta[:, None]).max(), err.max(), np.abs(cp).max()


def _head(seed=0):
    wl = workloads.WORKLOADS["tiny"].with_(B=1, H=1, N=1500, d=64, dv=64, K=128)
    mu, vr, lp = (p[0] for p in workloads.params(wl, seed=wl.seed + seed))
    return wl, mu, vr, lp


@pytest.mark.parametrize("case", ["normal", "peaked", "far rows", "small variances at the means",
                                  "large variances"])
def test_estimates_stay_inside_the_bound(case):
    wl, mu, vr, lp = _head()
    rng = np.random.default_rng(1)
    x = workloads.full_inputs(wl.with_(dist="peaked" if case == "peaked" else "normal"))[0][0, 0]
    if case == "far rows":
        x = 30.0 * x
    if case == "small variances at the means":     # sigma^2 ~ 0.0025, rows within 0.05 of a centre
        mu, vr = 3.0 * mu, np.full_like(vr, -6.0)
        x = (mu[rng.integers(0, 128, 600)] + 0.05 * rng.standard_normal((600, 64))).astype(np.float32)
    if case == "large variances":
        vr = np.full_like(vr, 8.0)
    ratio, _, _ = _estimate_error(mu, vr, lp, x.astype(np.float32))
    assert ratio <= 0.5, ratio


def test_constant_rounding_beyond_the_bound_stays_far_inside_the_margin():
    """A routing row at the origin with tiny variances and far means: the estimate is
    the fp32 constant c' alone (|c'| ~ 1e5), whose rounding exceeds delta = 1e-3, yet
    stays below 1e-6 |c'| and far inside the T = 30 keep margin, so every dropped
    component still has posterior below e^-29."""
    _, mu, vr, lp = _head()
    mu, vr = 3.0 * mu, np.full_like(vr, -6.0)
    ratio, err, cmax = _estimate_error(mu, vr, lp, np.zeros((4, 64), np.float32))
    assert cmax > 1e4 and ratio > 1.0            # the regime the 1e-3 does not cover
    assert err <= 1e-6 * cmax and err < 1.0 < T


@pytest.mark.parametrize("dist", ["normal", "peaked"])
def test_kept_set_posterior_equals_the_dense_one(dist):
    """The softmax over the kept set {k : l~_k >= max l~ - T - 2 delta} (a row whose
    second-best estimate falls below that threshold keeps its argmax alone, with
    posterior 1) differs from the dense posterior by at most the dropped mass,
    K e^-30 ~ 1.2e-11 of the row."""
    wl, mu, vr, lp = _head()
    x = workloads.full_inputs(wl.with_(dist=dist))[0][0, 0]
    est, delta, exact, _ = _estimates(mu, vr, lp, x)
    keep = est >= est.max(1, keepdims=True) - T - 2.0 * delta[:, None]
    dense = np.exp(exact - exact.max(1, keepdims=True))
    dense /= dense.sum(1, keepdims=True)
    kept = np.where(keep, np.exp(exact - exact.max(1, keepdims=True)), 0.0)
    kept /= kept.sum(1, keepdims=True)
    assert np.abs(kept - dense).max() <= 128 * np.exp(-30.0)
    single = keep.sum(1) == 1
    if dist == "peaked":
        assert single.mean() > 0.9           # most peaked rows take the single-component shortcut
    assert np.all(kept[single].max(1) == 1.0)
