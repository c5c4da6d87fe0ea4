"""The arithmetic of the tensor-core routings (d = 64), emulated on the CPU: the dense pass
of K = 128 and the full routing of the other K up to 512.

For the tiles the bounded routing leaves to the dense pass, every log-joint is
evaluated in the expanded form
  l~_k = [x^2 | x] . [-a_k / 2 | a_k mu_k] + c'_k
with both operands held as three bf16 planes (v = v0 + v1 + v2, each plane the
round-to-nearest of what the previous ones leave) and the six plane products
A2 W0, A1 W1, A1 W0, A0 W2, A0 W1, A0 W0 accumulated in fp32 in that order, one
16-wide K step at a time (the tensor core's accumulation), each product's values'
(odd) K steps before its squares' (even) ones as the kernels issue them; the
routing of 65 <= K <= 512 takes the products in the order its planes of W are at
hand, A1 W1, A0 W1, A2 W0, A1 W0, A0 W2, and A0 W0 last.  A tile whose rows
include one with S = A/2 sum x^2 + M sum |x| above 4096 (A = max a, M = max |a mu|
over the head) is evaluated exactly instead.  This checks that on the rows the
pass keeps the posteriors match the oracle's far inside the 1e-4 tolerance and
no worse than an fp32 evaluation of the direct form (x - mu)^2 / sigma^2 summed
feature by feature, that the error tracks S as the design states, and that fewer
planes or products do not suffice.  None of this code is used by the library.
"""
import numpy as np
import pytest
import torch

import oracle
from gaussian_mixture_sequence_gb300 import workloads

S_MAX = 4096.0
ALL_PASSES = [(2, 0), (1, 1), (1, 0), (0, 2), (0, 1), (0, 0)]
WIDE_PASSES = [(1, 1), (0, 1), (2, 0), (1, 0), (0, 2), (0, 0)]   # 65 <= K <= 512
KERNEL_KSTEPS = [1, 3, 5, 7, 0, 2, 4, 6]                          # the values' steps first


def _bf(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16).to(torch.float32).numpy()


def _planes(v, n=3):
    out, r = [], v.astype(np.float32)
    for _ in range(n):
        p = _bf(r)
        out.append(p)
        r = (r - p).astype(np.float32)
    return out


def _head(seed=0, K=128):
    wl = workloads.WORKLOADS["tiny"].with_(B=1, H=1, N=1024, d=64, dv=64, K=K)
    mu, vr, lp = (p[0] for p in workloads.params(wl, seed=wl.seed + seed))
    return wl, mu, vr, lp


def _emulate(mu, var_raw, logit_pi, x, passes=ALL_PASSES, nplanes=3, ksteps=KERNEL_KSTEPS):
    """(estimated log-joints [n, K] as the pass forms them, S [n]) for one head."""
    v32 = np.logaddexp(np.float32(0), var_raw.astype(np.float32)).astype(np.float32)
    s = (1.0 / np.sqrt(v32)).astype(np.float32)
    ms = (-mu.astype(np.float32) * s).astype(np.float32)
    lse = np.float32(np.logaddexp.reduce(logit_pi.astype(np.float32)))
    c = (logit_pi.astype(np.float32) - lse) - np.float32(0.5) * np.log(v32).sum(1, dtype=np.float32)
    cp = (c - np.float32(0.5) * (ms * ms).sum(1, dtype=np.float32)).astype(np.float32)
    w = np.concatenate([(-0.5 * s * s).astype(np.float32), (-s * ms).astype(np.float32)], 1)
    x = x.astype(np.float32)
    a = np.concatenate([(x * x).astype(np.float32), x], 1)
    ap, wp = _planes(a, nplanes), _planes(w, nplanes)
    acc = np.zeros((x.shape[0], w.shape[0]), np.float32)
    for i, j in passes:
        if i >= nplanes or j >= nplanes:
            continue
        for kk in ksteps:   # one MMA K step of 16 operand positions: exact products, one fp32 rounding
            cols = _kstep_columns(kk)
            step = ap[i][:, cols].astype(np.float64) @ wp[j][:, cols].T.astype(np.float64)
            acc = (acc + step).astype(np.float32)
    est = (acc + cp[None]).astype(np.float32)
    big_s = 0.5 * (s * s).max() * (x * x).sum(1) + np.abs(s * ms).max() * np.abs(x).sum(1)
    return est, big_s


def _kstep_columns(kk):
    """The 16 columns of [x^2 | x] in operand positions 16 kk .. 16 kk + 15: quarter q of
    the operand holds the squares of features 16 q .. 16 q + 15 (even steps), then their
    values (odd steps)."""
    q, val = kk // 2, kk % 2
    return np.arange(16 * q, 16 * q + 16) + (64 if val else 0)


def _exact_logits(mu, var_raw, logit_pi, x):
    v = np.logaddexp(0.0, var_raw.astype(np.float64))
    lpi = logit_pi.astype(np.float64) - np.logaddexp.reduce(logit_pi.astype(np.float64))
    dx = x.astype(np.float64)[:, None, :] - mu.astype(np.float64)[None]
    return lpi[None] - 0.5 * np.log(v).sum(1)[None] - 0.5 * (dx * dx / v[None]).sum(-1)


def _direct_fp32(mu, var_raw, logit_pi, x):
    """The direct form in fp32: y = x s - mu s, the squares summed feature by feature."""
    v32 = np.logaddexp(np.float32(0), var_raw.astype(np.float32)).astype(np.float32)
    s = (1.0 / np.sqrt(v32)).astype(np.float32)
    ms = (-mu.astype(np.float32) * s).astype(np.float32)
    y = (x.astype(np.float32)[:, None, :] * s[None] + ms[None]).astype(np.float32)
    acc = np.zeros(y.shape[:2], np.float32)
    for d in range(y.shape[2]):
        acc = (acc + y[:, :, d] * y[:, :, d]).astype(np.float32)
    lse = np.float32(np.logaddexp.reduce(logit_pi.astype(np.float32)))
    c = (logit_pi.astype(np.float32) - lse) - np.float32(0.5) * np.log(v32).sum(1, dtype=np.float32)
    return (c[None] - np.float32(0.5) * acc).astype(np.float32)


def _softmax(l):
    e = np.exp(l - l.max(1, keepdims=True))
    return e / e.sum(1, keepdims=True)


def _rows(case, n=512, seed=2, K=128):
    wl, mu, vr, lp = _head(K=K)
    rng = np.random.default_rng(seed)
    if case == "peaked":
        x = workloads.full_inputs(wl.with_(dist="peaked"))[0][0, 0][:n]
    else:
        scale = {"normal": 1.0, "narrow": 0.3, "wide 1.8": 1.8, "wide 2.0": 2.0}[case]
        x = (scale * rng.standard_normal((n, 64))).astype(np.float32)
    return mu, vr, lp, x


@pytest.mark.parametrize("case", ["normal", "narrow", "peaked", "wide 1.8", "wide 2.0"])
def test_dense_pass_matches_the_oracle_on_the_rows_it_keeps(case):
    mu, vr, lp, x = _rows(case)
    est, big_s = _emulate(mu, vr, lp, x)
    keep = big_s <= S_MAX
    assert keep.any()
    ref = oracle.responsibilities(mu[None], vr[None], lp[None], x[None])[0]
    err = np.abs(_softmax(est.astype(np.float64)) - ref)[keep].max()
    direct = np.abs(_softmax(_direct_fp32(mu, vr, lp, x).astype(np.float64)) - ref)[keep].max()
    assert err <= 2e-5, err                 # five times inside the 1e-4 tolerance
    assert err <= max(direct, 1e-6), (err, direct)


def test_error_tracks_the_magnitude_bound():
    """|l~ - l| stays below 2^-18 S on every row (S bounds the terms' magnitudes; the
    emulated error is a few fp32 units of it), over rows from S ~ 100 to S ~ 10^4."""
    mu, vr, lp, _ = _rows("normal")
    rng = np.random.default_rng(5)
    x = np.concatenate([(s * rng.standard_normal((64, 64))).astype(np.float32)
                        for s in (0.3, 0.7, 1.0, 1.5, 2.0, 3.0, 5.0)])
    est, big_s = _emulate(mu, vr, lp, x)
    err = np.abs(est - _exact_logits(mu, vr, lp, x)).max(1)
    assert big_s.min() < 300 and big_s.max() > 1e4
    assert np.all(err <= big_s * 2.0 ** -18), (err / big_s).max()


def test_rows_beyond_the_limit_are_the_far_ones():
    """N(0, 1) rows sit well under the limit (the tiles they fill take the tensor-core
    pass); rows three times wider are above it (their tiles go to the exact pass)."""
    mu, vr, lp, x = _rows("normal")
    _, s1 = _emulate(mu, vr, lp, x)
    _, s3 = _emulate(mu, vr, lp, 3.0 * x)
    assert s1.max() < 0.5 * S_MAX and np.median(s3) > S_MAX


@pytest.mark.parametrize("passes,nplanes", [
    (ALL_PASSES, 2),                            # two planes per operand (16 bits)
    ([(1, 0), (0, 1), (0, 0)], 3),              # the first-order products only
    ([(2, 0), (1, 1), (1, 0), (0, 1), (0, 0)], 3),   # A0 W2 dropped
    ([(2, 0), (1, 1), (0, 2), (0, 1), (0, 0)], 3),   # A1 W0 dropped
])
def test_fewer_planes_or_products_do_not_suffice(passes, nplanes):
    """Each plane and each of the six products is needed for the 1e-5 margin on N(0, 1)
    rows: with any one removed the emulated posteriors miss it."""
    mu, vr, lp, x = _rows("normal")
    est, _ = _emulate(mu, vr, lp, x, passes=passes, nplanes=nplanes)
    ref = oracle.responsibilities(mu[None], vr[None], lp[None], x[None])[0]
    assert np.abs(_softmax(est.astype(np.float64)) - ref).max() > 1e-5


@pytest.mark.parametrize("K,passes", [(32, ALL_PASSES), (64, ALL_PASSES), (100, WIDE_PASSES),
                                      (256, WIDE_PASSES), (512, WIDE_PASSES)])
@pytest.mark.parametrize("case", ["normal", "wide 2.0"])
def test_tensor_core_routing_orders_match_the_oracle(K, passes, case):
    """The full tensor-core routing of K != 128 (every component of every row, in the
    product order of its kernel) matches the oracle on the rows it keeps, as closely as
    an fp32 evaluation of the direct form."""
    mu, vr, lp, x = _rows(case, n=256, K=K)
    est, big_s = _emulate(mu, vr, lp, x, passes=passes)
    keep = big_s <= S_MAX
    assert keep.any()
    ref = oracle.responsibilities(mu[None], vr[None], lp[None], x[None])[0]
    err = np.abs(_softmax(est.astype(np.float64)) - ref)[keep].max()
    direct = np.abs(_softmax(_direct_fp32(mu, vr, lp, x).astype(np.float64)) - ref)[keep].max()
    assert err <= 2e-5, err
    assert err <= max(2 * direct, 1e-6), (err, direct)


def test_kstep_order_changes_only_the_rounding():
    """The odd-steps-first order of the kernels and the plain ascending order give
    log-joints within a few fp32 units of S of each other."""
    mu, vr, lp, x = _rows("normal")
    a, big_s = _emulate(mu, vr, lp, x)
    b, _ = _emulate(mu, vr, lp, x, ksteps=list(range(8)))
    assert np.all(np.abs(a - b).max(1) <= big_s * 2.0 ** -20)
    assert np.abs(a - b).max() > 0   # the orders do round differently
