"""The seeded input generator (CPU): every slice can be drawn alone, draws are
repeatable, and the distributions are the stated ones."""
import numpy as np
import pytest
import torch

from gaussian_mixture_sequence_gb300 import workloads

W = workloads.WORKLOADS


def test_a_slice_drawn_alone_equals_the_full_draw():
    wl = W["tiny"].with_(B=2, H=3, N=50, dist="peaked")
    q, k, v = workloads.full_inputs(wl)
    mu = workloads.params(wl)[0]
    for b in range(wl.B):
        for h in range(wl.H):
            qs, ks, vs = workloads.slice_inputs(wl, b, h)
            np.testing.assert_array_equal(qs, q[b, h])
            np.testing.assert_array_equal(ks, k[b, h])
            np.testing.assert_array_equal(vs, v[b, h])
            np.testing.assert_array_equal(workloads.slice_inputs(wl, b, h, mu=mu)[0], q[b, h])


def test_draws_repeat_and_seeds_differ():
    wl = W["tiny"].with_(B=1, H=2, N=20)
    a, b = workloads.full_inputs(wl), workloads.full_inputs(wl)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)
    c = workloads.full_inputs(wl, seed=wl.seed + 1)
    assert not np.array_equal(a[0], c[0])
    p1, p2 = workloads.params(wl), workloads.params(wl)
    for x, y in zip(p1, p2):
        np.testing.assert_array_equal(x, y)
    # Q_X, K_X and V are independent draws
    assert not np.array_equal(a[0], a[1])
    # the tokens after a prefill are new draws
    d = workloads.full_inputs(wl.with_(decode_steps=20), decode=True)
    assert not np.array_equal(d[0], a[0])


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    a = np.concatenate([rng.standard_normal(4096).astype(np.float32) * 10.0 ** rng.integers(-5, 5, 4096),
                        np.array([0.0, -0.0, 1.0, -1.0, 1.00390625, 1.01171875, 3e38, -3e38], np.float32)])
    # halfway cases: a bf16 value plus half an ulp of bf16 (ties go to even)
    base = rng.standard_normal(512).astype(np.float32)
    half = (base.view(np.uint32) & np.uint32(0xFFFF0000)) | np.uint32(0x8000)
    a = np.concatenate([a, half.view(np.float32)])
    ref = torch.from_numpy(a).to(torch.bfloat16).to(torch.float32).numpy()
    np.testing.assert_array_equal(workloads.round_bf16(a), ref)


def test_distributions():
    wl = W["tiny"].with_(B=1, H=2, N=4000, d=16, K=8)
    mu, var_raw, logit_pi = workloads.params(wl)
    assert mu.std() == pytest.approx(1.0, rel=0.1)
    assert var_raw.std() == pytest.approx(0.5, rel=0.1)          # r ~ N(0, 0.5^2)
    assert logit_pi.std() == pytest.approx(1.0, rel=0.3)
    q, k, v = workloads.full_inputs(wl)
    assert q.std() == pytest.approx(1.0, rel=0.05) and v.std() == pytest.approx(1.0, rel=0.05)
    # peaked: x = mu_c + 0.3 z, so the nearest centre is at squared distance about 0.09 d
    pk = wl.with_(dist="peaked")
    qp = workloads.full_inputs(pk)[0][0, 1]
    d2 = ((qp[:, None, :] - mu[1][None]) ** 2).sum(-1).min(1)
    assert d2.mean() == pytest.approx(0.09 * wl.d, rel=0.1)
    # every centre is used
    assert len(np.unique(((qp[:, None, :] - mu[1][None]) ** 2).sum(-1).argmin(1))) == wl.K


def test_bf16_inputs_are_representable():
    wl = W["tiny"].with_(x_dtype="bf16", v_dtype="bf16")
    for a in workloads.full_inputs(wl):
        np.testing.assert_array_equal(a, workloads.round_bf16(a))


def test_sample_slices():
    wl = W["causal_16k_peaked"]
    s = workloads.sample_slices(wl, 3)
    assert s == sorted(set(s)) and len(s) == 3 and s[-1] == wl.B * wl.H - 1
    assert workloads.sample_slices(wl, 3) == s                       # fixed
    assert workloads.sample_slices(wl, 100) == list(range(wl.B * wl.H))
