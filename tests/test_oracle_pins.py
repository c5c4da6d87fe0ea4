"""Pins of the fp64 oracle to things other than itself (CPU only).

Each test checks the oracle against what the GMA explainer page ("Gaussian
Mixture Attention: Linear-Time Sequence Mixing via Probabilistic Latent
Routing", technical summary, "핵심 메커니즘" and "변형 및 학습") or mathematics
fixes: a library GMM posterior (scikit-learn), the two-component logistic
closed form, brute-force N x N affinity, rank(Gamma_Q Gamma_K^T) <= K, the
causal prefix property, K = 1 means, equal-component identities and sequence
splitting.  None of them retypes the oracle's own code.
"""
import math

import numpy as np
import pytest
from scipy.special import softmax

from gaussian_mixture_sequence_gb300 import workloads as wlmod

TINY = wlmod.WORKLOADS["tiny"]


def _tiny(seed=None, K=None, N=None, d=None, dv=None):
    wl = TINY.with_(**{k: v for k, v in dict(K=K, N=N, d=d, dv=dv).items() if v is not None})
    mu, vr, lp = wlmod.params(wl, seed)
    qx, kx, v = wlmod.slice_inputs(wl, 0, 0, seed, mu)
    return wl, mu, vr, lp, qx[None], kx[None], v[None]


def _sklearn_posterior(mu, var_raw, logit_pi, x):
    """GMM posterior from scikit-learn's GaussianMixture (diagonal covariances).

    The parameters are reparameterised with library routines (numpy logaddexp
    for softplus, scipy softmax for the priors)."""
    sk = pytest.importorskip("sklearn.mixture")
    K, d = mu.shape
    g = sk.GaussianMixture(n_components=K, covariance_type="diag")
    cov = np.logaddexp(0.0, var_raw.astype(np.float64))
    g.weights_ = softmax(logit_pi.astype(np.float64))
    g.means_ = mu.astype(np.float64)
    g.covariances_ = cov
    g.precisions_cholesky_ = 1.0 / np.sqrt(cov)
    g.precisions_ = 1.0 / cov
    return g.predict_proba(x.astype(np.float64))


# ---------------------------------------------------------------- S0 -------

def test_s0_softplus_closed_forms(orc):
    r = np.array([0.0, math.log(math.e - 1.0), 50.0, -50.0, 1e-3, -1e-3])
    var, _ = orc.params(r.reshape(1, 1, -1), np.zeros((1, 1)))
    var = var.ravel()
    assert var[0] == pytest.approx(math.log(2.0), rel=1e-15)
    assert var[1] == pytest.approx(1.0, rel=1e-15)
    assert var[2] == pytest.approx(50.0 + math.exp(-50.0), rel=1e-15)
    assert var[3] == pytest.approx(math.exp(-50.0), rel=1e-14)
    # softplus(r) - softplus(-r) = r
    rr = np.random.default_rng(0).normal(0, 3, size=64)
    a, _ = orc.params(rr.reshape(1, 1, -1), np.zeros((1, 1)))
    b, _ = orc.params(-rr.reshape(1, 1, -1), np.zeros((1, 1)))
    np.testing.assert_allclose((a - b).ravel(), rr, rtol=0, atol=1e-13)


def test_s0_log_priors(orc):
    rng = np.random.default_rng(1)
    l = rng.normal(0, 2, size=(3, 11))
    _, log_pi = orc.params(np.zeros((3, 11, 2)), l)
    np.testing.assert_allclose(np.exp(log_pi).sum(1), 1.0, rtol=0, atol=1e-14)
    np.testing.assert_allclose(log_pi - log_pi[:, :1], l - l[:, :1], rtol=0, atol=1e-13)
    _, u = orc.params(np.zeros((1, 5, 1)), np.full((1, 5), 3.7))
    np.testing.assert_allclose(u, -math.log(5.0), rtol=1e-15)


# ---------------------------------------------------------------- S1 -------

@pytest.mark.parametrize("K,d,dist", [(8, 16, "normal"), (128, 64, "normal"), (32, 64, "peaked"),
                                      (3, 5, "normal")])
def test_s1_matches_library_gmm_posterior(orc, K, d, dist):
    wl = TINY.with_(K=K, d=d, N=300, dist=dist)
    mu, vr, lp = wlmod.params(wl)
    x = wlmod.slice_inputs(wl, 0, 0, mu=mu)[0]
    g = orc.responsibilities(mu, vr, lp, x[None])[0]
    ref = _sklearn_posterior(mu[0], vr[0], lp[0], x)
    np.testing.assert_allclose(g, ref, rtol=0, atol=1e-10)


def test_s1_two_component_logistic(orc):
    """d = 1, K = 2, equal variances: the posterior is the logistic function of a
    linear discriminant (the textbook Gaussian discriminant closed form)."""
    rng = np.random.default_rng(2)
    mu = np.array([[[0.7], [-1.3]]])
    r = 0.4
    var = math.log1p(math.exp(r))
    l = np.array([[0.25, -0.6]])
    x = rng.normal(0, 2, size=(1, 50, 1))
    g = orc.responsibilities(mu, np.full((1, 2, 1), r), l, x)[0]
    m1, m2 = 0.7, -1.3
    a = (m1 - m2) * x[0, :, 0] / var - (m1 * m1 - m2 * m2) / (2 * var) + (0.25 - (-0.6))
    expect = 1.0 / (1.0 + np.exp(-a))
    np.testing.assert_allclose(g[:, 0], expect, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(g[:, 1], 1.0 - expect, rtol=1e-12, atol=1e-15)


def test_s1_equal_components_give_priors(orc):
    rng = np.random.default_rng(3)
    K, d = 6, 4
    mu = np.tile(rng.normal(size=(1, 1, d)), (1, K, 1))
    vr = np.tile(rng.normal(size=(1, 1, d)), (1, K, 1))
    l = rng.normal(size=(1, K))
    g = orc.responsibilities(mu, vr, l, rng.normal(size=(1, 40, d)))[0]
    np.testing.assert_allclose(g, np.tile(softmax(l[0]), (40, 1)), rtol=1e-13)


def test_s1_component_permutation(orc):
    wl, mu, vr, lp, qx, _, _ = _tiny()
    perm = np.random.default_rng(4).permutation(wl.K)
    g = orc.responsibilities(mu, vr, lp, qx)[0]
    gp = orc.responsibilities(mu[:, perm], vr[:, perm], lp[:, perm], qx)[0]
    np.testing.assert_allclose(gp, g[:, perm], rtol=0, atol=1e-13)


def test_s1_rows_are_distributions_even_far_away(orc):
    wl, mu, vr, lp, qx, _, _ = _tiny()
    x = np.concatenate([qx[0], np.full((2, wl.d), 1e3), np.full((2, wl.d), -1e3)])
    g = orc.responsibilities(mu, vr, lp, x[None])[0]
    assert np.isfinite(g).all() and (g >= 0).all()
    np.testing.assert_allclose(g.sum(1), 1.0, rtol=0, atol=1e-12)
    # a token sitting on a component with a tiny variance belongs to it
    mu2, vr2 = mu.copy(), vr.copy()
    vr2[0, 3] = -30.0
    g2 = orc.responsibilities(mu2, vr2, lp, mu2[:, 3:4].astype(np.float64))[0]
    assert g2[0, 3] > 1 - 1e-12


# ------------------------------------------------------------- S2 + S3 -----

def _bruteforce(gq, gk, v, eps, causal):
    A = gq @ gk.T                        # the N x N affinity Gamma_Q Gamma_K^T
    if causal:
        A = np.tril(A)                   # j <= i
    return (A @ v) / (A.sum(1, keepdims=True) + eps)


@pytest.mark.parametrize("eps", [1e-6, 0.37])
@pytest.mark.parametrize("causal", [False, True])
def test_s2_s4_match_bruteforce_affinity(orc, eps, causal):
    """The latent-memory form equals materialising the N x N affinity, with
    responsibilities from the library GMM posterior."""
    wl, mu, vr, lp, qx, kx, v = _tiny()
    gq = _sklearn_posterior(mu[0], vr[0], lp[0], qx[0])
    gk = _sklearn_posterior(mu[0], vr[0], lp[0], kx[0])
    ref = _bruteforce(gq, gk, v[0].astype(np.float64), eps, causal)
    fn = orc.causal if causal else orc.bidir
    out = fn(mu, vr, lp, qx, kx, v, eps)[0]
    np.testing.assert_allclose(out, ref, rtol=1e-9, atol=1e-12)


def test_affinity_rank_at_most_K(orc):
    wl, mu, vr, lp, qx, kx, _ = _tiny()
    gq = orc.responsibilities(mu, vr, lp, qx)[0]
    gk = orc.responsibilities(mu, vr, lp, kx)[0]
    s = np.linalg.svd(gq @ gk.T, compute_uv=False)
    assert wl.N > wl.K
    assert s[wl.K:].max() < 1e-12 * s[0]
    assert s[wl.K - 1] > 1e-12 * s[0]


def test_bidir_K1_is_the_mean(orc):
    wl, mu, vr, lp, qx, kx, v = _tiny(K=1)
    eps = 0.25
    out = orc.bidir(mu, vr, lp, qx, kx, v, eps)[0]
    expect = v[0].astype(np.float64).sum(0) / (wl.N + eps)
    np.testing.assert_allclose(out, np.tile(expect, (wl.N, 1)), rtol=1e-12, atol=1e-15)


def test_bidir_equal_components_give_scaled_mean(orc):
    rng = np.random.default_rng(5)
    K, d, dv, N = 5, 3, 4, 64
    mu = np.tile(rng.normal(size=(1, 1, d)), (1, K, 1))
    vr = np.tile(rng.normal(size=(1, 1, d)), (1, K, 1))
    l = rng.normal(size=(1, K))
    v = rng.normal(size=(1, N, dv))
    eps = 0.1
    out = orc.bidir(mu, vr, l, rng.normal(size=(1, N, d)), rng.normal(size=(1, N, d)), v, eps)[0]
    pp = float((softmax(l[0]) ** 2).sum())
    expect = v[0].sum(0) * pp / (N * pp + eps)
    np.testing.assert_allclose(out, np.tile(expect, (N, 1)), rtol=1e-12)


def test_bidir_convexity_permutation_linearity(orc):
    wl, mu, vr, lp, qx, kx, v = _tiny()
    out = orc.bidir(mu, vr, lp, qx, kx, v, 1e-6)[0]
    assert (np.abs(out) <= np.abs(v[0]).max(0) + 1e-12).all()
    perm = np.random.default_rng(6).permutation(wl.N)
    outp = orc.bidir(mu, vr, lp, qx, kx[:, perm], v[:, perm], 1e-6)[0]
    np.testing.assert_allclose(outp, out, rtol=1e-11, atol=1e-14)
    v2 = np.random.default_rng(7).normal(size=v.shape)
    o2 = orc.bidir(mu, vr, lp, qx, kx, v2, 1e-6)[0]
    o12 = orc.bidir(mu, vr, lp, qx, kx, 2.0 * v - 3.0 * v2, 1e-6)[0]
    np.testing.assert_allclose(o12, 2.0 * out - 3.0 * o2, rtol=1e-10, atol=1e-12)
    ones = orc.bidir(mu, vr, lp, qx, kx, np.ones_like(v), 1e-6)[0]
    assert (ones < 1).all() and (ones > 1 - 1e-4).all()


# ---------------------------------------------------------------- S4 -------

def test_s4_causal_prefix_property(orc):
    """O_i depends on tokens j <= i only: perturbing later tokens leaves it bit-identical."""
    wl, mu, vr, lp, qx, kx, v = _tiny()
    out = orc.causal(mu, vr, lp, qx, kx, v, 1e-6)[0]
    rng = np.random.default_rng(8)
    for i in (0, 1, 63, 64, 200, wl.N - 2):
        q2, k2, v2 = qx.copy(), kx.copy(), v.copy()
        q2[0, i + 1:] += rng.normal(size=q2[0, i + 1:].shape).astype(np.float32)
        k2[0, i + 1:] += rng.normal(size=k2[0, i + 1:].shape).astype(np.float32)
        v2[0, i + 1:] += rng.normal(size=v2[0, i + 1:].shape).astype(np.float32)
        o2 = orc.causal(mu, vr, lp, q2, k2, v2, 1e-6)[0]
        assert np.array_equal(o2[: i + 1], out[: i + 1])
        assert not np.array_equal(o2[i + 1:], out[i + 1:])


def test_s4_K1_is_the_prefix_mean(orc):
    wl, mu, vr, lp, qx, kx, v = _tiny(K=1)
    eps = 0.5
    out = orc.causal(mu, vr, lp, qx, kx, v, eps)[0]
    cs = np.cumsum(v[0].astype(np.float64), 0)
    n = np.arange(1, wl.N + 1, dtype=np.float64)[:, None]
    np.testing.assert_allclose(out, cs / (n + eps), rtol=1e-12, atol=1e-15)


def test_s4_last_row_equals_bidir(orc):
    wl, mu, vr, lp, qx, kx, v = _tiny()
    c = orc.causal(mu, vr, lp, qx, kx, v, 1e-6)[0]
    b = orc.bidir(mu, vr, lp, qx, kx, v, 1e-6)[0]
    np.testing.assert_allclose(c[-1], b[-1], rtol=1e-12, atol=1e-15)
    assert not np.allclose(c[0], b[0])


def test_s4_state_carry_and_split(orc):
    """Splitting the sequence and carrying the state is exact, and the final
    state is the bidirectional write [Gamma_K^T V, Gamma_K^T 1]."""
    wl, mu, vr, lp, qx, kx, v = _tiny()
    full, st = orc.causal(mu, vr, lp, qx, kx, v, 1e-6, return_state=True)
    gk = _sklearn_posterior(mu[0], vr[0], lp[0], kx[0])
    expect = np.concatenate([(gk.T @ v[0].astype(np.float64)).ravel(), gk.sum(0)])
    np.testing.assert_allclose(st[0], expect, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(orc.write(mu, vr, lp, kx, v)[0], expect, rtol=1e-10, atol=1e-12)
    for m in (1, 100, 128):
        a, sa = orc.causal(mu, vr, lp, qx[:, :m], kx[:, :m], v[:, :m], 1e-6, return_state=True)
        b, sb = orc.causal(mu, vr, lp, qx[:, m:], kx[:, m:], v[:, m:], 1e-6, state_in=sa,
                           return_state=True)
        np.testing.assert_allclose(np.concatenate([a, b], 1), full, rtol=1e-11, atol=1e-14)
        np.testing.assert_allclose(sb, st, rtol=1e-12, atol=1e-12)


def test_bidir_is_write_then_read_and_splits(orc):
    """The bidirectional memory of a split sequence is the sum of the parts'
    memories (the exchange a sequence-split run would all-reduce)."""
    wl, mu, vr, lp, qx, kx, v = _tiny()
    b = orc.bidir(mu, vr, lp, qx, kx, v, 1e-6)
    s1 = orc.write(mu, vr, lp, kx[:, :77], v[:, :77])
    s2 = orc.write(mu, vr, lp, kx[:, 77:], v[:, 77:])
    np.testing.assert_allclose(orc.read(mu, vr, lp, qx, s1 + s2, 1e-6), b, rtol=1e-11, atol=1e-14)


# ----------------------------------------------------- cross-attention -----

@pytest.mark.parametrize("nq,nk", [(40, 256), (256, 40), (1, 7)])
def test_cross_matches_rectangular_bruteforce(orc, nq, nk):
    """Queries of one sequence read the memory written by the keys of another: the
    latent-memory form equals the rectangular affinity Gamma_Q Gamma_K^T (nq x nk)
    materialised from the library GMM posterior."""
    wl, mu, vr, lp, qx, kx, v = _tiny()
    q, k, vv = qx[:, :nq], kx[:, wl.N - nk:], v[:, wl.N - nk:]
    gq = _sklearn_posterior(mu[0], vr[0], lp[0], q[0])
    gk = _sklearn_posterior(mu[0], vr[0], lp[0], k[0])
    for eps in (1e-6, 0.37):
        ref = _bruteforce(gq, gk, vv[0].astype(np.float64), eps, False)
        out = orc.cross(mu, vr, lp, q, k, vv, eps)[0]
        assert out.shape == (nq, wl.dv)
        np.testing.assert_allclose(out, ref, rtol=1e-9, atol=1e-12)


def test_cross_special_cases(orc):
    """Equal lengths and the same rows give the bidirectional form; K = 1 gives the
    mean of the key sequence's values for every query; no keys give 0 / eps."""
    wl, mu, vr, lp, qx, kx, v = _tiny()
    np.testing.assert_array_equal(orc.cross(mu, vr, lp, qx, kx, v, 1e-6), orc.bidir(mu, vr, lp, qx, kx, v, 1e-6))
    wl1, mu1, vr1, lp1, q1, k1, v1 = _tiny(K=1)
    out = orc.cross(mu1, vr1, lp1, q1[:, :9], k1[:, 100:], v1[:, 100:], 0.25)[0]
    expect = v1[0, 100:].astype(np.float64).sum(0) / (wl1.N - 100 + 0.25)
    np.testing.assert_allclose(out, np.tile(expect, (9, 1)), rtol=1e-12, atol=1e-15)
    empty = orc.cross(mu, vr, lp, qx[:, :5], kx[:, :0], v[:, :0], 0.5)
    np.testing.assert_array_equal(empty, np.zeros((1, 5, wl.dv)))


# ----------------------------------------------------------- diagnostics -----

def test_usage_is_the_sum_and_argmax_of_the_posterior(orc):
    """Soft usage = column sums of Gamma, hard assignments = row argmax, summed per head
    over the slices of that head; checked against numpy on the library GMM posterior."""
    wl = TINY.with_(B=2, H=2, N=300, K=12, d=8)
    mu, vr, lp = wlmod.params(wl)
    xs, heads = [], []
    for b in range(wl.B):
        for h in range(wl.H):
            xs.append(wlmod.slice_inputs(wl, b, h, mu=mu)[0])
            heads.append(h)
    x = np.stack(xs)
    u, c, a, e = orc.usage(mu, vr, lp, x, heads=heads)
    for h in range(wl.H):
        g = np.concatenate([_sklearn_posterior(mu[h], vr[h], lp[h], x[s]) for s in range(len(xs))
                            if heads[s] == h])
        np.testing.assert_allclose(u[h], g.sum(0), rtol=1e-10, atol=1e-10)
        top2 = np.sort(g, 1)[:, -2:]
        clear = top2[:, 1] - top2[:, 0] > 1e-9        # rows whose argmax is not a near-tie
        assign = np.concatenate([a[s] for s in range(len(xs)) if heads[s] == h])
        np.testing.assert_array_equal(assign[clear], g.argmax(1)[clear])
        np.testing.assert_array_equal(c[h], np.bincount(assign, minlength=wl.K))
        p = u[h] / u[h].sum()
        np.testing.assert_allclose(e[h, 0], -(p * np.log(p)).sum() / np.log(wl.K), rtol=1e-12)
        q = c[h][c[h] > 0] / c[h].sum()
        np.testing.assert_allclose(e[h, 1], -(q * np.log(q)).sum() / np.log(wl.K), rtol=1e-12)
    assert u.sum() == pytest.approx(wl.B * wl.H * wl.N, rel=1e-12)
    assert c.sum() == wl.B * wl.H * wl.N


def test_usage_closed_forms(orc):
    """Equal components: every row's posterior is pi, so the soft usage is N pi, every row
    is assigned to argmax pi and the hard entropy is 0; K = 1: all mass on one component."""
    rng = np.random.default_rng(11)
    K, d, N = 7, 5, 90
    mu = np.tile(rng.normal(size=(1, 1, d)), (1, K, 1))
    vr = np.tile(rng.normal(size=(1, 1, d)), (1, K, 1))
    l = rng.normal(size=(1, K))
    u, c, a, e = orc.usage(mu, vr, l, rng.normal(size=(1, N, d)))
    pi = softmax(l[0])
    np.testing.assert_allclose(u[0], N * pi, rtol=1e-12)
    assert (a == pi.argmax()).all() and c[0, pi.argmax()] == N
    np.testing.assert_allclose(e[0, 0], -(pi * np.log(pi)).sum() / np.log(K), rtol=1e-12)
    assert e[0, 1] == 0.0
    # uniform priors and equal components: the soft usage has the largest entropy, 1
    u, c, a, e = orc.usage(mu, vr, np.zeros((1, K)), rng.normal(size=(1, N, d)))
    assert e[0, 0] == pytest.approx(1.0, rel=1e-12)
    assert (a == 0).all()                              # ties go to the lowest component
    wl1, mu1, vr1, lp1, q1, _, _ = _tiny(K=1)
    u, c, a, e = orc.usage(mu1, vr1, lp1, q1)
    assert u[0, 0] == pytest.approx(wl1.N, rel=1e-14) and c[0, 0] == wl1.N and (e == 0).all()


def test_usage_follows_component_permutation(orc):
    wl, mu, vr, lp, qx, _, _ = _tiny()
    perm = np.random.default_rng(12).permutation(wl.K)
    u, c, a, e = orc.usage(mu, vr, lp, qx)
    up, cp, ap, ep = orc.usage(mu[:, perm], vr[:, perm], lp[:, perm], qx)
    np.testing.assert_allclose(up[0], u[0, perm], rtol=1e-12)
    np.testing.assert_array_equal(cp[0], c[0, perm])
    np.testing.assert_allclose(ep, e, rtol=1e-12)


# ------------------------------------------------------------- gradients -----

def _torch_bruteforce_grads(mu, vr, lp, qx, kx, v, eps, W, causal):
    """Gradients of L = sum(W * O) by torch autograd through a brute-force fp64 forward
    (library softplus / log-softmax / softmax, the N x N affinity materialised): an
    implementation that shares nothing with the oracle."""
    torch = pytest.importorskip("torch")
    t = lambda a: torch.tensor(np.asarray(a, np.float64), requires_grad=True)
    mu_t, vr_t, lp_t, q_t, k_t, v_t = (t(a) for a in (mu[0], vr[0], lp[0], qx[0], kx[0], v[0]))
    var = torch.nn.functional.softplus(vr_t)
    logpi = torch.log_softmax(lp_t, 0)

    def post(x):
        ll = logpi[None] - 0.5 * (((x[:, None, :] - mu_t[None]) ** 2) / var[None] + torch.log(var)[None]
                                  + math.log(2 * math.pi)).sum(-1)
        return torch.softmax(ll, 1)

    A = post(q_t) @ post(k_t).T
    if causal:
        A = torch.tril(A)
    O = (A @ v_t) / (A.sum(1, keepdim=True) + eps)
    (O * torch.tensor(W[0])).sum().backward()
    return [a.grad.numpy() for a in (q_t, k_t, v_t, mu_t, vr_t, lp_t)]


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("eps", [1e-6, 0.3])
def test_backward_matches_autograd_of_bruteforce(orc, causal, eps):
    wl, mu, vr, lp, qx, kx, v = _tiny(N=96, K=6, d=5, dv=7)
    W = np.random.default_rng(21).normal(size=(1, wl.N, wl.dv))
    got = orc.backward(mu, vr, lp, qx, kx, v, eps, W, causal=causal)
    ref = _torch_bruteforce_grads(mu, vr, lp, qx, kx, v, eps, W, causal)
    names = ("dqx", "dkx", "dv", "dmu", "dvar_raw", "dlogit_pi")
    for name, a, b in zip(names, got, ref):
        a = a.reshape(b.shape)
        assert np.abs(a - b).max() <= 1e-9 * max(np.abs(b).max(), 1e-300), name


def test_backward_matches_central_differences(orc):
    """Every gradient against central differences of the oracle's own (pinned) forward."""
    wl, mu, vr, lp, qx, kx, v = _tiny(N=40, K=5, d=4, dv=3)
    rng = np.random.default_rng(22)
    W = rng.normal(size=(1, wl.N, wl.dv))
    eps = 1e-3
    for causal in (True, False):
        fwd = orc.causal if causal else orc.bidir
        args = [np.asarray(a, np.float64).copy() for a in (qx, kx, v, mu, vr, lp)]

        def loss(a):
            q, k, vv, m, r, l = a
            return float((fwd(m, r, l, q, k, vv, eps) * W).sum())

        grads = orc.backward(args[3], args[4], args[5], args[0], args[1], args[2], eps, W, causal=causal)
        for which in range(6):
            flat = args[which].reshape(-1)
            for idx in rng.choice(flat.size, size=min(6, flat.size), replace=False):
                h = 1e-5 * max(1.0, abs(flat[idx]))
                old = flat[idx]
                flat[idx] = old + h
                lp_ = loss(args)
                flat[idx] = old - h
                lm_ = loss(args)
                flat[idx] = old
                fd = (lp_ - lm_) / (2 * h)
                g = grads[which].reshape(-1)[idx]
                assert abs(g - fd) <= 1e-6 * max(1.0, abs(fd)), (causal, which, idx, g, fd)


def test_backward_structure(orc):
    """Causal: dL/dO_i touches only rows <= i through the queries' side, so the query-row
    gradient of row i does not depend on dL/dO of other rows; the value gradient of the
    last row comes from the last output alone; the logit gradient of a head sums to zero
    (softmax); K = 1: routing gradients vanish."""
    wl, mu, vr, lp, qx, kx, v = _tiny(N=50)
    rng = np.random.default_rng(23)
    W = rng.normal(size=(1, wl.N, wl.dv))
    dq, dk, dv, dmu, dvr, dlp = orc.backward(mu, vr, lp, qx, kx, v, 1e-6, W)
    W2 = W.copy()
    W2[0, :10] = rng.normal(size=(10, wl.dv))
    dq2, dk2, dv2, *_ = orc.backward(mu, vr, lp, qx, kx, v, 1e-6, W2)
    np.testing.assert_array_equal(dq2[0, 10:], dq[0, 10:])
    W3 = np.zeros_like(W)
    W3[0, -1] = W[0, -1]
    _, _, dv3, *_ = orc.backward(mu, vr, lp, qx, kx, v, 1e-6, W3)
    np.testing.assert_allclose(dv3[0, -1], dv[0, -1] - orc.backward(mu, vr, lp, qx, kx, v, 1e-6, W - W3)[2][0, -1],
                               rtol=1e-10, atol=1e-14)
    assert abs(dlp.sum()) < 1e-10 * np.abs(dlp).max()
    wl1, mu1, vr1, lp1, q1, k1, v1 = _tiny(K=1, N=30)
    g1 = orc.backward(mu1, vr1, lp1, q1, k1, v1, 1e-6, rng.normal(size=(1, 30, wl1.dv)))
    for a in (g1[0], g1[1], g1[3], g1[4], g1[5]):
        assert np.abs(a).max() == 0.0


# ---------------------------------------------------------------- S5 -------

def test_s5_decode_continues_prefill(orc):
    wl, mu, vr, lp, qx, kx, v = _tiny()
    m = 200
    full = orc.causal(mu, vr, lp, qx, kx, v, 1e-6)[0]
    _, st = orc.causal(mu, vr, lp, qx[:, :m], kx[:, :m], v[:, :m], 1e-6, return_state=True)
    for t in range(m, wl.N):
        o, st = orc.decode_step(mu, vr, lp, qx[:, t], kx[:, t], v[:, t], 1e-6, st)
        np.testing.assert_allclose(o[0], full[t], rtol=1e-11, atol=1e-14)


def test_oracle_heads_and_slices(orc):
    """Slices use their own head's parameters; a sampled subset equals the full run."""
    wl = wlmod.WORKLOADS["tiny"].with_(B=2, H=3, N=40)
    mu, vr, lp = wlmod.params(wl)
    qx, kx, v = wlmod.full_inputs(wl)
    S = wl.B * wl.H
    full = orc.causal(mu, vr, lp, qx.reshape(S, wl.N, -1), kx.reshape(S, wl.N, -1),
                      v.reshape(S, wl.N, -1), wl.eps)
    pick = [1, 5]
    sub = orc.causal(mu, vr, lp, qx.reshape(S, wl.N, -1)[pick], kx.reshape(S, wl.N, -1)[pick],
                     v.reshape(S, wl.N, -1)[pick], wl.eps, heads=[p % wl.H for p in pick])
    np.testing.assert_array_equal(sub, full[pick])
    one = orc.causal(mu[1:2], vr[1:2], lp[1:2], qx[1, 1][None], kx[1, 1][None], v[1, 1][None], wl.eps)
    np.testing.assert_array_equal(one[0], full[4])


def test_oracle_matches_its_recorded_values(orc):
    """Guards against drift: sampled values recorded by tests/golden/make_golden.py."""
    import json
    import os
    with open(os.path.join(os.path.dirname(__file__), "golden", "tiny_oracle.json")) as f:
        rec = json.load(f)
    wl, mu, vr, lp, qx, kx, v = _tiny()
    rows = rec["rows"]
    g = orc.responsibilities(mu, vr, lp, qx)[0]
    c, st = orc.causal(mu, vr, lp, qx, kx, v, wl.eps, return_state=True)
    b = orc.bidir(mu, vr, lp, qx, kx, v, wl.eps)
    np.testing.assert_allclose(g[rows], rec["gamma_q"], rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(c[0, rows], rec["causal"], rtol=1e-11, atol=1e-14)
    np.testing.assert_allclose(b[0, rows], rec["bidir"], rtol=1e-11, atol=1e-14)
    np.testing.assert_allclose(st[0], rec["state_final"], rtol=1e-12, atol=1e-13)
