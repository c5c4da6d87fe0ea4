"""GPU parity: the CUDA library, called through the C ABI, against the fp64
oracle on the same seeded inputs.

Tolerance (normwise per (b, h) slice: max|O - O_ref| / max|O_ref|):
1e-4 when the chunk products carry fp32 operands, 2e-2 when they are bf16
(accumulation in fp32 either way).  Large workloads are checked on a fixed
sample of slices at their full sizes, in the launch configuration the
benchmark uses.
"""
import numpy as np
import pytest
import torch

from gaussian_mixture_sequence_gb300 import workloads
from gpu_cases import DEV, TOL, Case, normwise, shape_of
import gaussian_mixture_sequence_gb300 as gma

pytestmark = pytest.mark.gpu
W = workloads.WORKLOADS


def _report(name, err, tol):
    print(f"{name}: normwise error {err:.3e} (tolerance {tol:.0e})")
    assert err <= tol, f"{name}: {err:.3e} > {tol:.0e}"


# ------------------------------------------------------------ S1 --------------

@pytest.mark.parametrize("wl,sample", [
    (W["tiny"], None),
    (W["tiny"].with_(K=1, B=2, H=2), None),
    (W["tiny"].with_(K=3, d=32, N=77), None),
    (W["tiny"].with_(K=200, d=128, N=300, H=2), None),
    # generic routing: odd K above 256 (64-row tiles, parameters in chunks), bf16 rows, d = 16
    (W["tiny"].with_(K=257, d=64, N=513, H=3, x_dtype="bf16"), None),
    (W["tiny"].with_(K=48, d=16, N=1000, B=2), None),
    (W["tiny"].with_(K=512, d=128, N=200, H=2), None),
    (W["causal_4k"], 4),
    (W["bidir_16k_peaked"], 3),
    # more chunks than SMs, ragged last chunk: persistent CTAs cross slice boundaries
    (W["tiny"].with_(mode="bidir", B=4, H=16, N=1100, d=64, dv=64, K=128), None),
    (W["tiny"].with_(mode="bidir", B=8, H=25, N=200, d=64, dv=64, K=128), None),
    (W["causal_8k_K512"], 2),
    (W["causal_64k_bf16"], 2),
    # the tensor-core routing for 17 <= K <= 64 (d = 64): padded widths, bf16 rows; K = 33 keeps
    # the CUDA-core kernel (fp32 rows of 33 are not 16-byte multiples)
    (W["tiny"].with_(K=40, d=64, N=1000, B=2, H=3), None),
    (W["tiny"].with_(K=64, d=64, N=777, H=2, x_dtype="bf16"), None),
    (W["tiny"].with_(K=20, d=64, N=300, H=2), None),
    (W["tiny"].with_(K=33, d=64, N=300, H=2), None),
    (W["causal_8k_K32"], 2),
    # the wide form (65 <= K <= 256 but 128, d = 64): chunks of 64 components through two
    # buffers (K = 256: a buffer refilled while the other is multiplied), output in halves
    (W["tiny"].with_(K=256, d=64, N=1000, B=2, H=2), None),
    (W["tiny"].with_(K=200, d=64, N=555, H=3, x_dtype="bf16"), None),
    (W["tiny"].with_(K=129, d=64, N=300, H=2), None),
    (W["tiny"].with_(K=100, d=64, N=777, H=2), None),
    (W["tiny"].with_(K=72, d=64, N=300, H=2, x_dtype="bf16"), None),
    (W["causal_8k_K256"], 2),
    # 256 < K <= 512 (d = 64): two CTAs per tile as a cluster, the softmax's row maxima and
    # sums exchanged between them
    (W["tiny"].with_(K=512, d=64, N=1000, B=2, H=2), None),
    (W["tiny"].with_(K=384, d=64, N=555, H=3, x_dtype="bf16"), None),
    (W["tiny"].with_(K=300, d=64, N=300, H=2), None),
])
def test_responsibilities(wl, sample):
    c = Case(wl, None if sample is None else workloads.sample_slices(wl, sample))
    for which in ("q", "k"):
        g = c.pick(c.gamma(which))
        ref = c.ref_gamma(which)
        assert np.abs(g.reshape(ref.shape).sum(-1) - 1).max() < 1e-5
        _report(f"gamma_{which} {wl.name} K={wl.K}", normwise(g, ref), TOL["f32"])


def test_responsibilities_adversarial_rows():
    """Rows that stress the component bound of the K = 128, d = 64 routing path:
    on a centre, midway between two centres, far from every centre (|x| = 1e3,
    logits ~ -1e6), and widely spread; each must match the oracle."""
    import oracle
    from gaussian_mixture_sequence_gb300 import gma
    from gpu_cases import shape_of
    wl = W["causal_4k"].with_(B=1, H=2, N=600)
    mu, vr, lp = workloads.params(wl)
    rng = np.random.default_rng(3)
    rows = []
    for h in range(wl.H):
        r = [mu[h, k] for k in range(0, 128, 8)]
        r += [0.5 * (mu[h, a] + mu[h, b]) for a, b in zip(range(0, 64), range(64, 128))]
        r += [np.full(64, 1e3, np.float32), np.full(64, -1e3, np.float32), np.full(64, 37.0, np.float32)]
        r += [rng.normal(0, 3.0, 64).astype(np.float32) for _ in range(100)]
        r += [rng.normal(0, 1.0, 64).astype(np.float32) for _ in range(wl.N - len(r))]
        rows.append(np.stack(r)[: wl.N])
    x = np.stack(rows)[None].astype(np.float32)              # [1, H, N, 64]
    dev = "cuda:0"
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    g = torch.empty(1, wl.H, wl.N, wl.K, device=dev)
    gma.gma_responsibilities(shape_of(wl), t(mu), t(vr), t(lp), t(x), g)
    ref = oracle.responsibilities(mu, vr, lp, x.reshape(wl.H, wl.N, 64))
    out = g.reshape(wl.H, wl.N, wl.K).cpu().numpy()
    _report("gamma adversarial rows", normwise(out, ref), TOL["f32"])
    assert np.abs(out.sum(-1) - 1).max() < 1e-5


@pytest.mark.parametrize("K,x_dtype", [(128, "f32"), (128, "bf16"), (64, "f32"), (40, "bf16"), (32, "f32"),
                                     (256, "f32"), (96, "bf16"), (512, "f32")])
def test_responsibilities_dense_tiles_across_scales(K, x_dtype):
    """Tiles of N(0, s^2) rows, one scale per tile of 128 rows, from s = 0.3 to s = 6.  At
    K = 128 the wide tiles keep many components and go to the dense passes, the tensor-core
    one below its magnitude limit (s up to about 2) and the exact one above it; at the
    other K every tile takes the tensor-core routing and the rows above the limit its exact
    path.  A last tile mixes N(0, 1) rows with one row of s = 6.  Each tile's posteriors
    must match the oracle's."""
    import oracle
    from gaussian_mixture_sequence_gb300 import gma
    from gpu_cases import shape_of
    scales = [0.3, 0.7, 1.0, 1.4, 1.8, 2.2, 3.0, 6.0]
    wl = W["causal_4k"].with_(B=1, H=2, N=128 * (len(scales) + 1) - 37, K=K, x_dtype=x_dtype)
    mu, vr, lp = workloads.params(wl)
    rng = np.random.default_rng(11)
    x = np.concatenate([s * rng.standard_normal((wl.H, 128, 64)) for s in scales] +
                       [rng.standard_normal((wl.H, 128 - 37, 64))], axis=1).astype(np.float32)
    x[:, 128 * len(scales) + 40] *= 6.0
    if x_dtype == "bf16":
        x = workloads.round_bf16(x)
    dev = "cuda:0"
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    xd = t(x[None]).to(torch.bfloat16) if x_dtype == "bf16" else t(x[None])
    g = torch.empty(1, wl.H, wl.N, wl.K, device=dev)
    gma.gma_responsibilities(shape_of(wl), t(mu), t(vr), t(lp), xd, g)
    ref = oracle.responsibilities(mu, vr, lp, x)
    out = g.reshape(wl.H, wl.N, wl.K).cpu().numpy()
    for j in range(len(scales) + 1):
        rows = slice(128 * j, min(wl.N, 128 * (j + 1)))
        _report(f"gamma tile {j} (scale {scales[j] if j < len(scales) else 'mixed'}) K={K} {x_dtype}",
                normwise(out[:, rows], ref[:, rows]), TOL["f32"])
    assert np.abs(out.sum(-1) - 1).max() < 1e-5


# --------------------------------------------------------- S2 + S3 -------------

@pytest.mark.parametrize("wl,sample", [
    (W["tiny"].with_(mode="bidir"), None),
    (W["tiny"].with_(mode="bidir", B=2, H=3, N=1000, d=32, dv=128, K=40), None),
    (W["tiny"].with_(mode="bidir", N=1, K=16), None),
    (W["tiny"].with_(mode="bidir", B=2, H=2, N=1000, d=64, dv=64, K=128), None),
    (W["tiny"].with_(mode="bidir", B=1, H=2, N=300, d=32, dv=128, K=128, gemm_dtype="bf16", v_dtype="bf16"), None),
    (W["bidir_16k_peaked"], 3),
    # more chunks than SMs, ragged last chunk: persistent CTAs cross slice boundaries
    (W["tiny"].with_(mode="bidir", B=4, H=16, N=1100, d=64, dv=64, K=128), None),
    (W["tiny"].with_(mode="bidir", B=8, H=25, N=200, d=64, dv=64, K=128), None),
    (W["causal_4k"].with_(mode="bidir", gemm_dtype="bf16"), 2),
    # tensor-core path with component groups
    (W["tiny"].with_(mode="bidir", B=2, H=2, N=1000, d=64, dv=64, K=256), None),
    (W["tiny"].with_(mode="bidir", B=2, H=2, N=900, d=64, dv=64, K=40), None),
    (W["causal_8k_K512"].with_(mode="bidir"), 2),
])
def test_bidir(wl, sample):
    c = Case(wl, None if sample is None else workloads.sample_slices(wl, sample))
    out = c.pick(c.bidir())
    _report(f"bidir {wl.name} N={wl.N} K={wl.K} dv={wl.dv}", normwise(out, c.ref_bidir()),
            TOL[wl.gemm_dtype])


# ------------------------------------------------------------ S4 --------------

CAUSAL = [
    (W["tiny"], None, 0),
    (W["tiny"], None, 16),
    (W["tiny"], None, 32),
    (W["tiny"].with_(K=1, N=300), None, 0),
    (W["tiny"].with_(N=1), None, 0),
    (W["tiny"].with_(B=2, H=3, N=1000, d=32, dv=128, K=40), None, 0),
    (W["tiny"].with_(N=257, K=24, dv=32), None, 16),
    (W["causal_4k"], 4, 0),
    (W["causal_4k"], 2, 64),
    (W["causal_4k_bf16"], 4, 0),
    (W["causal_4k_bf16"], 2, 64),
    (W["tiny"].with_(B=2, H=2, N=1000, d=64, dv=64, K=128), None, 0),
    (W["tiny"].with_(B=1, H=2, N=129, d=16, dv=64, K=128), None, 0),
    (W["tiny"].with_(B=1, H=1, N=1, d=64, dv=64, K=128), None, 0),
    (W["tiny"].with_(B=1, H=2, N=700, d=32, dv=128, K=128, gemm_dtype="bf16", v_dtype="bf16"), None, 0),
    # more chunks than SMs, ragged last chunk: persistent CTAs cross slice boundaries
    (W["tiny"].with_(B=4, H=16, N=1100, d=64, dv=64, K=128), None, 0),
    # two-chunk slices, three chunks per CTA: the state kernel's ranges span slices
    (W["tiny"].with_(B=8, H=25, N=200, d=64, dv=64, K=128), None, 0),
    (W["tiny"].with_(B=2, H=16, N=1100, d=64, dv=128, K=128, gemm_dtype="bf16", v_dtype="bf16"), None, 0),
    (W["causal_16k_peaked"], 3, 0),
    (W["causal_16k_peaked_bf16"], 2, 0),
    (W["causal_64k_bf16"], 2, 0),
    (W["causal_8k_K32"], 2, 0),
    (W["causal_8k_K64"], 2, 0),
    (W["causal_8k_K256"], 2, 0),
    (W["causal_8k_K512"], 2, 0),
    # tensor-core path with component groups: K < 128 padded, K = 256 / 384, bf16 and split operands,
    # ragged chunks, more chunks than SMs; K = 200 stays on CUDA cores (its routing, like that of
    # K = 100 and 256 at d = 64, takes the wide tensor-core form)
    (W["tiny"].with_(B=2, H=2, N=1000, d=64, dv=64, K=100), None, 0),
    (W["tiny"].with_(B=2, H=2, N=700, d=32, dv=64, K=8), None, 0),
    (W["tiny"].with_(B=2, H=2, N=1000, d=64, dv=64, K=256), None, 0),
    (W["tiny"].with_(B=1, H=3, N=1300, d=16, dv=64, K=384), None, 0),
    (W["tiny"].with_(B=1, H=2, N=700, d=32, dv=128, K=256, gemm_dtype="bf16", v_dtype="bf16"), None, 0),
    (W["tiny"].with_(B=4, H=16, N=1100, d=64, dv=64, K=512), None, 0),
    (W["tiny"].with_(B=1, H=2, N=600, d=64, dv=64, K=200), None, 0),
    # the tensor-core routing for 17 <= K <= 64 with padded widths, fp32 and bf16 rows
    (W["tiny"].with_(B=2, H=3, N=1000, d=64, dv=64, K=20), None, 0),
    (W["tiny"].with_(B=1, H=2, N=700, d=64, dv=64, K=48, x_dtype="bf16"), None, 0),
]


@pytest.mark.parametrize("wl,sample,chunk", CAUSAL, ids=[f"{w.name}-N{w.N}-K{w.K}-C{c}" for w, _, c in CAUSAL])
def test_causal(wl, sample, chunk):
    c = Case(wl, None if sample is None else workloads.sample_slices(wl, sample))
    out, st = c.causal(chunk=chunk, want_state=True)
    ref, ref_st = c.ref_causal(return_state=True)
    tol = TOL[wl.gemm_dtype]
    _report(f"causal {wl.name} N={wl.N} K={wl.K} C={chunk}", normwise(c.pick(out), ref), tol)
    _report(f"causal state {wl.name}", normwise(c.pick(st), ref_st), tol)


@pytest.mark.parametrize("K", [32, 128, 256])
def test_causal_state_carry(K):
    """Two calls chained through state_out -> state_in equal one call on the whole sequence."""
    wl = W["tiny"].with_(B=2, H=2, N=600, K=K, d=64, dv=64)
    c = Case(wl)
    q, k, v = c.dev["seq"]
    from gaussian_mixture_sequence_gb300 import gma
    from gpu_cases import shape_of
    m = 333
    o1 = torch.empty(wl.B, wl.H, m, wl.dv, device="cuda:0")
    o2 = torch.empty(wl.B, wl.H, wl.N - m, wl.dv, device="cuda:0")
    s1 = torch.empty(wl.B, wl.H, wl.K * wl.dv + wl.K, device="cuda:0")
    s2 = torch.empty_like(s1)
    gma.gma_forward_causal(shape_of(wl, N=m), *c.prm, q[:, :, :m].contiguous(), k[:, :, :m].contiguous(),
                           v[:, :, :m].contiguous(), o1, state_out=s1)
    gma.gma_forward_causal(shape_of(wl, N=wl.N - m), *c.prm, q[:, :, m:].contiguous(),
                           k[:, :, m:].contiguous(), v[:, :, m:].contiguous(), o2, state_in=s1, state_out=s2)
    ref, ref_st = c.ref_causal(return_state=True)
    out = torch.cat([o1, o2], 2)
    _report("causal split at 333", normwise(c.pick(out), ref), TOL["f32"])
    _report("causal split state", normwise(c.pick(s2), ref_st), TOL["f32"])
    # state_out may alias state_in
    gma.gma_forward_causal(shape_of(wl, N=wl.N - m), *c.prm, q[:, :, m:].contiguous(),
                           k[:, :, m:].contiguous(), v[:, :, m:].contiguous(), o2, state_in=s1, state_out=s1)
    assert torch.equal(s1, s2)
    # an empty sequence passes the state through
    s3 = torch.full_like(s1, 7.0)
    e = torch.empty(wl.B, wl.H, 0, wl.dv, device="cuda:0")
    z = torch.empty(wl.B, wl.H, 0, wl.d, device="cuda:0")
    gma.gma_forward_causal(shape_of(wl, N=0), *c.prm, z, z, e, e, state_in=s2, state_out=s3)
    assert torch.equal(s3, s2)


@pytest.mark.parametrize("K", [64, 128])
def test_causal_prefix_property_bitwise(K):
    """Perturbing tokens after position i leaves outputs 0..i bit-identical."""
    wl = W["tiny"].with_(B=1, H=2, N=700, K=K, d=64, dv=64)
    c = Case(wl)
    base = c.causal()
    q, k, v = c.dev["seq"]
    for i in (0, 63, 64, 127, 128, 255, 256, 400):
        c.dev["seq"] = (q.clone(), k.clone(), v.clone())
        for t in c.dev["seq"]:
            t[:, :, i + 1:] += 0.5
        out = c.causal()
        assert torch.equal(out[:, :, : i + 1], base[:, :, : i + 1]), i
        assert not torch.equal(out[:, :, i + 1:], base[:, :, i + 1:])
    c.dev["seq"] = (q, k, v)


@pytest.mark.parametrize("K,chunks", [(64, (16, 32, 64, 128)), (128, (16, 64, 128)), (256, (64, 128))])
def test_chunk_size_invariance(K, chunks):
    """The chunkwise form is exact: chunk lengths (and the tensor-core path at
    chunk 128 against the CUDA-core path at 16/64) agree to rounding."""
    wl = W["tiny"].with_(B=1, H=2, N=1000, K=K, d=64, dv=64)
    c = Case(wl)
    outs = [c.causal(chunk=ch) for ch in chunks]
    for o in outs[1:]:
        assert (o - outs[0]).abs().max().item() <= 1e-5 * outs[0].abs().max().item()


def test_repeatable_bitwise():
    wl = W["causal_4k"].with_(B=1, H=2, N=2000)
    c = Case(wl)
    a, b = c.causal(), c.causal()
    assert torch.equal(a, b)
    a, b = c.causal(chunk=64), c.causal(chunk=64)
    assert torch.equal(a, b)
    x, y = c.bidir(), c.bidir()
    assert torch.equal(x, y)


def test_unwritten_lo_planes_are_never_read():
    """On peaked inputs the routing of Q leaves the lo plane of a tile unwritten when every row
    keeps its argmax alone (the plane is zero) and the chunk output skips it.  A workspace that
    an N(0, 1) call filled with non-zero lo planes must give, on the peaked call after it,
    bitwise the output of a fresh workspace filled with NaN bytes, and match the oracle."""
    from gaussian_mixture_sequence_gb300 import gma
    from gpu_cases import shape_of
    wl_p = W["causal_16k_peaked"].with_(B=1, H=2, N=2048 + 77)
    wl_n = wl_p.with_(dist="normal")
    cp, cn = Case(wl_p), Case(wl_n)
    dev = "cuda:0"
    for mode, op, fn in (("causal", gma.OP_CAUSAL, gma.gma_forward_causal),
                         ("bidir", gma.OP_BIDIR, gma.gma_forward_bidir)):
        size = gma.gma_workspace_size(shape_of(wl_p), op)
        ws = torch.empty(size, dtype=torch.uint8, device=dev)
        out_n = torch.empty(wl_p.B, wl_p.H, wl_p.N, wl_p.dv, device=dev)
        fn(shape_of(wl_n), *cn.prm, *cn.dev["seq"], out_n, ws=ws)   # non-zero lo planes everywhere
        out_a = torch.empty_like(out_n)
        fn(shape_of(wl_p), *cp.prm, *cp.dev["seq"], out_a, ws=ws)
        fresh = torch.full((size,), 0xFF, dtype=torch.uint8, device=dev)   # NaN in every plane
        out_b = torch.empty_like(out_n)
        fn(shape_of(wl_p), *cp.prm, *cp.dev["seq"], out_b, ws=fresh)
        torch.cuda.synchronize()
        assert torch.equal(out_a, out_b), mode
        ref = cp.ref_causal() if mode == "causal" else cp.ref_bidir()
        _report(f"{mode} after a reused workspace", normwise(cp.pick(out_a), ref), TOL["f32"])


# ------------------------------------------------------------ S5 --------------

def _decode_run(c, prefill_state):
    from gaussian_mixture_sequence_gb300 import gma
    from gpu_cases import shape_of
    wl = c.wl
    q, k, v = c.dev["dec"]
    state = prefill_state.clone()
    outs = torch.empty(wl.B, wl.H, wl.decode_steps, wl.dv, device="cuda:0")
    ws = torch.empty(gma.gma_workspace_size(shape_of(wl), gma.OP_DECODE), dtype=torch.uint8,
                     device="cuda:0")
    o = torch.empty(wl.B, wl.H, wl.dv, device="cuda:0")
    qs, ks, vs = (t.permute(2, 0, 1, 3).contiguous() for t in (q, k, v))
    for t in range(wl.decode_steps):
        gma.gma_decode_step(shape_of(wl), *c.prm, qs[t], ks[t], vs[t], state, o, ws=ws)
        outs[:, :, t] = o
    return outs, state


@pytest.mark.parametrize("wl,sample", [
    (W["decode_b256"].with_(B=2, H=2, N=300, decode_steps=40, K=24, d=16, dv=32), None),
    # K not a multiple of 4: slices of the state are not 16-byte aligned (the scalar state pass)
    (W["decode_b256"].with_(B=1, H=3, N=70, decode_steps=12, K=7, d=16, dv=16), None),
    (W["decode_b256"].with_(B=2, H=2, N=130, decode_steps=9, K=128, d=64, dv=128), None),
    (W["decode_b256"], 3),
])
def test_decode_after_prefill(wl, sample):
    c = Case(wl, None if sample is None else workloads.sample_slices(wl, sample), decode=True)
    _, st = c.causal(want_state=True)
    outs, final = _decode_run(c, st)
    _, ref_st = c.ref_causal(return_state=True)
    q, k, v = c.host["dec"]
    ref = np.empty((len(c.slices), wl.decode_steps, wl.dv))
    import oracle
    for t in range(wl.decode_steps):
        ref[:, t], ref_st = oracle.decode_step(c.mu, c.vr, c.lp, q[:, t], k[:, t], v[:, t], wl.eps, ref_st,
                                               heads=c.heads)
    _report(f"decode {wl.name} B={wl.B}", normwise(c.pick(outs), ref), TOL["f32"])
    _report(f"decode state {wl.name}", normwise(c.pick(final), ref_st), TOL["f32"])


# ------------------------------------------------- host-buffer causal entry ----

@pytest.mark.parametrize("wl", [W["causal_16k_peaked"].with_(H=5, N=3000), W["tiny"].with_(B=3, H=2, N=300, K=128, d=64, dv=64),
                                W["tiny"].with_(B=2, H=3, N=257, K=40, d=32, dv=32)])
def test_causal_host_entry_matches_device_entry(wl):
    """The host-buffer entry copies in groups of slices and overlaps copies with compute:
    its output and final state equal the device entry's bit for bit (slices are independent)."""
    c = Case(wl)
    out_dev, st_dev = c.causal(want_state=True)
    q, k, v = (t.cpu().pin_memory() for t in c.dev["seq"])
    out_host = torch.empty(wl.B, wl.H, wl.N, wl.dv).pin_memory()
    st = torch.empty(wl.B, wl.H, wl.K * wl.dv + wl.K, device=DEV)
    gma.gma_forward_causal_host(shape_of(wl), *c.prm, q, k, v, out_host, state_out=st)
    torch.cuda.synchronize()
    assert torch.equal(out_host, out_dev.cpu())
    assert torch.equal(st, st_dev)
    _report(f"causal host entry {wl.name}", normwise(c.pick(out_host), c.ref_causal()), TOL[wl.gemm_dtype])
