"""Seeded synthetic workloads for Gaussian Mixture Attention (GMA).

This module only draws random numbers and names problem sizes.  It holds none
of the method's arithmetic (no softplus, no posterior, no mixing): both the
fp64 oracle and the CUDA library receive exactly the arrays produced here.

Every tensor is generated per (batch, head) slice from its own counter-keyed
PCG64 stream, ``SeedSequence([seed, tensor_code, b, h])``, so any slice can be
regenerated on its own (the oracle checks sampled slices of the large
workloads) and the values do not depend on the machine or on numpy's thread
count.  Per-head GMM parameters use ``SeedSequence([seed, tensor_code, h])``.

Value distributions are those of the benchmark and test workloads defined
below (the pages fix the model -- the diagonal GMM of the GMA explainer's
"핵심 메커니즘", with softplus variances and softmax mixture weights -- but
print no input distributions):

* mu_k ~ N(0, 1); raw variance r ~ N(0, 0.5^2) (0.5 read as a standard
  deviation); mixture logits l ~ N(0, 1).
* routing vectors Q_X, K_X and values V ~ N(0, 1), or, for the "peaked"
  workload, x = mu_c + 0.3 z with c uniform over the K centres of the head, so
  that the responsibilities concentrate on one component.
* bf16 workloads round the drawn fp32 values to bf16 (round to nearest even);
  the returned float32 arrays then hold exactly representable bf16 values.
"""
from __future__ import annotations

import dataclasses
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_CODES = {
    "mu": 1, "var_raw": 2, "logit_pi": 3,
    "qx": 4, "kx": 5, "v": 6,
    "qx_dec": 7, "kx_dec": 8, "v_dec": 9,
    "qcomp": 10, "kcomp": 11, "qcomp_dec": 12, "kcomp_dec": 13, "dout": 14,
}


@dataclasses.dataclass(frozen=True)
class Workload:
    """One problem size: shapes, dtypes, value distribution and default seed."""
    name: str
    B: int
    H: int
    N: int
    d: int            # d_route: width of Q_X and K_X rows
    dv: int           # d_v: width of V rows
    K: int            # number of Gaussian components
    mode: str         # "causal", "bidir", "decode" or "backward" (gradients of the causal form)
    eps: float = 1e-6
    x_dtype: str = "f32"      # storage of Q_X / K_X: "f32" or "bf16"
    v_dtype: str = "f32"      # storage of V
    gemm_dtype: str = "f32"   # chunk-product operand precision: "f32" or "bf16"
    dist: str = "normal"      # "normal" or "peaked"
    chunk: int = 0            # causal chunk length; 0 = the library's default
    decode_steps: int = 0     # decode workloads: steps after an N-token prefill
    seed: int = 1000

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The problem sizes the GMA hot path is measured and checked on.
WORKLOADS = {
    "tiny": Workload("tiny", 1, 1, 256, 16, 16, 8, "causal", seed=1000),
    "causal_4k": Workload("causal_4k", 4, 8, 4096, 64, 64, 128, "causal", seed=1001),
    "causal_4k_bf16": Workload("causal_4k_bf16", 4, 8, 4096, 64, 64, 128, "causal",
                               gemm_dtype="bf16", seed=1001),
    "bidir_16k_peaked": Workload("bidir_16k_peaked", 2, 16, 16384, 64, 64, 128, "bidir",
                                 dist="peaked", seed=1002),
    "causal_16k_peaked": Workload("causal_16k_peaked", 2, 16, 16384, 64, 64, 128, "causal",
                                  dist="peaked", seed=1002),
    # the same sequence with bf16 chunk-product operands (fp32 accumulation)
    "causal_16k_peaked_bf16": Workload("causal_16k_peaked_bf16", 2, 16, 16384, 64, 64, 128, "causal",
                                       gemm_dtype="bf16", dist="peaked", seed=1002),
    "causal_64k_bf16": Workload("causal_64k_bf16", 1, 16, 65536, 64, 128, 128, "causal",
                                x_dtype="bf16", v_dtype="bf16", gemm_dtype="bf16", seed=1003),
    "causal_8k_K32": Workload("causal_8k_K32", 4, 8, 8192, 64, 64, 32, "causal", seed=1004),
    "causal_8k_K64": Workload("causal_8k_K64", 4, 8, 8192, 64, 64, 64, "causal", seed=1004),
    "causal_8k_K256": Workload("causal_8k_K256", 4, 8, 8192, 64, 64, 256, "causal", seed=1004),
    "causal_8k_K512": Workload("causal_8k_K512", 4, 8, 8192, 64, 64, 512, "causal", seed=1004),
    "decode_b256": Workload("decode_b256", 256, 16, 4096, 64, 64, 128, "decode",
                            decode_steps=1024, seed=1005),
    # gradients of the causal form (dL/dO drawn N(0,1) per slice)
    "backward_4k": Workload("backward_4k", 4, 8, 4096, 64, 64, 128, "backward", seed=1001),
    "backward_16k_peaked": Workload("backward_16k_peaked", 2, 16, 16384, 64, 64, 128, "backward",
                                    dist="peaked", seed=1002),
}


def _rng(seed: int, *key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, *key])))


def round_bf16(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); returns float32."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return r.astype(np.uint32).view(np.float32).reshape(a.shape)


def params(wl: Workload, seed: int | None = None):
    """Per-head GMM parameters: mu [H,K,d], var_raw [H,K,d], logit_pi [H,K] (float32)."""
    seed = wl.seed if seed is None else seed
    mu = np.empty((wl.H, wl.K, wl.d), np.float32)
    var_raw = np.empty((wl.H, wl.K, wl.d), np.float32)
    logit_pi = np.empty((wl.H, wl.K), np.float32)
    for h in range(wl.H):
        mu[h] = _rng(seed, _CODES["mu"], h).standard_normal((wl.K, wl.d), dtype=np.float32)
        var_raw[h] = 0.5 * _rng(seed, _CODES["var_raw"], h).standard_normal(
            (wl.K, wl.d), dtype=np.float32)
        logit_pi[h] = _rng(seed, _CODES["logit_pi"], h).standard_normal(wl.K, dtype=np.float32)
    return mu, var_raw, logit_pi


def _route_slice(wl, seed, name, comp_name, b, h, n, mu_h):
    rng = _rng(seed, _CODES[name], b, h)
    z = rng.standard_normal((n, wl.d), dtype=np.float32)
    if wl.dist == "peaked":
        c = _rng(seed, _CODES[comp_name], b, h).integers(0, wl.K, size=n)
        z = mu_h[c] + np.float32(0.3) * z
    elif wl.dist != "normal":
        raise ValueError(f"unknown distribution {wl.dist!r}")
    return round_bf16(z) if wl.x_dtype == "bf16" else z


def slice_inputs(wl: Workload, b: int, h: int, seed: int | None = None, mu=None,
                 decode: bool = False):
    """Q_X [n,d], K_X [n,d], V [n,dv] of slice (b, h) as float32.

    ``decode=True`` returns the ``decode_steps`` tokens that follow the prefill
    of a decode workload instead of the N prefill tokens.
    """
    seed = wl.seed if seed is None else seed
    if mu is None:
        mu = params(wl, seed)[0]
    n = wl.decode_steps if decode else wl.N
    sfx = "_dec" if decode else ""
    qx = _route_slice(wl, seed, "qx" + sfx, "qcomp" + sfx, b, h, n, mu[h])
    kx = _route_slice(wl, seed, "kx" + sfx, "kcomp" + sfx, b, h, n, mu[h])
    v = _rng(seed, _CODES["v" + sfx], b, h).standard_normal((n, wl.dv), dtype=np.float32)
    if wl.v_dtype == "bf16":
        v = round_bf16(v)
    return qx, kx, v


def full_inputs(wl: Workload, seed: int | None = None, decode: bool = False, threads: int = 8):
    """Q_X [B,H,n,d], K_X [B,H,n,d], V [B,H,n,dv] (float32), all slices."""
    seed = wl.seed if seed is None else seed
    mu = params(wl, seed)[0]
    n = wl.decode_steps if decode else wl.N
    qx = np.empty((wl.B, wl.H, n, wl.d), np.float32)
    kx = np.empty((wl.B, wl.H, n, wl.d), np.float32)
    v = np.empty((wl.B, wl.H, n, wl.dv), np.float32)

    def fill(bh):
        b, h = divmod(bh, wl.H)
        qx[b, h], kx[b, h], v[b, h] = slice_inputs(wl, b, h, seed, mu, decode)

    with ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(fill, range(wl.B * wl.H)))
    return qx, kx, v


def sample_slices(wl: Workload, count: int, seed: int = 7):
    """A fixed, sorted sample of distinct (b, h) slice indices (always includes the last)."""
    total = wl.B * wl.H
    if count >= total:
        return list(range(total))
    rng = np.random.default_rng(seed)
    pick = set(rng.choice(total - 1, size=count - 1, replace=False).tolist())
    pick.add(total - 1)
    return sorted(pick)


def dout_slice(wl: Workload, b: int, h: int, seed: int | None = None):
    """dL/dO [N, dv] of slice (b, h) for the gradient workloads, N(0,1), float32."""
    seed = wl.seed if seed is None else seed
    return _rng(seed, _CODES["dout"], b, h).standard_normal((wl.N, wl.dv), dtype=np.float32)


def full_dout(wl: Workload, seed: int | None = None):
    """dL/dO [B, H, N, dv] for the gradient workloads."""
    g = np.empty((wl.B, wl.H, wl.N, wl.dv), np.float32)
    for b in range(wl.B):
        for h in range(wl.H):
            g[b, h] = dout_slice(wl, b, h, seed)
    return g
