"""fp64 CPU oracle for Gaussian Mixture Attention (GMA): numpy front end.

TEST INFRASTRUCTURE ONLY.  The tests, the smoke check and the CPU-baseline
leg of the benchmark are the only callers.  The product (the CUDA library and
its Python binding) never imports this package, and this package imports
nothing from the product.

The arithmetic lives in ``gma_oracle.c`` (plain C, double precision, one
token at a time, OpenMP across independent (batch, head) slices).  This file
only compiles it, converts arrays to float64 and calls it.  Every function
follows the GMA explainer page "Gaussian Mixture Attention: Linear-Time
Sequence Mixing via Probabilistic Latent Routing", technical summary,
sections "핵심 메커니즘" and "변형 및 학습"; see the C file for the step list.

Slices: routing inputs are ``[S, n, d]`` arrays of S independent sequences;
``heads[s]`` names the head whose parameters slice s uses (default: slice s
uses head s % H, matching a ``[B, H, n, d]`` tensor reshaped to ``[B*H, n, d]``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gma_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libgma_oracle.so")
_lock = threading.Lock()
_lib = None


def compile_to(src: str, lib: str) -> None:
    """gcc, plain IEEE double: no fast-math, no FMA contraction."""
    subprocess.check_call(["gcc", "-O2", "-std=c99", "-fopenmp", "-ffp-contract=off", "-fPIC",
                           "-shared", "-o", lib, src, "-lm"])


def build(force: bool = False) -> str:
    """Compile the oracle (once; again when the C source is newer).

    GMA_ORACLE_LIB, when set, names an already built library to load instead:
    the tests that plant a mistake in a copy of the oracle use it to run the
    pins against the mutated build."""
    override = os.environ.get("GMA_ORACLE_LIB")
    if override:
        return override
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        compile_to(_SRC, tmp)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i, dbl = ctypes.c_int, ctypes.c_double
            lib.gma_oracle_max_threads.restype = i
            lib.gma_oracle_set_threads.argtypes = [i]
            lib.gma_oracle_params.argtypes = [i, i, i, P, P, P, P]
            lib.gma_oracle_responsibilities.argtypes = [i, P, i, i, i, i, P, P, P, P, P]
            lib.gma_oracle_bidir.argtypes = [i, P, i, i, i, i, i, P, P, P, P, P, P, dbl, P]
            lib.gma_oracle_causal.argtypes = [i, P, i, i, i, i, i, P, P, P, P, P, P, dbl, P, P, P]
            lib.gma_oracle_write.argtypes = [i, P, i, i, i, i, i, P, P, P, P, P, P]
            lib.gma_oracle_read.argtypes = [i, P, i, i, i, i, i, P, P, P, P, P, dbl, P]
            lib.gma_oracle_decode_step.argtypes = [i, P, i, i, i, i, P, P, P, P, P, P, dbl, P, P]
            lib.gma_oracle_cross.argtypes = [i, P, i, i, i, i, i, i, P, P, P, P, P, P, dbl, P]
            lib.gma_oracle_usage.argtypes = [i, P, i, i, i, i, P, P, P, P, P, P, P, P]
            lib.gma_oracle_backward.argtypes = [i, P, i, i, i, i, i, i, P, P, P, P, P, P, dbl, P, P, P, P, P, P,
                                                P]
            _lib = lib
    return _lib


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _heads(S, H, heads):
    h = np.arange(S) % H if heads is None else np.asarray(heads)
    h = np.ascontiguousarray(h, dtype=np.int32)
    if h.shape != (S,) or (h < 0).any() or (h >= H).any():
        raise ValueError("heads must hold S head indices in [0, H)")
    return h


def max_threads() -> int:
    return _load().gma_oracle_max_threads()


def set_threads(n: int) -> None:
    _load().gma_oracle_set_threads(int(n))


def params(var_raw, logit_pi):
    """S0: (sigma^2 [H,K,d], log pi [H,K]) from raw variances and mixture logits."""
    vr, lp = _f64(var_raw), _f64(logit_pi)
    H, K, d = vr.shape
    var = np.empty_like(vr)
    log_pi = np.empty_like(lp)
    _load().gma_oracle_params(H, K, d, _p(vr), _p(lp), _p(var), _p(log_pi))
    return var, log_pi


def responsibilities(mu, var_raw, logit_pi, x, heads=None):
    """S1: gamma [S,n,K] = p(z=k | x) for routing rows x [S,n,d]."""
    mu, vr, lp, x = _f64(mu), _f64(var_raw), _f64(logit_pi), _f64(x)
    H, K, d = mu.shape
    S, n, _ = x.shape
    hs = _heads(S, H, heads)
    g = np.empty((S, n, K))
    _load().gma_oracle_responsibilities(S, _p(hs), H, n, d, K, _p(mu), _p(vr), _p(lp), _p(x), _p(g))
    return g


def write(mu, var_raw, logit_pi, kx, v, state=None, heads=None):
    """S2 alone: returns state + [Gamma_K^T V, Gamma_K^T 1] as [S, K*dv + K]."""
    mu, vr, lp = _f64(mu), _f64(var_raw), _f64(logit_pi)
    kx, v = _f64(kx), _f64(v)
    H, K, d = mu.shape
    S, n, dv = v.shape
    hs = _heads(S, H, heads)
    st = np.zeros((S, K * dv + K)) if state is None else _f64(state).reshape(S, K * dv + K).copy()
    _load().gma_oracle_write(S, _p(hs), H, n, d, dv, K, _p(mu), _p(vr), _p(lp), _p(kx), _p(v), _p(st))
    return st


def read(mu, var_raw, logit_pi, qx, state, eps, heads=None):
    """S3 alone: output [S,n,dv] of queries qx [S,n,d] reading the fixed state [S, K*dv + K]."""
    mu, vr, lp = _f64(mu), _f64(var_raw), _f64(logit_pi)
    qx = _f64(qx)
    H, K, d = mu.shape
    S, n, _ = qx.shape
    st = _f64(state).reshape(S, -1)
    dv = (st.shape[1] - K) // K
    hs = _heads(S, H, heads)
    out = np.empty((S, n, dv))
    _load().gma_oracle_read(S, _p(hs), H, n, d, dv, K, _p(mu), _p(vr), _p(lp), _p(qx), _p(st),
                            float(eps), _p(out))
    return out


def bidir(mu, var_raw, logit_pi, qx, kx, v, eps, heads=None):
    """S2+S3: bidirectional output [S,n,dv]."""
    mu, vr, lp = _f64(mu), _f64(var_raw), _f64(logit_pi)
    qx, kx, v = _f64(qx), _f64(kx), _f64(v)
    H, K, d = mu.shape
    S, n, dv = v.shape
    hs = _heads(S, H, heads)
    out = np.empty((S, n, dv))
    _load().gma_oracle_bidir(S, _p(hs), H, n, d, dv, K, _p(mu), _p(vr), _p(lp),
                             _p(qx), _p(kx), _p(v), float(eps), _p(out))
    return out


def causal(mu, var_raw, logit_pi, qx, kx, v, eps, heads=None, state_in=None, return_state=False):
    """S4: causal output [S,n,dv]; optionally also the final state [S, K*dv + K]."""
    mu, vr, lp = _f64(mu), _f64(var_raw), _f64(logit_pi)
    qx, kx, v = _f64(qx), _f64(kx), _f64(v)
    H, K, d = mu.shape
    S, n, dv = v.shape
    hs = _heads(S, H, heads)
    out = np.empty((S, n, dv))
    sin = None if state_in is None else _f64(state_in).reshape(S, K * dv + K)
    sout = np.empty((S, K * dv + K)) if return_state else None
    _load().gma_oracle_causal(S, _p(hs), H, n, d, dv, K, _p(mu), _p(vr), _p(lp),
                              _p(qx), _p(kx), _p(v), float(eps),
                              None if sin is None else _p(sin),
                              None if sout is None else _p(sout), _p(out))
    return (out, sout) if return_state else out


def decode_step(mu, var_raw, logit_pi, qx, kx, v, eps, state, heads=None):
    """S5: one decode step.  qx,kx [S,d], v [S,dv], state [S,K*dv+K] -> (out [S,dv], new state)."""
    mu, vr, lp = _f64(mu), _f64(var_raw), _f64(logit_pi)
    qx, kx, v = _f64(qx), _f64(kx), _f64(v)
    H, K, d = mu.shape
    S, dv = v.shape
    hs = _heads(S, H, heads)
    st = _f64(state).reshape(S, K * dv + K).copy()
    out = np.empty((S, dv))
    _load().gma_oracle_decode_step(S, _p(hs), H, d, dv, K, _p(mu), _p(vr), _p(lp),
                                   _p(qx), _p(kx), _p(v), float(eps), _p(st), _p(out))
    return out, st


def cross(mu, var_raw, logit_pi, qx, kx, v, eps, heads=None):
    """Cross-attention: queries qx [S,nq,d] read the memory written by kx [S,nk,d], v [S,nk,dv]."""
    mu, vr, lp = _f64(mu), _f64(var_raw), _f64(logit_pi)
    qx, kx, v = _f64(qx), _f64(kx), _f64(v)
    H, K, d = mu.shape
    S, nq, _ = qx.shape
    _, nk, dv = v.shape
    if kx.shape[:2] != (S, nk):
        raise ValueError("kx and v must hold the same key rows")
    hs = _heads(S, H, heads)
    out = np.empty((S, nq, dv))
    _load().gma_oracle_cross(S, _p(hs), H, nq, nk, d, dv, K, _p(mu), _p(vr), _p(lp),
                             _p(qx), _p(kx), _p(v), float(eps), _p(out))
    return out


def usage(mu, var_raw, logit_pi, x, heads=None):
    """Responsibility diagnostics of routing rows x [S,n,d], per head:
    (usage [H,K] soft sums, counts [H,K] hard-assignment counts (int64),
     assign [S,n] argmax per row (int32), entropy [H,2]: soft, hard, divided by log K)."""
    mu, vr, lp, x = _f64(mu), _f64(var_raw), _f64(logit_pi), _f64(x)
    H, K, d = mu.shape
    S, n, _ = x.shape
    hs = _heads(S, H, heads)
    u = np.empty((H, K))
    c = np.empty((H, K), dtype=np.int64)
    a = np.empty((S, n), dtype=np.int32)
    e = np.empty((H, 2))
    _load().gma_oracle_usage(S, _p(hs), H, n, d, K, _p(mu), _p(vr), _p(lp), _p(x), _p(u), _p(c), _p(a), _p(e))
    return u, c, a, e


def backward(mu, var_raw, logit_pi, qx, kx, v, eps, dout, causal=True, heads=None):
    """Gradients of the causal (or bidirectional) forward given dL/dO = dout [S,n,dv]:
    (dqx [S,n,d], dkx [S,n,d], dv [S,n,dv], dmu [H,K,d], dvar_raw [H,K,d], dlogit_pi [H,K]);
    the parameter gradients sum over the slices of each head and both routings."""
    mu, vr, lp = _f64(mu), _f64(var_raw), _f64(logit_pi)
    qx, kx, v, g = _f64(qx), _f64(kx), _f64(v), _f64(dout)
    H, K, d = mu.shape
    S, n, dv = v.shape
    hs = _heads(S, H, heads)
    dq, dk, dvv = np.empty((S, n, d)), np.empty((S, n, d)), np.empty((S, n, dv))
    dmu, dvr, dlp = np.empty((H, K, d)), np.empty((H, K, d)), np.empty((H, K))
    _load().gma_oracle_backward(S, _p(hs), H, n, d, dv, K, int(bool(causal)), _p(mu), _p(vr), _p(lp),
                                _p(qx), _p(kx), _p(v), float(eps), _p(g), _p(dq), _p(dk), _p(dvv),
                                _p(dmu), _p(dvr), _p(dlp))
    return dq, dk, dvv, dmu, dvr, dlp
