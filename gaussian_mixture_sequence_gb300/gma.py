"""Python binding of libgma (argument marshalling only).

Every function here has the name of the C entry point it calls (declared in
include/gma.h) and does nothing but check that the torch tensors it is given
match the declared layout, take their device pointers and the current CUDA
stream, and call the library.  All arithmetic happens in the library's CUDA
kernels.  There is no fallback: if ``libgma.so`` has not been built, or if the
library reports an error, these functions raise.

Workspace: when ``ws`` is not given, a uint8 tensor of
``gma_workspace_size`` bytes is taken from torch's caching allocator on the
tensors' device (memory plumbing, not computation).
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libgma.so")
_lib = None

F32, BF16 = 0, 1
OP_RESPONSIBILITIES, OP_BIDIR, OP_CAUSAL, OP_DECODE, OP_CAUSAL_HOST, OP_USAGE, OP_BACKWARD = 0, 1, 2, 3, 4, 5, 6
_DT = {"f32": F32, "bf16": BF16, torch.float32: F32, torch.bfloat16: BF16}
_TORCH_DT = {F32: torch.float32, BF16: torch.bfloat16}


class GMAError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn}: {msg} (status {status})")
        self.status = status


class Shape(ctypes.Structure):
    """Mirror of ``gma_shape``."""
    _fields_ = [("B", ctypes.c_int), ("H", ctypes.c_int), ("N", ctypes.c_int),
                ("d_route", ctypes.c_int), ("d_v", ctypes.c_int), ("K", ctypes.c_int),
                ("chunk", ctypes.c_int), ("eps", ctypes.c_float), ("x_dtype", ctypes.c_int),
                ("v_dtype", ctypes.c_int), ("gemm_dtype", ctypes.c_int)]

    @classmethod
    def make(cls, B, H, N, d_route, d_v, K, chunk=0, eps=1e-6, x_dtype="f32", v_dtype="f32",
             gemm_dtype="f32"):
        return cls(B, H, N, d_route, d_v, K, chunk, eps, _DT[x_dtype], _DT[v_dtype], _DT[gemm_dtype])


PROFILE_MAX_STAGES = 8


class Profile(ctypes.Structure):
    """Mirror of ``gma_profile``."""
    _fields_ = [("events", ctypes.c_void_p * (PROFILE_MAX_STAGES + 1)), ("n_stages", ctypes.c_int),
                ("stage_name", ctypes.c_char_p * PROFILE_MAX_STAGES)]


class _Params(ctypes.Structure):
    _fields_ = [("mu", ctypes.c_void_p), ("var_raw", ctypes.c_void_p), ("logit_pi", ctypes.c_void_p)]


def library_path() -> str:
    return _LIB_PATH


def load():
    """The loaded ctypes library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"{_LIB_PATH} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(_LIB_PATH)
        P, S = ctypes.c_void_p, ctypes.POINTER(Shape)
        lib.gma_workspace_size.argtypes = [S, ctypes.c_int]
        lib.gma_workspace_size.restype = ctypes.c_size_t
        lib.gma_status_string.argtypes = [ctypes.c_int]
        lib.gma_status_string.restype = ctypes.c_char_p
        lib.gma_last_cuda_error.argtypes = []
        lib.gma_last_cuda_error.restype = ctypes.c_char_p
        lib.gma_responsibilities.argtypes = [S, _Params, P, P, P, ctypes.c_size_t, P]
        lib.gma_forward_bidir.argtypes = [S, _Params, P, P, P, P, P, ctypes.c_size_t, P]
        lib.gma_forward_causal.argtypes = [S, _Params, P, P, P, P, P, P, P, ctypes.c_size_t, P]
        lib.gma_forward_causal_host.argtypes = [S, _Params, P, P, P, P, P, P, P, ctypes.c_size_t, P]
        lib.gma_decode_step.argtypes = [S, _Params, P, P, P, P, P, P, ctypes.c_size_t, P]
        lib.gma_decode_step_noalloc.argtypes = [S, _Params, P, P, P, P, P, P]
        lib.gma_forward_causal_profiled.argtypes = [S, _Params, P, P, P, P, P, P, P, ctypes.c_size_t, P,
                                                    ctypes.POINTER(Profile)]
        lib.gma_forward_bidir_profiled.argtypes = [S, _Params, P, P, P, P, P, ctypes.c_size_t, P,
                                                   ctypes.POINTER(Profile)]
        lib.gma_decode_step_profiled.argtypes = [S, _Params, P, P, P, P, P, P, ctypes.c_size_t, P,
                                                 ctypes.POINTER(Profile)]
        lib.gma_responsibility_stats.argtypes = [S, _Params, P, P, P, P, P, P, ctypes.c_size_t, P]
        lib.gma_cross_workspace_size.argtypes = [S, ctypes.c_int]
        lib.gma_cross_workspace_size.restype = ctypes.c_size_t
        lib.gma_forward_cross.argtypes = [S, ctypes.c_int, _Params, P, P, P, P, P, ctypes.c_size_t, P]
        lib.gma_backward.argtypes = [S, ctypes.c_int, _Params, P, P, P, P, P, P, P, P, P, P, P, ctypes.c_size_t, P]
        lib.gma_sync_status.argtypes = [P]
        lib.gma_test_wait_timeout.argtypes = [ctypes.c_longlong, P]
        for fn in ("gma_backward", "gma_responsibility_stats", "gma_forward_cross", "gma_sync_status",
                   "gma_test_wait_timeout", "gma_responsibilities", "gma_forward_bidir", "gma_forward_causal", "gma_decode_step",
                   "gma_forward_causal_host", "gma_forward_causal_profiled", "gma_decode_step_noalloc",
                   "gma_forward_bidir_profiled", "gma_decode_step_profiled"):
            getattr(lib, fn).restype = ctypes.c_int
        _lib = lib
    return _lib


def gma_status_string(status: int) -> str:
    return load().gma_status_string(int(status)).decode()


def gma_workspace_size(shape: Shape, op: int) -> int:
    return int(load().gma_workspace_size(ctypes.byref(shape), int(op)))


def _check(fn, status):
    if status != 0:
        msg = gma_status_string(status)
        if status == 5:
            msg += " (" + load().gma_last_cuda_error().decode() + ")"
        raise GMAError(fn, status, msg)


def _ptr(t, name, shape=None, dtype=None, device=None, optional=False):
    if t is None:
        if optional:
            return None
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.numel() == 0:
        return None
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    return t.data_ptr()


def _params(shape, mu, var_raw, logit_pi, dev):
    H, K, D = shape.H, shape.K, shape.d_route
    return _Params(_ptr(mu, "mu", (H, K, D), torch.float32, dev),
                   _ptr(var_raw, "var_raw", (H, K, D), torch.float32, dev),
                   _ptr(logit_pi, "logit_pi", (H, K), torch.float32, dev))


def _ws(shape, op, ws, dev):
    need = gma_workspace_size(shape, op)
    if ws is None:
        ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    return _ptr(ws, "ws", dtype=torch.uint8, device=dev), ws.numel()


def _stream(dev, stream):
    s = torch.cuda.current_stream(dev) if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def gma_responsibilities(shape: Shape, mu, var_raw, logit_pi, x, gamma, ws=None, stream=None):
    """gamma [B,H,N,K] (fp32) <- posterior responsibilities of routing rows x [B,H,N,d_route]."""
    dev = x.device
    s = shape
    xp = _ptr(x, "x", (s.B, s.H, s.N, s.d_route), _TORCH_DT[s.x_dtype], dev)
    gp = _ptr(gamma, "gamma", (s.B, s.H, s.N, s.K), torch.float32, dev)
    prm = _params(s, mu, var_raw, logit_pi, dev)
    wp, wn = _ws(s, OP_RESPONSIBILITIES, ws, dev)
    _check("gma_responsibilities",
           load().gma_responsibilities(ctypes.byref(s), prm, xp, gp, wp, wn, _stream(dev, stream)))
    return gamma


def gma_responsibility_stats(shape: Shape, mu, var_raw, logit_pi, x, usage, counts, entropy, assign=None,
                             ws=None, stream=None):
    """Per-head diagnostics of the responsibilities of routing rows x [B,H,N,d_route]:
    usage [H,K] fp32 (soft sums), counts [H,K] int64 (hard assignments), entropy [H,2]
    fp32 (normalised entropies of usage and counts), assign [B,H,N] int32 (optional)."""
    dev = x.device
    s = shape
    xp = _ptr(x, "x", (s.B, s.H, s.N, s.d_route), _TORCH_DT[s.x_dtype], dev)
    up = _ptr(usage, "usage", (s.H, s.K), torch.float32, dev)
    cp = _ptr(counts, "counts", (s.H, s.K), torch.int64, dev)
    ep = _ptr(entropy, "entropy", (s.H, 2), torch.float32, dev)
    ap = _ptr(assign, "assign", (s.B, s.H, s.N), torch.int32, dev, optional=True)
    prm = _params(s, mu, var_raw, logit_pi, dev)
    wp, wn = _ws(s, OP_USAGE, ws, dev)
    _check("gma_responsibility_stats",
           load().gma_responsibility_stats(ctypes.byref(s), prm, xp, up, cp, ep, ap, wp, wn, _stream(dev, stream)))
    return usage, counts, entropy


def gma_backward(shape: Shape, mu, var_raw, logit_pi, qx, kx, v, dout, dqx, dkx, dv, dmu, dvar_raw, dlogit_pi,
                 causal=True, ws=None, stream=None):
    """Gradients of the causal (or bidirectional) forward given dout = dL/dO [B,H,N,d_v] (fp32):
    dqx, dkx [B,H,N,d_route], dv [B,H,N,d_v], dmu, dvar_raw [H,K,d_route], dlogit_pi [H,K], all fp32."""
    dev = qx.device
    s = shape
    f32 = torch.float32
    q, k, vv, _ = _fwd_ptrs(s, qx, kx, v, dout, dev)
    g = _ptr(dout, "dout", (s.B, s.H, s.N, s.d_v), f32, dev)
    dq = _ptr(dqx, "dqx", (s.B, s.H, s.N, s.d_route), f32, dev)
    dk = _ptr(dkx, "dkx", (s.B, s.H, s.N, s.d_route), f32, dev)
    dvp = _ptr(dv, "dv", (s.B, s.H, s.N, s.d_v), f32, dev)
    dm = _ptr(dmu, "dmu", (s.H, s.K, s.d_route), f32, dev)
    dr = _ptr(dvar_raw, "dvar_raw", (s.H, s.K, s.d_route), f32, dev)
    dl = _ptr(dlogit_pi, "dlogit_pi", (s.H, s.K), f32, dev)
    prm = _params(s, mu, var_raw, logit_pi, dev)
    wp, wn = _ws(s, OP_BACKWARD, ws, dev)
    _check("gma_backward",
           load().gma_backward(ctypes.byref(s), int(bool(causal)), prm, q, k, vv, g, dq, dk, dvp, dm, dr, dl, wp, wn,
                               _stream(dev, stream)))
    return dqx, dkx, dv, dmu, dvar_raw, dlogit_pi


def gma_cross_workspace_size(shape: Shape, n_kv: int) -> int:
    return int(load().gma_cross_workspace_size(ctypes.byref(shape), int(n_kv)))


def gma_forward_cross(shape: Shape, mu, var_raw, logit_pi, qx, kx, v, out, ws=None, stream=None):
    """out [B,H,N,d_v]: queries qx [B,H,N,d_route] read the memory written by kx
    [B,H,n_kv,d_route] and v [B,H,n_kv,d_v] (n_kv taken from kx)."""
    dev = qx.device
    s = shape
    xdt, vdt = _TORCH_DT[s.x_dtype], _TORCH_DT[s.v_dtype]
    n_kv = kx.shape[2]
    q = _ptr(qx, "qx", (s.B, s.H, s.N, s.d_route), xdt, dev)
    k = _ptr(kx, "kx", (s.B, s.H, n_kv, s.d_route), xdt, dev)
    vv = _ptr(v, "v", (s.B, s.H, n_kv, s.d_v), vdt, dev)
    o = _ptr(out, "out", (s.B, s.H, s.N, s.d_v), torch.float32, dev)
    prm = _params(s, mu, var_raw, logit_pi, dev)
    need = gma_cross_workspace_size(s, n_kv)
    if ws is None:
        ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    wp = _ptr(ws, "ws", dtype=torch.uint8, device=dev)
    _check("gma_forward_cross",
           load().gma_forward_cross(ctypes.byref(s), n_kv, prm, q, k, vv, o, wp, ws.numel(), _stream(dev, stream)))
    return out


def _fwd_ptrs(s, qx, kx, v, out, dev):
    xdt, vdt = _TORCH_DT[s.x_dtype], _TORCH_DT[s.v_dtype]
    return (_ptr(qx, "qx", (s.B, s.H, s.N, s.d_route), xdt, dev),
            _ptr(kx, "kx", (s.B, s.H, s.N, s.d_route), xdt, dev),
            _ptr(v, "v", (s.B, s.H, s.N, s.d_v), vdt, dev),
            _ptr(out, "out", (s.B, s.H, s.N, s.d_v), torch.float32, dev))


def gma_forward_bidir(shape: Shape, mu, var_raw, logit_pi, qx, kx, v, out, ws=None, stream=None):
    """out [B,H,N,d_v] <- Gamma_Q Vt / (Gamma_Q Z + eps) with Vt, Z written by all N keys."""
    dev = qx.device
    q, k, vv, o = _fwd_ptrs(shape, qx, kx, v, out, dev)
    prm = _params(shape, mu, var_raw, logit_pi, dev)
    wp, wn = _ws(shape, OP_BIDIR, ws, dev)
    _check("gma_forward_bidir",
           load().gma_forward_bidir(ctypes.byref(shape), prm, q, k, vv, o, wp, wn, _stream(dev, stream)))
    return out


def gma_forward_causal(shape: Shape, mu, var_raw, logit_pi, qx, kx, v, out, state_in=None,
                       state_out=None, ws=None, stream=None):
    """out [B,H,N,d_v]: causal form; optional state_in / state_out [B,H,K*d_v+K] (fp32)."""
    dev = qx.device
    s = shape
    q, k, vv, o = _fwd_ptrs(s, qx, kx, v, out, dev)
    sshape = (s.B, s.H, s.K * s.d_v + s.K)
    si = _ptr(state_in, "state_in", sshape, torch.float32, dev, optional=True)
    so = _ptr(state_out, "state_out", sshape, torch.float32, dev, optional=True)
    prm = _params(s, mu, var_raw, logit_pi, dev)
    wp, wn = _ws(s, OP_CAUSAL, ws, dev)
    _check("gma_forward_causal",
           load().gma_forward_causal(ctypes.byref(s), prm, q, k, vv, si, so, o, wp, wn, _stream(dev, stream)))
    return out


def _host_ptr(t, name, shape, dtype):
    if not isinstance(t, torch.Tensor) or t.is_cuda:
        raise TypeError(f"{name} must be a host (CPU) tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if t.dtype != dtype:
        raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")
    return ctypes.c_void_p(t.data_ptr()) if t.numel() else None


def gma_forward_causal_host(shape: Shape, mu, var_raw, logit_pi, qx, kx, v, out, state_in=None,
                            state_out=None, ws=None, stream=None):
    """gma_forward_causal on host tensors qx, kx, v, out (page-locked for asynchronous copies);
    the library copies in and out itself, overlapping the copies with the computation.
    Parameters and the optional states are device tensors.  Returns after enqueueing."""
    dev = mu.device
    s = shape
    xdt, vdt = _TORCH_DT[s.x_dtype], _TORCH_DT[s.v_dtype]
    q = _host_ptr(qx, "qx", (s.B, s.H, s.N, s.d_route), xdt)
    k = _host_ptr(kx, "kx", (s.B, s.H, s.N, s.d_route), xdt)
    vv = _host_ptr(v, "v", (s.B, s.H, s.N, s.d_v), vdt)
    o = _host_ptr(out, "out", (s.B, s.H, s.N, s.d_v), torch.float32)
    sshape = (s.B, s.H, s.K * s.d_v + s.K)
    si = _ptr(state_in, "state_in", sshape, torch.float32, dev, optional=True)
    so = _ptr(state_out, "state_out", sshape, torch.float32, dev, optional=True)
    prm = _params(s, mu, var_raw, logit_pi, dev)
    wp, wn = _ws(s, OP_CAUSAL_HOST, ws, dev)
    _check("gma_forward_causal_host",
           load().gma_forward_causal_host(ctypes.byref(s), prm, q, k, vv, si, so, o, wp, wn, _stream(dev, stream)))
    return out


def gma_forward_causal_profiled(shape: Shape, mu, var_raw, logit_pi, qx, kx, v, out, events,
                                state_in=None, state_out=None, ws=None, stream=None):
    """gma_forward_causal with a CUDA event recorded before every launch and after the last.

    ``events`` holds PROFILE_MAX_STAGES + 1 timing-enabled ``torch.cuda.Event``
    objects that have been recorded at least once (so that they exist).
    Returns the names of the launches; events[i] precedes launch i."""
    dev = qx.device
    s = shape
    q, k, vv, o = _fwd_ptrs(s, qx, kx, v, out, dev)
    sshape = (s.B, s.H, s.K * s.d_v + s.K)
    si = _ptr(state_in, "state_in", sshape, torch.float32, dev, optional=True)
    so = _ptr(state_out, "state_out", sshape, torch.float32, dev, optional=True)
    prm = _params(s, mu, var_raw, logit_pi, dev)
    wp, wn = _ws(s, OP_CAUSAL, ws, dev)
    prof = _profile(events)
    _check("gma_forward_causal_profiled",
           load().gma_forward_causal_profiled(ctypes.byref(s), prm, q, k, vv, si, so, o, wp, wn,
                                              _stream(dev, stream), ctypes.byref(prof)))
    return [prof.stage_name[i].decode() for i in range(prof.n_stages)]


def _profile(events):
    if len(events) != PROFILE_MAX_STAGES + 1:
        raise ValueError(f"need {PROFILE_MAX_STAGES + 1} events")
    prof = Profile()
    for i, e in enumerate(events):
        prof.events[i] = e.cuda_event
    return prof


def gma_forward_bidir_profiled(shape: Shape, mu, var_raw, logit_pi, qx, kx, v, out, events, ws=None,
                               stream=None):
    """gma_forward_bidir with CUDA events around every launch (see gma_forward_causal_profiled)."""
    dev = qx.device
    q, k, vv, o = _fwd_ptrs(shape, qx, kx, v, out, dev)
    prm = _params(shape, mu, var_raw, logit_pi, dev)
    wp, wn = _ws(shape, OP_BIDIR, ws, dev)
    prof = _profile(events)
    _check("gma_forward_bidir_profiled",
           load().gma_forward_bidir_profiled(ctypes.byref(shape), prm, q, k, vv, o, wp, wn,
                                             _stream(dev, stream), ctypes.byref(prof)))
    return [prof.stage_name[i].decode() for i in range(prof.n_stages)]


def gma_decode_step_profiled(shape: Shape, mu, var_raw, logit_pi, qx, kx, v, state, out, events, ws=None,
                             stream=None):
    """gma_decode_step with CUDA events around every launch (see gma_forward_causal_profiled)."""
    dev = qx.device
    s = shape
    xdt, vdt = _TORCH_DT[s.x_dtype], _TORCH_DT[s.v_dtype]
    q = _ptr(qx, "qx", (s.B, s.H, s.d_route), xdt, dev)
    k = _ptr(kx, "kx", (s.B, s.H, s.d_route), xdt, dev)
    vv = _ptr(v, "v", (s.B, s.H, s.d_v), vdt, dev)
    st = _ptr(state, "state", (s.B, s.H, s.K * s.d_v + s.K), torch.float32, dev)
    o = _ptr(out, "out", (s.B, s.H, s.d_v), torch.float32, dev)
    prm = _params(s, mu, var_raw, logit_pi, dev)
    wp, wn = _ws(s, OP_DECODE, ws, dev)
    prof = _profile(events)
    _check("gma_decode_step_profiled",
           load().gma_decode_step_profiled(ctypes.byref(s), prm, q, k, vv, st, o, wp, wn, _stream(dev, stream),
                                           ctypes.byref(prof)))
    return [prof.stage_name[i].decode() for i in range(prof.n_stages)]


def gma_decode_step(shape: Shape, mu, var_raw, logit_pi, qx, kx, v, state, out, ws=None, stream=None):
    """One decode token per (b, h): state [B,H,K*d_v+K] updated in place, out [B,H,d_v]."""
    dev = qx.device
    s = shape
    xdt, vdt = _TORCH_DT[s.x_dtype], _TORCH_DT[s.v_dtype]
    q = _ptr(qx, "qx", (s.B, s.H, s.d_route), xdt, dev)
    k = _ptr(kx, "kx", (s.B, s.H, s.d_route), xdt, dev)
    vv = _ptr(v, "v", (s.B, s.H, s.d_v), vdt, dev)
    st = _ptr(state, "state", (s.B, s.H, s.K * s.d_v + s.K), torch.float32, dev)
    o = _ptr(out, "out", (s.B, s.H, s.d_v), torch.float32, dev)
    prm = _params(s, mu, var_raw, logit_pi, dev)
    wp, wn = _ws(s, OP_DECODE, ws, dev)
    _check("gma_decode_step",
           load().gma_decode_step(ctypes.byref(s), prm, q, k, vv, st, o, wp, wn, _stream(dev, stream)))
    return out


NOALLOC_SCRATCH_BYTES = 8 << 20


def gma_decode_step_noalloc(shape: Shape, mu, var_raw, logit_pi, qx, kx, v, state, out, stream=None):
    """gma_decode_step without a workspace: for callers that cannot allocate
    device memory.  The library keeps the step's scratch in a fixed device
    array of NOALLOC_SCRATCH_BYTES on every GPU that loads it; shapes that
    need more raise GMAError (status 4).  Calls must not overlap on the GPU."""
    dev = qx.device
    s = shape
    xdt, vdt = _TORCH_DT[s.x_dtype], _TORCH_DT[s.v_dtype]
    q = _ptr(qx, "qx", (s.B, s.H, s.d_route), xdt, dev)
    k = _ptr(kx, "kx", (s.B, s.H, s.d_route), xdt, dev)
    vv = _ptr(v, "v", (s.B, s.H, s.d_v), vdt, dev)
    st = _ptr(state, "state", (s.B, s.H, s.K * s.d_v + s.K), torch.float32, dev)
    o = _ptr(out, "out", (s.B, s.H, s.d_v), torch.float32, dev)
    prm = _params(s, mu, var_raw, logit_pi, dev)
    _check("gma_decode_step_noalloc",
           load().gma_decode_step_noalloc(ctypes.byref(s), prm, q, k, vv, st, o, _stream(dev, stream)))
    return out


TIMEOUT = 6


def gma_sync_status(device=None, stream=None):
    """Waits for the stream (default: the current stream of `device`, default the
    current device), then raises GMAError (status 6) if a bounded wait inside one of
    the library's kernels expired on that device since the last report."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    _check("gma_sync_status", load().gma_sync_status(_stream(dev, stream)))


def gma_test_wait_timeout(limit_cycles: int, device=None, stream=None):
    """Enqueues the library's test kernel whose one bounded wait expires after
    limit_cycles SM cycles (nothing is in flight when it gives up)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    _check("gma_test_wait_timeout", load().gma_test_wait_timeout(int(limit_cycles), _stream(dev, stream)))
