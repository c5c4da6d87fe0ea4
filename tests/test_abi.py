"""The C ABI without a GPU: the library loads, exports every declared entry
point, and rejects bad arguments on the host before touching CUDA."""
import ctypes
import os
import re

import pytest

from gaussian_mixture_sequence_gb300 import build as gbuild
from gaussian_mixture_sequence_gb300 import gma

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    gbuild.build()
    return gma.load()


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(gma_\w+)\s*\(", text))
    return names


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert {"gma_responsibilities", "gma_forward_bidir", "gma_forward_causal", "gma_decode_step",
            "gma_workspace_size", "gma_status_string"} <= names
    for n in sorted(names):
        assert hasattr(lib, n), f"libgma.so does not export {n}"


def test_status_strings(lib):
    for code in range(7):
        assert gma.gma_status_string(code) and gma.gma_status_string(code) != "unknown status"
    assert gma.gma_status_string(99) == "unknown status"


def _shape(**kw):
    base = dict(B=2, H=3, N=100, d_route=64, d_v=64, K=128)
    base.update(kw)
    return gma.Shape.make(**base)


def test_workspace_size(lib):
    s = _shape()
    for op in range(4):
        assert gma.gma_workspace_size(s, op) > 0
    assert gma.gma_workspace_size(_shape(d_route=48), gma.OP_CAUSAL) == 0
    assert gma.gma_workspace_size(_shape(K=513), gma.OP_CAUSAL) == 0
    assert gma.gma_workspace_size(s, 7) == 0
    # bf16 product operands halve the responsibility scratch
    f = gma.gma_workspace_size(_shape(N=4096), gma.OP_CAUSAL)
    b = gma.gma_workspace_size(_shape(N=4096, gemm_dtype="bf16"), gma.OP_CAUSAL)
    assert b < f


FAKE = 1 << 20  # aligned, never dereferenced: validation fails before any launch


def _call_causal(lib, shape, ptrs=None, ws_bytes=1 << 40):
    p = dict(mu=FAKE, var=FAKE, lp=FAKE, q=FAKE, k=FAKE, v=FAKE, si=None, so=None, o=FAKE, ws=FAKE)
    p.update(ptrs or {})
    prm = gma._Params(p["mu"], p["var"], p["lp"])
    sp = ctypes.byref(shape) if shape is not None else None
    return lib.gma_forward_causal(sp, prm, p["q"], p["k"], p["v"], p["si"], p["so"], p["o"], p["ws"],
                                  ws_bytes, None)


@pytest.mark.parametrize("kw,status", [
    (dict(d_route=48), 2), (dict(d_v=8), 2), (dict(K=600), 2), (dict(chunk=48), 2),
    (dict(K=200, chunk=128), 2), (dict(K=640, chunk=128), 2), (dict(d_v=128, chunk=128), 2),
    (dict(B=0), 1), (dict(N=-1), 1), (dict(K=0), 1), (dict(eps=-1.0), 1), (dict(eps=float("nan")), 1),
    (dict(B=300, H=300), 2),
])
def test_rejects_bad_shapes(lib, kw, status):
    assert _call_causal(lib, _shape(**kw)) == status


def test_rejects_bad_pointers_and_workspace(lib):
    s = _shape()
    assert _call_causal(lib, None) == 1
    assert _call_causal(lib, s, dict(q=None)) == 1
    assert _call_causal(lib, s, dict(mu=None)) == 1
    assert _call_causal(lib, s, dict(q=FAKE + 4)) == 3
    assert _call_causal(lib, s, dict(si=FAKE + 8)) == 3
    assert _call_causal(lib, s, dict(ws=None)) == 4
    need = gma.gma_workspace_size(s, gma.OP_CAUSAL)
    assert _call_causal(lib, s, ws_bytes=need - 1) == 4
    bad = gma.Shape.make(2, 3, 100, 64, 64, 128)
    bad.x_dtype = 5
    assert _call_causal(lib, bad) == 1


def test_host_entry_workspace_and_validation(lib):
    s = _shape(N=4096)
    # the host-buffer entry's scratch holds device copies of q, k, v and out, then the causal workspace
    need = gma.gma_workspace_size(s, gma.OP_CAUSAL_HOST)
    stage = 2 * 3 * 4096 * (2 * 64 * 4 + 64 * 4 + 64 * 4)   # B * H * N rows of q, k, v, out (fp32)
    assert need == gma.gma_workspace_size(s, gma.OP_CAUSAL) + stage
    prm = gma._Params(FAKE, FAKE, FAKE)
    call = lambda **kw: lib.gma_forward_causal_host(
        ctypes.byref(s), prm, kw.get("q", FAKE), kw.get("k", FAKE), kw.get("v", FAKE), None, None,
        kw.get("o", FAKE), kw.get("ws", FAKE), kw.get("wn", need), None)
    assert call(q=None) == 1
    assert call(o=None) == 1
    assert call(ws=None) == 4
    assert call(wn=need - 1) == 4
    assert call(ws=FAKE + 8) == 3
    assert lib.gma_last_cuda_error() == b"cudaSuccess"


def test_empty_sequence_is_a_no_op(lib):
    # N = 0: nothing to launch for the bidirectional form
    s = _shape(N=0)
    prm = gma._Params(FAKE, FAKE, FAKE)
    assert lib.gma_forward_bidir(ctypes.byref(s), prm, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 30, None) == 0
    assert lib.gma_responsibilities(ctypes.byref(s), prm, FAKE, FAKE, FAKE, 1 << 30, None) == 0


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(gma, "_lib", None)
    monkeypatch.setattr(gma, "_LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        gma.load()


def _prm():
    return gma._Params(FAKE, FAKE, FAKE)


def test_bidir_validation(lib):
    s = _shape(N=300)
    need = gma.gma_workspace_size(s, gma.OP_BIDIR)
    call = lambda shape=s, q=FAKE, k=FAKE, v=FAKE, o=FAKE, ws=FAKE, wn=need: lib.gma_forward_bidir(
        ctypes.byref(shape) if shape is not None else None, _prm(), q, k, v, o, ws, wn, None)
    assert call(shape=None) == 1
    assert call(q=None) == 1 and call(k=None) == 1 and call(v=None) == 1 and call(o=None) == 1
    assert call(v=FAKE + 4) == 3 and call(o=FAKE + 8) == 3
    assert call(ws=None) == 4 and call(wn=need - 1) == 4
    assert call(shape=_shape(d_route=48)) == 2 and call(shape=_shape(K=513)) == 2
    assert call(shape=_shape(eps=float("inf"))) == 1
    bad = gma._Params(FAKE, None, FAKE)
    assert lib.gma_forward_bidir(ctypes.byref(s), bad, FAKE, FAKE, FAKE, FAKE, FAKE, need, None) == 1
    bad = gma._Params(FAKE, FAKE, FAKE + 4)
    assert lib.gma_forward_bidir(ctypes.byref(s), bad, FAKE, FAKE, FAKE, FAKE, FAKE, need, None) == 3


def test_decode_validation(lib):
    s = _shape(B=4, N=0)
    need = gma.gma_workspace_size(s, gma.OP_DECODE)
    assert need > 0
    call = lambda q=FAKE, k=FAKE, v=FAKE, st=FAKE, o=FAKE, ws=FAKE, wn=need: lib.gma_decode_step(
        ctypes.byref(s), _prm(), q, k, v, st, o, ws, wn, None)
    # every pointer is required (one token per sequence, whatever N says)
    for kw in ("q", "k", "v", "st", "o"):
        assert call(**{kw: None}) == 1, kw
        assert call(**{kw: FAKE + 4}) == 3, kw
    assert call(ws=None) == 4 and call(wn=need - 1) == 4
    # the decode step's scratch holds only the prepared parameters: packed {1/sigma, -mu/sigma}
    # (16 bytes per component and feature pair) and c_k, each rounded up to 256 bytes
    up = lambda n: -(-n // 256) * 256
    assert need == up(s.H * s.K * (s.d_route // 2) * 16) + up(s.H * s.K * 4)


def test_responsibilities_validation(lib):
    s = _shape(N=300)
    need = gma.gma_workspace_size(s, gma.OP_RESPONSIBILITIES)
    call = lambda x=FAKE, g=FAKE, ws=FAKE, wn=need: lib.gma_responsibilities(
        ctypes.byref(s), _prm(), x, g, ws, wn, None)
    assert call(x=None) == 1 and call(g=None) == 1
    assert call(x=FAKE + 2) == 3 and call(g=FAKE + 12) == 3
    assert call(ws=None) == 4 and call(wn=need - 1) == 4
    # the caller's Gamma is the output: the scratch is smaller than a forward's
    assert need < gma.gma_workspace_size(s, gma.OP_CAUSAL)


def test_profiled_entries_need_a_profile(lib):
    s = _shape(N=300)
    wn = 1 << 40
    assert lib.gma_forward_causal_profiled(ctypes.byref(s), _prm(), FAKE, FAKE, FAKE, None, None, FAKE,
                                           FAKE, wn, None, None) == 1
    assert lib.gma_forward_bidir_profiled(ctypes.byref(s), _prm(), FAKE, FAKE, FAKE, FAKE, FAKE, wn, None,
                                          None) == 1
    assert lib.gma_decode_step_profiled(ctypes.byref(s), _prm(), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, wn,
                                        None, None) == 1
    # a profile whose events are missing is rejected before anything is recorded
    prof = gma.Profile()
    assert lib.gma_forward_causal_profiled(ctypes.byref(s), _prm(), FAKE, FAKE, FAKE, None, None, FAKE,
                                           FAKE, wn, None, ctypes.byref(prof)) == 1


def test_binding_refuses_host_tensors():
    """No CPU fallback: the device entries take CUDA tensors only, and say so before any call."""
    import torch
    s = _shape(B=1, H=1, N=8, d_route=64, d_v=64, K=128)
    x = torch.zeros(1, 1, 8, 64)
    o = torch.zeros(1, 1, 8, 64)
    p = (torch.zeros(1, 128, 64), torch.zeros(1, 128, 64), torch.zeros(1, 128))
    for call in (lambda: gma.gma_forward_causal(s, *p, x, x, x, o),
                 lambda: gma.gma_forward_bidir(s, *p, x, x, x, o),
                 lambda: gma.gma_responsibilities(s, *p, x, torch.zeros(1, 1, 8, 128))):
        with pytest.raises(TypeError, match="CUDA tensor"):
            call()


def test_timeout_hooks_validate_on_the_host(lib):
    """The timeout test hook rejects limits outside [1, 4e9] before any launch."""
    assert lib.gma_test_wait_timeout(0, None) == 1
    assert lib.gma_test_wait_timeout(-5, None) == 1
    assert lib.gma_test_wait_timeout(4000000001, None) == 1
    assert gma.gma_status_string(gma.TIMEOUT) == "a bounded device wait expired"


def test_cross_validation(lib):
    """Cross-attention: host-side checks of the key length, pointers and workspace."""
    s = _shape(N=300)
    need = gma.gma_cross_workspace_size(s, 1000)
    assert need > gma.gma_cross_workspace_size(s, 100) > 0
    assert gma.gma_cross_workspace_size(s, -1) == 0
    assert gma.gma_cross_workspace_size(_shape(d_route=48), 10) == 0
    # equal lengths: the bidirectional workspace
    assert gma.gma_cross_workspace_size(s, 300) == gma.gma_workspace_size(s, gma.OP_BIDIR)
    call = lambda n_kv=1000, q=FAKE, k=FAKE, v=FAKE, o=FAKE, ws=FAKE, wn=need: lib.gma_forward_cross(
        ctypes.byref(s), n_kv, _prm(), q, k, v, o, ws, wn, None)
    assert call(n_kv=-1) == 1
    assert call(q=None) == 1 and call(o=None) == 1 and call(k=None) == 1 and call(v=None) == 1
    assert call(k=FAKE + 4) == 3 and call(o=FAKE + 8) == 3
    assert call(ws=None) == 4 and call(wn=need - 1) == 4
    # no query rows: nothing to do, every pointer may be null
    s0 = _shape(N=0)
    assert lib.gma_forward_cross(ctypes.byref(s0), 50, _prm(), None, None, None, None, FAKE, 1 << 30, None) == 0


def test_stats_validation(lib):
    s = _shape(N=300)
    need = gma.gma_workspace_size(s, gma.OP_USAGE)
    assert need > 0
    call = lambda x=FAKE, u=FAKE, c=FAKE, e=FAKE, a=None, ws=FAKE, wn=need: lib.gma_responsibility_stats(
        ctypes.byref(s), _prm(), x, u, c, e, a, ws, wn, None)
    assert call(x=None) == 1 and call(u=None) == 1 and call(c=None) == 1 and call(e=None) == 1
    assert call(u=FAKE + 4) == 3 and call(a=FAKE + 4) == 3
    assert call(ws=None) == 4 and call(wn=need - 1) == 4
    assert gma.gma_workspace_size(_shape(K=513), gma.OP_USAGE) == 0


def test_backward_validation(lib):
    s = _shape(N=300)
    need = gma.gma_workspace_size(s, gma.OP_BACKWARD)
    assert need > gma.gma_workspace_size(s, gma.OP_CAUSAL)
    call = lambda causal=1, **kw: lib.gma_backward(
        ctypes.byref(s), causal, _prm(), *(kw.get(n, FAKE) for n in ("q", "k", "v", "g", "dq", "dk", "dv", "dm",
                                                                        "dr", "dl", "ws")),
        kw.get("wn", need), None)
    assert call(causal=2) == 1
    for n in ("q", "k", "v", "g", "dq", "dk", "dv", "dm", "dr", "dl"):
        assert call(**{n: None}) == 1, n
        assert call(**{n: FAKE + 4}) == 3, n
    assert call(ws=None) == 4 and call(wn=need - 1) == 4
    assert gma.gma_workspace_size(_shape(d_v=8), gma.OP_BACKWARD) == 0
    # the gradient pass ignores the chunk length and the product type of the shape
    assert gma.gma_workspace_size(_shape(N=300, chunk=16), gma.OP_BACKWARD) == need
    assert gma.gma_workspace_size(_shape(N=300, gemm_dtype="bf16"), gma.OP_BACKWARD) == need
