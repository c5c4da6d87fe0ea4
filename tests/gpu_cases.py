"""Shared helpers of the GPU parity tests: device inputs, library calls through
the C ABI binding, and the oracle on sampled (batch, head) slices."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import gaussian_mixture_sequence_gb300 as gma
from gaussian_mixture_sequence_gb300 import workloads

TOL = {"f32": 1e-4, "bf16": 2e-2}   # normwise relative error per (b, h) slice
DEV = "cuda:0"


def shape_of(wl, N=None, chunk=0):
    return gma.Shape.make(wl.B, wl.H, wl.N if N is None else N, wl.d, wl.dv, wl.K, chunk=chunk,
                          eps=wl.eps, x_dtype=wl.x_dtype, v_dtype=wl.v_dtype, gemm_dtype=wl.gemm_dtype)


def _tdt(name):
    return torch.bfloat16 if name == "bf16" else torch.float32


class Case:
    """Inputs of a workload on the device, with host copies of the checked slices.

    ``host_slices=None`` generates every slice on the host (exact seeded
    inputs); otherwise only those slices come from the seeded generator and
    the others are filled on the device with torch's generator (they are not
    compared, and slices are independent in the method)."""

    def __init__(self, wl, host_slices=None, decode=False):
        self.wl = wl
        self.S = wl.B * wl.H
        self.mu, self.vr, self.lp = workloads.params(wl)
        self.slices = list(range(self.S)) if host_slices is None else list(host_slices)
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
        self.prm = (t(self.mu), t(self.vr), t(self.lp))
        self.host = {}
        self.dev = {}
        for part, dec in (("seq", False), ("dec", True)) if decode else (("seq", False),):
            n = wl.decode_steps if dec else wl.N
            if host_slices is None:
                q, k, v = workloads.full_inputs(wl, decode=dec)
                self.host[part] = (q.reshape(self.S, n, -1), k.reshape(self.S, n, -1), v.reshape(self.S, n, -1))
                dq, dk, dv = t(q), t(k), t(v)
            else:
                g = torch.Generator(device=DEV).manual_seed(wl.seed + (7 if dec else 0))
                dq = torch.randn(wl.B, wl.H, n, wl.d, device=DEV, generator=g)
                dk = torch.randn(wl.B, wl.H, n, wl.d, device=DEV, generator=g)
                dv = torch.randn(wl.B, wl.H, n, wl.dv, device=DEV, generator=g)
                hq, hk, hv = [], [], []
                for s in self.slices:
                    b, h = divmod(s, wl.H)
                    q, k, v = workloads.slice_inputs(wl, b, h, mu=self.mu, decode=dec)
                    dq[b, h], dk[b, h], dv[b, h] = t(q), t(k), t(v)
                    hq.append(q); hk.append(k); hv.append(v)
                self.host[part] = (np.stack(hq), np.stack(hk), np.stack(hv))
            self.dev[part] = (dq.to(_tdt(wl.x_dtype)).contiguous(), dk.to(_tdt(wl.x_dtype)).contiguous(),
                              dv.to(_tdt(wl.v_dtype)).contiguous())

    @property
    def heads(self):
        return [s % self.wl.H for s in self.slices]

    def pick(self, t):
        """Rows of a [B,H,...] device tensor for the checked slices, as float64 numpy."""
        flat = t.reshape(self.S, *t.shape[2:]).float().cpu().numpy().astype(np.float64)
        return flat[self.slices] if len(self.slices) != self.S else flat

    def causal(self, chunk=0, state_in=None, want_state=False):
        wl = self.wl
        q, k, v = self.dev["seq"]
        out = torch.empty(wl.B, wl.H, wl.N, wl.dv, device=DEV)
        so = torch.empty(wl.B, wl.H, wl.K * wl.dv + wl.K, device=DEV) if want_state else None
        gma.gma_forward_causal(shape_of(wl, chunk=chunk), *self.prm, q, k, v, out, state_in=state_in,
                               state_out=so)
        return (out, so) if want_state else out

    def bidir(self):
        wl = self.wl
        q, k, v = self.dev["seq"]
        out = torch.empty(wl.B, wl.H, wl.N, wl.dv, device=DEV)
        gma.gma_forward_bidir(shape_of(wl), *self.prm, q, k, v, out)
        return out

    def gamma(self, which="q"):
        wl = self.wl
        x = self.dev["seq"][0 if which == "q" else 1]
        g = torch.empty(wl.B, wl.H, wl.N, wl.K, device=DEV)
        gma.gma_responsibilities(shape_of(wl), *self.prm, x, g)
        return g

    # --- oracle on the checked slices ---
    def ref_causal(self, state_in=None, return_state=False):
        q, k, v = self.host["seq"]
        return oracle.causal(self.mu, self.vr, self.lp, q, k, v, self.wl.eps, heads=self.heads,
                             state_in=state_in, return_state=return_state)

    def ref_bidir(self):
        q, k, v = self.host["seq"]
        return oracle.bidir(self.mu, self.vr, self.lp, q, k, v, self.wl.eps, heads=self.heads)

    def ref_gamma(self, which="q"):
        x = self.host["seq"][0 if which == "q" else 1]
        return oracle.responsibilities(self.mu, self.vr, self.lp, x, heads=self.heads)


def normwise(out, ref):
    """max over slices of max|out - ref| / max|ref| (slices along axis 0)."""
    out = np.asarray(out, np.float64).reshape(ref.shape[0], -1)
    ref = np.asarray(ref, np.float64).reshape(ref.shape[0], -1)
    num = np.abs(out - ref).max(1)
    den = np.abs(ref).max(1)
    return float((num / np.maximum(den, 1e-300)).max())
