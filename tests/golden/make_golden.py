"""Writes tests/golden/tiny_oracle.json: sampled fp64 oracle values on the tiny workload.

Calls only the oracle (and the seeded input generator).  The record guards the
oracle against silent drift; the oracle itself is pinned by test_oracle_pins.py.
Run from the repository root:  python tests/golden/make_golden.py
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from gaussian_mixture_sequence_gb300 import workloads  # noqa: E402

ROWS = [0, 1, 63, 64, 100, 255]


def main():
    wl = workloads.WORKLOADS["tiny"]
    mu, vr, lp = workloads.params(wl)
    qx, kx, v = workloads.slice_inputs(wl, 0, 0, mu=mu)
    g = oracle.responsibilities(mu, vr, lp, qx[None])[0]
    c, st = oracle.causal(mu, vr, lp, qx[None], kx[None], v[None], wl.eps, return_state=True)
    b = oracle.bidir(mu, vr, lp, qx[None], kx[None], v[None], wl.eps)
    rec = {
        "source": "fp64 oracle (oracle/gma_oracle.c) on workload 'tiny' (B=1,H=1,N=256,d=16,"
                  "dv=16,K=8, seed 1000); method per the GMA explainer 'Gaussian Mixture "
                  "Attention: Linear-Time Sequence Mixing via Probabilistic Latent Routing', "
                  "technical summary, sections 핵심 메커니즘 and 변형 및 학습",
        "rows": ROWS,
        "gamma_q": g[ROWS].tolist(),
        "causal": c[0, ROWS].tolist(),
        "bidir": b[0, ROWS].tolist(),
        "state_final": st[0].tolist(),
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_oracle.json")
    with open(path, "w") as f:
        json.dump(rec, f, indent=0)
    print("wrote", path)


if __name__ == "__main__":
    main()
