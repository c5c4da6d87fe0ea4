"""Host logic of bench.py on the CPU: the algorithmic work per launch behind
the roofline, the committed DRAM counters and when they stop applying, the
chunk length per workload, and the clock summary that decides whether a run
is kept."""
import os
import shutil

import pytest

import bench
from gaussian_mixture_sequence_gb300 import workloads

W = workloads.WORKLOADS


def test_chunk_length_per_workload():
    assert bench.eff_chunk(W["causal_16k_peaked"]) == 128                 # K = 128, d_v = 64: tensor cores
    assert bench.eff_chunk(W["causal_8k_K64"]) == 64                      # other K: CUDA cores, C = 64
    assert bench.eff_chunk(W["causal_64k_bf16"]) == 128                   # d_v = 128 with bf16 products
    assert bench.eff_chunk(W["causal_16k_peaked"].with_(dv=128)) == 64    # d_v = 128, fp32 products
    assert bench.eff_chunk(W["causal_16k_peaked"].with_(chunk=32)) == 32  # a caller's choice wins


def test_headline_bytes_per_launch():
    """Minimum bytes of one launch at the headline size (B=2, H=16, N=16384, d=d_v=64,
    K=128, fp32): its inputs once and its outputs once."""
    wl = W["causal_16k_peaked"]
    ht = 2 * 16 * 16384                        # head-tokens
    chunks = 2 * 16 * (16384 // 128)           # chunks of 128 rows
    state = 128 * 65 * 4                       # one fp32 memory block [Vt | Z]
    _, pipe, b = bench.stage_work("resp_q", wl)
    assert pipe == "tensor_bf16" and b == ht * (64 * 4 + 128 * 4)                # x in, Gamma out
    _, pipe, b = bench.stage_work("chunk_state_tc", wl)
    assert pipe == "tensor_bf16" and b == ht * (128 * 4 + 64 * 4) + chunks * state
    _, _, b = bench.stage_work("state_scan", wl)
    assert b == 2 * chunks * state                                              # partials in, memory out
    f, pipe, b = bench.stage_work("chunk_out_tc", wl)
    assert b == ht * (2 * 128 * 4 + 64 * 4 + 64 * 4) + chunks * state            # Gq, Gk, V in, O out
    assert b == pytest.approx(941.6e6, rel=1e-4)
    assert f == ht * (2 * 128 * 128 + 128 * 65 + 2 * 128 * 65)
    assert bench.stage_work("prep", wl)[2] == 0.0
    # the bidirectional total: every chunk's partial in, one block per (b, h) out
    assert bench.stage_work("state_reduce", W["bidir_16k_peaked"])[2] == (chunks + 2 * 16) * state
    # the CUDA-core path scans blocks of 256 rows
    g = W["causal_8k_K64"]
    assert bench.stage_work("state_scan", g)[2] == 2 * (4 * 8 * (8192 // 256)) * 64 * 65 * 4


def test_decode_bytes_per_launch():
    wl = W["decode_b256"]
    bh = wl.B * wl.H
    f, pipe, b = bench.stage_work("decode", wl)
    state = wl.K * (wl.dv + 1) * 4
    assert pipe == "alu"
    assert b == bh * (2 * state + 2 * wl.d * 4 + wl.dv * 4 + wl.dv * 4)         # state in and out, q, k, v, o
    assert f == bh * (8 * wl.K * wl.d + 4 * wl.K * (wl.dv + 1))


def test_measured_traffic_matches_algorithmic_bytes():
    """The committed ncu counters of the chunk-output kernel (the headline's dominant
    kernel) are within 5 % of its algorithmic bytes: no tile is read twice."""
    wl = W["causal_16k_peaked"]
    t = bench.traffic_record("chunk_out_tc", wl)
    assert t is not None, "profiles/dram_traffic.txt does not match the current kernel sources"
    assert t == pytest.approx(bench.stage_work("chunk_out_tc", wl)[2], rel=0.05)
    assert bench.traffic_record("decode", wl) is None                           # no counters recorded


def test_traffic_is_dropped_when_the_kernel_changes(tmp_path, monkeypatch):
    """A counter applies only while the kernel's source (with the shared headers) still
    hashes to the recorded value."""
    csrc = os.path.join(bench.ROOT, "gaussian_mixture_sequence_gb300", "csrc")
    root = tmp_path / "repo"
    shutil.copytree(csrc, root / "gaussian_mixture_sequence_gb300" / "csrc")
    shutil.copytree(os.path.join(bench.ROOT, "profiles"), root / "profiles")
    monkeypatch.setattr(bench, "ROOT", str(root))
    wl = W["causal_16k_peaked"]
    before = bench.traffic_record("chunk_out_tc", wl)
    assert before is not None
    p = root / "gaussian_mixture_sequence_gb300" / "csrc" / "gma_causal_tc.cu"
    p.write_text(p.read_text() + "\n// changed\n")
    assert bench.traffic_record("chunk_out_tc", wl) is None
    assert bench.traffic_record("resp_q", wl) is not None                      # other sources unchanged
    h = root / "gaussian_mixture_sequence_gb300" / "csrc" / "gma_tc.cuh"
    h.write_text(h.read_text() + "\n// changed\n")
    assert bench.traffic_record("resp_q", wl) is None                          # a shared header


def _sampler(rows):
    s = bench.ClockSampler.__new__(bench.ClockSampler)
    s.samples = [(float(i), r) for i, r in enumerate(rows)]
    s.proc = None
    return s


def test_clock_summary():
    ok = ["2070", "2070", "800.5", "0x0", "Not Active", "Not Active", "Not Active", "Not Active"]
    cap = ["1965", "2070", "1390.0", "0x4", "Not Active", "Not Active", "Not Active", "Active"]
    hot = ["1500", "2070", "1200.0", "0x40", "Not Active", "Active", "Not Active", "Not Active"]
    s = _sampler([ok, ok, cap, ok, ok])
    r = s.summary(0.0, 10.0)
    assert r["sm_mhz"] == 2070.0 and r["sm_max_mhz"] == 2070.0 and r["samples"] == 5
    assert r["reasons"] == ["sw_power_cap"] and r["power_w_max"] == 1390.0
    r = _sampler([ok, hot, hot]).summary(0.0, 10.0)
    assert r["reasons"] == ["hw_thermal_slowdown"] and r["sm_mhz"] == 1500.0
    # fewer than three samples in the window: the whole record is used
    r = _sampler([ok, ok, ok, cap]).summary(3.0, 3.0)
    assert r["samples"] == 4
    r = _sampler([]).summary(0.0, 1.0)
    assert r["samples"] == 0 and r["reasons"] == ["nvidia-smi unavailable"]


def test_tokens_per_step():
    assert bench.tokens_per_step(W["causal_16k_peaked"]) == 2 * 16384
    assert bench.tokens_per_step(W["decode_b256"]) == 256
