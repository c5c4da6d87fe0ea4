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
    assert bench.eff_chunk(W["causal_8k_K64"]) == 128                     # K < 128: padded to 128
    assert bench.eff_chunk(W["causal_8k_K512"]) == 128                    # whole groups of 128
    assert bench.eff_chunk(W["causal_8k_K64"].with_(K=200)) == 64         # other K: CUDA cores, C = 64
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
    g = W["causal_8k_K64"].with_(K=200)
    assert bench.stage_work("state_scan", g)[2] == 2 * (4 * 8 * (8192 // 256)) * 200 * 65 * 4


def test_algorithmic_bytes_follow_the_method_io():
    """The roofline charges each launch only with the method's own input and output
    (Q_X, K_X, V in once; O out once): materialised responsibilities and the carried
    memory are implementation overhead.  At the headline size the chunk-output launch
    is charged V in + O out, 512 bytes per head-token, and the whole step sums to
    (2 d + d_v) * 4 + 4 d_v bytes per head-token plus one more read of V (both the
    state pass and the output pass consume V)."""
    wl = W["causal_16k_peaked"]
    ht = 2 * 16 * 16384
    pk = dict(bench.FALLBACK)
    assert bench.algorithmic_work("chunk_out_tc", wl)[2] == ht * (64 * 4 + 64 * 4)
    assert bench.algorithmic_work("chunk_state_tc", wl)[2] == ht * 64 * 4
    assert bench.algorithmic_work("resp_q", wl, kept=1.0)[2] == ht * 64 * 4
    assert bench.algorithmic_work("state_scan", wl)[2] == 0.0
    assert bench.algorithmic_work("prep", wl)[2] == 0.0
    step = sum(bench.algorithmic_work(s, wl, kept=1.0)[2]
               for s in ("prep", "resp_q", "resp_k", "chunk_state_tc", "state_scan", "chunk_out_tc"))
    assert step == ht * ((2 * 64 + 64) * 4 + 4 * 64) + ht * 64 * 4
    # the bidirectional read writes O only
    assert bench.algorithmic_work("bidir_read_tc", W["bidir_16k_peaked"])[2] == ht * 64 * 4
    # bf16 inputs halve the input bytes
    g = W["causal_64k_bf16"]
    assert bench.algorithmic_work("chunk_out_tc", g)[2] == 65536 * 16 * (128 * 2 + 128 * 4)
    # the roofline of a 166 us chunk-output launch: HBM-bound, 268 MB / 166 us over the peak,
    # and the kernel-byte model beside it
    r = bench.roofline_of("chunk_out_tc", wl, 166e-6, pk)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["frac"] == pytest.approx(ht * 512 / 166e-6 / 1e9 / pk["hbm_gbs"])
    assert r["frac_kernel_bytes"] == pytest.approx(bench.stage_work("chunk_out_tc", wl)[2] / 166e-6 / 1e9
                                                   / pk["hbm_gbs"])
    assert r["frac_kernel_bytes"] > 3 * r["frac"]
    # the decode step's state is the method's memory: in and out are algorithmic bytes
    d = W["decode_b256"]
    assert bench.algorithmic_work("decode", d)[2] == bench.stage_work("decode", d)[2]


def test_bounded_routing_roofline():
    """With the bounded routing the FP32 work is the exact evaluation of the kept components
    and the bound GEMM is bf16 tensor work; the launch is HBM-bound when few are kept and
    FP32-bound when many are."""
    pk = dict(bench.FALLBACK)
    peaked = bench.roofline_of("resp_q", W["causal_16k_peaked"], 100e-6, pk, kept=1.0)
    assert peaked["bound"] == "hbm"
    dense = bench.roofline_of("resp_q", W["causal_4k"], 300e-6, pk, kept=64.0)
    assert dense["bound"] == "alu"
    assert dense["algorithmic_flop"] == 4 * 64 * 64.0 * 4 * 8 * 4096
    # the generic kernel (here d = 128) is charged the dense routing on the FP32 pipe
    g = bench.roofline_of("resp_q", W["causal_8k_K512"].with_(d=128), 2600e-6, pk)
    assert g["bound"] == "alu" and g["algorithmic_flop"] == 4 * 512 * 128 * 4 * 8 * 8192


def test_dense_pass_roofline():
    """The dense pass is tensor work: six bf16 passes of the [x^2 | x] W^T product (4 K d
    flop per row each; four with bf16 rows) over both routings' rows in dense tiles; the
    rows it takes carry no FP32 exact work in the bounded routing launches."""
    pk = dict(bench.FALLBACK)
    wl, wb = W["causal_4k"], W["causal_64k_bf16"]
    ht = wl.B * wl.H * wl.N
    r = bench.roofline_of("resp_dense", wl, 70e-6, pk, kept=3.0, dense=1.0)
    assert r["bound"] == "tensor" and r["algorithmic_flop"] == 2 * 6 * 4 * 128 * 64 * ht
    assert r["algorithmic_bytes"] == 0                # the routing rows are charged to resp_q / resp_k
    rb = bench.roofline_of("resp_dense", wb, 390e-6, pk, kept=3.0, dense=0.5)
    assert rb["algorithmic_flop"] == 0.5 * 2 * 4 * 4 * 128 * 64 * wb.B * wb.H * wb.N
    q = bench.roofline_of("resp_q", wl, 33e-6, pk, kept=3.0, dense=1.0)
    assert q["bound"] == "hbm" and q["algorithmic_bytes"] == ht * 64 * 4
    t, parts = bench.path_roofline_s(wl, pk, kept=3.0, dense=1.0)
    assert parts["alu_s"] == 0.0 and parts["mma_s"] > 0.0


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
    kernel) stay within its kernel-byte model (no tile is read twice) and above the model
    less the lo plane of Gamma_Q (256 B per head-token), which the kernel skips on
    the chunks whose rows all keep their argmax alone (most of the headline's)."""
    wl = W["causal_16k_peaked"]
    t = bench.traffic_record("chunk_out_tc", wl)
    if t is None:
        pytest.skip("profiles/dram_traffic.txt holds no counters for the current chunk-output source")
    model = bench.stage_work("chunk_out_tc", wl)[2]
    lo_q = wl.K * 2 * wl.B * wl.H * wl.N            # Gamma_Q's lo plane (bf16)
    # (ncu does not count dirty lines left in L2 at the end of a launch: 2 % below is allowed)
    assert 0.98 * (model - lo_q) <= t <= 1.05 * model, (t, model)
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
    # a record for the current sources of both kernels (written here, so that the test does not
    # depend on the committed counters being current)
    rec = root / "profiles" / "dram_traffic.txt"
    rec.write_text(rec.read_text() + "".join(
        f"{st} {bench.source_hash(st, wl)} {wl.name} 1000\n" for st in ("chunk_out_tc", "resp_q")))
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
    # a timed region shorter than the sampling period: the clock soak before it is used
    r = _sampler([hot, ok, ok, cap, ok]).summary(4.0, 4.5, 1.0)
    assert r["window"] == "soak+timed" and r["samples"] == 4 and r["reasons"] == ["sw_power_cap"]
    r = _sampler([ok, ok, ok, ok]).summary(0.0, 3.0, 0.0)
    assert r["window"] == "timed"


def test_tokens_per_step():
    assert bench.tokens_per_step(W["causal_16k_peaked"]) == 2 * 16384
    assert bench.tokens_per_step(W["decode_b256"]) == 256


def test_small_k_routing_roofline():
    """For 17 <= K <= 512 but 128 with d = 64 both routings are tensor work (the six bf16
    passes of a product 32, 64, 128, 256 or 512 components wide) and carry no FP32 work in
    the whole-step roofline."""
    pk = dict(bench.FALLBACK)
    wl = W["causal_8k_K32"]
    ht = wl.B * wl.H * wl.N
    f, pipe, _ = bench.stage_work("resp_q", wl)
    assert pipe == "tensor_bf16" and f == 6 * 4 * 32 * 64 * ht
    assert bench.stage_work("resp_q", W["causal_8k_K64"])[0] == 6 * 4 * 64 * 64 * ht
    r = bench.roofline_of("resp_q", wl, 100e-6, pk)
    assert r["bound"] in ("tensor", "hbm")
    t, parts = bench.path_roofline_s(wl, pk)
    assert parts["alu_s"] == 0.0
    f, pipe, _ = bench.stage_work("resp_q", W["causal_8k_K256"])
    assert pipe == "tensor_bf16" and f == 6 * 4 * 256 * 64 * ht
    assert bench.stage_work("resp_q", W["causal_8k_K256"].with_(K=100))[0] == 6 * 4 * 128 * 64 * ht
    assert bench.stage_work("resp_q", W["causal_8k_K256"].with_(x_dtype="bf16"))[0] == 4 * 4 * 256 * 64 * ht
    assert bench.stage_work("resp_q", W["causal_8k_K512"])[0] == 6 * 4 * 512 * 64 * ht
    # K = 128 has the bounded routing; K above 512 and d = 128 keep the CUDA-core routing
    assert not bench.tc_routing(W["causal_4k"])
    assert bench.stage_work("resp_q", W["causal_8k_K512"].with_(K=520))[1] == "alu"
    assert bench.stage_work("resp_q", W["causal_8k_K256"].with_(d=128))[1] == "alu"
