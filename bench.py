#!/usr/bin/env python
"""Causal GMA forward throughput on GB300 (tokens/s at N=16384, K=128).

One step = one full causal forward (parameter preparation, responsibilities
of Q_X and K_X, chunkwise write/read with the carried memory) over one batch
of seeded synthetic inputs already resident in HBM, through the library's C
ABI.  Prints one JSON line (rank 0).  See --help for options.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the fp64 oracle on the host cores

For N > 1 it is launched by torch.distributed.run, one rank per GPU; every
rank runs its own replica of the workload (weak scaling, no collective on the
data path) and the slowest rank's time sets the whole-job throughput.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GMA causal fwd tokens/sec at N=16K,K=128 (1 GB300); % of roofline"
SM_COUNT, FP32_LANES_PER_SM = 152, 128
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "sm_max_mhz": 2070.0}


def parse():
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["gma", "reference"], default="gma")
    p.add_argument("--workload", default="causal_16k_peaked")
    p.add_argument("--e2e-steps", type=int, default=10)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--batch", type=int, default=0,
                   help="run the workload with this many sequences instead of its own B (profiling captures)")
    p.add_argument("--clock-soak-s", type=float, default=1.0,
                   help="after the --warmup steps, run untimed steps for this many seconds right before "
                        "the timed region, so that the clock sampler (100 ms period) sees the GPU under "
                        "this load (reported as clock_soak, not as warm-up)")
    return p.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK), "fallback"


# ----------------------------------------------------------------- work model --

def eff_chunk(wl):
    """Chunk length the library uses for this workload (its default when 0)."""
    if wl.chunk:
        return wl.chunk
    tc = ((wl.K <= 128 or (wl.K % 128 == 0 and wl.K <= 512))
          and (wl.dv == 64 or (wl.dv == 128 and wl.gemm_dtype == "bf16")))
    return 128 if tc else 64


def stage_work(stage, wl):
    """Work of one launch of a stage as the kernel runs it: (flop, pipe, bytes),
    the bytes being everything the launch must move, the materialised
    responsibilities and the per-chunk memory included (the kernel-byte model;
    compare it with the DRAM counters).

    Per head-token (ht), with d = d_route, K components, d_v values, chunk C
    (flop):
      resp_q / resp_k     4*K*d on the FP32 pipe (one fp32x2 FMA for (x-mu)/sigma
                          and one for the square-accumulate, per component and
                          feature pair); for 17 <= K <= 64 and d = 64, the six (four
                          with bf16 rows) bf16 passes of [x^2 | x] W^T, K_N = 32 or
                          64 wide, on the tensor pipe
      resp_dense          24*K*d on the bf16 tensor pipe per row of the tiles the
                          bounded routings leave to the dense pass (K = 128, d = 64;
                          six passes of the three-plane product [x^2 | x] W^T, of
                          4*K*d each; 16*K*d with bf16 rows, whose zero planes are
                          skipped), both routings
      block_state /
      chunk_state_tc      2*K*(d_v+1)           (Gamma_K^T [V | 1])
      chunk_out(_tc)      2*C*K + C*(d_v+1) + 2*K*(d_v+1)   (P = Gq Gk^T, lower half
                          of P [V | 1], read of the carried memory); the CUDA-core
                          kernel also advances the memory: + 2*K*(d_v+1)
      bidir_read          2*K*(d_v+1)           (Gq [Vt | Z])
      decode (per (b,h))  8*K*d + 4*K*(d_v+1)   (two routings, update and read)
    Bytes are the minimum each launch must move: its inputs once and its
    outputs once (fp32 state of K*(d_v+1) per block of the scan, blocks of C
    rows on the tensor-core path and of 256 rows otherwise; for the decode
    step the whole state in and out).
    """
    K, d, dv = wl.K, wl.d, wl.dv
    xb = 2 if wl.x_dtype == "bf16" else 4
    vb = 2 if wl.v_dtype == "bf16" else 4
    gb = 2 if wl.gemm_dtype == "bf16" else 4
    st = 4.0 * K * (dv + 1)
    if wl.mode == "decode":
        bh = wl.B * wl.H
        if stage == "decode":
            return (8.0 * K * d + 4.0 * K * (dv + 1)) * bh, "alu", (2 * st + 2 * d * xb + dv * vb + 4 * dv) * bh
        return 0.0, "alu", 0.0
    ht = wl.B * wl.H * wl.N
    if wl.mode == "backward":
        return backward_work(wl)
    C = eff_chunk(wl)
    tc = stage.endswith("_tc")
    # blocks of the carried memory: chunks of C rows on the tensor-core path (its scan too),
    # blocks of 256 rows on the CUDA-core path
    blk = C if tc or (stage in ("state_scan", "state_reduce") and C == 128) else 256
    nblk = wl.B * wl.H * -(-wl.N // blk)
    if stage in ("resp_q", "resp_k"):
        # K = 128, d = 64: the bound GEMM [x^2 | x] W has the same 4*K*d flop per row and runs on the
        # tensor pipe (bf16); the exact evaluation of the kept components is data-dependent extra work.
        # 17 <= K <= 512 otherwise, d = 64: every log-joint on the tensor pipe, the dense pass's bf16
        # passes of a product K_N wide (K rounded up to 32, 64, 128, 256 or 512)
        if tc_routing(wl):
            kn = tc_width(K)
            return dense_passes(wl) * 4.0 * kn * d * ht, "tensor_bf16", (d * xb + K * gb) * ht
        pipe = "tensor_bf16" if bounded_routing(wl) else "alu"
        return 4.0 * K * d * ht, pipe, (d * xb + K * gb) * ht
    if stage == "resp_dense":
        # the dense pass over the tiles the bounded routings left to it, charged as if every tile
        # of both routings were dense (on the inputs where this stage dominates, nearly all are)
        return 2 * dense_passes(wl) * 4.0 * K * d * ht, "tensor_bf16", 2 * (d * xb + K * gb) * ht
    if stage in ("block_state", "chunk_state_tc"):
        return 2.0 * K * (dv + 1) * ht, ("tensor_bf16" if tc else "alu"), (K * gb + dv * vb) * ht + st * nblk
    if stage in ("chunk_out", "chunk_out_tc"):
        fl = 2.0 * C * K + C * (dv + 1) + 2.0 * K * (dv + 1) + (0 if tc else 2.0 * K * (dv + 1))
        return fl * ht, ("tensor_bf16" if tc else "alu"), (2 * K * gb + dv * vb + 4 * dv) * ht + st * nblk
    if stage in ("bidir_read", "bidir_read_tc"):
        return 2.0 * K * (dv + 1) * ht, ("tensor_bf16" if tc else "alu"), (K * gb + 4 * dv) * ht + st * wl.B * wl.H
    if stage == "state_scan":     # every block's partial in, its carried memory out
        return 0.0, "alu", 2.0 * st * nblk
    if stage == "state_reduce":   # every block's partial in, one total per (b, h) out
        return 0.0, "alu", st * (nblk + wl.B * wl.H)
    return 0.0, "alu", 0.0


def dense_passes(wl):
    """bf16 passes of the dense tensor-core routing, in units of one [x^2 | x] W^T product:
    six for fp32 rows; with bf16 rows the values' two lower planes and the squares' lowest
    plane are zero (32 of the 48 MMAs run)."""
    return 4.0 if wl.x_dtype == "bf16" else 6.0


def backward_work(wl):
    """Work of one gradient pass (causal form, chunks of C = 64 on CUDA cores), per head-token:
    FP32 flop: routing recomputed for Q_X and K_X (8 K d), dx (8 K d: y and the
    delta-weighted sum), the parameter partial sums (12 K d), and the chunk products of
    the forward recompute, the query side and the key/value side (three times those of
    the forward, 3 (4 K (d_v + 1) + 2 C K + C (d_v + 1)));
    bytes: Q_X, K_X, V and dL/dO in, dQ_X, dK_X and dV out (fp32)."""
    K, d, dv, C = wl.K, wl.d, wl.dv, 64
    xb = 2 if wl.x_dtype == "bf16" else 4
    vb = 2 if wl.v_dtype == "bf16" else 4
    ht = wl.B * wl.H * wl.N
    flop = (28.0 * K * d + 3.0 * (4.0 * K * (dv + 1) + 2.0 * C * K + C * (dv + 1))) * ht
    nbytes = (2 * d * xb + dv * vb + 4 * dv + 8 * d + 4 * dv) * ht
    return flop, "alu", nbytes


def algorithmic_work(stage, wl, kept=None, dense=None):
    """Algorithmic work of one launch of a stage, as the roofline charges it:
    (flop, pipe, bytes).

    Bytes: only the method's own input and output (read Q_X, K_X and V once,
    write O once; for the decode step also the recurrent state in and out,
    which is the method's memory).  Each launch is charged with the part of
    that I/O it consumes or produces:
      resp_q / resp_k      Q_X or K_X in
      chunk_state(_tc) /
      block_state          V in
      chunk_out(_tc)       V in, O out
      bidir_read(_tc)      O out
      scans, reductions,
      parameter prep       nothing
    Materialised responsibilities and the per-chunk carried memory are
    overhead of this implementation and are not counted (they appear in
    `stage_work`, the kernel-byte model).

    Flop: the method's contractions as `stage_work` counts them.  For the
    bounded routing (K = 128, d = 64) the flop are the bound GEMM on the bf16
    tensor pipe plus the exact evaluation of the kept components on the FP32
    pipe, whichever takes longer at its peak (`kept` = mean kept components per
    row outside the dense tiles and `dense` = fraction of rows in dense tiles,
    both measured); the dense pass is charged its tensor passes over that
    fraction of the rows; elsewhere the dense FP32 routing."""
    if wl.mode == "backward":
        return backward_work(wl)
    flop, pipe, _ = stage_work(stage, wl)
    if pipe == "tensor_bf16" and stage not in ("resp_q", "resp_k", "resp_dense"):   # routing: bf16 passes
        pipe = "tensor"   # the chunk products at the rate of their operand type (tf32 for fp32)
    d, dv = wl.d, wl.dv
    xb = 2 if wl.x_dtype == "bf16" else 4
    vb = 2 if wl.v_dtype == "bf16" else 4
    if wl.mode == "decode":
        return stage_work(stage, wl)
    ht = wl.B * wl.H * wl.N
    if stage in ("resp_q", "resp_k"):
        nbytes = d * xb * ht
        if bounded_routing(wl) and kept is not None:
            return 4.0 * d * kept * (1.0 - (dense or 0.0)) * ht, "alu_kept", nbytes
        return flop, pipe, nbytes
    if stage == "resp_dense":   # its routing rows were charged to resp_q / resp_k
        return flop * (1.0 if dense is None else dense), pipe, 0.0
    if stage in ("block_state", "chunk_state_tc"):
        return flop, pipe, dv * vb * ht
    if stage in ("chunk_out", "chunk_out_tc"):
        return flop, pipe, (dv * vb + 4 * dv) * ht
    if stage in ("bidir_read", "bidir_read_tc"):
        return flop, pipe, 4 * dv * ht
    return flop, pipe, 0.0


def roofline_of(stage, wl, t_launch, pk, kept=None, dense=None):
    """The roofline object of one launch taking t_launch seconds: the bound is the
    slower of its algorithmic flop at the pipe's peak and its algorithmic bytes at
    the measured HBM rate; `frac` = achieved / peak on that bound.  Also the same
    launch against the kernel-byte model (`kernel_bytes`, `frac_kernel_bytes`)."""
    flop, pipe, nbytes = algorithmic_work(stage, wl, kept, dense)
    if pipe == "alu_kept":   # bounded routing: the bound GEMM (tensor) or the kept exact work (FP32)
        t_fp = flop / pipe_peak("alu", wl, pk)
        t_tc = stage_work(stage, wl)[0] / pipe_peak("tensor_bf16", wl, pk)
        flop, pipe = (flop, "alu") if t_fp >= t_tc else (stage_work(stage, wl)[0], "tensor_bf16")
    t_flop = flop / pipe_peak(pipe, wl, pk) if flop else 0.0
    t_mem = nbytes / (pk["hbm_gbs"] * 1e9)
    if t_flop >= t_mem:
        bound = "alu" if pipe == "alu" else "tensor"
        achieved, peak, unit = flop / t_launch / 1e12, pipe_peak(pipe, wl, pk) / 1e12, "TFLOP/s"
    else:
        bound = "hbm"
        achieved, peak, unit = nbytes / t_launch / 1e9, pk["hbm_gbs"], "GB/s"
    kb = stage_work(stage, wl)[2]
    return {"bound": bound, "kernel": stage, "achieved": achieved, "peak": peak, "unit": unit,
            "frac": achieved / peak, "algorithmic_bytes": nbytes, "algorithmic_flop": flop,
            "kernel_bytes": kb, "frac_kernel_bytes": kb / t_launch / 1e9 / pk["hbm_gbs"]}


def bounded_routing(wl):
    """The library's routing kernel with the tensor-core bound applies (K = 128, d = 64)."""
    return wl.K == 128 and wl.d == 64


def tc_routing(wl):
    """The library's tensor-core routing for 17 <= K <= 512 applies (d = 64; K = 128 has the
    bounded routing instead)."""
    return wl.d == 64 and 17 <= wl.K <= 512 and not bounded_routing(wl)


def tc_width(K):
    """Components of the tensor-core routing's product: K rounded up to 32, 64, 128, 256 or
    512 (two CTAs of 256)."""
    return next(w for w in (32, 64, 128, 256, 512) if K <= w)


def pipe_peak(pipe, wl, pk):
    """Peak of a pipe in flop/s: FP32 lanes x 2 x max SM clock, or the tensor
    rate of the product operands (tf32 = measured bf16 x 1.1/2.25 nominal ratio)."""
    if pipe == "alu":
        return SM_COUNT * FP32_LANES_PER_SM * 2 * pk["sm_max_mhz"] * 1e6
    bf16 = pk["bf16_tflops"] * 1e12
    if pipe == "tensor_bf16":
        return bf16
    return bf16 if wl.gemm_dtype == "bf16" else bf16 * (1.1 / 2.25)


def path_roofline_s(wl, pk, kept=None, dense=None):
    """Roofline time of one step: max(FP32 time, HBM time of the minimum
    traffic, tensor time).  With the bounded routing (K = 128, d = 64) the FP32
    work is the exact evaluation of the kept components of the rows outside the
    dense tiles (two passes of 4*d flop each per kept component and row; `kept`
    = their mean kept components, `dense` = fraction of rows in dense tiles,
    both measured), and the bound GEMMs and the dense tiles' passes are tensor
    work; otherwise the FP32 work is the dense routing, 8*K*d flop per
    head-token."""
    fp32_peak = SM_COUNT * FP32_LANES_PER_SM * 2 * pk["sm_max_mhz"] * 1e6
    xb = 2 if wl.x_dtype == "bf16" else 4
    vb = 2 if wl.v_dtype == "bf16" else 4
    if wl.mode == "decode":
        bh = wl.B * wl.H
        t_alu = (8.0 * wl.K * wl.d + 4.0 * wl.K * (wl.dv + 1)) * bh / fp32_peak
        t_hbm = (8.0 * wl.K * (wl.dv + 1) + 2 * wl.d * xb + wl.dv * vb + 4 * wl.dv) * bh / (pk["hbm_gbs"] * 1e9)
        return max(t_alu, t_hbm), dict(alu_s=t_alu, hbm_s=t_hbm, mma_s=0.0)
    ht = wl.B * wl.H * wl.N
    if wl.mode == "backward":
        flop, _, nbytes = backward_work(wl)
        t_alu, t_hbm = flop / fp32_peak, nbytes / (pk["hbm_gbs"] * 1e9)
        return max(t_alu, t_hbm), dict(alu_s=t_alu, hbm_s=t_hbm, mma_s=0.0)
    t_hbm = ((2 * wl.d * xb + wl.dv * vb + 4 * wl.dv) * ht) / (pk["hbm_gbs"] * 1e9)
    C = eff_chunk(wl)
    if wl.mode == "bidir":
        mma = 4.0 * wl.K * (wl.dv + 1) * ht
    else:
        mma = (4.0 * wl.K * (wl.dv + 1) + 2.0 * C * wl.K + C * (wl.dv + 1)) * ht
    tens = pk["bf16_tflops"] * 1e12 * (1.0 if wl.gemm_dtype == "bf16" else 1.1 / 2.25)
    t_mma = mma / tens
    if bounded_routing(wl) and kept is not None:
        dn = dense or 0.0
        t_alu = 2 * 2 * 4.0 * wl.d * kept * (1.0 - dn) * ht / fp32_peak   # Q and K rows, two exact passes
        t_mma += (8.0 + 8.0 * dense_passes(wl) * dn) * wl.K * wl.d * ht / (pk["bf16_tflops"] * 1e12)
    elif tc_routing(wl):   # both routings on the tensor pipe
        t_alu = 0.0
        t_mma += 2 * stage_work("resp_q", wl)[0] / (pk["bf16_tflops"] * 1e12)
    else:
        t_alu = 8.0 * wl.K * wl.d * ht / fp32_peak
    return max(t_alu, t_hbm, t_mma), dict(alu_s=t_alu, hbm_s=t_hbm, mma_s=t_mma)


def tokens_per_step(wl):
    """Tokens (all H heads of a position) one step processes."""
    return wl.B if wl.mode == "decode" else wl.B * wl.N


# ----------------------------------------------------------------- clocks -----

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", gpu_id, f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            return
        self.th = threading.Thread(target=self._read, daemon=True)
        self.th.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) == 8:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1, t_soak=None):
        """Clock record of the timed region [t0, t1]; when it holds fewer than three
        samples, of the clock soak and the timed region [t_soak, t1] (the same load
        just before it), else of the whole record.  `window` says which."""
        window = "timed"
        win = [p for t, p in self.samples if t0 <= t <= t1]
        if len(win) < 3 and t_soak is not None:
            window = "soak+timed"
            win = [p for t, p in self.samples if t_soak <= t <= t1]
        if len(win) < 3:
            window = "run"
            win = [p for _, p in self.samples]
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[0]) for p in win if num(p[0]) is not None]
        mx = [num(p[1]) for p in win if num(p[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in win for i in range(4) if p[4 + i].lower().startswith("active")})
        pw = [num(p[2]) for p in win if num(p[2]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(win), "power_w_max": max(pw) if pw else None,
                "window": window}


# ----------------------------------------------------------------- helpers ----

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def replica_seed(wl, rank):
    """Seed of the inputs of rank `rank`: every rank runs its own replica of the workload
    (the (batch, head) slices are independent, so there is no exchange between ranks)."""
    return wl.seed + rank


def max_over_ranks(pg, x, device):
    """The maximum of a per-rank number over all ranks (`pg` None: one rank)."""
    if pg is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world, tokens_per_rank, ms):
    """Tokens per second of the whole job: every rank processes tokens_per_rank in ms (the
    slowest rank's time)."""
    return world * tokens_per_rank / (ms * 1e-3)


# The source file holding each stage's kernel; its hash (with the shared headers)
# keys the committed DRAM counters, so a changed kernel reports no traffic.
KERNEL_SOURCE = {
    "prep_params": "gma_resp.cu", "prep": "gma_resp_tc.cu", "resp_dense": "gma_resp_tc.cu",
    "chunk_state_tc": "gma_causal_tc.cu", "chunk_out_tc": "gma_causal_tc.cu", "bidir_read_tc": "gma_causal_tc.cu",
    "block_state": "gma_mix.cu", "state_scan": "gma_mix.cu", "state_reduce": "gma_mix.cu",
    "chunk_out": "gma_mix.cu", "bidir_read": "gma_mix.cu", "decode": "gma_decode.cu",
}


def traffic_record(stage, wl):
    """DRAM bytes per launch of `stage` on workload `wl` from the committed ncu
    summary, or None if the kernel's source changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    h = source_hash(stage, wl)
    for line in open(path):
        f = line.split()
        if len(f) >= 4 and not line.startswith("#") and f[0] == stage and f[1] == h and f[2] == wl.name:
            return float(f[3])
    return None


def source_hash(stage, wl):
    d = os.path.join(ROOT, "gaussian_mixture_sequence_gb300", "csrc")
    src = KERNEL_SOURCE.get(stage)
    if src is None:  # routing: the pruned kernel, the tensor-core kernels, else the generic one
        src = "gma_resp_tc.cu" if bounded_routing(wl) else ("gma_resp_gtc.cu" if tc_routing(wl) else "gma_resp.cu")
    if stage in ("state_scan", "state_reduce") and eff_chunk(wl) == 128:   # the tensor-core path's scan
        src = "gma_causal_tc.cu"
    m = hashlib.sha256()
    for fn in ("gma_internal.cuh", "gma_tc.cuh", src):
        m.update(open(os.path.join(d, fn), "rb").read())
    return m.hexdigest()[:16]


def _oracle_call(wl, mu, vr, lp, q, k, v, heads):
    """The oracle's form of the workload on [S, n, .] slices (decode: one step per slice)."""
    import numpy as np
    import oracle
    if wl.mode == "bidir":
        return oracle.bidir(mu, vr, lp, q, k, v, wl.eps, heads=heads)
    if wl.mode == "decode":
        S = q.shape[0]
        state = np.ones((S, wl.K * wl.dv + wl.K))
        return oracle.decode_step(mu, vr, lp, q[:, 0], k[:, 0], v[:, 0], wl.eps, state, heads=heads)
    if wl.mode == "backward":
        g = np.ones_like(v)   # dL/dO: any values cost the same
        return oracle.backward(mu, vr, lp, q, k, v, wl.eps, g, causal=True, heads=heads)
    return oracle.causal(mu, vr, lp, q, k, v, wl.eps, heads=heads)


def _host_slices(wl, S, n):
    """Seeded inputs of the first S (b, h) slices, first n tokens, as [S, n, .] arrays."""
    import numpy as np
    from gaussian_mixture_sequence_gb300 import workloads
    mu, vr, lp = workloads.params(wl)
    qs, ks, vs = [], [], []
    for s_ in range(S):
        b, h = divmod(s_, wl.H)
        q, k, v = workloads.slice_inputs(wl.with_(N=n), b, h, mu=mu)
        qs.append(q); ks.append(k); vs.append(v)
    return mu, vr, lp, np.stack(qs), np.stack(ks), np.stack(vs)


def cpu_baseline(wl):
    """The fp64 oracle as it stands, on a bounded sample of the same workload."""
    import oracle
    nthr = oracle.max_threads()
    if wl.mode == "decode":
        S, n = min(wl.B * wl.H, 1024 * max(1, nthr)), 1
    else:
        S, n = min(wl.B * wl.H, max(8, nthr)), wl.N
    mu, vr, lp, q, k, v = _host_slices(wl, S, n)
    heads = [s_ % wl.H for s_ in range(S)]
    t0 = time.perf_counter()
    reps = 0
    while True:
        _oracle_call(wl, mu, vr, lp, q, k, v, heads)
        reps += 1
        if wl.mode != "decode" or time.perf_counter() - t0 > 2.0:
            break
    dt = (time.perf_counter() - t0) / reps
    tokens = S * n / wl.H
    what = "one decode step of" if wl.mode == "decode" else f"the full length N={wl.N} of"
    return {"value": tokens / dt, "unit": "tokens/s", "cores": min(nthr, S), "kind": "oracle",
            "sample": f"{what} {S} of {wl.B * wl.H} (batch, head) sequences of workload {wl.name} "
                      f"(= {tokens:.0f} tokens of H={wl.H} heads), fp64, {dt:.3f} s wall per pass"}


# ----------------------------------------------------------------- reference --

def run_reference(args, wl, world, rank):
    if rank != 0:
        return
    import oracle
    nthr = oracle.max_threads()
    S = min(wl.B * wl.H, max(1, nthr) * (256 if wl.mode == "decode" else 1))
    heads = [s_ % wl.H for s_ in range(S)]
    if wl.mode == "decode":
        n = 1
    else:
        # size one step (a prefix of n tokens of S sequences) so that the whole run stays near 2 minutes
        mu, vr, lp, q, k, v = _host_slices(wl, S, 256)
        t0 = time.perf_counter()
        _oracle_call(wl, mu, vr, lp, q, k, v, heads)
        per_tok = (time.perf_counter() - t0) / 256
        n = int(max(64, min(wl.N, 120.0 / (args.steps + args.warmup) / max(per_tok, 1e-9))))
    mu, vr, lp, q, k, v = _host_slices(wl, S, n)
    for _ in range(args.warmup):
        _oracle_call(wl, mu, vr, lp, q, k, v, heads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_call(wl, mu, vr, lp, q, k, v, heads)
    dt = (time.perf_counter() - t0) / max(args.steps, 1)
    tokens = S * n / wl.H
    val = tokens / dt
    line = {
        "impl": "reference", "metric": METRIC if wl.mode == "causal" else f"GMA {wl.mode} tokens/sec",
        "value": val, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "B": wl.B, "H": wl.H, "N": wl.N, "d_route": wl.d, "d_v": wl.dv,
                   "K": wl.K, "chunk": eff_chunk(wl)},
        "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": min(nthr, S), "kind": "oracle",
                         "sample": f"each step: first {n} tokens of {S} (batch, head) sequences of {wl.name}"},
        "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------- runners ----

class Runner:
    """Device inputs of one workload and its profiled / plain step.

    Causal and bidirectional workloads use the seeded host generator (the same
    inputs the oracle sees); the decode workload draws its prefill and tokens
    on the device with a seeded torch generator (4 GB per tensor at batch 256
    would take minutes on the host) and builds the state with one causal
    prefill through the library."""

    def __init__(self, wl, dev, seed):
        import torch
        from gaussian_mixture_sequence_gb300 import gma, workloads
        self.wl, self.dev, self.gma = wl, dev, gma
        tdt = lambda s_: torch.bfloat16 if s_ == "bf16" else torch.float32
        mu, vr, lp = workloads.params(wl, seed)
        self.prm = tuple(torch.from_numpy(a).to(dev) for a in (mu, vr, lp))
        self.shape = gma.Shape.make(wl.B, wl.H, wl.N, wl.d, wl.dv, wl.K, chunk=wl.chunk, eps=wl.eps,
                                    x_dtype=wl.x_dtype, v_dtype=wl.v_dtype, gemm_dtype=wl.gemm_dtype)
        if wl.mode == "decode":
            g = torch.Generator(device=dev).manual_seed(seed)
            shp = lambda w: (wl.B, wl.H, wl.N, w)
            q, k, v = (torch.randn(*shp(w), device=dev, generator=g).to(tdt(t))
                       for w, t in ((wl.d, wl.x_dtype), (wl.d, wl.x_dtype), (wl.dv, wl.v_dtype)))
            self.state0 = torch.empty(wl.B, wl.H, wl.K * wl.dv + wl.K, device=dev)
            gma.gma_forward_causal(self.shape, *self.prm, q, k, v, torch.empty(shp(wl.dv), device=dev),
                                   state_out=self.state0)
            del q, k, v
            self.state = self.state0.clone()
            nt = 16   # a ring of decode tokens
            tok = lambda w, t: torch.randn(nt, wl.B, wl.H, w, device=dev, generator=g).to(tdt(t))
            self.tq, self.tk, self.tv = tok(wl.d, wl.x_dtype), tok(wl.d, wl.x_dtype), tok(wl.dv, wl.v_dtype)
            self.h_in = [t[0].cpu().pin_memory() for t in (self.tq, self.tk, self.tv)]
            self.d_in = [t[0].clone() for t in (self.tq, self.tk, self.tv)]
            self.out = torch.empty(wl.B, wl.H, wl.dv, device=dev)
            op = gma.OP_DECODE
        else:
            q, k, v = workloads.full_inputs(wl, seed)
            self.h_in = [torch.from_numpy(q).to(tdt(wl.x_dtype)).pin_memory(),
                         torch.from_numpy(k).to(tdt(wl.x_dtype)).pin_memory(),
                         torch.from_numpy(v).to(tdt(wl.v_dtype)).pin_memory()]
            self.d_in = [t.to(dev) for t in self.h_in]
            self.out = torch.empty(wl.B, wl.H, wl.N, wl.dv, device=dev)
            op = gma.OP_BIDIR if wl.mode == "bidir" else gma.OP_CAUSAL
            if wl.mode == "backward":
                op = gma.OP_BACKWARD
                self.h_in.append(torch.from_numpy(workloads.full_dout(wl, seed)).pin_memory())
                self.d_in.append(self.h_in[-1].to(dev))
                f32 = dict(device=dev, dtype=torch.float32)
                self.grads = (torch.empty(wl.B, wl.H, wl.N, wl.d, **f32), torch.empty(wl.B, wl.H, wl.N, wl.d, **f32),
                              torch.empty(wl.B, wl.H, wl.N, wl.dv, **f32), torch.empty(wl.H, wl.K, wl.d, **f32),
                              torch.empty(wl.H, wl.K, wl.d, **f32), torch.empty(wl.H, wl.K, **f32))
                self.h_grads = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in self.grads]
        self.ws = torch.empty(gma.gma_workspace_size(self.shape, op), dtype=torch.uint8, device=dev)
        self.h_out = torch.empty(self.out.shape, dtype=self.out.dtype).pin_memory()
        self.host_ws = (torch.empty(gma.gma_workspace_size(self.shape, gma.OP_CAUSAL_HOST), dtype=torch.uint8,
                                    device=dev) if wl.mode == "causal" else None)   # the host-buffer entry's
        self.i = 0

    def profiled(self, evs):
        g, wl = self.gma, self.wl
        if wl.mode == "backward":   # one launch sequence, timed as one stage
            import torch
            st = torch.cuda.current_stream(self.dev)
            evs[0].record(st)
            g.gma_backward(self.shape, *self.prm, *self.d_in, *self.grads, causal=True, ws=self.ws)
            evs[1].record(st)
            return ["backward"]
        if wl.mode == "decode":
            t = self.i % self.tq.shape[0]
            self.i += 1
            return g.gma_decode_step_profiled(self.shape, *self.prm, self.tq[t], self.tk[t], self.tv[t],
                                              self.state, self.out, evs, ws=self.ws)
        q, k, v = self.d_in
        if wl.mode == "bidir":
            return g.gma_forward_bidir_profiled(self.shape, *self.prm, q, k, v, self.out, evs, ws=self.ws)
        return g.gma_forward_causal_profiled(self.shape, *self.prm, q, k, v, self.out, evs, ws=self.ws)

    def e2e_step(self):
        """One step with host inputs in and the result out: the causal form through the
        host-buffer entry point (which overlaps its copies with the computation), the
        other forms through the plain entry points with the copies around them."""
        g, wl = self.gma, self.wl
        if wl.mode == "causal":
            g.gma_forward_causal_host(self.shape, *self.prm, *self.h_in, self.h_out, ws=self.host_ws)
            return
        for d, h in zip(self.d_in, self.h_in):
            d.copy_(h, non_blocking=True)
        if wl.mode == "backward":
            g.gma_backward(self.shape, *self.prm, *self.d_in, *self.grads, causal=True, ws=self.ws)
            for h, d in zip(self.h_grads, self.grads):
                h.copy_(d, non_blocking=True)
            return
        q, k, v = self.d_in
        if wl.mode == "decode":
            g.gma_decode_step(self.shape, *self.prm, q, k, v, self.state, self.out, ws=self.ws)
        elif wl.mode == "bidir":
            g.gma_forward_bidir(self.shape, *self.prm, q, k, v, self.out, ws=self.ws)
        else:
            g.gma_forward_causal(self.shape, *self.prm, q, k, v, self.out, ws=self.ws)
        self.h_out.copy_(self.out, non_blocking=True)

    def kept_per_row(self):
        """(mean number of components with a non-zero posterior per routing row
        outside the dense tiles -- the components the bounded routing evaluates
        exactly --, fraction of rows with every posterior non-zero -- the rows of
        the tiles the dense pass takes), from one responsibilities call on the Q_X
        and K_X rows outside the timed region."""
        import torch
        g, wl = self.gma, self.wl
        kept, dense = 0.0, 0.0
        for x in self.d_in[:2]:
            gam = torch.empty(wl.B, wl.H, wl.N, wl.K, device=self.dev)
            g.gma_responsibilities(self.shape, *self.prm, x, gam)
            cnt = (gam > 0).sum(-1)
            full = cnt == wl.K
            dense += full.float().mean().item()
            rest = cnt[~full]
            kept += rest.float().mean().item() if rest.numel() else 0.0
            del gam
        return kept / 2, dense / 2

    def resident_bytes(self):
        """Bytes a step streams from HBM that a repeat could find in L2: the state of the
        decode step, the device inputs otherwise."""
        wl = self.wl
        if wl.mode == "decode":
            return wl.B * wl.H * (wl.K * wl.dv + wl.K) * 4
        return self.io_bytes()[0]

    def io_bytes(self):
        out = (sum(t.numel() * t.element_size() for t in self.h_grads) if self.wl.mode == "backward"
               else self.h_out.numel() * self.h_out.element_size())
        return sum(t.numel() * t.element_size() for t in self.h_in), out


# ----------------------------------------------------------------- main -------

def main():
    args = parse()
    world, rank, local = dist_env()
    from gaussian_mixture_sequence_gb300 import workloads
    wl = workloads.WORKLOADS[args.workload]
    if args.batch > 0:
        wl = wl.with_(B=args.batch)
    if args.impl == "reference":
        return run_reference(args, wl, world, rank)

    import torch
    from gaussian_mixture_sequence_gb300 import gma

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    gma.load()
    run = Runner(wl, dev, replica_seed(wl, rank))
    stream = torch.cuda.current_stream(dev)
    NE = gma.PROFILE_MAX_STAGES + 1

    def new_events():
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(NE)]
        for e in evs:
            e.record(stream)
        return evs

    step_events = [new_events() for _ in range(args.steps)]
    warm_events = new_events()
    torch.cuda.synchronize(dev)

    props = torch.cuda.get_device_properties(dev)
    uuid = str(getattr(props, "uuid", ""))
    clocks = ClockSampler(("GPU-" + uuid) if uuid and not uuid.startswith("GPU-") else (uuid or str(local)))
    # warm-up: exactly --warmup steps
    for i in range(args.warmup):
        run.profiled(warm_events)
        if i % 20 == 19:
            torch.cuda.synchronize(dev)
    torch.cuda.synchronize(dev)
    # clock soak: untimed steps right before the timed region, so that nvidia-smi samples the
    # clocks under this load (a timed region of a few ms holds no 100 ms sample of its own)
    t_soak0 = time.time()
    n_soak = 0
    while time.time() - t_soak0 < args.clock_soak_s:
        run.profiled(warm_events)
        n_soak += 1
        if n_soak % 20 == 0:
            torch.cuda.synchronize(dev)
    torch.cuda.synchronize(dev)
    soak_s = time.time() - t_soak0

    # a step whose data would fit in L2 is preceded by a write of twice the L2 size; the
    # step's own events (before its first launch, after its last) then exclude that write
    l2 = int(getattr(props, "L2_cache_size", 0) or 129 * 2**20)
    resident = run.resident_bytes()
    flush = resident < 1.5 * l2
    fbuf = torch.empty(2 * l2 // 4, dtype=torch.float32, device=dev) if flush else None
    if pg:
        pg.barrier()
    torch.cuda.synchronize(dev)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_host0 = time.time()
    start.record(stream)
    names = None
    for i in range(args.steps):
        if flush:
            fbuf.zero_()
        names = run.profiled(step_events[i])
    end.record(stream)
    torch.cuda.synchronize(dev)
    t_host1 = time.time()
    if pg:
        pg.barrier()
    if flush:
        step_sum = sum(step_events[i][0].elapsed_time(step_events[i][len(names)]) for i in range(args.steps))
        total_ms = max_over_ranks(pg, step_sum, dev)
    else:
        total_ms = max_over_ranks(pg, start.elapsed_time(end), dev)
    clocks_summary = clocks.summary(t_host0, t_host1, t_soak0)

    ms = total_ms / args.steps
    tokens = tokens_per_step(wl)
    value = whole_job_rate(world, tokens, ms)
    stage_ms = {}
    for i, nm in enumerate(names):
        stage_ms[nm] = statistics.mean(step_events[s_][i].elapsed_time(step_events[s_][i + 1])
                                       for s_ in range(args.steps))
    dom = max(stage_ms, key=stage_ms.get)
    pk, pk_kind = peaks()
    kept, dense = (run.kept_per_row() if (bounded_routing(wl) and wl.mode in ("causal", "bidir"))
                   else (None, None))
    roof = roofline_of(dom, wl, stage_ms[dom] * 1e-3, pk, kept, dense)
    roof_s, roof_parts = path_roofline_s(wl, pk, kept, dense)

    # end to end through the plain public entry point: pinned host inputs in, result out, every step
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ne = max(1, min(args.e2e_steps, args.steps))
    for _ in range(2):   # untimed: the first calls create the copy streams and load the kernels
        run.e2e_step()
    torch.cuda.synchronize(dev)
    if pg:
        pg.barrier()
    e_start.record(stream)
    for _ in range(ne):
        run.e2e_step()
    e_end.record(stream)
    torch.cuda.synchronize(dev)
    e_ms = max_over_ranks(pg, e_start.elapsed_time(e_end) / ne, dev)
    clocks.stop()
    h2d, d2h = run.io_bytes()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wl)

    if rank == 0:
        tr = traffic_record(dom, wl)
        cfg = {"workload": wl.name, "mode": wl.mode, "B": wl.B, "H": wl.H, "N": wl.N, "d_route": wl.d,
               "d_v": wl.dv, "K": wl.K, "x_dtype": wl.x_dtype, "gemm_dtype": wl.gemm_dtype,
               "inputs": "peaked mixture around the K centres" if wl.dist == "peaked" else "N(0,1)"}
        what = "state" if wl.mode == "decode" else "inputs"
        if wl.mode == "decode":
            cfg["prefill"] = f"{wl.N} tokens (causal, on device)"
        else:
            cfg["chunk"] = eff_chunk(wl)
        if flush:
            cfg["l2"] = ("%s %.0f MB per step, under 1.5x L2 (%.0f MB): L2 flushed by a %.0f MB write before "
                         "each timed step, outside the step's events" % (what, resident / 1e6, l2 / 1e6, 2 * l2 / 1e6))
        else:
            cfg["l2"] = "%s %.0f MB per step, over 1.5x L2 (%.0f MB), no flush" % (what, resident / 1e6, l2 / 1e6)
        line = {
            "metric": METRIC if wl.mode == "causal" else f"GMA {wl.mode} tokens/sec ({wl.name})",
            "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32" if wl.gemm_dtype == "f32" else "f32+bf16",
            "data": "synthetic", "config": cfg,
            "roofline": {**roof, "traffic": tr,
                         "peak_source": ("152 SMs x 128 FP32 lanes x 2 x max SM clock (%s)" % pk_kind)
                         if roof["bound"] == "alu" else pk_kind},
            "path_roofline": {"tokens_per_s": tokens / roof_s, "frac": value / world / (tokens / roof_s),
                              **{k2.replace("_s", "_ms"): v2 * 1e3 for k2, v2 in roof_parts.items()},
                              "kept_components_per_row": kept, "dense_row_fraction": dense},
            "stages_ms": stage_ms,
            "gpu_launches": len(names) * args.steps,
            "clocks": clocks_summary,
            "clock_soak": {"steps": n_soak, "s": round(soak_s, 3)},
            "e2e": {"value": whole_job_rate(world, tokens, e_ms), "unit": "tokens/s", "ms_per_step": e_ms,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "entry": "gma_forward_causal_host" if wl.mode == "causal" else "device entry + torch copies"},
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if pg:
        pg.barrier()
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
