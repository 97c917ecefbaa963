"""Benchmark of the ternary pq2_0 x q8_K hot path on GB300.

One step = one pass of the hot path over one batch of synthetic input:
quantize the activations to q8_K, then the ternary matmul, through
tq_quantize_matmul (one fused launch up to 8 tokens; the load-time repack
runs once, before timing, and is reported separately). The headline
workload is the decode GEMV (32768 x 8192 weights, 1 token), measured in
Gweights/s; the 4-token and 64-token 17408 x 5120 tiles are measured in the
same run in GMAC/s, and the 64-block decode-step replay (23.82 G weights,
6.33 GB per step) at 1 and 512 tokens.

Timing: inputs resident in HBM; W >= 3 warm-up steps; K timed steps replayed
from a CUDA graph on one stream, bracketed by a barrier and a device
synchronize, timed with CUDA events, max over ranks. Weights rotate over
copies whose total exceeds twice the 129 MB L2, so every step streams its
weights from HBM. The GEMV's own duration is taken from events around each of
its launches inside the timed graph. `e2e` repeats the step through the
C ABI with host buffers (tq_matmul_host): pinned host -> device copy of the
activations, quantize, matmul, device -> pinned host copy of the outputs,
every step.

`--impl reference` times the plain C oracle on the host cores instead (a row
sample of the same workload per step).

Multi-GPU (torchrun): each rank runs its own copy of the workload on its own
GPU (weak scaling, no collective on the data path); the reported time is the
maximum over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

L2_BYTES = 129 * 1024 * 1024
PAGES_DECODE_GWEIGHTS = 390.5   # ciot README: t2x4 NEON, 32768 x 8192 matvec, 8 Oryon cores
# GB300 HBM3e nominal bandwidth (GB/s): context beside the measured copy peak.
HBM_NOMINAL_GBS = 7900.0
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# The tensor-core matmul runs e4m3 MMAs: its peak is the measured bf16 dense
# rate times the nominal e4m3 : bf16 ratio (4.5 : 2.25 PFLOP/s dense).
E4M3_PER_BF16 = 2.0


def mma_flops_per_flop(ntok: int) -> float:
    """MMA flops the tensor-core matmul executes per algorithmic flop: 2 (each
    int8 activation split exactly into two e4m3 parts, two MMA columns), a
    quarter more on 64-token tiles (a fifth MMA per group adds the activation
    sums), times the padding of the last token tile (16, 32 or 64 tokens)."""
    tile = 16 if ntok <= 16 else 32 if ntok <= 32 else 64
    padded = -(-ntok // tile) * tile
    return (2.5 if tile == 64 else 2.0) * padded / ntok

# Token counts the workspace forms (every call the benchmark makes) run as a
# GEMV, one weight pass: one fused launch, or from 4 tokens, where the
# workspace size is not 0 (3072 to 19968 columns), two (one kernel quantizes
# and stages the activations in the workspace, then the GEMV); above, two
# launches too (quantize and pack, then the tensor-core kernel). The forms
# without a workspace run the GEMV up to 16 tokens.
GEMV_MAX_TOKENS = 8


def staged(rows: int, cols: int, ntok: int) -> bool:
    import bit_matvec_gb300 as tq
    return ntok <= GEMV_MAX_TOKENS and tq.tq_matmul_workspace_bytes(rows, cols, ntok) > 0


def launches_per_matmul(rows: int, cols: int, ntok: int) -> int:
    """Kernels one tq_quantize_matmul call launches (for the shapes benchmarked: a
    GEMV whose activations fit its shared memory, or the tensor cores)."""
    return 2 if ntok > GEMV_MAX_TOKENS or staged(rows, cols, ntok) else 1


def gemv_kernel_name(rows: int, cols: int, ntok: int) -> str:
    if not staged(rows, cols, ntok):
        return "gemv_kernel (quantize fused in)"
    return "gemv_stage_kernel + gemv_mma_kernel (activations quantized and staged once)"

WORKLOADS = {
    "decode": "decode GEMV 32768x8192 pq2_0 x q8_K, ntok=1",
    "small_batch": "small-batch 17408x5120 pq2_0 x q8_K, ntok=4",
    "prefill": "prefill tile 17408x5120 pq2_0 x q8_K, ntok=64 (1% outliers x10)",
}


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20000)
    p.add_argument("--warmup", type=int, default=200)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default="decode", choices=list(WORKLOADS))
    p.add_argument("--no-extra", action="store_true", help="skip the 4- and 64-token tiles")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--e2e-streams", type=int, default=4,
                   help="streams the end-to-end steps alternate over (requests in flight)")
    p.add_argument("--no-cpu", action="store_true", help="skip the oracle CPU baseline")
    p.add_argument("--no-replay", action="store_true",
                   help="skip the 64-block decode-step replay (ntok 1 and 512)")
    p.add_argument("--no-read-ceiling", action="store_true",
                   help="skip the read-ceiling probe beside the GEMV's roofline")
    p.add_argument("--tensor-rates", action="store_true",
                   help="only measure library int8 / bf16 / f16 GEMM rates (operand-type choice)")
    return p.parse_args()


# ---------------------------------------------------------------- distributed plumbing

def dist_init(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if os.environ.get("TQ_BENCH_BACKEND", "nccl") == "nccl" else "gloo"
        dist.init_process_group(backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Largest value of x over all ranks (timing only, not the data path)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- peaks and clocks

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clock and throttle-reason samples every 100 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [v.strip() for v in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for name, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- workloads

def algorithmic_bytes(rows, cols, ntok):
    """What one matmul must move: packed weights, q8_K activations, f32 outputs."""
    w = rows * cols // 128 * 34
    x = ntok * cols // 256 * 292
    y = ntok * rows * 4
    return w + x + y


def quantize_bytes(ntok, cols):
    return ntok * cols * 4 + ntok * cols // 256 * 292


class Workload:
    def __init__(self, name, device):
        import torch
        import bit_matvec_gb300 as tq
        wpq, x, cfg = synth.workload(name)
        self.name, self.cfg = name, cfg
        self.rows, self.cols, self.ntok = cfg["rows"], cfg["cols"], cfg["ntok"]
        W = torch.from_numpy(wpq).to(device)
        wtq = tq.repacked_empty(self.rows, self.cols, device)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        tq.tq_repack(W, wtq, self.rows, self.cols)
        torch.cuda.synchronize()
        self.repack_s = time.perf_counter() - t0
        del W
        nbytes = wtq.numel()
        self.copies = max(2, -(-2 * L2_BYTES // nbytes) + 1)
        self.W = [wtq] + [wtq.clone() for _ in range(self.copies - 1)]
        self.x_host = x
        self.X = torch.from_numpy(x).to(device)
        self.Xq = tq.q8K_empty(self.ntok, self.cols, device)
        self.Y = torch.empty((self.ntok, self.rows), dtype=torch.float32, device=device)
        self.ws = tq.workspace_empty(self.rows, self.cols, self.ntok, device)
        self.device = device

    def step(self, i, stream=None):
        """quantize + matmul (one fused launch where nothing is staged)."""
        import bit_matvec_gb300 as tq
        tq.tq_quantize_matmul(self.W[i % self.copies], self.X, self.Xq, self.Y, self.rows,
                              self.cols, self.ntok, self.ws, stream)

    def matmul_only(self, i, stream=None):
        """The dominant kernel alone: for ntok <= GEMV_MAX_TOKENS the whole step (the
        fused GEMV, or the staging kernel and the GEMV), the workspace tensor-core
        matmul otherwise."""
        import bit_matvec_gb300 as tq
        if self.ntok <= GEMV_MAX_TOKENS:
            self.step(i, stream)
        else:
            tq.tq_matmul_ws(self.W[i % self.copies], self.Xq, self.Y, self.rows, self.cols,
                            self.ntok, self.ws, stream)

    def launches(self):
        # tq_quantize_matmul: one fused GEMV launch, or a staging (or
        # quantize-and-pack) kernel, then the GEMV (or tensor cores)
        return launches_per_matmul(self.rows, self.cols, self.ntok)

    def weights(self):
        return self.rows * self.cols

    def macs(self):
        return self.rows * self.cols * self.ntok


class ReplayWorkload:
    """The decode-step replay: 64 blocks x {Wqkv 15360x5120, Wo 5120x5120,
    W_gate and W_up 17408x5120, W_down 5120x17408} (23.82 G weights, 6.33 GB in
    64 x 5 distinct allocations, so every step streams them from HBM; each
    block's allocations hold copies of one synthetic block). One step = for
    every block and matrix: quantize that matrix's activations, matmul. The
    activations of a matrix are one seeded batch shared by the 64 blocks."""

    def __init__(self, ntok, device, blocks=synth.REPLAY_BLOCKS):
        import torch
        import bit_matvec_gb300 as tq
        self.ntok, self.blocks, self.device = ntok, blocks, device
        self.mats = []
        need = 0
        for m in range(len(synth.REPLAY_BLOCK)):
            wpq, x, rows, cols = synth.replay_matrix(m, ntok)
            W = torch.from_numpy(wpq).to(device)
            wtq = tq.repacked_empty(rows, cols, device)
            tq.tq_repack(W, wtq, rows, cols)
            torch.cuda.synchronize(device)
            del W
            self.mats.append(dict(
                rows=rows, cols=cols, W=[wtq] + [wtq.clone() for _ in range(blocks - 1)],
                X=torch.from_numpy(x).to(device), Xq=tq.q8K_empty(ntok, cols, device),
                Y=torch.empty((ntok, rows), dtype=torch.float32, device=device)))
            need = max(need, tq.tq_matmul_workspace_bytes(rows, cols, ntok))
        self.ws = torch.empty(max(1, need), dtype=torch.uint8, device=device)

    def step(self, stream=None):
        import bit_matvec_gb300 as tq
        for b in range(self.blocks):
            for m in self.mats:
                tq.tq_quantize_matmul(m["W"][b], m["X"], m["Xq"], m["Y"], m["rows"], m["cols"],
                                      self.ntok, self.ws, stream)

    def launches(self):
        return self.blocks * sum(launches_per_matmul(m["rows"], m["cols"], self.ntok)
                                 for m in self.mats)

    def weights(self):
        return self.blocks * sum(m["rows"] * m["cols"] for m in self.mats)

    def weight_bytes(self):
        return self.blocks * sum(m["W"][0].numel() for m in self.mats)

    def algorithmic_bytes(self):
        return self.blocks * sum(algorithmic_bytes(m["rows"], m["cols"], self.ntok)
                                 for m in self.mats)


def replay_read_ceiling(wl, steps, warmup, stream):
    """The same step's weight reads by the read-ceiling probe instead of the
    matmuls: one tq_probe_read_sum launch per matrix and block, in the step's
    order, each allowed to read before the one ahead of it ends (as the
    replay's GEMVs do), from one CUDA graph. The most any kernel that reads
    each matrix once per launch can expect."""
    import torch
    import bit_matvec_gb300 as tq
    out = torch.zeros(1, dtype=torch.int32, device=wl.device)

    def probe_step():
        for b in range(wl.blocks):
            for m in wl.mats:
                tq.tq_probe_read_sum(m["W"][b], out, True, stream)

    probe_step()
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        probe_step()
    for _ in range(max(warmup, 3)):
        g.replay()
    stream.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(steps):
        g.replay()
    end.record(stream)
    stream.synchronize()
    return start.elapsed_time(end) / steps


def measure_replay(ntok, steps, warmup, world, device, peaks, peak_kind, read_ceiling=False):
    """Device time of whole replay steps from one CUDA graph per step."""
    import torch
    wl = ReplayWorkload(ntok, device)
    stream = torch.cuda.Stream(device=device)
    stream.wait_stream(torch.cuda.current_stream(device))
    with torch.cuda.stream(stream):
        wl.step(stream)                                 # un-captured warm-up (kernel attributes)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            wl.step(stream)
        for _ in range(max(warmup, 3)):
            g.replay()
        stream.synchronize()
        barrier(world)
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for _ in range(steps):
            g.replay()
        end.record(stream)
        stream.synchronize()
        ms = max_over_ranks(start.elapsed_time(end) / steps, world, device)
        rc_ms = replay_read_ceiling(wl, steps, warmup, stream) if read_ceiling else None
    res = {"workload": f"decode-step replay, {wl.blocks} blocks x 5 matrices, ntok={ntok}",
           "ntok": ntok, "ms_per_step": ms, "steps": steps, "launches_per_step": wl.launches(),
           "weights_per_step": wl.weights(), "weight_bytes_per_step": wl.weight_bytes(),
           "timing": "CUDA graph of one whole step, CUDA events"}
    if ntok == 1:
        res["gweights_per_s"] = world * wl.weights() / (ms * 1e-3) / 1e9
        achieved = wl.algorithmic_bytes() / (ms * 1e-3) / 1e9
        peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
        res["roofline"] = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                           "frac": achieved / peak, "peak_source": peak_kind,
                           "frac_of_nominal": achieved / HBM_NOMINAL_GBS,
                           "note": "whole step (quantize + matmul launches) over algorithmic bytes"}
        if rc_ms is not None:
            wb = wl.weight_bytes()
            res["read_ceiling"] = {
                "ms_per_step": rc_ms, "bytes": wb, "gbs": wb / (rc_ms * 1e-3) / 1e9,
                "frac": wb / (rc_ms * 1e-3) / 1e9 / peak,
                "replay_vs_ceiling": rc_ms / ms,
                "how": "tq_probe_read_sum over the same weight buffers, one launch per matrix "
                       "and block in the step's order, reading early, one CUDA graph"}
    else:
        res["gmac_per_s"] = world * wl.weights() * ntok / (ms * 1e-3) / 1e9
        achieved = 2.0 * wl.weights() * ntok / (ms * 1e-3) / 1e12
        peak = E4M3_PER_BF16 * float(peaks.get("bf16_tflops_sustained",
                                               FALLBACK_PEAKS["bf16_tflops_sustained"]))
        res["roofline"] = {"bound": "tensor", "achieved": achieved, "peak": peak,
                           "unit": "TFLOP/s", "frac": achieved / peak,
                           "mma_busy_frac": achieved * mma_flops_per_flop(ntok) / peak,
                           "peak_source": f"{peak_kind} bf16 dense sustained (a long step) "
                                          f"x {E4M3_PER_BF16:g} (e4m3 : bf16 nominal)"}
    del wl
    torch.cuda.empty_cache()
    return res


def measure_read_ceiling(nbytes, device, warmup):
    """Read rate of the probe kernel (tq_probe_read_sum: a streaming sum, no
    other work) over buffers of nbytes rotating through more than twice the
    L2, in graphs of back-to-back launches: 'chained' lets each launch read
    before the previous one ends (as the independent GEMV chain does), and
    'wait_first' makes each wait for it first."""
    import torch
    import bit_matvec_gb300 as tq
    copies = max(2, -(-2 * L2_BYTES // nbytes) + 1)
    bufs = [torch.full((nbytes // 4,), i + 1, dtype=torch.int32, device=device)
            for i in range(copies)]
    out = torch.zeros(1, dtype=torch.int32, device=device)
    stream = torch.cuda.Stream(device=device)
    stream.wait_stream(torch.cuda.current_stream(device))
    G = copies * max(1, STEPS_PER_GRAPH // copies)
    res = {"bytes": nbytes, "copies": copies}
    with torch.cuda.stream(stream):
        for early in (True, False):
            for i in range(copies):
                tq.tq_probe_read_sum(bufs[i], out, early, stream)
            stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in range(G):
                    tq.tq_probe_read_sum(bufs[i % copies], out, early, stream)
            for _ in range(max(3, warmup // G + 1)):
                g.replay()
            stream.synchronize()
            reps = max(5, int(2e9 // (nbytes * G)))
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(reps):
                g.replay()
            b.record(stream)
            stream.synchronize()
            us = a.elapsed_time(b) / (reps * G) * 1e3
            res["chained" if early else "wait_first"] = {"us": us, "gbs": nbytes / us / 1e3}
    del bufs
    torch.cuda.empty_cache()
    return res


def measure_ptq1_stream(steps, warmup, world, device, peaks, peak_kind, ref_kernel_ms):
    """The decode workload's weights as the 1.75-bit ptq1_0 file, streamed and
    decoded by the GEMV itself (tq_matmul_ptq1_0_stream, one token), timed like
    the headline's matmul launches: back-to-back launches in graphs, weights
    rotating over copies larger than twice the L2."""
    import torch
    import bit_matvec_gb300 as tq
    cfg = synth.CONFIGS["decode"]
    rows, cols = cfg["rows"], cfg["cols"]
    s = synth.seeds(cfg["index"])
    wpt = synth.pack_ptq1_0(synth.ternary_codes(rows, cols, s["weights"]),
                            synth.group_scales(rows, cols, s["scales"]))
    W = torch.from_numpy(wpt).to(device)
    del wpt
    wt1 = torch.empty(tq.tq_ptq1_0_stream_bytes(rows, cols), dtype=torch.uint8, device=device)
    tq.tq_repack_ptq1_0_stream(W, wt1, rows, cols)
    del W
    copies = max(2, -(-2 * L2_BYTES // wt1.numel()) + 1)
    Ws = [wt1] + [wt1.clone() for _ in range(copies - 1)]
    X = torch.from_numpy(synth.activations(1, cols, s["acts"])).to(device)
    Xq = tq.q8K_empty(1, cols, device)
    tq.tq_quantize_q8K(X, Xq, 1, cols)
    Y = torch.empty((1, rows), dtype=torch.float32, device=device)
    stream = torch.cuda.Stream(device=device)
    stream.wait_stream(torch.cuda.current_stream(device))
    G = copies * max(1, STEPS_PER_GRAPH // copies)
    reps = max(1, steps // G)
    with torch.cuda.stream(stream):
        for i in range(max(warmup, 3)):
            tq.tq_matmul_ptq1_0_stream(Ws[i % copies], Xq, Y, rows, cols, 1, stream)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(G):
                tq.tq_matmul_ptq1_0_stream(Ws[i % copies], Xq, Y, rows, cols, 1, stream)
        for _ in range(3):
            g.replay()
        stream.synchronize()
        barrier(world)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            g.replay()
        b.record(stream)
        stream.synchronize()
    ms = max_over_ranks(a.elapsed_time(b) / (reps * G), world, device)
    wbytes = wt1.numel()
    abytes = wbytes + cols // 256 * 292 + rows * 4
    peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    res = {"workload": "decode GEMV 32768x8192 as the 1.75-bit ptq1_0 file, streamed and decoded "
                       "in the kernel, ntok=1",
           "ms_per_launch": ms, "launches": reps * G,
           "gweights_per_s": world * rows * cols / (ms * 1e-3) / 1e9,
           "weight_bytes": wbytes, "weight_gbs": wbytes / (ms * 1e-3) / 1e9,
           "roofline": {"bound": "hbm", "achieved": abytes / (ms * 1e-3) / 1e9, "peak": peak,
                        "unit": "GB/s", "frac": abytes / (ms * 1e-3) / 1e9 / peak,
                        "peak_source": peak_kind},
           "time_vs_2bit_stream": ms / ref_kernel_ms if ref_kernel_ms else None,
           "timing": f"graphs of {G} back-to-back launches, CUDA events"}
    del Ws
    torch.cuda.empty_cache()
    return res


# Steps per captured graph (a multiple of the weight copies): a decode graph
# holds many matmuls back to back, and consecutive kernels overlap only within
# one graph launch.
STEPS_PER_GRAPH = 40


def graph_plan(steps: int, copies: int):
    """(G, replays of the G-step graph, steps left for a second graph): G is the
    largest multiple of `copies` up to STEPS_PER_GRAPH (at least `copies`), and
    replays * G + rest == steps exactly."""
    G = copies * max(1, STEPS_PER_GRAPH // copies)
    reps, rest = divmod(steps, G)
    return G, reps, rest


def time_graph(wl: Workload, steps: int, warmup: int, world: int):
    """Device time per step, and the matmul kernel's average launch duration.

    Graph A holds G steps (quantize + matmul, cycling over the weight copies;
    G = the largest multiple of `copies` up to STEPS_PER_GRAPH, at least
    `copies`), and graph A' the steps % G left over: A replayed steps // G
    times and A' once, between two events, time exactly `steps` steps, with
    consecutive kernels overlapping as they do in a real decode (programmatic
    dependent launch). Graphs M and M' hold the matmul launches alone and are
    replayed the same way: the timed region's length over its launches is the
    kernel's average launch duration. Graph B (`copies` steps with events
    around each matmul, which serialise the kernels) gives the isolated
    per-launch time too.
    """
    import torch
    import bit_matvec_gb300 as tq
    stream = torch.cuda.Stream(device=wl.device)
    stream.wait_stream(torch.cuda.current_stream(wl.device))
    n = wl.copies

    def timing_event():
        try:   # recorded inside a graph as an external event node, readable after replay
            return torch.cuda.Event(enable_timing=True, external=True)
        except TypeError:
            return torch.cuda.Event(enable_timing=True)

    ev = [(timing_event(), timing_event()) for _ in range(n)]

    G, reps, rest = graph_plan(steps, n)

    # Dependent chain: step k > 0 of a graph quantizes the previous step's
    # output (its first ntok x cols values) instead of the seeded activations,
    # so each launch must wait for the one before it before reading them (its
    # weights, which no step writes, may still be requested first). Two output
    # buffers alternate; every graph launch starts again from the seeded X.
    import bit_matvec_gb300 as tq_mod
    need = wl.ntok * wl.cols
    if wl.ntok * wl.rows >= need:
        Yd = [torch.empty_like(wl.Y) for _ in range(2)]

        def dep_step(i, s):
            k = i % G
            X = wl.X if k == 0 else Yd[(k - 1) % 2].view(-1)[:need].view(wl.ntok, wl.cols)
            tq_mod.tq_quantize_matmul(wl.W[i % wl.copies], X, wl.Xq, Yd[k % 2], wl.rows, wl.cols,
                                      wl.ntok, wl.ws, s)
    else:
        dep_step = None

    def timed(graph, graph_rest):
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for _ in range(reps):
            graph.replay()
        if graph_rest is not None:
            graph_rest.replay()
        end.record(stream)
        stream.synchronize()
        return start.elapsed_time(end)

    def capture(fn, count):
        if count == 0:
            return None
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(count):
                fn(i, stream)
        return g

    with torch.cuda.stream(stream):
        for i in range(max(warmup, 3)):                 # un-captured warm-up (kernel attributes)
            wl.step(i, stream)
        stream.synchronize()
        ga, ga_rest = capture(wl.step, G), capture(wl.step, rest)
        gm, gm_rest = capture(wl.matmul_only, G), capture(wl.matmul_only, rest)
        gd, gd_rest = ((capture(dep_step, G), capture(dep_step, rest)) if dep_step
                       else (None, None))
        gb = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gb, stream=stream):
            for i in range(n):
                if wl.ntok > GEMV_MAX_TOKENS:
                    tq.tq_quantize_q8K(wl.X, wl.Xq, wl.ntok, wl.cols, stream)
                ev[i][0].record(stream)
                wl.matmul_only(i, stream)
                ev[i][1].record(stream)
        for g in (ga, gm, gb, gd):                      # graph warm-up replays
            if g is not None:
                for _ in range(max(1, -(-warmup // G))):
                    g.replay()
        for g in (ga_rest, gm_rest, gd_rest):
            if g is not None:
                g.replay()
        stream.synchronize()
        barrier(world)
        torch.cuda.synchronize(wl.device)
        total_ms = timed(ga, ga_rest)
        kern_ms = timed(gm, gm_rest) / steps
        dep_ms = timed(gd, gd_rest) / steps if gd is not None else None
        gb.replay()
        stream.synchronize()
        try:
            serial_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
        except RuntimeError:
            serial_ms = None
        barrier(world)
    how = (f"timed graphs of back-to-back matmul launches ({G} per graph, events around "
           f"the region)")
    return total_ms / steps, kern_ms, steps, how, serial_ms, dep_ms


def time_e2e(wl: Workload, steps: int, warmup: int, nstreams: int):
    """Through the C ABI with host buffers: one tq_matmul_host call per step
    (pinned host X -> device, quantize, matmul, device -> pinned host Y). Steps
    alternate over nstreams streams, each with its own host and device
    buffers, as a server pipelines independent requests: one step's copies run
    while another step's kernels do; every step still copies its own input in
    and its own result out."""
    import torch
    import bit_matvec_gb300 as tq
    lanes = []
    for _ in range(nstreams):
        lanes.append({
            "stream": torch.cuda.Stream(wl.device),
            "x_pin": torch.from_numpy(wl.x_host).pin_memory(),
            "y_pin": torch.empty((wl.ntok, wl.rows), dtype=torch.float32).pin_memory(),
            "X": torch.empty_like(wl.X), "Xq": torch.empty_like(wl.Xq),
            "Y": torch.empty_like(wl.Y), "ws": torch.empty_like(wl.ws)})

    def one(i):
        ln = lanes[i % nstreams]
        tq.tq_matmul_host(wl.W[i % wl.copies], ln["x_pin"], ln["X"], ln["Xq"], ln["Y"],
                          ln["y_pin"], wl.rows, wl.cols, wl.ntok, ln["ws"], ln["stream"])

    for i in range(max(warmup, 3)):
        one(i)
    torch.cuda.synchronize(wl.device)
    t0 = time.perf_counter()
    for i in range(steps):
        one(i)
    torch.cuda.synchronize(wl.device)
    dt = time.perf_counter() - t0
    return dt / steps, lanes[0]["x_pin"].numel() * 4, lanes[0]["y_pin"].numel() * 4


# ---------------------------------------------------------------- oracle timing

def cpu_info():
    """Host cores and CPU model of the machine the oracle is timed on."""
    model = None
    try:
        out = subprocess.run(["lscpu"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                             text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().lower().startswith("model name:"):
                model = ln.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if model is None:
        try:
            with open("/proc/cpuinfo") as f:
                for ln in f:
                    if ln.lower().startswith(("model name", "cpu part")):
                        model = ln.split(":", 1)[1].strip()
                        break
        except OSError:
            pass
    import platform
    return {"nproc": os.cpu_count(), "model": model, "machine": platform.machine()}


def _timed_loop(fn, budget_s):
    """Seconds per call of fn, repeated until budget_s has passed (at least once)."""
    n = 0
    t0 = time.perf_counter()
    while True:
        fn()
        n += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    return (time.perf_counter() - t0) / n, n


def oracle_matrix_time(rows, cols, ntok, x, seed_index, budget_s):
    """Estimated single-core seconds of the oracle for quantize + matmul of the
    whole rows x cols matrix: the quantizer timed on all of x, the matmul on a
    sample of rows scaled up by rows / sample (the matmul's time is linear in
    the rows). Returns (seconds, description)."""
    import oracle
    oracle.build()
    rpc = max(1, min(rows, (1 << 22) // (cols * ntok)))
    wsub = synth.pq2_0_weights(rpc, cols, seed_index)
    t_q, n_q = _timed_loop(lambda: oracle.quantize_q8K(x), budget_s * 0.2)
    xq = oracle.quantize_q8K(x)
    t_m, n_m = _timed_loop(lambda: oracle.matmul(wsub, xq, rpc, cols), budget_s * 0.8)
    est = t_q + t_m * rows / rpc
    return est, (f"quantize {ntok}x{cols} timed whole ({n_q} calls); matmul timed on {rpc} of "
                 f"{rows} rows ({n_m} calls) and scaled by {rows / rpc:.1f}")


def oracle_rate(name: str, budget_s: float):
    """The C oracle (single-threaded) on a workload: units per second,
    estimated from a row sample (oracle_matrix_time). Returns (rate, unit,
    sample description, cores used, seconds per full step)."""
    cfg = synth.CONFIGS[name]
    rows, cols, ntok = cfg["rows"], cfg["cols"], cfg["ntok"]
    s = synth.seeds(cfg["index"])
    x = synth.activations(ntok, cols, s["acts"], s["outliers"] if cfg["outliers"] else None)
    est, how = oracle_matrix_time(rows, cols, ntok, x, cfg["index"], budget_s)
    unit = "Gweights/s" if ntok == 1 else "GMAC/s"
    return rows * cols * ntok / est / 1e9, unit, how, 1, est


def oracle_replay_rate(ntok: int, budget_s: float, blocks=None):
    """The oracle on one decode-step replay: per matrix of a block, quantize +
    matmul estimated from a row sample; times the blocks. Returns (rate, unit,
    sample description, cores used, seconds per step)."""
    blocks = blocks or synth.REPLAY_BLOCKS
    total, weights, parts = 0.0, 0, []
    for m in range(len(synth.REPLAY_BLOCK)):
        _, x, rows, cols = synth.replay_matrix(m, ntok, rows=1)
        est, how = oracle_matrix_time(rows, cols, ntok, x, 0x100 + m,
                                      budget_s / len(synth.REPLAY_BLOCK))
        total += est
        weights += rows * cols
        parts.append(f"{rows}x{cols}: {how}")
    total *= blocks
    weights *= blocks
    unit = "Gweights/s" if ntok == 1 else "GMAC/s"
    return (weights * ntok / total / 1e9, unit,
            f"{blocks} blocks x 5 matrices, each estimated as: " + "; ".join(parts), 1, total)


def cpu_baseline_entry(rate, unit, sample, cores, step_s):
    return {"value": rate, "unit": unit, "cores": cores, "kind": "oracle", "sample": sample,
            "s_per_step": step_s, "host": cpu_info()}


def metric_name(unit, name):
    """The metric string both arms print for a workload."""
    return f"ternary matvec {unit} & HBM GB/s ({WORKLOADS[name]})"


def run_reference(args, rank, world):
    """--impl reference: the oracle on the host cores, --steps/--warmup of row samples."""
    if rank != 0:
        return
    name = args.workload
    cfg = synth.CONFIGS[name]
    # calibrate a per-step row sample so that warm-up + steps take about a minute
    per_row = oracle_rate(name, 1.0)[4] / cfg["rows"]
    total = max(1, args.steps + args.warmup)
    rows_step = int(max(1, min(cfg["rows"], 60.0 / total / per_row)))
    import oracle
    s = synth.seeds(cfg["index"])
    x = synth.activations(cfg["ntok"], cfg["cols"], s["acts"],
                          s["outliers"] if cfg["outliers"] else None)
    wsub = synth.pq2_0_weights(rows_step, cfg["cols"], cfg["index"])
    for _ in range(max(args.warmup, 0)):
        oracle.matmul(wsub, oracle.quantize_q8K(x), rows_step, cfg["cols"])
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.matmul(wsub, oracle.quantize_q8K(x), rows_step, cfg["cols"])
    dt = time.perf_counter() - t0
    ntok = cfg["ntok"]
    per_step = rows_step * cfg["cols"] * ntok
    value = per_step * args.steps / dt / 1e9
    unit = "Gweights/s" if ntok == 1 else "GMAC/s"
    sample = (f"each step: quantize + matmul of {rows_step} of {cfg['rows']} rows x "
              f"{cfg['cols']} cols, ntok={ntok}")
    line = {
        "impl": "reference",
        "metric": metric_name(unit, name),
        "value": value, "unit": unit, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int32 sums, f64 accumulation", "data": "synthetic (seeded splitmix64)",
        "config": {"workload": WORKLOADS[name], "rows": cfg["rows"], "cols": cfg["cols"],
                   "ntok": ntok, "sample_rows": rows_step},
        "cpu_baseline": {"value": value, "unit": unit, "cores": 1, "kind": "oracle",
                         "sample": sample, "host": cpu_info()},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- profile evidence

def code_text(src: str) -> str:
    """C/CUDA source without its comments (no string literal in the kernel
    sources holds a comment marker) and without the lines left empty: what
    the compiler sees of it, unchanged by adding or removing comment lines."""
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    return "\n".join(ln.rstrip() for ln in src.splitlines() if ln.strip())


def kernel_source_sha(files):
    """Hash of the kernel sources' code (comments stripped), so a profile taken
    on a kernel stays valid across comment-only edits."""
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "bit_matvec_gb300", "csrc", f), encoding="utf-8") as fh:
            h.update(code_text(fh.read()).encode())
    return h.hexdigest()[:16]


def profile_traffic(summary_name, files, launch_bytes_key="dram_bytes_per_launch"):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel source (same source hash); else None."""
    path = os.path.join(ROOT, "profiles", summary_name)
    try:
        with open(path) as f:
            kv = dict(ln.split(":", 1) for ln in f if ":" in ln and not ln.startswith("#"))
    except OSError:
        return None
    kv = {k.strip(): v.strip() for k, v in kv.items()}
    if kv.get("source_sha") != kernel_source_sha(files):
        return None
    try:
        return float(kv[launch_bytes_key])
    except (KeyError, ValueError):
        return None


GEMV_FILES = ("tq_gemv.cu", "tq_tcgen05.cuh", "tq_internal.cuh")
TC_FILES = ("tq_gemm_tc_ws.cu", "tq_tcgen05.cuh", "tq_internal.cuh")


def measure(name, args, rank, world, device, peaks, peak_kind, steps):
    wl = Workload(name, device)
    step_ms, kern_ms, done, kern_how, serial_ms, dep_ms = time_graph(wl, steps, args.warmup,
                                                                      world)
    step_ms = max_over_ranks(step_ms, world, device)
    abytes = algorithmic_bytes(wl.rows, wl.cols, wl.ntok)
    res = {"workload": WORKLOADS[name], "rows": wl.rows, "cols": wl.cols, "ntok": wl.ntok,
           "ms_per_step": step_ms, "steps": done, "weight_copies": wl.copies,
           "repack_ms": wl.repack_s * 1e3}
    if wl.ntok == 1:
        res["gweights_per_s"] = world * wl.weights() / (step_ms * 1e-3) / 1e9
    res["gmac_per_s"] = world * wl.macs() / (step_ms * 1e-3) / 1e9
    res["hbm_gbs_step"] = (abytes + quantize_bytes(wl.ntok, wl.cols)) / (step_ms * 1e-3) / 1e9
    if wl.ntok <= GEMV_MAX_TOKENS:
        achieved = abytes / (kern_ms * 1e-3) / 1e9
        peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
        traffic = profile_traffic(f"gemv_{name}_ncu.txt", GEMV_FILES)

        def frac_at(ms):
            return None if ms is None else abytes / (ms * 1e-3) / 1e9 / peak

        res["roofline"] = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                           "frac": achieved / peak, "traffic": traffic,
                           "frac_of_nominal": achieved / HBM_NOMINAL_GBS,
                           "kernel": gemv_kernel_name(wl.rows, wl.cols, wl.ntok),
                           "kernel_ms": kern_ms,
                           "kernel_timing": kern_how,
                           "frac_meaning": "frac: independent launches back to back in a graph "
                                           "(each reads nothing the one before writes, so it "
                                           "streams its weights and activations before that one "
                                           "ends); frac_dependent: each launch quantizes the "
                                           "previous launch's output, so it waits for it before "
                                           "reading activations (weights are still requested "
                                           "first); frac_serialised: events between launches, "
                                           "no overlap at all",
                           "kernel_ms_dependent": dep_ms, "frac_dependent": frac_at(dep_ms),
                           "kernel_ms_serialised": serial_ms,
                           "frac_serialised": frac_at(serial_ms),
                           "algorithmic_bytes": abytes, "peak_source": peak_kind}
    else:
        flops = 2.0 * wl.macs()
        achieved = flops / (kern_ms * 1e-3) / 1e12
        peak = E4M3_PER_BF16 * float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
        traffic = profile_traffic(f"gemm_tc_ws_{name}_ncu.txt", TC_FILES)
        res["roofline"] = {"bound": "tensor", "achieved": achieved, "peak": peak,
                           "unit": "TFLOP/s", "frac": achieved / peak, "traffic": traffic,
                           "mma_busy_frac": achieved * mma_flops_per_flop(wl.ntok) / peak,
                           "kernel": "act_pack + gemm_tc_ws_kernel (tcgen05 kind::f8f6f4, exact)",
                           "kernel_ms": kern_ms, "kernel_timing": kern_how,
                           "kernel_ms_dependent": dep_ms,
                           "kernel_ms_serialised": serial_ms, "algorithmic_flops": flops,
                           "peak_source": f"{peak_kind} bf16 dense x {E4M3_PER_BF16:g} "
                                          f"(e4m3 : bf16 nominal)"}
    return wl, res


def tensor_rates():
    """Dense tensor-core rate by operand type through the vendor GEMMs (int8 via
    torch._int_mm, bf16 and f16 via matmul), square n x n x n, 3 warm-up and 20
    timed launches with CUDA events. Decides which MMA kind the tensor-core
    path uses; prints one JSON line per size."""
    import torch
    torch.backends.cuda.matmul.allow_tf32 = False
    dev = torch.device("cuda", 0)

    def rate(fn, flops, reps=20):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            fn()
        b.record()
        torch.cuda.synchronize()
        return flops / (a.elapsed_time(b) / reps / 1e3) / 1e12

    g = torch.Generator(device=dev).manual_seed(1)
    for n in (4096, 8192, 16384):
        a8 = torch.randint(-127, 127, (n, n), dtype=torch.int8, device=dev, generator=g)
        b8 = torch.randint(-127, 127, (n, n), dtype=torch.int8, device=dev,
                           generator=g).t().contiguous().t()
        ab = torch.randn(n, n, dtype=torch.bfloat16, device=dev, generator=g)
        bb = torch.randn(n, n, dtype=torch.bfloat16, device=dev, generator=g)
        ah, bh = ab.half(), bb.half()
        print(json.dumps({"n": n,
                          "int8_tops": round(rate(lambda: torch._int_mm(a8, b8), 2 * n ** 3), 1),
                          "bf16_tflops": round(rate(lambda: ab @ bb, 2 * n ** 3), 1),
                          "f16_tflops": round(rate(lambda: ah @ bh, 2 * n ** 3), 1)}), flush=True)


def main():
    args = parse_args()
    if args.tensor_rates:
        tensor_rates()
        return
    rank, world, local = dist_init(args.gpus)
    if args.impl == "reference":
        run_reference(args, rank, world)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    import torch
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    from bit_matvec_gb300 import build as tq_build
    tq_build.build()
    peaks, peak_kind = measured_peaks()

    clocks = ClockSampler(local)
    clocks.start()
    wl, main_res = measure(args.workload, args, rank, world, device, peaks, peak_kind, args.steps)
    clocks.stop()

    want_cpu = rank == 0 and world == 1 and not args.no_cpu
    extra = {}
    if not args.no_extra:
        for name in ("small_batch", "prefill"):
            if name != args.workload:
                _, r = measure(name, args, rank, world, device, peaks, peak_kind,
                               max(64, args.steps // 10))
                if want_cpu:
                    r["cpu_baseline"] = cpu_baseline_entry(*oracle_rate(name, 5.0))
                extra[name] = r
    if not args.no_replay:
        for ntok, rsteps in ((1, 30), (512, 3)):
            r = measure_replay(ntok, rsteps, args.warmup // 100 + 1, world, device, peaks,
                               peak_kind, read_ceiling=ntok == 1 and not args.no_read_ceiling)
            if want_cpu:
                r["cpu_baseline"] = cpu_baseline_entry(*oracle_replay_rate(ntok, 5.0))
            extra[f"replay_ntok{ntok}"] = r
    if args.workload == "decode" and not args.no_extra:
        extra["ptq1_stream"] = measure_ptq1_stream(max(40, args.steps // 10), args.warmup, world,
                                                   device, peaks, peak_kind,
                                                   main_res["roofline"]["kernel_ms"])
    if wl.ntok <= GEMV_MAX_TOKENS and not args.no_read_ceiling:
        main_res["roofline"]["read_ceiling"] = measure_read_ceiling(
            main_res["roofline"]["algorithmic_bytes"] // 16 * 16, device, args.warmup)

    e2e = None
    if not args.no_e2e:
        e2e_steps = max(100, min(args.steps, 5000))
        # The median of five runs, each with its own pinned buffers: the host
        # copies' speed varies from run to run (measured 11.8 to 14 us per
        # step on the decode workload with the same build).
        e2e_runs = [time_e2e(wl, e2e_steps, args.warmup, args.e2e_streams) for _ in range(5)]
        e2e_runs.sort(key=lambda r: r[0])
        s_per_step, h2d, d2h = e2e_runs[2]
        s_per_step = max_over_ranks(s_per_step, world, device)
        units = wl.weights() if wl.ntok == 1 else wl.macs()
        e2e = {"value": world * units / s_per_step / 1e9,
               "unit": "Gweights/s" if wl.ntok == 1 else "GMAC/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
               "ms_per_step": s_per_step * 1e3, "streams": args.e2e_streams,
               "runs_ms_per_step": [r[0] * 1e3 for r in e2e_runs],
               "how": "tq_matmul_host per step from pinned host X to pinned host Y; "
                      f"steps alternate over {args.e2e_streams} streams with their own buffers "
                      "(independent requests in flight); host wall clock around all steps; "
                      "median of 5 runs"}
        if args.e2e_streams != 1:
            # the median of five runs: on one stream the copies' latency varies
            # from run to run (measured 25 to 34 us per step on the decode
            # workload with the same build)
            runs = sorted(time_e2e(wl, e2e_steps, args.warmup, 1)[0] for _ in range(5))
            s1 = max_over_ranks(runs[2], world, device)
            e2e["one_stream"] = {"value": world * units / s1 / 1e9, "ms_per_step": s1 * 1e3,
                                 "runs_ms_per_step": [r * 1e3 for r in runs],
                                 "how": "the same calls on one stream: each step's copy in, "
                                        "kernel and copy out run one after another (the "
                                        "latency of a single request); median of 5 runs"}

    cpu = None
    if want_cpu:
        cpu = cpu_baseline_entry(*oracle_rate(args.workload, 10.0))

    if rank == 0:
        unit = "Gweights/s" if wl.ntok == 1 else "GMAC/s"
        value = main_res["gweights_per_s"] if wl.ntok == 1 else main_res["gmac_per_s"]
        line = {
            "metric": metric_name(unit, args.workload),
            "value": value, "unit": unit, "n_gpus": world, "steps": main_res["steps"],
            "warmup": args.warmup, "ms_per_step": main_res["ms_per_step"],
            "higher_is_better": True, "scaling": "weak",
            "vs_baseline": (value / PAGES_DECODE_GWEIGHTS
                            if args.workload == "decode" else None),
            "dtype": "int8" if wl.ntok <= GEMV_MAX_TOKENS else "e4m3 (exact integer sums)",
            "data": "synthetic (seeded splitmix64; no model weights)",
            "config": {"workload": WORKLOADS[args.workload], "rows": wl.rows, "cols": wl.cols,
                       "ntok": wl.ntok,
                       "l2": f"{wl.copies} rotating weight copies "
                             f"({wl.copies * wl.W[0].numel() / 1e6:.0f} MB > 2x 129 MB L2)",
                       "timing": f"CUDA graphs of {graph_plan(args.steps, wl.copies)[0]} "
                                 f"quantize+matmul steps each, CUDA events"},
            "hbm_gbs": main_res["hbm_gbs_step"],
            "roofline": main_res["roofline"],
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": wl.launches() * main_res["steps"],
            "clocks": clocks.summary(),
            "repack_ms": main_res["repack_ms"],
            "also": extra,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
