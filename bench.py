#!/usr/bin/env python3
"""Benchmark of the tile-centric overlap path on GB300.

One step = one pass of the whole hot path over one batch of synthetic inputs:
  * AllGather-GEMM, R=8 emulated ranks, A_r [1024, 4096] ~ N(0,1),
    B [4096, 1792] ~ N(0, 0.02) -> C [8192, 1792]     (tl_ag_gemm)
  * GEMM-ReduceScatter, R=8, A_r [8192, 1792], B_r [1792, 4096]
    -> 8 row shards [1024, 4096]                      (tl_gemm_rs)
  * AllGather + grouped MoE GEMM, R=8 x [1024, 4096] tokens, top-2 of 32
    experts (Zipf 1.2), W_e [4096, 1408]               (tl_moe_ag_gemm)
Metric: whole-job TFLOP/s = algorithmic FLOPs of the step / device time.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With N > 1 (launched by torchrun) every rank runs the same step on its own GPU
(independent replicas, weak scaling); rank 0 prints the JSON line with the
max-over-ranks time.  ``--impl reference`` times the CPU oracle on a bounded
sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

AG = dict(R=8, M_shard=1024, K=4096, N=1792)
RS = dict(R=8, M=8192, K_r=1792, N=4096)
MOE = dict(R=8, T_r=1024, H=4096, N=1408, E=32, topk=2, zipf_s=1.2)
AG_FLOPS = 2 * AG["R"] * AG["M_shard"] * AG["N"] * AG["K"]
RS_FLOPS = 2 * RS["R"] * RS["M"] * RS["N"] * RS["K_r"]
# operands read once and the bf16 output written once (the emulated fp32 partial push and read are extra)
RS_BYTES = RS["R"] * (RS["M"] * RS["K_r"] + RS["K_r"] * RS["N"]) * 2 + RS["M"] * RS["N"] * 2
# the reduce-scatter's own data movement on emulated ranks: every fp32 partial written once and read once
RS_PARTIAL_BYTES = 2 * RS["R"] * RS["M"] * RS["N"] * 4
MOE_FLOPS = 2 * MOE["R"] * MOE["T_r"] * MOE["topk"] * MOE["N"] * MOE["H"]
METRIC = "fused AG-GEMM / GEMM-RS TFLOP/s on 1 GB300"
WORKLOAD = ("AG-GEMM R=8 [8192x4096]x[4096x1792] + GEMM-RS R=8 8x[8192x1792]x[1792x4096] "
            "+ MoE AG+grouped GEMM R=8 8192 tokens top-2/32 experts [16384x4096]x[4096x1408] "
            "(TP MLP up/down projection and MoE expert up-projection, emulated ranks)")


# DRAM traffic of one gemm_rs_kernel launch on this workload, from one ncu capture
# (dram__bytes_read.sum + dram__bytes_write.sum), valid only while the kernel's
# sources hash to what was captured.
RS_TRAFFIC_BYTES = 910_647_808 + 422_917_376
RS_TRAFFIC_SOURCES = ("tl_gemm_rs.cu", "tl_pair.cuh", "tl_common.cuh", "tl_ptx.cuh")
RS_TRAFFIC_SHA256 = "cf9195c3f8068f36a58b0341495c7a399ff00e2bb07379de374daa46f6c2e67f"


def rs_traffic():
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tile_centric_gemm_gb300", "csrc")
    for f in RS_TRAFFIC_SOURCES:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return RS_TRAFFIC_BYTES if h.hexdigest() == RS_TRAFFIC_SHA256 else None


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-overlap", action="store_true", help="skip the fused-vs-halves measurements")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--sweep", action="store_true",
                    help="AG-GEMM sweep (R in {2,4,8}, M in {1024..16384}, K=8192, N=1024; shards in HBM and "
                         "peer shards in pinned host memory): copy, GEMM, sequential and fused times, one JSON line")
    ap.add_argument("--no-extras", action="store_true", help="skip the measurements outside the step")
    ap.add_argument("--only", choices=["ag", "rs", "moe", "moe_down", "ag_attn", "gemm_vs_library", "allgather_ll"],
                    help="run one fused call of the step (W untimed, then K timed back to back) and print its "
                         "device time; for profiling a single kernel on the bench's workload")
    return ap.parse_args()


def dist_env():
    return int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")), \
        int(os.environ.get("LOCAL_RANK", "0"))


def max_over_ranks(pg, x):
    """The slowest rank's time: all-reduce MAX over the process group (None = one rank)."""
    if pg is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t[0])


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every 100 ms, timestamped."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                self.samples.append((time.time(), float(parts[0]), float(parts[1]), parts[3:7]))
            except ValueError:
                pass

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        window = "timed"
        if len(inside) < 3:
            inside = [s for s in self.samples if t0 - 1.0 <= s[0] <= t1 + 0.2]
            window = "timed+1s before"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in inside for i, v in enumerate(s[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(s[1] for s in inside), "sm_max_mhz": max(s[2] for s in inside),
                "reasons": reasons, "samples": len(inside), "window": window}


# ------------------------------------------------------------------ CPU oracle timing
class OracleSample:
    """The oracle, as it stands, on a row sample of the same workload: the AG-GEMM
    shards cut to `rows` rows each and the GEMM-RS operands cut to R*rows rows."""

    def __init__(self):
        from tile_centric_gemm_gb300 import inputs
        self.A, self.B = inputs.ag_gemm_inputs(AG["R"], AG["M_shard"], AG["K"], AG["N"], "normal", seed=0)
        self.Ar, self.Br = inputs.gemm_rs_inputs(RS["R"], RS["M"], RS["K_r"], RS["N"], seed=0)
        self.X, self.ids, self.W = inputs.moe_inputs(MOE["R"], MOE["T_r"], MOE["H"], MOE["N"], MOE["E"],
                                                     MOE["topk"], MOE["zipf_s"], seed=0)
        self.rows = 16

    def flops(self):
        return (2 * AG["R"] * self.rows * AG["N"] * AG["K"] + 2 * RS["R"] * (RS["R"] * self.rows) * RS["N"] * RS["K_r"]
                + 2 * MOE["R"] * self.rows * MOE["topk"] * MOE["N"] * MOE["H"])

    def describe(self):
        return (f"AG-GEMM with {self.rows} of {AG['M_shard']} rows per shard + GEMM-RS with "
                f"{RS['R'] * self.rows} of {RS['M']} rows + MoE with {self.rows} of {MOE['T_r']} tokens per shard "
                f"({self.flops() / 1e9:.1f} GFLOP; float64 numpy oracle)")

    def step(self):
        import oracle
        t0 = time.perf_counter()
        oracle.ag_gemm.ag_gemm([a[:self.rows] for a in self.A], self.B)
        oracle.gemm_rs.gemm_rs([a[:RS["R"] * self.rows] for a in self.Ar], self.Br)
        T_r = MOE["T_r"]
        keep = np.concatenate([np.arange(r * T_r, r * T_r + self.rows) for r in range(MOE["R"])])
        oracle.moe.moe_ag_gemm([x[:self.rows] for x in self.X], self.ids[keep], self.W)
        return time.perf_counter() - t0

    def size_to(self, seconds):
        """Grow the sample until one step takes about `seconds` (at most the full shard)."""
        while True:
            dt = self.step()
            if dt >= 0.5 * seconds or self.rows >= AG["M_shard"]:
                return dt
            self.rows = min(AG["M_shard"], self.rows * max(2, int(seconds / max(dt, 1e-3))))


def cpu_threads():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def time_oracle(budget_s=12.0):
    """(TFLOP/s, seconds, sample description) of the oracle on a ~budget_s sample."""
    o = OracleSample()
    o.size_to(budget_s)
    dt = o.step()
    return o.flops() / dt / 1e12, dt, o.describe()


def run_reference(args, world, rank):
    """The reference arm: the CPU oracle timed step by step on a bounded sample."""
    if rank != 0:
        return
    o = OracleSample()
    o.size_to(1.0)
    times = []
    for i in range(args.warmup + args.steps):
        dt = o.step()
        if i >= args.warmup:
            times.append(dt)
    t = statistics.mean(times)
    value = o.flops() / t / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "sample": o.describe()},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cpu_threads(), "kind": "oracle",
                             "sample": o.describe()},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU arm
class Workload:
    def __init__(self, B, torch):
        from tile_centric_gemm_gb300 import inputs
        self.B, self.torch = B, torch
        dev = "cuda"
        A, Bm = inputs.ag_gemm_inputs(AG["R"], AG["M_shard"], AG["K"], AG["N"], "normal", seed=0)
        Ar, Br = inputs.gemm_rs_inputs(RS["R"], RS["M"], RS["K_r"], RS["N"], seed=0)
        tb = inputs.to_torch_bf16
        # host (pinned) copies for the end-to-end measurement
        self.h_ag = [tb(a).pin_memory() for a in A] + [tb(Bm).pin_memory()]
        self.h_rs = [tb(a).pin_memory() for a in Ar] + [tb(b).pin_memory() for b in Br]
        self.d_ag = [t.to(dev) for t in self.h_ag]
        self.d_rs = [t.to(dev) for t in self.h_rs]
        R = AG["R"]
        M = R * AG["M_shard"]
        self.G = torch.empty(M, AG["K"], dtype=torch.bfloat16, device=dev)
        self.C = torch.empty(M, AG["N"], dtype=torch.bfloat16, device=dev)
        nf, _ = B.tl_ag_gemm_num_flags(R, AG["M_shard"], AG["K"])
        self.sig_ag = B.Signals(nf)
        Rr = RS["R"]
        self.out = [torch.empty(RS["M"] // Rr, RS["N"], dtype=torch.bfloat16, device=dev) for _ in range(Rr)]
        self.ws = torch.empty(B.tl_gemm_rs_workspace_size(Rr, RS["M"], RS["N"]) // 4, dtype=torch.float32,
                              device=dev)
        self.sig_rs = B.Signals(B.tl_gemm_rs_num_flags(Rr, RS["M"], RS["N"]))
        X, ids, W = inputs.moe_inputs(MOE["R"], MOE["T_r"], MOE["H"], MOE["N"], MOE["E"], MOE["topk"],
                                      MOE["zipf_s"], seed=0)
        self.h_moe = [tb(x).pin_memory() for x in X] + [tb(w).pin_memory() for w in W] + \
            [torch.from_numpy(ids).pin_memory()]
        self.d_moe = [t.to(dev) for t in self.h_moe]
        P = MOE["R"] * MOE["T_r"] * MOE["topk"]
        self.S = torch.empty(P, MOE["H"], dtype=torch.bfloat16, device=dev)
        self.Y = torch.empty(P, MOE["N"], dtype=torch.bfloat16, device=dev)
        self.perm = torch.empty(P, dtype=torch.int32, device=dev)
        self.offs = torch.empty(MOE["E"] + 1, dtype=torch.int32, device=dev)
        self.ws_moe = torch.empty(B.tl_moe_workspace_size(MOE["R"], MOE["T_r"], MOE["E"], MOE["topk"]) // 4,
                                  dtype=torch.int32, device=dev)
        self.sig_moe = B.Signals(B.tl_moe_num_flags(MOE["R"], MOE["T_r"], MOE["H"], MOE["topk"])[0])
        self.h_C = torch.empty_like(self.C, device="cpu").pin_memory()
        self.h_out = [torch.empty_like(o, device="cpu").pin_memory() for o in self.out]
        self.h_Y = torch.empty_like(self.Y, device="cpu").pin_memory()
        # set 0 = the tensors above; set 1 = a second copy of every input and of every
        # output read back, so that the end-to-end loop can copy one step's inputs in
        # while the previous step computes and its outputs go out
        self.sets = [dict(ag=self.d_ag, rs=self.d_rs, moe=self.d_moe, C=self.C, out=self.out, Y=self.Y),
                     dict(ag=[torch.empty_like(t) for t in self.d_ag], rs=[torch.empty_like(t) for t in self.d_rs],
                          moe=[torch.empty_like(t) for t in self.d_moe], C=torch.empty_like(self.C),
                          out=[torch.empty_like(o) for o in self.out], Y=torch.empty_like(self.Y))]
        self.epoch = 0
        self.launches_per_step = 4  # ag_gemm, gemm_rs, moe route, moe gemm

    def ag(self, b=0):
        self.epoch += 1
        R = AG["R"]
        d = self.sets[b]
        self.B.tl_ag_gemm(d["ag"][:R], d["ag"][R], self.G, d["C"], self.sig_ag, self.epoch)

    def rs(self, b=0):
        self.epoch += 1
        R = RS["R"]
        d = self.sets[b]
        self.B.tl_gemm_rs(d["rs"][:R], d["rs"][R:], d["out"], self.ws, self.sig_rs, self.epoch)

    def moe(self, b=0):
        self.epoch += 1
        R, E = MOE["R"], MOE["E"]
        d = self.sets[b]
        m = d["moe"]
        self.B.tl_moe_ag_gemm(m[:R], m[R + E], m[R:R + E], self.S, d["Y"], self.perm, self.offs, self.ws_moe,
                              self.sig_moe, self.epoch)

    def _weight(self, i):
        """Whether input i (in h_ag + h_rs + h_moe order) is a weight: B, the B_r, the W_e."""
        R, Rr, E = AG["R"], RS["R"], MOE["E"]
        n_ag, n_rs = len(self.h_ag), len(self.h_rs)
        if i < n_ag:
            return i == R
        if i < n_ag + n_rs:
            return i - n_ag >= Rr
        return MOE["R"] <= i - n_ag - n_rs < MOE["R"] + E

    def h2d(self, b=0, weights=True):
        """Copy set b's inputs in from pinned host memory: every operand, or (weights=False)
        the activations and the routing only, the weights staying resident."""
        d = self.sets[b]
        for i, (h, t) in enumerate(zip(self.h_ag + self.h_rs + self.h_moe, d["ag"] + d["rs"] + d["moe"])):
            if weights or not self._weight(i):
                t.copy_(h, non_blocking=True)

    def d2h(self, b=0):
        d = self.sets[b]
        self.h_C.copy_(d["C"], non_blocking=True)
        for h, t in zip(self.h_out, d["out"]):
            h.copy_(t, non_blocking=True)
        self.h_Y.copy_(d["Y"], non_blocking=True)

    def h2d_bytes(self, weights=True):
        return sum(t.numel() * t.element_size() for i, t in enumerate(self.h_ag + self.h_rs + self.h_moe)
                   if weights or not self._weight(i))

    def d2h_bytes(self):
        return self.h_C.numel() * 2 + sum(t.numel() * 2 for t in self.h_out) + self.h_Y.numel() * 2

    def check_status(self):
        for s in (self.sig_ag, self.sig_rs, self.sig_moe):
            code, where = self.B.tl_query_status(s)
            if code:
                raise RuntimeError(f"device error {code} at {where}")


def e2e_serial(torch, wl, E, stream, barrier, weights=True):
    """ms per step with the copies and the calls in one stream: H2D inputs (every
    operand, or the activations and routing with the weights resident), the three
    calls, D2H outputs, one step after the other."""
    wl.h2d()
    for _ in range(2):
        wl.h2d(weights=weights); wl.ag(); wl.rs(); wl.moe(); wl.d2h()
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(E):
        wl.h2d(weights=weights); wl.ag(); wl.rs(); wl.moe(); wl.d2h()
    e1.record(stream)
    barrier()
    return e0.elapsed_time(e1) / E


def e2e_pipelined(torch, wl, E, stream, barrier, weights=True):
    """ms per step over E steps, each copying its inputs in (every operand, or with
    weights=False the activations and routing, the weights loaded into both sets
    once before timing) and all of its outputs back, with two device sets: step i
    computes on set i % 2 while step i+1's inputs copy into the other set (copy-in
    stream) and step i-1's outputs copy out (copy-out stream).  The timed region
    runs from before the first copy-in to after the last copy-out."""
    wl.h2d(0)
    wl.h2d(1)
    cin, cout = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: [torch.cuda.Event(), torch.cuda.Event()]

    def run(n, e0=None):
        inputs_free, inputs_ready, outputs_ready, outputs_read = ev(), ev(), ev(), ev()
        if e0 is not None:
            e0.record(stream)
        cin.wait_stream(stream)
        cout.wait_stream(stream)
        for i in range(n):
            b = i & 1
            with torch.cuda.stream(cin):
                if i >= 2:
                    cin.wait_event(inputs_free[b])
                wl.h2d(b, weights=weights)
                inputs_ready[b].record(cin)
            stream.wait_event(inputs_ready[b])
            if i >= 2:
                stream.wait_event(outputs_read[b])
            wl.ag(b)
            wl.rs(b)
            wl.moe(b)
            inputs_free[b].record(stream)
            outputs_ready[b].record(stream)
            with torch.cuda.stream(cout):
                cout.wait_event(outputs_ready[b])
                wl.d2h(b)
                outputs_read[b].record(cout)
        stream.wait_stream(cin)
        stream.wait_stream(cout)

    run(2)
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    run(E, e0)
    e1.record(stream)
    barrier()
    return e0.elapsed_time(e1) / E


def flushed_time_us(torch, fn, flush, reps=7):
    """Median device time (CUDA events on the current stream) of fn() over reps
    runs, each after a write of a buffer larger than L2 (not timed; it also
    hides the host's launch latency), after one warm-up run."""
    return time_variants(torch, fn, flush, reps)["cold"]


def time_variants(torch, fn, flush, reps=7):
    """Device times of fn() in microseconds: 'cold' (median) and 'cold_min' with
    L2 flushed before every run by a write larger than L2, and 'warm' (median)
    with runs back to back, each bracketed by its own events."""
    fn()
    cold, warm = [], []
    for flushed in (True, False):
        for _ in range(reps):
            if flushed:
                flush.zero_()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            b.synchronize()
            (cold if flushed else warm).append(a.elapsed_time(b) * 1e3)
    return {"cold": statistics.median(cold), "cold_min": min(cold), "warm": statistics.median(warm)}


def decomposed_graph(torch, B, shards, Bm, G, C, sig, ws=None, library=False):
    """The prior-art decomposed schedule as a CUDA graph: the copy engine gathers
    shard after shard (rank 0 last) on a side stream while the main stream runs
    one GEMM per shard, the local shard 0 first, each after its copy's event.
    The per-shard GEMM is tl_gemm (split-K with a workspace), or torch.matmul
    with library=True."""
    R, Ms = len(shards), shards[0].shape[0]
    s1 = torch.cuda.Stream()

    def gemm(a, c):
        if library:
            torch.matmul(a, Bm, out=c)
        else:
            B.tl_gemm(a, Bm, c, sig, workspace=ws)

    def launches():
        main = torch.cuda.current_stream()
        start = torch.cuda.Event()
        start.record(main)
        s1.wait_event(start)
        evs = []
        with torch.cuda.stream(s1):
            for j in range(1, R):
                G[j * Ms:(j + 1) * Ms].copy_(shards[j], non_blocking=True)
                e = torch.cuda.Event()
                e.record(s1)
                evs.append(e)
            G[0:Ms].copy_(shards[0], non_blocking=True)
        gemm(shards[0], C[0:Ms])
        for j, e in zip(range(1, R), evs):
            main.wait_event(e)
            gemm(G[j * Ms:(j + 1) * Ms], C[j * Ms:(j + 1) * Ms])
        main.wait_stream(s1)

    launches()  # sets every kernel's launch attributes before the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        launches()
    return graph


def overlap_metrics(torch, B, wl):
    """The fused kernels against their halves run alone, one after the other, and
    (AG-GEMM) decomposed onto two streams (the copy engine and per-shard GEMMs,
    replayed from a CUDA graph so the host's launch rate does not bound it), plus
    torch.matmul on the same operands as a library reference.  The metrics use
    the cold-L2 medians; warm medians and cold minima are reported beside them."""
    R, Ms, K = AG["R"], AG["M_shard"], AG["K"]
    A, Bm = wl.d_ag[:R], wl.d_ag[R]
    sig1 = B.Signals(max(1, wl.sig_ag.num_flags))
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    ep = [10_000_000]
    C_lib = torch.empty_like(wl.C)

    def copy_only():
        ep[0] += 1
        B.tl_allgather(A, wl.G, sig1, ep[0])

    def gemm_only():
        B.tl_gemm(wl.G, Bm, wl.C, sig1)

    def seq():
        copy_only()
        gemm_only()

    # the decomposed schedule with each per-shard GEMM as fast as this library or the
    # library GEMM makes it: tl_gemm with split-K (a shard's 28 tiles fill 28 of 76 pairs
    # unsplit), and torch.matmul; t_decomposed is the faster of the two
    ws_shard = torch.zeros(max(16, B.tl_gemm_workspace_size(Ms, AG["N"], K) // 4), dtype=torch.float32,
                           device="cuda")
    graph = decomposed_graph(torch, B, A, Bm, wl.G, wl.C, sig1, ws_shard)
    graph_lib = decomposed_graph(torch, B, A, Bm, wl.G, wl.C, sig1, library=True)
    ag_t = {"copy": time_variants(torch, copy_only, flush), "gemm": time_variants(torch, gemm_only, flush),
            "seq": time_variants(torch, seq, flush), "decomposed": time_variants(torch, graph.replay, flush),
            "decomposed_torch_matmul": time_variants(torch, graph_lib.replay, flush),
            "fused": time_variants(torch, wl.ag, flush),
            "torch_matmul": time_variants(torch, lambda: torch.matmul(wl.G, Bm, out=C_lib), flush)}
    t_copy, t_gemm, t_seq = ag_t["copy"]["cold"], ag_t["gemm"]["cold"], ag_t["seq"]["cold"]
    t_dec = min(ag_t["decomposed"]["cold"], ag_t["decomposed_torch_matmul"]["cold"])
    t_fused = ag_t["fused"]["cold"]
    ag = {"t_copy_us": t_copy, "t_gemm_us": t_gemm, "t_seq_us": t_seq, "t_decomposed_us": t_dec,
          "t_decomposed_tl_gemm_splitk_us": ag_t["decomposed"]["cold"],
          "t_decomposed_torch_matmul_us": ag_t["decomposed_torch_matmul"]["cold"],
          "t_fused_us": t_fused, "t_torch_matmul_us": ag_t["torch_matmul"]["cold"],
          "speedup_vs_seq": t_seq / t_fused,
          "speedup_vs_decomposed": t_dec / t_fused,
          "fused_over_max_copy_gemm": t_fused / max(t_copy, t_gemm),
          "overlap_efficiency": (t_seq - t_fused) / min(t_copy, t_gemm),
          "copy_gbs": 2 * R * Ms * K * 2 / (t_copy * 1e-6) / 1e9,
          "warm_us": {k: v["warm"] for k, v in ag_t.items()},
          "cold_min_us": {k: v["cold_min"] for k, v in ag_t.items()}}
    # swizzle ablation: the fused kernel with its consumer in arrival order and in plain row
    # order, for the calling rank 0 (the two orders coincide) and a rank in the middle
    abl = {}
    for self_rank in (0, R // 2):
        for name, sw in (("arrival", B.TL_SWIZZLE_ARRIVAL), ("rows", B.TL_SWIZZLE_ROWS)):
            def fused_sw(self_rank=self_rank, sw=sw):
                ep[0] += 1
                B.tl_ag_gemm(A, Bm, wl.G, wl.C, sig1, ep[0], self_rank=self_rank, swizzle=sw)
            abl[f"self{self_rank}_{name}_us"] = flushed_time_us(torch, fused_sw, flush)
    ag["swizzle_ablation"] = abl
    # push against pull (talk summary, Technical Deep Dive: push needs one barrier, pull a
    # readiness barrier before the copy and a completion barrier after it), each with both
    # consumer orders, for a middle calling rank; the readiness flags are set before the
    # call, as a resident peer's would be
    ready = B.Signals(max(1, wl.sig_ag.num_flags))
    B.tl_tile_notify(ready, 0, wl.sig_ag.num_flags, 0x7FFF0000)
    pp = {}
    for mname, mode in (("push", B.TL_MODE_PUSH), ("pull", B.TL_MODE_PULL)):
        for name, sw in (("arrival", B.TL_SWIZZLE_ARRIVAL), ("rows", B.TL_SWIZZLE_ROWS)):
            def fused_mode(mode=mode, sw=sw):
                ep[0] += 1
                B.tl_ag_gemm(A, Bm, wl.G, wl.C, sig1, ep[0], self_rank=R // 2, swizzle=sw, mode=mode,
                             src_ready=ready if mode == B.TL_MODE_PULL else None)
            pp[f"{mname}_{name}_us"] = flushed_time_us(torch, fused_mode, flush)
    ag["push_pull_ablation"] = pp
    code, where = B.tl_query_status(ready)
    if code:
        raise RuntimeError(f"device error {code} at {where} on the readiness flags")
    # GEMM-RS: per-rank GEMMs with fp32 partials, then the rank-ordered ReduceScatter
    Rr, M, N = RS["R"], RS["M"], RS["N"]
    parts = [torch.empty(M, N, dtype=torch.float32, device="cuda") for _ in range(Rr)]

    def rs_gemm():
        for r in range(Rr):
            B.tl_gemm(wl.d_rs[r], wl.d_rs[Rr + r], None, sig1, C_f32=parts[r])

    def rs_reduce():
        B.tl_reduce_scatter(parts, wl.out)

    def rs_seq():
        rs_gemm()
        rs_reduce()

    lib_out = [torch.empty(M, N, dtype=torch.bfloat16, device="cuda") for _ in range(Rr)]

    def rs_torch_matmul():
        for r in range(Rr):
            torch.matmul(wl.d_rs[r], wl.d_rs[Rr + r], out=lib_out[r])

    rs_t = {"gemm": time_variants(torch, rs_gemm, flush, reps=5),
            "reduce": time_variants(torch, rs_reduce, flush, reps=5),
            "seq": time_variants(torch, rs_seq, flush, reps=5), "fused": time_variants(torch, wl.rs, flush, reps=5),
            "torch_matmul": time_variants(torch, rs_torch_matmul, flush, reps=5)}
    t_g, t_r, t_s, t_f = (rs_t[k]["cold"] for k in ("gemm", "reduce", "seq", "fused"))
    rs = {"t_gemm_us": t_g, "t_reduce_us": t_r, "t_seq_us": t_s, "t_fused_us": t_f,
          "t_torch_matmul_us": rs_t["torch_matmul"]["cold"],
          "speedup_vs_seq": t_s / t_f, "fused_over_max_gemm_reduce": t_f / max(t_g, t_r),
          "overlap_efficiency": (t_s - t_f) / min(t_g, t_r),
          "reduce_gbs": (Rr * M * N * 4 + M * N * 2) / (t_r * 1e-6) / 1e9,
          "warm_us": {k: v["warm"] for k, v in rs_t.items()},
          "cold_min_us": {k: v["cold_min"] for k, v in rs_t.items()}}
    del lib_out
    # the fused kernel with bf16 partials (half the emulated partial traffic) and with
    # the ring summation order, beside the default fp32 partials in rank order
    abl = {}
    sig_rs2 = B.Signals(wl.sig_rs.num_flags)
    for name, opt in (("bf16_partials", B.TL_RS_BF16_PARTIALS), ("ring_order", B.TL_RS_RING_ORDER),
                      ("bf16_partials_ring_order", B.TL_RS_BF16_PARTIALS | B.TL_RS_RING_ORDER)):
        def rs_opt(opt=opt):
            ep[0] += 1
            B.tl_gemm_rs(wl.d_rs[:Rr], wl.d_rs[Rr:], wl.out, wl.ws, sig_rs2, ep[0], options=opt)
        abl[f"{name}_us"] = flushed_time_us(torch, rs_opt, flush, reps=5)
    rs["options_ablation"] = abl
    # MoE AllGather + grouped GEMM (routing included) in its two data modes: pull (the
    # consumer side gathers sorted rows in the order the tiles run) and push (source
    # shards scatter their tokens, tiles run by the latest arrival among their barriers)
    R_m, E_m = MOE["R"], MOE["E"]
    m = wl.d_moe
    moe_pp = {}
    for mname, mode in (("pull", B.TL_MODE_PULL), ("push", B.TL_MODE_PUSH)):
        sig_m = B.Signals(B.tl_moe_num_flags(R_m, MOE["T_r"], MOE["H"], MOE["topk"], mode=mode)[0])

        def moe_mode(mode=mode, sig_m=sig_m):
            ep[0] += 1
            B.tl_moe_ag_gemm(m[:R_m], m[R_m + E_m], m[R_m:R_m + E_m], wl.S, wl.Y, wl.perm, wl.offs, wl.ws_moe,
                             sig_m, ep[0], mode=mode, self_rank=R_m // 2)
        moe_pp[f"{mname}_us"] = flushed_time_us(torch, moe_mode, flush)
        code, where = B.tl_query_status(sig_m)
        if code:
            raise RuntimeError(f"device error {code} at {where} in the MoE {mname} measurement")
    moe_pp["note"] = "cold L2, median of 7, caller rank 4, routing kernel included"
    for s in (sig1, sig_rs2, wl.sig_ag, wl.sig_rs):
        code, where = B.tl_query_status(s)
        if code:
            raise RuntimeError(f"device error {code} at {where} in the overlap measurements")
    del parts, flush
    return {"ag_gemm": ag, "gemm_rs": rs, "moe_push_pull": moe_pp}


SWEEP = dict(R=(2, 4, 8), M=(1024, 2048, 4096, 8192, 16384), K=8192, N=1024)


def run_sweep(torch, B, peaks):
    """The AG-GEMM sweep: fused time against the copy and the GEMM alone, from a cold L2."""
    K, N = SWEEP["K"], SWEEP["N"]
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    rows = []
    for placement in ("hbm", "pinned_host"):
        for R in SWEEP["R"]:
            for M in SWEEP["M"]:
                Ms = M // R
                gen = torch.Generator(device="cuda")
                shards = []
                for r in range(R):
                    gen.manual_seed(r)
                    a = torch.randn(Ms, K, generator=gen, device="cuda").to(torch.bfloat16)
                    # rank 0 is the caller; the others sit behind the slower link in the pinned-host case
                    shards.append(a.cpu().pin_memory() if placement == "pinned_host" and r != 0 else a)
                gen.manual_seed(1000)
                Bm = (torch.randn(K, N, generator=gen, device="cuda") * 0.02).to(torch.bfloat16)
                G = torch.empty(M, K, dtype=torch.bfloat16, device="cuda")
                C = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
                sig = B.Signals(B.tl_ag_gemm_num_flags(R, Ms, K)[0])
                ep = [0]
                # split-K workspaces (zeroed; None where the tiles already fill the SMs); the
                # per-shard GEMMs of the decomposed schedule run one after another on one stream
                ws_ag, ws_gemm, ws_shard = (torch.zeros(n, dtype=torch.uint8, device="cuda") if n else None for n in (
                    B.tl_ag_gemm_workspace_size(R, Ms, K, N), B.tl_gemm_workspace_size(M, N, K),
                    B.tl_gemm_workspace_size(Ms, N, K)))

                def copy_only():
                    ep[0] += 1
                    B.tl_allgather(shards, G, sig, ep[0])

                def gemm_only():
                    B.tl_gemm(G, Bm, C, sig, workspace=ws_gemm)

                def seq():
                    copy_only()
                    gemm_only()

                def fused():
                    ep[0] += 1
                    B.tl_ag_gemm(shards, Bm, G, C, sig, ep[0], workspace=ws_ag)

                C_lib = torch.empty_like(C)
                graph = decomposed_graph(torch, B, shards, Bm, G, C, sig, ws_shard)
                graph_lib = decomposed_graph(torch, B, shards, Bm, G, C_lib, sig, library=True)
                t_copy = flushed_time_us(torch, copy_only, flush, reps=5)
                t_gemm = flushed_time_us(torch, gemm_only, flush, reps=5)
                t_seq = flushed_time_us(torch, seq, flush, reps=5)
                # the decomposed schedule with either per-shard GEMM; the faster one is reported
                t_dec_tl = flushed_time_us(torch, graph.replay, flush, reps=5)
                t_dec_lib = flushed_time_us(torch, graph_lib.replay, flush, reps=5)
                t_dec = min(t_dec_tl, t_dec_lib)
                t_fused = flushed_time_us(torch, fused, flush, reps=5)
                t_lib = flushed_time_us(torch, lambda: torch.matmul(G, Bm, out=C_lib), flush, reps=5)
                del graph, graph_lib
                code, where = B.tl_query_status(sig)
                if code:
                    raise RuntimeError(f"device error {code} at {where} in the sweep (R={R}, M={M}, {placement})")
                flops = 2 * M * N * K
                host_bytes = (R - 1) * Ms * K * 2 if placement == "pinned_host" else 0
                splits = (B.tl_ag_gemm_workspace_size(R, Ms, K, N) - 1024) // (-(-M // 256) * -(-N // 256) * 262144) \
                    if ws_ag is not None else 1
                rows.append({"placement": placement, "R": R, "M": M, "splits": int(splits),
                             "t_copy_us": t_copy, "t_gemm_us": t_gemm,
                             "t_seq_us": t_seq, "t_decomposed_us": t_dec,
                             "t_decomposed_tl_gemm_splitk_us": t_dec_tl, "t_decomposed_torch_matmul_us": t_dec_lib,
                             "t_fused_us": t_fused,
                             "t_torch_matmul_us": t_lib, "speedup_vs_decomposed": t_dec / t_fused,
                             "tflops": flops / (t_fused * 1e-6) / 1e12,
                             "frac_of_peak": flops / (t_fused * 1e-6) / 1e12 / peaks["bf16_tflops"],
                             "fused_over_max": t_fused / max(t_copy, t_gemm),
                             "speedup_vs_seq": t_seq / t_fused,
                             "overlap_efficiency": (t_seq - t_fused) / min(t_copy, t_gemm),
                             "copy_gbs": 2 * M * K * 2 / (t_copy * 1e-6) / 1e9,
                             "host_read_gbs": host_bytes / (t_copy * 1e-6) / 1e9 if host_bytes else None})
                del shards, G, C, C_lib, Bm, sig, ws_ag, ws_gemm, ws_shard
    del flush
    return rows


# the down side of the step's MoE layer: same routing; I_r = the up side's per-rank columns, Hd = its hidden size
MOE_DOWN = dict(R=MOE["R"], T_r=MOE["T_r"], topk=MOE["topk"], E=MOE["E"], I_r=MOE["N"], Hd=MOE["H"])
MOE_DOWN_FLOPS = 2 * MOE_DOWN["R"] * (MOE_DOWN["R"] * MOE_DOWN["T_r"] * MOE_DOWN["topk"]) * MOE_DOWN["Hd"] * \
    MOE_DOWN["I_r"]


class MoeDown:
    """The MoE layer's down-projection side on the bench's routing (the step's MoE
    call leaves it in its workspace): per-rank H_r [P, I_r] ~ N(0,1), W2_r
    [E*I_r, Hd] ~ N(0,0.02), gates uniform and normalised per token, drawn on the
    device from seeded generators (the weights alone are 3 GB)."""

    def __init__(self, B, torch, wl):
        c = MOE_DOWN
        self.B, self.torch, self.wl = B, torch, wl
        P = c["R"] * c["T_r"] * c["topk"]
        g = torch.Generator(device="cuda")
        self.H, self.W2 = [], []
        for r in range(c["R"]):
            g.manual_seed(4000 + r)
            self.H.append(torch.randn(P, c["I_r"], generator=g, device="cuda").to(torch.bfloat16))
            g.manual_seed(5000 + r)
            self.W2.append((torch.randn(c["E"] * c["I_r"], c["Hd"], generator=g, device="cuda") * 0.02)
                           .to(torch.bfloat16))
        g.manual_seed(6000)
        gates = torch.rand(c["R"] * c["T_r"], c["topk"], generator=g, device="cuda")
        self.gates = (gates / gates.sum(dim=1, keepdim=True)).contiguous()
        self.out = [torch.empty(c["T_r"], c["Hd"], dtype=torch.bfloat16, device="cuda") for _ in range(c["R"])]
        nbytes = B.tl_moe_down_workspace_size(c["R"], c["T_r"], c["topk"], c["E"], c["Hd"])
        self.work = torch.empty(nbytes // 4, dtype=torch.float32, device="cuda")
        self.sig = B.Signals(B.tl_moe_down_num_flags(c["R"], c["T_r"], c["topk"], c["E"], c["Hd"]))
        self.epoch = 0

    def run(self, options=0):
        self.epoch += 1
        self.B.tl_moe_down(self.H, self.W2, self.gates, self.wl.ws_moe, self.out, self.work, self.sig, self.epoch,
                           topk=MOE_DOWN["topk"], E=MOE_DOWN["E"], options=options)

    def check_status(self):
        code, where = self.B.tl_query_status(self.sig)
        if code:
            raise RuntimeError(f"device error {code} at {where} in the MoE down projection")


# AllGather-KV attention (sequence parallel): 8 ranks x 8192 tokens (a 64K context), 32 query heads
# over 8 key/value heads, head dim 128; rank 0's view (every rank does the same work when not causal)
AG_ATTN = dict(R=8, S_shard=8192, H=32, H_kv=8, D=128)


def attn_flops(c, causal, self_rank):
    """4 * D flops per visible (query, key) pair and head (S = Q K^T and O = P V)."""
    S = c["S_shard"]
    pairs = S * (self_rank * S) + S * (S + 1) // 2 if causal else S * c["R"] * S
    return 4 * c["D"] * c["H"] * pairs


class AgAttn:
    """AllGather-KV attention on the device: Q [S, H, D], K_r / V_r [S, H_kv, D]
    ~ N(0,1), drawn on the device from seeded generators."""

    def __init__(self, B, torch):
        c = AG_ATTN
        self.B, self.torch = B, torch
        g = torch.Generator(device="cuda")
        g.manual_seed(7000)
        self.Q = torch.randn(c["S_shard"], c["H"], c["D"], generator=g, device="cuda").to(torch.bfloat16)
        self.K, self.V = [], []
        for r in range(c["R"]):
            g.manual_seed(8000 + r)
            self.K.append(torch.randn(c["S_shard"], c["H_kv"], c["D"], generator=g, device="cuda").to(torch.bfloat16))
            g.manual_seed(9000 + r)
            self.V.append(torch.randn(c["S_shard"], c["H_kv"], c["D"], generator=g, device="cuda").to(torch.bfloat16))
        self.Kg = torch.empty(c["R"] * c["S_shard"], c["H_kv"], c["D"], dtype=torch.bfloat16, device="cuda")
        self.Vg = torch.empty_like(self.Kg)
        self.O = torch.empty(c["S_shard"], c["H"], c["D"], dtype=torch.bfloat16, device="cuda")
        self.L = torch.empty(c["H"], c["S_shard"], dtype=torch.float32, device="cuda")
        self.sig = B.Signals(B.tl_ag_attn_num_flags(c["R"], c["S_shard"]))
        self.sig_ag = B.Signals(B.tl_ag_gemm_num_flags(c["R"], c["S_shard"], c["H_kv"] * c["D"], 0)[0])
        self.epoch = 0

    def run(self, causal=False, self_rank=0):
        self.epoch += 1
        self.B.tl_ag_attn(self.Q, self.K, self.V, self.Kg, self.Vg, self.O, self.sig, self.epoch,
                          self_rank=self_rank, causal=causal, lse=self.L)

    def copy_only(self):
        """The key and value AllGathers alone (the stand-alone AllGather, two calls)."""
        c = AG_ATTN
        flat = lambda ts: [t.view(c["S_shard"], c["H_kv"] * c["D"]) for t in ts]
        self.epoch += 1
        self.B.tl_allgather(flat(self.K), self.Kg.view(-1, c["H_kv"] * c["D"]), self.sig_ag, self.epoch)
        self.epoch += 1
        self.B.tl_allgather(flat(self.V), self.Vg.view(-1, c["H_kv"] * c["D"]), self.sig_ag, self.epoch)

    def torch_decomposed(self):
        """torch: gather by concatenation, then scaled_dot_product_attention with grouped heads."""
        F = self.torch.nn.functional
        q = self.Q.permute(1, 0, 2).unsqueeze(0)
        k = self.torch.cat(self.K).permute(1, 0, 2).unsqueeze(0)
        v = self.torch.cat(self.V).permute(1, 0, 2).unsqueeze(0)
        return F.scaled_dot_product_attention(q, k, v, enable_gqa=True)

    def torch_cudnn(self):
        """torch: gather by concatenation, then the cuDNN fused attention (key/value heads
        expanded to the query heads when the backend takes no grouped heads)."""
        from torch.nn.attention import SDPBackend, sdpa_kernel
        F = self.torch.nn.functional
        q = self.Q.permute(1, 0, 2).unsqueeze(0)
        k = self.torch.cat(self.K).permute(1, 0, 2).unsqueeze(0)
        v = self.torch.cat(self.V).permute(1, 0, 2).unsqueeze(0)
        with sdpa_kernel([SDPBackend.CUDNN_ATTENTION]):
            try:
                return F.scaled_dot_product_attention(q, k, v, enable_gqa=True)
            except RuntimeError:
                g = q.shape[1] // k.shape[1]
                return F.scaled_dot_product_attention(q, k.repeat_interleave(g, dim=1),
                                                      v.repeat_interleave(g, dim=1))

    def check_status(self):
        for s in (self.sig, self.sig_ag):
            code, where = self.B.tl_query_status(s)
            if code:
                raise RuntimeError(f"device error {code} at {where} in the AllGather-KV attention")


# AllGather through the slow link (pinned host memory) at small messages: R=8 ranks, K=4096
# bf16 columns, 1..128 rows per shard (8 KB..1 MB)
LL_SIZES = dict(R=8, K=4096, M_shard=(1, 4, 16, 64, 128))


def ll_extras(torch, B, reps=7, batch=16):
    """Latency of one AllGather whose peer shards cross the slow link (pinned host memory):
    the flag-in-data protocol (tl_allgather_ll, 8-byte words of 4 data bytes + epoch) against
    the separate-flag protocol on the same link (data, system fence, flag), and against
    tl_allgather reading peer shards that sit in host memory with their readiness flags set
    (pull mode: one readiness wait per chunk).  Device time per call: batches of calls
    enqueued behind a GPU sleep, timed with CUDA events; the median over batches."""
    from tile_centric_gemm_gb300 import inputs
    R, K = LL_SIZES["R"], LL_SIZES["K"]
    rows = []
    for Ms in LL_SIZES["M_shard"]:
        A = [inputs.to_torch_bf16(inputs.normal_bf16((Ms, K), 1200 + r)).cuda() for r in range(R)]
        A_host = [A[0]] + [a.cpu().pin_memory() for a in A[1:]]
        link = torch.zeros(B.tl_allgather_ll_link_bytes(R, Ms, K), dtype=torch.uint8).pin_memory()
        G = torch.empty(R * Ms, K, dtype=torch.bfloat16, device="cuda")
        nfl = R * B.tl_ag_gemm_num_flags(R, Ms, K)[0]
        sig = B.Signals(max(nfl, R * Ms))
        ready = B.Signals(max(nfl, R * Ms))
        B.tl_tile_notify(ready, 0, ready.num_flags, 0x7FFF0000)
        ep = [0]

        def ll(protocol):
            ep[0] += 1
            B.tl_allgather_ll(A, link, G, sig, ep[0], protocol=protocol)

        def ag_host():
            ep[0] += 1
            B.tl_allgather(A_host, G, sig, ep[0], mode=B.TL_MODE_PULL, src_ready=ready)

        res = {"shard_bytes": Ms * K * 2}
        for name, fn in (("flag_in_data", lambda: ll(B.TL_LL_FLAG_IN_DATA)),
                         ("separate_flag", lambda: ll(B.TL_LL_SEPARATE_FLAG)), ("tl_allgather_host_pull", ag_host)):
            fn()
            ts = []
            for _ in range(reps):
                # the GPU first sleeps while the host enqueues a batch of calls, so the events
                # time the calls back to back on the device, not the host's launch rate
                torch.cuda._sleep(3_000_000)
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                for _ in range(batch):
                    fn()
                b.record()
                b.synchronize()
                ts.append(a.elapsed_time(b) * 1e3 / batch)
            res[name + "_us"] = statistics.median(ts)
        for s in (sig, ready):
            code, where = B.tl_query_status(s)
            if code:
                raise RuntimeError(f"device error {code} at {where} in the slow-link AllGather")
        res["speedup_flag_in_data_vs_separate_flag"] = res["separate_flag_us"] / res["flag_in_data_us"]
        rows.append(res)
        del A, A_host, link, G
    return {"config": LL_SIZES, "link": "pinned host memory", "rows": rows,
            "what": "one AllGather of R shards through the slow link; device time per call, batches of "
                    "back-to-back calls enqueued behind a GPU sleep"}


def attn_extras(torch, B, peaks, peak_src):
    a = AgAttn(B, torch)
    c = AG_ATTN
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    out = {"config": c, "what": "AllGather of the key/value shards fused with the attention over them, one launch; "
                                "flops = 4 * D * H * visible (query, key) pairs",
           "peak_tflops": peaks["bf16_tflops"], "peak_source": f"{peak_src} bf16 burst"}
    for name, causal, self_rank in (("full", False, 0), ("causal_last_rank", True, c["R"] - 1),
                                    ("causal_middle_rank", True, c["R"] // 2 - 1)):
        t = flushed_time_us(torch, lambda: a.run(causal, self_rank), flush, reps=5)
        fl = attn_flops(c, causal, self_rank)
        out[name] = {"us": t, "tflops": fl / (t * 1e-6) / 1e12, "self_rank": self_rank, "causal": causal,
                     "frac": fl / (t * 1e-6) / 1e12 / peaks["bf16_tflops"]}
    a.check_status()
    t_copy = flushed_time_us(torch, a.copy_only, flush, reps=5)
    a.check_status()
    kv_bytes = 2 * c["R"] * c["S_shard"] * c["H_kv"] * c["D"] * 2
    out["copy_only"] = {"us": t_copy, "gbs": 2 * kv_bytes / (t_copy * 1e-6) / 1e9,
                        "what": "tl_allgather of K then V (read + write bytes / time)"}
    try:
        t_torch = flushed_time_us(torch, a.torch_decomposed, flush, reps=3)
        fl = attn_flops(c, False, 0)
        out["torch_cat_sdpa"] = {"us": t_torch, "tflops": fl / (t_torch * 1e-6) / 1e12,
                                 "speedup_of_fused": t_torch / out["full"]["us"]}
    except Exception as ex:  # a torch build without a fused attention for this device
        out["torch_cat_sdpa"] = {"unavailable": str(ex).splitlines()[0][:200]}
    try:
        t_cudnn = flushed_time_us(torch, a.torch_cudnn, flush, reps=3)
        fl = attn_flops(c, False, 0)
        out["torch_cat_cudnn_sdpa"] = {"us": t_cudnn, "tflops": fl / (t_cudnn * 1e-6) / 1e12,
                                       "speedup_of_fused": t_cudnn / out["full"]["us"]}
    except Exception as ex:  # no cuDNN attention for this device or build
        out["torch_cat_cudnn_sdpa"] = {"unavailable": str(ex).splitlines()[0][:200]}
    # the copy runs inside the fused launch; alone it would add this much to a copy-then-attend schedule
    out["copy_frac_of_fused"] = t_copy / out["full"]["us"]
    del a, flush
    return out


def main():
    args = parse()
    world, rank, local_rank = dist_env()
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from tile_centric_gemm_gb300 import binding as B

    torch.cuda.set_device(local_rank)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
        pg = dist

    def barrier():
        torch.cuda.synchronize()
        if pg:
            pg.barrier()

    peaks, peak_src = load_peaks()
    if args.sweep:
        rows = run_sweep(torch, B, peaks)
        if rank == 0:
            print(json.dumps({"sweep": "AG-GEMM K=8192 N=1024, bf16 N(0,1) x N(0,0.02), cold L2, median of 5",
                              "peak_tflops": peaks["bf16_tflops"], "rows": rows}), flush=True)
        return
    wl = Workload(B, torch)
    stream = torch.cuda.current_stream()
    if args.only:
        if args.only == "moe_down":
            wl.moe()  # the routing the down projection reads
            down = MoeDown(B, torch, wl)
            fn, flops = down.run, MOE_DOWN_FLOPS
        elif args.only == "ag_attn":
            attn = AgAttn(B, torch)
            fn, flops = attn.run, attn_flops(AG_ATTN, False, 0)
        elif args.only == "allgather_ll":
            # one slow-link AllGather (flag in data) of 8 ranks x 16 rows x 4096 columns (128 KB per
            # shard), the link in pinned host memory; "flops" stands for the bytes gathered
            from tile_centric_gemm_gb300 import inputs as _in
            Ms_ll = 16
            A_ll = [_in.to_torch_bf16(_in.normal_bf16((Ms_ll, 4096), 1200 + r)).cuda() for r in range(8)]
            link = torch.zeros(B.tl_allgather_ll_link_bytes(8, Ms_ll, 4096), dtype=torch.uint8).pin_memory()
            G_ll = torch.empty(8 * Ms_ll, 4096, dtype=torch.bfloat16, device="cuda")
            sig_ll = B.Signals(8 * Ms_ll)
            ep_ll = [0]

            def fn():
                ep_ll[0] += 1
                B.tl_allgather_ll(A_ll, link, G_ll, sig_ll, ep_ll[0])
            flops = 8 * Ms_ll * 4096 * 2
        elif args.only == "gemm_vs_library":
            # the compute half of the AG-GEMM alone (tl_gemm on the gathered matrix), then the
            # library GEMM on the same operands: one launch of each per call, for profiling them
            # side by side; the time printed covers both
            wl.ag()
            C_lib = torch.empty_like(wl.C)
            sig_g = B.Signals(1)

            def fn():
                B.tl_gemm(wl.G, wl.d_ag[AG["R"]], wl.C, sig_g)
                torch.matmul(wl.G, wl.d_ag[AG["R"]], out=C_lib)
            flops = 2 * AG_FLOPS
        else:
            fn = {"ag": wl.ag, "rs": wl.rs, "moe": wl.moe}[args.only]
            flops = {"ag": AG_FLOPS, "rs": RS_FLOPS, "moe": MOE_FLOPS}[args.only]
        for _ in range(args.warmup):
            fn()
        barrier()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(args.steps):
            fn()
        b.record(stream)
        barrier()
        wl.check_status()
        us = a.elapsed_time(b) * 1e3 / max(1, args.steps)
        if rank == 0:
            print(json.dumps({"only": args.only, "us_per_call": us, "tflops": flops / (us * 1e-6) / 1e12,
                              "calls": args.steps, "warmup": args.warmup}), flush=True)
        return
    for _ in range(max(3, args.warmup)):
        wl.ag()
        wl.rs()
        wl.moe()
    wl.check_status()

    sampler = ClockSampler(local_rank)
    time.sleep(0.3)
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    barrier()
    t_host0 = time.time()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(K):
        ev[i][0].record(stream)
        wl.ag()
        ev[i][1].record(stream)
        wl.rs()
        ev[i][2].record(stream)
        wl.moe()
        ev[i][3].record(stream)
    end.record(stream)
    barrier()
    t_host1 = time.time()
    sampler.stop()
    wl.check_status()
    total_ms = start.elapsed_time(end)
    ag_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(K)]
    rs_ms = [ev[i][1].elapsed_time(ev[i][2]) for i in range(K)]
    moe_ms = [ev[i][2].elapsed_time(ev[i][3]) for i in range(K)]
    ms_per_step = total_ms / K
    ms_per_step = max_over_ranks(pg, ms_per_step)
    step_flops = AG_FLOPS + RS_FLOPS + MOE_FLOPS
    value = world * step_flops / (ms_per_step * 1e-3) / 1e12

    # end to end through the public API with host buffers: every step copies its inputs in
    # from pinned host memory, runs the three calls and reads its outputs back
    E = max(3, args.e2e_steps)
    e2e_serial_ms = max_over_ranks(pg, e2e_serial(torch, wl, E, stream, barrier, weights=False))
    e2e_ms = max_over_ranks(pg, e2e_pipelined(torch, wl, E, stream, barrier, weights=False))
    e2e_all_ms = max_over_ranks(pg, e2e_pipelined(torch, wl, E, stream, barrier, weights=True))
    wl.check_status()

    rs_avg = statistics.mean(rs_ms)
    ag_avg = statistics.mean(ag_ms)
    moe_avg = statistics.mean(moe_ms)
    achieved = RS_FLOPS / (rs_avg * 1e-3) / 1e12
    peak = peaks["bf16_tflops"]
    clocks = sampler.summary(t_host0, t_host1)
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "ag": AG, "rs": RS, "moe": MOE, "step_gflop": step_flops / 1e9,
                   "l2": "inputs larger than L2: a step touches ~2.3 GB (129 MB L2); no flush",
                   "parallelism": f"{world} independent replica(s), 8 emulated ranks each"},
        "breakdown": {"ag_gemm_us": ag_avg * 1e3, "ag_gemm_tflops": AG_FLOPS / (ag_avg * 1e-3) / 1e12,
                      "gemm_rs_us": rs_avg * 1e3, "gemm_rs_tflops": achieved,
                      "moe_us": moe_avg * 1e3, "moe_tflops": MOE_FLOPS / (moe_avg * 1e-3) / 1e12},
        "roofline": {"bound": "tensor", "kernel": "gemm_rs_kernel", "achieved": achieved, "peak": peak,
                     "unit": "TFLOP/s", "frac": achieved / peak, "peak_source": f"{peak_src} bf16 burst",
                     "frac_of_sustained": achieved / peaks.get("bf16_tflops_sustained", peak),
                     "traffic": rs_traffic(), "traffic_unit": "bytes per launch (ncu DRAM read + write)",
                     "algorithmic_bytes": RS_BYTES,
                     "algorithmic_bytes_with_partials": RS_BYTES + RS_PARTIAL_BYTES,
                     # every call of the step against the same peak (CUDA events around each call)
                     "per_call": {
                         name: {"kernels": kern, "achieved": fl / (us * 1e-3) / 1e12,
                                "frac": fl / (us * 1e-3) / 1e12 / peak,
                                "frac_of_sustained": fl / (us * 1e-3) / 1e12 / peaks.get("bf16_tflops_sustained", peak)}
                         for name, kern, fl, us in (
                             ("ag_gemm", "ag_gemm_kernel", AG_FLOPS, ag_avg),
                             ("gemm_rs", "gemm_rs_kernel", RS_FLOPS, rs_avg),
                             ("moe_ag_gemm", "moe_route_kernel + moe_gemm_kernel (useful flops, no padding)",
                              MOE_FLOPS, moe_avg))}},
        "clocks": clocks,
        "e2e": {"value": world * step_flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": wl.h2d_bytes(weights=False),
                "d2h_bytes_per_step": wl.d2h_bytes(),
                "inputs": "activations (A shards, A_r, token shards) and top-k ids copied in every step; the "
                          "weights (B, B_r, W_e) are model state, loaded once before the timed region",
                "how": "double-buffered: step i+1's inputs copy in on a copy stream while step i computes, "
                       "step i's outputs copy out on a third stream",
                "serial_ms_per_step": e2e_serial_ms,
                "serial_value": world * step_flops / (e2e_serial_ms * 1e-3) / 1e12,
                "all_operands": {"value": world * step_flops / (e2e_all_ms * 1e-3) / 1e12,
                                 "ms_per_step": e2e_all_ms, "h2d_bytes_per_step": wl.h2d_bytes(),
                                 "what": "the same, with every weight copied in every step as well"}},
        "gpu_launches": K * wl.launches_per_step,
    }
    if not args.no_overlap:
        line["overlap"] = overlap_metrics(torch, B, wl)
    if not args.no_extras:
        # outside the step: the MoE layer's down-projection side on the step's routing
        down = MoeDown(B, torch, wl)
        flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
        t = flushed_time_us(torch, down.run, flush, reps=5)
        t_bf16 = flushed_time_us(torch, lambda: down.run(options=B.TL_RS_BF16_PARTIALS), flush, reps=5)
        down.check_status()
        line["extras"] = {"moe_down": {"us": t, "tflops": MOE_DOWN_FLOPS / (t * 1e-6) / 1e12, "config": MOE_DOWN,
                                       "bf16_partials_us": t_bf16,
                                       "bf16_partials_tflops": MOE_DOWN_FLOPS / (t_bf16 * 1e-6) / 1e12,
                                       "what": "grouped GEMM -> ReduceScatter over ranks -> gate-weighted "
                                               "TopK-reduce -> scatter, one call (two launches); fp32 partials, "
                                               "and bf16 partials (TL_RS_BF16_PARTIALS)"}}
        del down, flush
        line["extras"]["ag_attn"] = attn_extras(torch, B, peaks, peak_src)
        line["extras"]["allgather_ll"] = ll_extras(torch, B)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tf, dt, sample = time_oracle()
        line["cpu_baseline"] = {"value": tf, "unit": "TFLOP/s", "cores": cpu_threads(), "kind": "oracle",
                                "sample": sample, "seconds": dt}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
