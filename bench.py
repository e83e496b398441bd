"""Benchmark: batch-1 decode of the 8B-shaped ternary model on GB300.

One step = one decode token through the library's public C ABI (nt_decode_step, persistent
launcher): in-step int8 quantization of every projection input, all 36 x {q, k, v, o, gate,
up, down} ternary projections, then the int8 output projection over 151,936 x 4,096 with the
greedy arg-max. Inputs are seeded and synthetic with the workloads' shapes and value mixes;
weights are resident in HBM before timing, and every step streams 2.37 GB (>> the 129 MB L2),
so no L2 flush is needed between steps.

Prints ONE JSON line (rank 0). `--impl reference` times the CPU oracle instead (the only
other place this script runs oracle code besides the cpu_baseline leg).
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from synth import workloads as wl  # noqa: E402

METRIC = "8B-shape decode weight-stream µs/token; achieved HBM GB/s vs GB300 peak"
WORKLOAD = ("8B-shaped batch-1 decode token: 36 layers x ternary {q,k,v,o,gate,up,down} "
            "GEMVs (2-bit trits, 16/uint32, per-row fp32 scales) + int8 output table "
            "151936x4096 with greedy argmax")
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "persist_kernel_decode8b_traffic.txt")
KERNEL_SOURCES = ["packed_weight_gemv_gb300/csrc/nt_persist.cu",
                  "packed_weight_gemv_gb300/csrc/nt_internal.cuh",
                  "packed_weight_gemv_gb300/csrc/nt_step.cuh",
                  "packed_weight_gemv_gb300/csrc/nt_kernels.cuh"]


def step_bytes(B: int = 1, n_layers: int = wl.DECODER_8B_LAYERS) -> int:
    """Algorithmic bytes of one decode token: the projection stream (packed trits, row scales,
    int8 activations, fp32 outputs, activation scales), the fp32 inputs the step quantizes
    (read once, int8 written once -- counted in the activations), and the output projection
    (table, row scales, hidden, logits, arg-max)."""
    fp32_inputs = 4 * B * sum(K for (_, K) in wl.DECODER_8B.values()) * n_layers
    fp32_inputs += 4 * B * wl.HEAD_K
    return wl.packed_bytes_per_token(n_layers=n_layers, B=B) + wl.head_bytes(B=B) + fp32_inputs


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def read_traffic():
    """DRAM bytes per launch from the committed ncu summary, if it was taken on this exact
    kernel source; else None."""
    try:
        kv = {}
        with open(PROFILE_TRAFFIC) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("kernel_source_sha256_16") != kernel_source_hash():
            return None
        return int(kv["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


def measured_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def mark(self, start: bool):
        if start:
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        return parse_clock_samples(out)


def parse_clock_samples(out: str) -> dict:
    """Median SM clock, the maximum clock and every throttle reason seen Active, from
    nvidia-smi's `--format=csv,noheader,nounits` rows of ClockSampler.FIELDS. Rows that do not
    parse (a truncated last line, "[N/A]") are skipped."""
    rows = [r for r in csv.reader(io.StringIO(out)) if len(r) >= 9]
    sm, mx, reasons = [], None, set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for r in rows:
        try:
            sm.append(float(r[1]))
            mx = float(r[2])
        except ValueError:
            continue
        for n, v in zip(names, r[5:9]):
            if v.strip().lower() == "active":
                reasons.add(n)
    return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
            "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------------------
# Replicas: one process per GPU, each decoding its own tokens; the job's time is the slowest
# rank's. Collectives here only align the start and take the maximum.
# ---------------------------------------------------------------------------------------

def max_over_ranks(torch, x: float, world: int, device) -> float:
    """The largest of every rank's x; x itself on one rank. A collective when world > 1: every
    rank calls it at the same point."""
    if world <= 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_us_per_token(slowest_us: float, tokens_per_rank: int, world: int) -> float:
    """Whole-job microseconds per token: `world` replicas each decoded tokens_per_rank tokens in
    a window as long as the slowest rank's time."""
    return slowest_us / (tokens_per_rank * world)


def host_timed_job(torch, step, n: int, world: int, device, sync=None) -> float:
    """Whole-job microseconds per token of n calls step(0) ... step(n - 1) on every rank, timed
    on the host: the ranks start together after a barrier, sync() (if given) ends each rank's
    window, and the job's window is the slowest rank's."""
    if world > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    for i in range(n):
        step(i)
    if sync is not None:
        sync()
    us = (time.perf_counter() - t0) * 1e6
    return job_us_per_token(max_over_ranks(torch, us, world, device), n, world)


# ---------------------------------------------------------------------------------------
# Our arm
# ---------------------------------------------------------------------------------------

def build_inputs(torch, nt, dev, n_layers=wl.DECODER_8B_LAYERS):
    """Device-resident model: tiled weights, scales; fp32 inputs in one buffer."""
    projs = wl.decoder_projections(n_layers)
    head = wl.head()
    K_total = sum(p.K for p in projs) + head.K
    x_all = torch.empty(K_total, dtype=torch.float32, device=dev)
    dp, off = [], 0
    for p in projs:
        w_plain = torch.from_numpy(p.w_plain.view(np.int32)).to(dev)
        w = torch.empty(nt.nt_repack_size(p.N, p.K), dtype=torch.uint8, device=dev)
        nt.nt_repack_ternary(w_plain, p.N, p.K, w)
        del w_plain
        x = x_all[off:off + p.K]
        x.copy_(torch.from_numpy(p.x[0]))
        off += p.K
        dp.append(dict(N=p.N, K=p.K, w=w, s_w=torch.from_numpy(p.s_w).to(dev), x=x,
                       q=torch.empty(p.K, dtype=torch.int8, device=dev),
                       s_x=torch.empty(1, dtype=torch.float32, device=dev),
                       y=torch.empty(p.N, dtype=torch.float32, device=dev)))
        p.w_plain = None  # regenerated on demand for the parity sample
    hx = x_all[off:off + head.K]
    hx.copy_(torch.from_numpy(head.x[0]))
    hd = dict(T=torch.from_numpy(head.T).to(dev), s=torch.from_numpy(head.s_T).to(dev),
              V=head.V, K=head.K, x=hx, q=torch.empty(head.K, dtype=torch.int8, device=dev),
              sx=torch.empty(1, dtype=torch.float32, device=dev),
              logits=torch.empty(head.V, dtype=torch.float32, device=dev),
              argmax=torch.empty(1, dtype=torch.int32, device=dev))
    torch.cuda.synchronize()
    return projs, head, dp, hd, x_all


def parity_gate(oracle, projs, head, dp, hd, layers=(0, 35)):
    """Sampled parity before any timing: every projection of the sampled layers and the full
    output projection, against the oracle (acc-derived fp32 within 1e-6, arg-max exact)."""
    for p, d in zip(projs, dp):
        layer = int(p.name.split(".")[0][1:])
        if layer not in layers:
            continue
        pi = wl.PROJ_NAMES.index(p.name.split(".")[1])
        full = wl.projection(wl.WL_DECODE, layer, pi, p.N, p.K)
        q, s = oracle.quantize(full.x)
        if not (np.array_equal(d["q"].cpu().numpy(), q[0]) and d["s_x"].cpu().numpy()[0] == s[0]):
            return f"{p.name}: int8 codes differ"
        _, y, _ = oracle.gemv(full.w_plain, full.s_w, p.N, p.K, q[0], s)
        got = d["y"].cpu().numpy().astype(np.float64)
        if np.any(np.abs(got - y) > 1e-6 * np.abs(y.astype(np.float64))):
            return f"{p.name}: outputs differ"
    q, s = oracle.quantize(head.x)
    logits, am, _ = oracle.logits_argmax(head.T, head.s_T, head.V, head.K, q, s)
    got = hd["logits"].cpu().numpy().astype(np.float64)
    if np.any(np.abs(got - logits[0]) > 1e-6 * np.abs(logits[0].astype(np.float64))):
        return "output projection logits differ"
    if int(hd["argmax"].cpu().item()) != int(am[0]):
        return "arg-max differs"
    return "pass"


def time_steps(torch, plan, steps, stream, nvtx_name=None):
    """Device time of `steps` consecutive steps (CUDA events on the launching stream). The
    NVTX range lets `ncu --nvtx --nvtx-include <name>/` list exactly these launches."""
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    if nvtx_name:
        torch.cuda.nvtx.range_push(nvtx_name)
    ev0.record(stream)
    for _ in range(steps):
        plan.nt_decode_step(stream)
    ev1.record(stream)
    torch.cuda.synchronize()
    if nvtx_name:
        torch.cuda.nvtx.range_pop()
    return ev0.elapsed_time(ev1) * 1e3  # microseconds


def step_distribution(torch, plan, steps, stream):
    """Per-step device times of `steps` consecutive steps: one CUDA event between every two
    steps on the launching stream (events add no work between the launches). Median, 10th and
    90th percentile in microseconds."""
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    torch.cuda.synchronize()
    ev[0].record(stream)
    for i in range(steps):
        plan.nt_decode_step(stream)
        ev[i + 1].record(stream)
    torch.cuda.synchronize()
    return percentiles_us([ev[i].elapsed_time(ev[i + 1]) * 1e3 for i in range(steps)])


def percentiles_us(d) -> dict:
    d = np.asarray(d, dtype=np.float64)
    return {"n": int(d.size), "median": round(float(np.median(d)), 2),
            "p10": round(float(np.percentile(d, 10)), 2), "p90": round(float(np.percentile(d, 90)), 2),
            "min": round(float(d.min()), 2), "max": round(float(d.max()), 2)}


def cpu_baseline(oracle, budget_s=12.0):
    """The oracle on a bounded sample of the same workload, scaled to microseconds per token:
    a whole decoder layer (7 projections, the layer's int8 quantization included) and a
    slice of the output table, repeated while under the time budget."""
    layer = [wl.projection(wl.WL_DECODE, 0, i, *wl.DECODER_8B[n]) for i, n in enumerate(wl.PROJ_NAMES)]
    hv = 8192
    head = wl.head(V=hv)
    t_layer, t_head, n = 0.0, 0.0, 0
    while n == 0 or (t_layer + t_head) * (n + 1) / n < budget_s:
        t0 = time.perf_counter()
        for p in layer:
            q, s = oracle.quantize(p.x)
            oracle.gemv(p.w_plain, p.s_w, p.N, p.K, q[0], s)
        t1 = time.perf_counter()
        q, s = oracle.quantize(head.x)
        oracle.logits_argmax(head.T, head.s_T, hv, head.K, q, s)
        t2 = time.perf_counter()
        t_layer += t1 - t0
        t_head += t2 - t1
        n += 1
    us = (t_layer / n * wl.DECODER_8B_LAYERS + t_head / n * wl.HEAD_V / hv) * 1e6
    return {"value": round(us, 1), "unit": "us/token", "cores": oracle.threads(), "kind": "oracle",
            "sample": (f"1 of 36 decoder layers (7 projections, seed-0 inputs) + {hv} of "
                       f"151936 output-table rows, {n} repetition(s), scaled to one token")}


class OracleRounds:
    """The oracle timed per workload at one thread and at every core, one round at a time, so
    that its rounds can interleave with the GPU's: the single 1536 x 512 GEMV (config 1), one
    decoder layer of the 8B-shaped step (scaled to the 36-layer token, config 2) and 8,192 rows of
    the output table (scaled to 151,936, config 3); throughput in GB/s of packed weight bytes."""

    def __init__(self, oracle):
        self.o = oracle
        self.cores = os.cpu_count() or 1
        self.single = wl.single_gemv()
        self.layer = [wl.projection(wl.WL_DECODE, 0, i, *wl.DECODER_8B[n]) for i, n in enumerate(wl.PROJ_NAMES)]
        self.hv = 8192
        self.head = wl.head(V=self.hv)
        self.rows = {}

    def _time(self, fn, min_s):
        n, t0 = 0, time.perf_counter()
        while True:
            fn()
            n += 1
            dt = time.perf_counter() - t0
            if dt >= min_s:
                return dt / n

    def round(self):
        o, p1, h = self.o, self.single, self.head
        q1, s1 = o.quantize(p1.x)
        ql = [o.quantize(p.x) for p in self.layer]
        qh, sh = o.quantize(h.x)
        res = {}
        for th in (1, self.cores):
            o.set_threads(th)
            t1 = self._time(lambda: o.gemv(p1.w_plain, p1.s_w, p1.N, p1.K, q1[0], s1), 0.2)
            tl = self._time(lambda: [o.gemv(p.w_plain, p.s_w, p.N, p.K, q[0], s)
                                     for p, (q, s) in zip(self.layer, ql)], 0.5)
            th_ = self._time(lambda: o.logits_argmax(h.T, h.s_T, self.hv, h.K, qh, sh), 0.3)
            res[th] = (t1, tl, th_)
        o.set_threads(0)
        for th, v in res.items():
            self.rows.setdefault(th, []).append(v)

    def summary(self):
        p1 = self.single
        b1 = p1.N * p1.K // 4
        bl = wl.packed_bytes_per_token(n_layers=1)
        bh = self.hv * self.head.K
        out = {}
        for th, rows in self.rows.items():
            t1, tl, th_ = (statistics.median(c) for c in zip(*rows))
            out[f"threads_{th}"] = {
                "config1_single_gemv": {"us_per_call": round(t1 * 1e6, 2), "GBps_packed": round(b1 / t1 / 1e9, 3)},
                "config2_decode_projections": {"us_per_token": round(tl * wl.DECODER_8B_LAYERS * 1e6, 1),
                                               "GBps_packed": round(bl / tl / 1e9, 3)},
                "config3_lm_head": {"us_per_token": round(th_ * wl.HEAD_V / self.hv * 1e6, 1),
                                    "GBps_packed": round(bh / th_ / 1e9, 3)},
            }
        return out


def time_single_gemv(torch, nt, oracle, dev, stream, peak):
    """The single 1536 x 512 GEMV of the first workload, per call: with its weights resident in L2
    (the same matrix every call) and cold (a rotating pool of copies larger than 4 x L2, one
    copy per call). The calls are captured in a CUDA graph and replayed, so the host's per-call
    cost is not timed; parity against the oracle first."""
    p = wl.single_gemv()
    q, s = oracle.quantize(p.x)
    acc, y, _ = oracle.gemv(p.w_plain, p.s_w, p.N, p.K, q[0], s)
    w = torch.empty(nt.nt_repack_size(p.N, p.K), dtype=torch.uint8, device=dev)
    nt.nt_repack_ternary(torch.from_numpy(p.w_plain.view(np.int32)).to(dev), p.N, p.K, w)
    sw = torch.from_numpy(p.s_w).to(dev)
    qd, sd = torch.from_numpy(q[0]).to(dev), torch.from_numpy(s).to(dev)
    yd = torch.empty(p.N, dtype=torch.float32, device=dev)
    ad = torch.empty(p.N, dtype=torch.int32, device=dev)
    nt.nt_ternary_gemv(w, nt.NT_LAYOUT_TILED, sw, p.N, p.K, qd, sd, yd, ad, stream=stream)
    torch.cuda.synchronize()
    ok = np.array_equal(ad.cpu().numpy(), acc) and np.all(
        np.abs(yd.cpu().numpy().astype(np.float64) - y) <= 1e-6 * np.abs(y.astype(np.float64)))
    nbytes = p.N * p.K // 4 + 4 * p.N + p.K + 4 * p.N + 4
    l2 = 129 * 2 ** 20
    pool_n = -(-4 * l2 // (w.numel() + 4 * p.N))
    ws = w.unsqueeze(0).repeat(pool_n, 1)
    sws = sw.unsqueeze(0).repeat(pool_n, 1)

    def graph_of(calls):
        for _ in range(2):
            calls()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            calls()
        return g

    def hot():
        st = torch.cuda.current_stream()
        for _ in range(pool_n):
            nt.nt_ternary_gemv(w, nt.NT_LAYOUT_TILED, sw, p.N, p.K, qd, sd, yd, stream=st)

    def cold():
        st = torch.cuda.current_stream()
        for i in range(pool_n):
            nt.nt_ternary_gemv(ws[i], nt.NT_LAYOUT_TILED, sws[i], p.N, p.K, qd, sd, yd, stream=st)

    res = {}
    for name, calls in (("l2_resident", hot), ("cold_rotating_pool", cold)):
        g = graph_of(calls)
        g.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(3):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / (3 * pool_n)
        gbs = nbytes / (us * 1e-6) / 1e9
        res[name] = {"us_per_call": round(us, 3), "GBps": round(gbs, 1), "frac_of_hbm": round(gbs / peak, 4)}
        del g
    del ws, sws
    torch.cuda.empty_cache()
    return dict(res, bytes_per_call=nbytes, calls_per_replay=pool_n, kernel="gemv_tiled_kernel",
                pool_bytes=int(pool_n * (w.numel() + 4 * p.N)), parity="pass" if ok else "differs",
                what="1536x512 trits (seed 0), batch 1, nt_ternary_gemv calls replayed as a CUDA graph")


def run_ours(args, rank, world):
    import torch

    import oracle
    from packed_weight_gemv_gb300 import nt

    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    nt.nt_device_check()
    L = args.layers
    projs, head, dp, hd, x_all = build_inputs(torch, nt, dev, L)
    stream = torch.cuda.current_stream()
    plan = nt.DecodePlan(L, 1, dp, hd, nt.NT_STEP_INDEPENDENT, nt.NT_LAUNCH_PERSISTENT)
    for _ in range(args.warmup):
        plan.nt_decode_step(stream)
    torch.cuda.synchronize()
    if plan.nt_decode_step_status() != nt.NT_OK:
        raise RuntimeError("persistent step reported a timeout during warm-up")
    parity = parity_gate(oracle, projs, head, dp, hd, layers=(0, L - 1)) if rank == 0 else "pass"
    if parity != "pass":
        raise RuntimeError(f"parity gate failed: {parity}")

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.mark(True)
    us = time_steps(torch, plan, args.steps, stream, nvtx_name="nt_timed")
    clocks.mark(False)
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    if plan.nt_decode_step_status() != nt.NT_OK:
        raise RuntimeError("persistent step reported a timeout in the timed region")
    us = max_over_ranks(torch, us, world, dev)
    per_step_us = us / args.steps
    value = job_us_per_token(us, args.steps, world)
    # after the timed region: the spread of single steps (at least 50), this rank's
    dist_steps = step_distribution(torch, plan, max(50, min(args.steps, 2000)), stream)
    if plan.nt_decode_step_status() != nt.NT_OK:
        raise RuntimeError("persistent step reported a timeout in the per-step timing")

    # Serial end to end through the same public call: every step copies its fp32 inputs from
    # pinned host memory, runs, and reads its token back to the host before the next step
    # starts, as a dependent single-stream decode must.
    x_host = torch.empty(x_all.numel(), dtype=torch.float32, pin_memory=True)
    x_host.copy_(x_all.cpu())
    am_host = torch.empty(2, dtype=torch.int32, pin_memory=True)

    def serial_step():
        x_all.copy_(x_host, non_blocking=True)
        plan.nt_decode_step(stream)
        am_host[0:1].copy_(hd["argmax"], non_blocking=True)
        stream.synchronize()

    serial_steps = max(1, min(args.steps, 2000))
    for _ in range(3):
        serial_step()
    e2e_serial_us = host_timed_job(torch, lambda i: serial_step(), serial_steps, world, dev)
    if int(am_host[0]) != int(hd["argmax"].item()):
        raise RuntimeError("serial end-to-end: the token read back differs from the device's")

    # The same serial loop recorded once into a CUDA graph (copy in, step, token out) and
    # replayed per token: a single-launch persistent step takes the same launch parameters on
    # every call, so the recorded step stays valid.
    graph = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(graph, stream=torch.cuda.Stream()):  # recorded on a side stream
        x_all.copy_(x_host, non_blocking=True)
        plan.nt_decode_step()  # the capturing stream is the current one here
        am_host[1:2].copy_(hd["argmax"], non_blocking=True)
    graph_stream = torch.cuda.current_stream()

    def graph_step():
        graph.replay()
        graph_stream.synchronize()

    for _ in range(3):
        graph_step()
    e2e_graph_us = host_timed_job(torch, lambda i: graph_step(), serial_steps, world, dev)
    if int(am_host[1]) != int(hd["argmax"].item()) or plan.nt_decode_step_status() != nt.NT_OK:
        raise RuntimeError("graph end-to-end: the token read back differs from the device's")
    del graph

    # The same serial loop with no copy call: a second plan whose fp32 inputs are views of the
    # pinned host buffer, read by the step's first phase over the host link (this part's
    # coherent CPU-GPU link; every byte still crosses it every step). Its outputs must equal
    # the device-input plan's.
    dp_zc, off = [], 0
    for d in dp:
        dp_zc.append(dict(d, x=x_host[off:off + d["K"]], q=torch.empty_like(d["q"]),
                          s_x=torch.empty_like(d["s_x"]), y=torch.empty_like(d["y"])))
        off += d["K"]
    hd_zc = dict(hd, x=x_host[off:off + head.K], q=torch.empty_like(hd["q"]), sx=torch.empty_like(hd["sx"]),
                 logits=torch.empty_like(hd["logits"]), argmax=torch.empty_like(hd["argmax"]))
    plan_zc = nt.DecodePlan(L, 1, dp_zc, hd_zc, nt.NT_STEP_INDEPENDENT, nt.NT_LAUNCH_PERSISTENT)

    def zero_copy_step():
        plan_zc.nt_decode_step(stream)
        am_host[1:2].copy_(hd_zc["argmax"], non_blocking=True)
        stream.synchronize()

    for _ in range(3):
        zero_copy_step()
    e2e_zero_copy_us = host_timed_job(torch, lambda i: zero_copy_step(), serial_steps, world, dev)
    serial_step()  # the device-input plan's outputs for the same inputs
    torch.cuda.synchronize()
    if (plan_zc.nt_decode_step_status() != nt.NT_OK or int(am_host[1]) != int(hd["argmax"].item())
            or not torch.equal(hd_zc["logits"], hd["logits"])
            or not all(torch.equal(a["q"], b["q"]) and torch.equal(a["y"], b["y"]) for a, b in zip(dp, dp_zc))):
        raise RuntimeError("zero-copy end-to-end: outputs differ from the device-input plan's")
    plan_zc.close()
    del dp_zc, hd_zc

    # Pipelined end to end through the same public call, with pinned host buffers: every step
    # copies its fp32 inputs host->device, runs the step and reads the emitted token back.
    # Inputs and token are double-buffered: step i+1's copy (on its own stream) overlaps step
    # i's compute and waits until step i-1 has finished with the buffers it overwrites; the
    # token is read back on a third stream. Possible only because the workload supplies every
    # step's inputs (a dependent decode cannot do this: the serial figure above is its cost).
    x_alt = torch.empty_like(x_all)
    dp_alt, off = [], 0
    for d in dp:
        dp_alt.append(dict(d, x=x_alt[off:off + d["K"]]))
        off += d["K"]
    hd_alt = dict(hd, x=x_alt[off:off + head.K], argmax=torch.empty_like(hd["argmax"]))
    plans = [plan, nt.DecodePlan(L, 1, dp_alt, hd_alt, nt.NT_STEP_INDEPENDENT, nt.NT_LAUNCH_PERSISTENT)]
    bufs, am_dev = [x_all, x_alt], [hd["argmax"], hd_alt["argmax"]]
    copy_stream, read_stream = torch.cuda.Stream(), torch.cuda.Stream()
    copied = [torch.cuda.Event() for _ in range(2)]
    consumed = [torch.cuda.Event() for _ in range(2)]
    read = [torch.cuda.Event() for _ in range(2)]
    for k in range(2):
        consumed[k].record(stream)
        read[k].record(stream)

    def e2e_step(i):
        # inputs of step i into buffer set k on the copy stream once step i - 2 has consumed
        # them; the token read back on its own stream, so the next step never waits for it
        k = i % 2
        copy_stream.wait_event(consumed[k])
        with torch.cuda.stream(copy_stream):
            bufs[k].copy_(x_host, non_blocking=True)
            copied[k].record(copy_stream)
        stream.wait_event(copied[k])
        stream.wait_event(read[k])
        plans[k].nt_decode_step(stream)
        consumed[k].record(stream)
        read_stream.wait_event(consumed[k])
        with torch.cuda.stream(read_stream):
            am_host[k:k + 1].copy_(am_dev[k], non_blocking=True)
            read[k].record(read_stream)

    e2e_steps = max(1, min(args.steps, 2000))
    for i in range(4):
        e2e_step(i)
    torch.cuda.synchronize()
    e2e_us = host_timed_job(torch, e2e_step, e2e_steps, world, dev, sync=torch.cuda.synchronize)
    if plans[1].nt_decode_step_status() != nt.NT_OK:
        raise RuntimeError("end-to-end steps reported a timeout")
    plans[1].close()

    # The oracle's protocol: GPU steps and the oracle's samples in interleaved rounds (the
    # oracle at one thread and at every core, per workload), medians reported.
    rounds = None
    if rank == 0 and world == 1:
        orc = OracleRounds(oracle)
        gpu_rounds = []
        for _ in range(3):
            n_r = max(3, min(args.steps, 300))
            gpu_rounds.append(time_steps(torch, plan, n_r, stream) / n_r)
            orc.round()
        rounds = dict(orc.summary(), rounds=3, gpu_us_per_token_by_round=[round(u, 2) for u in gpu_rounds],
                      cores_available=orc.cores)

    # Breakdown (not the headline): the other launchers and modes over the same inputs.
    extra = {}
    n_extra = max(3, min(args.steps, 300))
    for name, mode, launcher in [("ordered_persistent", nt.NT_STEP_ORDERED, nt.NT_LAUNCH_PERSISTENT),
                                 ("independent_graph", nt.NT_STEP_INDEPENDENT, nt.NT_LAUNCH_GRAPH),
                                 ("ordered_graph", nt.NT_STEP_ORDERED, nt.NT_LAUNCH_GRAPH),
                                 ("ordered_stream", nt.NT_STEP_ORDERED, nt.NT_LAUNCH_STREAM),
                                 ("chained_persistent", nt.NT_STEP_CHAINED, nt.NT_LAUNCH_PERSISTENT),
                                 ("chained_graph", nt.NT_STEP_CHAINED, nt.NT_LAUNCH_GRAPH)]:
        pl = nt.DecodePlan(L, 1, dp, hd, mode, launcher)
        for _ in range(3):
            pl.nt_decode_step(stream)
        extra[name + "_us_per_token"] = round(time_steps(torch, pl, n_extra, stream) / n_extra, 2)
        if pl.nt_decode_step_status() != nt.NT_OK:
            raise RuntimeError(f"{name}: step reported a timeout")
        pl.close()
    # Components of the step, each timed alone (CUDA events, inputs larger than L2): the ternary
    # weight stream without the output projection, the output projection on its own (the
    # standalone call), and the offline repack of the largest matrix shape.
    peak, peak_kind = measured_peak()
    comp = {}

    def frac(nbytes_, us_):
        gbs = nbytes_ / (us_ * 1e-6) / 1e9
        return {"us": round(us_, 2), "bytes": int(nbytes_), "GBps": round(gbs, 1), "frac": round(gbs / peak, 4)}

    pl = nt.DecodePlan(L, 1, dp, None, nt.NT_STEP_INDEPENDENT, nt.NT_LAUNCH_PERSISTENT)
    for _ in range(3):
        pl.nt_decode_step(stream)
    us_stream = time_steps(torch, pl, n_extra, stream) / n_extra
    if pl.nt_decode_step_status() != nt.NT_OK:
        raise RuntimeError("weight stream: step reported a timeout")
    pl.close()
    stream_bytes = wl.packed_bytes_per_token(n_layers=L) + 4 * sum(p.K for p in projs)
    comp["weight_stream"] = dict(frac(stream_bytes, us_stream), kernel="persist_kernel",
                                 what=f"{L} layers x 7 ternary projections, inputs quantized in the step")
    # the per-call API: one nt_ternary_gemv per projection (inputs already quantized by the step)
    def gemv_calls():
        st = torch.cuda.current_stream()  # the capture stream inside torch.cuda.graph
        for d in dp:
            nt.nt_ternary_gemv(d["w"], nt.NT_LAYOUT_TILED, d["s_w"], d["N"], d["K"], d["q"], d["s_x"], d["y"],
                               stream=st)

    for _ in range(3):
        gemv_calls()
    torch.cuda.synchronize()
    gemv_graph = torch.cuda.CUDAGraph()  # replayed, so the host's per-call cost is not timed
    with torch.cuda.graph(gemv_graph):
        gemv_calls()
    gemv_graph.replay()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(10):
        gemv_graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    del gemv_graph
    comp["gemv_per_call"] = dict(frac(wl.packed_bytes_per_token(n_layers=L), e0.elapsed_time(e1) * 1e3 / 10),
                                 kernel="gemv_tiled_kernel",
                                 what=f"{len(dp)} nt_ternary_gemv calls, batch 1, replayed as a CUDA graph "
                                      "(each call a separate kernel: latency-bound for 1-12 MB matrices)")
    # one large per-call GEMV (268 MB of packed trits, more than L2): the kernel's streaming rate
    bN, bK = 65536, 16384
    r1 = torch.randint(-2 ** 31, 2 ** 31 - 1, (bN * bK // 16,), dtype=torch.int32, device=dev)
    r2 = torch.randint(-2 ** 31, 2 ** 31 - 1, (bN * bK // 16,), dtype=torch.int32, device=dev)
    low = r1 & 0x55555555
    big_plain = low | ((low & r2) << 1)  # fields 00 / 01 / 11 only
    del r1, r2, low
    big_w = torch.empty(nt.nt_repack_size(bN, bK), dtype=torch.uint8, device=dev)
    nt.nt_repack_ternary(big_plain, bN, bK, big_w, stream=stream)
    del big_plain
    big_q = torch.randint(-127, 128, (bK,), dtype=torch.int8, device=dev)
    big_sw = torch.full((bN,), 0.01, dtype=torch.float32, device=dev)
    big_sx = torch.full((1,), 0.02, dtype=torch.float32, device=dev)
    big_y = torch.empty(bN, dtype=torch.float32, device=dev)
    for _ in range(3):
        nt.nt_ternary_gemv(big_w, nt.NT_LAYOUT_TILED, big_sw, bN, bK, big_q, big_sx, big_y, stream=stream)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(10):
        nt.nt_ternary_gemv(big_w, nt.NT_LAYOUT_TILED, big_sw, bN, bK, big_q, big_sx, big_y, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize()
    big_bytes = bN * bK // 4 + 4 * bN + bK + 4 * bN + 4
    comp["gemv_per_call_large"] = dict(frac(big_bytes, e0.elapsed_time(e1) * 1e3 / 10), kernel="gemv_tiled_kernel",
                                       what=f"one nt_ternary_gemv call, {bN}x{bK} trits (268 MB), batch 1")
    # the same matrix for 8 vectors in one nt_ternary_gemm call: with a workspace on the tensor
    # cores, without one on the dp4a kernel
    gB = 8
    g_q = torch.randint(-127, 128, (gB, bK), dtype=torch.int8, device=dev)
    g_sx = torch.full((gB,), 0.02, dtype=torch.float32, device=dev)
    g_y = torch.empty((gB, bN), dtype=torch.float32, device=dev)
    g_ws = torch.zeros(nt.nt_ternary_gemm_workspace_size(bN, bK, gB, nt.NT_LAYOUT_TILED), dtype=torch.uint8, device=dev)
    g_us = {}
    for label, ws in (("tc", g_ws), ("dp4a", None)):
        for _ in range(3):
            nt.nt_ternary_gemm(big_w, nt.NT_LAYOUT_TILED, big_sw, bN, bK, g_q, g_sx, gB, g_y, ws=ws, stream=stream)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(10):
            nt.nt_ternary_gemm(big_w, nt.NT_LAYOUT_TILED, big_sw, bN, bK, g_q, g_sx, gB, g_y, ws=ws, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize()
        g_us[label] = e0.elapsed_time(e1) * 1e3 / 10
    g_bytes = bN * bK // 4 + 4 * bN + gB * bK + 4 * gB * bN + 4 * gB
    comp["gemm_per_call_large_b8"] = dict(frac(g_bytes, g_us["tc"]), kernel="gemv_tc8_kernel",
                                          dp4a_us=round(g_us["dp4a"], 2),
                                          what=f"one nt_ternary_gemm call, {bN}x{bK} trits, batch {gB}, with a "
                                               "workspace (tensor cores); dp4a_us: the same call without one")
    del big_w, big_q, big_sw, big_sx, big_y, g_q, g_sx, g_y, g_ws
    hws = torch.zeros(nt.nt_int8_logits_workspace_size(head.V, head.K, 1), dtype=torch.uint8, device=dev)
    hq_o, hs_o = oracle.quantize(head.x)
    am_oracle = int(oracle.logits_argmax(head.T, head.s_T, head.V, head.K, hq_o, hs_o)[1][0])
    nt.nt_quantize_act(hd["x"], hd["q"], hd["sx"], stream)

    def head_call():
        nt.nt_int8_logits_argmax(hd["T"], hd["s"], head.V, head.K, hd["q"], hd["sx"], 1, hd["logits"],
                                 hd["argmax"], hws, stream)

    for _ in range(3):
        head_call()
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(n_extra):
        head_call()
    e1.record(stream)
    torch.cuda.synchronize()
    if nt.nt_workspace_status(hws) != nt.NT_OK:
        raise RuntimeError("standalone output projection: a bounded wait ran out")
    if int(hd["argmax"].item()) != am_oracle:
        raise RuntimeError("standalone output projection: arg-max differs from the oracle's")
    comp["lm_head"] = dict(frac(wl.head_bytes(B=1), e0.elapsed_time(e1) * 1e3 / n_extra),
                           kernel="persist_kernel (implicit schedule, programmatic dependent launch)",
                           what=f"int8 table {head.V}x{head.K}, fp32 logits, greedy arg-max")
    comp["single_gemv_config1"] = time_single_gemv(torch, nt, oracle, dev, stream, peak)
    rN, rK = wl.DECODER_8B["gate"]
    r1 = torch.randint(-2 ** 31, 2 ** 31 - 1, (rN * rK // 16,), dtype=torch.int32, device=dev)
    r2 = torch.randint(-2 ** 31, 2 ** 31 - 1, (rN * rK // 16,), dtype=torch.int32, device=dev)
    low = r1 & 0x55555555
    w_plain = low | ((low & r2) << 1)  # fields 00 / 01 / 11 only (no invalid 10)
    del r1, r2, low
    w_t = torch.empty(nt.nt_repack_size(rN, rK), dtype=torch.uint8, device=dev)
    for _ in range(3):
        nt.nt_repack_ternary(w_plain, rN, rK, w_t, stream=stream)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(20):
        nt.nt_repack_ternary(w_plain, rN, rK, w_t, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize()
    comp["repack"] = dict(frac(2 * rN * rK // 4, e0.elapsed_time(e1) * 1e3 / 20), kernel="repack_kernel",
                          what=f"plain -> tiled, {rN}x{rK} trits (read + write)")
    del w_plain, w_t, hws

    plan.nt_decode_step(stream)  # chained plans rewrote the codes: requantize the supplied inputs
    torch.cuda.synchronize()
    parity_after = parity_gate(oracle, projs, head, dp, hd, layers=(L // 2,)) if rank == 0 else "pass"

    nbytes = step_bytes(n_layers=L)
    achieved = nbytes / (per_step_us * 1e-6) / 1e9
    cpu = cpu_baseline(oracle) if (rank == 0 and world == 1) else None
    if cpu is not None and rounds is not None:
        cpu["per_config_interleaved"] = rounds
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "us/token",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(per_step_us / 1e3, 5),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "int8 x ternary -> int32, fp32 epilogue",
        "data": "synthetic (seeded SplitMix64; workload shapes and value mixes)",
        "config": {"workload": WORKLOAD if L == wl.DECODER_8B_LAYERS else
                   WORKLOAD.replace("36 layers", f"{L} of 36 layers (profiling case)"),
                   "batch": 1, "mode": "independent",
                   "launcher": "persistent", "bytes_per_step": nbytes,
                   "l2": "inputs larger than L2 (2.37 GB streamed per step vs 129 MB L2)",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": read_traffic(),
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured" else peak_kind,
                     "kernel": "persist_kernel", "frac_of_8TBps_spec": round(achieved / 8000.0, 4)},
        "cpu_baseline": cpu,
        "e2e": {"value": round(e2e_serial_us, 2), "unit": "us/token", "mode": "serial",
                "h2d_bytes_per_step": int(x_all.numel() * 4), "d2h_bytes_per_step": 4},
        "e2e_graph": {"value": round(e2e_graph_us, 2), "unit": "us/token", "mode": "serial",
                      "h2d_bytes_per_step": int(x_all.numel() * 4), "d2h_bytes_per_step": 4,
                      "what": "copy in, step and token out recorded once into a CUDA graph, replayed per token"},
        "e2e_zero_copy": {"value": round(e2e_zero_copy_us, 2), "unit": "us/token", "mode": "serial",
                          "h2d_bytes_per_step": int(x_all.numel() * 4), "d2h_bytes_per_step": 4,
                          "what": "no copy call: the step reads its inputs from pinned host memory over the host link"},
        "e2e_pipelined": {"value": round(e2e_us, 2), "unit": "us/token",
                          "h2d_bytes_per_step": int(x_all.numel() * 4), "d2h_bytes_per_step": 4,
                          "what": "step i+1's input copy overlaps step i (inputs supplied, not produced)"},
        "step_distribution": dict(dist_steps, unit="us", what="single steps, one event between every two, "
                                  "after the timed region (this rank)"),
        "gpu_launches": args.steps,
        "clocks": clk,
        "parity": parity if parity_after == "pass" else f"after timing: {parity_after}",
        "breakdown": extra,
        "components": comp,
    }
    plan.close()
    if rank == 0:
        print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------------------
# Reference arm: the CPU oracle, as it stands, on a bounded sample per step
# ---------------------------------------------------------------------------------------

def run_reference(args):
    import oracle

    oracle.build()
    layer = [wl.projection(wl.WL_DECODE, 0, i, *wl.DECODER_8B[n]) for i, n in enumerate(wl.PROJ_NAMES)]
    hv = 2048
    head = wl.head(V=hv)
    trits_layer = sum(p.N * p.K for p in layer)

    def sample(rows_frac):
        # rows_frac of every projection of one layer + the same fraction of the table slice
        t0 = time.perf_counter()
        for p in layer:
            n = max(4, int(p.N * rows_frac))
            q, s = oracle.quantize(p.x)
            oracle.gemv(p.w_plain[:n], p.s_w[:n], n, p.K, q[0], s)
        hn = max(1, int(hv * rows_frac))
        q, s = oracle.quantize(head.x)
        oracle.logits_argmax(head.T[:hn], head.s_T[:hn], hn, head.K, q, s)
        return time.perf_counter() - t0

    t1 = sample(0.05)  # calibration
    budget = 90.0
    per_step = budget / max(1, args.steps + args.warmup)
    frac = min(1.0, max(0.002, 0.05 * per_step / max(t1, 1e-6)))
    for _ in range(args.warmup):
        sample(frac)
    total = 0.0
    for _ in range(args.steps):
        total += sample(frac)
    sampled_trits = sum(max(4, int(p.N * frac)) * p.K for p in layer)
    hn = max(1, int(hv * frac))
    # scale: layer part to 36 layers, table part to 151,936 rows (by MAC count)
    macs_sample = sampled_trits + hn * head.K
    macs_token = trits_layer * wl.DECODER_8B_LAYERS + wl.HEAD_V * wl.HEAD_K
    us = total / args.steps * macs_token / macs_sample * 1e6
    line = {
        "impl": "reference", "metric": METRIC, "value": round(us, 1), "unit": "us/token",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total / args.steps * 1e3, 3), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "int64 sums, fp32 epilogue",
        "data": "synthetic (seeded SplitMix64; workload shapes and value mixes)",
        "config": {"workload": WORKLOAD, "batch": 1},
        "cpu_baseline": {"value": round(us, 1), "unit": "us/token", "cores": oracle.threads(),
                         "kind": "oracle",
                         "sample": (f"per step: {frac:.4f} of the rows of one decoder layer's 7 "
                                    f"projections + {hn} output-table rows; scaled to one "
                                    "token by multiply-accumulate count")},
        "e2e": {"value": round(us, 1), "unit": "us/token", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------------------
# Batched sweep (not the headline line): the same 36-layer projection set and output table
# with B independent activation vectors per step
# ---------------------------------------------------------------------------------------

def run_sweep(args):
    import torch

    import oracle
    from packed_weight_gemv_gb300 import nt

    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    nt.nt_device_check()
    L = args.layers
    projs, head, dp, hd, _ = build_inputs(torch, nt, dev, L)
    stream = torch.cuda.current_stream()
    peak, peak_kind = measured_peak()
    for B in args.batches:
        dpB, hosts = [], []
        for p, d in zip(projs, dp):
            layer, name = p.name.split(".")
            x = wl.projection_x(wl.WL_DECODE, int(layer[1:]), wl.PROJ_NAMES.index(name), p.K, B)
            hosts.append(x)
            dpB.append(dict(N=p.N, K=p.K, w=d["w"], s_w=d["s_w"], x=torch.from_numpy(x).to(dev),
                            q=torch.empty((B, p.K), dtype=torch.int8, device=dev),
                            s_x=torch.empty(B, dtype=torch.float32, device=dev),
                            y=torch.empty((B, p.N), dtype=torch.float32, device=dev)))
        hx = wl.head_x(B=B)
        hdB = dict(T=hd["T"], s=hd["s"], V=head.V, K=head.K, x=torch.from_numpy(hx).to(dev),
                   q=torch.empty((B, head.K), dtype=torch.int8, device=dev),
                   sx=torch.empty(B, dtype=torch.float32, device=dev),
                   logits=torch.empty((B, head.V), dtype=torch.float32, device=dev),
                   argmax=torch.empty(B, dtype=torch.int32, device=dev))
        res = {}
        for lname, launcher in (("persistent", nt.NT_LAUNCH_PERSISTENT), ("graph", nt.NT_LAUNCH_GRAPH)):
            if lname not in args.launchers:
                continue
            for d in dpB:
                d["y"].zero_()
            hdB["logits"].zero_()
            plan = nt.DecodePlan(L, B, dpB, hdB, nt.NT_STEP_INDEPENDENT, launcher)
            for _ in range(args.warmup):
                plan.nt_decode_step(stream)
            torch.cuda.synchronize()
            parity = "pass"
            for i in range(len(wl.PROJ_NAMES)):  # every projection of layer 0
                p = projs[i]
                full = wl.projection(wl.WL_DECODE, 0, i, p.N, p.K)
                q, s = oracle.quantize(hosts[i])
                _, y, _ = oracle.gemm(full.w_plain, full.s_w, p.N, p.K, q, s)
                got = dpB[i]["y"].cpu().numpy().astype(np.float64)
                if np.any(np.abs(got - y) > 1e-6 * np.abs(y.astype(np.float64))):
                    parity = f"{p.name} differs"
            q, s = oracle.quantize(hx)
            logits, am, _ = oracle.logits_argmax(head.T, head.s_T, head.V, head.K, q, s)
            if not np.array_equal(hdB["argmax"].cpu().numpy(), am):
                parity = "arg-max differs"
            got = hdB["logits"].cpu().numpy().astype(np.float64)
            if np.any(np.abs(got - logits) > 1e-6 * np.abs(logits.astype(np.float64))):
                parity = "logits differ"
            steps = max(3, min(args.steps, 500))
            us = time_steps(torch, plan, steps, stream) / steps
            if launcher == nt.NT_LAUNCH_PERSISTENT and plan.nt_decode_step_status() != nt.NT_OK:
                parity = "timeout reported"
            nbytes = step_bytes(B=B, n_layers=L)
            gbs = nbytes / (us * 1e-6) / 1e9
            res[lname] = {"us_per_step": round(us, 2), "us_per_token": round(us / B, 2),
                          "achieved_GBps": round(gbs, 1), "frac": round(gbs / peak, 4), "parity": parity}
            plan.close()
        best = min(res, key=lambda k: res[k]["us_per_step"])
        print(json.dumps({"metric": "batched decode sweep", "batch": B, "steps": steps,
                          **res[best], "launcher": best, "peak_GBps": peak, "peak_source": peak_kind,
                          "bytes_per_step": nbytes, "by_launcher": res,
                          "projections": "dp4a (persistent); f16 mma.sync tensor cores for projections and output projection (graph, B >= 2)"}), flush=True)


# ---------------------------------------------------------------------------------------
# Speculative verify pass (not the headline line): B positions (the last emitted token and
# B - 1 drafts) gathered from the input table into layer 0's q, k and v, every projection,
# the output projection and the acceptance of the longest agreeing draft prefix, in one step
# ---------------------------------------------------------------------------------------

def run_verify(args):
    import torch

    import oracle
    from packed_weight_gemv_gb300 import nt

    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    nt.nt_device_check()
    L = args.layers
    projs, head, dp, hd, _ = build_inputs(torch, nt, dev, L)
    emb = wl.embedding(B=8)
    eT, es = torch.from_numpy(emb.T).to(dev), torch.from_numpy(emb.s_T).to(dev)
    stream = torch.cuda.current_stream()
    for B in (2, 4, 8):
        tokens = emb.tokens[:B].copy()
        ex = torch.empty((B, emb.K), dtype=torch.float32, device=dev)
        dpB, hosts = [], []
        for i, (p, d) in enumerate(zip(projs, dp)):
            layer, name = p.name.split(".")
            x = wl.projection_x(wl.WL_DECODE, int(layer[1:]), wl.PROJ_NAMES.index(name), p.K, B)
            hosts.append(x)
            dpB.append(dict(N=p.N, K=p.K, w=d["w"], s_w=d["s_w"],
                            x=ex if i < 3 else torch.from_numpy(x).to(dev),
                            q=torch.empty((B, p.K), dtype=torch.int8, device=dev),
                            s_x=torch.empty(B, dtype=torch.float32, device=dev),
                            y=torch.empty((B, p.N), dtype=torch.float32, device=dev)))
        hx = wl.head_x(B=B)
        hdB = dict(T=hd["T"], s=hd["s"], V=head.V, K=head.K, x=torch.from_numpy(hx).to(dev),
                   q=torch.empty((B, head.K), dtype=torch.int8, device=dev),
                   sx=torch.empty(B, dtype=torch.float32, device=dev),
                   logits=torch.empty((B, head.V), dtype=torch.float32, device=dev),
                   argmax=torch.empty(B, dtype=torch.int32, device=dev))
        # drafts that agree with the greedy tokens at every position (a fully accepted pass)
        q, s = oracle.quantize(hx)
        _, greedy, _ = oracle.logits_argmax(head.T, head.s_T, head.V, head.K, q, s)
        greedy = np.asarray(greedy, dtype=np.int32)
        draft = wl.draft_tokens(greedy, B - 1, head.V)
        emit = torch.empty(B, dtype=torch.int32, device=dev)
        n_emit = torch.empty(1, dtype=torch.int32, device=dev)
        embed = dict(T=eT, s=es, V=emb.V, K=emb.K, tokens=torch.from_numpy(tokens).to(dev), x=ex)
        verify = dict(draft=torch.from_numpy(draft).to(dev), emit=emit, n=n_emit)
        res = {}
        for lname, launcher in (("persistent", nt.NT_LAUNCH_PERSISTENT), ("graph", nt.NT_LAUNCH_GRAPH)):
            plan = nt.DecodePlan(L, B, dpB, hdB, nt.NT_STEP_INDEPENDENT, launcher, embed=embed, verify=verify)
            base = nt.DecodePlan(L, B, dpB, hdB, nt.NT_STEP_INDEPENDENT, launcher)
            for _ in range(args.warmup):
                base.nt_decode_step(stream)
                plan.nt_decode_step(stream)
            torch.cuda.synchronize()
            parity = "pass"
            xe, _ = oracle.embed_rows(emb.T, emb.s_T, emb.V, emb.K, tokens)
            if not np.array_equal(ex.cpu().numpy().view(np.uint32), xe.view(np.uint32)):
                parity = "gathered rows differ"
            for i in range(len(wl.PROJ_NAMES)):  # every projection of layer 0
                p = projs[i]
                full = wl.projection(wl.WL_DECODE, 0, i, p.N, p.K)
                qi, si = oracle.quantize(xe if i < 3 else hosts[i])
                _, y, _ = oracle.gemm(full.w_plain, full.s_w, p.N, p.K, qi, si)
                got = dpB[i]["y"].cpu().numpy().astype(np.float64)
                if np.any(np.abs(got - y) > 1e-6 * np.abs(y.astype(np.float64))):
                    parity = f"{p.name} differs"
            if not np.array_equal(hdB["argmax"].cpu().numpy(), greedy):
                parity = "arg-max differs"
            want = oracle.verify_accept(draft, greedy)
            if int(n_emit.item()) != want.size or not np.array_equal(emit.cpu().numpy()[:want.size], want):
                parity = "emitted tokens differ"
            steps = max(3, min(args.steps, 300))
            us_base = time_steps(torch, base, steps, stream) / steps
            us = time_steps(torch, plan, steps, stream) / steps
            if plan.nt_decode_step_status() != nt.NT_OK or base.nt_decode_step_status() != nt.NT_OK:
                parity = "timeout reported"
            res[lname] = {"us_per_pass": round(us, 2), "us_per_pass_without_gather_accept": round(us_base, 2),
                          "us_per_token_if_all_accepted": round(us / B, 2), "tokens_emitted": int(n_emit.item()),
                          "parity": parity}
            plan.close()
            base.close()
        best = min(res, key=lambda k: res[k]["us_per_pass"])
        print(json.dumps({"metric": "speculative verify pass", "positions": B, "steps": steps, **res[best],
                          "launcher": best, "by_launcher": res,
                          "gather_bytes": B * (emb.K + 4 + 4 * emb.K)}), flush=True)


# ---------------------------------------------------------------------------------------
# Attention over the key-value cache (not the headline line): the 36 layers' grouped-query
# attention of one new position at several context lengths
# ---------------------------------------------------------------------------------------

def run_attention(args):
    import torch

    from oracle import layer_ops as lo
    from packed_weight_gemv_gb300 import nt

    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    nt.nt_device_check()
    L, Hq, Hkv, D = args.layers, 32, 8, 128
    peak, peak_kind = measured_peak()
    stream = torch.cuda.current_stream()
    for T in (args.contexts or (4096, 16384, 32768)):
        # one cache per layer, bf16 N(0,1) keys and values (the layers' contents differ only by
        # seed; the attention's cost does not depend on the values)
        kb = wl.bf16_normal(Hkv * T * D, 0, wl.tag(wl.WL_ATTN, T, 1, 0))
        vb = wl.bf16_normal(Hkv * T * D, 0, wl.tag(wl.WL_ATTN, T, 2, 0))
        kc = [torch.from_numpy(kb.view(np.int16)).to(dev) for _ in range(L)]
        vc = [torch.from_numpy(vb.view(np.int16)).to(dev) for _ in range(L)]
        q = wl.normal(L * Hq * D, 0, wl.tag(wl.WL_ATTN, T, 3, 0)).reshape(L, 1, Hq, D)
        qd = torch.from_numpy(q).to(dev)
        out = torch.empty((L, 1, Hq, D), device=dev)
        ws = torch.zeros(nt.nt_attention_workspace_size(1, Hq, Hkv, T), dtype=torch.uint8, device=dev)

        def one_token():
            for l in range(L):
                nt.nt_attention_decode(qd[l], kc[l], vc[l], 1, Hq, Hkv, D, T, T, out[l], ws)

        for _ in range(max(3, args.warmup)):
            one_token()
        torch.cuda.synchronize()
        want = lo.attention_decode(q[0], lo.from_bf16_bits(kb.reshape(Hkv, T, D)),
                                   lo.from_bf16_bits(vb.reshape(Hkv, T, D)), T)
        vmax = float(np.abs(lo.from_bf16_bits(vb)).max())
        err = float(np.abs(out[0].cpu().numpy().astype(np.float64) - want).max())
        parity = "pass" if err <= 3e-5 * vmax else f"max error {err:.3g}"
        steps = max(3, min(args.steps, 200))
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            one_token()
        graph.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            graph.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / steps
        nbytes = L * 2 * Hkv * T * D * 2
        gbs = nbytes / (us * 1e-6) / 1e9
        print(json.dumps({"metric": "attention over the key-value cache (36 layers, 1 position)",
                          "context": T, "steps": steps, "us_per_token": round(us, 2),
                          "cache_bytes_per_token": nbytes, "achieved_GBps": round(gbs, 1),
                          "peak_GBps": peak, "frac": round(gbs / peak, 4), "peak_source": peak_kind,
                          "launches_per_token": L, "parity": parity}), flush=True)
        del graph, kc, vc, qd, out, ws
        torch.cuda.empty_cache()


# ---------------------------------------------------------------------------------------
# Chained decode with the attention side (not the headline line): every stage quantizes the
# previous one's output; norms, rotary embedding, cache append, attention, SiLU gate
# ---------------------------------------------------------------------------------------

def run_layer_attention(args):
    import torch

    import oracle
    from oracle import layer_ops as lo
    from packed_weight_gemv_gb300 import nt

    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    nt.nt_device_check()
    L = args.layers
    projs, head, dp, hd, _ = build_inputs(torch, nt, dev, L)
    Hkv, d = 8, 4096
    stream = torch.cuda.current_stream()
    gam = [torch.from_numpy(wl.scales(d, 1.0, 0, wl.tag(wl.WL_ATTN, l, 4, 0))).to(dev) for l in range(2 * L + 1)]
    for T in (args.contexts or (4096, 16384)):
        pos = T - 1
        kb = wl.bf16_normal(Hkv * T * 128, 0, wl.tag(wl.WL_ATTN, T, 1, 0)).reshape(Hkv, T, 128)
        vb = wl.bf16_normal(Hkv * T * 128, 0, wl.tag(wl.WL_ATTN, T, 2, 0)).reshape(Hkv, T, 128)
        kc = [torch.from_numpy(kb.view(np.int16)).to(dev) for _ in range(L)]
        vc = [torch.from_numpy(vb.view(np.int16)).to(dev) for _ in range(L)]
        att = dict(k_cache=kc, v_cache=vc, t_stride=T, pos=pos, norm_attn=gam[:L], norm_ffn=gam[L:2 * L],
                   norm_final=gam[2 * L])
        # parity first: the first two layers as their own chained plan against the oracle
        L2 = min(2, L)
        layers = []
        for l in range(L2):
            mats = []
            for i in range(7):
                full = wl.projection(wl.WL_DECODE, l, i, projs[7 * l + i].N, projs[7 * l + i].K)
                mats.append((full.w_plain, full.s_w, full.N, full.K))
            layers.append(mats)
        g_np = [g.cpu().numpy() for g in gam]
        kf = [lo.from_bf16_bits(kb).copy() for _ in range(L2)]
        vf = [lo.from_bf16_bits(vb).copy() for _ in range(L2)]
        want = oracle.decode_chained_attention(layers, wl.projection_x(wl.WL_DECODE, 0, 0, d, 1), (head.T, head.s_T, head.V, head.K),
                                               kf, vf, pos, g_np[:L2], g_np[L:L + L2], g_np[2 * L])
        line = {"metric": "chained decode with attention", "context": T, "layers": L}
        kv = L * 2 * Hkv * T * 128 * 2
        arms = (("persistent", nt.NT_LAUNCH_PERSISTENT, 3 * L + 1), ("graph", nt.NT_LAUNCH_GRAPH, L * 12 + 2))
        for name, launcher, launches in [a for a in arms if a[0] in args.launchers]:
            p2 = nt.DecodePlan(L2, 1, dp[:7 * L2], hd, nt.NT_STEP_CHAINED, launcher,
                               attention=dict(att, k_cache=kc[:L2], v_cache=vc[:L2], norm_attn=gam[:L2],
                                              norm_ffn=gam[L:L + L2]))
            p2.nt_decode_step(stream)
            torch.cuda.synchronize()
            parity = "pass"
            for i in range(7 * L2):
                y = dp[i]["y"].cpu().numpy().reshape(1, -1).astype(np.float64)
                if np.abs(y - want["y"][i]).max() > 2e-3 * np.abs(want["y"][i]).max():
                    parity = f"{projs[i].name} differs"
            p2.close()
            # the caches' row at pos is rewritten by every step with the same values
            plan = nt.DecodePlan(L, 1, dp, hd, nt.NT_STEP_CHAINED, launcher, attention=att)
            for _ in range(max(3, args.warmup)):
                plan.nt_decode_step(stream)
            steps = max(3, min(args.steps, 100))
            us = time_steps(torch, plan, steps, stream) / steps
            line[name] = {"us_per_token": round(us, 2), "launches_per_token": launches,
                          "GBps_weights_plus_cache": round((step_bytes(n_layers=L) + kv) / (us * 1e-6) / 1e9, 1),
                          "parity_first_two_layers": parity}
            plan.close()
        line.update(steps=steps, weight_bytes=step_bytes(n_layers=L), cache_bytes=kv)
        print(json.dumps(line), flush=True)
        del kc, vc
        torch.cuda.empty_cache()


# ---------------------------------------------------------------------------------------
# Prefill (not the headline line): the 28-layer small model at M = 2048 and 8192 tokens on
# the tensor-core GEMM
# ---------------------------------------------------------------------------------------

def run_prefill(args):
    import torch

    import oracle
    from packed_weight_gemv_gb300 import nt

    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    nt.nt_device_check()
    shapes, L = wl.SMALL_28, wl.SMALL_28_LAYERS
    mats = []
    for layer in range(L):
        for pi, name in enumerate(wl.PROJ_NAMES):
            N, K = shapes[name]
            w = wl.ternary_plain(N, K, 0, wl.tag(wl.WL_PREFILL, layer, pi, wl.ROLE_TRITS))
            s_w = wl.scales(N, np.sqrt(K), 0, wl.tag(wl.WL_PREFILL, layer, pi, wl.ROLE_ROW_SCALE))
            wt = torch.empty(nt.nt_repack_size(N, K), dtype=torch.uint8, device=dev)
            nt.nt_repack_ternary(torch.from_numpy(w.view(np.int32)).to(dev), N, K, wt)
            mats.append(dict(name=f"L{layer}.{name}", N=N, K=K, w=wt, s_w=torch.from_numpy(s_w).to(dev),
                             host_w=w if layer == 0 else None, host_sw=s_w if layer == 0 else None))
    macs = sum(m["N"] * m["K"] for m in mats)
    peak = 1872.8
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peak = float(json.load(f)["bf16_tflops"])
    except (OSError, KeyError, ValueError):
        pass
    stream = torch.cuda.current_stream()
    for M in (args.tokens or wl.PREFILL_TOKENS):
        # One fp32 input per distinct K (shared by the layers: values do not change the work),
        # quantized per token inside the timed pass, then every projection's GEMM.
        xs = {K: torch.from_numpy(wl.normal(M * K, 0, wl.tag(wl.WL_PREFILL, 99, K, wl.ROLE_X))
                                  .reshape(M, K)).to(dev) for K in sorted({m["K"] for m in mats})}
        qs = {K: torch.empty((M, K), dtype=torch.int8, device=dev) for K in xs}
        ss = {K: torch.empty(M, dtype=torch.float32, device=dev) for K in xs}
        ys = [torch.empty((M, m["N"]), dtype=torch.float32, device=dev) for m in mats]

        # q/k/v and gate/up read one input each: one call per group (one activation conversion,
        # one tile set); o and down alone
        groups = []
        for layer in range(L):
            b = 7 * layer
            groups += [[b, b + 1, b + 2], [b + 3], [b + 4, b + 5], [b + 6]]
        wsg = torch.empty(max(nt.nt_ternary_gemm_multi_workspace_size([mats[i]["N"] for i in g], mats[g[0]]["K"], M)
                              for g in groups[:4]), dtype=torch.uint8, device=dev)

        def one_pass():  # on the current stream (the capture stream while a graph records)
            for K in xs:
                nt.nt_quantize_act(xs[K], qs[K], ss[K])
            for g in groups:
                K = mats[g[0]]["K"]
                nt.nt_ternary_gemm_multi([mats[i]["w"] for i in g], [mats[i]["s_w"] for i in g],
                                         [mats[i]["N"] for i in g], K, qs[K], ss[K], M, [ys[i] for i in g], None, wsg)

        for _ in range(max(1, args.warmup)):
            one_pass()
        torch.cuda.synchronize()
        # parity: the first layer's projections on 64 sampled tokens
        rows = np.linspace(0, M - 1, 64).astype(np.int64)
        parity = "pass"
        for K in xs:
            xq, xs_ = oracle.quantize(xs[K].cpu().numpy()[rows])
            if not np.array_equal(qs[K].cpu().numpy()[rows], xq):
                parity = "int8 codes differ"
        for m, y in zip(mats[:7], ys[:7]):
            xq, xs_ = oracle.quantize(xs[m["K"]].cpu().numpy()[rows])
            _, yo, _ = oracle.gemm(m["host_w"], m["host_sw"], m["N"], m["K"], xq, xs_)
            got = y.cpu().numpy()[rows].astype(np.float64)
            if np.any(np.abs(got - yo) > 1e-6 * np.abs(yo.astype(np.float64))):
                parity = f"{m['name']} differs"
        n_pass = max(2, min(args.steps, 20))
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for _ in range(n_pass):
            one_pass()
        ev1.record(stream)
        torch.cuda.synchronize()
        ms_eager = ev0.elapsed_time(ev1) / n_pass
        # The same calls captured once in a CUDA graph and replayed (no host work per call).
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            one_pass()
        graph.replay()
        torch.cuda.synchronize()
        ev0.record(stream)
        for _ in range(n_pass):
            graph.replay()
        ev1.record(stream)
        torch.cuda.synchronize()
        ms = ev0.elapsed_time(ev1) / n_pass
        tflops = 2.0 * M * macs / (ms * 1e-3) / 1e12
        out_bytes = 4 * M * sum(m["N"] for m in mats)
        print(json.dumps({"metric": "prefill ternary GEMM (28-layer small model)", "tokens": M,
                          "passes": n_pass, "ms_per_pass": round(ms, 3),
                          "ms_per_pass_eager": round(ms_eager, 3),
                          "tflops": round(tflops, 1), "peak_tflops_bf16": peak,
                          "frac_of_bf16_peak": round(tflops / peak, 4),
                          "output_GBps": round(out_bytes / (ms * 1e-3) / 1e9, 1),
                          "parity": parity}), flush=True)
        del graph
        del xs, qs, ss, ys, wsg
        torch.cuda.empty_cache()


# ---------------------------------------------------------------------------------------
# Step timeline (not the headline line): where the time between stages of the ordered and
# chained persistent steps goes, from the plan's per-CTA %globaltimer stamps
# ---------------------------------------------------------------------------------------

def run_timeline(args):
    import torch

    from packed_weight_gemv_gb300 import nt

    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    nt.nt_device_check()
    L = args.layers
    projs, head, dp, hd, _ = build_inputs(torch, nt, dev, L)
    stream = torch.cuda.current_stream()
    kinds = {1: "o", 2: "gate_up", 3: "down", 0: "qkv"}
    for mode, name in ((nt.NT_STEP_ORDERED, "ordered"), (nt.NT_STEP_CHAINED, "chained")):
        plan = nt.DecodePlan(L, 1, dp, hd, mode, nt.NT_LAUNCH_PERSISTENT)
        G, S = plan.nt_decode_plan_trace_layout()
        n_pre = S - 4 * L  # barriers before the first stage boundary (input quantization)
        steps = max(3, min(args.steps, 200))
        us = time_steps(torch, plan, steps, stream) / steps
        tr = torch.zeros(G * (S + 1) * 4, dtype=torch.int64, device=dev)
        plan.nt_decode_plan_set_trace(tr)
        for _ in range(3):
            plan.nt_decode_step(stream)
        torch.cuda.synchronize()
        t = tr.cpu().numpy().reshape(G, S + 1, 4).astype(np.int64)
        t = (t - t[:, 0, 0].min()) / 1000.0
        acc = {}
        for b in range(1, S + 1):
            done, pas, act = t[:, b, 0], t[:, b, 1], t[:, b, 2]
            nxt = t[:, b + 1, 0] if b < S else t[:, 0, 1]
            i = b - n_pre
            k = "quantize" if i <= 0 else ("head" if i == 4 * L else kinds[i % 4])
            acc.setdefault(k, []).append((done.max() - np.median(done), pas.min() - done.max(),
                                          np.median(act - pas), np.median(nxt) - np.median(act)))
        by = {k: dict(zip(("tail_us", "barrier_release_us", "stage_input_us", "stage_work_us"),
                          [round(float(x), 2) for x in np.mean(v, axis=0)]), count=len(v)) for k, v in acc.items()}
        print(json.dumps({"metric": "step timeline", "mode": name, "layers": L, "us_per_token": round(us, 2),
                          "barriers": S, "trace_span_us": round(float(t[:, 0, 1].max()), 1), "before_stage": by,
                          "what": ("per boundary, averaged per stage kind: tail = last CTA done - median CTA done; "
                                   "barrier_release = first CTA past the barrier - last CTA done; stage_input = "
                                   "median (activations ready - barrier passed; chained: the stage input quantized "
                                   "from L2); stage_work = median next done - median activations ready")}),
              flush=True)
        plan.nt_decode_plan_set_trace(None)
        plan.close()


# ---------------------------------------------------------------------------------------
# One prefill-shaped GEMM (not the headline line): a single nt_ternary_gemm call of M tokens
# against one N x K ternary matrix on the tensor cores -- the case the prefill kernel's
# profiles are taken on
# ---------------------------------------------------------------------------------------

def run_gemm(args):
    import torch

    import oracle
    from packed_weight_gemv_gb300 import nt

    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    nt.nt_device_check()
    M, N, K = args.gemm
    w = wl.ternary_plain(N, K, 0, wl.tag(wl.WL_PREFILL, 98, 0, wl.ROLE_TRITS))
    s_w = wl.scales(N, np.sqrt(K), 0, wl.tag(wl.WL_PREFILL, 98, 0, wl.ROLE_ROW_SCALE))
    x = wl.normal(M * K, 0, wl.tag(wl.WL_PREFILL, 98, K, wl.ROLE_X)).reshape(M, K)
    q, s = oracle.quantize(x)
    wt = torch.empty(nt.nt_repack_size(N, K), dtype=torch.uint8, device=dev)
    nt.nt_repack_ternary(torch.from_numpy(w.view(np.int32)).to(dev), N, K, wt)
    swd, qd, sd = torch.from_numpy(s_w).to(dev), torch.from_numpy(q).to(dev), torch.from_numpy(s).to(dev)
    y = torch.empty((M, N), dtype=torch.float32, device=dev)
    ws = torch.zeros(nt.nt_ternary_gemm_workspace_size(N, K, M, nt.NT_LAYOUT_TILED), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    for _ in range(max(3, args.warmup)):
        nt.nt_ternary_gemm(wt, nt.NT_LAYOUT_TILED, swd, N, K, qd, sd, M, y, ws=ws, stream=stream)
    torch.cuda.synchronize()
    rows = np.linspace(0, M - 1, 16).astype(np.int64)
    _, yo, _ = oracle.gemm(w, s_w, N, K, q[rows], s[rows])
    got = y.cpu().numpy()[rows].astype(np.float64)
    parity = "pass" if np.all(np.abs(got - yo) <= 1e-6 * np.abs(yo.astype(np.float64))) else "differs"
    steps = max(3, min(args.steps, 200))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        nt.nt_ternary_gemm(wt, nt.NT_LAYOUT_TILED, swd, N, K, qd, sd, M, y, ws=ws, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / steps
    if nt.nt_workspace_status(ws) != nt.NT_OK:
        parity = "timeout reported"
    print(json.dumps({"metric": "prefill ternary GEMM, one call", "M": M, "N": N, "K": K, "calls": steps,
                      "us_per_call": round(us, 2), "tflops": round(2.0 * M * N * K / (us * 1e-6) / 1e12, 1),
                      "kernels": "act_f16_kernel + gemm_tc_kernel", "parity_16_tokens": parity}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--layers", type=int, default=wl.DECODER_8B_LAYERS,
                    help="decoder layers in the step (36 = the 8B-shaped workload; fewer only "
                         "for small profiling captures)")
    ap.add_argument("--sweep", action="store_true",
                    help="batched sweep B = 1, 2, 4, 8, 16 (one JSON line per batch)")
    ap.add_argument("--batches", type=lambda v: [int(x) for x in v.split(",")], default=[1, 2, 4, 8, 16],
                    help="--sweep: batch sizes to run")
    ap.add_argument("--verify", action="store_true",
                    help="speculative verify passes of 2, 4 and 8 positions (gather + step + acceptance)")
    ap.add_argument("--attention", action="store_true",
                    help="attention over the key-value cache at 4K/16K/32K context (36 layers)")
    ap.add_argument("--layer-attention", action="store_true",
                    help="chained decode with norms, rotary embedding and attention at 4K/16K context")
    ap.add_argument("--tokens", type=lambda v: [int(x) for x in v.split(",")], default=None,
                    help="--prefill: token counts to run (default 2048,8192)")
    ap.add_argument("--contexts", type=lambda v: [int(x) for x in v.split(",")], default=None,
                    help="--attention / --layer-attention: context lengths to run")
    ap.add_argument("--launchers", type=lambda v: v.split(","), default=["persistent", "graph"],
                    help="--layer-attention, --sweep: launchers to time (persistent,graph)")
    ap.add_argument("--prefill", action="store_true",
                    help="prefill GEMMs of the 28-layer small model at 2048 and 8192 tokens")
    ap.add_argument("--timeline", action="store_true",
                    help="per-boundary step timeline of the ordered and chained persistent steps")
    ap.add_argument("--gemm", type=lambda v: [int(x) for x in v.split(",")], default=None,
                    help="one prefill-shaped GEMM M,N,K (the profiling case of the prefill kernel)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            run_reference(args)
        return
    if args.sweep:
        run_sweep(args)
        return
    if args.verify:
        run_verify(args)
        return
    if args.attention:
        run_attention(args)
        return
    if args.layer_attention:
        run_layer_attention(args)
        return
    if args.prefill:
        run_prefill(args)
        return
    if args.gemm:
        run_gemm(args)
        return
    if args.timeline:
        run_timeline(args)
        return
    if world > 1:
        import torch

        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        torch.distributed.init_process_group("nccl")
    run_ours(args, rank, world)
    if world > 1:
        import torch

        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
