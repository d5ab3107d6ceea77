"""Benchmark of the GDP prefill hot path on GB300 (one JSON line on rank 0).

A step is one pass of the prefill path over the bf16 prefill workload
(B=2, T=4096, H=HV=16, K=V=128, M=2, chunk 64): gdp_prefill_prepare on the
post-conv activations (G=H: one key/query group per head) followed by
gdp_chunk_fwd with the in-kernel L2 norm of q and k, producing o [B,T,HV,V]
fp32 and the final state. Inputs are synthetic (seeded N(0,1) activations,
the pages' gate-input distributions) and resident in HBM before the timed
region; L2 is flushed before every timed step by a 256 MiB write followed by
a 256 MiB read, so that no step data is cached and the flush's own dirty lines
are written back before the step starts rather than inside its first kernel.

value = expanded tokens (B*T*M) per second over all ranks; e2e = the same
through the C ABI with the step's inputs copied from pinned host memory and
o copied back inside the timed region. roofline = the dominant kernel's
achieved bandwidth (or flop rate) against the measured peak. Per-kernel times
come from CUDA events recorded on the launching stream (the library's
stage-event hook). Multi-GPU: each rank runs its own copy of the workload, no
collective on the data path (weak scaling).

--impl reference times the CPU oracle (the plain fp64 walk that the tests use
as ground truth) on a bounded sample per step of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "GDP prefill tokens/sec (T·M) and % of bf16 TC peak; prepare GB/s vs HBM"
WORKLOAD = dict(B=2, T=4096, H=16, HV=16, G=16, K=128, V=128, M=2, BT=64)
DECODE = dict(n=256, S=4, M=2, H=32, G=8, P=128, N=128)
# Device-side pause (~1 ms) between the L2 flush and the start event of a timed
# step, so that the launches of the step are all queued before it starts: the
# kernel-timed value then holds no host (Python/ctypes) launch latency. The e2e
# figure keeps every host cost.
HOST_LEAD_CYCLES = 2_000_000
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) per launch of each
# kernel at the bench workload, from one `ncu --set full` capture of
# `bench.py --only prefill --steps 2 --warmup 3`. A kernel's entry is removed
# whenever the kernel changes after the capture.
TRAFFIC = {"wy": 351.9e6, "scan_out": 429.0e6, "prepare": 279.5e6}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------------------------------
# algorithmic work: the method's own tensors and flops, never the intermediates of
# this design (w, u, decay records, v_new or chunk states that kernels hand to each
# other)
# ----------------------------------------------------------------------------------

def method_work(Tt, N_seq, H, HV, K, V, M, BT, fused):
    """Algorithmic flops and bytes of one chunked forward over Tt tokens (all
    sequences) in N_seq sequences, apportioned to the kernels.

    Bytes are the fused floor of the method: q, k, v (bf16), beta, g (fp32) read,
    o (fp32) and the final state (fp32) written. A kernel is charged the method
    tensors it reads or writes: WY reads k, v, beta, g; the state scan reads k, g
    and writes the state; the output reads q, k, g and writes o (the fused scan +
    output does both). Flops: the chunked algebra at chunk BT per expanded token
    and value head, 2 BT (2K + V) for the transition block, its inverse and w, u;
    4 K V for the state recurrence; 2 BT (K + V) + 2 K V / M for the output (one
    multiply-add = 2 flops; the hi/lo operand passes of this design are not
    counted)."""
    E = Tt * M
    b_q, b_k, b_v = Tt * H * K * 2, E * H * K * 2, E * HV * V * 2
    b_beta, b_g = E * HV * 4, Tt * HV * 4
    b_o, b_state = Tt * HV * V * 4, N_seq * HV * K * V * 4
    f_wy = E * HV * 2 * BT * (2 * K + V)
    f_h = E * HV * 4 * K * V
    f_o = E * HV * (2 * BT * (K + V) + 2 * K * V / M)
    out = {"E": E,
           "chunk_bytes": b_q + b_k + b_v + b_beta + b_g + b_o + b_state,
           "flops": {"wy": f_wy, "h": f_h, "o": f_o, "scan_out": f_h + f_o,
                     "chunk": f_wy + f_h + f_o},
           "bytes": {"wy": b_k + b_v + b_beta + b_g,
                     "h": b_k + b_g + b_state,
                     "o": b_q + b_k + b_g + b_o,
                     "scan_out": b_q + b_k + b_g + b_o + b_state}}
    out["kernels"] = ("wy", "scan_out") if fused else ("wy", "h", "o")
    return out


def prepare_bytes(n, T, M, H, G, P, N, decode):
    """Bytes the prepare map moves: x and ba read; q, k, v, beta, g written."""
    rows = n * T
    D = M * H * P + M * G * N + G * N
    L = T * M
    qrows = L if decode else T
    return (rows * D * 2 + rows * (M * H + H) * 2 + n * qrows * H * N * 2 + n * L * H * N * 2
            + n * L * H * P * 2 + n * L * H * 4 + n * (L if decode else T) * H * 4)


def algorithmic(w=WORKLOAD):
    """Algorithmic work per step of the headline prefill workload."""
    B, T, H, HV, G, K, V, M, BT = (w[k] for k in ("B", "T", "H", "HV", "G", "K", "V", "M", "BT"))
    out = method_work(B * T, B, H, HV, K, V, M, BT, fused=(M == 2))
    out["prepare_bytes"] = prepare_bytes(B, T, M, H, G, V, K, False)
    return out


def roof_entry(ms, flops, nbytes, tc, hbm):
    """Achieved rates of one kernel against its algorithmic work and its binding
    roofline (the larger of the tensor-core time and the HBM time at the peaks)."""
    sec = ms * 1e-3
    tf = flops / sec / 1e12
    gbs = nbytes / sec / 1e9
    bound = "tensor" if flops / (tc * 1e12) >= nbytes / (hbm * 1e9) else "hbm"
    return {"ms": ms, "TFLOPs": tf, "tc_frac": tf / tc, "GBps": gbs, "hbm_frac": gbs / hbm,
            "alg_bytes": nbytes, "alg_flops": flops,
            "bound": bound, "frac": tf / tc if bound == "tensor" else gbs / hbm}


# ----------------------------------------------------------------------------------
# clocks sampled during the timed region
# ----------------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                self.rows.append(parts)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[0]) for r in self.rows if num(r[0]) is not None]
        mx = [num(r[1]) for r in self.rows if num(r[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4)
                          if r[4 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(self.rows)}


# ----------------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------------

def make_inputs(dev, seed=0):
    import synth_inputs as si
    w = WORKLOAD
    d = si.prepare_inputs(w["B"], w["T"], w["M"], w["H"], w["G"], w["V"], w["K"], seed=seed)
    return d


class Prefill:
    """Buffers and one step of the prefill path, all on `dev`."""

    def __init__(self, gdp, d, dev):
        w = WORKLOAD
        self.gdp = gdp
        B, T, H, G, K, V, M = w["B"], w["T"], w["H"], w["G"], w["K"], w["V"], w["M"]
        self.x = d["x"].to(dev)
        self.ba = d["ba"].to(dev)
        self.A_log = d["A_log"].to(dev)
        self.dt_bias = d["dt_bias"].to(dev)
        bf = torch.bfloat16
        self.pre = (torch.empty(B, T, H, K, dtype=bf, device=dev),
                    torch.empty(B, T * M, H, K, dtype=bf, device=dev),
                    torch.empty(B, T * M, H, V, dtype=bf, device=dev),
                    torch.empty(B, T * M, H, dtype=torch.float32, device=dev),
                    torch.empty(B, T, H, dtype=torch.float32, device=dev))
        self.o = torch.empty(B, T, H, V, dtype=torch.float32, device=dev)
        self.fs = torch.empty(B, H, K, V, dtype=torch.float32, device=dev)
        need = gdp.gdp_chunk_fwd_workspace_size(B, T, B, H, H, K, V, M, w["BT"], bf)
        self.ws = torch.empty(need, dtype=torch.uint8, device=dev)
        off = gdp.gdp_chunk_fwd_stage_offsets(B, T, B, H, H, K, V, M, w["BT"], bf)
        self.path, self.fused = off[5], off[7] == 1

    def step(self, ev_prep=None):
        w = WORKLOAD
        if ev_prep is not None:
            ev_prep[0].record()
        self.gdp.gdp_prefill_prepare(self.x, self.ba, self.A_log, self.dt_bias, w["M"], w["H"],
                                     w["G"], w["V"], w["K"], out=self.pre)
        if ev_prep is not None:
            ev_prep[1].record()
        q, k, v, beta, g = self.pre
        self.gdp.gdp_chunk_fwd(q, k, v, beta, g, chunk_size=w["BT"], num_householder=w["M"],
                               use_qk_l2norm=True, workspace=self.ws, out=(self.o, self.fs))


def launches_per_step(fused: bool) -> int:
    # prepare, chunk tables, WY, then the scan with the output fused into it
    # (one launch) or the scan and the output kernel (two)
    return 1 + 1 + 1 + (1 if fused else 2)


def kernel_names(pf) -> tuple:
    return ("wy", "scan_out") if pf.fused else ("wy", "h", "o")


def kernel_rooflines(times, alg, tc, hbm, fused):
    """Per-kernel roof entries from the stage-event times of a chunked forward."""
    stage_ms = {"wy": statistics.mean(times["wy"]), "h": statistics.mean(times["h"]),
                "o": statistics.mean(times["o"])}
    if fused:  # stage events 3 and 4 are recorded back to back
        stage_ms = {"wy": stage_ms["wy"], "scan_out": stage_ms["h"] + stage_ms["o"]}
    kern = {n: roof_entry(stage_ms[n], alg["flops"][n], alg["bytes"][n], tc, hbm)
            for n in alg["kernels"]}
    kern["tables"] = {"ms": statistics.mean(times["tables"])}
    return kern


def roofline_object(name, k, tc, hbm, pk_src, traffic):
    """The bench line's roofline object for kernel `name` (entry `k`)."""
    if k["bound"] == "hbm":
        roof = {"kernel": name, "bound": "hbm", "achieved": k["GBps"], "peak": hbm,
                "unit": "GB/s", "frac": k["hbm_frac"], "peak_source": pk_src + " (hbm_gbs)"}
    else:
        roof = {"kernel": name, "bound": "tensor", "achieved": k["TFLOPs"], "peak": tc,
                "unit": "TFLOP/s", "frac": k["tc_frac"],
                "peak_source": pk_src + " (bf16_tflops, burst)"}
    roof["algorithmic_bytes"] = k["alg_bytes"]
    roof["traffic"] = traffic
    roof["traffic_over_algorithmic"] = None if traffic is None else traffic / k["alg_bytes"]
    return roof


def run_ours(args, rank, world, dev):
    import linear_attention_ssm_gdp_gb300 as gdp
    gdp.load()
    pk, pk_src = peaks()
    alg = algorithmic()
    d = make_inputs(dev)
    pf = Prefill(gdp, d, dev)
    flush = L2Flush(dev)
    stage = [torch.cuda.Event(enable_timing=True) for _ in range(gdp.GDP_STAGE_EVENTS)]
    prep_ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    step_ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    gdp.gdp_set_stage_events(stage)

    for _ in range(args.warmup):
        flush()
        pf.step()
    torch.cuda.synchronize()

    sampler = ClockSampler(torch.cuda.current_device() if dev.index is None else dev.index)
    sampler.start()
    time.sleep(0.3)
    times = {"step": [], "prepare": [], "tables": [], "wy": [], "h": [], "o": []}
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    # the timed steps: only the two step events in the stream, no stage events between
    # the kernels (each event record is one more stream operation between launches)
    gdp.gdp_set_stage_events(None)
    for _ in range(args.steps):
        flush()
        torch.cuda._sleep(HOST_LEAD_CYCLES)  # the host queues the whole step meanwhile
        step_ev[0].record()
        pf.step()
        step_ev[1].record()
        torch.cuda.synchronize()
        times["step"].append(step_ev[0].elapsed_time(step_ev[1]))
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    # per-kernel breakdown: the same steps again with events at the stage boundaries
    gdp.gdp_set_stage_events(stage)
    for _ in range(max(5, min(args.steps, 20))):
        flush()
        torch.cuda._sleep(HOST_LEAD_CYCLES)
        pf.step(prep_ev)
        torch.cuda.synchronize()
        times["prepare"].append(prep_ev[0].elapsed_time(prep_ev[1]))
        times["tables"].append(stage[0].elapsed_time(stage[1]))
        times["wy"].append(stage[1].elapsed_time(stage[2]))
        times["h"].append(stage[2].elapsed_time(stage[3]))
        times["o"].append(stage[3].elapsed_time(stage[4]))
    torch.cuda.synchronize()
    # keep the GPU busy a little longer so the sampler sees load, then stop
    extra_t0 = time.time()
    while time.time() - extra_t0 < 0.5:
        pf.step()
    torch.cuda.synchronize()
    sampler.stop()
    gdp.gdp_set_stage_events(None)

    ms = max_over_ranks(statistics.mean(times["step"]), world, dev)
    units = alg["E"] * world
    value = units / (ms * 1e-3)

    # per-kernel rooflines against the method's algorithmic work; the step is
    # well under a millisecond, so the tensor peak is the measured burst figure
    hbm = pk["hbm_gbs"]
    tc = pk["bf16_tflops"]
    kern = kernel_rooflines(times, alg, tc, hbm, pf.fused)
    prep_ms = statistics.mean(times["prepare"])
    kern["prepare"] = roof_entry(prep_ms, 0, alg["prepare_bytes"], tc, hbm)
    chunk_ms = kern["tables"]["ms"] + sum(kern[n]["ms"] for n in alg["kernels"])
    chunk_tf = alg["flops"]["chunk"] / (chunk_ms * 1e-3) / 1e12
    chunk_gbs = alg["chunk_bytes"] / (chunk_ms * 1e-3) / 1e9
    dominant = max(("prepare",) + alg["kernels"], key=lambda n: kern[n]["ms"])
    traffic = TRAFFIC.get(dominant) if args.traffic is None else args.traffic
    roof = roofline_object(dominant, kern[dominant], tc, hbm, pk_src, traffic)

    full = args.only == "all"
    e2e = run_e2e(args, gdp, d, dev, pf) if full else None
    decode = run_decode(args, gdp, dev, pk) if full else None
    prep_eager = run_prepare_eager(args, gdp, dev) if full else None
    ungated = run_ungated(args, gdp, dev, pk, pk_src, pf) if full else None
    varlen = run_varlen(args, gdp, dev, pk, pk_src) if full else None
    gva = run_gva(args, gdp, dev, pk, pk_src) if full else None
    clocks = sampler.summary()
    w = WORKLOAD
    line = {
        "metric": METRIC, "value": value, "unit": "expanded tokens/s (B*T*M)",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) activations and gate inputs)",
        "config": workload_config(world),
        "chunk_path": ("tensor-core" if pf.path == 1 else "generic")
        + (", scan and output fused" if pf.fused else ""),
        "roofline": roof,
        "chunk": {"ms": chunk_ms, "TFLOPs": chunk_tf, "tc_frac": chunk_tf / tc,
                  "GBps_fused_floor": chunk_gbs, "hbm_frac": chunk_gbs / hbm},
        "prepare": {"ms": prep_ms, "GBps": kern["prepare"]["GBps"],
                    "hbm_frac": kern["prepare"]["frac"]},
        "kernels": kern,
        "decode": decode,
        "prepare_vs_eager": prep_eager,
        "ungated": ungated,
        "config2_varlen": varlen,
        "config3_gva": gva,
        "e2e": e2e,
        "gpu_launches": launches_per_step(pf.fused) * args.steps,
        "clocks": clocks,
        "peaks": {"hbm_gbs": hbm, "bf16_tflops": tc, "source": pk_src,
                  "note": "burst tensor peak: every timed step is under a few ms"},
    }
    if rank == 0 and full and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(d, min_seconds=args.cpu_seconds,
                                            max_seconds=max(30.0, args.cpu_seconds))
    return line


def eager_prepare(x, ba, A_log, dt_bias, M, H, G, P, N, decode):
    """The prepare step as the pages' eager PyTorch composition (the comparator
    the fused prepare kernel replaces): the value/key/query splits, the group
    expansion and the copy folding as torch copies, the gates as fp32 torch
    ops. Same outputs, bit for bit, as gdp_{prefill,decode}_prepare."""
    import torch.nn.functional as F
    n, T = x.shape[:2]
    hpg = H // G
    kb, qb = M * H * P, M * H * P + M * G * N
    v = x[..., :kb].reshape(n, T, M, H, P).reshape(n, T * M, H, P)
    k = x[..., kb:qb].reshape(n, T, M, G, N).repeat_interleave(hpg, dim=3).reshape(n, T * M, H, N)
    qx = x[..., qb:].reshape(n, T, G, N).repeat_interleave(hpg, dim=2)
    beta = torch.sigmoid(ba[..., :M * H].float().reshape(n, T * M, H))
    gt = -torch.exp(A_log.float()) * F.softplus(ba[..., M * H:].float() + dt_bias.float())
    if decode:
        q = torch.zeros(n, T, M, H, N, dtype=x.dtype, device=x.device)
        q[:, :, M - 1] = qx
        g = torch.zeros(n, T, M, H, dtype=torch.float32, device=x.device)
        g[:, :, 0] = gt
        return q.reshape(n, T * M, H, N), k, v, beta, g.reshape(n, T * M, H)
    return qx.contiguous(), k, v, beta, gt


def run_prepare_eager(args, gdp, dev):
    """The fused prepare kernel against the eager composition, both timed with
    CUDA events after an L2 flush, on the prefill and the decode workloads."""
    import synth_inputs as si
    flush = L2Flush(dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    out = {}
    for name, decode in (("prefill", False), ("decode", True)):
        if decode:
            w = DECODE
            n, S, M, H, G, P, N = w["n"], w["S"], w["M"], w["H"], w["G"], w["P"], w["N"]
            d = si.prepare_inputs(n, S, M, H, G, P, N, seed=1)
        else:
            w = WORKLOAD
            M, H, G, P, N = w["M"], w["H"], w["G"], w["V"], w["K"]
            d = make_inputs(dev)
        x, ba = d["x"].to(dev), d["ba"].to(dev)
        A_log, dt_bias = d["A_log"].to(dev), d["dt_bias"].to(dev)
        fused = gdp.gdp_decode_prepare if decode else gdp.gdp_prefill_prepare
        ref = eager_prepare(x, ba, A_log, dt_bias, M, H, G, P, N, decode)
        got = fused(x, ba, A_log, dt_bias, M, H, G, P, N)
        exact = all(torch.equal(a, b) for a, b in zip(got, ref))
        times = {}
        for label, fn in (("fused", lambda: fused(x, ba, A_log, dt_bias, M, H, G, P, N, out=got)),
                          ("eager", lambda: eager_prepare(x, ba, A_log, dt_bias, M, H, G, P, N,
                                                          decode))):
            for _ in range(3):
                fn()
            t = []
            for _ in range(max(5, min(args.steps, 20))):
                flush()
                torch.cuda._sleep(HOST_LEAD_CYCLES)
                ev[0].record()
                fn()
                ev[1].record()
                torch.cuda.synchronize()
                t.append(ev[0].elapsed_time(ev[1]))
            times[label] = statistics.mean(t) * 1e3
        out[name] = {"fused_us": times["fused"], "eager_us": times["eager"],
                     "eager_over_fused": times["eager"] / times["fused"], "bit_exact": exact}
    return out


def run_e2e(args, gdp, d, dev, pf):
    """Whole-job throughput through the C ABI with host buffers. Every step
    copies its inputs (x, ba) from pinned host memory, runs the two calls and
    copies o and the final state back, all inside the timed region. Steps
    alternate between two CUDA streams with their own device buffers and
    workspaces, so a step's uploads overlap the previous step's kernels and
    downloads (the way a caller streaming batches would run it)."""
    w = WORKLOAD
    hx = d["x"].pin_memory()
    hba = d["ba"].pin_memory()
    lanes = [pf, Prefill(gdp, d, dev)]
    streams = [torch.cuda.Stream(dev), torch.cuda.Stream(dev)]
    hout = [(torch.empty(pf.o.shape, dtype=torch.float32).pin_memory(),
             torch.empty(pf.fs.shape, dtype=torch.float32).pin_memory()) for _ in lanes]
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]

    def one(i):
        p, s, (ho, hfs) = lanes[i % 2], streams[i % 2], hout[i % 2]
        with torch.cuda.stream(s):
            p.x.copy_(hx, non_blocking=True)
            p.ba.copy_(hba, non_blocking=True)
            p.step()
            ho.copy_(p.o, non_blocking=True)
            hfs.copy_(p.fs, non_blocking=True)

    for i in range(4):
        one(i)
    torch.cuda.synchronize()
    n = max(4, min(args.steps, 20))
    cur = torch.cuda.current_stream(dev)
    ev[0].record(cur)
    for s in streams:
        s.wait_stream(cur)
    for i in range(n):
        one(i)
    for s in streams:
        cur.wait_stream(s)
    ev[1].record(cur)
    torch.cuda.synchronize()
    ms = ev[0].elapsed_time(ev[1]) / n
    bi = hx.numel() * hx.element_size() + hba.numel() * hba.element_size()
    bo = hout[0][0].numel() * 4 + hout[0][1].numel() * 4
    return {"value": w["B"] * w["T"] * w["M"] / (ms * 1e-3),
            "unit": "expanded tokens/s (B*T*M)", "ms_per_step": ms,
            "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
            "steps": n, "overlap": "two streams, alternating steps"}


class L2Flush:
    """Evicts L2 (129 MB on GB300): a 256 MiB write, then a 256 MiB read so that
    the written lines leave L2 before the timed work, not during it."""

    def __init__(self, dev):
        n = 256 * 1024 * 1024 // 4
        self.w = torch.empty(n, dtype=torch.float32, device=dev)
        self.r = torch.ones(n, dtype=torch.float32, device=dev)

    def __call__(self):
        self.w.fill_(1.0)
        self.r.sum()


def run_decode(args, gdp, dev, pk):
    """Decode step (prepare + recurrent update), n=256 S=4 M=2 H=32 G=8 P=N=128."""
    import synth_inputs as si
    w = DECODE
    n, S, M, H, G, P, N = w["n"], w["S"], w["M"], w["H"], w["G"], w["P"], w["N"]
    d = si.prepare_inputs(n, S, M, H, G, P, N, seed=1)
    x, ba = d["x"].to(dev), d["ba"].to(dev)
    A_log, dt_bias = d["A_log"].to(dev), d["dt_bias"].to(dev)
    state = si.decode_state(n, H, N, P).to(dev)
    outs = gdp.gdp_decode_prepare(x, ba, A_log, dt_bias, M, H, G, P, N)
    o = torch.empty(n, S * M, H, P, device=dev)
    flush = L2Flush(dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    for _ in range(3):
        gdp.gdp_decode_prepare(x, ba, A_log, dt_bias, M, H, G, P, N, out=outs)
        gdp.gdp_recurrent_update(*outs, state, use_qk_l2norm=True, out=o)
    torch.cuda.synchronize()
    tp, tr = [], []
    for _ in range(max(5, min(args.steps, 50))):
        flush()
        torch.cuda._sleep(HOST_LEAD_CYCLES)
        ev[0].record()
        gdp.gdp_decode_prepare(x, ba, A_log, dt_bias, M, H, G, P, N, out=outs)
        ev[1].record()
        gdp.gdp_recurrent_update(*outs, state, use_qk_l2norm=True, out=o)
        ev[2].record()
        torch.cuda.synchronize()
        tp.append(ev[0].elapsed_time(ev[1]))
        tr.append(ev[1].elapsed_time(ev[2]))
    D = M * H * P + M * G * N + G * N
    L = S * M
    prep_bytes = (n * S * D * 2 + n * S * (M * H + H) * 2 + n * L * H * (2 * N + P) * 2
                  + 2 * n * L * H * 4)
    rec_bytes = (2 * n * H * N * P * 4 + n * L * H * (2 * N + P) * 2 + 2 * n * L * H * 4
                 + n * L * H * P * 4)
    mp, mr = statistics.mean(tp), statistics.mean(tr)
    hbm = pk["hbm_gbs"]
    # the same update through a state pool (decode serving): 2n pool entries,
    # requests on a seeded permutation of them, every 16th request padding (-1)
    gen = torch.Generator().manual_seed(3)
    slot = torch.randperm(2 * n, generator=gen)[:n].to(torch.int32)
    slot[::16] = -1
    slot = slot.to(dev)
    pool = si.decode_state(2 * n, H, N, P).to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    for _ in range(3):
        gdp.gdp_recurrent_update_slots(*outs, pool, slot, use_qk_l2norm=True, status=status,
                                       out=o)
    torch.cuda.synchronize()
    ts = []
    for _ in range(max(5, min(args.steps, 50))):
        flush()
        torch.cuda._sleep(HOST_LEAD_CYCLES)
        ev[0].record()
        gdp.gdp_recurrent_update_slots(*outs, pool, slot, use_qk_l2norm=True, status=status,
                                       out=o)
        ev[1].record()
        torch.cuda.synchronize()
        ts.append(ev[0].elapsed_time(ev[1]))
    live = int((slot >= 0).sum())
    ms_slots = statistics.mean(ts)
    slot_bytes = rec_bytes - (n - live) * (2 * H * N * P * 4)  # padding moves no state
    slots = torch.arange(n, dtype=torch.int32, device=dev)
    conv = time_conv_prepare(gdp, dev, x, ba, A_log, dt_bias, M, H, G, P, N, None, outs,
                             prep_bytes, hbm, decode=True, slots=slots)
    return {"workload": "decode n256 S4 M2 H32 G8 P128 N128 (fp32 state)",
            "conv_prepare": conv,
            "prepare_us": mp * 1e3, "prepare_GBps": prep_bytes / (mp * 1e-3) / 1e9,
            "prepare_hbm_frac": prep_bytes / (mp * 1e-3) / 1e9 / hbm,
            "update_us": mr * 1e3, "update_GBps": rec_bytes / (mr * 1e-3) / 1e9,
            "update_hbm_frac": rec_bytes / (mr * 1e-3) / 1e9 / hbm,
            "update_slots": {"us": ms_slots * 1e3, "pool_entries": 2 * n, "live_requests": live,
                             "GBps": slot_bytes / (ms_slots * 1e-3) / 1e9,
                             "hbm_frac": slot_bytes / (ms_slots * 1e-3) / 1e9 / hbm,
                             "status": int(status.item())},
            "requests_per_s": n / ((mp + mr) * 1e-3)}


# ----------------------------------------------------------------------------------
# the other prefill workloads: measured in the same run, reported beside the headline
# ----------------------------------------------------------------------------------

def _time_chunk_steps(gdp, step, stage, flush, steps, warmup, prep_ev=None):
    """Times `step()` (one pass of the workload) with CUDA events after an L2 flush;
    returns per-step, prepare and stage times (ms) as lists."""
    step_ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    for _ in range(warmup):
        flush()
        step()
    torch.cuda.synchronize()
    times = {"step": [], "prepare": [], "tables": [], "wy": [], "h": [], "o": []}
    # whole steps without the library's stage events, then the per-stage breakdown
    gdp.gdp_set_stage_events(None)
    for _ in range(steps):
        flush()
        torch.cuda._sleep(HOST_LEAD_CYCLES)
        step_ev[0].record()
        step()
        step_ev[1].record()
        torch.cuda.synchronize()
        times["step"].append(step_ev[0].elapsed_time(step_ev[1]))
    gdp.gdp_set_stage_events(stage)
    for _ in range(steps):
        flush()
        torch.cuda._sleep(HOST_LEAD_CYCLES)
        step()
        torch.cuda.synchronize()
        if prep_ev is not None:
            times["prepare"].append(prep_ev[0].elapsed_time(prep_ev[1]))
        times["tables"].append(stage[0].elapsed_time(stage[1]))
        times["wy"].append(stage[1].elapsed_time(stage[2]))
        times["h"].append(stage[2].elapsed_time(stage[3]))
        times["o"].append(stage[3].elapsed_time(stage[4]))
    return times


def _workload_summary(name, times, alg, tc, hbm, pk_src, fused, prep_bytes=None):
    ms = statistics.mean(times["step"])
    kern = kernel_rooflines(times, alg, tc, hbm, fused)
    chunk_ms = kern["tables"]["ms"] + sum(kern[n]["ms"] for n in alg["kernels"])
    out = {"workload": name, "ms_per_step": ms, "value": alg["E"] / (ms * 1e-3),
           "unit": "expanded tokens/s", "kernels": kern,
           "chunk": {"ms": chunk_ms,
                     "TFLOPs": alg["flops"]["chunk"] / (chunk_ms * 1e-3) / 1e12,
                     "GBps_fused_floor": alg["chunk_bytes"] / (chunk_ms * 1e-3) / 1e9,
                     "hbm_frac": alg["chunk_bytes"] / (chunk_ms * 1e-3) / 1e9 / hbm,
                     "tc_frac": alg["flops"]["chunk"] / (chunk_ms * 1e-3) / 1e12 / tc}}
    names = alg["kernels"]
    if prep_bytes is not None:
        pm = statistics.mean(times["prepare"])
        kern["prepare"] = roof_entry(pm, 0, prep_bytes, tc, hbm)
        out["prepare"] = {"us": pm * 1e3, "bytes": prep_bytes, "GBps": kern["prepare"]["GBps"],
                          "hbm_frac": kern["prepare"]["hbm_frac"]}
        names = ("prepare",) + names
    dom = max(names, key=lambda n: kern[n]["ms"])
    out["binding"] = roofline_object(dom, kern[dom], tc, hbm, pk_src, None)
    return out


def run_varlen(args, gdp, dev, pk, pk_src):
    """Packed varlen prefill from prepare: 16 requests, lengths ~U(64, 2048) (seed 0),
    H=HV=32, G=8, P=N=128, M=3, chunk 64; a step is gdp_prefill_prepare on x
    [1, T, M*H*P + M*G*N + G*N] followed by gdp_chunk_fwd with cu_seqlens."""
    import synth_inputs as si
    w = si.WORKLOADS["varlen_bf16"].dims
    M, H, G, P, N, BT = w["M"], w["H"], w["G"], w["P"], w["N"], w["BT"]
    lens = si.varlen_lengths(w["n_seq"], seed=0)
    cu = si.cu_seqlens_of(lens).to(dev)
    T = int(cu[-1])
    d = si.prepare_inputs(1, T, M, H, G, P, N, seed=0)
    x, ba = d["x"].to(dev), d["ba"].to(dev)
    A_log, dt_bias = d["A_log"].to(dev), d["dt_bias"].to(dev)
    bf = torch.bfloat16
    pre = (torch.empty(1, T, H, N, dtype=bf, device=dev),
           torch.empty(1, T * M, H, N, dtype=bf, device=dev),
           torch.empty(1, T * M, H, P, dtype=bf, device=dev),
           torch.empty(1, T * M, H, dtype=torch.float32, device=dev),
           torch.empty(1, T, H, dtype=torch.float32, device=dev))
    nseq = len(lens)
    o = torch.empty(1, T, H, P, dtype=torch.float32, device=dev)
    fs = torch.empty(nseq, H, N, P, dtype=torch.float32, device=dev)
    ws = torch.empty(gdp.gdp_chunk_fwd_workspace_size(1, T, nseq, H, H, N, P, M, BT, bf),
                     dtype=torch.uint8, device=dev)
    off = gdp.gdp_chunk_fwd_stage_offsets(1, T, nseq, H, H, N, P, M, BT, bf)
    stage = [torch.cuda.Event(enable_timing=True) for _ in range(gdp.GDP_STAGE_EVENTS)]
    prep_ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]

    def step():
        prep_ev[0].record()
        gdp.gdp_prefill_prepare(x, ba, A_log, dt_bias, M, H, G, P, N, out=pre)
        prep_ev[1].record()
        q, k, v, beta, g = pre
        gdp.gdp_chunk_fwd(q, k, v, beta, g, cu_seqlens=cu, chunk_size=BT, num_householder=M,
                          use_qk_l2norm=True, workspace=ws, out=(o, fs))

    gdp.gdp_set_stage_events(stage)
    times = _time_chunk_steps(gdp, step, stage, L2Flush(dev), max(3, min(args.steps, 10)), 3,
                              prep_ev)
    gdp.gdp_set_stage_events(None)
    conv = time_conv_prepare(gdp, dev, x, ba, A_log, dt_bias, M, H, G, P, N, cu, pre,
                             prepare_bytes(1, T, M, H, G, P, N, False), pk["hbm_gbs"])
    fused = off[7] == 1
    alg = method_work(T, nseq, H, H, N, P, M, BT, fused)
    out = _workload_summary(
        f"varlen bf16 {nseq} requests U(64,2048) T={T} H=HV=32 G8 K=V=128 M3 BT64 "
        "(prepare + chunk_fwd with cu_seqlens)", times, alg, pk["bf16_tflops"], pk["hbm_gbs"],
        pk_src, fused, prepare_bytes(1, T, M, H, G, P, N, False))
    out["tokens"] = T
    out["conv_prepare"] = conv
    return out


def time_conv_prepare(gdp, dev, x, ba, A_log, dt_bias, M, H, G, P, N, cu, pre, prep_bytes, hbm,
                      W=4, decode=False, slots=None):
    """The short causal conv (width W, SiLU) fused into prepare on the same workload:
    x stands in for the pre-conv activations; conv weights and states are synthetic
    (seeded). Bytes: prepare's plus the conv states read and written."""
    C = x.shape[-1]
    gen = torch.Generator(device=dev)
    gen.manual_seed(1)
    w = torch.randn(C, W, device=dev, generator=gen) * 0.5
    b = torch.randn(C, device=dev, generator=gen) * 0.1
    nst = (cu.numel() - 1) if cu is not None else x.shape[0]
    if decode:
        pool = torch.randn(slots.numel() * 2, C, W - 1, device=dev, generator=gen).to(x.dtype)
        st_bytes = 2 * slots.numel() * C * (W - 1) * x.element_size()
        fn = lambda: gdp.gdp_decode_conv_prepare(x, w, b, ba, A_log, dt_bias, M, H, G, P, N,
                                                 pool, slots, out=pre)
    else:
        st0 = torch.randn(nst, C, W - 1, device=dev, generator=gen).to(x.dtype)
        st_bytes = 2 * nst * C * (W - 1) * x.element_size()
        fn = lambda: gdp.gdp_prefill_conv_prepare(x, w, b, ba, A_log, dt_bias, M, H, G, P, N,
                                                  conv_state=st0, cu_seqlens=cu, out=pre)
    flush = L2Flush(dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    for _ in range(3):
        fn()
    ts = []
    for _ in range(10):
        flush()
        torch.cuda._sleep(HOST_LEAD_CYCLES)
        ev[0].record()
        fn()
        ev[1].record()
        torch.cuda.synchronize()
        ts.append(ev[0].elapsed_time(ev[1]))
    us = statistics.mean(ts) * 1e3
    nbytes = prep_bytes + st_bytes
    return {"W": W, "us": us, "bytes": nbytes, "GBps": nbytes / (us * 1e-6) / 1e9,
            "hbm_frac": nbytes / (us * 1e-6) / 1e9 / hbm}


def run_ungated(args, gdp, dev, pk, pk_src, pf):
    """The headline workload's chunked forward without decay (g = None, the pages'
    USE_G = false), on the q, k, v, beta the prepare step produced."""
    w = WORKLOAD
    q, k, v, beta, _ = pf.pre
    stage = [torch.cuda.Event(enable_timing=True) for _ in range(gdp.GDP_STAGE_EVENTS)]

    def step():
        gdp.gdp_chunk_fwd(q, k, v, beta, None, chunk_size=w["BT"], num_householder=w["M"],
                          use_qk_l2norm=True, workspace=pf.ws, out=(pf.o, pf.fs))

    gdp.gdp_set_stage_events(stage)
    times = _time_chunk_steps(gdp, step, stage, L2Flush(dev), max(5, min(args.steps, 20)), 3)
    gdp.gdp_set_stage_events(None)
    alg = method_work(w["B"] * w["T"], w["B"], w["H"], w["HV"], w["K"], w["V"], w["M"], w["BT"],
                      pf.fused)
    alg["bytes"] = {n: b - w["B"] * w["T"] * w["HV"] * 4 if n != "h" else b
                    for n, b in alg["bytes"].items()}  # no g is read
    alg["chunk_bytes"] -= w["B"] * w["T"] * w["HV"] * 4
    return _workload_summary("prefill bf16 B2 T4096 H16 HV16 K128 V128 M2 BT64, ungated "
                             "(g = None; chunk_fwd only)", times, alg, pk["bf16_tflops"],
                             pk["hbm_gbs"], pk_src, pf.fused)


def run_gva(args, gdp, dev, pk, pk_src):
    """GVA prefill: B=4, T=8192, H=8, HV=32, K=128, V=256, M=2, chunk 64; a step is
    gdp_chunk_fwd on q, k, v, beta, g already in HBM. Inputs are drawn on the device
    (seeded): q, k, v ~ N(0,1) bf16; beta = sigmoid(N(0,1)); g = -exp(A_log)
    softplus(N(0,1) + dt_bias) with A_log ~ U(0, ln 16), dt_bias ~ N(0, 0.5^2)."""
    import torch.nn.functional as F
    B, T, H, HV, K, V, M, BT = 4, 8192, 8, 32, 128, 256, 2, 64
    gen = torch.Generator(device=dev)
    gen.manual_seed(0)
    bf = torch.bfloat16
    q = torch.randn(B, T, H, K, device=dev, generator=gen).to(bf)
    k = torch.randn(B, T * M, H, K, device=dev, generator=gen).to(bf)
    v = torch.randn(B, T * M, HV, V, device=dev, generator=gen).to(bf)
    beta = torch.sigmoid(torch.randn(B, T * M, HV, device=dev, generator=gen))
    A_log = torch.rand(HV, device=dev, generator=gen) * math.log(16.0)
    dt_bias = torch.randn(HV, device=dev, generator=gen) * 0.5
    g = -torch.exp(A_log) * F.softplus(torch.randn(B, T, HV, device=dev, generator=gen) + dt_bias)
    o = torch.empty(B, T, HV, V, dtype=torch.float32, device=dev)
    fs = torch.empty(B, HV, K, V, dtype=torch.float32, device=dev)
    ws = torch.empty(gdp.gdp_chunk_fwd_workspace_size(B, T, B, H, HV, K, V, M, BT, bf),
                     dtype=torch.uint8, device=dev)
    off = gdp.gdp_chunk_fwd_stage_offsets(B, T, B, H, HV, K, V, M, BT, bf)
    stage = [torch.cuda.Event(enable_timing=True) for _ in range(gdp.GDP_STAGE_EVENTS)]

    def step():
        gdp.gdp_chunk_fwd(q, k, v, beta, g, chunk_size=BT, num_householder=M,
                          use_qk_l2norm=True, workspace=ws, out=(o, fs))

    gdp.gdp_set_stage_events(stage)
    times = _time_chunk_steps(gdp, step, stage, L2Flush(dev), max(3, min(args.steps, 6)), 3)
    gdp.gdp_set_stage_events(None)
    fused = off[7] == 1
    alg = method_work(B * T, B, H, HV, K, V, M, BT, fused)
    return _workload_summary("GVA bf16 B4 T8192 H8 HV32 K128 V256 M2 BT64 (chunk_fwd)", times,
                             alg, pk["bf16_tflops"], pk["hbm_gbs"], pk_src, fused)


# ----------------------------------------------------------------------------------
# CPU oracle (baseline / reference arm)
# ----------------------------------------------------------------------------------

def _oracle_sample(d, rows, heads, t_len):
    """Oracle prepare + fp64 walk over batch rows [0, rows), value heads [0, heads) and
    the first t_len tokens of the prefill workload; returns expanded token-heads done."""
    import oracle
    w = WORKLOAD
    x = d["x"][:rows, :t_len]
    ba = d["ba"][:rows, :t_len]
    q, k, v, beta, g = oracle.prepare(x, ba, d["A_log"], d["dt_bias"], w["M"], w["H"], w["G"],
                                      w["V"], w["K"], decode=False)
    hs = slice(0, heads)
    oracle.walk(q[:, :, hs], k[:, :, hs], v[:, :, hs], beta[:, :, hs], g[:, :, hs], w["M"],
                w["K"] ** -0.5, l2norm=True)
    return rows * t_len * w["M"] * heads


def _oracle_rate(d):
    """Calibration: expanded token-heads per second of the oracle on a small sample."""
    w = WORKLOAD
    t0 = time.perf_counter()
    done = _oracle_sample(d, 1, w["HV"], 128)
    return done / max(time.perf_counter() - t0, 1e-9)


def cpu_baseline(d, min_seconds=10.0, max_seconds=30.0):
    """The oracle as it stands on the host cores: the whole prefill workload (both batch
    rows, all heads, all tokens), repeated until about min_seconds of CPU work; if one
    pass would exceed max_seconds, a prefix of the tokens instead."""
    import oracle
    oracle.build()
    w = WORKLOAD
    full = w["B"] * w["T"] * w["M"] * w["HV"]
    est = full / _oracle_rate(d)
    if est <= max_seconds / 4:  # re-estimate on one whole pass (threads warm, all rows)
        t0 = time.perf_counter()
        _oracle_sample(d, w["B"], w["HV"], w["T"])
        est = time.perf_counter() - t0
    if est <= max_seconds:
        rows, t_len = w["B"], w["T"]
        reps = max(1, min(math.ceil(min_seconds / max(est, 1e-9)), int(max_seconds / max(est, 1e-9))))
    else:
        rows, reps = 1, 1
        t_len = max(64, int(w["T"] * (0.5 * max_seconds) / (est / w["B"])))
    done, t0 = 0, time.perf_counter()
    for _ in range(reps):
        done += _oracle_sample(d, rows, w["HV"], t_len)
    dt = time.perf_counter() - t0
    value = done / w["HV"] / dt  # expanded tokens (all heads) per second
    return {"value": value, "unit": "expanded tokens/s (B*T*M)", "cores": oracle.max_threads(),
            "kind": "oracle",
            "sample": f"{reps} x (batch rows 0..{rows - 1}, all {w['HV']} heads, first {t_len} "
                      f"tokens x {w['M']} copies): oracle prepare + fp64 walk, {dt:.1f} s"}


def workload_config(world: int) -> dict:
    """The bench line's `config`, the same for both arms."""
    w = WORKLOAD
    return {"workload": "prefill bf16 B2 T4096 H16 HV16 K128 V128 M2 BT64 "
                        "(prepare + chunk_fwd, G=16, in-kernel qk L2 norm)",
            "B": w["B"], "T": w["T"], "H": w["H"], "HV": w["HV"], "G": w["G"],
            "K": w["K"], "V": w["V"], "M": w["M"], "chunk_size": w["BT"],
            "parallelism": f"replicas x{world} (no collective)",
            "l2": "flushed before every timed step (256 MiB write, then a 256 MiB read)"}


def run_reference(args, rank, world, budget_seconds=150.0):
    """Reference arm: the CPU oracle, rank 0 only. Each step is batch row 0, all heads,
    a token prefix sized so that warm-up + timed steps take about budget_seconds."""
    if rank != 0:
        return None
    import oracle
    oracle.build()
    d = make_inputs(torch.device("cpu"))
    w = WORKLOAD
    heads = w["HV"]
    rate = _oracle_rate(d)
    per_step = budget_seconds / max(1, args.steps + args.warmup)
    t_len = int(min(w["T"], max(64, rate * per_step / (w["M"] * heads))))
    for _ in range(args.warmup):
        _oracle_sample(d, 1, heads, t_len)
    ts = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        _oracle_sample(d, 1, heads, t_len)
        ts.append(time.perf_counter() - t0)
    per_step = statistics.mean(ts)
    value = (t_len * w["M"]) / per_step  # expanded tokens (all heads) per second
    sample = (f"per step: batch row 0, all {heads} heads, first {t_len} of {w['T']} tokens "
              f"x {w['M']} copies: oracle prepare + fp64 walk")
    cores = oracle.max_threads()
    return {"metric": METRIC, "value": value, "unit": "expanded tokens/s (B*T*M)",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": per_step * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(world),
            "impl": "reference",
            "cpu_baseline": {"kind": "oracle", "cores": cores, "sample": sample, "value": value},
            "e2e": {"value": value, "unit": "expanded tokens/s (B*T*M)",
                    "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def max_over_ranks(ms: float, world: int, device) -> float:
    """Slowest rank's step time (every rank calls this; world 1 returns ms)."""
    if world <= 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="minimum CPU seconds of oracle work for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--traffic", type=float, default=None,
                    help="ncu DRAM bytes per launch of the dominant kernel, if measured")
    ap.add_argument("--only", default="all",
                    choices=["all", "prefill", "decode", "varlen", "gva"],
                    help="profiling runs: time only the prefill step (no e2e, decode or CPU "
                         "baseline), only the decode step, or only the varlen / GVA workload")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    if world > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device())
    if args.only in ("decode", "varlen", "gva"):
        import linear_attention_ssm_gdp_gb300 as gdp
        gdp.load()
        pk, pk_src = peaks()
        if args.only == "decode":
            line = {"decode": run_decode(args, gdp, dev, pk)}
        elif args.only == "varlen":
            line = {"config2_varlen": run_varlen(args, gdp, dev, pk, pk_src)}
        else:
            line = {"config3_gva": run_gva(args, gdp, dev, pk, pk_src)}
    else:
        line = run_ours(args, rank, world, dev)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
