#!/usr/bin/env python3
"""Benchmark of the MMQ hot path on GB300 (one JSON line on rank 0).

A step is one pass of the whole path over one batch: q8_1 activation quantization followed by the
block-quantized GEMM (for W8A8 the GEMM alone; for MoE quantization, routing and the grouped GEMM).
The default workload is the 7B-shaped Q4_0 prefill GEMM (M=2048 tokens, N=4096, K=4096) on seeded
synthetic data.  Timing: W warm-up steps, then K timed steps, each bracketed by CUDA events on the
launching stream, with a 256 MiB write between steps so that L2 (129 MB) starts cold; device time is
the sum of step durations, max over ranks.  `e2e` repeats the step through the C-ABI with the
activations copied from pinned host memory and the output copied back inside the timed region.

--impl reference times the CPU oracle (test infrastructure, plain C) on a bounded sample of the same
workload on the host cores and prints the same line with "impl": "reference".
Multi-GPU (torchrun): every rank runs an independent replica of the workload; value is the sum of
the units all ranks processed over the slowest rank's time ("scaling": "weak").
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from block_quantized_int8_q8_gb300 import synth  # noqa: E402

METRIC = "effective int8 TOPS (2MNK/t) & prefill tok/s per type/shape; % of GB300 int8 peak"
FLUSH_BYTES = 256 << 20


class L2Flush:
    """Leaves L2 (129 MB) cold between timed steps: writes a FLUSH_BYTES buffer, and in "write-read" mode
    then reads a second one of the same size, so that the written buffer's dirty lines are written back
    before the timed step starts instead of while it runs."""

    def __init__(self, dev, mode):
        import torch
        self.mode = mode
        self.wbuf = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.rbuf = torch.ones(FLUSH_BYTES // 4, dtype=torch.int32, device=dev) if mode == "write-read" else None

    def __call__(self):
        import torch
        self.wbuf.zero_()
        if self.rbuf is not None:
            torch.amax(self.rbuf)

    DESCRIBE = {"write-read": "flushed between timed steps (256 MiB write, then 256 MiB read: no dirty lines left)",
                "write": "flushed between timed steps (256 MiB write)"}


FLUSH_MODE = "write-read"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ------------------------------------------------------------------------------------------ helpers
def max_over_ranks(x: float, device=None) -> float:
    """The largest value of x over all ranks (1 rank: x).  The job's time is its slowest replica's."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_step: float, world: int, steps: int, seconds: float) -> float:
    """Whole-job rate: every rank processes units_per_step per step (weak scaling), over the slowest
    rank's time."""
    return units_per_step * world * steps / seconds


def workload_ops(name: str) -> tuple[float, int]:
    """(2*M*N*K of the whole step, tokens per step); MoE counts every (token, slot) row."""
    w = synth.WORKLOADS[name]
    rows = w["M"] * w.get("slots", 1)
    return 2.0 * rows * w["N"] * w["K"], w["M"]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# Source files that define each GEMM kernel (device code and its launch); a change to any of them
# voids the DRAM traffic recorded for that kernel.
KERNEL_SOURCES = {
    "mmq_gemm_tma_kernel": ["gemm_tma.cuh", "gemm_tma.cu", "gemm.cuh", "mmq_device.cuh", "internal.h"],
    "mmq_w8a8_tma_kernel": ["gemm_w8a8_tma.cuh", "gemm_tma.cu", "gemm.cuh", "mmq_device.cuh", "internal.h"],
    "mmq_gemm_kernel": ["gemm.cuh", "gemm_q8_0.cu", "gemm_q4_0.cu", "gemm_q4_k.cu", "gemm_iq1_m.cu",
                        "mmq_device.cuh", "internal.h"],
    "mmvq_kernel": ["gemv.cu", "gemv.h", "gemm.cuh", "mmq_device.cuh", "internal.h"],
}


def kernel_source_hash(kernel: str) -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "block_quantized_int8_q8_gb300", "csrc")
    for fn in sorted(KERNEL_SOURCES[kernel]):
        with open(os.path.join(csrc, fn), "rb") as f:
            h.update(fn.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, kernel: str):
    """DRAM bytes per GEMM launch from the committed ncu summary, if taken on the current kernels."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    ent = rec.get(workload)
    if not ent or ent.get("kernel") != kernel or ent.get("kernel_hash") != kernel_source_hash(kernel):
        return None
    return ent.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling while the timed region runs."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = None

    def start(self):
        try:
            self.path = os.path.join("/tmp", f"mmq_clocks_{os.getpid()}.csv")
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader",
                                          "-lms", "20", "-i", self.gpu_id], stdout=self.out,
                                         stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def mark(self, t0: float, t1: float):
        """Wall-clock window (time.time()) of the timed region; samples outside it are ignored."""
        self.window = (t0, t1)

    def stop(self):
        import datetime
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        sm, mx, pw, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                cols = [c.strip() for c in line.split(",")]
                if len(cols) < 9:
                    continue
                try:
                    ts = datetime.datetime.strptime(cols[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    w = getattr(self, "window", None)
                    if w and not (w[0] - 0.03 <= ts <= w[1] + 0.03):
                        continue
                    sm.append(float(cols[1].split()[0]))
                    mx.append(float(cols[2].split()[0]))
                    pw.append(float(cols[3].split()[0]))
                except ValueError:
                    continue
                for nm, v in zip(names, cols[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(nm)
        os.remove(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None, "reasons": sorted(reasons), "samples": len(sm)}


def gpu_id_for_smi(torch, dev_index: int) -> str:
    try:
        p = torch.cuda.get_device_properties(dev_index)
        uuid = getattr(p, "uuid", None)
        if uuid:
            u = str(uuid)
            return u if u.startswith("GPU-") else "GPU-" + u
        bus = getattr(p, "pci_bus_id", None)
        dom = getattr(p, "pci_domain_id", 0)
        devn = getattr(p, "pci_device_id", 0)
        if bus is not None:
            return f"{dom:08x}:{bus:02x}:{devn:02x}.0"
    except Exception:
        pass
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        return vis.split(",")[dev_index]
    return str(dev_index)


# ------------------------------------------------------------------------------------------ CPU oracle
def oracle_step_sample(pb, rows):
    """One CPU-oracle pass over a sample of token rows (quantize those rows, then the blockwise GEMM)."""
    import oracle
    if pb.wtype == synth.W8A8:
        return oracle.w8a8(pb.fields.W, pb.fields.ws, pb.X[rows], pb.xs[rows])
    q, d, s = oracle.quantize_q8_1(pb.x[rows])
    if pb.ids is not None:
        return oracle.gemm_id(pb.wtype, pb.W, pb.experts, q, d, s, pb.ids[rows], pb.N)
    return oracle.gemm(pb.wtype, pb.W, q, d, s, pb.N)


def cpu_rows_for(pb, target_s: float):
    """Token rows of a sample that takes about target_s seconds on the host cores."""
    # fit t(rows) = fixed (weight decode) + rows * per_row from two probe sizes
    sizes = [min(4, pb.M), min(16, pb.M)]
    ts = []
    for n in sizes:
        t = time.perf_counter()
        oracle_step_sample(pb, list(range(n)))
        ts.append(time.perf_counter() - t)
    per_row = max((ts[1] - ts[0]) / max(sizes[1] - sizes[0], 1), 1e-9) if sizes[1] > sizes[0] else ts[0]
    fixed = max(ts[0] - per_row * sizes[0], 0.0)
    n = int(max(1, min(pb.M, (target_s - fixed) / per_row)))
    return list(range(n))


def cpu_baseline(pb, name, target_s=10.0):
    """The oracle on a bounded sample of the workload: as many token rows as fit in about target_s (all of
    them for the smaller workloads), repeated until about target_s of wall time has been spent."""
    import oracle
    rows = cpu_rows_for(pb, target_s)
    t = time.perf_counter()
    oracle_step_sample(pb, rows)
    first = time.perf_counter() - t
    reps = max(1, min(100, int(target_s / max(first, 1e-3)) - 1))
    t = time.perf_counter()
    for _ in range(reps):
        oracle_step_sample(pb, rows)
    dt = (time.perf_counter() - t) / reps
    ops_full, tokens = workload_ops(name)
    ops = ops_full * len(rows) / pb.M
    return {"value": ops / dt / 1e12, "unit": "TOPS", "cores": oracle.max_threads(), "kind": "oracle",
            "sample": f"{len(rows)} of {pb.M} token rows of {name}, quantize + blockwise GEMM, timed over "
                      f"{reps} passes after one untimed ({dt * reps:.1f} s on the host cores)",
            "tok_per_s": len(rows) / dt}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    pb = synth.workload(args.workload)
    ops_full, tokens = workload_ops(args.workload)
    rows = cpu_rows_for(pb, args.ref_step_s)
    for _ in range(args.warmup):
        oracle_step_sample(pb, rows)
    times = []
    for _ in range(args.steps):
        t = time.perf_counter()
        oracle_step_sample(pb, rows)
        times.append(time.perf_counter() - t)
    ops = ops_full * len(rows) / pb.M
    total = sum(times)
    value = ops * args.steps / total / 1e12
    import oracle
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TOPS", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": total / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8 x q8_1 (CPU oracle)",
            "data": "synthetic", "config": workload_config(args.workload),
            "tok_per_s": len(rows) * args.steps / total,
            "cpu_baseline": {"value": value, "unit": "TOPS", "cores": oracle.max_threads(), "kind": "oracle",
                             "sample": f"{len(rows)} of {pb.M} token rows per step (quantize + blockwise GEMM)"},
            "e2e": {"value": value, "unit": "TOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)
    return 0


def rescale_ceiling(wt, ops, ffma_tflops):
    """FP32-pipe ceiling of the per-block rescale: each 32-k element-block (64 ops of the contraction)
    costs two FP32 instructions (scale product, fused multiply-add), three for Q4_K (min term)."""
    if not ffma_tflops or wt == synth.W8A8:
        return None
    instr = 3 if wt == synth.Q4_K else 2
    fp32_instr_per_s = ffma_tflops * 1e12 / 2
    return {"ffma_tflops": ffma_tflops, "fp32_instr_per_element_block": instr, "element_blocks": ops / 64,
            "ceiling_tops": fp32_instr_per_s / instr * 64 / 1e12}


def workload_config(name):
    w = synth.WORKLOADS[name]
    cfg = {"workload": name, "wtype": synth.TYPE_NAMES[w["wtype"]].upper(), "M_tokens": w["M"], "N": w["N"],
           "K": w["K"], "seed": w["seed"], "l2": L2Flush.DESCRIBE[FLUSH_MODE]}
    if "experts" in w:
        cfg.update(experts=w["experts"], slots=w["slots"])
    return cfg


# ------------------------------------------------------------------------------------------ GPU arm
# ------------------------------------------------------------------------------------------ GPU legs
def setup_workload(name, dev, eager, warmup, flush):
    """Inputs, output and the two legs (quantize; GEMM with MoE routing and gather) of one workload on
    the device, warmed up and, unless eager, captured as CUDA graphs that are replayed every step (every
    kernel runs again on every replay; the L2 flush stays an eager launch between steps)."""
    import torch
    from block_quantized_int8_q8_gb300 import api
    pb = synth.workload(name)
    wt = pb.wtype
    M, N, K = pb.M, pb.N, pb.K
    ops, tokens = workload_ops(name)
    W = torch.from_numpy(pb.W.reshape(-1)).to(dev)
    is_moe = pb.ids is not None
    xq = ids = ws = None
    if wt == synth.W8A8:
        x = torch.from_numpy(synth.pack_w8a8_acts(pb.X, pb.xs)).to(dev)
        out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        launches_per_step = 1
    else:
        x = torch.from_numpy(pb.x).to(dev)
        xq = torch.empty(api.q8_1_bytes(M, K), dtype=torch.uint8, device=dev)
        if is_moe:
            ids = torch.from_numpy(pb.ids).to(dev)
            out = torch.empty((M, pb.ids.shape[1], N), dtype=torch.float32, device=dev)
            ws = torch.empty(api.gemm_id_workspace_bytes(M, K, pb.ids.shape[1], pb.experts), dtype=torch.uint8,
                             device=dev)
            # quantize, routing (one single-block launch up to 65536 rows and 1024 experts, else four),
            # operand gather, grouped GEMM
            small = M * pb.ids.shape[1] <= 65536 and pb.experts <= 1024
            moe_tma = K % 256 == 0 and (wt != synth.IQ1_M or K % 1024 == 0)
            launches_per_step = (4 if small else 7) if moe_tma else 6
            if M <= 8:
                launches_per_step = 2       # quantize, matrix-vector kernel reading the ids itself
        else:
            out = torch.empty((M, N), dtype=torch.float32, device=dev)
            # quantize, GEMM (plus the zeroing of the K-split tail tiles' rows on the tile path)
            launches_per_step = 2

    def gemm_call(xin=None, o=None):
        xin = x if xin is None else xin
        o = out if o is None else o
        if wt == synth.W8A8:
            api.gemm(wt, W, xin, M, N, K, out=o)
        elif is_moe:
            api.gemm_id(wt, W, pb.experts, xq, ids, M, N, K, out=o, workspace=ws)
        else:
            api.gemm(wt, W, xq, M, N, K, out=o)

    def quant_call(xin=None):
        if wt != synth.W8A8:
            api.quantize_q8_1(x if xin is None else xin, out=xq)

    for _ in range(warmup):
        flush()
        quant_call()
        gemm_call()
    torch.cuda.synchronize()
    assert api.read_device_errors() == 0
    run_quant, run_gemm = quant_call, gemm_call
    timed_as = "API calls issued eagerly"
    if not eager:
        def capture(fn):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                fn()
            return g
        try:
            g_gemm = capture(gemm_call)
            g_quant = capture(quant_call) if wt != synth.W8A8 else None
        except RuntimeError as exc:     # keep the measurement: time the eager calls and say why
            print(f"bench: CUDA-graph capture failed ({exc}); timing eager calls", file=sys.stderr)
            torch.cuda.synchronize()
            timed_as = f"API calls issued eagerly (graph capture failed: {str(exc)[:120]})"
        else:
            run_gemm = g_gemm.replay
            if g_quant is not None:
                run_quant = g_quant.replay
            timed_as = "CUDA-graph replay of each leg (quantize; GEMM), every kernel re-run per step"
        for _ in range(2):
            flush()
            run_quant()
            run_gemm()
        torch.cuda.synchronize()
        assert api.read_device_errors() == 0
    tma_path = wt != synth.W8A8 and K % 256 == 0 and (wt != synth.IQ1_M or K % 1024 == 0)
    kernel = "mmq_w8a8_tma_kernel" if wt == synth.W8A8 else ("mmq_gemm_tma_kernel" if tma_path else "mmq_gemm_kernel")
    if wt != synth.W8A8 and M <= 8:
        kernel = "mmvq_kernel"
    return dict(pb=pb, wt=wt, M=M, N=N, K=K, ops=ops, tokens=tokens, x=x, out=out, ids=ids, ws=ws,
                quant_call=quant_call,
                gemm_call=gemm_call, run_quant=run_quant, run_gemm=run_gemm, timed_as=timed_as,
                launches_per_step=launches_per_step, kernel=kernel)


def timed_steps(wl, steps, flush, stream):
    """`steps` timed steps (L2 flush, quantize leg, GEMM leg), CUDA events on the launching stream;
    per-step (step, GEMM, quantize) milliseconds."""
    import torch
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    for i in range(steps):
        flush()
        ev[i][0].record(stream)
        wl["run_quant"]()
        ev[i][1].record(stream)
        wl["run_gemm"]()
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    step_ms = [ev[i][0].elapsed_time(ev[i][2]) for i in range(steps)]
    gemm_ms = [ev[i][1].elapsed_time(ev[i][2]) for i in range(steps)]
    quant_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(steps)]
    return step_ms, gemm_ms, quant_ms


def fewtoken_bytes(wl) -> int:
    """Algorithmic bytes of one matrix-vector launch: the weight rows it reads (a MoE call reads only the
    experts its tokens route to), the q8_1 codes and (d, s) pairs of the M tokens, the f32 outputs."""
    pb, M, N, K = wl["pb"], wl["M"], wl["N"], wl["K"]
    if pb.ids is not None:
        w = len(np.unique(pb.ids)) * (pb.W.nbytes // pb.experts)
        rows = pb.ids.size
    else:
        w, rows = pb.W.nbytes, M
    return int(w + M * K + M * (K // 32) * 8 + rows * N * 4)


def decode_stream(wl, dev, stream, replays=20):
    """Few-token (M <= 8) weights as a decode pass sees them: R layers, each its own copy of the weight
    matrix (the bytes R layers read together at least twice the L2, so every layer's weights come from
    HBM), one CUDA graph of R x (quantize, GEMM) replayed `replays` times between two CUDA events; and the
    same with the GEMMs alone.  No flush is needed: each layer's weights are read once per pass and evicted
    by the others.  A MoE layer reads only the experts its tokens route to."""
    import torch
    from block_quantized_int8_q8_gb300 import api
    pb, wt, M, N, K = wl["pb"], wl["wt"], wl["M"], wl["N"], wl["K"]
    if pb.ids is not None:
        wbytes = len(np.unique(pb.ids)) * (pb.W.nbytes // pb.experts)
    else:
        wbytes = pb.W.nbytes
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or (132 << 20)
    R = int(min(128, max(8, -(-(2 * l2) // wbytes))))
    Ws = [torch.from_numpy(pb.W.reshape(-1)).to(dev) for _ in range(R)]
    x, out = wl["x"], wl["out"]
    xq = torch.empty(api.q8_1_bytes(M, K), dtype=torch.uint8, device=dev)

    def layers(with_quant):
        for W in Ws:
            if with_quant:
                api.quantize_q8_1(x, out=xq)
            if pb.ids is not None:
                api.gemm_id(wt, W, pb.experts, xq, wl["ids"], M, N, K, out=out, workspace=wl["ws"])
            else:
                api.gemm(wt, W, xq, M, N, K, out=out)

    res = {"layers": R, "weight_bytes_per_layer": wbytes, "replays": replays}
    for key, wq in (("layer_us", True), ("gemm_us", False)):
        layers(wq)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            layers(wq)
        for _ in range(3):
            g.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(replays):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        res[key] = e0.elapsed_time(e1) * 1e3 / (replays * R)
        del g
    res["gemm_weight_GBps"] = wbytes / (res["gemm_us"] * 1e-6) / 1e9
    del Ws
    torch.cuda.empty_cache()
    return res


def workloads_block(dev, stream, flush, steps, warmup, peak, eager, gpu_id):
    """Every workload of the suite (the five configurations, W8A8 at both token counts, the dense IQ1_M
    shape and q6_K) timed with the headline's protocol, `steps` steps each."""
    import torch
    from block_quantized_int8_q8_gb300 import api
    res = {}
    sampler = ClockSampler(gpu_id)
    sampler.start()
    tw0 = time.time()
    for name in synth.WORKLOADS:
        wl = setup_workload(name, dev, eager, warmup, flush)
        step_ms, gemm_ms, quant_ms = timed_steps(wl, steps, flush, stream)
        errs = api.read_device_errors()
        step = statistics.mean(step_ms) / 1e3
        gemm = statistics.mean(gemm_ms) / 1e3
        res[name] = {"config": workload_config(name), "kernel": wl["kernel"],
                     "step_tops": wl["ops"] / step / 1e12, "gemm_only_tops": wl["ops"] / gemm / 1e12,
                     "step_ms": step * 1e3, "gemm_ms": gemm * 1e3, "quantize_ms": statistics.mean(quant_ms),
                     "tok_per_s": wl["tokens"] / step, "frac_of_peak": wl["ops"] / gemm / 1e12 / peak,
                     "steps": steps, "device_errors": errs}
        del wl
        torch.cuda.empty_cache()
    sampler.mark(tw0, time.time())
    return res, sampler.stop()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["mmq", "reference"], default="mmq")
    ap.add_argument("--workload", choices=sorted(synth.WORKLOADS), default="q4_0_7b")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--flush", choices=["write", "write-read"], default="write-read",
                    help="L2 flush between timed steps: a 256 MiB write, optionally followed by a 256 MiB read")
    ap.add_argument("--workload-steps", type=int, default=100,
                    help="timed steps per workload of the 'workloads' block (0: leave the block out)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-step-s", type=float, default=2.0)
    ap.add_argument("--cpu-baseline-s", type=float, default=10.0)
    ap.add_argument("--eager", action="store_true",
                    help="time the API calls as issued from Python instead of CUDA-graph replays of each leg")
    ap.add_argument("--tokens", type=int, default=0,
                    help="token count M in place of the workload's (same weights and K; a token-count study)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.tokens > 0:
        # a derived workload: the named one with M tokens (same weights, K, seed and routing recipe)
        derived = f"{args.workload}_m{args.tokens}"
        synth.WORKLOADS[derived] = dict(synth.WORKLOADS[args.workload], M=args.tokens)
        args.workload = derived

    if args.impl == "reference":
        return run_reference(args)

    import torch
    import torch.distributed as dist
    from block_quantized_int8_q8_gb300 import _build, api

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    _build.build()
    api.load()

    name = args.workload
    global FLUSH_MODE
    FLUSH_MODE = args.flush
    flush = L2Flush(dev, args.flush)
    stream = torch.cuda.current_stream()
    wl = setup_workload(name, dev, args.eager, args.warmup, flush)
    pb, wt, M, N, K = wl["pb"], wl["wt"], wl["M"], wl["N"], wl["K"]
    ops, tokens = wl["ops"], wl["tokens"]
    x, out, quant_call, gemm_call = wl["x"], wl["out"], wl["quant_call"], wl["gemm_call"]
    timed_as, launches_per_step = wl["timed_as"], wl["launches_per_step"]

    # ---------------------------------------------------------------- timed region
    K_steps = args.steps
    sampler = ClockSampler(gpu_id_for_smi(torch, local))
    sampler.start()
    time.sleep(0.15)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    tw0 = time.time()
    step_ms, gemm_ms, quant_ms = timed_steps(wl, K_steps, flush, stream)
    if world > 1:
        dist.barrier()
    wall = time.perf_counter() - wall0
    sampler.mark(tw0, time.time())
    clocks = sampler.stop()
    dev_total = max_over_ranks(sum(step_ms) / 1e3, dev)
    errs = api.read_device_errors()

    # ---------------------------------------------------------------- end to end through the C ABI
    e2e = None
    if args.e2e_steps > 0:
        if wt == synth.W8A8:
            host_in = torch.from_numpy(synth.pack_w8a8_acts(pb.X, pb.xs)).pin_memory()
        else:
            host_in = torch.from_numpy(pb.x).pin_memory()
        host_out = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
        # Steps pipelined over two device buffer sets: step i's input copy (copy stream) and step i-1's
        # result copy (second copy stream) overlap the compute of the step before; every step still
        # copies its whole input in and its whole result out inside the timed region.
        xs_dev = [x, torch.empty_like(x)]
        outs_dev = [out, torch.empty_like(out)]
        s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        ev_in = [torch.cuda.Event() for _ in range(2)]      # input copy landed
        ev_used = [torch.cuda.Event() for _ in range(2)]    # compute no longer reads the input buffer
        ev_res = [torch.cuda.Event() for _ in range(2)]     # result written
        ev_drained = [torch.cuda.Event() for _ in range(2)] # result copied out

        def pipelined(n):
            for i in range(n):
                b = i & 1
                with torch.cuda.stream(s_in):
                    if i >= 2:
                        s_in.wait_event(ev_used[b])
                    xs_dev[b].copy_(host_in, non_blocking=True)
                    ev_in[b].record(s_in)
                stream.wait_event(ev_in[b])
                if i >= 2:
                    stream.wait_event(ev_drained[b])
                quant_call(xs_dev[b])
                if wt != synth.W8A8:
                    ev_used[b].record(stream)
                gemm_call(xs_dev[b], outs_dev[b])
                if wt == synth.W8A8:
                    ev_used[b].record(stream)
                ev_res[b].record(stream)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(ev_res[b])
                    host_out[b].copy_(outs_dev[b], non_blocking=True)
                    ev_drained[b].record(s_out)
            for b in range(min(n, 2)):
                stream.wait_event(ev_drained[b])

        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        pipelined(2)
        torch.cuda.synchronize()
        e0.record(stream)
        s_in.wait_event(e0)
        pipelined(args.e2e_steps)
        e1.record(stream)
        torch.cuda.synchronize()
        assert torch.equal(outs_dev[(args.e2e_steps - 1) & 1].cpu(), host_out[(args.e2e_steps - 1) & 1]), \
            "pipelined result copy differs from the device result"
        e2e_s = max_over_ranks(e0.elapsed_time(e1) / 1e3, dev)
        e2e = {"value": job_throughput(ops, world, args.e2e_steps, e2e_s) / 1e12, "unit": "TOPS",
               "h2d_bytes_per_step": host_in.numel() * host_in.element_size(),
               "d2h_bytes_per_step": host_out[0].numel() * host_out[0].element_size(),
               "steps": args.e2e_steps,
               "note": "weights resident in HBM; activations in, outputs out (pinned host buffers), steps "
                       "pipelined: input copy, compute and result copy of consecutive steps overlap"}

    # ---------------------------------------------------------------- roofline and peaks
    peaks, peak_src = measured_peaks()
    gemm_avg = statistics.mean(gemm_ms) / 1e3
    achieved = ops / gemm_avg / 1e12
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    # the block types run the TMA-fed kernel (dense and MoE; IQ1_M when K % 1024 == 0; the matrix-vector
    # kernel for eight tokens or fewer), W8A8 its own TMA-fed kernel; the remaining shapes the general kernel
    kernel = wl["kernel"]
    roofline = {"bound": "tensor", "kernel": kernel, "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak, "traffic": recorded_traffic(name, kernel),
                "peak_source": f"{peak_src} dense bf16 burst (fp16 operands, same nominal rate)",
                "flops_per_launch": ops}
    if kernel == "mmvq_kernel":
        # a few tokens: every weight byte is used M times at most, the kernel is bound by reading them
        hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
        nbytes = fewtoken_bytes(wl)
        roofline.update(bound="hbm", achieved=nbytes / gemm_avg / 1e9, peak=hbm, unit="GB/s",
                        frac=nbytes / gemm_avg / 1e9 / hbm, peak_source=f"{peak_src} HBM copy bandwidth",
                        bytes_per_launch=nbytes)
        roofline.pop("flops_per_launch")
    int8_peak = ffma = None
    try:
        import ctypes
        plib = ctypes.CDLL(_build.PEAKS_LIB)
        plib.mmq_peak_int8_mma_sync.argtypes = [ctypes.POINTER(ctypes.c_double), ctypes.c_int, ctypes.c_void_p]
        plib.mmq_peak_ffma.argtypes = [ctypes.POINTER(ctypes.c_double), ctypes.c_int, ctypes.c_void_p]
        v = ctypes.c_double(0)
        if plib.mmq_peak_int8_mma_sync(ctypes.byref(v), 4096, ctypes.c_void_p(stream.cuda_stream)) == 0:
            int8_peak = v.value
        if plib.mmq_peak_ffma(ctypes.byref(v), 4096, ctypes.c_void_p(stream.cuda_stream)) == 0:
            ffma = v.value
    except OSError:
        pass

    value = job_throughput(ops, world, K_steps, dev_total) / 1e12
    line = {"metric": METRIC, "value": value, "unit": "TOPS", "n_gpus": world, "steps": K_steps,
            "warmup": args.warmup, "ms_per_step": dev_total / K_steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "s8 x s8 -> exact block dot (fp16 tensor cores, f32 accumulate), f32 rescale",
            "data": "synthetic",
            "config": workload_config(name), "timing": timed_as,
            "tok_per_s": job_throughput(tokens, world, K_steps, dev_total),
            # context, not the roofline: the GEMM runs on the fp16 tensor pipe (roofline above); this is the
            # rate of the legacy warp-level int8 MMA, the only int8 tensor instruction sm_103a keeps
            "legacy_int8_mma_sync": {"tops": int8_peak, "step_pct_of_it": (100.0 * value / world / int8_peak)
                                     if int8_peak else None,
                                     "source": "measured live: mma.sync.m16n8k32.s8 throughput probe"},
            "gemm_ms": statistics.mean(gemm_ms), "quantize_ms": statistics.mean(quant_ms),
            "gemm_only_tops": ops / gemm_avg / 1e12,
            "roofline": roofline,
            "rescale_ceiling": rescale_ceiling(wt, ops, ffma),
            "e2e": e2e, "gpu_launches": launches_per_step * K_steps, "clocks": clocks,
            "wall_s": wall, "device_errors": errs}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:   # the oracle baseline is a one-GPU figure
        line["cpu_baseline"] = cpu_baseline(pb, name, args.cpu_baseline_s)
    if world == 1 and wl["kernel"] == "mmvq_kernel":
        line["decode_stream"] = decode_stream(wl, dev, stream)
    if world == 1 and args.workload_steps > 0:
        # every configuration, timed after the headline with the same protocol (one GPU)
        del wl, x, out
        torch.cuda.empty_cache()
        line["workloads"], line["workloads_clocks"] = workloads_block(
            dev, stream, flush, args.workload_steps, args.warmup, peak, args.eager, gpu_id_for_smi(torch, local))
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
