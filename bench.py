#!/usr/bin/env python3
"""Benchmark of the keep-quant GEMV / MoE routed-expert path (libggq) on GB300.

Headline workload (one "step"): the non-grouped K-quant GEMV, W = 14336 x 4096
in each of Q8_0, Q4_K, Q5_K and Q6_K, at 1, 2, 4 and 8 tokens (16 GEMVs; x is
quantized to Q8_K once per token count and shared by the four formats).
Metric: packed weight bytes streamed per second (GB/s) and its fraction of the
measured HBM copy bandwidth.  Each format has 8 weight copies; one step reads
a different copy for each token count, so no copy is read twice within a step
(736 MB per step, 1.47 GB live, far larger than the 129 MB L2).  The step is
captured once in a CUDA graph and replayed.

Roofline of the GEMV kernels: each (format, token count) GEMV is timed as a
chain of 8 back-to-back launches over the 8 copies (one captured graph, CUDA
events around its replays), so a launch's duration includes its share of the
launch boundaries as it runs inside a decode step; the same launches timed one
by one with events around each (which breaks the overlap of consecutive
launches) are reported beside it.

Secondary lines (same JSON, "workloads"): the Q4_0 1024 x 4096 GEMV, the
4096 x 14336 long-row GEMV (Q8_0, Q6_K at 1 and 8 tokens), the Q2_K and Q3_K
GEMV on the 14336 x 4096 shape (1 and 8 tokens), the MoE decode
layer (128 experts, H 2048, I 768, Q4_K gate/up, Q6_K down, top-8, 1-4
tokens), the MXFP4 routed experts (256 experts, H 4096, I 2048, top-8, 1-512
tokens) and the 4096-token prefill layer; MoE GB/s counts the distinct
experts actually selected.  From 5 tokens the MoE lines run the workloads'
own route (expert-sorted tiles); where the library's default differs (direct
calls of 4 tokens, up to 32 tokens), a "_direct4" line times that beside it.

--impl reference times the CPU oracle on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import ctypes
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

import ggq_synth as syn  # noqa: E402

KQ = syn.GEMV_KQUANT
FMTS = KQ["fmts"]
TOKENS = KQ["T"]
N, K = KQ["N"], KQ["K"]
ROTATE = 8
CHAIN = 8  # launches per timed chain of one GEMV
METRIC = "decode GEMV/MoE packed-weight GB/s (% of HBM); prefill expert GEMM int8 TOPS"


TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic_kquant_gemv_step.json")


# sources of the decode GEMV kernels (k_stream, k_gemv_mma) that the stored traffic was taken on
GEMV_SOURCES = ("ggq_device.cuh", "ggq_stream.cuh", "ggq_mmav.cuh", "ggq_k_gemv_a.cu", "ggq_k_gemv_b.cu", "ggq_k_mmav.cu",
                "ggq_internal.h", "ggq_plan.h")


def _code_only(text):
    """Source text without comments and with whitespace runs collapsed, so that
    documentation edits leave the hash (and the stored measurement) valid."""
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def csrc_hash():
    """Hash of the GEMV kernel code (comments excluded): a stored DRAM-traffic
    figure applies only to the kernels it was taken on."""
    import hashlib
    d = os.path.join(ROOT, "gguf_block_quant_ggq_gb300", "csrc")
    h = hashlib.sha256()
    for f in GEMV_SOURCES:
        with open(os.path.join(d, f), encoding="utf-8") as fh:
            h.update(f.encode() + b"\0" + _code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def stored_traffic():
    """Mean DRAM bytes (read + write) per GEMV launch of one step, from the ncu summary, or None if stale."""
    try:
        with open(TRAFFIC_FILE) as f:
            t = json.load(f)
        return float(t["mean_traffic_bytes"]) if t.get("csrc_hash") == csrc_hash() else None
    except Exception:
        return None


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def tensor_peak():
    """Dense 16-bit tensor peak in TFLOP/s (measured cuBLAS bf16 burst; f16 runs at the same rate)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


# ----------------------------------------------------------------- CUDA runtime (events in graphs)

class Cudart:
    def __init__(self):
        self.lib = None
        for name in ("libcudart.so.13", "libcudart.so", "/usr/local/cuda/lib64/libcudart.so"):
            try:
                self.lib = ctypes.CDLL(name)
                break
            except OSError:
                continue
        if self.lib is None:
            raise RuntimeError("libcudart not found")
        self.lib.cudaEventElapsedTime.argtypes = [ctypes.POINTER(ctypes.c_float), ctypes.c_void_p, ctypes.c_void_p]
        self.lib.cudaEventRecordWithFlags.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint]
        self.lib.cudaEventSynchronize.argtypes = [ctypes.c_void_p]

    def event(self):
        e = ctypes.c_void_p()
        assert self.lib.cudaEventCreate(ctypes.byref(e)) == 0
        return e

    def record(self, ev, stream, external=False):
        rc = self.lib.cudaEventRecordWithFlags(ev, ctypes.c_void_p(stream.cuda_stream), 1 if external else 0)
        if rc != 0:
            raise RuntimeError(f"cudaEventRecordWithFlags rc={rc}")

    def elapsed_ms(self, a, b):
        self.lib.cudaEventSynchronize(b)
        ms = ctypes.c_float()
        rc = self.lib.cudaEventElapsedTime(ctypes.byref(ms), a, b)
        if rc != 0:
            raise RuntimeError(f"cudaEventElapsedTime rc={rc}")
        return ms.value


# ----------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index=0):
        self.proc = None
        self.lines = []
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm), "power_w_max": max(power) if power else None}


# ----------------------------------------------------------------- distributed plumbing

def dist_init(n_gpus):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("gloo", rank=rank, world_size=world)
    return rank, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world):
    if world <= 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbps(bytes_per_rank_step, world, ms_per_step):
    """Whole-job throughput: every rank streams the same per-step bytes (weak
    scaling, independent replicas), divided by the slowest rank's time."""
    return bytes_per_rank_step * world / (ms_per_step / 1e3) / 1e9


# ----------------------------------------------------------------- CPU oracle timing

def oracle_sample_rate(target_s=12.0):
    """The oracle's integer-dot GEMV over the headline workload, on a row
    sample sized for ~target_s seconds on all host cores.  Returns (GB/s of
    packed weights, cores, sample description, seconds)."""
    import oracle as orc
    cores = os.cpu_count() or 1
    orc.set_threads(cores)
    g = syn.rng(KQ["index"], 900)
    xq = {T: orc.quantize("Q8_K", syn.activations(T, K, g)) for T in TOKENS}
    probe_rows = 64
    Wp = {f: syn.weights(f, probe_rows, K, g) for f in FMTS}
    t0 = time.perf_counter()
    for f in FMTS:
        for T in TOKENS:
            orc.gemv(f, Wp[f], probe_rows, K, xq[T], T)
    dt = time.perf_counter() - t0
    rows = int(max(probe_rows, min(N, probe_rows * target_s / max(dt, 1e-6))))
    W = {f: syn.weights(f, rows, K, g) for f in FMTS}
    reps = 0
    t0 = time.perf_counter()
    while True:  # whole passes over the sample until ~target_s / 2 of CPU time
        for f in FMTS:
            for T in TOKENS:
                orc.gemv(f, W[f], rows, K, xq[T], T)
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= target_s / 2 or reps >= 50:
            break
    nbytes = sum(rows * syn.row_bytes(f, K) for f in FMTS) * len(TOKENS) * reps
    sample = (f"{rows} of {N} rows of each of Q8_0/Q4_K/Q5_K/Q6_K (K={K}) at T=1,2,4,8, {reps} pass(es): "
              f"{nbytes / 1e6:.1f} MB of packed weights, oracle integer-dot GEMV, {cores} OpenMP threads")
    return nbytes / dt / 1e9, orc.threads(), sample, dt, rows


def run_reference(args, rank, world):
    if rank != 0:
        return
    import oracle as orc
    orc.build()
    cores = os.cpu_count() or 1
    orc.set_threads(cores)
    g = syn.rng(KQ["index"], 900)
    xq = {T: orc.quantize("Q8_K", syn.activations(T, K, g)) for T in TOKENS}
    # bounded sample: each step is 256 rows of every matrix, all token counts
    rows = 256
    W = {f: syn.weights(f, rows, K, g) for f in FMTS}

    def step():
        for f in FMTS:
            for T in TOKENS:
                orc.gemv(f, W[f], rows, K, xq[T], T)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    nbytes = sum(rows * syn.row_bytes(f, K) for f in FMTS) * len(TOKENS)
    value = nbytes * args.steps / dt / 1e9
    sample = (f"{rows} of {N} rows per matrix per step (Q8_0/Q4_K/Q5_K/Q6_K, K={K}, T=1,2,4,8), "
              f"{nbytes / 1e6:.2f} MB packed weights per step")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8 dot, f64 epilogue",
        "data": "synthetic (seeded)",
        "config": {"workload": "kquant_gemv_14336x4096_T1-2-4-8 (CPU oracle, row sample)", "sample": sample},
        "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": orc.threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------- GPU arm

def run_gpu(args, rank, world):
    import torch

    import gguf_block_quant_ggq_gb300 as ggq
    from gguf_block_quant_ggq_gb300 import _build

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    _build.build()
    ctx = ggq.Context(local)
    rt = Cudart()
    hbm_peak, peak_kind = peaks()

    # ---- inputs (seeded; per-rank replica: same workload on every GPU)
    Wdev = {}
    for fi, f in enumerate(FMTS):
        g = syn.rng(KQ["index"], 10 + fi)
        w0 = torch.from_numpy(syn.weights(f, N, K, g)).cuda()
        Wdev[f] = [w0] + [w0.clone() for _ in range(ROTATE - 1)]  # distinct addresses, same bytes
    gx = syn.rng(KQ["index"], 200)
    x_host = {T: torch.from_numpy(syn.activations(T, K, gx)).pin_memory() for T in TOKENS}
    x_dev = {T: x_host[T].cuda() for T in TOKENS}
    xq_dev = {T: torch.empty((T, syn.row_bytes("Q8_K", K)), dtype=torch.uint8, device="cuda") for T in TOKENS}
    y_dev = {(f, T): torch.empty((T, N), dtype=torch.float32, device="cuda") for f in FMTS for T in TOKENS}
    ctx.reserve(max_tokens=8, max_k=K)
    # each token count reads its own copy of every format: nothing is re-read within a step
    plan = []
    for f in FMTS:
        for c, T in enumerate(TOKENS):
            plan.append((f, T, c))
    wbytes = {f: N * syn.row_bytes(f, K) for f in FMTS}
    step_wbytes = sum(wbytes[f] for f, _, _ in plan)
    # algorithmic bytes of one GEMV launch: packed W + quantized x + fp32 y
    alg_bytes = {(f, T): wbytes[f] + T * syn.row_bytes("Q8_K", K) + T * N * 4 for f in FMTS for T in TOKENS}

    kev = [(rt.event(), rt.event()) for _ in plan]
    stream = torch.cuda.Stream()
    ctx.set_static_weights(True)  # weights are never written while calls run: kernels overlap

    def step(events):
        s = torch.cuda.current_stream()
        for T in TOKENS:
            ctx.quantize_act("Q8_K", x_dev[T], out=xq_dev[T])
        for j, (f, T, c) in enumerate(plan):
            if events:
                rt.record(kev[j][0], s, True)
            ctx.mul_mat_vec_q(f, Wdev[f][c], N, K, xq_dev[T], T, Y=y_dev[(f, T)])
            if events:
                rt.record(kev[j][1], s, True)

    # eager warm-up (sets kernel attributes outside capture), then capture the
    # step twice: plain (timed; consecutive kernels overlap through programmatic
    # dependent launch) and with an event pair around every GEMV (kernel times)
    with torch.cuda.stream(stream):
        for _ in range(2):
            step(False)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step(False)
    graph_ev = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph_ev, stream=stream):
        step(True)
    torch.cuda.synchronize()

    t_ev = (rt.event(), rt.event())
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    barrier(world)
    clocks = ClockSampler(local)
    time.sleep(0.3)
    torch.cuda.synchronize()
    rt.record(t_ev[0], stream)
    with torch.cuda.stream(stream):
        for _ in range(args.steps):
            graph.replay()
    rt.record(t_ev[1], stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    barrier(world)
    total_ms = max_over_ranks(rt.elapsed_ms(*t_ev), world)
    ms_per_step = total_ms / args.steps
    value = job_gbps(step_wbytes, world, ms_per_step)

    # isolated launches: events around every GEMV inside the second graph, median of 5 replays
    samples = {k: [] for k in plan}
    with torch.cuda.stream(stream):
        for _ in range(5):
            graph_ev.replay()
            torch.cuda.synchronize()
            for j, key in enumerate(plan):
                samples[key].append(rt.elapsed_ms(*kev[j]))
    isolated = {(f, T): statistics.median(samples[(f, T, c)]) for (f, T, c) in plan}
    # kernel durations in a chain: CHAIN back-to-back launches of one GEMV over the
    # copies (> 2x L2 between reuses), one captured graph, events around 5 replays
    chain = {}
    for f in FMTS:
        for T in TOKENS:
            def one_chain(f=f, T=T):
                for c in range(CHAIN):
                    ctx.mul_mat_vec_q(f, Wdev[f][c % ROTATE], N, K, xq_dev[T], T, Y=y_dev[(f, T)])
            chain[(f, T)] = _graph_time(one_chain, 5, rt, stream) / CHAIN
    sum_alg = sum(alg_bytes[k] for k in chain)
    sum_ms = sum(chain.values())
    achieved = sum_alg / (sum_ms / 1e3) / 1e9
    iso_achieved = sum_alg / (sum(isolated.values()) / 1e3) / 1e9
    # which kernel the library runs for (format, tokens): the dp4a streaming kernel at
    # one token and, for Q8_0 and Q5_K, at two; the tensor-path GEMV otherwise
    streamed = [k for k in chain if k[1] <= 2]
    fam = {"k_gemv_mma": [k for k in chain if k not in streamed], "k_stream": streamed}
    families = {name: round(sum(alg_bytes[k] for k in ks) / (sum(chain[k] for k in ks) / 1e3) / 1e9 / hbm_peak, 4)
                for name, ks in fam.items()}
    breakdown = {f"{f}_T{T}": {"us": round(ms * 1e3, 2), "GBps": round(alg_bytes[(f, T)] / (ms / 1e3) / 1e9, 1),
                               "isolated_us": round(isolated[(f, T)] * 1e3, 2)}
                 for (f, T), ms in chain.items()}

    # ---- end to end through the public API with host buffers: the step's inputs
    # (every token count's x, one pinned buffer) in one host-to-device copy, the
    # step's calls (ggq_quantize_act per token count, ggq_mul_mat_vec_q per GEMV),
    # and all 16 outputs (one device buffer) back in one device-to-host copy
    rows_x = sum(TOKENS)
    xh_all = torch.empty((rows_x, K), dtype=torch.float32).pin_memory()
    xd_all = torch.empty((rows_x, K), dtype=torch.float32, device="cuda")
    xh, xd, r = {}, {}, 0
    for T in TOKENS:
        xh[T], xd[T] = xh_all[r:r + T], xd_all[r:r + T]
        xh[T].copy_(x_host[T])
        r += T
    yd_all = torch.empty((len(FMTS) * rows_x, N), dtype=torch.float32, device="cuda")
    yh_all = torch.empty((len(FMTS) * rows_x, N), dtype=torch.float32).pin_memory()
    yd, r = {}, 0
    for f in FMTS:
        for T in TOKENS:
            yd[(f, T)] = yd_all[r:r + T]
            r += T
    h2d = xh_all.numel() * 4
    d2h = yh_all.numel() * 4

    def e2e_step():
        xd_all.copy_(xh_all, non_blocking=True)
        for T in TOKENS:
            ctx.quantize_act("Q8_K", xd[T], out=xq_dev[T])
        for (f, T, c) in plan:
            ctx.mul_mat_vec_q(f, Wdev[f][c], N, K, xq_dev[T], T, Y=yd[(f, T)])
        yh_all.copy_(yd_all, non_blocking=True)

    ctx.set_static_weights(False)  # the public call as a generic caller makes it
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            e2e_step()
        torch.cuda.synchronize()
        e_ev = (rt.event(), rt.event())
        rt.record(e_ev[0], stream)
        for _ in range(args.steps):
            e2e_step()
        rt.record(e_ev[1], stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(rt.elapsed_ms(*e_ev), world) / args.steps
    e2e_value = job_gbps(step_wbytes, world, e2e_ms)
    ctx.sync_status()

    # ---- secondary workloads (1 GPU lines, rank 0 only)
    workloads = {}
    if rank == 0 and not args.headline_only:
        workloads = secondary_workloads(ctx, rt, hbm_peak)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, cores, sample, secs, _ = oracle_sample_rate()
        cpu = {"value": round(v, 4), "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample,
               "seconds": round(secs, 2)}

    gpu_launches = (len(TOKENS) + len(plan)) * args.steps  # 4 quantize + 16 GEMV kernels per step
    traffic = stored_traffic()
    if traffic is not None:
        traffic = round(traffic)
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "int8 (dp4a, int8 mma) and f16 mma on integer-valued operands; f32 scales",
            "data": "synthetic (seeded)",
            "config": {"workload": "kquant_gemv_14336x4096_Q8_0-Q4_K-Q5_K-Q6_K_T1-2-4-8",
                       "packed_weight_bytes_per_step": step_wbytes,
                       "l2": f"inputs larger than L2: {ROTATE} copies per format ({sum(wbytes.values()) * ROTATE / 1e6:.0f} "
                             "MB live), each read once per step, no L2 flush",
                       "graph": "one step captured in a CUDA graph, replayed",
                       "fraction_of_hbm": round(value / world / hbm_peak, 4), "peak": f"{hbm_peak} GB/s ({peak_kind})"},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                         "frac": round(achieved / hbm_peak, 4), "traffic": traffic,
                         "algorithmic_bytes_per_launch": round(sum_alg / len(chain)),
                         "kernel": "decode GEMV kernels (k_stream dp4a at T=1 and 2, k_gemv_mma tensor "
                                   "path at T=4 and 8): "
                                   "all 16 launches of a step; algorithmic bytes = packed W + Q8_K x + fp32 y",
                         "traffic_source": "mean dram__bytes_read.sum + dram__bytes_write.sum per GEMV launch of "
                                           "one step (ncu; profiles/traffic_kquant_gemv_step.json), null when the "
                                           "kernel sources changed since",
                         "timing": f"average launch duration in a chain of {CHAIN} back-to-back launches of each "
                                   "GEMV (CUDA events around 5 replays of the captured chain on its stream)",
                         "frac_by_kernel": families,
                         "isolated_frac": round(iso_achieved / hbm_peak, 4),
                         "isolated_timing": "CUDA events around each GEMV inside the captured step (no overlap "
                                            "with the neighbouring launches), median of 5 replays",
                         "peak_kind": peak_kind, "per_launch": breakdown},
            "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4)},
            "gpu_launches": gpu_launches,
            "clocks": clk,
            "cpu_baseline": cpu,
            "workloads": workloads,
        }
        print(json.dumps(line), flush=True)
    ctx.close()


def _moe_route(T, E, k):
    """The route ggq_moe_experts takes by default: one direct launch pair up to
    4 tokens, direct calls of 4 tokens up to 32 tokens while the pairs number
    at most 2 E, else expert-sorted tiles."""
    if T <= 4:
        return "direct"
    return "direct, calls of 4 tokens" if T <= 32 and T * k <= 2 * E else "expert-sorted"


def _graph_time(fn, reps, rt, stream, warm=2):
    """Capture fn() once; return the mean ms of one replay over `reps` replays."""
    import torch
    with torch.cuda.stream(stream):
        for _ in range(warm):
            fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    torch.cuda.synchronize()
    for _ in range(3):
        g.replay()
    ev = (rt.event(), rt.event())
    torch.cuda.synchronize()
    rt.record(ev[0], stream)
    with torch.cuda.stream(stream):
        for _ in range(reps):
            g.replay()
    rt.record(ev[1], stream)
    torch.cuda.synchronize()
    return rt.elapsed_ms(*ev) / reps


def secondary_workloads(ctx, rt, hbm_peak):
    import torch

    out = {}
    stream = torch.cuda.Stream()
    # Q4_0 1024 x 4096, T = 1: 64 rotating copies (151 MB) per replay
    cfg = syn.GEMV_Q4_0
    Nq, Kq = cfg["N"], cfg["K"]
    gq = syn.rng(cfg["index"], 0)
    copies = [torch.from_numpy(syn.weights("Q4_0", Nq, Kq, gq)).cuda() for _ in range(64)]
    xq4 = torch.from_numpy(syn.activations(1, Kq, syn.rng(cfg["index"], 1))).cuda()
    y4 = torch.empty((1, Nq), dtype=torch.float32, device="cuda")
    ctx.reserve(max_tokens=1, max_k=Kq)

    def q4():
        for Wc in copies:
            ctx.mul_mat_vec("Q4_0", Wc, Nq, Kq, xq4, Y=y4, reserve=False)

    ms = _graph_time(q4, 5, rt, stream)
    bytes_ = len(copies) * Nq * syn.row_bytes("Q4_0", Kq)
    out["q4_0_gemv_1024x4096_T1"] = {"GBps": round(bytes_ / (ms / 1e3) / 1e9, 1),
                                     "frac": round(bytes_ / (ms / 1e3) / 1e9 / hbm_peak, 4),
                                     "us_per_call": round(ms * 1e3 / len(copies), 2)}
    del copies

    # long rows: the 4096 x 14336 down-projection shape at T = 1 and 8 (rows of
    # 15232 B in Q8_0, 11760 B in Q6_K stream in row chunks); 3 rotating copies
    ctx.set_static_weights(True)
    NL, KL = 4096, 14336
    ctx.reserve(max_tokens=8, max_k=KL)
    for fmt in ("Q8_0", "Q6_K"):
        gl = syn.rng(KQ["index"], 300 + FMTS.index(fmt))
        lcopies = [torch.from_numpy(syn.weights(fmt, NL, KL, gl)).cuda() for _ in range(3)]
        for T in (1, 8):
            xl = torch.from_numpy(syn.activations(T, KL, gl)).cuda()
            yl = torch.empty((T, NL), dtype=torch.float32, device="cuda")
            xql = torch.empty((T, syn.row_bytes("Q8_K", KL)), dtype=torch.uint8, device="cuda")
            ctx.quantize_act("Q8_K", xl, out=xql)
            torch.cuda.synchronize()

            def longrow():
                for Wc in lcopies:
                    ctx.mul_mat_vec_q(fmt, Wc, NL, KL, xql, T, Y=yl)

            ms = _graph_time(longrow, 10, rt, stream)
            bytes_ = len(lcopies) * NL * syn.row_bytes(fmt, KL)
            out[f"{fmt.lower()}_gemv_{NL}x{KL}_T{T}"] = {
                "GBps": round(bytes_ / (ms / 1e3) / 1e9, 1), "frac": round(bytes_ / (ms / 1e3) / 1e9 / hbm_peak, 4),
                "us_per_call": round(ms * 1e3 / len(lcopies), 2)}
        del lcopies

    # the 2- and 3-bit K-quants on the headline shape (14336 x 4096) at T = 1 and 8
    # (the dp4a streaming kernel at every token count); 4 rotating copies > 2x L2
    ctx.set_static_weights(True)
    N2, K2 = syn.GEMV_KQUANT["N"], syn.GEMV_KQUANT["K"]
    ctx.reserve(max_tokens=8, max_k=K2)
    for fmt in ("Q2_K", "Q3_K"):
        g2 = syn.rng(syn.GEMV_KQUANT["index"], 400 + syn.WEIGHT_FORMATS.index(fmt))
        lc = [torch.from_numpy(syn.weights(fmt, N2, K2, g2)).cuda() for _ in range(4)]
        for T in (1, 8):
            x2 = torch.from_numpy(syn.activations(T, K2, g2)).cuda()
            xq2 = torch.empty((T, syn.row_bytes("Q8_K", K2)), dtype=torch.uint8, device="cuda")
            ctx.quantize_act("Q8_K", x2, out=xq2)
            y2 = torch.empty((T, N2), dtype=torch.float32, device="cuda")
            torch.cuda.synchronize()

            def lowbit():
                for Wc in lc:
                    ctx.mul_mat_vec_q(fmt, Wc, N2, K2, xq2, T, Y=y2)

            ms = _graph_time(lowbit, 10, rt, stream)
            bytes_ = len(lc) * N2 * syn.row_bytes(fmt, K2)
            out[f"{fmt.lower()}_gemv_{N2}x{K2}_T{T}"] = {
                "GBps": round(bytes_ / (ms / 1e3) / 1e9, 1), "frac": round(bytes_ / (ms / 1e3) / 1e9 / hbm_peak, 4),
                "us_per_call": round(ms * 1e3 / len(lc), 2)}
        del lc
    torch.cuda.empty_cache()

    # MoE layers: rotate seeded router-logit sets so the expert sets differ per call
    ctx.set_static_weights(True)
    for cfg, E, Ts in ((syn.MOE_DECODE, syn.MOE_DECODE["E"], (1, 2, 3, 4)),
                       (syn.MOE_MXFP4, syn.MOE_MXFP4["E"], (1, 2, 3, 4, 5, 32, 128, 512)),
                       (syn.MOE_PREFILL, syn.MOE_PREFILL["E"], (4096,))):
        H, I, k = cfg["H"], cfg["I"], cfg["k"]
        g = syn.rng(cfg["index"], 1)
        banks = [torch.from_numpy(syn.expert_bank(cfg[n], E, r, c, g)).cuda()
                 for n, r, c in (("gate", I, H), ("up", I, H), ("down", H, I))]
        w8 = ctx.moe_weights(cfg["gate"], banks[0], cfg["up"], banks[1], cfg["down"], banks[2])
        per_expert = 2 * I * syn.row_bytes(cfg["gate"], H) + H * syn.row_bytes(cfg["down"], I)
        for T in Ts:
            R = 16 if T <= 8 else (4 if T <= 512 else 2)
            xs = [torch.from_numpy(syn.activations(T, H, g)).cuda() for _ in range(R)]
            lgs = [syn.router_logits(T, E, g, cfg.get("zipf")) for _ in range(R)]
            # distinct experts per layer: top-k by logit (stable sort keeps ties on the lower index)
            distinct = sum(len(np.unique(np.argsort(-lg, axis=1, kind="stable")[:, :k])) for lg in lgs)
            lgd = [torch.from_numpy(lg).cuda() for lg in lgs]
            ys = torch.empty((T, H), dtype=torch.float32, device="cuda")
            ctx.reserve(max_tokens=T, n_experts=E, hidden=H, inter=I, top_k=k)

            def moe():
                for r in range(R):
                    ctx.moe_experts(w8, E, H, I, k, xs[r], logits=lgd[r], Y=ys, reserve=False)

            # 5 tokens and up: the workload's own route (expert-sorted tiles, the direct
            # route held to 4 tokens) under the workload's name, and the library's
            # default (direct calls of 4 tokens where those apply) beside it
            base = f"moe_{cfg['gate'].lower()}_{cfg['down'].lower()}_E{E}_H{H}_I{I}_T{T}"
            runs = [(base, 4 if T > 4 else 32)]
            if T > 4 and _moe_route(T, E, k) != "expert-sorted":
                runs.append((base + "_direct4", 32))
            ops = 2.0 * T * k * 3 * I * H * R  # int multiply-adds x 2
            for name, dmax in runs:
                ctx.set_direct_route_max_tokens(dmax)
                ms = _graph_time(moe, 3 if T > 512 else 5, rt, stream)
                gbps = distinct * per_expert / (ms / 1e3) / 1e9
                out[name] = {"GBps": round(gbps, 1), "frac": round(gbps / hbm_peak, 4),
                             "us_per_layer": round(ms * 1e3 / R, 2), "distinct_experts_per_layer": distinct / R,
                             "int_TOPS": round(ops / (ms / 1e3) / 1e12, 2),
                             "route": _moe_route(T, E, k) if dmax > 4 else ("direct" if T <= 4 else "expert-sorted")}
            ctx.set_direct_route_max_tokens(32)
            name = base
            if T > 4 and cfg["gate"] in ("Q8_0", "Q4_K") and cfg["down"] in ("Q8_0", "Q4_K"):
                # the grouped GEMM runs the integer multiply-adds on 16-bit tensor cores (f16
                # operands holding integers): against the measured dense 16-bit peak
                tp, tkind = tensor_peak()
                out[name]["tensor_frac"] = round(ops / (ms / 1e3) / 1e12 / tp, 4)
                out[name]["tensor_peak"] = f"{tp} TFLOP/s dense bf16/f16 ({tkind})"
        del banks, w8
        torch.cuda.empty_cache()
    ctx.set_static_weights(False)
    ctx.sync_status()
    return out


def profile_case(args):
    """Small launch sequences for ncu captures (not a benchmark).
    gemv: 4 warm-up launches of a 14336 x 4096 GEMV at T=1, then one at T=1, one
          at T=2 and one at T=8, over 5 rotating weight copies (165 MB for Q4_K > L2).
    longrow: the same for the 4096 x 14336 shape (rows streamed in chunks;
          3 rotating copies, 187 MB for Q8_0).
    moe:  the MoE decode layer (128 experts, H 2048, I 768, Q4_K/Q6_K, top-8)
          at T tokens: 2 warm-up layers, then 1 layer.
    mxfp4: the MXFP4 expert layer (256 experts, H 4096, I 2048, top-8) at T
          tokens: 2 warm-up layers, then 1 layer.
    prefill: the expert-sorted route on the prefill workload at T tokens
          (128 experts, H 4096, I 1536, Q8_0 gate/up, Q4_K down, Zipf 1.1)."""
    import torch

    import gguf_block_quant_ggq_gb300 as ggq
    from gguf_block_quant_ggq_gb300 import _build

    _build.build()
    ctx = ggq.Context(0)
    if args.profile_case == "headline":
        # one step of the headline workload (one copy per format): 4 quantizations,
        # 16 GEMVs; run twice, the second pass is the one to capture
        Ws = {f: torch.from_numpy(syn.weights(f, N, K, syn.rng(KQ["index"], 10 + fi))).cuda()
              for fi, f in enumerate(FMTS)}
        gx = syn.rng(KQ["index"], 200)
        xs = {T: torch.from_numpy(syn.activations(T, K, gx)).cuda() for T in TOKENS}
        ctx.reserve(max_tokens=8, max_k=K)
        for _ in range(2):
            xq = {T: ctx.quantize_act("Q8_K", xs[T]) for T in TOKENS}
            for f in FMTS:
                for T in TOKENS:
                    ctx.mul_mat_vec_q(f, Ws[f], N, K, xq[T], T)
    elif args.profile_case == "longrow":
        # the 4096 x 14336 down-projection shape (rows streamed in chunks): 4 warm-up
        # launches at T=1 over 3 rotating copies (> L2), then one at T=1 and one at T=8
        fmt, NL, KL = args.fmt, 4096, 14336
        Ws = [torch.from_numpy(syn.weights(fmt, NL, KL, syn.rng(1, 300 + i))).cuda() for i in range(3)]
        ctx.reserve(max_tokens=8, max_k=KL)
        xq = {T: ctx.quantize_act("Q8_K", torch.from_numpy(syn.activations(T, KL, syn.rng(1, 350 + T))).cuda())
              for T in (1, 8)}
        for i in range(4):
            ctx.mul_mat_vec_q(fmt, Ws[i % 3], NL, KL, xq[1], 1)
        ctx.mul_mat_vec_q(fmt, Ws[1], NL, KL, xq[1], 1)
        ctx.mul_mat_vec_q(fmt, Ws[2], NL, KL, xq[8], 8)
    elif args.profile_case == "gemv":
        fmt = args.fmt
        Ws = [torch.from_numpy(syn.weights(fmt, N, K, syn.rng(1, i))).cuda() for i in range(5)]
        xq = {T: ctx.quantize_act("Q8_K", torch.from_numpy(syn.activations(T, K, syn.rng(1, 50 + T))).cuda())
              for T in (1, 2, 8)}
        for i in range(4):
            ctx.mul_mat_vec_q(fmt, Ws[i % 5], N, K, xq[1], 1)
        ctx.mul_mat_vec_q(fmt, Ws[4], N, K, xq[1], 1)
        ctx.mul_mat_vec_q(fmt, Ws[1], N, K, xq[2], 2)
        ctx.mul_mat_vec_q(fmt, Ws[0], N, K, xq[8], 8)
    else:
        cfg = {"moe": syn.MOE_DECODE, "mxfp4": syn.MOE_MXFP4, "prefill": syn.MOE_PREFILL}[args.profile_case]
        E, H, I, k = cfg["E"], cfg["H"], cfg["I"], cfg["k"]
        g = syn.rng(cfg["index"], 1)
        banks = [torch.from_numpy(syn.expert_bank(cfg[n], E, r, c, g)).cuda()
                 for n, r, c in (("gate", I, H), ("up", I, H), ("down", H, I))]
        w8 = ctx.moe_weights(cfg["gate"], banks[0], cfg["up"], banks[1], cfg["down"], banks[2])
        T = args.tokens
        ctx.set_direct_route_max_tokens(args.direct_max)
        for r in range(3):
            x = torch.from_numpy(syn.activations(T, H, g)).cuda()
            lg = torch.from_numpy(syn.router_logits(T, E, g, cfg.get("zipf"))).cuda()
            ctx.moe_experts(w8, E, H, I, k, x, logits=lg)
    torch.cuda.synchronize()
    ctx.sync_status()
    ctx.close()
    print("profile case done")


def summarize_ncu(path):
    """Per-launch DRAM traffic of the last 16 GEMV launches in an ncu CSV log."""
    import csv
    rows = []
    with open(path) as f:
        lines = [ln for ln in f if ln.startswith('"')]
    for r in csv.DictReader(lines):
        rows.append(r)
    launches = {}
    for r in rows:
        name = r["Kernel Name"]
        if not ("k_stream" in name or "k_gemv_mma" in name):
            continue
        key = int(r["ID"])
        d = launches.setdefault(key, {"kernel": name.split("(")[0]})
        val = float(r["Metric Value"].replace(",", ""))
        unit = r["Metric Unit"]
        scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "ns": 1e-3, "nsecond": 1e-3, "us": 1,
                 "usecond": 1, "ms": 1e3, "msecond": 1e3}
        if r["Metric Name"].startswith("dram__bytes"):
            d[r["Metric Name"]] = val * scale.get(unit, 1)
        elif r["Metric Name"] == "gpu__time_duration.sum":
            d["us"] = val * scale.get(unit, 1)
    last = [launches[k] for k in sorted(launches)][-len(FMTS) * len(TOKENS):]
    plan = [(f, T) for f in FMTS for T in TOKENS]
    out = []
    for (f, T), d in zip(plan, last):
        alg = N * syn.row_bytes(f, K) + T * syn.row_bytes("Q8_K", K) + T * N * 4
        tr = d.get("dram__bytes_read.sum", 0.0) + d.get("dram__bytes_write.sum", 0.0)
        out.append({"launch": f"{f}_T{T}", "kernel": d["kernel"], "us_cold": round(d.get("us", 0.0), 2),
                    "dram_bytes": round(tr), "algorithmic_bytes": alg, "ratio": round(tr / alg, 4)})
    summary = {
        "csrc_hash": csrc_hash(),
        "command": "python bench.py --profile-case headline && ncu --metrics gpu__time_duration.sum,"
                   "dram__bytes_read.sum,dram__bytes_write.sum --clock-control none -k regex:'k_stream|k_gemv_mma' "
                   f"--csv --log-file {path} python bench.py --profile-case headline && "
                   f"python bench.py --summarize-ncu {path}",
        "mean_traffic_bytes": round(sum(o["dram_bytes"] for o in out) / len(out)),
        "mean_algorithmic_bytes": round(sum(o["algorithmic_bytes"] for o in out) / len(out)),
        "launches": out,
    }
    os.makedirs(os.path.dirname(TRAFFIC_FILE), exist_ok=True)
    with open(TRAFFIC_FILE, "w") as f:
        json.dump(summary, f, indent=1)
    print(json.dumps({k: summary[k] for k in ("mean_traffic_bytes", "mean_algorithmic_bytes", "csrc_hash")}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ggq", choices=["ggq", "reference"])
    ap.add_argument("--headline-only", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile-case", choices=["headline", "gemv", "longrow", "moe", "mxfp4", "prefill"], default=None,
                    help="run a small launch sequence for an ncu capture instead of the benchmark")
    ap.add_argument("--fmt", default="Q4_K")
    ap.add_argument("--summarize-ncu", metavar="CSV", default=None,
                    help="write the per-launch DRAM traffic of a --profile-case headline ncu capture "
                         "(metrics gpu__time_duration.sum, dram__bytes_read.sum, dram__bytes_write.sum) "
                         "to profiles/traffic_kquant_gemv_step.json")
    ap.add_argument("--tokens", type=int, default=1)
    ap.add_argument("--direct-max", type=int, default=32,
                    help="--profile-case moe/mxfp4/prefill: the direct MoE route's token limit (4: sorted tiles from 5)")
    args = ap.parse_args()
    if args.summarize_ncu:
        summarize_ncu(args.summarize_ncu)
        return
    if args.profile_case:
        profile_case(args)
        return
    if args.warmup < 3:
        args.warmup = 3
    rank, world = dist_init(args.gpus)
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_gpu(args, rank, world)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
