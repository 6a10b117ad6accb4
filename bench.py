"""Denoiser-step benchmark: target rows/s and TFLOP/s of the 32-block step
(dim 4096, 32 heads x 128, mlp 12288, f16 operands / f32 accumulation) of
a 64x64 target image against a 4114-row prefix (Text(18) + condition
Image(64,64)), on synthetic seeded inputs.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle, timed on a sample

One JSON line on rank 0. Multi-GPU: independent replicas (one process per
GPU, launched by torch.distributed.run), no data-path collective; the
barrier and the max-over-ranks time only frame the measurement.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "step32_cond4114_n4096"
METRIC = "denoiser-step target rows/s & TFLOP/s (32 blocks, 1024² = 4096 rows) vs f16 peak"
UNIT = "target rows/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    p.add_argument("--workload", default=DEFAULT_WORKLOAD)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-rows", type=int, default=0,
                   help="query rows of the CPU sample (0 = all target rows)")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-fp8", action="store_true", help="skip the FP8 (E4M3) variant leg")
    p.add_argument("--source-shas", action="store_true",
                   help="print the source hashes the DRAM traffic records are keyed by, and exit")
    p.add_argument("--dtype", default="f16", choices=["f16", "bf16"],
                   help="16-bit type of the weights and activation rows (the metric is quoted on f16)")
    return p.parse_args(argv)


def workload_of(args):
    """The named workload in the requested 16-bit type."""
    import dataclasses

    from synthetic import qi21_inputs as S
    w = S.WORKLOADS[args.workload]
    if w.dtype != args.dtype:
        w = dataclasses.replace(w, name=f"{w.name}_{args.dtype}", dtype=args.dtype)
    return w


# ------------------------------------------------------------ accounting --

def pass_flops(w, n_rows, vis_sum):
    """(gemm, attention) flops of one pass over n_rows rows and all layers:
    GEMM 2 M (3H^2 + H^2 + 2HI + HI), attention 4 H sum_i visible(i)."""
    H, I, L = w.dim, w.mlp_hidden, w.layers
    gemm = 2.0 * n_rows * (4 * H * H + 3 * H * I) * L
    attn = 4.0 * H * float(vis_sum) * L
    return gemm, attn


def class_work(w, n_rows, vis_sum):
    """Algorithmic work of ONE launch of each kernel class in a step:
    (kind, amount) with kind 'flop' (tensor bound) or 'byte' (HBM bound)."""
    H, I, M = w.dim, w.mlp_hidden, n_rows
    return {
        "qkv": ("flop", 2.0 * M * 3 * H * H),
        "o": ("flop", 2.0 * M * H * H),
        "gateup": ("flop", 2.0 * M * 2 * I * H),
        "down": ("flop", 2.0 * M * H * I),
        "attention": ("flop", 4.0 * H * float(vis_sum)),
        # x f32 read + xn f16 write per row
        "rowop": ("byte", float(M) * H * (4 + 2)),
        # q, k f16 read + write, cos/sin f32 read
        "qkrope": ("byte", float(M) * (2 * H * 2 * 2 + 2 * 64 * 4)),
        "kvcopy": ("byte", float(M) * 2 * H * 2 * 2),
        "misc": ("byte", 4.0 * H * 4 * 2),
        # tokens f32 read + x f32 written / x f32 read + velocity written
        "embed": ("byte", float(M) * (64 + H) * 4),
        "final": ("byte", float(M) * (H + 64) * 4),
    }


# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) of
# each kernel class, from an ncu capture of a few launches of the one-layer
# workload block_cond4114_n4096, whose launches have exactly the shapes of a
# layer of the default workload, with the sha256 of the kernel's sources at
# capture time. Reported only while those sources are unchanged.
NCU_TRAFFIC = {
    # class: (source file, sha256 of its sources at capture, bytes per launch)
    "qkv": ("k_gemm.cu", "684e0dfa6f26be902ffa2091e0bbd5f73ffb7508c27d53d6cf67a68be0300ce5", 259934293),
    "o": ("k_gemm.cu", "684e0dfa6f26be902ffa2091e0bbd5f73ffb7508c27d53d6cf67a68be0300ce5", 185210411),
    "gateup": ("k_gemm.cu", "684e0dfa6f26be902ffa2091e0bbd5f73ffb7508c27d53d6cf67a68be0300ce5", 342851072),
    "down": ("k_gemm.cu", "684e0dfa6f26be902ffa2091e0bbd5f73ffb7508c27d53d6cf67a68be0300ce5", 535644373),
    "attention": ("k_attn.cu", "0c223df4c70c62f3cb0d40456fdc9cf7b63bea42920efa7e17d68ecacd84aafe", 187213056),
    "rowop": ("k_rows.cu", "847de743ecc98efdc1094293875279186e0aeb33cd001f79547e2cc5163ce983", 67706453),
}

# The workloads whose launches have the captured shapes.
TRAFFIC_WORKLOADS = ("step32_cond4114_n4096", "block_cond4114_n4096")


def kernel_source_sha(fname):
    """sha256 over a kernel's translation unit and the headers it includes
    from csrc/ (ptx.cuh, internal.h)."""
    import hashlib
    h = hashlib.sha256()
    for f in (fname, "ptx.cuh", "internal.h"):
        with open(os.path.join(ROOT, "diffusion_transformer_denoiser_qi21_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def measured_traffic(kernel_class, workload):
    """ncu DRAM bytes per launch of a kernel class, or None if there is no
    capture for this workload or the kernel's sources changed since."""
    if workload not in TRAFFIC_WORKLOADS or kernel_class not in NCU_TRAFFIC:
        return None
    fname, sha, nbytes = NCU_TRAFFIC[kernel_class]
    try:
        if kernel_source_sha(fname) != sha:
            return None
    except OSError:
        return None
    return float(nbytes)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except OSError:
        return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------ replicas --

def aggregate(elapsed_s, rows_per_step, steps, dist=None, device="cpu"):
    """Whole-job throughput of independent replicas: every rank processed
    rows_per_step x steps rows; the job took the slowest rank's time.
    Returns (max elapsed seconds over ranks, rows/s over all ranks)."""
    import torch
    world = 1
    t = torch.tensor([float(elapsed_s)], dtype=torch.float64, device=device)
    if dist is not None and dist.is_initialized():
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        world = dist.get_world_size()
    t_max = float(t.item())
    return t_max, rows_per_step * steps * world / t_max


# ---------------------------------------------------------------- clocks --

class ClockSampler:
    """nvidia-smi samples every 200 ms during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, mx, reasons, power = [], [], set(), []
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1].split()[0]))
                mx.append(float(f[2].split()[0]))
                power.append(float(f[3].split()[0]))
            except ValueError:
                continue
            for name, val in zip(self.NAMES, f[5:9]):
                if val == "Active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


# ---------------------------------------------------------- CPU baseline --

class OracleSample:
    """The oracle on layer 0 of the step, as a bounded sample of the
    workload: the keys/values of all n target rows (against the layer-0
    prefix cache, computed once, untimed) plus the query side (q, attention,
    O, FFN) of r target rows; each part timed and scaled to n rows and L
    layers."""

    def __init__(self, w):
        from oracle import qi21_oracle as O
        from synthetic import qi21_inputs as S
        self.O, self.w = O, w
        self.cfg = O.cfg_of(w)
        segs = w.segs(0)
        self.lp = O.prefix_len(segs)
        self.W = S.layer_weights(w, 0)
        cp, sp = O.rope_tables(O.positions(segs)[:self.lp], self.cfg["axes"], self.cfg["theta"])
        vis = O.prefix_visibility(segs)
        _, self.kp, self.vp = O.block(S.x_prefix(w, 0), self.W, S.mods0(w), cp, sp, self.cfg, None, vis,
                                      rows=[0])
        self.ct, self.st = O.target_rope(segs, self.cfg["axes"], self.cfg["theta"])
        self.x = S.x_target(w)
        self.m = S.mods_t(w)

    def layer_seconds(self, r):
        """(estimated seconds of one full layer on all n rows, seconds spent)."""
        import numpy as np
        O, n = self.O, self.w.n_target
        r = n if r <= 0 else min(r, n)
        t0 = time.perf_counter()
        O.block(self.x, self.W, self.m, self.ct, self.st, self.cfg, (self.kp, self.vp), None, rows=np.arange(r))
        t1 = time.perf_counter()
        if r == n:
            return t1 - t0, t1 - t0
        O.block(self.x, self.W, self.m, self.ct, self.st, self.cfg, (self.kp, self.vp), None, rows=[0])
        t2 = time.perf_counter()
        t_kv = t2 - t1
        return t_kv + ((t1 - t0) - t_kv) * (n / r), t2 - t0

    def describe(self, r):
        n, L = self.w.n_target, self.w.layers
        r = n if r <= 0 else min(r, n)
        return (f"oracle (numpy float64, BLAS matmuls) on layer 0 of {L}: K/V of all {n} target rows "
                f"against the {self.lp}-row layer-0 cache + the query side of {r} of {n} rows; "
                f"time scaled to {n} rows x {L} layers")


def oracle_layer_sample(w, r):
    """(rows/s, seconds spent, description) of one timed oracle sample."""
    smp = OracleSample(w)
    t_layer, spent = smp.layer_seconds(r)
    return w.n_target / (t_layer * w.layers), spent, smp.describe(r)


def cpu_cores():
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        v = os.environ.get(var)
        if v and v.isdigit():
            return int(v)
    return os.cpu_count() or 1


# ------------------------------------------------------------ reference --

def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    w = workload_of(args)
    r = args.cpu_rows if args.cpu_rows > 0 else 128
    smp = OracleSample(w)
    desc = smp.describe(r)
    times, spent = [], []
    for i in range(args.warmup + args.steps):
        t_layer, t_spent = smp.layer_seconds(r)
        if i >= args.warmup:
            times.append(t_layer)
            spent.append(t_spent)
    t_layer = statistics.median(times)
    value = w.n_target / (t_layer * w.layers)
    ms = t_layer * w.layers * 1e3
    cores = cpu_cores()
    n_q = w.n_target if r <= 0 else min(r, w.n_target)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": _config(w, args.gpus),
        # each "step" is a timed sample of one layer, scaled to the whole
        # step: ms_per_step is that estimate, not a measured step
        "extrapolated": True,
        "measured": {"seconds_per_sample": statistics.median(spent), "samples": len(spent),
                     "what": f"layer 0 of {w.layers}: K/V of all {w.n_target} target rows + the query side "
                             f"of {n_q} rows"},
        "extrapolation": {"query_rows_factor": w.n_target / n_q, "layers_factor": w.layers},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def _config(w, n_gpus):
    return {"workload": w.name, "dim": w.dim, "heads": w.heads, "head_dim": w.head_dim,
            "mlp_hidden": w.mlp_hidden, "layers": w.layers,
            "prefix_rows": [w.prefix_rows(s) for s in range(w.nseq)], "target_rows": w.n_target,
            "sequences": w.nseq, "parallelism": f"replicas x{n_gpus}",
            "l2": "inputs larger than L2: every step streams all 32 layers' weights (13.96 GB f16) "
                  "and K/V caches"}


# -------------------------------------------------------------- GPU arm --

def run_gpu(args):
    import torch

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    import diffusion_transformer_denoiser_qi21_gb300 as q
    from diffusion_transformer_denoiser_qi21_gb300.make import build as make
    from synthetic import device as D
    from synthetic import qi21_inputs as S

    make()
    w = workload_of(args)
    t0 = time.perf_counter()
    dw = D.DeviceWorkload(w)
    torch.cuda.synchronize()
    t_setup = time.perf_counter() - t0
    n_rows = w.nseq * w.n_target
    lp = [c.lp for c in dw.caches]
    vis_sum = sum(w.n_target * (lp_s + w.n_target) for lp_s in lp)
    gemm_f, attn_f = pass_flops(w, n_rows, vis_sum)
    flops_step = gemm_f + attn_f
    stream = torch.cuda.current_stream()

    def barrier():
        if dist is not None:
            dist.barrier()

    # prefill (once per prompt), timed on its own
    dw.prefill_all()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(2):
        dw.prefill_all()
    e1.record(stream)
    torch.cuda.synchronize()
    prefill_ms = e0.elapsed_time(e1) / 2
    if q.device_status() != 0:
        raise RuntimeError("a kernel gave up waiting during the prefill")

    for _ in range(args.warmup):
        dw.step()
    torch.cuda.synchronize()

    # per-class device times: the same steps launched directly with the
    # library's per-launch events on (kept out of the headline timing)
    _, launches0 = q.profile_read()
    q.profile_enable(True)
    torch.cuda.synchronize()
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    p0.record(stream)
    for _ in range(args.steps):
        dw.step()
    p1.record(stream)
    torch.cuda.synchronize()
    direct_ms = p0.elapsed_time(p1) / args.steps
    class_ms, launches1 = q.profile_read()
    q.profile_enable(False)
    if q.device_status() != 0:
        raise RuntimeError("a kernel gave up waiting during the profiled steps")
    launches = {k: launches1[k] - launches0[k] for k in launches1}
    launches_per_step = sum(launches.values()) / args.steps

    # the step as one recorded CUDA graph (x_target -> x_out with mods_t),
    # replayed for the headline
    graph = q.graph_step_batch(dw.g, dw.layers, dw.caches, dw.x_target, dw.x_out, dw.mods_t, dw.ws)
    for _ in range(args.warmup):
        graph.launch(stream)
    torch.cuda.synchronize()

    gpu_index = local
    vis_dev = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis_dev:
        ids = [v.strip() for v in vis_dev.split(",") if v.strip()]
        if local < len(ids) and ids[local].isdigit():
            gpu_index = int(ids[local])
    clocks = ClockSampler(gpu_index)
    clocks.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        graph.launch(stream)
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier()
    elapsed_ms = ev0.elapsed_time(ev1)
    clk = clocks.stop()
    if q.device_status() != 0:
        raise RuntimeError("a kernel gave up waiting during the timed steps")
    # every replay runs the recorded step's kernels
    gpu_launches = int(round(launches_per_step * args.steps))

    t_max_s, value = aggregate(elapsed_ms * 1e-3, n_rows, args.steps, dist, device="cuda")
    t_max_ms = t_max_s * 1e3
    tflops = flops_step * args.steps * world / t_max_s / 1e12

    # end to end through host buffers: pinned x in, x out back each step
    e2e = None
    if not args.no_e2e:
        x_host = torch.empty_like(dw.x_target, device="cpu").pin_memory()
        x_host.copy_(dw.x_target.cpu())
        out_host = torch.empty_like(x_host).pin_memory()
        m_host = dw.mods_t.cpu().pin_memory()
        barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            # the recorded step reads x_target and mods_t, writes x_out
            dw.x_target.copy_(x_host, non_blocking=True)
            dw.mods_t.copy_(m_host, non_blocking=True)
            graph.launch(stream)
            out_host.copy_(dw.x_out, non_blocking=True)
        torch.cuda.synchronize()
        t_e2e = time.perf_counter() - t0
        _, e2e_value = aggregate(t_e2e, n_rows, args.steps, dist, device="cuda")
        h2d = x_host.numel() * 4 + m_host.numel() * 4
        e2e = {"value": e2e_value, "unit": UNIT,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(out_host.numel() * 4)}

    peaks, peak_src = load_peaks()
    work = class_work(w, n_rows, vis_sum)
    classes = {}
    total_cls = sum(class_ms.values()) or 1.0
    for k, ms in class_ms.items():
        nl = launches.get(k, 0)
        if nl == 0 or ms <= 0:
            continue
        kind, amount = work[k]
        per_launch_s = ms * 1e-3 / nl
        if kind == "flop":
            ach = amount / per_launch_s / 1e12
            peak = peaks["bf16_tflops_sustained"]
            unit = "TFLOP/s"
        else:
            ach = amount / per_launch_s / 1e9
            peak = peaks["hbm_gbs"]
            unit = "GB/s"
        classes[k] = {"ms_per_step": ms / args.steps, "share": ms / total_cls, "launches": nl,
                      "achieved": ach, "unit": unit, "frac": ach / peak}
    dom = max(classes, key=lambda k: classes[k]["ms_per_step"])
    dk = classes[dom]
    kind, amount = work[dom]
    roofline = {
        "kernel": dom, "bound": "tensor" if kind == "flop" else "hbm", "achieved": dk["achieved"],
        "peak": peaks["bf16_tflops_sustained"] if kind == "flop" else peaks["hbm_gbs"],
        "unit": dk["unit"], "frac": dk["frac"], "traffic": measured_traffic(dom, w.name),
        "traffic_unit": "bytes per launch",
        "peak_source": f"{peak_src}: " + ("bf16_tflops_sustained (f16 dense rate = bf16 dense rate)"
                                          if kind == "flop" else "hbm_gbs"),
        "algorithmic_per_launch": amount,
    }
    gemm_ms = sum(classes[k]["ms_per_step"] for k in ("qkv", "o", "gateup", "down") if k in classes)
    attn_ms = classes.get("attention", {}).get("ms_per_step", 0.0)
    fractions = {
        "gemm_tflops": gemm_f / (gemm_ms * 1e-3) / 1e12 if gemm_ms else None,
        "attention_tflops": attn_f / (attn_ms * 1e-3) / 1e12 if attn_ms else None,
    }
    fractions["gemm_frac"] = (fractions["gemm_tflops"] or 0) / peaks["bf16_tflops_sustained"]
    fractions["attention_frac"] = (fractions["attention_tflops"] or 0) / peaks["bf16_tflops_sustained"]

    # the whole sampler call of the pages (t -> modulation; tokens -> embed
    # -> blocks -> final -> velocity), timed on its own beside the step metric
    denoise = None
    if not args.no_e2e:
        tw = {k: torch.from_numpy(v).cuda() for k, v in S.timestep_weights(w).items()}
        mods_c = torch.empty(4 * w.dim, device="cuda")
        fs_c = torch.empty(w.dim, device="cuda")
        t_work = torch.empty(2 * w.dim, device="cuda")

        def sampler_call(t):
            q.timestep_mods(t, tw["t_lin1"], tw["t_lin2"], tw["modulation"], tw["norm_out"], mods_c, fs_c,
                            work=t_work)
            q.denoise_batch(dw.g, dw.layers, dw.caches, tok, w_in, mods_c, fs_c, w_out, vel, dw.ws)

        tok = torch.from_numpy(S.tokens(w)).cuda()
        if w.nseq > 1:
            tok = tok.repeat(w.nseq, 1).contiguous()
        w_in = torch.from_numpy(S.w_in(w)).cuda()
        w_out = torch.from_numpy(S.w_out(w)).cuda()
        vel = torch.empty((n_rows, 64), device="cuda")
        for i in range(2):
            sampler_call(0.9 - 0.1 * i)
        q.profile_enable(True)
        torch.cuda.synchronize()
        d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        d0.record(stream)
        nd = max(2, args.steps // 2)
        for i in range(nd):
            sampler_call(0.7 - 0.5 * i / nd)
        d1.record(stream)
        torch.cuda.synchronize()
        dms, _ = q.profile_read()
        q.profile_enable(False)
        ms = d0.elapsed_time(d1) / nd
        temb_ms = dms["temb"] / nd
        temb_bytes = 4.0 * sum(v.numel() for v in tw.values())
        denoise = {"ms": ms, "rows_per_s": n_rows / (ms * 1e-3), "calls": nd,
                   "what": "timestep_mods + embed + step over all blocks + final, per call",
                   "embed_ms": dms["embed"] / nd, "final_ms": dms["final"] / nd, "temb_ms": temb_ms,
                   "temb_gbs": temb_bytes / (temb_ms * 1e-3) / 1e9 if temb_ms else None}
        if q.device_status() != 0:
            raise RuntimeError("a kernel gave up waiting during the denoiser calls")

    # the FP8 (E4M3 W8A8) variant of the same step, reported beside the
    # f16 headline (its own precision; not the metric's)
    fp8 = None
    if not args.no_fp8 and w.dtype == "f16":
        l8 = [q.pack_layer_fp8(dw.g, l) for l in dw.layers]
        ws8 = torch.empty(q.workspace_bytes_fp8(dw.g, max([n_rows] + lp)), dtype=torch.uint8, device="cuda")
        for s_, c_ in enumerate(dw.caches):
            q.prefill_fp8(dw.g, l8, c_, dw.x_prefix[s_], dw.mods0, ws8)
        out8 = torch.empty_like(dw.x_target)
        for _ in range(args.warmup):
            q.step_batch_fp8(dw.g, l8, dw.caches, dw.x_target, out8, dw.mods_t, ws8)
        q.profile_enable(True)
        torch.cuda.synchronize()
        for _ in range(args.steps):
            q.step_batch_fp8(dw.g, l8, dw.caches, dw.x_target, out8, dw.mods_t, ws8)
        torch.cuda.synchronize()
        cms8, _ = q.profile_read()
        q.profile_enable(False)
        g8 = q.graph_step_batch_fp8(dw.g, l8, dw.caches, dw.x_target, out8, dw.mods_t, ws8)
        for _ in range(args.warmup):
            g8.launch(stream)
        torch.cuda.synchronize()
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        for _ in range(args.steps):
            g8.launch(stream)
        f1.record(stream)
        torch.cuda.synchronize()
        g8.free()
        if q.device_status() != 0:
            raise RuntimeError("a kernel gave up waiting during the FP8 steps")
        ms8 = f0.elapsed_time(f1) / args.steps
        fp8_peak = 2.0 * peaks["bf16_tflops_sustained"]
        gm8 = {}
        for k in ("qkv", "o", "gateup", "down"):
            if cms8.get(k, 0) > 0:
                tf = work[k][1] * launches.get(k, 0) / args.steps / (cms8[k] / args.steps * 1e-3) / 1e12
                gm8[k] = {"ms_per_step": cms8[k] / args.steps, "tflops": tf, "frac_of_fp8_peak": tf / fp8_peak}
        gms8 = sum(v["ms_per_step"] for v in gm8.values())
        fp8 = {"ms_per_step": ms8, "rows_per_s": n_rows / (ms8 * 1e-3), "tflops": flops_step / (ms8 * 1e-3) / 1e12,
               "gemm_tflops": gemm_f / (gms8 * 1e-3) / 1e12 if gms8 else None,
               "fp8_peak": fp8_peak, "fp8_peak_source": "2 x measured bf16_tflops_sustained (nominal 4.5 / 2.25)",
               "gemms": gm8, "quant_ms_per_step": cms8.get("quant", 0.0) / args.steps,
               "attention_ms_per_step": cms8.get("attention", 0.0) / args.steps,
               "launch": "one recorded CUDA graph per step; per-class times from direct launches with events"}
        del l8, ws8, out8
        torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rps, spent, desc = oracle_layer_sample(w, args.cpu_rows)
        cpu = {"value": rps, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle", "sample": desc,
               "seconds": spent}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": t_max_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
            "config": _config(w, world), "tflops": tflops, "flops_per_step": flops_step,
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": gpu_launches,
            "clocks": clk, "classes": classes, "fractions": fractions,
            "prefill": {"ms": prefill_ms, "rows": lp, "rows_per_s": sum(lp) / (prefill_ms * 1e-3)},
            "launch": {"timed": "one recorded CUDA graph per step (qi21_graph_step_batch)",
                       "direct_profiled_ms_per_step": direct_ms},
            "denoise": denoise,
            "fp8": fp8,
            "setup_s": t_setup,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    args = parse(argv)
    if args.source_shas:
        print(json.dumps({f: kernel_source_sha(f) for f in ("k_gemm.cu", "k_attn.cu", "k_rows.cu")}))
        return 0
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
