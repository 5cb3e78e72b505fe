#!/usr/bin/env python
"""Decode-step throughput of LowRAM compressed decode attention on B300.

A step is one model decode step: L sequential ``lowram_decode_attn`` calls, one per layer, each over all B
sequences of the workload (selection keys for every stored token, exact top-S, value regeneration for the
selected tokens, split softmax and merge).  The compressed cache (latent coefficients, bases, predictor
weights, residual lists) is written once by ``lowram_compress`` before timing and stays resident in HBM.
Inputs are seeded synthetic tensors shaped like the workload; nothing is read from disk.

Timing: W warm-up steps, then K steps.  L2 is flushed (a 256 MB buffer is zeroed) before every layer call,
outside the CUDA events that bracket the call, so each call reads its cache cold from HBM (consecutive
layers of a group share the latent coefficients, which would otherwise stay in L2).  Two events per call on
the launching stream bracket it; ``value`` = 1000 / (mean over steps of the summed call times).  One more
step with events between the kernels (which serialises them) gives the per-kernel breakdown.  Multi-GPU (torchrun): every rank runs its own replica of the workload (no data-path collective);
the slowest rank's time and the sum of work give the job's throughput.

    python bench.py [--steps K] [--warmup W] [--workload llama8b] [--impl lowram|reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from decode_attention_19_b300 import synth  # noqa: E402

METRIC = "compressed decode-attn steps/s"
UNIT = "steps/s"
L2_BYTES = 126 * 1024 * 1024
NOMINAL_SM = 148
FP32_LANES_PER_SM = 128


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["lowram", "reference"], default="lowram")
    ap.add_argument("--workload", default="llama8b", choices=list(synth.WORKLOADS))
    ap.add_argument("--B", type=int, default=0)
    ap.add_argument("--T", type=int, default=0)
    ap.add_argument("--layers", type=int, default=0, help="layers per step (default: the workload's L)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-dense", dest="dense", action="store_false",
                    help="skip the uncompressed-cache comparator (timed by default)")
    ap.add_argument("--fit-basis", action="store_true",
                    help="time lowram_fit_basis (the group's cross-layer key basis) on the workload's group shape")
    ap.add_argument("--fit-iters", type=int, default=8)
    ap.add_argument("--fit-predictor", action="store_true",
                    help="time one Adam step of lowram_fit_predictor on the workload's layer shape")
    ap.add_argument("--evict-plan", action="store_true",
                    help="time lowram_attention_mass + lowram_evict_plan on the workload's prompt (T_nominal tokens)")
    ap.add_argument("--window", type=int, default=32, help="observation-window queries for --evict-plan")
    return ap.parse_args()


def workload(args) -> synth.Workload:
    w = synth.WORKLOADS[args.workload]
    kw = {}
    if args.B:
        kw["B"] = args.B
    if args.T:
        kw["T"] = args.T
    if args.layers:
        if args.layers % w.G:
            raise SystemExit(f"--layers {args.layers}: must be a multiple of the layer-group size G={w.G}")
        kw["L"] = args.layers
    return w.with_(**kw) if kw else w


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "sm_max_mhz": 2032.0}, \
        "fallback"


# ------------------------------------------------------------------------------------------------
# algorithmic work per call (bytes, flops) -- the roofline's numerators
# ------------------------------------------------------------------------------------------------
def coef_bytes_per_token(w):
    if w.coef_fmt == "int4":
        return w.r // 2 + 2 * (w.r // 32)
    return w.r * (4 if w.coef_fmt == "f32" else 2)


def algorithmic(w):
    """Per decode call: bytes that must move (cache read once, keys written/read, outputs) and FLOPs."""
    act = 4 if w.act == "f32" else 2
    res_row = w.d * (4 if w.res_fmt == "f32" else 2 if w.res_fmt == "bf16" else 1) + (2 if w.res_fmt == "int8" else 0)
    S = w.S_eff
    bytes_ = (w.B * w.T * coef_bytes_per_token(w)                       # latent coefficients
              + w.H_kv * w.d * w.r * act + 2 * w.H_kv * w.d * w.m * act   # basis + predictor
              + w.B * w.H_kv * w.n_res * 4                                # residual indices
              + w.B * w.H_kv * math.ceil(w.rho * S) * res_row             # residual rows touched (~rho of S)
              + 2 * w.B * w.H_kv * w.T * 4                                # selection keys written + read
              + w.B * w.H_q * w.d * (act + 4))                            # q in, out
    f_keys = 2.0 * w.B * w.T * w.H_kv * w.d * w.r
    f_sel = 2.0 * w.B * w.H_kv * S * w.r * w.d
    f_mlp = 4.0 * w.B * w.H_kv * S * w.d * w.m
    return bytes_, f_keys, f_sel, f_mlp


def job_throughput(ms_per_step_local: float, world: int, dist=None, device=None):
    """Whole-job steps/s of `world` replicas that each ran the same per-rank work: the slowest rank's step
    time bounds the job (max over ranks, the only collective), and the job completes `world` steps in it.
    Returns (steps/s, max ms per step)."""
    ms = float(ms_per_step_local)
    if dist is not None and world > 1:
        t = torch.tensor([ms], device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return world * 1000.0 / ms, ms


def gpu_backlog(ms=10.0):
    """Queue a GPU-side wait (outside every timed event pair) so the host runs ahead of the GPU: a host
    hiccup while it enqueues a step then cannot leave the GPU idle between an event and the kernel after it."""
    if hasattr(torch.cuda, "_sleep"):
        torch.cuda._sleep(int(ms * 1e-3 * 2.0e9))


def launches_per_call(w, tc_path):
    """Kernels one decode call launches: keys, selection, values and the merge of the values' chunk records, plus,
    for an int4 cache on the tensor cores, the one kernel that makes the fp16 copies of the coefficients and the
    basis (the exact bf16 split behind LOWRAM_FLAG_INT4_EXACT_SPLIT takes two, and the bench does not set it)."""
    copy = 1 if (tc_path and w.coef_fmt == "int4") else 0
    if w.S_eff == 0:
        return 2 + copy
    return 4 + copy


def kernel_digest(paths):
    h = hashlib.sha256()
    for p in sorted(paths):
        h.update(open(p, "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(name, src_files):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", name)
    if not os.path.exists(path):
        return None
    kv = {}
    for line in open(path):
        if ":" in line and not line.startswith("#"):
            k, v = line.split(":", 1)
            kv[k.strip()] = v.strip()
    if kv.get("kernel_source_digest") != kernel_digest(src_files):
        return None
    try:
        return float(kv["dram_bytes_per_launch_full_size"])
    except (KeyError, ValueError):
        return None


# ------------------------------------------------------------------------------------------------
# clocks during the timed region
# ------------------------------------------------------------------------------------------------
class _Nvml:
    """Read-only NVML queries through the driver's libnvidia-ml (the Python binding when present, else ctypes):
    current and maximum SM clock and the active clock-event reasons of one GPU."""
    NVML_CLOCK_SM = 1

    def __init__(self, uuid):
        try:
            import pynvml
            pynvml.nvmlInit()
            self.py = pynvml
            self.h = pynvml.nvmlDeviceGetHandleByUUID(uuid)
            self.reasons = getattr(pynvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                pynvml.nvmlDeviceGetCurrentClocksThrottleReasons
            return
        except ImportError:
            self.py = None
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit_v2 failed")
        self.h = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.h)) != 0:
            raise RuntimeError("nvmlDeviceGetHandleByUUID failed")
        self.lib, self.ct = lib, ctypes
        self.reason_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def max_sm_mhz(self):
        if self.py is not None:
            return float(self.py.nvmlDeviceGetMaxClockInfo(self.h, self.py.NVML_CLOCK_SM))
        v = self.ct.c_uint()
        self.lib.nvmlDeviceGetMaxClockInfo(self.h, self.NVML_CLOCK_SM, self.ct.byref(v))
        return float(v.value)

    def sample(self):
        try:
            if self.py is not None:
                return float(self.py.nvmlDeviceGetClockInfo(self.h, self.py.NVML_CLOCK_SM)), int(self.reasons(self.h))
            mhz, why = self.ct.c_uint(), self.ct.c_ulonglong()
            if self.lib.nvmlDeviceGetClockInfo(self.h, self.NVML_CLOCK_SM, self.ct.byref(mhz)) != 0:
                return None
            if self.reason_fn(self.h, self.ct.byref(why)) != 0:
                return None
            return float(mhz.value), int(why.value)
        except Exception:   # noqa: BLE001 -- a missed sample is skipped
            return None


class Clocks:
    """SM clock and throttle reasons sampled every 2 ms on a host thread (NVML reads only) while the timed
    region runs; nvidia-smi at its 200 ms minimum period if NVML cannot be used."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    # NVML clock-event reason bits
    REASONS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20, "hw_thermal_slowdown": 0x40}

    def __init__(self, dev):
        self.proc = None
        self.f = None
        self.thread = None
        self.samples = []
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        ident = uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
        self.nvml_error = None
        try:
            nv = _Nvml(ident)
            self.max_mhz = nv.max_sm_mhz()
            self.stop_event = threading.Event()

            def run():
                while not self.stop_event.is_set():
                    got = nv.sample()
                    if got is not None:
                        self.samples.append(got)
                    time.sleep(0.002)

            self.thread = threading.Thread(target=run, daemon=True)
            self.thread.start()
            return
        except Exception as e:   # noqa: BLE001 -- fall back to nvidia-smi below
            self.nvml_error = repr(e)
            self.thread = None
        try:
            self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", ident, f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except (OSError, RuntimeError):
            self.proc = None

    def stop(self):
        if self.thread is not None:
            self.stop_event.set()
            self.thread.join(timeout=5)
            if not self.samples:
                return None
            reasons = sorted(n for n, bit in self.REASONS.items() if any(w & bit for _, w in self.samples))
            return {"sm_mhz": statistics.median(m for m, _ in self.samples), "sm_max_mhz": self.max_mhz,
                    "reasons": reasons, "samples": len(self.samples), "source": "NVML every 2 ms"}
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.seek(0)
        rows = [r.split(",") for r in self.f.read().strip().splitlines() if r.strip()]
        os.unlink(self.f.name)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "source": "nvidia-smi, 200 ms", "nvml_error": self.nvml_error}


# ------------------------------------------------------------------------------------------------
# the compressed cache of the whole model (all layer groups), written by lowram_compress
# ------------------------------------------------------------------------------------------------
def build_cache(w, dev):
    import torch.nn.functional as F

    import decode_attention_19_b300 as L
    act = torch.bfloat16 if w.act == "bf16" else torch.float32
    fmt = {"f32": L.LOWRAM_F32, "bf16": L.LOWRAM_BF16, "int4": L.LOWRAM_INT4_G32, "int8": L.LOWRAM_INT8_VEC}
    pos = synth.eviction_positions(w).to(dev) if w.T_nominal else None
    groups, compress_ms = [], []
    for gi in range(w.groups):
        raw = synth.draw_group(w, gi, with_noise=False)
        C = raw["coef"].to(dev)
        gen = torch.Generator(device=dev).manual_seed(synth.sub_seed(w.seed, w.name, gi, "noise-device"))
        keys, vals = [], []
        for l in range(w.G):
            K = (C.view(-1, w.r) @ raw["basis"][l].to(dev).float().T).view(w.B, w.T, w.H_kv, w.d)
            Hh = F.silu(torch.einsum("bthd,hmd->bthm", K, raw["w1"][l].to(dev).float()))
            V = torch.einsum("bthm,hdm->bthd", Hh, raw["w2"][l].to(dev).float())
            V += 0.3 * torch.randn(V.shape, device=dev, generator=gen)
            keys.append(K.to(act))
            vals.append(V.to(act).contiguous())
            del K, Hh, V
        kg = torch.stack(keys, dim=2).contiguous()
        del keys
        Wst = torch.cat([b.double() for b in raw["basis"]]).to(dev)
        proj = torch.linalg.pinv(Wst).float().contiguous()
        bases = [b.to(dev) for b in raw["basis"]]
        w1s = [x.to(dev) for x in raw["w1"]]
        w2s = [x.to(dev) for x in raw["w2"]]
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        r = L.lowram_compress(kg, vals, proj, bases, w1s, w2s, n_res=w.n_res, coef_dtype=fmt[w.coef_fmt],
                              res_dtype=fmt[w.res_fmt], pos=pos)
        e1.record()
        torch.cuda.synchronize()
        compress_ms.append(e0.elapsed_time(e1))
        del kg, vals, C
        groups.append(dict(coef=r["coef"], coef_scale=r["coef_scale"], bases=bases, w1s=w1s, w2s=w2s,
                           res_idx=r["res_idx"], res_val=r["res_val"],
                           res_scale=r["res_scale"] if r["res_scale"] is not None else [None] * w.G))
        torch.cuda.empty_cache()
    return groups, pos, compress_ms


def layer_args(w, groups, layer):
    g = groups[layer // w.G]
    l = layer % w.G
    return dict(coef=g["coef"], coef_scale=g["coef_scale"], basis=g["bases"][l], w1=g["w1s"][l], w2=g["w2s"][l],
                res_idx=g["res_idx"][l] if w.n_res else None, res_val=g["res_val"][l] if w.n_res else None,
                res_scale=g["res_scale"][l] if w.n_res else None)


# ------------------------------------------------------------------------------------------------
# CPU oracle sample (cpu_baseline and the reference arm)
# ------------------------------------------------------------------------------------------------
def oracle_sample_inputs(w, n_seq=1):
    """One layer call restricted to n_seq sequences, built on the CPU from the seeded draws."""
    import oracle as O
    ws = w.with_(B=n_seq)
    raw = synth.draw_group(ws, 0, with_noise=False)
    coef = raw["coef"].to(torch.bfloat16 if w.coef_fmt == "bf16" else torch.float32)
    coef_vals = O.f64(coef)
    if w.coef_fmt == "int4":
        packed, sc = O.quant_int4_g32(raw["coef"])
        coef_vals = O.dequant_int4_g32(packed, sc)
    ridx, rval = synth.placeholder_residuals(ws, 0)
    res_vals = O.f64(rval.to(torch.bfloat16)) if w.res_fmt != "int8" else O.dequant_int8_vec(*O.quant_int8_vec(rval))
    pos = synth.eviction_positions(ws) if w.T_nominal else None
    return dict(q=synth.draw_query(ws, 0), coef=coef_vals, basis=raw["basis"][0], w1=raw["w1"][0], w2=raw["w2"][0],
                res_idx=ridx if w.n_res else None, res_val=res_vals if w.n_res else None, pos=pos)


def time_oracle_sample(w, inp, reps):
    import oracle as O
    ts = []
    for _ in range(reps):
        t0 = time.perf_counter()
        O.decode(inp["q"], inp["coef"], inp["basis"], inp["w1"], inp["w2"], S=w.S, theta=w.theta, pos=inp["pos"],
                 res_idx=inp["res_idx"], res_val=inp["res_val"])
        ts.append(time.perf_counter() - t0)
    return ts


def run_reference(args, rank):
    """The oracle as it stands, timed on the host cores: each step is one layer call for one sequence,
    scaled to the workload's steps/s (B sequences x L layers per step)."""
    if rank != 0:
        return
    import oracle as O
    w = workload(args)
    inp = oracle_sample_inputs(w)
    time_oracle_sample(w, inp, args.warmup)
    ts = time_oracle_sample(w, inp, args.steps)
    t_step = statistics.mean(ts) * w.B * w.L
    v = 1.0 / t_step
    cores = O.max_threads()
    sample = f"one layer call of 1 of {w.B} sequences (all {w.H_kv} kv-heads, T={w.T}); x{w.B * w.L} per step"
    line = {"metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": t_step * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": w.name, "B": w.B, "T": w.T, "layers": w.L, "S": w.S, "n_res": w.n_res},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------------------------
# main arm
# ------------------------------------------------------------------------------------------------
def main():
    args = parse()
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local = int(os.environ.get("LOCAL_RANK", 0))
    if args.impl == "reference":
        run_reference(args, rank)
        return
    import decode_attention_19_b300 as L

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    w = workload(args)
    pk, pk_kind = peaks()
    if args.fit_basis:
        if rank == 0:
            fit_bench(w, dev, args, pk)
        return
    if args.fit_predictor:
        if rank == 0:
            fit_predictor_bench(w, dev, args, pk)
        return
    if args.evict_plan:
        if rank == 0:
            evict_bench(w, dev, args, pk)
        return
    groups, pos, compress_ms = build_cache(w, dev)
    cos, sin = L.lowram_rope_table(w.d, w.theta, w.T_nominal or w.T)
    qs = [synth.draw_query(w, l).to(dev) for l in range(w.L)]
    shape_probe = L.decode_shape(qs[0], groups[0]["coef"], groups[0]["w1s"][0], S=w.S, n_res=w.n_res,
                                 max_pos=cos.shape[1], res_dtype=1, coef_int4=w.coef_fmt == "int4")
    ws = torch.zeros(L.lowram_decode_workspace_size(shape_probe), dtype=torch.uint8, device=dev)
    out = torch.empty((w.B, w.H_q, w.d), dtype=torch.float32, device=dev)
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
    args_l = [layer_args(w, groups, l) for l in range(w.L)]

    def call(l, q=None, events=None):
        a = args_l[l]
        return L.lowram_decode_attn(qs[l] if q is None else q, a["coef"], a["basis"], a["w1"], a["w2"], rope_cos=cos,
                                    rope_sin=sin, S=w.S, coef_scale=a["coef_scale"], pos=pos, res_idx=a["res_idx"],
                                    res_val=a["res_val"], res_scale=a["res_scale"], out=out, workspace=ws,
                                    want_lse=False, events=events)

    # warm-up
    for _ in range(args.warmup):
        for l in range(w.L):
            flush.zero_()
            call(l)
    torch.cuda.synchronize()
    if L.lowram_get_error(ws):
        raise RuntimeError("device check word set during warm-up")

    # timed region: K steps x L calls; one event before and one after each call, none between its kernels (so
    # the kernels' programmatic dependent launches overlap as they do in use)
    evs = [[[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(w.L)] for _ in range(args.steps)]
    for step in evs:
        for e5 in step:
            for e in e5:
                e.record()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = Clocks(dev)
    t_wall = time.perf_counter()
    for s in range(args.steps):
        gpu_backlog()
        for l in range(w.L):
            flush.zero_()
            e5 = evs[s][l]
            call(l, events=[e5[0], None, None, None, e5[4]])
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    clk = clocks.stop()
    call_ms = np.array([[evs[s][l][0].elapsed_time(evs[s][l][4]) for l in range(w.L)] for s in range(args.steps)])
    step_ms = call_ms.sum(axis=1)
    value, ms_per_step = job_throughput(float(step_ms.mean()), world, dist, dev)

    # per-kernel breakdown (three more steps with events between the kernels, which serialise them; median
    # over the calls)
    n_bd = 3
    stage = np.zeros((n_bd * w.L, 4))
    bev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(n_bd * w.L)]
    for e5 in bev:
        for e in e5:
            e.record()
    torch.cuda.synchronize()
    for i in range(n_bd * w.L):
        if i % w.L == 0:
            gpu_backlog()
        flush.zero_()
        call(i % w.L, events=bev[i])
    torch.cuda.synchronize()
    for i in range(n_bd * w.L):
        for k in range(4):
            stage[i, k] = bev[i][k].elapsed_time(bev[i][k + 1])
    per_kernel_ms = np.median(stage, axis=0)    # K1 keys, K2 select, K3 values (+ merge), K4 merge
    names = ["score", "select", "vregen", "merge"]
    dom = int(np.argmax(per_kernel_ms))

    # back-to-back (no flush) for context
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for l in range(w.L):
        call(l)
    e1.record()
    torch.cuda.synchronize()
    ms_b2b = e0.elapsed_time(e1)

    # end to end through the public API: every step copies its inputs (the L layer calls' queries) from pinned host
    # memory in one transfer before its first call, and reads its results (the L outputs) back to pinned host memory
    # in one transfer after its last call; each call writes its own output buffer.  The timed intervals are the L
    # calls, the first including the upload and the last the download (the L2 flush between calls stays outside).
    e2e = None
    if not args.no_e2e:
        q_host = torch.stack([q.cpu() for q in qs]).pin_memory()                       # [L, B, H_q, d]
        out_host = torch.empty((w.L, w.B, w.H_q, w.d), dtype=torch.float32).pin_memory()
        q_dev = torch.empty((w.L,) + tuple(qs[0].shape), dtype=qs[0].dtype, device=dev)
        out_dev = torch.empty((w.L, w.B, w.H_q, w.d), dtype=torch.float32, device=dev)
        st = torch.cuda.current_stream()

        def call_e2e(l):
            a = args_l[l]
            L.lowram_decode_attn(q_dev[l], a["coef"], a["basis"], a["w1"], a["w2"], rope_cos=cos, rope_sin=sin, S=w.S,
                                 coef_scale=a["coef_scale"], pos=pos, res_idx=a["res_idx"], res_val=a["res_val"],
                                 res_scale=a["res_scale"], out=out_dev[l], workspace=ws, want_lse=False)

        def e2e_loop(backlog):
            """Mean ms per step of the events around the L calls, and the host's mean microseconds inside the
            binding per call.  Without the backlog the host enqueues each call only after the previous one
            returned, so host time the GPU waits for shows up between the events."""
            step_ms, host_us = [], []
            for s in range(args.warmup + args.steps):
                pairs = []
                if backlog:
                    gpu_backlog()
                for l in range(w.L):
                    flush.zero_()
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record()
                    if l == 0:
                        q_dev.copy_(q_host, non_blocking=True)
                    t0 = time.perf_counter()
                    call_e2e(l)
                    t1 = time.perf_counter()
                    if l == w.L - 1:
                        out_host.copy_(out_dev, non_blocking=True)
                    b.record()
                    pairs.append((a, b))
                    if s >= args.warmup:
                        host_us.append((t1 - t0) * 1e6)
                st.synchronize()
                if s >= args.warmup:
                    step_ms.append(sum(a.elapsed_time(b) for a, b in pairs))
            return float(np.mean(step_ms)), float(np.mean(host_us))

        ms_plain, host_us_call = e2e_loop(backlog=False)
        ms_backlog, _ = e2e_loop(backlog=True)
        e2e_value, m = job_throughput(ms_plain, world, dist, dev)
        e2e = {"value": e2e_value, "unit": UNIT,
               "h2d_bytes_per_step": q_host.numel() * q_host.element_size(),
               "d2h_bytes_per_step": out_host.numel() * out_host.element_size(), "ms_per_step": m,
               "host_us_per_call": host_us_call,
               "how": "host enqueues call after call (no queued GPU wait ahead); events around each call, the "
                      "first including the query upload and the last the output download",
               "ms_per_step_host_ahead": job_throughput(ms_backlog, world, dist, dev)[1]}

    # roofline of the dominant kernel
    bytes_call, f_keys, f_sel, f_mlp = algorithmic(w)
    src = [os.path.join(ROOT, "decode_attention_19_b300", "csrc", f) for f in
           ("tc_decode.cu", "tc_common.cuh", "common.cuh", "kernels.h")]
    tc_path = L.lowram_decode_uses_tensor_cores(shape_probe)
    k1_ms = per_kernel_ms[0]
    if tc_path:
        # the key pass is timed alone (events on both sides, L2 flushed before), for ~70 us: the burst peak
        peak_tf = pk["bf16_tflops"]
        roof = {"bound": "tensor", "achieved": f_keys / (k1_ms * 1e-3) / 1e12, "peak": peak_tf, "unit": "TFLOP/s",
                "peak_kind": f"{pk_kind} bf16 burst"}
    else:
        peak_tf = NOMINAL_SM * FP32_LANES_PER_SM * 2 * pk.get("sm_max_mhz", 2032.0) * 1e6 / 1e12
        roof = {"bound": "alu", "achieved": f_keys / (k1_ms * 1e-3) / 1e12, "peak": peak_tf, "unit": "TFLOP/s",
                "peak_kind": "fp32 FMA: 148 SMs x 128 lanes x 2 FLOP x max SM clock"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["kernel"] = "score (selection keys of every token)"
    traffic = profiled_traffic("score_tc_llama8b.md", src) if w.name == "llama8b" else None
    roof["traffic"] = traffic
    t_bytes_us = bytes_call / (pk["hbm_gbs"] * 1e9) * 1e6
    # a decode call lasts ~0.1 ms between L2 flushes: the burst bf16 peak applies (the sustained one is also given)
    t_alg_us = max(t_bytes_us, (f_keys + f_sel + f_mlp) / (pk["bf16_tflops"] * 1e12) * 1e6)
    t_lit_us = max(t_bytes_us, f_mlp / (pk["bf16_tflops"] * 1e12) * 1e6)
    t_alg_sus_us = max(t_bytes_us, (f_keys + f_sel + f_mlp) / (pk["bf16_tflops_sustained"] * 1e12) * 1e6)
    call_us = ms_per_step * 1e3 / w.L

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16" if w.act == "bf16" else "f32", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "T": w.T, "T_nominal": w.T_nominal or w.T, "layers": w.L,
                       "G": w.G, "H_q": w.H_q, "H_kv": w.H_kv, "d": w.d, "r": w.r, "m": w.m, "S": w.S,
                       "n_res": w.n_res, "coef": w.coef_fmt, "res": w.res_fmt,
                       "l2": "flushed before every layer call (256 MB zero fill, outside the timed events)",
                       "parallelism": f"replicas x{world}"},
            "tokens_heads_per_s": w.B * w.T * w.H_q / (call_us * 1e-6) * world,
            "hbm_gbs_algorithmic": bytes_call / (call_us * 1e-6) / 1e9,
            "roofline_call": {"t_call_us": call_us, "bytes_per_call": bytes_call,
                              "t_bytes_us": t_bytes_us, "literal_roof_us": t_lit_us, "algorithmic_roof_us": t_alg_us,
                              "frac_literal": t_lit_us / call_us, "frac_algorithmic": t_alg_us / call_us,
                              "peak": "bf16 burst (measured)", "algorithmic_roof_us_sustained": t_alg_sus_us,
                              "frac_algorithmic_sustained": t_alg_sus_us / call_us},
            "per_kernel_us": {n: float(v) * 1e3 for n, v in zip(names, per_kernel_ms)},
            "dominant_kernel": names[dom],
            "roofline": roof,
            "ms_per_step_no_flush": ms_b2b, "wall_ms_per_step": t_wall * 1e3 / args.steps,
            "compress_ms_per_group": float(np.mean(compress_ms)),
            "gpu_launches": args.steps * w.L * launches_per_call(w, tc_path),
            "clocks": clk, "peaks": pk_kind}
    if e2e:
        line["e2e"] = e2e
        line["host_us_per_call"] = e2e["host_us_per_call"]
    if args.dense and w.act == "bf16":   # before the CPU baseline, while the GPU is still at its working clocks
        line["dense_comparator"] = dense_bench(w, dev, qs, flush, args)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle as O
        inp = oracle_sample_inputs(w)
        ts = time_oracle_sample(w, inp, 3)
        t_step = statistics.median(ts) * w.B * w.L
        line["cpu_baseline"] = {"value": 1.0 / t_step, "unit": UNIT, "cores": O.max_threads(), "kind": "oracle",
                                "sample": f"one layer call of 1 of {w.B} sequences (all kv-heads, T={w.T}), "
                                          f"median of 3, x{w.B * w.L} per step"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def fit_bench(w, dev, args, pk):
    """lowram_fit_basis on one layer group of the workload: keys [B, T, G, H_kv, d] of rank r with a decaying
    spectrum plus noise (seeded, made on the GPU), timed with CUDA events over --steps calls after --warmup."""
    import decode_attention_19_b300 as L
    B, T, G, H_kv, d, r = w.B, w.T, w.G, w.H_kv, w.d, w.r
    D, N = G * H_kv * d, B * T
    g = torch.Generator(device=dev).manual_seed(11)
    U, _ = torch.linalg.qr(torch.randn((D, r), generator=g, device=dev))
    sig = torch.logspace(1.0, 0.0, r, device=dev)
    keys = torch.randn((N, r), generator=g, device=dev) * sig @ U.T
    keys = (keys + 0.05 * torch.randn((N, D), generator=g, device=dev)).to(torch.bfloat16).view(B, T, G, H_kv, d)
    del U
    ws = None
    for _ in range(args.warmup):
        proj, bases, ws = L.lowram_fit_basis(keys, r, iters=args.fit_iters, workspace=ws)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for a, b in ev:
        a.record()
        proj, bases, ws = L.lowram_fit_basis(keys, r, iters=args.fit_iters, workspace=ws)
        b.record()
    torch.cuda.synchronize()
    if L.lowram_get_error(ws):
        raise RuntimeError("device check word set by lowram_fit_basis")
    ms = float(np.median([a.elapsed_time(b) for a, b in ev]))
    # rebuild error of the fitted subspace against the optimal one (the noise floor): a sampled check
    Kf = keys.view(N, D)[:8192].float()
    P = proj.float()
    err = float(torch.linalg.norm(Kf - (Kf @ P.T) @ P) / torch.linalg.norm(Kf))
    it = args.fit_iters + 1          # iterations plus the final Cholesky QR
    flops = N * D * D + args.fit_iters * 2.0 * D * D * r + it * (4.0 * D * r * r + 2.0 * r ** 3 / 3.0)
    peak_tf = NOMINAL_SM * FP32_LANES_PER_SM * 2 * pk.get("sm_max_mhz", 2032.0) * 1e6 / 1e12
    achieved = flops / (ms * 1e-3) / 1e12
    print(json.dumps({
        "metric": "fitted key basis: time per layer group", "value": ms, "unit": "ms", "higher_is_better": False,
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name, "B": B, "T": T, "G": G, "H_kv": H_kv, "d": d, "r": r, "D": D,
                   "iters": args.fit_iters, "keys": "bf16, rank r (spectrum 10..1) + 0.05 noise"},
        "rebuild_rel_err_sampled": err,
        "roofline": {"bound": "alu", "achieved": achieved, "peak": peak_tf, "unit": "TFLOP/s",
                     "frac": achieved / peak_tf, "traffic": None,
                     "peak_kind": "fp32 FMA: 148 SMs x 128 lanes x 2 FLOP x max SM clock (a reference scale: the Gram "
                                  "matrix and Z = G Q run on the tensor cores as six bf16 products each, Z^T Z and "
                                  "the Cholesky in fp64 on the CUDA cores)",
                     "work": "float32-equivalent: Gram N*D^2 (symmetric) + per iteration 2*D^2*r + 4*D*r^2 + 2r^3/3"}}))


def fit_predictor_bench(w, dev, args, pk):
    """lowram_fit_predictor on one layer of the workload (all kv-heads, B*T prompt tokens): the time of one full-batch
    Adam step (gradient of every head's predictor + the update), from --steps steps after --warmup."""
    import decode_attention_19_b300 as L
    B, T, H_kv, d, m = w.B, w.T, w.H_kv, w.d, w.m
    g = torch.Generator(device=dev).manual_seed(12)
    keys = torch.randn((B, T, H_kv, d), generator=g, device=dev).to(torch.bfloat16)
    values = (0.5 * torch.tanh(keys.float().flip(-1)) + 0.1 * torch.randn((B, T, H_kv, d), generator=g, device=dev))
    values = values.to(torch.bfloat16)
    params = [torch.randn(s, generator=g, device=dev) * sc for s, sc in
              (((H_kv, m, d), d ** -0.5), ((H_kv, m), 0.1), ((H_kv, d, m), m ** -0.5), ((H_kv, d), 0.1))]
    L.lowram_fit_predictor(keys, values, *params, steps=max(1, args.warmup), lr=1e-3)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    losses = L.lowram_fit_predictor(keys, values, *params, steps=args.steps, lr=1e-3)
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / args.steps
    flops = 10.0 * B * T * d * m * H_kv            # forward (2 products), backward (3 products), 2 FLOP per MAC
    peak_tf = NOMINAL_SM * FP32_LANES_PER_SM * 2 * pk.get("sm_max_mhz", 2032.0) * 1e6 / 1e12
    achieved = flops / (ms * 1e-3) / 1e12
    ls = losses.float().cpu().numpy()
    print(json.dumps({
        "metric": "predictor fit: time per Adam step per layer", "value": ms, "unit": "ms", "higher_is_better": False,
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name, "B": B, "T": T, "H_kv": H_kv, "d": d, "m": m, "inputs": "bf16 keys/values"},
        "loss_first_last": [float(ls[0].mean()), float(ls[-1].mean())],
        "roofline": {"bound": "alu", "achieved": achieved, "peak": peak_tf, "unit": "TFLOP/s",
                     "frac": achieved / peak_tf, "traffic": None,
                     "peak_kind": "fp32 FMA: 148 SMs x 128 lanes x 2 FLOP x max SM clock (a reference scale: the five "
                                  "products run on the tensor cores as six bf16 products each)",
                     "work": "float32-equivalent: 10 * B*T * d * m * H_kv per step"}}))


def evict_bench(w, dev, args, pk):
    """The heavy-hitter eviction plan of one layer's prompt: attention mass of a --window query window over the
    T_nominal prompt tokens (rotated K, bf16), then the kept tokens (64 sinks, 2048 recents, to w.T)."""
    import decode_attention_19_b300 as L
    Tn = w.T_nominal or w.T
    g = torch.Generator(device=dev).manual_seed(13)
    q = (torch.randn((w.B, args.window, w.H_q, w.d), generator=g, device=dev) * 2 * w.d ** -0.5).to(torch.bfloat16)
    k = torch.randn((w.B, Tn, w.H_kv, w.d), generator=g, device=dev).to(torch.bfloat16)
    n_sink, n_recent = 64, min(2048, Tn // 4)
    T_keep = max(w.T, n_sink + n_recent) if w.T < Tn else Tn // 4 + n_sink + n_recent
    # workspaces allocated once, outside the timed region (the calls would otherwise allocate them each time)
    B_, W_, H_q_, d_ = q.shape
    ws_mass = torch.zeros(L.lowram_attention_mass_workspace_size(B_, Tn, W_, H_q_, w.H_kv, d_, L.LOWRAM_BF16),
                          dtype=torch.uint8, device=dev)
    ws_plan = torch.zeros(L.lowram_evict_plan_workspace_size(w.B, Tn), dtype=torch.uint8, device=dev)

    def plan():
        return L.lowram_evict_plan(L.lowram_attention_mass(q, k, workspace=ws_mass), n_sink=n_sink,
                                   n_recent=n_recent, T_keep=T_keep, workspace=ws_plan)
    for _ in range(max(1, args.warmup)):
        keep = plan()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for a, b in ev:
        a.record()
        keep = plan()
        b.record()
    torch.cuda.synchronize()
    ms = float(np.median([a.elapsed_time(b) for a, b in ev]))
    em = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for a, b in em:
        a.record()
        L.lowram_attention_mass(q, k, workspace=ws_mass)
        b.record()
    torch.cuda.synchronize()
    mass_ms = float(np.median([a.elapsed_time(b) for a, b in em]))
    # bytes: the window's log-sum-exp pass and the mass pass each read K once; FLOPs: the logits, twice
    kbytes = w.B * Tn * w.H_kv * w.d * 2
    flops = 2 * 2.0 * w.B * Tn * args.window * w.H_q * w.d
    # bf16: both passes stream K through the tensor cores, so the mass is HBM-bound (K read twice)
    print(json.dumps({
        "metric": "eviction plan: time per layer", "value": ms, "unit": "ms", "higher_is_better": False,
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "T_prompt": Tn, "window": args.window, "H_q": w.H_q,
                   "H_kv": w.H_kv, "d": w.d, "n_sink": n_sink, "n_recent": n_recent, "T_keep": T_keep},
        "kept_first_row_head": keep[0, :4].tolist(),
        "mass_ms": mass_ms,
        "roofline": {"bound": "hbm", "achieved": 2 * kbytes / (mass_ms * 1e-3) / 1e9, "peak": pk["hbm_gbs"],
                     "unit": "GB/s", "frac": 2 * kbytes / (mass_ms * 1e-3) / 1e9 / pk["hbm_gbs"], "traffic": None,
                     "kernel": "attention mass (log-sum-exp pass, fold, mass pass)",
                     "work": "K read once per pass: 2 * B*T * H_kv*d * 2 bytes"},
        "work": {"K_bytes": kbytes, "bytes_read_estimate": 2 * kbytes, "flops": flops,
                 "tensor_tflops": flops / (mass_ms * 1e-3) / 1e12}}))


def dense_bench(w, dev, qs, flush, args):
    """Same kernel family on an uncompressed bf16 cache at the same shape (explicit rotated K and V)."""
    import decode_attention_19_b300 as L
    Tn = w.T_nominal or w.T
    n_layers = min(w.L, 4)
    g = torch.Generator(device=dev).manual_seed(7)
    ks = [torch.randn((w.B, Tn, w.H_kv, w.d), device=dev, generator=g).to(torch.bfloat16) for _ in range(n_layers)]
    vs = [torch.randn((w.B, Tn, w.H_kv, w.d), device=dev, generator=g).to(torch.bfloat16) for _ in range(n_layers)]
    out = torch.empty((w.B, w.H_q, w.d), dtype=torch.float32, device=dev)
    ws = torch.zeros(L.lowram_dense_workspace_size(w.B, Tn, w.H_q, w.H_kv, w.d), dtype=torch.uint8, device=dev)
    ts = []
    for it in range(args.warmup + args.steps):
        for l in range(n_layers):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            L.lowram_dense_decode_attn(qs[l], ks[l], vs[l], out=out, workspace=ws, want_lse=False)
            b.record()
            if it >= args.warmup:
                ts.append((a, b))
    torch.cuda.synchronize()
    t_call = float(np.mean([a.elapsed_time(b) for a, b in ts]))
    kv_bytes = 2 * w.B * Tn * w.H_kv * w.d * 2
    return {"t_call_us": t_call * 1e3, "T": Tn, "kv_bytes_per_call": kv_bytes,
            "hbm_gbs": kv_bytes / (t_call * 1e-3) / 1e9, "steps_per_s_equiv": 1000.0 / (t_call * w.L)}


if __name__ == "__main__":
    main()
