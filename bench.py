#!/usr/bin/env python3
"""Benchmark of the W4A16 GEMM on GB300 (one JSON line on stdout).

A step is one call of the hot path (wq4_mm, or wq4_grouped_mm for the grouped workload) on one
batch of seeded synthetic input already resident in HBM; every weight is prepacked before timing
(prepack is the offline step of the method). Each workload keeps R rotating copies of all its
inputs (each weight prepacked into its own blob; R x working set > 3 x L2), and a CUDA graph of
L = max(K, R) launches walks them, so the data each launch reads was evicted from L2 by the
launches in between. After an untimed soak, 7 replays are timed with CUDA events on the launching
stream (max over ranks); the line reports the median per launch and the min / max.

The default run measures the five workloads one after the other, each with constant weights
(WQ4_OPT_CONST_WEIGHTS: weights prepacked once and not written by pending work, so the kernels
start streaming them before the kernel ahead completes) and in plain stream order. The headline
(value, roofline, e2e, cpu_baseline) is the decode workload with constant weights; its
stream-ordered number is in "stream_ordered", and every workload's own line (rate, roofline,
clocks, and its stream-ordered figures) is under "workloads".

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--stream-order]
                  [--impl reference]

Variants of a workload (measured like the workload itself; the default line uses none):
  --group-size G / --no-scales   other group sizes, or uint4b8 without scales (direct conversion)
  --epilogue                     Y = X.dequant(W)^T + C + bias through wq4_mm_ex (C, bias read)
  --float-zeros                  the workload's weight in the float-zero format (value = q s + zf)
  --device-m                     grouped workload with its token counts in device memory
  --dev-ptrs                     grouped workload with its X / W / Y pointers in device memory

With N > 1 (launched by torch.distributed.run) every rank runs its own replica of the workload
(weak scaling; the GEMM needs no exchange) and value = all ranks' work / max time.
--impl reference times the CPU oracle (fp64 NumPy) on this host's cores instead.
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
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import wq4_inputs as I  # noqa: E402

METRIC = "W4A16 GEMM TFLOP/s and HBM GB/s vs GB300 roofline, M=8..4096 (1 GPU)"
DEFAULT_WORKLOAD = "decode_m8_n4096_k4096_bf16_u4b8"
L2_BYTES = 129 * 1024 * 1024
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16": p["bf16_tflops"], "bf16_sust": p["bf16_tflops_sustained"],
                "src": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16": 1900.0, "bf16_sust": 1700.0, "src": "fallback"}


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "weight_only_quantized_wq4_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode())
            h.update(fh.read())
    return h.hexdigest()[:16]


def variant_of(args):
    """Non-default variant flags as config entries (empty for the plain workload)."""
    v = {}
    if args.group_size != I.GROUP:
        v["group_size"] = args.group_size
    if args.no_scales:
        v["scales"] = "none (direct conversion)"
    if args.epilogue:
        v["epilogue"] = "Y = acc + C + bias (wq4_mm_ex)"
    if args.device_m:
        v["token_counts"] = "device memory (wq4_grouped_mm_device_m)"
    if getattr(args, "dev_ptrs", False):
        v["pointers"] = "device memory (wq4_grouped_mm_dev_ptrs)"
    if getattr(args, "float_zeros", False):
        v["qtype"] = "u4_fzp (value = q s + zf, float zero per group and row)"
    return v


def make_inputs(args):
    """The workload's seeded problems, drawn with the variant's group size / scales."""
    spec = dict(I.WORKLOADS[args.workload])
    kind = spec.pop("kind")
    if args.no_scales and spec["qtype"] != I.U4B8:
        raise SystemExit("--no-scales applies to uint4b8 weights")
    if getattr(args, "float_zeros", False):
        spec["qtype"] = I.U4_FZP
    if kind == "mm":
        return I.make_problem(**spec, group_size=args.group_size, scaled=not args.no_scales)
    if args.group_size != I.GROUP or args.no_scales or args.epilogue:
        raise SystemExit("--group-size, --no-scales and --epilogue apply to single-problem workloads")
    return I.make_grouped(**spec)


def variant_bytes(p, args):
    """Algorithmic bytes of one problem under the variant: the scales it really has, and C and
    bias read by the epilogue."""
    b = I.algorithmic_bytes(p.M, p.N, p.K, p.qtype, args.group_size)
    if args.no_scales:
        b -= 2 * (p.K // args.group_size) * p.N
    if args.epilogue:
        b += 2 * p.M * p.N + 2 * p.N
    return b


def workload_shapes(name, probs):
    if isinstance(probs, list):
        Ms = [p.M for p in probs]
        byts = sum(I.algorithmic_bytes(p.M, p.N, p.K, p.qtype) for p in probs)
        flops = sum(I.algorithmic_flops(p.M, p.N, p.K) for p in probs)
        cfg = {"workload": name, "problems": len(probs), "M_list": Ms, "N": probs[0].N, "K": probs[0].K,
               "group_size": 128, "qtype": probs[0].qtype}
        return byts, flops, cfg, probs[0].dtype
    p = probs
    cfg = {"workload": name, "M": p.M, "N": p.N, "K": p.K, "group_size": 128, "qtype": p.qtype}
    return I.algorithmic_bytes(p.M, p.N, p.K, p.qtype), I.algorithmic_flops(p.M, p.N, p.K), cfg, p.dtype


def bound_of(byts, flops, pk):
    # ridge point of the measured rooflines
    return "tensor" if flops / byts > (pk["bf16"] * 1e12) / (pk["hbm_gbs"] * 1e9) else "hbm"


class ClockSampler:
    """nvidia-smi samples (every 100 ms) of SM clock and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = []
        for ts, line in self.lines:
            if t0 <= ts <= t1:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 8:
                    rows.append(parts)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[4 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------------------------ GPU arm
ALL_WORKLOADS = ["tiny_m16_n256_k512_fp16_u4b8", "decode_m8_n4096_k4096_bf16_u4b8", "asym_m128_n14336_k4096_bf16_u4zp",
                 "prefill_m4096_n4096_k14336_bf16_u4b8", "grouped_8x_n14336_k4096_summ1024_bf16_u4b8"]
REPLAYS = 7


class Workload:
    """One workload resident in HBM: R rotating copies of every input (each weight prepacked with
    wq4_prepack into its own blob), so that the data each launch reads was evicted from L2 by the
    launches in between, and the call a step makes."""

    def __init__(self, args, name, dev, use_variant):
        import torch
        import weight_only_quantized_wq4_gb300 as wq4
        self.name = name
        self.args = args
        self.dev = dev
        vargs = args if use_variant else argparse.Namespace(group_size=I.GROUP, no_scales=False, epilogue=False,
                                                           device_m=False, float_zeros=False, dev_ptrs=False,
                                                           workload=name)
        self.vargs = vargs
        probs = make_inputs(argparse.Namespace(**dict(vars(vargs), workload=name)))
        self.probs = probs
        self.grouped = isinstance(probs, list)
        dev_ptrs = getattr(vargs, "dev_ptrs", False)
        if (vargs.device_m or dev_ptrs) and not self.grouped:
            raise SystemExit("--device-m and --dev-ptrs apply to the grouped workload")
        if vargs.device_m and dev_ptrs:
            raise SystemExit("--device-m and --dev-ptrs are separate calls")
        plist = probs if self.grouped else [probs]
        self.plist = plist
        byts, flops, cfg, dtype = workload_shapes(name, probs)
        self.variant = variant_of(vargs)
        if self.variant:
            byts = sum(variant_bytes(p, vargs) for p in plist)
            cfg = dict(cfg, **self.variant)
        self.byts, self.flops, self.cfg, self.dtype = byts, flops, cfg, dtype
        tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
        self.tdt = tdt
        G = vargs.group_size

        def c16(bits):
            return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(tdt).to(dev)

        def c32(words):
            return torch.from_numpy(np.ascontiguousarray(words).view(np.int32)).to(dev)

        def zeros(p):
            if p.Z is None:
                return None
            return c16(p.Z) if p.qtype == I.U4_FZP else c32(p.Z)

        src = [(c32(p.Wq), c16(p.S_bits) if p.S_bits is not None else None, zeros(p)) for p in plist]

        def blobs():
            return [wq4.prepack(wq, sc, z, qtype=p.qtype, group_size=G, dtype=dtype) for (wq, sc, z), p in zip(src, plist)]

        base_X = [c16(p.X_bits) if p.M > 0 else torch.empty((0, p.K), dtype=tdt, device=dev) for p in plist]
        self.base_W = blobs()
        rng = np.random.default_rng(7)
        self.base_C = [c16(I.f32_to_bits(rng.standard_normal((p.M, p.N)).astype(np.float32), dtype)) for p in plist] \
            if vargs.epilogue else None
        self.base_b = [c16(I.f32_to_bits(rng.standard_normal(p.N).astype(np.float32), dtype)) for p in plist] \
            if vargs.epilogue else None
        qtype = plist[0].qtype
        if vargs.device_m:
            self.ws_bytes = wq4.grouped_device_m_workspace_bytes(len(plist))
        elif dev_ptrs:
            self.ws_bytes = wq4.grouped_dev_ptrs_workspace_bytes([p.M for p in plist], [p.N for p in plist],
                                                                 [p.K for p in plist], G)
        elif self.grouped:
            self.ws_bytes = wq4.grouped_workspace_bytes([p.M for p in plist], [p.N for p in plist], [p.K for p in plist],
                                                        G, plist[0].qtype)
        else:
            self.ws_bytes = wq4.workspace_bytes(plist[0].M, plist[0].N, plist[0].K, G, plist[0].qtype)
        self.set_bytes = sum(x.numel() * 2 for x in base_X) + sum(w.numel() for w in self.base_W) + \
            sum(p.M * p.N * 2 for p in plist) * (2 if vargs.epilogue else 1) + self.ws_bytes
        M_dev = torch.tensor([p.M for p in plist], dtype=torch.int32, device=dev) if vargs.device_m else None
        self.R = max(2, math.ceil(3 * L2_BYTES / self.set_bytes))
        self.copies = []
        for r in range(self.R):
            Xs = [x.clone() for x in base_X]
            Ws = self.base_W if r == 0 else blobs()
            Ys = [torch.empty((p.M, p.N), dtype=tdt, device=dev) for p in plist]
            ws = wq4.alloc_workspace(self.ws_bytes, dev)
            Cs = [c.clone() for c in self.base_C] if vargs.epilogue else None
            self.copies.append((Xs, Ws, Ys, ws, Cs))
        del src
        torch.cuda.synchronize()
        grouped = self.grouped

        ptr_arrays = {}     # device pointer arrays per set of buffers, made before any timing or capture

        def dev_ptr_arrays(Xs, Ws, Ys):
            key = tuple(t.data_ptr() for t in Xs + Ws + Ys)
            if key not in ptr_arrays:
                ptr_arrays[key] = [torch.tensor([t.data_ptr() for t in ts], dtype=torch.int64, device=dev)
                                   for ts in (Xs, Ws, Ys)]
            return ptr_arrays[key]

        if dev_ptrs:
            for Xs, Ws, Ys, _, _ in self.copies:
                dev_ptr_arrays(Xs, Ws, Ys)
        self.dev_ptr_arrays = dev_ptr_arrays

        def call(Xs, Ws, Ys, ws, Cs, bias):
            if dev_ptrs:
                wq4.grouped_mm_dev_ptrs([p.M for p in plist], [p.N for p in plist], [p.K for p in plist],
                                        *dev_ptr_arrays(Xs, Ws, Ys), dtype=dtype, qtype=qtype, workspace=ws,
                                        group_size=G)
            elif vargs.device_m:
                wq4.grouped_mm_device_m(Xs, Ws, M_dev, [p.N for p in plist], qtype=qtype, workspace=ws, outs=Ys,
                                        group_size=G)
            elif grouped:
                wq4.grouped_mm(Xs, Ws, [p.N for p in plist], qtype=qtype, workspace=ws, outs=Ys, group_size=G)
            elif vargs.epilogue:
                wq4.mm(Xs[0], Ws[0], plist[0].N, qtype=qtype, workspace=ws, out=Ys[0], group_size=G, C=Cs[0],
                       beta=1.0, bias=bias[0])
            else:
                wq4.mm(Xs[0], Ws[0], plist[0].N, qtype=qtype, workspace=ws, out=Ys[0], group_size=G)

        self.call = call
        # device counts: the tile-table kernel too; device pointers: one set-up launch per 128 problems
        self.launches_per_step = 2 if vargs.device_m else (1 + (len(plist) + 127) // 128 if dev_ptrs else 1)

    def step(self, c):
        Xs, Ws, Ys, ws, Cs = self.copies[c % self.R]
        self.call(Xs, Ws, Ys, ws, Cs, self.base_b)

    def time(self, steps, warmup, world, soak_s, no_graph=False):
        """W eager warm-up steps, then a CUDA graph of L = max(steps, R) launches (so one replay walks
        every rotating copy); after an untimed soak of replays, REPLAYS timed replays, each between
        a barrier and a synchronize, timed with CUDA events on the launching stream; per-launch
        times (max over ranks) and the wall-clock window of soak + timing (for the clock record)."""
        import torch
        import weight_only_quantized_wq4_gb300 as wq4
        L = max(steps, self.R)
        stream = torch.cuda.Stream(self.dev)
        with torch.cuda.stream(stream):
            for i in range(warmup):
                self.step(i)
            torch.cuda.synchronize()
            graph = None
            if not no_graph:
                graph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(graph, stream=stream):
                    for i in range(L):
                        self.step(i)
                torch.cuda.synchronize()
        assert wq4.get_last_error(self.dev) == 0

        def replay():
            with torch.cuda.stream(stream):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                if graph is not None:
                    graph.replay()
                else:
                    for i in range(L):
                        self.step(i)
                e1.record(stream)
                e1.synchronize()
                return e0.elapsed_time(e1)

        t_soak = time.time()
        replay()
        while time.time() - t_soak < soak_s:
            replay()
        per_launch = []
        for _ in range(REPLAYS):
            _barrier(world)
            torch.cuda.synchronize()
            ms = replay()
            torch.cuda.synchronize()
            per_launch.append(_max_over_ranks(ms, world) / L)
        t_end = time.time()
        _barrier(world)
        assert wq4.get_last_error(self.dev) == 0
        del graph
        return per_launch, L, t_soak, t_end


def summarize(w, per_launch, L, pk, world, clocks):
    """Median per-launch time, both rates, the roofline of the bound this workload sits under."""
    ms = statistics.median(per_launch)
    gbs = w.byts / (ms * 1e-3) / 1e9
    tfl = w.flops / (ms * 1e-3) / 1e12
    bound = bound_of(w.byts, w.flops, pk)
    traffic = None
    try:
        if w.variant:
            raise LookupError("no capture of the variant")
        with open(PROFILE_TRAFFIC) as f:
            tr = json.load(f)
        ent = tr.get(w.name)
        if ent and ent.get("kernel_hash") == kernel_source_hash():
            traffic = ent["bytes_per_launch"]
    except Exception:
        pass
    if bound == "hbm":
        roof = {"bound": "hbm", "achieved": round(gbs, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": round(gbs / pk["hbm_gbs"], 4), "traffic": traffic,
                "peak_source": pk["src"] + " (burst copy)"}
        value, unit = gbs * world, "GB/s"
    else:
        roof = {"bound": "tensor", "achieved": round(tfl, 1), "peak": pk["bf16"], "unit": "TFLOP/s",
                "frac": round(tfl / pk["bf16"], 4), "traffic": traffic,
                "peak_source": pk["src"] + " (bf16 burst)",
                "frac_vs_sustained": round(tfl / pk["bf16_sust"], 4)}
        value, unit = tfl * world, "TFLOP/s"
    return {"value": round(value, 3), "unit": unit, "ms_per_step": ms,
            "ms_per_step_min": min(per_launch), "ms_per_step_max": max(per_launch),
            "tflops": round(tfl, 3), "gbs": round(gbs, 1), "roofline": roof, "clocks": clocks,
            "launches_per_replay": L, "bound": bound}


def run_gpu(args, rank, world, local_rank):
    import torch
    import weight_only_quantized_wq4_gb300 as wq4

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    wq4.build()
    wq4.load_library()
    if args.a_in_smem:
        wq4.set_option(wq4.OPT_A_IN_SMEM, 1)
    pk = peaks()
    names = [args.workload] if args.workload else ALL_WORKLOADS
    headline = args.workload or DEFAULT_WORKLOAD
    soak = 0.0 if args.profile_run else 1.0

    sampler = ClockSampler(local_rank)
    if not args.profile_run:
        sampler.start()
        time.sleep(0.3)
    results = {}
    head = None
    for name in names:
        w = Workload(args, name, dev, use_variant=(name == headline))
        modes = [("stream", 0)]
        if not args.stream_order:
            modes = [("const", 1), ("stream", 0)]        # constant weights first: the reported figure
        out = {}
        for mode, cw in modes:
            wq4.set_option(wq4.OPT_CONST_WEIGHTS, cw)
            per, L, t0, t1 = w.time(args.steps, args.warmup, world, soak, args.no_graph)
            out[mode] = summarize(w, per, L, pk, world, sampler.summary(t0, t1) if not args.profile_run else None)
        wq4.set_option(wq4.OPT_CONST_WEIGHTS, 0)
        first = out[modes[0][0]]
        entry = dict(first, config=w.cfg, weights="constant (WQ4_OPT_CONST_WEIGHTS)" if modes[0][0] == "const"
                     else "stream order")
        if len(modes) > 1:
            entry["stream_ordered"] = {k: out["stream"][k] for k in ("value", "unit", "ms_per_step", "ms_per_step_min",
                                                                    "ms_per_step_max", "roofline", "clocks")}
        results[name] = entry
        if name == headline:
            head = (w, first, out.get("stream"), modes[0][0])
        else:
            del w
            torch.cuda.empty_cache()
    sampler.stop()

    w, first, stream_res, mode = head
    bound = first["bound"]
    # end to end through the public API from pinned host buffers: H2D of the step's inputs (the
    # activations and the prepacked weight), the call, D2H of the result. The weight is written by
    # a copy on the stream every step, so this runs in stream order (no constant-weight promise).
    e2e = None if args.profile_run else run_e2e(args, w.plist, w.base_W, w.base_C, w.base_b, w.call, w.ws_bytes, dev,
                                                 w.tdt, w.byts, w.flops, bound)
    cfg = dict(w.cfg, weights=("constant: prepacked once, read before the kernel ahead completes "
                               "(WQ4_OPT_CONST_WEIGHTS=1)") if mode == "const" else "stream order",
               l2="rotating %d input copies (%.0f MB, each weight prepacked into its own blob) > L2" % (
                   w.R, w.R * w.set_bytes / 1e6),
               launch=("CUDA graph of %d launches" % first["launches_per_replay"]) if not args.no_graph
               else "eager launches",
               timing="median of %d replays (per-launch min %.6f ms, max %.6f ms)" % (
                   REPLAYS, first["ms_per_step_min"], first["ms_per_step_max"]),
               parallelism="replicas" if world > 1 else "single GPU")
    out = {
        "metric": METRIC, "value": first["value"], "unit": first["unit"], "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": first["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic (seeded numpy, wq4_inputs)", "config": cfg,
        "tflops": first["tflops"], "gbs": first["gbs"], "frac_hbm_nominal_8tbs": round(first["gbs"] / 8000.0, 4),
        "roofline": first["roofline"],
        "gpu_launches": first["launches_per_replay"] * w.launches_per_step * REPLAYS,
        "clocks": first["clocks"],
        "e2e": e2e,
        "stream_ordered": results[headline].get("stream_ordered"),
        "workloads": results,
    }
    if w.variant:
        out["cpu_baseline"] = None   # the oracle's row-sampled step covers the plain workloads only
    elif rank == 0 and world == 1 and not args.no_cpu_baseline and not args.profile_run:
        out["cpu_baseline"] = cpu_baseline(headline, w.probs, w.byts, w.flops, bound, budget_s=args.cpu_seconds)
    return out


def run_e2e(args, plist, base_W, base_C, base_b, call, ws_bytes, dev, tdt, byts, flops, bound):
    """The same call from pinned host buffers: H2D of the step's inputs (activations, prepacked
    weight, and C and bias with the epilogue), the call, D2H of the result."""
    import torch
    import weight_only_quantized_wq4_gb300 as wq4
    steps = max(3, min(args.steps, 20))
    hX = [torch.from_numpy(np.ascontiguousarray(p.X_bits).view(np.int16)).view(tdt).pin_memory() for p in plist]
    hW = [w.cpu().pin_memory() for w in base_W]
    hC = [c.cpu().pin_memory() for c in base_C] if base_C is not None else []
    hb = [b.cpu().pin_memory() for b in base_b] if base_b is not None else []
    hY = [torch.empty((p.M, p.N), dtype=tdt).pin_memory() for p in plist]
    dX = [torch.empty_like(x, device=dev) for x in hX]
    dW = [torch.empty_like(w, device=dev) for w in hW]
    dC = [torch.empty_like(c, device=dev) for c in hC]
    db = [torch.empty_like(b, device=dev) for b in hb]
    dY = [torch.empty((p.M, p.N), dtype=tdt, device=dev) for p in plist]
    ws = wq4.alloc_workspace(ws_bytes, dev)
    stream = torch.cuda.Stream(dev)
    h2d = sum(t.numel() * t.element_size() for t in hX + hW + hC + hb)
    d2h = sum(y.numel() * 2 for y in hY)

    def one():
        for a, b in zip(dX + dW + dC + db, hX + hW + hC + hb):
            a.copy_(b, non_blocking=True)
        call(dX, dW, dY, ws, dC or None, db or None)
        for a, b in zip(hY, dY):
            a.copy_(b, non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(3):
            one()
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            one()
        e1.record(stream)
        e1.synchronize()
    ms = e0.elapsed_time(e1) / steps
    if bound == "hbm":
        v, u = byts / (ms * 1e-3) / 1e9, "GB/s"
    else:
        v, u = flops / (ms * 1e-3) / 1e12, "TFLOP/s"
    return {"value": round(v, 3), "unit": u, "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "ms_per_step": ms, "steps": steps}


# ------------------------------------------------------------------------------------ CPU oracle
def _rows_of(p, n):
    """The sub-problem made of the first n weight rows (outputs Y[:, :n] of the full problem)."""
    return I.Problem(p.M, n, p.K, p.dtype, p.qtype, p.X_bits, p.q[:n], p.Wq[:n], p.S_bits[:, :n],
                     None if p.z is None else p.z[:, :n], None if p.Z is None else p.Z[:, :n // 8])


def oracle_step(probs, frac):
    """The oracle on a fraction of every problem's weight rows (its dequantisation and product
    both scale linearly with the rows)."""
    import oracle as O
    plist = probs if isinstance(probs, list) else [probs]
    out = []
    for p in plist:
        if p.M == 0:
            continue
        n = max(128, int(round(p.N * frac / 128)) * 128) if frac < 1 else p.N
        out.append(O.mm_problem(_rows_of(p, n)))
    return out


def calibrate(probs, seconds):
    """Fraction of weight rows that makes one oracle step take about `seconds`."""
    plist = probs if isinstance(probs, list) else [probs]
    f0 = min(1.0, 1024.0 / max(p.N for p in plist))
    t0 = time.perf_counter()
    oracle_step(probs, f0)
    dt = time.perf_counter() - t0
    f = min(1.0, f0 * seconds / max(dt, 1e-6))
    n_rows = max(p.N for p in plist)
    return max(128.0 / n_rows, round(f * n_rows / 128) * 128 / n_rows)


def _sample_text(probs, frac):
    plist = probs if isinstance(probs, list) else [probs]
    if frac >= 1:
        return "the whole step"
    return "the first %d of %d weight rows of every problem (all tokens), time scaled by %d/%d" % (
        max(128, int(round(plist[0].N * frac / 128)) * 128), plist[0].N, plist[0].N,
        max(128, int(round(plist[0].N * frac / 128)) * 128))


def _scaled_step_time(probs, frac, dt):
    plist = probs if isinstance(probs, list) else [probs]
    if frac >= 1:
        return dt
    n = max(128, int(round(plist[0].N * frac / 128)) * 128)
    return dt * plist[0].N / n


def _as_metric(bound, byts, flops, dt):
    if bound == "hbm":
        return byts / dt / 1e9, "GB/s"
    return flops / dt / 1e12, "TFLOP/s"


def cpu_baseline(name, probs, byts, flops, bound, budget_s=15.0):
    """The oracle as it stands on this host's cores, about budget_s seconds of work."""
    frac = calibrate(probs, 1.0)
    oracle_step(probs, frac)          # warm-up
    t0 = time.perf_counter()
    n = 0
    while True:
        oracle_step(probs, frac)
        n += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = _scaled_step_time(probs, frac, (time.perf_counter() - t0) / n)
    v, u = _as_metric(bound, byts, flops, dt)
    return {"value": v, "unit": u, "cores": os.cpu_count(), "kind": "oracle",
            "sample": "%d repetition(s) of %s" % (n, _sample_text(probs, frac)),
            "seconds_per_step": dt, "note": "fp64 NumPy dequantise + matmul; a baseline, not a target"}


def run_reference(args, rank, world):
    pk = peaks()
    name = args.workload or DEFAULT_WORKLOAD
    probs = I.make_workload(name)
    byts, flops, cfg, dtype = workload_shapes(name, probs)
    bound = bound_of(byts, flops, pk)
    per_step = max(0.05, min(2.0, 120.0 / (args.steps + args.warmup)))
    frac = calibrate(probs, per_step)
    for _ in range(args.warmup):
        oracle_step(probs, frac)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(probs, frac)
    dt = _scaled_step_time(probs, frac, (time.perf_counter() - t0) / args.steps)
    v, u = _as_metric(bound, byts, flops, dt)
    sample = "each step: " + _sample_text(probs, frac)
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": u, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded numpy, wq4_inputs)", "config": cfg,
            "cpu_baseline": {"value": v, "unit": u, "cores": os.cpu_count(), "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": u, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ------------------------------------------------------------------------------------ ranks
def _barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _max_over_ranks(v, world):
    if world <= 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=None, choices=sorted(I.WORKLOADS),
                    help="one workload only (default: all five, the decode one as the headline)")
    ap.add_argument("--impl", default="wq4", choices=["wq4", "reference"])
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--a-in-smem", action="store_true", help="dequantised operand via shared memory")
    ap.add_argument("--stream-order", action="store_true",
                    help="every workload in stream order only (default: constant weights, WQ4_OPT_CONST_WEIGHTS, "
                         "then stream order)")
    ap.add_argument("--group-size", type=int, default=I.GROUP, help="variant: quantisation group size")
    ap.add_argument("--no-scales", action="store_true", help="variant: uint4b8 weights without scales")
    ap.add_argument("--epilogue", action="store_true", help="variant: Y = acc + C + bias (wq4_mm_ex)")
    ap.add_argument("--device-m", action="store_true", help="variant: grouped token counts in device memory")
    ap.add_argument("--dev-ptrs", action="store_true", help="variant: grouped X / W / Y pointers in device memory")
    ap.add_argument("--float-zeros", action="store_true", help="variant: the weight in the float-zero format")
    ap.add_argument("--profile-run", action="store_true",
                    help="only warm-up and the timed replay (for profiler runs): no soak, e2e or CPU baseline")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args, rank, world)), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    out = run_gpu(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
