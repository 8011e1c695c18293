#!/usr/bin/env python3
"""Benchmark of the activation-sparse (TwELL) FFN hot path on one GB300.

One step = one pass of the whole hot path over one batch of synthetic input:
the training forward (gate GEMM + ReLU + TwELL pack, hybrid split, fused sparse
up/down, dense fallback rows, saved activations) and the sparse backward with
the L1 term, on the gated bf16 FFN with T=4096, d_model=2048, d_ff=8192,
tile 128, K=8, ~99% sparse (bias -2.33), lambda = 1e-4.  ``--mode fwd`` times
the inference forward alone.

Prints ONE JSON line (rank 0).  Multi-GPU: every rank runs its own replica of
the workload (weak scaling, no collective on the data path); the timed region
is bracketed by a barrier and a device synchronisation, and the time is the
maximum over ranks.

``--impl reference`` times the CPU oracle instead (a bounded sample of the
same workload per step) and prints the same line with "impl": "reference".
"""
from __future__ import annotations

import argparse
import csv
import datetime
import ctypes
import hashlib
import io
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "sparse-FFN tokens/s at 99% sparsity vs dense cuBLAS; gather HBM GB/s vs 8 TB/s"


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--mode", choices=["train", "fwd"], default="train")
    ap.add_argument("--workload", default="c2",
                    help="c2 | c3 | c4:<bias>:<K> (shapes of the pages' setting)")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--no-dense", action="store_true", help="skip the cuBLAS dense FFN")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-energy", action="store_true",
                    help="skip the saved-memory and energy-per-token leg")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--shard", choices=["replicas", "tokens"], default="replicas",
                    help="N > 1: one replica of the workload per rank (weak scaling), or the "
                         "batch's tokens split over the ranks with the weight gradients summed "
                         "by an all-reduce in every step (strong scaling)")
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the compact records of the other workloads' forward")
    ap.add_argument("--compare-formats", action="store_true",
                    help="forward: TwELL against classic row-ELL and against an unfused pack "
                         "(dense gate GEMM + standalone conversion), same inputs")
    ap.add_argument("--dense-density", type=float, default=0.0,
                    help="the dispatcher's density threshold (0: the library default; "
                         "< 0: off; a tiny value forces the all-dense path)")
    ap.add_argument("--dh-density", type=float, default=0.0,
                    help="backward: slot density above which dh comes from the tensor-core "
                         "GEMM read at the slots (0: the library default; < 0: always the "
                         "gather SDDMM; a tiny value: always the GEMM)")
    ap.add_argument("--gather-passes", type=int, default=0,
                    help="passes of the gather kernels over their matrices / d_model columns "
                         "(0: the library's choice from L2 size; 1: one pass)")
    return ap.parse_args()


def workload_of(name: str, train: bool) -> synth.Workload:
    if name == "c1":
        w = synth.config1()
    elif name == "c2":
        w = synth.config5() if train else synth.config2()
    elif name == "c3":
        w = synth.config3()
    elif name.startswith("c4"):
        _, b, k = name.split(":")
        w = synth.config4(float(b), int(k))
    else:
        raise SystemExit(f"unknown workload {name}")
    if train and not w.train:
        w = synth.scaled(w, lam=1e-4, train=True)
    return w


def describe(w: synth.Workload, train: bool) -> str:
    from scipy.stats import norm
    zero = 100.0 * norm.cdf(-w.bias) if w.bias < 0 else 100.0 * (1 - norm.cdf(w.bias))
    kind = f"training step (fwd+bwd, L1 lambda={w.lam})" if train else "inference forward"
    s = (f"{kind} of the {'gated' if w.gated else 'plain'} ReLU FFN, {w.dtype}, T={w.T} "
         f"d_model={w.D} d_ff={w.F}, TwELL tile {w.C} K={w.K}, gate bias {w.bias} "
         f"(~{zero:.1f}% zero)")
    if w.hot_tokens:
        s += f", first {w.hot_tokens} of every {w.seq_len} tokens at bias {w.bias + w.hot_bias:.2f}"
    return s


class ClockSampler:
    """nvidia-smi samples of the SM clock and throttle reasons while running."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(index), f"--query-gpu=timestamp,{self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in csv.reader(io.StringIO(out)):
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                continue
            for nm, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(nm)
        busy = [c for c in sm if c >= 0.5 * max(sm)] if sm else []
        return {"sm_mhz": float(np.median(busy)) if busy else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def upload(torch, dev, v):
    if v is None:
        return None
    if v.dtype == np.uint16:
        return torch.from_numpy(v.view(np.int16)).view(torch.bfloat16).to(dev)
    return torch.from_numpy(v).to(dev)


class Bench:
    """Device state of one workload: inputs, TwELL buffers, workspace, outputs
    and the step (forward, or forward + backward) through the C ABI."""

    def __init__(self, torch, tw, w, train, dev, args, a=None):
        self.torch, self.tw, self.w, self.train, self.dev = torch, tw, w, train, dev
        self.a = synth.generate(w) if a is None else a
        self.dtype = tw.TWELL_BF16 if w.dtype == "bf16" else tw.TWELL_F32
        tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
        self.d = d = {k: upload(torch, dev, self.a[k]) for k in ("x", "Wg", "Wu", "Wd", "bg", "rb", "dy")}
        T, D, F = w.T, w.D, w.F
        self.bufs = tw.TwellBuffers(T, F, w.C, w.K, self.dtype, train=train, device=dev,
                                    dense_density=args.dense_density,
                                    dh_density=args.dh_density,
                                    gather_passes=args.gather_passes)
        self.ws, self.nws = tw.workspace(T, D, F, w.C, w.K, self.dtype, train, device=dev)
        self.y = torch.empty((T, D), dtype=tdt, device=dev)
        self.dx = self.dWg = self.dWu = self.dWd = self.dbg = None
        if train:
            self.dx = torch.empty_like(d["x"])
            self.dWg = torch.empty((F, D), dtype=torch.float32, device=dev)
            self.dWu = torch.empty_like(self.dWg) if w.gated else None
            self.dWd = torch.empty_like(self.dWg)
            self.dbg = torch.empty((F,), dtype=torch.float32, device=dev)
        self.stream = torch.cuda.current_stream(dev)
        self.sh = self.stream.cuda_stream

    def step(self, x=None, dy=None, y_out=None, dx_out=None):
        tw, d, w = self.tw, self.d, self.w
        xx = d["x"] if x is None else x
        tw.twell_ffn_forward(xx, d["Wg"], d["bg"], d["rb"], d["Wu"], d["Wd"], w.D, int(self.train),
                             self.bufs.t, self.y if y_out is None else y_out, self.ws, self.nws,
                             self.sh)
        if self.train:
            tw.twell_ffn_backward(xx, d["Wg"], d["Wu"], d["Wd"], self.bufs.t,
                                  d["dy"] if dy is None else dy, w.lam, w.D,
                                  self.dx if dx_out is None else dx_out, self.dWg, self.dbg,
                                  self.dWu, self.dWd, self.ws, self.nws, self.sh)

    def status(self):
        return self.tw.twell_get_status(self.bufs.t, self.sh)

    def dispatch(self):
        """Rows the dispatcher sent to the dense path (control block n_rows) in
        a lone forward and in the backward that follows it, and whether the
        backward took dh from the tensor-core GEMM."""
        torch, tw, d, w = self.torch, self.tw, self.d, self.w
        tw.twell_ffn_forward(d["x"], d["Wg"], d["bg"], d["rb"], d["Wu"], d["Wd"], w.D,
                             int(self.train), self.bufs.t, self.y, self.ws, self.nws, self.sh)
        torch.cuda.synchronize(self.dev)
        rows_f = int(self.ws[:4].view(torch.int32).item())
        rows_b, dh_gemm = 0, False
        if self.train:
            tw.twell_ffn_backward(d["x"], d["Wg"], d["Wu"], d["Wd"], self.bufs.t, d["dy"], w.lam,
                                  w.D, self.dx, self.dWg, self.dbg, self.dWu, self.dWd, self.ws,
                                  self.nws, self.sh)
            torch.cuda.synchronize(self.dev)
            rows_b = int(self.ws[:4].view(torch.int32).item())
            dh_gemm = bool(self.ws[24:28].view(torch.int32).item())  # control block: dh_gemm
        return rows_f, rows_b, dh_gemm


def make_timer(torch, dev, stream, flush_buf):
    per_step = []

    def timed(fn, steps, flush=True):
        """Sum of per-step device times (CUDA events on the launching stream),
        with the L2 flushed by a large write before every step (flush=False:
        back to back, warm L2); the per-step times are kept in per_step."""
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        for e0, e1 in evs:
            if flush:
                flush_buf.fill_(1)
            e0.record(stream)
            fn()
            e1.record(stream)
        torch.cuda.synchronize(dev)
        per_step[:] = [e0.elapsed_time(e1) for e0, e1 in evs]
        return sum(per_step)

    return timed, per_step


def kernel_profile(torch, lib, b, flush_buf, prof_steps):
    """Per-kernel times inside the step: events the library records between
    its own launches on the launch stream (one stream while this is on)."""
    lib.twell_profile_begin()
    for _ in range(prof_steps):
        flush_buf.fill_(1)
        b.step()
    torch.cuda.synchronize(b.dev)
    cap = 64 * prof_steps
    ids = (ctypes.c_int * cap)()
    ms = (ctypes.c_float * cap)()
    nl = (ctypes.c_int * cap)()
    cnt = ctypes.c_int(0)
    lib.twell_kernel_name.restype = ctypes.c_char_p
    lib.twell_profile_end_ex(cap, ids, ms, nl, ctypes.byref(cnt))
    per = {}
    for i in range(min(cnt.value, cap)):
        per.setdefault(lib.twell_kernel_name(ids[i]).decode(), []).append(ms[i])
    launches_per_step = sum(nl[i] for i in range(min(cnt.value, cap))) / prof_steps
    kern = {k: {"launches_per_step": len(v) / prof_steps, "avg_ms": float(np.mean(v)),
                "ms_per_step": float(np.sum(v)) / prof_steps} for k, v in per.items()}
    return kern, launches_per_step


def dominant_roofline(kern, rl, workload, train, gceil):
    """The contract's roofline object for the kernel with the largest time
    per step.  A tensor-core kernel is read against the measured bf16 peak.
    A gather kernel whose rows are served from L2 (the weight rows it
    re-reads fit in L2; ncu DRAM bytes are a small fraction of its
    algorithmic bytes) is read against the rate this GPU reaches on the same
    random-row gather pattern, measured in the same run (bound "l2"); its
    figures against the HBM copy peak are kept beside it, both on algorithmic
    bytes and on the ncu DRAM bytes."""
    dominant = max((k for k in kern if k in rl), key=lambda k: kern[k]["ms_per_step"],
                   default=None)
    if not dominant:
        return None
    r = rl[dominant]
    traffic = traffic_for(dominant, workload, train)
    src = "random-row gather probe on the same matrix and pair count"
    if isinstance(gceil, dict):  # per kernel: the rows it gathers (weight or token rows)
        src = gceil.get("_source", {}).get(dominant, src)
        gceil = gceil.get(dominant)
    if r["bound"] != "hbm" or not gceil:
        return {"kernel": dominant, "bound": r["bound"], "achieved": round(r["achieved"], 2),
                "peak": r["peak"], "unit": r["unit"], "frac": round(r["frac"], 4),
                "traffic": traffic, "peak_source": r["peak_source"]}
    sec = kern[dominant]["avg_ms"] / 1e3
    hbm = {"peak_gbs": r["peak"], "peak_source": r["peak_source"],
           "frac_algorithmic_bytes": round(r["frac"], 4),
           "frac_dram_bytes": (round(traffic / sec / 1e9 / r["peak"], 4) if traffic else None)}
    return {"kernel": dominant, "bound": "l2", "achieved": round(r["achieved"], 2),
            "peak": round(gceil, 1), "unit": "GB/s", "frac": round(r["achieved"] / gceil, 4),
            "traffic": traffic,
            "peak_source": f"measured in this run: {src} (the memory level that serves these "
                           "gathers)",
            "hbm": hbm}


def measure(torch, lib, b, timed, per_step, flush_buf, args, steps, w_key, full=True):
    """Time one workload: the sparse step (cold L2), per-kernel times and
    rooflines, the gather ceiling, and the two dense cuBLAS arms."""
    w, train = b.w, b.train
    for _ in range(3):
        b.step()
    code, n_ovf = b.status()
    if code != 0:
        raise SystemExit(f"device status {code} after warm-up ({w.name})")
    ms = timed(b.step, steps) / steps
    med = sorted(per_step)[len(per_step) // 2]
    code, n_ovf = b.status()
    if code != 0:
        raise SystemExit(f"device status {code} after the timed steps ({w.name})")
    kern, launches = kernel_profile(torch, lib, b, flush_buf, 5 if not full else max(5, min(50, steps)))
    nnz = b.bufs.nnz.cpu().numpy().astype(np.int64)
    rows_f, rows_b, dh_gemm = b.dispatch()
    rl = kernel_rooflines(kern, w, nnz, train, rows_f, rows_b, dh_gemm)
    gceil = gceil_x = None
    if any(r.get("bound") == "hbm" for k, r in rl.items() if not k.startswith("_")):
        # weight rows (up/down, dh, dx) and, for the weight-gradient gather,
        # token rows of x (the rows it gathers: x and dy, T x d_model each)
        gceil = gather_ceiling(torch, b.dev, b.d["Wu"] if w.gated else b.d["Wd"], w,
                               rl["_counts"]["pairs_all"], timed, b.sh)
        if "bwd_dw_gather" in rl:
            gceil_x = gather_ceiling(torch, b.dev, b.d["x"], w, rl["_counts"]["pairs_all"], timed,
                                     b.sh, n_rows=w.T)
        for k, r in rl.items():
            c = gceil_x if k == "bwd_dw_gather" else gceil
            if r.get("bound") == "hbm" and c:
                r["frac_of_l2_gather"] = r["achieved"] / c
    ceilings = dict({k: gceil for k in rl if not k.startswith("_")},
                    bwd_dw_gather=gceil_x,
                    _source={"bwd_dw_gather": "random-row gather probe on x (token rows, as this "
                                              "kernel gathers x and dy rows), same pair count"})
    dense = None if args.no_dense else dense_arms(torch, b.d, w, train, timed, args, steps)
    row_ovf = (nnz > w.K).any(axis=0)
    rec = {"ms_per_step": round(ms, 5), "median_ms": round(med, 5),
           "tokens_per_s": round(w.T / (ms / 1e3), 1),
           "roofline": dominant_roofline(kern, rl, w_key, train, ceilings),
           "path": {"forward_all_dense": bool(rows_f >= w.T), "forward_dense_rows": rows_f,
                    "backward_dense_rows": rows_b if train else None,
                    "backward_dh_gemm": dh_gemm if train else None},
           "sparsity": {"active_frac": float(nnz.sum() / (w.T * w.F)), "n_ovf": int(row_ovf.sum())},
           "l2_gather_gbs": round(gceil, 1) if gceil else None,
           "l2_gather_token_rows_gbs": round(gceil_x, 1) if gceil_x else None}
    if dense:
        rec["dense_cublas"] = dense["eager"]
        rec["dense_gemm_only"] = dense["gemm_only"]
        rec["speedup_vs_dense"] = round(dense["eager"]["ms_per_step"] / ms, 4)
        rec["speedup_vs_dense_gemm_only"] = round(dense["gemm_only"]["ms_per_step"] / ms, 4)
    return rec, kern, rl, launches, nnz


SWEEP = ("c2", "c3", "c4:-1.28:8", "c4:-1.64:8", "c4:-2.33:8", "c4:-2.58:8", "c1")
# training steps of the larger workloads beside the headline one
SWEEP_TRAIN = ("c3", "c4:-2.58:8", "c4:-2.33:8")


def sweep(torch, tw, lib, dev, args, timed, per_step, flush_buf):
    """Compact records of the inference forward of the other workloads (the
    pages' shapes) and of the training step of the larger ones, each with
    its own dominant-kernel roofline and the two dense cuBLAS arms on the
    same inputs."""
    out = {}
    for key, train in [(k, False) for k in SWEEP] + [(k, True) for k in SWEEP_TRAIN]:
        w = workload_of(key, train)
        b = Bench(torch, tw, w, train, dev, args)
        rec, _, _, _, _ = measure(torch, lib, b, timed, per_step, flush_buf, args,
                                  20 if train else 30, key, full=False)
        rec = {"workload": describe(w, train), "dtype": w.dtype, **rec}
        out[f"{key}:{'train' if train else 'fwd'}"] = rec
        del b
        torch.cuda.empty_cache()
    return out


def run_ours(args, rank, world, local_rank):
    import torch
    import activation_sparse_transformer_gate_gb300 as tw
    from activation_sparse_transformer_gate_gb300 import _build

    if rank == 0:
        _build.build(variants=("", "hooks"))
    if world > 1:
        torch.distributed.barrier()
    lib = tw.load()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    torch.backends.cuda.matmul.allow_tf32 = False  # the fp32 dense arm stays fp32
    train = args.mode == "train"
    w = workload_of(args.workload, train)
    sharded = args.shard == "tokens" and world > 1
    if sharded:
        # token-sharded step: this rank's contiguous range of the batch; the
        # weight gradients are summed over the ranks inside the step
        from activation_sparse_transformer_gate_gb300 import shard
        a = synth.generate(w)
        t0, t1 = shard.token_range(w.T, rank, world)
        if t1 <= t0:
            raise SystemExit(f"rank {rank} has no tokens: T={w.T} over {world} ranks")
        a = {k: (v[t0:t1] if k in ("x", "dy", "rb") and v is not None else v) for k, v in a.items()}
        b = Bench(torch, tw, synth.scaled(w, T=t1 - t0), train, dev, args, a=a)
        local_step = b.step

        def sharded_step():
            local_step()
            if train:
                shard.allreduce_weight_grads([b.dWg, b.dWu, b.dWd, b.dbg])

        b.step = sharded_step
    else:
        b = Bench(torch, tw, w, train, dev, args)
    T = w.T
    stream = b.stream
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush_buf = torch.empty((max(2 * l2, 256 << 20),), dtype=torch.uint8, device=dev)
    timed, per_step = make_timer(torch, dev, stream, flush_buf)

    for _ in range(max(args.warmup, 3)):
        b.step()
    code, n_ovf = b.status()
    if code != 0:
        raise SystemExit(f"device status {code} after warm-up")
    sampler = None if (args.no_clocks or rank != 0) else ClockSampler(local_rank)
    if sampler:
        time.sleep(0.2)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    total_ms = timed(b.step, args.steps)
    step_ms = sorted(per_step)
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    total_ms = max_over_ranks(torch, total_ms, world, dev)
    clocks = sampler.stop() if sampler else None
    code, n_ovf = b.status()
    if code != 0:
        raise SystemExit(f"device status {code} after the timed region")
    ms_step = total_ms / args.steps
    value = (T if sharded else T * world) / (ms_step / 1e3)
    if rank != 0:
        return None
    if sharded:
        b.step = local_step  # the measurements below are of this rank's own work
    n_warm = max(10, min(args.steps, 100))
    warm_ms = timed(b.step, n_warm, flush=False) / n_warm

    rec, kern, rl, launches_per_step, nnz = measure(
        torch, lib, b, timed, per_step, flush_buf, args, max(10, min(args.steps, 200)),
        args.workload, full=True)
    d, bufs, ws, nws, y, sh = b.d, b.bufs, b.ws, b.nws, b.y, b.sh
    formats = (format_comparison(torch, lib, d, w, bufs, ws, nws, y, sh, timed, args)
               if (args.compare_formats and not train and w.gated) else None)
    e2e = None if args.no_e2e else end_to_end(torch, d, b.step, y, b.dx, w, train, timed, args,
                                              stream, flush_buf)
    mem = energy = None
    if not args.no_energy:
        mem, energy = memory_and_energy(torch, dev, local_rank, d, w, train, b.step, bufs, nws,
                                        int(row_ovf_count(bufs, w)))
        if w.dtype == "bf16":
            # 256 rows: the dense path still takes up to two row tiles; 64:
            # below one 128-row tile, no dense-path buffers at all (every row
            # on the gathers, as at this sparsity anyway)
            for key, cap in (("capped_step", 256), ("capped_step_no_dense_path", 64)):
                cm = capped_memory(torch, tw, b, timed, cap)
                mem[key] = cm
                mem[key.replace("capped_step", "capped_vs_dense_peak")] = round(
                    cm["measured_peak_extra_bytes"] /
                    max(mem["dense_step_peak_beyond_outputs_bytes"], 1), 4)
    cpu = None if (args.no_cpu or world > 1) else cpu_baseline(b.a, w, train, args.cpu_seconds)
    del b, d, bufs, ws, y
    torch.cuda.empty_cache()
    sub = None if (args.no_sweep or world > 1) else sweep(torch, tw, lib, dev, args, timed,
                                                          per_step, flush_buf)

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": round(ms_step, 5),
        "step_ms": {"median": round(step_ms[len(step_ms) // 2], 5), "min": round(step_ms[0], 5),
                    "warm_l2_mean": round(warm_ms, 5)},
        "higher_is_better": True, "scaling": "strong" if sharded else "weak",
        "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic (seeded numpy PCG64; shapes and sparsity of the pages' FFN setting)",
        "config": {"workload": describe(w, train), "T": T, "d_model": w.D, "d_ff": w.F,
                   "tile": w.C, "K": w.K, "step": "fwd+bwd" if train else "fwd",
                   "l2": f"flushed before every timed step ({flush_buf.numel() >> 20} MiB write)",
                   "parallelism": (f"token-sharded x{world} (dW all-reduce in the step)"
                                   if sharded else f"replicas x{world}")},
        "roofline": rec["roofline"],
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": int(round(launches_per_step * args.steps)),
        "clocks": clocks,
        "kernels": {k: {kk: round(vv, 5) for kk, vv in v.items()} for k, v in kern.items()},
        "kernel_roofline": {k: {kk: (round(vv, 4) if isinstance(vv, float) else vv)
                                for kk, vv in v.items()} for k, v in rl.items()},
        "sparsity": rec["sparsity"],
        "path": rec["path"],
        "l2_gather_gbs": rec["l2_gather_gbs"],
        "l2_gather_token_rows_gbs": rec["l2_gather_token_rows_gbs"],
        "memory": mem,
        "energy": energy,
    }
    if formats:
        line["format_comparison"] = formats
    for k in ("dense_cublas", "dense_gemm_only", "speedup_vs_dense", "speedup_vs_dense_gemm_only"):
        if k in rec:
            line[k] = rec[k]
    if sub:
        line["workloads"] = sub
    return line


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        j = json.load(open(p))
        return {"hbm_gbs": float(j["hbm_gbs"]), "bf16_tflops": float(j["bf16_tflops"]),
                "bf16_tflops_sustained": float(j.get("bf16_tflops_sustained", j["bf16_tflops"])),
                "source": "of measured (MEASURED_PEAKS.json)"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "of fallback (no MEASURED_PEAKS.json)"}


def tw_hooks():
    """The test-hooks build of the library (the gather probe lives there, not
    in libtwell.so)."""
    import activation_sparse_transformer_gate_gb300 as tw
    from activation_sparse_transformer_gate_gb300 import _build
    _build.build(variants=("hooks",))
    return tw.load(_build.lib_path("hooks"))


def fp32_alu_tflops() -> float:
    """fp32 FFMA peak of one GB300: 152 SMs x 128 fp32 lanes x 2 flop x the
    2.07 GHz maximum SM clock."""
    return 152 * 128 * 2 * 2.07e9 / 1e12


def gather_ceiling(torch, dev, W, w, pairs, timed, sh, n_rows=None):
    """GB/s at which the GPU gathers `pairs` rows of W (n_rows x d_model,
    default F rows) in a uniform random order with plain 16-byte loads: the
    measured ceiling for the sparse kernels' row gathers (L2-served when W
    fits in L2), timed like the step (events on the stream, L2 flushed
    before every run)."""
    if pairs < 1:
        return None
    rng = np.random.default_rng(7)
    n_rows = w.F if n_rows is None else n_rows
    rows = torch.from_numpy(rng.integers(0, n_rows, size=pairs).astype(np.int32)).to(dev)
    blocks = 6 * torch.cuda.get_device_properties(dev).multi_processor_count
    out = torch.empty((blocks * 8,), dtype=torch.int32, device=dev)
    hooks = tw_hooks()
    f = hooks.twell_test_gather_probe
    f.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                  ctypes.c_void_p, ctypes.c_void_p]
    row_bytes = w.D * (2 if w.dtype == "bf16" else 4)

    def run():
        rc = f(W.data_ptr(), row_bytes, rows.data_ptr(), pairs, blocks, out.data_ptr(), sh)
        if rc != 0:
            raise SystemExit(f"gather probe failed: {rc}")

    for _ in range(3):
        run()
    n = 20
    ms = timed(run, n) / n
    return pairs * row_bytes / (ms / 1e3) / 1e9


def kernel_rooflines(kern, w, nnz, train, rows_f=0, rows_b=0, dh_gemm=False):
    """Achieved rate of each kernel from its algorithmic work per step:
    bytes for the gather kernels (rows gathered + rows streamed + TwELL),
    flops for the gate GEMM and for the dense-path GEMMs (rows_f / rows_b
    rows of the forward / backward; fp16 operands, one GEMM per product),
    bytes for the fp16 weight copies of the dense path; divided by the
    kernel's device time per step (a gather kernel split into passes over
    its matrices or columns launches once per pass, each with its share of
    the work).  See the design notes for the per-unit figures."""
    peaks = load_peaks()
    D, F, T, K = w.D, w.F, w.T, w.K
    es = 2 if w.dtype == "bf16" else 4
    row_ovf = (nnz > K).any(axis=0)
    sparse_rows = int((~row_ovf).sum())
    pairs = int(np.minimum(nnz, K)[:, ~row_ovf].sum())          # pairs of TwELL rows
    pairs_all = int(nnz.sum())                                    # incl. overflow rows
    twell = (F // w.C) * T * ((1 + es) * K + 1)
    nw = 2 if w.gated else 1  # weight rows gathered per pair in the forward

    def gathered(rows):
        """Pairs and tokens the gather kernels take when `rows` rows are on
        the dense path (all: none; the overflow rows: the TwELL rows only)."""
        if rows >= T:
            return 0, 0
        if rows > 0:
            return pairs, sparse_rows
        return pairs_all, T

    pf, tf = gathered(rows_f)
    pb, tb = gathered(rows_b)
    ng = 3 if w.gated else 2  # dW problems (dWg, [dWu,] dWd)
    wrk = {
        # per pair: W_up (gated) + W_down rows; per token: x row in (gated), y
        # row out; TwELL read
        "twell_updown_fused": ("hbm", (pf * nw * D * es + tf * D * es * nw + twell) if tf else 0),
        # dh SDDMM: per pair a W_down row, u in and dz/du/h out; per token the dy row
        "bwd_slots_sddmm": ("hbm", pb * (D * es + es + 12) + tb * D * es),
        # dx SpMM: per pair W_gate (+ W_up) rows and dz/du in; per token the dx row out
        "bwd_dx_spmm": ("hbm", pb * (nw * D * es + 8) + tb * D * es),
        # per pair: x + dy rows and its 16-byte list record {token, dz, du, h};
        # the fp32 dW rows and dbg out
        "bwd_dw_gather": ("hbm", pb * (2 * D * es + 16) + (ng * F * D * 4 + F * 4 if tb else 0)),
        # bf16: tcgen05 tensor cores; fp32: CUDA-core FFMA (no TF32)
        "gate_gemm_relu_twell": ("tensor" if es == 2 else "alu", 2.0 * T * D * F),
    }
    if dh_gemm:  # dh from the full product dy W_down^T, read at the slots
        del wrk["bwd_slots_sddmm"]
        wrk["bwd_dh_gemm_sampled"] = ("tensor", 2.0 * T * D * F)
    wrk = {k: v for k, v in wrk.items() if v[1] > 0}
    for k, rows, mult in (("dense_rows_gate_up", rows_f, 1), ("dense_rows_down", rows_f, 1),
                          ("bwd_dense_dh_gemm", rows_b, 1),
                          ("bwd_dense_dx_gemm", rows_b, 2 if w.gated else 1),
                          ("bwd_dense_dw_gemm", rows_b, ng)):
        if rows > 0:
            wrk[k] = ("tensor", 2.0 * mult * rows * D * F)
    # fp16 copies of the weights the dense-path GEMMs take (read bf16, write
    # fp16): W_down in the forward (gated), W_down, W_gate (, W_up) in the backward
    n16 = ((1 if w.gated and rows_f > 0 else 0) + (ng if train and rows_b > 0 else 0))
    if n16 and es == 2:
        wrk["weights_to_f16"] = ("hbm", n16 * F * D * 4)
    out = {}
    for k, (bound, work) in wrk.items():
        if k not in kern:
            continue
        sec = kern[k]["ms_per_step"] / 1e3
        src = peaks["source"]
        if bound == "hbm":
            ach, peak, unit = work / sec / 1e9, peaks["hbm_gbs"], "GB/s"
        elif bound == "alu":  # fp32 FFMA on the CUDA cores
            ach, peak, unit = work / sec / 1e12, fp32_alu_tflops(), "TFLOP/s"
            src = ("derived: 152 SMs x 128 fp32 lanes x 2 flop per FFMA x 2.07 GHz maximum "
                   "SM clock")
        else:  # timed inside back-to-back steps: the sustained (power-capped) peak
            ach, peak, unit = work / sec / 1e12, peaks["bf16_tflops_sustained"], "TFLOP/s"
        out[k] = dict(bound=bound, achieved=ach, peak=peak, unit=unit, frac=ach / peak,
                      algorithmic=work, peak_source=src)
        if k == "bwd_dh_gemm_sampled":
            # the same values as the SDDMM it replaces, rated on that SDDMM's
            # bytes (the method's own work) beside the dense product's flops
            sb = pb * (D * es + es + 12) + tb * D * es
            out[k]["sddmm_bytes"] = sb
            out[k]["sddmm_equivalent_gbs"] = sb / sec / 1e9
    out.setdefault("_counts", {"bound": "-", "pairs_twell_rows": pairs, "pairs_all": pairs_all,
                               "sparse_rows": sparse_rows, "dense_path_rows_fwd": rows_f,
                               "dense_path_rows_bwd": rows_b})
    return out


def kernel_source_hash() -> str:
    """Hash of the library's sources with comments and blank space removed,
    so that a capture stays matched to its kernels across comment edits."""
    import re
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "activation_sparse_transformer_gate_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        text = open(os.path.join(csrc, f), encoding="utf-8").read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        text = re.sub(r"\s+", " ", text)
        h.update(f.encode() + b"\0" + text.encode())
    return h.hexdigest()[:16]


def traffic_for(kernel, workload, train):
    """DRAM bytes per launch from a committed ncu capture, if it was taken on
    the current kernel sources (null otherwise)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        e = json.load(open(p)).get(f"{kernel}|{workload}|{'train' if train else 'fwd'}")
    except ValueError:
        return None
    if not e or e.get("source_hash") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


def row_ovf_count(bufs, w):
    """Overflow rows of the current TwELL (a row overflows if any tile does)."""
    nnz = bufs.nnz.cpu().numpy()
    return int((nnz > w.K).any(axis=0).sum())


def dense_step_fn(torch, d, w, train):
    """One step of the same FFN with cuBLAS GEMMs through torch (bf16 operands,
    fp32 accumulation): forward, and for training the backward with the L1
    term."""
    x, Wg, Wu, Wd, rb, dy = d["x"], d["Wg"], d["Wu"], d["Wd"], d["rb"], d["dy"]
    bgb = d["bg"].to(x.dtype)
    lam = w.lam

    def step():
        z = torch.addmm(bgb, x, Wg.t())
        if rb is not None:
            z = z + rb.to(x.dtype)[:, None]
        g = torch.relu(z)
        if Wu is None:
            h = g
            y = h @ Wd
            if not train:
                return y
            dh = dy @ Wd.t() + lam * torch.sign(h)
            dz = torch.where(z > 0, dh, torch.zeros_like(dh))
            return (dz @ Wg, dz.t() @ x, h.t() @ dy, dz.float().sum(0))
        u = x @ Wu.t()
        h = g * u
        y = h @ Wd
        if not train:
            return y
        dh = dy @ Wd.t() + lam * torch.sign(h)
        dz = torch.where(z > 0, dh * u, torch.zeros_like(dh))
        du = dh * g
        return (dz @ Wg + du @ Wu, dz.t() @ x, du.t() @ x, h.t() @ dy, dz.float().sum(0))

    return step


class PowerSampler:
    """nvidia-smi power.draw samples (20 ms) with their timestamps."""

    def __init__(self, index: int):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(index), "--query-gpu=timestamp,power.draw",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return []
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        samples = []
        for r in csv.reader(io.StringIO(out)):
            if len(r) < 2:
                continue
            try:
                ts = datetime.datetime.strptime(r[0].strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
                samples.append((ts, float(r[1])))
            except ValueError:
                continue
        return samples


def capped_memory(torch, tw, b, timed, cap=256):
    """The same step with buffers and a workspace sized for at most `cap`
    overflow rows and `cap` dense-path rows (twell_t.dense_rows_cap): the
    device memory it needs beyond its inputs and outputs, measured as the
    high-water mark of the allocator around the allocation and a step (the
    library allocates nothing itself), and its time."""
    w, dev, train = b.w, b.dev, b.train
    T, D, F = w.T, w.D, w.F
    torch.cuda.synchronize(dev)
    base = torch.cuda.memory_allocated(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    bufs = tw.TwellBuffers(T, F, w.C, w.K, b.dtype, ovf_cap=cap, train=train, device=dev,
                           dense_rows_cap=cap)
    ws, nws = tw.workspace(T, D, F, w.C, w.K, b.dtype, train, device=dev, dense_rows_cap=cap)
    d = b.d

    def step():
        tw.twell_ffn_forward(d["x"], d["Wg"], d["bg"], d["rb"], d["Wu"], d["Wd"], D, int(train),
                             bufs.t, b.y, ws, nws, b.sh)
        if train:
            tw.twell_ffn_backward(d["x"], d["Wg"], d["Wu"], d["Wd"], bufs.t, d["dy"], w.lam, D,
                                  b.dx, b.dWg, b.dbg, b.dWu, b.dWd, ws, nws, b.sh)

    for _ in range(3):
        step()
    code, n_ovf = tw.twell_get_status(bufs.t, b.sh)
    peak = torch.cuda.max_memory_allocated(dev) - base
    ms = timed(step, 20) / 20
    buf_bytes = sum(t.numel() * t.element_size() for t in
                    (bufs.idx, bufs.val, bufs.nnz, bufs.ovf_rows, bufs.g_fb, bufs.u_val, bufs.u_fb,
                     bufs.n_ovf, bufs.status) if t is not None)
    out = {"dense_rows_cap": cap, "ovf_cap": cap, "status": code, "n_ovf": n_ovf,
           "buffers_bytes": int(buf_bytes), "workspace_bytes": int(nws),
           "measured_peak_extra_bytes": int(peak), "ms_per_step": round(ms, 5)}
    del bufs, ws
    torch.cuda.empty_cache()
    return out


def memory_and_energy(torch, dev, index, d, w, train, ours_step, bufs, nws, n_ovf, seconds=2.5):
    """Saved-activation bytes (forward -> backward) and device memory of the
    sparse path against the dense one, and energy per token of each measured
    with the GPU's energy counter over a few seconds of back-to-back steps."""
    T, F = w.T, w.F
    es = 2  # bf16
    nt = F // w.C
    twell = nt * T * (w.K * (1 + es) + 1) + (nt * T * w.K * es if train else 0)
    fb = n_ovf * F * es * (2 if train else 1) + 4 * n_ovf
    dense_step = dense_step_fn(torch, d, w, train)
    dense_step()
    torch.cuda.synchronize(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    base = torch.cuda.memory_allocated(dev)
    dense_step()
    torch.cuda.synchronize(dev)
    dense_peak = torch.cuda.max_memory_allocated(dev) - base
    buf_bytes = sum(t.numel() * t.element_size() for t in
                    (bufs.idx, bufs.val, bufs.nnz, bufs.ovf_rows, bufs.g_fb, bufs.u_val, bufs.u_fb)
                    if t is not None)
    mem = {
        "saved_activation_bytes_sparse": twell + fb,
        "saved_activation_bytes_dense": (3 * T * F * es) if train else 0,
        "note_saved": "sparse: TwELL idx/val/nnz (+u at the slots) and the used overflow rows; "
                      "dense: z, u, h [T][F] bf16 kept for the backward",
        "dense_step_peak_extra_bytes": int(dense_peak),
        # the dense step's outputs (y, and for training dx, the three weight
        # gradients in bf16 and dbg) are part of its peak; the sparse path's
        # outputs are the caller's preallocated tensors
        "dense_step_peak_beyond_outputs_bytes": int(dense_peak - (
            T * w.D * es + ((T * w.D * es + 3 * F * w.D * es + 4 * F) if train else 0))),
        "sparse_buffers_allocated_bytes": int(buf_bytes),
        "sparse_workspace_bytes": int(nws),
        "note_alloc": "buffers sized for ovf_cap = T overflow rows and a workspace sized for the "
                      "all-dense fallback: allocations, not what a step keeps",
    }

    def joules_per_token(fn):
        """Mean board power over a few seconds of back-to-back steps x their
        time / tokens (power samples inside the loop's wall-clock window)."""
        fn()
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        n = 0
        while time.perf_counter() - t0 < 0.3:
            fn()
            n += 1
        torch.cuda.synchronize(dev)
        per = (time.perf_counter() - t0) / n
        reps = max(10, int(seconds / per))
        ps = PowerSampler(index)
        time.sleep(0.5)
        w0 = time.time()
        t0 = time.perf_counter()
        for _ in range(reps):
            fn()
        torch.cuda.synchronize(dev)
        wall = time.perf_counter() - t0
        w1 = time.time()
        samples = ps.stop()
        inside = [pw for ts, pw in samples if w0 + 0.1 <= ts <= w1]
        if len(inside) < 5:
            return None
        watts = float(np.mean(inside))
        return {"j_per_token": watts * wall / (reps * T), "mean_w": watts, "samples": len(inside),
                "s": round(wall, 3)}

    es_, ed_ = joules_per_token(ours_step), joules_per_token(dense_step)
    energy = None
    if es_ and ed_:
        energy = {"sparse_j_per_token": es_["j_per_token"], "dense_j_per_token": ed_["j_per_token"],
                  "ratio": es_["j_per_token"] / ed_["j_per_token"],
                  "sparse_mean_w": es_["mean_w"], "dense_mean_w": ed_["mean_w"],
                  "how": f"mean nvidia-smi power.draw (20 ms samples) x time over >= {seconds} s of "
                         "back-to-back steps (no L2 flush), whole board"}
    return mem, energy


def dense_gemm_only_fn(torch, d, w, train):
    """The dense FFN's GEMMs alone, with the same shapes and operand types as
    the eager arm and preallocated outputs, no element-wise work: 3 GEMMs
    forward (gate, up, down; 2 for the plain FFN) and 6 more for the
    backward (dh, the two dx products, dW_gate, dW_up, dW_down).  A floor
    for any dense implementation that runs these products on cuBLAS."""
    x, Wg, Wu, Wd, dy = d["x"], d["Wg"], d["Wu"], d["Wd"], d["dy"]
    T, F, D = w.T, w.F, w.D
    z = torch.empty((T, F), dtype=x.dtype, device=x.device)
    u = torch.empty_like(z) if Wu is not None else None
    y = torch.empty((T, D), dtype=x.dtype, device=x.device)
    if train:
        dh = torch.empty_like(z)
        dx = torch.empty_like(y)
        dWg = torch.empty((F, D), dtype=x.dtype, device=x.device)
        dWu = torch.empty_like(dWg) if Wu is not None else None
        dWd = torch.empty_like(dWg)

    def step():
        torch.matmul(x, Wg.t(), out=z)
        if u is not None:
            torch.matmul(x, Wu.t(), out=u)
        torch.matmul(z, Wd, out=y)            # (z stands in for h: same shape, same cost)
        if not train:
            return
        torch.matmul(dy, Wd.t(), out=dh)
        torch.matmul(dh, Wg, out=dx)
        if u is not None:
            dx.addmm_(u, Wu)                  # (u stands in for du)
        torch.matmul(dh.t(), x, out=dWg)
        if dWu is not None:
            torch.matmul(z.t(), x, out=dWu)
        torch.matmul(z.t(), dy, out=dWd)

    return step


def dense_arms(torch, d, w, train, timed, args, steps):
    """The same FFN on cuBLAS through torch (bf16 operands with fp32
    accumulation; fp32 with TF32 off for the fp32 workload), timed like the
    sparse step: "eager" with torch's element-wise ops between the GEMMs,
    "gemm_only" the GEMMs alone."""
    out = {}
    for name, fn in (("eager", dense_step_fn(torch, d, w, train)),
                     ("gemm_only", dense_gemm_only_fn(torch, d, w, train))):
        for _ in range(max(args.warmup, 3)):
            fn()
        ms = timed(fn, steps) / steps
        what = ("torch %s matmul (cuBLAS) dense FFN%s%s" %
                (w.dtype, " fwd+bwd" if train else " fwd",
                 ": GEMMs only, no element-wise work" if name == "gemm_only" else ""))
        out[name] = {"ms_per_step": round(ms, 5), "tokens_per_s": round(w.T / (ms / 1e3), 1),
                     "what": what, "steps": steps}
    return out


def format_comparison(torch, lib, d, w, bufs, ws, nws, y, sh, timed, args):
    """What the TwELL format and its fused pack buy, on the same inputs
    (forward).  Times, with cold L2 before each step:
      twell_fused_pack: twell_pack (gate GEMM with the ReLU + TwELL epilogue,
        overflow list, backup rows);
      twell_unfused_pack: the gate GEMM writing the dense activation matrix
        H (cuBLAS through torch, bias, ReLU, bf16) + twell_pack_dense(H);
      twell_forward: twell_ffn_forward (gate + pack + up/down);
      rowell_forward: H as above + row-ELL pack (width E = the densest row)
        + the row-ELL up/down projection.
    and the bytes each format keeps (indices, values, counts)."""
    import activation_sparse_transformer_gate_gb300 as tw
    T, D, F = w.T, w.D, w.F
    H = torch.empty((T, F), dtype=torch.bfloat16, device=d["x"].device)

    bg16 = d["bg"].to(torch.bfloat16)
    rb16 = None if d["rb"] is None else d["rb"].to(torch.bfloat16)[:, None]

    def gate_dense():  # cuBLAS GEMM with the bias into H (bf16), then row bias and ReLU in place
        torch.addmm(bg16, d["x"], d["Wg"].t(), out=H)
        if rb16 is not None:
            H.add_(rb16)
        H.relu_()

    # width of row-ELL: the densest row of this input
    tw.twell_ffn_forward(d["x"], d["Wg"], d["bg"], d["rb"], d["Wu"], d["Wd"], D, 0, bufs.t, y,
                         ws, nws, sh)
    gate_dense()
    torch.cuda.synchronize()
    E = int((H > 0).sum(dim=1).max().item())
    re = tw.RowEllBuffers(T, F, E, tw.TWELL_BF16, device=d["x"].device)
    y2 = torch.empty_like(y)

    legs = {
        "twell_fused_pack": lambda: tw.twell_pack(d["x"], d["Wg"], d["bg"], d["rb"], D, bufs.t,
                                                  ws, nws, sh),
        "twell_unfused_pack": lambda: (gate_dense(), tw.twell_pack_dense(H, bufs.t, sh)),
        "twell_forward": lambda: tw.twell_ffn_forward(d["x"], d["Wg"], d["bg"], d["rb"], d["Wu"],
                                                      d["Wd"], D, 0, bufs.t, y, ws, nws, sh),
        "rowell_forward": lambda: (gate_dense(), tw.twell_rowell_pack_dense(H, re.t, sh),
                                   tw.twell_rowell_forward(d["x"], d["Wu"], d["Wd"], D, re.t, y2,
                                                           sh)),
    }
    out = {}
    steps = max(10, min(args.steps, 100))
    for k, fn in legs.items():
        for _ in range(3):
            fn()
        out[k] = {"ms": round(timed(fn, steps) / steps, 5)}
    code = int(re.status[0].item())
    nt = F // w.C
    out["bytes"] = {"twell_idx_val_nnz": nt * T * w.K * 3 + nt * T,
                    "rowell_idx_val_nnz": T * E * 4 + T * 4, "rowell_width_E": E,
                    "twell_K_per_tile": w.K, "dense_H": T * F * 2}
    out["rowell_status"] = code
    out["note"] = ("the unfused legs round z + bias to bf16 before the ReLU (a cuBLAS GEMM "
                   "output), so their activations differ slightly from the fused epilogue's")
    return out


def end_to_end(torch, d, step, y, dx, w, train, timed, args, stream, flush_buf):
    """Pinned host inputs copied in and the step's outputs copied out, every
    step, around the same C-ABI calls.  value: the copies run on a second
    stream, double-buffered, so that the next step's inputs go in and the
    previous step's outputs come out while a step computes (what a data
    loader's prefetch does); the timed region spans all the steps and ends
    when every copy has completed.  serial_ms_per_step: copy in, step, copy
    out, one after the other."""
    hx = d["x"].cpu().pin_memory()
    hdy = d["dy"].cpu().pin_memory() if train else None
    hy = [torch.empty(y.shape, dtype=y.dtype).pin_memory() for _ in range(2)]
    hdx = [torch.empty(dx.shape, dtype=dx.dtype).pin_memory() for _ in range(2)] if train else None
    gx = [torch.empty_like(d["x"]) for _ in range(2)]
    gdy = [torch.empty_like(d["dy"]) for _ in range(2)] if train else None
    gy = [torch.empty_like(y) for _ in range(2)]
    gdx = [torch.empty_like(dx) for _ in range(2)] if train else None

    def serial_step():
        gx[0].copy_(hx, non_blocking=True)
        if train:
            gdy[0].copy_(hdy, non_blocking=True)
        step(gx[0], gdy[0] if train else None)
        hy[0].copy_(y, non_blocking=True)
        if train:
            hdx[0].copy_(dx, non_blocking=True)

    cs = torch.cuda.Stream(device=stream.device)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def h2d(b):
        gx[b].copy_(hx, non_blocking=True)
        if train:
            gdy[b].copy_(hdy, non_blocking=True)
        ev_in[b].record(cs)

    def pipelined(K):
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        cs.wait_stream(stream)
        with torch.cuda.stream(cs):
            h2d(0)
        for i in range(K):
            b = i % 2
            flush_buf.fill_(1)
            stream.wait_event(ev_in[b])
            if i >= 2:
                stream.wait_event(ev_out[b])  # step i-2's outputs are out of this buffer
            step(gx[b], gdy[b] if train else None, gy[b], gdx[b] if train else None)
            ev_done[b].record(stream)
            with torch.cuda.stream(cs):
                if i + 1 < K:
                    h2d(1 - b)  # (its buffers were released by step i-1's read-out, in order)
                cs.wait_event(ev_done[b])
                hy[b].copy_(gy[b], non_blocking=True)
                if train:
                    hdx[b].copy_(gdx[b], non_blocking=True)
                ev_out[b].record(cs)
        stream.wait_stream(cs)
        t1.record(stream)
        torch.cuda.synchronize(stream.device)
        return t0.elapsed_time(t1) / K

    def flush_only(K):
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(K):
            flush_buf.fill_(1)
        t1.record(stream)
        torch.cuda.synchronize(stream.device)
        return t0.elapsed_time(t1) / K

    for _ in range(3):
        serial_step()
    steps = max(10, min(args.steps, 200))
    ms_serial = timed(serial_step, steps) / steps
    pipelined(3)
    ms = pipelined(steps)
    ms_flush = flush_only(steps)
    h2d_bytes = hx.numel() * 2 + (hdy.numel() * 2 if train else 0)
    d2h_bytes = hy[0].numel() * 2 + (hdx[0].numel() * 2 if train else 0)
    return {"value": round(w.T / (ms / 1e3), 1), "unit": "tokens/s",
            "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": d2h_bytes,
            "ms_per_step": round(ms, 5), "steps": steps,
            "copies": "double-buffered on a second stream, overlapping the neighbouring steps",
            "l2_flush_ms_per_step": round(ms_flush, 5),
            "note_flush": "the timed region also holds the write of a 2 x L2 buffer before every "
                          "step (cold L2, as for value); l2_flush_ms_per_step is that write's "
                          "own time, not subtracted",
            "serial_ms_per_step": round(ms_serial, 5),
            "serial_tokens_per_s": round(w.T / (ms_serial / 1e3), 1),
            "outputs_copied": "y" + (" and dx; the fp32 weight gradients (dW_gate, dW_up, "
                                     "dW_down, dbg) stay on the device for an optimizer step "
                                     "there" if train else "")}


def oracle_sample(a, w, train, S, Fs):
    """The oracle on S tokens and the first Fs neurons of the workload: the
    FFN cost is linear in both, so tokens/s scales by Fs/F exactly."""
    import oracle
    dt = w.dtype
    x = a["x"][:S]
    rb = None if a["rb"] is None else a["rb"][:S]
    Wg, Wu, Wd, bg = a["Wg"][:Fs], a["Wu"][:Fs], a["Wd"][:Fs], a["bg"][:Fs]
    t0 = time.perf_counter()
    oracle.ffn_dense(x, Wg, bg, rb, Wu, Wd, dt, dt)
    if train:
        oracle.ffn_backward(x, Wg, bg, rb, Wu, Wd, a["dy"][:S], w.lam, dt, dt)
    return time.perf_counter() - t0


def cpu_baseline(a, w, train, seconds):
    import oracle
    oracle.build()
    S = 2
    t = oracle_sample(a, w, train, S, w.F)
    S = int(max(2, min(w.T, S * seconds / max(t, 1e-3))))
    t = oracle_sample(a, w, train, S, w.F)
    cores = oracle.get_threads()
    # the same oracle on one host core, on a smaller sample of the same rows
    oracle.set_threads(1)
    try:
        S1 = max(1, S // max(cores, 1))
        t1 = oracle_sample(a, w, train, S1, w.F)
    finally:
        oracle.set_threads(cores)
    return {"value": round(S / t, 3), "unit": "tokens/s", "cores": cores,
            "kind": "oracle",
            "sample": f"first {S} tokens of the workload, all {w.F} neurons, "
                      f"{'dense fwd+bwd' if train else 'dense fwd'} in fp64 C loops (OpenMP over "
                      f"tokens/neurons), {t:.1f} s",
            "single_thread": {"value": round(S1 / t1, 3), "unit": "tokens/s",
                              "sample": f"first {S1} tokens, {t1:.1f} s on 1 core"}}


def max_over_ranks(torch, value: float, world: int, device) -> float:
    """The slowest rank's value (every rank contributes its own and receives
    the maximum): the job takes as long as its slowest replica."""
    if world <= 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def run_reference(args, rank, world):
    """The CPU oracle as the reference arm: each step is a bounded sample of
    the workload (S tokens x Fs neurons), scaled to tokens/s of the full FFN."""
    if rank != 0:
        return None
    import oracle
    oracle.build()
    train = args.mode == "train"
    w = workload_of(args.workload, train)
    a = synth.generate(w, rows=64)
    budget = min(10.0, 150.0 / (args.steps + max(args.warmup, 3)))
    S, Fs = 1, w.F
    t = oracle_sample(a, w, train, S, Fs)
    while t > budget and Fs > 64:
        Fs //= 2
        t = oracle_sample(a, w, train, S, Fs)
    while t * 2 < budget and S < 64:
        S *= 2
        t = oracle_sample(a, w, train, S, Fs)
    for _ in range(max(args.warmup, 3)):
        oracle_sample(a, w, train, S, Fs)
    tot = sum(oracle_sample(a, w, train, S, Fs) for _ in range(args.steps))
    ms_step = tot / args.steps * 1e3
    value = S * Fs / w.F / (ms_step / 1e3)
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": max(args.warmup, 3),
        "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded numpy PCG64)",
        "config": {"workload": describe(w, train), "T": w.T, "d_model": w.D, "d_ff": w.F,
                   "tile": w.C, "K": w.K, "step": "fwd+bwd" if train else "fwd"},
        "cpu_baseline": {"value": round(value, 4), "unit": "tokens/s", "kind": "oracle",
                         "cores": oracle.get_threads(),
                         "sample": f"per step: {S} token(s) x {Fs} of {w.F} neurons "
                                   f"(cost linear in both), dense {'fwd+bwd' if train else 'fwd'}"},
        "e2e": {"value": round(value, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    import torch
    if world > 1:
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    try:
        line = run_ours(args, rank, world, local_rank)
        if line is not None:
            print(json.dumps(line), flush=True)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
