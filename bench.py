#!/usr/bin/env python
"""Throughput of the fused attention hot path (forward + backward) on one GB300 per rank.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload c4] [--impl ours]

A step is one pass of the whole hot path over one batch of synthetic input: attn_fwd
then (where the workload has a backward) attn_bwd, both through the C ABI. The headline
workload is c4, the video-DiT self-attention (B1 H40 S32760 D128, the largest
single-GPU configuration); the same run also times the GQA training step (c3: the
long-sequence forward + backward), the varlen DiT self-attention (c4v) and the DiT
cross-attention (c5), reported under ``also`` in the same JSON line. The value is
TFLOP/s with the pages' counting rule (4 * B * Hq * Sq * Skv_eff * D for the forward,
2.5 x that for the backward), inputs already resident in HBM; L2 is flushed (a 512 MiB
write) before every step, outside the timed events. ``e2e`` is the same metric with the
inputs copied from pinned host memory and every output copied back, inside the timed
region (a forward-only workload through attn_fwd_host, which overlaps the copies with
the compute chunk by chunk of kv heads). Under torchrun each rank runs an independent replica (attention over
independent batches and heads needs no exchange); the time is the max over ranks.

``--impl reference`` times the float64 CPU oracle instead, on the host cores, on a
bounded sample of the same workload per step (rank 0 only).
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import tempfile
import sys
import time

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, HERE)

from attention_sm_flash_gb300 import metrics, workloads  # noqa: E402

METRIC = "attention fwd/bwd TFLOP/s (bf16) and % of GB300 dense BF16 tensor peak"
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}
DEFAULT_ALSO = "c3,c4v,c5,c4@paged256,dec1@dense,dec1@split,sq64@dense,sq64@split,vae_f32,c1"
# the fp32 forward runs three TF32 tensor-core products per multiply: its peak in
# algorithmic fp32 FLOP/s is the TF32 dense peak / 3, the TF32 peak being the measured
# bf16 peak x the nominal TF32 : bf16 ratio (1.1 : 2.25 PFLOP/s dense per GPU)
TF32_PER_BF16 = 1.1 / 2.25


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="c4", choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--also", default=DEFAULT_ALSO,
                    help="comma-separated workloads timed after the headline one, in the "
                         "same process, each as key[@mode] with mode dense (default), split "
                         "(attn_fwd_splitkv) or pagedN (attn_fwd_paged, N-key pages); empty: "
                         "none")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="CPU work in the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    return ap.parse_args()


def load_peaks():
    path = os.path.join(HERE, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def workload_config(w, inp):
    lens = inp["kv_lens"]
    fwd = metrics.fwd_flops(w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.D, w.causal, lens)
    bwd = metrics.bwd_flops(w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.D, w.causal, lens) if w.has_bwd else 0.0
    pairs = metrics.visible_pairs(w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.causal, lens)
    cfg = {"workload": f"{w.key} {w.name}", "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Sq": w.Sq,
           "Skv": w.Skv, "Skv_eff": round(pairs / (w.B * w.Hq * w.Sq), 2), "D": w.D,
           "causal": w.causal, "kv_lens": w.lens_kind, "scale": round(w.scale, 6),
           "step": "attn_fwd + attn_bwd" if w.has_bwd else "attn_fwd",
           "parallelism": "replicas (independent problem per rank, no collective)"}
    return cfg, fwd, bwd


# ----------------------------------------------------------------------- CPU oracle
def oracle_sample(w, inp, target_s):
    """A bounded slice of the workload for the float64 oracle, sized to ~target_s.

    Returns (run, flops, description). Training workloads use whole (batch, kv head)
    groups, forward + backward; the long-sequence workloads use query rows of head 0.
    """
    import oracle

    g = w.Hq // w.Hkv
    lens = inp["kv_lens"]

    def unit_group(b, kvh):
        sl = slice(kvh * g, (kvh + 1) * g)
        q = inp["q"][b:b + 1, :, sl]
        k = inp["k"][b:b + 1, :, kvh:kvh + 1]
        v = inp["v"][b:b + 1, :, kvh:kvh + 1]
        ln = None if lens is None else lens[b:b + 1, kvh:kvh + 1]
        fl = metrics.fwd_flops(1, g, 1, w.Sq, w.Skv, w.D, w.causal, ln)
        if w.has_bwd:
            do = inp["do"][b:b + 1, :, sl]
            fl *= 3.5

            def run():
                oracle.forward(q, k, v, w.scale, w.causal, ln)
                oracle.backward(q, k, v, do, w.scale, w.causal, ln)
        else:
            def run():
                oracle.forward(q, k, v, w.scale, w.causal, ln)
        return run, fl

    if w.Sq * w.Skv <= 4096 * 4096:
        units = [(b, kvh) for b in range(w.B) for kvh in range(w.Hkv)]
        run0, fl0 = unit_group(*units[0])
        t0 = time.perf_counter()
        run0()
        dt = max(time.perf_counter() - t0, 1e-4)
        n = int(max(1, min(len(units), round(target_s / dt))))
        runs = [unit_group(*u) for u in units[:n]]

        def run():
            for r, _ in runs:
                r()
        return run, sum(f for _, f in runs), f"{n} of {len(units)} (batch, kv-head) groups, " \
            f"{'fwd+bwd' if w.has_bwd else 'fwd'}, all query heads of each group"
    # long sequences: rows of head 0
    q = inp["q"][0:1, :, 0:1]
    k = inp["k"][0:1, :, 0:1]
    v = inp["v"][0:1, :, 0:1]
    ln = None if lens is None else lens[0:1, 0:1]

    def rows_run(nrows):
        rows = np.arange(nrows)

        def run():
            oracle.forward_rows(q, k, v, w.scale, w.causal, ln, 0, 0, rows)
        L = w.Skv if ln is None else int(ln[0, 0])
        return run, 4.0 * w.D * nrows * L

    r, _ = rows_run(64)
    t0 = time.perf_counter()
    r()
    dt = max(time.perf_counter() - t0, 1e-4)
    nrows = int(max(64, min(w.Sq, 64 * target_s / dt)))
    run, fl = rows_run(nrows)
    return run, fl, f"{nrows} query rows of (batch 0, head 0), fwd, all valid keys"


def cpu_info():
    cores = len(os.sched_getaffinity(0))
    threads = None
    try:
        from threadpoolctl import threadpool_info
        threads = max((i.get("num_threads", 0) for i in threadpool_info()), default=None)
    except Exception:
        pass
    return cores, threads


def cpu_baseline(w, inp, seconds):
    run, fl, desc = oracle_sample(w, inp, seconds)
    t0 = time.perf_counter()
    run()
    dt = time.perf_counter() - t0
    cores, threads = cpu_info()
    return {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": threads or cores,
            "host_cores": cores, "kind": "oracle", "sample": desc, "seconds": round(dt, 2)}


# ------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index, enabled=True):
        self.index = str(index)
        self.proc = None
        self.path = None
        if not enabled:
            return
        try:
            fd, self.path = tempfile.mkstemp(prefix=f"attn_clocks_{os.getpid()}_", suffix=".csv")
            self.fh = os.fdopen(fd, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            rows = [[p.strip() for p in line.split(",")] for line in f]
        try:
            os.remove(self.path)
        except OSError:
            pass
        rows = [r for r in rows if len(r) >= 9]
        seen = {r[0] for r in rows}
        want = self.index if self.index in seen else (seen.pop() if len(seen) == 1 else None)
        for parts in rows:
                if parts[0] != want:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for n, val in zip(names, parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx) if mx else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# --------------------------------------------------------------------- replicas
def reduce_max(x: float, device) -> float:
    """The max of a per-rank scalar over all ranks (the identity without a process group)."""
    t = torch.tensor([x], dtype=torch.float64, device=device)
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_rank_step: float, ms_max: float, world: int) -> float:
    """Whole-job throughput: every rank's work over the slowest rank's step time."""
    return world * flops_per_rank_step / (ms_max * 1e-3) / 1e12


# --------------------------------------------------------------------------- ours
def bwd_kernel_estimates(key, dtype, bwd_ms, fwd_flops, peak):
    """Per-kernel estimates for one backward call: each kernel's share of the recorded ncu
    durations (profiles/bwd_kernel_durations.txt) times the call's CUDA-event time, and the
    TFLOP/s of the GEMMs it executes over that time; None without a record for the current
    code of the backward's kernels."""
    path = os.path.join(HERE, "profiles", "bwd_kernel_durations.txt")
    if not os.path.exists(path) or not bwd_ms:
        return None
    from attention_sm_flash_gb300 import build as libbuild
    stamp = libbuild.source_digest(libbuild.OP_SOURCES.get(("attn_bwd", dtype)))
    rows = []
    with open(path) as f:
        for line in f:
            parts = line.split()
            if line.startswith("#") or len(parts) != 5 or parts[0] != f"attn_bwd:{key}":
                continue
            if parts[4] != stamp:
                return None
            rows.append((parts[1], int(parts[2]), float(parts[3])))
    total = sum(r[2] for r in rows)
    if not rows or total <= 0:
        return None
    out = []
    for name, gemms, us in rows:
        ms = bwd_ms * us / total
        tf = gemms * fwd_flops / 2 / (ms * 1e-3) / 1e12 if gemms else None
        out.append({"kernel": name, "gemms": gemms, "ncu_share": round(us / total, 4),
                    "ms_est": round(ms, 5), "tflops_est": round(tf, 1) if tf else None,
                    "frac_est": round(tf / peak, 4) if tf else None})
    return out


def traffic_for(kernel_key, dtype="bf16"):
    """DRAM bytes per call recorded from an ncu capture of the current sources of that
    operation's kernels, or None (no record, or the kernels changed since)."""
    path = os.path.join(HERE, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    from attention_sm_flash_gb300 import build as libbuild
    op = kernel_key.split(":")[0]
    stamp = libbuild.source_digest(libbuild.OP_SOURCES.get((op, dtype)))
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 3 and not line.startswith("#") and parts[0] == kernel_key:
                if len(parts) >= 4 and parts[3] != stamp:
                    return None
                return float(parts[2])
    return None


def fwd_bytes(w, lens) -> float:
    """Algorithmic HBM bytes of one forward: Q read and O written once, LSE written, and
    the valid rows of K and V read once."""
    el = 2 if w.dtype == "bf16" else 4
    valid = (w.B * w.Hkv * w.Skv if lens is None else int(lens.to(torch.int64).sum()))
    return 2.0 * w.B * w.Sq * w.Hq * w.D * el + 4.0 * w.B * w.Hq * w.Sq + 2.0 * valid * w.D * el


class Workbench:
    """One workload's device buffers and its timed step (attn_fwd, then attn_bwd where the
    workload has a backward) on one stream, L2 flushed before every step. ``mode``: dense
    (attn_fwd), split (attn_fwd_splitkv) or pagedN (attn_fwd_paged over shuffled N-key
    pages holding the same keys)."""

    def __init__(self, w, inp, dev, stream, flush_buf, mode="dense"):
        from attention_sm_flash_gb300 import attn

        self.attn, self.w, self.inp, self.stream, self.flush_buf = attn, w, inp, stream, flush_buf
        self.mode = mode
        self.q = inp["q"].to(dev)
        self.do = inp["do"].to(dev) if w.has_bwd else None
        self.lens = inp["kv_lens"].to(dev) if inp["kv_lens"] is not None else None
        self.o = torch.empty_like(self.q)
        self.lse = torch.empty((w.B, w.Hq, w.Sq), dtype=torch.float32, device=dev)
        if mode.startswith("paged"):
            ps = int(mode[len("paged"):])
            lens = ([w.Skv] * w.B if inp["kv_lens"] is None else
                    [int(x) for x in inp["kv_lens"][:, 0]])
            kp, vp, bt, _ = workloads.make_paged(inp["k"], inp["v"], lens, ps, seed=w.seed)
            self.k, self.v, self.bt = kp.to(dev), vp.to(dev), bt.to(dev)
            self.seq = torch.tensor(lens, dtype=torch.int32, device=dev)
        else:
            self.k, self.v = inp["k"].to(dev), inp["v"].to(dev)
        if mode == "split":
            need = attn.attn_fwd_splitkv_workspace_size(w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.D,
                                                        attn.ATTN_BF16)
            self.fws = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
        if w.has_bwd:
            self.dq, self.dk, self.dv = (torch.empty_like(t) for t in (self.q, self.k, self.v))
            code = attn.ATTN_BF16 if w.dtype == "bf16" else attn.ATTN_F32
            ws_bytes = attn.attn_bwd_workspace_size(w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.D, code)
            self.ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)

    def fwd(self):
        w = self.w
        if self.mode == "split":
            self.attn.attn_fwd_splitkv(self.q, self.k, self.v, self.o, self.lse, w.causal,
                                       w.scale, self.lens, self.fws, self.stream)
        elif self.mode.startswith("paged"):
            self.attn.attn_fwd_paged(self.q, self.k, self.v, self.bt, self.seq, self.o,
                                     self.lse, w.causal, w.scale, self.stream)
        else:
            self.attn.attn_fwd(self.q, self.k, self.v, self.o, self.lse, w.causal, w.scale,
                               self.lens, self.stream)

    def bwd(self):
        w = self.w
        self.attn.attn_bwd(self.q, self.k, self.v, self.o, self.do, self.lse, self.dq, self.dk,
                           self.dv, w.causal, w.scale, self.lens, self.ws, self.stream)

    def run_steps(self, n):
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
        for e in evs:
            self.flush_buf.zero_()
            e[0].record(self.stream)
            self.fwd()
            e[1].record(self.stream)
            if self.w.has_bwd:
                self.bwd()
            e[2].record(self.stream)
        return evs

    def measure(self, steps, warmup, world, sampler_index, clocks_on):
        """(fwd_ms list, bwd_ms list, clocks, launches, wall seconds) of ``steps`` timed
        steps, barrier + synchronize on both sides."""
        self.run_steps(max(warmup, 3))
        torch.cuda.synchronize()
        sampler = ClockSampler(sampler_index, enabled=clocks_on)
        # clock pre-roll (untimed): about half a second of steps so clocks settle under load
        t_end = time.perf_counter() + 0.5
        while time.perf_counter() < t_end:
            self.run_steps(1)
            torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        n0 = self.attn.attn_launch_count()
        t0 = time.perf_counter()
        evs = self.run_steps(steps)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
        launches = self.attn.attn_launch_count() - n0
        if world > 1:
            torch.distributed.barrier()
        clocks = sampler.stop()
        fwd_ms = [e[0].elapsed_time(e[1]) for e in evs]
        bwd_ms = [e[1].elapsed_time(e[2]) for e in evs]
        return fwd_ms, bwd_ms, clocks, launches, wall


def tensor_peak(w, peaks, peak_src):
    bf16 = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    if w.dtype == "bf16":
        return bf16, "tensor", f"bf16 dense burst, {peak_src}"
    return (bf16 * TF32_PER_BF16 / 3.0, "tensor",
            f"fp32 as 3 TF32 products: bf16 dense burst ({peak_src}) x 1.1/2.25 / 3")


def also_entry(bench, args, world, sampler_index, peaks, peak_src, dev):
    """The figures of one extra workload for the ``also`` key of the JSON line."""
    w = bench.w
    cfg, fwd_fl, bwd_fl = workload_config(w, bench.inp)
    fwd_ms, bwd_ms, clocks, launches, _ = bench.measure(args.steps, args.warmup, world,
                                                          sampler_index, not args.no_clocks)
    fm = reduce_max(statistics.mean(fwd_ms), dev)
    bm = reduce_max(statistics.mean(bwd_ms), dev) if w.has_bwd else 0.0
    peak, bound, note = tensor_peak(w, peaks, peak_src)
    fwd_t = whole_job_tflops(fwd_fl, fm, world)
    gbs = world * fwd_bytes(w, bench.inp["kv_lens"]) / (fm * 1e-3) / 1e9
    hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    call = {"dense": "attn_fwd", "split": "attn_fwd_splitkv"}.get(bench.mode, "attn_fwd_paged")
    out = {"workload": cfg["workload"], "Skv_eff": cfg["Skv_eff"], "step": cfg["step"],
           "forward_call": call,
           "fwd_gbs": round(gbs, 1), "fwd_hbm_frac": round(gbs / world / hbm, 4),
           "value": round(whole_job_tflops(fwd_fl + bwd_fl, fm + bm, world), 3),
           "ms_per_step": round(fm + bm, 5), "fwd_ms": round(fm, 5),
           "fwd_tflops": round(fwd_t, 3), "fwd_frac": round(fwd_t / world / peak, 4),
           "bound": bound, "peak": peak, "peak_source": note, "gpu_launches": int(launches),
           "clocks": clocks}
    if w.has_bwd:
        bwd_t = whole_job_tflops(bwd_fl, bm, world)
        out.update({"bwd_ms": round(bm, 5), "bwd_tflops": round(bwd_t, 3),
                    "bwd_frac": round(bwd_t / world / peak, 4),
                    "bwd_traffic": traffic_for(f"attn_bwd:{w.key}", w.dtype),
                    "bwd_per_kernel_est": bwd_kernel_estimates(w.key, w.dtype, bm, fwd_fl, peak)})
    if w.key != "c3":
        op = {"dense": "attn_fwd", "split": "attn_fwd_splitkv"}.get(bench.mode, "attn_fwd_paged")
        out["fwd_traffic"] = traffic_for(f"{op}:{w.key}", w.dtype)
    return out


def run_ours(args, rank, world, local_rank):
    from attention_sm_flash_gb300 import attn
    from attention_sm_flash_gb300 import build as libbuild

    if not os.path.exists(attn.LIB_PATH):
        libbuild.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    sampler_index = (local_rank if "CUDA_VISIBLE_DEVICES" not in os.environ else
                     os.environ["CUDA_VISIBLE_DEVICES"].split(",")[local_rank])
    w = workloads.get(args.workload)
    inp = workloads.make_inputs(w)
    cfg, fwd_fl, bwd_fl = workload_config(w, inp)
    step_fl = fwd_fl + bwd_fl
    td = w.torch_dtype
    stream = torch.cuda.current_stream(dev)
    flush_buf = torch.empty(256 * 1024 * 1024, dtype=torch.int16, device=dev)  # 512 MiB
    bench = Workbench(w, inp, dev, stream, flush_buf)
    fwd_ms, bwd_ms, clocks, launches, wall = bench.measure(args.steps, args.warmup, world,
                                                           sampler_index, not args.no_clocks)
    step_ms = [a + b for a, b in zip(fwd_ms, bwd_ms)]
    ms = statistics.mean(step_ms)
    ms_max = reduce_max(ms, dev)
    value = whole_job_tflops(step_fl, ms_max, world)
    q, k, v, do, lens, o, lse = bench.q, bench.k, bench.v, bench.do, bench.lens, bench.o, bench.lse

    # e2e: the same step through the C ABI from pinned host buffers, outputs copied back.
    # A forward-only workload goes through attn_fwd_host (the copies overlapped with the
    # compute, chunk by chunk of kv heads); a training step copies its inputs in, runs
    # attn_fwd and attn_bwd and copies its outputs out.
    e2e = None
    if not args.no_e2e and not w.has_bwd:
        hq, hk, hv = (inp[n].pin_memory() for n in ("q", "k", "v"))
        hl = inp["kv_lens"].pin_memory() if inp["kv_lens"] is not None else None
        ho = torch.empty(o.shape, dtype=td).pin_memory()
        hlse = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
        code = attn.ATTN_BF16 if w.dtype == "bf16" else attn.ATTN_F32
        hws = torch.empty(max(attn.attn_fwd_host_workspace_size(w.B, w.Hq, w.Hkv, w.Sq, w.Skv,
                                                                w.D, code), 1),
                          dtype=torch.uint8, device=dev)
        h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hl) if t is not None)
        d2h = sum(t.numel() * t.element_size() for t in (ho, hlse))

        def e2e_step():
            attn.attn_fwd_host(hq, hk, hv, ho, hlse, w.causal, w.scale, hl, hws, stream)

        for _ in range(max(args.warmup, 3)):
            e2e_step()
        torch.cuda.synchronize()
        s_ev, e_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s_ev.record(stream)
        for _ in range(args.steps):
            e2e_step()
        e_ev.record(stream)
        torch.cuda.synchronize()
        e2e_ms = reduce_max(s_ev.elapsed_time(e_ev) / args.steps, dev)
        e2e = {"value": whole_job_tflops(step_fl, e2e_ms, world), "unit": "TFLOP/s",
               "ms_per_step": e2e_ms, "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "call": "attn_fwd_host"}
    elif not args.no_e2e:
        hq, hk, hv = (inp[n].pin_memory() for n in ("q", "k", "v"))
        hdo = inp["do"].pin_memory() if w.has_bwd else None
        hl = inp["kv_lens"].pin_memory() if inp["kv_lens"] is not None else None
        outs_h = [torch.empty(o.shape, dtype=td).pin_memory(),
                  torch.empty(lse.shape, dtype=torch.float32).pin_memory()]
        outs_d = [o, lse]
        if w.has_bwd:
            outs_h += [torch.empty(t.shape, dtype=td).pin_memory()
                       for t in (bench.dq, bench.dk, bench.dv)]
            outs_d += [bench.dq, bench.dk, bench.dv]
        h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hdo, hl) if t is not None)
        d2h = sum(t.numel() * t.element_size() for t in outs_h)

        def e2e_step():
            q.copy_(hq, non_blocking=True)
            k.copy_(hk, non_blocking=True)
            v.copy_(hv, non_blocking=True)
            if hdo is not None:
                do.copy_(hdo, non_blocking=True)
            if hl is not None:
                lens.copy_(hl, non_blocking=True)
            bench.fwd()
            if w.has_bwd:
                bench.bwd()
            for hd, dd in zip(outs_h, outs_d):
                hd.copy_(dd, non_blocking=True)

        for _ in range(max(args.warmup, 3)):
            e2e_step()
        torch.cuda.synchronize()
        s_ev, e_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s_ev.record(stream)
        for _ in range(args.steps):
            e2e_step()
        e_ev.record(stream)
        torch.cuda.synchronize()
        e2e_ms = reduce_max(s_ev.elapsed_time(e_ev) / args.steps, dev)
        e2e = {"value": whole_job_tflops(step_fl, e2e_ms, world), "unit": "TFLOP/s",
               "ms_per_step": e2e_ms, "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "call": "attn_fwd + attn_bwd"}

    peaks, peak_src = load_peaks()
    fwd_mean = statistics.mean(fwd_ms)
    bwd_mean = statistics.mean(bwd_ms) if w.has_bwd else 0.0
    dom = "attn_bwd" if bwd_mean > fwd_mean else "attn_fwd"
    dom_fl = bwd_fl if dom == "attn_bwd" else fwd_fl
    dom_ms = bwd_mean if dom == "attn_bwd" else fwd_mean
    achieved = dom_fl / (dom_ms * 1e-3) / 1e12
    peak, bound, peak_note = tensor_peak(w, peaks, peak_src)
    kernels = {"attn_fwd": ("fwd_sm103_kernel (one launch per call)" if w.dtype == "bf16"
                            else "fwd_tf32x3_kernel (one launch per call)"),
               "attn_bwd": "bwd_delta + bwd_dq + bwd_dkdv (+ group reduce) kernels of one call"}
    roofline = {"bound": bound, "achieved": round(achieved, 3), "peak": peak,
                "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                "traffic": traffic_for(f"{dom}:{w.key}", w.dtype), "kernel": kernels[dom],
                "call": dom, "peak_source": peak_note,
                "algorithmic_flops_per_launch": dom_fl}
    if dom == "attn_bwd":
        roofline["per_kernel_est"] = bwd_kernel_estimates(w.key, w.dtype, bwd_mean, fwd_fl, peak)
    bf16_peak = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_max, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.dtype == "bf16" else "f32",
        "data": "synthetic: seeded N(0,1) inputs with the pages' shapes (no real activations)",
        "config": dict(cfg, l2="flushed (512 MiB write) before every step, outside the "
                               "timed events"),
        "pct_of_bf16_peak": round(100 * value / world / bf16_peak, 2),
        "peak_source": peak_src,
        "fwd_tflops": round(fwd_fl / (fwd_mean * 1e-3) / 1e12, 3),
        "bwd_tflops": round(bwd_fl / (bwd_mean * 1e-3) / 1e12, 3) if w.has_bwd else None,
        "fwd_ms": round(fwd_mean, 5), "bwd_ms": round(bwd_mean, 5) if w.has_bwd else None,
        "wall_s_timed": round(wall, 4),
        "e2e": e2e, "gpu_launches": int(launches), "roofline": roofline,
        "clocks": clocks, "library": attn.build_info(),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, inp, args.cpu_seconds)
    # the other graded workloads, timed the same way in the same process
    del bench, q, k, v, do, lens, o, lse
    also = {}
    for entry in [x for x in args.also.split(",") if x and x != w.key]:
        key, _, mode = entry.partition("@")
        wa = workloads.get(key)
        ba = Workbench(wa, workloads.make_inputs(wa), dev, stream, flush_buf, mode or "dense")
        also[entry] = also_entry(ba, args, world, sampler_index, peaks, peak_src, dev)
        del ba
        torch.cuda.empty_cache()
    if also:
        line["also"] = also
    if rank == 0:
        print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------- reference
def run_reference(args, world):
    w = workloads.get(args.workload)
    inp = workloads.make_inputs(w)
    cfg, _, _ = workload_config(w, inp)
    budget = 150.0  # seconds for warmup + steps together
    per_step = max(0.2, min(10.0, budget / max(1, args.steps + args.warmup)))
    run, fl, desc = oracle_sample(w, inp, per_step)
    for _ in range(args.warmup):
        run()
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        run()
        times.append(time.perf_counter() - t0)
    ms = 1e3 * statistics.mean(times)
    value = fl / (ms * 1e-3) / 1e12
    cores, threads = cpu_info()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic: seeded N(0,1) inputs with the pages' shapes",
        "config": cfg,
        "cpu_baseline": {"kind": "oracle", "cores": threads or cores, "host_cores": cores,
                         "sample": desc, "value": value, "unit": "TFLOP/s"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            run_reference(args, world)
        return
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
