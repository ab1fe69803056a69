"""Decode-attention benchmark: one step = the whole hot path over one batch.

A step on the 31B-shaped decode batch (B 64, L ~ U[8192, 32768], 32 query
heads; local 16 KV heads hd256 window 1024; global 4 KV heads hd512) is:
KV append (local) -> local decode (+ split-KV combine if planned) -> KV
append (global) -> global decode -> split-KV combine.  All of it runs in
libga's CUDA kernels through the C ABI.

Printed: one JSON line with the metric (algorithmic HBM GB/s of the step),
the roofline of the dominant kernel (global decode), the end-to-end figure
through host buffers, the CPU oracle baseline and the SM clocks seen.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("decode-attention HBM GB/s and % of GB300 peak; attended KV-tokens/sec per layer")
NOMINAL_HBM_GBS = 8000.0
WORKLOAD_INDEX = 3          # the 31B-shaped decode batch


def measured_peak_gbs():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            return float(json.load(fh)["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_split_kv_gqa_gb300", "csrc")
    for fn in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, fn), "rb") as fh:
            h.update(fn.encode() + fh.read())
    return h.hexdigest()[:16]


def committed_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if the kernel
    sources are unchanged since it was taken; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as fh:
            rec = json.load(fh).get(kernel)
    except Exception:
        return None
    if not rec or rec.get("source_hash") != kernel_source_hash():
        return None
    return rec.get("bytes_per_launch")


class ClockSampler:
    """nvidia-smi samples of SM clocks / throttle reasons during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ workload

def build_step(device, seed, rows=0):
    import torch
    from paged_split_kv_gqa_gb300 import ga
    from paged_split_kv_gqa_gb300 import metrics as M
    from paged_split_kv_gqa_gb300 import workloads as W

    wl = W.config(WORKLOAD_INDEX, seed=seed)
    if rows:
        wl = W.Workload(wl.name + f" (first {rows} rows)", wl.seq_lens[:rows].copy(),
                        wl.page_size, wl.local, wl.global_)
    fams = {}
    for fam in wl.families():
        fi = W.make_family_inputs(wl, fam, device=device, seed=seed,
                                  release_old=(fam.window > 0))
        plan = ga.ga_plan_splits(wl.seq_lens, num_q_heads=fam.num_q_heads,
                                 num_kv_heads=fam.num_kv_heads, head_dim=fam.head_dim,
                                 window=fam.window, flags=ga.GA_PLAN_EXTERNAL_COMBINE)
        ws = ga.workspace_for(plan, device)
        po, plse, _ = ga.workspace_views(plan, ws) if ws is not None else (None, None, None)
        esz = 1 if fam.kv_dtype == W.KV_E4M3 else 2
        fams[fam.name] = dict(
            fam=fam, fi=fi, plan=plan, ws=ws, po=po, plse=plse,
            out=torch.empty_like(fi.q), pos=(fi.seq_lens - 1).contiguous(),
            scale=1.0 / math.sqrt(fam.head_dim),
            bytes=M.decode_bytes(wl.seq_lens, num_q_heads=fam.num_q_heads,
                                 num_kv_heads=fam.num_kv_heads, head_dim=fam.head_dim,
                                 window=fam.window, page_size=wl.page_size,
                                 kv_bytes_per_elem=esz),
            append_bytes=M.append_bytes(wl.batch, num_kv_heads=fam.num_kv_heads,
                                        head_dim=fam.head_dim, kv_bytes_per_elem=esz),
            keys=int(M.attended_keys(wl.seq_lens, fam.window).sum()))
    err = torch.zeros(1, dtype=torch.int32, device=device)
    return wl, fams, err


def launch_family(ga, f, err, events=None):
    """append + decode (+ combine) of one family on the current stream.
    Returns the number of kernels launched."""
    fi, fam, plan = f["fi"], f["fam"], f["plan"]
    ga.ga_kv_append(fi.k_new, fi.v_new, fi.k_pool, fi.v_pool, fi.page_table, f["pos"],
                    k_scale=fi.k_scale, v_scale=fi.v_scale, err_word=err)
    kw = dict(scale=f["scale"], plan=plan, workspace=f["ws"], out=f["out"], k_scale=fi.k_scale,
              v_scale=fi.v_scale, err_word=err)
    if events is not None:
        events[0].record()
    if fam.window > 0:
        ga.ga_decode_local_hd256(fi.q, fi.k_pool, fi.v_pool, fi.page_table, fi.seq_lens,
                                 window=fam.window, **kw)
    else:
        ga.ga_decode_global_hd512(fi.q, fi.k_pool, fi.v_pool, fi.page_table, fi.seq_lens, **kw)
    if events is not None:
        events[1].record()
    n = 2
    if plan.mode != ga.GA_SPLIT_NONE:
        ga.ga_splitkv_combine(f["po"], f["plse"], plan, fi.seq_lens, fi.page_table.shape[1],
                              f["out"], err_word=err)
        n += 1
    return n


# ------------------------------------------------------------------ CPU oracle

def oracle_sample(fams_cpu, rows, nthreads=0):
    """Run the oracle on the sampled rows of both families; returns seconds."""
    from oracle import oracle as O
    t0 = time.perf_counter()
    for f in fams_cpu:
        O.decode(f.q, f.k_pool, f.v_pool, f.page_table, f.seq_lens,
                 num_kv_heads=f.family.num_kv_heads, window=f.family.window,
                 scale=1.0 / math.sqrt(f.family.head_dim), kv_dtype=f.family.kv_dtype,
                 k_scale=f.k_scale, v_scale=f.v_scale, rows=rows, nthreads=nthreads)
    return time.perf_counter() - t0


def cpu_sample_inputs(seed, nrows):
    """CPU copies of a bounded sample of the same workload: the first nrows
    rows of the batch (same lengths), drawn on the host."""
    from paged_split_kv_gqa_gb300 import metrics as M
    from paged_split_kv_gqa_gb300 import workloads as W
    wl = W.config(WORKLOAD_INDEX, seed=seed)
    sub = W.Workload(wl.name, wl.seq_lens[:nrows].copy(), wl.page_size, wl.local, wl.global_)
    fams = [W.make_family_inputs(sub, fam, device="cpu", seed=seed,
                                 release_old=(fam.window > 0)) for fam in sub.families()]
    nbytes = sum(M.decode_bytes(sub.seq_lens, num_q_heads=f.num_q_heads,
                                num_kv_heads=f.num_kv_heads, head_dim=f.head_dim,
                                window=f.window, page_size=sub.page_size,
                                kv_bytes_per_elem=2) for f in sub.families())
    keys = {f.name: int(M.attended_keys(sub.seq_lens, f.window).sum()) for f in sub.families()}
    return fams, nbytes, keys


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def run_cpu_baseline(seed, target_s=12.0):
    from oracle import oracle as O
    nrows = 2
    fams, nbytes, _ = cpu_sample_inputs(seed, nrows)
    t = oracle_sample(fams, None)
    # grow the sample toward ~target_s of CPU work (bounded)
    while t < target_s / 4 and nrows < 16:
        nrows = min(16, nrows * 2)
        fams, nbytes, _ = cpu_sample_inputs(seed, nrows)
        t = oracle_sample(fams, None)
    return {"value": nbytes / t / 1e9, "unit": "GB/s", "cores": O.max_threads(), "kind": "oracle",
            "sample": f"first {nrows} rows of the 31B-shaped batch, both families, fp64 C "
                      f"oracle with OpenMP, {t:.2f} s"}


# ------------------------------------------------------------------ arms

def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
            int(os.environ.get("WORLD_SIZE", 1)))


def run_reference(args):
    """The reference arm: the CPU oracle as it stands on the host cores."""
    rank, _, world = dist_env()
    if rank != 0:
        return
    from oracle import oracle as O
    nrows = 2
    fams, nbytes, keys = cpu_sample_inputs(args.seed, nrows)
    for _ in range(args.warmup):
        oracle_sample(fams, None)
    times = [oracle_sample(fams, None) for _ in range(args.steps)]
    t = sum(times) / len(times)
    value = nbytes / t / 1e9
    cb = {"value": value, "unit": "GB/s", "cores": O.max_threads(), "kind": "oracle",
          "sample": f"first {nrows} rows of the 31B-shaped batch per step, both families"}
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": t * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "31B-shaped decode, sampled rows", "batch": nrows},
            "cpu_baseline": cb,
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ga(args):
    import torch
    from paged_split_kv_gqa_gb300 import ga

    rank, local_rank, world = dist_env()
    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
        pg = dist
    wl, fams, err = build_step(device, args.seed + rank, args.rows)
    loc, glo = fams["local"], fams["global"]
    stream = torch.cuda.current_stream()

    def step(ev_local=None, ev_global=None):
        n = launch_family(ga, loc, err, ev_local)
        n += launch_family(ga, glo, err, ev_global)
        return n

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    if int(err.item()) != 0:
        raise RuntimeError(f"device error word {int(err.item())} during warm-up")

    # ---- device-timed region: K steps, events around each decode launch
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)] for _ in range(2)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches = 0
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clocks:
        start.record()
        for k in range(args.steps):
            launches += step(ev[0][k], ev[1][k])
        end.record()
        torch.cuda.synchronize()
    elapsed = start.elapsed_time(end) / 1e3
    if pg:
        t = torch.tensor([elapsed], device=device)
        pg.all_reduce(t, op=pg.ReduceOp.MAX)
        elapsed = float(t.item())
    if int(err.item()) != 0:
        raise RuntimeError(f"device error word {int(err.item())}")
    local_ms = [a.elapsed_time(b) for a, b in ev[0]]
    global_ms = [a.elapsed_time(b) for a, b in ev[1]]

    step_bytes = sum(f["bytes"] + f["append_bytes"] for f in fams.values())
    value = step_bytes * args.steps * world / elapsed / 1e9
    peak, peak_kind = measured_peak_gbs()
    g_avg = sum(global_ms) / len(global_ms) / 1e3
    l_avg = sum(local_ms) / len(local_ms) / 1e3
    g_ach = glo["bytes"] / g_avg / 1e9
    l_ach = loc["bytes"] / l_avg / 1e9
    traffic = committed_traffic("decode_global_hd512")

    # ---- end to end through host buffers: H2D inputs, the C-ABI calls, D2H outputs
    e2e = None
    if not args.no_e2e:
        host = {}
        for name, f in fams.items():
            fi = f["fi"]
            host[name] = {k: getattr(fi, k).cpu().pin_memory() for k in ("q", "k_new", "v_new",
                                                                         "seq_lens")}
            host[name]["pos"] = f["pos"].cpu().pin_memory()
            host[name]["out"] = torch.empty_like(f["out"], device="cpu").pin_memory()
        h2d = sum(t.numel() * t.element_size() for h in host.values()
                  for k, t in h.items() if k != "out")
        d2h = sum(h["out"].numel() * h["out"].element_size() for h in host.values())

        def e2e_step():
            n = 0
            for name, f in fams.items():
                fi, h = f["fi"], host[name]
                fi.q.copy_(h["q"], non_blocking=True)
                fi.k_new.copy_(h["k_new"], non_blocking=True)
                fi.v_new.copy_(h["v_new"], non_blocking=True)
                fi.seq_lens.copy_(h["seq_lens"], non_blocking=True)
                f["pos"].copy_(h["pos"], non_blocking=True)
                n += launch_family(ga, f, err)
                h["out"].copy_(f["out"], non_blocking=True)
            return n

        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        if pg:
            pg.barrier()
        s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s2.record()
        for _ in range(args.steps):
            e2e_step()
        e2.record()
        torch.cuda.synchronize()
        t_e2e = s2.elapsed_time(e2) / 1e3
        if pg:
            t = torch.tensor([t_e2e], device=device)
            pg.all_reduce(t, op=pg.ReduceOp.MAX)
            t_e2e = float(t.item())
        e2e = {"value": step_bytes * args.steps * world / t_e2e / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": t_e2e / args.steps * 1e3}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = run_cpu_baseline(args.seed)

    if rank == 0:
        def plan_desc(p):
            return {"mode": ["none", "count", "chunk"][p.mode], "chunk_pages": p.chunk_pages,
                    "units": p.units, "grid": p.grid}

        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": max(3, args.warmup),
            "ms_per_step": elapsed / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {
                "workload": ("31B-shaped decode: B64, L~U[8192,32768] seed 0, 32 q heads; local "
                             "16 kv hd256 window 1024 (bf16); global 4 kv hd512 (bf16); "
                             "page 16, shuffled page pool")
                            + (f" -- PROFILING SUBSET: first {args.rows} rows" if args.rows else ""),
                "global_batch": wl.batch * world, "step": "append+decode(+combine), both families",
                "l2": "inputs larger than L2 (global KV pools ~10.4 GB, local ~1.1 GB); no flush",
                "plans": {n: plan_desc(f["plan"]) for n, f in fams.items()},
            },
            "pct_of_peak": {"measured": value / peak, "nominal_8TBs": value / NOMINAL_HBM_GBS},
            "families": {
                n: {"decode_ms": (g_avg if n == "global" else l_avg) * 1e3,
                    "decode_gbs": g_ach if n == "global" else l_ach,
                    "attended_kv_tokens_per_s_per_layer":
                        f["keys"] / (g_avg if n == "global" else l_avg),
                    "algorithmic_bytes": f["bytes"]}
                for n, f in fams.items()},
            "roofline": {"kernel": "decode_global_hd512 (decode kernel, combine excluded)",
                         "bound": "hbm", "achieved": g_ach, "peak": peak,
                         "peak_kind": peak_kind, "unit": "GB/s", "frac": g_ach / peak,
                         "traffic": traffic},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches,
            "clocks": clocks.summary(),
        }
        print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ga", choices=["ga", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--rows", type=int, default=0,
                    help="profiling only: the first N rows of the batch (not a bench line)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ga(args)


if __name__ == "__main__":
    main()
