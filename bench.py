"""Decode-attention benchmark: one step = the whole hot path over one batch.

A step on the 31B-shaped decode batch (the default workload: B 64, L ~
U[8192, 32768], 32 query heads; local 16 KV heads hd256 window 1024; global 4
KV heads hd512) is: KV append (local) -> local decode (+ split-KV combine if
planned) -> KV append (global) -> global decode -> split-KV combine, each
append inside its decode launch (`--separate-append` launches it apart).
All of it runs in libga's CUDA kernels through the C ABI.  --workload ragged runs
the 50-local (fp8) + 10-global layer sweep instead.

Printed: one JSON line with the metric (algorithmic HBM GB/s of the step),
the roofline of the dominant kernel (global decode), the end-to-end figure
through host buffers, the CPU oracle baseline and the SM clocks seen.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference] [--workload W]
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


def measured_peak_gbs():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            return float(json.load(fh)["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# The sources a one-query decode launch's DRAM traffic depends on: both
# decode kernels (mma.sync and tcgen05), the headers they include, and the
# host code that encodes their tensor maps and makes their plans.  (The
# public header is left out: what of it the kernels use is restated by
# ga_internal.h and ga_api.cu, and its comments change with the docs.)
_CSRC = "paged_split_kv_gqa_gb300/csrc/"
DECODE_SOURCES = tuple(_CSRC + f for f in (
    "ga_api.cu", "ga_decode.cu", "ga_decode_tc.cu", "ga_decode_common.cuh", "ga_device.cuh",
    "ga_geometry.h", "ga_internal.h"))


def kernel_source_hash(files=DECODE_SOURCES):
    h = hashlib.sha256()
    for fn in sorted(files):
        with open(os.path.join(ROOT, fn), "rb") as fh:
            h.update(fn.encode() + fh.read())
    return h.hexdigest()[:16]


def committed_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary of this kernel in
    this workload's default step, if the decode sources are unchanged since
    it was taken; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as fh:
            rec = json.load(fh).get(kernel)
    except Exception:
        return None
    if (not rec or rec.get("workload") != workload
            or rec.get("source_hash") != kernel_source_hash()):
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

WORKLOADS = {"31b": 3, "12b": 2, "long": 4, "ragged": 5}


MQ_UNIT_FLAGS = {"auto": 0, "tc": "GA_PLAN_TENSOR_CORE_UNITS", "cp": "GA_PLAN_COLUMN_PARALLEL_UNITS"}
DEALS = {"round-robin": 0, "rows-by-size": 1}      # ga_plan.schedule


def make_layer(device, wl, fam, seed, layer, kv_alias=False, splits=0, q_len=1, mq_units="auto",
               fp8_units=0, separate_append=False, deal="auto"):
    """One layer's inputs.  q_len > 1: a multi-query step (q_len new tokens
    per row at its last positions, e.g. a speculative-decoding verify): the
    pools keep the union of the queries' windows, q / out are
    [B, Hq, q_len, D] and q_len tokens are appended per row."""
    import dataclasses

    import torch
    from paged_split_kv_gqa_gb300 import ga
    from paged_split_kv_gqa_gb300 import metrics as M
    from paged_split_kv_gqa_gb300 import workloads as W

    S = q_len
    alloc = fam if S == 1 else dataclasses.replace(fam, window=M.union_window(fam.window, S))
    fi = W.make_family_inputs(wl, alloc, device=device, seed=seed, layer=layer,
                              release_old=(fam.window > 0))
    if S == 1:
        q, kn, vn = fi.q, fi.k_new[None], fi.v_new[None]
    else:
        g = torch.Generator().manual_seed(seed * 7919 + layer * 31 + 5)
        B, Hq, D = fi.q.shape
        q = torch.randn(B, Hq, S, D, generator=g).to(torch.bfloat16).to(device)
        kn = torch.randn((S,) + tuple(fi.k_new.shape), generator=g).to(torch.bfloat16).to(device)
        vn = torch.randn((S,) + tuple(fi.v_new.shape), generator=g).to(torch.bfloat16).to(device)
    pos = torch.stack([fi.seq_lens - S + i for i in range(S)]).to(torch.int32).contiguous()
    alias = kv_alias and fam.window == 0
    if alias:                      # K == V: one pool serves both (global family)
        fi.v_pool = fi.k_pool
        fi.v_scale = fi.k_scale
    unit_flag = MQ_UNIT_FLAGS[mq_units]
    plan = ga.ga_plan_splits(wl.seq_lens, num_q_heads=fam.num_q_heads,
                             num_kv_heads=fam.num_kv_heads, head_dim=fam.head_dim,
                             window=fam.window, requested_splits=splits,
                             flags=ga.GA_PLAN_EXTERNAL_COMBINE |
                             (ga.GA_PLAN_KV_E4M3 if fam.kv_dtype == W.KV_E4M3 else 0) |
                             (getattr(ga, unit_flag) if unit_flag else 0), q_len=S)
    if fp8_units and fam.kv_dtype == W.KV_E4M3 and fam.window > 0:
        plan.kv_heads_per_unit = fp8_units        # A/B: force the E4M3 unit width
    if deal != "auto" and plan.mode in (ga.GA_SPLIT_NONE, ga.GA_SPLIT_CHUNK) and S == 1:
        plan.schedule = DEALS[deal]               # A/B: force how units are dealt to CTAs
    ws = ga.workspace_for(plan, device)
    po, plse, _ = ga.workspace_views(plan, ws) if ws is not None else (None, None, None)
    esz = 1 if fam.kv_dtype == W.KV_E4M3 else 2
    return dict(
        separate_append=separate_append,
        fam=fam, fi=fi, plan=plan, ws=ws, po=po, plse=plse, q=q, kn=kn, vn=vn, pos=pos,
        out=torch.empty_like(q), scale=1.0 / math.sqrt(fam.head_dim),
        bytes=M.decode_bytes(wl.seq_lens, num_q_heads=fam.num_q_heads,
                             num_kv_heads=fam.num_kv_heads, head_dim=fam.head_dim,
                             window=fam.window, page_size=wl.page_size, kv_bytes_per_elem=esz,
                             kv_alias=alias, q_len=S),
        append_bytes=S * M.append_bytes(wl.batch, num_kv_heads=fam.num_kv_heads,
                                        head_dim=fam.head_dim, kv_bytes_per_elem=esz),
        keys=int(M.attended_keys(wl.seq_lens, M.union_window(fam.window, S)).sum()))


def workload_config(workload, seed, fp8="none"):
    """The named workload; fp8 ("local", "global", "both") stores those
    families' KV pools as E4M3 with per-head scales instead of bf16."""
    import dataclasses

    from paged_split_kv_gqa_gb300 import workloads as W
    wl = W.config(WORKLOADS[workload], seed=seed)
    if fp8 == "none":
        return wl
    loc, glo = wl.local, wl.global_
    if fp8 in ("local", "both"):
        loc = dataclasses.replace(loc, kv_dtype=W.KV_E4M3)
    if fp8 in ("global", "both"):
        glo = dataclasses.replace(glo, kv_dtype=W.KV_E4M3)
    return W.Workload(wl.name, wl.seq_lens, wl.page_size, loc, glo, wl.local_layers,
                      wl.global_layers)


def build_step(device, seed, workload="31b", rows=0, pools=4, kv_alias=False, splits=0,
               q_len=1, fp8="none", mq_units="auto", fp8_units=0, separate_append=False,
               deal="auto"):
    """The layers one step launches, in order.  31b / 12b / long: one local and
    one global layer.  ragged: 50 local + 10 global layers in 5:1 order, the
    layers of a family rotating over `pools` distinct KV pools (each > L2).
    splits: 0 lets the planner choose, s > 0 asks every plan for s chunks per row."""
    import torch
    from paged_split_kv_gqa_gb300 import workloads as W

    wl = workload_config(workload, seed, fp8)
    if rows:
        wl = W.Workload(wl.name + f" (first {rows} rows)", wl.seq_lens[:rows].copy(),
                        wl.page_size, wl.local, wl.global_, wl.local_layers, wl.global_layers)
    npool = pools if workload == "ragged" else 1
    sets = {fam.name: [make_layer(device, wl, fam, seed, i, kv_alias, splits, q_len, mq_units,
                                  fp8_units, separate_append, deal)
                       for i in range(npool)]
            for fam in wl.families()}
    if workload == "ragged":
        schedule, nl, ng = [], 0, 0
        per = wl.local_layers // wl.global_layers           # 5 local, then 1 global
        for _ in range(wl.global_layers):
            for _ in range(per):
                schedule.append(sets["local"][nl % npool]); nl += 1
            schedule.append(sets["global"][ng % npool]); ng += 1
    else:
        schedule = [sets["local"][0], sets["global"][0]]
    err = torch.zeros(1, dtype=torch.int32, device=device)
    return wl, schedule, sets, err


def launch_layer(ga, f, err, events=None):
    """append + decode (+ combine) of one layer on the current stream.  A
    one-query step appends inside the decode launch (the decode call with the
    append fused) unless the layer asks for the append kernel first
    (`separate_append`).  Returns the number of kernels launched."""
    fi, fam, plan = f["fi"], f["fam"], f["plan"]
    S = f["kn"].shape[0]
    fused = S == 1 and not f["separate_append"]
    if not fused:
        for i in range(S):             # this step's new token(s) of every row
            ga.ga_kv_append(f["kn"][i], f["vn"][i], fi.k_pool, fi.v_pool, fi.page_table,
                            f["pos"][i], k_scale=fi.k_scale, v_scale=fi.v_scale, err_word=err)
    kw = dict(scale=f["scale"], plan=plan, workspace=f["ws"], out=f["out"], k_scale=fi.k_scale,
              v_scale=fi.v_scale, err_word=err)
    if events is not None:
        events[0].record()
    if fused and fam.window > 0:
        ga.ga_decode_local_hd256_append(f["kn"][0], f["vn"][0], f["q"], fi.k_pool, fi.v_pool,
                                        fi.page_table, fi.seq_lens, window=fam.window, **kw)
    elif fused:
        ga.ga_decode_global_hd512_append(f["kn"][0], f["vn"][0], f["q"], fi.k_pool, fi.v_pool,
                                         fi.page_table, fi.seq_lens, **kw)
    elif fam.window > 0:
        ga.ga_decode_local_hd256(f["q"], fi.k_pool, fi.v_pool, fi.page_table, fi.seq_lens,
                                 window=fam.window, **kw)
    else:
        ga.ga_decode_global_hd512(f["q"], fi.k_pool, fi.v_pool, fi.page_table, fi.seq_lens,
                                  **kw)
    if events is not None:
        events[1].record()
    # the decode launch, plus the append kernel(s) when not fused (or when a
    # kv head's query heads span several units: the call appends first)
    n = 1 + (S if not fused else (1 if fam.num_q_heads // fam.num_kv_heads > 8 else 0))
    if plan.mode != ga.GA_SPLIT_NONE:
        ga.ga_splitkv_combine(f["po"], f["plse"], plan, fi.seq_lens, fi.page_table.shape[1],
                              f["out"], err_word=err)
        n += 1
    return n


# ------------------------------------------------------------------ CPU oracle

def oracle_sample(fams_cpu, nthreads=0):
    """Run the oracle on every row of the sampled inputs (nthreads 0: all
    host cores); returns seconds."""
    from oracle import oracle as O
    t0 = time.perf_counter()
    for f in fams_cpu:
        fn = O.decode_mq if f.q.dim() == 4 else O.decode      # [B, Hq, S, D]: S queries
        fn(f.q, f.k_pool, f.v_pool, f.page_table, f.seq_lens,
           num_kv_heads=f.family.num_kv_heads, window=f.family.window,
           scale=1.0 / math.sqrt(f.family.head_dim), kv_dtype=f.family.kv_dtype,
           k_scale=f.k_scale, v_scale=f.v_scale, nthreads=nthreads)
    return time.perf_counter() - t0


def cpu_sample_inputs(seed, nrows, workload, fp8="none"):
    """CPU copies of a bounded sample of the same workload: its first nrows
    rows (same lengths), one layer per family, drawn on the host."""
    from paged_split_kv_gqa_gb300 import metrics as M
    from paged_split_kv_gqa_gb300 import workloads as W
    wl = workload_config(workload, seed, fp8)
    sub = W.Workload(wl.name, wl.seq_lens[:nrows].copy(), wl.page_size, wl.local, wl.global_)
    fams = [W.make_family_inputs(sub, fam, device="cpu", seed=seed,
                                 release_old=(fam.window > 0)) for fam in sub.families()]
    nbytes = sum(M.decode_bytes(sub.seq_lens, num_q_heads=f.num_q_heads,
                                num_kv_heads=f.num_kv_heads, head_dim=f.head_dim,
                                window=f.window, page_size=sub.page_size,
                                kv_bytes_per_elem=1 if f.kv_dtype == W.KV_E4M3 else 2)
                 for f in sub.families())
    return fams, nbytes


def gather_rows_to_host(layer, nrows):
    """Host copies of the first nrows rows of a device layer: only the pages
    those rows reference, renumbered, plus their q, table and lengths."""
    import numpy as np
    import torch
    from paged_split_kv_gqa_gb300 import workloads as W
    fi = layer["fi"]
    table = fi.page_table[:nrows].cpu().numpy()
    used = np.unique(table[table >= 0])
    remap = np.full(max(int(fi.num_pages), 1), -1, dtype=np.int64)
    remap[used] = np.arange(len(used))
    sub = np.where(table >= 0, remap[np.maximum(table, 0)], -1).astype(np.int32)
    idx = torch.as_tensor(used, device=fi.k_pool.device)
    q = layer["q"][:nrows].cpu()
    if q.dim() == 4 and q.shape[2] == 1:
        q = q[:, :, 0].contiguous()
    return W.FamilyInputs(layer["fam"], q, fi.k_pool.index_select(0, idx).cpu(),
                          fi.v_pool.index_select(0, idx).cpu(),
                          None if fi.k_scale is None else fi.k_scale.cpu(),
                          None if fi.v_scale is None else fi.v_scale.cpu(),
                          torch.from_numpy(sub), fi.seq_lens[:nrows].cpu(), None, None,
                          len(used))


def run_cpu_baseline(sets, batch, target_s=10.0):
    """The oracle as it stands on the host cores, on the first rows of the
    bench's own inputs (one layer per family), the sample grown toward about
    target_s / 2 .. target_s of work or the whole batch."""
    from oracle import oracle as O
    from paged_split_kv_gqa_gb300 import metrics as M
    from paged_split_kv_gqa_gb300 import workloads as W
    nrows = min(batch, 4)
    while True:
        fams = [gather_rows_to_host(layers[0], nrows) for layers in sets.values()]
        t = oracle_sample(fams)
        if t >= target_s / 2 or nrows >= batch:
            break
        nrows = min(batch, max(nrows + 1, int(nrows * min(8.0, 0.75 * target_s / max(t, 1e-3)))))
    def sample_bytes(fs):
        lens = fs[0].seq_lens.numpy()
        return sum(M.decode_bytes(lens, num_q_heads=f.family.num_q_heads,
                                  num_kv_heads=f.family.num_kv_heads, head_dim=f.family.head_dim,
                                  window=f.family.window, page_size=16,
                                  kv_bytes_per_elem=1 if f.family.kv_dtype == W.KV_E4M3 else 2,
                                  q_len=f.q.shape[2] if f.q.dim() == 4 else 1)
                   for f in fs)
    nbytes = sample_bytes(fams)
    # the same oracle on one core, on the first row only (a few seconds)
    one = [gather_rows_to_host(layers[0], 1) for layers in sets.values()]
    t1 = oracle_sample(one, nthreads=1)
    return {"value": nbytes / t / 1e9, "unit": "GB/s", "cores": O.max_threads(), "kind": "oracle",
            "sample": f"first {nrows} of {batch} rows of the bench batch, one layer per family, "
                      f"fp64 C oracle with OpenMP on all cores, {t:.2f} s",
            "single_thread": {"value": sample_bytes(one) / t1 / 1e9, "unit": "GB/s", "cores": 1,
                              "sample": f"first row, one layer per family, {t1:.2f} s"}}


# ------------------------------------------------------------------ arms

def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
            int(os.environ.get("WORLD_SIZE", 1)))


def workload_text(args):
    text = WORKLOAD_TEXT[args.workload]
    if args.rows:
        text += f" -- PROFILING SUBSET: first {args.rows} rows"
    if args.workload == "ragged":
        text += f"; {args.pools} distinct pools per family rotated over the layers"
    if args.kv_alias:
        text += "; global family with K == V (one pool, read once)"
    if args.fp8 != "none":
        text += f"; {args.fp8} family KV stored as fp8-e4m3 with per-head scales"
    if args.splits:
        text += f"; split-KV count fixed at {args.splits} chunks per row"
    if args.q_len > 1:
        text += (f"; {args.q_len} query tokens per row at its last positions (causal "
                 f"within the chunk), {args.q_len} appends per row and layer")
    if args.fp8_units:
        text += f"; E4M3 sliding-family units of {args.fp8_units} kv heads forced"
    if args.separate_append:
        text += "; append kernel launched before each decode (not fused)"
    if args.deal != "auto":
        text += f"; unsplit and chunked plans deal units {args.deal}"
    if args.mq_units != "auto":
        text += {"tc": "; tcgen05 units of 64 columns forced",
                 "cp": "; column-parallel mma.sync units forced"}[args.mq_units]
    return text


def host_schedule(args, wl):
    """The step's layers as the bench runs them, with each layer's algorithmic
    decode bytes, computed on the host (the same object for a layer that is
    repeated, as the bench's rotated pools are)."""
    from paged_split_kv_gqa_gb300 import metrics as M
    from paged_split_kv_gqa_gb300 import workloads as W

    def layer(fam):
        esz = 1 if fam.kv_dtype == W.KV_E4M3 else 2
        return {"bytes": M.decode_bytes(wl.seq_lens, num_q_heads=fam.num_q_heads,
                                        num_kv_heads=fam.num_kv_heads, head_dim=fam.head_dim,
                                        window=fam.window, page_size=wl.page_size,
                                        kv_bytes_per_elem=esz,
                                        kv_alias=args.kv_alias and fam.window == 0,
                                        q_len=args.q_len)}
    if args.workload != "ragged":
        return [layer(wl.local), layer(wl.global_)]
    loc = [layer(wl.local) for _ in range(args.pools)]
    glo = [layer(wl.global_) for _ in range(args.pools)]
    schedule, nl, ng = [], 0, 0
    per = wl.local_layers // wl.global_layers
    for _ in range(wl.global_layers):
        for _ in range(per):
            schedule.append(loc[nl % args.pools])
            nl += 1
        schedule.append(glo[ng % args.pools])
        ng += 1
    return schedule


def line_config(args, wl, world):
    """The `config` of the JSON line, the same for the GPU arm and the
    reference arm: the workload, the whole-job batch and what keeps each timed
    repetition reading from HBM."""
    return {"workload": workload_text(args), "global_batch": wl.batch * world,
            "parallelism": f"replicas x{world}: one independent batch per rank, no exchange",
            "l2": l2_claim(host_schedule(args, wl))}


def run_reference(args):
    """The reference arm: the CPU oracle as it stands on the host cores."""
    rank, _, world = dist_env()
    if rank != 0:
        return
    from oracle import oracle as O
    nrows = 2
    wl = workload_config(args.workload, args.seed, args.fp8)
    if args.rows:
        from paged_split_kv_gqa_gb300 import workloads as W
        wl = W.Workload(wl.name, wl.seq_lens[:args.rows].copy(), wl.page_size, wl.local,
                        wl.global_, wl.local_layers, wl.global_layers)
    fams, nbytes = cpu_sample_inputs(args.seed, nrows, args.workload, args.fp8)
    for _ in range(args.warmup):
        oracle_sample(fams)
    times = [oracle_sample(fams) for _ in range(args.steps)]
    t = sum(times) / len(times)
    value = nbytes / t / 1e9
    cb = {"value": value, "unit": "GB/s", "cores": O.max_threads(), "kind": "oracle",
          "sample": f"first {nrows} rows of the {args.workload} batch per step, one layer per "
                    f"family"}
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": t * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": line_config(args, wl, world),
            "cpu_baseline": cb,
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


WORKLOAD_TEXT = {
    "31b": "31B-shaped decode: B64, L~U[8192,32768] seed 0, 32 q heads; local 16 kv hd256 window "
           "1024 (bf16); global 4 kv hd512 (bf16); page 16, shuffled page pool",
    "12b": "12B-shaped decode: B32, L~U[512,4096] (rows 0-2 = 1023/1024/1025), 16 q heads; local "
           "8 kv hd256 window 1024; global 2 kv hd512; bf16; page 16",
    "long": "long-context 31B-shaped decode: B4, L=131072, 32 q heads; local 16 kv hd256 window "
            "1024; global 4 kv hd512; bf16; page 16",
    "ragged": "ragged 31B-shaped decode: B256, lognormal L (median 2048, sigma 1, clip "
              "[1,65536]); 50 local (fp8-e4m3, per-head scales) + 10 global (bf16) layers in 5:1 "
              "order; page 16",
}


L2_BYTES = 129 << 20     # GB300 L2 (nominal 129 MB; 126.5 MiB as reported)


def l2_claim(schedule):
    """What keeps each timed decode reading from HBM, computed for this step:
    a byte of a layer's KV is read again only after that layer's other bytes
    and the other layers' reads in between (cyclically over replayed steps)
    have streamed through L2.  If that reuse distance exceeds L2 for every
    layer, no flush is needed and the line says so; if not, it says that too."""
    n = len(schedule)
    reuse = []
    for i, layer in enumerate(schedule):
        b, j = layer["bytes"], (i + 1) % n
        while schedule[j] is not layer:
            b += schedule[j]["bytes"]
            j = (j + 1) % n
        reuse.append(b)
    least = min(reuse) if reuse else 0
    if least > L2_BYTES:
        return (f"no flush: every byte of KV is re-read only after >= {least / 1e6:.0f} MB "
                f"of other reads (> {L2_BYTES / 1e6:.0f} MB L2)")
    return (f"NOT flushed: KV bytes can be re-read after only {least / 1e6:.0f} MB of other "
            f"reads (< {L2_BYTES / 1e6:.0f} MB L2); L2 hits possible")


def one_page_rows_ms(ga, layer, err, device, reps=21):
    """The fixed part of a decode launch of this family: the same decode call
    (batch, heads, pools, table, a plan made the same way; the combine is
    timed apart, as for the family's own figure) with every row cut to one
    page (16 keys), median of `reps` launches timed with CUDA events.  The
    family's launch time minus this is the time spent streaming its KV."""
    import torch
    fi, fam, plan = layer["fi"], layer["fam"], layer["plan"]
    B = fi.seq_lens.numel()
    S = plan.q_len
    lens = torch.full((B,), max(16, S), dtype=torch.int32, device=device)
    p16 = ga.ga_plan_splits([max(16, S)] * B, num_q_heads=fam.num_q_heads,
                            num_kv_heads=fam.num_kv_heads, head_dim=fam.head_dim,
                            window=fam.window, flags=plan.flags, q_len=S)
    ws = ga.workspace_for(p16, device)
    out = torch.empty_like(layer["out"])
    kw = dict(scale=layer["scale"], plan=p16, workspace=ws, out=out, k_scale=fi.k_scale,
              v_scale=fi.v_scale, err_word=err)

    def call():
        if fam.window > 0:
            ga.ga_decode_local_hd256(layer["q"], fi.k_pool, fi.v_pool, fi.page_table, lens,
                                     window=fam.window, **kw)
        else:
            ga.ga_decode_global_hd512(layer["q"], fi.k_pool, fi.v_pool, fi.page_table, lens,
                                      **kw)

    for _ in range(3):
        call()
    ts = []
    for _ in range(reps):
        if hasattr(torch.cuda, "_sleep"):     # the host enqueues ahead of the GPU
            torch.cuda._sleep(1_000_000)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        call()
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    return sorted(ts)[len(ts) // 2]


def run_unit_cost(args):
    """Profiling only (no bench line): the fixed and per-unit cost of each
    decode kernel on the 31B shapes.  Rows of 1, 4, 16 or 64 pages, one kv
    head per unit, no split, 2 to 16 units per CTA; each launch timed alone
    with CUDA events (median of 15), and a least-squares line through the
    times: intercept = the launch's fixed part, slope = one unit's time.
    The stream time of a unit at the measured copy bandwidth's per-SM share
    is printed beside it."""
    import torch
    from paged_split_kv_gqa_gb300 import _build
    _build.build()
    from paged_split_kv_gqa_gb300 import ga
    from paged_split_kv_gqa_gb300 import workloads as W
    device = "cuda"
    err = torch.zeros(1, dtype=torch.int32, device=device)
    sms = ga.num_sms()
    peak, _ = measured_peak_gbs()
    wl31 = W.config(3)
    for fam0 in (wl31.local, wl31.global_):
        for kv in (W.KV_BF16, W.KV_E4M3):
            fam = W.Family(fam0.name, fam0.num_q_heads, fam0.num_kv_heads, fam0.head_dim,
                           fam0.window, kv)
            for npg in (1, 4, 16, 64):
                pts = []
                for upc in (2, 4, 8, 16):
                    B = max(1, upc * sms // fam.num_kv_heads)
                    lens = np.full(B, 16 * npg, dtype=np.int32)
                    wl = W.Workload("unit-cost", lens, 16, fam, fam)
                    fi = W.make_family_inputs(wl, fam, device=device, seed=args.seed + 1)
                    plan = ga.ga_plan_splits(
                        lens, num_q_heads=fam.num_q_heads, num_kv_heads=fam.num_kv_heads,
                        head_dim=fam.head_dim, window=fam.window, requested_splits=1,
                        flags=ga.GA_PLAN_KV_E4M3 if kv == W.KV_E4M3 else 0)
                    plan.kv_heads_per_unit = 1
                    ws = ga.workspace_for(plan, device)
                    kw = dict(scale=1.0 / math.sqrt(fam.head_dim), plan=plan, workspace=ws,
                              out=torch.empty_like(fi.q), k_scale=fi.k_scale,
                              v_scale=fi.v_scale, err_word=err)

                    def call():
                        if fam.window > 0:
                            ga.ga_decode_local_hd256(fi.q, fi.k_pool, fi.v_pool, fi.page_table,
                                                     fi.seq_lens, window=fam.window, **kw)
                        else:
                            ga.ga_decode_global_hd512(fi.q, fi.k_pool, fi.v_pool, fi.page_table,
                                                      fi.seq_lens, **kw)
                    for _ in range(3):
                        call()
                    ts = []
                    for _ in range(15):
                        if hasattr(torch.cuda, "_sleep"):
                            torch.cuda._sleep(1_000_000)
                        a = torch.cuda.Event(enable_timing=True)
                        b = torch.cuda.Event(enable_timing=True)
                        a.record()
                        call()
                        b.record()
                        torch.cuda.synchronize()
                        ts.append(a.elapsed_time(b))
                    pts.append((B * fam.num_kv_heads / sms, sorted(ts)[len(ts) // 2] * 1e3))
                    del fi, ws, kw
                    torch.cuda.empty_cache()
                slope, icpt = np.polyfit([x for x, _ in pts], [y for _, y in pts], 1)
                esz = 1 if kv == W.KV_E4M3 else 2
                unit_bytes = 2 * npg * 16 * fam.head_dim * esz
                print(json.dumps({
                    "family": fam.name, "kv_dtype": "e4m3" if kv == W.KV_E4M3 else "bf16",
                    "pages_per_unit": npg, "units_per_cta_us": [[round(x, 2), round(y, 2)]
                                                                 for x, y in pts],
                    "fixed_us": round(float(icpt), 2), "us_per_unit": round(float(slope), 2),
                    "unit_stream_us_at_peak_share": round(unit_bytes / (peak * 1e3 / sms), 2)}),
                    flush=True)
    torch.cuda.synchronize()
    if int(err.item()) != 0:
        raise RuntimeError(f"device error word {int(err.item()):#x}")


def run_ga(args):
    import torch
    from paged_split_kv_gqa_gb300 import ga

    rank, local_rank, world = dist_env()
    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    pg = None
    # under torchrun (even with one rank) the barrier and the max over ranks
    # run through the process group, as they do on N GPUs
    if world > 1 or "LOCAL_WORLD_SIZE" in os.environ:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
        pg = dist
    wl, schedule, sets, err = build_step(device, args.seed + rank, args.workload, args.rows,
                                         args.pools, args.kv_alias, args.splits, args.q_len,
                                         args.fp8, args.mq_units, args.fp8_units,
                                         args.separate_append, args.deal)

    def step(evs=None):
        n = 0
        for i, layer in enumerate(schedule):
            n += launch_layer(ga, layer, err, None if evs is None else evs[i])
        return n

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    if int(err.item()) != 0:
        raise RuntimeError(f"device error word {int(err.item())} during warm-up")

    # --graph: the whole step captured once in a CUDA graph and replayed
    graph, per_step = None, 0
    if not args.eager:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            per_step = step()
        graph.replay()
        torch.cuda.synchronize()

    # ---- device-timed region: K steps (eager: events around each decode launch)
    ev_steps = min(args.steps, 50) if graph is not None else args.steps
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in schedule] for _ in range(ev_steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches = 0
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clocks:
        start.record()
        for k in range(args.steps):
            if graph is not None:
                graph.replay()
                launches += per_step
            else:
                launches += step(ev[k])
        end.record()
        torch.cuda.synchronize()
    elapsed = start.elapsed_time(end) / 1e3
    if graph is not None:          # per-family kernel times from an eager pass
        # a GPU-side wait first, so the host enqueues the whole pass before it
        # runs and no decode's events include host launch overhead
        if hasattr(torch.cuda, "_sleep"):
            torch.cuda._sleep(100_000_000)
        for k in range(ev_steps):
            step(ev[k])
        torch.cuda.synchronize()
    if pg:
        t = torch.tensor([elapsed], device=device)
        pg.all_reduce(t, op=pg.ReduceOp.MAX)
        elapsed = float(t.item())
    if int(err.item()) != 0:
        raise RuntimeError(f"device error word {int(err.item())}")

    # per family: decode-kernel time and algorithmic bytes over all its launches
    fam_ms, fam_bytes, fam_keys, fam_n = {}, {}, {}, {}
    for k in range(ev_steps):
        for i, layer in enumerate(schedule):
            name = layer["fam"].name
            a, b = ev[k][i]
            fam_ms[name] = fam_ms.get(name, 0.0) + a.elapsed_time(b)
            fam_bytes[name] = fam_bytes.get(name, 0) + layer["bytes"]
            fam_keys[name] = fam_keys.get(name, 0) + layer["keys"]
            fam_n[name] = fam_n.get(name, 0) + 1
    families = {}
    for name in fam_ms:
        t = fam_ms[name] / 1e3
        families[name] = {
            "launches_per_step": fam_n[name] // ev_steps,
            "decode_ms_per_launch": fam_ms[name] / fam_n[name],
            "decode_gbs": fam_bytes[name] / t / 1e9,
            "algorithmic_bytes_per_launch": fam_bytes[name] // fam_n[name],
            "attended_kv_tokens_per_s_per_layer": fam_keys[name] / t,
            "kv_dtype": "e4m3" if sets[name][0]["fam"].kv_dtype else "bf16"}
    for name in families:
        families[name]["one_page_rows_ms"] = one_page_rows_ms(ga, sets[name][0], err, device)
    dominant = max(fam_ms, key=fam_ms.get)
    step_bytes = sum(layer["bytes"] + layer["append_bytes"] for layer in schedule)
    value = step_bytes * args.steps * world / elapsed / 1e9
    peak, peak_kind = measured_peak_gbs()
    dom_ach = families[dominant]["decode_gbs"]
    kname = "decode_global_hd512" if dominant == "global" else "decode_local_hd256"
    if families[dominant]["kv_dtype"] == "e4m3":
        kname += "_e4m3"
    # the committed counters cover a workload's default step: the planner's
    # plans and deal, the workload's own KV dtypes, the append fused
    default_step = (not args.rows and not args.splits and not args.kv_alias
                    and args.q_len == 1 and args.fp8 == "none" and args.deal == "auto"
                    and not args.fp8_units and not args.separate_append
                    and (args.workload != "ragged" or args.pools == 4))
    traffic = committed_traffic(kname, args.workload) if default_step else None

    # ---- end to end through host buffers: H2D inputs, the C-ABI calls, D2H outputs
    e2e = None
    if not args.no_e2e:
        host = {}
        uniq = [layer for fam_layers in sets.values() for layer in fam_layers]
        for layer in uniq:
            fi = layer["fi"]
            # positions only where an append kernel reads them (the fused
            # append takes L - 1 from seq_lens)
            keys = ("q", "kn", "vn") if (layer["kn"].shape[0] == 1 and
                                         not layer["separate_append"]) else ("q", "kn", "vn", "pos")
            h = {k: layer[k].cpu().pin_memory() for k in keys}
            h["seq_lens"] = fi.seq_lens.cpu().pin_memory()
            h["out"] = torch.empty_like(layer["out"], device="cpu").pin_memory()
            host[id(layer)] = h
        h2d = sum(t.numel() * t.element_size() for layer in schedule
                  for k, t in host[id(layer)].items() if k != "out")
        d2h = sum(host[id(layer)]["out"].numel() * 2 for layer in schedule)

        # Host copies run on two side streams so that a layer's inputs land
        # and its output is read back while other layers decode.  The step
        # is software-pipelined: it starts with the read-back of the previous
        # step's last output and ends by copying in the next step's first
        # inputs, so no copy waits at a step boundary.  A prologue (first
        # inputs) and an epilogue (last read-back) inside the timed region
        # complete the first and last step: every step still moves its own
        # inputs in and its result out within the clock.  Events order each
        # use of a layer's buffers after the previous decode / read-back of
        # the same buffers.  The step (copies + C-ABI calls on three streams
        # forked from and joined into the launching one) is captured once in
        # a CUDA graph and replayed like the device-timed step; --eager
        # enqueues it from Python every step instead.
        h2d_stream, d2h_stream = torch.cuda.Stream(device), torch.cuda.Stream(device)
        first, final = schedule[0], schedule[-1]
        assert first is not final

        def copy_inputs(layer):
            h = host[id(layer)]
            for k in ("q", "kn", "vn", "pos"):
                if k in h:
                    layer[k].copy_(h[k], non_blocking=True)
            layer["fi"].seq_lens.copy_(h["seq_lens"], non_blocking=True)

        def read_back(layer):
            host[id(layer)]["out"].copy_(layer["out"], non_blocking=True)

        def e2e_body():
            cs = torch.cuda.current_stream(device)
            fork = torch.cuda.Event()
            fork.record(cs)
            h2d_stream.wait_event(fork)
            d2h_stream.wait_event(fork)
            joins = []
            with torch.cuda.stream(d2h_stream):        # the previous step's result
                read_back(final)
                prev = torch.cuda.Event()
                prev.record(d2h_stream)
            joins.append(prev)
            last, n = {}, 0
            for j, layer in enumerate(schedule):
                i = id(layer)
                e = {k: torch.cuda.Event() for k in ("done", "inputs", "copied")}
                if j > 0:                              # (the first inputs came with the last step)
                    if i in last:
                        h2d_stream.wait_event(last[i]["done"])     # its last decode is over
                    with torch.cuda.stream(h2d_stream):
                        copy_inputs(layer)
                        e["inputs"].record(h2d_stream)
                    cs.wait_event(e["inputs"])
                if i in last:
                    cs.wait_event(last[i]["copied"])   # its last read-back is over
                elif layer is final:
                    cs.wait_event(prev)
                n += launch_layer(ga, layer, err)
                e["done"].record(cs)
                if j < len(schedule) - 1:              # (the last one is read back next step)
                    d2h_stream.wait_event(e["done"])
                    with torch.cuda.stream(d2h_stream):
                        read_back(layer)
                        e["copied"].record(d2h_stream)
                    joins.append(e["copied"])
                last[i] = e
            h2d_stream.wait_event(last[id(first)]["done"])
            with torch.cuda.stream(h2d_stream):        # the next step's first inputs
                copy_inputs(first)
                nxt = torch.cuda.Event()
                nxt.record(h2d_stream)
            joins.append(nxt)
            for ev_ in joins:                          # join every side-stream copy
                cs.wait_event(ev_)
            return n

        copy_inputs(first)                             # prime (outside any timing)
        torch.cuda.synchronize()
        e2e_graph = None
        if not args.eager:
            e2e_body()                                 # warm the allocator / plans
            torch.cuda.synchronize()
            e2e_graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(e2e_graph):
                e2e_body()

        def e2e_step():
            if e2e_graph is not None:
                e2e_graph.replay()
            else:
                e2e_body()

        def time_e2e(step_fn):
            for _ in range(3):
                step_fn()
            torch.cuda.synchronize()
            if pg:
                pg.barrier()
            s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s2.record()
            copy_inputs(first)                         # prologue: step 0's first inputs
            for _ in range(args.steps):
                step_fn()
            read_back(final)                           # epilogue: the last step's result
            e2.record()
            torch.cuda.synchronize()
            t = s2.elapsed_time(e2) / 1e3
            if pg:
                tt = torch.tensor([t], device=device)
                pg.all_reduce(tt, op=pg.ReduceOp.MAX)
                t = float(tt.item())
            return t

        t_e2e = time_e2e(e2e_step)
        # every read-back must equal its device output (deterministic kernels,
        # same inputs each step): a read-back that raced its decode would not
        outputs_match = all(torch.equal(host[id(layer)]["out"], layer["out"].cpu())
                            for layer in {id(layer): layer for layer in schedule}.values())
        e2e = {"value": step_bytes * args.steps * world / t_e2e / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": t_e2e / args.steps * 1e3,
               "read_back_matches_device": bool(outputs_match),
               "mode": "eager" if e2e_graph is None else "graph_replay",
               "copies": "pinned host buffers; H2D and D2H on two side streams overlapping "
                         "other layers' decode; a step reads back the previous step's last "
                         "output first and copies in the next step's first inputs last "
                         "(prologue and epilogue inside the timed region); "
                         + ("every copy and C-ABI call enqueued from Python each step"
                            if e2e_graph is None else
                            "the step's copies and calls replayed from one CUDA graph")}
        if e2e_graph is not None:
            # the same pipelined step with every C-ABI call (argument checks,
            # tensor-map encoding, launch) made from the host each step, as a
            # caller that does not capture graphs pays it
            t_eager = time_e2e(e2e_body)
            eager_match = all(torch.equal(host[id(layer)]["out"], layer["out"].cpu())
                              for layer in {id(layer): layer for layer in schedule}.values())
            e2e["eager"] = {"value": step_bytes * args.steps * world / t_eager / 1e9,
                            "unit": "GB/s", "ms_per_step": t_eager / args.steps * 1e3,
                            "read_back_matches_device": bool(eager_match),
                            "how": "same copies; every copy and C-ABI call enqueued from "
                                   "Python (ctypes) each step, no graph"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = run_cpu_baseline(sets, wl.batch)

    # The practical HBM read ceiling on this GPU (own read-only stream kernel,
    # 4 GiB > L2, after the timed region): the decode kernels' second denominator
    ceiling = None
    if rank == 0 and not args.rows:
        buf = torch.empty(4 << 30, dtype=torch.uint8, device=device)
        sink = torch.zeros(1, dtype=torch.int64, device=device)
        for _ in range(2):
            ga.ga_read_stream(buf, sink)
        s3, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s3.record()
        for _ in range(10):
            ga.ga_read_stream(buf, sink)
        e3.record()
        torch.cuda.synchronize()
        ceiling = buf.numel() * 10 / (s3.elapsed_time(e3) / 1e3) / 1e9
        del buf

    if rank == 0:
        def plan_desc(p):
            return {"mode": ["none", "count", "chunk"][p.mode], "splits": p.splits,
                    "chunk_pages": p.chunk_pages, "col_tile": p.col_tile,
                    "units": p.units, "grid": p.grid}

        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": max(3, args.warmup),
            "ms_per_step": elapsed / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": line_config(args, wl, world),
            "step": f"{len(schedule)} layers, each append+decode(+combine)"
                    + ("" if args.eager else "; captured in one CUDA graph, replayed"),
            "plans": {n: plan_desc(layers[0]["plan"]) for n, layers in sets.items()},
            "pct_of_peak": {"measured": value / peak, "nominal_8TBs": value / NOMINAL_HBM_GBS},
            "families": families,
            "roofline": {"kernel": f"{kname} (decode kernel, combine excluded)",
                         "bound": "hbm", "achieved": dom_ach, "peak": peak,
                         "peak_kind": peak_kind, "unit": "GB/s", "frac": dom_ach / peak,
                         "frac_of_nominal_8TBs": dom_ach / NOMINAL_HBM_GBS,
                         "read_ceiling_gbs": ceiling,
                         "frac_of_read_ceiling": (dom_ach / ceiling) if ceiling else None,
                         "read_ceiling_kernel": "ga_read_stream: own read-only stream, 16-byte "
                                                "loads, 4 GiB, 10 passes",
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
    ap.add_argument("--workload", default="31b", choices=sorted(WORKLOADS))
    ap.add_argument("--kv-alias", action="store_true",
                    help="global family with K == V: one pool, each block read once")
    ap.add_argument("--eager", action="store_true",
                    help="launch every call from Python in the timed loop instead of replaying "
                         "one captured CUDA graph of the step")
    ap.add_argument("--pools", type=int, default=4,
                    help="ragged workload: distinct KV pools per family rotated over layers")
    ap.add_argument("--rows", type=int, default=0,
                    help="profiling only: the first N rows of the batch (not a bench line)")
    ap.add_argument("--splits", type=int, default=0,
                    help="split-KV chunks per row for every plan (0 = planner's choice)")
    ap.add_argument("--q-len", type=int, default=1,
                    help="query tokens per row (> 1: a multi-query / speculative-verify step)")
    ap.add_argument("--fp8", default="none", choices=["none", "local", "global", "both"],
                    help="store these families' KV pools as fp8-e4m3 with per-head scales")
    ap.add_argument("--separate-append", action="store_true",
                    help="one-query steps launch the append kernel before the decode instead "
                         "of the decode call with the append fused (A/B)")
    ap.add_argument("--deal", default="auto", choices=["auto"] + sorted(DEALS),
                    help="how one-query plans (unsplit, or in fixed-size chunks) deal work "
                         "units to the CTAs: the "
                         "planner's choice, or forced (A/B)")
    ap.add_argument("--fp8-units", type=int, default=0,
                    help="kv heads per unit of the E4M3 sliding-family decode (1, or 8 / group): "
                         "forces the width the planner would otherwise choose (A/B)")
    ap.add_argument("--mq-units", default="auto", choices=sorted(MQ_UNIT_FLAGS),
                    help="multi-query units for more than 8 (query, head) columns per kv head: "
                         "the planner's choice, tcgen05 units of 64 columns, or column-parallel "
                         "mma.sync units of 32")
    ap.add_argument("--unit-cost", action="store_true",
                    help="profiling only: fixed and per-unit cost of each decode kernel on the "
                         "31B shapes (one JSON line per kernel and unit length, no bench line)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    if args.unit_cost:
        return run_unit_cost(args)
    world = dist_env()[2]
    if "WORLD_SIZE" in os.environ and args.gpus != world:
        ap.error(f"--gpus {args.gpus} but {world} ranks were launched")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ga(args)


if __name__ == "__main__":
    main()
