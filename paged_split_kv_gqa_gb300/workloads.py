"""Seeded synthetic decode workloads (Gemma-4-shaped).

This module only draws inputs: sequence lengths, page tables, bf16 q / K / V,
fp8 codes with their per-head scales, and the new token of a decode step.  It
holds none of the attention arithmetic, and it is the one module both the CUDA
path's tests and the CPU oracle's tests use.

Shapes follow the pages: the local family is sliding-window attention at
head_dim 256 with a 1024-token window, the global family full attention at
head_dim 512 with fewer KV heads ("[Model] Gemma 4 M1 12B", Description;
"[Model] Gemma 4 M3 31B", Description and Acceptance Criteria).  31B global
decode is 32 query heads over 4 KV heads ("visible-cx/Gemma-4-31B-CoreAI",
hybrid-pf64 numerics gate).  The opt-in FP8 pool is for the sliding family
("[Model] Gemma 4 M2 26B-A4B", Proposed Plan).

Recipe (all seeds 0 unless given): every random tensor has its own
``torch.Generator`` seeded from (seed, tag); bf16 values are N(0, 1);
physical pages are a random permutation of a pool with spare pages; spare
pages and never-attended slots can be filled with NaN ("poison") so that a
read the definition does not make shows up in the output.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import numpy as np
import torch

PAGE_SIZE = 16
KV_BF16 = 0
KV_E4M3 = 1

_TAGS = {"q": 1, "k": 2, "v": 3, "lens": 4, "perm": 5, "k_new": 6, "v_new": 7, "noise": 8}


def generator(seed: int, tag: str, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 1000003 + _TAGS[tag] * 7919 + 17)
    return g


@dataclasses.dataclass(frozen=True)
class Family:
    name: str            # "local" or "global"
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    window: int          # 0 = global (whole context)
    kv_dtype: int = KV_BF16


@dataclasses.dataclass
class Workload:
    name: str
    seq_lens: np.ndarray          # [B] int32, host copy
    page_size: int
    local: Family
    global_: Family
    local_layers: int = 1
    global_layers: int = 1

    @property
    def batch(self) -> int:
        return int(len(self.seq_lens))

    def families(self) -> List[Family]:
        return [self.local, self.global_]


def _lens_uniform(B, lo, hi, seed):
    g = generator(seed, "lens")
    return torch.randint(lo, hi + 1, (B,), generator=g, dtype=torch.int64).numpy().astype(np.int32)


def config(index: int, seed: int = 0) -> Workload:
    """The five workload shapes: 1 tiny, 2 12B, 3 31B, 4 long context, 5 ragged."""
    if index == 1:
        lens = np.array([40, 33], dtype=np.int32)
        return Workload("tiny: B2 L{40,33} local 4q/2kv hd256 W32, global 4q/1kv hd512",
                        lens, PAGE_SIZE,
                        Family("local", 4, 2, 256, 32), Family("global", 4, 1, 512, 0))
    if index == 2:
        lens = _lens_uniform(32, 512, 4096, seed)
        lens[0], lens[1], lens[2] = 1023, 1024, 1025
        return Workload("12B-shaped: B32 L~U[512,4096] (rows 0-2 = 1023/1024/1025) 16q, "
                        "local 8kv hd256 W1024, global 2kv hd512", lens, PAGE_SIZE,
                        Family("local", 16, 8, 256, 1024), Family("global", 16, 2, 512, 0))
    if index == 3:
        lens = _lens_uniform(64, 8192, 32768, seed)
        return Workload("31B-shaped: B64 L~U[8192,32768] 32q, local 16kv hd256 W1024, "
                        "global 4kv hd512", lens, PAGE_SIZE,
                        Family("local", 32, 16, 256, 1024), Family("global", 32, 4, 512, 0))
    if index == 4:
        lens = np.full(4, 131072, dtype=np.int32)
        return Workload("long-context 31B-shaped: B4 L=131072, 32q, local 16kv hd256 W1024, "
                        "global 4kv hd512", lens, PAGE_SIZE,
                        Family("local", 32, 16, 256, 1024), Family("global", 32, 4, 512, 0))
    if index == 5:
        g = generator(seed, "lens")
        z = torch.randn(256, generator=g, dtype=torch.float64).numpy()
        lens = np.clip(np.rint(np.exp(math.log(2048.0) + 1.0 * z)), 1, 65536).astype(np.int32)
        return Workload("ragged 31B-shaped: B256 lognormal L (median 2048, sigma 1, clip "
                        "[1,65536]), local fp8-e4m3 16kv hd256 W1024, global bf16 4kv hd512, "
                        "50 local + 10 global layers", lens, PAGE_SIZE,
                        Family("local", 32, 16, 256, 1024, KV_E4M3),
                        Family("global", 32, 4, 512, 0), local_layers=50, global_layers=10)
    raise ValueError(f"no workload {index}")


# ------------------------------------------------------------------ layout

def allocated_logical_pages(L: int, page_size: int, window: int, release_old: bool):
    """Logical pages a KV manager keeps for a row of length L.

    All pages 0 .. ceil(L / P) - 1, except that with release_old a sliding-
    window family releases every page whose newest slot is older than the
    window (its slots p*P .. p*P+P-1 are all < L - window).
    """
    n = -(-int(L) // page_size)
    pages = list(range(n))
    if release_old and window > 0:
        pages = [p for p in pages if (p + 1) * page_size > L - window]
    return pages


@dataclasses.dataclass
class FamilyInputs:
    family: Family
    q: torch.Tensor            # [B, Hq, D] bf16
    k_pool: torch.Tensor       # [num_pages, Hkv, P, D] bf16 or uint8 (e4m3 codes)
    v_pool: torch.Tensor
    k_scale: Optional[torch.Tensor]   # [Hkv] fp32 (fp8 only)
    v_scale: Optional[torch.Tensor]
    page_table: torch.Tensor   # [B, stride] int32
    seq_lens: torch.Tensor     # [B] int32
    k_new: torch.Tensor        # [B, Hkv, D] bf16
    v_new: torch.Tensor
    num_pages: int


BF16_NAN_BITS = 0x7FC0
E4M3_NAN_CODE = 0x7F


def make_family_inputs(wl: Workload, fam: Family, *, device="cpu", seed: int = 0,
                       spare_pages: Optional[int] = None, poison: bool = False,
                       release_old: bool = False, stride_pad: int = 0,
                       layer: int = 0) -> FamilyInputs:
    """Draw one layer's inputs for one family of a workload.

    spare_pages: pool pages beyond those allocated (default ~3% + 3).
    poison: NaN-fill spare pages and slots no query of this step attends
      (slots at or beyond L in a row's last page; for a windowed family the
      slots older than the window).
    release_old: page-table entries of released pages are -1 and no pool page
      backs them (sliding-window family only).
    """
    P = wl.page_size
    B = wl.batch
    Hq, Hkv, D = fam.num_q_heads, fam.num_kv_heads, fam.head_dim
    s = seed + 101 * layer + (0 if fam.name == "local" else 50)
    lens = wl.seq_lens.astype(np.int64)
    per_row = [allocated_logical_pages(int(L), P, fam.window, release_old) for L in lens]
    n_alloc = sum(len(r) for r in per_row)
    if spare_pages is None:
        spare_pages = n_alloc // 32 + 3
    num_pages = n_alloc + spare_pages
    stride = max(1, max((-(-int(L) // P) for L in lens), default=1)) + stride_pad
    perm = torch.randperm(num_pages, generator=generator(s, "perm")).numpy().astype(np.int64)
    table = np.full((B, stride), -1, dtype=np.int32)
    k = 0
    for b, pages in enumerate(per_row):
        for p in pages:
            table[b, p] = perm[k]
            k += 1
    dev = torch.device(device)
    gq = generator(s, "q", "cpu")
    q = torch.randn(B, Hq, D, generator=gq, dtype=torch.float32).to(torch.bfloat16).to(dev)
    shape = (num_pages, Hkv, P, D)
    gdev = "cuda" if dev.type == "cuda" else "cpu"
    gk = generator(s, "k", gdev)
    gv = generator(s, "v", gdev)
    kf = torch.randn(shape, generator=gk, device=dev, dtype=torch.bfloat16)
    vf = torch.randn(shape, generator=gv, device=dev, dtype=torch.bfloat16)
    k_scale = v_scale = None
    if fam.kv_dtype == KV_E4M3:
        k_scale = (kf.abs().amax(dim=(0, 2, 3)).float() / 448.0).clamp_min(1e-12)
        v_scale = (vf.abs().amax(dim=(0, 2, 3)).float() / 448.0).clamp_min(1e-12)
        k_pool = _to_e4m3_codes(kf, k_scale)
        v_pool = _to_e4m3_codes(vf, v_scale)
        del kf, vf
    else:
        k_pool, v_pool = kf, vf
    if poison:
        _poison(k_pool, v_pool, table, lens, fam, P, perm[:n_alloc])
    kn = torch.randn(B, Hkv, D, generator=generator(s, "k_new"), dtype=torch.float32)
    vn = torch.randn(B, Hkv, D, generator=generator(s, "v_new"), dtype=torch.float32)
    return FamilyInputs(fam, q, k_pool, v_pool,
                        None if k_scale is None else k_scale.to(dev),
                        None if v_scale is None else v_scale.to(dev),
                        torch.from_numpy(table).to(dev),
                        torch.from_numpy(lens.astype(np.int32)).to(dev),
                        kn.to(torch.bfloat16).to(dev), vn.to(torch.bfloat16).to(dev),
                        num_pages)


def _to_e4m3_codes(x: torch.Tensor, scale: torch.Tensor) -> torch.Tensor:
    y = (x.float() / scale.view(1, -1, 1, 1)).clamp(-448.0, 448.0)
    return y.to(torch.float8_e4m3fn).view(torch.uint8)


def _nan_fill(pool: torch.Tensor, fam: Family):
    if fam.kv_dtype == KV_E4M3:
        return E4M3_NAN_CODE
    return float("nan")


def _poison(k_pool, v_pool, table, lens, fam: Family, P: int, used: np.ndarray):
    """NaN-fill spare pages and never-attended slots (see make_family_inputs)."""
    num_pages = k_pool.shape[0]
    dev = k_pool.device
    fill = _nan_fill(k_pool, fam)
    used_mask = np.zeros(num_pages, dtype=bool)
    used_mask[used] = True
    whole = list(np.nonzero(~used_mask)[0])          # spare pages
    partial = []                                     # (page, slot_lo, slot_hi)
    for b, L in enumerate(lens):
        L = int(L)
        if L <= 0:
            continue
        if L % P:
            partial.append((int(table[b, (L - 1) // P]), L % P, P))
        if fam.window > 0 and L > fam.window:
            oldest = L - fam.window           # first attended position
            for p in range(0, oldest // P):
                if table[b, p] >= 0:
                    whole.append(int(table[b, p]))
            if oldest % P:
                page = int(table[b, oldest // P])
                partial.append((page, 0, oldest % P))
    if whole:
        idx = torch.as_tensor(np.array(whole, dtype=np.int64), device=dev)
        k_pool[idx] = fill
        v_pool[idx] = fill
    for page, lo, hi in partial:
        k_pool[page, :, lo:hi, :] = fill
        v_pool[page, :, lo:hi, :] = fill


def sample_rows(B: int, n: int, seed: int = 0) -> np.ndarray:
    """n distinct row indices (always including the first and last row)."""
    if n >= B:
        return np.arange(B, dtype=np.int32)
    g = torch.Generator().manual_seed(seed + 4242)
    mid = torch.randperm(max(B - 2, 1), generator=g)[: max(n - 2, 0)].numpy() + 1
    rows = sorted(set([0, B - 1] + [int(x) for x in mid]))
    return np.array(rows[:n], dtype=np.int32)
