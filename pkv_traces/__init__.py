"""Seeded synthetic decode traces for paged-KV GQA decode attention.

This module is the one piece shared by the CUDA path's tests/bench and the
CPU oracle's tests: it draws inputs (lengths, block tables, q/K/V values) and
holds none of the attention arithmetic.  Everything is a pure function of
(config id, seed) so both sides consume the same fp16 bytes.

Trace families follow "PersistentKV: Page-Aware Decode Scheduling for
Long-Context LLM Serving on Commodity GPUs", technical summary, Methodology
section 3 "Evaluation protocol": synthetic Bucketed, Bimodal, Uniform and
Zipf-like traces isolating context length, active batch and length
irregularity.  The pages give no generator parameters; the shapes below are
the five workloads this library is measured on:

  1  B=1  Hq=8  Hkv=2 d=128 P=16  N=1024, 64 pages drawn without replacement
     from a 128-page pool, random order; S=4 splits (C=256)
  2  B=1  Hq=32 Hkv=8 d=128 P=16  N=32768, block table a random permutation of
     a 2048-page pool; S=32 splits of C=1024; keys scaled by 0.5
  3  B=8  Hq=32 Hkv=8 d=128 P=16  bimodal: 4 rows ~U[512,2048], 4 rows
     ~U[24576,32768] (row order shuffled); C=1024; pool = sum of pages, shuffled
  4  B=4 or 8, Hq=32 Hkv=8 d=128 P=16  truncated Zipf s=1.2 on [16,32768]
  5  B=64 Hq=64 Hkv=8 d=128 P=16  U[128,65536]; pool sum ceil((N+256)/P)
     pages shuffled so 256 appended tokens per row fit; 256 decode steps; the
     workload names no split size: C=4096 (the fastest measured on GB300,
     where each split's fp32 partial state costs write traffic)

Seeds: results use the held-out seed 20260623, policy thresholds the
calibration seed 20260622 (technical summary, "Results", first paragraph).
Random streams: ``numpy.random.default_rng([seed, cfg_id])``.  Values are
fp32 standard normals rounded to fp16 (round-to-nearest-even by numpy).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import numpy as np

HELDOUT_SEED = 20260623
CALIBRATION_SEED = 20260622

ZIPF_S = 1.2
ZIPF_LO, ZIPF_HI = 16, 32768


@dataclasses.dataclass
class Trace:
    """One decode batch: shapes, lengths and the paged layout (no values)."""

    name: str
    cfg_id: int
    seed: int
    B: int
    Hq: int
    Hkv: int
    d: int
    page_size: int
    split_tokens: int
    num_pages: int
    seq_lens: np.ndarray          # int32 [B]
    block_table: np.ndarray       # int32 [B, bt_stride]; unused entries = -1
    k_scale: float = 1.0          # K values multiplied by this before the fp16 cast
    steps: int = 1                # decode steps (config 5 appends one token per step)
    path_hint: str = "policy"     # 'bucketed' | 'workqueue' | 'policy' | 'single'

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def bt_stride(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def n_max(self) -> int:
        return int(self.seq_lens.max()) if self.B else 0

    def kv_bytes(self) -> int:
        """Algorithmic K+V bytes of one decode step: sum_i N_i * Hkv * d * 2 * 2."""
        return int(self.seq_lens.astype(np.int64).sum()) * self.Hkv * self.d * 2 * 2

    def rng(self, stream: int) -> np.random.Generator:
        return np.random.default_rng([self.seed, self.cfg_id, stream])


# ----------------------------------------------------------------- lengths

def zipf_lengths(rng: np.random.Generator, n: int, s: float = ZIPF_S,
                 lo: int = ZIPF_LO, hi: int = ZIPF_HI) -> np.ndarray:
    """Truncated discrete power law P(N) proportional to N^-s on integers [lo, hi].

    "Clipped" is read as truncation; sampled by inverse CDF on the exact pmf.
    """
    support = np.arange(lo, hi + 1, dtype=np.float64)
    pmf = support ** (-s)
    cdf = np.cumsum(pmf)
    cdf /= cdf[-1]
    u = rng.random(n)
    idx = np.searchsorted(cdf, u, side="left")
    return (lo + idx).astype(np.int32)


def _scatter_pages(rng: np.random.Generator, pages_per_row: Sequence[int],
                   num_pages: Optional[int] = None) -> tuple[np.ndarray, int]:
    """Give each row its pages from a shuffled pool; returns (block_table, num_pages)."""
    total = int(sum(pages_per_row))
    if num_pages is None:
        num_pages = total
    num_pages = max(1, num_pages)  # a pool holds at least one page
    assert num_pages >= total
    perm = rng.permutation(num_pages)[:total].astype(np.int32)
    stride = max(1, max(pages_per_row) if len(pages_per_row) else 1)
    bt = np.full((len(pages_per_row), stride), -1, dtype=np.int32)
    pos = 0
    for i, n in enumerate(pages_per_row):
        bt[i, :n] = perm[pos:pos + n]
        pos += n
    return bt, num_pages


def _pages(n: int, P: int) -> int:
    return (n + P - 1) // P


# ----------------------------------------------------------------- configs

def make_trace(cfg_id: int, seed: int = HELDOUT_SEED, B: Optional[int] = None,
               len_scale: float = 1.0) -> Trace:
    """Build the (lengths, block table) part of workload ``cfg_id`` (1..5).

    len_scale (workloads 3 and 5 only) multiplies every drawn length (rounded,
    at least 1) before the pages are laid out: the same batch structure with a
    smaller pool, for profiler captures that must stay small."""
    rng = np.random.default_rng([seed, cfg_id])
    if len_scale != 1.0 and cfg_id not in (3, 5):
        raise ValueError("len_scale applies to workloads 3 and 5")
    scaled = lambda a: np.maximum(1, np.rint(a * len_scale)).astype(np.int32) \
        if len_scale != 1.0 else a
    P = 16
    if cfg_id == 1:
        N = 1024
        pool = 128
        pages = rng.choice(pool, size=N // P, replace=False).astype(np.int32)
        return Trace("bucketed-short", 1, seed, 1, 8, 2, 128, P, 256, pool,
                     np.array([N], np.int32), pages[None, :].copy(),
                     path_hint="bucketed")
    if cfg_id == 2:
        N = 32768
        pool = 2048
        pages = rng.permutation(pool).astype(np.int32)
        return Trace("bucketed-long", 2, seed, 1, 32, 8, 128, P, 1024, pool,
                     np.array([N], np.int32), pages[None, :].copy(), k_scale=0.5,
                     path_hint="bucketed")
    if cfg_id == 3:
        short = rng.integers(512, 2048, size=4, endpoint=True)
        long_ = rng.integers(24576, 32768, size=4, endpoint=True)
        lens = scaled(np.concatenate([short, long_])[rng.permutation(8)].astype(np.int32))
        bt, pool = _scatter_pages(rng, [_pages(int(n), P) for n in lens])
        return Trace("bimodal", 3, seed, 8, 32, 8, 128, P, 1024, pool, lens, bt,
                     path_hint="workqueue")
    if cfg_id == 4:
        b = 8 if B is None else int(B)
        lens = zipf_lengths(rng, b)
        bt, pool = _scatter_pages(rng, [_pages(int(n), P) for n in lens])
        return Trace(f"zipf-B{b}", 4, seed, b, 32, 8, 128, P, 1024, pool, lens, bt,
                     path_hint="policy")
    if cfg_id == 5:
        lens = scaled(rng.integers(128, 65536, size=64, endpoint=True).astype(np.int32))
        bt, pool = _scatter_pages(rng, [_pages(int(n) + 256, P) for n in lens])
        return Trace("uniform-B64", 5, seed, 64, 64, 8, 128, P, 4096, pool, lens, bt,
                     steps=256, path_hint="workqueue")
    raise ValueError(f"unknown config {cfg_id}")


def custom_trace(seq_lens: Sequence[int], Hq: int, Hkv: int, d: int = 128, P: int = 16,
                 C: int = 256, seed: int = HELDOUT_SEED, extra_pages: int = 0,
                 extra_cols: int = 0, share_prefix_pages: int = 0,
                 name: str = "custom", tag: int = 100) -> Trace:
    """A trace with given lengths, for edge cases.

    extra_pages: pool pages that no row references (a pool larger than needed).
    extra_cols: unused block-table columns (a row stride wider than needed).
    share_prefix_pages: rows 1.. reuse row 0's first pages (read-only prefix sharing).
    """
    rng = np.random.default_rng([seed, tag, len(seq_lens), Hq, Hkv, d, P, C])
    lens = np.asarray(seq_lens, dtype=np.int32)
    per_row = [_pages(int(n), P) for n in lens]
    bt, pool = _scatter_pages(rng, per_row, sum(per_row) + extra_pages)
    if extra_cols:
        bt = np.concatenate([bt, np.full((len(lens), extra_cols), -1, np.int32)], axis=1)
    if share_prefix_pages and len(lens) > 1:
        for i in range(1, len(lens)):
            k = min(share_prefix_pages, per_row[i], per_row[0])
            bt[i, :k] = bt[0, :k]
    return Trace(name, tag, seed, len(lens), Hq, Hkv, d, P, C, pool, lens, bt)


# ----------------------------------------------------------------- values

def gen_q(tr: Trace) -> np.ndarray:
    """q [B, Hq, d] fp16, standard normal."""
    return tr.rng(1).standard_normal((tr.B, tr.Hq, tr.d), dtype=np.float32).astype(np.float16)


def gen_kv(tr: Trace, poison_unused: bool = False) -> tuple[np.ndarray, np.ndarray]:
    """k_cache, v_cache [num_pages, P, Hkv, d] fp16 on the host (NHD page layout).

    poison_unused fills every slot that no row's valid tokens reference with
    NaN, so a read outside the row-local bounds shows up in the output.
    """
    shape = (tr.num_pages, tr.page_size, tr.Hkv, tr.d)
    k = tr.rng(2).standard_normal(shape, dtype=np.float32)
    if tr.k_scale != 1.0:
        k *= np.float32(tr.k_scale)
    k = k.astype(np.float16)
    v = tr.rng(3).standard_normal(shape, dtype=np.float32).astype(np.float16)
    if poison_unused:
        used = used_slot_mask(tr)
        k[~used] = np.float16(np.nan)
        v[~used] = np.float16(np.nan)
    return k, v


def used_slot_mask(tr: Trace) -> np.ndarray:
    """bool [num_pages, P]: slots holding some row's valid token."""
    used = np.zeros((tr.num_pages, tr.page_size), dtype=bool)
    for i in range(tr.B):
        n = int(tr.seq_lens[i])
        t = np.arange(n)
        used[tr.block_table[i, t // tr.page_size], t % tr.page_size] = True
    return used


def gen_kv_torch(tr: Trace, device: str = "cuda"):
    """k_cache, v_cache as torch fp16 tensors drawn by torch's seeded generator.

    Used for pools too large to draw on the host in reasonable time (config 5):
    same distribution, a different (torch) stream seeded from (seed, cfg_id).
    """
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(tr.seed * 1000 + tr.cfg_id)
    shape = (tr.num_pages, tr.page_size, tr.Hkv, tr.d)
    k = torch.empty(shape, dtype=torch.float16, device=device)
    v = torch.empty(shape, dtype=torch.float16, device=device)
    # draw in slabs so the fp32 temporary stays small
    slab = max(1, (1 << 26) // (tr.page_size * tr.Hkv * tr.d))
    for t, mult in ((k, tr.k_scale), (v, 1.0)):
        for p0 in range(0, tr.num_pages, slab):
            p1 = min(tr.num_pages, p0 + slab)
            x = torch.randn((p1 - p0,) + shape[1:], generator=g, device=device,
                            dtype=torch.float32)
            if mult != 1.0:
                x.mul_(mult)
            t[p0:p1].copy_(x)
    return k, v


def gen_append_tokens(tr: Trace, step: int) -> tuple[np.ndarray, np.ndarray]:
    """K/V of the token appended to every row at decode step ``step``: [B, Hkv, d] fp16."""
    rng = np.random.default_rng([tr.seed, tr.cfg_id, 10, step])
    k = rng.standard_normal((tr.B, tr.Hkv, tr.d), dtype=np.float32)
    if tr.k_scale != 1.0:
        k *= np.float32(tr.k_scale)
    v = rng.standard_normal((tr.B, tr.Hkv, tr.d), dtype=np.float32)
    return k.astype(np.float16), v.astype(np.float16)


def gen_step_q(tr: Trace, step: int) -> np.ndarray:
    """q for decode step ``step`` of a multi-step trace: [B, Hq, d] fp16."""
    if step == 0:
        return gen_q(tr)
    rng = np.random.default_rng([tr.seed, tr.cfg_id, 11, step])
    return rng.standard_normal((tr.B, tr.Hq, tr.d), dtype=np.float32).astype(np.float16)


def allocation_split(tr: Trace) -> tuple[np.ndarray, np.ndarray]:
    """For decode loops that allocate pages on the device: the block table with
    only the pages each row's current tokens fill (the rest set to -1), and the
    remaining pool pages as a free list in the shuffled order the table gave
    them (returned reversed, so the first page a row would take is on top)."""
    bt = tr.block_table.copy()
    free = []
    for i in range(tr.B):
        n = _pages(int(tr.seq_lens[i]), tr.page_size)
        row = bt[i]
        free.extend(row[n:][row[n:] >= 0].tolist())
        row[n:] = -1
    return bt, np.array(free[::-1], dtype=np.int32)
