#!/usr/bin/env python3
"""Benchmark: decode-attention KV-read GB/s and microseconds per decode step.

Default workload (N=1): B=64 uniform lengths U[128, 65536], Hq=64, Hkv=8
(G=8), d=128, page_size 16, a shuffled pool sized to the total length, the
compact workqueue with C=4096, and every step appending one token per row
(an append launch that allocates pages from a device free list, then the
decode, which builds the workqueue's plan itself, and the merge) -- the largest workload that fits one
GPU.  `--config 1..4` selects the smaller workloads (1: B=1 N=1024; 2: B=1
N=32768 bucketed split; 3: B=8 bimodal; 4: B=8 Zipf).

One JSON line on rank 0:
  value        K+V bytes of the step's valid tokens / device time per step
               (CUDA events around K back-to-back steps replayed from CUDA
               graphs of at least 8 chained steps; inputs resident in HBM;
               inputs larger than L2, or KV pools rotated so the data a step
               reads is not in L2)
  roofline     the decode kernel: algorithmic K+V bytes per launch / its
               duration per launch in a CUDA graph of back-to-back decode
               launches chained by programmatic dependent launch, as inside
               the step; the per-launch event-bracketed times (launched alone)
               are reported apart under `isolated`
  e2e          the same metric through the C ABI's host-buffer step
               (pkv_decode_step_host, or pkv_append_decode_step_host when the
               workload appends): the step's inputs copied from pinned host
               memory, the step, its outputs copied back, synchronized; wall
               clock per step.  `e2e.graph_loop` times the Python
               HostDecodeLoop (one captured graph per step) beside it
  cpu_baseline the float64 oracle on the host cores on a bounded sample
`--merge fused` merges on the decode kernel's tail; on the workqueue the decode
builds its own plan (no plan launch; an appending step's append launch then
only appends and allocates) unless `--plan separate`.  `--len-scale f` scales the B=8 / B=64 workloads' lengths by f (small
cases for profiler captures).  `--impl reference` times the oracle alone (the
reference arm).
Multi-GPU (torchrun): every rank runs an independent replica (no collective
on the data path); value sums the ranks' bytes over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "decode-attention KV-read GB/s (% of GB300 HBM peak); µs per decode step"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e nominal (8 stacks at 3996 MHz), context for the copy peak

WORKLOADS = {
    1: "B=1 GQA decode Hq=8 Hkv=2 d=128 N=1024 P=16 (64 pages of a 128-page pool) S=4 (C=256)",
    2: "B=1 long-context bucketed Hq=32 Hkv=8 d=128 N=32768 P=16 (2048-page pool permutation) "
       "S=32 (C=1024), keys x0.5",
    3: "B=8 bimodal (4x U[512,2048], 4x U[24576,32768]) Hq=32 Hkv=8 d=128 P=16 C=1024 workqueue",
    4: "B=8 Zipf s=1.2 on [16,32768] Hq=32 Hkv=8 d=128 P=16, policy route",
    5: "B=64 uniform U[128,65536] Hq=64 Hkv=8 d=128 P=16 C=4096 workqueue, +1 token/row/step",
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--impl", default="pkv", choices=["pkv", "reference"])
    ap.add_argument("--config", type=int, default=5, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--path", default="policy", choices=["policy", "bucketed", "workqueue", "single"])
    ap.add_argument("--no-graph", action="store_true", help="launch steps eagerly")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--merge", default="separate", choices=["fused", "separate"],
                    help="split paths: merge on the decode's tail, or in a second kernel")
    ap.add_argument("--plan", default="in-decode", choices=["in-decode", "separate"],
                    help="workqueue without appends: the decode builds its own plan, or a plan kernel")
    ap.add_argument("--len-scale", type=float, default=1.0,
                    help="scale the lengths of the B=8 bimodal and B=64 uniform workloads")
    ap.add_argument("--split-tokens", type=int, default=None,
                    help="split size C on the split paths, instead of the workload's")
    return ap.parse_args()


def workload_name(cfg_id: int, len_scale: float = 1.0) -> str:
    name = WORKLOADS[cfg_id]
    return name if len_scale == 1.0 else f"{name}, lengths x{len_scale:g}"


def default_steps(cfg_id):
    # about a second of timed device work per run
    return {1: 20000, 2: 40000, 3: 10000, 4: 20000, 5: 256}[cfg_id]


# ------------------------------------------------------------------ ranks

def dist_setup(args):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
        pg = dist
    return rank, local, ws, pg


def barrier(pg):
    if pg is not None:
        pg.barrier()


def reduce_max(pg, x: float) -> float:
    if pg is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(kv_bytes_per_rank: int, ms_per_step_max: float, world: int) -> float:
    """Replicas: every rank streams its own step; the job's throughput is all
    ranks' bytes over the slowest rank's time per step."""
    return kv_bytes_per_rank * world / (ms_per_step_max * 1e-3) / 1e9


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples, each stamped on arrival, kept if inside [t0, t1]."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, index: int):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        self.th = threading.Thread(target=self._read, daemon=True)
        self.th.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self, t0, t1):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        inside = [s for t, s in self.samples if t0 <= t <= t1 + 0.2]
        if not inside:
            inside = [s for _, s in self.samples]
        sm, mx, reasons = [], [], set()
        for s in inside:
            try:
                sm.append(float(s[0]))
                mx.append(float(s[1]))
            except (ValueError, IndexError):
                continue
            for name, val in zip(self.NAMES, s[3:7]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ helpers

def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        j = json.load(open(p))
        return float(j["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def _code_only(text: str) -> str:
    """C++ source without comments, blank lines or trailing blanks: what the
    compiler sees (these files hold no comment markers inside string literals)."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def decode_source_hash() -> str:
    """Identity of the decode kernel's code, so that an ncu summary taken on it
    stays attached to it across comment edits and to nothing else."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_gqa_09_gb300", "csrc")
    for f in ("decode.cu", "pkv_device.cuh", "pkv_kernels.h", "plan_map.cuh"):
        h.update(_code_only(open(os.path.join(csrc, f)).read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(cfg_id: int):
    """DRAM bytes per decode launch from the committed ncu summary, if it was
    taken on the current decode kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", f"decode_config{cfg_id}_traffic.md")
    try:
        txt = open(p).read()
    except OSError:
        return None
    m_hash = re.search(r"kernel_source_sha:\s*([0-9a-f]+)", txt)
    m_tr = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", txt)
    if not (m_hash and m_tr) or m_hash.group(1) != decode_source_hash():
        return None
    return int(m_tr.group(1))


def cpu_baseline_run(tr, q, k, v, seconds: float, sample_of: str = "the workload"):
    """The oracle, as it stands, on this host's cores: repeated whole decode
    steps of the workload (or, for large workloads, a row-prefix sample) for
    about `seconds` on all cores, then a quarter of that on one thread; returns
    (GB/s of K+V processed on all cores, cores, description, one-thread GB/s)."""
    import oracle
    cores = oracle.max_threads()
    lens = tr.seq_lens
    # sample: the whole batch when one step fits in the budget, else one row prefix
    t = time.perf_counter()
    oracle.attention(q[:1], k, v, tr.block_table[:1], np.minimum(lens[:1], 2048), tr.scale)
    probe = time.perf_counter() - t
    per_tok = probe / min(int(lens[0]), 2048)
    total_tok = int(lens.sum())
    if per_tok * total_tok <= seconds / 2:
        sample_lens, sample_q, sample_bt = lens, q, tr.block_table
        desc = f"whole decode steps of {sample_of}"
    else:
        n = max(16, min(int(lens[0]), int(seconds / 4 / per_tok)))
        sample_lens = np.array([n], np.int32)
        sample_q, sample_bt = q[:1], tr.block_table[:1]
        desc = f"row 0, first {n} tokens, all {tr.Hq} query heads, repeated"
    bytes_per = int(sample_lens.astype(np.int64).sum()) * tr.Hkv * tr.d * 4

    def timed(budget, nthreads):
        reps, t0 = 0, time.perf_counter()
        while True:
            oracle.attention(sample_q, k, v, sample_bt, sample_lens, tr.scale, nthreads=nthreads)
            reps += 1
            el = time.perf_counter() - t0
            if el >= budget:
                return bytes_per * reps / el / 1e9, reps, el

    gbs, reps, el = timed(seconds, 0)
    one, reps1, el1 = timed(seconds / 4, 1)
    return gbs, cores, f"{desc}; {reps} reps in {el:.1f} s ({reps1} in {el1:.1f} s on one thread)", one


# ------------------------------------------------------------------ reference arm

def run_reference(args, rank, ws, pg):
    import oracle
    import pkv_traces as T
    if rank != 0:
        return
    tr = T.make_trace(args.config, len_scale=args.len_scale)
    steps = args.steps if args.steps is not None else default_steps(args.config)
    warm = args.warmup if args.warmup is not None else 3
    # the sample per step: row 0 prefix, sized so that all steps fit in ~60 s
    if tr.num_pages * tr.page_size * tr.Hkv * tr.d <= (1 << 28):
        q = T.gen_q(tr)
        k, v = T.gen_kv(tr)
    else:
        tr, q, k, v = _row0_sample(tr)
    budget = 60.0 / max(1, steps + warm)
    t = time.perf_counter()
    oracle.attention(q[:1], k, v, tr.block_table[:1], np.minimum(tr.seq_lens[:1], 256), tr.scale)
    per_tok = (time.perf_counter() - t) / min(256, int(tr.seq_lens[0]))
    n = int(max(16, min(int(tr.seq_lens[0]), budget / max(per_tok, 1e-9))))
    sl = np.array([n], np.int32)
    for _ in range(warm):
        oracle.attention(q[:1], k, v, tr.block_table[:1], sl, tr.scale)
    t0 = time.perf_counter()
    for _ in range(steps):
        oracle.attention(q[:1], k, v, tr.block_table[:1], sl, tr.scale)
    el = time.perf_counter() - t0
    gbs = n * tr.Hkv * tr.d * 4 * steps / el / 1e9
    desc = f"per step: row 0, first {n} of {int(tr.seq_lens[0])} tokens, all {tr.Hq} query heads"
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": UNIT, "n_gpus": ws,
        "steps": steps, "warmup": warm, "ms_per_step": el / steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": workload_name(args.config, args.len_scale),
                                       "seed": tr.seed},
        "cpu_baseline": {"value": gbs, "unit": UNIT, "cores": oracle.max_threads(),
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": gbs, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def _row0_sample(tr):
    """A one-row trace shaped like row 0 of `tr` with its own host K/V, for
    workloads whose pool is too large to draw on the host."""
    import pkv_traces as T
    sub = T.custom_trace([int(tr.seq_lens[0])], tr.Hq, tr.Hkv, tr.d, tr.page_size,
                         tr.split_tokens, seed=tr.seed, tag=tr.cfg_id)
    k, v = T.gen_kv(sub)
    return sub, T.gen_q(sub), k, v


# ------------------------------------------------------------------ our arm

def run_pkv(args, rank, local, ws, pg):
    import torch

    import pkv_traces as T
    from paged_kv_gqa_09_gb300 import _lib, api
    from paged_kv_gqa_09_gb300 import build as build_mod

    build_mod.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    # everything runs on one non-default stream (graph capture needs one)
    stream = torch.cuda.Stream(dev)
    torch.cuda.set_stream(stream)
    L = _lib.load()
    cfg_id = args.config
    tr = T.make_trace(cfg_id, len_scale=args.len_scale)
    steps = args.steps if args.steps is not None else default_steps(cfg_id)
    warm = max(3, args.warmup if args.warmup is not None else 5)
    appends = tr.steps > 1
    if appends:  # the block table holds room for tr.steps appended tokens per row
        steps = min(steps, tr.steps - 1)
    big = tr.num_pages * tr.page_size * tr.Hkv * tr.d * 2 > (1 << 30)

    # ---- inputs (host copies kept for the oracle baseline)
    q_h = T.gen_q(tr)
    if big:
        k0, v0 = T.gen_kv_torch(tr, "cuda")
        k_h = v_h = None
    else:
        k_h, v_h = T.gen_kv(tr)
        k0 = torch.from_numpy(k_h).to(dev)
        v0 = torch.from_numpy(v_h).to(dev)
    pool_bytes = 2 * k0.numel() * 2
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    R = max(1, math.ceil(3 * l2 / pool_bytes) + 1) if pool_bytes < 3 * l2 else 1
    pools = [(k0, v0)] + [(k0.clone(), v0.clone()) for _ in range(R - 1)]
    q = torch.from_numpy(q_h).to(dev)
    bt = torch.from_numpy(tr.block_table).to(dev)
    sl = torch.from_numpy(tr.seq_lens).to(dev)
    sl_init = sl.clone()
    shape = api.make_shape(q, k0, bt)

    # ---- path: the one the workload names, else the policy's route (or --path)
    pol = api.pkv_policy_default()
    path, C = api.pkv_policy(tr.B, tr.n_max + (tr.steps if tr.steps > 1 else 0), pol)
    named = {"bucketed": 0, "workqueue": 1, "single": 2}
    if tr.path_hint in named:
        path = named[tr.path_hint]
    forced = named.get(args.path)
    if forced is not None:
        path = forced
    if path != 2 and tr.path_hint != "policy":
        C = tr.split_tokens  # the workload fixes its split size (S splits)
    if path != 2 and args.split_tokens:
        C = args.split_tokens
    n_max_run = tr.n_max + (tr.steps if appends else 0)
    bucket = n_max_run if path == 0 else 0
    fused = args.merge == "fused" and path != 2
    # with appends the append launch then allocates pages only and the decode plans
    self_plan = (args.plan == "in-decode" and path == 1 and not fused
                 and tr.B <= api.PKV_SELF_PLAN_MAX_B)
    plan_mode = api.PKV_PLAN_IN_DECODE if self_plan else api.PKV_PLAN_SEPARATE
    cfg = api.make_cfg(path, C, bucket, 0, api.PKV_MERGE_FUSED if fused else api.PKV_MERGE_SEPARATE,
                       plan_mode)
    wsb = torch.zeros(api.pkv_plan_workspace_size(shape, cfg), dtype=torch.uint8, device=dev)
    npart = api.pkv_partials_size(shape, cfg)
    part = torch.empty(max(npart // 4, 4), dtype=torch.float32, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=dev)
    kn = torch.from_numpy(T.gen_append_tokens(tr, 0)[0]).to(dev)
    vn = torch.from_numpy(T.gen_append_tokens(tr, 0)[1]).to(dev)
    if appends:
        # on the workqueue, pages are allocated on the device as rows grow: each
        # row starts with the pages its tokens fill and the rest of the shuffled
        # pool is the free list; other paths use the pre-assigned table
        bt_alloc, free_np = T.allocation_split(tr) if path == 1 else (tr.block_table, np.zeros(1, np.int32))
        bt_init = torch.from_numpy(np.ascontiguousarray(bt_alloc)).to(dev)
        bt.copy_(bt_init)
        free_pages = torch.from_numpy(free_np).to(dev)
        free_count = torch.tensor([free_np.size], dtype=torch.int32, device=dev)
        free_init = free_count.clone()
    sp = stream.cuda_stream
    P = lambda t: t.data_ptr() if t is not None else None
    sref, cref = _ctypes_refs(shape, cfg)

    def step(r):
        kk, vv = pools[r]
        if appends and path == 1:
            # append + page allocation + plan in one launch, then decode and merge
            rc = L.pkv_append_plan(sref, cref, P(wsb), P(kn), P(vn), P(bt), P(sl), P(free_pages),
                                   P(free_count), P(kk), P(vv), sp)
            _lib.check(rc, "pkv_append_plan")
            if fused:
                _lib.check(L.pkv_decode_merge(sref, cref, P(wsb), P(q), P(kk), P(vv), P(bt), P(sl),
                                              P(part), P(o), P(lse), sp), "pkv_decode_merge")
                return
            _lib.check(L.pkv_decode(sref, cref, P(wsb), P(q), P(kk), P(vv), P(bt), P(sl), P(part), sp),
                       "pkv_decode")
            _lib.check(L.pkv_merge(sref, cref, P(wsb), P(sl), P(part), P(o), P(lse), sp), "pkv_merge")
            return
        if appends:
            rc = L.pkv_append(sref, P(wsb), P(kn), P(vn), P(bt), P(sl), P(kk), P(vv), sp)
            _lib.check(rc, "pkv_append")
        rc = L.pkv_decode_step(sref, cref, P(wsb), P(q), P(kk), P(vv), P(bt), P(sl),
                               P(part) if npart else None, P(o), P(lse), sp)
        _lib.check(rc, "pkv_decode_step")

    def reset_lengths():
        sl.copy_(sl_init)
        if appends:
            bt.copy_(bt_init)
            free_count.copy_(free_init)

    # ---- warm-up (eager), then capture the step graphs
    for w in range(warm):
        step(w % R)
    torch.cuda.synchronize()
    st, msg = api.pkv_get_error(wsb)
    if st != 0:
        raise RuntimeError(f"device error during warm-up: {msg}")
    api.pkv_reset_counters()
    step(0)
    torch.cuda.synchronize()
    c = api.pkv_get_counters()
    launches_per_step = sum(c.values())
    # graphs: one of G consecutive steps (pools 0..R-1 in turn, G a multiple of
    # R and at least 8), so that each step's kernels chain into the next step's
    # by programmatic dependent launch (which stops at a graph boundary), and
    # single steps for a remainder of K mod G
    G = R * -(-8 // R)
    graphs = None
    if not args.no_graph:
        try:
            loop_graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(loop_graph, stream=stream):
                for r in range(G):
                    step(r % R)
            singles = []
            for r in range(R):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    step(r)
                singles.append(g)
            loop_graph.replay()
            torch.cuda.synchronize()
            graphs = (loop_graph, singles)
        except Exception as e:  # capture unsupported: eager launches
            print(f"# graph capture failed ({e}); timing eager launches", file=sys.stderr)
            graphs = None
    if appends:
        reset_lengths()
        torch.cuda.synchronize()

    kv_step = tr.kv_bytes()
    if appends:  # every step appends first: step s reads N_i + s + 1 tokens per row
        kv_step = int((int(tr.seq_lens.astype(np.int64).sum()) + tr.B * (1 + (steps - 1) / 2))
                      * tr.Hkv * tr.d * 4)

    # ---- timed region: K steps back to back
    sampler = ClockSampler(_gpu_id(torch, dev)) if rank == 0 else None
    barrier(pg)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    t_wall0 = time.time()
    e0.record(stream)
    if graphs:
        for _ in range(steps // G):
            graphs[0].replay()
        for r in range(steps % G):
            graphs[1][r % R].replay()
    else:
        for s in range(steps):
            step(s % R)
    e1.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    barrier(pg)
    ms = e0.elapsed_time(e1) / steps
    ms_max = reduce_max(pg, ms)
    clocks = sampler.stop(t_wall0, t_wall1) if sampler else None
    st, msg = api.pkv_get_error(wsb)
    if st != 0:
        raise RuntimeError(f"device error in the timed region: {msg}")

    # ---- the decode kernel (roofline)
    if appends:
        reset_lengths()
    if path != 2:
        L.pkv_plan(sref, cref, P(sl), P(wsb), sp)

    def kernel(s):
        kk, vv = pools[s % R]
        if path == 2:
            rc = L.pkv_single_pass(sref, P(wsb), P(q), P(kk), P(vv), P(bt), P(sl), P(o), P(lse), sp)
        else:
            rc = (L.pkv_decode_merge(sref, cref, P(wsb), P(q), P(kk), P(vv), P(bt), P(sl), P(part),
                                     P(o), P(lse), sp) if fused else
                  L.pkv_decode(sref, cref, P(wsb), P(q), P(kk), P(vv), P(bt), P(sl), P(part), sp))
        _lib.check(rc, "decode")

    # (1) the basis of the roofline: the kernel as it runs inside the step --
    # G launches back to back in one CUDA graph (pools in turn), each chained
    # to the one before by programmatic dependent launch, replayed; events only
    # around the replays, so the per-launch time is the kernel's share of a
    # step loop with the other launches of the step taken out
    kern_launches = G * max(1, min(steps, 2000) // G)
    kgraph = None
    if graphs:
        try:
            kgraph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(kgraph, stream=stream):
                for s in range(G):
                    kernel(s)
            kgraph.replay()
            torch.cuda.synchronize()
        except Exception as e:
            print(f"# decode graph capture failed ({e}); chaining eager launches", file=sys.stderr)
            kgraph = None
    c0 = torch.cuda.Event(enable_timing=True)
    c1 = torch.cuda.Event(enable_timing=True)
    c0.record(stream)
    if kgraph is not None:
        for _ in range(kern_launches // G):
            kgraph.replay()
    else:
        for s in range(kern_launches):
            kernel(s)
    c1.record(stream)
    torch.cuda.synchronize()
    chained_ms = c0.elapsed_time(c1) / kern_launches
    # (2) each launch alone, with events around it: adds the launch, ramp-up
    # and drain that a chain hides (reported apart, not the roofline basis)
    iso_launches = min(steps, 2000)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(iso_launches)]
    for s in range(iso_launches):
        evs[s][0].record(stream)
        kernel(s)
        evs[s][1].record(stream)
    torch.cuda.synchronize()
    launch_ms = sorted(a.elapsed_time(b) for a, b in evs)
    iso_ms = statistics.mean(launch_ms)
    pct = lambda f: launch_ms[min(len(launch_ms) - 1, int(f * len(launch_ms)))] * 1e3
    st, msg = api.pkv_get_error(wsb)
    if st != 0:
        raise RuntimeError(f"device error while timing the decode kernel: {msg}")
    kv_launch = tr.kv_bytes()
    peak, peak_src = peaks()
    achieved = kv_launch / (chained_ms * 1e-3) / 1e9
    achieved_iso = kv_launch / (iso_ms * 1e-3) / 1e9

    # ---- end to end through the C ABI with pinned host buffers
    e2e = None
    if not args.no_e2e:
        if appends:
            reset_lengths()
        e2e = run_e2e_cabi(L, torch, tr, q_h, pools, dev, sref, cref, cfg, wsb, part if npart else None,
                           steps, appends, path)
        # the Python serving loop (one captured graph per step), beside it
        if appends:
            reset_lengths()
        e2e["graph_loop"] = run_e2e(api, torch, tr, q_h, pools, dev, path, C, steps, appends, kn, vn,
                                    wsb, cfg.merge, cfg.plan)

    traffic = profiled_traffic(cfg_id) if args.len_scale == 1.0 else None
    total = whole_job_gbs(kv_step, ms_max, ws)
    cpu = None
    if rank == 0 and not args.no_cpu:
        if k_h is None:
            tr_s, qb, k_s, v_s = _row0_sample(tr)
            of = f"row 0 of the workload ({int(tr.seq_lens[0])} tokens, all {tr.Hq} query heads)"
        else:
            tr_s, qb, k_s, v_s = tr, q_h, k_h, v_h
            of = "the workload"
        val, cores, desc, one = cpu_baseline_run(tr_s, qb, k_s, v_s, args.cpu_seconds, of)
        cpu = {"value": val, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc,
               "single_thread_value": one}
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": total, "unit": UNIT, "n_gpus": ws, "steps": steps,
        "warmup": warm, "ms_per_step": ms_max, "us_per_step": ms_max * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic",
        "config": {
            "workload": workload_name(cfg_id, args.len_scale), "path": ["bucketed-split", "workqueue", "single-pass"][path],
            "merge": ("fused" if fused else "separate") if path != 2 else None,
            "plan": ("in-decode" if self_plan else "append+plan kernel" if appends else "plan kernel")
                    if path == 1 else None,
            "launches_per_step": launches_per_step,
            "split_tokens": C, "kv_bytes_per_step": kv_step, "seed": tr.seed,
            "l2": (f"{R} KV pools rotated ({R * pool_bytes / 2**20:.0f} MiB > L2 {l2 / 2**20:.0f} MiB)"
                   if R > 1 else f"inputs ({pool_bytes / 2**30:.1f} GiB) larger than L2"),
            "graph": bool(graphs), "graph_steps": G if graphs else 0, "parallelism": f"replicas x{ws}",
        },
        "hbm_frac": total / ws / peak,
        "roofline": {"bound": "hbm",
                     "kernel": ("decode_merge" if fused else "decode") if path != 2 else "single_pass",
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_source": peak_src, "traffic": traffic,
                     "bytes_per_launch": kv_launch, "us_per_launch": chained_ms * 1e3,
                     "timing": f"CUDA events around replays of a CUDA graph of {G} back-to-back "
                               f"launches chained by programmatic dependent launch (as inside the "
                               f"step); {kern_launches} launches",
                     "share_of_step": chained_ms / ms,
                     "frac_of_nominal_hbm": achieved / NOMINAL_HBM_GBS,
                     "isolated": {"us_per_launch": iso_ms * 1e3,
                                  "us_per_launch_p10_p50_p90": [pct(0.1), pct(0.5), pct(0.9)],
                                  "achieved": achieved_iso, "frac": achieved_iso / peak,
                                  "how": f"{iso_launches} launches, each alone between two "
                                         "events (launch, ramp-up and drain included)"}},
        "gpu_launches": launches_per_step * steps,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)


def _gpu_id(torch, dev):
    """nvidia-smi -i selector for this CUDA device (its UUID, else its index)."""
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return str(dev.index)


def _ctypes_refs(shape, cfg):
    import ctypes
    return ctypes.byref(shape), ctypes.byref(cfg)


def run_e2e_cabi(L, torch, tr, q_h, pools, dev, sref, cref, cfg, wsb, part, steps, appends, path):
    """The C ABI's host-buffer step, once per step on the wall clock: every call
    takes the step's inputs from pinned host memory (q and the block table and
    lengths; or, when the workload appends, q and the new K/V token -- the table
    and lengths being device state the step advances), which its kernels read in
    place, runs the step, has its last kernel write o and lse into pinned host
    memory and synchronizes the stream."""
    import pkv_traces as T
    from paged_kv_gqa_09_gb300 import _lib
    R = len(pools)
    sp = torch.cuda.current_stream(dev).cuda_stream
    P = lambda t: t.data_ptr() if t is not None else None
    h_q = torch.from_numpy(q_h).pin_memory()
    d_q = torch.empty(h_q.shape, dtype=torch.float16, device=dev)
    h_o = torch.empty(h_q.shape, dtype=torch.float16).pin_memory()
    d_o = torch.empty_like(d_q)
    h_lse = torch.empty(h_q.shape[:2], dtype=torch.float32).pin_memory()
    d_lse = torch.empty(h_q.shape[:2], dtype=torch.float32, device=dev)
    qb, ob, lb = h_q.numel() * 2, h_o.numel() * 2, h_lse.numel() * 4
    if appends:
        kn_h, vn_h = T.gen_append_tokens(tr, 0)
        h_kn = torch.from_numpy(kn_h).pin_memory()
        h_vn = torch.from_numpy(vn_h).pin_memory()
        d_kn, d_vn = torch.empty_like(h_kn, device=dev), torch.empty_like(h_vn, device=dev)
        # as in the device loop: on the workqueue the rows' pages come from a
        # device free list as they grow
        bt0, free_np = T.allocation_split(tr) if path == 1 else (tr.block_table, None)
        d_bt = torch.from_numpy(np.ascontiguousarray(bt0)).to(dev)
        d_sl = torch.from_numpy(tr.seq_lens).to(dev)
        free = torch.from_numpy(free_np).to(dev) if free_np is not None else None
        cnt = torch.tensor([free_np.size], dtype=torch.int32, device=dev) if free is not None else None
        steps = min(steps, tr.steps - 4)  # the block table holds room for tr.steps tokens per row
        h2d = qb + 2 * h_kn.numel() * 2
    else:
        h_bt = torch.from_numpy(np.ascontiguousarray(tr.block_table)).pin_memory()
        h_sl = torch.from_numpy(tr.seq_lens).pin_memory()
        d_bt = torch.empty(h_bt.shape, dtype=torch.int32, device=dev)
        d_sl = torch.empty(h_sl.shape, dtype=torch.int32, device=dev)
        steps = min(steps, 4000)
        h2d = qb + h_bt.numel() * 4 + h_sl.numel() * 4
    per_tok = tr.Hkv * tr.d * 4
    sl0 = int(tr.seq_lens.astype(np.int64).sum())
    appended = [0]

    def one(s):
        kk, vv = pools[s % R]
        if appends:
            rc = L.pkv_append_decode_step_host(
                sref, cref, P(wsb), P(part), P(h_q), P(d_q), P(h_kn), P(h_vn), P(d_kn), P(d_vn),
                P(d_bt), P(d_sl), P(free), P(cnt), P(kk), P(vv), P(d_o), P(h_o), P(d_lse), P(h_lse),
                sp)
            _lib.check(rc, "pkv_append_decode_step_host")
            appended[0] += 1
        else:
            rc = L.pkv_decode_step_host(sref, cref, P(wsb), P(part), P(h_q), P(d_q), P(h_bt),
                                        P(d_bt), P(h_sl), P(d_sl), P(kk), P(vv), P(d_o), P(h_o),
                                        P(d_lse), P(h_lse), sp)
            _lib.check(rc, "pkv_decode_step_host")
        return (sl0 + tr.B * appended[0]) * per_tok

    for s in range(3):
        one(s)
    kv = 0
    t0 = time.perf_counter()
    for s in range(steps):
        kv += one(s)
    el = time.perf_counter() - t0
    from paged_kv_gqa_09_gb300 import api
    st, msg = api.pkv_get_error(wsb)
    if st != 0:
        raise RuntimeError(f"device error in the end-to-end steps: {msg}")
    name = "pkv_append_decode_step_host" if appends else "pkv_decode_step_host"
    return {"value": kv / el / 1e9, "unit": UNIT, "us_per_step": el / steps * 1e6, "steps": steps,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": ob + lb,
            "timing": f"synchronized wall clock per step: one {name} call (C ABI) per step -- "
                      + ("q and the new token" if appends else "q, block table and lengths")
                      + " read in place from pinned memory by the step's kernels, o/lse written "
                        "in place into pinned memory by the last kernel, stream synchronized"}


def run_e2e(api, torch, tr, q_h, pools, dev, path, C, steps, appends, kn, vn, wsb, merge, plan):
    """Public-API steps with host buffers (HostDecodeLoop, one captured graph per
    step): the step's kernels read q, the block table and the lengths (or, when
    the workload appends, q and the new K/V token, the table and lengths being
    device state the step advances) from pinned host memory and write o and lse
    there; every step is synchronized; timed on the wall clock."""
    import pkv_traces as T
    R = len(pools)
    n_max = int(tr.seq_lens.max()) + (tr.steps if appends else 0)
    q_pin = torch.from_numpy(q_h).pin_memory()
    sl0 = tr.seq_lens.astype(np.int64)
    qb = q_pin.numel() * 2
    d2h = qb + q_pin.shape[0] * q_pin.shape[1] * 4
    steps = min(steps, 4000 if not appends else tr.steps - 4)
    stream = torch.cuda.current_stream(dev)
    per_tok = tr.Hkv * tr.d * 4
    loops = []
    for kk, vv in pools:
        if appends:
            # as in the device loop: on the workqueue the rows' pages are taken
            # from a device free list as they grow
            bt0, free_np = T.allocation_split(tr) if path == 1 else (tr.block_table, None)
            fp = torch.from_numpy(free_np).to(dev) if free_np is not None else None
            fc = torch.tensor([free_np.size], dtype=torch.int32, device=dev) if fp is not None else None
            lp = api.HostDecodeLoop(kk, vv, tr.B, tr.Hq, tr.bt_stride, n_max, path=path,
                                    split_tokens=C, merge=merge, append=True, free_pages=fp,
                                    free_count=fc, plan=plan)
            lp.set_state(torch.from_numpy(np.ascontiguousarray(bt0)), torch.from_numpy(tr.seq_lens))
            lp.h_kn.copy_(kn.cpu())
            lp.h_vn.copy_(vn.cpu())
        else:
            lp = api.HostDecodeLoop(kk, vv, tr.B, tr.Hq, tr.bt_stride, n_max, path=path,
                                    split_tokens=C, merge=merge, plan=plan)
            lp.h_bt.copy_(torch.from_numpy(tr.block_table))
            lp.h_sl.copy_(torch.from_numpy(tr.seq_lens))
        lp.h_q.copy_(q_pin)
        lp.capture(stream)  # with appends, this runs the first step (one token)
        loops.append(lp)
    h2d = qb + (2 * kn.numel() * 2 if appends else tr.block_table.size * 4 + tr.B * 4)
    # as for the C-ABI leg, the step's inputs sit in the pinned buffers already
    # (writing them there is the caller's work); each step moves them to the
    # device and its outputs back
    appended = [1 if appends else 0]  # tokens each row has gained so far
    kv_total = [0]

    def one(s):
        lp = loops[s % R]
        lp.step_graph()
        if appends:
            appended[0] += 1
        kv_total[0] += (int(sl0.sum()) + tr.B * appended[0]) * per_tok

    for s in range(3):
        one(s)
    kv_total[0] = 0
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for s in range(steps):
        one(s)
    el = time.perf_counter() - t0
    return {"value": kv_total[0] / el / 1e9, "unit": UNIT, "us_per_step": el / steps * 1e6,
            "steps": steps, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "timing": "synchronized wall clock per step (HostDecodeLoop graph: the step's kernels "
                      + ("append the staged token, then " if appends else "")
                      + "read their host inputs from pinned memory in place and write o/lse there)"}


def main():
    args = parse()
    rank, local, ws, pg = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, rank, ws, pg)
    else:
        run_pkv(args, rank, local, ws, pg)
    if pg is not None:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
