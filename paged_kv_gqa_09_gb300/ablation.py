"""Scheduling ablation on the current GPU: the compact workqueue against the
exact-length-bucket scheme it replaces and the length-bucketed rectangular
grid ("PersistentKV: Page-Aware Decode Scheduling for Long-Context LLM Serving
on Commodity GPUs", technical summary, Results, "Scheduling overhead":
launches per step 16.00 -> 2.00 on B=8 bimodal traces, merge-state traffic
about -37%).

For each B=8 trace (bimodal, uniform, Zipf-like; held-out seed) and route it
reports: attention launches per step (library counters; the workqueue's plan
launch apart), merge-state bytes (fp32 states written by the split kernel plus
read by the merge, from pkv_step_model), device time per step (CUDA events
over back-to-back steps) and synchronized wall-clock per step (host launches
included, as the pages time).  A fourth time replays CUDA graphs of 20
consecutive steps: the same launches with the host's issue rate out of the
picture (the exact-length scheme's 16 launches per step are otherwise limited
by the host).

Usage (GPU):  python -m paged_kv_gqa_09_gb300.ablation [--reps 200]
"""
from __future__ import annotations

import argparse
import statistics
import sys
import time

import numpy as np

import pkv_traces as T


def traces():
    rng = np.random.default_rng([T.HELDOUT_SEED, 55])
    uni = rng.integers(4096, 32768, size=8, endpoint=True).astype(np.int32)
    out = [("bimodal", T.make_trace(3)), ("zipf", T.make_trace(4, B=8))]
    tr_u = T.custom_trace(uni.tolist(), 32, 8, 128, 16, 1024, seed=T.HELDOUT_SEED, tag=56)
    out.insert(1, ("uniform U[4096,32768]", tr_u))
    return out


def main(argv=None):
    import torch

    from paged_kv_gqa_09_gb300 import _lib, api

    ap = argparse.ArgumentParser()
    ap.add_argument("--reps", type=int, default=200)
    a = ap.parse_args(argv)
    rows = []
    for name, tr in traces():
        q = torch.from_numpy(T.gen_q(tr)).cuda()
        k, v = T.gen_kv_torch(tr, "cuda")
        bt = torch.from_numpy(tr.block_table).cuda()
        sl = torch.from_numpy(tr.seq_lens).cuda()
        shape = api.make_shape(q, k, bt)
        o = torch.empty_like(q)
        lse = torch.empty(q.shape[:2], dtype=torch.float32, device="cuda")
        C = tr.split_tokens
        wq_cfg = api.make_cfg(_lib.PKV_PATH_WORKQUEUE, C)
        bk_cfg = api.make_cfg(_lib.PKV_PATH_BUCKETED_SPLIT, C, tr.n_max)
        bufs = {}
        for key, cfg in (("wq", wq_cfg), ("bk", bk_cfg)):
            ws = torch.zeros(api.pkv_plan_workspace_size(shape, cfg), dtype=torch.uint8, device="cuda")
            part = torch.empty(api.pkv_partials_size(shape, cfg) // 4, dtype=torch.float32, device="cuda")
            bufs[key] = (cfg, ws, part)
        ex_ws = torch.zeros(64, dtype=torch.uint8, device="cuda")
        ex_part = torch.empty(bufs["bk"][2].numel(), dtype=torch.float32, device="cuda")
        cache = {}

        def run(route):
            if route == "exact-length buckets":
                api.exact_length_buckets_step(q, k, v, bt, sl, tr.seq_lens, C, o, lse, ws=ex_ws,
                                              partials=ex_part, rows_cache=cache)
            else:
                cfg, ws, part = bufs["wq" if route == "workqueue" else "bk"]
                api.pkv_decode_step(shape, cfg, ws, q, k, v, bt, sl, part, o, lse)

        model_path = {"workqueue": 1, "length-bucketed grid": 0, "exact-length buckets": 3}
        for route in ("workqueue", "length-bucketed grid", "exact-length buckets"):
            for _ in range(5):
                run(route)
            torch.cuda.synchronize()
            api.pkv_reset_counters()
            run(route)
            torch.cuda.synchronize()
            cnt = api.pkv_get_counters()
            attn = cnt["decode_launches"] + cnt["merge_launches"] + cnt["single_pass_launches"]
            model = api.pkv_step_model(model_path[route], shape, C, tr.n_max, tr.seq_lens)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(a.reps):
                run(route)
            e1.record()
            torch.cuda.synchronize()
            dev_us = e0.elapsed_time(e1) / a.reps * 1e3
            # the same steps replayed from a graph (buffers and row lists are
            # warm, so the captured calls allocate nothing)
            per_graph = 20
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                run(route)
            torch.cuda.current_stream().wait_stream(side)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                for _ in range(per_graph):
                    run(route)
            graph.replay()
            torch.cuda.synchronize()
            replays = max(1, a.reps // per_graph)
            e0.record()
            for _ in range(replays):
                graph.replay()
            e1.record()
            torch.cuda.synchronize()
            graph_us = e0.elapsed_time(e1) / (replays * per_graph) * 1e3
            wall = []
            for _ in range(min(a.reps, 100)):
                torch.cuda.synchronize()
                t0 = time.perf_counter()
                run(route)
                torch.cuda.synchronize()
                wall.append((time.perf_counter() - t0) * 1e6)
            rows.append((name, route, attn, cnt["plan_launches"], model["merge_state_bytes"],
                         dev_us, graph_us, statistics.median(wall), tr.kv_bytes()))
        for key in ("wq", "bk"):
            st, msg = api.pkv_get_error(bufs[key][1])
            if st:
                raise RuntimeError(msg)
        st, msg = api.pkv_get_error(ex_ws)
        if st:
            raise RuntimeError(msg)
    print("| trace (B=8) | route | attention launches / step | plan launches | merge-state MB | "
          "device us/step | graph us/step | sync wall us/step | KV GB/s (graph) |")
    print("|---|---|---|---|---|---|---|---|---|")
    for name, route, attn, plan, msb, dev_us, graph_us, wall_us, kvb in rows:
        print(f"| {name} | {route} | {attn} | {plan} | {msb / 1e6:.2f} | {dev_us:.1f} | "
              f"{graph_us:.1f} | {wall_us:.1f} | {kvb / graph_us / 1e3:.0f} |")
    return 0


if __name__ == "__main__":
    sys.exit(main())
