"""Multi-rank host logic of bench.py on CPU (gloo, world size 2, 127.0.0.1):
the barrier, the max over ranks of the per-step time and the whole-job
throughput.  The path itself runs replicas with no collective on the data
path, so this is all the exchange there is."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    r, local, ws, pg = bench.dist_setup(None)
    assert (r, local, ws) == (rank, rank, world) and pg is not None
    bench.barrier(pg)
    ms = 1.0 + rank  # rank 1 is the slow one
    ms_max = bench.reduce_max(pg, ms)
    out.put((rank, ms_max, bench.whole_job_gbs(1000, ms_max, ws)))
    pg.destroy_process_group()


def test_two_rank_barrier_and_max_over_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    res = sorted(q.get(timeout=5) for _ in range(2))
    assert [ms for _, ms, _ in res] == [2.0, 2.0]
    # 1000 bytes per rank, 2 ranks, 2 ms per step -> 1e-3 GB/s
    assert all(abs(g - 2000 / 2e-3 / 1e9) < 1e-12 for _, _, g in res)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.reduce_max(None, 3.5) == 3.5
    assert bench.whole_job_gbs(134217728, 0.0201, 1) == pytest.approx(6677.5, rel=1e-3)


def test_cpu_baseline_times_all_cores_and_one_thread():
    """The cpu_baseline leg: the oracle as it stands on the small case, timed
    on all cores and on one thread, in GB/s of K+V."""
    import bench
    import pkv_traces as T
    tr = T.make_trace(1)
    k, v = T.gen_kv(tr)
    gbs, cores, desc, one = bench.cpu_baseline_run(tr, T.gen_q(tr), k, v, 0.2)
    assert gbs > 0 and one > 0 and cores >= 1
    assert "whole decode steps" in desc and "one thread" in desc


# ------------------------------------------------------------------ the reference arm's line

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _reference_lines(nproc):
    import subprocess
    import sys
    args = ["bench.py", "--impl", "reference", "--gpus", str(nproc), "--steps", "2", "--warmup", "1",
            "--config", "1"]
    if nproc > 1:
        cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={nproc}",
               "--master-addr", "127.0.0.1", "--master-port", str(_free_port())] + args
    else:
        cmd = [sys.executable] + args
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    return [line for line in r.stdout.splitlines() if line.startswith("{")]


@pytest.mark.parametrize("nproc", [1, 2])
def test_reference_arm_prints_one_contract_line(nproc):
    """The oracle timed on the host cores: one JSON line from rank 0 only, with
    the base contract's keys, a cpu_baseline describing the run, and an e2e
    that moves no bytes."""
    import json
    lines = _reference_lines(nproc)
    assert len(lines) == 1
    d = json.loads(lines[0])
    import bench
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "GB/s"
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["higher_is_better"] is True
    assert (d["n_gpus"], d["steps"], d["warmup"]) == (nproc, 2, 1)
    assert d["vs_baseline"] is None and d["data"] == "synthetic" and d["dtype"] == "f64"
    assert d["scaling"] == "weak" and "workload" in d["config"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
