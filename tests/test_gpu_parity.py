"""GPU parity: libpkv (through its C ABI) against the float64 oracle.

Every case draws seeded inputs once on the host, runs the oracle on the CPU
and the CUDA path on the GPU, and compares element by element: the task list
and launch counts bit-exactly, neutral states bit-exactly, outputs within the
stated tolerance |x - y| <= 3e-3 + 1e-2 |y|.
"""
import numpy as np
import pytest
import torch

import oracle
import pkv_traces as T
from plan_order import balance_order
from paged_kv_gqa_09_gb300 import _lib, api

from gpu_util import (check_error_free, close, close_lse, dev, oracle_out, read_plan, run_path,
                      shape_of, upload)

pytestmark = pytest.mark.gpu

BUCKETED, WORKQUEUE, SINGLE = (_lib.PKV_PATH_BUCKETED_SPLIT, _lib.PKV_PATH_WORKQUEUE,
                               _lib.PKV_PATH_SINGLE_PASS)


@pytest.fixture(scope="module", autouse=True)
def _lib_loaded():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_gqa_09_gb300 import build
    build.build()
    _lib.load()


def case(lens, Hq=8, Hkv=2, d=128, P=16, C=64, seed=3, **kw):
    tr = T.custom_trace(lens, Hq, Hkv, d, P, C, seed=seed, **kw)
    q = T.gen_q(tr)
    k, v = T.gen_kv(tr, poison_unused=True)
    return tr, q, k, v


# ------------------------------------------------------------------ plan

@pytest.mark.parametrize("lens,C", [
    ([1, 0, 1024, 1025, 17], 256),
    ([0, 0, 0], 64),
    ([5000, 3, 64, 64, 100000, 7, 0, 2048], 1024),
    (list(range(1, 300, 7)), 16),
    # more rows than one plan block: a totals pass, then chunk by chunk
    (np.random.default_rng(7).integers(0, 600, 2500).tolist(), 64),
    ([64] * 1024 + [65], 64),
])
def test_plan_matches_oracle_bit_exact(lens, C):
    Hq, Hkv = 32, 8
    P = 16
    tr = T.custom_trace(lens, Hq, Hkv, 128, P, C, extra_cols=2)
    shape = shape_of(tr)
    cfg = api.make_cfg(WORKQUEUE, C)
    ws = torch.zeros(api.pkv_plan_workspace_size(shape, cfg), dtype=torch.uint8, device="cuda")
    api.pkv_plan(shape, cfg, dev(tr.seq_lens), ws)
    torch.cuda.synchronize()
    count, off, tasks, h, ordered = read_plan(ws, tr.B, with_order=True)
    want, want_off = oracle.plan_compact(tr.seq_lens, Hq, Hkv, C)
    assert count == want.shape[0]
    assert np.array_equal(off, want_off)
    assert np.array_equal(tasks, want)
    assert h[0] == 0 and h[6] == 0
    check_error_free(ws)
    # the decode walks a balance-ordered copy of the same records
    # (plan_order.py: full-length splits first, then the shorter last splits
    # from the longest length class down)
    expect = want[balance_order(want, lens, C)] if count else want
    assert np.array_equal(ordered, expect)


@pytest.mark.parametrize("cfg_id", [3, 5])
def test_plan_matches_oracle_on_workloads(cfg_id):
    tr = T.make_trace(cfg_id)
    shape = shape_of(tr)
    cfg = api.make_cfg(WORKQUEUE, tr.split_tokens)
    ws = torch.zeros(api.pkv_plan_workspace_size(shape, cfg), dtype=torch.uint8, device="cuda")
    api.pkv_plan(shape, cfg, dev(tr.seq_lens), ws)
    torch.cuda.synchronize()
    count, off, tasks, _ = read_plan(ws, tr.B)
    want, want_off = oracle.plan_compact(tr.seq_lens, tr.Hq, tr.Hkv, tr.split_tokens)
    assert count == want.shape[0] and np.array_equal(tasks, want) and np.array_equal(off, want_off)


def test_plan_capacity_overflow_is_reported():
    """A plan that exceeds its capacity writes no task, reports PKV_ECAPACITY,
    and the merge writes NaN (outputs and partial states start at zero here, so
    a missing write would show)."""
    tr = T.custom_trace([300, 700], 8, 2, 128, 16, 64)
    shape = shape_of(tr)
    cfg = api.make_cfg(WORKQUEUE, 64, 0, max_tasks=5)
    d = upload(tr, T.gen_q(tr), *T.gen_kv(tr))
    ws = torch.zeros(api.pkv_plan_workspace_size(shape, cfg), dtype=torch.uint8, device="cuda")
    part = torch.zeros(api.pkv_partials_size(shape, cfg) // 4, dtype=torch.float32, device="cuda")
    o = torch.zeros((tr.B, tr.Hq, tr.d), dtype=torch.float16, device="cuda")
    lse = torch.zeros((tr.B, tr.Hq), dtype=torch.float32, device="cuda")
    api.pkv_decode_step(shape, cfg, ws, d["q"], d["k"], d["v"], d["bt"], d["sl"], part, o, lse)
    st, msg = api.pkv_get_error(ws)
    assert st == _lib.PKV_ECAPACITY, msg
    assert torch.isnan(o.float()).all() and torch.isnan(lse).all()
    assert read_plan(ws, tr.B)[0] == 0  # no task count


# ------------------------------------------------------------------ partials

def partial_views(part, tr, slots):
    d = tr.d
    acc = part[:slots * d].view(slots, d).cpu().numpy().astype(np.float64)
    m = part[slots * d:slots * d + slots].cpu().numpy().astype(np.float64)
    l = part[slots * d + slots:slots * (d + 2)].cpu().numpy().astype(np.float64)
    return m, l, acc


@pytest.mark.parametrize("rect", [False, True])
def test_partial_states_match_oracle(rect):
    tr, q, k, v = case([200, 1, 64, 130, 0], Hq=8, Hkv=2, C=64)
    d = upload(tr, q, k, v)
    shape = shape_of(tr)
    C = 64
    S_b = -(-tr.n_max // C)
    path = BUCKETED if rect else WORKQUEUE
    cfg = api.make_cfg(path, C, tr.n_max if rect else 0)
    ws = torch.zeros(api.pkv_plan_workspace_size(shape, cfg), dtype=torch.uint8, device="cuda")
    slots = api.pkv_partials_size(shape, cfg) // ((tr.d + 2) * 4)
    part = torch.full((slots * (tr.d + 2),), float("nan"), dtype=torch.float32, device="cuda")
    api.pkv_plan(shape, cfg, d["sl"], ws)
    api.pkv_decode(shape, cfg, ws, d["q"], d["k"], d["v"], d["bt"], d["sl"], part)
    torch.cuda.synchronize()
    check_error_free(ws)
    m, l, acc = partial_views(part, tr, slots)
    mo, lo, acco = oracle.partials(q, k, v, tr.block_table, tr.seq_lens, tr.scale, C,
                                   rect=rect, S_b=S_b)
    n = mo.shape[0]
    m, l, acc = m[:n], l[:n], acc[:n]
    neutral = lo == 0
    if rect:
        assert neutral.any()
    # neutral states are written bit-exactly: m = -inf, l = +0, acc = +0
    mb = part[slots * tr.d:slots * tr.d + n].cpu().numpy().view(np.uint32)
    lb = part[slots * tr.d + slots:slots * tr.d + slots + n].cpu().numpy().view(np.uint32)
    ab = part[:n * tr.d].view(n, tr.d).cpu().numpy().view(np.uint32)
    assert np.all(mb[neutral] == 0xFF800000)
    assert np.all(lb[neutral] == 0) and np.all(ab[neutral] == 0)
    live = ~neutral
    assert np.max(np.abs(m[live] - mo[live])) < 1e-4
    # l and acc are relative to m: compare the normalized split outputs and l
    assert np.max(np.abs(l[live] / lo[live] - 1)) < 2e-4
    on = acc[live] / l[live][:, None]
    ref = acco[live] / lo[live][:, None]
    assert np.all(np.abs(on - ref) <= 3e-3 + 1e-2 * np.abs(ref))


# ------------------------------------------------------------------ outputs on the workloads

@pytest.mark.parametrize("cfg_id,path", [
    (1, BUCKETED), (1, WORKQUEUE), (1, SINGLE),
    (2, BUCKETED), (2, WORKQUEUE),
    (3, WORKQUEUE), (3, BUCKETED), (3, SINGLE),
])
def test_workload_outputs_match_oracle(cfg_id, path):
    tr = T.make_trace(cfg_id)
    q = T.gen_q(tr)
    k, v = T.gen_kv(tr)
    d = upload(tr, q, k, v)
    o, lse, ws, _ = run_path(tr, d, path)
    check_error_free(ws)
    oref, lref = oracle_out(tr, q, k, v)
    close(o, oref)
    close_lse(lse, lref)


@pytest.mark.parametrize("B", [4, 8])
def test_zipf_policy_route_matches_oracle(B):
    tr = T.make_trace(4, B=B)
    q = T.gen_q(tr)
    k, v = T.gen_kv(tr)
    d = upload(tr, q, k, v)
    dec = api.PagedDecoder()
    o, lse = dec.step(d["q"], d["k"], d["v"], d["bt"], d["sl"], tr.n_max)
    torch.cuda.synchronize()
    check_error_free(dec.workspace(d["q"].device))
    oref, lref = oracle_out(tr, q, k, v)
    close(o, oref)
    close_lse(lse, lref)
    for path in (BUCKETED, WORKQUEUE, SINGLE):
        o2, l2, ws, _ = run_path(tr, d, path)
        check_error_free(ws)
        close(o2, oref)


@pytest.mark.parametrize("cfg_id,B", [(3, 8), (4, 4), (4, 8)])
def test_learned_cost_model_route_matches_oracle(cfg_id, B):
    """PagedDecoder(learned=True) routes each batch by pkv_policy_learned (the
    learned cost model of the pages' future work) on (B, N_max, N_sum) and runs
    that route's step: the launches are the route's, the outputs match the
    oracle."""
    tr = T.make_trace(4, B=B) if cfg_id == 4 else T.make_trace(cfg_id)
    q = T.gen_q(tr)
    k, v = T.gen_kv(tr)
    d = upload(tr, q, k, v)
    n_sum = int(tr.seq_lens.astype(np.int64).sum())
    path, C = api.pkv_policy_learned(tr.B, tr.n_max, n_sum)
    dec = api.PagedDecoder(learned=True)
    cfg = dec.plan_cfg(tr.B, tr.n_max, n_sum=n_sum)
    assert (cfg.path, cfg.split_tokens if path != SINGLE else C) == (path, C)
    api.pkv_reset_counters()
    o, lse = dec.step(d["q"], d["k"], d["v"], d["bt"], d["sl"], tr.n_max, n_sum=n_sum)
    torch.cuda.synchronize()
    c = api.pkv_get_counters()
    if path == SINGLE:
        assert (c["single_pass_launches"], c["decode_launches"], c["merge_launches"]) == (1, 0, 0)
    else:
        assert (c["decode_launches"], c["merge_launches"]) == (1, 1)
        assert c["plan_launches"] == 0  # bucketed, or the workqueue planning in its decode
    check_error_free(dec.workspace(d["q"].device))
    oref, lref = oracle_out(tr, q, k, v)
    close(o, oref)
    close_lse(lse, lref)


# ------------------------------------------------------------------ edge cases

P_C = [(8, 64), (16, 16), (16, 48), (16, 256), (32, 64), (64, 128), (128, 256), (256, 512)]


@pytest.mark.parametrize("P,C", P_C)
@pytest.mark.parametrize("path", [BUCKETED, WORKQUEUE, SINGLE])
def test_boundary_lengths(P, C, path):
    lens = sorted({1, P - 1, P, P + 1, C - 1, C, C + 1, 2 * C + 3, 0, 63, 64, 65})
    lens = [n for n in lens if n >= 0]
    tr, q, k, v = case(lens, Hq=8, Hkv=2, d=128, P=P, C=C, seed=P * 1000 + C)
    d = upload(tr, q, k, v)
    o, lse, ws, _ = run_path(tr, d, path)
    check_error_free(ws)
    oref, lref = oracle_out(tr, q, k, v)
    close(o, oref)
    close_lse(lse, lref)


@pytest.mark.parametrize("Hq,Hkv,dd", [(4, 4, 128), (16, 2, 128), (8, 8, 64), (16, 2, 64),
                                       (12, 4, 128), (6, 2, 64)])
@pytest.mark.parametrize("path", [BUCKETED, WORKQUEUE, SINGLE])
def test_group_sizes_and_head_dims(Hq, Hkv, dd, path):
    tr, q, k, v = case([333, 17, 1000, 64], Hq=Hq, Hkv=Hkv, d=dd, P=16, C=128, seed=Hq * 7 + dd)
    d = upload(tr, q, k, v)
    o, lse, ws, _ = run_path(tr, d, path)
    check_error_free(ws)
    oref, lref = oracle_out(tr, q, k, v)
    close(o, oref)
    close_lse(lse, lref)


@pytest.mark.parametrize("B,Hq,Hkv,dd", [(64, 32, 8, 128), (64, 32, 8, 64), (400, 6, 2, 128),
                                        (600, 4, 2, 128)])
@pytest.mark.parametrize("path", [BUCKETED, WORKQUEUE])
def test_merge_with_a_warp_per_row_and_head(B, Hq, Hkv, dd, path):
    """Batches of at least 2048 (row, head) pairs merge with one warp per pair
    and four heads of a row per CTA (Hq = 6: the row's second CTA has two idle
    warps; B = 600: the workqueue merge reads its offsets after the wait);
    rows of 0 to 11 splits, empty rows included."""
    rng = np.random.default_rng(B * 10 + Hq + dd)
    lens = rng.integers(0, 700, size=B)
    lens[::17] = 0
    lens[5] = 704  # exactly 11 splits of C = 64
    tr, q, k, v = case(lens.tolist(), Hq=Hq, Hkv=Hkv, d=dd, P=16, C=64, seed=B + Hq + dd)
    d = upload(tr, q, k, v)
    o, lse, ws, _ = run_path(tr, d, path)
    check_error_free(ws)
    oref, lref = oracle_out(tr, q, k, v)
    close(o, oref)
    close_lse(lse, lref)


def test_random_batches_on_every_path():
    """Seeded random batches on the bucketed split, the workqueue (plan
    kernel) and the single pass: B up to 64, page sizes 8..256, C = 1..8
    pages, Hkv 1..8, G 1..8, d 64 or 128, rows of 0 to 40 pages."""
    rng = np.random.default_rng(20261204)
    for n in range(16):
        B = int(rng.choice([1, 2, 5, 16, 64]))
        P = int(rng.choice([8, 16, 32, 256]))
        C = P * int(rng.choice([1, 2, 8]))
        Hkv, G, dd = int(rng.choice([1, 2, 8])), int(rng.choice([1, 3, 8])), int(rng.choice([64, 128]))
        lens = rng.integers(0, 40 * P + 1, size=B)
        lens[rng.random(B) < 0.15] = 0
        tr, q, k, v = case(lens.tolist(), Hq=Hkv * G, Hkv=Hkv, d=dd, P=P, C=C, seed=100 + n)
        d = upload(tr, q, k, v)
        oref, lref = oracle_out(tr, q, k, v)
        for path in (BUCKETED, WORKQUEUE, SINGLE):
            o, lse, ws, _ = run_path(tr, d, path)
            check_error_free(ws)
            close(o, oref, f"case {n}, path {path}")
            close_lse(lse, lref)


def test_wide_table_shared_pages_and_big_pool():
    tr, q, k, v = case([500, 300, 77, 0, 1], Hq=8, Hkv=2, P=16, C=128, extra_pages=40,
                       extra_cols=5, share_prefix_pages=10)
    assert np.array_equal(tr.block_table[1, :10], tr.block_table[0, :10])
    d = upload(tr, q, k, v)
    oref, lref = oracle_out(tr, q, k, v)
    for path in (BUCKETED, WORKQUEUE, SINGLE):
        o, lse, ws, _ = run_path(tr, d, path)
        check_error_free(ws)
        close(o, oref)
        close_lse(lse, lref)


def test_empty_batch_rows_and_zero_lengths():
    tr, q, k, v = case([0, 0, 5], Hq=8, Hkv=2)
    d = upload(tr, q, k, v)
    oref, lref = oracle_out(tr, q, k, v)
    for path in (BUCKETED, WORKQUEUE, SINGLE):
        o, lse, ws, _ = run_path(tr, d, path)
        check_error_free(ws)
        assert torch.all(o[:2] == 0)
        assert torch.all(lse[:2] == float("-inf"))
        close(o, oref)


def test_empty_batch_through_the_python_api():
    """B = 0 through PagedDecoder on every route: no launch, empty outputs."""
    k = torch.zeros((4, 16, 2, 128), dtype=torch.float16, device="cuda")
    q = torch.zeros((0, 8, 128), dtype=torch.float16, device="cuda")
    bt = torch.zeros((0, 4), dtype=torch.int32, device="cuda")
    sl = torch.zeros((0,), dtype=torch.int32, device="cuda")
    api.pkv_reset_counters()
    for path in (BUCKETED, WORKQUEUE, SINGLE):
        for merge in (_lib.PKV_MERGE_SEPARATE, _lib.PKV_MERGE_FUSED):
            o, lse = api.PagedDecoder(merge=merge).step(q, k, k, bt, sl, 0, path=path,
                                                        split_tokens=16)
            assert o.shape == (0, 8, 128) and lse.shape == (0, 8)
    torch.cuda.synchronize()
    assert sum(api.pkv_get_counters().values()) == 0


def test_one_very_long_row():
    """N = 262144 tokens in one row (16384 pages): 256 splits for the merge to
    combine on the split paths (also fused), 128 block-table segments per
    task on the single pass."""
    tr, q, k, v = case([262144], Hq=8, Hkv=2, P=16, C=1024, seed=41)
    d = upload(tr, q, k, v)
    oref, lref = oracle_out(tr, q, k, v)
    for path, merge in ((BUCKETED, _lib.PKV_MERGE_SEPARATE), (WORKQUEUE, _lib.PKV_MERGE_SEPARATE),
                        (SINGLE, _lib.PKV_MERGE_SEPARATE), (BUCKETED, _lib.PKV_MERGE_FUSED),
                        (WORKQUEUE, _lib.PKV_MERGE_FUSED)):
        o, lse, ws, _ = run_path(tr, d, path, merge=merge)
        check_error_free(ws)
        close(o, oref, f"o on path {path} merge {merge}")
        close_lse(lse, lref)


def test_outputs_are_deterministic():
    tr = T.make_trace(3)
    q = T.gen_q(tr)
    k, v = T.gen_kv(tr)
    d = upload(tr, q, k, v)
    a = run_path(tr, d, WORKQUEUE)[0]
    b = run_path(tr, d, WORKQUEUE)[0]
    assert torch.equal(a, b)


def test_extreme_scores_stay_finite():
    tr, q, k, v = case([900, 40], Hq=8, Hkv=2, C=128)
    k[:] = np.float16(0.0)
    q[:] = np.float16(30.0)
    rng = np.random.default_rng(1)
    idx = rng.choice(tr.num_pages, size=4, replace=False)
    k[idx] = np.float16(20.0)   # a few pages with very large scores
    d = upload(tr, q, k, v)
    oref, lref = oracle_out(tr, q, k, v)
    for path in (BUCKETED, WORKQUEUE, SINGLE):
        o, lse, ws, _ = run_path(tr, d, path)
        check_error_free(ws)
        close(o, oref)
        close_lse(lse, lref)


# ------------------------------------------------------------------ launch counts

@pytest.mark.parametrize("path,expect", [(BUCKETED, dict(decode_launches=1, merge_launches=1)),
                                         (WORKQUEUE, dict(plan_launches=1, decode_launches=1,
                                                          merge_launches=1)),
                                         (SINGLE, dict(single_pass_launches=1))])
def test_launch_counts_match_model(path, expect):
    tr = T.make_trace(3)
    d = upload(tr, T.gen_q(tr), *T.gen_kv(tr))
    api.pkv_reset_counters()
    run_path(tr, d, path)
    got = api.pkv_get_counters()
    full = dict(plan_launches=0, decode_launches=0, merge_launches=0, single_pass_launches=0,
                append_launches=0)
    full.update(expect)
    assert got == full
    model = oracle.counters(path, tr.seq_lens, tr.Hq, tr.Hkv, tr.d, tr.split_tokens,
                            -(-tr.n_max // tr.split_tokens))
    attn = got["decode_launches"] + got["merge_launches"] + got["single_pass_launches"]
    assert attn == model.attn_launches and got["plan_launches"] == model.plan_launches


# ------------------------------------------------------------------ device-side checks

@pytest.mark.parametrize("path", [BUCKETED, WORKQUEUE])
def test_state_traffic_is_what_the_kernels_write_and_read(path):
    """The merge-state counts of the step model (behind the pages' merge-state
    traffic comparison, Results, 'Scheduling overhead') against the kernels
    themselves.  Written: every slot the split decode changes in a buffer
    filled with a marker.  Read: with every slot outside the counted set
    replaced by a state that would ruin any merge using it (l = 1, m = 0,
    acc = NaN) the merge is bit-identical; replacing the counted slots of
    split j ruins exactly the rows that have a split j."""
    lens = [100, 3000, 40, 0, 1024, 2049]
    Hq, Hkv, d, C = 8, 2, 64, 256
    tr, q, k, v = case(lens, Hq, Hkv, d, 16, C)
    dd = upload(tr, q, k, v)
    shape = shape_of(tr)
    S_b = -(-max(lens) // C)
    cfg = api.make_cfg(path, C, max(lens) if path == BUCKETED else 0)
    ws = torch.zeros(api.pkv_plan_workspace_size(shape, cfg), dtype=torch.uint8, device="cuda")
    npart = api.pkv_partials_size(shape, cfg) // 4
    slots = npart // (d + 2)
    part = torch.full((npart,), 1234.5, dtype=torch.float32, device="cuda")
    if path == WORKQUEUE:
        api.pkv_plan(shape, cfg, dd["sl"], ws)
    api.pkv_decode(shape, cfg, ws, dd["q"], dd["k"], dd["v"], dd["bt"], dd["sl"], part)
    torch.cuda.synchronize()
    check_error_free(ws)
    acc = part[:slots * d].view(slots, d)
    m, l = part[slots * d:slots * (d + 1)], part[slots * (d + 1):]
    written = int(((l != 1234.5) | (m != 1234.5)).sum())
    model = api.pkv_step_model(path, shape, C, max(lens), lens)
    assert written == model["states_written"] == oracle.counters(
        path, lens, Hq, Hkv, d, C, S_b).states_written
    n = [-(-x // C) for x in lens]
    off = np.concatenate([[0], np.cumsum(n)])
    split_slots = {}  # split j -> the counted slots of every row's split j
    for i, ni in enumerate(n):
        for j in range(ni):
            base = (i * S_b + j) * Hq if path == BUCKETED else (off[i] + j) * Hq
            split_slots.setdefault(j, []).extend(range(base, base + Hq))
    counted = sorted(s_ for v_ in split_slots.values() for s_ in v_)
    assert len(counted) == model["states_read"] == oracle.counters(
        path, lens, Hq, Hkv, d, C, S_b).states_read
    o0 = torch.empty((tr.B, Hq, d), dtype=torch.float16, device="cuda")
    api.pkv_merge(shape, cfg, ws, dd["sl"], part, o0)
    clean = part.clone()

    def ruin(idx):
        t = clean.clone()
        ix = torch.tensor(idx, dtype=torch.long, device="cuda")
        t[slots * d:slots * (d + 1)][ix] = 0.0
        t[slots * (d + 1):][ix] = 1.0
        t[:slots * d].view(slots, d)[ix] = float("nan")
        o = torch.empty_like(o0)
        api.pkv_merge(shape, cfg, ws, dd["sl"], t, o)
        torch.cuda.synchronize()
        return o.float().cpu().numpy()

    others = sorted(set(range(slots)) - set(counted))
    if others:
        assert np.array_equal(ruin(others), o0.float().cpu().numpy(), equal_nan=True)
    base_o = o0.float().cpu().numpy()
    for j, idx in split_slots.items():
        got = ruin(idx)
        for i, ni in enumerate(n):
            if ni > j:
                assert np.isnan(got[i]).all(), (j, i)
            else:
                assert np.array_equal(got[i], base_o[i]), (j, i)


def test_bad_page_id_is_reported_not_faulted():
    tr, q, k, v = case([100, 50], Hq=8, Hkv=2, C=64)
    tr.block_table[1, 2] = tr.num_pages + 7     # out of range
    d = upload(tr, q, k, v)
    for path in (BUCKETED, WORKQUEUE, SINGLE):
        o, lse, ws, _ = run_path(tr, d, path)
        st, msg = api.pkv_get_error(ws)
        assert st == _lib.PKV_EDEVICE and "row 1" in msg, msg
        # row 0 is untouched by the bad entry
        tr0 = T.custom_trace([100], 8, 2, 128, 16, 64)
        tr0.block_table = tr.block_table[:1, :7].copy()
        tr0.num_pages = tr.num_pages
        oref, _ = oracle.attention(q[:1], k, v, tr0.block_table, tr.seq_lens[:1], tr.scale)
        close(o[:1], oref)


def test_row_longer_than_bucket_is_reported():
    tr, q, k, v = case([300, 100], Hq=8, Hkv=2, C=64)
    d = upload(tr, q, k, v)
    o, lse, ws, _ = run_path(tr, d, BUCKETED, C=64, bucket=128)
    st, msg = api.pkv_get_error(ws)
    assert st == _lib.PKV_EDEVICE and "row 0" in msg, msg
    api.pkv_get_error(ws)  # cleared
    assert api.pkv_get_error(ws)[0] == 0


# ------------------------------------------------------------------ append

def test_append_writes_the_next_slot():
    tr, q, k, v = case([15, 16, 40, 0], Hq=8, Hkv=2, P=16, C=64, extra_cols=2, extra_pages=8)
    # give every row one more page for the new token
    free = [p for p in range(tr.num_pages) if p not in set(tr.block_table[tr.block_table >= 0].tolist())]
    for i in range(tr.B):
        n = int(tr.seq_lens[i])
        if tr.block_table[i, n // 16] < 0:
            tr.block_table[i, n // 16] = free.pop()
    d = upload(tr, q, k, v)
    kn, vn = T.gen_append_tokens(tr, 0)
    shape = shape_of(tr)
    ws = torch.zeros(64, dtype=torch.uint8, device="cuda")
    api.pkv_reset_counters()
    api.pkv_append(shape, ws, dev(kn), dev(vn), d["bt"], d["sl"], d["k"], d["v"])
    torch.cuda.synchronize()
    check_error_free(ws)
    assert api.pkv_get_counters()["append_launches"] == 1
    assert np.array_equal(d["sl"].cpu().numpy(), tr.seq_lens + 1)
    kc, vc = d["k"].cpu().numpy(), d["v"].cpu().numpy()
    for i in range(tr.B):
        n = int(tr.seq_lens[i])
        pg, sl = tr.block_table[i, n // 16], n % 16
        assert np.array_equal(kc[pg, sl], kn[i]) and np.array_equal(vc[pg, sl], vn[i])
    # nothing else changed
    mask = np.ones(k.shape[:2], bool)
    for i in range(tr.B):
        n = int(tr.seq_lens[i])
        mask[tr.block_table[i, n // 16], n % 16] = False
    assert np.array_equal(kc[mask].view(np.uint16), k[mask].view(np.uint16))


# ------------------------------------------------------------------ host-buffer step

@pytest.mark.parametrize("cfg_id,path", [(1, BUCKETED), (3, WORKQUEUE), (3, SINGLE)])
def test_host_buffer_step_matches_oracle(cfg_id, path):
    tr = T.make_trace(cfg_id)
    q = T.gen_q(tr)
    k, v = T.gen_kv(tr)
    kd, vd = dev(k), dev(v)
    loop = api.HostDecodeLoop(kd, vd, tr.B, tr.Hq, tr.bt_stride, tr.n_max, path=path,
                              split_tokens=tr.split_tokens)
    hq = torch.from_numpy(q).pin_memory()
    hbt = torch.from_numpy(tr.block_table).pin_memory()
    hsl = torch.from_numpy(tr.seq_lens).pin_memory()
    oref, lref = oracle_out(tr, q, k, v)
    for _ in range(2):
        o, lse = loop.step(hq, hbt, hsl)
        close(o, oref)
        close_lse(lse, lref)
    check_error_free(loop.ws)


@pytest.mark.parametrize("pinned", [True, False])
def test_host_buffer_step_outputs_in_place_or_copied(pinned):
    """pkv_decode_step_host reads page-locked q, block table and lengths in
    place and writes page-locked h_o / h_lse straight from the step's last
    kernel (the device buffers stay untouched); pageable buffers go through the
    device ones.  Both match the oracle."""
    tr = T.make_trace(3)
    q = T.gen_q(tr)
    k, v = T.gen_kv(tr)
    d = upload(tr, q, k, v)
    shape = shape_of(tr)
    cfg = api.make_cfg(WORKQUEUE, tr.split_tokens, 0, 0, 0, _lib.PKV_PLAN_IN_DECODE)
    ws = torch.zeros(api.pkv_plan_workspace_size(shape, cfg), dtype=torch.uint8, device="cuda")
    part = torch.empty(api.pkv_partials_size(shape, cfg) // 4, dtype=torch.float32, device="cuda")
    host = (lambda t: t.pin_memory()) if pinned else (lambda t: t)
    hq = host(torch.from_numpy(q))
    hbt = host(torch.from_numpy(tr.block_table))
    hsl = host(torch.from_numpy(tr.seq_lens))
    h_o = host(torch.full(q.shape, float("nan"), dtype=torch.float16))
    h_lse = host(torch.full(q.shape[:2], float("nan"), dtype=torch.float32))
    d_o = torch.full(q.shape, float("nan"), dtype=torch.float16, device="cuda")
    d_lse = torch.full(q.shape[:2], float("nan"), dtype=torch.float32, device="cuda")
    d_q = torch.full(q.shape, float("nan"), dtype=torch.float16, device="cuda")
    d_bt = torch.full_like(d["bt"], -7)
    d_sl = torch.full_like(d["sl"], -7)
    api.pkv_decode_step_host(shape, cfg, ws, part, hq, d_q, hbt, d_bt, hsl, d_sl, d["k"],
                             d["v"], d_o, h_o, d_lse, h_lse)
    check_error_free(ws)
    oref, lref = oracle_out(tr, q, k, v)
    close(h_o, oref)
    close_lse(h_lse, lref)
    if pinned:  # every host buffer used in place: the device ones were never written
        assert torch.isnan(d_o.float()).all() and torch.isnan(d_lse).all()
        assert torch.isnan(d_q.float()).all() and (d_bt == -7).all() and (d_sl == -7).all()
    else:
        assert torch.equal(d_o.cpu(), h_o) and torch.equal(d_lse.cpu(), h_lse)
        assert torch.equal(d_q.cpu(), hq) and torch.equal(d_bt.cpu(), hbt) and torch.equal(d_sl.cpu(), hsl)


# ------------------------------------------------------------------ exact-length buckets

def test_exact_length_buckets_match_oracle_and_launch_twice_per_length():
    """The scheme the pages compare against: one split + merge launch pair per
    distinct length; 8 distinct lengths on the bimodal B=8 trace -> 16
    launches, where the workqueue needs 2 (plus the plan)."""
    tr = T.make_trace(3)
    q = T.gen_q(tr)
    k, v = T.gen_kv(tr)
    d = upload(tr, q, k, v)
    o = torch.full((tr.B, tr.Hq, tr.d), float("nan"), dtype=torch.float16, device="cuda")
    lse = torch.full((tr.B, tr.Hq), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.zeros(64, dtype=torch.uint8, device="cuda")
    api.pkv_reset_counters()
    groups = api.exact_length_buckets_step(d["q"], d["k"], d["v"], d["bt"], d["sl"], tr.seq_lens,
                                           tr.split_tokens, o, lse, ws=ws)
    torch.cuda.synchronize()
    check_error_free(ws)
    c = api.pkv_get_counters()
    assert groups == 8
    assert c["decode_launches"] + c["merge_launches"] == 16 and c["plan_launches"] == 0
    oref, lref = oracle_out(tr, q, k, v)
    close(o, oref)
    close_lse(lse, lref)


def test_exact_length_buckets_with_empty_and_repeated_lengths():
    """Rows sharing a length run in one group; rows without tokens run as one
    more group that gives them o = 0, lse = -inf."""
    lens = [300, 0, 64, 300, 1, 0, 64, 1000]
    tr, q, k, v = case(lens, 8, 2, 128, 16, 64)
    d = upload(tr, q, k, v)
    o = torch.full((tr.B, tr.Hq, tr.d), float("nan"), dtype=torch.float16, device="cuda")
    lse = torch.full((tr.B, tr.Hq), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.zeros(64, dtype=torch.uint8, device="cuda")
    api.pkv_reset_counters()
    groups = api.exact_length_buckets_step(d["q"], d["k"], d["v"], d["bt"], d["sl"], tr.seq_lens,
                                           64, o, lse, ws=ws)
    torch.cuda.synchronize()
    check_error_free(ws)
    assert groups == 4 + 1  # lengths 1, 64, 300, 1000, then the empty rows
    c = api.pkv_get_counters()
    assert c["decode_launches"] + c["merge_launches"] == 2 * groups
    oref, lref = oracle_out(tr, q, k, v)
    close(o, oref)
    close_lse(lse, lref)


def test_row_list_step_leaves_other_rows_untouched():
    tr, q, k, v = case([300, 50, 300, 0, 128], Hq=8, Hkv=2, C=64)
    d = upload(tr, q, k, v)
    o = torch.full((tr.B, tr.Hq, tr.d), 7.0, dtype=torch.float16, device="cuda")
    lse = torch.full((tr.B, tr.Hq), 7.0, dtype=torch.float32, device="cuda")
    rows = torch.tensor([2, 0], dtype=torch.int32, device="cuda")
    shape = shape_of(tr)
    cfg = api.make_cfg(BUCKETED, 64, 300)
    sub = _lib.Shape(2, tr.Hq, tr.Hkv, tr.d, tr.page_size, tr.num_pages, tr.bt_stride, tr.scale)
    part = torch.empty(api.pkv_partials_size(sub, cfg) // 4, dtype=torch.float32, device="cuda")
    ws = torch.zeros(64, dtype=torch.uint8, device="cuda")
    api.pkv_decode_step_rows(shape, cfg, ws, rows, d["q"], d["k"], d["v"], d["bt"], d["sl"], part,
                             o, lse)
    torch.cuda.synchronize()
    check_error_free(ws)
    oref, lref = oracle_out(tr, q, k, v)
    close(o[[0, 2]], oref[[0, 2]])
    close_lse(lse[[0, 2]], lref[[0, 2]])
    assert torch.all(o[[1, 3, 4]] == 7.0) and torch.all(lse[[1, 3, 4]] == 7.0)
    # a row id outside the batch is reported, not faulted
    bad = torch.tensor([0, 9], dtype=torch.int32, device="cuda")
    api.pkv_decode_step_rows(shape, cfg, ws, bad, d["q"], d["k"], d["v"], d["bt"], d["sl"], part,
                             o, lse)
    st, msg = api.pkv_get_error(ws)
    assert st == _lib.PKV_EDEVICE and "row list" in msg, msg


@pytest.mark.parametrize("cfg_id,path,in_place", [(2, BUCKETED, True), (3, WORKQUEUE, True),
                                                  (1, SINGLE, True), (3, WORKQUEUE, False)])
def test_host_loop_graph_step_matches_oracle(cfg_id, path, in_place):
    """The captured host step: its kernels read q, the block table and the
    lengths from pinned host memory in place (the plan too, on the workqueue),
    or from one copy of them, and write o / lse into pinned host memory."""
    tr = T.make_trace(cfg_id)
    q = T.gen_q(tr)
    k, v = T.gen_kv(tr)
    loop = api.HostDecodeLoop(dev(k), dev(v), tr.B, tr.Hq, tr.bt_stride, tr.n_max,
                              path=path, split_tokens=tr.split_tokens, inputs_in_place=in_place)
    loop.h_q.copy_(torch.from_numpy(q))
    loop.h_bt.copy_(torch.from_numpy(tr.block_table))
    loop.h_sl.copy_(torch.from_numpy(tr.seq_lens))
    s = torch.cuda.Stream()
    loop.capture(s)
    oref, lref = oracle_out(tr, q, k, v)
    for _ in range(2):
        o, lse = loop.step_graph()
        close(o, oref)
        close_lse(lse, lref)
    # the next step's query, written into the pinned input, is what the kernels read
    q2 = T.gen_step_q(tr, 1)
    loop.h_q.copy_(torch.from_numpy(q2))
    o, lse = loop.step_graph()
    oref2, lref2 = oracle_out(tr, q2, k, v)
    close(o, oref2)
    close_lse(lse, lref2)
    check_error_free(loop.ws)


# ------------------------------------------------------------------ bounded waits

def test_a_starved_barrier_times_out_and_the_context_stays_usable():
    """A barrier wait that nothing completes (test hook) runs out after its
    bound; the kernel reports PKV_ETIMEOUT and returns, and the next launch on
    the same context is correct."""
    tr = T.make_trace(1)
    q = T.gen_q(tr)
    k, v = T.gen_kv(tr)
    d = upload(tr, q, k, v)
    L = _lib.load()
    assert L.pkv_test_starve_next_decodes(1) == 0
    try:
        o, lse, ws, _ = run_path(tr, d, BUCKETED)
    finally:
        L.pkv_test_starve_next_decodes(0)
    st, msg = api.pkv_get_error(ws)
    assert st == _lib.PKV_ETIMEOUT, msg
    o, lse, ws, _ = run_path(tr, d, BUCKETED)
    check_error_free(ws)
    oref, lref = oracle_out(tr, q, k, v)
    close(o, oref)


# ------------------------------------------------------------------ dynamic task claims

def _claim_counters(ws):
    h = ws[:64].view(torch.int32).cpu().numpy()
    return int(h[7]), int(h[8])  # next_task, done_ctas


def test_workqueue_claims_reset_between_launches():
    """The workqueue decode hands tasks out from a counter in the workspace
    header; the last CTA of a launch zeroes it, so repeated decodes on one
    plan and workspace each process every task (bit-identical outputs)."""
    tr = T.make_trace(3)
    q = T.gen_q(tr)
    k, v = T.gen_kv(tr)
    d = upload(tr, q, k, v)
    shape = shape_of(tr)
    cfg = api.make_cfg(WORKQUEUE, tr.split_tokens)
    ws = torch.zeros(api.pkv_plan_workspace_size(shape, cfg), dtype=torch.uint8, device="cuda")
    part = torch.empty(api.pkv_partials_size(shape, cfg) // 4, dtype=torch.float32, device="cuda")
    api.pkv_plan(shape, cfg, d["sl"], ws)
    outs = []
    for _ in range(4):
        part.fill_(float("nan"))
        o = torch.empty((tr.B, tr.Hq, tr.d), dtype=torch.float16, device="cuda")
        lse = torch.empty((tr.B, tr.Hq), dtype=torch.float32, device="cuda")
        api.pkv_decode(shape, cfg, ws, d["q"], d["k"], d["v"], d["bt"], d["sl"], part)
        api.pkv_merge(shape, cfg, ws, d["sl"], part, o, lse)
        torch.cuda.synchronize()
        assert _claim_counters(ws) == (0, 0)
        outs.append((o, lse))
    check_error_free(ws)
    oref, lref = oracle_out(tr, q, k, v)
    close(outs[0][0], oref)
    close_lse(outs[0][1], lref)
    for o, lse in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(lse, outs[0][1])


def test_a_starved_workqueue_launch_resets_its_claims():
    """A CTA that times out stops claiming; the others take the remaining
    tasks, every CTA still counts itself done, and the next launch on the same
    workspace starts from a zeroed counter."""
    tr = T.make_trace(3)
    q = T.gen_q(tr)
    k, v = T.gen_kv(tr)
    d = upload(tr, q, k, v)
    L = _lib.load()
    assert L.pkv_test_starve_next_decodes(1) == 0
    try:
        o, lse, ws, _ = run_path(tr, d, WORKQUEUE)
    finally:
        L.pkv_test_starve_next_decodes(0)
    st, msg = api.pkv_get_error(ws)
    assert st == _lib.PKV_ETIMEOUT, msg
    assert _claim_counters(ws) == (0, 0)
    o, lse, ws, _ = run_path(tr, d, WORKQUEUE, ws=ws)
    check_error_free(ws)
    oref, lref = oracle_out(tr, q, k, v)
    close(o, oref)
    close_lse(lse, lref)


# ------------------------------------------------------------------ the timed launch configuration

@pytest.mark.parametrize("cfg_id,path,merge", [(2, BUCKETED, _lib.PKV_MERGE_SEPARATE),
                                               (3, WORKQUEUE, _lib.PKV_MERGE_SEPARATE),
                                               (1, SINGLE, _lib.PKV_MERGE_SEPARATE),
                                               (2, BUCKETED, _lib.PKV_MERGE_FUSED),
                                               (3, WORKQUEUE, _lib.PKV_MERGE_FUSED)])
def test_chained_graph_steps_match_oracle(cfg_id, path, merge):
    """bench.py times CUDA graphs of consecutive steps whose kernels chain by
    programmatic dependent launch: a step's decode may start while the previous
    step's merge still reads the partial states.  Replaying such a graph (four
    steps on the same workspace, partials and outputs) must give the oracle's
    result every time."""
    tr = T.make_trace(cfg_id)
    q = T.gen_q(tr)
    k, v = T.gen_kv(tr)
    d = upload(tr, q, k, v)
    shape = shape_of(tr)
    cfg = api.make_cfg(path, tr.split_tokens, tr.n_max if path == BUCKETED else 0, 0, merge)
    ws = torch.zeros(max(64, api.pkv_plan_workspace_size(shape, cfg)), dtype=torch.uint8,
                     device="cuda")
    npart = api.pkv_partials_size(shape, cfg)
    part = torch.empty(max(npart // 4, 4), dtype=torch.float32, device="cuda") if npart else None
    o = torch.empty((tr.B, tr.Hq, tr.d), dtype=torch.float16, device="cuda")
    lse = torch.empty((tr.B, tr.Hq), dtype=torch.float32, device="cuda")
    k2, v2 = d["k"].clone(), d["v"].clone()  # a second pool, as the bench rotates them
    st = torch.cuda.Stream()

    def steps():
        for r in range(4):
            kk, vv = (d["k"], d["v"]) if r % 2 == 0 else (k2, v2)
            api.pkv_decode_step(shape, cfg, ws, d["q"], kk, vv, d["bt"], d["sl"], part, o, lse,
                                stream=st)

    with torch.cuda.stream(st):
        steps()
        st.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            steps()
    oref, lref = oracle_out(tr, q, k, v)
    for _ in range(3):
        with torch.cuda.stream(st):
            o.fill_(float("nan"))
            g.replay()
        st.synchronize()
        check_error_free(ws)
        close(o, oref)
        close_lse(lse, lref)
