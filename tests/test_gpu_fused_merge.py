"""GPU parity of the fused merge (PKV_MERGE_FUSED, pkv_decode_merge) against
the float64 oracle, and its bookkeeping.

The fused step computes what pkv_decode + pkv_merge compute -- the exact
log-sum-exp merge of "Sequence splitting" -- with the merge run on the decode's
tail: the CTAs meet at a grid-wide barrier, then share out the (row, query
head) merges.  Besides the outputs (the parity tolerance
|x - y| <= 3e-3 + 1e-2 |y|), these tests check that the header's counters
(task claims, barrier) are back at zero after every launch, also after a
timeout, that rows without tokens and workqueue overflows give the merge
kernel's outputs, that reruns are bit-identical, and the launch counts.
"""
import numpy as np
import pytest
import torch

import pkv_traces as T
from paged_kv_gqa_09_gb300 import _lib, api

from gpu_util import (check_error_free, close, close_lse, dev, header_counters, oracle_out,
                      run_path, shape_of, upload)

pytestmark = pytest.mark.gpu

BUCKETED, WORKQUEUE = _lib.PKV_PATH_BUCKETED_SPLIT, _lib.PKV_PATH_WORKQUEUE
FUSED, SEPARATE = _lib.PKV_MERGE_FUSED, _lib.PKV_MERGE_SEPARATE


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


def fused(tr, d, path, **kw):
    """One fused step; checks it left no device error and every counter at 0."""
    o, lse, ws, part = run_path(tr, d, path, merge=FUSED, **kw)
    check_error_free(ws)
    assert not any(header_counters(ws).values()), "header counters not reset"
    return o, lse, ws, part


def against_oracle(tr, q, k, v, path, **kw):
    d = upload(tr, q, k, v)
    o, lse, _, _ = fused(tr, d, path, **kw)
    oref, lref = oracle_out(tr, q, k, v)
    close(o, oref)
    close_lse(lse, lref)


# ------------------------------------------------------------------ parity

@pytest.mark.parametrize("cfg_id,path", [
    (1, BUCKETED), (1, WORKQUEUE), (2, BUCKETED), (2, WORKQUEUE), (3, WORKQUEUE), (3, BUCKETED),
])
def test_fused_workload_outputs_match_oracle(cfg_id, path):
    tr = T.make_trace(cfg_id)
    q = T.gen_q(tr)
    k, v = T.gen_kv(tr)
    against_oracle(tr, q, k, v, path)


P_C = [(8, 64), (16, 16), (16, 48), (32, 64), (64, 128), (256, 512)]


@pytest.mark.parametrize("P,C", P_C)
@pytest.mark.parametrize("path", [BUCKETED, WORKQUEUE])
def test_fused_boundary_lengths(P, C, path):
    """Rows of 0 tokens (no task), of one split (o from registers) and of
    several splits (merged after the grid-wide barrier), around page and split ends."""
    lens = sorted({0, 1, P - 1, P, P + 1, C - 1, C, C + 1, 2 * C + 3, 63, 64, 65})
    tr, q, k, v = case(lens, P=P, C=C, seed=P * 1000 + C)
    against_oracle(tr, q, k, v, path)


@pytest.mark.parametrize("Hq,Hkv,dd", [(4, 4, 128), (16, 2, 128), (8, 8, 64), (16, 2, 64),
                                       (12, 4, 128), (6, 2, 64)])
@pytest.mark.parametrize("path", [BUCKETED, WORKQUEUE])
def test_fused_group_sizes_and_head_dims(Hq, Hkv, dd, path):
    """G = 1..8 query heads per KV head (each merged head is one unit of the
    tail's work), d = 64 and 128."""
    tr, q, k, v = case([333, 17, 1000, 64], Hq=Hq, Hkv=Hkv, d=dd, P=16, C=128, seed=Hq * 7 + dd)
    against_oracle(tr, q, k, v, path)


@pytest.mark.parametrize("path", [BUCKETED, WORKQUEUE])
def test_fused_rows_with_many_splits(path):
    """Rows of up to 101 splits: each merging warp folds a quarter of them."""
    tr, q, k, v = case([100 * 64 + 5, 33 * 64, 32 * 64, 31 * 64 + 1, 64], Hq=16, Hkv=2, C=64,
                       seed=11)
    against_oracle(tr, q, k, v, path)


# ------------------------------------------------------------------ edge cases

@pytest.mark.parametrize("path", [BUCKETED, WORKQUEUE])
def test_fused_empty_rows_get_zero_and_minus_inf(path):
    tr, q, k, v = case([0, 0, 5, 0, 700], Hq=8, Hkv=2)
    d = upload(tr, q, k, v)
    o, lse, _, _ = fused(tr, d, path)
    assert torch.all(o[[0, 1, 3]] == 0)
    assert torch.all(lse[[0, 1, 3]] == float("-inf"))
    oref, lref = oracle_out(tr, q, k, v)
    close(o, oref)
    close_lse(lse, lref)


def test_fused_workqueue_overflow_writes_nan_and_reports():
    """No task runs after an overflow: every row gets NaN, and the merge phase
    must not combine the (here zero-filled) states no task wrote."""
    tr, q, k, v = case([300, 700], Hq=8, Hkv=2)
    d = upload(tr, q, k, v)
    shape = shape_of(tr)
    cfg = api.make_cfg(WORKQUEUE, 64, 0, 5, FUSED)
    ws = torch.zeros(api.pkv_plan_workspace_size(shape, cfg), dtype=torch.uint8, device="cuda")
    part = torch.zeros(api.pkv_partials_size(shape, cfg) // 4, dtype=torch.float32, device="cuda")
    o = torch.zeros((tr.B, tr.Hq, tr.d), dtype=torch.float16, device="cuda")
    lse = torch.zeros((tr.B, tr.Hq), dtype=torch.float32, device="cuda")
    api.pkv_decode_step(shape, cfg, ws, d["q"], d["k"], d["v"], d["bt"], d["sl"], part, o, lse)
    st, msg = api.pkv_get_error(ws)
    assert st == _lib.PKV_ECAPACITY, msg
    assert torch.isnan(o.float()).all() and torch.isnan(lse).all()
    assert not any(header_counters(ws).values())


def test_fused_equals_separate_and_reruns_bit_identically():
    """Each (row, head) is merged by one CTA reading its states in a fixed
    order, so reruns are bit-identical whichever CTAs ran which tasks."""
    for cfg_id, path in ((3, WORKQUEUE), (1, BUCKETED), (2, BUCKETED)):
        tr = T.make_trace(cfg_id)
        q = T.gen_q(tr)
        k, v = T.gen_kv(tr)
        d = upload(tr, q, k, v)
        a, la, _, _ = fused(tr, d, path)
        b, lb, _, _ = fused(tr, d, path)
        assert torch.equal(a, b) and torch.equal(la, lb)
        s, ls, ws, _ = run_path(tr, d, path, merge=SEPARATE)
        check_error_free(ws)
        assert (a.float() - s.float()).abs().max().item() <= 2e-3
        fin = torch.isfinite(ls)
        assert torch.equal(fin, torch.isfinite(la))
        assert (la[fin] - ls[fin]).abs().max().item() <= 1e-4


def test_fused_steps_reuse_one_workspace():
    """Counters reset themselves: consecutive steps on one workspace (as a
    serving loop runs them) stay correct while the lengths change (each row
    stays within the pages it owns)."""
    import oracle
    tr, q, k, v = case([900, 64, 0, 2000, 130], Hq=8, Hkv=2, C=128)
    d = upload(tr, q, k, v)
    full = tr.seq_lens.copy()
    for path in (BUCKETED, WORKQUEUE):
        ws = None
        for step in range(6):
            lens = (full * (6 - step) // 6).astype(np.int32)
            lens[1] = full[1] if step % 2 else 0
            d["sl"] = dev(lens)
            o, lse, ws, _ = fused(tr, d, path, bucket=int(full.max()) if path == BUCKETED else 0,
                                  ws=ws)
            oref, lref = oracle.attention(q, k, v, tr.block_table, lens, tr.scale)
            close(o, oref)
            close_lse(lse, lref)


def test_fused_row_list_step_leaves_other_rows_untouched():
    tr, q, k, v = case([300, 50, 300, 0, 128], Hq=8, Hkv=2, C=64)
    d = upload(tr, q, k, v)
    o = torch.full((tr.B, tr.Hq, tr.d), 7.0, dtype=torch.float16, device="cuda")
    lse = torch.full((tr.B, tr.Hq), 7.0, dtype=torch.float32, device="cuda")
    rows = torch.tensor([2, 0, 3], dtype=torch.int32, device="cuda")
    shape = shape_of(tr)
    cfg = api.make_cfg(BUCKETED, 64, 300, 0, FUSED)
    sub = _lib.Shape(3, tr.Hq, tr.Hkv, tr.d, tr.page_size, tr.num_pages, tr.bt_stride, tr.scale)
    part = torch.empty(api.pkv_partials_size(sub, cfg) // 4, dtype=torch.float32, device="cuda")
    ws = torch.zeros(api.pkv_plan_workspace_size(shape, cfg), dtype=torch.uint8, device="cuda")
    api.pkv_reset_counters()
    api.pkv_decode_step_rows(shape, cfg, ws, rows, d["q"], d["k"], d["v"], d["bt"], d["sl"], part,
                             o, lse)
    torch.cuda.synchronize()
    check_error_free(ws)
    assert api.pkv_get_counters()["decode_launches"] == 1
    assert api.pkv_get_counters()["merge_launches"] == 0
    assert not any(header_counters(ws).values())
    oref, lref = oracle_out(tr, q, k, v)
    close(o[[0, 2, 3]], oref[[0, 2, 3]])
    close_lse(lse[[0, 2, 3]], lref[[0, 2, 3]])
    assert torch.all(o[[1, 4]] == 7.0) and torch.all(lse[[1, 4]] == 7.0)


@pytest.mark.parametrize("path,expect", [(BUCKETED, dict(decode_launches=1)),
                                         (WORKQUEUE, dict(plan_launches=1, decode_launches=1))])
def test_fused_launch_counts(path, expect):
    tr = T.make_trace(3)
    d = upload(tr, T.gen_q(tr), *T.gen_kv(tr))
    api.pkv_reset_counters()
    fused(tr, d, path)
    full = dict(plan_launches=0, decode_launches=0, merge_launches=0, single_pass_launches=0,
                append_launches=0)
    full.update(expect)
    assert api.pkv_get_counters() == full


def test_decode_merge_entry_point_ignores_the_cfg_field():
    """pkv_decode_merge always merges on its tail (after pkv_plan on the
    workqueue), whatever cfg.merge says."""
    tr = T.make_trace(3)
    q = T.gen_q(tr)
    k, v = T.gen_kv(tr)
    d = upload(tr, q, k, v)
    shape = shape_of(tr)
    cfg = api.make_cfg(WORKQUEUE, tr.split_tokens, 0, 0, SEPARATE)
    ws = torch.zeros(api.pkv_plan_workspace_size(shape, cfg), dtype=torch.uint8, device="cuda")
    part = torch.empty(api.pkv_partials_size(shape, cfg) // 4, dtype=torch.float32, device="cuda")
    o = torch.full((tr.B, tr.Hq, tr.d), float("nan"), dtype=torch.float16, device="cuda")
    lse = torch.full((tr.B, tr.Hq), float("nan"), dtype=torch.float32, device="cuda")
    api.pkv_plan(shape, cfg, d["sl"], ws)
    api.pkv_decode_merge(shape, cfg, ws, d["q"], d["k"], d["v"], d["bt"], d["sl"], part, o, lse)
    torch.cuda.synchronize()
    check_error_free(ws)
    assert not any(header_counters(ws).values())
    oref, lref = oracle_out(tr, q, k, v)
    close(o, oref)
    close_lse(lse, lref)


def test_paged_decoder_switches_shapes_on_one_workspace():
    """PagedDecoder with the fused merge zeroes its workspace when the
    configuration changes: the counters' place moves with the shape."""
    dec = api.PagedDecoder(merge=FUSED)
    runs = []
    for lens, path in (([4000, 9000, 1, 0, 7000, 300, 5000, 8000], WORKQUEUE),
                       ([20000], BUCKETED), ([700, 2000, 4100], WORKQUEUE),
                       ([4000, 9000, 1, 0, 7000, 300, 5000, 8000], WORKQUEUE)):
        tr, q, k, v = case(lens, Hq=32, Hkv=8, C=1024, seed=len(lens))
        d = upload(tr, q, k, v)
        o, lse = dec.step(d["q"], d["k"], d["v"], d["bt"], d["sl"], tr.n_max, path=path,
                          split_tokens=1024)
        torch.cuda.synchronize()
        check_error_free(dec.workspace(d["q"].device))
        oref, lref = oracle_out(tr, q, k, v)
        close(o, oref)
        close_lse(lse, lref)
        runs.append(path)
    assert dec.merge == FUSED and len(runs) == 4


# ------------------------------------------------------------------ bounded waits

def test_fused_timeout_reports_and_the_next_step_is_correct():
    """A starved CTA (test hook) times out, still arrives at the grid-wide
    barrier so that no other CTA waits for it, and the launch reports
    PKV_ETIMEOUT; the barrier's count is back at zero and the next fused step
    on the same workspace is correct."""
    tr = T.make_trace(1)
    q = T.gen_q(tr)
    k, v = T.gen_kv(tr)
    d = upload(tr, q, k, v)
    L = _lib.load()
    assert L.pkv_test_starve_next_decodes(1) == 0
    try:
        o, lse, ws, _ = run_path(tr, d, BUCKETED, merge=FUSED)
    finally:
        L.pkv_test_starve_next_decodes(0)
    st, msg = api.pkv_get_error(ws)
    assert st == _lib.PKV_ETIMEOUT, msg
    assert header_counters(ws)["bar_count"] == 0
    o, lse, ws, _ = fused(tr, d, BUCKETED, ws=ws)
    oref, lref = oracle_out(tr, q, k, v)
    close(o, oref)
    close_lse(lse, lref)
