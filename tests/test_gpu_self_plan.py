"""GPU parity of the self-planning workqueue decode (PKV_PLAN_IN_DECODE).

"PersistentKV: Page-Aware Decode Scheduling for Long-Context LLM Serving on
Commodity GPUs", technical summary, Methodology 1, "Row-local bounds" and
"Compact workqueue": the plan (n_i = ceil(N*_i / C), offsets, the compact task
list) is the same whether the plan kernel builds it or the decode kernel does;
here every CTA of the decode derives its tasks from the lengths and the launch
writes the plan into the workspace.  Checked against the oracle: the plan
bit-exactly, outputs within |x - y| <= 3e-3 + 1e-2 |y|, and bit-identical to
the two-launch (plan kernel) step.
"""
import numpy as np
import pytest
import torch

import oracle
from plan_order import balance_order
import pkv_traces as T
from paged_kv_gqa_09_gb300 import _lib, api

from gpu_util import (check_error_free, close, close_lse, dev, header_counters, oracle_out, read_plan,
                      run_path, shape_of, upload)

pytestmark = pytest.mark.gpu

WORKQUEUE = _lib.PKV_PATH_WORKQUEUE
IN_DECODE, SEPARATE = _lib.PKV_PLAN_IN_DECODE, _lib.PKV_PLAN_SEPARATE


@pytest.fixture(scope="module", autouse=True)
def _lib_loaded():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_gqa_09_gb300 import build
    build.build()
    _lib.load()


def expected_order(want, lens, C):
    """The balance order (plan_order.py) of the canonical list `want`."""
    return want[balance_order(want, lens, C)] if len(want) else want


def check_plan(ws, tr, C):
    count, off, tasks, h, ordered = read_plan(ws, tr.B, with_order=True)
    want, want_off = oracle.plan_compact(tr.seq_lens, tr.Hq, tr.Hkv, C)
    assert count == want.shape[0]
    assert h[5] == want_off[-1] and h[6] == 0      # state rows, no overflow
    assert np.array_equal(off, want_off)
    assert np.array_equal(tasks, want)
    assert np.array_equal(ordered, expected_order(want, tr.seq_lens, C))
    lens = np.clip(tr.seq_lens, 0, None)
    sb = np.concatenate([[0], np.cumsum(lens % C != 0)])[:-1]
    t0 = (64 + 4 * (tr.B + 1) + 15) // 16 * 16
    got_sb = ws[ws.numel() - 4 * tr.B:].view(torch.int32).cpu().numpy()
    assert t0 < ws.numel() and np.array_equal(got_sb, sb)


@pytest.mark.parametrize("lens,C,Hq,Hkv", [
    ([1, 0, 1024, 1025, 17], 256, 32, 8),
    ([0, 0, 0, 5], 64, 8, 2),
    ([5000, 3, 64, 64, 20000, 7, 0, 2048], 1024, 32, 8),
    (list(range(1, 300, 7)), 16, 16, 2),
    ([64] * 40 + [65], 64, 8, 8),
    ([777], 256, 8, 1),
])
def test_plan_and_outputs_match_oracle(lens, C, Hq, Hkv):
    tr = T.custom_trace(lens, Hq, Hkv, 128, 16, C, seed=5, extra_cols=2)
    q = T.gen_q(tr)
    k, v = T.gen_kv(tr, poison_unused=True)
    d = upload(tr, q, k, v)
    api.pkv_reset_counters()
    o, lse, ws, _ = run_path(tr, d, WORKQUEUE, C=C, plan=IN_DECODE)
    check_error_free(ws)
    c = api.pkv_get_counters()
    assert (c["plan_launches"], c["decode_launches"], c["merge_launches"]) == (0, 1, 1)
    check_plan(ws, tr, C)
    assert header_counters(ws) == {"next_task": 0, "done_ctas": 0, "bar_count": 0}
    oref, lref = oracle_out(tr, q, k, v)
    close(o, oref)
    close_lse(lse, lref)


@pytest.mark.parametrize("cfg_id,B", [(1, None), (2, None), (3, None), (4, 4), (4, 8)])
def test_workloads_match_oracle_and_the_plan_kernel_step(cfg_id, B):
    tr = T.make_trace(cfg_id) if B is None else T.make_trace(cfg_id, B=B)
    q = T.gen_q(tr)
    k, v = T.gen_kv(tr)
    d = upload(tr, q, k, v)
    o, lse, ws, _ = run_path(tr, d, WORKQUEUE, plan=IN_DECODE)
    check_error_free(ws)
    check_plan(ws, tr, tr.split_tokens)
    oref, lref = oracle_out(tr, q, k, v)
    close(o, oref)
    close_lse(lse, lref)
    # the same tasks, each computed by one CTA in the same way: bit-identical
    o2, lse2, ws2, _ = run_path(tr, d, WORKQUEUE, plan=SEPARATE)
    check_error_free(ws2)
    assert torch.equal(o, o2) and torch.equal(lse, lse2)


@pytest.mark.parametrize("B", [_lib.PKV_SELF_PLAN_MAX_B, _lib.PKV_SELF_PLAN_MAX_B + 1])
def test_largest_self_planned_batch_and_the_one_above(B):
    """B = 512 plans in the decode; B = 513 takes the plan kernel (same results)."""
    rng = np.random.default_rng(11)
    lens = rng.integers(0, 700, B)
    lens[rng.choice(B, 20, replace=False)] = 0
    tr = T.custom_trace(lens.tolist(), 8, 2, 64, 16, 128, seed=9)
    q = T.gen_q(tr)
    k, v = T.gen_kv(tr)
    d = upload(tr, q, k, v)
    api.pkv_reset_counters()
    o, lse, ws, _ = run_path(tr, d, WORKQUEUE, plan=IN_DECODE)
    check_error_free(ws)
    assert api.pkv_get_counters()["plan_launches"] == (0 if B <= _lib.PKV_SELF_PLAN_MAX_B else 1)
    check_plan(ws, tr, 128)
    oref, lref = oracle_out(tr, q, k, v)
    close(o, oref)
    close_lse(lse, lref)


def test_capacity_overflow_is_reported():
    """Too many tasks for the workspace: nothing is decoded, PKV_ECAPACITY,
    header overflow set, and the merge writes NaN (outputs start at zero)."""
    tr = T.custom_trace([300, 700], 8, 2, 128, 16, 64)
    shape = shape_of(tr)
    cfg = api.make_cfg(WORKQUEUE, 64, 0, 5, _lib.PKV_MERGE_SEPARATE, IN_DECODE)
    d = upload(tr, T.gen_q(tr), *T.gen_kv(tr))
    ws = torch.zeros(api.pkv_plan_workspace_size(shape, cfg), dtype=torch.uint8, device="cuda")
    part = torch.zeros(api.pkv_partials_size(shape, cfg) // 4, dtype=torch.float32, device="cuda")
    o = torch.zeros((tr.B, tr.Hq, tr.d), dtype=torch.float16, device="cuda")
    lse = torch.zeros((tr.B, tr.Hq), dtype=torch.float32, device="cuda")
    api.pkv_decode_step(shape, cfg, ws, d["q"], d["k"], d["v"], d["bt"], d["sl"], part, o, lse)
    torch.cuda.synchronize()
    h = ws[:64].view(torch.int32).cpu().numpy()
    assert h[4] == 0 and h[6] == 1
    st, msg = api.pkv_get_error(ws)
    assert st == _lib.PKV_ECAPACITY, msg
    assert torch.isnan(o.float()).all() and torch.isnan(lse).all()
    assert torch.count_nonzero(part) == 0   # no state written


@pytest.mark.parametrize("bad", [-5, 10 ** 6])
def test_bad_lengths_are_treated_as_the_plan_kernel_treats_them(bad):
    """A negative length reads as 0 and one beyond the table as the table's
    reach; either is reported.  The self-planned step and the plan-kernel step
    then agree bit for bit."""
    tr = T.custom_trace([100, 200, 300], 8, 2, 128, 16, 64)
    q = T.gen_q(tr)
    k, v = T.gen_kv(tr)
    sl = tr.seq_lens.copy()
    sl[1] = bad
    d = upload(tr, q, k, v)
    d["sl"] = dev(sl)
    outs = []
    for plan in (IN_DECODE, SEPARATE):
        o, lse, ws, _ = run_path(tr, d, WORKQUEUE, plan=plan)
        st, msg = api.pkv_get_error(ws)
        assert st == _lib.PKV_EDEVICE, msg
        outs.append((o, lse))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


def test_chained_graph_steps_match_oracle():
    """Four PDL-chained steps in one CUDA graph, replayed three times on one
    workspace: each step's decode plans for itself, and the claim counters it
    leaves behind start the next one from zero."""
    tr = T.make_trace(3)
    q = T.gen_q(tr)
    k, v = T.gen_kv(tr)
    d = upload(tr, q, k, v)
    shape = shape_of(tr)
    cfg = api.make_cfg(WORKQUEUE, tr.split_tokens, 0, 0, _lib.PKV_MERGE_SEPARATE, IN_DECODE)
    ws = torch.zeros(api.pkv_plan_workspace_size(shape, cfg), dtype=torch.uint8, device="cuda")
    part = torch.empty(api.pkv_partials_size(shape, cfg) // 4, dtype=torch.float32, device="cuda")
    o = torch.empty((tr.B, tr.Hq, tr.d), dtype=torch.float16, device="cuda")
    lse = torch.empty((tr.B, tr.Hq), dtype=torch.float32, device="cuda")
    k2, v2 = d["k"].clone(), d["v"].clone()
    st = torch.cuda.Stream()

    def steps():
        for r in range(4):
            kk, vv = (d["k"], d["v"]) if r % 2 == 0 else (k2, v2)
            api.pkv_decode_step(shape, cfg, ws, d["q"], kk, vv, d["bt"], d["sl"], part, o, lse,
                                stream=st)

    api.pkv_reset_counters()
    with torch.cuda.stream(st):
        steps()
        st.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            steps()
    c = api.pkv_get_counters()
    assert c["plan_launches"] == 0 and c["decode_launches"] == c["merge_launches"] == 8
    oref, lref = oracle_out(tr, q, k, v)
    for _ in range(3):
        with torch.cuda.stream(st):
            o.fill_(float("nan"))
            g.replay()
        st.synchronize()
        check_error_free(ws)
        close(o, oref)
        close_lse(lse, lref)
    check_plan(ws, tr, tr.split_tokens)


def test_host_loop_graph_and_paged_decoder():
    tr = T.make_trace(4, B=8)
    q = T.gen_q(tr)
    k, v = T.gen_kv(tr)
    d = upload(tr, q, k, v)
    oref, lref = oracle_out(tr, q, k, v)
    dec = api.PagedDecoder(plan=IN_DECODE)
    o, lse = dec.step(d["q"], d["k"], d["v"], d["bt"], d["sl"], tr.n_max, path=WORKQUEUE)
    torch.cuda.synchronize()
    check_error_free(dec.workspace(d["q"].device))
    close(o, oref)
    close_lse(lse, lref)
    loop = api.HostDecodeLoop(d["k"], d["v"], tr.B, tr.Hq, tr.bt_stride, tr.n_max, path=WORKQUEUE,
                              split_tokens=tr.split_tokens, plan=IN_DECODE)
    loop.h_q.copy_(torch.from_numpy(q))
    loop.h_bt.copy_(torch.from_numpy(tr.block_table))
    loop.h_sl.copy_(torch.from_numpy(tr.seq_lens))
    st = torch.cuda.Stream()
    loop.capture(st)
    for _ in range(2):
        ho, hl = loop.step_graph()
        check_error_free(loop.ws)
        close(ho, oref)
        close_lse(hl, lref)


def test_random_batches_match_oracle():
    """Seeded random batches -- B up to 512, page sizes 8..64, C = 1..16 pages,
    Hkv 1..8, G 1..8, d 64 or 128, lengths from 0 to 20 splits with empty rows
    mixed in -- through both plan modes: the plan (header, offsets, canonical
    and balance-ordered lists) bit-exact against the oracle and the definition
    of the order, the outputs within tolerance."""
    rng = np.random.default_rng(20261203)
    for case in range(24):
        B = int(rng.choice([1, 3, 8, 31, 33, 64, 200, 512]))
        P = int(rng.choice([8, 16, 64]))
        C = P * int(rng.choice([1, 2, 4, 16]))
        Hkv, G, d = int(rng.choice([1, 2, 8])), int(rng.choice([1, 4, 8])), int(rng.choice([64, 128]))
        maxlen = int(rng.choice([C, 4 * C, 20 * C])) if B < 200 else min(int(rng.choice([C, 4 * C])), 1024)
        lens = rng.integers(0, min(maxlen, 16384) + 1, size=B)
        lens[rng.random(B) < 0.1] = 0
        tr = T.custom_trace(lens.tolist(), Hkv * G, Hkv, d, P, C, seed=case, extra_cols=1)
        q = T.gen_q(tr)
        k, v = T.gen_kv(tr, poison_unused=True)
        d_in = upload(tr, q, k, v)
        oref, lref = oracle_out(tr, q, k, v)
        want, want_off = oracle.plan_compact(tr.seq_lens, tr.Hq, tr.Hkv, C)
        for plan in (IN_DECODE, SEPARATE):
            o, lse, ws, _ = run_path(tr, d_in, WORKQUEUE, plan=plan)
            check_error_free(ws)
            count, off, tasks, h, ordered = read_plan(ws, tr.B, with_order=True)
            assert count == want.shape[0], (case, plan)
            assert np.array_equal(off, want_off) and np.array_equal(tasks, want), (case, plan)
            assert np.array_equal(ordered, expected_order(want, tr.seq_lens, C)), (case, plan)
            close(o, oref, f"case {case}, plan mode {plan}")
            close_lse(lse, lref)
