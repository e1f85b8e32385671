"""The step's KV write fused into the workqueue plan (pkv_append_plan), with
pages allocated on the device from a free list, over a multi-step decode
loop.  A host mirror applies the documented rule (rows whose new token starts
a page take free_pages[count - 1 - rank] in row order) to its own copy of the
cache, block table and lengths; the oracle runs on that mirror."""
import numpy as np
import pytest
import torch

import oracle
import pkv_traces as T
from paged_kv_gqa_09_gb300 import _lib, api

from gpu_util import check_error_free, close, close_lse, dev, shape_of

pytestmark = pytest.mark.gpu

P, HQ, HKV, D, C = 16, 8, 2, 128, 64


@pytest.fixture(scope="module", autouse=True)
def _lib_loaded():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_gqa_09_gb300 import build
    build.build()
    _lib.load()


def setup(lens0, steps, spare_pages):
    tr = T.custom_trace(lens0, HQ, HKV, D, P, C, extra_pages=spare_pages,
                        extra_cols=steps // P + 2, tag=700)
    k, v = T.gen_kv(tr)
    used = set(tr.block_table[tr.block_table >= 0].tolist())
    rng = np.random.default_rng([T.HELDOUT_SEED, 701])
    free = [int(x) for x in rng.permutation(tr.num_pages) if int(x) not in used]
    return tr, k, v, free


def mirror_append(tr, k_h, v_h, bt_h, lens_h, free_h, count, kn, vn):
    cap = tr.bt_stride * P
    need = [i for i in range(tr.B) if lens_h[i] % P == 0 and lens_h[i] < cap]
    for rank, i in enumerate(need):
        bt_h[i, lens_h[i] // P] = free_h[count - 1 - rank]
    count -= len(need)
    for i in range(tr.B):
        pg, sl = bt_h[i, lens_h[i] // P], lens_h[i] % P
        k_h[pg, sl], v_h[pg, sl] = kn[i], vn[i]
        lens_h[i] += 1
    return count


@pytest.mark.parametrize("merge,plan", [(_lib.PKV_MERGE_SEPARATE, _lib.PKV_PLAN_SEPARATE),
                                        (_lib.PKV_MERGE_FUSED, _lib.PKV_PLAN_SEPARATE),
                                        (_lib.PKV_MERGE_SEPARATE, _lib.PKV_PLAN_IN_DECODE),
                                        (_lib.PKV_MERGE_FUSED, _lib.PKV_PLAN_IN_DECODE)])
def test_fused_append_allocates_pages_and_matches_oracle(merge, plan):
    """With merge == FUSED the loop runs two launches per step: append + plan,
    then the decode with the merge on its tail (pkv_decode_merge).  With the
    separate merge and plan == IN_DECODE the append launch only appends and
    allocates, and the decode builds the plan."""
    steps = 40
    tr, k, v, free = setup([15, 16, 40, 0, 33, 64, 1], steps, spare_pages=30)
    k_h, v_h = k.copy(), v.copy()
    bt_h, lens_h, count = tr.block_table.copy(), tr.seq_lens.astype(np.int64).copy(), len(free)
    kd, vd, btd, sld = dev(k), dev(v), dev(tr.block_table), dev(tr.seq_lens)
    freed = dev(np.array(free, np.int32))
    cnt = torch.tensor([len(free)], dtype=torch.int32, device="cuda")
    shape = shape_of(tr)
    cfg = api.make_cfg(_lib.PKV_PATH_WORKQUEUE, C, 0, 0, merge, plan)
    deferred = merge == _lib.PKV_MERGE_SEPARATE and plan == _lib.PKV_PLAN_IN_DECODE
    ws = torch.zeros(api.pkv_plan_workspace_size(shape, cfg), dtype=torch.uint8, device="cuda")
    part = torch.empty(api.pkv_partials_size(shape, cfg) // 4, dtype=torch.float32, device="cuda")
    o = torch.empty((tr.B, HQ, D), dtype=torch.float16, device="cuda")
    lse = torch.empty((tr.B, HQ), dtype=torch.float32, device="cuda")
    api.pkv_reset_counters()
    for step in range(steps):
        kn, vn = T.gen_append_tokens(tr, step)
        q = T.gen_step_q(tr, step)
        count = mirror_append(tr, k_h, v_h, bt_h, lens_h, free, count, kn, vn)
        api.pkv_append_plan(shape, cfg, ws, dev(kn), dev(vn), btd, sld, kd, vd, freed, cnt)
        if merge == _lib.PKV_MERGE_FUSED:
            api.pkv_decode_merge(shape, cfg, ws, dev(q), kd, vd, btd, sld, part, o, lse)
        else:
            api.pkv_decode(shape, cfg, ws, dev(q), kd, vd, btd, sld, part)
            api.pkv_merge(shape, cfg, ws, sld, part, o, lse)
        if step in (0, 7, 23, steps - 1):
            torch.cuda.synchronize()
            check_error_free(ws)
            assert np.array_equal(btd.cpu().numpy(), bt_h)
            assert np.array_equal(sld.cpu().numpy(), lens_h)
            assert int(cnt.item()) == count
            oref, lref = oracle.attention(q, k_h, v_h, bt_h, lens_h.astype(np.int32), tr.scale)
            close(o, oref, f"o at step {step}")
            close_lse(lse, lref)
    c = api.pkv_get_counters()
    if deferred:
        assert c["plan_launches"] == 0 and c["append_launches"] == steps  # the decode plans
    else:
        assert c["plan_launches"] == steps and c["append_launches"] == 0  # append + plan in one
    assert c["decode_launches"] == steps
    assert c["merge_launches"] == (0 if merge == _lib.PKV_MERGE_FUSED else steps)
    used = bt_h[bt_h >= 0]
    assert len(np.unique(used)) == used.size                               # no page handed out twice


@pytest.mark.parametrize("plan", [_lib.PKV_PLAN_SEPARATE, _lib.PKV_PLAN_IN_DECODE])
def test_fused_append_reports_an_empty_free_list(plan):
    tr, k, v, free = setup([16, 32, 5], steps=4, spare_pages=1)
    kd, vd, btd, sld = dev(k), dev(v), dev(tr.block_table), dev(tr.seq_lens)
    freed = dev(np.array(free, np.int32))
    cnt = torch.tensor([len(free)], dtype=torch.int32, device="cuda")
    shape = shape_of(tr)
    cfg = api.make_cfg(_lib.PKV_PATH_WORKQUEUE, C, plan=plan)
    ws = torch.zeros(api.pkv_plan_workspace_size(shape, cfg), dtype=torch.uint8, device="cuda")
    kn, vn = T.gen_append_tokens(tr, 0)
    api.pkv_append_plan(shape, cfg, ws, dev(kn), dev(vn), btd, sld, kd, vd, freed, cnt)
    st, msg = api.pkv_get_error(ws)
    # rows 0 and 1 both start a page, only one page is free: row 0 gets it
    assert st == _lib.PKV_EDEVICE and "no free page" in msg, msg
    assert sld.cpu().numpy().tolist() == [17, 32, 6]
    assert int(cnt.item()) == 0
    assert btd.cpu().numpy()[0, 1] == free[len(free) - 1]


@pytest.mark.parametrize("page,dd,hkv,nrows", [(P, D, HKV, 300), (8, 64, 8, 300), (64, 128, 1, 300),
                                               (256, 64, 4, 300), (P, D, HKV, 512)])
def test_row_parallel_append_matches_the_plan_kernels_append(page, dd, hkv, nrows):
    """The append launch that leaves the plan to the decode (one CTA per row,
    each counting the rows before it that need a page) against the plan
    kernel's fused append (one CTA, a block scan), on two copies of the same
    state: 300 or 512 rows, most of them starting a page, and a free list of 160
    pages that runs out at the first step (rows left without a page keep
    asking).  Every step must leave the same block table, lengths, free count,
    error status and cache contents."""
    rng = np.random.default_rng([T.HELDOUT_SEED, 702, page, nrows])
    nmax = 40 if page <= 16 else 6
    lens0 = (rng.integers(0, nmax, nrows) * page
             + rng.integers(0, 3, nrows) * (rng.random(nrows) < 0.3)).tolist()
    tr = T.custom_trace(lens0, hkv * 2, hkv, dd, page, max(C, page), extra_pages=160, extra_cols=2,
                        tag=703)
    k, v = T.gen_kv(tr)
    used = set(tr.block_table[tr.block_table >= 0].tolist())
    free = np.array([x for x in rng.permutation(tr.num_pages) if int(x) not in used], np.int32)
    assert free.size == 160
    shape = shape_of(tr)
    states = []
    for plan in (_lib.PKV_PLAN_SEPARATE, _lib.PKV_PLAN_IN_DECODE):
        cfg = api.make_cfg(_lib.PKV_PATH_WORKQUEUE, max(C, page), plan=plan)
        ws = torch.zeros(api.pkv_plan_workspace_size(shape, cfg), dtype=torch.uint8, device="cuda")
        states.append(dict(cfg=cfg, ws=ws, k=dev(k), v=dev(v), bt=dev(tr.block_table),
                           sl=dev(tr.seq_lens), free=dev(free),
                           cnt=torch.tensor([free.size], dtype=torch.int32, device="cuda")))
    statuses = []
    for step in range(4):
        kn, vn = T.gen_append_tokens(tr, step)
        seen = []
        for s_ in states:
            api.pkv_append_plan(shape, s_["cfg"], s_["ws"], dev(kn), dev(vn), s_["bt"], s_["sl"],
                                s_["k"], s_["v"], s_["free"], s_["cnt"])
            st, _ = api.pkv_get_error(s_["ws"])
            seen.append((st, s_["bt"].cpu().numpy(), s_["sl"].cpu().numpy(), int(s_["cnt"].item())))
        a, b = seen
        assert a[0] == b[0], f"step {step}: status {a[0]} vs {b[0]}"
        assert np.array_equal(a[1], b[1]), f"step {step}: block tables differ"
        assert np.array_equal(a[2], b[2]), f"step {step}: lengths differ"
        assert a[3] == b[3], f"step {step}: free counts differ"
        assert torch.equal(states[0]["k"], states[1]["k"]) and torch.equal(states[0]["v"], states[1]["v"])
        statuses.append(a[0])
    assert int(states[0]["cnt"].item()) == 0
    assert statuses == [_lib.PKV_EDEVICE] * 4  # the exhausted list is reported every step
    # rows that got a page advanced; the others kept their length
    grew = states[1]["sl"].cpu().numpy() - np.asarray(lens0)
    assert grew.max() == 4 and grew.min() < 4


@pytest.mark.parametrize("path,alloc", [(_lib.PKV_PATH_WORKQUEUE, True),
                                        (_lib.PKV_PATH_BUCKETED_SPLIT, False)])
def test_host_loop_append_graph_matches_mirror(path, alloc):
    """HostDecodeLoop in append mode: each captured step appends the staged
    token (on the workqueue fused into the plan, with device page allocation)
    and decodes, reading q and the token from pinned memory and writing o / lse
    there; the block table and lengths stay on the device.  Checked against the
    host mirror of the append rule and the oracle."""
    steps = 24
    tr, k, v, free = setup([15, 16, 40, 0, 33, 64, 1], steps, spare_pages=30)
    k_h, v_h = k.copy(), v.copy()
    bt_h, lens_h, count = tr.block_table.copy(), tr.seq_lens.astype(np.int64).copy(), len(free)
    if not alloc:
        # the bucketed path writes into pages the table already names
        for i in range(tr.B):
            for col in range(tr.bt_stride):
                if bt_h[i, col] < 0:
                    bt_h[i, col] = free[count - 1]
                    count -= 1
    kd, vd = dev(k), dev(v)
    freed = dev(np.array(free, np.int32)) if alloc else None
    cnt = torch.tensor([count], dtype=torch.int32, device="cuda") if alloc else None
    loop = api.HostDecodeLoop(kd, vd, tr.B, HQ, tr.bt_stride, int(lens_h.max()) + steps + 1, path=path,
                              split_tokens=C, append=True, free_pages=freed, free_count=cnt)
    loop.set_state(torch.from_numpy(bt_h.astype(np.int32)), torch.from_numpy(lens_h.astype(np.int32)))
    st = torch.cuda.Stream()
    for step in range(steps):
        kn, vn = T.gen_append_tokens(tr, step)
        q = T.gen_step_q(tr, step)
        loop.h_q.copy_(torch.from_numpy(q))
        loop.h_kn.copy_(torch.from_numpy(kn))
        loop.h_vn.copy_(torch.from_numpy(vn))
        if alloc:
            count = mirror_append(tr, k_h, v_h, bt_h, lens_h, free, count, kn, vn)
        else:  # the page is already in the table
            for i in range(tr.B):
                pg, sl = bt_h[i, lens_h[i] // P], lens_h[i] % P
                k_h[pg, sl], v_h[pg, sl] = kn[i], vn[i]
                lens_h[i] += 1
        if step == 0:
            loop.capture(st)  # runs step 0 eagerly
            torch.cuda.synchronize()
            o, lse = loop.h_o, loop.h_lse
        else:
            o, lse = loop.step_graph()
        if step in (0, 1, 9, steps - 1):
            check_error_free(loop.ws)
            assert np.array_equal(loop.sl.cpu().numpy(), lens_h)
            if alloc:
                assert np.array_equal(loop.bt.cpu().numpy(), bt_h)
                assert int(cnt.item()) == count
            oref, lref = oracle.attention(q, k_h, v_h, bt_h, lens_h.astype(np.int32), tr.scale)
            close(o, oref, f"o at step {step}")
            close_lse(lse, lref)


@pytest.mark.parametrize("path,merge,alloc,pinned", [
    (_lib.PKV_PATH_WORKQUEUE, _lib.PKV_MERGE_SEPARATE, True, True),
    (_lib.PKV_PATH_WORKQUEUE, _lib.PKV_MERGE_SEPARATE, True, False),
    (_lib.PKV_PATH_WORKQUEUE, _lib.PKV_MERGE_FUSED, True, True),
    (_lib.PKV_PATH_WORKQUEUE, _lib.PKV_MERGE_SEPARATE, False, True),
    (_lib.PKV_PATH_BUCKETED_SPLIT, _lib.PKV_MERGE_SEPARATE, False, True),
    (_lib.PKV_PATH_BUCKETED_SPLIT, _lib.PKV_MERGE_SEPARATE, False, False),
    (_lib.PKV_PATH_SINGLE_PASS, _lib.PKV_MERGE_SEPARATE, False, True)])
def test_append_decode_step_host_matches_mirror(path, merge, alloc, pinned):
    """pkv_append_decode_step_host, one synchronized C call per step: q and
    the new token come from host memory, o / lse land in host memory, the
    block table and lengths advance on the device.  With page-locked host
    buffers q and the new token are read and o / lse written in place (the
    device staging for them stays untouched); with pageable ones every buffer
    goes through its device copy.  Checked against the host mirror of the append
    rule and the oracle."""
    steps = 20
    tr, k, v, free = setup([15, 16, 40, 0, 33, 64, 1], steps, spare_pages=30)
    k_h, v_h = k.copy(), v.copy()
    bt_h, lens_h, count = tr.block_table.copy(), tr.seq_lens.astype(np.int64).copy(), len(free)
    if not alloc:
        for i in range(tr.B):
            for col in range(tr.bt_stride):
                if bt_h[i, col] < 0:
                    bt_h[i, col] = free[count - 1]
                    count -= 1
    kd, vd = dev(k), dev(v)
    btd, sld = dev(bt_h.astype(np.int32)), dev(lens_h.astype(np.int32))
    freed = dev(np.array(free, np.int32)) if alloc else None
    cnt = torch.tensor([count], dtype=torch.int32, device="cuda") if alloc else None
    shape = shape_of(tr)
    n_max = int(lens_h.max()) + steps + 1
    cfg = api.make_cfg(path, C, n_max if path == _lib.PKV_PATH_BUCKETED_SPLIT else 0, 0, merge,
                       _lib.PKV_PLAN_IN_DECODE)  # the append launch plans; the field is ignored
    ws = torch.zeros(api.pkv_plan_workspace_size(shape, cfg), dtype=torch.uint8, device="cuda")
    npart = api.pkv_partials_size(shape, cfg)
    part = torch.empty(max(npart // 4, 4), dtype=torch.float32, device="cuda") if npart else None
    host = (lambda t: t.pin_memory()) if pinned else (lambda t: t)
    h_q = host(torch.empty((tr.B, HQ, D), dtype=torch.float16))
    h_kn = host(torch.empty((tr.B, HKV, D), dtype=torch.float16))
    h_vn = host(torch.empty((tr.B, HKV, D), dtype=torch.float16))
    h_o = host(torch.full((tr.B, HQ, D), float("nan"), dtype=torch.float16))
    h_lse = host(torch.full((tr.B, HQ), float("nan"), dtype=torch.float32))
    d_q = torch.full((tr.B, HQ, D), float("nan"), dtype=torch.float16, device="cuda")
    d_kn = torch.full((tr.B, HKV, D), float("nan"), dtype=torch.float16, device="cuda")
    d_vn = torch.full_like(d_kn, float("nan"))
    d_o = torch.full_like(d_q, float("nan"))
    d_lse = torch.full((tr.B, HQ), float("nan"), dtype=torch.float32, device="cuda")
    for step in range(steps):
        kn, vn = T.gen_append_tokens(tr, step)
        q = T.gen_step_q(tr, step)
        h_q.copy_(torch.from_numpy(q))
        h_kn.copy_(torch.from_numpy(kn))
        h_vn.copy_(torch.from_numpy(vn))
        if alloc:
            count = mirror_append(tr, k_h, v_h, bt_h, lens_h, free, count, kn, vn)
        else:
            for i in range(tr.B):
                pg, sl = bt_h[i, lens_h[i] // P], lens_h[i] % P
                k_h[pg, sl], v_h[pg, sl] = kn[i], vn[i]
                lens_h[i] += 1
        api.pkv_append_decode_step_host(shape, cfg, ws, part, h_q, d_q, h_kn, h_vn, d_kn, d_vn,
                                        btd, sld, kd, vd, d_o, h_o, d_lse, h_lse, freed, cnt)
        if step in (0, 1, 9, steps - 1):  # the call has synchronized: h_o is final
            check_error_free(ws)
            assert np.array_equal(sld.cpu().numpy(), lens_h)
            assert np.array_equal(btd.cpu().numpy(), bt_h)
            if alloc:
                assert int(cnt.item()) == count
            oref, lref = oracle.attention(q, k_h, v_h, bt_h, lens_h.astype(np.int32), tr.scale)
            close(h_o, oref, f"o at step {step}")
            close_lse(h_lse, lref)
            staged = [d_q, d_kn, d_vn, d_o, d_lse]
            if pinned:  # used in place: the device staging was never written
                assert all(torch.isnan(t.float()).all() for t in staged)
            else:       # copied through it
                assert torch.equal(d_o.cpu(), h_o) and torch.equal(d_kn.cpu(), h_kn)
                assert torch.equal(d_q.cpu(), h_q)


def test_append_decode_step_host_checks_before_enqueueing():
    """A free list on a path without device allocation is refused before any
    copy or launch: the lengths stay as they were."""
    tr, k, v, free = setup([15, 16], steps=4, spare_pages=4)
    kd, vd, btd, sld = dev(k), dev(v), dev(tr.block_table), dev(tr.seq_lens)
    freed = dev(np.array(free, np.int32))
    cnt = torch.tensor([len(free)], dtype=torch.int32, device="cuda")
    shape = shape_of(tr)
    cfg = api.make_cfg(_lib.PKV_PATH_BUCKETED_SPLIT, C, 64)
    ws = torch.zeros(api.pkv_plan_workspace_size(shape, cfg), dtype=torch.uint8, device="cuda")
    part = torch.empty(api.pkv_partials_size(shape, cfg) // 4, dtype=torch.float32, device="cuda")
    h_q = torch.zeros((tr.B, HQ, D), dtype=torch.float16).pin_memory()
    h_kn = torch.zeros((tr.B, HKV, D), dtype=torch.float16).pin_memory()
    d_q = torch.empty((tr.B, HQ, D), dtype=torch.float16, device="cuda")
    d_kn = torch.empty((tr.B, HKV, D), dtype=torch.float16, device="cuda")
    with pytest.raises(_lib.PkvError) as ei:
        api.pkv_append_decode_step_host(shape, cfg, ws, part, h_q, d_q, h_kn, h_kn, d_kn, d_kn,
                                        btd, sld, kd, vd, d_q.clone(), h_q.clone(), None, None,
                                        freed, cnt)
    assert ei.value.status == _lib.PKV_EINVAL
    torch.cuda.synchronize()
    assert sld.cpu().numpy().tolist() == [15, 16]
