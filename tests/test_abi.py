"""CPU tests of libpkv's C ABI: symbols, argument validation, policy and the
host-side step model.  No call here launches a kernel."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import pkv_traces as T
from paged_kv_gqa_09_gb300 import _lib, api
from paged_kv_gqa_09_gb300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    build_mod.build()
    return _lib.load()


def header_symbols():
    src = open(os.path.join(ROOT, "include", "pkv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(L):
    declared = header_symbols()
    assert len(declared) >= 16
    for name in declared:
        assert hasattr(L, name), name
    assert sorted(_lib.EXPORTS) == declared
    assert L.pkv_version() == 2


def shape(**kw):
    base = dict(B=2, Hq=8, Hkv=2, d=128, page_size=16, num_pages=64, bt_stride=16, scale=0.088)
    base.update(kw)
    return _lib.Shape(*[base[k] for k, _ in _lib.Shape._fields_])


def cfg(path=_lib.PKV_PATH_WORKQUEUE, C=256, bucket=0, max_tasks=0, merge=0, plan=0):
    return _lib.PlanCfg(path, C, bucket, max_tasks, merge, plan)


FAKE = 1 << 20  # 16-byte aligned, never dereferenced: validation fails first


@pytest.mark.parametrize("kw,status", [
    (dict(Hq=6, Hkv=4), _lib.PKV_EINVAL),
    (dict(d=96), _lib.PKV_EUNSUPPORTED),
    (dict(Hq=32, Hkv=2), _lib.PKV_EUNSUPPORTED),      # G = 16
    (dict(page_size=24), _lib.PKV_EUNSUPPORTED),
    (dict(page_size=4), _lib.PKV_EUNSUPPORTED),
    (dict(page_size=512), _lib.PKV_EUNSUPPORTED),
    (dict(B=-1), _lib.PKV_EINVAL),
    (dict(num_pages=0), _lib.PKV_EINVAL),
    (dict(scale=float("nan")), _lib.PKV_EINVAL),
])
def test_bad_shapes_are_rejected(L, kw, status):
    s, c = shape(**kw), cfg()
    rc = L.pkv_plan(ctypes.byref(s), ctypes.byref(c), FAKE, FAKE, None)
    assert rc == status, _lib.last_error()
    assert _lib.last_error()
    assert L.pkv_plan_workspace_size(ctypes.byref(s), ctypes.byref(c)) == 0


def test_bad_cfg_and_pointers_are_rejected(L):
    s = shape()
    assert L.pkv_plan(ctypes.byref(s), ctypes.byref(cfg(C=100)), FAKE, FAKE, None) == _lib.PKV_EINVAL
    assert L.pkv_plan(ctypes.byref(s), ctypes.byref(cfg(path=7)), FAKE, FAKE, None) == _lib.PKV_EINVAL
    c = cfg()
    assert L.pkv_plan(ctypes.byref(s), ctypes.byref(c), None, FAKE, None) == _lib.PKV_EINVAL
    assert "seq_lens" in _lib.last_error()
    assert L.pkv_plan(ctypes.byref(s), ctypes.byref(c), FAKE + 4, FAKE, None) == _lib.PKV_EINVAL
    assert "aligned" in _lib.last_error()
    args = [FAKE] * 7
    args[3] = FAKE + 2  # k_cache misaligned
    assert L.pkv_decode(ctypes.byref(s), ctypes.byref(c), *args, None) == _lib.PKV_EINVAL
    assert L.pkv_decode(ctypes.byref(s), ctypes.byref(cfg(path=2)), *([FAKE] * 7), None) == _lib.PKV_EINVAL
    assert L.pkv_merge(ctypes.byref(s), ctypes.byref(c), FAKE, FAKE, FAKE, None, None, None) == _lib.PKV_EINVAL
    assert L.pkv_single_pass(ctypes.byref(s), FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, None,
                             None) == _lib.PKV_EINVAL
    assert L.pkv_append(ctypes.byref(s), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None) == _lib.PKV_EINVAL
    assert L.pkv_plan(None, ctypes.byref(c), FAKE, FAKE, None) == _lib.PKV_EINVAL
    assert L.pkv_get_error(None, None) == _lib.PKV_EINVAL


def test_empty_batch_is_a_no_op(L):
    """B = 0: every launching call returns PKV_OK without looking at its
    pointers (NULL here) or the GPU."""
    s = shape(B=0)
    for path in (_lib.PKV_PATH_BUCKETED_SPLIT, _lib.PKV_PATH_WORKQUEUE, _lib.PKV_PATH_SINGLE_PASS):
        for merge in (0, 1):
            c = cfg(path=path, merge=merge)
            args = (ctypes.byref(s), ctypes.byref(c))
            assert L.pkv_decode_step(*args, None, None, None, None, None, None, None, None, None,
                                     None) == 0
            assert L.pkv_decode_step_noalloc(*args, None, None, None, None, None, None, None,
                                             None) == 0
            assert L.pkv_decode_step_host(*args, None, None, None, None, None, None, None, None,
                                          None, None, None, None, None, None, None) == 0
            assert L.pkv_append_decode_step_host(*args, *([None] * 19)) == 0
            if path != _lib.PKV_PATH_SINGLE_PASS:
                assert L.pkv_plan(*args, None, None, None) == 0
                assert L.pkv_decode(*args, None, None, None, None, None, None, None, None) == 0
                assert L.pkv_decode_merge(*args, None, None, None, None, None, None, None, None,
                                          None, None) == 0
                assert L.pkv_merge(*args, None, None, None, None, None, None) == 0
    assert L.pkv_single_pass(ctypes.byref(s), None, None, None, None, None, None, None, None,
                             None) == 0
    assert L.pkv_append(ctypes.byref(s), None, None, None, None, None, None, None, None) == 0
    wq = cfg()
    assert L.pkv_append_plan(ctypes.byref(s), ctypes.byref(wq), *([None] * 10)) == 0


def test_unknown_merge_mode_is_rejected(L):
    s = shape()
    for bad in (-1, 2):
        c = cfg(merge=bad)
        assert L.pkv_plan_workspace_size(ctypes.byref(s), ctypes.byref(c)) == 0
        assert L.pkv_decode_merge(ctypes.byref(s), ctypes.byref(c), FAKE, FAKE, FAKE, FAKE, FAKE,
                                  FAKE, FAKE, FAKE, None, None) == _lib.PKV_EINVAL
    ok = cfg(merge=_lib.PKV_MERGE_FUSED)
    assert L.pkv_plan_workspace_size(ctypes.byref(s), ctypes.byref(ok)) > 0


def test_unknown_plan_mode_is_rejected(L):
    s = shape()
    for bad in (-1, 2):
        c = cfg(plan=bad)
        assert L.pkv_plan_workspace_size(ctypes.byref(s), ctypes.byref(c)) == 0
        assert L.pkv_decode_step(ctypes.byref(s), ctypes.byref(c), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                                 FAKE, FAKE, None, None) == _lib.PKV_EINVAL
    for path in (_lib.PKV_PATH_WORKQUEUE, _lib.PKV_PATH_BUCKETED_SPLIT):
        ok = cfg(path=path, plan=_lib.PKV_PLAN_IN_DECODE)
        # the workspace is the same whichever kernel builds the plan
        same = cfg(path=path)
        assert (L.pkv_plan_workspace_size(ctypes.byref(s), ctypes.byref(ok)) ==
                L.pkv_plan_workspace_size(ctypes.byref(s), ctypes.byref(same)) > 0)


def test_state_slots_beyond_int32_are_refused(L):
    """State slots are int32 in the task records and the kernels: a split
    configuration whose partial-state buffer would hold more than 2^31 - 1 slots
    is refused before any launch (it could only wrap to a negative index)."""
    s = shape()
    wq = cfg(max_tasks=1 << 30)                      # 2^30 tasks x G=4 slots
    rect = cfg(path=_lib.PKV_PATH_BUCKETED_SPLIT, C=16, bucket=0x7fffffff)  # 2 x 2^27 x 8 slots
    for c in (wq, rect):
        assert L.pkv_decode(ctypes.byref(s), ctypes.byref(c), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                            FAKE, None) == _lib.PKV_EUNSUPPORTED
        assert L.pkv_merge(ctypes.byref(s), ctypes.byref(c), FAKE, FAKE, FAKE, FAKE, FAKE,
                           None) == _lib.PKV_EUNSUPPORTED
        assert "int32" in _lib.last_error()
    assert L.pkv_plan(ctypes.byref(s), ctypes.byref(wq), FAKE, FAKE, None) == _lib.PKV_EUNSUPPORTED


def test_plan_is_a_noop_off_the_workqueue(L):
    s = shape()
    for p in (_lib.PKV_PATH_BUCKETED_SPLIT, _lib.PKV_PATH_SINGLE_PASS):
        assert L.pkv_plan(ctypes.byref(s), ctypes.byref(cfg(path=p)), FAKE, FAKE, None) == 0


def test_workspace_and_partial_sizes(L):
    s = shape(B=3, Hq=32, Hkv=8, d=128, bt_stride=64, page_size=16)
    # workqueue: header + offsets (aligned) + 16 B per task; default capacity Hkv*B*ceil(1024/C)
    c = cfg(C=256)
    tasks_off = (64 + 4 * 4 + 15) // 16 * 16
    cap = 8 * 3 * 4
    # canonical list, its balance-ordered copy, one int per row
    assert L.pkv_plan_workspace_size(ctypes.byref(s), ctypes.byref(c)) == tasks_off + 32 * cap + 4 * 3
    assert L.pkv_partials_size(ctypes.byref(s), ctypes.byref(c)) == cap * 4 * (128 + 2) * 4
    c = cfg(C=256, max_tasks=10)
    assert L.pkv_partials_size(ctypes.byref(s), ctypes.byref(c)) == 10 * 4 * 130 * 4
    r = cfg(path=_lib.PKV_PATH_BUCKETED_SPLIT, C=256, bucket=600)
    assert L.pkv_plan_workspace_size(ctypes.byref(s), ctypes.byref(r)) == tasks_off
    assert L.pkv_partials_size(ctypes.byref(s), ctypes.byref(r)) == 3 * 3 * 32 * 130 * 4
    one = cfg(path=_lib.PKV_PATH_SINGLE_PASS)
    assert L.pkv_plan_workspace_size(ctypes.byref(s), ctypes.byref(one)) == tasks_off
    assert L.pkv_partials_size(ctypes.byref(s), ctypes.byref(one)) == 0


def test_policy_routes_by_batch_and_length(L):
    """Methodology 2: by (B, N_max) to the bucketed split, the workqueue or the
    single-kernel route, with calibrated cut-offs."""
    P = _lib
    custom = _lib.PolicyCfg(1000, 1, 2000, 8, 512, 256)
    assert api.pkv_policy(1, 1000, custom) == (P.PKV_PATH_BUCKETED_SPLIT, 256)
    assert api.pkv_policy(1, 999, custom)[0] == P.PKV_PATH_SINGLE_PASS
    assert api.pkv_policy(9, 2000, custom) == (P.PKV_PATH_WORKQUEUE, 512)
    assert api.pkv_policy(9, 1999, custom)[0] == P.PKV_PATH_SINGLE_PASS
    assert api.pkv_policy(4, 10 ** 6, custom)[0] == P.PKV_PATH_SINGLE_PASS   # the pages' B=4 gap
    assert api.pkv_policy(0, 10 ** 6, custom)[0] == P.PKV_PATH_SINGLE_PASS   # empty batch
    d = api.pkv_policy_default()
    assert d.split_tokens > 0 and d.bucketed_split_tokens > 0
    path, C = api.pkv_policy(1, d.bucketed_min_tokens)
    assert path == P.PKV_PATH_BUCKETED_SPLIT and C == d.bucketed_split_tokens
    assert api.pkv_policy(64, 65536)[0] == P.PKV_PATH_WORKQUEUE
    with pytest.raises(_lib.PkvError):
        api.pkv_policy(-1, 5)
    with pytest.raises(_lib.PkvError):
        api.pkv_policy(1, 5, _lib.PolicyCfg(0, 1, 0, 8, 0, 256))
    # the workqueue's split size doubling with the batch, up to its largest
    grow = _lib.PolicyCfg(1000, 1, 2000, 8, 512, 256, 4096, 256)
    assert api.pkv_policy(9, 2000, grow) == (P.PKV_PATH_WORKQUEUE, 512)      # 9 x 4 pairs
    assert api.pkv_policy(64, 8192, grow) == (P.PKV_PATH_WORKQUEUE, 2048)    # 64 x 4 pairs
    assert api.pkv_policy(64, 8193, grow) == (P.PKV_PATH_WORKQUEUE, 4096)
    assert api.pkv_policy(64, 10 ** 7, grow) == (P.PKV_PATH_WORKQUEUE, 4096)  # capped
    assert api.pkv_policy(1, 10 ** 6, grow)[1] == 256                         # bucketed C unchanged
    with pytest.raises(_lib.PkvError):
        api.pkv_policy(9, 2000, _lib.PolicyCfg(1000, 1, 2000, 8, 512, 256, 4096, -1))
    keep = _lib.PolicyCfg(1000, 1, 2000, 8, 256, 256, 4096, 32, 16)   # the longest row keeps 16
    assert api.pkv_policy(8, 2903, keep) == (P.PKV_PATH_WORKQUEUE, 256)
    assert api.pkv_policy(64, 65536, keep) == (P.PKV_PATH_WORKQUEUE, 4096)
    with pytest.raises(_lib.PkvError):
        api.pkv_policy(9, 2000, _lib.PolicyCfg(1000, 1, 2000, 8, 512, 256, 4096, 32, -1))


@pytest.mark.parametrize("cfg_id", [1, 2, 3, 4, 5])
def test_step_model_matches_oracle_counters(L, cfg_id):
    tr = T.make_trace(cfg_id)
    s = _lib.Shape(tr.B, tr.Hq, tr.Hkv, tr.d, tr.page_size, tr.num_pages, tr.bt_stride, tr.scale)
    C = tr.split_tokens
    S_b = -(-tr.n_max // C)
    for path in (0, 1, 2, 3):
        got = api.pkv_step_model(path, s, C, tr.n_max, tr.seq_lens)
        want = oracle.counters(path, tr.seq_lens, tr.Hq, tr.Hkv, tr.d, C, S_b)
        assert got == vars(want), (path, got, vars(want))


def test_counters_start_at_zero_and_reset(L):
    api.pkv_reset_counters()
    assert set(api.pkv_get_counters().values()) == {0}


def test_learned_policy_matches_the_fitted_feature_map(L):
    """pkv_policy_learned (C) against the calibration script's feature map
    (Python) on the default GB300 model: same route on a grid of batches."""
    from paged_kv_gqa_09_gb300 import calibrate
    m = api.pkv_cost_model_default()
    assert m.n_routes == len(calibrate.routes()) == 11
    routes = [(m.route[r].path, m.route[r].split_tokens, np.array(m.route[r].w[:], np.float64))
              for r in range(m.n_routes)]
    assert {p for p, _, _ in routes} == {0, 1, 2}
    rng = np.random.default_rng(3)
    for _ in range(400):
        B = int(rng.integers(1, 129))
        n_max = int(rng.integers(1, 70000))
        n_sum = int(rng.integers(n_max, B * n_max + 1))
        f = calibrate.features(B, n_max, n_sum)
        t = [float(f @ w) for _, _, w in routes]
        best = int(np.argmin(t))
        if sorted(t)[1] - t[best] < 1e-4:   # a near tie: float32 weights may pick either
            continue
        got = api.pkv_policy_learned(B, n_max, n_sum)
        assert got == (routes[best][0], routes[best][1]), (B, n_max, n_sum)
    assert api.pkv_policy_learned(0, 100, 0)[0] == _lib.PKV_PATH_SINGLE_PASS
    assert api.pkv_policy_learned(4, 0, 0)[0] == _lib.PKV_PATH_SINGLE_PASS
    with pytest.raises(_lib.PkvError):
        api.pkv_policy_learned(-1, 5, 5)
    bad = api.pkv_cost_model_default()
    bad.n_routes = 0
    with pytest.raises(_lib.PkvError):
        api.pkv_policy_learned(1, 5, 5, bad)


def test_learned_policy_prefers_workqueue_for_ragged_and_split_for_b1(L):
    # B=1 long context -> a split path; B=64 uniform long -> not the bucketed grid
    p1, _ = api.pkv_policy_learned(1, 32768, 32768)
    assert p1 in (_lib.PKV_PATH_BUCKETED_SPLIT, _lib.PKV_PATH_WORKQUEUE)
    p2, _ = api.pkv_policy_learned(16, 32768, 16 * 900)       # one long row, the rest short
    assert p2 == _lib.PKV_PATH_WORKQUEUE


def test_host_append_step_checks_arguments_first(L):
    """pkv_append_decode_step_host refuses bad arguments before it copies or
    launches anything (so with no GPU it never reaches the device)."""
    s = shape()
    wq = cfg()
    args = [FAKE] * 19
    # host q missing
    a = list(args)
    a[2] = None
    assert L.pkv_append_decode_step_host(ctypes.byref(s), ctypes.byref(wq), *a) == _lib.PKV_EINVAL
    # a free list without its count
    a = list(args)
    a[11] = None
    assert L.pkv_append_decode_step_host(ctypes.byref(s), ctypes.byref(wq), *a) == _lib.PKV_EINVAL
    # a free list off the workqueue
    rect = cfg(path=_lib.PKV_PATH_BUCKETED_SPLIT)
    assert L.pkv_append_decode_step_host(ctypes.byref(s), ctypes.byref(rect), *args) == _lib.PKV_EINVAL
    assert "WORKQUEUE" in _lib.last_error()
    # an unaligned device pointer
    a = list(args)
    a[3] = FAKE + 8  # d_q
    assert L.pkv_append_decode_step_host(ctypes.byref(s), ctypes.byref(wq), *a) == _lib.PKV_EINVAL


def test_learned_route_of_the_decoder_needs_the_total_tokens(L):
    dec = api.PagedDecoder(learned=True)
    with pytest.raises(ValueError):
        dec.route(8, 32768)
    assert dec.route(8, 32768, 8 * 900) == api.pkv_policy_learned(8, 32768, 8 * 900)
    assert api.PagedDecoder().route(8, 32768) == api.pkv_policy(8, 32768)


def test_the_test_hook_needs_the_opt_in(L, monkeypatch):
    """pkv_test_starve_next_decodes is inert unless PKV_TEST_HOOKS=1."""
    monkeypatch.setenv("PKV_TEST_HOOKS", "0")
    assert L.pkv_test_starve_next_decodes(1) == _lib.PKV_EUNSUPPORTED
    assert "PKV_TEST_HOOKS" in _lib.last_error()
    monkeypatch.setenv("PKV_TEST_HOOKS", "1")
    assert L.pkv_test_starve_next_decodes(0) == 0


@pytest.mark.parametrize("lens", [[5, 5, 7, 0, 7, 9], [0, 0], [], [3], [9, 8, 7, 8, 9, 0, 1]])
def test_exact_length_groups(L, lens):
    """The exact-length-bucket scheme's launch groups, built by the library on
    the host: each distinct non-zero length once, ascending, with its rows in
    order; the rows without tokens last."""
    rows, start, glen = api.pkv_exact_length_groups(lens)
    want = sorted({n for n in lens if n > 0})
    assert glen.tolist() == want
    for g, n in enumerate(want):
        assert rows[start[g]:start[g + 1]].tolist() == [i for i, x in enumerate(lens) if x == n]
    assert rows[start[-1]:].tolist() == [i for i, x in enumerate(lens) if x == 0]
    assert len(rows) == len(lens)
    # the step model's exact-bucket launch count is two per group
    if lens:
        s = shape(B=len(lens), bt_stride=1)
        m = api.pkv_step_model(_lib.PATH_EXACT_BUCKETS, s, 16, 16, lens)
        assert m["attn_launches"] == 2 * len(want)


def test_exact_length_groups_rejects_bad_input(L):
    with pytest.raises(_lib.PkvError):
        api.pkv_exact_length_groups([3, -1])
