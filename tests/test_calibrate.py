"""Host logic of the policy calibration (CPU only).

"PersistentKV: Page-Aware Decode Scheduling for Long-Context LLM Serving on
Commodity GPUs", technical summary, Methodology 2: a policy routes each decode
step by batch size B and longest context N_max, with thresholds calibrated on
one seed and checked on a held-out seed.  The calibration script searches those
thresholds in Python; the library applies them in C.  These tests pin the search
on a planted optimum, tie the Python rule to the C rule, and tie the frozen C
defaults to the committed calibration record.
"""
import ast
import itertools
import os
import re

import numpy as np
import pytest

from paged_kv_gqa_09_gb300 import _lib, api, calibrate

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PATH_OF = {"bucketed": _lib.PKV_PATH_BUCKETED_SPLIT, "workqueue": _lib.PKV_PATH_WORKQUEUE,
           "single": _lib.PKV_PATH_SINGLE_PASS}


@pytest.fixture(scope="module")
def L():
    try:
        return _lib.load()
    except _lib.PkvLibraryError as e:
        pytest.skip(f"libpkv.so not built: {e}")


def planted_results(params, rng):
    """A timing table over the calibration grid whose best route is, on every
    trace, the one the planted parameters choose; the others are 5-60% slower."""
    out = []
    for fam, B, n_max in itertools.product(calibrate.FAMILIES, calibrate.BATCHES, calibrate.NMAX):
        best = calibrate.choose(params, B, n_max)
        us = {f"{n}:{c}": float(rng.uniform(1.05, 1.6)) * 10.0 for n, c in calibrate.routes()}
        us[best] = 10.0
        out.append({"family": fam, "B": B, "n_max": n_max, "kv_bytes": 0, "us": us})
    return out


@pytest.mark.parametrize("planted", [
    (1024, 4, 2048, 1, 512, 512, 512, 0, 0),        # one fixed workqueue C
    (4096, 1, 8192, 8, 1024, 1024, 1024, 0, 0),     # the pages' own routing: B=1 split, B>=8 workqueue
    (0, 0, 256, 2, 2048, 128, 2048, 0, 0),          # no bucketed route at all
    (16384, 2, 1024, 1, 512, 1024, 4096, 256, 0),   # the workqueue's C growing with the batch
    (16384, 1, 1024, 1, 256, 1024, 4096, 32, 16),   # ... while the longest row keeps 16 splits
])
def test_fit_recovers_a_planted_policy(planted):
    rng = np.random.default_rng(11)
    res = planted_results(planted, rng)
    params, score = calibrate.fit(res)
    assert score == pytest.approx(1.0, abs=1e-12)
    assert calibrate.regret(params, res) == pytest.approx((1.0, 1.0), abs=1e-12)
    for r in res:   # parameters may differ where the grid cannot tell them apart; choices may not
        assert calibrate.choose(params, r["B"], r["n_max"]) == calibrate.choose(planted, r["B"], r["n_max"])


def test_regret_is_the_mean_and_max_of_chosen_over_best():
    params = (1024, 1, 1 << 30, 1 << 30, 512, 256, 512, 0, 0)  # B=1, N_max>=1024 -> bucketed:256, else single
    res = [{"B": 1, "n_max": 2048, "us": {"bucketed:256": 12.0, "single:0": 6.0}},
           {"B": 8, "n_max": 2048, "us": {"bucketed:256": 3.0, "single:0": 9.0}},
           {"B": 8, "n_max": 64, "us": {"bucketed:256": 9.0, "single:0": 9.0}}]
    mean, worst = calibrate.regret(params, res)
    assert worst == pytest.approx(3.0)
    assert mean == pytest.approx((2.0 + 3.0 + 1.0) / 3)


def test_python_rule_is_the_c_rule(L):
    """calibrate.choose (what the search scores) and pkv_policy (what runs) route
    every (B, N_max) alike, including both sides of every cut-off."""
    rng = np.random.default_rng(5)
    cfgs = [api.pkv_policy_default(), _lib.PolicyCfg(1000, 1, 2000, 8, 512, 256, 512, 0),
            _lib.PolicyCfg(0, 64, 0, 1, 256, 2048, 256, 0),
            _lib.PolicyCfg(1 << 30, 0, 1 << 30, 1 << 30, 1024, 1024, 1024, 0),
            _lib.PolicyCfg(16384, 2, 1024, 1, 512, 1024, 4096, 256),
            _lib.PolicyCfg(0, 0, 0, 1, 256, 1024, 2048, 16),
            _lib.PolicyCfg(16384, 1, 1024, 1, 256, 1024, 4096, 32, 16)]
    for c in cfgs:
        params = (c.bucketed_min_tokens, c.bucketed_max_batch, c.workqueue_min_tokens,
                  c.workqueue_min_batch, c.split_tokens, c.bucketed_split_tokens,
                  c.workqueue_max_split_tokens, c.workqueue_target_splits,
                  c.workqueue_min_long_splits)
        bs = {0, 1, 2, 3, 4, 5, 8, 9, 64, 65, c.bucketed_max_batch, c.bucketed_max_batch + 1,
              c.workqueue_min_batch, c.workqueue_min_batch - 1}
        ns = {0, 1, 256, 32768, c.bucketed_min_tokens, c.bucketed_min_tokens - 1,
              c.workqueue_min_tokens, c.workqueue_min_tokens - 1}
        ns |= {int(x) for x in rng.integers(0, 70000, size=20)}
        for B, n in itertools.product(bs, ns):
            if B < 0 or n < 0 or n > 2 ** 31 - 1:
                continue
            name, C = calibrate.choose(params, B, n).split(":")
            path, split = api.pkv_policy(B, n, c)
            assert path == PATH_OF[name], (params, B, n)
            if name != "single":
                assert split == int(C), (params, B, n)


def test_frozen_defaults_are_the_calibration_record(L):
    """The C defaults equal the parameters the committed calibration record says
    were frozen from the GB300 fit."""
    text = open(os.path.join(ROOT, "profiles", "policy_calibration.md")).read()
    m = re.search(r"Frozen in `pkv_policy_default`: (\{[^}]*\})", text)
    assert m, "calibration record lacks its frozen-parameter line"
    rec = ast.literal_eval(m.group(1))
    d = api.pkv_policy_default()
    assert {k: getattr(d, k) for k, _ in _lib.PolicyCfg._fields_} == rec


@pytest.mark.parametrize("family", calibrate.FAMILIES)
def test_length_families(family):
    rng = np.random.default_rng(7)
    for B, n_max in itertools.product(calibrate.BATCHES, calibrate.NMAX):
        n = calibrate.lengths(family, B, n_max, rng)
        assert n.shape == (B,) and n.dtype == np.int32
        assert n.max() == n_max and n.min() >= 1
        if family == "bucketed":
            assert (n == n_max).all()
        elif family == "uniform":
            assert n.min() >= max(1, n_max // 8)
        elif family == "bimodal" and B >= 2:
            assert (n <= max(1, n_max // 4)).sum() >= B // 2 - 1   # the argmax row may be reset
            assert (n >= 3 * n_max // 4).sum() >= B - B // 2
        else:
            assert n.min() >= min(16, n_max)


def test_workqueue_split_rule():
    """The workqueue's C doubles from its smallest value while the batch holds
    more than the target number of (row, split) pairs, up to its largest."""
    assert calibrate.wq_split(64, 65536, 512, 4096, 256) == 4096
    assert calibrate.wq_split(8, 32768, 512, 4096, 256) == 1024    # 8 x 32 = 256 pairs
    assert calibrate.wq_split(8, 32769, 512, 4096, 256) == 2048
    assert calibrate.wq_split(1, 1000, 512, 4096, 256) == 512
    assert calibrate.wq_split(64, 65536, 512, 4096, 0) == 512      # target 0: fixed C
    assert calibrate.wq_split(64, 10 ** 7, 256, 1024, 16) == 1024  # capped
    # the longest row keeps at least 16 splits: a ragged batch of short rows
    assert calibrate.wq_split(8, 2903, 256, 4096, 32, 16) == 256
    assert calibrate.wq_split(8, 8192, 256, 4096, 32, 16) == 512    # 8192 / 1024 would leave 8
    assert calibrate.wq_split(64, 65536, 256, 4096, 32, 16) == 4096


def test_near_ties_go_to_the_better_device_time():
    """Parameter sets within the calibration's resolution (TIE) of the best
    wall-clock regret are told apart by device-time regret; a set outside it
    never wins on device time alone, and without device times the wall clock
    decides."""
    best, near, far = 1.040, 1.040 * calibrate.TIE * 0.9999, 1.040 * calibrate.TIE * 1.001
    assert calibrate._pick([(best, 1.05, "a"), (near, 1.01, "b")])[2] == "b"
    assert calibrate._pick([(best, 1.05, "a"), (far, 1.00, "c")])[2] == "a"
    assert calibrate._pick([(near, None, "b"), (best, None, "a")])[2] == "a"
