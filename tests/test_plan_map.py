"""The balance-order map of the self-planning workqueue decode, on the CPU.

"PersistentKV: Page-Aware Decode Scheduling for Long-Context LLM Serving on
Commodity GPUs", technical summary, Methodology 1, "Compact workqueue": the
decode's CTAs take the plan's tasks in balance order (every full-length split,
by row, then split, then kv head -- the kv heads of one split side by side --
then the shorter last splits, longest length class first, by row and kv head;
`plan_order.py` states it).  When the decode builds the plan itself it maps a
position t to its task from two per-row prefix sums and the class-ordered list
of rows with a shorter split (plan_map.cuh, a host-and-device function).  Here
that map, compiled for the host, is compared with the oracle's canonical task
list reordered by the definition: the same record at every position, and each
position's index in the canonical list.
"""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
from plan_order import balance_order, short_rows

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "paged_kv_gqa_09_gb300", "csrc")


@pytest.fixture(scope="module")
def pmap(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    out = tmp_path_factory.mktemp("plan_map") / "libplan_map.so"
    subprocess.run([nvcc, "-O2", "-std=c++17", "-shared", "-Xcompiler", "-fPIC", "-I", CSRC, "-o", str(out),
                    os.path.join(ROOT, "tests", "plan_map_host.cu")], check=True)
    L = ctypes.CDLL(str(out))
    vp, ci = ctypes.c_void_p, ctypes.c_int
    L.plan_map_all.argtypes = [ci, vp, vp, vp, ci, ci, ci, ci, vp, vp]
    return L


def check(L, lens, C, Hkv, G):
    lens = np.asarray(lens, dtype=np.int32)
    B, Hq = lens.size, Hkv * G
    canon, off = oracle.plan_compact(lens, Hq, Hkv, C)
    T = canon.shape[0]
    order = balance_order(canon, lens, C)
    F = np.concatenate([[0], np.cumsum(lens // C)]).astype(np.int32)
    R = np.concatenate([[0], np.cumsum(lens % C != 0)]).astype(np.int32)
    S = np.zeros(max(B, 1), np.int16)
    S[:R[-1]] = short_rows(lens, C)
    rec = np.zeros((max(T, 1), 4), np.int32)
    lex = np.zeros(max(T, 1), np.int64)
    L.plan_map_all(B, F.ctypes.data, R.ctypes.data, S.ctypes.data, Hkv, Hq, G, T, rec.ctypes.data,
                   lex.ctypes.data)
    assert np.array_equal(rec[:T], canon[order]), (lens.tolist(), C)
    assert np.array_equal(lex[:T], order)
    assert np.array_equal(F + R, off)  # the map's prefix sums are the plan's offsets
    return T


@pytest.mark.parametrize("lens,C", [
    ([1, 0, 1024, 1025, 17], 256),
    ([0, 0, 0, 5], 64),
    ([64, 128, 192], 64),                  # no shorter splits
    ([1, 2, 3, 4, 5], 64),                 # only shorter splits
    ([0] * 30 + [70] + [0] * 30, 16),      # one row among empty ones
    ([777], 256),
    ([10, 250, 130, 70, 255, 31, 32, 224], 256),  # every length class, out of order
])
@pytest.mark.parametrize("Hkv,G", [(1, 1), (2, 4), (8, 8)])
def test_map_matches_the_plan_on_edge_cases(pmap, lens, C, Hkv, G):
    check(pmap, lens, C, Hkv, G)


def test_map_matches_the_plan_on_random_batches(pmap):
    rng = np.random.default_rng(20260622)
    tasks = 0
    for _ in range(300):
        B = int(rng.integers(1, 48))
        C = int(rng.choice([16, 64, 256, 1024]))
        kind = int(rng.integers(0, 3))
        if kind == 0:
            lens = rng.integers(0, 5 * C, size=B)
        elif kind == 1:
            lens = rng.choice([0, 1, C - 1, C, C + 1, 2 * C], size=B)
        else:
            lens = rng.integers(0, 2, size=B) * rng.integers(1, 4, size=B) * C
        tasks += check(pmap, lens, C, int(rng.choice([1, 2, 8])), int(rng.choice([1, 4, 8])))
    assert tasks > 10000


def test_map_at_the_largest_self_planned_batch(pmap):
    rng = np.random.default_rng(7)
    check(pmap, rng.integers(0, 3000, size=512), 256, 8, 8)
    check(pmap, [1] * 512, 16, 2, 4)


def test_balance_order_definition_on_a_worked_case():
    """The definition itself, on a batch small enough to order by hand:
    C = 256, one kv head, rows of 300, 100, 250 and 512 tokens.  Full splits:
    row 0 split 0, row 3 splits 0 and 1.  Shorter splits: row 0 44 tokens
    (class 1), row 1 100 (class 3), row 2 250 (class 7)."""
    lens = np.array([300, 100, 250, 512])
    canon, _ = oracle.plan_compact(lens, 1, 1, 256)
    got = canon[balance_order(canon, lens, 256)][:, :3].tolist()
    # full splits: row 0 split 0, row 3 splits 0 and 1; then rows 2, 1, 0 by class
    assert got == [[0, 0, 0], [3, 0, 0], [3, 0, 1], [2, 0, 0], [1, 0, 0], [0, 0, 1]]
    assert short_rows(lens, 256).tolist() == [2, 1, 0]
