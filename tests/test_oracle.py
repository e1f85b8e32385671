"""Pins for the float64 oracle: checks against things other than the oracle itself.

Brute force (dense attention by torch's float64 SDPA on un-paged tensors),
closed forms, invariants, direct enumeration of the plan and the launch counts
the pages print.  Passages: "PersistentKV: Page-Aware Decode Scheduling for
Long-Context LLM Serving on Commodity GPUs", technical summary, Methodology 1
(GQA, layout, sequence splitting, row-local bounds, compact workqueue) and
Results ("Scheduling overhead").
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import logsumexp

import oracle
import pkv_traces as T

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------ helpers

def small_case(lens, Hq=8, Hkv=2, d=64, P=16, C=32, seed=1, k_scale=1.0, extra_pages=0):
    tr = T.custom_trace(lens, Hq, Hkv, d, P, C, seed=seed, extra_pages=extra_pages)
    tr.k_scale = k_scale
    q = T.gen_q(tr)
    k, v = T.gen_kv(tr)
    return tr, q, k, v


def unpage(cache, bt_row, n, P):
    """Gather a row's first n tokens into a contiguous [n, Hkv, d] array (numpy indexing)."""
    t = np.arange(n)
    return cache[bt_row[t // P], t % P]


def brute_force(tr, q, k, v):
    """Dense attention by torch SDPA in float64 with KV heads repeated G times."""
    G = tr.G
    o = np.zeros((tr.B, tr.Hq, tr.d))
    lse = np.full((tr.B, tr.Hq), -np.inf)
    for i in range(tr.B):
        n = int(tr.seq_lens[i])
        if n == 0:
            continue
        K = torch.from_numpy(unpage(k, tr.block_table[i], n, tr.page_size).astype(np.float64))
        V = torch.from_numpy(unpage(v, tr.block_table[i], n, tr.page_size).astype(np.float64))
        K = K.permute(1, 0, 2).repeat_interleave(G, dim=0)   # [Hq, n, d]
        V = V.permute(1, 0, 2).repeat_interleave(G, dim=0)
        Q = torch.from_numpy(q[i].astype(np.float64))[:, None, :]  # [Hq, 1, d]
        out = torch.nn.functional.scaled_dot_product_attention(
            Q[None], K[None], V[None], scale=tr.scale)[0, :, 0, :]
        o[i] = out.numpy()
        s = (Q @ K.transpose(1, 2))[:, 0, :].numpy() * tr.scale  # [Hq, n]
        lse[i] = logsumexp(s, axis=1)
    return o, lse


def run_oracle(tr, q, k, v):
    return oracle.attention(q, k, v, tr.block_table, tr.seq_lens, tr.scale)


# ------------------------------------------------------------ fp16 decode

def test_half_decode_matches_golden_values():
    rows = [ln.split() for ln in open(os.path.join(GOLDEN, "fp16_values.txt"))
            if ln.strip() and not ln.startswith("#")]
    bits = np.array([int(h, 16) for h, _ in rows], dtype=np.uint16)
    want = np.array([float(x) for _, x in rows])
    got = oracle.half_to_double(bits)
    for b, g, w in zip(bits, got, want):
        if math.isnan(w):
            assert math.isnan(g), hex(b)
        else:
            assert g == w and math.copysign(1, g) == math.copysign(1, w), hex(b)


def test_half_decode_all_patterns_match_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.half_to_double(bits)
    want = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


# ------------------------------------------------------------ brute force

@pytest.mark.parametrize("lens,Hq,Hkv,d,P", [
    ([37, 1, 64, 200], 8, 2, 64, 16),
    ([100], 4, 4, 128, 16),          # G = 1: plain multi-head attention
    ([5, 33, 0, 77], 8, 1, 32, 8),   # one KV head shared by all, an empty row
    ([130, 17], 16, 2, 128, 32),     # G = 8
])
def test_oracle_matches_dense_sdpa(lens, Hq, Hkv, d, P):
    tr, q, k, v = small_case(lens, Hq, Hkv, d, P)
    o, lse = run_oracle(tr, q, k, v)
    ob, lseb = brute_force(tr, q, k, v)
    assert np.max(np.abs(o - ob)) < 1e-12
    fin = np.isfinite(lseb)
    assert np.array_equal(fin, np.isfinite(lse))
    assert np.max(np.abs(lse[fin] - lseb[fin])) < 1e-12
    assert np.all(lse[~fin] == -np.inf)


def test_empty_row_gives_zero_and_neg_inf():
    tr, q, k, v = small_case([0, 3], Hq=4, Hkv=2, d=32)
    o, lse = run_oracle(tr, q, k, v)
    assert np.all(o[0] == 0.0) and np.all(lse[0] == -np.inf)
    assert np.all(np.isfinite(o[1]))


# ------------------------------------------------------------ closed forms

def test_identical_keys_give_mean_of_v():
    tr, q, k, v = small_case([45], Hq=4, Hkv=2, d=64)
    k[:] = k[0, 0]                      # every token's key identical (per head)
    o, _ = run_oracle(tr, q, k, v)
    V = unpage(v, tr.block_table[0], 45, tr.page_size).astype(np.float64)  # [n, Hkv, d]
    mean = V.mean(axis=0)
    for h in range(tr.Hq):
        assert np.max(np.abs(o[0, h] - mean[h // tr.G])) < 1e-14


def test_length_one_gives_v0():
    tr, q, k, v = small_case([1, 1], Hq=8, Hkv=4, d=64)
    o, lse = run_oracle(tr, q, k, v)
    for i in range(2):
        V0 = v[tr.block_table[i, 0], 0].astype(np.float64)      # [Hkv, d]
        K0 = k[tr.block_table[i, 0], 0].astype(np.float64)
        for h in range(tr.Hq):
            assert np.array_equal(o[i, h], V0[h // tr.G])
            s = tr.scale * float(q[i, h].astype(np.float64) @ K0[h // tr.G])
            assert abs(lse[i, h] - s) < 1e-12


def test_zero_query_gives_mean_of_v():
    tr, q, k, v = small_case([29], Hq=4, Hkv=1, d=32)
    q[:] = 0
    o, lse = run_oracle(tr, q, k, v)
    V = unpage(v, tr.block_table[0], 29, tr.page_size).astype(np.float64)
    assert np.max(np.abs(o[0] - V.mean(axis=0)[0])) < 1e-14
    assert np.allclose(lse, math.log(29), atol=1e-14)


def test_constant_v_gives_constant():
    tr, q, k, v = small_case([61, 7], Hq=8, Hkv=2, d=64)
    c = np.linspace(-3, 3, tr.d).astype(np.float16)
    v[:] = c
    o, _ = run_oracle(tr, q, k, v)
    assert np.max(np.abs(o - c.astype(np.float64))) < 1e-14


def test_dominant_key_selects_its_value():
    tr, q, k, v = small_case([50], Hq=2, Hkv=1, d=32)
    q[:] = 0
    q[0, :, 3] = 1.0
    k[:] = 0
    t_star = 17
    pg, sl = tr.block_table[0, t_star // tr.page_size], t_star % tr.page_size
    k[pg, sl, 0, 3] = 60000.0
    o, lse = run_oracle(tr, q, k, v)
    assert np.array_equal(o[0, 0], v[pg, sl, 0].astype(np.float64))
    assert abs(lse[0, 0] - tr.scale * 60000.0) < 1e-9


def test_identical_queries_in_group_give_identical_outputs():
    tr, q, k, v = small_case([90, 40], Hq=8, Hkv=2, d=64)
    q[:, 1] = q[:, 0]
    q[:, 2] = q[:, 0]
    q[:, 5] = q[:, 4]
    o, _ = run_oracle(tr, q, k, v)
    assert np.array_equal(o[:, 1], o[:, 0]) and np.array_equal(o[:, 2], o[:, 0])
    assert np.array_equal(o[:, 5], o[:, 4])
    # heads 0 and 4 read different KV heads, so they differ
    assert not np.allclose(o[:, 0], o[:, 4])


# ------------------------------------------------------------ invariants

def test_page_relabelling_is_bit_identical():
    tr, q, k, v = small_case([70, 33, 1], Hq=8, Hkv=2, d=64, extra_pages=9)
    o1, l1 = run_oracle(tr, q, k, v)
    perm = np.random.default_rng(5).permutation(tr.num_pages)   # new page p holds old page perm[p]
    inv = np.argsort(perm)
    k2, v2 = k[perm], v[perm]
    bt2 = tr.block_table.copy()
    m = bt2 >= 0
    bt2[m] = inv[bt2[m]]
    o2, l2 = oracle.attention(q, k2, v2, bt2, tr.seq_lens, tr.scale)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


@pytest.mark.parametrize("C", [8, 16, 48, 64, 1000])
def test_split_merge_matches_unsplit(C):
    tr, q, k, v = small_case([130, 1, 64, 0, 65], Hq=8, Hkv=2, d=32, P=16)
    o, lse = run_oracle(tr, q, k, v)
    m, l, acc = oracle.partials(q, k, v, tr.block_table, tr.seq_lens, tr.scale, C)
    o2, lse2 = oracle.merge(m, l, acc, tr.seq_lens, tr.Hq, C)
    assert np.max(np.abs(o - o2)) < 1e-12
    fin = np.isfinite(lse)
    assert np.array_equal(fin, np.isfinite(lse2))
    assert np.max(np.abs(lse[fin] - lse2[fin])) < 1e-12


def test_rect_partials_merge_to_the_same_output():
    tr, q, k, v = small_case([130, 1, 64, 0, 65], Hq=8, Hkv=2, d=32, P=16)
    C, S_b = 32, 5
    o, lse = run_oracle(tr, q, k, v)
    m, l, acc = oracle.partials(q, k, v, tr.block_table, tr.seq_lens, tr.scale, C,
                                rect=True, S_b=S_b)
    o2, _ = oracle.merge(m, l, acc, tr.seq_lens, tr.Hq, C, rect=True, S_b=S_b)
    assert np.max(np.abs(o - o2)) < 1e-12


def test_output_is_linear_in_v():
    tr, q, k, v = small_case([77, 20], Hq=4, Hkv=2, d=32)
    rng = np.random.default_rng(9)
    v1 = rng.integers(-8, 8, size=v.shape).astype(np.float16)
    v2 = rng.integers(-8, 8, size=v.shape).astype(np.float16)
    o1, _ = oracle.attention(q, k, v1, tr.block_table, tr.seq_lens, tr.scale)
    o2, _ = oracle.attention(q, k, v2, tr.block_table, tr.seq_lens, tr.scale)
    o12, _ = oracle.attention(q, k, (v1 + v2).astype(np.float16), tr.block_table,
                              tr.seq_lens, tr.scale)
    o3, _ = oracle.attention(q, k, (3 * v1).astype(np.float16), tr.block_table,
                             tr.seq_lens, tr.scale)
    assert np.max(np.abs(o12 - (o1 + o2))) < 1e-12
    assert np.max(np.abs(o3 - 3 * o1)) < 1e-12


def test_scores_follow_scale():
    tr, q, k, v = small_case([40], Hq=4, Hkv=2, d=64)
    _, lse1 = oracle.attention(q, k, v, tr.block_table, tr.seq_lens, 0.1)
    _, lse0 = oracle.attention(q, k, v, tr.block_table, tr.seq_lens, 0.0)
    assert np.allclose(lse0, math.log(40), atol=1e-14)
    assert not np.allclose(lse1, lse0)


# ------------------------------------------------------------ partial states

def test_partials_definition_against_dense_scores():
    tr, q, k, v = small_case([100, 37], Hq=4, Hkv=2, d=32, P=16)
    C = 32
    m, l, acc = oracle.partials(q, k, v, tr.block_table, tr.seq_lens, tr.scale, C)
    _, offsets = oracle.plan_compact(tr.seq_lens, tr.Hq, tr.Hkv, C)
    for i in range(tr.B):
        n = int(tr.seq_lens[i])
        K = unpage(k, tr.block_table[i], n, tr.page_size).astype(np.float64)
        V = unpage(v, tr.block_table[i], n, tr.page_size).astype(np.float64)
        for h in range(tr.Hq):
            g = h // tr.G
            s = tr.scale * (K[:, g, :] @ q[i, h].astype(np.float64))
            for j in range((n + C - 1) // C):
                sl = slice(j * C, min(n, (j + 1) * C))
                slot = (offsets[i] + j) * tr.Hq + h
                assert m[slot] == np.max(s[sl])
                w = np.exp(s[sl] - m[slot])
                assert abs(l[slot] - w.sum()) < 1e-12
                assert np.max(np.abs(acc[slot] - w @ V[sl, g, :])) < 1e-12


def test_neutral_states_are_exact():
    tr, q, k, v = small_case([20, 70], Hq=4, Hkv=2, d=32)
    C, S_b = 32, 4
    m, l, acc = oracle.partials(q, k, v, tr.block_table, tr.seq_lens, tr.scale, C,
                                rect=True, S_b=S_b)
    _, empty = oracle.plan_rect(tr.seq_lens, tr.Hq, tr.Hkv, C, S_b)
    neg_inf_bits = np.array([-np.inf]).view(np.uint64)[0]
    for i in range(tr.B):
        for j in range(S_b):
            for h in range(tr.Hq):
                slot = (i * S_b + j) * tr.Hq + h
                if j * C >= tr.seq_lens[i]:
                    assert np.array([m[slot]]).view(np.uint64)[0] == neg_inf_bits
                    assert np.array([l[slot]]).view(np.uint64)[0] == 0
                    assert not np.any(np.array(acc[slot]).view(np.uint64))
                else:
                    assert np.isfinite(m[slot]) and l[slot] >= 1.0


def test_single_split_state_is_the_output():
    tr, q, k, v = small_case([45, 9], Hq=4, Hkv=2, d=32)
    o, lse = run_oracle(tr, q, k, v)
    m, l, acc = oracle.partials(q, k, v, tr.block_table, tr.seq_lens, tr.scale, 4096)
    for i in range(tr.B):
        for h in range(tr.Hq):
            slot = i * tr.Hq + h
            assert np.max(np.abs(acc[slot] / l[slot] - o[i, h])) < 1e-13
            assert abs(m[slot] + math.log(l[slot]) - lse[i, h]) < 1e-12


# ------------------------------------------------------------ plan

def brute_force_tasks(lens, Hq, Hkv, C):
    """All (i, g, j) with a non-empty split, lexicographic; state rows counted directly."""
    G = Hq // Hkv
    out = []
    for i, n in enumerate(lens):
        rows_before = sum(-(-int(x) // C) for x in lens[:i])
        for g, j in itertools.product(range(Hkv), range(-(-int(n) // C))):
            if j * C < n:
                out.append((i, g, j, (rows_before + j) * Hq + g * G))
    return np.array(out, dtype=np.int32).reshape(-1, 4)


@pytest.mark.parametrize("lens,C", [
    ([1, 0, 1024, 1025, 17], 256),
    ([0, 0], 16),
    ([5000, 3, 64, 64, 100000], 1024),
])
def test_plan_matches_enumeration(lens, C):
    Hq, Hkv = 32, 8
    tasks, offsets = oracle.plan_compact(lens, Hq, Hkv, C)
    want = brute_force_tasks(lens, Hq, Hkv, C)
    assert tasks.shape == want.shape and np.array_equal(tasks, want)
    n = [-(-x // C) for x in lens]
    assert list(offsets) == [sum(n[:i]) for i in range(len(lens) + 1)]
    assert tasks.shape[0] == Hkv * sum(n)


def test_plan_closed_forms_on_workloads():
    tr1 = T.make_trace(1)
    tasks, _ = oracle.plan_compact(tr1.seq_lens, tr1.Hq, tr1.Hkv, tr1.split_tokens)
    assert tasks.shape[0] == 2 * 4          # Hkv=2, S=4
    tr2 = T.make_trace(2)
    tasks, _ = oracle.plan_compact(tr2.seq_lens, tr2.Hq, tr2.Hkv, tr2.split_tokens)
    assert tasks.shape[0] == 8 * 32         # Hkv=8, S=32


def test_rect_plan_enumeration():
    lens, Hq, Hkv, C, S_b = [100, 0, 300], 8, 2, 64, 5
    tasks, empty = oracle.plan_rect(lens, Hq, Hkv, C, S_b)
    want = [(i, g, j, (i * S_b + j) * Hq + g * (Hq // Hkv))
            for i in range(3) for g in range(Hkv) for j in range(S_b)]
    assert np.array_equal(tasks, np.array(want, dtype=np.int32))
    assert list(empty) == [int(j * C >= lens[i]) for i, g, j, _ in want]


# ------------------------------------------------------------ counters

def test_launch_counts_reproduce_the_pages_bimodal_figures():
    gold = json.load(open(os.path.join(GOLDEN, "launch_counts.json")))
    tr = T.make_trace(3)
    assert len(set(tr.seq_lens.tolist())) == 8    # eight distinct lengths
    ex = oracle.counters(oracle.PATH_EXACT_BUCKETS, tr.seq_lens, tr.Hq, tr.Hkv, tr.d, 1024)
    wq = oracle.counters(oracle.PATH_WORKQUEUE, tr.seq_lens, tr.Hq, tr.Hkv, tr.d, 1024)
    assert ex.attn_launches == gold["exact_length_buckets_launches_per_step"]
    assert wq.attn_launches == gold["compact_workqueue_launches_per_step"]


def _state_traffic_enumerated(lens, Hq, Hkv, C, S_b):
    """States written by the split step and read by the merge, enumerated from
    the plans' records rather than from the counter model's sums: the
    rectangular grid writes one state per query head of every cell (an empty
    cell gets the neutral state) and the merge reads the cells a row's length
    reaches; the compact queue lists only those cells."""
    G = Hq // Hkv
    rect, empty = oracle.plan_rect(lens, Hq, Hkv, C, S_b)
    comp, _ = oracle.plan_compact(lens, Hq, Hkv, C)
    return {"rect": (len(rect) * G, int((empty == 0).sum()) * G),
            "compact": (len(comp) * G, len(comp) * G)}


@pytest.mark.parametrize("seed", [T.HELDOUT_SEED, T.CALIBRATION_SEED, 1, 2])
def test_merge_state_counts_match_the_enumerated_plans(seed):
    """The counter model behind the pages' merge-state traffic comparison
    (Results, 'Scheduling overhead') against the plans' records, on the B=8
    bimodal batch of several draws and on edge cases (empty rows, a length at
    a split boundary, one split)."""
    cases = [(T.make_trace(3, seed=seed).seq_lens, 32, 8, 1024)]
    if seed == T.HELDOUT_SEED:
        cases += [([100, 3000, 40, 0, 1024, 2049], 8, 2, 256), ([0, 0, 5], 8, 8, 16),
                  ([256], 4, 1, 256)]
    for lens, Hq, Hkv, C in cases:
        S_b = max(1, -(-int(np.max(lens)) // C))
        got = _state_traffic_enumerated(lens, Hq, Hkv, C, S_b)
        r = oracle.counters(oracle.PATH_BUCKETED, lens, Hq, Hkv, 128, C, S_b)
        w = oracle.counters(oracle.PATH_WORKQUEUE, lens, Hq, Hkv, 128, C)
        assert (r.states_written, r.states_read) == got["rect"]
        assert (w.states_written, w.states_read) == got["compact"]
        for c in (r, w):
            assert c.merge_state_bytes == (c.states_written + c.states_read) * (128 + 2) * 4


def test_counters_closed_forms():
    tr = T.make_trace(2)
    c = oracle.counters(oracle.PATH_BUCKETED, tr.seq_lens, tr.Hq, tr.Hkv, tr.d, 1024, 32)
    assert c.kv_bytes == 128 * 1024 * 1024
    assert c.tasks == c.grid_tasks == 256 and c.attn_launches == 2 and c.plan_launches == 0
    assert c.merge_state_bytes == 2 * 32 * 32 * (128 + 2) * 4
    s = oracle.counters(oracle.PATH_SINGLE, [5, 0, 7], 8, 2, 64, 16)
    assert s.attn_launches == 1 and s.merge_state_bytes == 0 and s.tasks == 6
    # compact writes and reads the same states; rectangular writes the neutral cells too
    lens = [100, 3000, 40]
    r = oracle.counters(oracle.PATH_BUCKETED, lens, 8, 2, 64, 1024, 3)
    w = oracle.counters(oracle.PATH_WORKQUEUE, lens, 8, 2, 64, 1024)
    assert w.states_written == w.states_read == (1 + 3 + 1) * 8
    assert r.states_written == 3 * 3 * 8 and r.states_read == w.states_read
    assert w.merge_state_bytes < r.merge_state_bytes
    # exact-length buckets: one (split, merge) pair per distinct non-zero length
    e = oracle.counters(oracle.PATH_EXACT_BUCKETS, [5, 5, 7, 0, 7, 9], 8, 2, 64, 16)
    assert e.attn_launches == 2 * 3


# ------------------------------------------------------------ traces

def test_traces_are_deterministic_and_shaped():
    a, b = T.make_trace(5), T.make_trace(5)
    assert np.array_equal(a.seq_lens, b.seq_lens) and np.array_equal(a.block_table, b.block_table)
    assert a.B == 64 and a.G == 8 and a.seq_lens.min() >= 128 and a.seq_lens.max() <= 65536
    # each row owns enough pages for 256 appended tokens, pages are distinct
    used = a.block_table[a.block_table >= 0]
    assert len(np.unique(used)) == used.size == a.num_pages
    assert np.all((a.block_table >= 0).sum(1) == (a.seq_lens + 256 + 15) // 16)
    c3 = T.make_trace(3)
    assert sorted((c3.seq_lens >= 24576).tolist()) == [False] * 4 + [True] * 4
    z = T.zipf_lengths(np.random.default_rng(0), 20000)
    assert z.min() >= 16 and z.max() <= 32768 and 150 < np.median(z) < 230
    c1 = T.make_trace(1)
    assert len(np.unique(c1.block_table)) == 64 and c1.block_table.max() < 128
    cal, held = T.make_trace(3, seed=T.CALIBRATION_SEED), T.make_trace(3)
    assert not np.array_equal(cal.seq_lens, held.seq_lens)
