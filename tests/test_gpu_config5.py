"""Full-size uniform workload (B=64, Hq=64, Hkv=8, G=8, lengths U[128, 65536],
256 decode steps each appending one token per row) in captured CUDA graphs of
whole steps -- the fused append + page allocation + plan launch, the decode and
the merge on the compact workqueue -- one step per graph (a serving loop) or 8
consecutive steps per graph chained by programmatic dependent launch (how the
benchmark times it), each step's q and new token copied into its own fixed
buffers before a replay.  The ~8.6 GB pool is drawn on the GPU by torch's
seeded generator; the oracle checks sampled rows (all 64 heads each) at steps
0, 1 and 255 from host copies of exactly those rows' pages, found through the
block table as the device allocated it (later steps only add pages and tokens
past a step's lengths, so the final table serves every earlier step)."""
import numpy as np
import pytest
import torch

import oracle
import pkv_traces as T
from paged_kv_gqa_09_gb300 import _lib, api

from gpu_util import check_error_free, close, close_lse, dev, shape_of

pytestmark = pytest.mark.gpu

SAMPLE_ROWS = [0, 17, 38, 63]
CHECK_STEPS = {0, 1, 255}


def row_oracle(tr, q_step, kc, vc, bt, seq_lens, rows):
    """Oracle on the sampled rows from host copies of their pages."""
    o = np.zeros((len(rows), tr.Hq, tr.d))
    lse = np.zeros((len(rows), tr.Hq))
    for r, i in enumerate(rows):
        n = int(seq_lens[i])
        npg = -(-n // tr.page_size)
        pages = bt[i, :npg]
        kp = kc[torch.from_numpy(pages.astype(np.int64)).cuda()].cpu().numpy()
        vp = vc[torch.from_numpy(pages.astype(np.int64)).cuda()].cpu().numpy()
        bt_local = np.arange(npg, dtype=np.int32)[None, :]
        oo, ll = oracle.attention(q_step[i:i + 1], kp, vp, bt_local, np.array([n], np.int32),
                                  tr.scale)
        o[r], lse[r] = oo[0], ll[0]
    return o, lse


@pytest.mark.parametrize("per_graph,plan", [(1, _lib.PKV_PLAN_SEPARATE), (8, _lib.PKV_PLAN_SEPARATE),
                                           (8, _lib.PKV_PLAN_IN_DECODE)])
def test_uniform_b64_decode_loop_matches_oracle(per_graph, plan):
    """plan = IN_DECODE is the benchmark's step: the append launch only appends
    and allocates (one CTA per row) and the decode builds the plan itself."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tr = T.make_trace(5)
    assert tr.steps % per_graph == 0
    k, v = T.gen_kv_torch(tr, "cuda")
    bt_alloc, free_np = T.allocation_split(tr)  # rows start with the pages their tokens fill
    bt = dev(np.ascontiguousarray(bt_alloc))
    sl = dev(tr.seq_lens)
    free = dev(free_np)
    cnt = torch.tensor([free_np.size], dtype=torch.int32, device="cuda")
    shape = shape_of(tr)
    cfg = api.make_cfg(_lib.PKV_PATH_WORKQUEUE, tr.split_tokens, plan=plan)
    ws = torch.zeros(api.pkv_plan_workspace_size(shape, cfg), dtype=torch.uint8, device="cuda")
    part = torch.empty(api.pkv_partials_size(shape, cfg) // 4, dtype=torch.float32, device="cuda")
    S = per_graph
    o = torch.empty((S, tr.B, tr.Hq, tr.d), dtype=torch.float16, device="cuda")
    lse = torch.empty((S, tr.B, tr.Hq), dtype=torch.float32, device="cuda")
    q_buf = torch.empty((S, tr.B, tr.Hq, tr.d), dtype=torch.float16, device="cuda")
    kn_buf = torch.empty((S, tr.B, tr.Hkv, tr.d), dtype=torch.float16, device="cuda")
    vn_buf = torch.empty_like(kn_buf)
    st = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(st):
        with torch.cuda.graph(g, stream=st):  # captured, not run
            for j in range(S):
                api.pkv_append_plan(shape, cfg, ws, kn_buf[j], vn_buf[j], bt, sl, k, v, free, cnt,
                                    stream=st)
                api.pkv_decode(shape, cfg, ws, q_buf[j], k, v, bt, sl, part, stream=st)
                api.pkv_merge(shape, cfg, ws, sl, part, o[j], lse[j], stream=st)
    lens0 = tr.seq_lens.copy()
    checked = 0
    for first in range(0, tr.steps, S):
        qs = {}
        with torch.cuda.stream(st):
            for j in range(S):
                kn, vn = T.gen_append_tokens(tr, first + j)
                qs[first + j] = T.gen_step_q(tr, first + j)
                q_buf[j].copy_(torch.from_numpy(qs[first + j]), non_blocking=False)
                kn_buf[j].copy_(torch.from_numpy(kn), non_blocking=False)
                vn_buf[j].copy_(torch.from_numpy(vn), non_blocking=False)
            g.replay()
        due = [s for s in range(first, first + S) if s in CHECK_STEPS]
        if not due:
            continue
        st.synchronize()
        check_error_free(ws)
        assert np.array_equal(sl.cpu().numpy(), lens0 + first + S)
        bt_now = bt.cpu().numpy()
        for s in due:
            lens = lens0 + s + 1
            oref, lref = row_oracle(tr, qs[s], k, v, bt_now, lens, SAMPLE_ROWS)
            close(o[s - first][SAMPLE_ROWS], oref, f"o at step {s}")
            close_lse(lse[s - first][SAMPLE_ROWS], lref)
            checked += 1
    st.synchronize()
    assert checked == len(CHECK_STEPS)
    used = bt.cpu().numpy()
    used = used[used >= 0]
    assert len(np.unique(used)) == used.size  # no page handed out twice
