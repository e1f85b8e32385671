"""Full-size uniform workload (B=64, Hq=64, Hkv=8, G=8, lengths U[128, 65536],
256 decode steps each appending one token per row), in the launch
configuration the benchmark times: one captured CUDA graph per step holding
the fused append + page allocation + plan launch, the decode and the merge on
the compact workqueue, the step's q and new token copied into fixed buffers
before each replay.  The ~8.6 GB pool is drawn on the GPU by torch's seeded
generator; the oracle checks sampled rows (all 64 heads each) at steps 0, 1
and 255 from host copies of exactly those rows' pages, found through the block
table as the device allocated it."""
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


def test_uniform_b64_decode_loop_matches_oracle():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tr = T.make_trace(5)
    k, v = T.gen_kv_torch(tr, "cuda")
    bt_alloc, free_np = T.allocation_split(tr)  # rows start with the pages their tokens fill
    bt = dev(np.ascontiguousarray(bt_alloc))
    sl = dev(tr.seq_lens)
    free = dev(free_np)
    cnt = torch.tensor([free_np.size], dtype=torch.int32, device="cuda")
    shape = shape_of(tr)
    cfg = api.make_cfg(_lib.PKV_PATH_WORKQUEUE, tr.split_tokens)
    ws = torch.zeros(api.pkv_plan_workspace_size(shape, cfg), dtype=torch.uint8, device="cuda")
    part = torch.empty(api.pkv_partials_size(shape, cfg) // 4, dtype=torch.float32, device="cuda")
    o = torch.empty((tr.B, tr.Hq, tr.d), dtype=torch.float16, device="cuda")
    lse = torch.empty((tr.B, tr.Hq), dtype=torch.float32, device="cuda")
    q_buf = torch.empty((tr.B, tr.Hq, tr.d), dtype=torch.float16, device="cuda")
    kn_buf = torch.empty((tr.B, tr.Hkv, tr.d), dtype=torch.float16, device="cuda")
    vn_buf = torch.empty_like(kn_buf)
    st = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(st):
        with torch.cuda.graph(g, stream=st):  # captured, not run
            api.pkv_append_plan(shape, cfg, ws, kn_buf, vn_buf, bt, sl, k, v, free, cnt, stream=st)
            api.pkv_decode(shape, cfg, ws, q_buf, k, v, bt, sl, part, stream=st)
            api.pkv_merge(shape, cfg, ws, sl, part, o, lse, stream=st)
    lens = tr.seq_lens.copy()
    checked = 0
    for step in range(tr.steps):
        kn, vn = T.gen_append_tokens(tr, step)
        q = T.gen_step_q(tr, step)
        with torch.cuda.stream(st):
            q_buf.copy_(torch.from_numpy(q), non_blocking=False)
            kn_buf.copy_(torch.from_numpy(kn), non_blocking=False)
            vn_buf.copy_(torch.from_numpy(vn), non_blocking=False)
            g.replay()
        lens += 1
        if step in CHECK_STEPS:
            st.synchronize()
            check_error_free(ws)
            assert np.array_equal(sl.cpu().numpy(), lens)
            bt_now = bt.cpu().numpy()
            oref, lref = row_oracle(tr, q, k, v, bt_now, lens, SAMPLE_ROWS)
            close(o[SAMPLE_ROWS], oref, f"o at step {step}")
            close_lse(lse[SAMPLE_ROWS], lref)
            checked += 1
    st.synchronize()
    assert checked == len(CHECK_STEPS)
    used = bt.cpu().numpy()
    used = used[used >= 0]
    assert len(np.unique(used)) == used.size  # no page handed out twice
