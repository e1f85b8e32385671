"""Full-size uniform workload (B=64, Hq=64, Hkv=8, G=8, lengths U[128, 65536],
256 decode steps each appending one token per row), in the launch
configuration the benchmark times: append + plan + decode + merge per step on
the compact workqueue.  The ~8.6 GB pool is drawn on the GPU by torch's seeded
generator; the oracle checks sampled rows (all 64 heads each) at steps 0, 1
and 255 from host copies of exactly those rows' pages."""
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
    bt = dev(tr.block_table)
    sl = dev(tr.seq_lens)
    shape = shape_of(tr)
    cfg = api.make_cfg(_lib.PKV_PATH_WORKQUEUE, tr.split_tokens)
    ws = torch.zeros(api.pkv_plan_workspace_size(shape, cfg), dtype=torch.uint8, device="cuda")
    part = torch.empty(api.pkv_partials_size(shape, cfg) // 4, dtype=torch.float32, device="cuda")
    o = torch.empty((tr.B, tr.Hq, tr.d), dtype=torch.float16, device="cuda")
    lse = torch.empty((tr.B, tr.Hq), dtype=torch.float32, device="cuda")
    lens = tr.seq_lens.copy()
    checked = 0
    for step in range(tr.steps):
        kn, vn = T.gen_append_tokens(tr, step)
        q = T.gen_step_q(tr, step)
        api.pkv_append(shape, ws, dev(kn), dev(vn), bt, sl, k, v)
        lens += 1
        api.pkv_decode_step(shape, cfg, ws, dev(q), k, v, bt, sl, part, o, lse)
        if step in CHECK_STEPS:
            torch.cuda.synchronize()
            check_error_free(ws)
            assert np.array_equal(sl.cpu().numpy(), lens)
            oref, lref = row_oracle(tr, q, k, v, tr.block_table, lens, SAMPLE_ROWS)
            close(o[SAMPLE_ROWS], oref, f"o at step {step}")
            close_lse(lse[SAMPLE_ROWS], lref)
            checked += 1
    assert checked == len(CHECK_STEPS)
