"""Helpers shared by the GPU parity tests (not a test module)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import pkv_traces as T
from paged_kv_gqa_09_gb300 import api, _lib

# Parity tolerance for fp16 outputs against the float64 oracle, applied
# element-wise in allclose form: |x - y| <= ATOL + RTOL * |y|.
ATOL, RTOL = 3e-3, 1e-2
# lse (fp32): scores are exact fp16 products summed in fp32 and the exponent
# is evaluated with a 2^-22 relative error, so 1e-3 absolute is generous.
LSE_ATOL = 1e-3


def dev(x, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(x)).cuda()
    return t if dtype is None else t.to(dtype)


def upload(tr: T.Trace, q, k, v):
    return dict(q=dev(q), k=dev(k), v=dev(v), bt=dev(tr.block_table), sl=dev(tr.seq_lens))


def shape_of(tr: T.Trace):
    return _lib.Shape(tr.B, tr.Hq, tr.Hkv, tr.d, tr.page_size, tr.num_pages, tr.bt_stride,
                      float(tr.scale))


def run_path(tr: T.Trace, d: dict, path: int, C: int | None = None, bucket: int | None = None,
             max_tasks: int = 0, want_lse: bool = True, merge: int = _lib.PKV_MERGE_SEPARATE,
             ws: torch.Tensor | None = None, plan: int = _lib.PKV_PLAN_SEPARATE):
    """One decode step through pkv_decode_step; returns (o, lse, ws, partials).
    A given workspace `ws` is reused (it must be zeroed once before first use)."""
    shape = shape_of(tr)
    C = tr.split_tokens if C is None else C
    if bucket is None:
        bucket = tr.n_max if path == _lib.PKV_PATH_BUCKETED_SPLIT else 0
    cfg = api.make_cfg(path, C, bucket, max_tasks, merge, plan)
    if ws is None:
        ws = torch.zeros(max(64, api.pkv_plan_workspace_size(shape, cfg)), dtype=torch.uint8,
                         device="cuda")
    npart = api.pkv_partials_size(shape, cfg)
    part = torch.full((max(npart // 4, 4),), float("nan"), dtype=torch.float32, device="cuda")
    o = torch.full((tr.B, tr.Hq, tr.d), float("nan"), dtype=torch.float16, device="cuda")
    lse = torch.full((tr.B, tr.Hq), float("nan"), dtype=torch.float32, device="cuda") if want_lse else None
    api.pkv_decode_step(shape, cfg, ws, d["q"], d["k"], d["v"], d["bt"], d["sl"],
                        part if npart else None, o, lse)
    torch.cuda.synchronize()
    return o, lse, ws, part


def check_error_free(ws):
    st, msg = api.pkv_get_error(ws)
    assert st == 0, msg


def close(o_gpu: torch.Tensor, o_ref: np.ndarray, what: str = "o"):
    x = o_gpu.float().cpu().numpy().astype(np.float64)
    bad = ~(np.abs(x - o_ref) <= ATOL + RTOL * np.abs(o_ref))
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(
            f"{what}: {bad.sum()} of {bad.size} elements outside |x-y| <= {ATOL} + {RTOL}|y|; "
            f"max abs err {np.nanmax(np.abs(x - o_ref)):.3g}; first {idx.tolist()} "
            f"gpu {x[tuple(idx[0])]} ref {o_ref[tuple(idx[0])]}")
    return float(np.max(np.abs(x - o_ref))) if x.size else 0.0


def close_lse(lse_gpu: torch.Tensor, lse_ref: np.ndarray):
    x = lse_gpu.cpu().numpy().astype(np.float64)
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(x), fin), "lse finiteness differs"
    assert np.all(x[~fin] == lse_ref[~fin])
    if fin.any():
        err = np.max(np.abs(x[fin] - lse_ref[fin]))
        assert err <= LSE_ATOL, f"lse max abs err {err}"


def header_counters(ws: torch.Tensor) -> dict:
    """The decode's counters in the workspace header, all zero between launches:
    the workqueue's task claims and the fused merge's grid-barrier count."""
    h = ws[:64].view(torch.int32).cpu().numpy()
    return {"next_task": int(h[7]), "done_ctas": int(h[8]), "bar_count": int(h[9])}


def read_plan(ws: torch.Tensor, B: int, with_order: bool = False):
    h = ws[:64].view(torch.int32).cpu().numpy()
    count = int(h[4])
    off = ws[64:64 + 4 * (B + 1)].view(torch.int32).cpu().numpy()
    t0 = (64 + 4 * (B + 1) + 15) // 16 * 16
    tasks = ws[t0:t0 + 16 * count].view(torch.int32).cpu().numpy().reshape(-1, 4)
    if not with_order:
        return count, off, tasks, h
    cap = (ws.numel() - t0 - 4 * B) // 32  # workspace = t0 + 32 * cap + short_before[B]
    o0 = t0 + 16 * cap
    ordered = ws[o0:o0 + 16 * count].view(torch.int32).cpu().numpy().reshape(-1, 4)
    return count, off, tasks, h, ordered


def oracle_out(tr, q, k, v):
    return oracle.attention(q, k, v, tr.block_table, tr.seq_lens, tr.scale)
