"""pkv_decode_step_noalloc: the decode step for callers that cannot allocate
device memory (code inside an allocator's callbacks, plugins of runtimes that
own every device allocation, paths that must avoid the allocator's implicit
synchronisation).  It runs the same kernels as pkv_decode_step with the
library's static scratch array instead of caller buffers.

The test calls it through the C ABI twice in a row on each path -- the second
call sees the array as the first left it -- and checks both outputs against
pkv_decode_step within the parity tolerance.  It builds and loads the library
itself, so it passes alone in a fresh process as well as after the rest of the
suite; this file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import pkv_traces as T
from paged_kv_gqa_09_gb300 import _lib, api

from gpu_util import ATOL, LSE_ATOL, RTOL, run_path, shape_of, upload

pytestmark = pytest.mark.gpu

PATHS = (_lib.PKV_PATH_BUCKETED_SPLIT, _lib.PKV_PATH_WORKQUEUE, _lib.PKV_PATH_SINGLE_PASS)


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_gqa_09_gb300 import build
    build.build()
    return _lib.load()


def _noalloc(L, tr, d, cfg):
    shape = shape_of(tr)
    o = torch.full((tr.B, tr.Hq, tr.d), float("nan"), dtype=torch.float16, device="cuda")
    lse = torch.full((tr.B, tr.Hq), float("nan"), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    rc = L.pkv_decode_step_noalloc(ctypes.byref(shape), ctypes.byref(cfg), d["q"].data_ptr(),
                                   d["k"].data_ptr(), d["v"].data_ptr(), d["bt"].data_ptr(),
                                   d["sl"].data_ptr(), o.data_ptr(), lse.data_ptr(), stream)
    assert rc == 0, _lib.last_error()
    torch.cuda.synchronize()
    return o, lse


@pytest.mark.parametrize("path,merge,plan", [(p, _lib.PKV_MERGE_SEPARATE, 0) for p in PATHS] +
                         [(p, _lib.PKV_MERGE_FUSED, 0) for p in PATHS[:2]] +
                         [(_lib.PKV_PATH_WORKQUEUE, _lib.PKV_MERGE_SEPARATE, _lib.PKV_PLAN_IN_DECODE)])
def test_noalloc_matches_decode_step_twice(lib, path, merge, plan):
    """With the fused merge the header also holds the grid barrier's counters,
    which the call zeroes with the rest of the header, over whatever the
    previous call left there; with the plan built in the decode, the decode
    writes the plan into the same scratch."""
    tr = T.make_trace(3)  # B=8 bimodal, ~491 MB of K+V
    q = T.gen_q(tr)
    k, v = T.gen_kv(tr)
    d = upload(tr, q, k, v)
    o_ref, lse_ref, _, _ = run_path(tr, d, path)
    C = tr.split_tokens
    cfg = api.make_cfg(path, C, tr.n_max if path == _lib.PKV_PATH_BUCKETED_SPLIT else 0, 0, merge, plan)
    ref = o_ref.float().cpu().numpy()
    lref = lse_ref.cpu().numpy()
    for call in range(2):
        o, lse = _noalloc(lib, tr, d, cfg)
        x = o.float().cpu().numpy()
        assert np.all(np.abs(x - ref) <= ATOL + RTOL * np.abs(ref)), f"call {call}"
        assert np.max(np.abs(lse.cpu().numpy() - lref)) <= LSE_ATOL, f"call {call}"


def test_noalloc_rejects_steps_beyond_its_scratch(lib):
    tr = T.make_trace(5)  # B=64 workqueue: its partial states need far more than the array
    shape = shape_of(tr)
    cfg = api.make_cfg(_lib.PKV_PATH_WORKQUEUE, tr.split_tokens)
    assert api.pkv_partials_size(shape, cfg) > _lib.NOALLOC_SCRATCH_BYTES
    fake = 1 << 20
    rc = lib.pkv_decode_step_noalloc(ctypes.byref(shape), ctypes.byref(cfg), fake, fake, fake,
                                     fake, fake, fake, None, None)
    assert rc == _lib.PKV_ECAPACITY
    assert "scratch" in _lib.last_error()
