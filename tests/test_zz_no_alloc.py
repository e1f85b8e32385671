"""pkv_decode_step_noalloc: the decode step for callers that cannot allocate
device memory (code inside an allocator's callbacks, plugins of runtimes that
own every device allocation, paths that must avoid the allocator's implicit
synchronisation).  It runs the same kernels as pkv_decode_step with the
library's static scratch array instead of caller buffers.

The tests call it through the C ABI twice in a row on each path -- the second
call sees the array as the first left it -- and check both outputs against
pkv_decode_step within the parity tolerance, and against the float64 oracle
directly.  Further cases leave the array's header dirty on purpose (a
workqueue overflow, a timed-out grid barrier) and check that the next call is
still right, and that calls after the first allocate no device memory.  The
module builds and loads the library itself, so it passes alone in a fresh
process as well as after the rest of the suite; it is named to be collected
last.
"""
import ctypes

import numpy as np
import pytest
import torch

import pkv_traces as T
from paged_kv_gqa_09_gb300 import _lib, api

from gpu_util import (ATOL, LSE_ATOL, RTOL, close, close_lse, oracle_out, run_path, shape_of,
                      upload)

pytestmark = pytest.mark.gpu

PATHS = (_lib.PKV_PATH_BUCKETED_SPLIT, _lib.PKV_PATH_WORKQUEUE, _lib.PKV_PATH_SINGLE_PASS)


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_gqa_09_gb300 import build
    build.build()
    return _lib.load()


@pytest.fixture(scope="module")
def bimodal(lib):
    """B=8 bimodal workload (~491 MB of K+V) on the device, with its oracle."""
    tr = T.make_trace(3)
    q = T.gen_q(tr)
    k, v = T.gen_kv(tr)
    d = upload(tr, q, k, v)
    oref, lref = oracle_out(tr, q, k, v)
    return tr, d, oref, lref


def _outputs(tr):
    o = torch.full((tr.B, tr.Hq, tr.d), float("nan"), dtype=torch.float16, device="cuda")
    lse = torch.full((tr.B, tr.Hq), float("nan"), dtype=torch.float32, device="cuda")
    return o, lse


def _call(L, tr, d, cfg, o, lse):
    shape = shape_of(tr)
    stream = torch.cuda.current_stream().cuda_stream
    return L.pkv_decode_step_noalloc(ctypes.byref(shape), ctypes.byref(cfg), d["q"].data_ptr(),
                                     d["k"].data_ptr(), d["v"].data_ptr(), d["bt"].data_ptr(),
                                     d["sl"].data_ptr(), o.data_ptr(), lse.data_ptr(), stream)


def _noalloc(L, tr, d, cfg):
    o, lse = _outputs(tr)
    rc = _call(L, tr, d, cfg, o, lse)
    assert rc == 0, _lib.last_error()
    torch.cuda.synchronize()
    return o, lse


def _cfg(tr, path, merge=_lib.PKV_MERGE_SEPARATE, plan=_lib.PKV_PLAN_SEPARATE, max_tasks=0):
    bucket = tr.n_max if path == _lib.PKV_PATH_BUCKETED_SPLIT else 0
    return api.make_cfg(path, tr.split_tokens, bucket, max_tasks, merge, plan)


def _matches(o, lse, o_ref, lse_ref, oref, lref, what):
    """Within the parity tolerance of pkv_decode_step's outputs and of the oracle."""
    x = o.float().cpu().numpy()
    ref = o_ref.float().cpu().numpy()
    assert np.all(np.abs(x - ref) <= ATOL + RTOL * np.abs(ref)), what
    assert np.max(np.abs(lse.cpu().numpy() - lse_ref.cpu().numpy())) <= LSE_ATOL, what
    close(o, oref, f"{what}: o against the oracle")
    close_lse(lse, lref)


@pytest.mark.parametrize("path,merge,plan", [(p, _lib.PKV_MERGE_SEPARATE, 0) for p in PATHS] +
                         [(p, _lib.PKV_MERGE_FUSED, 0) for p in PATHS[:2]] +
                         [(_lib.PKV_PATH_WORKQUEUE, _lib.PKV_MERGE_SEPARATE, _lib.PKV_PLAN_IN_DECODE)])
def test_noalloc_matches_decode_step_twice(lib, bimodal, path, merge, plan):
    """With the fused merge the header also holds the grid barrier's counters,
    which the call zeroes with the rest of the header, over whatever the
    previous call left there; with the plan built in the decode, the decode
    writes the plan into the same scratch."""
    tr, d, oref, lref = bimodal
    o_ref, lse_ref, _, _ = run_path(tr, d, path)
    cfg = _cfg(tr, path, merge, plan)
    for call in range(2):
        o, lse = _noalloc(lib, tr, d, cfg)
        _matches(o, lse, o_ref, lse_ref, oref, lref, f"call {call}")


def test_noalloc_after_a_workqueue_overflow(lib, bimodal):
    """Call 1 leaves the array's header dirty: a task capacity far below the
    batch's tasks makes the plan record an overflow (error word, overflow flag,
    zero task count) and the merge write NaN.  Call 2, with the capacity the
    batch needs, must not see any of it."""
    tr, d, oref, lref = bimodal
    o_ref, lse_ref, _, _ = run_path(tr, d, _lib.PKV_PATH_WORKQUEUE)
    o, _ = _noalloc(lib, tr, d, _cfg(tr, _lib.PKV_PATH_WORKQUEUE, max_tasks=8))
    assert torch.isnan(o.float()).all()  # the overflow's documented outputs
    for plan in (_lib.PKV_PLAN_SEPARATE, _lib.PKV_PLAN_IN_DECODE):
        o, lse = _noalloc(lib, tr, d, _cfg(tr, _lib.PKV_PATH_WORKQUEUE, plan=plan))
        _matches(o, lse, o_ref, lse_ref, oref, lref, f"after an overflow, plan mode {plan}")


def test_noalloc_after_a_timed_out_barrier(lib):
    """Call 1 runs the fused merge with the bounded-wait test hook: one CTA
    never fills its first stage, its wait gives up after about a second and the
    grid barrier's counters are left as the timeout found them.  Call 2 clears
    the header first and must merge correctly."""
    tr = T.make_trace(1)  # B=1, N=1024: the shape the fused-merge timeout test uses
    q = T.gen_q(tr)
    k, v = T.gen_kv(tr)
    d = upload(tr, q, k, v)
    oref, lref = oracle_out(tr, q, k, v)
    o_ref, lse_ref, _, _ = run_path(tr, d, _lib.PKV_PATH_BUCKETED_SPLIT)
    cfg = _cfg(tr, _lib.PKV_PATH_BUCKETED_SPLIT, merge=_lib.PKV_MERGE_FUSED)
    assert lib.pkv_test_starve_next_decodes(1) == 0, _lib.last_error()
    try:
        _noalloc(lib, tr, d, cfg)
    finally:
        lib.pkv_test_starve_next_decodes(0)
    o, lse = _noalloc(lib, tr, d, cfg)
    _matches(o, lse, o_ref, lse_ref, oref, lref, "after a timed-out barrier")


def test_noalloc_calls_after_the_first_allocate_nothing(lib, bimodal):
    """After one set-up call per configuration (which may load the library's
    kernels and the array onto the device), further calls leave the device's
    free memory exactly as it was."""
    tr, d, oref, lref = bimodal
    cfgs = [_cfg(tr, p) for p in PATHS] + [
        _cfg(tr, _lib.PKV_PATH_WORKQUEUE, plan=_lib.PKV_PLAN_IN_DECODE),
        _cfg(tr, _lib.PKV_PATH_WORKQUEUE, merge=_lib.PKV_MERGE_FUSED)]
    outs = [_outputs(tr) for _ in cfgs]
    for cfg, (o, lse) in zip(cfgs, outs):  # set-up
        assert _call(lib, tr, d, cfg, o, lse) == 0, _lib.last_error()
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        for cfg, (o, lse) in zip(cfgs, outs):
            assert _call(lib, tr, d, cfg, o, lse) == 0, _lib.last_error()
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    for o, lse in outs:
        close(o, oref, "o after the repeated calls")


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
