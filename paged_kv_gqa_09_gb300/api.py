"""Python binding of libpkv with the C ABI's names (argument marshalling only).

Device buffers are torch CUDA tensors (PyTorch provides memory and streams);
every step of the decode path runs in libpkv's kernels.  Each function checks
that its tensors live on the current CUDA device with the dtype and layout the
C ABI expects -- a host tensor handed to a kernel would fault -- then forwards
raw pointers and the current stream.
"""
from __future__ import annotations

import ctypes
import math
from typing import Optional, Sequence

import numpy as np
import torch

from . import _lib
from ._lib import (PKV_MERGE_FUSED, PKV_MERGE_SEPARATE, PKV_PATH_BUCKETED_SPLIT,
                   PKV_PATH_SINGLE_PASS, PKV_PATH_WORKQUEUE, PKV_PLAN_IN_DECODE,
                   PKV_PLAN_SEPARATE, PKV_SELF_PLAN_MAX_B, Counters,
                   PlanCfg, PolicyCfg, Shape, StepModel, check)

__all__ = [
    "Shape", "PlanCfg", "PolicyCfg", "make_shape", "make_cfg",
    "pkv_plan_workspace_size", "pkv_partials_size", "pkv_plan", "pkv_decode", "pkv_merge",
    "pkv_decode_merge", "PKV_MERGE_SEPARATE", "PKV_MERGE_FUSED", "PKV_PLAN_SEPARATE",
    "PKV_PLAN_IN_DECODE", "PKV_SELF_PLAN_MAX_B", "pkv_single_pass",
    "pkv_decode_step", "pkv_decode_step_noalloc",
    "pkv_decode_step_host", "pkv_append_decode_step_host", "pkv_decode_step_rows",
    "exact_length_buckets_step", "pkv_exact_length_groups", "pkv_append",
    "pkv_append_plan", "pkv_policy", "pkv_policy_default",
    "pkv_cost_model_default", "pkv_policy_learned",
    "pkv_get_counters", "pkv_reset_counters", "pkv_step_model", "pkv_get_error", "pkv_version",
    "PagedDecoder", "HostDecodeLoop",
]


# ------------------------------------------------------------------ helpers

def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dev(t: Optional[torch.Tensor], name: str, dtype: torch.dtype, nullable: bool = False) -> int:
    if t is None:
        if nullable:
            return 0
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (got {t.device})")
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"{name} is on {t.device}, current device is cuda:{torch.cuda.current_device()}")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype} (got {t.dtype})")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _ws(t: torch.Tensor, name: str = "workspace") -> int:
    if not (isinstance(t, torch.Tensor) and t.is_cuda and t.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    return t.data_ptr()


def make_shape(q: torch.Tensor, k_cache: torch.Tensor, block_table: torch.Tensor,
               scale: Optional[float] = None) -> Shape:
    """Shape from q [B,Hq,d], k_cache [num_pages,P,Hkv,d], block_table [B,bt_stride]."""
    B, Hq, d = q.shape
    num_pages, P, Hkv, d2 = k_cache.shape
    if d2 != d or block_table.shape[0] != B:
        raise ValueError("q, k_cache and block_table disagree on d or B")
    return Shape(B, Hq, Hkv, d, P, num_pages, int(block_table.shape[1]),
                 float(1.0 / math.sqrt(d) if scale is None else scale))


def make_cfg(path: int, split_tokens: int = 1024, bucket_len: int = 0, max_tasks: int = 0,
             merge: int = PKV_MERGE_SEPARATE, plan: int = PKV_PLAN_SEPARATE) -> PlanCfg:
    return PlanCfg(int(path), int(split_tokens), int(bucket_len), int(max_tasks), int(merge), int(plan))


# ------------------------------------------------------------------ C ABI

def pkv_version() -> int:
    return _lib.load().pkv_version()


def pkv_plan_workspace_size(shape: Shape, cfg: PlanCfg) -> int:
    n = _lib.load().pkv_plan_workspace_size(ctypes.byref(shape), ctypes.byref(cfg))
    if n == 0:
        raise _lib.PkvError(_lib.PKV_EINVAL, "pkv_plan_workspace_size", _lib.last_error())
    return int(n)


def pkv_partials_size(shape: Shape, cfg: PlanCfg) -> int:
    return int(_lib.load().pkv_partials_size(ctypes.byref(shape), ctypes.byref(cfg)))


def pkv_plan(shape, cfg, seq_lens, ws, stream=None) -> None:
    L = _lib.load()
    check(L.pkv_plan(ctypes.byref(shape), ctypes.byref(cfg), _dev(seq_lens, "seq_lens", torch.int32),
                     _ws(ws), _stream(stream)), "pkv_plan")


def pkv_decode(shape, cfg, ws, q, k_cache, v_cache, block_table, seq_lens, partials,
               stream=None) -> None:
    L = _lib.load()
    part = _dev(partials, "partials", torch.float32, nullable=shape.B == 0)
    check(L.pkv_decode(ctypes.byref(shape), ctypes.byref(cfg), _ws(ws),
                       _dev(q, "q", torch.float16), _dev(k_cache, "k_cache", torch.float16),
                       _dev(v_cache, "v_cache", torch.float16),
                       _dev(block_table, "block_table", torch.int32),
                       _dev(seq_lens, "seq_lens", torch.int32),
                       part, _stream(stream)), "pkv_decode")


def pkv_merge(shape, cfg, ws, seq_lens, partials, o, lse=None, stream=None) -> None:
    L = _lib.load()
    part = _dev(partials, "partials", torch.float32, nullable=shape.B == 0)
    check(L.pkv_merge(ctypes.byref(shape), ctypes.byref(cfg), _ws(ws),
                      _dev(seq_lens, "seq_lens", torch.int32), part, _dev(o, "o", torch.float16),
                      _dev(lse, "lse", torch.float32, nullable=True), _stream(stream)), "pkv_merge")


def pkv_decode_merge(shape, cfg, ws, q, k_cache, v_cache, block_table, seq_lens, partials, o,
                     lse=None, stream=None) -> None:
    L = _lib.load()
    part = _dev(partials, "partials", torch.float32, nullable=shape.B == 0)
    check(L.pkv_decode_merge(ctypes.byref(shape), ctypes.byref(cfg), _ws(ws),
                             _dev(q, "q", torch.float16), _dev(k_cache, "k_cache", torch.float16),
                             _dev(v_cache, "v_cache", torch.float16),
                             _dev(block_table, "block_table", torch.int32),
                             _dev(seq_lens, "seq_lens", torch.int32),
                             part, _dev(o, "o", torch.float16),
                             _dev(lse, "lse", torch.float32, nullable=True), _stream(stream)),
          "pkv_decode_merge")


def pkv_single_pass(shape, ws, q, k_cache, v_cache, block_table, seq_lens, o, lse=None,
                    stream=None) -> None:
    L = _lib.load()
    check(L.pkv_single_pass(ctypes.byref(shape), _ws(ws), _dev(q, "q", torch.float16),
                            _dev(k_cache, "k_cache", torch.float16),
                            _dev(v_cache, "v_cache", torch.float16),
                            _dev(block_table, "block_table", torch.int32),
                            _dev(seq_lens, "seq_lens", torch.int32), _dev(o, "o", torch.float16),
                            _dev(lse, "lse", torch.float32, nullable=True), _stream(stream)),
          "pkv_single_pass")


def pkv_decode_step(shape, cfg, ws, q, k_cache, v_cache, block_table, seq_lens, partials, o,
                    lse=None, stream=None) -> None:
    L = _lib.load()
    part = _dev(partials, "partials", torch.float32,
                nullable=cfg.path == PKV_PATH_SINGLE_PASS or shape.B == 0)
    check(L.pkv_decode_step(ctypes.byref(shape), ctypes.byref(cfg), _ws(ws),
                            _dev(q, "q", torch.float16), _dev(k_cache, "k_cache", torch.float16),
                            _dev(v_cache, "v_cache", torch.float16),
                            _dev(block_table, "block_table", torch.int32),
                            _dev(seq_lens, "seq_lens", torch.int32), part,
                            _dev(o, "o", torch.float16),
                            _dev(lse, "lse", torch.float32, nullable=True), _stream(stream)),
          "pkv_decode_step")


def pkv_decode_step_noalloc(shape, cfg, q, k_cache, v_cache, block_table, seq_lens, o, lse=None,
                            stream=None) -> None:
    """pkv_decode_step with the library's static scratch: for callers that
    cannot allocate device memory (see include/pkv.h for the size limit and the
    rules on overlapping calls)."""
    L = _lib.load()
    check(L.pkv_decode_step_noalloc(ctypes.byref(shape), ctypes.byref(cfg),
                                    _dev(q, "q", torch.float16),
                                    _dev(k_cache, "k_cache", torch.float16),
                                    _dev(v_cache, "v_cache", torch.float16),
                                    _dev(block_table, "block_table", torch.int32),
                                    _dev(seq_lens, "seq_lens", torch.int32),
                                    _dev(o, "o", torch.float16),
                                    _dev(lse, "lse", torch.float32, nullable=True),
                                    _stream(stream)), "pkv_decode_step_noalloc")


def pkv_decode_step_rows(shape, cfg, ws, rows, q, k_cache, v_cache, block_table, seq_lens,
                         partials, o, lse=None, stream=None) -> None:
    """Bucketed split step over the batch rows listed in `rows` (int32, device)."""
    L = _lib.load()
    check(L.pkv_decode_step_rows(ctypes.byref(shape), ctypes.byref(cfg), _ws(ws),
                                 _dev(rows, "rows", torch.int32), int(rows.numel()),
                                 _dev(q, "q", torch.float16), _dev(k_cache, "k_cache", torch.float16),
                                 _dev(v_cache, "v_cache", torch.float16),
                                 _dev(block_table, "block_table", torch.int32),
                                 _dev(seq_lens, "seq_lens", torch.int32),
                                 _dev(partials, "partials", torch.float32, nullable=shape.B == 0),
                                 _dev(o, "o", torch.float16),
                                 _dev(lse, "lse", torch.float32, nullable=True), _stream(stream)),
          "pkv_decode_step_rows")


def pkv_exact_length_groups(seq_lens_host) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """(rows, group_start, group_len) of the exact-length-bucket scheme from the
    host lengths (see include/pkv.h): group g is rows[group_start[g] :
    group_start[g + 1]] of length group_len[g]; rows[group_start[-1]:] have no
    tokens."""
    sl = np.ascontiguousarray(np.asarray(seq_lens_host, dtype=np.int32))
    B = sl.size
    rows = np.zeros(max(B, 1), np.int32)
    start = np.zeros(B + 1, np.int32)
    glen = np.zeros(max(B, 1), np.int32)
    ng = ctypes.c_int32()
    check(_lib.load().pkv_exact_length_groups(sl.ctypes.data, B, rows.ctypes.data, start.ctypes.data,
                                              glen.ctypes.data, ctypes.byref(ng)),
          "pkv_exact_length_groups")
    g = int(ng.value)
    return rows[:B], start[:g + 1], glen[:g]


def exact_length_buckets_step(q, k_cache, v_cache, block_table, seq_lens, seq_lens_host,
                              split_tokens: int, o, lse=None, ws=None, partials=None,
                              rows_cache: Optional[dict] = None, stream=None):
    """The exact-length-bucket scheme the compact workqueue replaces (Results,
    "Scheduling overhead"): one bucketed split + merge launch pair per distinct
    non-zero row length, each over the rows of that length (the groups come from
    pkv_exact_length_groups, every step), and one more pair over the rows of
    length 0, if any, which gives them o = 0, lse = -inf.  `seq_lens_host` is
    the host copy of the lengths.  With `rows_cache` the device row lists and
    launch arguments of a grouping seen before are reused.  Returns the number
    of launch pairs."""
    shape = make_shape(q, k_cache, block_table)
    rows, start, glen = pkv_exact_length_groups(seq_lens_host)
    key = (split_tokens, rows.tobytes(), start.tobytes(), shape.num_pages, shape.bt_stride)
    launches = rows_cache.get(key) if rows_cache is not None else None
    if launches is None:
        dev = q.device
        groups = [(int(glen[g]), rows[start[g]:start[g + 1]]) for g in range(glen.size)]
        if start[-1] < rows.size:
            groups.append((0, rows[start[-1]:]))  # no tokens: neutral states, o = 0
        launches = []
        for n, rws in groups:
            cfg = make_cfg(PKV_PATH_BUCKETED_SPLIT, split_tokens, n if n > 0 else split_tokens)
            sub = Shape(len(rws), shape.Hq, shape.Hkv, shape.d, shape.page_size, shape.num_pages,
                        shape.bt_stride, shape.scale)
            launches.append((cfg, torch.from_numpy(np.ascontiguousarray(rws)).to(dev),
                             pkv_partials_size(sub, cfg) // 4))
        if rows_cache is not None:
            rows_cache[key] = launches
    for cfg, rows_t, need_p in launches:
        part = partials if partials is not None and partials.numel() >= need_p else \
            torch.empty(max(need_p, 4), dtype=torch.float32, device=q.device)
        w = ws if ws is not None else torch.zeros(64, dtype=torch.uint8, device=q.device)
        pkv_decode_step_rows(shape, cfg, w, rows_t, q, k_cache, v_cache, block_table, seq_lens,
                             part, o, lse, stream)
    return len(launches)


def _host(t: Optional[torch.Tensor], name: str, dtype: torch.dtype, nullable: bool = False) -> int:
    if t is None:
        if nullable:
            return 0
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor) or t.is_cuda:
        raise ValueError(f"{name} must be a host (CPU) tensor")
    if t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {dtype} tensor")
    return t.data_ptr()


def pkv_decode_step_host(shape, cfg, ws, partials, h_q, q, h_block_table, block_table, h_seq_lens,
                         seq_lens, k_cache, v_cache, o, h_o, lse=None, h_lse=None,
                         stream=None) -> None:
    """One synchronized decode step with host inputs/outputs (see include/pkv.h)."""
    L = _lib.load()
    part = _dev(partials, "partials", torch.float32,
                nullable=cfg.path == PKV_PATH_SINGLE_PASS or shape.B == 0)
    check(L.pkv_decode_step_host(
        ctypes.byref(shape), ctypes.byref(cfg), _ws(ws), part, _host(h_q, "h_q", torch.float16),
        _dev(q, "q", torch.float16), _host(h_block_table, "h_block_table", torch.int32, True),
        _dev(block_table, "block_table", torch.int32),
        _host(h_seq_lens, "h_seq_lens", torch.int32, True), _dev(seq_lens, "seq_lens", torch.int32),
        _dev(k_cache, "k_cache", torch.float16), _dev(v_cache, "v_cache", torch.float16),
        _dev(o, "o", torch.float16), _host(h_o, "h_o", torch.float16),
        _dev(lse, "lse", torch.float32, nullable=True), _host(h_lse, "h_lse", torch.float32, True),
        _stream(stream)), "pkv_decode_step_host")


def pkv_append_decode_step_host(shape, cfg, ws, partials, h_q, q, h_k_new, h_v_new, k_new, v_new,
                                block_table, seq_lens, k_cache, v_cache, o, h_o, lse=None,
                                h_lse=None, free_pages=None, free_count=None, stream=None) -> None:
    """One synchronized serving-loop step with host q / new token in and o / lse
    out: append (allocating pages from the free list when given), decode, merge
    (see include/pkv.h)."""
    L = _lib.load()
    part = _dev(partials, "partials", torch.float32,
                nullable=cfg.path == PKV_PATH_SINGLE_PASS or shape.B == 0)
    check(L.pkv_append_decode_step_host(
        ctypes.byref(shape), ctypes.byref(cfg), _ws(ws), part, _host(h_q, "h_q", torch.float16),
        _dev(q, "q", torch.float16), _host(h_k_new, "h_k_new", torch.float16),
        _host(h_v_new, "h_v_new", torch.float16), _dev(k_new, "k_new", torch.float16),
        _dev(v_new, "v_new", torch.float16), _dev(block_table, "block_table", torch.int32),
        _dev(seq_lens, "seq_lens", torch.int32),
        _dev(free_pages, "free_pages", torch.int32, nullable=True),
        _dev(free_count, "free_count", torch.int32, nullable=True),
        _dev(k_cache, "k_cache", torch.float16), _dev(v_cache, "v_cache", torch.float16),
        _dev(o, "o", torch.float16), _host(h_o, "h_o", torch.float16),
        _dev(lse, "lse", torch.float32, nullable=True), _host(h_lse, "h_lse", torch.float32, True),
        _stream(stream)), "pkv_append_decode_step_host")


def pkv_append(shape, ws, k_new, v_new, block_table, seq_lens, k_cache, v_cache,
               stream=None) -> None:
    L = _lib.load()
    check(L.pkv_append(ctypes.byref(shape), _ws(ws), _dev(k_new, "k_new", torch.float16),
                       _dev(v_new, "v_new", torch.float16),
                       _dev(block_table, "block_table", torch.int32),
                       _dev(seq_lens, "seq_lens", torch.int32),
                       _dev(k_cache, "k_cache", torch.float16),
                       _dev(v_cache, "v_cache", torch.float16), _stream(stream)), "pkv_append")


def pkv_append_plan(shape, cfg, ws, k_new, v_new, block_table, seq_lens, k_cache, v_cache,
                    free_pages=None, free_count=None, stream=None) -> None:
    """Append one token per row (allocating pages from the free list when
    given), then build the workqueue plan -- one launch."""
    L = _lib.load()
    check(L.pkv_append_plan(ctypes.byref(shape), ctypes.byref(cfg), _ws(ws),
                            _dev(k_new, "k_new", torch.float16), _dev(v_new, "v_new", torch.float16),
                            _dev(block_table, "block_table", torch.int32),
                            _dev(seq_lens, "seq_lens", torch.int32),
                            _dev(free_pages, "free_pages", torch.int32, nullable=True),
                            _dev(free_count, "free_count", torch.int32, nullable=True),
                            _dev(k_cache, "k_cache", torch.float16),
                            _dev(v_cache, "v_cache", torch.float16), _stream(stream)),
          "pkv_append_plan")


def pkv_policy_default() -> PolicyCfg:
    c = PolicyCfg()
    _lib.load().pkv_policy_default(ctypes.byref(c))
    return c


def pkv_policy(B: int, n_max: int, cfg: Optional[PolicyCfg] = None) -> tuple[int, int]:
    path, split = ctypes.c_int32(), ctypes.c_int32()
    check(_lib.load().pkv_policy(int(B), int(n_max), ctypes.byref(cfg) if cfg is not None else None,
                                 ctypes.byref(path), ctypes.byref(split)), "pkv_policy")
    return int(path.value), int(split.value)


def pkv_cost_model_default() -> _lib.CostModel:
    m = _lib.CostModel()
    _lib.load().pkv_cost_model_default(ctypes.byref(m))
    return m


def pkv_policy_learned(B: int, n_max: int, n_sum: int,
                       model: Optional[_lib.CostModel] = None) -> tuple[int, int]:
    path, split = ctypes.c_int32(), ctypes.c_int32()
    check(_lib.load().pkv_policy_learned(int(B), int(n_max), int(n_sum),
                                         ctypes.byref(model) if model is not None else None,
                                         ctypes.byref(path), ctypes.byref(split)),
          "pkv_policy_learned")
    return int(path.value), int(split.value)


def pkv_get_counters() -> dict:
    c = Counters()
    check(_lib.load().pkv_get_counters(ctypes.byref(c)), "pkv_get_counters")
    return {name: int(getattr(c, name)) for name, _ in Counters._fields_}


def pkv_reset_counters() -> None:
    check(_lib.load().pkv_reset_counters(), "pkv_reset_counters")


def pkv_step_model(path: int, shape: Shape, split_tokens: int, bucket_len: int,
                   seq_lens: Sequence[int]) -> dict:
    sl = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32))
    out = StepModel()
    check(_lib.load().pkv_step_model(int(path), ctypes.byref(shape), int(split_tokens),
                                     int(bucket_len), sl.ctypes.data, ctypes.byref(out)),
          "pkv_step_model")
    return {name: int(getattr(out, name)) for name, _ in StepModel._fields_}


def pkv_get_error(ws: torch.Tensor, stream=None) -> tuple[int, str]:
    """Synchronize the stream and read/clear the device error word -> (status, detail)."""
    L = _lib.load()
    st = L.pkv_get_error(_ws(ws), _stream(stream))
    return int(st), (_lib.last_error() if st != 0 else "")


# ------------------------------------------------------------------ engine

class PagedDecoder:
    """Owns the workspace and partial-state buffers for one (shape, path) and
    runs whole decode steps: pkv_policy (host) then pkv_decode_step.  With
    `learned` (or a `cost_model`) the route comes from pkv_policy_learned, the
    cost model the pages name as future work, instead of the thresholds.

    Buffers come from the torch caching allocator on the current device and are
    reused across steps; they are resized when a larger configuration arrives.
    `merge` picks how split states are combined (a second kernel by default,
    or PKV_MERGE_FUSED: on the decode's tail) and `plan` where the workqueue's
    plan is built (by the decode kernel by default, for batches of up to
    PKV_SELF_PLAN_MAX_B rows; PKV_PLAN_SEPARATE: its own launch); the workspace
    is zeroed whenever the configuration changes, so that each configuration
    starts from a clean header.
    """

    def __init__(self, policy: Optional[PolicyCfg] = None, max_split_tasks: int = 0,
                 merge: int = PKV_MERGE_SEPARATE, plan: int = PKV_PLAN_IN_DECODE,
                 learned: bool = False, cost_model: Optional[_lib.CostModel] = None):
        self.policy = policy
        self.max_split_tasks = max_split_tasks
        self.merge = merge
        self.plan = plan
        self.learned = learned or cost_model is not None
        self.cost_model = cost_model
        self._ws: dict = {}
        self._part: dict = {}
        self._key: dict = {}

    def route(self, B: int, n_max: int, n_sum: Optional[int] = None) -> tuple[int, int]:
        """(path, split_tokens) for a batch: the calibrated thresholds, or with
        `learned` the cost model's fastest route, which also needs the batch's
        total tokens n_sum."""
        if not self.learned:
            return pkv_policy(B, n_max, self.policy)
        if n_sum is None:
            raise ValueError("the learned cost model needs n_sum, the batch's total tokens")
        return pkv_policy_learned(B, n_max, int(n_sum), self.cost_model)

    def plan_cfg(self, B: int, n_max: int, path: Optional[int] = None,
                 split_tokens: Optional[int] = None, n_sum: Optional[int] = None) -> PlanCfg:
        p, c = self.route(B, n_max, n_sum) if (path is None or split_tokens is None) else \
            (path, split_tokens)
        if path is not None:
            p = path
        if split_tokens is not None:
            c = split_tokens
        bucket = n_max if p == PKV_PATH_BUCKETED_SPLIT else 0
        return make_cfg(p, c, bucket, self.max_split_tasks if p == PKV_PATH_WORKQUEUE else 0,
                        self.merge, self.plan)

    def buffers(self, shape: Shape, cfg: PlanCfg, device) -> tuple[torch.Tensor, Optional[torch.Tensor]]:
        nws = pkv_plan_workspace_size(shape, cfg)
        npart = pkv_partials_size(shape, cfg)
        ws = self._ws.get(device)
        key = (tuple(getattr(shape, f) for f, _ in shape._fields_),
               tuple(getattr(cfg, f) for f, _ in cfg._fields_))
        if ws is None or ws.numel() < nws:
            ws = torch.zeros(max(nws, 64), dtype=torch.uint8, device=device)
            self._ws[device] = ws
        elif self._key.get(device) != key:
            ws.zero_()
        self._key[device] = key
        part = None
        if npart:
            part = self._part.get(device)
            if part is None or part.numel() * 4 < npart:
                part = torch.empty(npart // 4, dtype=torch.float32, device=device)
                self._part[device] = part
        return ws, part

    def step(self, q, k_cache, v_cache, block_table, seq_lens, n_max: int,
             path: Optional[int] = None, split_tokens: Optional[int] = None,
             o: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
             want_lse: bool = True, scale: Optional[float] = None, stream=None,
             n_sum: Optional[int] = None):
        """One decode step; n_max is the longest row and n_sum the total of the
        lengths (host scalars the caller knows; n_sum only for `learned`)."""
        shape = make_shape(q, k_cache, block_table, scale)
        cfg = self.plan_cfg(shape.B, int(n_max), path, split_tokens, n_sum)
        ws, part = self.buffers(shape, cfg, q.device)
        if o is None:
            o = torch.empty_like(q)
        if lse is None and want_lse:
            lse = torch.empty(q.shape[:2], dtype=torch.float32, device=q.device)
        pkv_decode_step(shape, cfg, ws, q, k_cache, v_cache, block_table, seq_lens, part, o, lse,
                        stream)
        return o, lse

    def workspace(self, device) -> Optional[torch.Tensor]:
        return self._ws.get(device)


class HostDecodeLoop:
    """A serving loop whose per-step inputs (q, block table, lengths) and outputs
    (o, lse) live in host memory while the KV cache stays on the device: one
    pkv_decode_step_host call per step (copies in, decode, copies out, sync).

    The shape and path are fixed at construction (policy route for the given
    B and n_max unless `path` is given); device staging buffers, the workspace
    and the partial-state buffer are allocated once; outputs land in pinned
    host tensors `h_o` and `h_lse`, reused across steps.

    With `append`, every captured step first writes one new K/V token per row
    (pinned staging `h_kn`, `h_vn` [B, Hkv, d]) into its page and advances the
    lengths, then decodes: the block table and lengths are device-resident
    state, loaded once by `set_state()` and advanced by the step's kernels.  On
    the workqueue the append is pkv_append_plan (which also plans unless the
    decode does), and with `free_pages` / `free_count` (device int32) a token
    that starts a page takes one from that free list.  `n_max` must then cover
    the lengths the loop will reach.  `merge` and `plan` choose the step's
    launches as in PagedDecoder.
    """

    def __init__(self, k_cache: torch.Tensor, v_cache: torch.Tensor, B: int, Hq: int, bt_stride: int,
                 n_max: int, path: Optional[int] = None, split_tokens: Optional[int] = None,
                 policy: Optional[PolicyCfg] = None, scale: Optional[float] = None,
                 max_tasks: int = 0, merge: int = PKV_MERGE_SEPARATE, inputs_in_place: bool = True,
                 append: bool = False, free_pages: Optional[torch.Tensor] = None,
                 free_count: Optional[torch.Tensor] = None, plan: int = PKV_PLAN_IN_DECODE):
        dev = k_cache.device
        self.inputs_in_place = inputs_in_place
        self.append = append
        if (free_pages is None) != (free_count is None):
            raise ValueError("free_pages and free_count go together")
        d = int(k_cache.shape[3])
        # the step's inputs (q | block table | lengths) and outputs (o | lse) each
        # live in one buffer, on the device and pinned on the host, so that a
        # step moves them with one copy each way
        a16 = lambda n: (n + 15) // 16 * 16
        qb, btb, slb = B * Hq * d * 2, B * bt_stride * 4, B * 4
        ob, lb = qb, B * Hq * 4
        in_sizes, out_sizes = [a16(qb), a16(btb), a16(slb)], [a16(ob), a16(lb)]
        self.d_in = torch.empty(sum(in_sizes), dtype=torch.uint8, device=dev)
        self.h_in = torch.empty(sum(in_sizes), dtype=torch.uint8).pin_memory()
        self.d_out = torch.empty(sum(out_sizes), dtype=torch.uint8, device=dev)
        self.h_out = torch.empty(sum(out_sizes), dtype=torch.uint8).pin_memory()

        def views(buf, sizes, specs):
            out, off = [], 0
            for size, (n, dtype, shape) in zip(sizes, specs):
                out.append(buf[off:off + n].view(dtype).view(shape))
                off += size
            return out

        in_specs = [(qb, torch.float16, (B, Hq, d)), (btb, torch.int32, (B, bt_stride)),
                    (slb, torch.int32, (B,))]
        out_specs = [(ob, torch.float16, (B, Hq, d)), (lb, torch.float32, (B, Hq))]
        self.q, self.bt, self.sl = views(self.d_in, in_sizes, in_specs)
        self.h_q, self.h_bt, self.h_sl = views(self.h_in, in_sizes, in_specs)
        self.o, self.lse = views(self.d_out, out_sizes, out_specs)
        self.h_o, self.h_lse = views(self.h_out, out_sizes, out_specs)
        self.shape = make_shape(self.q, k_cache, self.bt, scale)
        p, c = pkv_policy(B, n_max, policy)
        if path is not None:
            p = path
        if split_tokens is not None:
            c = split_tokens
        self.cfg = make_cfg(p, c, n_max if p == PKV_PATH_BUCKETED_SPLIT else 0,
                            max_tasks if p == PKV_PATH_WORKQUEUE else 0, merge, plan)
        self.ws = torch.zeros(pkv_plan_workspace_size(self.shape, self.cfg), dtype=torch.uint8, device=dev)
        npart = pkv_partials_size(self.shape, self.cfg)
        self.partials = torch.empty(max(npart // 4, 4), dtype=torch.float32, device=dev) if npart else None
        self.k, self.v = k_cache, v_cache
        if append:
            if free_pages is not None and p != PKV_PATH_WORKQUEUE:
                raise ValueError("device page allocation comes with the workqueue's fused append")
            hkv = int(k_cache.shape[2])
            self.h_new = torch.empty((2, B, hkv, d), dtype=torch.float16).pin_memory()
            self.d_new = torch.empty((2, B, hkv, d), dtype=torch.float16, device=dev)
            self.h_kn, self.h_vn = self.h_new[0], self.h_new[1]
            self.free_pages = _dev(free_pages, "free_pages", torch.int32, nullable=True)
            self.free_count = _dev(free_count, "free_count", torch.int32, nullable=True)
            self._free = (free_pages, free_count)  # keeps them alive
        self._fn = _lib.load().pkv_decode_step_host
        self._refs = (ctypes.byref(self.shape), ctypes.byref(self.cfg))
        self._graph = None
        self._graph_stream = None

    def step(self, h_q: torch.Tensor, h_block_table: Optional[torch.Tensor] = None,
             h_seq_lens: Optional[torch.Tensor] = None, stream=None):
        """Run one synchronized step; returns the pinned host (o, lse)."""
        st = _stream(stream)
        rc = self._fn(self._refs[0], self._refs[1], self.ws.data_ptr(),
                      self.partials.data_ptr() if self.partials is not None else None,
                      h_q.data_ptr(), self.q.data_ptr(),
                      h_block_table.data_ptr() if h_block_table is not None else None,
                      self.bt.data_ptr(),
                      h_seq_lens.data_ptr() if h_seq_lens is not None else None, self.sl.data_ptr(),
                      self.k.data_ptr(), self.v.data_ptr(), self.o.data_ptr(), self.h_o.data_ptr(),
                      self.lse.data_ptr(), self.h_lse.data_ptr(), st)
        check(rc, "pkv_decode_step_host")
        return self.h_o, self.h_lse

    def set_state(self, h_block_table: torch.Tensor, h_seq_lens: torch.Tensor) -> None:
        """Append mode: load the block table and lengths the step's kernels then
        advance on the device (synchronous)."""
        self.bt.copy_(h_block_table)
        self.sl.copy_(h_seq_lens)
        torch.cuda.synchronize(self.bt.device)

    def capture(self, stream: Optional[torch.cuda.Stream] = None) -> None:
        """Capture one whole host step as a CUDA graph: the step's kernels, the
        last of which writes o and lse straight into the pinned `h_o`, `h_lse`
        (page-locked host memory is addressable from kernels under unified
        addressing, so no copy back is needed).  With `inputs_in_place` the
        kernels also read the pinned inputs `h_q`, `h_bt`, `h_sl` where they are;
        otherwise one copy moves them to the device first.  In place every split
        of a row re-reads its q rows, and every kv head its block-table entries,
        over the host link; those reads overlap the KV stream (on GB300 in place
        measured no slower than the copy from B=1 to B=64).  Afterwards each step is
        `step_graph()`: write the inputs into the staging tensors, one graph
        launch, one synchronize.  Capture needs a non-default stream.  The
        capture runs the step once eagerly first: in append mode that is a real
        step, appending the token staged in `h_kn`, `h_vn`."""
        st = stream if stream is not None else torch.cuda.current_stream()
        if st.cuda_stream == torch.cuda.default_stream(st.device).cuda_stream:
            raise ValueError("capture needs a non-default stream")
        L = _lib.load()
        part = self.partials.data_ptr() if self.partials is not None else None

        src = (self.h_q, self.h_bt, self.h_sl) if self.inputs_in_place else (self.q, self.bt, self.sl)
        if self.append:  # table and lengths are device state; q and the new tokens come in
            new = self.h_new if self.inputs_in_place else self.d_new
            src = (self.h_q if self.inputs_in_place else self.q, self.bt, self.sl)
        sref, cref = self._refs
        ho, hl = self.h_o.data_ptr(), self.h_lse.data_ptr()

        def body():
            if not self.inputs_in_place:
                if self.append:
                    self.q.copy_(self.h_q, non_blocking=True)
                    self.d_new.copy_(self.h_new, non_blocking=True)
                else:
                    self.d_in.copy_(self.h_in, non_blocking=True)
            q_, bt_, sl_ = (t.data_ptr() for t in src)
            if self.append and self.cfg.path == PKV_PATH_WORKQUEUE:
                check(L.pkv_append_plan(sref, cref, self.ws.data_ptr(), new[0].data_ptr(),
                                        new[1].data_ptr(), bt_, sl_, self.free_pages,
                                        self.free_count, self.k.data_ptr(), self.v.data_ptr(),
                                        st.cuda_stream), "pkv_append_plan")
                if self.cfg.merge == PKV_MERGE_FUSED:
                    check(L.pkv_decode_merge(sref, cref, self.ws.data_ptr(), q_, self.k.data_ptr(),
                                             self.v.data_ptr(), bt_, sl_, part, ho, hl, st.cuda_stream),
                          "pkv_decode_merge")
                else:
                    check(L.pkv_decode(sref, cref, self.ws.data_ptr(), q_, self.k.data_ptr(),
                                       self.v.data_ptr(), bt_, sl_, part, st.cuda_stream), "pkv_decode")
                    check(L.pkv_merge(sref, cref, self.ws.data_ptr(), sl_, part, ho, hl,
                                      st.cuda_stream), "pkv_merge")
                return
            if self.append:
                check(L.pkv_append(sref, self.ws.data_ptr(), new[0].data_ptr(), new[1].data_ptr(),
                                   bt_, sl_, self.k.data_ptr(), self.v.data_ptr(), st.cuda_stream),
                      "pkv_append")
            check(L.pkv_decode_step(sref, cref, self.ws.data_ptr(), q_, self.k.data_ptr(),
                                    self.v.data_ptr(), bt_, sl_, part, ho, hl, st.cuda_stream),
                  "pkv_decode_step")

        with torch.cuda.stream(st):
            body()  # an eager step first (binds lazily-created state)
            st.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=st):
                body()
        self._graph, self._graph_stream = g, st

    def step_graph(self):
        """Replay the captured step and wait for it; returns the pinned (o, lse)."""
        if self._graph is None:
            raise RuntimeError("capture() first")
        # a graph replays on the current stream: it must be the capture stream,
        # so that the synchronize below waits for this very replay (switching
        # costs a few microseconds, so only when needed)
        if torch.cuda.current_stream().cuda_stream == self._graph_stream.cuda_stream:
            self._graph.replay()
        else:
            with torch.cuda.stream(self._graph_stream):
                self._graph.replay()
        self._graph_stream.synchronize()
        return self.h_o, self.h_lse
