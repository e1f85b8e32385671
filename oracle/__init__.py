"""float64 CPU oracle for paged-KV GQA decode attention (test infrastructure).

Only the tests, the package smoke check and the benchmark's CPU-baseline leg
may import this module.  The product path never does; the oracle shares no
code with the CUDA library (see ``pkv_oracle.c`` for the passages followed
and the readings taken).

The C source is compiled with gcc into ``oracle/_build/liboracle.so`` by
:func:`build` (called from ``__graft_entry__.build()`` and, lazily, on first
use).  Arrays are exchanged as numpy buffers: fp16 inputs are passed as their
raw uint16 bits and converted to double inside the oracle.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lib: Optional[ctypes.CDLL] = None

OK, EBADARG, EBADPAGE, ETOOLONG, ENOMEM = 0, -1, -2, -3, -4

PATH_BUCKETED, PATH_WORKQUEUE, PATH_SINGLE, PATH_EXACT_BUCKETS = 0, 1, 2, 3


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP when available); returns the .so path."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        # a planted-mistake copy of the oracle (tests/test_oracle_mutants.py) is
        # loaded from here instead of the real build
        path = os.environ.get("PKV_ORACLE_LIB") or build()
        L = ctypes.CDLL(path)
        i32, i64, f64, vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
        L.pkvo_half_to_double.argtypes = [ctypes.c_uint16]
        L.pkvo_half_to_double.restype = f64
        L.pkvo_half_array_to_double.argtypes = [vp, vp, i64]
        L.pkvo_half_array_to_double.restype = None
        L.pkvo_max_threads.argtypes = []
        L.pkvo_max_threads.restype = ctypes.c_int
        L.pkvo_attention.argtypes = [i32] * 7 + [f64] + [vp] * 7 + [i32]
        L.pkvo_attention.restype = ctypes.c_int
        L.pkvo_plan_compact.argtypes = [i32, i32, i32, i32, vp, vp, i64, vp]
        L.pkvo_plan_compact.restype = i64
        L.pkvo_plan_rect.argtypes = [i32, i32, i32, i32, i32, vp, vp, i64, vp]
        L.pkvo_plan_rect.restype = i64
        L.pkvo_partials.argtypes = ([i32] * 7 + [f64] + [vp] * 5 + [i32, i32, i32]
                                    + [vp] * 3 + [i64, i32])
        L.pkvo_partials.restype = ctypes.c_int
        L.pkvo_merge.argtypes = [i32] * 6 + [vp] * 6
        L.pkvo_merge.restype = ctypes.c_int
        L.pkvo_counters.argtypes = [i32] * 7 + [vp, vp]
        L.pkvo_counters.restype = ctypes.c_int
        _lib = L
    return _lib


def _p(a: np.ndarray) -> int:
    return a.ctypes.data


def _bits(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a)
    assert a.dtype == np.float16, a.dtype
    return a.view(np.uint16)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


class OracleError(RuntimeError):
    pass


def _check(rc: int, what: str) -> None:
    if rc != OK:
        raise OracleError(f"{what} failed with status {rc}")


def max_threads() -> int:
    return int(lib().pkvo_max_threads())


def half_to_double(bits: np.ndarray) -> np.ndarray:
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(bits.shape, dtype=np.float64)
    lib().pkvo_half_array_to_double(_p(bits), _p(out), bits.size)
    return out


def attention(q, k_cache, v_cache, block_table, seq_lens, scale: float,
              nthreads: int = 0):
    """Plain float64 paged GQA decode attention -> (o [B,Hq,d], lse [B,Hq])."""
    qb, kb, vb = _bits(q), _bits(k_cache), _bits(v_cache)
    bt, sl = _i32(block_table), _i32(seq_lens)
    B, Hq, d = qb.shape
    num_pages, P, Hkv, d2 = kb.shape
    assert d2 == d and vb.shape == kb.shape and bt.shape[0] == B and sl.shape == (B,)
    o = np.empty((B, Hq, d), dtype=np.float64)
    lse = np.empty((B, Hq), dtype=np.float64)
    rc = lib().pkvo_attention(B, Hq, Hkv, d, P, num_pages, bt.shape[1], float(scale),
                              _p(qb), _p(kb), _p(vb), _p(bt), _p(sl), _p(o), _p(lse),
                              int(nthreads))
    _check(rc, "pkvo_attention")
    return o, lse


def plan_compact(seq_lens, Hq: int, Hkv: int, C: int):
    """Canonical compact workqueue -> (tasks int32 [T,4], offsets int32 [B+1])."""
    sl = _i32(seq_lens)
    B = sl.shape[0]
    offsets = np.empty(B + 1, dtype=np.int32)
    T = lib().pkvo_plan_compact(B, Hq, Hkv, C, _p(sl), None, 0, _p(offsets))
    if T < 0:
        _check(int(T), "pkvo_plan_compact")
    tasks = np.empty((max(T, 1), 4), dtype=np.int32)
    T2 = lib().pkvo_plan_compact(B, Hq, Hkv, C, _p(sl), _p(tasks), T, _p(offsets))
    assert T2 == T
    return tasks[:T], offsets


def plan_rect(seq_lens, Hq: int, Hkv: int, C: int, S_b: int):
    """Rectangular bucketed grid -> (tasks int32 [B*Hkv*S_b,4], empty int32 [...])."""
    sl = _i32(seq_lens)
    B = sl.shape[0]
    T = B * Hkv * S_b
    tasks = np.empty((max(T, 1), 4), dtype=np.int32)
    empty = np.empty(max(T, 1), dtype=np.int32)
    T2 = lib().pkvo_plan_rect(B, Hq, Hkv, C, S_b, _p(sl), _p(tasks), T, _p(empty))
    if T2 < 0:
        _check(int(T2), "pkvo_plan_rect")
    assert T2 == T
    return tasks[:T], empty[:T]


def n_slots(seq_lens, Hq: int, C: int, rect: bool, S_b: int = 0) -> int:
    sl = np.asarray(seq_lens, dtype=np.int64)
    if rect:
        return int(sl.shape[0]) * S_b * Hq
    return int(((sl + C - 1) // C).sum()) * Hq


def partials(q, k_cache, v_cache, block_table, seq_lens, scale: float, C: int,
             rect: bool = False, S_b: int = 0, nthreads: int = 0):
    """Per-split partial states (m [slots], l [slots], acc [slots, d]) in float64."""
    qb, kb, vb = _bits(q), _bits(k_cache), _bits(v_cache)
    bt, sl = _i32(block_table), _i32(seq_lens)
    B, Hq, d = qb.shape
    num_pages, P, Hkv, _ = kb.shape
    ns = n_slots(sl, Hq, C, rect, S_b)
    m = np.empty(max(ns, 1), dtype=np.float64)
    l = np.empty(max(ns, 1), dtype=np.float64)
    acc = np.empty((max(ns, 1), d), dtype=np.float64)
    rc = lib().pkvo_partials(B, Hq, Hkv, d, P, num_pages, bt.shape[1], float(scale),
                             _p(qb), _p(kb), _p(vb), _p(bt), _p(sl), C, int(rect), S_b,
                             _p(m), _p(l), _p(acc), ns, int(nthreads))
    _check(rc, "pkvo_partials")
    return m[:ns], l[:ns], acc[:ns]


def merge(m, l, acc, seq_lens, Hq: int, C: int, rect: bool = False, S_b: int = 0):
    """Exact LSE merge of partial states -> (o [B,Hq,d], lse [B,Hq])."""
    m = np.ascontiguousarray(m, dtype=np.float64)
    l = np.ascontiguousarray(l, dtype=np.float64)
    acc = np.ascontiguousarray(acc, dtype=np.float64)
    sl = _i32(seq_lens)
    B = sl.shape[0]
    d = acc.shape[1]
    o = np.empty((B, Hq, d), dtype=np.float64)
    lse = np.empty((B, Hq), dtype=np.float64)
    rc = lib().pkvo_merge(B, Hq, d, C, int(rect), S_b, _p(sl), _p(m), _p(l), _p(acc),
                          _p(o), _p(lse))
    _check(rc, "pkvo_merge")
    return o, lse


@dataclass
class Counters:
    attn_launches: int
    plan_launches: int
    tasks: int
    grid_tasks: int
    states_written: int
    states_read: int
    merge_state_bytes: int
    kv_bytes: int


def counters(path: int, seq_lens, Hq: int, Hkv: int, d: int, C: int, S_b: int = 0) -> Counters:
    """Launch and traffic model of one decode step (see pkvo_counters)."""
    sl = _i32(seq_lens)
    buf = np.zeros(8, dtype=np.int64)
    rc = lib().pkvo_counters(path, sl.shape[0], Hq, Hkv, d, C, S_b, _p(sl), _p(buf))
    _check(rc, "pkvo_counters")
    return Counters(*[int(x) for x in buf])
