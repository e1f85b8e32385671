"""The workqueue's balance order, written from its definition (not a test module).

"PersistentKV: Page-Aware Decode Scheduling for Long-Context LLM Serving on
Commodity GPUs", technical summary, Methodology 1, "Compact workqueue": the
plan's tasks are the non-empty (row, kv head, split) intervals; the library
also writes them in the order its decode CTAs claim them, and these helpers
state that order so the tests can check both the plan kernel and the
self-planning decode against it:
  1. every full-length split (C tokens), by row, then split, then kv head;
  2. every shorter last split (N_i mod C tokens), by length class
     floor(8 * (N_i mod C) / C) from the longest class down, then by row,
     then kv head.
"""
import numpy as np

SHORT_CLASSES = 8


def short_class(r, C):
    """Length class of a shorter split of r tokens (0 < r < C)."""
    return (np.asarray(r, dtype=np.int64) * SHORT_CLASSES) // C


def short_rows(lens, C):
    """The rows that end in a shorter split, in balance order."""
    lens = np.clip(np.asarray(lens, dtype=np.int64), 0, None)
    rows = np.flatnonzero(lens % C != 0)
    cls = short_class(lens[rows] % C, C)
    return rows[np.lexsort((rows, -cls))]


def balance_order(want, lens, C):
    """Indices into the canonical task list `want` ({row, kv head, split,
    slot} records in (row, kv head, split) order) in balance order."""
    want = np.asarray(want)
    if not len(want):
        return np.zeros(0, dtype=np.int64)
    lens = np.clip(np.asarray(lens, dtype=np.int64), 0, None)
    n = -(-lens // C)
    row, g, j = want[:, 0], want[:, 1], want[:, 2]
    short = (lens[row] % C != 0) & (j == n[row] - 1)
    full = np.flatnonzero(~short)
    full = full[np.lexsort((g[full], j[full], row[full]))]
    sh = np.flatnonzero(short)
    cls = short_class(lens[row[sh]] % C, C)
    sh = sh[np.lexsort((g[sh], row[sh], -cls))]
    return np.concatenate([full, sh]).astype(np.int64)
