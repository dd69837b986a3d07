"""Routing plan: top-k expert ids -> grouped-contiguous row layout.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

What is computed (MoonEP PR #38, "fit planning block size to device SMEM
limit", background section: the planning kernel keeps a per-expert histogram
and per-warp scratch and places each routed row in its expert's column; its
correctness section checks every output against an independent reference and
against planning invariants.  humming PR #129, first section: the rows routed
to one expert form one contiguous range):

* flatten ``topk_ids[M, k]`` in row-major order: source index s = t*k + j;
* counts[e] = number of s whose id is e;
* ``expert_offsets`` = exclusive prefix sum of counts, length E+1, so expert e
  owns sorted rows [off[e], off[e+1]);
* a stable permutation: inside one expert, rows keep ascending s.
  ``sorted_to_src[r]`` is the s placed at sorted row r; ``src_to_sorted`` is
  its inverse.

Readings where the pages are silent: ties inside an expert are broken by
ascending s (a stable counting sort); ids outside [0, E) are dropped from the
layout (not counted, ``src_to_sorted[s] = -1``) and reported as a count.
"""
from __future__ import annotations

import numpy as np


def plan_expert_offsets(topk_ids: np.ndarray, E: int):
    """Return ``(expert_offsets[E+1], sorted_to_src[R'], src_to_sorted[R], n_invalid)``.

    ``R = M*k`` source rows; ``R'`` = number of in-range ids (= R when every
    id is in [0, E)).  ``sorted_to_src`` is padded with -1 up to length R so
    both permutation arrays have the caller's length R.
    """
    flat = np.asarray(topk_ids, dtype=np.int64).reshape(-1)
    R = flat.shape[0]
    valid = (flat >= 0) & (flat < E)
    counts = np.bincount(flat[valid], minlength=E).astype(np.int64)
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    src_valid = np.nonzero(valid)[0]
    order = np.argsort(flat[src_valid], kind="stable")
    sorted_src = src_valid[order]
    sorted_to_src = np.full(R, -1, dtype=np.int64)
    sorted_to_src[: sorted_src.shape[0]] = sorted_src
    src_to_sorted = np.full(R, -1, dtype=np.int64)
    src_to_sorted[sorted_src] = np.arange(sorted_src.shape[0], dtype=np.int64)
    n_invalid = int(R - sorted_src.shape[0])
    return (offsets.astype(np.int32), sorted_to_src.astype(np.int32),
            src_to_sorted.astype(np.int32), n_invalid)
