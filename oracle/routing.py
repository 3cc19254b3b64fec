"""Routing of (token, k) assignments to experts -- plain definitions.

Follows the dispatch steps that the DeepGEMM SM90 MegaMoE dev log lists in
its Phase 2 entry (count each expert's assignments, record for every slot
which token and top-k position it came from), restricted to one GPU:

* counts[e]   = number of assignments (t, j) with topk_idx[t, j] == e;
* offsets[e]  = sum of counts[e'] for e' < e  (offsets has E + 1 entries);
* perm[slot]  = the flat index t*k + j of the assignment stored at ``slot``;
  within one expert the assignments keep ascending flat order (stable), so
  the permutation is unique;
* inv[t*k+j]  = its slot, or -1 for an empty slot (topk_idx == -1).

topk_idx == -1 marks an empty slot; any other value outside [0, E) is an
error.
"""
from __future__ import annotations

import numpy as np


def check_indices(topk_idx, E: int) -> np.ndarray:
    flat = np.asarray(topk_idx, dtype=np.int64).reshape(-1)
    bad = (flat < -1) | (flat >= E)
    if np.any(bad):
        raise ValueError(f"topk_idx outside [-1, {E}) at flat index {int(np.argmax(bad))}")
    return flat


def route(topk_idx, E: int):
    """Return (counts[E], offsets[E+1], perm[n_valid], inv[T*k]) as int64 arrays."""
    flat = check_indices(topk_idx, E)
    valid = flat >= 0
    counts = np.bincount(flat[valid], minlength=E).astype(np.int64)
    offsets = np.zeros(E + 1, dtype=np.int64)
    np.cumsum(counts, out=offsets[1:])
    key = np.where(valid, flat, E)                 # empty slots sort after every expert
    order = np.argsort(key, kind="stable")
    n_valid = int(valid.sum())
    perm = order[:n_valid].astype(np.int64)
    inv = np.full(flat.shape[0], -1, dtype=np.int64)
    inv[perm] = np.arange(n_valid, dtype=np.int64)
    return counts, offsets, perm, inv
