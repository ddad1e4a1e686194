"""CPU oracle for reading a flattened custom tree mask — TEST INFRASTRUCTURE.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may use
this module.  It shares no code with the CUDA library.

What it computes.  A serving framework hands verify attention a flattened
boolean mask instead of a parent array: for request b, a row-major
[T, P_b + T] array whose entry (i, k) says whether tree node i may attend key
k (k < P_b: a prefix row; k >= P_b: tree node k - P_b).  The pages built this
mask on the host ("Chunk 66.1": the mask-build took 0.18 ms); the verify
kernels here want the tree itself.  For a tree mask the visible tree nodes of
node i are i and its ancestors, and the ancestors have smaller indices along
the chain, so

    parent(i) = the largest j < i that node i sees, or -1 if it sees none,

and the mask is a tree mask exactly when every node sees itself, every node
sees all prefix rows, and node i sees precisely {i} plus what parent(i) sees.
A mask that breaks one of these is reported as such (the kernels cannot
express it) and its parent row is still derived by the rule above.
"""
from __future__ import annotations

from typing import Dict, List, Sequence

import numpy as np


def tree_from_mask(mask_rows: np.ndarray, prefix_len: int) -> Dict[str, object]:
    """One request: ``mask_rows`` [T, P + T] of 0/1.  Returns parents,
    the visible tree set of each node (as a sorted list) and the three checks."""
    m = np.asarray(mask_rows).astype(bool)
    T = m.shape[0]
    P = int(prefix_len)
    assert m.shape[1] == P + T
    sees = [set(int(j) for j in np.nonzero(m[i, P:])[0]) for i in range(T)]
    parents: List[int] = []
    for i in range(T):
        below = [j for j in sees[i] if j < i]
        parents.append(max(below) if below else -1)
    self_ok = all(i in sees[i] for i in range(T))
    prefix_ok = bool(m[:, :P].all()) if P > 0 else True
    chain_ok = all(sees[i] == ({i} | (sees[parents[i]] if parents[i] >= 0 else set())) for i in range(T))
    return {"parents": parents, "sees": [sorted(s) for s in sees],
            "self_ok": self_ok, "prefix_ok": prefix_ok, "chain_ok": chain_ok,
            "valid": self_ok and prefix_ok and chain_ok}


def trees_from_flat_mask(flat: np.ndarray, mask_indptr: Sequence[int], prefix_lens: Sequence[int],
                         n_nodes: int) -> Dict[str, object]:
    """All requests: ``flat`` is the concatenation of the per-request row-major
    masks, request b starting at element ``mask_indptr[b]``.  Returns
    parents [B, T] and a per-request validity flag."""
    B = len(prefix_lens)
    T = n_nodes
    parents = np.zeros((B, T), np.int64)
    valid = np.zeros(B, bool)
    for b in range(B):
        P = int(prefix_lens[b])
        start = int(mask_indptr[b])
        rows = np.asarray(flat[start:start + T * (P + T)]).reshape(T, P + T)
        r = tree_from_mask(rows, P)
        parents[b] = r["parents"]
        valid[b] = r["valid"]
    return {"parents": parents, "valid": valid}
