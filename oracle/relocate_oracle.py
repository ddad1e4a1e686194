"""CPU oracle for Tier-1 KV relocation — TEST INFRASTRUCTURE.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may use
this module.  It shares no code with the CUDA library.

What it computes.  On a token-granular pool (page_size=1) a request's KV rows
end up scattered after churn.  Tier-1 relocation ("Chunk 66.1", magik.net
seg_66/chunk_1: "Tier 1 (live relocation)", deferred there) moves them into
one contiguous region so that the contiguous fast path applies:

    for each request b with rows idx_b[0..n_b) and destination start d_b:
        pool[d_b + k] = pool[idx_b[k]]      (values as they were before the call)
        idx_b[k]      = d_b + k
    the old row numbers are returned so the caller can release them.

The pages give no more than the name and its purpose; the reading (the
caller's allocator picks each destination start, the destination rows must
not hold any row the batch reads, every index must lie in the pool, and a
call that breaks a rule changes nothing) is recorded in the design notes.
"""
from __future__ import annotations

from typing import Dict, Sequence

import torch


def relocation_errors(pool_rows: int, kv_indices: Sequence[int], kv_indptr: Sequence[int],
                      dest_base: Sequence[int]) -> Dict[str, bool]:
    """Which rule a call breaks: bad_index (an index outside the pool),
    bad_dest (a destination region outside the pool), overlap (destination
    regions overlap each other, or a row the batch reads lies in one)."""
    B = len(dest_base)
    bad_index = any(not (0 <= int(i) < pool_rows) for i in kv_indices)
    dest_rows = []
    bad_dest = False
    for b in range(B):
        n = int(kv_indptr[b + 1]) - int(kv_indptr[b])
        d = int(dest_base[b])
        if d < 0 or d + n > pool_rows:
            bad_dest = True
        dest_rows.extend(range(d, d + n))
    overlap = len(dest_rows) != len(set(dest_rows)) or bool(set(dest_rows) & {int(i) for i in kv_indices})
    return {"bad_index": bad_index, "bad_dest": bad_dest, "overlap": overlap}


def relocate(kv_pool: torch.Tensor, kv_indices: torch.Tensor, kv_indptr: torch.Tensor,
             dest_base: torch.Tensor):
    """Returns (new_pool, new_indices, old_indices, errors).  When any rule is
    broken the pool and the indices come back unchanged and old_indices is a
    copy of the indices."""
    pool_rows = int(kv_pool.shape[0])
    idx = [int(v) for v in kv_indices.tolist()]
    ptr = [int(v) for v in kv_indptr.tolist()]
    dst = [int(v) for v in dest_base.tolist()]
    err = relocation_errors(pool_rows, idx, ptr, dst)
    new_pool = kv_pool.clone()
    new_idx = kv_indices.clone()
    if any(err.values()):
        return new_pool, new_idx, kv_indices.clone(), err
    for b in range(len(dst)):
        for k in range(ptr[b + 1] - ptr[b]):
            new_pool[dst[b] + k] = kv_pool[idx[ptr[b] + k]]
            new_idx[ptr[b] + k] = dst[b] + k
    return new_pool, new_idx, kv_indices.clone(), err
