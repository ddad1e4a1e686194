"""CPU oracle for greedy DDTree acceptance and KV commit — TEST INFRASTRUCTURE.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may use
this module.  It shares no code with the CUDA library.

What it computes.  After the verify forward, the target model has scored the
draft tree: ``logits[0]`` is its prediction at the end of the prefix (for the
children of the prefix end, the roots) and ``logits[1 + i]`` its prediction
after tree node ``i``.  Greedy acceptance walks the tree from the prefix end:

    cur = prefix end;  y = argmax(logits[0])
    while some child c of cur has draft[c] == y:
        take the smallest such c;  accept c;  cur = c;  y = argmax(logits[1 + c])
    next_token = y                         (the target's own token after the path)

The accepted nodes' KV rows become committed context in path order; the other
tree rows are released.  ``argmax`` takes the first index among equal maxima.

Sources: "Chunk 66.0" (magik.net seg_66/chunk_0) reports the DDTree commit
length (7-8 tokens per step with predictable text, 1 with hard text) — the
number of tokens a verify step commits.  The pages do not spell out the
acceptance rule; the greedy walk above (the target's argmax must equal the
drafted token at every step, smallest node index on a tie between siblings,
the final argmax is the extra committed token) is the plain reading, recorded
with the other readings in the design notes.  ``argmax(logits).item()`` as the
sampling step appears in the capture-safety inventory of page 3.
"""
from __future__ import annotations

from typing import Dict, List, Sequence, Tuple

import numpy as np
import torch


def argmax_rows(logits: torch.Tensor) -> np.ndarray:
    """First index of the maximum of each row (last dimension), compared as
    float64 values of the given (bf16) logits."""
    x = logits.detach().to(torch.float64).cpu().numpy()
    return np.argmax(x, axis=-1).astype(np.int64)


def children(parent: Sequence[int], node: int) -> List[int]:
    """Children of ``node`` (-1 = the prefix end) in increasing node order."""
    return [c for c, p in enumerate(parent) if int(p) == node]


def greedy_path(pred: Sequence[int], draft: Sequence[int], parent: Sequence[int]) -> Tuple[List[int], int]:
    """The greedy walk.  ``pred[0]`` is the argmax at the prefix end and
    ``pred[1 + i]`` the argmax after node i.  Returns (accepted nodes in path
    order, next token)."""
    cur, y = -1, int(pred[0])
    path: List[int] = []
    while True:
        hit = [c for c in children(parent, cur) if int(draft[c]) == y]
        if not hit:
            return path, y
        cur = hit[0]
        path.append(cur)
        y = int(pred[1 + cur])


def accept_request(logits: torch.Tensor, draft: Sequence[int], parent: Sequence[int],
                   tree_rows: Sequence[int]) -> Dict[str, object]:
    """One request: ``logits`` [T+1, V], ``draft`` and ``parent`` [T], and
    ``tree_rows`` [T], the KV pool rows of the tree nodes in node order.

    Returns accept_len, path, next_token, commit (pool rows of the accepted
    nodes in path order) and freed (pool rows of the other nodes in node
    order)."""
    pred = argmax_rows(logits)
    path, nxt = greedy_path(pred, draft, parent)
    on_path = set(path)
    return {
        "accept_len": len(path),
        "path": path,
        "next_token": nxt,
        "commit": [int(tree_rows[i]) for i in path],
        "freed": [int(tree_rows[i]) for i in range(len(parent)) if i not in on_path],
    }


def accept_batched(logits: torch.Tensor, draft: torch.Tensor, parent: torch.Tensor,
                   kv_indices: torch.Tensor, kv_indptr: torch.Tensor,
                   prefix_lens: torch.Tensor) -> Dict[str, np.ndarray]:
    """All requests, in the padded layouts the device entry point writes:
    accept_len [B], next_token [B], accepted_nodes [B, T] (-1 padded),
    commit_indices [B, T] and freed_indices [B, T] (-1 padded)."""
    B, T = parent.shape
    out = {
        "accept_len": np.zeros(B, np.int64),
        "next_token": np.zeros(B, np.int64),
        "accepted_nodes": np.full((B, T), -1, np.int64),
        "commit_indices": np.full((B, T), -1, np.int64),
        "freed_indices": np.full((B, T), -1, np.int64),
    }
    for b in range(B):
        base = int(kv_indptr[b]) + int(prefix_lens[b])
        rows = [int(v) for v in kv_indices[base:base + T].tolist()]
        r = accept_request(logits[b], draft[b].tolist(), parent[b].tolist(), rows)
        n = r["accept_len"]
        out["accept_len"][b] = n
        out["next_token"][b] = r["next_token"]
        out["accepted_nodes"][b, :n] = r["path"]
        out["commit_indices"][b, :n] = r["commit"]
        out["freed_indices"][b, :T - n] = r["freed"]
    return out
