"""Float64 CPU oracle for DDTree verify attention (MLA, absorbed form).

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
link this package; only the tests, the smoke check and the benchmark's CPU
baseline leg do.  It shares no code with the CUDA library.

What it computes (the plain definition, no blocking or online softmax):

  For request b with prefix length P, index list idx (P prefix rows then the
  T draft-tree rows in node order) and parents ``parent`` (-1 = root that
  hangs off the prefix end, otherwise parent[i] < i):

    anc*(i)  = {i} u anc*(parent[i])          (empty past -1)
    K(i)     = {idx[0..P-1]} u {idx[P+j] : j in anc*(i)}
    s_k      = sm_scale * (q_lat[i,h] . pool[k, :512] + q_rope[i,h] . pool[k, 512:])
    O[i,h]   = sum_k softmax(s)_k * pool[k, :512]      (k in K(i))
    LSE[i,h] = ln sum_k exp(s_k)

Sources: "DDTree verify attention" is the target-model forward that scores
every node of the drafter's token tree in one pass (magik.net, "Chunk 66.0":
verify attention locked to Triton MLA at page_size=1; "Chunk 66.1": the
mask-build on the host and the owned verify kernel).  The pages do not write
the formula out; the reading above (self-attention to the node itself, roots
under the prefix end, tree rows last in the index list, natural-log LSE with
the scale inside) is the plain reading recorded in the design notes.  The
split/merge identity in :func:`merge_partials` is the "partial+reduce"
KV-split design of ``verify_attn_flash.cu`` ("Chunk 66.0").

All arithmetic is float64; bf16 inputs convert to float64 exactly.
"""
from __future__ import annotations

import math
from typing import Iterable, List, Optional, Sequence, Tuple

import torch

LATENT_DIM = 512
ROPE_DIM = 64
ROW_DIM = LATENT_DIM + ROPE_DIM

F64 = torch.float64


def ancestor_sets(tree_parent: Sequence[int]) -> List[set]:
    """anc*(i): node i and every node reached by following parents to -1.

    Raises ValueError on a parent that is not -1 and not an earlier node
    (the tree is given in topological order)."""
    par = [int(p) for p in tree_parent]
    out: List[set] = []
    for i, p in enumerate(par):
        if p < -1 or p >= i:
            raise ValueError(f"parent[{i}] = {p} is not -1 and not an earlier node")
        s = {i}
        if p >= 0:
            s |= out[p]
        out.append(s)
    return out


def ancestor_mask(tree_parent: Sequence[int]) -> torch.Tensor:
    """Boolean [T, T]: mask[i, j] is True when tree node j is in anc*(i)."""
    sets = ancestor_sets(tree_parent)
    T = len(sets)
    m = torch.zeros(T, T, dtype=torch.bool)
    for i, s in enumerate(sets):
        for j in s:
            m[i, j] = True
    return m


def ancestor_bits(tree_parent: Sequence[int]) -> List[int]:
    """Per node the ancestor set as an integer bitmask (bit j = node j)."""
    return [sum(1 << j for j in s) for s in ancestor_sets(tree_parent)]


def key_mask(prefix_len: int, tree_parent: Sequence[int]) -> torch.Tensor:
    """Boolean [T, P+T]: every node sees the whole prefix, then its ancestors."""
    T = len(tree_parent)
    m = torch.ones(T, prefix_len + T, dtype=torch.bool)
    m[:, prefix_len:] = ancestor_mask(tree_parent)
    return m


def verify_request(q_latent: torch.Tensor, q_rope: torch.Tensor, kv_pool: torch.Tensor,
                   kv_indices: torch.Tensor, prefix_len: int, tree_parent: Sequence[int],
                   sm_scale: float, nodes: Optional[Iterable[int]] = None,
                   heads: Optional[Iterable[int]] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """One request.  q_latent [T, H, 512], q_rope [T, H, 64], kv_indices [P+T].

    Returns (O [n, h, 512], LSE [n, h]) in float64 for the selected nodes
    (default all) and heads (default all), in the order given.
    """
    T, H = q_latent.shape[0], q_latent.shape[1]
    P = int(prefix_len)
    idx = kv_indices.to(torch.int64)
    if idx.numel() != P + T:
        raise ValueError("kv_indices must hold P prefix rows then T tree rows")
    nodes = list(range(T)) if nodes is None else [int(n) for n in nodes]
    heads = list(range(H)) if heads is None else [int(h) for h in heads]

    # Gather the request's key rows into one dense float64 matrix [P+T, 576].
    K = kv_pool.index_select(0, idx).to(F64)
    V = K[:, :LATENT_DIM]
    allowed = key_mask(P, tree_parent)  # [T, P+T]

    O = torch.empty(len(nodes), len(heads), LATENT_DIM, dtype=F64)
    L = torch.empty(len(nodes), len(heads), dtype=F64)
    hsel = torch.tensor(heads, dtype=torch.int64)
    for a, i in enumerate(nodes):
        q = torch.cat([q_latent[i].to(F64), q_rope[i].to(F64)], dim=-1)[hsel]  # [h, 576]
        s = sm_scale * (q @ K.T)                                               # [h, P+T]
        s = s.masked_fill(~allowed[i].unsqueeze(0), float("-inf"))
        m = s.max(dim=-1, keepdim=True).values
        e = torch.exp(s - m)
        l = e.sum(dim=-1, keepdim=True)
        O[a] = (e @ V) / l
        L[a] = (m + torch.log(l)).squeeze(-1)
    return O, L


def verify_batched(q_latent: torch.Tensor, q_rope: torch.Tensor, kv_pool: torch.Tensor,
                   kv_indices: torch.Tensor, kv_indptr: torch.Tensor, prefix_lens: torch.Tensor,
                   tree_parent: torch.Tensor, sm_scale: float) -> Tuple[torch.Tensor, torch.Tensor]:
    """All requests; q_* are [B*T, H, d]; returns O [B*T, H, 512], LSE [B*T, H]."""
    B, T = tree_parent.shape
    outs, lses = [], []
    for b in range(B):
        lo, hi = int(kv_indptr[b]), int(kv_indptr[b + 1])
        o, l = verify_request(q_latent[b * T:(b + 1) * T], q_rope[b * T:(b + 1) * T], kv_pool,
                              kv_indices[lo:hi], int(prefix_lens[b]),
                              tree_parent[b].tolist(), sm_scale)
        outs.append(o)
        lses.append(l)
    return torch.cat(outs), torch.cat(lses)


def partial_over_keys(q: torch.Tensor, K: torch.Tensor, allowed: torch.Tensor,
                      sm_scale: float) -> Tuple[torch.Tensor, torch.Tensor]:
    """Attention of query rows q [r, 576] over one subset of keys K [n, 576]
    with a per-(row, key) allow mask [r, n].  Returns the subset's normalised
    output O_s [r, 512] and its log-sum-exp lse_s [r] (-inf and 0 when a row
    has no allowed key in the subset)."""
    s = sm_scale * (q.to(F64) @ K.to(F64).T)
    s = s.masked_fill(~allowed, float("-inf"))
    m = s.max(dim=-1, keepdim=True).values
    empty = torch.isinf(m) & (m < 0)
    m = torch.where(empty, torch.zeros_like(m), m)
    e = torch.exp(s - m)
    l = e.sum(dim=-1, keepdim=True)
    O = torch.where(empty, torch.zeros(1, dtype=F64), (e @ K.to(F64)[:, :LATENT_DIM]) / torch.where(empty, torch.ones_like(l), l))
    lse = torch.where(empty, torch.full_like(m, float("-inf")), m + torch.log(l)).squeeze(-1)
    return O, lse


def merge_partials(o_parts: Sequence[torch.Tensor], lse_parts: Sequence[torch.Tensor]
                   ) -> Tuple[torch.Tensor, torch.Tensor]:
    """Merge split-KV partials (the "reduce" of partial+reduce):
    lse = ln sum_s exp(lse_s);  O = sum_s exp(lse_s - lse) * O_s."""
    lse_stack = torch.stack([l.to(F64) for l in lse_parts])          # [S, r]
    o_stack = torch.stack([o.to(F64) for o in o_parts])              # [S, r, 512]
    lse = torch.logsumexp(lse_stack, dim=0)                          # [r]
    w = torch.exp(lse_stack - lse.unsqueeze(0))                      # [S, r]
    w = torch.nan_to_num(w, nan=0.0)
    O = (w.unsqueeze(-1) * o_stack).sum(dim=0)
    return O, lse
