"""Seeded synthetic inputs for DDTree verify attention.

This module only draws inputs: a bf16 latent KV pool, a page_size=1 index
table, draft-tree parent arrays and bf16 queries.  It holds none of the
attention arithmetic, so the float64 oracle and the CUDA path can both be fed
from it without sharing any of the method's code.

Shapes follow the workloads on the magik.net pages ("Chunk 66.0": TP8 with 8
heads per rank, prefixes from 1k to 185k tokens, page_size=1 KV on a churned
pool; "Chunk 66.1": NSPLIT tuning for the 8-head regime).  The numeric
distributions (N(0,1) rounded to bf16) and the five named workloads are the
synthetic stand-ins described in the design notes; there is no dataset.

Draw order per workload is fixed: pool -> indices -> trees -> queries, from
one CPU ``torch.Generator`` seeded with the workload's seed.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional

import torch

LATENT_DIM = 512
ROPE_DIM = 64
ROW_DIM = LATENT_DIM + ROPE_DIM  # 576 bf16 = 1152 bytes per KV row


@dataclass
class VerifyInputs:
    """One batch of verify-attention inputs (CPU tensors).

    kv_pool      bf16  [pool_rows, 576]      latent (512) + rope (64) per token
    kv_indices   int32 [sum_b (P_b + T)]     per request: P_b prefix rows then
                                             T tree rows in node order
    kv_indptr    int32 [B + 1]               request b owns kv_indices[indptr[b]:indptr[b+1]]
    prefix_lens  int32 [B]
    tree_parent  int32 [B, T]                -1 = root under the prefix end, else < i
    q_latent     bf16  [B*T, H, 512]
    q_rope       bf16  [B*T, H, 64]
    """

    name: str
    kv_pool: torch.Tensor
    kv_indices: torch.Tensor
    kv_indptr: torch.Tensor
    prefix_lens: torch.Tensor
    tree_parent: torch.Tensor
    q_latent: torch.Tensor
    q_rope: torch.Tensor
    sm_scale: float
    n_heads: int
    n_nodes: int
    meta: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return int(self.prefix_lens.numel())

    @property
    def pool_rows(self) -> int:
        return int(self.kv_pool.shape[0])


def _bf16(x: torch.Tensor) -> torch.Tensor:
    # fp32 -> bf16 with round-to-nearest-even (torch's conversion rule).
    return x.to(torch.bfloat16)


def chain_tree(n_nodes: int) -> List[int]:
    """parent[i] = i - 1; node 0 hangs off the prefix end (-1)."""
    return [i - 1 for i in range(n_nodes)]


def uniform_tree(n_nodes: int, g: torch.Generator) -> List[int]:
    """parent[i] uniform over {-1, 0, ..., i-1}."""
    out = []
    for i in range(n_nodes):
        out.append(int(torch.randint(-1, i, (1,), generator=g)))
    return out


def bounded_tree(n_nodes: int, g: torch.Generator, max_children: int = 4,
                 max_depth: int = 8) -> List[int]:
    """parent[i] uniform over {-1} and the earlier nodes that still have fewer
    than ``max_children`` children and depth < ``max_depth`` (root depth 1).
    The -1 pseudo-root is capped at ``max_children`` children as well."""
    parent: List[int] = []
    depth: List[int] = []
    children = {-1: 0}
    for i in range(n_nodes):
        cands = [-1] if children[-1] < max_children else []
        cands += [j for j in range(i) if children[j] < max_children and depth[j] < max_depth]
        if not cands:  # cannot happen for n_nodes <= 4 * (4**8 - 1) / 3
            raise ValueError("tree capacity exhausted")
        p = cands[int(torch.randint(0, len(cands), (1,), generator=g))]
        parent.append(p)
        depth.append(1 if p < 0 else depth[p] + 1)
        children[p] += 1
        children[i] = 0
    return parent


def make_inputs(name: str, *, batch: int, n_heads: int, prefixes: List[int], n_nodes: int,
                tree: str, pool_rows: int, index_mode: str, seed: int,
                sm_scale: Optional[float] = None, q_scale: float = 1.0,
                kv_scale: float = 1.0) -> VerifyInputs:
    """Draw one workload.

    index_mode:
      "sample"       each request draws P_b+T distinct rows (a prefix of one
                     random permutation per request: without replacement)
      "permutation"  same as "sample"; named for the Tiny workload
      "contiguous"   the defragmented copy of "sample": the request's rows are
                     moved to rows [0, P+T) of a re-ordered pool and the
                     indices become arange (batch 1 only)
      "interleaved"  one random permutation of the whole pool cut consecutively
                     into the requests' P_b+T chunks (requests interleave)
    tree: "chain" | "uniform" | "bounded"
    """
    assert len(prefixes) == batch
    g = torch.Generator().manual_seed(seed)
    pool = _bf16(torch.randn(pool_rows, ROW_DIM, generator=g) * kv_scale)

    lens = [p + n_nodes for p in prefixes]
    if sum(lens) > pool_rows:
        raise ValueError("pool too small for the requests")
    idx_parts = []
    if index_mode in ("sample", "permutation", "contiguous"):
        for L in lens:
            idx_parts.append(torch.randperm(pool_rows, generator=g)[:L])
    elif index_mode == "interleaved":
        perm = torch.randperm(pool_rows, generator=g)
        off = 0
        for L in lens:
            idx_parts.append(perm[off:off + L])
            off += L
    else:
        raise ValueError(index_mode)

    if index_mode == "contiguous":
        if batch != 1:
            raise ValueError("contiguous mode is defined for batch 1")
        rows = idx_parts[0]
        used = torch.zeros(pool_rows, dtype=torch.bool)
        used[rows] = True
        rest = torch.nonzero(~used).flatten()
        order = torch.cat([rows, rest])  # new row k holds old row order[k]
        pool = pool[order].contiguous()
        idx_parts = [torch.arange(rows.numel())]

    parents = []
    for _ in range(batch):
        if tree == "chain":
            parents.append(chain_tree(n_nodes))
        elif tree == "uniform":
            parents.append(uniform_tree(n_nodes, g))
        elif tree == "bounded":
            parents.append(bounded_tree(n_nodes, g))
        else:
            raise ValueError(tree)

    q = _bf16(torch.randn(batch * n_nodes, n_heads, ROW_DIM, generator=g) * q_scale)
    indptr = [0]
    for L in lens:
        indptr.append(indptr[-1] + L)
    return VerifyInputs(
        name=name,
        kv_pool=pool,
        kv_indices=torch.cat(idx_parts).to(torch.int32).contiguous(),
        kv_indptr=torch.tensor(indptr, dtype=torch.int32),
        prefix_lens=torch.tensor(prefixes, dtype=torch.int32),
        tree_parent=torch.tensor(parents, dtype=torch.int32).reshape(batch, n_nodes),
        q_latent=q[..., :LATENT_DIM].contiguous(),
        q_rope=q[..., LATENT_DIM:].contiguous(),
        sm_scale=(1.0 / math.sqrt(192.0)) if sm_scale is None else float(sm_scale),
        n_heads=n_heads,
        n_nodes=n_nodes,
        meta=dict(tree=tree, index_mode=index_mode, seed=seed, prefixes=list(prefixes)),
    )


# The five named workloads.  "k" prefixes: 1k=1024 ... 131k=131072, 185k=185*1024.
MIXED_PREFIXES = [1024, 4096, 8192, 16384, 32768, 65536, 131072, 189440]

WORKLOADS = {
    "tiny": dict(batch=1, n_heads=8, prefixes=[256], n_nodes=4, tree="chain",
                 pool_rows=1024, index_mode="permutation", seed=0),
    "tp8_slice": dict(batch=1, n_heads=8, prefixes=[4096], n_nodes=16, tree="uniform",
                      pool_rows=262144, index_mode="sample", seed=1),
    "long_scattered": dict(batch=1, n_heads=8, prefixes=[65536], n_nodes=32, tree="uniform",
                           pool_rows=262144, index_mode="sample", seed=2),
    "long_contiguous": dict(batch=1, n_heads=8, prefixes=[65536], n_nodes=32, tree="uniform",
                            pool_rows=262144, index_mode="contiguous", seed=2),
    "unsharded_heads": dict(batch=1, n_heads=128, prefixes=[32768], n_nodes=64, tree="bounded",
                            pool_rows=131072, index_mode="sample", seed=3),
    "mixed_batch": dict(batch=8, n_heads=8, prefixes=MIXED_PREFIXES, n_nodes=32, tree="uniform",
                        pool_rows=524288, index_mode="interleaved", seed=4),
}


def workload(name: str, **overrides) -> VerifyInputs:
    cfg = dict(WORKLOADS[name])
    cfg.update(overrides)
    return make_inputs(name, **cfg)


def algorithmic_cost(inp: VerifyInputs) -> dict:
    """Algorithmic bytes and FLOPs of one verify call (no re-reads, no
    workspace traffic): each needed KV row once (1152 B) plus its 4-byte index,
    Q (576 bf16 per row), O (512 bf16) + LSE (fp32) per row, 4 B per parent;
    FLOPs = 2*(576+512) per (query row, attended key)."""
    T, H = inp.n_nodes, inp.n_heads
    byts = 0
    flops = 0
    for b in range(inp.batch):
        P = int(inp.prefix_lens[b])
        par = inp.tree_parent[b].tolist()
        depth_sum = 0
        for i in range(T):
            d, j = 0, i
            while j >= 0:
                d += 1
                j = par[j]
            depth_sum += d
        byts += (P + T) * (ROW_DIM * 2 + 4)
        flops += H * (T * P + depth_sum) * (2 * ROW_DIM + 2 * LATENT_DIM)
    rows = inp.batch * T * H
    byts += rows * ROW_DIM * 2 + rows * (LATENT_DIM * 2 + 4) + 4 * inp.batch * T
    return dict(bytes=byts, flops=flops)


# ---------------------------------------------------------------- acceptance
@dataclass
class AcceptInputs:
    """Inputs of the greedy-acceptance step after a verify forward.

    logits        [B, T+1, V] bf16: row 0 is the target's prediction at the
                  prefix end, row 1+i its prediction after tree node i
    draft_tokens  [B, T] int32: the drafted token of each tree node
    tree_parent   [B, T] int32 (-1 = child of the prefix end, else < i)
    kv_indices    int32: per request P prefix rows then T tree rows
    kv_indptr     [B+1] int32, prefix_lens [B] int32
    planted       [B, T+1] int64: the token given the largest logit of each
                  row by construction (test bookkeeping only)
    """
    logits: torch.Tensor
    draft_tokens: torch.Tensor
    tree_parent: torch.Tensor
    kv_indices: torch.Tensor
    kv_indptr: torch.Tensor
    prefix_lens: torch.Tensor
    planted: torch.Tensor
    pool_rows: int
    meta: dict

    @property
    def batch(self) -> int:
        return int(self.tree_parent.shape[0])

    @property
    def n_nodes(self) -> int:
        return int(self.tree_parent.shape[1])

    @property
    def vocab(self) -> int:
        return int(self.logits.shape[2])


def make_accept_inputs(name: str, *, batch: int, n_nodes: int, vocab: int, prefixes: List[int],
                       tree: str, pool_rows: int, p_match: float, seed: int,
                       planted_logit: float = 10.0) -> AcceptInputs:
    """Draw one acceptance workload (order: indices -> trees -> logits -> drafts).

    Logits are N(0,1) rounded to bf16, except one planted token per row that
    gets ``planted_logit`` (far above any N(0,1) draw over the vocabulary, so
    it is the row's unique largest value).  Among the children of each node
    (and of the prefix end), with probability ``p_match`` one child, chosen
    uniformly, drafts the parent row's planted token; every other child
    drafts a distinct other token.  That gives a tree in which the draft
    agrees with the target along a random root-to-node path, like a drafter
    whose guesses are right most of the time.
    """
    assert len(prefixes) == batch
    g = torch.Generator().manual_seed(seed)
    total = sum(P + n_nodes for P in prefixes)
    if total > pool_rows:
        raise ValueError("pool too small for the requests")
    perm = torch.randperm(pool_rows, generator=g)[:total].to(torch.int32)
    indptr = [0]
    for P in prefixes:
        indptr.append(indptr[-1] + P + n_nodes)
    parents = []
    for _ in range(batch):
        if tree == "chain":
            parents.append(chain_tree(n_nodes))
        elif tree == "uniform":
            parents.append(uniform_tree(n_nodes, g))
        elif tree == "bounded":
            parents.append(bounded_tree(n_nodes, g))
        else:
            raise ValueError(tree)
    logits = torch.randn(batch, n_nodes + 1, vocab, generator=g)
    planted = torch.randint(0, vocab, (batch, n_nodes + 1), generator=g)
    for b in range(batch):
        for r in range(n_nodes + 1):
            logits[b, r, int(planted[b, r])] = planted_logit
    drafts = torch.empty(batch, n_nodes, dtype=torch.int32)
    for b in range(batch):
        par = parents[b]
        for p in [-1] + list(range(n_nodes)):
            kids = [c for c in range(n_nodes) if par[c] == p]
            if not kids:
                continue
            target = int(planted[b, 0 if p < 0 else 1 + p])
            match = kids[int(torch.randint(0, len(kids), (1,), generator=g))] \
                if float(torch.rand(1, generator=g)) < p_match else -1
            used = {target}
            for c in kids:
                if c == match:
                    drafts[b, c] = target
                    continue
                # A fresh token when the vocabulary has one left, else any
                # token other than the target (siblings may then repeat).
                for _ in range(64):
                    tok = int(torch.randint(0, vocab, (1,), generator=g))
                    if tok not in used:
                        break
                else:
                    tok = (target + 1) % vocab
                used.add(tok)
                drafts[b, c] = tok
    return AcceptInputs(
        logits=_bf16(logits),
        draft_tokens=drafts,
        tree_parent=torch.tensor(parents, dtype=torch.int32),
        kv_indices=perm,
        kv_indptr=torch.tensor(indptr, dtype=torch.int32),
        prefix_lens=torch.tensor(prefixes, dtype=torch.int32),
        planted=planted,
        pool_rows=pool_rows,
        meta=dict(tree=tree, p_match=p_match, seed=seed, prefixes=list(prefixes)),
    )


# DeepSeek-V3's vocabulary has 129,280 tokens; prefixes as in the verify workloads.
ACCEPT_WORKLOADS = {
    "accept_small": dict(batch=2, n_nodes=8, vocab=1000, prefixes=[16, 40], tree="uniform",
                         pool_rows=4096, p_match=0.8, seed=10),
    "accept_long": dict(batch=1, n_nodes=32, vocab=129280, prefixes=[65536], tree="bounded",
                        pool_rows=262144, p_match=0.9, seed=11),
    "accept_batch": dict(batch=8, n_nodes=32, vocab=129280, prefixes=MIXED_PREFIXES, tree="bounded",
                         pool_rows=524288, p_match=0.9, seed=12),
}


def accept_workload(name: str, **overrides) -> AcceptInputs:
    cfg = dict(ACCEPT_WORKLOADS[name])
    cfg.update(overrides)
    return make_accept_inputs(name, **cfg)


# ---------------------------------------------------------------- relocation
@dataclass
class RelocateInputs:
    """A churned pool and where each request's rows should move.

    kv_pool    [pool_rows, 576] bf16
    kv_indices int32: per request its P + T rows, scattered over the lower
               part of the pool (sampled without replacement)
    kv_indptr  [B+1] int32
    dest_base  [B] int32: consecutive free regions in the top part of the pool
    """
    kv_pool: torch.Tensor
    kv_indices: torch.Tensor
    kv_indptr: torch.Tensor
    dest_base: torch.Tensor
    meta: dict

    @property
    def batch(self) -> int:
        return int(self.dest_base.shape[0])

    @property
    def pool_rows(self) -> int:
        return int(self.kv_pool.shape[0])


def make_relocate_inputs(name: str, *, prefixes: List[int], n_nodes: int, pool_rows: int,
                         seed: int) -> RelocateInputs:
    """Draw order: pool -> source rows -> (destinations follow from the sizes).

    The top sum(P + T) rows of the pool are the free destination area, one
    region per request in request order; the sources are sampled without
    replacement from the rows below it, so no destination holds a source."""
    g = torch.Generator().manual_seed(seed)
    sizes = [P + n_nodes for P in prefixes]
    total = sum(sizes)
    if 2 * total > pool_rows:
        raise ValueError("pool too small")
    pool = _bf16(torch.randn(pool_rows, ROW_DIM, generator=g))
    src = torch.randperm(pool_rows - total, generator=g)[:total].to(torch.int32)
    indptr = [0]
    dest = []
    for n in sizes:
        dest.append(pool_rows - total + indptr[-1])
        indptr.append(indptr[-1] + n)
    return RelocateInputs(kv_pool=pool, kv_indices=src, kv_indptr=torch.tensor(indptr, dtype=torch.int32),
                          dest_base=torch.tensor(dest, dtype=torch.int32),
                          meta=dict(prefixes=list(prefixes), n_nodes=n_nodes, seed=seed))


RELOCATE_WORKLOADS = {
    "relocate_small": dict(prefixes=[0, 17, 300], n_nodes=4, pool_rows=2048, seed=20),
    "relocate_long": dict(prefixes=[65536], n_nodes=32, pool_rows=262144, seed=21),
    "relocate_batch": dict(prefixes=MIXED_PREFIXES, n_nodes=32, pool_rows=1048576, seed=22),
}


def relocate_workload(name: str, **overrides) -> RelocateInputs:
    cfg = dict(RELOCATE_WORKLOADS[name])
    cfg.update(overrides)
    return make_relocate_inputs(name, **cfg)


# ---------------------------------------------------------------- tree masks
def tree_mask(parents: List[int], prefix_len: int) -> torch.Tensor:
    """The flattened-mask input format for one request: uint8 [T, P + T],
    row i = 1 for every prefix row and for node i and each node on its parent
    chain.  (Input construction: the form a serving framework builds on the
    host and hands over instead of the parent array.)"""
    T = len(parents)
    m = torch.zeros(T, prefix_len + T, dtype=torch.uint8)
    m[:, :prefix_len] = 1
    for i in range(T):
        j = i
        while j >= 0:
            m[i, prefix_len + j] = 1
            j = parents[j]
    return m


def flat_tree_masks(tree_parent: torch.Tensor, prefix_lens: torch.Tensor):
    """All requests' masks concatenated row-major; returns (flat uint8 mask,
    int64 element offsets [B+1])."""
    parts, indptr = [], [0]
    for b in range(tree_parent.shape[0]):
        m = tree_mask(tree_parent[b].tolist(), int(prefix_lens[b]))
        parts.append(m.reshape(-1))
        indptr.append(indptr[-1] + m.numel())
    return torch.cat(parts), torch.tensor(indptr, dtype=torch.int64)
