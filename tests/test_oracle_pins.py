"""Pins for the float64 oracle, independent of the oracle's own code.

Each test checks the oracle against something it does not compute itself:
library attention routines (SDPA, the CPU flash kernel's log-sum-exp),
networkx for tree ancestry, closed forms, a pure-Python brute force over every
tree of up to 5 nodes, and invariances.  A dropped rope term, a wrong scale,
a log2 LSE, a mask that misses the node itself or an ancestor, or tree rows in
the wrong order each fail at least one of them.
"""
import itertools
import json
import math
import os

import networkx as nx
import pytest
import torch
import torch.nn.functional as F

from oracle import (ancestor_bits, ancestor_mask, merge_partials, partial_over_keys,
                    verify_batched, verify_request)
from speculative_decode_tree_gb300.workloads import make_inputs, uniform_tree

F64 = torch.float64
HERE = os.path.dirname(os.path.abspath(__file__))


def _inputs(P, T, H, tree="uniform", pool_rows=None, seed=7, **kw):
    pool_rows = pool_rows or max(64, 2 * (P + T))
    return make_inputs("pin", batch=1, n_heads=H, prefixes=[P], n_nodes=T, tree=tree,
                       pool_rows=pool_rows, index_mode="sample", seed=seed, **kw)


def _rows(inp):
    """Gathered key rows by plain Python indexing (not index_select)."""
    idx = [int(i) for i in inp.kv_indices.tolist()]
    return torch.stack([inp.kv_pool[i].to(F64) for i in idx])


def _nx_ancestors(parent):
    g = nx.DiGraph()
    g.add_nodes_from(range(len(parent)))
    for i, p in enumerate(parent):
        if p >= 0:
            g.add_edge(p, i)
    return [nx.ancestors(g, i) | {i} for i in range(len(parent))]


def _sdpa(q, K, allowed, scale):
    """Library attention in float64: returns O [T,H,512] and LSE [T,H]."""
    T, H, _ = q.shape
    add = torch.zeros(allowed.shape, dtype=F64).masked_fill(~allowed, float("-inf"))
    qq = q.permute(1, 0, 2).unsqueeze(0)                         # [1,H,T,576]
    kk = K.unsqueeze(0).unsqueeze(0).expand(1, H, -1, -1)        # [1,H,n,576]
    vv = K[:, :512].unsqueeze(0).unsqueeze(0).expand(1, H, -1, -1)
    o = F.scaled_dot_product_attention(qq, kk, vv, attn_mask=add, scale=scale)
    # The CPU flash kernel also returns the natural-log LSE; it wants equal
    # head sizes, so feed the full rows as V (its first 512 output columns
    # are the same attention output).
    _, lse = torch.ops.aten._scaled_dot_product_flash_attention_for_cpu(
        qq.contiguous(), kk.contiguous(), kk.contiguous(), 0.0, False, attn_mask=add, scale=scale)[:2]
    return o[0].permute(1, 0, 2), lse[0].permute(1, 0)


def _q(inp):
    return torch.cat([inp.q_latent.to(F64), inp.q_rope.to(F64)], dim=-1)


def _run(inp):
    return verify_request(inp.q_latent, inp.q_rope, inp.kv_pool, inp.kv_indices,
                          int(inp.prefix_lens[0]), inp.tree_parent[0].tolist(), inp.sm_scale)


def test_single_node_is_plain_mla_decode():
    inp = _inputs(P=37, T=1, H=3)
    O, L = _run(inp)
    allowed = torch.ones(1, 38, dtype=torch.bool)
    Os, Ls = _sdpa(_q(inp), _rows(inp), allowed, inp.sm_scale)
    torch.testing.assert_close(O, Os, rtol=1e-12, atol=1e-13)
    torch.testing.assert_close(L, Ls, rtol=1e-12, atol=1e-13)


def test_chain_is_causal_attention():
    P, T = 20, 6
    inp = _inputs(P=P, T=T, H=4, tree="chain")
    O, L = _run(inp)
    allowed = torch.cat([torch.ones(T, P, dtype=torch.bool),
                         torch.ones(T, T, dtype=torch.bool).tril()], dim=1)
    Os, Ls = _sdpa(_q(inp), _rows(inp), allowed, inp.sm_scale)
    torch.testing.assert_close(O, Os, rtol=1e-12, atol=1e-13)
    torch.testing.assert_close(L, Ls, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_random_tree_matches_sdpa_with_networkx_ancestors(seed):
    P, T = 33, 16
    inp = _inputs(P=P, T=T, H=2, seed=seed)
    parent = inp.tree_parent[0].tolist()
    anc = _nx_ancestors(parent)
    allowed = torch.zeros(T, P + T, dtype=torch.bool)
    allowed[:, :P] = True
    for i in range(T):
        for j in anc[i]:
            allowed[i, P + j] = True
    O, L = _run(inp)
    Os, Ls = _sdpa(_q(inp), _rows(inp), allowed, inp.sm_scale)
    torch.testing.assert_close(O, Os, rtol=1e-12, atol=1e-13)
    torch.testing.assert_close(L, Ls, rtol=1e-12, atol=1e-13)
    # The mask helpers agree with networkx too.
    m = ancestor_mask(parent)
    bits = ancestor_bits(parent)
    for i in range(T):
        assert set(torch.nonzero(m[i]).flatten().tolist()) == anc[i]
        assert bits[i] == sum(1 << j for j in anc[i])


def test_pool_permutation_invariance_is_exact():
    inp = _inputs(P=50, T=8, H=2, pool_rows=200)
    O, L = _run(inp)
    g = torch.Generator().manual_seed(99)
    perm = torch.randperm(inp.pool_rows, generator=g)      # new row r holds old row perm[r]
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(perm.numel())
    pool2 = inp.kv_pool[perm]
    idx2 = inv[inp.kv_indices.long()].to(torch.int32)
    O2, L2 = verify_request(inp.q_latent, inp.q_rope, pool2, idx2, 50,
                            inp.tree_parent[0].tolist(), inp.sm_scale)
    assert torch.equal(O, O2) and torch.equal(L, L2)


def test_constant_scores_give_mean_of_values():
    """q = 0 makes every score 0: O is the mean of V over K(i) and
    LSE = ln |K(i)| = ln(P + depth(i))."""
    P, T = 29, 12
    inp = _inputs(P=P, T=T, H=2, seed=5)
    inp.q_latent.zero_()
    inp.q_rope.zero_()
    O, L = _run(inp)
    parent = inp.tree_parent[0].tolist()
    rows = _rows(inp)
    for i in range(T):
        chain, j = [], i
        while j >= 0:
            chain.append(j)
            j = parent[j]
        keys = list(range(P)) + [P + j for j in chain]
        mean = rows[keys, :512].mean(dim=0)
        for h in range(2):
            torch.testing.assert_close(O[i, h], mean, rtol=1e-12, atol=1e-14)
            assert abs(float(L[i, h]) - math.log(P + len(chain))) < 1e-12


def test_identical_keys_give_that_value():
    """All key rows equal: every weight is equal, O is that row's V and
    LSE = s + ln |K(i)| with s = scale * q.k."""
    P, T = 10, 5
    inp = _inputs(P=P, T=T, H=1, tree="chain", seed=11)
    row = inp.kv_pool[int(inp.kv_indices[0])].clone()
    inp.kv_pool[:] = row
    O, L = _run(inp)
    k = [float(x) for x in row.to(F64)]
    for i in range(T):
        q = [float(x) for x in torch.cat([inp.q_latent[i, 0], inp.q_rope[i, 0]]).to(F64)]
        s = inp.sm_scale * math.fsum(a * b for a, b in zip(q, k))
        torch.testing.assert_close(O[i, 0], row[:512].to(F64), rtol=1e-12, atol=1e-14)
        assert abs(float(L[i, 0]) - (s + math.log(P + i + 1))) < 1e-11


def test_rope_and_latent_columns_each_count():
    P, T = 40, 6
    inp = _inputs(P=P, T=T, H=2, seed=13)
    parent = inp.tree_parent[0].tolist()
    anc = _nx_ancestors(parent)
    allowed = torch.zeros(T, P + T, dtype=torch.bool)
    allowed[:, :P] = True
    for i in range(T):
        for j in anc[i]:
            allowed[i, P + j] = True
    # Rope only: zero the latent query.
    inp.q_latent.zero_()
    O, L = _run(inp)
    rows = _rows(inp)
    q = _q(inp)
    Os, Ls = _sdpa(q, rows, allowed, inp.sm_scale)
    torch.testing.assert_close(O, Os, rtol=1e-12, atol=1e-13)
    torch.testing.assert_close(L, Ls, rtol=1e-12, atol=1e-13)
    assert float(L.std()) > 0.05  # the rope columns really moved the scores
    # Latent only: zero the rope columns of the pool.
    inp2 = _inputs(P=P, T=T, H=2, seed=13)
    inp2.kv_pool[:, 512:] = 0
    O2, L2 = _run(inp2)
    Os2, Ls2 = _sdpa(_q(inp2), _rows(inp2), allowed, inp2.sm_scale)
    torch.testing.assert_close(O2, Os2, rtol=1e-12, atol=1e-13)
    torch.testing.assert_close(L2, Ls2, rtol=1e-12, atol=1e-13)


def _python_reference(q, keys, P, parent, scale):
    """Pure-Python brute force: path walk per (i, j), math.fsum, no max shift."""
    T = len(parent)
    out = []
    for i in range(T):
        vis = list(range(P))
        for j in range(T):
            a = i
            while a >= 0 and a != j:
                a = parent[a]
            if a == j:
                vis.append(P + j)
        per_head = []
        for qh in q[i]:
            s = [scale * math.fsum(x * y for x, y in zip(qh, keys[k])) for k in vis]
            e = [math.exp(v) for v in s]
            den = math.fsum(e)
            o = [math.fsum(e[n] * keys[k][d] for n, k in enumerate(vis)) / den for d in range(512)]
            per_head.append((o, math.log(den)))
        out.append(per_head)
    return out


@pytest.mark.parametrize("P", [0, 3])
def test_bruteforce_every_tree_of_five_nodes(P):
    T, H = 5, 2
    inp = _inputs(P=P, T=T, H=H, pool_rows=64, seed=17 + P)
    keys = [[float(x) for x in r] for r in _rows(inp)]
    q = [[[float(x) for x in torch.cat([inp.q_latent[i, h], inp.q_rope[i, h]]).to(F64)]
          for h in range(H)] for i in range(T)]
    # Scores do not depend on the tree: precompute the pure-Python score table.
    n_trees = 0
    for parent in itertools.product(*[range(-1, i) for i in range(T)]):
        parent = list(parent)
        n_trees += 1
        O, L = verify_request(inp.q_latent, inp.q_rope, inp.kv_pool, inp.kv_indices, P,
                              parent, inp.sm_scale)
        if n_trees % 24 != 1 and n_trees != 120:
            # Mask-only check for the rest (the full 512-wide brute force on
            # every tree is slow in pure Python): compare LSE, which moves
            # with every key added to or dropped from K(i).
            for i in range(T):
                a, vis = i, []
                while a >= 0:
                    vis.append(P + a)
                    a = parent[a]
                vis += list(range(P))
                for h in range(H):
                    s = [inp.sm_scale * math.fsum(x * y for x, y in zip(q[i][h], keys[k])) for k in vis]
                    assert abs(float(L[i, h]) - math.log(math.fsum(math.exp(v) for v in s))) < 1e-12
            continue
        ref = _python_reference(q, keys, P, parent, inp.sm_scale)
        for i in range(T):
            for h in range(H):
                o, l = ref[i][h]
                assert abs(float(L[i, h]) - l) < 1e-12
                assert torch.allclose(O[i, h], torch.tensor(o, dtype=F64), rtol=1e-12, atol=1e-13)
    assert n_trees == 120  # 1*2*3*4*5 parent arrays


def test_split_and_merge_equals_dense():
    """LSE over a union is the log-add of LSEs over disjoint parts; the merged
    output equals the dense one.  Includes parts where a row has no allowed key."""
    P, T, H = 70, 8, 2
    inp = _inputs(P=P, T=T, H=H, seed=23)
    O, L = _run(inp)
    rows = _rows(inp)
    parent = inp.tree_parent[0].tolist()
    allowed = torch.zeros(T, P + T, dtype=torch.bool)
    allowed[:, :P] = True
    for i, s in enumerate(_nx_ancestors(parent)):
        for j in s:
            allowed[i, P + j] = True
    q = _q(inp).reshape(T * H, 576)
    allow_r = allowed.repeat_interleave(H, dim=0)
    bounds = [0, 13, 14, 50, P, P + 3, P + T]  # ragged parts; the tree split in two
    o_parts, l_parts = [], []
    for a, b in zip(bounds[:-1], bounds[1:]):
        o, l = partial_over_keys(q, rows[a:b], allow_r[:, a:b], inp.sm_scale)
        o_parts.append(o)
        l_parts.append(l)
    assert torch.isinf(l_parts[-1]).any()  # some rows see none of the last tree keys
    Om, Lm = merge_partials(o_parts, l_parts)
    torch.testing.assert_close(Om.reshape(T, H, 512), O, rtol=1e-12, atol=1e-13)
    torch.testing.assert_close(Lm.reshape(T, H), L, rtol=1e-12, atol=1e-13)


def test_spiked_tree_keys_pin_the_mask():
    """Tree rows' rope column 0 is large and so is q_rope[0]: tree scores beat
    prefix scores by ~70 nats, so O[i] is the mean of V over anc*(i) alone."""
    P, T, H = 256, 16, 2
    inp = _inputs(P=P, T=T, H=H, seed=29)
    inp.q_latent.zero_()
    inp.q_rope.zero_()
    inp.q_rope[..., 0] = 8.0
    tree_rows = inp.kv_indices[P:].long()
    inp.kv_pool[tree_rows, 512] = 128.0
    O, L = _run(inp)
    rows = _rows(inp)
    anc = _nx_ancestors(inp.tree_parent[0].tolist())
    for i in range(T):
        mean = rows[[P + j for j in sorted(anc[i])], :512].mean(dim=0)
        for h in range(H):
            torch.testing.assert_close(O[i, h], mean, rtol=1e-12, atol=1e-12)
            assert abs(float(L[i, h]) - (inp.sm_scale * 1024.0 + math.log(len(anc[i])))) < 1e-9


def test_batched_equals_per_request():
    inp = make_inputs("pin", batch=3, n_heads=2, prefixes=[5, 0, 17], n_nodes=4, tree="uniform",
                      pool_rows=100, index_mode="interleaved", seed=31)
    O, L = verify_batched(inp.q_latent, inp.q_rope, inp.kv_pool, inp.kv_indices, inp.kv_indptr,
                          inp.prefix_lens, inp.tree_parent, inp.sm_scale)
    for b in range(3):
        lo, hi = int(inp.kv_indptr[b]), int(inp.kv_indptr[b + 1])
        o, l = verify_request(inp.q_latent[4 * b:4 * b + 4], inp.q_rope[4 * b:4 * b + 4],
                              inp.kv_pool, inp.kv_indices[lo:hi], int(inp.prefix_lens[b]),
                              inp.tree_parent[b].tolist(), inp.sm_scale)
        assert torch.equal(O[4 * b:4 * b + 4], o) and torch.equal(L[4 * b:4 * b + 4], l)


def test_invalid_parent_rejected():
    with pytest.raises(ValueError):
        ancestor_mask([-1, 1])
    with pytest.raises(ValueError):
        ancestor_mask([-2])


def test_closed_form_golden_cases():
    """Hand-derived cases in tests/golden/closed_form.json (see its notes)."""
    with open(os.path.join(HERE, "golden", "closed_form.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        P, T = c["prefix_len"], len(c["tree_parent"])
        pool = torch.zeros(len(c["key_rows"]), 576, dtype=torch.bfloat16)
        for r, entries in enumerate(c["key_rows"]):
            for d, v in entries.items():
                pool[r, int(d)] = v
        ql = torch.zeros(T, 1, 512, dtype=torch.bfloat16)
        qr = torch.zeros(T, 1, 64, dtype=torch.bfloat16)
        for d, v in c["query"].items():
            d = int(d)
            if d < 512:
                ql[:, 0, d] = v
            else:
                qr[:, 0, d - 512] = v
        idx = torch.tensor(c["kv_indices"], dtype=torch.int32)
        O, L = verify_request(ql, qr, pool, idx, P, c["tree_parent"], c["sm_scale"])
        for i, exp in enumerate(c["expected"]):
            assert abs(float(L[i, 0]) - eval(exp["lse"], {"math": math})) < 1e-13
            for d, e in exp["out"].items():
                assert abs(float(O[i, 0, int(d)]) - eval(e, {"math": math})) < 1e-13
