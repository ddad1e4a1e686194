"""The synthetic inputs match the workloads they stand in for: shapes, tree
shapes, index-table structure and value distribution of the five verify
configurations (batch, heads, nodes, prefixes, pool, index mode), drawn with
their fixed seeds.  No GPU and no attention arithmetic here."""
import math

import pytest
import torch

from speculative_decode_tree_gb300.workloads import (LATENT_DIM, MIXED_PREFIXES, ROPE_DIM, WORKLOADS,
                                                     bounded_tree, workload)

# Restated configuration of each workload: (batch, heads, prefixes, nodes, tree, pool rows, index mode).
EXPECTED = {
    "tiny": (1, 8, [256], 4, "chain", 1024, "permutation"),
    "tp8_slice": (1, 8, [4096], 16, "uniform", 262144, "sample"),
    "long_scattered": (1, 8, [65536], 32, "uniform", 262144, "sample"),
    "long_contiguous": (1, 8, [65536], 32, "uniform", 262144, "contiguous"),
    "unsharded_heads": (1, 128, [32768], 64, "bounded", 131072, "sample"),
    "mixed_batch": (8, 8, [1024, 4096, 8192, 16384, 32768, 65536, 131072, 189440], 32, "uniform", 524288,
                    "interleaved"),
}


def test_named_configurations():
    assert set(WORKLOADS) == set(EXPECTED)
    for name, (b, h, prefixes, t, tree, pool, mode) in EXPECTED.items():
        cfg = WORKLOADS[name]
        assert (cfg["batch"], cfg["n_heads"], list(cfg["prefixes"]), cfg["n_nodes"], cfg["tree"],
                cfg["pool_rows"], cfg["index_mode"]) == (b, h, prefixes, t, tree, pool, mode), name
    assert MIXED_PREFIXES[-1] == 185 * 1024


def _depths(parent):
    d = []
    for i, p in enumerate(parent):
        assert -1 <= p < i
        d.append(1 if p < 0 else d[p] + 1)
    return d


@pytest.mark.parametrize("name", sorted(EXPECTED))
def test_drawn_inputs_have_the_stated_structure(name):
    b, h, prefixes, t, tree, pool_rows, mode = EXPECTED[name]
    inp = workload(name)
    assert inp.batch == b and inp.n_heads == h and inp.n_nodes == t and inp.pool_rows == pool_rows
    assert inp.kv_pool.dtype == torch.bfloat16 and tuple(inp.kv_pool.shape) == (pool_rows, LATENT_DIM + ROPE_DIM)
    assert tuple(inp.q_latent.shape) == (b * t, h, LATENT_DIM) and inp.q_latent.dtype == torch.bfloat16
    assert tuple(inp.q_rope.shape) == (b * t, h, ROPE_DIM) and inp.q_rope.dtype == torch.bfloat16
    assert inp.prefix_lens.tolist() == prefixes
    assert math.isclose(inp.sm_scale, 1.0 / math.sqrt(192.0))
    lens = [p + t for p in prefixes]
    assert inp.kv_indptr.tolist() == [sum(lens[:k]) for k in range(b + 1)]
    idx = inp.kv_indices.long()
    assert idx.numel() == sum(lens) and int(idx.min()) >= 0 and int(idx.max()) < pool_rows
    for k in range(b):  # page_size=1: each request's rows are distinct pool rows
        part = idx[inp.kv_indptr[k]:inp.kv_indptr[k + 1]]
        assert part.unique().numel() == part.numel()
    if mode == "interleaved":  # one permutation of the pool cut into the requests
        assert idx.unique().numel() == idx.numel()
    if mode == "contiguous":
        assert torch.equal(idx, torch.arange(sum(lens)))
    for k in range(b):
        parent = inp.tree_parent[k].tolist()
        depth = _depths(parent)
        if tree == "chain":
            assert parent == list(range(-1, t - 1))
        if tree == "bounded":
            kids = {}
            for p in parent:
                kids[p] = kids.get(p, 0) + 1
            assert max(kids.values()) <= 4 and max(depth) <= 8


def test_contiguous_is_the_defragmented_copy_of_scattered():
    s = workload("long_scattered")
    c = workload("long_contiguous")
    n = int(s.kv_indptr[-1])
    # Same seed: the contiguous pool's first rows are the scattered request's rows in order.
    assert torch.equal(c.kv_pool[:n].view(torch.int16), s.kv_pool[s.kv_indices.long()].view(torch.int16))
    assert torch.equal(c.tree_parent, s.tree_parent)
    assert torch.equal(c.q_latent.view(torch.int16), s.q_latent.view(torch.int16))


def test_values_are_standard_normal_rounded_to_bf16():
    inp = workload("tp8_slice")
    x = inp.kv_pool[:20000].float()
    assert abs(float(x.mean())) < 0.01 and abs(float(x.std()) - 1.0) < 0.01
    assert torch.equal(x.to(torch.bfloat16).float(), x)  # exactly representable: drawn in bf16
    q = inp.q_latent.float()
    assert abs(float(q.mean())) < 0.05 and abs(float(q.std()) - 1.0) < 0.05


def test_same_seed_same_inputs():
    a, b = workload("tiny"), workload("tiny")
    for f in ("kv_pool", "q_latent", "q_rope"):  # bitwise, through the bf16 bit patterns
        assert torch.equal(getattr(a, f).view(torch.int16), getattr(b, f).view(torch.int16)), f
    for f in ("kv_indices", "tree_parent"):
        assert torch.equal(getattr(a, f), getattr(b, f)), f


def test_bounded_tree_respects_both_limits_at_full_size():
    g = torch.Generator().manual_seed(123)
    for _ in range(20):
        parent = bounded_tree(64, g)
        kids = {}
        for p in parent:
            kids[p] = kids.get(p, 0) + 1
        assert max(kids.values()) <= 4 and max(_depths(parent)) <= 8


# Algorithmic bytes and GFLOP per call from the scope table of the verify path
# (bytes = sum (P+T)(1152+4) + T H (1152 + 1028) + 4T, FLOPs = H (T P + sum depth) 2176,
# worked out there for one sample tree per config): the roofline denominators
# the benchmark divides by must agree with them.
TABLE = {"tiny": (0.37, 0.018), "tp8_slice": (5.03, 1.14), "long_scattered": (76.4, 36.5),
         "unsharded_heads": (55.8, 584.0), "mixed_batch": (523.0, 250.0)}


@pytest.mark.parametrize("name", sorted(TABLE))
def test_algorithmic_cost_matches_the_scope_table(name):
    from speculative_decode_tree_gb300.workloads import algorithmic_cost
    mb, gflop = TABLE[name]
    c = algorithmic_cost(workload(name))
    assert abs(c["bytes"] / 1e6 - mb) <= 0.01 * mb, c
    assert abs(c["flops"] / 1e9 - gflop) <= 0.01 * gflop, c
