"""GPU parity of greedy acceptance + commit: the CUDA path through the C ABI
against the oracle on the same seeded inputs.  Every output is an integer,
so the comparison is exact."""
import numpy as np
import pytest
import torch

from oracle import accept_batched
from speculative_decode_tree_gb300 import binding as B
from speculative_decode_tree_gb300.runner import DeviceAccept
from speculative_decode_tree_gb300.workloads import AcceptInputs, accept_workload, make_accept_inputs

pytestmark = pytest.mark.gpu

KEYS = ("accept_len", "next_token", "accepted_nodes", "commit_indices", "freed_indices")


def _check(inp, what=""):
    da = DeviceAccept(inp)
    da.run()
    torch.cuda.synchronize()
    assert da.status() == 0, what
    got = da.outputs()
    ref = accept_batched(inp.logits, inp.draft_tokens, inp.tree_parent, inp.kv_indices, inp.kv_indptr,
                         inp.prefix_lens)
    for k in KEYS:
        np.testing.assert_array_equal(got[k], ref[k], err_msg=f"{what}: {k}")
    return da, ref


@pytest.mark.parametrize("name", ["accept_small", "accept_long", "accept_batch"])
def test_workloads(name):
    _check(accept_workload(name), name)


@pytest.mark.parametrize("vocab", [2, 7, 1001, 4096, 4097, 129280])
@pytest.mark.parametrize("tree", ["chain", "uniform", "bounded"])
def test_vocab_sizes_and_trees(vocab, tree):
    inp = make_accept_inputs("v", batch=3, n_nodes=12, vocab=vocab, prefixes=[0, 5, 33], tree=tree,
                             pool_rows=512, p_match=0.9, seed=vocab + len(tree))
    _check(inp, f"vocab {vocab} {tree}")


@pytest.mark.parametrize("T", [1, 2, 31, 32, 33, 63, 64])
def test_node_counts(T):
    inp = make_accept_inputs("t", batch=2, n_nodes=T, vocab=3000, prefixes=[7, 0], tree="bounded",
                             pool_rows=1024, p_match=0.95, seed=T)
    _check(inp, f"T={T}")


def test_chain_fully_accepted():
    inp = make_accept_inputs("c", batch=1, n_nodes=64, vocab=50000, prefixes=[100], tree="chain",
                             pool_rows=4096, p_match=1.0, seed=5)
    da, ref = _check(inp, "chain")
    assert int(ref["accept_len"][0]) == 64


def _with_logits(inp: AcceptInputs, logits: torch.Tensor) -> AcceptInputs:
    return AcceptInputs(logits=logits.to(torch.bfloat16), draft_tokens=inp.draft_tokens,
                        tree_parent=inp.tree_parent, kv_indices=inp.kv_indices, kv_indptr=inp.kv_indptr,
                        prefix_lens=inp.prefix_lens, planted=inp.planted, pool_rows=inp.pool_rows,
                        meta=inp.meta)


def test_ties_across_segments_take_the_first_index():
    # Equal maxima far apart (different argmax segments) and inside one
    # segment; an all-zero row (every index ties, and -0.0 equals +0.0).
    base = make_accept_inputs("tie", batch=1, n_nodes=4, vocab=129280, prefixes=[3], tree="chain",
                              pool_rows=256, p_match=1.0, seed=9)
    x = torch.zeros(1, 5, 129280)
    x[0, 0, [70000, 129279, 555]] = 4.0          # first index 555
    x[0, 1, [9, 10]] = 2.5                        # first index 9
    x[0, 2, :] = -1.0
    x[0, 2, [128000, 64000]] = -0.5               # first index 64000
    x[0, 3, 1::2] = -0.0                          # row 3: zeros and negative zeros -> 0
    x[0, 4, 77] = 1.0
    draft = torch.tensor([[555, 9, 64000, 0]], dtype=torch.int32)
    inp = _with_logits(base, x)
    inp.draft_tokens = draft
    da, ref = _check(inp, "ties")
    assert ref["accepted_nodes"][0].tolist() == [0, 1, 2, 3]
    assert int(ref["next_token"][0]) == 77


def test_two_calls_in_a_row_and_graph_replay():
    inp = accept_workload("accept_batch")
    da = DeviceAccept(inp)
    da.run()
    da.run()     # the argmax keys of the first call must not leak into the second
    torch.cuda.synchronize()
    ref = accept_batched(inp.logits, inp.draft_tokens, inp.tree_parent, inp.kv_indices, inp.kv_indptr,
                         inp.prefix_lens)
    for k in KEYS:
        np.testing.assert_array_equal(da.outputs()[k], ref[k])
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        da.run(s)
    s.synchronize()
    with torch.cuda.graph(g, stream=s):
        da.run(s)
    other = accept_workload("accept_batch", seed=99)
    da.logits.copy_(other.logits)
    da.draft.copy_(other.draft_tokens)
    da.parent.copy_(other.tree_parent)
    g.replay()
    torch.cuda.synchronize()
    ref2 = accept_batched(other.logits, other.draft_tokens, other.tree_parent, inp.kv_indices,
                          inp.kv_indptr, inp.prefix_lens)
    for k in KEYS:
        np.testing.assert_array_equal(da.outputs()[k], ref2[k], err_msg=k)


def test_bad_parent_and_bad_length_are_flagged():
    inp = accept_workload("accept_small")
    bad = inp.tree_parent.clone()
    bad[0, 3] = 3                                  # not an earlier node
    inp2 = _with_logits(inp, inp.logits.float())
    inp2.tree_parent = bad
    da = DeviceAccept(inp2)
    da.run()
    assert da.status() & B.DDTREE_ST_BAD_PARENT
    inp3 = _with_logits(inp, inp.logits.float())
    inp3.prefix_lens = inp.prefix_lens + 1         # lengths disagree with kv_indptr
    da = DeviceAccept(inp3)
    da.run()
    assert da.status() & B.DDTREE_ST_BAD_LENGTH
    out = da.outputs()
    assert (out["commit_indices"] == -1).all() and (out["freed_indices"] == -1).all()
