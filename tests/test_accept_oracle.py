"""Pins of the greedy-acceptance oracle against cases whose answer is known
without running it: hand-worked trees, the tie rules, and an independent
characterisation of the accepted path checked on every tree of up to five
nodes."""
import itertools
import random

import numpy as np
import pytest
import torch

from oracle.accept_oracle import accept_batched, accept_request, argmax_rows, greedy_path


def _rows(planted, vocab=16, base=0.0):
    """Logit rows that are `base` everywhere except 5.0 at the planted token."""
    x = torch.full((len(planted), vocab), base)
    for r, tok in enumerate(planted):
        x[r, tok] = 5.0
    return x.to(torch.bfloat16)


def test_argmax_takes_first_of_equal_maxima():
    x = torch.tensor([[1.0, 3.0, 3.0, 2.0], [7.0, 7.0, 7.0, 7.0], [-4.0, -2.5, -9.0, -2.5]],
                     dtype=torch.bfloat16)
    assert argmax_rows(x).tolist() == [1, 0, 1]


def test_argmax_compares_bf16_values():
    # 1.0 and 1.0 + 2^-9 round to the same bf16 value: a tie, so index 0.
    x = torch.tensor([[1.0, 1.0 + 2.0 ** -9]]).to(torch.bfloat16)
    assert argmax_rows(x).tolist() == [0]


def test_chain_with_every_draft_right_accepts_everything():
    T = 6
    planted = [3, 9, 1, 14, 0, 7, 11]          # row r: prefix end (r=0), then node r-1
    parent = [i - 1 for i in range(T)]
    draft = [planted[i] for i in range(T)]     # node i's parent row is row i
    rows = [100 + i for i in range(T)]
    r = accept_request(_rows(planted), draft, parent, rows)
    assert r["path"] == [0, 1, 2, 3, 4, 5]
    assert r["accept_len"] == 6
    assert r["next_token"] == 11               # the target's token after the last node
    assert r["commit"] == rows and r["freed"] == []


def test_wrong_first_draft_accepts_nothing():
    planted = [3, 9, 1]
    r = accept_request(_rows(planted), [4, 9], [-1, 0], [50, 51])
    assert r["accept_len"] == 0 and r["path"] == []
    assert r["next_token"] == 3
    assert r["commit"] == [] and r["freed"] == [50, 51]


def test_sibling_tie_takes_smaller_index_even_if_the_other_branch_is_longer():
    # Roots 0 and 1 both draft the prefix-end token 2.  Node 1 has a matching
    # child (node 2) while node 0 has none; the walk still takes node 0.
    planted = [2, 6, 8, 5]          # rows: prefix end, node 0, node 1, node 2
    parent = [-1, -1, 1]
    draft = [2, 2, 8]
    r = accept_request(_rows(planted), draft, parent, [10, 11, 12])
    assert r["path"] == [0]
    assert r["next_token"] == 6
    assert r["freed"] == [11, 12]


def test_hand_worked_tree():
    #        prefix end
    #        /        \
    #      n0          n1
    #     /  \          |
    #   n2    n3        n4
    #   |
    #   n5 -- n6
    # Target tokens: end->7, n0->4, n1->9, n2->1, n3->2, n4->3, n5->8, n6->0.
    # Drafts: n0=7 (right), n1=5, n2=3, n3=4 (right: n0's target is 4),
    # n4=9, n5=1, n6=8.  The walk: end predicts 7 -> n0; n0 predicts 4 -> n3
    # (n2 drafted 3); n3 predicts 2 -> n3 has no children: stop with token 2.
    planted = [7, 4, 9, 1, 2, 3, 8, 0]
    parent = [-1, -1, 0, 0, 1, 2, 5]
    draft = [7, 5, 3, 4, 9, 1, 8]
    rows = [200, 201, 202, 203, 204, 205, 206]
    r = accept_request(_rows(planted), draft, parent, rows)
    assert r["path"] == [0, 3]
    assert r["next_token"] == 2
    assert r["commit"] == [200, 203]
    assert r["freed"] == [201, 202, 204, 205, 206]


def _accepted_by_definition(pred, draft, parent):
    """Independent characterisation for trees whose siblings draft distinct
    tokens: node x is accepted iff its draft equals the prediction of its
    parent row and its parent is accepted (or is the prefix end).  Such nodes
    form one root path; the next token is the prediction after the deepest."""
    T = len(parent)
    ok = [False] * T
    for x in range(T):                           # parents come before children
        p = parent[x]
        row = 0 if p < 0 else 1 + p
        ok[x] = draft[x] == pred[row] and (p < 0 or ok[p])
    acc = [x for x in range(T) if ok[x]]

    def depth(x):
        d = 0
        while x >= 0:
            d += 1
            x = parent[x]
        return d
    acc.sort(key=depth)
    nxt = pred[0] if not acc else pred[1 + acc[-1]]
    return acc, nxt


def _all_parent_arrays(T):
    return itertools.product(*[range(-1, i) for i in range(T)])


@pytest.mark.parametrize("T", [1, 2, 3, 4, 5])
def test_every_small_tree_matches_the_definition(T):
    rng = random.Random(T)
    vocab = 6
    for parent in _all_parent_arrays(T):
        parent = list(parent)
        for _ in range(3):
            pred = [rng.randrange(vocab) for _ in range(T + 1)]
            draft = [0] * T
            for p in [-1] + list(range(T)):
                kids = [c for c in range(T) if parent[c] == p]
                if not kids:
                    continue
                toks = rng.sample(range(vocab), len(kids))      # distinct among siblings
                want = pred[0 if p < 0 else 1 + p]
                if want not in toks and rng.random() < 0.7:      # often one child is right
                    toks[rng.randrange(len(kids))] = want
                for c, t in zip(kids, toks):
                    draft[c] = t
            path, nxt = greedy_path(pred, draft, parent)
            acc, nxt2 = _accepted_by_definition(pred, draft, parent)
            assert path == acc and nxt == nxt2, (parent, pred, draft)


def test_commit_and_freed_partition_the_tree_rows():
    g = torch.Generator().manual_seed(3)
    T, vocab = 9, 12
    parent = [-1, 0, 0, 1, -1, 3, 5, 2, 6]
    logits = torch.randn(T + 1, vocab, generator=g).to(torch.bfloat16)
    pred = argmax_rows(logits).tolist()
    draft = [pred[0 if p < 0 else 1 + p] if i in (0, 1, 3, 5) else (pred[0 if p < 0 else 1 + p] + 1) % vocab
             for i, p in enumerate(parent)]
    rows = list(range(500, 500 + T))
    r = accept_request(logits, draft, parent, rows)
    assert r["path"] == [0, 1, 3, 5]
    assert sorted(r["commit"] + r["freed"]) == rows
    assert r["commit"] == [rows[i] for i in r["path"]]


def test_batched_layout_pads_with_minus_one():
    planted = [[3, 9, 1], [5, 5, 2]]
    logits = torch.stack([_rows(planted[0]), _rows(planted[1])])
    draft = torch.tensor([[3, 9], [0, 0]], dtype=torch.int32)
    parent = torch.tensor([[-1, 0], [-1, -1]], dtype=torch.int32)
    kv = torch.tensor([7, 8, 70, 71, 9, 90, 91], dtype=torch.int32)   # request 0: P=2, request 1: P=1
    indptr = torch.tensor([0, 4, 7], dtype=torch.int32)
    plen = torch.tensor([2, 1], dtype=torch.int32)
    out = accept_batched(logits, draft, parent, kv, indptr, plen)
    assert out["accept_len"].tolist() == [2, 0]
    assert out["next_token"].tolist() == [1, 5]
    assert out["accepted_nodes"].tolist() == [[0, 1], [-1, -1]]
    assert out["commit_indices"].tolist() == [[70, 71], [-1, -1]]
    assert out["freed_indices"].tolist() == [[-1, -1], [90, 91]]
