"""Pins of the flattened-mask reader: masks built independently from known
trees (networkx ancestry) give those trees back, and every way a mask can fail
to be a tree mask is caught."""
import itertools

import numpy as np
import pytest
import torch

from oracle.mask_oracle import tree_from_mask, trees_from_flat_mask
from speculative_decode_tree_gb300.workloads import flat_tree_masks, tree_mask

nx = pytest.importorskip("networkx")


def _nx_mask(parents, P):
    g = nx.DiGraph()
    g.add_nodes_from(range(len(parents)))
    g.add_edges_from((p, i) for i, p in enumerate(parents) if p >= 0)
    T = len(parents)
    m = np.zeros((T, P + T), np.uint8)
    m[:, :P] = 1
    for i in range(T):
        for j in nx.ancestors(g, i) | {i}:
            m[i, P + j] = 1
    return m


@pytest.mark.parametrize("T", [1, 2, 3, 4, 5])
@pytest.mark.parametrize("P", [0, 3])
def test_every_small_tree_round_trips(T, P):
    for parents in itertools.product(*[range(-1, i) for i in range(T)]):
        parents = list(parents)
        m = _nx_mask(parents, P)
        r = tree_from_mask(m, P)
        assert r["parents"] == parents and r["valid"], parents
        # the generator's mask builder agrees with the networkx construction
        assert np.array_equal(tree_mask(parents, P).numpy(), m)


def test_hand_worked_mask():
    # Prefix of 2; nodes: 0 root, 1 root, 2 child of 0, 3 child of 2.
    m = np.array([[1, 1, 1, 0, 0, 0],
                  [1, 1, 0, 1, 0, 0],
                  [1, 1, 1, 0, 1, 0],
                  [1, 1, 1, 0, 1, 1]], np.uint8)
    r = tree_from_mask(m, 2)
    assert r["parents"] == [-1, -1, 0, 2] and r["valid"]


def test_broken_masks_are_caught():
    good = _nx_mask([-1, 0, 1, 0], 2)
    no_self = good.copy(); no_self[2, 2 + 2] = 0
    assert not tree_from_mask(no_self, 2)["self_ok"]
    prefix_hole = good.copy(); prefix_hole[1, 0] = 0
    assert not tree_from_mask(prefix_hole, 2)["prefix_ok"]
    sibling = good.copy(); sibling[3, 2 + 2] = 1          # node 3 (child of 0) also sees node 2 (0 -> 1 -> 2)
    r = tree_from_mask(sibling, 2)
    assert not r["chain_ok"] and r["parents"][3] == 2     # the rule still names the largest seen node
    later = good.copy(); later[1, 2 + 3] = 1              # node 1 sees a later node
    assert not tree_from_mask(later, 2)["chain_ok"]
    skip = _nx_mask([-1, 0, 1, 2], 2); skip[3, 2 + 1] = 0  # node 3 sees 2 and 0 but not 1 (2's parent)
    assert not tree_from_mask(skip, 2)["chain_ok"]
    for bad in (no_self, prefix_hole, sibling, later, skip):
        assert not tree_from_mask(bad, 2)["valid"]


def test_flat_batch_layout():
    parents = torch.tensor([[-1, 0, 0], [-1, -1, 1]], dtype=torch.int32)
    plen = torch.tensor([4, 0], dtype=torch.int32)
    flat, indptr = flat_tree_masks(parents, plen)
    assert indptr.tolist() == [0, 3 * 7, 3 * 7 + 3 * 3]
    out = trees_from_flat_mask(flat.numpy(), indptr.tolist(), plen.tolist(), 3)
    assert out["parents"].tolist() == parents.tolist() and out["valid"].all()
