"""GPU parity of the flattened-mask reader: exact parents and ancestor bits
against the oracle on every verify workload's trees, the broken-mask flags,
and verify attention run on the recovered tree matching the original bit for
bit."""
import numpy as np
import pytest
import torch

from oracle import ancestor_bits, trees_from_flat_mask
from speculative_decode_tree_gb300 import binding as B
from speculative_decode_tree_gb300.runner import DeviceVerify
from speculative_decode_tree_gb300.workloads import flat_tree_masks, make_inputs, tree_mask
from parity_util import cached_workload

pytestmark = pytest.mark.gpu


def _read(flat, indptr, plen, T, B_):
    parent = torch.full((B_, T), -9, dtype=torch.int32, device="cuda")
    anc = torch.zeros(B_, T, dtype=torch.int64, device="cuda")
    ws = torch.empty(B.ddtree_tree_from_mask_workspace_size(B_, T), dtype=torch.uint8, device="cuda")
    B.ddtree_tree_from_mask(flat.cuda(), indptr.cuda(), plen.cuda(), parent, ws, anc)
    torch.cuda.synchronize()
    return parent.cpu(), anc.cpu(), B.ddtree_verify_mla_check(ws)


@pytest.mark.parametrize("name", ["tiny", "tp8_slice", "long_scattered", "unsharded_heads", "mixed_batch"])
def test_workload_trees_round_trip(name):
    inp = cached_workload(name)
    flat, indptr = flat_tree_masks(inp.tree_parent, inp.prefix_lens)
    parent, anc, status = _read(flat, indptr, inp.prefix_lens, inp.n_nodes, inp.batch)
    assert status == 0
    assert torch.equal(parent, inp.tree_parent)
    ref = trees_from_flat_mask(flat.numpy(), indptr.tolist(), inp.prefix_lens.tolist(), inp.n_nodes)
    assert np.array_equal(parent.numpy(), ref["parents"]) and ref["valid"].all()
    for b in range(inp.batch):
        want = [int(x) for x in ancestor_bits(inp.tree_parent[b].tolist())]
        got = [int(x) & ((1 << 64) - 1) for x in anc[b].tolist()]
        assert got == want, (name, b)


@pytest.mark.parametrize("P,T", [(0, 1), (1, 1), (0, 64), (15, 33), (17, 64), (4099, 7)])
def test_odd_sizes_and_bool_masks(P, T):
    g = torch.Generator().manual_seed(P * 100 + T)
    parents = [int(torch.randint(-1, i, (1,), generator=g)) for i in range(T)]
    flat, indptr = flat_tree_masks(torch.tensor([parents, parents[::1]], dtype=torch.int32),
                                   torch.tensor([P, P + 3], dtype=torch.int32))
    parent, anc, status = _read(flat.bool(), indptr, torch.tensor([P, P + 3], dtype=torch.int32), T, 2)
    assert status == 0
    assert parent.tolist() == [parents, parents]


def test_broken_masks_and_lengths_are_flagged():
    parents = [-1, 0, 1, 0]
    P = 21
    good = tree_mask(parents, P)
    cases = []
    m = good.clone(); m[2, P + 2] = 0; cases.append(m)          # a node that does not see itself
    m = good.clone(); m[1, 13] = 0; cases.append(m)             # a hole in the prefix
    m = good.clone(); m[3, P + 2] = 1; cases.append(m)          # node 3 sees a node off its chain
    for m in cases:
        flat = m.reshape(-1)
        parent, anc, status = _read(flat, torch.tensor([0, flat.numel()]), torch.tensor([P], dtype=torch.int32), 4, 1)
        assert status & B.DDTREE_ST_BAD_MASK
        ref = trees_from_flat_mask(flat.numpy(), [0, flat.numel()], [P], 4)
        assert parent[0].tolist() == ref["parents"][0].tolist() and not ref["valid"][0]
    flat = good.reshape(-1)
    parent, anc, status = _read(flat, torch.tensor([0, flat.numel() - 1]), torch.tensor([P], dtype=torch.int32), 4, 1)
    assert status & B.DDTREE_ST_BAD_LENGTH and parent[0].tolist() == [-1] * 4


def test_verify_on_the_recovered_tree_is_bitwise_equal():
    inp = make_inputs("m", batch=3, n_heads=8, prefixes=[5000, 0, 777], n_nodes=24, tree="uniform",
                      pool_rows=65536, index_mode="sample", seed=31)
    dv = DeviceVerify(inp)
    dv.run()
    torch.cuda.synchronize()
    out0, lse0 = dv.out.clone(), dv.lse.clone()
    flat, indptr = flat_tree_masks(inp.tree_parent, inp.prefix_lens)
    ws = torch.empty(B.ddtree_tree_from_mask_workspace_size(3, 24), dtype=torch.uint8, device="cuda")
    dv.tree_parent.fill_(-1)
    B.ddtree_tree_from_mask(flat.cuda(), indptr.cuda(), dv.prefix_lens, dv.tree_parent, ws)
    dv.run()
    torch.cuda.synchronize()
    assert B.ddtree_verify_mla_check(ws) == 0 and dv.status() == 0
    assert torch.equal(dv.out, out0) and torch.equal(dv.lse, lse0)
