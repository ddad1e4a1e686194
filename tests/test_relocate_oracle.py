"""Pins of the KV-relocation oracle: hand-worked moves, the rules a call must
keep, and the property that matters downstream, that verify attention gives
the same result on the relocated rows."""
import torch

from oracle.relocate_oracle import relocate, relocation_errors
from oracle.verify_oracle import verify_request


def _pool(rows, width=4):
    # Row r holds the values r*10 + column: every row is distinguishable.
    return (torch.arange(rows)[:, None] * 10 + torch.arange(width)[None, :]).to(torch.bfloat16)


def test_hand_worked_single_request():
    pool = _pool(12)
    new_pool, new_idx, old_idx, err = relocate(pool, torch.tensor([5, 2, 7], dtype=torch.int32),
                                              torch.tensor([0, 3], dtype=torch.int32),
                                              torch.tensor([8], dtype=torch.int32))
    assert not any(err.values())
    assert new_idx.tolist() == [8, 9, 10]
    assert old_idx.tolist() == [5, 2, 7]
    assert torch.equal(new_pool[8], pool[5]) and torch.equal(new_pool[9], pool[2]) and torch.equal(new_pool[10], pool[7])
    assert torch.equal(new_pool[:8], pool[:8]) and torch.equal(new_pool[11], pool[11])  # nothing else moves


def test_two_requests_sharing_a_row_and_an_empty_request():
    pool = _pool(16)
    idx = torch.tensor([3, 4, 4, 9, 1], dtype=torch.int32)      # request 0: [3, 4], request 1: [4, 9, 1]
    ptr = torch.tensor([0, 2, 2, 5], dtype=torch.int32)         # request 1 is empty
    dst = torch.tensor([10, 15, 12], dtype=torch.int32)
    new_pool, new_idx, old_idx, err = relocate(pool, idx, ptr, dst)
    assert not any(err.values())
    assert new_idx.tolist() == [10, 11, 12, 13, 14]
    for k, src in enumerate([3, 4, 4, 9, 1]):
        assert torch.equal(new_pool[new_idx[k]], pool[src])


def test_rules_leave_everything_unchanged():
    pool = _pool(16)
    cases = [
        ([3, 4], [0, 2], [4], "overlap"),          # destination covers a row being read
        ([3, 4, 5], [0, 1, 3], [8, 8], "overlap"),  # two destination regions overlap
        ([3, 16], [0, 2], [8], "bad_index"),        # index past the pool
        ([3, -1], [0, 2], [8], "bad_index"),
        ([3, 4], [0, 2], [15], "bad_dest"),         # destination runs past the pool
        ([3, 4], [0, 2], [-1], "bad_dest"),
    ]
    for idx, ptr, dst, which in cases:
        err = relocation_errors(16, idx, ptr, dst)
        assert err[which], (idx, ptr, dst)
        new_pool, new_idx, old_idx, err2 = relocate(pool, torch.tensor(idx, dtype=torch.int32),
                                                   torch.tensor(ptr, dtype=torch.int32),
                                                   torch.tensor(dst, dtype=torch.int32))
        assert torch.equal(new_pool, pool) and new_idx.tolist() == idx and old_idx.tolist() == idx


def test_verify_attention_is_unchanged_by_relocation():
    g = torch.Generator().manual_seed(7)
    rows, P, T, H = 300, 40, 6, 2
    pool = torch.randn(rows, 576, generator=g).to(torch.bfloat16)
    idx = torch.randperm(200, generator=g)[:P + T].to(torch.int32)        # rows below 200
    parent = [-1, 0, 0, 1, -1, 4]
    ql = torch.randn(T, H, 512, generator=g).to(torch.bfloat16)
    qr = torch.randn(T, H, 64, generator=g).to(torch.bfloat16)
    O0, L0 = verify_request(ql, qr, pool, idx, P, parent, 0.0721)
    new_pool, new_idx, _, err = relocate(pool, idx, torch.tensor([0, P + T], dtype=torch.int32),
                                         torch.tensor([220], dtype=torch.int32))
    assert not any(err.values())
    assert new_idx.tolist() == list(range(220, 220 + P + T))
    O1, L1 = verify_request(ql, qr, new_pool, new_idx, P, parent, 0.0721)
    assert torch.equal(O0, O1) and torch.equal(L0, L1)
