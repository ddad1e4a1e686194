"""GPU parity of Tier-1 KV relocation against the oracle (byte-exact pool,
indices and old indices), its all-or-nothing checks, and the end-to-end
property: verify attention on the relocated rows equals verify attention on
the scattered rows, bit for bit."""
import pytest
import torch

from oracle import relocate
from speculative_decode_tree_gb300 import binding as B
from speculative_decode_tree_gb300.runner import DeviceVerify
from speculative_decode_tree_gb300.workloads import RelocateInputs, relocate_workload, workload

pytestmark = pytest.mark.gpu


def _run(inp: RelocateInputs, with_old=True):
    pool = inp.kv_pool.cuda()
    idx = inp.kv_indices.cuda()
    ptr = inp.kv_indptr.cuda()
    dst = inp.dest_base.cuda()
    old = torch.full_like(idx, -7) if with_old else None
    ws = torch.empty(B.ddtree_relocate_kv_workspace_size(pool.shape[0]), dtype=torch.uint8, device="cuda")
    B.ddtree_relocate_kv(pool, idx, ptr, dst, int(inp.kv_indptr[-1]), ws, old)
    torch.cuda.synchronize()
    return pool, idx, old, B.ddtree_verify_mla_check(ws)


def _compare(inp, what):
    pool, idx, old, status = _run(inp)
    ref_pool, ref_idx, ref_old, err = relocate(inp.kv_pool, inp.kv_indices, inp.kv_indptr, inp.dest_base)
    assert status == 0 and not any(err.values()), what
    assert torch.equal(idx.cpu(), ref_idx), what
    assert torch.equal(old.cpu(), ref_old), what
    assert torch.equal(pool.cpu().view(torch.int16), ref_pool.view(torch.int16)), what


@pytest.mark.parametrize("name", ["relocate_small", "relocate_long"])
def test_workloads(name):
    _compare(relocate_workload(name), name)


def test_batch_workload():
    # 448,768 rows over 8 requests in a 1M-row pool; the oracle copies row by row.
    _compare(relocate_workload("relocate_batch"), "relocate_batch")


@pytest.mark.parametrize("prefixes,T", [([0], 1), ([1], 1), ([0, 0, 5], 2), ([63, 64, 65], 3)])
def test_small_and_empty_requests(prefixes, T):
    inp = relocate_workload("relocate_small", prefixes=prefixes, n_nodes=T, pool_rows=1024, seed=len(prefixes) + T)
    _compare(inp, f"{prefixes} {T}")


def _bad(inp, **kw):
    d = dict(kv_pool=inp.kv_pool, kv_indices=inp.kv_indices, kv_indptr=inp.kv_indptr,
             dest_base=inp.dest_base, meta=inp.meta)
    d.update(kw)
    return RelocateInputs(**d)


def test_checks_leave_pool_and_indices_untouched():
    inp = relocate_workload("relocate_small")
    n_rows = inp.pool_rows
    cases = {
        "overlap: destination covers a source": (_bad(inp, dest_base=torch.tensor(
            [int(inp.kv_indices[5]), int(inp.dest_base[1]), int(inp.dest_base[2])], dtype=torch.int32)),
            B.DDTREE_ST_OVERLAP),
        "overlap: two destinations": (_bad(inp, dest_base=torch.tensor(
            [int(inp.dest_base[1]), int(inp.dest_base[1]), int(inp.dest_base[2])], dtype=torch.int32)),
            B.DDTREE_ST_OVERLAP),
        "index past the pool": (_bad(inp, kv_indices=torch.where(torch.arange(inp.kv_indices.numel()) == 3,
                                                                 torch.tensor(n_rows, dtype=torch.int32),
                                                                 inp.kv_indices)), B.DDTREE_ST_BAD_INDEX),
        "destination past the pool": (_bad(inp, dest_base=torch.tensor(
            [int(inp.dest_base[0]), int(inp.dest_base[1]), n_rows - 3], dtype=torch.int32)),
            B.DDTREE_ST_BAD_LENGTH),
    }
    for what, (bad, bit) in cases.items():
        pool, idx, old, status = _run(bad)
        assert status & bit, what
        assert torch.equal(pool.cpu().view(torch.int16), bad.kv_pool.view(torch.int16)), what
        assert torch.equal(idx.cpu(), bad.kv_indices), what
        assert torch.equal(old.cpu(), bad.kv_indices), what


def test_verify_on_relocated_rows_is_bitwise_unchanged():
    import dataclasses
    base = workload("long_scattered")
    n = int(base.kv_indptr[-1])
    # The scattered rows cover the whole pool, so give the pool n free rows on
    # top for the destination region.
    grown = torch.cat([base.kv_pool, torch.zeros(n, base.kv_pool.shape[1], dtype=base.kv_pool.dtype)])
    inp = dataclasses.replace(base, kv_pool=grown)
    dv = DeviceVerify(inp)
    dv.run()
    torch.cuda.synchronize()
    assert dv.status() == 0
    out0, lse0 = dv.out.clone(), dv.lse.clone()
    ws = torch.empty(B.ddtree_relocate_kv_workspace_size(inp.pool_rows), dtype=torch.uint8, device="cuda")
    dst = torch.tensor([base.pool_rows], dtype=torch.int32, device="cuda")
    B.ddtree_relocate_kv(dv.kv_pool, dv.kv_indices, dv.kv_indptr, dst, n, ws)
    torch.cuda.synchronize()
    assert B.ddtree_verify_mla_check(ws) == 0
    assert torch.equal(dv.kv_indices.cpu(), torch.arange(base.pool_rows, base.pool_rows + n, dtype=torch.int32))
    dv.run()
    torch.cuda.synchronize()
    assert dv.status() == 0
    assert torch.equal(dv.out, out0) and torch.equal(dv.lse, lse0)


def test_two_calls_in_a_row_reuse_the_workspace():
    inp = relocate_workload("relocate_small")
    pool = inp.kv_pool.cuda()
    idx = inp.kv_indices.cuda()
    ptr = inp.kv_indptr.cuda()
    ws = torch.empty(B.ddtree_relocate_kv_workspace_size(pool.shape[0]), dtype=torch.uint8, device="cuda")
    # First move to the top region, then back down to a region of the (now free) low rows.
    B.ddtree_relocate_kv(pool, idx, ptr, inp.dest_base.cuda(), int(inp.kv_indptr[-1]), ws)
    moved = idx.clone()
    low = torch.tensor([0, int(inp.kv_indptr[1]), int(inp.kv_indptr[2])], dtype=torch.int32)
    # The low region [0, total) may hold original source rows: after the first
    # move nothing reads them, so the second call is valid.
    B.ddtree_relocate_kv(pool, idx, ptr, low.cuda(), int(inp.kv_indptr[-1]), ws)
    torch.cuda.synchronize()
    assert B.ddtree_verify_mla_check(ws) == 0
    ref_pool, ref_idx, _, _ = relocate(inp.kv_pool, inp.kv_indices, inp.kv_indptr, inp.dest_base)
    ref_pool2, ref_idx2, _, err = relocate(ref_pool, moved.cpu(), inp.kv_indptr, low)
    assert not any(err.values())
    assert torch.equal(idx.cpu(), ref_idx2)
    assert torch.equal(pool.cpu().view(torch.int16), ref_pool2.view(torch.int16))


def test_overlapping_destinations_within_one_warp_are_caught():
    # Two small requests whose destination regions overlap by a few rows that
    # fall in the same 32-row group (the same warp marks both).
    inp = relocate_workload("relocate_small", prefixes=[6, 6], n_nodes=2, pool_rows=1024, seed=3)
    top = int(inp.dest_base[0])
    bad = _bad(inp, dest_base=torch.tensor([top, top + 5], dtype=torch.int32))
    pool, idx, old, status = _run(bad)
    assert status & B.DDTREE_ST_OVERLAP
    assert torch.equal(idx.cpu(), bad.kv_indices)
