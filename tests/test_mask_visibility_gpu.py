"""GPU parity where a wrong ancestor mask would show.

At long prefixes the tree keys carry a tiny share of the softmax mass, so a
wrong mask can still pass the output tolerance.  These cases make the tree
keys score ~70 nats above the prefix keys ("spiked" keys), so each node's
output is the mean of V over its own ancestors: a mask that adds or drops a
single tree key moves O by far more than the tolerance.  The tree segment is
placed where the kernels' mask arithmetic changes: across a 128-key tile
boundary, across a split boundary of the library's own plan, and in the
65,536-key production plan with both 128-row tiles of the cluster of four
holding tree nodes.  Every row is compared with the float64 oracle, and the
oracle with one parent link cut is checked to differ (so the case can see a
mask error at all).

Also here: queries passed as strided views of one [nodes, heads, 576] tensor
(the unsharded-heads shape), and a wait bound so short that every kernel wait
expires: the call must report DDTREE_ST_TIMEOUT, return finite outputs, and
leave the device usable for the next call.
"""
import pytest
import torch

from speculative_decode_tree_gb300 import binding as B
from speculative_decode_tree_gb300.runner import DeviceVerify
from speculative_decode_tree_gb300.workloads import make_inputs
from parity_util import assert_within_tolerance, cached_workload, oracle_rows

pytestmark = pytest.mark.gpu

KERNELS = [B.DDTREE_KERNEL_SIMT, B.DDTREE_KERNEL_TC, B.DDTREE_KERNEL_TC2]
SPIKE_Q, SPIKE_K = 8.0, 128.0   # q_rope[..., 0] and the tree rows' first rope column


def _spiked(P, T, H, seed, pool_rows=None, tree="uniform"):
    pool_rows = pool_rows or max(1024, 2 * (P + T) + 64)
    inp = make_inputs("spiked", batch=1, n_heads=H, prefixes=[P], n_nodes=T, tree=tree,
                      pool_rows=pool_rows, index_mode="sample", seed=seed)
    inp.q_latent.zero_()
    inp.q_rope.zero_()
    inp.q_rope[..., 0] = SPIKE_Q
    inp.kv_pool[inp.kv_indices[P:].long(), 512] = SPIKE_K
    return inp


def _check_mask_visible(inp, out):
    """Cutting one node's parent link moves the oracle by >= 0.1 at that node,
    and the GPU output stays on the right side of that gap."""
    O_ref, _ = oracle_rows(inp, 0)
    par = inp.tree_parent[0].tolist()
    depth = []
    for p in par:
        depth.append(1 if p < 0 else depth[p] + 1)
    i = max(range(len(par)), key=lambda j: depth[j])
    if par[i] < 0:
        pytest.skip("forest of roots only: no parent link to cut")
    saved = inp.tree_parent.clone()
    inp.tree_parent[0, i] = -1
    O_wrong, _ = oracle_rows(inp, 0, nodes=[i])
    inp.tree_parent.copy_(saved)
    assert float((O_wrong[0] - O_ref[i]).abs().max()) >= 0.1
    assert float((out[i].double().cpu() - O_wrong[0]).abs().max()) >= 0.09


def _run_all_rows(inp, kernel, what, plan=None):
    dv = DeviceVerify(inp, kernel=kernel, plan=plan)
    dv.run()
    torch.cuda.synchronize()
    assert dv.status() == 0, what
    O_ref, L_ref = oracle_rows(inp, 0)
    assert_within_tolerance(dv.out, dv.lse, O_ref, L_ref, what)
    _check_mask_visible(inp, dv.out)
    return dv


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("P,T,H", [(120, 16, 8), (100, 32, 8), (250, 64, 2), (127, 2, 8)])
def test_spiked_tree_across_a_tile_boundary(kernel, P, T, H):
    """Tree keys P .. P+T-1 straddle key 128 (the tensor-core kernels' tile)
    and key 32 multiples (the CUDA-core kernel's tile)."""
    inp = _spiked(P, T, H, seed=1000 + P + T, tree="chain" if T <= 4 else "uniform")
    _run_all_rows(inp, kernel, f"tile boundary P={P} T={T} H={H} kernel={kernel}")


def _split_crossing_prefix(kernel, T, H, lo, hi, pool_rows):
    """A prefix length in [lo, hi) whose plan on this device puts a split
    boundary strictly inside the tree segment [P, P+T)."""
    for P in range(lo, hi):
        plan = B.ddtree_verify_mla_plan_ex(1, T, H, [P], pool_rows, 0, kernel)
        c = plan.chunk_keys
        first_boundary_after_P = (P // c + 1) * c
        if plan.total_splits > 1 and first_boundary_after_P < P + T:
            return P, plan
    pytest.skip("no prefix in range puts a split boundary inside the tree")


@pytest.mark.parametrize("kernel", KERNELS)
def test_spiked_tree_across_a_split_boundary(kernel):
    T, H = 32, 8
    P, plan = _split_crossing_prefix(kernel, T, H, 2900, 3400, 8192)
    inp = _spiked(P, T, H, seed=77, pool_rows=8192)
    _run_all_rows(inp, kernel, f"split boundary P={P} chunk={plan.chunk_keys} kernel={kernel}", plan=plan)


@pytest.mark.parametrize("where", ["tile_start", "tile_crossing", "split_crossing"])
def test_spiked_tree_in_the_65k_production_plan(where):
    """The long-prefix shape (65,536 keys, 32 nodes, 8 heads, 262,144-row
    pool) in the plan the benchmark runs: the cluster-of-four kernel with both
    row tiles live (nodes 16..31 are the second tile), every row compared."""
    T, H, rows = 32, 8, 262144
    if where == "tile_start":
        P = 65536
    elif where == "tile_crossing":
        P = 65536 - 16
    else:
        P, _ = _split_crossing_prefix(B.DDTREE_KERNEL_AUTO, T, H, 65536 - 2048, 65536 + 2048, rows)
    inp = _spiked(P, T, H, seed=2, pool_rows=rows)
    dv = DeviceVerify(inp)
    assert dv.plan.kernel == B.DDTREE_KERNEL_TC2 and dv.plan.row_tiles == 2
    dv.run()
    torch.cuda.synchronize()
    assert dv.status() == 0
    O_ref, L_ref = oracle_rows(inp, 0)
    assert_within_tolerance(dv.out, dv.lse, O_ref, L_ref, f"65k {where} P={P}")
    _check_mask_visible(inp, dv.out)


def test_strided_queries_unsharded_shape():
    """Q given as one [64, 128, 576] tensor: q_latent and q_rope are views
    with a row stride of 576 elements (plan fields q_*_row_stride)."""
    inp = cached_workload("unsharded_heads")
    dv = DeviceVerify(inp)
    dv.run()
    torch.cuda.synchronize()
    ref_out, ref_lse = dv.out.clone(), dv.lse.clone()
    q = torch.cat([inp.q_latent, inp.q_rope], dim=-1).cuda().contiguous()   # [64, 128, 576]
    plan = B.ddtree_verify_mla_plan(inp.batch, inp.n_nodes, inp.n_heads, inp.prefix_lens.tolist(),
                                    inp.pool_rows)
    plan.q_latent_row_stride = 576
    plan.q_rope_row_stride = 576
    dv.out.zero_()
    dv.lse.zero_()
    B.ddtree_verify_mla_batched(plan, q[..., :512], q[..., 512:], dv.kv_pool, dv.kv_indices, dv.kv_indptr,
                                dv.prefix_lens, dv.tree_parent, inp.sm_scale, dv.out, dv.lse, dv.workspace)
    torch.cuda.synchronize()
    assert dv.status() == 0
    assert torch.equal(dv.out, ref_out) and torch.equal(dv.lse, ref_lse)
    nodes = [0, 63]
    O_ref, L_ref = oracle_rows(inp, 0, nodes=nodes)
    assert_within_tolerance(dv.out[nodes], dv.lse[nodes], O_ref, L_ref, "strided Q")


@pytest.mark.parametrize("P", [1000, 65536])
def test_expired_wait_reports_timeout_with_finite_outputs(P):
    """A 1 us bound makes the kernels' waits expire: the status word says
    TIMEOUT, the outputs are finite (zeros), and a following call with the
    default bound is correct."""
    T, H = 32, 8
    inp = make_inputs("timeout", batch=1, n_heads=H, prefixes=[P], n_nodes=T, tree="uniform",
                      pool_rows=max(4096, 2 * (P + T)), index_mode="sample", seed=5)
    dv = DeviceVerify(inp)
    assert dv.plan.kernel == B.DDTREE_KERNEL_TC2
    dv.plan.wait_limit_us = 1
    dv.out.fill_(float("nan"))
    dv.lse.fill_(float("nan"))
    dv.run()
    torch.cuda.synchronize()
    assert dv.status() & B.DDTREE_ST_TIMEOUT
    if dv.plan.fused_combine:
        assert torch.isfinite(dv.out.float()).all()
        assert bool((dv.out.float() == 0).all())
    dv.plan.wait_limit_us = 0
    dv.run()
    torch.cuda.synchronize()
    assert dv.status() == 0
    nodes = [0, T - 1]
    O_ref, L_ref = oracle_rows(inp, 0, nodes=nodes)
    assert_within_tolerance(dv.out[nodes], dv.lse[nodes], O_ref, L_ref, "after timeout")
