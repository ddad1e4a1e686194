"""The entry point that allocates nothing (ddtree_verify_mla_noalloc).

It exists for callers that cannot call cudaMalloc where they run verify
attention; its partial results live in a fixed scratch array built into the
library (DDTREE_NOALLOC_SCRATCH_BYTES) instead of a caller-provided workspace.
These checks call it through the C ABI on two shapes in a row and compare
each result with the float64 oracle under the parity tolerance:

  * the 65,536-key prefix shape, whose usual plan needs more partial storage
    than the scratch holds, so the call runs fewer, longer splits;
  * a 3,000-key prefix, reusing the same scratch right after.

A shape whose partials cannot fit even with one split is rejected with
DDTREE_EWORKSPACE before anything is launched.  The file is named to be
collected last, so a run that stops at the first failure has already run
every other test; it also passes alone in a fresh process.
"""
import pytest
import torch

from speculative_decode_tree_gb300 import binding as B
from speculative_decode_tree_gb300.workloads import make_inputs
from parity_util import assert_within_tolerance, oracle_rows

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 8 << 20  # DDTREE_NOALLOC_SCRATCH_BYTES in include/ddtree_verify.h


def _device_inputs(inp, dev):
    return (inp.q_latent.to(dev), inp.q_rope.to(dev), inp.kv_pool.to(dev), inp.kv_indices.to(dev),
            inp.tree_parent.to(dev))


def test_noalloc_matches_the_oracle_twice_and_shrinks_its_splits():
    from speculative_decode_tree_gb300.build import build
    build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    shapes = [
        dict(P=65536, T=32, H=8, seed=2, shrinks=True),    # usual plan's partials exceed the scratch
        dict(P=3000, T=16, H=8, seed=5, shrinks=False),    # fits as planned; reuses the same scratch
    ]
    for s in shapes:
        inp = make_inputs("noalloc", batch=1, n_heads=s["H"], prefixes=[s["P"]], n_nodes=s["T"],
                          tree="uniform", pool_rows=2 * (s["P"] + s["T"]) + 1024,
                          index_mode="sample", seed=s["seed"])
        plan = B.ddtree_verify_mla_plan(1, inp.n_nodes, inp.n_heads, [s["P"]], 0)
        assert (plan.workspace_bytes > SCRATCH_BYTES) == s["shrinks"], plan.workspace_bytes
        q_l, q_r, pool, idx, par = _device_inputs(inp, dev)
        out = torch.full((inp.n_nodes, inp.n_heads, 512), float("nan"), dtype=torch.bfloat16, device=dev)
        lse = torch.full((inp.n_nodes, inp.n_heads), float("nan"), dtype=torch.float32, device=dev)
        B.ddtree_verify_mla_noalloc(q_l, q_r, pool, idx, s["P"], par, inp.n_nodes, inp.n_heads,
                                    inp.sm_scale, out, lse)
        torch.cuda.synchronize()
        O_ref, L_ref = oracle_rows(inp, 0)
        assert_within_tolerance(out, lse, O_ref, L_ref, f"noalloc P={s['P']}")


def test_noalloc_rejects_a_shape_beyond_the_scratch():
    dev = torch.device("cuda", 0)
    T, H, P = 64, 128, 1000       # 8,192 query rows: one split's partials alone exceed the scratch
    inp = make_inputs("noalloc_big", batch=1, n_heads=H, prefixes=[P], n_nodes=T, tree="bounded",
                      pool_rows=4096, index_mode="sample", seed=9)
    q_l, q_r, pool, idx, par = _device_inputs(inp, dev)
    out = torch.zeros(T, H, 512, dtype=torch.bfloat16, device=dev)
    lse = torch.zeros(T, H, dtype=torch.float32, device=dev)
    with pytest.raises(B.DDTreeError) as e:
        B.ddtree_verify_mla_noalloc(q_l, q_r, pool, idx, P, par, T, H, inp.sm_scale, out, lse)
    assert e.value.code == B.DDTREE_EWORKSPACE
