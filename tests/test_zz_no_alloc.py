"""The entry point that allocates nothing (ddtree_verify_mla_noalloc).

It exists for callers that cannot call cudaMalloc where they run verify
attention; its partial results live in a scratch array built into the
library instead of a caller-provided workspace.  These checks call it through
the C ABI twice in a row, with different shapes, and compare each result with
the regular workspace entry point under the parity tolerance.  The file is
named to be collected last, so a run that stops at the first failure has
already run every other test.
"""
import pytest
import torch

from speculative_decode_tree_gb300 import binding as B
from speculative_decode_tree_gb300.workloads import make_inputs
from parity_util import assert_within_tolerance

pytestmark = pytest.mark.gpu


def _regular(inp, dev):
    q_l, q_r = inp.q_latent.to(dev), inp.q_rope.to(dev)
    pool, idx, par = inp.kv_pool.to(dev), inp.kv_indices.to(dev), inp.tree_parent.to(dev)
    P = int(inp.prefix_lens[0])
    plan = B.ddtree_verify_mla_plan(1, inp.n_nodes, inp.n_heads, [P], 0)
    ws = torch.empty(B.ddtree_verify_mla_workspace_size(plan), dtype=torch.uint8, device=dev)
    out = torch.empty(inp.n_nodes, inp.n_heads, 512, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(inp.n_nodes, inp.n_heads, dtype=torch.float32, device=dev)
    B.ddtree_verify_mla(q_l, q_r, pool, idx, P, par, inp.n_nodes, inp.n_heads, inp.sm_scale, out, lse, ws)
    return (q_l, q_r, pool, idx, par, P), out, lse


def test_noalloc_matches_workspace_entry_point_twice():
    from speculative_decode_tree_gb300.build import build
    build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    shapes = [
        dict(P=65536, T=32, H=8, tree="uniform", seed=2),   # needs fewer splits to fit the scratch
        dict(P=3000, T=16, H=8, tree="uniform", seed=5),    # smaller shape reusing the same scratch
    ]
    for s in shapes:
        inp = make_inputs("noalloc", batch=1, n_heads=s["H"], prefixes=[s["P"]], n_nodes=s["T"],
                          tree=s["tree"], pool_rows=2 * (s["P"] + s["T"]) + 1024,
                          index_mode="sample", seed=s["seed"])
        (q_l, q_r, pool, idx, par, P), out_ref, lse_ref = _regular(inp, dev)
        out = torch.full_like(out_ref, float("nan"))
        lse = torch.full_like(lse_ref, float("nan"))
        B.ddtree_verify_mla_noalloc(q_l, q_r, pool, idx, P, par, inp.n_nodes, inp.n_heads,
                                    inp.sm_scale, out, lse)
        torch.cuda.synchronize()
        assert_within_tolerance(out, lse, out_ref.double().cpu(), lse_ref.double().cpu(),
                                f"noalloc P={P}")
