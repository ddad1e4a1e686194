"""The product path has no CPU fallback: without the compiled library, or when
handed host tensors, the entry points raise instead of computing anything."""
import pytest
import torch

from speculative_decode_tree_gb300 import binding as B
from speculative_decode_tree_gb300.workloads import make_inputs


def test_missing_library_raises(monkeypatch, tmp_path):
    monkeypatch.setattr(B, "LIB_PATH", str(tmp_path / "absent.so"))
    monkeypatch.setattr(B, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        B.library()
    inp = make_inputs("t", batch=1, n_heads=2, prefixes=[16], n_nodes=2, tree="chain", pool_rows=64,
                      index_mode="permutation", seed=0)
    with pytest.raises(RuntimeError, match="not built"):
        B.ddtree_verify_mla(inp.q_latent, inp.q_rope, inp.kv_pool, inp.kv_indices, 16, inp.tree_parent[0],
                            2, 2, inp.sm_scale, torch.empty(2, 2, 512, dtype=torch.bfloat16),
                            torch.empty(2, 2), torch.empty(1 << 20, dtype=torch.uint8))


def test_host_tensors_are_rejected_before_any_call():
    # The library is present (built by the ABI tests' fixture or here); the
    # wrapper must still refuse host memory rather than copy or compute.
    from speculative_decode_tree_gb300.build import build
    build()
    inp = make_inputs("t", batch=1, n_heads=2, prefixes=[16], n_nodes=2, tree="chain", pool_rows=64,
                      index_mode="permutation", seed=0)
    with pytest.raises(TypeError, match="must be a CUDA tensor"):
        B.ddtree_verify_mla(inp.q_latent, inp.q_rope, inp.kv_pool, inp.kv_indices, 16, inp.tree_parent[0],
                            2, 2, inp.sm_scale, torch.empty(2, 2, 512, dtype=torch.bfloat16),
                            torch.empty(2, 2), torch.empty(1 << 20, dtype=torch.uint8))
    with pytest.raises(TypeError, match="must be a CUDA tensor"):
        B.ddtree_verify_mla_noalloc(inp.q_latent, inp.q_rope, inp.kv_pool, inp.kv_indices, 16,
                                    inp.tree_parent[0], 2, 2, inp.sm_scale,
                                    torch.empty(2, 2, 512, dtype=torch.bfloat16), torch.empty(2, 2))


def test_batched_and_bound_calls_reject_host_tensors():
    # The batched wrapper and the bound call check their tensors before
    # anything else (no device lookup first, no copy, no compute).
    from speculative_decode_tree_gb300.build import build
    build()
    inp = make_inputs("t", batch=1, n_heads=2, prefixes=[16], n_nodes=2, tree="chain", pool_rows=64,
                      index_mode="permutation", seed=0)
    plan = B.Plan()
    plan.batch, plan.n_nodes, plan.n_heads, plan.rows_per_req = 1, 2, 2, 4
    args = (plan, inp.q_latent, inp.q_rope, inp.kv_pool, inp.kv_indices, inp.kv_indptr, inp.prefix_lens,
            inp.tree_parent, inp.sm_scale, torch.empty(2, 2, 512, dtype=torch.bfloat16), torch.empty(2, 2),
            torch.empty(1 << 20, dtype=torch.uint8))
    with pytest.raises(TypeError, match="must be a CUDA tensor"):
        B.ddtree_verify_mla_batched(*args)
    with pytest.raises(TypeError, match="must be a CUDA tensor"):
        B.BoundVerify(*args)
