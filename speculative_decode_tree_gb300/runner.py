"""Device buffers for one verify batch, driven through the C ABI.

Holds the inputs on the GPU, the plan, the caller-owned workspace and the
outputs, and calls the batched entry point.  Plumbing only: all compute runs
in the library's kernels.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import binding as B
from .workloads import VerifyInputs


class DeviceVerify:
    def __init__(self, inp: VerifyInputs, device: str = "cuda", kernel: Optional[int] = None,
                 check_pool: bool = True, plan: Optional[B.Plan] = None):
        dev = torch.device(device)
        self.inp = inp
        self.kv_pool = inp.kv_pool.to(dev)
        self.kv_indices = inp.kv_indices.to(dev)
        self.kv_indptr = inp.kv_indptr.to(dev)
        self.prefix_lens = inp.prefix_lens.to(dev)
        self.tree_parent = inp.tree_parent.to(dev).contiguous()
        self.q_latent = inp.q_latent.to(dev)
        self.q_rope = inp.q_rope.to(dev)
        pool_rows = inp.pool_rows if check_pool else 0
        if plan is not None:
            self.plan = plan
        elif kernel is None:
            self.plan = B.ddtree_verify_mla_plan(inp.batch, inp.n_nodes, inp.n_heads,
                                                 inp.prefix_lens.tolist(), pool_rows)
        else:
            self.plan = B.ddtree_verify_mla_plan_ex(inp.batch, inp.n_nodes, inp.n_heads,
                                                    inp.prefix_lens.tolist(), pool_rows, 0, kernel)
        rows = inp.batch * inp.n_nodes
        self.out = torch.empty(rows, inp.n_heads, 512, dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty(rows, inp.n_heads, dtype=torch.float32, device=dev)
        self.workspace = torch.empty(B.ddtree_verify_mla_workspace_size(self.plan),
                                     dtype=torch.uint8, device=dev)

    def run(self, stream=None) -> None:
        B.ddtree_verify_mla_batched(self.plan, self.q_latent, self.q_rope, self.kv_pool,
                                    self.kv_indices, self.kv_indptr, self.prefix_lens,
                                    self.tree_parent, self.inp.sm_scale, self.out, self.lse,
                                    self.workspace, stream)

    def run_timed(self, stage_events, stream=None) -> None:
        B.ddtree_verify_mla_batched_timed(self.plan, self.q_latent, self.q_rope, self.kv_pool,
                                          self.kv_indices, self.kv_indptr, self.prefix_lens,
                                          self.tree_parent, self.inp.sm_scale, self.out, self.lse,
                                          self.workspace, stage_events, stream)

    def run_single(self, stream=None) -> None:
        """The single-request entry point (batch 1)."""
        assert self.inp.batch == 1
        B.ddtree_verify_mla(self.q_latent, self.q_rope, self.kv_pool, self.kv_indices,
                            int(self.inp.prefix_lens[0]), self.tree_parent, self.inp.n_nodes,
                            self.inp.n_heads, self.inp.sm_scale, self.out, self.lse,
                            self.workspace, stream)

    def status(self, stream=None) -> int:
        return B.ddtree_verify_mla_check(self.workspace, stream)


class DeviceAccept:
    """Device copies of an acceptance workload and its output buffers."""

    def __init__(self, inp, device: str = "cuda"):
        dev = torch.device(device)
        self.inp = inp
        self.logits = inp.logits.to(dev).contiguous()
        self.draft = inp.draft_tokens.to(dev).contiguous()
        self.parent = inp.tree_parent.to(dev).contiguous()
        self.kv_indices = inp.kv_indices.to(dev)
        self.kv_indptr = inp.kv_indptr.to(dev)
        self.prefix_lens = inp.prefix_lens.to(dev)
        nb, nt = inp.batch, inp.n_nodes
        i32 = torch.int32
        self.accept_len = torch.empty(nb, dtype=i32, device=dev)
        self.next_token = torch.empty(nb, dtype=i32, device=dev)
        self.accepted_nodes = torch.empty(nb, nt, dtype=i32, device=dev)
        self.commit_indices = torch.empty(nb, nt, dtype=i32, device=dev)
        self.freed_indices = torch.empty(nb, nt, dtype=i32, device=dev)
        self.workspace = torch.empty(B.ddtree_accept_greedy_workspace_size(nb, nt), dtype=torch.uint8,
                                     device=dev)

    def run(self, stream=None) -> None:
        B.ddtree_accept_greedy(self.logits, self.draft, self.parent, self.kv_indices, self.kv_indptr,
                               self.prefix_lens, self.accept_len, self.next_token, self.accepted_nodes,
                               self.commit_indices, self.freed_indices, self.workspace, stream)

    def status(self, stream=None) -> int:
        return B.ddtree_verify_mla_check(self.workspace, stream)

    def outputs(self) -> dict:
        return {"accept_len": self.accept_len.cpu().numpy(), "next_token": self.next_token.cpu().numpy(),
                "accepted_nodes": self.accepted_nodes.cpu().numpy(),
                "commit_indices": self.commit_indices.cpu().numpy(),
                "freed_indices": self.freed_indices.cpu().numpy()}

