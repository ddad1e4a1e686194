"""Helpers shared by the GPU parity tests: oracle evaluation on selected rows
and the tolerance check (|O - O_ref| <= 1e-2 + 1e-2 |O_ref|,
|LSE - LSE_ref| <= 2e-3)."""
from __future__ import annotations

import functools

import torch

from oracle import verify_request
from speculative_decode_tree_gb300.workloads import VerifyInputs, workload

O_ATOL = 1e-2
O_RTOL = 1e-2
LSE_ATOL = 2e-3


def oracle_rows(inp: VerifyInputs, b: int, nodes=None, heads=None):
    T = inp.n_nodes
    lo, hi = int(inp.kv_indptr[b]), int(inp.kv_indptr[b + 1])
    return verify_request(inp.q_latent[b * T:(b + 1) * T], inp.q_rope[b * T:(b + 1) * T],
                          inp.kv_pool, inp.kv_indices[lo:hi], int(inp.prefix_lens[b]),
                          inp.tree_parent[b].tolist(), inp.sm_scale, nodes=nodes, heads=heads)


def assert_within_tolerance(O, L, O_ref, L_ref, what=""):
    O = O.detach().to("cpu", torch.float64)
    L = L.detach().to("cpu", torch.float64)
    assert torch.isfinite(O).all() and torch.isfinite(L).all(), what + ": non-finite output"
    err = (O - O_ref).abs()
    bound = O_ATOL + O_RTOL * O_ref.abs()
    worst = float((err - bound).max())
    assert worst <= 0, f"{what}: O exceeds tolerance by {worst:.3e} (max err {float(err.max()):.3e})"
    lerr = float((L - L_ref).abs().max())
    assert lerr <= LSE_ATOL, f"{what}: LSE error {lerr:.3e}"
    rel_rms = float(((O - O_ref).pow(2).mean() / O_ref.pow(2).mean().clamp_min(1e-30)).sqrt())
    return dict(max_err=float(err.max()), lse_err=lerr, rel_rms=rel_rms)


@functools.lru_cache(maxsize=2)
def cached_workload(name: str) -> VerifyInputs:
    return workload(name)
