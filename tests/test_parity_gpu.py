"""GPU parity: the CUDA path through the C ABI against the float64 oracle on
the same seeded inputs, element by element.  Small shapes compare every
row; the five full-size workloads compare every row where the oracle is
quick and sampled rows elsewhere, in the launch configuration the
benchmark times (the plan the library picks)."""
import pytest
import torch

from oracle import ancestor_bits
from speculative_decode_tree_gb300 import binding as B
from speculative_decode_tree_gb300.runner import DeviceVerify
from speculative_decode_tree_gb300.workloads import make_inputs
from parity_util import assert_within_tolerance, cached_workload, oracle_rows

pytestmark = pytest.mark.gpu

KERNELS = [B.DDTREE_KERNEL_SIMT, B.DDTREE_KERNEL_TC, B.DDTREE_KERNEL_TC2]


def _compare_all(inp, kernel=None, what=""):
    dv = DeviceVerify(inp, kernel=kernel)
    dv.run()
    torch.cuda.synchronize()
    assert dv.status() == 0
    T, H = inp.n_nodes, inp.n_heads
    for b in range(inp.batch):
        O_ref, L_ref = oracle_rows(inp, b)
        assert_within_tolerance(dv.out[b * T:(b + 1) * T], dv.lse[b * T:(b + 1) * T], O_ref, L_ref,
                                f"{what} request {b}")
    return dv


SMALL = [
    # (P, T, H, tree, batch)
    (256, 4, 8, "chain", 1),
    (0, 1, 1, "chain", 1),
    (1, 1, 8, "chain", 1),
    (0, 5, 2, "uniform", 1),
    (37, 16, 8, "uniform", 1),
    (1000, 32, 8, "uniform", 1),
    (4097, 16, 8, "uniform", 1),
    (300, 64, 2, "bounded", 1),
    (129, 3, 128, "uniform", 1),
    (2000, 8, 16, "uniform", 1),
]


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("shape", SMALL, ids=[f"P{s[0]}_T{s[1]}_H{s[2]}_{s[3]}" for s in SMALL])
def test_small_shapes_match_oracle(shape, kernel):
    P, T, H, tree, batch = shape
    inp = make_inputs("small", batch=batch, n_heads=H, prefixes=[P] * batch, n_nodes=T, tree=tree,
                      pool_rows=max(1024, 2 * (P + T)), index_mode="sample", seed=P + 7 * T + H)
    _compare_all(inp, kernel, f"P={P} T={T} H={H}")


def _random_shapes(n: int, seed: int):
    """Seeded draws of (batch, T, H, prefixes, tree, index mode): plans of
    every kind the library picks by default (split counts, fused merge or
    not, one or two row tiles, empty and one-key prefixes)."""
    import random
    r = random.Random(seed)
    shapes = []
    for _ in range(n):
        batch = r.randint(1, 4)
        T = r.choice([1, 3, 8, 16, 31, 32, 48, 64])
        H = r.choice([1, 2, 4, 8, 16])
        while T * H > 512:
            H //= 2
        prefixes = [r.choice([0, 1, r.randint(2, 300), r.randint(300, 4000)]) for _ in range(batch)]
        shapes.append((batch, T, H, prefixes, r.choice(["chain", "uniform", "bounded"]),
                       r.choice(["sample", "interleaved"])))
    return shapes


def _wide_shapes(n: int, seed: int):
    """Seeded draws with many heads and few nodes: three to eight row tiles,
    so the quad kernel runs several row pairs of one split side by side."""
    import random
    r = random.Random(seed)
    shapes = []
    for _ in range(n):
        batch = r.randint(1, 3)
        H = r.choice([32, 64, 128])
        T = r.choice([t for t in (2, 3, 4, 5, 8, 12, 16, 24, 32) if 256 < t * H <= 1024])
        prefixes = [r.choice([0, r.randint(1, 500), r.randint(500, 3000)]) for _ in range(batch)]
        shapes.append((batch, T, H, prefixes, r.choice(["chain", "uniform", "bounded"]),
                       r.choice(["sample", "interleaved"])))
    return shapes


RANDOM = _random_shapes(12, seed=20261203) + _wide_shapes(6, seed=1203) + [
    # longer prefixes: several splits per request, fused merge over many of them
    (2, 16, 8, [20000, 9000], "uniform", "interleaved"),
    (1, 32, 8, [30000], "bounded", "sample"),
]


@pytest.mark.parametrize("kernel", [None, B.DDTREE_KERNEL_TC2], ids=["auto", "tc2"])
@pytest.mark.parametrize("shape", RANDOM, ids=[f"B{s[0]}_T{s[1]}_H{s[2]}_P{sum(s[3])}_{s[4]}_{s[5]}" for s in RANDOM])
def test_random_plans_match_oracle(shape, kernel):
    batch, T, H, prefixes, tree, mode = shape
    pool_rows = max(1024, 2 * sum(p + T for p in prefixes))
    inp = make_inputs("random", batch=batch, n_heads=H, prefixes=prefixes, n_nodes=T, tree=tree,
                      pool_rows=pool_rows, index_mode=mode, seed=batch + 3 * T + 11 * H + sum(prefixes))
    dv = _compare_all(inp, kernel, f"B={batch} T={T} H={H} P={prefixes} {tree} {mode}")
    if kernel is not None:
        assert dv.plan.kernel == kernel


@pytest.mark.parametrize("kernel", KERNELS)
def test_rows_at_both_ends_of_the_pool(kernel):
    """Keys in the pool's first and last rows: four whole tiles of one run that
    ends at the last row (the quad kernel loads such tiles as 2-D TMA boxes),
    then row 0 and the last row again among scattered rows."""
    T, H, P, pool_rows = 16, 8, 1000, 4096
    inp = make_inputs("ends", batch=1, n_heads=H, prefixes=[P], n_nodes=T, tree="uniform",
                      pool_rows=pool_rows, index_mode="sample", seed=77)
    inp.kv_indices[:512] = torch.arange(pool_rows - 512, pool_rows, dtype=torch.int32)
    inp.kv_indices[512] = 0
    inp.kv_indices[700] = pool_rows - 1
    inp.kv_indices[P + T - 1] = pool_rows - 1
    _compare_all(inp, kernel, f"pool ends, kernel {kernel}")


@pytest.mark.parametrize("kernel", KERNELS)
def test_ragged_batch_matches_oracle(kernel):
    prefixes = [0, 5, 777, 64, 1, 2049, 31, 300]
    inp = make_inputs("ragged", batch=8, n_heads=4, prefixes=prefixes, n_nodes=12, tree="uniform",
                      pool_rows=8192, index_mode="interleaved", seed=41)
    _compare_all(inp, kernel, "ragged batch")


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("P", [0, 16, 256, 4096])
def test_spiked_tree_keys_make_the_mask_visible(P, kernel):
    """Tree keys score ~70 nats above prefix keys, so each node's output is
    the mean of V over its ancestors: a wrong mask moves O far past tolerance."""
    T, H = 16, 8
    inp = make_inputs("spiked", batch=1, n_heads=H, prefixes=[P], n_nodes=T, tree="uniform",
                      pool_rows=max(1024, 2 * (P + T)), index_mode="sample", seed=53 + P)
    inp.q_latent.zero_()
    inp.q_rope.zero_()
    inp.q_rope[..., 0] = 8.0
    inp.kv_pool[inp.kv_indices[P:].long(), 512] = 128.0
    dv = _compare_all(inp, kernel, f"spiked P={P}")
    # The mask is visible: dropping one node's deepest ancestor changes O by >= 0.1.
    O_ref, _ = oracle_rows(inp, 0)
    par = inp.tree_parent[0].tolist()
    for i in range(T):
        if par[i] >= 0:
            wrong = list(par)
            wrong[i] = -1
            inp2 = make_inputs("spiked", batch=1, n_heads=H, prefixes=[P], n_nodes=T, tree="uniform",
                               pool_rows=max(1024, 2 * (P + T)), index_mode="sample", seed=53 + P)
            inp2.kv_pool = inp.kv_pool
            inp2.q_latent, inp2.q_rope = inp.q_latent, inp.q_rope
            inp2.tree_parent = torch.tensor([wrong], dtype=torch.int32)
            O_wrong, _ = oracle_rows(inp2, 0)
            assert float((O_wrong[i] - O_ref[i]).abs().max()) >= 0.1
            assert float((dv.out[i].double().cpu() - O_wrong[i]).abs().max()) >= 0.09
            break


@pytest.mark.parametrize("name", ["tiny", "tp8_slice", "long_scattered"])
def test_full_workload_all_rows(name):
    inp = cached_workload(name)
    _compare_all(inp, None, name)


def test_long_contiguous_equals_scattered_bitwise():
    a = DeviceVerify(cached_workload("long_scattered"))
    a.run()
    b = DeviceVerify(cached_workload("long_contiguous"))
    b.run()
    torch.cuda.synchronize()
    assert torch.equal(a.out, b.out) and torch.equal(a.lse, b.lse)
    inp = cached_workload("long_contiguous")
    O_ref, L_ref = oracle_rows(inp, 0, nodes=[0, 31])
    assert_within_tolerance(b.out[[0, 31]], b.lse[[0, 31]], O_ref, L_ref, "long_contiguous")


def test_unsharded_heads_sampled_rows():
    inp = cached_workload("unsharded_heads")
    dv = DeviceVerify(inp)
    dv.run()
    torch.cuda.synchronize()
    assert dv.status() == 0
    par = inp.tree_parent[0].tolist()
    depth = []
    for i, p in enumerate(par):
        depth.append(1 if p < 0 else depth[p] + 1)
    deepest = max(range(len(par)), key=lambda i: depth[i])
    nodes = sorted({0, 1, 31, 63, deepest})
    O_ref, L_ref = oracle_rows(inp, 0, nodes=nodes)
    assert_within_tolerance(dv.out[nodes], dv.lse[nodes], O_ref, L_ref, "unsharded_heads")


def test_mixed_batch_sampled_rows():
    inp = cached_workload("mixed_batch")
    dv = DeviceVerify(inp)
    dv.run()
    torch.cuda.synchronize()
    assert dv.status() == 0
    T = inp.n_nodes
    for b in range(inp.batch):
        nodes = [0, 17, 31]
        O_ref, L_ref = oracle_rows(inp, b, nodes=nodes)
        rows = [b * T + n for n in nodes]
        assert_within_tolerance(dv.out[rows], dv.lse[rows], O_ref, L_ref, f"mixed request {b}")


def test_single_request_entry_point_matches_batched():
    inp = make_inputs("single", batch=1, n_heads=8, prefixes=[3000], n_nodes=16, tree="uniform",
                      pool_rows=8192, index_mode="sample", seed=61)
    dv = DeviceVerify(inp, check_pool=False)
    dv.run()
    o1, l1 = dv.out.clone(), dv.lse.clone()
    dv.out.zero_()
    dv.run_single()
    torch.cuda.synchronize()
    assert torch.equal(o1, dv.out) and torch.equal(l1, dv.lse)


def test_ancestor_mask_stage_bit_exact():
    g = torch.Generator().manual_seed(71)
    B_, T = 5, 64
    par = []
    for b in range(B_):
        par.append([int(torch.randint(-1, i, (1,), generator=g)) for i in range(T)])
    parent = torch.tensor(par, dtype=torch.int32, device="cuda")
    anc = torch.empty(B_ * T, dtype=torch.int64, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.ddtree_build_ancestor_mask(parent, B_, T, anc, status)
    torch.cuda.synchronize()
    got = [v & ((1 << 64) - 1) for v in anc.tolist()]
    want = sum((ancestor_bits(p) for p in par), [])
    assert got == want and int(status) == 0
    parent[1, 7] = 9  # not an earlier node
    B.ddtree_build_ancestor_mask(parent, B_, T, anc, status)
    torch.cuda.synchronize()
    assert int(status) & B.DDTREE_ST_BAD_PARENT


def test_bad_device_data_is_flagged_not_dereferenced():
    inp = make_inputs("bad", batch=1, n_heads=8, prefixes=[500], n_nodes=8, tree="uniform",
                      pool_rows=2048, index_mode="sample", seed=73)
    dv = DeviceVerify(inp)
    dv.kv_indices[3] = inp.pool_rows + 1000
    dv.kv_indices[4] = -5
    dv.run()
    torch.cuda.synchronize()
    assert dv.status() & B.DDTREE_ST_BAD_INDEX
    assert torch.isfinite(dv.out.float()).all()
    dv2 = DeviceVerify(inp)
    dv2.tree_parent[0, 5] = 6
    dv2.run()
    torch.cuda.synchronize()
    assert dv2.status() & B.DDTREE_ST_BAD_PARENT
    dv3 = DeviceVerify(inp)
    dv3.prefix_lens[0] = 500 + dv3.plan.chunk_keys * 3  # longer than planned
    dv3.kv_indptr[1] = 500 + dv3.plan.chunk_keys * 3 + 8
    dv3.run()
    torch.cuda.synchronize()
    assert dv3.status() & B.DDTREE_ST_BAD_LENGTH


def test_graph_capture_and_replay_with_new_inputs_and_shorter_prefix():
    P, T, H = 6000, 16, 8
    inp = make_inputs("graph", batch=1, n_heads=H, prefixes=[P], n_nodes=T, tree="uniform",
                      pool_rows=16384, index_mode="sample", seed=79)
    dv = DeviceVerify(inp)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        dv.run()  # warm-up (sets kernel attributes) outside capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        dv.run()
    # New queries and indices, same shapes.
    inp2 = make_inputs("graph", batch=1, n_heads=H, prefixes=[P], n_nodes=T, tree="uniform",
                       pool_rows=16384, index_mode="sample", seed=83)
    inp2.kv_pool = inp.kv_pool
    dv.q_latent.copy_(inp2.q_latent)
    dv.q_rope.copy_(inp2.q_rope)
    dv.kv_indices.copy_(inp2.kv_indices)
    dv.tree_parent.copy_(inp2.tree_parent)
    g.replay()
    torch.cuda.synchronize()
    O_ref, L_ref = oracle_rows(inp2, 0)
    assert_within_tolerance(dv.out, dv.lse, O_ref, L_ref, "graph replay")
    eager = DeviceVerify(inp2)
    eager.run()
    torch.cuda.synchronize()
    assert torch.equal(eager.out, dv.out) and torch.equal(eager.lse, dv.lse)
    # Shorter prefix on replay: lengths are read on the device.
    P2 = 2500
    idx_short = torch.cat([inp2.kv_indices[:P2], inp2.kv_indices[P:]])
    dv.kv_indices[:P2 + T].copy_(idx_short)
    dv.prefix_lens.fill_(P2)
    dv.kv_indptr[1] = P2 + T
    g.replay()
    torch.cuda.synchronize()
    assert dv.status() == 0
    inp3 = make_inputs("graph", batch=1, n_heads=H, prefixes=[P2], n_nodes=T, tree="uniform",
                       pool_rows=16384, index_mode="sample", seed=83)
    inp3.kv_pool, inp3.q_latent, inp3.q_rope = inp.kv_pool, inp2.q_latent, inp2.q_rope
    inp3.kv_indices, inp3.tree_parent = idx_short.to(torch.int32), inp2.tree_parent
    O_ref3, L_ref3 = oracle_rows(inp3, 0)
    assert_within_tolerance(dv.out, dv.lse, O_ref3, L_ref3, "graph replay, shorter prefix")


@pytest.mark.parametrize("kernel", KERNELS)
def test_graph_replay_batched_with_changing_lengths(kernel):
    """One plan for the longest lengths, captured once; replays with new,
    shorter and unequal prefix lengths, new indices and new trees must match
    eager execution bit for bit and the oracle within tolerance."""
    T, H = 24, 16                                     # 384 rows per request: three row tiles
    plan_prefixes = [3000, 5000, 800]
    base = make_inputs("gb", batch=3, n_heads=H, prefixes=plan_prefixes, n_nodes=T, tree="uniform",
                       pool_rows=32768, index_mode="sample", seed=91)
    dv = DeviceVerify(base, kernel=kernel)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        dv.run()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        dv.run()
    for step, prefixes in enumerate([[100, 4999, 0], [3000, 1, 800], [2048, 2048, 17]]):
        new = make_inputs("gb", batch=3, n_heads=H, prefixes=prefixes, n_nodes=T, tree="bounded",
                          pool_rows=32768, index_mode="sample", seed=92 + step)
        new.kv_pool = base.kv_pool
        n = int(new.kv_indptr[-1])
        dv.q_latent.copy_(new.q_latent)
        dv.q_rope.copy_(new.q_rope)
        dv.kv_indices[:n].copy_(new.kv_indices)
        dv.kv_indptr.copy_(new.kv_indptr)
        dv.prefix_lens.copy_(new.prefix_lens)
        dv.tree_parent.copy_(new.tree_parent)
        g.replay()
        torch.cuda.synchronize()
        assert dv.status() == 0, prefixes
        eager = DeviceVerify(new, kernel=kernel, plan=dv.plan)
        eager.run()
        torch.cuda.synchronize()
        assert torch.equal(eager.out, dv.out) and torch.equal(eager.lse, dv.lse), prefixes
        for b in range(3):
            O_ref, L_ref = oracle_rows(new, b)
            assert_within_tolerance(dv.out[b * T:(b + 1) * T], dv.lse[b * T:(b + 1) * T], O_ref, L_ref,
                                    f"replay {prefixes} request {b}")


def test_bound_call_matches_the_batched_call_and_sees_new_inputs_in_place():
    """BoundVerify marshals its buffers once; each call reads their current
    contents (new queries written in place between calls)."""
    inp = make_inputs("bound", batch=2, n_heads=8, prefixes=[3000, 700], n_nodes=16, tree="uniform",
                      pool_rows=8192, index_mode="interleaved", seed=5)
    dv = DeviceVerify(inp)
    dv.run()
    ref_out, ref_lse = dv.out.clone(), dv.lse.clone()
    out, lse = torch.empty_like(dv.out), torch.empty_like(dv.lse)
    call = B.BoundVerify(dv.plan, dv.q_latent, dv.q_rope, dv.kv_pool, dv.kv_indices, dv.kv_indptr, dv.prefix_lens,
                         dv.tree_parent, inp.sm_scale, out, lse, dv.workspace)
    call()
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)
    # New queries in the same buffers: the bound call computes with them.
    other = make_inputs("bound2", batch=2, n_heads=8, prefixes=[3000, 700], n_nodes=16, tree="uniform",
                        pool_rows=8192, index_mode="interleaved", seed=6)
    dv.q_latent.copy_(other.q_latent)
    dv.q_rope.copy_(other.q_rope)
    call()
    torch.cuda.synchronize()
    assert dv.status() == 0
    from oracle import verify_request
    T = inp.n_nodes
    for b in range(inp.batch):
        lo, hi = int(inp.kv_indptr[b]), int(inp.kv_indptr[b + 1])
        O_ref, L_ref = verify_request(other.q_latent[b * T:(b + 1) * T], other.q_rope[b * T:(b + 1) * T],
                                      inp.kv_pool, inp.kv_indices[lo:hi], int(inp.prefix_lens[b]),
                                      inp.tree_parent[b].tolist(), inp.sm_scale)
        assert_within_tolerance(out[b * T:(b + 1) * T], lse[b * T:(b + 1) * T], O_ref, L_ref, f"bound request {b}")
