"""C-ABI checks that need no GPU: the library loads, exports every entry
point include/ddtree_verify.h declares, plans deterministically, and rejects
bad arguments on the host before touching a device."""
import ctypes
import os
import re

import pytest

from speculative_decode_tree_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"DDTREE_API\s+[\w\s\*]+?\b(ddtree_\w+)\s*\(", text)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    from speculative_decode_tree_gb300.build import build
    build()
    return B.library()


def test_every_declared_symbol_is_exported(lib):
    declared = _declared()
    assert len(declared) >= 8
    for name in declared:
        assert hasattr(lib, name), name
    assert set(B.EXPORTS) <= set(declared)


def test_status_strings(lib):
    for code in range(0, 7):
        assert B.ddtree_status_str(code)
    assert B.ddtree_status_str(99) == "unknown status"


def test_plan_fills_the_sms_and_sizes_the_workspace(lib):
    p = B.ddtree_verify_mla_plan_ex(1, 32, 8, [65536], 262144, 148, B.DDTREE_KERNEL_SIMT)
    assert p.rows_per_req == 256 and p.row_tile == 32 and p.row_tiles == 8
    assert p.chunk_keys % p.tile_keys == 0
    items = p.row_tiles * p.total_splits
    assert items >= 4 * 148 * 0.9
    assert p.total_splits == -(-(65536 + 32) // p.chunk_keys)
    ws = B.ddtree_verify_mla_workspace_size(p)
    assert ws == p.workspace_bytes and ws % 256 == 0
    # status block, fp32 LSE per (split, row), bf16 partial O per (split, row)
    assert ws >= 256 + p.total_splits * 256 * 4 + p.total_splits * 256 * 512 * 2
    # Deterministic.
    q = B.ddtree_verify_mla_plan_ex(1, 32, 8, [65536], 262144, 148, B.DDTREE_KERNEL_SIMT)
    assert p.as_dict() == q.as_dict()


def test_plan_batch_splits_sum_per_request(lib):
    prefixes = [1024, 4096, 8192, 16384, 32768, 65536, 131072, 189440]
    p = B.ddtree_verify_mla_plan_ex(8, 32, 8, prefixes, 524288, 148, B.DDTREE_KERNEL_SIMT)
    assert p.total_splits == sum(-(-(P + 32) // p.chunk_keys) for P in prefixes)
    assert p.max_keys == 189440 + 32


# The five verify workloads' shapes (batch, heads, nodes, prefixes).
WORKLOAD_SHAPES = {
    "tiny": (1, 8, 4, [256]),
    "tp8_slice": (1, 8, 16, [4096]),
    "long_scattered": (1, 8, 32, [65536]),
    "unsharded_heads": (1, 128, 64, [32768]),
    "mixed_batch": (8, 8, 32, [1024, 4096, 8192, 16384, 32768, 65536, 131072, 189440]),
}


@pytest.mark.parametrize("name", sorted(WORKLOAD_SHAPES))
@pytest.mark.parametrize("num_sms", [144, 148, 152])
def test_cluster_plans_fit_one_wave_after_per_request_rounding(lib, name, num_sms):
    """A cluster kernel's work items (row groups x every request's own split
    count) fit the clusters the SMs hold at once, with the shortest such
    chunk: one chunk shorter would need a second wave."""
    b, h, t, prefixes = WORKLOAD_SHAPES[name]
    p = B.ddtree_verify_mla_plan_ex(b, t, h, prefixes, 1 << 20, num_sms)
    if p.kernel == B.DDTREE_KERNEL_SIMT:
        return
    csize = 4 if p.kernel == B.DDTREE_KERNEL_TC2 else 2
    row_groups = (p.row_tiles + 1) // 2 if p.kernel == B.DDTREE_KERNEL_TC2 else p.row_tiles
    capacity = num_sms // csize

    def items(chunk):
        return row_groups * sum(-(-(P + t) // chunk) for P in prefixes)

    assert p.total_splits == sum(-(-(P + t) // p.chunk_keys) for P in prefixes)
    assert p.chunk_keys % p.tile_keys == 0
    if row_groups * b <= capacity:
        assert items(p.chunk_keys) <= capacity
        if p.chunk_keys > p.tile_keys:
            assert items(p.chunk_keys - p.tile_keys) > capacity
    else:
        assert p.chunk_keys >= max(prefixes) + t
    assert p.fused_combine == 0  # explicit SM counts never fuse (no residency guarantee known)


@pytest.mark.parametrize("args", [
    (0, 4, 8), (1, 0, 8), (1, 65, 8), (1, 4, 0), (1, 4, 129), (1025, 4, 8),
])
def test_plan_rejects_bad_sizes(lib, args):
    b, t, h = args
    with pytest.raises(B.DDTreeError) as e:
        B.ddtree_verify_mla_plan_ex(b, t, h, [16] * max(b, 1), 1024, 148)
    assert e.value.code == B.DDTREE_EINVAL


def test_plan_rejects_negative_prefix(lib):
    with pytest.raises(B.DDTreeError):
        B.ddtree_verify_mla_plan_ex(2, 4, 8, [16, -1], 1024, 148)


def test_null_pointers_rejected_before_device_use(lib):
    p = B.ddtree_verify_mla_plan_ex(1, 4, 8, [256], 1024, 148)
    rc = lib.ddtree_verify_mla_batched(ctypes.byref(p), None, None, None, None, None, None, None,
                                       0.1, None, None, None, 0, None)
    assert rc == B.DDTREE_EINVAL


def test_tampered_plan_rejected(lib):
    p = B.ddtree_verify_mla_plan_ex(1, 4, 8, [256], 1024, 148)
    p.workspace_bytes -= 256
    fake = ctypes.c_void_p(256)  # never dereferenced: validation fails first
    rc = lib.ddtree_verify_mla_batched(ctypes.byref(p), fake, fake, fake, fake, fake, fake, fake,
                                       0.1, fake, fake, fake, 1 << 20, None)
    assert rc == B.DDTREE_EINVAL


def test_misaligned_pointer_rejected(lib):
    p = B.ddtree_verify_mla_plan_ex(1, 4, 8, [256], 1024, 148)
    ok = ctypes.c_void_p(1 << 12)
    bad = ctypes.c_void_p((1 << 12) + 8)
    rc = lib.ddtree_verify_mla_batched(ctypes.byref(p), bad, ok, ok, ok, ok, ok, ok,
                                       0.1, ok, ok, ok, 1 << 30, None)
    assert rc == B.DDTREE_EINVAL


def test_small_workspace_rejected(lib):
    p = B.ddtree_verify_mla_plan_ex(1, 4, 8, [256], 1024, 148)
    ok = ctypes.c_void_p(1 << 12)
    rc = lib.ddtree_verify_mla_batched(ctypes.byref(p), ok, ok, ok, ok, ok, ok, ok,
                                       0.1, ok, ok, ok, p.workspace_bytes - 1, None)
    assert rc == B.DDTREE_EWORKSPACE


def test_nonfinite_scale_rejected(lib):
    p = B.ddtree_verify_mla_plan_ex(1, 4, 8, [256], 1024, 148)
    ok = ctypes.c_void_p(1 << 12)
    rc = lib.ddtree_verify_mla_batched(ctypes.byref(p), ok, ok, ok, ok, ok, ok, ok,
                                       float("nan"), ok, ok, ok, 1 << 30, None)
    assert rc == B.DDTREE_EINVAL


def test_no_device_reports_unsupported(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    p = B.Plan()
    arr = (ctypes.c_int32 * 1)(256)
    rc = lib.ddtree_verify_mla_plan(1, 4, 8, ctypes.cast(arr, ctypes.c_void_p), 1024, ctypes.byref(p))
    assert rc == B.DDTREE_EUNSUPPORTED


def test_accept_workspace_size(lib):
    # status block + keys (8 B per scored row) + counters (4 B per request), each rounded to 256
    assert B.ddtree_accept_greedy_workspace_size(1, 32) == 256 + 512 + 256
    assert B.ddtree_accept_greedy_workspace_size(8, 64) == 256 + 4352 + 256
    for bad in [(0, 4), (1, 0), (1, 65), (1025, 4)]:
        assert B.ddtree_accept_greedy_workspace_size(*bad) == 0


# The five verify workloads' shapes (batch, heads, nodes, prefixes).
WORKLOAD_SHAPES = {
    "tiny": (1, 8, 4, [256]),
    "tp8_slice": (1, 8, 16, [4096]),
    "long_scattered": (1, 8, 32, [65536]),
    "unsharded_heads": (1, 128, 64, [32768]),
    "mixed_batch": (8, 8, 32, [1024, 4096, 8192, 16384, 32768, 65536, 131072, 189440]),
}


@pytest.mark.parametrize("name", sorted(WORKLOAD_SHAPES))
@pytest.mark.parametrize("num_sms", [144, 148, 152])
def test_cluster_plans_fit_one_wave_after_per_request_rounding(lib, name, num_sms):
    """A cluster kernel's work items (row groups x every request's own split
    count) fit the clusters the SMs hold at once, with the shortest such
    chunk: one chunk shorter would need a second wave."""
    b, h, t, prefixes = WORKLOAD_SHAPES[name]
    p = B.ddtree_verify_mla_plan_ex(b, t, h, prefixes, 1 << 20, num_sms)
    if p.kernel == B.DDTREE_KERNEL_SIMT:
        return
    csize = 4 if p.kernel == B.DDTREE_KERNEL_TC2 else 2
    row_groups = (p.row_tiles + 1) // 2 if p.kernel == B.DDTREE_KERNEL_TC2 else p.row_tiles
    capacity = num_sms // csize

    def items(chunk):
        return row_groups * sum(-(-(P + t) // chunk) for P in prefixes)

    assert p.total_splits == sum(-(-(P + t) // p.chunk_keys) for P in prefixes)
    assert p.chunk_keys % p.tile_keys == 0
    if row_groups * b <= capacity:
        assert items(p.chunk_keys) <= capacity
        if p.chunk_keys > p.tile_keys:
            assert items(p.chunk_keys - p.tile_keys) > capacity
    else:
        assert p.chunk_keys >= max(prefixes) + t
    assert p.fused_combine == 0  # explicit SM counts never fuse (no residency guarantee known)


@pytest.mark.parametrize("args", [(0, 4, 100), (1, 0, 100), (1, 65, 100), (1, 4, 0), (1, 4, (1 << 26) + 1)])
def test_accept_rejects_bad_sizes(lib, args):
    buf = ctypes.create_string_buffer(4096)
    p = ctypes.cast(ctypes.addressof(buf) + (-ctypes.addressof(buf)) % 256, ctypes.c_void_p)
    rc = lib.ddtree_accept_greedy(*args, *([p] * 12), 4096 - 256, None)
    assert rc == B.DDTREE_EINVAL


def test_accept_rejects_null_and_small_workspace(lib):
    buf = ctypes.create_string_buffer(4096)
    p = ctypes.cast(ctypes.addressof(buf) + (-ctypes.addressof(buf)) % 256, ctypes.c_void_p)
    ptrs = [p] * 12
    assert lib.ddtree_accept_greedy(1, 4, 100, None, *ptrs[1:], 1024, None) == B.DDTREE_EINVAL
    rc = lib.ddtree_accept_greedy(1, 4, 100, *ptrs, 16, None)
    assert rc == B.DDTREE_EWORKSPACE


def test_relocate_workspace_size(lib):
    assert B.ddtree_relocate_kv_workspace_size(1) == 256 + 256
    assert B.ddtree_relocate_kv_workspace_size(262144) == 256 + 32768        # one bit per row
    assert B.ddtree_relocate_kv_workspace_size(0) == 0
    assert B.ddtree_relocate_kv_workspace_size(1 << 31) == 0


def test_relocate_rejects_bad_arguments(lib):
    buf = ctypes.create_string_buffer(8192)
    p = ctypes.cast(ctypes.addressof(buf) + (-ctypes.addressof(buf)) % 256, ctypes.c_void_p)
    ok = dict(batch=1, total=4, pool=p, rows=100, idx=p, ptr=p, dst=p, old=None, ws=p, wsb=4096)

    def call(**kw):
        a = dict(ok, **kw)
        return lib.ddtree_relocate_kv(a["batch"], a["total"], a["pool"], a["rows"], a["idx"], a["ptr"],
                                      a["dst"], a["old"], a["ws"], a["wsb"], None)
    assert call(batch=0) == B.DDTREE_EINVAL
    assert call(rows=0) == B.DDTREE_EINVAL
    assert call(total=101) == B.DDTREE_EINVAL
    assert call(pool=None) == B.DDTREE_EINVAL
    assert call(ptr=ctypes.c_void_p(p.value + 2)) == B.DDTREE_EINVAL
    assert call(wsb=16) == B.DDTREE_EWORKSPACE


def test_mask_reader_workspace_and_rejections(lib):
    assert B.ddtree_tree_from_mask_workspace_size(1, 32) == 256 + 256 + 256
    assert B.ddtree_tree_from_mask_workspace_size(0, 4) == 0
    assert B.ddtree_tree_from_mask_workspace_size(1, 65) == 0
    buf = ctypes.create_string_buffer(4096)
    p = ctypes.cast(ctypes.addressof(buf) + (-ctypes.addressof(buf)) % 256, ctypes.c_void_p)
    assert lib.ddtree_tree_from_mask(0, 4, p, p, p, p, None, p, 2048, None) == B.DDTREE_EINVAL
    assert lib.ddtree_tree_from_mask(1, 4, None, p, p, p, None, p, 2048, None) == B.DDTREE_EINVAL
    assert lib.ddtree_tree_from_mask(1, 4, p, ctypes.c_void_p(p.value + 4), p, p, None, p, 2048, None) == B.DDTREE_EINVAL
    assert lib.ddtree_tree_from_mask(1, 4, p, p, p, p, None, p, 16, None) == B.DDTREE_EWORKSPACE
