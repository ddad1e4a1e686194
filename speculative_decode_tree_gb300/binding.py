"""Thin Python binding of the C ABI in include/ddtree_verify.h.

Argument marshalling only: tensors become device pointers, the current torch
stream becomes the cudaStream_t, return codes become exceptions.  Every step
of the verify path runs in the library's CUDA kernels; there is no CPU
fallback, and loading fails loudly when the library has not been built.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_lib", "libddtree_verify.so")

DDTREE_OK = 0
DDTREE_EINVAL = 1
DDTREE_EWORKSPACE = 2
DDTREE_EUNSUPPORTED = 3
DDTREE_ELAUNCH = 4
DDTREE_EDEVICE_DATA = 5
DDTREE_ECUDA = 6

DDTREE_ST_BAD_INDEX = 0x1
DDTREE_ST_BAD_PARENT = 0x2
DDTREE_ST_BAD_LENGTH = 0x4
DDTREE_ST_TIMEOUT = 0x8
DDTREE_ST_OVERLAP = 0x10
DDTREE_ST_BAD_MASK = 0x20

DDTREE_KERNEL_AUTO = 0
DDTREE_KERNEL_SIMT = 1
DDTREE_KERNEL_TC = 2
DDTREE_KERNEL_TC2 = 3

EXPORTS = (
    "ddtree_verify_mla_plan", "ddtree_verify_mla_plan_ex", "ddtree_verify_mla_workspace_size",
    "ddtree_verify_mla", "ddtree_verify_mla_batched", "ddtree_build_ancestor_mask",
    "ddtree_verify_mla_check", "ddtree_status_str", "ddtree_verify_mla_batched_timed",
    "ddtree_verify_mla_noalloc", "ddtree_accept_greedy_workspace_size", "ddtree_accept_greedy",
    "ddtree_relocate_kv_workspace_size", "ddtree_relocate_kv",
    "ddtree_tree_from_mask_workspace_size", "ddtree_tree_from_mask",
)


class Plan(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32), ("n_nodes", ctypes.c_int32), ("n_heads", ctypes.c_int32),
        ("rows_per_req", ctypes.c_int32), ("pool_rows", ctypes.c_int64),
        ("max_keys", ctypes.c_int32), ("kernel", ctypes.c_int32), ("tile_keys", ctypes.c_int32),
        ("chunk_keys", ctypes.c_int32), ("total_splits", ctypes.c_int32),
        ("row_tile", ctypes.c_int32), ("row_tiles", ctypes.c_int32), ("num_sms", ctypes.c_int32),
        ("q_latent_row_stride", ctypes.c_int32), ("q_rope_row_stride", ctypes.c_int32),
        ("workspace_bytes", ctypes.c_int64), ("off_partial_lse", ctypes.c_int64),
        ("off_partial_o", ctypes.c_int64), ("fused_combine", ctypes.c_int32),
        ("wait_limit_us", ctypes.c_int32), ("reserved", ctypes.c_int32 * 6),
    ]

    def as_dict(self) -> dict:
        return {k: getattr(self, k) for k, _ in self._fields_ if k != "reserved"}


class DDTreeError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {code} ({ddtree_status_str(code)})")


_lib = None


def library() -> ctypes.CDLL:
    """Load the in-tree library once; raise if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"CUDA library not built: {LIB_PATH} is missing "
                           "(run speculative_decode_tree_gb300.build.build())")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    P = ctypes.POINTER(Plan)
    L.ddtree_verify_mla_plan.argtypes = [i32, i32, i32, vp, i64, P]
    L.ddtree_verify_mla_plan_ex.argtypes = [i32, i32, i32, vp, i64, i32, i32, P]
    L.ddtree_verify_mla_workspace_size.argtypes = [P]
    L.ddtree_verify_mla_workspace_size.restype = sz
    L.ddtree_verify_mla.argtypes = [vp, vp, vp, vp, i32, vp, i32, i32, f32, vp, vp, vp, vp]
    L.ddtree_verify_mla_batched.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, f32, vp, vp, vp, sz, vp]
    L.ddtree_verify_mla_batched_timed.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, f32, vp, vp, vp, sz,
                                                  vp, vp]
    L.ddtree_build_ancestor_mask.argtypes = [vp, i32, i32, vp, vp, vp]
    L.ddtree_verify_mla_noalloc.argtypes = [vp, vp, vp, vp, i32, vp, i32, i32, f32, vp, vp, vp]
    L.ddtree_verify_mla_check.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_uint32)]
    L.ddtree_status_str.argtypes = [i32]
    L.ddtree_status_str.restype = ctypes.c_char_p
    L.ddtree_accept_greedy_workspace_size.argtypes = [i32, i32]
    L.ddtree_accept_greedy_workspace_size.restype = sz
    L.ddtree_accept_greedy.argtypes = [i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.ddtree_accept_greedy.restype = i32
    L.ddtree_relocate_kv_workspace_size.argtypes = [i64]
    L.ddtree_relocate_kv_workspace_size.restype = sz
    L.ddtree_relocate_kv.argtypes = [i32, i64, vp, i64, vp, vp, vp, vp, vp, sz, vp]
    L.ddtree_relocate_kv.restype = i32
    L.ddtree_tree_from_mask_workspace_size.argtypes = [i32, i32]
    L.ddtree_tree_from_mask_workspace_size.restype = sz
    L.ddtree_tree_from_mask.argtypes = [i32, i32, vp, vp, vp, vp, vp, vp, sz, vp]
    L.ddtree_tree_from_mask.restype = i32
    for name in ("ddtree_verify_mla_plan", "ddtree_verify_mla_plan_ex", "ddtree_verify_mla",
                 "ddtree_verify_mla_batched", "ddtree_build_ancestor_mask", "ddtree_verify_mla_check",
                 "ddtree_verify_mla_batched_timed", "ddtree_verify_mla_noalloc"):
        getattr(L, name).restype = i32
    _lib = L
    return L


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _dev(t: torch.Tensor, dtype: torch.dtype, name: str, numel: Optional[int] = None,
         contiguous: bool = True, device: Optional[int] = None) -> int:
    """Device pointer of `t` after checking what the kernels rely on: a CUDA
    tensor of `dtype` on the current device (`device`, when the caller looked
    it up once for several tensors), contiguous (unless the caller checks its
    layout), holding at least `numel` elements.  The C ABI trusts the sizes it
    derives itself, so an undersized or foreign buffer is rejected here,
    before any launch."""
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    cur = torch.cuda.current_device() if device is None else device
    if t.get_device() != cur:
        raise ValueError(f"{name} is on {t.device}, not the current device cuda:{cur}")
    if contiguous and not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if numel is not None and t.numel() < numel:
        raise ValueError(f"{name} holds {t.numel()} elements, needs at least {numel}")
    return t.data_ptr()


def _q(t: torch.Tensor, name: str, rows: int, width: int, row_stride: int, device: Optional[int] = None) -> int:
    """Pointer of a query operand: `rows` rows of `width` bf16 values whose
    starts are `row_stride` elements apart (width when 0), e.g. views
    q[..., :512] and q[..., 512:] of one [tokens, heads, 576] tensor."""
    stride = row_stride or width
    _dev(t, torch.bfloat16, name, contiguous=False, device=device)
    shape, strides = t.shape, t.stride()
    if len(shape) < 2 or shape[-1] != width or strides[-1] != 1 or t.numel() != rows * width:
        raise ValueError(f"{name} must be [..., {width}] with {rows} rows of unit-stride elements")
    expect = stride
    for d in range(len(shape) - 2, -1, -1):  # every leading dimension steps whole rows
        if shape[d] > 1 and strides[d] != expect:
            raise ValueError(f"{name}: row stride must be {stride} elements (plan q_*_row_stride)")
        expect *= shape[d]
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(rc: int, where: str) -> None:
    if rc != DDTREE_OK:
        raise DDTreeError(rc, where)


def ddtree_status_str(code: int) -> str:
    return library().ddtree_status_str(int(code)).decode()


def ddtree_verify_mla_plan(batch: int, n_nodes: int, n_heads: int, prefix_lens: Sequence[int],
                           pool_rows: int) -> Plan:
    arr = (ctypes.c_int32 * max(len(prefix_lens), 1))(*[int(p) for p in prefix_lens])
    plan = Plan()
    _check(library().ddtree_verify_mla_plan(batch, n_nodes, n_heads, ctypes.cast(arr, ctypes.c_void_p),
                                            int(pool_rows), ctypes.byref(plan)), "plan")
    return plan


def ddtree_verify_mla_plan_ex(batch: int, n_nodes: int, n_heads: int, prefix_lens: Sequence[int],
                              pool_rows: int, num_sms: int, kernel: int = DDTREE_KERNEL_AUTO) -> Plan:
    arr = (ctypes.c_int32 * max(len(prefix_lens), 1))(*[int(p) for p in prefix_lens])
    plan = Plan()
    _check(library().ddtree_verify_mla_plan_ex(batch, n_nodes, n_heads, ctypes.cast(arr, ctypes.c_void_p),
                                               int(pool_rows), int(num_sms), int(kernel),
                                               ctypes.byref(plan)), "plan_ex")
    return plan


def ddtree_verify_mla_workspace_size(plan: Plan) -> int:
    return int(library().ddtree_verify_mla_workspace_size(ctypes.byref(plan)))


def ddtree_verify_mla(q_latent, q_rope, kv_pool, kv_indices, prefix_len: int, tree_parent,
                      n_nodes: int, n_heads: int, sm_scale: float, out, lse, workspace,
                      stream=None) -> None:
    bf, i32 = torch.bfloat16, torch.int32
    lib = library()
    rows = int(n_nodes) * int(n_heads)
    args = (_dev(q_latent, bf, "q_latent", rows * 512), _dev(q_rope, bf, "q_rope", rows * 64),
            _dev(kv_pool, bf, "kv_pool"), _dev(kv_indices, i32, "kv_indices", int(prefix_len) + int(n_nodes)),
            int(prefix_len), _dev(tree_parent, i32, "tree_parent", int(n_nodes)),
            int(n_nodes), int(n_heads), float(sm_scale), _dev(out, bf, "out", rows * 512),
            _dev(lse, torch.float32, "lse", rows))
    # The workspace must hold what the library's own plan for this shape needs.
    plan = ddtree_verify_mla_plan(1, n_nodes, n_heads, [prefix_len], 0)
    rc = lib.ddtree_verify_mla(*args, _dev(workspace, torch.uint8, "workspace", plan.workspace_bytes),
                               _stream(stream))
    _check(rc, "ddtree_verify_mla")


def ddtree_verify_mla_noalloc(q_latent, q_rope, kv_pool, kv_indices, prefix_len: int, tree_parent,
                              n_nodes: int, n_heads: int, sm_scale: float, out, lse,
                              stream=None) -> None:
    """ddtree_verify_mla without a workspace: for callers that cannot allocate
    device memory; the partials use the library's built-in scratch array."""
    bf, i32 = torch.bfloat16, torch.int32
    rows = int(n_nodes) * int(n_heads)
    rc = library().ddtree_verify_mla_noalloc(
        _dev(q_latent, bf, "q_latent", rows * 512), _dev(q_rope, bf, "q_rope", rows * 64),
        _dev(kv_pool, bf, "kv_pool"), _dev(kv_indices, i32, "kv_indices", int(prefix_len) + int(n_nodes)),
        int(prefix_len), _dev(tree_parent, i32, "tree_parent", int(n_nodes)),
        int(n_nodes), int(n_heads), float(sm_scale), _dev(out, bf, "out", rows * 512),
        _dev(lse, torch.float32, "lse", rows), _stream(stream))
    _check(rc, "ddtree_verify_mla_noalloc")


def _batched_args(plan: Plan, q_latent, q_rope, kv_pool, kv_indices, kv_indptr, prefix_lens, tree_parent,
                  sm_scale, out, lse, workspace):
    bf, i32 = torch.bfloat16, torch.int32
    b, t, rows = plan.batch, plan.n_nodes, plan.batch * plan.rows_per_req
    pool_numel = plan.pool_rows * 576 if plan.pool_rows > 0 else None
    ql = _q(q_latent, "q_latent", rows, 512, plan.q_latent_row_stride)  # a CUDA tensor on the current device
    d = q_latent.get_device()  # so the current device, for the call's other tensors
    return (ctypes.byref(plan), ql,
            _q(q_rope, "q_rope", rows, 64, plan.q_rope_row_stride, d),
            _dev(kv_pool, bf, "kv_pool", pool_numel, device=d),
            _dev(kv_indices, i32, "kv_indices", device=d), _dev(kv_indptr, i32, "kv_indptr", b + 1, device=d),
            _dev(prefix_lens, i32, "prefix_lens", b, device=d), _dev(tree_parent, i32, "tree_parent", b * t, device=d),
            float(sm_scale), _dev(out, bf, "out", rows * 512, device=d), _dev(lse, torch.float32, "lse", rows, device=d),
            _dev(workspace, torch.uint8, "workspace", plan.workspace_bytes, device=d), workspace.numel())


def ddtree_verify_mla_batched(plan: Plan, q_latent, q_rope, kv_pool, kv_indices, kv_indptr,
                              prefix_lens, tree_parent, sm_scale: float, out, lse, workspace,
                              stream=None) -> None:
    rc = library().ddtree_verify_mla_batched(
        *_batched_args(plan, q_latent, q_rope, kv_pool, kv_indices, kv_indptr, prefix_lens, tree_parent,
                       sm_scale, out, lse, workspace), _stream(stream))
    _check(rc, "ddtree_verify_mla_batched")


class BoundVerify:
    """ddtree_verify_mla_batched with its arguments checked and marshalled
    once, for callers whose buffers stay the same from call to call (a decode
    loop with static buffers).  Calling the object launches the verify on
    `stream`.  It keeps references to the plan and tensors; they must not be
    resized or moved in place (`resize_`, `set_`) while the object is used."""

    def __init__(self, plan: Plan, q_latent, q_rope, kv_pool, kv_indices, kv_indptr, prefix_lens,
                 tree_parent, sm_scale: float, out, lse, workspace):
        self._keep = (plan, q_latent, q_rope, kv_pool, kv_indices, kv_indptr, prefix_lens, tree_parent,
                      out, lse, workspace)
        self._args = _batched_args(plan, q_latent, q_rope, kv_pool, kv_indices, kv_indptr, prefix_lens,
                                   tree_parent, sm_scale, out, lse, workspace)
        self._fn = library().ddtree_verify_mla_batched

    def __call__(self, stream=None) -> None:
        _check(self._fn(*self._args, _stream(stream)), "ddtree_verify_mla_batched")


def ddtree_verify_mla_batched_timed(plan: Plan, q_latent, q_rope, kv_pool, kv_indices, kv_indptr,
                                    prefix_lens, tree_parent, sm_scale: float, out, lse, workspace,
                                    stage_events, stream=None) -> None:
    """As ddtree_verify_mla_batched, recording three torch.cuda.Event objects
    (before the partial kernel, between partial and combine, after combine)."""
    evs = (ctypes.c_void_p * 3)(*[None if e is None else e.cuda_event for e in stage_events])
    rc = library().ddtree_verify_mla_batched_timed(
        *_batched_args(plan, q_latent, q_rope, kv_pool, kv_indices, kv_indptr, prefix_lens, tree_parent,
                       sm_scale, out, lse, workspace), _stream(stream), ctypes.cast(evs, ctypes.c_void_p))
    _check(rc, "ddtree_verify_mla_batched_timed")


def ddtree_build_ancestor_mask(tree_parent, batch: int, n_nodes: int, anc_out, status=None,
                               stream=None) -> None:
    rc = library().ddtree_build_ancestor_mask(
        _dev(tree_parent, torch.int32, "tree_parent"), int(batch), int(n_nodes),
        _dev(anc_out, torch.int64, "anc_out"),
        None if status is None else _dev(status, torch.int32, "status"), _stream(stream))
    _check(rc, "ddtree_build_ancestor_mask")


def ddtree_verify_mla_check(workspace, stream=None) -> int:
    """Synchronising read of the device status word; returns its DDTREE_ST_* bits."""
    v = ctypes.c_uint32(0)
    rc = library().ddtree_verify_mla_check(_dev(workspace, torch.uint8, "workspace"), _stream(stream),
                                           ctypes.byref(v))
    if rc not in (DDTREE_OK, DDTREE_EDEVICE_DATA):
        raise DDTreeError(rc, "ddtree_verify_mla_check")
    return int(v.value)


def ddtree_accept_greedy_workspace_size(batch: int, n_nodes: int) -> int:
    return int(library().ddtree_accept_greedy_workspace_size(int(batch), int(n_nodes)))


def ddtree_accept_greedy(logits: torch.Tensor, draft_tokens: torch.Tensor, tree_parent: torch.Tensor,
                         kv_indices: torch.Tensor, kv_indptr: torch.Tensor, prefix_lens: torch.Tensor,
                         accept_len: torch.Tensor, next_token: torch.Tensor, accepted_nodes: torch.Tensor,
                         commit_indices: torch.Tensor, freed_indices: torch.Tensor, workspace: torch.Tensor,
                         stream=None) -> None:
    """Greedy acceptance + commit (include/ddtree_accept.h).  logits [B, T+1, V]
    bf16; the int32 outputs are [B] and [B, T]."""
    B, T1, V = logits.shape
    T = T1 - 1
    if not logits.is_contiguous():
        raise ValueError("logits must be contiguous")
    i32 = torch.int32
    _check(library().ddtree_accept_greedy(
        B, T, V, _dev(logits, torch.bfloat16, "logits"), _dev(draft_tokens, i32, "draft_tokens"),
        _dev(tree_parent, i32, "tree_parent"), _dev(kv_indices, i32, "kv_indices"),
        _dev(kv_indptr, i32, "kv_indptr"), _dev(prefix_lens, i32, "prefix_lens"),
        _dev(accept_len, i32, "accept_len"), _dev(next_token, i32, "next_token"),
        _dev(accepted_nodes, i32, "accepted_nodes"), _dev(commit_indices, i32, "commit_indices"),
        _dev(freed_indices, i32, "freed_indices"), _dev(workspace, torch.uint8, "workspace"),
        workspace.numel(), _stream(stream)), "accept_greedy")


def ddtree_relocate_kv_workspace_size(pool_rows: int) -> int:
    return int(library().ddtree_relocate_kv_workspace_size(int(pool_rows)))


def ddtree_relocate_kv(kv_pool: torch.Tensor, kv_indices: torch.Tensor, kv_indptr: torch.Tensor,
                       dest_base: torch.Tensor, total_rows: int, workspace: torch.Tensor,
                       old_indices: Optional[torch.Tensor] = None, stream=None) -> None:
    """Tier-1 relocation (include/ddtree_relocate.h): moves each request's rows
    to [dest_base[b], dest_base[b] + n_b) and rewrites kv_indices in place."""
    i32 = torch.int32
    _check(library().ddtree_relocate_kv(
        int(dest_base.numel()), int(total_rows), _dev(kv_pool, torch.bfloat16, "kv_pool"), int(kv_pool.shape[0]),
        _dev(kv_indices, i32, "kv_indices"), _dev(kv_indptr, i32, "kv_indptr"), _dev(dest_base, i32, "dest_base"),
        None if old_indices is None else _dev(old_indices, i32, "old_indices"),
        _dev(workspace, torch.uint8, "workspace"), workspace.numel(), _stream(stream)), "relocate_kv")


def ddtree_tree_from_mask_workspace_size(batch: int, n_nodes: int) -> int:
    return int(library().ddtree_tree_from_mask_workspace_size(int(batch), int(n_nodes)))


def ddtree_tree_from_mask(custom_mask: torch.Tensor, mask_indptr: torch.Tensor, prefix_lens: torch.Tensor,
                          tree_parent: torch.Tensor, workspace: torch.Tensor,
                          anc_bits: Optional[torch.Tensor] = None, stream=None) -> None:
    """Flattened custom tree mask -> parent array (include/ddtree_mask.h).
    custom_mask uint8 (or bool) flat; tree_parent int32 [B, T] output."""
    m = custom_mask.view(torch.uint8) if custom_mask.dtype == torch.bool else custom_mask
    B_, T = tree_parent.shape
    _check(library().ddtree_tree_from_mask(
        int(B_), int(T), _dev(m, torch.uint8, "custom_mask"), _dev(mask_indptr, torch.int64, "mask_indptr"),
        _dev(prefix_lens, torch.int32, "prefix_lens"), _dev(tree_parent, torch.int32, "tree_parent"),
        None if anc_bits is None else _dev(anc_bits, torch.int64, "anc_bits"),
        _dev(workspace, torch.uint8, "workspace"), workspace.numel(), _stream(stream)), "tree_from_mask")
