"""GB300 fused linear cross-entropy (FLCE): Python binding of libflce.so.

The loss of a language-model head, mean over non-ignored rows of
CE(softcap(m * h W^T), label), with token accuracy, predicted tokens, grad_h
and an fp32 grad_W accumulator, computed by hand-written sm_103a kernels
without keeping the [tokens, vocab] logits (Liger-Kernel, "Muse Glimmer"
support, Summary and Details / Softcap; DeepSeek-V3 support, Summary and
Memory; SpecForge DSpine PR, Changes: flattened frozen projection and the
CE-only prepass).

This module only marshals arguments: it checks dtypes and devices, flattens
leading row dimensions ([B, k, S, H] -> [N, H], the DSpine page's flattened
proposal rows), allocates outputs and a cached workspace with torch, and calls
the C ABI on torch's current CUDA stream. Every step of the computation runs
in the library's kernels; CPU tensors are rejected, there is no fallback.
"""
from __future__ import annotations

import ctypes
from typing import Optional

import torch

from . import _lib
from ._lib import (FLCE_FLAG_KMAJOR_BWD, FLCE_FLAG_RECOMPUTE, FLCE_FLAG_SIMT_GEMM, FLCE_FLAG_TEST_STALL,  # noqa: F401
                   FLCE_FLAG_TILE128, FLCE_FLAG_TILE256, FLCE_FLAG_CTA_PAIR, FLCE_FLAG_F32_3PASS, FLCE_FLAG_VP_STORED,
                   FLCE_MODE_CE_ONLY, FLCE_MODE_FORWARD,
                   FLCE_MODE_FORWARD_BACKWARD, FLCE_REDUCTION_MEAN, FLCE_REDUCTION_SUM, FlceError, FlceParams)

__all__ = [
    "flce_ce_only", "flce_ce_only_noalloc", "flce_forward", "flce_forward_backward",
    "flce_forward_backward_from_host", "flce_ce_only_from_host", "flce_cross_entropy",
    "flce_scale_gradient", "flce_workspace_size", "flce_chunk_rows", "flce_chunk_rows_for_budget", "flce_release_workspaces", "flce_get_status", "flce_launch_count",
    "flce_profile_begin",
    "flce_profile_read", "linear_cross_entropy", "FusedLinearCrossEntropyLoss", "FlceError",
    "flce_vp_forward", "flce_vp_backward", "flce_vp_workspace", "vocab_parallel_linear_cross_entropy", "vp_shard_table",
    "vp_gather_partials", "vp_reduce_grad_h",
]

_REDUCTIONS = {"mean": FLCE_REDUCTION_MEAN, "sum": FLCE_REDUCTION_SUM, "none": _lib.FLCE_REDUCTION_NONE}
_workspaces: dict = {}


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(device: torch.device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _params(n_rows: int, hidden: int, vocab: int, ld_h: int, ld_w: int, softcap: float, out_mult: float,
            ignore_index: int, reduction: str, grad_scale: float, chunk_rows: int, flags: int,
            timeout_ns: int, vocab_slab: int = 0, dtype: int = 0) -> FlceParams:
    if reduction not in _REDUCTIONS:
        raise ValueError(f"reduction must be one of {sorted(_REDUCTIONS)}")
    p = FlceParams()
    _lib.lib().flce_default_params(ctypes.byref(p))
    p.n_rows, p.hidden, p.vocab = n_rows, hidden, vocab
    p.ld_h, p.ld_w = ld_h, ld_w
    p.softcap, p.out_mult = float(softcap), float(out_mult)
    p.ignore_index = int(ignore_index)
    p.reduction = _REDUCTIONS[reduction]
    p.grad_scale = float(grad_scale)
    p.chunk_rows = int(chunk_rows)
    p.flags = int(flags)
    p.timeout_ns = int(timeout_ns)
    p.vocab_slab = int(vocab_slab)
    p.dtype = int(dtype)
    return p


def _rows2d(h: torch.Tensor, H: int) -> torch.Tensor:
    h2 = h.reshape(-1, H)
    if h2.stride(1) != 1 or h2.stride(0) % 8 != 0 or h2.data_ptr() % 16 != 0:
        h2 = h2.contiguous()
    return h2


def _dtype_code(t: torch.Tensor) -> int:
    return _lib.FLCE_DTYPE_F32 if t.dtype == torch.float32 else _lib.FLCE_DTYPE_BF16


def _check(h: torch.Tensor, W: torch.Tensor, labels: torch.Tensor):
    for name, t in (("h", h), ("W", W), ("labels", labels)):
        if not isinstance(t, torch.Tensor) or t.device.type != "cuda":
            raise ValueError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    if h.dtype not in (torch.bfloat16, torch.float32) or W.dtype != h.dtype:
        raise ValueError("h and W must both be bfloat16, or both float32 (tf32 tensor-core path)")
    if labels.dtype != torch.int64:
        raise ValueError("labels must be int64")
    if W.dim() != 2 or h.shape[-1] != W.shape[1]:
        raise ValueError("W must be [V, H] and h [..., H]")
    if labels.shape != h.shape[:-1]:
        raise ValueError("labels must have h's leading shape")
    if h.device != W.device or h.device != labels.device:
        raise ValueError("h, W and labels must be on one device")


def _workspace(device: torch.device, nbytes: int) -> torch.Tensor:
    """The cached workspace of (device, current stream): calls on one stream
    reuse it in stream order; calls on different streams never share one."""
    dev = device.index if device.index is not None else torch.cuda.current_device()
    key = (dev, torch.cuda.current_stream(dev).cuda_stream)
    ws = _workspaces.get(key)
    if ws is None or ws.numel() < nbytes:
        _workspaces.pop(key, None)
        ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
        _workspaces[key] = ws
    return ws


def flce_chunk_rows_for_budget(n_rows: int, hidden: int, vocab: int, budget_bytes: int, *,
                               mode: int = FLCE_MODE_FORWARD_BACKWARD, need_grad_h: bool = True,
                               need_grad_W: bool = True, flags: int = 0, dtype=torch.bfloat16) -> int:
    """The largest chunk (a multiple of 128 rows, at most 32768) whose workspace
    fits in budget_bytes, from flce_workspace_size; 0 if not even 128 rows fit
    (then the recompute backward, FLCE_FLAG_RECOMPUTE, needs far less)."""
    best, lo, hi = 0, 1, 32768 // 128
    code = _lib.FLCE_DTYPE_F32 if dtype == torch.float32 else _lib.FLCE_DTYPE_BF16
    while lo <= hi:                      # the workspace grows with the chunk
        mid = (lo + hi) // 2
        p = _params(n_rows, hidden, vocab, 0, 0, 0.0, 1.0, -100, "mean", 1.0, mid * 128, flags, 0, 0, code)
        need = int(_lib.lib().flce_workspace_size(ctypes.byref(p), mode, int(need_grad_h), int(need_grad_W)))
        if 0 < need <= budget_bytes:
            best, lo = mid * 128, mid + 1
        else:
            hi = mid - 1
    return best


def flce_release_workspaces() -> None:
    """Drops the cached workspaces (one per device and stream, grown to the
    largest call so far); torch's allocator then holds the memory for reuse.
    Call it after the last use on a stream, not while a call may still run."""
    _workspaces.clear()


def _native(device: torch.device, name: str, *args):
    """Calls a C entry point with `device` current. The library takes the SM
    count, its per-device setup and the static scratch array from the current
    device, so it must be the device that owns the tensors and the stream."""
    with torch.cuda.device(device):
        return getattr(_lib.lib(), name)(*args)


def _raise(rc: int, what: str):
    if rc != 0:
        raise FlceError(rc, what)


def flce_workspace_size(n_rows: int, hidden: int, vocab: int, mode: int = FLCE_MODE_FORWARD_BACKWARD,
                        need_grad_h: bool = True, need_grad_W: bool = True, chunk_rows: int = 0,
                        flags: int = 0, dtype=torch.bfloat16) -> int:
    """Bytes of device workspace a call with these arguments needs (dtype: of h and W)."""
    p = _params(n_rows, hidden, vocab, 0, 0, 0.0, 1.0, -100, "mean", 1.0, chunk_rows, flags, 0, 0,
                _lib.FLCE_DTYPE_F32 if dtype == torch.float32 else _lib.FLCE_DTYPE_BF16)
    return int(_lib.lib().flce_workspace_size(ctypes.byref(p), mode, int(need_grad_h), int(need_grad_W)))


def flce_chunk_rows(n_rows: int, hidden: int, vocab: int, mode: int = FLCE_MODE_FORWARD_BACKWARD,
                    need_grad_h: bool = True, need_grad_W: bool = True, chunk_rows: int = 0,
                    flags: int = 0, dtype=torch.bfloat16) -> int:
    """Rows per chunk a call with these arguments uses (the library's choice when chunk_rows is 0)."""
    p = _params(n_rows, hidden, vocab, 0, 0, 0.0, 1.0, -100, "mean", 1.0, chunk_rows, flags, 0, 0,
                _lib.FLCE_DTYPE_F32 if dtype == torch.float32 else _lib.FLCE_DTYPE_BF16)
    return int(_lib.lib().flce_chunk_rows(ctypes.byref(p), mode, int(need_grad_h), int(need_grad_W)))


def _prepare(h, W, labels, softcap, out_mult, ignore_index, reduction, grad_scale, chunk_rows, flags,
             timeout_ns, mode, need_gh, need_gw, vocab_slab=0):
    _check(h, W, labels)
    H = W.shape[1]
    V = W.shape[0]
    h2 = _rows2d(h, H)
    if W.stride(1) != 1 or W.stride(0) % 8 != 0 or W.data_ptr() % 16 != 0:
        W = W.contiguous()
    lab = labels.reshape(-1).contiguous()
    p = _params(h2.shape[0], H, V, h2.stride(0), W.stride(0), softcap, out_mult, ignore_index, reduction,
                grad_scale, chunk_rows, flags, timeout_ns, vocab_slab, _dtype_code(h2))
    nbytes = _lib.lib().flce_workspace_size(ctypes.byref(p), mode, int(need_gh), int(need_gw))
    if nbytes == 0:
        raise FlceError(_lib.FLCE_ERR_ARG, "flce_workspace_size")
    ws = _workspace(h.device, nbytes)
    return p, h2, W, lab, ws, nbytes


def flce_ce_only(h, W, labels, *, softcap=0.0, out_mult=1.0, ignore_index=-100, reduction="mean",
                 chunk_rows=0, flags=0, timeout_ns=0):
    """CE-only pass (no gradients, no saved state). Returns (loss, token_accuracy)
    as 0-d fp32 CUDA tensors."""
    p, h2, W, lab, ws, nbytes = _prepare(h, W, labels, softcap, out_mult, ignore_index, reduction, 1.0,
                                         chunk_rows, flags, timeout_ns, FLCE_MODE_CE_ONLY, False, False)
    loss = torch.empty((), dtype=torch.float32, device=h.device)
    acc = torch.empty((), dtype=torch.float32, device=h.device)
    rc = _native(h.device, "flce_ce_only", ctypes.byref(p), _ptr(h2), _ptr(W), _ptr(lab), _ptr(loss), _ptr(acc),
                                 _ptr(ws), nbytes, _stream_handle(h.device))
    _raise(rc, "flce_ce_only")
    return loss, acc


def flce_ce_only_noalloc(h, W, labels, *, softcap=0.0, out_mult=1.0, ignore_index=-100, reduction="mean",
                         chunk_rows=0, flags=0, timeout_ns=0):
    """CE-only pass through the entry point that allocates no device memory in the
    library (its scratch is a fixed 64 MiB device array), for callers that cannot
    allocate. Returns (loss, token_accuracy, status) as 0-d CUDA tensors; the
    outputs themselves are allocated here by torch, as any caller would."""
    _check(h, W, labels)
    H = W.shape[1]
    h2 = _rows2d(h, H)
    if W.stride(1) != 1 or W.stride(0) % 8 != 0 or W.data_ptr() % 16 != 0:
        W = W.contiguous()
    lab = labels.reshape(-1).contiguous()
    p = _params(h2.shape[0], H, W.shape[0], h2.stride(0), W.stride(0), softcap, out_mult, ignore_index,
                reduction, 1.0, chunk_rows, flags, timeout_ns, 0, _dtype_code(h2))
    dev = h.device
    loss = torch.empty((), dtype=torch.float32, device=dev)
    acc = torch.empty((), dtype=torch.float32, device=dev)
    status = torch.zeros((), dtype=torch.int32, device=dev)
    rc = _native(dev, "flce_ce_only_noalloc", ctypes.byref(p), _ptr(h2), _ptr(W), _ptr(lab), _ptr(loss), _ptr(acc),
                                         _ptr(status), _stream_handle(dev))
    _raise(rc, "flce_ce_only_noalloc")
    return loss, acc, status


def flce_forward(h, W, labels, *, softcap=0.0, out_mult=1.0, ignore_index=-100, reduction="mean",
                 return_predicted=True, return_lse=False, chunk_rows=0, flags=0, timeout_ns=0):
    """Forward only. Returns dict(loss, token_accuracy, predicted, lse); per-row
    outputs have h's leading shape."""
    p, h2, W, lab, ws, nbytes = _prepare(h, W, labels, softcap, out_mult, ignore_index, reduction, 1.0,
                                         chunk_rows, flags, timeout_ns, FLCE_MODE_FORWARD, False, False)
    dev = h.device
    loss = torch.empty((), dtype=torch.float32, device=dev)
    acc = torch.empty((), dtype=torch.float32, device=dev)
    pred = torch.empty(h2.shape[0], dtype=torch.int64, device=dev) if return_predicted else None
    lse = torch.empty(h2.shape[0], dtype=torch.float32, device=dev) if return_lse else None
    rc = _native(dev, "flce_forward", ctypes.byref(p), _ptr(h2), _ptr(W), _ptr(lab), _ptr(loss), _ptr(acc),
                                 _ptr(pred), _ptr(lse), _ptr(ws), nbytes, _stream_handle(dev))
    _raise(rc, "flce_forward")
    lead = h.shape[:-1]
    return {"loss": loss, "token_accuracy": acc,
            "predicted": None if pred is None else pred.view(lead),
            "lse": None if lse is None else lse.view(lead)}


def flce_forward_backward(h, W, labels, *, grad_W: Optional[torch.Tensor] = None, need_grad_h=True,
                          softcap=0.0, out_mult=1.0, ignore_index=-100, reduction="mean", grad_scale=1.0,
                          return_predicted=False, chunk_rows=0, flags=0, timeout_ns=0, low_memory=False,
                          vocab_slab=0):
    """Forward + backward. grad_W: fp32 [V, H] CUDA tensor ACCUMULATED in place
    (grad_W += dL/dW), or None for a frozen W. Returns dict(loss,
    token_accuracy, predicted, grad_h, grad_W); grad_h (bf16) has h's shape.
    low_memory=True selects the recompute backward (FLCE_FLAG_RECOMPUTE): no
    logits kept, dlogits formed per vocab slab of vocab_slab columns."""
    if low_memory:
        flags |= FLCE_FLAG_RECOMPUTE
    if grad_W is not None:
        if grad_W.dtype != torch.float32 or grad_W.shape != W.shape or not grad_W.is_contiguous():
            raise ValueError("grad_W must be a contiguous fp32 tensor shaped like W")
        if grad_W.device != W.device:
            raise ValueError("grad_W must be on W's device")
    p, h2, W, lab, ws, nbytes = _prepare(h, W, labels, softcap, out_mult, ignore_index, reduction, grad_scale,
                                         chunk_rows, flags, timeout_ns, FLCE_MODE_FORWARD_BACKWARD,
                                         need_grad_h, grad_W is not None, vocab_slab)
    dev = h.device
    loss = torch.empty((), dtype=torch.float32, device=dev)
    acc = torch.empty((), dtype=torch.float32, device=dev)
    pred = torch.empty(h2.shape[0], dtype=torch.int64, device=dev) if return_predicted else None
    gh = torch.empty((h2.shape[0], W.shape[1]), dtype=h2.dtype, device=dev) if need_grad_h else None
    rc = _native(dev, "flce_forward_backward", ctypes.byref(p), _ptr(h2), _ptr(W), _ptr(lab), _ptr(loss), _ptr(acc),
                                          _ptr(pred), _ptr(gh), _ptr(grad_W), _ptr(ws), nbytes,
                                          _stream_handle(dev))
    _raise(rc, "flce_forward_backward")
    lead = h.shape[:-1]
    return {"loss": loss, "token_accuracy": acc,
            "predicted": None if pred is None else pred.view(lead),
            "grad_h": None if gh is None else gh.view(h.shape), "grad_W": grad_W}


# ---------------------------------------------------------------- vocab-parallel
def _vp_params(h2, W, softcap, out_mult, ignore_index, reduction, grad_scale, chunk_rows, flags, timeout_ns,
               vocab_slab=0):
    return _params(h2.shape[0], W.shape[1], W.shape[0], h2.stride(0), W.stride(0), softcap, out_mult, ignore_index,
                   reduction, grad_scale, chunk_rows, flags, timeout_ns, vocab_slab, _dtype_code(h2))


def _vp_workspace(dev, nbytes: int, workspace: Optional[torch.Tensor], flags: int) -> torch.Tensor:
    if workspace is None:
        if flags & FLCE_FLAG_VP_STORED:
            raise ValueError("FLCE_FLAG_VP_STORED keeps the logits in the workspace between the two calls: "
                             "pass the same workspace= (from flce_vp_workspace) to both")
        return _workspace(dev, nbytes)
    if workspace.dtype != torch.uint8 or workspace.device != dev or workspace.numel() < nbytes:
        raise ValueError(f"workspace must be a uint8 tensor of at least {nbytes} bytes on {dev}")
    return workspace


def flce_vp_workspace(h, W_shard, *, keep_logits=False, backward=True, need_grad_h=True, need_grad_W=True,
                      chunk_rows=0, vocab_slab=0, flags=0) -> torch.Tensor:
    """A device workspace (uint8) for flce_vp_forward / flce_vp_backward on
    these shapes. With keep_logits (FLCE_FLAG_VP_STORED) one workspace serves
    both calls and holds the shard's logits between them."""
    H = W_shard.shape[1]
    h2 = _rows2d(h, H)
    if keep_logits:
        flags |= FLCE_FLAG_VP_STORED
    p = _vp_params(h2, W_shard, 0.0, 1.0, -100, "mean", 1.0, chunk_rows, flags, 0, vocab_slab)
    nbytes = _native(h.device, "flce_vp_workspace_size", ctypes.byref(p), int(backward), int(need_grad_h),
                     int(need_grad_W))
    if nbytes == 0:
        raise FlceError(_lib.FLCE_ERR_ARG, "flce_vp_workspace_size")
    return torch.empty(nbytes, dtype=torch.uint8, device=h.device)


def flce_vp_forward(h, W_shard, labels, vocab_offset: int, vocab_total: int, *, softcap=0.0, out_mult=1.0,
                    ignore_index=-100, chunk_rows=0, flags=0, timeout_ns=0,
                    workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Forward of one vocab shard (W_shard holds the rows of vocab ids
    [vocab_offset, vocab_offset + V_k) of vocab_total): returns this shard's
    per-row partials, an fp32 [4, N] CUDA tensor (max, sum of exp, argmax id
    as int32 bits, label logit or 0). With FLCE_FLAG_VP_STORED in flags the
    shard's logits stay in `workspace` for flce_vp_backward."""
    _check(h, W_shard, labels)
    H = W_shard.shape[1]
    h2 = _rows2d(h, H)
    if W_shard.stride(1) != 1 or W_shard.stride(0) % 8 != 0 or W_shard.data_ptr() % 16 != 0:
        W_shard = W_shard.contiguous()
    lab = labels.reshape(-1).contiguous()
    p = _vp_params(h2, W_shard, softcap, out_mult, ignore_index, "mean", 1.0, chunk_rows, flags, timeout_ns)
    nbytes = _native(h.device, "flce_vp_workspace_size", ctypes.byref(p), 0, 0, 0)
    if nbytes == 0:
        raise FlceError(_lib.FLCE_ERR_ARG, "flce_vp_workspace_size")
    ws = _vp_workspace(h.device, nbytes, workspace, flags)
    part = torch.empty((4, h2.shape[0]), dtype=torch.float32, device=h.device)
    rc = _native(h.device, "flce_vp_forward", ctypes.byref(p), int(vocab_offset), int(vocab_total), _ptr(h2),
                 _ptr(W_shard), _ptr(lab), _ptr(part), _ptr(ws), nbytes, _stream_handle(h.device))
    _raise(rc, "flce_vp_forward")
    return part


def flce_vp_backward(h, W_shard, labels, all_partials: torch.Tensor, shard_offsets, vocab_offset: int,
                     vocab_total: int, *, grad_h_partial: Optional[torch.Tensor] = None,
                     grad_W: Optional[torch.Tensor] = None, softcap=0.0, out_mult=1.0, ignore_index=-100,
                     reduction="mean", grad_scale=1.0, return_predicted=True, return_lse=False, chunk_rows=0,
                     vocab_slab=0, flags=0, timeout_ns=0, workspace: Optional[torch.Tensor] = None) -> dict:
    """Backward of one vocab shard given every shard's partials ([S, 4, N], in
    shard order) and the shard table (S + 1 vocab offsets). grad_h_partial
    (fp32 [N, H]) and grad_W (this shard's fp32 [V_k, H]) are ACCUMULATED in
    place when given. Returns dict(loss, token_accuracy, predicted, lse).
    With FLCE_FLAG_VP_STORED it reads the logits that flce_vp_forward kept in
    `workspace` (the same params and workspace as that call)."""
    _check(h, W_shard, labels)
    H = W_shard.shape[1]
    h2 = _rows2d(h, H)
    if W_shard.stride(1) != 1 or W_shard.stride(0) % 8 != 0 or W_shard.data_ptr() % 16 != 0:
        W_shard = W_shard.contiguous()
    lab = labels.reshape(-1).contiguous()
    N = h2.shape[0]
    S = len(shard_offsets) - 1
    if (all_partials.dtype != torch.float32 or tuple(all_partials.shape) != (S, 4, N)
            or all_partials.device != h.device):
        raise ValueError("all_partials must be an fp32 [S, 4, N] tensor on h's device")
    all_partials = all_partials.contiguous()
    for name, t, shape in (("grad_h_partial", grad_h_partial, (N, H)), ("grad_W", grad_W, tuple(W_shard.shape))):
        if t is not None and (t.dtype != torch.float32 or tuple(t.shape) != shape or not t.is_contiguous()
                              or t.device != h.device):
            raise ValueError(f"{name} must be a contiguous fp32 {shape} tensor on h's device")
    p = _vp_params(h2, W_shard, softcap, out_mult, ignore_index, reduction, grad_scale, chunk_rows, flags,
                   timeout_ns, vocab_slab)
    nbytes = _native(h.device, "flce_vp_workspace_size", ctypes.byref(p), 1, int(grad_h_partial is not None),
                     int(grad_W is not None))
    if nbytes == 0:
        raise FlceError(_lib.FLCE_ERR_ARG, "flce_vp_workspace_size")
    ws = _vp_workspace(h.device, nbytes, workspace, flags)
    dev = h.device
    loss = torch.empty((), dtype=torch.float32, device=dev)
    acc = torch.empty((), dtype=torch.float32, device=dev)
    pred = torch.empty(N, dtype=torch.int64, device=dev) if return_predicted else None
    lse = torch.empty(N, dtype=torch.float32, device=dev) if return_lse else None
    offs = (ctypes.c_int64 * (S + 1))(*[int(o) for o in shard_offsets])
    rc = _native(dev, "flce_vp_backward", ctypes.byref(p), int(vocab_offset), int(vocab_total), S, offs,
                 _ptr(all_partials), _ptr(h2), _ptr(W_shard), _ptr(lab), _ptr(loss), _ptr(acc), _ptr(pred), _ptr(lse),
                 _ptr(grad_h_partial), _ptr(grad_W), _ptr(ws), nbytes, _stream_handle(dev))
    _raise(rc, "flce_vp_backward")
    lead = h.shape[:-1]
    return {"loss": loss, "token_accuracy": acc, "predicted": None if pred is None else pred.view(lead),
            "lse": None if lse is None else lse.view(lead)}


def _world(group) -> int:
    """Ranks in `group` (None: the default group), 1 without torch.distributed."""
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized():
        return 1
    return dist.get_world_size(group)


def vp_shard_table(vocab_offset: int, vocab_shard: int, group=None):
    """(offsets, order): the S + 1 vocab offsets of the shards of `group` (None:
    the default group) in vocab order, and the ranks in that order, from every
    rank's (offset, size). The shards must tile [0, vocab_total) without gaps
    or overlap."""
    import torch.distributed as dist
    mine = torch.tensor([int(vocab_offset), int(vocab_shard)], dtype=torch.int64)
    if _world(group) == 1:
        table = [mine]
    else:
        if dist.get_backend(group) == "nccl":  # NCCL exchanges device tensors only
            mine = mine.to(torch.device("cuda", torch.cuda.current_device()))
        table = [torch.empty_like(mine) for _ in range(_world(group))]
        dist.all_gather(table, mine, group=group)
    rows = sorted((int(t[0]), int(t[1]), r) for r, t in enumerate(table))
    offsets, order = [0], []
    for off, size, r in rows:
        if off != offsets[-1] or size <= 0:
            raise ValueError(f"vocab shards do not tile the vocabulary: {[(o, s) for o, s, _ in rows]}")
        offsets.append(off + size)
        order.append(r)
    return offsets, order


def vp_gather_partials(partials: torch.Tensor, order, group=None) -> torch.Tensor:
    """Every rank's [4, N] partials gathered and put in vocab order ([S, 4, N])."""
    import torch.distributed as dist
    if _world(group) == 1:
        return partials.unsqueeze(0)
    W = _world(group)
    out = torch.empty((W, *partials.shape), dtype=partials.dtype, device=partials.device)
    dist.all_gather(list(out.unbind(0)), partials.contiguous(), group=group)
    return out[torch.as_tensor(order, device=out.device)].contiguous()


def vp_reduce_grad_h(grad_h_partial: torch.Tensor, group=None) -> torch.Tensor:
    """Sums the shards' fp32 grad_h parts over `group` (in place)."""
    import torch.distributed as dist
    if _world(group) > 1:
        dist.all_reduce(grad_h_partial, op=dist.ReduceOp.SUM, group=group)
    return grad_h_partial


def vocab_parallel_linear_cross_entropy(h, W_shard, labels, vocab_offset: int, *, group=None,
                                        grad_W: Optional[torch.Tensor] = None, need_grad_h=True, softcap=0.0,
                                        out_mult=1.0, ignore_index=-100, reduction="mean", grad_scale=1.0,
                                        chunk_rows=0, vocab_slab=0, keep_logits=False) -> dict:
    """The fused head with W split by vocabulary rows over the ranks of
    `group` (one shard per rank, any order): shard forward, all-gather of the
    per-row partials (16 bytes per row and rank), shard backward, all-reduce of
    the fp32 grad_h parts, rounded to h's dtype by the library's kernel. Every
    rank gets the same loss, token accuracy and predictions; grad_W (this
    rank's fp32 [V_k, H], optional) is accumulated in place. keep_logits keeps
    each shard's logits between its forward and backward
    (FLCE_FLAG_VP_STORED: 6 N H V_k flops instead of 8, O(N V_k) memory)."""
    offsets, order = vp_shard_table(vocab_offset, W_shard.shape[0], group)
    V = offsets[-1]
    flags = FLCE_FLAG_VP_STORED if keep_logits else 0
    ws = flce_vp_workspace(h, W_shard, keep_logits=True, chunk_rows=chunk_rows) if keep_logits else None
    part = flce_vp_forward(h, W_shard, labels, vocab_offset, V, softcap=softcap, out_mult=out_mult,
                           ignore_index=ignore_index, chunk_rows=chunk_rows, flags=flags, workspace=ws)
    allp = vp_gather_partials(part, order, group)
    gh32 = None
    if need_grad_h:
        gh32 = torch.zeros((h.reshape(-1, h.shape[-1]).shape[0], h.shape[-1]), dtype=torch.float32, device=h.device)
    out = flce_vp_backward(h, W_shard, labels, allp, offsets, vocab_offset, V, grad_h_partial=gh32, grad_W=grad_W,
                           softcap=softcap, out_mult=out_mult, ignore_index=ignore_index, reduction=reduction,
                           grad_scale=grad_scale, chunk_rows=chunk_rows, vocab_slab=vocab_slab, flags=flags,
                           workspace=ws)
    gh = None
    if gh32 is not None:
        vp_reduce_grad_h(gh32, group)
        gh = flce_scale_gradient(gh32, None, out_dtype=h.dtype).view(h.shape)
    out["grad_h"] = gh
    out["grad_W"] = grad_W
    return out


_copy_streams: dict = {}


def _host_inputs(h, W, labels, softcap, out_mult, ignore_index, reduction, grad_scale, chunk_rows, flags,
                 timeout_ns, vocab_slab, mode, need_gh, need_gw):
    """Checks and marshals the host-input calls: h and labels on the host, W on
    the device; returns (params, h rows, W, labels, workspace, bytes, copy stream)."""
    for name, t in (("h", h), ("labels", labels)):
        if not isinstance(t, torch.Tensor) or t.device.type != "cpu":
            raise ValueError(f"{name} must be a host (CPU) tensor here")
    if not isinstance(W, torch.Tensor) or W.device.type != "cuda" or W.dim() != 2 or \
            W.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("W must be a bf16 or fp32 [V, H] CUDA tensor")
    if h.dtype != W.dtype or h.shape[-1] != W.shape[1]:
        raise ValueError("h must be [..., H] with W's H and dtype")
    if labels.dtype != torch.int64 or labels.shape != h.shape[:-1]:
        raise ValueError("labels must be int64 with h's leading shape")
    H, V = W.shape[1], W.shape[0]
    h2 = h.reshape(-1, H)
    if h2.stride(1) != 1 or h2.stride(0) % 8 != 0:
        h2 = h2.contiguous()
    if W.stride(1) != 1 or W.stride(0) % 8 != 0 or W.data_ptr() % 16 != 0:
        W = W.contiguous()
    lab = labels.reshape(-1).contiguous()
    p = _params(h2.shape[0], H, V, h2.stride(0), W.stride(0), softcap, out_mult, ignore_index, reduction,
                grad_scale, chunk_rows, flags, timeout_ns, vocab_slab, _dtype_code(W))
    nbytes = _lib.lib().flce_workspace_size(ctypes.byref(p), mode, int(need_gh), int(need_gw))
    if nbytes == 0:
        raise FlceError(_lib.FLCE_ERR_ARG, "flce_workspace_size")
    dev = W.device
    ws = _workspace(dev, nbytes)
    idx = dev.index if dev.index is not None else torch.cuda.current_device()
    cs = _copy_streams.get(idx)
    if cs is None:
        cs = _copy_streams[idx] = torch.cuda.Stream(device=idx)
    return p, h2, W, lab, ws, nbytes, cs


def flce_forward_backward_from_host(h, W, labels, *, grad_W: Optional[torch.Tensor] = None, need_grad_h=True,
                                    softcap=0.0, out_mult=1.0, ignore_index=-100, reduction="mean",
                                    grad_scale=1.0, return_predicted=False, chunk_rows=0, flags=0, timeout_ns=0,
                                    low_memory=False, vocab_slab=0):
    """Forward + backward with h ([..., H], bf16 or fp32 like W) and labels
    (int64) in host memory, page-locked for the copies to overlap the kernels: the library
    copies h chunk by chunk on a side stream while it computes the previous
    chunk. W, grad_W and the returned grad_h / predicted are CUDA tensors on
    the current device; loss and token_accuracy come back as 0-d page-locked
    host tensors, valid once the current stream has been synchronised (h and
    labels must stay unchanged until then)."""
    if low_memory:
        flags |= FLCE_FLAG_RECOMPUTE
    if grad_W is not None and (grad_W.dtype != torch.float32 or grad_W.shape != W.shape or
                               not grad_W.is_contiguous() or grad_W.device != W.device):
        raise ValueError("grad_W must be a contiguous fp32 tensor shaped like W, on W's device")
    p, h2, W, lab, ws, nbytes, cs = _host_inputs(h, W, labels, softcap, out_mult, ignore_index, reduction,
                                                 grad_scale, chunk_rows, flags, timeout_ns, vocab_slab,
                                                 _lib.FLCE_MODE_FORWARD_BACKWARD_HOST, need_grad_h,
                                                 grad_W is not None)
    dev, H = W.device, W.shape[1]
    loss = torch.empty((), dtype=torch.float32).pin_memory()
    acc = torch.empty((), dtype=torch.float32).pin_memory()
    pred = torch.empty(h2.shape[0], dtype=torch.int64, device=dev) if return_predicted else None
    gh = torch.empty((h2.shape[0], H), dtype=W.dtype, device=dev) if need_grad_h else None
    rc = _native(
        dev, "flce_forward_backward_from_host", ctypes.byref(p), _ptr(h2), _ptr(W), _ptr(lab), _ptr(loss), _ptr(acc), _ptr(pred), _ptr(gh), _ptr(grad_W),
        _ptr(ws), nbytes, _stream_handle(dev), ctypes.c_void_p(cs.cuda_stream))
    _raise(rc, "flce_forward_backward_from_host")
    lead = h.shape[:-1]
    return {"loss": loss, "token_accuracy": acc, "predicted": None if pred is None else pred.view(lead),
            "grad_h": None if gh is None else gh.view(*lead, H), "grad_W": grad_W}


def flce_ce_only_from_host(h, W, labels, *, softcap=0.0, out_mult=1.0, ignore_index=-100, reduction="mean",
                           chunk_rows=0, flags=0, timeout_ns=0):
    """CE-only pass with h and labels in (page-locked) host memory, copied by
    the library chunk by chunk under its kernels. Returns (loss,
    token_accuracy) as 0-d page-locked host tensors, valid once the current
    stream has been synchronised."""
    p, h2, W, lab, ws, nbytes, cs = _host_inputs(h, W, labels, softcap, out_mult, ignore_index, reduction, 1.0,
                                                 chunk_rows, flags, timeout_ns, 0, _lib.FLCE_MODE_CE_ONLY_HOST,
                                                 False, False)
    loss = torch.empty((), dtype=torch.float32).pin_memory()
    acc = torch.empty((), dtype=torch.float32).pin_memory()
    rc = _native(W.device, "flce_ce_only_from_host", ctypes.byref(p), _ptr(h2), _ptr(W), _ptr(lab), _ptr(loss), _ptr(acc),
                                           _ptr(ws), nbytes, _stream_handle(W.device),
                                           ctypes.c_void_p(cs.cuda_stream))
    _raise(rc, "flce_ce_only_from_host")
    return loss, acc


def flce_cross_entropy(logits, labels, *, softcap=0.0, out_mult=1.0, ignore_index=-100, reduction="mean",
                       grad_scale=1.0, row_scale: Optional[torch.Tensor] = None, need_grad=True,
                       grad_in_place=False, return_predicted=True, chunk_rows=0):
    """Cross-entropy on materialised logits [..., V] (bf16 or fp32 CUDA tensor).
    Returns dict(loss, token_accuracy, predicted, row_loss, grad_logits); with
    reduction="none" the gradient is that of sum_i row_scale_i * row_loss_i.
    grad_in_place=True writes dL/dlogits over the logits."""
    if not isinstance(logits, torch.Tensor) or logits.device.type != "cuda":
        raise ValueError("logits must be a CUDA tensor (the library has no CPU path)")
    if logits.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("logits must be bfloat16 or float32")
    if labels.dtype != torch.int64 or labels.shape != logits.shape[:-1] or labels.device != logits.device:
        raise ValueError("labels must be int64 with logits' leading shape, on its device")
    V = logits.shape[-1]
    x = logits.reshape(-1, V)
    if x.stride(1) != 1:
        x = x.contiguous()
    if grad_in_place and x.data_ptr() != logits.data_ptr():
        raise ValueError("grad_in_place needs logits whose rows can be viewed as [N, V] in place")
    lab = labels.reshape(-1).contiguous()
    N = x.shape[0]
    rs = None
    if row_scale is not None:
        rs = row_scale.reshape(-1).to(dtype=torch.float32).contiguous()
        if rs.numel() != N or rs.device != logits.device:
            raise ValueError("row_scale must hold one value per row, on the logits' device")
    p = _params(N, 8, V, 0, 0, softcap, out_mult, ignore_index, reduction, grad_scale, chunk_rows, 0, 0)
    nbytes = _lib.lib().flce_workspace_size(ctypes.byref(p), _lib.FLCE_MODE_CROSS_ENTROPY, 0, 0)
    if nbytes == 0:
        raise FlceError(_lib.FLCE_ERR_ARG, "flce_workspace_size")
    dev = logits.device
    ws = _workspace(dev, nbytes)
    loss = torch.empty((), dtype=torch.float32, device=dev)
    acc = torch.empty((), dtype=torch.float32, device=dev)
    pred = torch.empty(N, dtype=torch.int64, device=dev) if return_predicted else None
    row_loss = torch.empty(N, dtype=torch.float32, device=dev)
    grad = None
    if need_grad:
        grad = x if grad_in_place else torch.empty_like(x)
    dt = _lib.FLCE_DTYPE_BF16 if x.dtype == torch.bfloat16 else _lib.FLCE_DTYPE_F32
    rc = _native(dev, "flce_cross_entropy", ctypes.byref(p), _ptr(x), dt, x.stride(0), _ptr(lab), _ptr(loss), _ptr(acc),
                                       _ptr(pred), _ptr(row_loss), _ptr(rs), _ptr(grad), _ptr(ws), nbytes,
                                       _stream_handle(dev))
    _raise(rc, "flce_cross_entropy")
    lead = logits.shape[:-1]
    return {"loss": loss, "token_accuracy": acc, "predicted": None if pred is None else pred.view(lead),
            "row_loss": row_loss.view(lead), "grad_logits": None if grad is None else grad.view(logits.shape)}


def flce_scale_gradient(x: torch.Tensor, scale: Optional[torch.Tensor] = None, *, out_dtype=None,
                        out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """out = scale * x in out_dtype (bf16 results rounded to nearest even),
    computed by the library's kernel. x: contiguous bf16 or fp32 CUDA tensor;
    scale: fp32 CUDA tensor of one element, or None for 1; out=x scales in
    place (same dtype only)."""
    if not isinstance(x, torch.Tensor) or x.device.type != "cuda":
        raise ValueError("x must be a CUDA tensor (the library has no CPU path)")
    out_dtype = x.dtype if out_dtype is None else out_dtype
    for t in (x.dtype, out_dtype):
        if t not in (torch.bfloat16, torch.float32):
            raise ValueError("x and out must be bfloat16 or float32")
    if not x.is_contiguous():
        raise ValueError("x must be contiguous")
    if scale is not None:
        if (not isinstance(scale, torch.Tensor) or scale.device != x.device or scale.dtype != torch.float32
                or scale.numel() != 1):
            raise ValueError("scale must be a one-element fp32 tensor on x's device")
    if out is None:
        out = torch.empty(x.shape, dtype=out_dtype, device=x.device)
    elif out.dtype != out_dtype or out.shape != x.shape or not out.is_contiguous() or out.device != x.device:
        raise ValueError("out must be a contiguous tensor of x's shape and device in out_dtype")
    rc = _native(x.device, "flce_scale_gradient", _ptr(x), _dtype_code(x), _ptr(out), _dtype_code(out), x.numel(),
                                        _ptr(scale), _stream_handle(x.device))
    _raise(rc, "flce_scale_gradient")
    return out


class _LinearCrossEntropy(torch.autograd.Function):
    """Autograd node of the fused head. The forward runs the fused
    forward+backward with grad_scale 1 and keeps grad_h and grad_W, the way the
    pages' fused linear-cross-entropy functions do (DeepSeek-V3 page, Summary:
    the fused loss inside the model's forward, logits never kept); the backward
    only multiplies them by the upstream gradient of the loss."""

    @staticmethod
    def forward(ctx, h, W, labels, softcap, out_mult, ignore_index, reduction, chunk_rows, low_memory):
        need_gh, need_gW = ctx.needs_input_grad[0], ctx.needs_input_grad[1]
        ctx.w_dtype = W.dtype
        if not (need_gh or need_gW):
            loss, acc = flce_ce_only(h, W, labels, softcap=softcap, out_mult=out_mult, ignore_index=ignore_index,
                                     reduction=reduction, chunk_rows=chunk_rows)
            ctx.save_for_backward(None, None)
        else:
            gW = torch.zeros(W.shape, dtype=torch.float32, device=W.device) if need_gW else None
            out = flce_forward_backward(h, W, labels, grad_W=gW, need_grad_h=need_gh, softcap=softcap,
                                        out_mult=out_mult, ignore_index=ignore_index, reduction=reduction,
                                        chunk_rows=chunk_rows, low_memory=low_memory)
            loss, acc = out["loss"], out["token_accuracy"]
            ctx.save_for_backward(out["grad_h"], gW)
        ctx.mark_non_differentiable(acc)
        return loss, acc

    @staticmethod
    def backward(ctx, grad_loss, grad_acc):
        # The saved gradients are scaled in place (no second copy of grad_h, or
        # of an fp32 grad_W). Their version counters are bumped so that a second
        # backward through the same node (retain_graph=True) raises autograd's
        # in-place modification error instead of scaling them twice.
        gh, gW = ctx.saved_tensors
        g = grad_loss.reshape(1)
        if gh is not None:
            flce_scale_gradient(gh, g, out=gh)
            _bump_version(gh)
        if gW is not None:
            in_place = ctx.w_dtype == torch.float32
            gW_saved = gW
            gW = flce_scale_gradient(gW, g, out=gW if in_place else None, out_dtype=ctx.w_dtype)
            if in_place:
                _bump_version(gW_saved)
        return gh, gW, None, None, None, None, None, None, None


def _bump_version(t: torch.Tensor) -> None:
    """Marks t as modified in place (its data was written through the C ABI)."""
    inc = getattr(torch.autograd.graph, "increment_version", None)
    if inc is not None:
        inc(t)
    else:
        torch._C._increment_version(t)


def linear_cross_entropy(h, W, labels, *, softcap=0.0, out_mult=1.0, ignore_index=-100, reduction="mean",
                         chunk_rows=0, low_memory=False):
    """Differentiable fused head loss: returns (loss, token_accuracy). Gradients
    flow to h and to W where they require grad; a W that does not (a frozen
    projection, SpecForge DSpine PR, Changes) costs no grad_W work. W's
    gradient is accumulated in fp32 inside the call and handed to autograd in
    W's dtype."""
    if reduction not in ("mean", "sum"):
        raise ValueError("reduction must be 'mean' or 'sum' (per-row losses: flce_cross_entropy)")
    return _LinearCrossEntropy.apply(h, W, labels, float(softcap), float(out_mult), int(ignore_index), reduction,
                                     int(chunk_rows), bool(low_memory))


class FusedLinearCrossEntropyLoss(torch.nn.Module):
    """Module form of linear_cross_entropy: loss(h, W, labels) -> loss, or
    (loss, token_accuracy) with return_token_accuracy=True."""

    def __init__(self, *, softcap=0.0, out_mult=1.0, ignore_index=-100, reduction="mean", chunk_rows=0,
                 low_memory=False, return_token_accuracy=False):
        super().__init__()
        self.kw = dict(softcap=softcap, out_mult=out_mult, ignore_index=ignore_index, reduction=reduction,
                       chunk_rows=chunk_rows, low_memory=low_memory)
        self.return_token_accuracy = return_token_accuracy

    def forward(self, h, W, labels):
        loss, acc = linear_cross_entropy(h, W, labels, **self.kw)
        return (loss, acc) if self.return_token_accuracy else loss


def flce_get_status(device=None, workspace: Optional[torch.Tensor] = None) -> int:
    """Synchronises the current stream and returns the device status word of
    the last call on the cached workspace of this device and stream, or on
    `workspace` when given (0 = no device error)."""
    if workspace is not None:
        dev = workspace.device
        ws = workspace
    else:
        dev = torch.device("cuda", torch.cuda.current_device() if device is None else device)
        ws = _workspaces.get((dev.index, torch.cuda.current_stream(dev).cuda_stream))
    if ws is None:
        return 0
    st = ctypes.c_int32(0)
    _raise(_native(dev, "flce_get_status", _ptr(ws), _stream_handle(dev), ctypes.byref(st)), "flce_get_status")
    return int(st.value)


def flce_launch_count() -> int:
    return int(_lib.lib().flce_launch_count())


def flce_profile_begin(enable: bool = True) -> None:
    _lib.lib().flce_profile_begin(int(enable))


def flce_profile_read() -> dict:
    """{kernel name: (launches, total ms)} of the launches recorded since flce_profile_begin(True)."""
    n = _lib.FLCE_NUM_KERNELS
    launches = (ctypes.c_int64 * n)()
    ms = (ctypes.c_double * n)()
    rc = _lib.lib().flce_profile_read(launches, ms, n)
    if rc < 0:
        raise FlceError(-rc, "flce_profile_read")
    L = _lib.lib()
    return {L.flce_kernel_name(i).decode(): (int(launches[i]), float(ms[i])) for i in range(n) if launches[i]}
