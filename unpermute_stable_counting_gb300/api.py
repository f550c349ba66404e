"""PyTorch-facing binding of the C ABI (include/moe_reorder.h).

Argument marshalling only: shapes, dtypes and device pointers of torch CUDA
tensors go to the library; every step of every operation runs in the
library's CUDA kernels. PyTorch supplies device memory (outputs and the
workspace, when the caller does not pass them) and the current stream.
"""
from __future__ import annotations

import ctypes

import torch

from ._native import int64_array, lib

DT_F16, DT_BF16, DT_INT8, DT_F32 = 0, 1, 2, 3
_TORCH_TO_DT = {torch.float16: DT_F16, torch.bfloat16: DT_BF16, torch.float32: DT_F32}
_DT_TO_TORCH = {DT_F16: torch.float16, DT_BF16: torch.bfloat16, DT_INT8: torch.int8,
                DT_F32: torch.float32}

MR_OK = 0
MR_BATCHING_FULL_TAIL = 1


class MoeReorderError(RuntimeError):
    def __init__(self, status: int, where: str):
        text = lib().mr_status_string(status).decode()
        super().__init__(f"{where} failed with status {status}: {text}")
        self.status = status


def _check(status: int, where: str) -> None:
    if status != MR_OK:
        raise MoeReorderError(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _require_cuda(name, t, dtype=None, strided=False):
    if t is None:
        return
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not strided and not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise TypeError(f"{name} must have dtype {dtype}, got {t.dtype}")


def _stream(stream, device):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


# ---------------------------------------------------------------------------
# FFN-worker batching
# ---------------------------------------------------------------------------

def batching_workspace_size(expert_num: int, max_out_shape, token_dtype: int, layer_num: int,
                            need_schedule: int = 0) -> int:
    ws = ctypes.c_uint64(0)
    shape = int64_array(max_out_shape)
    _check(lib().ffnwb_batching_get_workspace_size(expert_num, shape, token_dtype, need_schedule,
                                                   layer_num, ctypes.byref(ws)),
           "ffnwb_batching_get_workspace_size")
    return int(ws.value)


def batching_outputs(Y: int, H: int, expert_num: int, token_dtype: int, device,
                     with_sorted_indices: bool = False) -> dict:
    """Allocate the output tensors of one batching call."""
    i32 = dict(dtype=torch.int32, device=device)
    return dict(
        y=torch.empty((Y, H), dtype=_DT_TO_TORCH[token_dtype], device=device),
        groupList=torch.empty((expert_num, 2), dtype=torch.int64, device=device),
        sessionIds=torch.empty(Y, **i32), microBatchIds=torch.empty(Y, **i32),
        tokenIds=torch.empty(Y, **i32), expertOffsets=torch.empty(Y, **i32),
        dynamicScale=torch.empty(Y, dtype=torch.float32, device=device) if token_dtype == DT_INT8 else None,
        actualTokenNum=torch.empty(1, dtype=torch.int64, device=device),
        sortedIndices=torch.empty(Y, **i32) if with_sorted_indices else None)


def ffnwb_batching(expert_ids, token_data, session_ids, micro_batch_ids, *, expert_num: int,
                   max_out_shape, token_dtype: int, layer_num: int = 1, layer_id: int = 0,
                   token_ids=None, scales=None, scale_stride: int = 4, token_row_stride=None,
                   need_schedule: int = 0, with_sorted_indices: bool = False, out: dict | None = None,
                   workspace=None, stream=None, full_tail: bool = False) -> dict:
    """Run the batching on the current CUDA stream.

    token_data: CUDA tensor whose first dimension is the Y slots; row s starts
    at token_row_stride bytes * s (default: the tensor's own row stride).
    full_tail: also gather the rows (and ids) of the masked slots.
    Returns the output dict (see batching_outputs)."""
    A, BS, K1, H = (int(v) for v in max_out_shape)
    Y = A * BS * K1
    for name, t in (("expert_ids", expert_ids), ("session_ids", session_ids),
                    ("micro_batch_ids", micro_batch_ids), ("token_ids", token_ids)):
        _require_cuda(name, t, torch.int32)
    _require_cuda("token_data", token_data)
    _require_cuda("scales", scales, strided=True)
    if token_row_stride is None:
        token_row_stride = token_data.stride(0) * token_data.element_size()
    dev = token_data.device
    if out is None:
        out = batching_outputs(Y, H, expert_num, token_dtype, dev, with_sorted_indices)
    if workspace is None:
        ws = batching_workspace_size(expert_num, max_out_shape, token_dtype, layer_num, need_schedule)
        workspace = torch.empty(max(ws, 1), dtype=torch.uint8, device=dev)
    shape = int64_array(max_out_shape)
    args = [_ptr(expert_ids), int(layer_id), _ptr(token_data), int(token_row_stride), _ptr(scales),
            int(scale_stride), _ptr(session_ids), _ptr(micro_batch_ids), _ptr(token_ids),
            int(expert_num), shape, int(token_dtype), int(need_schedule), int(layer_num),
            _ptr(out["y"]), _ptr(out["groupList"]), _ptr(out["sessionIds"]),
            _ptr(out["microBatchIds"]), _ptr(out["tokenIds"]), _ptr(out["expertOffsets"]),
            _ptr(out.get("dynamicScale")), _ptr(out["actualTokenNum"]), _ptr(out.get("sortedIndices"))]
    tail = [_ptr(workspace), int(workspace.numel()), _stream(stream, dev)]
    if full_tail:
        st = lib().ffnwb_batching_ex(*args, MR_BATCHING_FULL_TAIL, *tail)
    else:
        st = lib().ffnwb_batching(*args, *tail)
    _check(st, "ffnwb_batching")
    return out


def batching_context_workspace_size(expert_num: int, max_out_shape, token_dtype: int,
                                    layer_num: int, need_schedule: int = 0) -> int:
    ws = ctypes.c_uint64(0)
    _check(lib().ffnwb_batching_context_get_workspace_size(
        expert_num, int64_array(max_out_shape), token_dtype, need_schedule, layer_num,
        ctypes.byref(ws)), "ffnwb_batching_context_get_workspace_size")
    return int(ws.value)


def ffnwb_batching_context(schedule_context, *, expert_num: int, max_out_shape, token_dtype: int,
                           layer_num: int = 1, need_schedule: int = 0,
                           wait_timeout_us: int = 1_000_000, out: dict | None = None,
                           workspace=None, stream=None, full_tail: bool = False) -> dict:
    """Batching from a ScheduleContext (a CUDA tensor of its 1024 bytes) on the
    current stream. Returns the batching outputs plus scheduleStatus (int32 [1]):
    blocks not ready with need_schedule = 1, or -1 for a context that does not fit.
    full_tail: also gather the rows (and ids) of the context's masked slots."""
    _require_cuda("schedule_context", schedule_context)
    if schedule_context.numel() * schedule_context.element_size() < 1024:
        raise ValueError("schedule_context must hold 1024 bytes")
    A, BS, K1, H = (int(v) for v in max_out_shape)
    dev = schedule_context.device
    if out is None:
        out = batching_outputs(A * BS * K1, H, expert_num, token_dtype, dev)
    if out.get("scheduleStatus") is None:
        out["scheduleStatus"] = torch.zeros(1, dtype=torch.int32, device=dev)
    if workspace is None:
        ws = batching_context_workspace_size(expert_num, max_out_shape, token_dtype, layer_num,
                                             need_schedule)
        workspace = torch.empty(max(ws, 1), dtype=torch.uint8, device=dev)
    args = [_ptr(schedule_context), int(expert_num), int64_array(max_out_shape), int(token_dtype),
            int(need_schedule), int(layer_num), int(wait_timeout_us), _ptr(out["y"]),
            _ptr(out["groupList"]), _ptr(out["sessionIds"]), _ptr(out["microBatchIds"]),
            _ptr(out["tokenIds"]), _ptr(out["expertOffsets"]), _ptr(out.get("dynamicScale")),
            _ptr(out["actualTokenNum"]), _ptr(out["scheduleStatus"])]
    tail = [_ptr(workspace), int(workspace.numel()), _stream(stream, dev)]
    if full_tail:
        st = lib().ffnwb_batching_context_ex(*args, MR_BATCHING_FULL_TAIL, *tail)
    else:
        st = lib().ffnwb_batching_context(*args, *tail)
    _check(st, "ffnwb_batching_context")
    return out


# ---------------------------------------------------------------------------
# Routing-map unpermute
# ---------------------------------------------------------------------------

def _unpermute_shapes(permuted_tokens, sorted_indices, probs, padded_mode, restore_shape):
    tdt = _TORCH_TO_DT.get(permuted_tokens.dtype)
    if tdt is None:
        raise TypeError(f"permuted_tokens dtype {permuted_tokens.dtype} is not f16/bf16/f32")
    rows, H = int(permuted_tokens.shape[0]), int(permuted_tokens.shape[1])
    n = int(sorted_indices.numel())
    if probs is not None:
        pdt = _TORCH_TO_DT.get(probs.dtype)
        if pdt is None:
            raise TypeError(f"probs dtype {probs.dtype} is not f16/bf16/f32")
        T, Eu = int(probs.shape[0]), int(probs.shape[1])
    else:
        pdt, Eu = tdt, 0
        if restore_shape is None:
            raise ValueError("restore_shape is required without probs")
        T = int(restore_shape[0])
    return tdt, pdt, rows, H, n, T, Eu


def unpermute_workspace_size(rows: int, H: int, token_dtype: int, n: int, has_probs: bool,
                             probs_dtype: int, T: int, Eu: int, padded_mode: bool,
                             restore_shape=None) -> int:
    ws = ctypes.c_uint64(0)
    rs = int64_array(restore_shape) if restore_shape is not None else None
    _check(lib().moe_unpermute_get_workspace_size(rows, H, token_dtype, n, int(has_probs),
                                                  probs_dtype, T, Eu, int(padded_mode), rs,
                                                  ctypes.byref(ws)),
           "moe_unpermute_get_workspace_size")
    return int(ws.value)


def unpermute_outputs(T: int, H: int, n: int, token_dtype: int, probs_dtype: int | None, device) -> dict:
    return dict(
        unpermutedTokens=torch.empty((T, H), dtype=_DT_TO_TORCH[token_dtype], device=device),
        outIndex=torch.empty(n, dtype=torch.int32, device=device),
        permuteTokenId=torch.empty(n, dtype=torch.int32, device=device),
        permuteProbs=(torch.empty(n, dtype=_DT_TO_TORCH[probs_dtype], device=device)
                      if probs_dtype is not None else None))


def moe_unpermute(permuted_tokens, sorted_indices, routing_map=None, probs=None, *,
                  padded_mode: bool = False, restore_shape=None, out: dict | None = None,
                  workspace=None, stream=None) -> dict:
    """Run the unpermute on the current CUDA stream. Returns unpermutedTokens,
    outIndex, permuteTokenId and permuteProbs (None without probs)."""
    _require_cuda("permuted_tokens", permuted_tokens)
    _require_cuda("sorted_indices", sorted_indices, torch.int32)
    _require_cuda("routing_map", routing_map, (torch.int8, torch.bool, torch.uint8))
    _require_cuda("probs", probs)
    tdt, pdt, rows, H, n, T, Eu = _unpermute_shapes(permuted_tokens, sorted_indices, probs,
                                                     padded_mode, restore_shape)
    dev = permuted_tokens.device
    if out is None:
        out = unpermute_outputs(T, H, n, tdt, pdt if probs is not None else None, dev)
    if workspace is None:
        ws = unpermute_workspace_size(rows, H, tdt, n, probs is not None, pdt, T, Eu, padded_mode,
                                      restore_shape)
        workspace = torch.empty(max(ws, 1), dtype=torch.uint8, device=dev)
    rs = int64_array(restore_shape) if restore_shape is not None else None
    st = lib().moe_unpermute(
        _ptr(permuted_tokens), _ptr(sorted_indices), _ptr(routing_map), _ptr(probs), rows, H, tdt,
        n, pdt, T, Eu, int(bool(padded_mode)), rs, _ptr(out["unpermutedTokens"]),
        _ptr(out["outIndex"]), _ptr(out["permuteTokenId"]), _ptr(out.get("permuteProbs")),
        _ptr(workspace), int(workspace.numel()), _stream(stream, dev))
    _check(st, "moe_unpermute")
    return out


def permute_workspace_size(T: int, H: int, token_dtype: int, Eu: int, topk: int = 0,
                           padded_mode: bool = False, capacity: int = 0) -> int:
    ws = ctypes.c_uint64(0)
    _check(lib().moe_permute_get_workspace_size(T, H, token_dtype, Eu, topk, int(padded_mode),
                                                capacity, ctypes.byref(ws)),
           "moe_permute_get_workspace_size")
    return int(ws.value)


def moe_permute(tokens, routing_map, *, topk: int = 0, padded_mode: bool = False, capacity: int = 0,
                out: dict | None = None, workspace=None, stream=None) -> dict:
    """Permute tokens [T, H] by routing_map [T, Eu] on the current stream.
    Returns permutedTokens, sortedIndices and permutedRows (int32 [1])."""
    _require_cuda("tokens", tokens)
    _require_cuda("routing_map", routing_map, (torch.int8, torch.bool, torch.uint8))
    tdt = _TORCH_TO_DT.get(tokens.dtype)
    if tdt is None:
        raise TypeError(f"tokens dtype {tokens.dtype} is not f16/bf16/f32")
    T, H = int(tokens.shape[0]), int(tokens.shape[1])
    Eu = int(routing_map.shape[1])
    rows = Eu * capacity if padded_mode else T * topk
    dev = tokens.device
    if out is None:
        out = dict(permutedTokens=torch.empty((rows, H), dtype=tokens.dtype, device=dev),
                   sortedIndices=torch.empty(rows, dtype=torch.int32, device=dev),
                   permutedRows=torch.zeros(1, dtype=torch.int32, device=dev))
    if workspace is None:
        ws = permute_workspace_size(T, H, tdt, Eu, topk, padded_mode, capacity)
        workspace = torch.empty(max(ws, 1), dtype=torch.uint8, device=dev)
    st = lib().moe_permute(_ptr(tokens), _ptr(routing_map), T, H, tdt, Eu, int(topk),
                           int(bool(padded_mode)), int(capacity), _ptr(out["permutedTokens"]),
                           _ptr(out["sortedIndices"]), _ptr(out.get("permutedRows")),
                           _ptr(workspace), int(workspace.numel()), _stream(stream, dev))
    _check(st, "moe_permute")
    return out


_ID_TO_DT = {torch.int32: 4, torch.int64: 5}


def moe_update_expert(expert_ids, eplb_table, *, local_rank: int = 0, world_size: int,
                      balance_mode: int = 0, scales=None, threshold=None, active=None,
                      out: dict | None = None, stream=None) -> dict:
    """Map expert_ids [BS, K] (int32/int64) to physical instances through
    eplb_table [E, F] int32 and, with scales [BS, K] and threshold [K] (or
    [1, K]), prune them. Strided views are passed by their strides (no copy).
    Returns balancedExpertIds and balancedActiveMask (None without scales)."""
    _require_cuda("expert_ids", expert_ids, (torch.int32, torch.int64), strided=True)
    _require_cuda("eplb_table", eplb_table, (torch.int32,), strided=True)
    BS, K = int(expert_ids.shape[0]), int(expert_ids.shape[1])
    E, F = int(eplb_table.shape[0]), int(eplb_table.shape[1])
    dev = expert_ids.device
    sdt = 3
    if scales is not None:
        _require_cuda("scales", scales, strided=True)
        sdt = _TORCH_TO_DT.get(scales.dtype)
        if sdt is None:
            raise TypeError(f"scales dtype {scales.dtype} is not f16/bf16/f32")
    if threshold is not None:
        _require_cuda("threshold", threshold, (torch.float32,), strided=True)
    if active is not None:
        _require_cuda("active", active, (torch.bool, torch.uint8), strided=True)
    if out is None:
        out = dict(balancedExpertIds=torch.empty((BS, K), dtype=expert_ids.dtype, device=dev),
                   balancedActiveMask=(torch.empty((BS, K), dtype=torch.bool, device=dev)
                                       if scales is not None else None))
    bal, msk = out["balancedExpertIds"], out.get("balancedActiveMask")
    z = (0, 0)
    strides = (tuple(expert_ids.stride()) + tuple(eplb_table.stride())
               + (tuple(scales.stride()) if scales is not None else z)
               + ((threshold.stride(-1),) if threshold is not None else (0,))
               + ((active.stride(0),) if active is not None else (0,))
               + tuple(bal.stride()) + (tuple(msk.stride()) if msk is not None else (1, 1)))
    st = lib().moe_update_expert(_ptr(expert_ids), _ID_TO_DT[expert_ids.dtype], _ptr(eplb_table),
                                 _ptr(scales), sdt, _ptr(threshold), _ptr(active), BS, K, E, F,
                                 int(local_rank), int(world_size), int(balance_mode),
                                 int64_array(strides), _ptr(bal), _ptr(msk), _stream(stream, dev))
    _check(st, "moe_update_expert")
    return out


def profile_set_events(events) -> None:
    """Attach cudaEvents (torch.cuda.Event, created with enable_timing) to the
    library's phase markers for this thread; None to detach."""
    if not events:
        _check(lib().mr_profile_set_events(None, 0), "mr_profile_set_events")
        return
    for e in events:
        if not e.cuda_event:  # torch creates the CUDA event on its first record
            e.record()
    arr = (ctypes.c_void_p * len(events))(*[ctypes.c_void_p(e.cuda_event) for e in events])
    _check(lib().mr_profile_set_events(arr, len(events)), "mr_profile_set_events")
