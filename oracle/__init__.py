"""CPU parity oracle (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline /
reference leg may import this package. The product path never does.

The arithmetic lives in ``oracle.cpp`` (plain single-threaded C++17, built
with ``-ffp-contract=off``); this module only compiles it and marshals numpy
arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import fcntl
import hashlib
import os
import platform
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")
_CFLAGS = ["-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]
# A prebuilt oracle library to load instead (the mutation tests point this at a
# copy of the oracle with a planted mistake).
_LIB_OVERRIDE = os.environ.get("USC_ORACLE_LIB")
_lib = None

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32


def compile_library(src: str, out: str) -> str:
    """Compile one oracle source file into a shared library."""
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["g++"] + _CFLAGS + ["-o", tmp, src]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _digest() -> str:
    """SHA-256 of the oracle source, the compile command and the machine type:
    the library is rebuilt whenever its stamp differs (content, not times)."""
    h = hashlib.sha256()
    with open(_SRC, "rb") as f:
        h.update(f.read())
    h.update(" ".join(_CFLAGS).encode() + platform.machine().encode())
    return h.hexdigest()


def _stale() -> bool:
    stamp = _LIB + ".sha256"
    if not os.path.exists(_LIB) or not os.path.exists(stamp):
        return True
    with open(stamp) as f:
        return f.read().strip() != _digest()


def build(force: bool = False) -> str:
    """Compile oracle.cpp into liboracle.so (next to it), one builder at a time."""
    if force or _stale():
        with open(os.path.join(_HERE, ".build.lock"), "w") as lk:
            fcntl.flock(lk, fcntl.LOCK_EX)
            try:
                if force or _stale():
                    compile_library(_SRC, _LIB)
                    with open(_LIB + ".sha256", "w") as f:
                        f.write(_digest() + "\n")
            finally:
                fcntl.flock(lk, fcntl.LOCK_UN)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        if _LIB_OVERRIDE:
            lib = ctypes.CDLL(_LIB_OVERRIDE)
        else:
            build()
            lib = ctypes.CDLL(_LIB)
        lib.oracle_batching.restype = _I32
        lib.oracle_batching.argtypes = [
            _P, _I32, _P, _I64, _P, _I64, _P, _P, _P,
            _I64, _I64, _I64, _I64, _I64, _I64, _I64,
            _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I32]
        lib.oracle_batching_context.restype = _I32
        lib.oracle_batching_context.argtypes = [
            _P, _P, _P, _I64, _I64, _I64, _I64, _I64, _I64, _I64, _I64,
            _P, _P, _P, _P, _P, _P, _P, _P, _P, _I32]
        lib.oracle_permute.restype = _I32
        lib.oracle_permute.argtypes = [_P, _P, _I64, _I64, _I32, _I64, _I64, _I32, _I64, _P, _P, _P]
        lib.oracle_update_expert.restype = _I32
        lib.oracle_update_expert.argtypes = [_P, _I32, _P, _P, _I32, _P, _P, _I64, _I64, _I64, _I64,
                                             _I64, _I64, _P, _P]
        lib.oracle_unpermute.restype = _I32
        lib.oracle_unpermute.argtypes = [
            _P, _P, _P, _P, _I64, _I64, _I32, _I64, _I32, _I64, _I64, _I32,
            _P, _P, _P, _P]
        for name in ("oracle_half_to_float", "oracle_float_to_half", "oracle_bf16_to_float",
                     "oracle_float_to_bf16"):
            getattr(lib, name).restype = None
            getattr(lib, name).argtypes = [_P, _P, _I64]
        _lib = lib
    return _lib


def _ptr(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be contiguous"
    return a.ctypes.data


# -- conversions (exported for the conversion pins) -------------------------

def half_to_float(bits: np.ndarray) -> np.ndarray:
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(bits.shape, dtype=np.float32)
    _load().oracle_half_to_float(_ptr(bits), _ptr(out), bits.size)
    return out


def float_to_half(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().oracle_float_to_half(_ptr(x), _ptr(out), x.size)
    return out


def bf16_to_float(bits: np.ndarray) -> np.ndarray:
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(bits.shape, dtype=np.float32)
    _load().oracle_bf16_to_float(_ptr(bits), _ptr(out), bits.size)
    return out


def float_to_bf16(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().oracle_float_to_bf16(_ptr(x), _ptr(out), x.size)
    return out


# -- the two operations -------------------------------------------------------

ELEM_BYTES = {0: 2, 1: 2, 2: 1, 3: 4}


def batching(inp: dict, *, with_gather_idx: bool = False, full_tail: bool = False) -> dict:
    """Run the batching oracle on a ``workloads.make_batching`` dict.
    Returns y (uint8 [Y, H*s]), groupList, sessionIds, microBatchIds, tokenIds,
    expertOffsets, dynamicScale (None unless int8), actualTokenNum (int),
    sortedIndices (slot -> output row or -1) and optionally gather_idx.
    full_tail applies the gather and the id lookups to the masked rows too."""
    Y, H, dt = inp["Y"], inp["H"], inp["tokenDtype"]
    E = inp["expertNum"]
    row_bytes = H * ELEM_BYTES[dt]
    y = np.zeros((Y, row_bytes), dtype=np.uint8)
    gl = np.empty((E, 2), dtype=np.int64)
    sess = np.empty(Y, dtype=np.int32)
    micro = np.empty(Y, dtype=np.int32)
    tok = np.empty(Y, dtype=np.int32)
    eoff = np.empty(Y, dtype=np.int32)
    dyn = np.zeros(Y, dtype=np.float32) if dt == 2 else None
    atn = np.zeros(1, dtype=np.int64)
    sidx = np.empty(Y, dtype=np.int32)
    gidx = np.empty(Y, dtype=np.int32) if with_gather_idx else None
    scales = inp.get("scales")
    scale_stride = 4 if scales is not None else 0
    td = np.ascontiguousarray(inp["token_data"])
    rc = _load().oracle_batching(
        _ptr(np.ascontiguousarray(inp["expert_ids"], dtype=np.int32)), inp["layer_id"],
        _ptr(td), inp["row_stride"], _ptr(scales), scale_stride,
        _ptr(inp["session_in"]), _ptr(inp["micro_in"]), _ptr(inp.get("token_in")),
        E, inp["A"], inp["BS"], inp["K1"], H, dt, inp["layerNum"],
        _ptr(y), _ptr(gl), _ptr(sess), _ptr(micro), _ptr(tok), _ptr(eoff), _ptr(dyn),
        _ptr(atn), _ptr(sidx), _ptr(gidx), int(bool(full_tail)))
    if rc != 0:
        raise ValueError(f"oracle_batching rejected its arguments (code {rc})")
    out = dict(y=y, groupList=gl, sessionIds=sess, microBatchIds=micro, tokenIds=tok,
               expertOffsets=eoff, dynamicScale=dyn, actualTokenNum=int(atn[0]),
               sortedIndices=sidx)
    if with_gather_idx:
        out["gather_idx"] = gidx
    return out


def batching_context(ctx: np.ndarray, token_info: np.ndarray, token_data: np.ndarray, *,
                     expertNum: int, maxOutShape, tokenDtype: int, needSchedule: int,
                     layerNum: int, full_tail: bool = False) -> dict:
    """Run the ScheduleContext batching oracle. ctx: the 1024 context bytes;
    token_info / token_data: host copies of the buffers the context points to.
    full_tail: as for ``batching``, for the slots the context holds."""
    A, BS, K1, H = (int(v) for v in maxOutShape)
    Y, E = A * BS * K1, int(expertNum)
    row_bytes = H * ELEM_BYTES[tokenDtype]
    y = np.zeros((Y, row_bytes), dtype=np.uint8)
    gl = np.empty((E, 2), dtype=np.int64)
    sess, micro, tok, eoff = (np.empty(Y, dtype=np.int32) for _ in range(4))
    dyn = np.zeros(Y, dtype=np.float32) if tokenDtype == 2 else None
    atn = np.zeros(1, dtype=np.int64)
    status = np.zeros(1, dtype=np.int32)
    rc = _load().oracle_batching_context(
        _ptr(np.ascontiguousarray(ctx, dtype=np.uint8)), _ptr(np.ascontiguousarray(token_info)),
        _ptr(np.ascontiguousarray(token_data)), E, A, BS, K1, H, int(tokenDtype), int(needSchedule),
        int(layerNum), _ptr(y), _ptr(gl), _ptr(sess), _ptr(micro), _ptr(tok), _ptr(eoff), _ptr(dyn),
        _ptr(atn), _ptr(status), int(bool(full_tail)))
    if rc != 0:
        raise ValueError(f"oracle_batching_context rejected its arguments (code {rc})")
    return dict(y=y, groupList=gl, sessionIds=sess, microBatchIds=micro, tokenIds=tok,
                expertOffsets=eoff, dynamicScale=dyn, actualTokenNum=int(atn[0]),
                status=int(status[0]))


def permute(tokens: np.ndarray, routing_map: np.ndarray, *, tokenDtype: int, topK: int = 0,
            padded: int = 0, capacity: int = 0) -> dict:
    """Run the permute oracle. tokens: storage [T, H] (uint16 bits or float32);
    routing_map: int8/bool [T, Eu]. Returns permuted (storage [rows, H]),
    sortedIndices and rows (rows written, not padded / kept, padded)."""
    T, H = tokens.shape
    Eu = routing_map.shape[1]
    rows = Eu * capacity if padded else T * topK
    permuted = np.zeros((rows, H), dtype=tokens.dtype)
    si = np.empty(rows, dtype=np.int32)
    rows_out = np.zeros(1, dtype=np.int32)
    rc = _load().oracle_permute(
        _ptr(np.ascontiguousarray(tokens)), _ptr(np.ascontiguousarray(routing_map).view(np.int8)), T, H,
        int(tokenDtype), Eu, int(topK), int(padded), int(capacity), _ptr(permuted), _ptr(si),
        _ptr(rows_out))
    if rc != 0:
        raise ValueError(f"oracle_permute rejected its arguments (code {rc})")
    return dict(permuted=permuted, sortedIndices=si, rows=int(rows_out[0]))


def update_expert(expert_ids: np.ndarray, table: np.ndarray, *, local_rank: int, balance_mode: int,
                  scales: np.ndarray | None = None, scales_dtype: int = 3,
                  threshold: np.ndarray | None = None, active: np.ndarray | None = None) -> dict:
    """Run the MoeUpdateExpert oracle. expert_ids [BS, K] int32/int64; table
    [moeExpertNum, F] int32; scales storage [BS, K]; threshold float32 [K];
    active bool [BS]. Returns balancedExpertIds and balancedActiveMask (or None)."""
    ids = np.ascontiguousarray(expert_ids)
    BS, K = ids.shape
    E, F = table.shape
    out = np.empty_like(ids)
    mask = np.zeros((BS, K), np.uint8) if (scales is not None and threshold is not None) else None
    rc = _load().oracle_update_expert(
        _ptr(ids), ids.dtype.itemsize, _ptr(np.ascontiguousarray(table, dtype=np.int32)),
        _ptr(None if scales is None else np.ascontiguousarray(scales)), int(scales_dtype),
        _ptr(None if threshold is None else np.ascontiguousarray(threshold, dtype=np.float32)),
        _ptr(None if active is None else np.ascontiguousarray(active).astype(np.uint8)),
        BS, K, E, F, int(local_rank), int(balance_mode), _ptr(out), _ptr(mask))
    if rc != 0:
        raise ValueError(f"oracle_update_expert rejected its arguments (code {rc})")
    return dict(balancedExpertIds=out, balancedActiveMask=None if mask is None else mask.astype(bool))


def unpermute(inp: dict) -> dict:
    """Run the unpermute oracle on a ``workloads.make_unpermute_*`` dict (keys
    permuted, sortedIndices, routingMap, probs, permutedRows, H, tokenDtype, n,
    probsDtype, T, Eu, padded). Returns unpermuted (storage dtype [T, H]),
    outIndex, permuteTokenId, permuteProbs (None without probs)."""
    T, H, dt, n = inp["T"], inp["H"], inp["tokenDtype"], inp["n"]
    probs = inp.get("probs")
    pdt = inp["probsDtype"]
    store = np.float32 if dt == 3 else np.uint16
    out = np.zeros((T, H), dtype=store)
    oidx = np.empty(n, dtype=np.int32)
    ptid = np.empty(n, dtype=np.int32)
    pp = None
    if probs is not None:
        pp = np.zeros(n, dtype=np.float32 if pdt == 3 else np.uint16)
    rmap = inp.get("routingMap") if probs is not None else None
    rc = _load().oracle_unpermute(
        _ptr(np.ascontiguousarray(inp["permuted"])), _ptr(np.ascontiguousarray(inp["sortedIndices"])),
        _ptr(None if rmap is None else np.ascontiguousarray(rmap)),
        _ptr(None if probs is None else np.ascontiguousarray(probs)),
        inp["permutedRows"], H, dt, n, pdt, T, inp.get("Eu", 0), int(inp["padded"]),
        _ptr(out), _ptr(oidx), _ptr(ptid), _ptr(pp))
    if rc != 0:
        raise ValueError(f"oracle_unpermute rejected its arguments (code {rc})")
    return dict(unpermuted=out, outIndex=oidx, permuteTokenId=ptid, permuteProbs=pp)
