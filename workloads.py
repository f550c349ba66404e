"""Seeded synthetic inputs for the MoE expert-grouped token reorder.

This module only draws inputs. It holds none of the arithmetic of the two
operations (no sort of slots by expert, no gather, no weighted reduction), so
the CPU oracle and the CUDA path can both be fed from it without sharing any
of the method's code. Every array is a numpy array in host memory; the same
bytes go to both sides.

Workload recipes follow the shapes and distributions of the pages' workloads:

* batching ("aclnnFfnWorkerBatching", 参数说明 and 调用示例): Y = A*BS*(topK+1)
  slots, each with a local expert id (masked slots carry INT32_MAX), a hidden
  row (fp16/bf16 ~ N(0,1), or int8 with a trailing fp32 dynamic scale), and
  session / micro-batch / token ids;
* unpermute ("MoeTokenUnpermuteWithRoutingMap 算子全解析", 参数说明 and
  补充说明): permutedTokens, sortedIndices, a (tokens, experts) routing map
  and probs, in the padded (expert capacity) or the slot layout.

Random streams are numpy PCG64 generators seeded with [seed, tag, block], so
a value does not depend on how many threads drew it.
"""
from __future__ import annotations

import concurrent.futures as _fut
import os

import numpy as np
import torch

INT32_MAX = 2**31 - 1

DT_F16, DT_BF16, DT_INT8, DT_F32 = 0, 1, 2, 3
DTYPE_NAMES = {DT_F16: "f16", DT_BF16: "bf16", DT_INT8: "int8", DT_F32: "f32"}
ELEM_BYTES = {DT_F16: 2, DT_BF16: 2, DT_INT8: 1, DT_F32: 4}

_ROW_BLOCK = 2048
_TAG_HIDDEN, _TAG_IDS, _TAG_MASK, _TAG_SESS, _TAG_SCALE, _TAG_ROUTE, _TAG_PROBS = range(7)


def _rng(seed: int, *tags: int) -> np.random.Generator:
    return np.random.default_rng([int(seed), *[int(t) for t in tags]])


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def _to_storage(x32: np.ndarray, dtype: int) -> np.ndarray:
    """fp32 samples -> storage of the given float dtype (uint16 bits for 16-bit
    types, float32 itself for fp32). Uses torch's own round-to-nearest-even
    conversion."""
    if dtype == DT_F32:
        return np.ascontiguousarray(x32, dtype=np.float32)
    tdt = torch.float16 if dtype == DT_F16 else torch.bfloat16
    t = torch.from_numpy(np.ascontiguousarray(x32)).to(tdt)
    return t.view(torch.int16).numpy().view(np.uint16)


def normal_rows(rows: int, H: int, dtype: int, seed: int, tag: int = _TAG_HIDDEN) -> np.ndarray:
    """rows x H values ~ N(0,1) in the given float dtype (uint16 bits or float32).
    Drawn block by block in parallel; block b uses stream [seed, tag, b]."""
    out = np.empty((rows, H), dtype=np.float32 if dtype == DT_F32 else np.uint16)
    nblk = (rows + _ROW_BLOCK - 1) // _ROW_BLOCK

    def fill(b: int) -> None:
        r0 = b * _ROW_BLOCK
        r1 = min(rows, r0 + _ROW_BLOCK)
        x = _rng(seed, tag, b).standard_normal((r1 - r0, H), dtype=np.float32)
        out[r0:r1] = _to_storage(x, dtype)

    if nblk <= 1:
        for b in range(nblk):
            fill(b)
    else:
        with _fut.ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(fill, range(nblk)))
    return out


def zipf_ids(n: int, num: int, s: float, rng: np.random.Generator) -> np.ndarray:
    """n draws of a Zipf(s) law over ranks 1..num, returned as rank-1 (id 0 is
    the most frequent). Inverse-CDF sampling."""
    w = np.arange(1, num + 1, dtype=np.float64) ** (-float(s))
    cdf = np.cumsum(w) / w.sum()
    u = rng.random(n)
    return np.minimum(np.searchsorted(cdf, u, side="right"), num - 1).astype(np.int32)


# ---------------------------------------------------------------------------
# Batching inputs
# ---------------------------------------------------------------------------

def make_batching(*, A: int, BS: int, K1: int, E: int, H: int, dtype: int, layerNum: int = 1,
                  layer_id: int = 0, ids: str = "uniform", zipf_s: float = 1.1, mask: float = 0.1,
                  session: int = 2, micro: int = 4, token_ids: bool = True, seed: int = 0,
                  separate_scales: bool = False) -> dict:
    """Flat-tensor inputs of one batching call.

    expert_ids: local ids in [0, E/layerNum); masked slots carry INT32_MAX.
    token_data: uint8 [Y, row_stride]; fp16/bf16 rows hold H values, int8 rows
    hold H int8 values followed by a little-endian fp32 dynamic scale
    (row_stride = H + 4) unless separate_scales, in which case the scales are a
    separate float32 [Y] array and row_stride = H.
    """
    Y = A * BS * K1
    L = max(layerNum, 1)
    El = E // L
    rng_ids = _rng(seed, _TAG_IDS)
    if ids == "uniform":
        expert = rng_ids.integers(0, El, size=Y, dtype=np.int64).astype(np.int32)
    elif ids == "zipf":
        expert = zipf_ids(Y, El, zipf_s, rng_ids)
    elif ids == "mod":
        expert = (np.arange(Y) % El).astype(np.int32)
    else:
        raise ValueError(ids)
    if mask > 0:
        m = _rng(seed, _TAG_MASK).random(Y) < mask
        expert = np.where(m, np.int32(INT32_MAX), expert).astype(np.int32)

    scales = None
    if dtype == DT_INT8:
        rng_h = _rng(seed, _TAG_HIDDEN)
        data = rng_h.integers(-127, 128, size=(Y, H), dtype=np.int16).astype(np.int8)
        sc = _rng(seed, _TAG_SCALE).lognormal(mean=-4.0, sigma=0.5, size=Y).astype(np.float32)
        if separate_scales:
            token_data = data.view(np.uint8).copy()
            scales = sc
            row_stride = H
        else:
            token_data = np.empty((Y, H + 4), dtype=np.uint8)
            token_data[:, :H] = data.view(np.uint8)
            token_data[:, H:] = sc.view(np.uint8).reshape(Y, 4)
            row_stride = H + 4
    else:
        token_data = normal_rows(Y, H, dtype, seed).view(np.uint8).reshape(Y, H * ELEM_BYTES[dtype])
        row_stride = H * ELEM_BYTES[dtype]

    rng_s = _rng(seed, _TAG_SESS)
    session_in = rng_s.integers(0, session, size=Y, dtype=np.int64).astype(np.int32)
    micro_in = rng_s.integers(0, micro, size=Y, dtype=np.int64).astype(np.int32)
    token_in = np.arange(Y, dtype=np.int32) if token_ids else None
    return dict(expert_ids=expert, layer_id=int(layer_id), token_data=token_data,
                row_stride=int(row_stride), scales=scales, session_in=session_in,
                micro_in=micro_in, token_in=token_in, expertNum=int(E), A=int(A), BS=int(BS),
                K1=int(K1), H=int(H), tokenDtype=int(dtype), layerNum=int(layerNum), Y=int(Y))


# ---------------------------------------------------------------------------
# Unpermute inputs
# ---------------------------------------------------------------------------

def _softmax_rows(logits: np.ndarray, keep: np.ndarray) -> np.ndarray:
    """Softmax in float64 over the kept entries of each row, 0 elsewhere."""
    z = np.where(keep, logits, -np.inf)
    zmax = np.max(z, axis=1, keepdims=True)
    zmax = np.where(np.isfinite(zmax), zmax, 0.0)
    e = np.where(keep, np.exp(z - zmax), 0.0)
    s = e.sum(axis=1, keepdims=True)
    return np.where(s > 0, e / np.where(s > 0, s, 1.0), 0.0)


def make_unpermute_topk(*, T: int, k: int, Eu: int, H: int, dtype: int, probs_dtype: int | None,
                        choices=(6, 7, 8), seed: int = 1, rows: int | None = None) -> dict:
    """Not-padded (slot layout) inputs: each token picks n ~ U(choices)
    experts, the top-n of N(0,1) logits (ties to the lower expert id).
    permutedTokens rows are the expert-major order of the (token, expert)
    pairs, as the permute step that precedes the unpermute lays them out;
    sortedIndices[t*k + j] = row of t's j-th chosen expert (ascending expert
    id), -1 for unused slots. probs = softmax over the chosen experts, 0
    elsewhere (None -> no probs)."""
    rng = _rng(seed, _TAG_ROUTE)
    nsel = rng.choice(np.asarray(choices, dtype=np.int64), size=T)
    logits = rng.standard_normal((T, Eu))
    order = np.argsort(-logits, axis=1, kind="stable")
    keep = np.zeros((T, Eu), dtype=bool)
    for t in range(T):
        keep[t, order[t, :nsel[t]]] = True
    routing = keep.astype(np.int8)
    # rows: pairs ordered by (expert, token)
    tt, ee = np.nonzero(keep)                      # row-major: by token, then expert
    pair_order = np.lexsort((tt, ee))              # by expert, then token
    row_of_pair = np.empty(len(tt), dtype=np.int64)
    row_of_pair[pair_order] = np.arange(len(tt))
    sorted_idx = np.full(T * k, -1, dtype=np.int32)
    # a token's pairs come in ascending expert id: slot j of the token is its
    # j-th pair
    j = np.arange(len(tt)) - np.searchsorted(tt, tt)
    sorted_idx[tt * k + j] = row_of_pair
    nrows = T * k if rows is None else rows
    permuted = normal_rows(nrows, H, dtype, seed)
    probs = None
    if probs_dtype is not None:
        p64 = _softmax_rows(logits, keep)
        probs = _to_storage(p64.astype(np.float32), probs_dtype)
    return dict(permuted=permuted, sortedIndices=sorted_idx, routingMap=routing, probs=probs,
                permutedRows=int(nrows), H=int(H), tokenDtype=int(dtype), n=int(T * k),
                probsDtype=int(probs_dtype if probs_dtype is not None else dtype), T=int(T),
                Eu=int(Eu), padded=0)


def make_unpermute_padded(*, T: int, Eu: int, k: int, H: int, dtype: int, probs_dtype: int | None,
                          mult: int = 37, seed: int = 3, capacity: int | None = None) -> dict:
    """Padded (expert capacity) inputs with balanced routing: token t goes to
    experts (mult*t + (Eu/k)*j) mod Eu for j < k, so with Eu a power of two,
    mult odd and T a multiple of Eu every expert gets T*k/Eu tokens.
    sortedIndices[e*capacity + r] = r-th smallest token routed to e, -1 in the
    expert's unused slots; capacity = the largest expert load, or the given
    capacity when larger (slack slots). probs = Dirichlet(1) over the token's k
    experts (normalised Exp(1) draws)."""
    step = Eu // k
    routing = np.zeros((T, Eu), dtype=np.int8)
    t = np.arange(T)
    cols = np.stack([(mult * t + step * j) % Eu for j in range(k)], axis=1)  # [T, k]
    routing[t[:, None], cols] = 1
    counts = routing.sum(axis=0)
    cap = max(int(counts.max()), int(capacity or 0))
    sorted_idx = np.full(Eu * cap, -1, dtype=np.int32)
    e_idx, t_idx = np.nonzero(routing.T)            # expert-major, tokens ascending
    first = np.searchsorted(e_idx, np.arange(Eu))   # each expert's first pair
    sorted_idx[e_idx * cap + (np.arange(len(e_idx)) - first[e_idx])] = t_idx
    permuted = normal_rows(Eu * cap, H, dtype, seed)
    probs = None
    if probs_dtype is not None:
        # Exp(1) draws for the token's k experts only, normalised (Dirichlet(1))
        g = _rng(seed, _TAG_PROBS).exponential(1.0, size=(T, k))
        p = np.zeros((T, Eu), dtype=np.float32)
        p[t[:, None], cols] = (g / g.sum(axis=1, keepdims=True)).astype(np.float32)
        probs = _to_storage(p, probs_dtype)
    return dict(permuted=permuted, sortedIndices=sorted_idx, routingMap=routing, probs=probs,
                permutedRows=int(Eu * cap), H=int(H), tokenDtype=int(dtype), n=int(Eu * cap),
                probsDtype=int(probs_dtype if probs_dtype is not None else dtype), T=int(T),
                Eu=int(Eu), padded=1, capacity=cap)


def make_roundtrip_probs(*, T: int, k: int, slot_unmasked: np.ndarray, probs_dtype: int,
                         seed: int = 4) -> tuple[np.ndarray, np.ndarray]:
    """Routing map and probs of the round trip, with one column per slot of a
    token: routingMap[t, j] = slot t*k+j is unmasked; probs = softmax of
    N(0,1) logits over the k slots of the token."""
    routing = slot_unmasked.reshape(T, k).astype(np.int8)
    logits = _rng(seed, _TAG_PROBS).standard_normal((T, k))
    p64 = _softmax_rows(logits, np.ones((T, k), dtype=bool))
    return routing, _to_storage(p64.astype(np.float32), probs_dtype)


# ---------------------------------------------------------------------------
# The five workloads (sizes and distributions of the pages' workloads)
# ---------------------------------------------------------------------------

BATCHING_TINY = dict(A=2, BS=8, K1=3, E=8, H=128, dtype=DT_F16, layerNum=1, layer_id=0,
                     ids="uniform", mask=0.10, session=2, micro=4, token_ids=True, seed=0)
BATCHING_INT8_DECODE = dict(A=64, BS=32, K1=9, E=256, H=7168, dtype=DT_INT8, layerNum=1,
                            layer_id=0, ids="zipf", zipf_s=1.1, mask=0.15, session=64,
                            micro=64, token_ids=True, seed=2)
UNPERMUTE_TOPK = dict(T=4096, k=8, Eu=64, H=4096, dtype=DT_BF16, probs_dtype=DT_BF16, seed=1)
UNPERMUTE_PADDED = dict(T=16384, Eu=128, k=4, H=4096, dtype=DT_F16, probs_dtype=DT_F32, seed=3)
# the same routing with capacity twice the load: half of the expert slots are padding
UNPERMUTE_PADDED_SLACK = dict(UNPERMUTE_PADDED, capacity=1024)
# a decode-sized step: 64 tokens, each routed to 6-8 of 64 experts, H = 7168 bf16
UNPERMUTE_DECODE = dict(T=64, k=8, Eu=64, H=7168, dtype=DT_BF16, probs_dtype=DT_BF16, seed=7)
ROUNDTRIP_BATCHING = dict(A=256, BS=64, K1=9, E=1024, H=7168, dtype=DT_BF16, layerNum=4,
                          layer_id=2, ids="zipf", zipf_s=1.2, mask=0.05, session=256, micro=64,
                          token_ids=True, seed=4)
ROUNDTRIP_PROBS_DTYPE = DT_BF16

# Shapes that take the library's other paths, for measuring those kernels:
# the round trip's slots and keys with 16-byte rows (its index kernels alone);
# a routing map of more than 4M entries (the three-kernel maskedSelect); rows
# that are not whole 16-byte vectors (the element-wise gather-reduce); and a
# padded sort of more than 2^22 keys (LSD passes, then the row pointers).
ROUNDTRIP_BATCHING_INDEX = dict(ROUNDTRIP_BATCHING, H=8)
UNPERMUTE_LARGE_MAP = dict(T=32768, k=8, Eu=256, H=512, dtype=DT_BF16, probs_dtype=DT_BF16, seed=8)
UNPERMUTE_ODD_H = dict(UNPERMUTE_TOPK, H=4095)
UNPERMUTE_PADDED_LSD = dict(T=1 << 22, Eu=2, k=1, H=8, dtype=DT_F16, probs_dtype=DT_F32, seed=9)


# ---------------------------------------------------------------------------
# ScheduleContext inputs ("aclnnFfnWorkerBatching", 调用示例: the packed
# 1024-byte ScheduleContext and the FfnArea token_info / token_data buffers)
# ---------------------------------------------------------------------------

CTX_BYTES = 1024
CTX_FFN_OFFSET = 384  # CommonArea 128 + ControlArea 128 + AttentionArea 128


def make_token_info(*, sessions: int, micro: int, mbs: int, sel: int, expert_ids: np.ndarray,
                    layer_ids, flags) -> np.ndarray:
    """token_info_buf bytes: per (session, micro-batch) block, sessions outer,
    i32 flag, i32 layer_id, then mbs*sel i32 expert ids (FfnDataDesc)."""
    blocks = sessions * micro
    per = mbs * sel
    ids = np.asarray(expert_ids, dtype=np.int32).reshape(blocks, per)
    out = np.empty((blocks, 2 + per), dtype=np.int32)
    out[:, 0] = np.broadcast_to(np.asarray(flags, dtype=np.int32), (blocks,))
    out[:, 1] = np.broadcast_to(np.asarray(layer_ids, dtype=np.int32), (blocks,))
    out[:, 2:] = ids
    return out.view(np.uint8).reshape(-1)


def pack_schedule_context(*, sessions: int, micro: int, mbs: int, sel: int, expert_num: int,
                          info_ptr: int, info_size: int, data_ptr: int, data_size: int,
                          run_flag: int = 1) -> np.ndarray:
    """The packed ScheduleContext (1024 bytes) with the CommonArea counts and
    the FfnArea token_info / token_data buffer addresses and sizes."""
    ctx = np.zeros(CTX_BYTES, dtype=np.uint8)
    common = np.array([sessions, micro, mbs, sel, expert_num, 0, 0, 0], dtype=np.uint32)
    ctx[0:32] = common.view(np.uint8)
    ctx[128:132] = np.array([run_flag], dtype=np.int32).view(np.uint8)
    ffn = np.array([info_ptr, info_size, data_ptr, data_size], dtype=np.uint64)
    ctx[CTX_FFN_OFFSET:CTX_FFN_OFFSET + 32] = ffn.view(np.uint8)
    return ctx


# ---------------------------------------------------------------------------
# MoeUpdateExpert inputs ("MoeUpdateExpert", 参数说明 and 约束说明)
# ---------------------------------------------------------------------------

def make_eplb_table(*, moe_expert_num: int, world_size: int, place_per_rank: int,
                    seed: int = 0) -> np.ndarray:
    """eplbTable [moeExpertNum, F] int32: column 0 the instance count (1 ..
    worldSize), then the instance ids; every one of the worldSize *
    place_per_rank instances hosts one logical expert (ids not repeated)."""
    rng = _rng(seed, _TAG_ROUTE)
    n_inst = world_size * place_per_rank
    assert n_inst >= moe_expert_num
    perm = rng.permutation(n_inst)
    rows = [[int(perm[e])] for e in range(moe_expert_num)]
    for inst in perm[moe_expert_num:]:
        e = int(rng.integers(0, moe_expert_num))
        if len(rows[e]) < world_size:
            rows[e].append(int(inst))
    F = max(len(r) for r in rows) + 1
    table = np.zeros((moe_expert_num, F), dtype=np.int32)
    for e, r in enumerate(rows):
        table[e, 0] = len(r)
        table[e, 1:1 + len(r)] = r
    return table


def make_update_expert(*, BS: int, K: int, moe_expert_num: int, world_size: int,
                       place_per_rank: int, scales_dtype: int = DT_F32, id_dtype=np.int32,
                       active_frac: float = 0.8, seed: int = 0) -> dict:
    """Each token picks K distinct experts; scales descend within a token
    (sorted softmax of N(0,1) logits); thresholds [K] float32; activeMask is a
    prefix of trues."""
    rng = _rng(seed, _TAG_IDS)
    ids = np.stack([rng.choice(moe_expert_num, size=K, replace=False) for _ in range(BS)]).astype(id_dtype)
    logits = _rng(seed, _TAG_PROBS).standard_normal((BS, K))
    p = np.exp(logits - logits.max(axis=1, keepdims=True))
    p = -np.sort(-(p / p.sum(axis=1, keepdims=True)), axis=1)
    scales = _to_storage(p.astype(np.float32), scales_dtype)
    threshold = np.full(K, 0.5 / K, dtype=np.float32)
    active = np.zeros(BS, dtype=bool)
    active[:int(round(active_frac * BS))] = True
    table = make_eplb_table(moe_expert_num=moe_expert_num, world_size=world_size,
                            place_per_rank=place_per_rank, seed=seed)
    return dict(expert_ids=ids, table=table, scales=scales, scales_dtype=scales_dtype,
                threshold=threshold, active=active, world_size=world_size)


# The page's maxima (BS 512, K 16) with 512 logical experts over 128 ranks x 8
# instances: 1024 instances, so experts are replicated up to the rank count.
UPDATE_EXPERT = dict(BS=512, K=16, moe_expert_num=512, world_size=128, place_per_rank=8,
                     scales_dtype=DT_BF16, seed=6)
