"""Pins of the ScheduleContext batching oracle.

The context oracle parses the packed ScheduleContext and its token_info /
token_data buffers ("aclnnFfnWorkerBatching", 调用示例). It is pinned to the
page's own example (outputs derived by hand), to the flat-array batching
oracle (already pinned) on the same slots, and to hand-worked cases for
per-block layers, unready blocks and invalid contexts.
"""
import json
import os

import numpy as np
import pytest

import oracle
import workloads as w

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def build(*, sessions, micro, mbs, sel, E, H, dtype, ids, layers=0, flags=1, layerNum=1, A=None,
          BS=None, K1=None, seed=0, expert_num=None, info_size=None, data_size=None,
          data_ptr=0x2000):
    """Host context + buffers for the oracle; the 'addresses' are placeholders
    (the oracle reads the host copies and checks only that they are non-NULL)."""
    blocks = sessions * micro
    per = mbs * sel
    slots = blocks * per
    info = w.make_token_info(sessions=sessions, micro=micro, mbs=mbs, sel=sel, expert_ids=ids,
                             layer_ids=layers, flags=flags)
    es = w.ELEM_BYTES[dtype]
    stride = H * es + (4 if dtype == 2 else 0)
    data = np.random.default_rng(seed).integers(0, 256, size=slots * stride, dtype=np.uint8)
    El = E // max(layerNum, 1)
    ctx = w.pack_schedule_context(sessions=sessions, micro=micro, mbs=mbs, sel=sel,
                                  expert_num=El if expert_num is None else expert_num,
                                  info_ptr=0x1000, info_size=info.size if info_size is None else info_size,
                                  data_ptr=data_ptr,
                                  data_size=data.size if data_size is None else data_size)
    shape = (A or sessions, BS or micro * mbs, K1 or sel, H)
    return ctx, info, data, shape, stride


def run(ctx, info, data, shape, E, dtype, need, layerNum=1):
    return oracle.batching_context(ctx, info, data, expertNum=E, maxOutShape=shape, tokenDtype=dtype,
                                   needSchedule=need, layerNum=layerNum)


@pytest.mark.parametrize("need", [0, 1])
def test_page_example_through_the_context(need):
    """The example program's ScheduleContext: 1 session, 1 micro-batch of 8
    tokens, 9 selected experts, 8 experts, H = 4096 fp16 rows of 0x0001, flag 1,
    layer 0, ids i % 8."""
    g = json.load(open(os.path.join(GOLDEN, "ffnwb_example.json")))
    p = g["inputs"]
    Y = p["A"] * p["BS"] * p["K1"]
    info = w.make_token_info(sessions=1, micro=1, mbs=8, sel=9, expert_ids=np.arange(Y) % 8,
                             layer_ids=0, flags=1)
    data = np.full((Y, p["H"]), 1, dtype=np.uint16).view(np.uint8).reshape(-1)
    ctx = w.pack_schedule_context(sessions=1, micro=1, mbs=8, sel=9, expert_num=8, info_ptr=0x1000,
                                  info_size=info.size, data_ptr=0x2000, data_size=data.size)
    o = run(ctx, info, data, (p["A"], p["BS"], p["K1"], p["H"]), 8, 0, need)
    assert o["status"] == 0
    assert o["groupList"].tolist() == [[e, 9] for e in range(8)]
    assert o["actualTokenNum"] == 72
    assert np.array_equal(o["tokenIds"], [e + 8 * r for e in range(8) for r in range(9)])
    assert np.array_equal(o["expertOffsets"], np.arange(Y) % 9)
    assert np.all(o["y"].view(np.uint16) == 1)
    assert np.all(o["sessionIds"] == 0) and np.all(o["microBatchIds"] == 0)


@pytest.mark.parametrize("dtype,seed", [(0, 1), (1, 2), (2, 3)])
def test_matches_flat_batching_oracle(dtype, seed):
    """With one layer for every block, the context path equals the flat-array
    batching on the same slots, session = block // micro, micro = block % micro,
    token id = slot index."""
    sessions, micro, mbs, sel, E, H = 3, 2, 4, 5, 16, 24
    rng = np.random.default_rng(seed)
    slots = sessions * micro * mbs * sel
    ids = rng.integers(-2, 18, size=slots).astype(np.int32)
    ctx, info, data, shape, stride = build(sessions=sessions, micro=micro, mbs=mbs, sel=sel, E=E,
                                           H=H, dtype=dtype, ids=ids, seed=seed)
    o = run(ctx, info, data, shape, E, dtype, 0)
    blocks = np.arange(slots) // (mbs * sel)
    flat = dict(expert_ids=ids, layer_id=0, token_data=data.reshape(slots, stride), row_stride=stride,
                scales=None, session_in=(blocks // micro).astype(np.int32),
                micro_in=(blocks % micro).astype(np.int32), token_in=None, expertNum=E,
                A=shape[0], BS=shape[1], K1=shape[2], H=H, tokenDtype=dtype, layerNum=1, Y=slots)
    f = oracle.batching(flat)
    for k in ("groupList", "sessionIds", "microBatchIds", "tokenIds", "expertOffsets"):
        assert np.array_equal(o[k], f[k]), k
    assert o["actualTokenNum"] == f["actualTokenNum"]
    U = f["actualTokenNum"]
    assert np.array_equal(o["y"][:U], f["y"][:U])
    if dtype == 2:
        assert np.array_equal(o["dynamicScale"][:U].view(np.uint32), f["dynamicScale"][:U].view(np.uint32))


def test_per_block_layers_by_hand():
    """Two blocks of 2 slots, E_l = 2, layers 1 and 0: keys 1*2+id and 0*2+id.
    Block 0 (layer 1) ids [1, 0] -> keys [3, 2]; block 1 (layer 0) ids [0, 1]
    -> keys [0, 1]. Stable order: slots 2, 3, 1, 0."""
    ids = np.array([1, 0, 0, 1], np.int32)
    ctx, info, data, shape, _ = build(sessions=2, micro=1, mbs=2, sel=1, E=4, H=8, dtype=1, ids=ids,
                                      layers=np.array([1, 0]), layerNum=2)
    o = run(ctx, info, data, shape, 4, 1, 0, layerNum=2)
    assert o["tokenIds"].tolist() == [2, 3, 1, 0]
    assert o["groupList"].tolist() == [[0, 1], [1, 1], [2, 1], [3, 1]]
    assert o["sessionIds"].tolist() == [1, 1, 0, 0]
    # a block whose layer is out of range is masked
    ctx, info, data, shape, _ = build(sessions=2, micro=1, mbs=2, sel=1, E=4, H=8, dtype=1, ids=ids,
                                      layers=np.array([5, 0]), layerNum=2)
    o = run(ctx, info, data, shape, 4, 1, 0, layerNum=2)
    assert o["tokenIds"].tolist() == [2, 3, -1, -1] and o["actualTokenNum"] == 2


def test_unready_blocks_are_masked_with_need_schedule():
    """needSchedule = 1: blocks whose flag is not 1 take no part; status counts
    them. needSchedule = 0 ignores the flags."""
    ids = np.zeros(12, np.int32)
    ctx, info, data, shape, _ = build(sessions=3, micro=1, mbs=2, sel=2, E=1, H=8, dtype=0, ids=ids,
                                      flags=np.array([1, 0, 1]))
    o = run(ctx, info, data, shape, 1, 0, 1)
    assert o["status"] == 1 and o["actualTokenNum"] == 8
    assert o["tokenIds"][:8].tolist() == [0, 1, 2, 3, 8, 9, 10, 11]
    o = run(ctx, info, data, shape, 1, 0, 0)
    assert o["status"] == 0 and o["actualTokenNum"] == 12


@pytest.mark.parametrize("bad", ["too_many_slots", "expert_num", "null_data", "small_info", "small_data",
                                 "zero_sessions", "misaligned_info"])
def test_invalid_context_masks_everything(bad):
    ids = np.zeros(8, np.int32)
    kw = dict(sessions=2, micro=1, mbs=2, sel=2, E=2, H=8, dtype=1, ids=ids)
    if bad == "too_many_slots":
        kw.update(A=1)                      # outputs sized for 4 slots, context has 8
    elif bad == "expert_num":
        kw.update(expert_num=3)
    elif bad == "null_data":
        kw.update(data_ptr=0)
    elif bad == "small_info":
        kw.update(info_size=10)
    elif bad == "small_data":
        kw.update(data_size=16)
    ctx, info, data, shape, _ = build(**kw)
    if bad == "zero_sessions":
        ctx[0:4] = 0
    if bad == "misaligned_info":
        ctx[384:392] = np.array([0x1002], np.uint64).view(np.uint8)
    o = run(ctx, info, data, shape, 2, 1, 0)
    assert o["status"] == -1 and o["actualTokenNum"] == 0
    assert np.all(o["tokenIds"] == -1) and np.all(o["groupList"] == 0)
