"""Pins of the batching oracle's full-tail option: the formulas of
"aclnnFfnWorkerBatching", 计算公式 (y[i] = token_data[gather_idx[i]]) and the
id lookup of 功能说明 step 3, applied to every row, the masked tail included.

The pins do not go through the oracle's own sort: they rebuild gather_idx with
numpy's stable argsort of the keys and index the inputs with it."""
import numpy as np
import pytest

import oracle
import workloads as w

from test_oracle_context_pins import build


def keys_of(inp):
    El = inp["expertNum"] // max(inp["layerNum"], 1)
    ids = inp["expert_ids"].astype(np.int64)
    return np.where((ids >= 0) & (ids < El), inp["layer_id"] * El + ids, inp["expertNum"])


@pytest.mark.parametrize("dt,seed,sep", [(0, 0, False), (1, 1, False), (2, 2, False), (2, 3, True)])
def test_every_row_follows_the_library_argsort(dt, seed, sep):
    inp = w.make_batching(A=3, BS=8, K1=5, E=24, H=40, dtype=dt, layerNum=2, layer_id=1, mask=0.3,
                          session=3, micro=5, seed=seed, separate_scales=sep)
    o = oracle.batching(inp, full_tail=True)
    gidx = np.argsort(keys_of(inp), kind="stable")
    row_bytes = inp["H"] * w.ELEM_BYTES[dt]
    td = inp["token_data"].reshape(inp["Y"], -1)
    assert np.array_equal(o["y"], td[gidx, :row_bytes])
    assert np.array_equal(o["sessionIds"], inp["session_in"][gidx])
    assert np.array_equal(o["microBatchIds"], inp["micro_in"][gidx])
    assert np.array_equal(o["tokenIds"], inp["token_in"][gidx])
    if dt == 2:
        sc = inp["scales"] if sep else td[:, row_bytes:row_bytes + 4].copy().view(np.float32).reshape(-1)
        assert np.array_equal(o["dynamicScale"].view(np.uint32), sc[gidx].view(np.uint32))
    U = o["actualTokenNum"]
    assert 0 < U < inp["Y"]
    assert (o["expertOffsets"][U:] == -1).all()


def test_prefix_and_counts_match_the_default_mode():
    inp = w.make_batching(A=2, BS=16, K1=3, E=8, H=16, dtype=1, mask=0.25, seed=4, token_ids=False)
    a = oracle.batching(inp)
    b = oracle.batching(inp, full_tail=True)
    U = a["actualTokenNum"]
    assert b["actualTokenNum"] == U
    for k in ("groupList", "expertOffsets", "sortedIndices"):
        assert np.array_equal(a[k], b[k]), k
    for k in ("sessionIds", "microBatchIds", "tokenIds"):
        assert np.array_equal(a[k][:U], b[k][:U])
        assert (a[k][U:] == -1).all()
    assert np.array_equal(a["y"][:U], b["y"][:U])
    assert not a["y"][U:].any()                       # untouched (zeros) by default
    # token ids default to the slot index: the tail rows hold the masked slots ascending
    masked = np.flatnonzero(keys_of(inp) == inp["expertNum"])
    assert np.array_equal(b["tokenIds"][U:], masked)


def test_full_tail_rows_are_a_permutation_of_the_inputs():
    inp = w.make_batching(A=4, BS=4, K1=4, E=16, H=8, dtype=0, mask=0.5, seed=5)
    o = oracle.batching(inp, full_tail=True)
    td = inp["token_data"].reshape(inp["Y"], -1)
    got = sorted(map(bytes, o["y"]))
    want = sorted(map(bytes, td[:, :16]))
    assert got == want


@pytest.mark.parametrize("dt", [1, 2])
def test_context_tail_stops_at_the_context_slots(dt):
    """4 sessions x 2 micro x 4 tokens x 2 slots = 64 slots in a Y = 96 output:
    masked slots of the context are gathered with their ids; rows for the 32
    slots the context does not have stay untouched, ids -1."""
    rng = np.random.default_rng(6)
    ids = rng.integers(-1, 10, size=64).astype(np.int32)
    ctx, info, data, shape, stride = build(sessions=4, micro=2, mbs=4, sel=2, E=8, H=16, dtype=dt,
                                           ids=ids, A=6, seed=7)
    o = oracle.batching_context(ctx, info, data, expertNum=8, maxOutShape=shape, tokenDtype=dt,
                                needSchedule=0, layerNum=1, full_tail=True)
    key = np.where((ids >= 0) & (ids < 8), ids, 8)
    gidx = np.argsort(key, kind="stable")
    rows = data.reshape(64, stride)
    rb = 16 * w.ELEM_BYTES[dt]
    assert np.array_equal(o["y"][:64], rows[gidx, :rb])
    assert not o["y"][64:].any()
    assert np.array_equal(o["tokenIds"][:64], gidx)
    assert np.array_equal(o["sessionIds"][:64], gidx // 16)          # 16 slots per session
    assert np.array_equal(o["microBatchIds"][:64], (gidx // 8) % 2)  # 8 slots per block
    assert (o["tokenIds"][64:] == -1).all() and (o["expertOffsets"][o["actualTokenNum"]:] == -1).all()
    if dt == 2:
        assert np.array_equal(o["dynamicScale"][:64].view(np.uint32),
                              rows[gidx, rb:rb + 4].copy().view(np.uint32).reshape(-1))


def test_invalid_context_gathers_nothing():
    ids = np.zeros(16, np.int32)
    ctx, info, data, shape, _ = build(sessions=2, micro=1, mbs=4, sel=2, E=2, H=8, dtype=1, ids=ids,
                                      expert_num=3)
    o = oracle.batching_context(ctx, info, data, expertNum=2, maxOutShape=shape, tokenDtype=1,
                                needSchedule=0, layerNum=1, full_tail=True)
    assert o["status"] == -1 and o["actualTokenNum"] == 0
    assert not o["y"].any() and (o["tokenIds"] == -1).all()
