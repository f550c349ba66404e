"""The batching's full-tail option on the GPU vs the oracle: 计算公式 of
"aclnnFfnWorkerBatching" applied to every row, the masked tail included
(flat arrays and ScheduleContext). Rows, ids and scales are compared byte for
byte; rows that must stay untouched are checked against a fill pattern."""
import numpy as np
import pytest
import torch

import oracle
import workloads as w

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import unpermute_stable_counting_gb300 as usc  # noqa: E402

from _gpu_util import dev, to_dev  # noqa: E402
from test_gpu_context import device_context  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def filled_outputs(Y, H, E, dt):
    out = usc.batching_outputs(Y, H, E, dt, dev(), with_sorted_indices=True)
    out["y"].view(torch.uint8).fill_(0xA5)
    if out["dynamicScale"] is not None:
        out["dynamicScale"].view(torch.uint8).fill_(0xA5)
    return out


def run_flat(inp, full_tail):
    Y, H, E, dt = inp["Y"], inp["H"], inp["expertNum"], inp["tokenDtype"]
    out = filled_outputs(Y, H, E, dt)
    usc.ffnwb_batching(to_dev(inp["expert_ids"]), to_dev(inp["token_data"]), to_dev(inp["session_in"]),
                       to_dev(inp["micro_in"]), expert_num=E,
                       max_out_shape=(inp["A"], inp["BS"], inp["K1"], H), token_dtype=dt,
                       layer_num=inp["layerNum"], layer_id=inp["layer_id"],
                       token_ids=to_dev(inp["token_in"]) if inp.get("token_in") is not None else None,
                       scales=to_dev(inp["scales"]) if inp.get("scales") is not None else None,
                       token_row_stride=inp["row_stride"], with_sorted_indices=True, out=out,
                       full_tail=full_tail)
    torch.cuda.synchronize()
    return out


def check(out, ref, Y, rows_written):
    """rows_written: rows the oracle wrote (the rest must keep the fill)."""
    y = out["y"].contiguous().view(torch.uint8).cpu().numpy().reshape(Y, -1)
    assert np.array_equal(y[:rows_written], ref["y"][:rows_written])
    assert (y[rows_written:] == 0xA5).all()
    assert int(out["actualTokenNum"][0]) == ref["actualTokenNum"]
    for k in ("groupList", "sessionIds", "microBatchIds", "tokenIds", "expertOffsets"):
        assert np.array_equal(out[k].cpu().numpy(), ref[k]), k
    if out["dynamicScale"] is not None:
        d = out["dynamicScale"].cpu().numpy().view(np.uint32)
        assert np.array_equal(d[:rows_written], ref["dynamicScale"][:rows_written].view(np.uint32))
        assert (d[rows_written:] == 0xA5A5A5A5).all()


@pytest.mark.parametrize("dt,sep,mask,seed", [(0, False, 0.3, 0), (1, False, 0.05, 1), (2, False, 0.2, 2),
                                              (2, True, 0.2, 3), (1, False, 1.0, 4), (1, False, 0.0, 5)])
def test_flat_full_tail(dt, sep, mask, seed):
    inp = w.make_batching(A=5, BS=16, K1=9, E=96, H=200 if dt != 2 else 320, dtype=dt, layerNum=3,
                          layer_id=1, ids="zipf", mask=mask, session=5, micro=16, seed=seed,
                          separate_scales=sep)
    ref = oracle.batching(inp, full_tail=True)
    out = run_flat(inp, True)
    check(out, ref, inp["Y"], inp["Y"])
    assert np.array_equal(out["sortedIndices"].cpu().numpy(), ref["sortedIndices"])
    # the default on the same inputs leaves the tail alone
    ref0 = oracle.batching(inp)
    out0 = run_flat(inp, False)
    check(out0, ref0, inp["Y"], ref0["actualTokenNum"])


def test_flat_full_tail_int8_decode_shape():
    inp = w.make_batching(**w.BATCHING_INT8_DECODE)
    ref = oracle.batching(inp, full_tail=True)
    check(run_flat(inp, True), ref, inp["Y"], inp["Y"])


@pytest.mark.parametrize("dtype,need,seed", [(1, 0, 1), (2, 0, 2), (0, 1, 3)])
def test_context_full_tail(dtype, need, seed):
    """8 x 4 blocks of 16 x 9 slots in outputs with two more sessions of rows:
    the context's masked slots (bad ids, out-of-range layers, blocks not
    ready) are gathered, the rows past its slots keep the fill."""
    sessions, micro, mbs, sel, H, L = 8, 4, 16, 9, 136 if dtype != 2 else 128, 2
    E = 64 * L
    rng = np.random.default_rng(seed)
    ids = rng.integers(-1, 64 + 3, size=sessions * micro * mbs * sel).astype(np.int32)
    lay = rng.integers(0, L + 1, size=sessions * micro)
    flags = (rng.random(sessions * micro) < 0.8).astype(np.int32) if need else 1
    ctx_d, host, keep = device_context(sessions=sessions, micro=micro, mbs=mbs, sel=sel, E=E, H=H,
                                       dtype=dtype, ids=ids, layers=lay, flags=flags, layerNum=L,
                                       seed=seed)
    shape = (sessions + 2, micro * mbs, sel, H)
    Y = shape[0] * shape[1] * shape[2]
    slots = sessions * micro * mbs * sel
    out = filled_outputs(Y, H, E, dtype)
    out["scheduleStatus"] = torch.zeros(1, dtype=torch.int32, device=dev())
    usc.ffnwb_batching_context(ctx_d, expert_num=E, max_out_shape=shape, token_dtype=dtype, layer_num=L,
                               need_schedule=need, wait_timeout_us=20_000, out=out, full_tail=True)
    torch.cuda.synchronize()
    ref = oracle.batching_context(*host, expertNum=E, maxOutShape=shape, tokenDtype=dtype,
                                  needSchedule=need, layerNum=L, full_tail=True)
    assert int(out["scheduleStatus"][0]) == ref["status"]
    check(out, ref, Y, slots)


def test_context_default_still_leaves_the_tail():
    ids = np.random.default_rng(9).integers(-2, 40, size=4 * 2 * 8 * 3).astype(np.int32)
    ctx_d, host, keep = device_context(sessions=4, micro=2, mbs=8, sel=3, E=32, H=64, dtype=1, ids=ids)
    shape = (5, 16, 3, 64)
    Y = 5 * 16 * 3
    out = filled_outputs(Y, 64, 32, 1)
    usc.ffnwb_batching_context(ctx_d, expert_num=32, max_out_shape=shape, token_dtype=1, out=out)
    torch.cuda.synchronize()
    ref = oracle.batching_context(*host, expertNum=32, maxOutShape=shape, tokenDtype=1, needSchedule=0,
                                  layerNum=1)
    check(out, ref, Y, ref["actualTokenNum"])


def test_full_size_full_tail_sampled():
    """The round trip's batching (Y = 147456, H = 7168 bf16, 5% masked) with the
    option: every id output bit-exact, and 4096 sampled rows of y (all masked
    rows among them) equal to the source row of their slot."""
    inp = w.make_batching(**w.ROUNDTRIP_BATCHING)
    Y, H = inp["Y"], inp["H"]
    ref = oracle.batching(inp, full_tail=True, with_gather_idx=True)
    out = run_flat(inp, True)
    for k in ("groupList", "sessionIds", "microBatchIds", "tokenIds", "expertOffsets"):
        assert np.array_equal(out[k].cpu().numpy(), ref[k]), k
    U = ref["actualTokenNum"]
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([rng.choice(U, 2048, replace=False), np.arange(U, Y)[:2048]]))
    y = out["y"].view(torch.uint8).reshape(Y, -1)[torch.from_numpy(rows).to(dev())].cpu().numpy()
    td = inp["token_data"].reshape(Y, -1)
    assert np.array_equal(y, td[ref["gather_idx"][rows], :2 * H])
