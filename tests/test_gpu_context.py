"""Batching from a ScheduleContext on the GPU vs the context oracle.

The context and its buffers are built in device memory the way the batching
page's example program lays them out; the kernels read the context on the
device. With needSchedule = 1 the kernel waits, bounded by a timeout, for
each block's flag: a flag that nothing sets makes the wait run out, the
block is masked and the status word counts it; the GPU stays usable.
"""
import time

import numpy as np
import pytest
import torch

import oracle
import workloads as w

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import unpermute_stable_counting_gb300 as usc  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def device_context(*, sessions, micro, mbs, sel, E, H, dtype, ids, layers=0, flags=1, layerNum=1,
                   seed=0, data=None, base_offset=0):
    """Device buffers + a device copy of the packed context pointing at them
    (the token rows base_offset bytes into their allocation).
    Returns (ctx_dev, host pieces for the oracle, keep-alive tensors)."""
    dev = torch.device("cuda:0")
    info = w.make_token_info(sessions=sessions, micro=micro, mbs=mbs, sel=sel, expert_ids=ids,
                             layer_ids=layers, flags=flags)
    slots = sessions * micro * mbs * sel
    stride = H * w.ELEM_BYTES[dtype] + (4 if dtype == 2 else 0)
    if data is None:
        data = np.random.default_rng(seed).integers(0, 256, size=slots * stride, dtype=np.uint8)
    info_d = torch.from_numpy(info).to(dev)
    padded = np.zeros(data.size + base_offset, dtype=np.uint8)
    padded[base_offset:] = data
    data_d = torch.from_numpy(padded).to(dev)
    El = E // max(layerNum, 1)
    ctx = w.pack_schedule_context(sessions=sessions, micro=micro, mbs=mbs, sel=sel, expert_num=El,
                                  info_ptr=info_d.data_ptr(), info_size=info.size,
                                  data_ptr=data_d.data_ptr() + base_offset, data_size=data.size)
    ctx_d = torch.from_numpy(ctx).to(dev)
    return ctx_d, (ctx, info, data), (info_d, data_d)


def run_both(ctx_d, host, shape, E, dtype, need, layerNum=1, timeout_us=1_000_000):
    got = usc.ffnwb_batching_context(ctx_d, expert_num=E, max_out_shape=shape, token_dtype=dtype,
                                     layer_num=layerNum, need_schedule=need,
                                     wait_timeout_us=timeout_us)
    torch.cuda.synchronize()
    ref = oracle.batching_context(*host, expertNum=E, maxOutShape=shape, tokenDtype=dtype,
                                  needSchedule=need, layerNum=layerNum)
    Y = shape[0] * shape[1] * shape[2]
    g = {k: v.cpu().numpy() for k, v in got.items() if v is not None and k != "y"}
    U = ref["actualTokenNum"]
    assert int(g["actualTokenNum"][0]) == U
    assert int(g["scheduleStatus"][0]) == ref["status"]
    for k in ("groupList", "sessionIds", "microBatchIds", "tokenIds", "expertOffsets"):
        assert np.array_equal(g[k], ref[k]), k
    y = got["y"].contiguous().view(torch.uint8).cpu().numpy().reshape(Y, -1)
    assert np.array_equal(y[:U], ref["y"][:U])
    if dtype == 2:
        assert np.array_equal(g["dynamicScale"][:U].view(np.uint32), ref["dynamicScale"][:U].view(np.uint32))
    return g, ref


@pytest.mark.parametrize("need", [0, 1])
def test_page_example_context(need):
    Y, H = 72, 4096
    data = np.full((Y, H), 1, dtype=np.uint16).view(np.uint8).reshape(-1)
    ctx_d, host, keep = device_context(sessions=1, micro=1, mbs=8, sel=9, E=8, H=H, dtype=0,
                                       ids=np.arange(Y) % 8, data=data)
    g, _ = run_both(ctx_d, host, (1, 8, 9, H), 8, 0, need)
    assert g["groupList"].tolist() == [[e, 9] for e in range(8)]
    assert int(g["actualTokenNum"][0]) == 72 and int(g["scheduleStatus"][0]) == 0


@pytest.mark.parametrize("dtype,layers,L,seed", [(0, 0, 1, 1), (1, "mixed", 4, 2), (2, "mixed", 2, 3),
                                                 (1, 0, 1, 4)])
def test_random_contexts(dtype, layers, L, seed):
    sessions, micro, mbs, sel, H = 8, 4, 16, 9, 136 if dtype != 2 else 128
    E = 64 * L
    rng = np.random.default_rng(seed)
    slots = sessions * micro * mbs * sel
    ids = rng.integers(-1, 64 + 2, size=slots).astype(np.int32)
    lay = rng.integers(0, L + 1, size=sessions * micro) if layers == "mixed" else 0
    ctx_d, host, keep = device_context(sessions=sessions, micro=micro, mbs=mbs, sel=sel, E=E, H=H,
                                       dtype=dtype, ids=ids, layers=lay, layerNum=L, seed=seed)
    # outputs sized larger than the context's slots: the extra rows are tail
    run_both(ctx_d, host, (sessions + 2, micro * mbs, sel, H), E, dtype, 0, layerNum=L)


@pytest.mark.parametrize("dtype,off,H,sessions", [(1, 0, 4096, 4), (1, 2, 4096, 4), (1, 4, 4096, 4),
                                                   (1, 8, 4096, 4), (0, 12, 4096, 4), (2, 0, 4096, 4),
                                                   (2, 4, 4096, 4), (1, 0, 64, 32), (0, 6, 64, 32)])
def test_token_buffer_alignment(dtype, off, H, sessions):
    # 16-bit rows take the flat gather (rows of 8 KB over 1152 slots; rows of
    # 128 bytes over 9216 slots, its short-row form), whose source address is
    # read on the device and checked there: an aligned base, and bases 2 to 12
    # bytes past a 16-byte boundary (the word and byte forms); INT8 rows with
    # their scale stay with the warp kernel
    micro, mbs, sel = 2, 16, 9
    rng = np.random.default_rng(40 + off + H)
    slots = sessions * micro * mbs * sel
    ids = rng.integers(-1, 66, size=slots).astype(np.int32)
    ctx_d, host, keep = device_context(sessions=sessions, micro=micro, mbs=mbs, sel=sel, E=64, H=H,
                                       dtype=dtype, ids=ids, seed=off, base_offset=off)
    run_both(ctx_d, host, (sessions, micro * mbs, sel, H), 64, dtype, 0)


@pytest.mark.parametrize("dtype,off", [(1, 0), (1, 6), (0, 2), (2, 0), (2, 4)])
def test_small_context_one_block(dtype, off):
    # 144 slots of 128-byte rows (INT8: 68 bytes): one block sorts, scatters
    # and gathers the rows; token buffers aligned and not
    sessions, micro, mbs, sel, H = 2, 1, 8, 9, 64
    rng = np.random.default_rng(70 + off + dtype)
    ids = rng.integers(-1, 10, size=sessions * micro * mbs * sel).astype(np.int32)
    ctx_d, host, keep = device_context(sessions=sessions, micro=micro, mbs=mbs, sel=sel, E=8, H=H,
                                       dtype=dtype, ids=ids, seed=off, base_offset=off)
    run_both(ctx_d, host, (sessions + 1, micro * mbs, sel, H), 8, dtype, 0)


def test_need_schedule_all_ready():
    ids = np.random.default_rng(5).integers(0, 32, size=4 * 2 * 8 * 3).astype(np.int32)
    ctx_d, host, keep = device_context(sessions=4, micro=2, mbs=8, sel=3, E=32, H=64, dtype=1, ids=ids)
    g, _ = run_both(ctx_d, host, (4, 16, 3, 64), 32, 1, 1)
    assert int(g["scheduleStatus"][0]) == 0


def test_need_schedule_wait_runs_out_and_status_reports_it():
    """Three blocks never get their flag: the wait ends at the timeout, those
    blocks are masked, status = 3, and the GPU keeps working afterwards."""
    sessions, micro = 4, 2
    flags = np.ones(sessions * micro, np.int32)
    flags[[1, 4, 7]] = 0
    ids = np.random.default_rng(6).integers(0, 16, size=sessions * micro * 4 * 2).astype(np.int32)
    ctx_d, host, keep = device_context(sessions=sessions, micro=micro, mbs=4, sel=2, E=16, H=32,
                                       dtype=0, ids=ids, flags=flags)
    t0 = time.perf_counter()
    g, ref = run_both(ctx_d, host, (4, 8, 2, 32), 16, 0, 1, timeout_us=20_000)
    elapsed = time.perf_counter() - t0
    assert int(g["scheduleStatus"][0]) == 3 == ref["status"]
    assert elapsed < 10.0
    # the context stays usable: the same call without waiting, then again
    run_both(ctx_d, host, (4, 8, 2, 32), 16, 0, 0)
    g, _ = run_both(ctx_d, host, (4, 8, 2, 32), 16, 0, 1, timeout_us=20_000)
    assert int(g["scheduleStatus"][0]) == 3


@pytest.mark.parametrize("bad", ["too_many_slots", "expert_num", "small_data"])
def test_invalid_context(bad):
    ids = np.zeros(2 * 1 * 2 * 2, np.int32)
    ctx_d, host, keep = device_context(sessions=2, micro=1, mbs=2, sel=2, E=2, H=8, dtype=1, ids=ids)
    ctx = host[0].copy()
    shape = (2, 2, 2, 8)
    if bad == "too_many_slots":
        shape = (1, 2, 2, 8)
    elif bad == "expert_num":
        ctx[16:20] = np.array([3], np.uint32).view(np.uint8)
    else:
        ctx[408:416] = np.array([16], np.uint64).view(np.uint8)
    ctx_d = torch.from_numpy(ctx).to("cuda:0")
    g, _ = run_both(ctx_d, (ctx,) + host[1:], shape, 2, 1, 0)
    assert int(g["scheduleStatus"][0]) == -1 and int(g["actualTokenNum"][0]) == 0
