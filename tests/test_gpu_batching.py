"""Batching: CUDA path vs the oracle, bit for bit, on the same seeded inputs."""
import numpy as np
import pytest
import torch

import oracle
import workloads as w

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from _gpu_util import assert_batching_equal, batching_numpy, run_batching, to_dev  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def check(inp, **kw):
    ref = oracle.batching(inp)
    got = batching_numpy(run_batching(inp, **kw), inp)
    assert_batching_equal(got, ref, with_sorted=kw.get("with_sorted", True))
    return got, ref


def test_tiny_workload():
    check(w.make_batching(**w.BATCHING_TINY))


def test_page_example():
    """The batching page's example program: 72 slots, ids i % 8, H = 4096 fp16
    rows of 0x0001."""
    Y, H = 72, 4096
    td = np.full((Y, H), 1, dtype=np.uint16).view(np.uint8).reshape(Y, 2 * H)
    inp = dict(expert_ids=(np.arange(Y) % 8).astype(np.int32), layer_id=0, token_data=td,
               row_stride=2 * H, scales=None, session_in=np.zeros(Y, np.int32),
               micro_in=np.zeros(Y, np.int32), token_in=None, expertNum=8, A=1, BS=8, K1=9, H=H,
               tokenDtype=0, layerNum=1, Y=Y)
    got, _ = check(inp)
    assert got["groupList"].tolist() == [[e, 9] for e in range(8)]
    assert got["actualTokenNum"] == 72
    assert np.array_equal(got["expertOffsets"], np.arange(Y) % 9)


def test_int8_decode_workload():
    check(w.make_batching(**w.BATCHING_INT8_DECODE))


@pytest.mark.slow
def test_roundtrip_batching_full_size():
    check(w.make_batching(**w.ROUNDTRIP_BATCHING))


FUZZ = [
    # (A, BS, K1, E, H, dtype, layerNum, ids, mask)
    (1, 1, 1, 1, 1, 0, 1, "uniform", 0.0),
    (2, 3, 5, 8, 7, 1, 1, "uniform", 0.3),
    (3, 7, 9, 16, 8, 2, 2, "zipf", 0.2),
    (4, 16, 33, 8192, 129, 0, 1, "uniform", 0.1),      # E = 8192: 8193 buckets in one pass
    (4, 16, 33, 8192, 16, 2, 8, "zipf", 0.0),
    (5, 64, 7, 1, 24, 1, 1, "uniform", 0.5),           # a single expert
    (3, 100, 7, 64, 64, 1, 1, "mod", 0.0),             # 2100 slots: two tiles + ragged tail
    (8, 128, 9, 256, 40, 2, 1, "zipf", 0.15),          # 9216 slots, int8 row stride H + 4
    (2, 4, 3, 12, 5, 0, 3, "uniform", 1.0),            # every slot masked
    (16, 64, 64, 4096, 16, 1, 16, "zipf", 0.05),       # 65536 slots, 32 tiles
    (1024, 4, 8, 512, 8, 1, 1, "zipf", 0.1),           # A at its maximum (1024)
    (1024, 64, 32, 8192, 8, 1, 8, "zipf", 0.05),       # 2.1M slots (1024 tiles), 8192 experts
    (2, 4, 5, 16, 65536, 1, 1, "zipf", 0.1),           # 128 KB rows
    (2, 4, 5, 16, 65536, 2, 1, "zipf", 0.1),           # 64 KB int8 rows + scale (stride 65540)
    (3, 683, 1, 16, 24, 1, 1, "zipf", 0.1),            # 2049 slots: one-launch sort, 5 tiles, ragged
    (8, 64, 9, 4097, 8, 2, 1, "uniform", 0.2),         # 4608 slots, 4098 keys: one-launch sort's key limit
    (64, 64, 8, 4096, 8, 1, 1, "zipf", 0.05),          # 32768 slots: one-launch sort at 64 tiles
    (3, 10923, 1, 4097, 8, 0, 1, "uniform", 0.1),      # 32769 slots: past it, the kernel chain
    (4, 64, 9, 8192, 8, 1, 1, "zipf", 0.1),            # 2304 slots, 8193 keys: chain (key limit)
    (64, 64, 64, 1, 8, 1, 1, "uniform", 0.0),          # 262144 slots of one key: 128 full tiles of it
    (256, 64, 9, 1024, 8, 1, 4, "zipf", 0.05),         # the round trip's 147456 slots and 1025 keys
]


@pytest.mark.parametrize("A,BS,K1,E,H,dt,L,ids,mask", FUZZ)
def test_fuzz_shapes(A, BS, K1, E, H, dt, L, ids, mask):
    inp = w.make_batching(A=A, BS=BS, K1=K1, E=E, H=H, dtype=dt, layerNum=L, layer_id=L - 1,
                          ids=ids, zipf_s=1.1, mask=mask, session=7, micro=5,
                          seed=A * 1000 + E + H)
    check(inp)


def test_layer_zero_and_invalid_ids():
    inp = w.make_batching(A=2, BS=8, K1=4, E=10, H=32, dtype=1, layerNum=0, layer_id=0, seed=3,
                          mask=0.0)
    rng = np.random.default_rng(0)
    ids = inp["expert_ids"].copy()
    pick = rng.random(ids.size) < 0.25
    ids[pick] = rng.choice([-1, -2**31, 10, 11, 2**31 - 1], size=int(pick.sum()))
    inp["expert_ids"] = ids
    check(inp)


def test_token_ids_null_and_no_sorted_indices():
    inp = w.make_batching(A=4, BS=8, K1=3, E=16, H=64, dtype=0, seed=11, token_ids=False)
    check(inp, with_sorted=False)


def test_int8_separate_scales_and_odd_stride():
    inp = w.make_batching(A=4, BS=16, K1=5, E=32, H=96, dtype=2, seed=12, separate_scales=True)
    check(inp)
    # interleaved int8 rows whose length is not a multiple of 4 bytes
    inp = w.make_batching(A=4, BS=16, K1=5, E=32, H=97, dtype=2, seed=13)
    check(inp)


def test_unaligned_row_stride():
    """fp16 rows padded to a stride that is not a multiple of 16 bytes."""
    inp = w.make_batching(A=2, BS=16, K1=5, E=16, H=40, dtype=0, seed=14)
    Y, rb = inp["Y"], 80
    td = np.zeros((Y, rb + 6), np.uint8)
    td[:, :rb] = inp["token_data"]
    inp["token_data"] = td
    inp["row_stride"] = rb + 6
    check(inp)


def test_two_calls_reuse_workspace_and_side_stream():
    import unpermute_stable_counting_gb300 as usc
    a = w.make_batching(A=4, BS=32, K1=9, E=64, H=128, dtype=1, seed=21)
    b = w.make_batching(A=4, BS=32, K1=9, E=64, H=128, dtype=1, seed=22, ids="zipf")
    ws = torch.empty(usc.batching_workspace_size(64, (4, 32, 9, 128), 1, 1), dtype=torch.uint8,
                     device="cuda:0")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        ra = batching_numpy(run_batching(a, workspace=ws, stream=s), a)
        rb = batching_numpy(run_batching(b, workspace=ws, stream=s), b)
    assert_batching_equal(ra, oracle.batching(a))
    assert_batching_equal(rb, oracle.batching(b))


def test_tail_rows_untouched():
    """Rows i >= U of y are not written."""
    import unpermute_stable_counting_gb300 as usc
    inp = w.make_batching(A=2, BS=8, K1=3, E=8, H=64, dtype=1, mask=0.4, seed=31)
    out = usc.batching_outputs(inp["Y"], 64, 8, 1, "cuda:0", True)
    out["y"].fill_(7.0)
    got = batching_numpy(run_batching(inp, out=out), inp)
    U = got["actualTokenNum"]
    assert U < inp["Y"]
    tail = out["y"][U:].float()
    assert bool((tail == 7.0).all())


@pytest.mark.parametrize("H", [16, 48, 4112, 7168])
def test_int8_rows_with_interleaved_scale_shift_path(H):
    """INT8 rows of stride H + 4 start at 4-byte offsets 0, 4, 8, 12: the
    16-byte windows path (H a multiple of 16) and its last-vector tail."""
    inp = w.make_batching(A=2, BS=16, K1=9, E=64, H=H, dtype=2, ids="zipf", mask=0.1, seed=H)
    check(inp)


def test_int8_rows_unaligned_buffer_base():
    """A token buffer whose base is not 16-byte aligned takes the word path."""
    inp = w.make_batching(A=2, BS=16, K1=9, E=64, H=64, dtype=2, ids="zipf", mask=0.1, seed=5)
    raw = inp["token_data"].reshape(-1)
    buf = torch.zeros(raw.size + 16, dtype=torch.uint8, device="cuda:0")
    buf[4:4 + raw.size] = torch.from_numpy(raw).to("cuda:0")
    view = buf[4:4 + raw.size].view(inp["Y"], -1)
    assert view.data_ptr() % 16 == 4
    check(inp, token_data=view)
