"""MoeUpdateExpert on the GPU vs the oracle ("MoeUpdateExpert", 功能说明 and
参数说明): the mapping is integer work, compared bit for bit; the pruning mask
compares the same fp32 values on both sides."""
import numpy as np
import pytest
import torch

import oracle
import workloads as w

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import unpermute_stable_counting_gb300 as usc  # noqa: E402

from _gpu_util import dev, float_tensor, to_dev  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def run_both(inp, *, local_rank, mode, prune=True, active=True, strided=False):
    sdt = inp["scales_dtype"]
    ids_h, tab_h = inp["expert_ids"], inp["table"]
    ref = oracle.update_expert(ids_h, tab_h, local_rank=local_rank, balance_mode=mode,
                               scales=inp["scales"] if prune else None, scales_dtype=sdt,
                               threshold=inp["threshold"] if prune else None,
                               active=inp["active"] if (prune and active) else None)
    ids, tab = to_dev(ids_h), to_dev(tab_h)
    sc = float_tensor(inp["scales"], sdt) if prune else None
    thr = to_dev(inp["threshold"]) if prune else None
    act = to_dev(inp["active"]) if (prune and active) else None
    out = None
    if strided:
        # every tensor a strided view inside a larger buffer
        BS, K = ids_h.shape
        E, F = tab_h.shape
        big = torch.full((K, 3 * BS), -7, dtype=ids.dtype, device=dev())
        big[:, ::3] = ids.T
        ids = big[:, ::3].T                          # strides (3, 3*BS)
        bt = torch.zeros((E, 2 * F + 1), dtype=torch.int32, device=dev())
        bt[:, 1::2] = tab
        tab = bt[:, 1::2]                            # strides (2F+1, 2)
        if prune:
            bs = torch.zeros((BS, 2 * K), dtype=sc.dtype, device=dev())
            bs[:, K:] = sc
            sc = bs[:, K:]
            thr = thr.repeat_interleave(2)[::2].reshape(1, K)
            if act is not None:
                ba = torch.zeros((BS, 4), dtype=torch.bool, device=dev())
                ba[:, 2] = act
                act = ba[:, 2]
        ob = torch.full((BS, K, 2), -5, dtype=ids.dtype, device=dev())
        mb = torch.zeros((K, BS), dtype=torch.bool, device=dev())
        out = dict(balancedExpertIds=ob[:, :, 1], balancedActiveMask=mb.T if prune else None)
    got = usc.moe_update_expert(ids, tab, local_rank=local_rank, world_size=inp["world_size"],
                                balance_mode=mode, scales=sc, threshold=thr, active=act, out=out)
    torch.cuda.synchronize()
    g_ids = got["balancedExpertIds"].cpu().numpy()
    assert g_ids.dtype == ids_h.dtype
    assert np.array_equal(g_ids, ref["balancedExpertIds"])
    if prune:
        assert np.array_equal(got["balancedActiveMask"].cpu().numpy(), ref["balancedActiveMask"])
    else:
        assert got["balancedActiveMask"] is None
    if strided:
        assert (ob[:, :, 0] == -5).all()             # the gaps of the output view are untouched
    return got, ref


TABLE = np.array([[1, 7, 0, 0], [2, 3, 5, 0], [3, 1, 4, 6]], np.int32)


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("idt", [np.int32, np.int64])
def test_hand_table(mode, idt):
    ids = np.array([[0, 1, 2], [2, 1, 0], [1, 2, 0], [-1, 3, 2]], idt)
    scales = np.array([[0.6, 0.3, 0.1], [0.5, 0.25, 0.25], [0.9, 0.06, 0.04], [1, 1, 1]], np.float32)
    inp = dict(expert_ids=ids, table=TABLE, scales=scales, scales_dtype=3,
               threshold=np.array([0.2, 0.26, 0.1], np.float32),
               active=np.array([1, 1, 0, 1], bool), world_size=4)
    got, ref = run_both(inp, local_rank=2, mode=mode)
    assert ref["balancedExpertIds"][3].tolist()[:2] == [-1, -1]


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("sdt", [0, 1, 3])
@pytest.mark.parametrize("idt", [np.int32, np.int64])
def test_generated(mode, sdt, idt):
    inp = w.make_update_expert(BS=200, K=8, moe_expert_num=96, world_size=32, place_per_rank=6,
                               scales_dtype=sdt, id_dtype=idt, seed=10 + sdt + 3 * mode)
    run_both(inp, local_rank=13, mode=mode)
    run_both(inp, local_rank=0, mode=mode, active=False)
    run_both(inp, local_rank=31, mode=mode, prune=False)


@pytest.mark.parametrize("mode", [0, 1])
def test_strided_views(mode):
    inp = w.make_update_expert(BS=64, K=6, moe_expert_num=40, world_size=16, place_per_rank=4,
                               scales_dtype=1, id_dtype=np.int64, seed=21)
    run_both(inp, local_rank=5, mode=mode, strided=True)


@pytest.mark.parametrize("mode", [0, 1])
def test_maximum_sizes(mode):
    """BS 512, K 16, 1024 experts over 256 ranks x 4 instances (each count 1),
    and 512 experts over 128 x 8 (redundant instances)."""
    for E, ws, ppr, seed in [(1024, 256, 4, 30), (512, 128, 8, 31)]:
        inp = w.make_update_expert(BS=512, K=16, moe_expert_num=E, world_size=ws, place_per_rank=ppr,
                                   scales_dtype=1, seed=seed + mode)
        run_both(inp, local_rank=ws - 1, mode=mode)


def test_invalid_ids_counts_and_nan_scales():
    rng = np.random.default_rng(40)
    inp = w.make_update_expert(BS=33, K=5, moe_expert_num=20, world_size=8, place_per_rank=5,
                               scales_dtype=0, seed=40)
    ids = inp["expert_ids"].copy()
    ids[rng.random(ids.shape) < 0.2] = -3
    ids[rng.random(ids.shape) < 0.1] = 20                 # == moeExpertNum
    ids[0, 0] = np.iinfo(np.int32).max
    tab = inp["table"].copy()
    tab[3, 0] = 0                                         # count 0
    tab[4, 0] = tab.shape[1]                              # count past F - 1
    sc = inp["scales"].copy()
    sc[1, :] = 0x7E00                                     # fp16 NaN: not below the threshold
    sc[2, 0] = 0xFC00                                     # -inf: pruned
    inp = dict(inp, expert_ids=ids, table=tab, scales=sc)
    for mode in (0, 1):
        got, ref = run_both(inp, local_rank=7, mode=mode)
        assert (ref["balancedExpertIds"] == -1).sum() > 0
        assert ref["balancedActiveMask"][1].tolist() == [bool(inp["active"][1])] * 5


def test_back_to_back_on_a_side_stream():
    inp = w.make_update_expert(BS=128, K=8, moe_expert_num=64, world_size=16, place_per_rank=8,
                               scales_dtype=3, seed=50)
    s = torch.cuda.Stream()
    ids, tab = to_dev(inp["expert_ids"]), to_dev(inp["table"])
    sc, thr, act = to_dev(inp["scales"]), to_dev(inp["threshold"]), to_dev(inp["active"])
    with torch.cuda.stream(s):
        outs = [usc.moe_update_expert(ids, tab, local_rank=r, world_size=16, balance_mode=0,
                                      scales=sc, threshold=thr, active=act) for r in range(16)]
    s.synchronize()
    for r in (0, 7, 15):
        ref = oracle.update_expert(inp["expert_ids"], inp["table"], local_rank=r, balance_mode=0,
                                   scales=inp["scales"], scales_dtype=3, threshold=inp["threshold"],
                                   active=inp["active"])
        assert np.array_equal(outs[r]["balancedExpertIds"].cpu().numpy(), ref["balancedExpertIds"])
