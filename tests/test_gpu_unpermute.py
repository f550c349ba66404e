"""Unpermute: CUDA path vs the oracle on the same seeded inputs. Index and
prob outputs bit for bit; unpermutedTokens within the stated tolerance (and,
by construction of the kernels, bit for bit as well)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as w

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from _gpu_util import assert_unpermute_equal, run_unpermute, unpermute_numpy  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def check(inp, **kw):
    ref = oracle.unpermute(inp)
    got = unpermute_numpy(run_unpermute(inp, **kw), inp)
    assert_unpermute_equal(got, ref, inp)
    return got, ref


def test_page_example_padded():
    inp = dict(permuted=np.ones((2, 2), np.float32), sortedIndices=np.array([1, 1], np.int32),
               routingMap=np.ones((2, 2), np.int8), probs=np.ones((2, 2), np.float32),
               permutedRows=2, H=2, tokenDtype=3, n=2, probsDtype=3, T=2, Eu=2, padded=1)
    got, _ = check(inp)
    assert got["unpermuted"].tolist() == [[0.0, 0.0], [2.0, 2.0]]


def test_topk_workload():
    check(w.make_unpermute_topk(**w.UNPERMUTE_TOPK))


def test_padded_workload():
    check(w.make_unpermute_padded(**w.UNPERMUTE_PADDED))


def test_padded_slack_workload():
    """Capacity twice the routed load: half of the 131072 slots are padding."""
    check(w.make_unpermute_padded(**w.UNPERMUTE_PADDED_SLACK))


COMBOS = [(0, 0), (0, 3), (1, 1), (1, 3), (3, 3)]


@pytest.mark.parametrize("dt,pdt", COMBOS)
@pytest.mark.parametrize("with_probs", [True, False])
def test_not_padded_dtypes(dt, pdt, with_probs):
    inp = w.make_unpermute_topk(T=300, k=6, Eu=24, H=136, dtype=dt,
                                probs_dtype=pdt if with_probs else None, choices=(1, 3, 6),
                                seed=dt * 10 + pdt)
    check(inp)


@pytest.mark.parametrize("dt,pdt", COMBOS)
@pytest.mark.parametrize("with_probs", [True, False])
def test_padded_dtypes(dt, pdt, with_probs):
    inp = w.make_unpermute_padded(T=512, Eu=32, k=4, H=72, dtype=dt,
                                  probs_dtype=pdt if with_probs else None, mult=5,
                                  seed=dt * 10 + pdt)
    check(inp)


@pytest.mark.parametrize("H", [1, 7, 9, 33])
@pytest.mark.parametrize("padded", [0, 1])
def test_odd_hidden_scalar_path(H, padded):
    if padded:
        inp = w.make_unpermute_padded(T=64, Eu=16, k=4, H=H, dtype=1, probs_dtype=3, mult=3, seed=H)
    else:
        inp = w.make_unpermute_topk(T=70, k=5, Eu=12, H=H, dtype=0, probs_dtype=0,
                                    choices=(2, 5), seed=H)
    check(inp)


def test_invalid_indices_duplicates_and_zero_probs():
    rng = np.random.default_rng(5)
    inp = w.make_unpermute_topk(T=257, k=7, Eu=20, H=64, dtype=1, probs_dtype=3, choices=(1, 4, 7),
                                seed=5)
    si = inp["sortedIndices"]
    pick = rng.random(si.size) < 0.1
    si[pick] = rng.choice([-7, -1, inp["permutedRows"], 2**31 - 1], size=int(pick.sum()))
    dup = rng.random(si.size) < 0.1
    si[dup] = rng.integers(0, 50, size=int(dup.sum()))
    inp["probs"][rng.random(inp["probs"].shape) < 0.2] = 0.0
    check(inp)
    p = w.make_unpermute_padded(T=128, Eu=16, k=4, H=64, dtype=0, probs_dtype=0, mult=7, seed=6)
    si = p["sortedIndices"]
    pick = rng.random(si.size) < 0.1
    si[pick] = rng.choice([-1, 128, 999], size=int(pick.sum()))
    dup = rng.random(si.size) < 0.15
    si[dup] = rng.integers(0, 8, size=int(dup.sum()))
    check(p)


def test_topk_512_and_empty_tokens():
    """topK_num = 512 (the largest allowed), most slots unused."""
    T, k, H = 12, 512, 32
    inp = w.make_unpermute_topk(T=T, k=k, Eu=600, H=H, dtype=1, probs_dtype=1, choices=(0, 3, 512),
                                seed=9)
    check(inp)


@pytest.mark.parametrize("padded", [0, 1])
def test_wide_rows(padded):
    """65536-element rows (512 hidden chunks of 64 vectors per token)."""
    if padded:
        inp = w.make_unpermute_padded(T=64, Eu=16, k=2, H=65536, dtype=1, probs_dtype=3, mult=3, seed=43)
    else:
        inp = w.make_unpermute_topk(T=24, k=4, Eu=12, H=65536, dtype=1, probs_dtype=1, choices=(2, 4), seed=44)
    check(inp)


@pytest.mark.parametrize("T,Eu", [(40, 10), (2000, 16), (70000, 64)])
def test_more_routing_ones_than_slots(T, Eu):
    """maskedSelect output longer than n: truncated. The map sizes take the
    small-map path, the one-kernel maskedSelect and the three-kernel one."""
    inp = w.make_unpermute_topk(T=T, k=4, Eu=Eu, H=16, dtype=3, probs_dtype=3, choices=(4,), seed=3)
    inp["routingMap"][:] = 1
    inp["probs"] = np.random.default_rng(3).random((T, Eu)).astype(np.float32)
    check(inp)


@pytest.mark.parametrize("Eu,off", [(67, 0), (64, 1), (64, 4)])
def test_large_map_layouts(Eu, off):
    """Routing maps past the one-kernel maskedSelect (more than 4M entries):
    an expert count that is not a multiple of 4 (column masks one expert per
    lane; the scatter's 16-entry loads cross token rows), and maps 1 and 4
    bytes past a 16-byte boundary (the byte and 4-byte forms)."""
    T = (1 << 22) // Eu + 64
    inp = w.make_unpermute_topk(T=T, k=4, Eu=Eu, H=8, dtype=1, probs_dtype=1, choices=(1, 4), seed=Eu + off)
    assert T * Eu > (1 << 22)
    ref = oracle.unpermute(inp)
    got = unpermute_numpy(run_unpermute(inp, map_offset=off), inp)
    assert_unpermute_equal(got, ref, inp)


@pytest.mark.parametrize("rows_extra", [0, 5])
def test_no_probs_restore_shape(rows_extra):
    """Branches (3)/(4) take the token count from restoreShape."""
    inp = w.make_unpermute_topk(T=100, k=3, Eu=8, H=24, dtype=3, probs_dtype=None, choices=(1, 3),
                                seed=4, rows=300 + rows_extra)
    check(inp)


SORT_CASES = {
    # one counting-sort pass over every key (up to 4096 keys)
    "one_pass": lambda: w.make_unpermute_topk(T=500, k=8, Eu=32, H=16, dtype=1, probs_dtype=1,
                                              choices=(2, 8), seed=15),
    "one_pass_padded": lambda: w.make_unpermute_padded(T=4032, Eu=64, k=2, H=16, dtype=0,
                                                       probs_dtype=3, mult=9, seed=16),
    # two levels (a coarse pass, then a block per coarse bucket), ragged tile counts
    "two_level_not_padded": lambda: w.make_unpermute_topk(T=1000, k=6, Eu=32, H=16, dtype=1, probs_dtype=1,
                                                          choices=(2, 6), seed=11),
    "two_level_padded": lambda: w.make_unpermute_padded(T=8192, Eu=64, k=2, H=16, dtype=0,
                                                        probs_dtype=3, mult=9, seed=10),
    "two_level_wide_not_padded": lambda: w.make_unpermute_topk(T=20000, k=8, Eu=32, H=16, dtype=1,
                                                               probs_dtype=1, choices=(3, 8), seed=13),
    "two_level_wide_padded": lambda: w.make_unpermute_padded(T=32768, Eu=64, k=2, H=16, dtype=0,
                                                             probs_dtype=3, mult=7, seed=14),
    # padded, the first key count past one pass (T = 4096: 4097 keys), and a
    # token count that leaves the last coarse bucket part-filled (T = 5000,
    # 32 fine keys) with slack capacity (padding slots)
    "two_level_padded_4097_keys": lambda: w.make_unpermute_padded(T=4096, Eu=16, k=2, H=8, dtype=0,
                                                                  probs_dtype=3, mult=5, seed=25),
    "two_level_padded_ragged_slack": lambda: w.make_unpermute_padded(T=5000, Eu=8, k=2, H=8, dtype=1,
                                                                     probs_dtype=3, mult=3, capacity=1500,
                                                                     seed=24),
    # not padded, the first key count past one pass: 4096 rows, 3-bit fine keys
    "two_level_not_padded_4097_keys": lambda: w.make_unpermute_topk(T=1024, k=4, Eu=8, H=8, dtype=1,
                                                                    probs_dtype=1, choices=(1, 4), seed=21),
    # not padded at the two-level limit (2^22 keys: 4097 coarse buckets, 10-bit
    # fine keys) and one row past it (LSD passes)
    "two_level_not_padded_max": lambda: permutation_case((1 << 22) - 1, seed=22),
    "passes_not_padded_past_max": lambda: permutation_case(1 << 22, seed=23),
    # padded keys beyond 2^22: LSD passes and the CSR kernel
    "passes_padded_4m": lambda: w.make_unpermute_padded(T=1 << 22, Eu=16, k=1, H=4, dtype=0,
                                                        probs_dtype=3, mult=5, seed=19),
    # two levels beside a small routing map (the gather-reduce selects the
    # weights), without probs, with a map of 9 experts, and over 128 and 129
    # tiles of 2048 entries
    "two_level_small_map": lambda: w.make_unpermute_topk(T=512, k=10, Eu=32, H=16, dtype=1, probs_dtype=1,
                                                         choices=(3, 10), seed=26),
    "two_level_no_probs": lambda: permutation_case(100000, seed=27),
    "two_level_nine_experts": lambda: w.make_unpermute_topk(T=4096, k=9, Eu=9, H=16, dtype=1, probs_dtype=1,
                                                            choices=(7, 9), seed=28),
    "two_level_128_tiles": lambda: w.make_unpermute_topk(T=32768, k=8, Eu=16, H=8, dtype=1, probs_dtype=3,
                                                         choices=(5, 8), seed=29),
    "two_level_129_tiles": lambda: permutation_case(262145, seed=30),
    # 32800 tokens x 512 slots: 16.8M rows, 25-bit keys (topK_num at its maximum)
    "three_passes": lambda: w.make_unpermute_topk(T=32800, k=512, Eu=16, H=8, dtype=1, probs_dtype=1,
                                                  choices=(1, 2), seed=17),
}


def permutation_case(rows, seed, invalid=0.1):
    """Not padded, topK = 1, no probs: sortedIndices is a random permutation
    of the rows with a fraction replaced by invalid indices (-1 and rows)."""
    rng = np.random.default_rng(seed)
    si = rng.permutation(rows).astype(np.int32)
    bad = rng.random(rows) < invalid
    si[bad] = np.where(rng.random(int(bad.sum())) < 0.5, -1, rows).astype(np.int32)
    return dict(permuted=w.normal_rows(rows, 4, 0, seed), sortedIndices=si, routingMap=None, probs=None,
                permutedRows=rows, H=4, tokenDtype=0, n=rows, probsDtype=0, T=rows, Eu=0, padded=0)


@pytest.mark.parametrize("case", list(SORT_CASES))
def test_index_sort_paths(case):
    """The index sort's forms: one counting-sort pass over every key; up to
    2^22 keys a coarse pass on the high bits and a per-bucket fine sort (padded,
    it also writes the row pointers; not padded, the invalid entries are
    placed by the coarse pass); and two or three LSD passes beyond that (keys
    beyond 2^24 take three)."""
    check(SORT_CASES[case]())


@pytest.mark.parametrize("T,k", [(2048, 4), (16384, 9)])
def test_not_padded_invalid_rows_and_duplicates(T, k):
    """Two-level not-padded sort with 40% invalid slots (all in the coarse
    bucket that the coarse pass places) and one row index repeated in 10% of
    the slots (one fine key with thousands of entries, many 256-entry chunks
    in one block)."""
    inp = w.make_unpermute_topk(T=T, k=k, Eu=2 * k, H=24, dtype=1, probs_dtype=1, choices=(k,), seed=T + k)
    rng = np.random.default_rng(T)
    si = inp["sortedIndices"].copy()
    bad = rng.random(si.size) < 0.4
    si[bad] = np.where(rng.random(int(bad.sum())) < 0.5, -1, T * k + 3).astype(np.int32)
    dup = rng.random(si.size) < 0.1
    si[dup & ~bad] = 77
    check(dict(inp, sortedIndices=si))


@pytest.mark.parametrize("padded", [0, 1])
def test_maximum_experts(padded):
    """8192 experts (the most the maskedSelect and padded layouts take)."""
    if padded:
        inp = w.make_unpermute_padded(T=8192, Eu=8192, k=2, H=16, dtype=1, probs_dtype=3, mult=3, seed=18)
    else:
        inp = w.make_unpermute_topk(T=96, k=8, Eu=8192, H=24, dtype=1, probs_dtype=1, choices=(1, 8),
                                    seed=18)
    check(inp)


SMALL_MAP_CASES = {
    # T * Eu at the small-map limit (16384 entries: the weights are selected in
    # the gather-reduce) and just past it (the maskedSelect kernels)
    "at_limit": lambda: w.make_unpermute_topk(T=256, k=8, Eu=64, H=64, dtype=1, probs_dtype=1,
                                              choices=(3, 8), seed=31),
    "past_limit": lambda: w.make_unpermute_topk(T=257, k=8, Eu=64, H=64, dtype=1, probs_dtype=1,
                                                choices=(3, 8), seed=32),
    # more than 32 slots per token (several slot groups), fp32 probs with fp16 rows
    "wide_topk": lambda: w.make_unpermute_topk(T=48, k=40, Eu=128, H=72, dtype=0, probs_dtype=3,
                                               choices=(17, 40), seed=33),
    # a wide map of few tokens: 4000 experts, the expert starts scanned in 16 steps
    "many_experts": lambda: w.make_unpermute_topk(T=2, k=8, Eu=4000, H=8, dtype=1, probs_dtype=1,
                                                  choices=(1, 8), seed=34),
    # too wide for the 32 KB of shared memory (8192 experts): the maskedSelect kernels
    "too_wide": lambda: w.make_unpermute_topk(T=1, k=8, Eu=8192, H=8, dtype=1, probs_dtype=1,
                                              choices=(8,), seed=35),
    # one token, one slot
    "single": lambda: w.make_unpermute_topk(T=1, k=1, Eu=3, H=8, dtype=3, probs_dtype=3, choices=(1,),
                                            seed=36),
    # past the small-map limit (the maskedSelect kernels): more than 32 slots
    # per token, and several units per warp with runs of two chunks
    "wide_topk_past_limit": lambda: w.make_unpermute_topk(T=600, k=40, Eu=128, H=72, dtype=0, probs_dtype=3,
                                                      choices=(9, 40), seed=38),
    # the one-kernel maskedSelect at its limit (4096 tiles of 1024 map entries)
    # and past it (column bitmasks, prefix and scatter kernels)
    "one_kernel_select_at_limit": lambda: w.make_unpermute_topk(T=65536, k=2, Eu=64, H=8, dtype=1,
                                                                probs_dtype=1, choices=(1, 2), seed=40),
    "select_chain_past_limit": lambda: w.make_unpermute_topk(T=65600, k=2, Eu=64, H=8, dtype=1,
                                                             probs_dtype=3, choices=(1, 2), seed=41),
    "runs_past_limit": lambda: w.make_unpermute_topk(T=3000, k=6, Eu=48, H=2048, dtype=1, probs_dtype=3,
                                                 choices=(2, 6), seed=39),
}


@pytest.mark.parametrize("case", list(SMALL_MAP_CASES))
def test_small_map_weights(case):
    """Not padded with probs: the weights (and permuteProbs) selected by the
    gather-reduce from a small routing map, at and around the size limits;
    larger maps through the one-kernel maskedSelect, and past its limit the
    three-kernel one."""
    check(SMALL_MAP_CASES[case]())


def test_small_map_empty_and_invalid():
    """An empty routing map (permuteProbs all 0, nothing added) and invalid
    slot indices beside valid ones."""
    inp = w.make_unpermute_topk(T=40, k=4, Eu=16, H=16, dtype=1, probs_dtype=1, choices=(2, 4), seed=37)
    check(dict(inp, routingMap=np.zeros_like(inp["routingMap"])))
    si = inp["sortedIndices"].copy()
    si[::3] = -1
    si[1::7] = inp["permutedRows"] + 5
    check(dict(inp, sortedIndices=si))


@pytest.mark.parametrize("T,Eu", [(8192, 64), (16384, 128)])
def test_padded_invalid_rows_and_duplicates(T, Eu):
    """Two-level padded sort with 40% invalid rows (-1 and >= T: one fine
    bucket of thousands of rows, many 256-row chunks) and repeated tokens."""
    inp = w.make_unpermute_padded(T=T, Eu=Eu, k=2, H=24, dtype=1, probs_dtype=3, mult=3, seed=20)
    rng = np.random.default_rng(T)
    si = inp["sortedIndices"].copy()
    bad = rng.random(si.size) < 0.4
    si[bad] = np.where(rng.random(bad.sum()) < 0.5, -1, T + 7).astype(np.int32)
    dup = rng.random(si.size) < 0.1
    si[dup & ~bad] = 5                       # token 5 many times over
    inp = dict(inp, sortedIndices=si)
    check(inp)


def test_workspace_reuse_and_side_stream():
    import unpermute_stable_counting_gb300 as usc
    a = w.make_unpermute_topk(T=200, k=8, Eu=32, H=64, dtype=1, probs_dtype=1, seed=41)
    b = w.make_unpermute_padded(T=256, Eu=32, k=4, H=64, dtype=0, probs_dtype=3, mult=3, seed=42)
    s = torch.cuda.Stream()
    ws = torch.empty(1 << 22, dtype=torch.uint8, device="cuda:0")
    with torch.cuda.stream(s):
        ga = unpermute_numpy(run_unpermute(a, workspace=ws, stream=s), a)
        gb = unpermute_numpy(run_unpermute(b, workspace=ws, stream=s), b)
        ga2 = unpermute_numpy(run_unpermute(a, workspace=ws, stream=s), a)
    assert_unpermute_equal(ga, oracle.unpermute(a), a)
    assert_unpermute_equal(gb, oracle.unpermute(b), b)
    assert_unpermute_equal(ga2, oracle.unpermute(a), a)
