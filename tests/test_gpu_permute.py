"""Routing-map permute on the GPU vs the oracle, bit for bit, and the
GPU permute -> unpermute chain vs the oracle's."""
import numpy as np
import pytest
import torch

import oracle
import workloads as w

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import unpermute_stable_counting_gb300 as usc  # noqa: E402
from _gpu_util import (assert_unpermute_equal, float_numpy, float_tensor, to_dev,  # noqa: E402
                       unpermute_numpy)


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def routing(T, Eu, lo, hi, seed):
    rng = np.random.default_rng(seed)
    m = np.zeros((T, Eu), np.int8)
    for t in range(T):
        m[t, rng.choice(Eu, size=int(rng.integers(lo, hi + 1)), replace=False)] = 1
    return m


def check(x, m, dt, **kw):
    ref = oracle.permute(x, m, tokenDtype=dt, **kw)
    got = usc.moe_permute(float_tensor(x, dt), to_dev(m), topk=kw.get("topK", 0),
                          padded_mode=bool(kw.get("padded", 0)), capacity=kw.get("capacity", 0))
    torch.cuda.synchronize()
    rows = int(got["permutedRows"].item())
    assert rows == ref["rows"]
    assert np.array_equal(got["sortedIndices"].cpu().numpy(), ref["sortedIndices"])
    gp = float_numpy(got["permutedTokens"], dt)
    if kw.get("padded", 0):
        assert np.array_equal(gp.view(np.uint8), ref["permuted"].view(np.uint8))
    else:
        assert np.array_equal(gp[:rows].view(np.uint8), ref["permuted"][:rows].view(np.uint8))
    return got, ref


def test_hand_worked_example():
    x = np.array([[1.0, 2.0], [3.0, 4.0], [5.0, 6.0]], np.float32)
    m = np.array([[1, 1], [0, 1], [1, 0]], np.int8)
    got, _ = check(x, m, 3, topK=2)
    assert got["sortedIndices"].tolist() == [0, 2, 3, -1, 1, -1]
    check(x, m, 3, padded=1, capacity=1)
    check(x, m, 3, padded=1, capacity=3)


@pytest.mark.parametrize("dt", [0, 1, 3])
@pytest.mark.parametrize("Eu,k", [(10, 4), (64, 8), (100, 6), (8192, 3)])
def test_not_padded(dt, Eu, k):
    T, H = 300, 136
    m = routing(T, Eu, 0, k, seed=Eu + dt)
    check(w.normal_rows(T, H, dt, seed=dt), m, dt, topK=k)


@pytest.mark.parametrize("dt", [0, 1, 3])
@pytest.mark.parametrize("cap", [1, 7, 40])
def test_padded_with_drops(dt, cap):
    T, Eu, H = 257, 24, 72
    m = routing(T, Eu, 1, 5, seed=cap + 10 * dt)
    check(w.normal_rows(T, H, dt, seed=dt), m, dt, padded=1, capacity=cap)


@pytest.mark.parametrize("H", [1, 7, 33])
def test_odd_hidden(H):
    m = routing(70, 12, 0, 4, seed=H)
    check(w.normal_rows(70, H, 1, seed=H), m, 1, topK=4)
    check(w.normal_rows(70, H, 0, seed=H), m, 0, padded=1, capacity=9)


def test_more_experts_than_topk_and_overflowing_rows():
    x = w.normal_rows(40, 16, 3, seed=2)
    m = routing(40, 20, 3, 9, seed=4)            # some tokens over topK = 4
    check(x, m, 3, topK=4)
    m = np.ones((40, 20), np.int8)               # 800 pairs, 40 * 2 = 80 rows
    check(x, m, 3, topK=2)


@pytest.mark.parametrize("padded", [0, 1])
def test_permute_then_unpermute_chain(padded):
    """GPU permute -> GPU unpermute (with probs) vs the oracle's chain."""
    T, Eu, H = 512, 32, 256
    x = w.normal_rows(T, H, 1, seed=7)
    if padded:
        u = w.make_unpermute_padded(T=T, Eu=Eu, k=4, H=H, dtype=1, probs_dtype=3, mult=5, seed=8)
        m, probs, kw = u["routingMap"], u["probs"], dict(padded=1, capacity=u["n"] // Eu)
    else:
        u = w.make_unpermute_topk(T=T, k=8, Eu=Eu, H=H, dtype=1, probs_dtype=1, choices=(4, 8), seed=8)
        m, probs, kw = u["routingMap"], u["probs"], dict(topK=8)
    ref_p = oracle.permute(x, m, tokenDtype=1, **kw)
    rows = ref_p["permuted"].shape[0]
    pdt = 3 if padded else 1
    ui = dict(permuted=ref_p["permuted"], sortedIndices=ref_p["sortedIndices"], routingMap=m,
              probs=probs, permutedRows=rows, H=H, tokenDtype=1, n=rows, probsDtype=pdt, T=T, Eu=Eu,
              padded=padded)
    ref_u = oracle.unpermute(ui)
    gp = usc.moe_permute(float_tensor(x, 1), to_dev(m), topk=kw.get("topK", 0),
                         padded_mode=bool(padded), capacity=kw.get("capacity", 0))
    if not padded:
        # rows past the pairs are not written by the permute; the unpermute never reads them
        gp["permutedTokens"][int(gp["permutedRows"].item()):] = 0
    gu = usc.moe_unpermute(gp["permutedTokens"], gp["sortedIndices"], to_dev(m), float_tensor(probs, pdt),
                           padded_mode=bool(padded))
    torch.cuda.synchronize()
    assert_unpermute_equal(unpermute_numpy(gu, ui), ref_u, ui)
