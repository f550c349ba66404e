"""Pins of the routing-map permute oracle (the step the unpermute page names
as its producer, "MoeTokenUnpermuteWithRoutingMap 算子全解析", 算子定位)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as w


def test_hand_worked_example():
    """T=3 tokens, 2 experts, map [[1,1],[0,1],[1,0]], topK 2.
    Rows, expert-major: e0 -> tokens 0, 2 (rows 0, 1); e1 -> tokens 0, 1
    (rows 2, 3). Slots: t0 -> [0, 2], t1 -> [3, -1], t2 -> [1, -1].
    Padded with capacity 1: e0 keeps t0, e1 keeps t0."""
    x = np.array([[1.0, 2.0], [3.0, 4.0], [5.0, 6.0]], np.float32)
    m = np.array([[1, 1], [0, 1], [1, 0]], np.int8)
    o = oracle.permute(x, m, tokenDtype=3, topK=2)
    assert o["sortedIndices"].tolist() == [0, 2, 3, -1, 1, -1]
    assert o["permuted"].tolist() == [[1, 2], [5, 6], [1, 2], [3, 4], [0, 0], [0, 0]]
    assert o["rows"] == 4
    o = oracle.permute(x, m, tokenDtype=3, padded=1, capacity=1)
    assert o["sortedIndices"].tolist() == [0, 0]
    assert o["permuted"].tolist() == [[1, 2], [1, 2]] and o["rows"] == 2
    o = oracle.permute(x, m, tokenDtype=3, padded=1, capacity=3)
    assert o["sortedIndices"].tolist() == [0, 2, -1, 0, 1, -1]
    assert o["permuted"][2].tolist() == [0, 0] and o["rows"] == 4


@pytest.mark.parametrize("seed", range(6))
def test_rows_follow_library_nonzero_of_transposed_map(seed):
    rng = np.random.default_rng(seed)
    T, Eu, H, k = 37, 11, 5, 11
    m = (rng.random((T, Eu)) < 0.3).astype(np.int8)
    x = rng.standard_normal((T, H)).astype(np.float32)
    o = oracle.permute(x, m, tokenDtype=3, topK=k)
    nz = torch.nonzero(torch.from_numpy(m).T)          # (expert, token) pairs, expert-major
    toks = nz[:, 1].numpy()
    assert o["rows"] == len(toks)
    assert np.array_equal(o["permuted"][:len(toks)], x[toks])


@pytest.mark.parametrize("seed", range(4))
def test_slot_layout_matches_the_generators(seed):
    """The unpermute inputs drawn by workloads.py lay rows out the same way."""
    u = w.make_unpermute_topk(T=50, k=6, Eu=12, H=8, dtype=3, probs_dtype=None, choices=(1, 3, 6),
                              seed=seed)
    x = np.random.default_rng(seed).standard_normal((50, 8)).astype(np.float32)
    o = oracle.permute(x, u["routingMap"], tokenDtype=3, topK=6)
    assert np.array_equal(o["sortedIndices"], u["sortedIndices"])
    p = w.make_unpermute_padded(T=64, Eu=16, k=4, H=8, dtype=3, probs_dtype=None, mult=5, seed=seed)
    cap = p["n"] // 16
    x64 = np.random.default_rng(1).standard_normal((64, 8)).astype(np.float32)
    o = oracle.permute(x64, p["routingMap"], tokenDtype=3, padded=1, capacity=cap)
    assert np.array_equal(o["sortedIndices"], p["sortedIndices"])


@pytest.mark.parametrize("dt", [0, 1])
def test_unpermute_of_permute_without_probs_counts_copies(dt):
    """Branch (4) of the unpermute applied to the permute: each token gets its
    own row once per routed expert, so out[t] = RNE(n_t * x[t]) exactly (n_t <=
    8 copies of a 16-bit value add exactly in fp32)."""
    rng = np.random.default_rng(dt)
    T, Eu, H, k = 40, 10, 16, 8
    m = np.zeros((T, Eu), np.int8)
    for t in range(T):
        m[t, rng.choice(Eu, size=rng.integers(0, k + 1), replace=False)] = 1
    x = w.normal_rows(T, H, dt, seed=3)
    o = oracle.permute(x, m, tokenDtype=dt, topK=k)
    u = dict(permuted=o["permuted"], sortedIndices=o["sortedIndices"], routingMap=None, probs=None,
             permutedRows=T * k, H=H, tokenDtype=dt, n=T * k, probsDtype=dt, T=T, Eu=0, padded=0)
    out = oracle.unpermute(u)["unpermuted"]
    tdt = torch.float16 if dt == 0 else torch.bfloat16
    xf = torch.from_numpy(x.view(np.int16)).view(tdt).float()
    n = torch.from_numpy(m.sum(axis=1).astype(np.float32))[:, None]
    ref = (0.0 + xf * n).to(tdt).view(torch.int16).numpy().view(np.uint16)  # 0 + (-0) = +0
    assert np.array_equal(out, ref)


def test_padded_unpermute_of_permute_weights_sum_to_one():
    """Padded branch (1) on the permute of x with Dirichlet probs over each
    token's experts (no token dropped): out[t] = x[t] * sum_e probs[t, e] = x[t]."""
    p = w.make_unpermute_padded(T=128, Eu=16, k=4, H=12, dtype=3, probs_dtype=3, mult=5, seed=2)
    cap = p["n"] // 16
    x = np.random.default_rng(3).standard_normal((128, 12)).astype(np.float32)
    o = oracle.permute(x, p["routingMap"], tokenDtype=3, padded=1, capacity=cap)
    u = dict(p, permuted=o["permuted"], sortedIndices=o["sortedIndices"])
    out = oracle.unpermute(u)["unpermuted"]
    ref = x.astype(np.float64) * p["probs"].astype(np.float64).sum(axis=1)[:, None]
    assert np.allclose(out, ref, rtol=1e-6, atol=1e-7)


def test_tokens_over_topk_and_rows_over_capacity():
    """A token routed to more experts than topK keeps its first topK slots; a
    pair whose row is not below topK*T gets no slot."""
    x = np.arange(8, dtype=np.float32).reshape(4, 2)
    m = np.array([[1, 1, 1], [0, 0, 0], [0, 0, 0], [0, 0, 0]], np.int8)
    o = oracle.permute(x, m, tokenDtype=3, topK=2)
    # rows: e0 t0 -> 0, e1 t0 -> 1, e2 t0 -> 2; slots of t0: [0, 1] (the third is dropped)
    assert o["sortedIndices"].tolist() == [0, 1, -1, -1, -1, -1, -1, -1]
    assert o["rows"] == 3
    m = np.ones((4, 3), np.int8)                       # 12 pairs, topK*T = 4 rows
    o = oracle.permute(x, m, tokenDtype=3, topK=1)
    assert o["rows"] == 4
    assert o["sortedIndices"].tolist() == [0, 1, 2, 3]   # expert 0's rows, t0..t3
