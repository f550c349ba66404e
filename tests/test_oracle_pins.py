"""Pins of the CPU oracle to things other than itself.

Each test ties one part of the oracle to what the pages or the mathematics fix:
the pages' worked examples (tests/golden/), library routines (numpy, torch),
closed forms, invariants and brute force on tiny inputs. None of them calls the
CUDA path.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as w

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------
# fp16 / bf16 conversions (library pins: numpy float16, torch bfloat16)
# ---------------------------------------------------------------------------

def _edge_floats():
    rng = np.random.default_rng(123)
    vals = [0.0, -0.0, 1.0, -1.0, 65504.0, 65519.99, 65520.0, 1e9, -1e9, np.inf, -np.inf,
            2.0**-24, 2.0**-25, 2.0**-25 * 1.0000001, 3 * 2.0**-26, 2.0**-14, 2.0**-14 - 2.0**-25,
            1.0 + 2.0**-11, 1.0 + 3 * 2.0**-11, 1.0 + 2.0**-8, 1.0 + 3 * 2.0**-8, 1.0e-40, -1.0e-45,
            3.0e38, -3.4e38]
    vals += list(rng.standard_normal(20000).astype(np.float32))
    vals += list((rng.standard_normal(20000) * 1e-5).astype(np.float32))
    vals += list((rng.standard_normal(5000) * 7e4).astype(np.float32))
    # exact ties of binary16 / bfloat16: midpoints between neighbours
    h = rng.integers(0, 0x7bff, 4000).astype(np.uint16)
    lo = h.view(np.float16).astype(np.float64)
    hi = (h + 1).view(np.float16).astype(np.float64)
    vals += list(((lo + hi) / 2).astype(np.float32))
    b = rng.integers(0, 0x7f7f, 4000).astype(np.uint32)
    lo = (b << 16).view(np.float32).astype(np.float64)
    hi = ((b + 1) << 16).view(np.float32).astype(np.float64)
    vals += list(((lo + hi) / 2).astype(np.float32))
    x = np.asarray(vals, dtype=np.float32)
    return np.concatenate([x, -x])


def test_half_to_float_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float32)
    got = oracle.half_to_float(bits)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_float_to_half_rne():
    x = _edge_floats()
    ref = x.astype(np.float16).view(np.uint16)
    got = oracle.float_to_half(x)
    assert np.array_equal(got, ref)
    assert np.isnan(oracle.half_to_float(oracle.float_to_half(np.array([np.nan], np.float32))))[0]


def test_bf16_to_float_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    got = oracle.bf16_to_float(bits)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_float_to_bf16_rne():
    x = _edge_floats()
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.float_to_bf16(x)
    assert np.array_equal(got, ref)


# ---------------------------------------------------------------------------
# Batching
# ---------------------------------------------------------------------------

def _batching_from_spec(A, BS, K1, E, H, dtype, ids, layerNum=1, layer_id=0, sessions=None,
                        micros=None, token_in=None, fill_bits=None, seed=0):
    Y = A * BS * K1
    es = w.ELEM_BYTES[dtype]
    if fill_bits is not None:
        td = np.full((Y, H), fill_bits, dtype=np.uint16).view(np.uint8).reshape(Y, H * es)
    else:
        td = np.random.default_rng(seed).integers(0, 256, size=(Y, H * es + (4 if dtype == 2 else 0)),
                                                   dtype=np.uint8)
    return dict(expert_ids=np.asarray(ids, dtype=np.int32), layer_id=layer_id, token_data=td,
                row_stride=td.shape[1], scales=None,
                session_in=np.zeros(Y, np.int32) if sessions is None else np.asarray(sessions, np.int32),
                micro_in=np.zeros(Y, np.int32) if micros is None else np.asarray(micros, np.int32),
                token_in=token_in, expertNum=E, A=A, BS=BS, K1=K1, H=H, tokenDtype=dtype,
                layerNum=layerNum, Y=Y)


def test_batching_page_example():
    """The example program of the batching page, outputs derived by hand."""
    g = json.load(open(os.path.join(GOLDEN, "ffnwb_example.json")))
    p = g["inputs"]
    Y = p["A"] * p["BS"] * p["K1"]
    inp = _batching_from_spec(p["A"], p["BS"], p["K1"], p["E"], p["H"], p["tokenDtype"],
                              ids=np.arange(Y) % p["E"], fill_bits=1)
    o = oracle.batching(inp, with_gather_idx=True)
    assert o["groupList"].tolist() == [[e, 9] for e in range(8)]
    assert o["actualTokenNum"] == 72
    expect_g = np.array([e + 8 * r for e in range(8) for r in range(9)], dtype=np.int32)
    assert np.array_equal(o["gather_idx"], expect_g)
    assert np.array_equal(o["tokenIds"], expect_g)
    assert np.array_equal(o["expertOffsets"], np.arange(Y) % 9)
    assert np.all(o["y"].view(np.uint16) == 1)
    assert np.all(o["sessionIds"] == 0) and np.all(o["microBatchIds"] == 0)


def _brute_batching(ids, E, layerNum, layer_id):
    """Hand enumeration: walk the key values in ascending order and, for each,
    the slots in ascending order."""
    L = max(layerNum, 1)
    El = E // L
    keys = [layer_id * El + int(v) if 0 <= int(v) < El else E for v in ids]
    order = []
    for val in range(E + 1):
        for s in range(len(ids)):
            if keys[s] == val:
                order.append(s)
    return keys, order


@pytest.mark.parametrize("seed", range(40))
def test_batching_brute_force_tiny(seed):
    rng = np.random.default_rng(1000 + seed)
    A, BS, K1 = int(rng.integers(1, 3)), int(rng.integers(1, 4)), int(rng.integers(1, 4))
    Y = A * BS * K1
    layerNum = int(rng.choice([0, 1, 2, 4]))
    L = max(layerNum, 1)
    El = int(rng.integers(1, 4))
    E = El * L
    layer_id = int(rng.integers(0, L))
    choices = list(range(El)) + [-1, El, 2**31 - 1, -2**31]
    ids = rng.choice(choices, size=Y)
    sess = rng.integers(0, 5, size=Y)
    micro = rng.integers(0, 5, size=Y)
    tok = rng.integers(0, 1000, size=Y).astype(np.int32) if seed % 2 else None
    dt = int(rng.choice([0, 1, 2]))
    inp = _batching_from_spec(A, BS, K1, E, 3, dt, ids, layerNum, layer_id, sess, micro, tok, seed=seed)
    o = oracle.batching(inp, with_gather_idx=True)
    keys, order = _brute_batching(ids, E, layerNum, layer_id)
    U = sum(1 for k in keys if k < E)
    assert list(o["gather_idx"]) == order
    assert o["actualTokenNum"] == U
    rows = []
    for i, s in enumerate(order[:U]):
        if not rows or rows[-1][0] != keys[s]:
            rows.append([keys[s], 0])
        rows[-1][1] += 1
    rows += [[0, 0]] * (E - len(rows))
    assert o["groupList"].tolist() == rows
    td = inp["token_data"]
    H = 3
    es = w.ELEM_BYTES[dt]
    for i in range(Y):
        if i < U:
            s = order[i]
            assert bytes(o["y"][i]) == bytes(td[s, :H * es])
            assert o["sessionIds"][i] == sess[s] and o["microBatchIds"][i] == micro[s]
            assert o["tokenIds"][i] == (tok[s] if tok is not None else s)
            first = next(j for j in range(U) if keys[order[j]] == keys[s])
            assert o["expertOffsets"][i] == i - first
            if dt == 2:
                assert o["dynamicScale"][i].tobytes() == bytes(td[s, H:H + 4])
        else:
            assert o["sessionIds"][i] == -1 and o["tokenIds"][i] == -1
            assert o["microBatchIds"][i] == -1 and o["expertOffsets"][i] == -1
    inv = [-1] * Y
    for i in range(U):
        inv[order[i]] = i
    assert list(o["sortedIndices"]) == inv


def _check_batching_invariants(inp, o):
    ids = inp["expert_ids"].astype(np.int64)
    E = inp["expertNum"]
    L = max(inp["layerNum"], 1)
    El = E // L
    valid = (ids >= 0) & (ids < El)
    key = np.where(valid, inp["layer_id"] * El + ids, E)
    U = int(valid.sum())
    g = o["gather_idx"].astype(np.int64)
    # library pin: numpy's stable argsort gives the same permutation
    assert np.array_equal(g, np.argsort(key, kind="stable"))
    # sum of counts = actual token num = U
    gl = o["groupList"]
    assert int(gl[:, 1].sum()) == o["actualTokenNum"] == U
    # gather_idx[:U] is a permutation of the unmasked slots, keys nondecreasing,
    # slots increasing inside a group
    assert np.array_equal(np.sort(g[:U]), np.nonzero(valid)[0])
    ks = key[g[:U]]
    assert np.all(np.diff(ks) >= 0)
    same = np.diff(ks) == 0
    assert np.all(np.diff(g[:U])[same] > 0)
    # group list compacted, strictly increasing keys, offsets agree
    G = int((gl[:, 1] > 0).sum())
    assert np.all(gl[G:] == 0) and np.all(np.diff(gl[:G, 0]) > 0)
    assert np.array_equal(np.repeat(gl[:G, 0], gl[:G, 1]), ks)
    off = np.concatenate([np.arange(c) for c in gl[:G, 1]]) if G else np.zeros(0, np.int64)
    assert np.array_equal(o["expertOffsets"][:U], off)
    assert np.all(o["expertOffsets"][U:] == -1)
    # y rows are byte copies of the source rows
    rb = o["y"].shape[1]
    assert np.array_equal(o["y"][:U], inp["token_data"][g[:U], :rb])
    # the multiset of session / micro ids of the unmasked slots is preserved
    assert np.array_equal(np.sort(o["sessionIds"][:U]), np.sort(inp["session_in"][valid]))
    assert np.array_equal(np.sort(o["microBatchIds"][:U]), np.sort(inp["micro_in"][valid]))
    if inp["tokenDtype"] == 2:
        H = inp["H"]
        sc = inp["token_data"][:, H:H + 4].copy().view(np.float32).ravel() if inp["scales"] is None \
            else inp["scales"]
        assert np.array_equal(o["dynamicScale"][:U].view(np.uint32), sc[g[:U]].view(np.uint32))


def test_batching_invariants_tiny_config():
    inp = w.make_batching(**w.BATCHING_TINY)
    _check_batching_invariants(inp, oracle.batching(inp, with_gather_idx=True))


@pytest.mark.parametrize("E,layerNum,dtype,sep", [(256, 1, 2, False), (1024, 4, 1, False),
                                                   (8192, 1, 0, False), (64, 2, 2, True)])
def test_batching_invariants_medium(E, layerNum, dtype, sep):
    inp = w.make_batching(A=8, BS=16, K1=9, E=E, H=40, dtype=dtype, layerNum=layerNum,
                          layer_id=layerNum - 1, ids="zipf", zipf_s=1.2, mask=0.2, session=8,
                          micro=4, seed=E + layerNum, separate_scales=sep)
    _check_batching_invariants(inp, oracle.batching(inp, with_gather_idx=True))


def test_batching_all_masked_and_none_masked():
    inp = w.make_batching(A=2, BS=4, K1=3, E=16, H=8, dtype=0, mask=1.0, seed=5)
    o = oracle.batching(inp, with_gather_idx=True)
    assert o["actualTokenNum"] == 0 and np.all(o["groupList"] == 0)
    assert np.all(o["tokenIds"] == -1) and np.all(o["sortedIndices"] == -1)
    inp = w.make_batching(A=2, BS=4, K1=3, E=1, H=8, dtype=1, mask=0.0, seed=6)
    o = oracle.batching(inp, with_gather_idx=True)
    assert o["actualTokenNum"] == 24 and o["groupList"].tolist() == [[0, 24]]
    assert np.array_equal(o["gather_idx"], np.arange(24))


# ---------------------------------------------------------------------------
# Unpermute
# ---------------------------------------------------------------------------

def _f32(bits, dt):
    if dt == 3:
        return np.asarray(bits, np.float32)
    if dt == 0:
        return np.asarray(bits, np.uint16).view(np.float16).astype(np.float32)
    return torch.from_numpy(np.asarray(bits, np.uint16).view(np.int16)).view(torch.bfloat16).float().numpy()


def _store(x32, dt):
    if dt == 3:
        return x32.astype(np.float32)
    tdt = torch.float16 if dt == 0 else torch.bfloat16
    return torch.from_numpy(np.ascontiguousarray(x32, np.float32)).to(tdt).view(torch.int16).numpy().view(np.uint16)


def test_unpermute_page_example():
    g = json.load(open(os.path.join(GOLDEN, "unpermute_example.json")))
    p = g["inputs"]
    inp = dict(permuted=np.asarray(p["permuted"], np.float32),
               sortedIndices=np.asarray(p["sortedIndices"], np.int32),
               routingMap=np.asarray(p["routingMap"], np.int8), probs=np.asarray(p["probs"], np.float32),
               permutedRows=2, H=2, tokenDtype=3, n=2, probsDtype=3, T=2, Eu=2, padded=1)
    o = oracle.unpermute(inp)
    ex = g["expected_by_formula"]
    assert o["unpermuted"].tolist() == ex["unpermuted"]
    assert o["outIndex"].tolist() == ex["outIndex"]
    assert o["permuteTokenId"].tolist() == ex["permuteTokenId"]
    assert o["permuteProbs"].tolist() == ex["permuteProbs"]


def _rand_unpermute_topk(seed, T=24, k=5, Eu=7, H=6, dt=1, pdt=1, probs=True, rows=None, extra_invalid=True):
    inp = w.make_unpermute_topk(T=T, k=k, Eu=Eu, H=H, dtype=dt, probs_dtype=pdt if probs else None,
                                choices=(1, 2, 3, k), seed=seed, rows=rows)
    if extra_invalid:
        rng = np.random.default_rng(seed)
        si = inp["sortedIndices"]
        pick = rng.random(si.size) < 0.1
        si[pick] = rng.choice([-5, -1, inp["permutedRows"], inp["permutedRows"] + 7], size=int(pick.sum()))
    return inp


@pytest.mark.parametrize("seed", range(12))
def test_masked_select_matches_torch(seed):
    """Branch (2) permuteProbs = probs.T.maskedSelect(routingMap.T): pinned to
    torch.masked_select on the transposed tensors, truncated / zero padded to n."""
    inp = _rand_unpermute_topk(seed, dt=[0, 1, 3][seed % 3], pdt=[0, 3, 1, 3][seed % 4])
    if seed % 5 == 0:  # more ones than slots: truncation
        inp["routingMap"][:] = 1
    o = oracle.unpermute(inp)
    pr = torch.from_numpy(_f32(inp["probs"], inp["probsDtype"]).astype(np.float64))
    m = torch.from_numpy(inp["routingMap"] != 0)
    sel = torch.masked_select(pr.T, m.T).numpy()
    n = inp["n"]
    ref = np.zeros(n)
    ref[:min(n, sel.size)] = sel[:n]
    assert np.array_equal(_f32(o["permuteProbs"], inp["probsDtype"]).astype(np.float64), ref)


@pytest.mark.parametrize("seed", range(12))
def test_sort_outputs_match_numpy_stable_argsort(seed):
    rng = np.random.default_rng(seed)
    padded = seed % 2
    if padded:
        inp = w.make_unpermute_padded(T=32, Eu=8, k=2, H=4, dtype=0, probs_dtype=None, mult=3, seed=seed)
        si = inp["sortedIndices"]
        si[rng.random(si.size) < 0.15] = rng.choice([-1, 32, 99])
        si[rng.random(si.size) < 0.3] = rng.integers(0, 32)  # duplicates
        o = oracle.unpermute(inp)
        key = np.where((si >= 0) & (si < inp["T"]), si, inp["T"])
        order = np.argsort(key, kind="stable")
        assert np.array_equal(o["outIndex"], order)
        assert np.array_equal(o["permuteTokenId"], si[order])
    else:
        inp = _rand_unpermute_topk(seed, probs=False)
        si = inp["sortedIndices"]
        si[rng.random(si.size) < 0.2] = rng.integers(0, inp["permutedRows"])  # duplicates
        o = oracle.unpermute(inp)
        key = np.where((si >= 0) & (si < inp["permutedRows"]), si, -1)
        order = np.argsort(key, kind="stable")
        assert np.array_equal(o["outIndex"], order)
        assert np.array_equal(o["permuteTokenId"], order // (inp["permutedRows"] // inp["T"]))


def _fp64_reference(inp, pp64):
    """Weighted sum in float64 with numpy's unbuffered scatter-add, and the
    bound sum |terms| used for the tolerance."""
    T, H = inp["T"], inp["H"]
    x = _f32(inp["permuted"], inp["tokenDtype"]).reshape(-1, H).astype(np.float64)
    si = inp["sortedIndices"].astype(np.int64)
    n = inp["n"]
    ref = np.zeros((T, H))
    mag = np.zeros((T, H))
    if inp["padded"]:
        valid = (si >= 0) & (si < T)
        rows = np.nonzero(valid)[0]
        tok = si[rows]
        wgt = pp64[rows] if pp64 is not None else np.ones(rows.size)
    else:
        k = inp["permutedRows"] // T
        valid = (si >= 0) & (si < inp["permutedRows"])
        slots = np.nonzero(valid)[0]
        rows = si[slots]
        tok = slots // k
        wgt = pp64[slots] if pp64 is not None else np.ones(slots.size)
    np.add.at(ref, tok, x[rows] * wgt[:, None])
    np.add.at(mag, tok, np.abs(x[rows] * wgt[:, None]))
    return ref, mag


@pytest.mark.parametrize("seed", range(16))
def test_accumulation_matches_fp64(seed):
    """The fp32 accumulation against a float64 numpy scatter-add of the same
    terms, within fp32 accumulation error plus the final cast's half ulp.
    A wrong row, token, weight or sign fails this by O(1)."""
    dt = [0, 1, 3][seed % 3]
    padded = seed % 2
    has_probs = seed % 4 < 2
    if padded:
        inp = w.make_unpermute_padded(T=64, Eu=16, k=4, H=24, dtype=dt,
                                      probs_dtype=(3 if seed % 3 else dt) if has_probs else None,
                                      mult=5, seed=seed)
    else:
        inp = _rand_unpermute_topk(seed, T=40, k=6, Eu=9, H=24, dt=dt, pdt=3 if seed % 3 else dt,
                                   probs=has_probs)
    o = oracle.unpermute(inp)
    pp64 = _f32(o["permuteProbs"], inp["probsDtype"]).astype(np.float64) if has_probs else None
    if has_probs and not padded:
        # pin the weights to the library masked_select before using them
        pr = torch.from_numpy(_f32(inp["probs"], inp["probsDtype"]).astype(np.float64))
        sel = torch.masked_select(pr.T, torch.from_numpy(inp["routingMap"] != 0).T).numpy()
        ref_pp = np.zeros(inp["n"])
        ref_pp[:min(inp["n"], sel.size)] = sel[:inp["n"]]
        assert np.array_equal(pp64, ref_pp)
    if has_probs and padded:
        # pad-kernel lookup probs[sortedIndices[i], i // capacity], checked
        # against the expert that owns row i in the capacity layout
        cap = inp["n"] // inp["Eu"]
        pr = _f32(inp["probs"], inp["probsDtype"]).astype(np.float64)
        for i, t in enumerate(inp["sortedIndices"]):
            e = i // cap
            assert pp64[i] == (pr[t, e] if 0 <= t < inp["T"] else 0.0)
    ref, mag = _fp64_reference(inp, pp64)
    got = _f32(o["unpermuted"], dt).astype(np.float64)
    k = max(1, inp["n"] // inp["T"])
    half_ulp = {0: 2.0**-11, 1: 2.0**-8, 3: 0.0}[dt]
    tol = (k + 2) * 2.0**-24 * mag + half_ulp * np.abs(ref) + 1e-30
    assert np.all(np.abs(got - ref) <= tol * 1.0001 + (2.0**-24 if dt == 0 else 0.0))


def test_skip_rules():
    """Invalid indices and zero probs contribute nothing, even when the row
    they point at holds NaN or inf."""
    T, k, H = 3, 2, 4
    permuted = np.zeros((T * k, H), np.float32)
    permuted[0] = np.nan
    permuted[1] = np.inf
    permuted[2] = 1.5
    permuted[3] = -2.0
    si = np.array([0, 2, 1, 3, -1, 6], np.int32)  # slot 0 -> NaN row (weight 0), 2 -> inf row (weight 0)
    rmap = np.ones((T, k), np.int8)
    # permuteProbs = probs.T.maskedSelect(map.T) = [p00, p10, p20, p01, p11, p21]
    probs = np.array([[0.0, 0.5], [2.0, 0.25], [0.0, 1.0]], np.float32)
    pp = probs.T.ravel()  # [0, 2, 0, 0.5, 0.25, 1]
    assert pp[0] == 0 and pp[2] == 0
    inp = dict(permuted=permuted, sortedIndices=si, routingMap=rmap, probs=probs, permutedRows=T * k,
               H=H, tokenDtype=3, n=T * k, probsDtype=3, T=T, Eu=k, padded=0)
    o = oracle.unpermute(inp)
    out = o["unpermuted"]
    assert np.all(np.isfinite(out))
    assert np.array_equal(out[0], np.full(H, 1.5 * 2.0, np.float32))   # slot 1: row 2 * pp[1]
    assert np.array_equal(out[1], np.full(H, -2.0 * 0.5, np.float32))  # slot 3: row 3 * pp[3]; slot 2 skipped
    assert np.array_equal(out[2], np.zeros(H, np.float32))             # slot 4 = -1, slot 5 out of range


@pytest.mark.parametrize("dt", [0, 1, 3])
def test_row_permutation_special_case(dt):
    """Branch (4) with topK = 1 and no invalid slot is a row permutation:
    out[t] = permuted[sortedIndices[t]] bit for bit (0 + x is exact)."""
    T, H = 50, 16
    rng = np.random.default_rng(dt)
    x = w.normal_rows(T, H, dt, seed=7)
    si = rng.permutation(T).astype(np.int32)
    inp = dict(permuted=x, sortedIndices=si, routingMap=None, probs=None, permutedRows=T, H=H,
               tokenDtype=dt, n=T, probsDtype=dt, T=T, Eu=0, padded=0)
    o = oracle.unpermute(inp)
    ref = x[si]
    if dt == 3:
        assert np.array_equal(o["unpermuted"].view(np.uint32), ref.view(np.uint32))
    else:
        assert np.array_equal(o["unpermuted"], ref)


@pytest.mark.parametrize("dt,seed", [(1, 0), (0, 1), (1, 2)])
def test_roundtrip_closed_form(dt, seed):
    """unpermute(batching(x)) with the slot-column routing map equals, per
    token, the probs-weighted sum of the token's own slot rows. The closed form
    needs no sort: sequential fp32 adds over the token's k slots of
    token_data * maskedSelect weight (torch.masked_select), then one RNE cast."""
    A, BS, K1, H = 4, 8, 5, 12
    inp = w.make_batching(A=A, BS=BS, K1=K1, E=32, H=H, dtype=dt, layerNum=2, layer_id=1, ids="zipf",
                          zipf_s=1.2, mask=0.2, session=4, micro=4, seed=seed)
    b = oracle.batching(inp)
    T, k = A * BS, K1
    unmasked = (inp["expert_ids"] >= 0) & (inp["expert_ids"] < 16)
    rmap, probs = w.make_roundtrip_probs(T=T, k=k, slot_unmasked=unmasked, probs_dtype=dt, seed=seed)
    u = dict(permuted=b["y"], sortedIndices=b["sortedIndices"], routingMap=rmap, probs=probs,
             permutedRows=T * k, H=H, tokenDtype=dt, n=T * k, probsDtype=dt, T=T, Eu=k, padded=0)
    o = oracle.unpermute(u)
    # closed form
    pr = torch.from_numpy(_f32(probs, dt).astype(np.float32))
    pp = torch.masked_select(pr.T, torch.from_numpy(rmap != 0).T).numpy()
    w32 = np.zeros(T * k, np.float32)
    w32[:pp.size] = pp
    x = _f32(inp["token_data"].view(np.uint16), dt).reshape(T * k, H)
    acc = np.zeros((T, H), np.float32)
    for j in range(k):
        s = np.arange(T) * k + j
        use = unmasked[s] & (w32[s] != 0)
        term = (x[s] * w32[s][:, None]).astype(np.float32)
        acc = np.where(use[:, None], (acc + term).astype(np.float32), acc)
    assert np.array_equal(o["unpermuted"], _store(acc, dt))


def test_padded_roundtrip_weights_sum_to_one():
    """Padded round trip: if permuted[r] = x[sortedIndices[r]] then
    out[t] = x[t] * sum_e probs[t, e] = x[t] (Dirichlet rows sum to 1)."""
    T, Eu, k, H = 64, 16, 4, 10
    inp = w.make_unpermute_padded(T=T, Eu=Eu, k=k, H=H, dtype=3, probs_dtype=3, mult=5, seed=9)
    x = w.normal_rows(T, H, 3, seed=11)
    inp["permuted"] = np.ascontiguousarray(x[inp["sortedIndices"]])
    o = oracle.unpermute(inp)
    psum = inp["probs"].astype(np.float64).sum(axis=1)
    ref = x.astype(np.float64) * psum[:, None]
    assert np.allclose(o["unpermuted"], ref, rtol=1e-6, atol=1e-7)
    assert np.allclose(o["unpermuted"], x, rtol=1e-5, atol=1e-6)


@pytest.mark.parametrize("padded", [0, 1])
def test_accumulation_order_is_ascending(padded):
    """Terms are added in ascending slot (not padded) or row (padded) order.
    Hand-worked fp32 case: 0 + 1 + 1e8 - 1e8 = 0 in that order (1 is lost
    against 1e8), while the reverse order keeps the 1."""
    H = 4
    vals = np.array([1.0, 1e8, -1e8], np.float32)
    permuted = np.repeat(vals[:, None], H, axis=1).astype(np.float32)
    if padded:
        si = np.array([0, 0, 0], np.int32)       # token 0 three times, rows 0, 1, 2
        inp = dict(permuted=permuted, sortedIndices=si, routingMap=None, probs=None, permutedRows=3,
                   H=H, tokenDtype=3, n=3, probsDtype=3, T=1, Eu=0, padded=1)
    else:
        si = np.array([0, 1, 2], np.int32)       # one token, topK = 3
        inp = dict(permuted=permuted, sortedIndices=si, routingMap=None, probs=None, permutedRows=3,
                   H=H, tokenDtype=3, n=3, probsDtype=3, T=1, Eu=0, padded=0)
    o = oracle.unpermute(inp)
    assert np.array_equal(o["unpermuted"], np.zeros((1, H), np.float32))
    # reversed rows: 0 - 1e8 + 1e8 + 1 = 1
    inp["permuted"] = np.ascontiguousarray(permuted[::-1])
    o = oracle.unpermute(inp)
    assert np.array_equal(o["unpermuted"], np.ones((1, H), np.float32))
