"""The library's calls inside a CUDA graph: a batching + unpermute round trip,
the permute, and MoeUpdateExpert are captured once (torch.cuda.graph, which
captures the current stream; the not-padded unpermute forks its index sort
onto the library's auxiliary stream and joins it back inside the capture),
then replayed on new inputs copied into the captured buffers. Every replay
must equal the oracle on those inputs."""
import numpy as np
import pytest
import torch

import oracle
import workloads as w

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import unpermute_stable_counting_gb300 as usc  # noqa: E402

from _gpu_util import dev, float_numpy  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


SPEC = dict(A=4, BS=16, K1=9, E=64, H=264, dtype=1, layerNum=2, layer_id=1, ids="zipf", zipf_s=1.2,
            mask=0.1, session=4, micro=16, token_ids=True)


def roundtrip_inputs(seed):
    inp = w.make_batching(**SPEC, seed=seed)
    T, k = SPEC["A"] * SPEC["BS"], SPEC["K1"]
    El = SPEC["E"] // SPEC["layerNum"]
    unmasked = (inp["expert_ids"] >= 0) & (inp["expert_ids"] < El)
    rmap, probs = w.make_roundtrip_probs(T=T, k=k, slot_unmasked=unmasked, probs_dtype=1, seed=seed)
    return inp, rmap, probs


def oracle_roundtrip(inp, rmap, probs):
    b = oracle.batching(inp)
    T, k, H = SPEC["A"] * SPEC["BS"], SPEC["K1"], SPEC["H"]
    u = dict(permuted=b["y"].view(np.uint16).reshape(inp["Y"], H), sortedIndices=b["sortedIndices"],
             routingMap=rmap, probs=probs, permutedRows=inp["Y"], H=H, tokenDtype=1, n=T * k,
             probsDtype=1, T=T, Eu=k, padded=0)
    return b, oracle.unpermute(u)


def test_roundtrip_graph_replays():
    inp, rmap, probs = roundtrip_inputs(1)
    T, k, H, Y, E = SPEC["A"] * SPEC["BS"], SPEC["K1"], SPEC["H"], inp["Y"], SPEC["E"]
    shape = (SPEC["A"], SPEC["BS"], SPEC["K1"], H)
    g = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev())
    d = dict(ids=g(inp["expert_ids"]), td=g(inp["token_data"]).view(torch.bfloat16).view(Y, H),
             sess=g(inp["session_in"]), micro=g(inp["micro_in"]), tok=g(inp["token_in"]), rmap=g(rmap),
             probs=g(probs.view(np.int16)).view(torch.bfloat16).view(T, k))
    bout = usc.batching_outputs(Y, H, E, 1, dev(), with_sorted_indices=True)
    uout = usc.unpermute_outputs(T, H, T * k, 1, 1, dev())
    bws = torch.empty(usc.batching_workspace_size(E, shape, 1, SPEC["layerNum"]), dtype=torch.uint8,
                      device=dev())
    uws = torch.empty(usc.unpermute_workspace_size(Y, H, 1, T * k, True, 1, T, k, False), dtype=torch.uint8,
                      device=dev())

    def step():
        usc.ffnwb_batching(d["ids"], d["td"], d["sess"], d["micro"], expert_num=E, max_out_shape=shape,
                           token_dtype=1, layer_num=SPEC["layerNum"], layer_id=SPEC["layer_id"],
                           token_ids=d["tok"], with_sorted_indices=True, out=bout, workspace=bws)
        usc.moe_unpermute(bout["y"], bout["sortedIndices"], d["rmap"], d["probs"], out=uout, workspace=uws)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()                                   # warm-up outside the capture (first-use setup)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for seed in (1, 2, 3):
        inp, rmap, probs = roundtrip_inputs(seed)
        new = dict(ids=inp["expert_ids"], td=inp["token_data"], sess=inp["session_in"], micro=inp["micro_in"],
                   tok=inp["token_in"], rmap=rmap, probs=probs.view(np.int16))
        for n, a in new.items():
            d[n].view(-1).view(torch.uint8).copy_(torch.from_numpy(np.ascontiguousarray(a)).view(-1)
                                                  .view(torch.uint8).to(dev()))
        graph.replay()
        torch.cuda.synchronize()
        bref, uref = oracle_roundtrip(inp, rmap, probs)
        U = bref["actualTokenNum"]
        assert int(bout["actualTokenNum"][0]) == U
        assert np.array_equal(bout["groupList"].cpu().numpy(), bref["groupList"])
        y = bout["y"].view(torch.uint8).cpu().numpy().reshape(Y, -1)
        assert np.array_equal(y[:U], bref["y"][:U])
        assert np.array_equal(bout["sortedIndices"].cpu().numpy(), bref["sortedIndices"])
        assert np.array_equal(float_numpy(uout["unpermutedTokens"], 1), uref["unpermuted"])
        assert np.array_equal(uout["outIndex"].cpu().numpy(), uref["outIndex"])
        assert np.array_equal(uout["permuteTokenId"].cpu().numpy(), uref["permuteTokenId"])


def test_permute_and_update_expert_graph_replays():
    T, Eu, H = 200, 24, 72
    u = w.make_unpermute_topk(T=T, k=6, Eu=Eu, H=8, dtype=1, probs_dtype=None, choices=(1, 6), seed=4)
    x = torch.empty((T, H), dtype=torch.bfloat16, device=dev())
    rm = torch.empty((T, Eu), dtype=torch.int8, device=dev())
    ue = w.make_update_expert(BS=64, K=8, moe_expert_num=32, world_size=8, place_per_rank=8, scales_dtype=3,
                              seed=5)
    ids = torch.empty(ue["expert_ids"].shape, dtype=torch.int32, device=dev())
    tab = torch.from_numpy(ue["table"]).to(dev())
    sc, thr, act = (torch.from_numpy(ue[n]).to(dev()) for n in ("scales", "threshold", "active"))
    ws = torch.empty(usc.permute_workspace_size(T, H, 1, Eu, 6), dtype=torch.uint8, device=dev())
    pout, uout = None, None

    def step():
        nonlocal pout, uout
        pout = usc.moe_permute(x, rm, topk=6, out=pout, workspace=ws)
        uout = usc.moe_update_expert(ids, tab, local_rank=3, world_size=8, balance_mode=1, scales=sc,
                                     threshold=thr, active=act, out=uout)

    rm.copy_(torch.from_numpy(u["routingMap"]).to(dev()))
    step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for seed in (6, 7):
        rng = np.random.default_rng(seed)
        xv = w.normal_rows(T, H, 1, seed=seed)
        mv = (rng.random((T, Eu)) < 0.2).astype(np.int8)
        idv = rng.integers(-1, 34, size=ue["expert_ids"].shape).astype(np.int32)
        x.view(torch.int16).copy_(torch.from_numpy(xv.view(np.int16)).to(dev()))
        rm.copy_(torch.from_numpy(mv).to(dev()))
        ids.copy_(torch.from_numpy(idv).to(dev()))
        graph.replay()
        torch.cuda.synchronize()
        ref = oracle.permute(xv, mv, tokenDtype=1, topK=6)
        assert np.array_equal(pout["sortedIndices"].cpu().numpy(), ref["sortedIndices"])
        rows = ref["rows"]
        assert int(pout["permutedRows"][0]) == rows
        got = pout["permutedTokens"].view(torch.int16).cpu().numpy().view(np.uint16)[:rows]
        assert np.array_equal(got, ref["permuted"][:rows])
        uref = oracle.update_expert(idv, ue["table"], local_rank=3, balance_mode=1, scales=ue["scales"],
                                    scales_dtype=3, threshold=ue["threshold"], active=ue["active"])
        assert np.array_equal(uout["balancedExpertIds"].cpu().numpy(), uref["balancedExpertIds"])
        assert np.array_equal(uout["balancedActiveMask"].cpu().numpy(), uref["balancedActiveMask"])
