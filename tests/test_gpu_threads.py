"""Calls from several host threads at once, each on its own stream. The
not-padded unpermute forks its index sort onto the library's one auxiliary
stream per device and joins it back with shared events under a lock; two
threads must still each get their own, correct results. (ctypes releases the
interpreter lock during the library calls, so the calls overlap.)"""
import threading

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


def unpermute_case(seed):
    u = w.make_unpermute_topk(T=300, k=8, Eu=32, H=200, dtype=1, probs_dtype=1, choices=(3, 8), seed=seed)
    g = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev())
    b = lambda a: g(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    d = dict(perm=b(u["permuted"]), si=g(u["sortedIndices"]), rm=g(u["routingMap"]), pr=b(u["probs"]))
    return u, d


def batching_case(seed):
    inp = w.make_batching(A=3, BS=16, K1=9, E=48, H=136, dtype=1, layerNum=1, layer_id=0, ids="zipf",
                          mask=0.1, session=3, micro=16, seed=seed)
    g = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev())
    d = dict(ids=g(inp["expert_ids"]), td=g(inp["token_data"]), sess=g(inp["session_in"]),
             micro=g(inp["micro_in"]), tok=g(inp["token_in"]))
    return inp, d


def test_two_threads_unpermute_and_batching():
    cases = [unpermute_case(s) for s in (11, 12)]
    bcases = [batching_case(s) for s in (13, 14)]
    refs = [oracle.unpermute(u) for u, _ in cases]
    brefs = [oracle.batching(inp) for inp, _ in bcases]
    errors, results = [], [None, None]
    start = threading.Barrier(2)

    def worker(j):
        try:
            u, d = cases[j]
            inp, bd = bcases[j]
            stream = torch.cuda.Stream()
            outs = []
            start.wait()
            with torch.cuda.stream(stream):
                for _ in range(20):
                    o = usc.moe_unpermute(d["perm"], d["si"], d["rm"], d["pr"], padded_mode=False)
                    bo = usc.ffnwb_batching(bd["ids"], bd["td"], bd["sess"], bd["micro"],
                                            expert_num=inp["expertNum"],
                                            max_out_shape=(inp["A"], inp["BS"], inp["K1"], inp["H"]),
                                            token_dtype=1, layer_num=1, layer_id=0, token_ids=bd["tok"])
                    outs.append((o, bo))
            stream.synchronize()
            results[j] = outs
        except Exception as exc:  # reported by the main thread
            errors.append(exc)

    threads = [threading.Thread(target=worker, args=(j,)) for j in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    assert not errors, errors
    for j in range(2):
        ref, bref = refs[j], brefs[j]
        U = bref["actualTokenNum"]
        for o, bo in results[j]:
            assert np.array_equal(float_numpy(o["unpermutedTokens"], 1), ref["unpermuted"])
            assert np.array_equal(o["outIndex"].cpu().numpy(), ref["outIndex"])
            assert np.array_equal(o["permuteTokenId"].cpu().numpy(), ref["permuteTokenId"])
            assert int(bo["actualTokenNum"][0]) == U
            assert np.array_equal(bo["groupList"].cpu().numpy(), bref["groupList"])
            y = bo["y"].view(torch.uint8).cpu().numpy().reshape(bref["y"].shape[0], -1)
            assert np.array_equal(y[:U], bref["y"][:U])
