"""Round trip on the GPU: batching, then the not-padded unpermute of its
output y with the slot -> row map as sortedIndices, against the same chain
run by the oracle."""
import numpy as np
import pytest
import torch

import oracle
import workloads as w

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import unpermute_stable_counting_gb300 as usc  # noqa: E402
from _gpu_util import (assert_batching_equal, assert_unpermute_equal, batching_numpy,  # noqa: E402
                       float_tensor, run_batching, to_dev, unpermute_numpy)


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def roundtrip(spec):
    inp = w.make_batching(**spec)
    bref = oracle.batching(inp)
    res = run_batching(inp)
    assert_batching_equal(batching_numpy(res, inp), bref)
    T, k = inp["A"] * inp["BS"], inp["K1"]
    El = inp["expertNum"] // max(inp["layerNum"], 1)
    unmasked = (inp["expert_ids"] >= 0) & (inp["expert_ids"] < El)
    pdt = w.ROUNDTRIP_PROBS_DTYPE
    rmap, probs = w.make_roundtrip_probs(T=T, k=k, slot_unmasked=unmasked, probs_dtype=pdt,
                                         seed=spec["seed"])
    dt = inp["tokenDtype"]
    # oracle chain
    u = dict(permuted=bref["y"].view(np.uint16).reshape(inp["Y"], inp["H"]),
             sortedIndices=bref["sortedIndices"], routingMap=rmap, probs=probs,
             permutedRows=inp["Y"], H=inp["H"], tokenDtype=dt, n=T * k, probsDtype=pdt, T=T, Eu=k,
             padded=0)
    uref = oracle.unpermute(u)
    # GPU chain: y and sortedIndices stay on the device
    got = usc.moe_unpermute(res["y"], res["sortedIndices"], to_dev(rmap), float_tensor(probs, pdt),
                            padded_mode=False)
    torch.cuda.synchronize()
    assert_unpermute_equal(unpermute_numpy(got, u), uref, u)


def test_roundtrip_small():
    roundtrip(dict(A=8, BS=16, K1=9, E=64, H=256, dtype=1, layerNum=4, layer_id=2, ids="zipf",
                   zipf_s=1.2, mask=0.05, session=8, micro=4, token_ids=True, seed=4))


@pytest.mark.slow
def test_roundtrip_full_size():
    roundtrip(w.ROUNDTRIP_BATCHING)
