"""Helpers of the GPU parity tests: run the CUDA path on the numpy inputs of
workloads.py and compare with the oracle's numpy outputs."""
import numpy as np
import torch

import unpermute_stable_counting_gb300 as usc

TORCH_DT = {0: torch.float16, 1: torch.bfloat16, 3: torch.float32}
# |got - ref| <= rtol * |ref| + atol, per token dtype (the stated tolerances)
TOL = {3: (1e-5, 1e-6), 0: (2.0**-10, 1e-4), 1: (2.0**-7, 1e-3)}


def dev():
    return torch.device("cuda:0")


def to_dev(a, d=None):
    return torch.from_numpy(np.ascontiguousarray(a)).to(d or dev())


def float_tensor(a, dt, d=None):
    """numpy storage (uint16 bits or float32) -> torch CUDA tensor of dtype dt."""
    a = np.ascontiguousarray(a)
    if dt == 3:
        return torch.from_numpy(a.astype(np.float32, copy=False)).to(d or dev())
    return torch.from_numpy(a.view(np.int16)).view(TORCH_DT[dt]).to(d or dev())


def float_numpy(t, dt):
    t = t.detach().cpu()
    if dt == 3:
        return t.numpy()
    return t.view(torch.int16).numpy().view(np.uint16)


def run_batching(inp, *, with_sorted=True, stream=None, workspace=None, out=None, token_ids=True,
                 token_data=None):
    d = dev()
    td = to_dev(inp["token_data"]) if token_data is None else token_data
    res = usc.ffnwb_batching(
        to_dev(inp["expert_ids"]), td, to_dev(inp["session_in"]), to_dev(inp["micro_in"]),
        expert_num=inp["expertNum"], max_out_shape=(inp["A"], inp["BS"], inp["K1"], inp["H"]),
        token_dtype=inp["tokenDtype"], layer_num=inp["layerNum"], layer_id=inp["layer_id"],
        token_ids=to_dev(inp["token_in"]) if (token_ids and inp.get("token_in") is not None) else None,
        scales=to_dev(inp["scales"]) if inp.get("scales") is not None else None,
        token_row_stride=inp["row_stride"], with_sorted_indices=with_sorted, stream=stream,
        workspace=workspace, out=out)
    torch.cuda.synchronize()
    return res


def batching_numpy(res, inp):
    Y = inp["Y"]
    o = {k: (v.cpu().numpy() if v is not None else None) for k, v in res.items() if k != "y"}
    o["y"] = res["y"].contiguous().view(torch.uint8).cpu().numpy().reshape(Y, -1)
    o["actualTokenNum"] = int(o["actualTokenNum"][0])
    return o


def assert_batching_equal(got, ref, with_sorted=True):
    U = ref["actualTokenNum"]
    assert got["actualTokenNum"] == U
    assert np.array_equal(got["groupList"], ref["groupList"])
    for k in ("sessionIds", "microBatchIds", "tokenIds", "expertOffsets"):
        assert np.array_equal(got[k], ref[k]), k
    if with_sorted:
        assert np.array_equal(got["sortedIndices"], ref["sortedIndices"])
    assert np.array_equal(got["y"][:U], ref["y"][:U]), "y rows differ"
    if ref["dynamicScale"] is not None:
        assert np.array_equal(got["dynamicScale"][:U].view(np.uint32),
                              ref["dynamicScale"][:U].view(np.uint32))


def offset_dev(a, offset):
    """A device copy of `a` starting `offset` bytes into its allocation."""
    raw = np.ascontiguousarray(a)
    buf = torch.zeros(raw.nbytes + offset, dtype=torch.uint8, device="cuda")
    buf[offset:] = torch.from_numpy(raw.view(np.uint8).reshape(-1)).cuda()
    return buf[offset:].view(TORCH_RAW[raw.dtype]).view(*raw.shape)


TORCH_RAW = {np.dtype(np.int8): torch.int8, np.dtype(np.uint8): torch.uint8}


def run_unpermute(inp, *, stream=None, workspace=None, out=None, pass_restore=None, map_offset=0):
    probs = inp.get("probs")
    dt, pdt = inp["tokenDtype"], inp["probsDtype"]
    rs = None
    if probs is None or pass_restore:
        rs = (inp["T"], inp["H"])
    rmap = None
    if probs is not None:
        rmap = offset_dev(inp["routingMap"], map_offset) if map_offset else to_dev(inp["routingMap"])
    res = usc.moe_unpermute(
        float_tensor(inp["permuted"], dt), to_dev(inp["sortedIndices"]),
        rmap,
        float_tensor(probs, pdt) if probs is not None else None,
        padded_mode=bool(inp["padded"]), restore_shape=rs, stream=stream, workspace=workspace,
        out=out)
    torch.cuda.synchronize()
    return res


def unpermute_numpy(res, inp):
    return dict(unpermuted=float_numpy(res["unpermutedTokens"], inp["tokenDtype"]),
                outIndex=res["outIndex"].cpu().numpy(),
                permuteTokenId=res["permuteTokenId"].cpu().numpy(),
                permuteProbs=(float_numpy(res["permuteProbs"], inp["probsDtype"])
                              if res.get("permuteProbs") is not None else None))


def as_f64(a, dt):
    if dt == 3:
        return np.asarray(a, np.float32).astype(np.float64)
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(TORCH_DT[dt])
    return t.double().numpy()


def assert_unpermute_equal(got, ref, inp, exact=True):
    dt = inp["tokenDtype"]
    assert np.array_equal(got["outIndex"], ref["outIndex"])
    assert np.array_equal(got["permuteTokenId"], ref["permuteTokenId"])
    if ref["permuteProbs"] is not None:
        assert np.array_equal(got["permuteProbs"].view(np.uint8), ref["permuteProbs"].view(np.uint8))
    g = as_f64(got["unpermuted"], dt)
    r = as_f64(ref["unpermuted"], dt)
    rtol, atol = TOL[dt]
    bad = ~(np.abs(g - r) <= rtol * np.abs(r) + atol)
    assert not bad.any(), f"{int(bad.sum())} elements outside the tolerance"
    if exact:
        # the kernels add the same rounded terms in the same order as the oracle
        assert np.array_equal(got["unpermuted"].view(np.uint8), ref["unpermuted"].view(np.uint8))
