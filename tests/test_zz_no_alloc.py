"""ffnwb_batching_noalloc: the batching for callers that cannot allocate
device memory when they call (for example an engine plugin whose host
reserved all device memory up front). It uses a fixed scratch array inside
the library instead of a caller-provided workspace. Its results must equal
the CPU oracle's and the regular entry point's, call after call, even though
every call reuses the same scratch array, and calls after the first on a
device must not change how much device memory is in use.

This file sorts last so that a run stopping at its first failure has already
run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads as w

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

MR_ERR_WORKSPACE = 561002


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    from unpermute_stable_counting_gb300 import _native
    return _native.lib()


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda:0")


def _outputs(inp):
    import unpermute_stable_counting_gb300 as usc
    return usc.batching_outputs(inp["Y"], inp["H"], inp["expertNum"], inp["tokenDtype"], "cuda:0",
                                with_sorted_indices=True)


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def noalloc_args(inp):
    """Device copies of the inputs and the outputs of one call."""
    d = dict(ids=_dev(inp["expert_ids"]), td=_dev(inp["token_data"]), sess=_dev(inp["session_in"]),
             micro=_dev(inp["micro_in"]),
             tok=_dev(inp["token_in"]) if inp.get("token_in") is not None else None,
             sc=_dev(inp["scales"]) if inp.get("scales") is not None else None)
    return d, _outputs(inp)


def call_noalloc(lib, inp, d, out):
    from unpermute_stable_counting_gb300 import _native
    shape = _native.int64_array((inp["A"], inp["BS"], inp["K1"], inp["H"]))
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.ffnwb_batching_noalloc(
        _p(d["ids"]), inp["layer_id"], _p(d["td"]), inp["row_stride"], _p(d["sc"]), 4,
        _p(d["sess"]), _p(d["micro"]), _p(d["tok"]), inp["expertNum"], shape, inp["tokenDtype"], 0,
        inp["layerNum"], _p(out["y"]), _p(out["groupList"]), _p(out["sessionIds"]),
        _p(out["microBatchIds"]), _p(out["tokenIds"]), _p(out["expertOffsets"]),
        _p(out.get("dynamicScale")), _p(out["actualTokenNum"]), _p(out["sortedIndices"]), stream)


def run_noalloc(lib, inp):
    d, out = noalloc_args(inp)
    st = call_noalloc(lib, inp, d, out)
    torch.cuda.synchronize()
    return st, out


def as_numpy(out, inp):
    o = {k: (v.cpu().numpy() if v is not None else None) for k, v in out.items() if k != "y"}
    o["y"] = out["y"].contiguous().view(torch.uint8).cpu().numpy().reshape(inp["Y"], -1)
    o["actualTokenNum"] = int(o["actualTokenNum"][0])
    return o


def assert_matches_oracle(out, inp):
    """Bit for bit: every batching output is an integer or a byte copy."""
    got, ref = as_numpy(out, inp), oracle.batching(inp)
    U = ref["actualTokenNum"]
    assert got["actualTokenNum"] == U
    for k in ("groupList", "sessionIds", "microBatchIds", "tokenIds", "expertOffsets", "sortedIndices"):
        assert np.array_equal(got[k], ref[k]), k
    assert np.array_equal(got["y"][:U], ref["y"][:U]), "y rows differ"
    if ref["dynamicScale"] is not None:
        assert np.array_equal(got["dynamicScale"][:U].view(np.uint32), ref["dynamicScale"][:U].view(np.uint32))


def run_regular(inp):
    import unpermute_stable_counting_gb300 as usc
    res = usc.ffnwb_batching(
        _dev(inp["expert_ids"]), _dev(inp["token_data"]), _dev(inp["session_in"]),
        _dev(inp["micro_in"]), expert_num=inp["expertNum"],
        max_out_shape=(inp["A"], inp["BS"], inp["K1"], inp["H"]), token_dtype=inp["tokenDtype"],
        layer_num=inp["layerNum"], layer_id=inp["layer_id"],
        token_ids=_dev(inp["token_in"]) if inp.get("token_in") is not None else None,
        scales=_dev(inp["scales"]) if inp.get("scales") is not None else None,
        token_row_stride=inp["row_stride"], with_sorted_indices=True)
    torch.cuda.synchronize()
    return res


def assert_same(a, b, Y):
    """Batching outputs are integers and byte copies: the tolerance is zero."""
    U = int(b["actualTokenNum"].item())
    assert int(a["actualTokenNum"].item()) == U
    for k in ("groupList", "sessionIds", "microBatchIds", "tokenIds", "expertOffsets",
              "sortedIndices"):
        assert torch.equal(a[k], b[k]), k
    ya = a["y"].view(torch.uint8).reshape(Y, -1)[:U]
    yb = b["y"].view(torch.uint8).reshape(Y, -1)[:U]
    assert torch.equal(ya, yb)
    if b.get("dynamicScale") is not None:
        assert torch.equal(a["dynamicScale"][:U].view(torch.int32), b["dynamicScale"][:U].view(torch.int32))


def two_workloads():
    # the INT8 decode workload (its sort takes the one-launch cooperative
    # form) and 8192 experts (8193 keys: the kernel chain)
    first = w.make_batching(**w.BATCHING_INT8_DECODE)
    second = w.make_batching(A=4, BS=16, K1=33, E=8192, H=136, dtype=w.DT_BF16, layerNum=1,
                             layer_id=0, ids="zipf", zipf_s=1.1, mask=0.1, session=4, micro=4,
                             seed=77)
    return first, second


def test_noalloc_matches_oracle_and_regular_entry_point_twice_in_a_row(lib):
    for inp in two_workloads():
        st, got = run_noalloc(lib, inp)
        assert st == 0
        assert_matches_oracle(got, inp)
        assert_same(got, run_regular(inp), inp["Y"])


def test_noalloc_calls_allocate_nothing(lib):
    """After a first call on the device (which loads the library's code and
    its scratch array under lazy module loading), further calls leave the
    device's free memory and the caching allocator's counts unchanged."""
    runs = [(inp,) + noalloc_args(inp) for inp in two_workloads()]
    for inp, d, out in runs:
        assert call_noalloc(lib, inp, d, out) == 0
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    alloc0, reserved0 = torch.cuda.memory_allocated(), torch.cuda.memory_reserved()
    for _ in range(3):
        for inp, d, out in runs:
            assert call_noalloc(lib, inp, d, out) == 0
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, (free0, free1)
    assert torch.cuda.memory_allocated() == alloc0
    assert torch.cuda.memory_reserved() == reserved0
    for inp, d, out in runs:
        assert_matches_oracle(out, inp)


def test_noalloc_rejects_work_beyond_its_scratch(lib):
    """A call that needs more scratch than the fixed array holds is refused
    before anything is launched."""
    from unpermute_stable_counting_gb300 import _native
    shape = _native.int64_array((1024, 64, 64, 16))   # 4M slots: far more than 4 MiB of scratch
    one = torch.zeros(16, dtype=torch.int32, device="cuda:0")
    st = lib.ffnwb_batching_noalloc(
        _p(one), 0, _p(one), 32, None, 4, _p(one), _p(one), None, 8192, shape, 1, 0, 1, _p(one),
        _p(one), _p(one), _p(one), _p(one), _p(one), None, _p(one), None,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == MR_ERR_WORKSPACE
