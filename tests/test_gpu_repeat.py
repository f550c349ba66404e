"""Repeated unpermute calls on two streams at once: every result must equal
the first one bit for bit, and the first one the oracle. Covers each form of
the weights' maskedSelect (inside the gather-reduce, the cooperative kernel,
the three-kernel chain), the padded path and the no-probs path, with the
index sort forked onto the library's auxiliary stream by both streams."""
import numpy as np
import pytest
import torch

import oracle
import workloads as w

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import unpermute_stable_counting_gb300 as usc  # noqa: E402

from _gpu_util import assert_unpermute_equal, float_tensor, to_dev, unpermute_numpy  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


CASES = {
    "small_map": lambda: w.make_unpermute_topk(T=64, k=8, Eu=64, H=512, dtype=1, probs_dtype=1, seed=7),
    "one_kernel_select": lambda: w.make_unpermute_topk(T=3000, k=6, Eu=48, H=256, dtype=1, probs_dtype=3,
                                                       choices=(2, 6), seed=39),
    "select_chain": lambda: w.make_unpermute_topk(T=65600, k=2, Eu=64, H=8, dtype=1, probs_dtype=3,
                                                  choices=(1, 2), seed=41),
    "padded_slack": lambda: w.make_unpermute_padded(T=2048, Eu=32, k=2, H=64, dtype=0, probs_dtype=3,
                                                    mult=5, capacity=256, seed=42),
    "no_probs": lambda: w.make_unpermute_topk(T=300, k=8, Eu=32, H=200, dtype=1, probs_dtype=None,
                                              choices=(3, 8), seed=5),
}


@pytest.mark.parametrize("case", list(CASES))
def test_repeated_calls_on_two_streams(case):
    inp = CASES[case]()
    ref = oracle.unpermute(inp)
    probs = inp.get("probs")
    dt, pdt = inp["tokenDtype"], inp["probsDtype"]
    perm = float_tensor(inp["permuted"], dt)
    si = to_dev(inp["sortedIndices"])
    rm = to_dev(inp["routingMap"]) if probs is not None else None
    pr = float_tensor(probs, pdt) if probs is not None else None
    rs = None if probs is not None else (inp["T"], inp["H"])
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = [None, None]
    first = None
    for it in range(60):
        for j, st in enumerate(streams):
            with torch.cuda.stream(st):
                outs[j] = usc.moe_unpermute(perm, si, rm, pr, padded_mode=bool(inp["padded"]), restore_shape=rs,
                                            out=outs[j])
        if it % 10 == 9:
            torch.cuda.synchronize()
            for j in range(2):
                got = unpermute_numpy(outs[j], inp)
                if first is None:
                    assert_unpermute_equal(got, ref, inp)
                    first = got
                for k, v in got.items():
                    if v is not None:
                        assert np.array_equal(v.view(np.uint8), first[k].view(np.uint8)), (it, j, k)


def test_capture_on_one_stream_beside_eager_calls_on_another():
    """A not-padded unpermute captured on stream A while an eager one runs on
    stream B: each caller stream has its own auxiliary stream, so the eager
    call's sort fork does not touch the capture (with one auxiliary stream
    shared by both, the eager fork would record into a capturing stream).
    The replayed graph and the eager call must both equal the oracle."""
    a = w.make_unpermute_topk(T=512, k=8, Eu=64, H=256, dtype=1, probs_dtype=1, choices=(4, 8), seed=61)
    b = w.make_unpermute_topk(T=700, k=6, Eu=32, H=128, dtype=1, probs_dtype=1, choices=(2, 6), seed=62)

    def prep(inp):
        d = dict(perm=float_tensor(inp["permuted"], inp["tokenDtype"]), si=to_dev(inp["sortedIndices"]),
                 rm=to_dev(inp["routingMap"]), pr=float_tensor(inp["probs"], inp["probsDtype"]))
        n, T = inp["n"], inp["T"]
        d["out"] = usc.unpermute_outputs(T, inp["H"], n, inp["tokenDtype"], inp["probsDtype"], "cuda:0")
        ws = usc.unpermute_workspace_size(inp["permutedRows"], inp["H"], inp["tokenDtype"], n, True,
                                          inp["probsDtype"], T, inp["Eu"], False)
        d["ws"] = torch.empty(max(ws, 1), dtype=torch.uint8, device="cuda:0")
        return d

    da, db = prep(a), prep(b)
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()

    def call(d, st):
        usc.moe_unpermute(d["perm"], d["si"], d["rm"], d["pr"], padded_mode=False, out=d["out"],
                          workspace=d["ws"], stream=st)

    # first calls outside any capture create each stream's auxiliary stream
    call(da, sa)
    call(db, sb)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=sa, capture_error_mode="thread_local"):
        call(da, sa)
        call(db, sb)  # eager, on another stream, during the capture
    sb.synchronize()
    assert_unpermute_equal(unpermute_numpy(db["out"], b), oracle.unpermute(b), b)
    for v in da["out"].values():
        if v is not None:
            v.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert_unpermute_equal(unpermute_numpy(da["out"], a), oracle.unpermute(a), a)


def test_many_caller_streams():
    """Not-padded unpermutes on more caller streams than the library keeps
    auxiliary streams for (64 per device): past that the sort runs in the
    caller's stream. Every result must equal the oracle."""
    inp = w.make_unpermute_topk(T=300, k=6, Eu=24, H=64, dtype=1, probs_dtype=1, choices=(2, 6), seed=63)
    ref = oracle.unpermute(inp)
    perm = float_tensor(inp["permuted"], inp["tokenDtype"])
    si, rm, pr = to_dev(inp["sortedIndices"]), to_dev(inp["routingMap"]), float_tensor(inp["probs"], inp["probsDtype"])
    streams = [torch.cuda.Stream() for _ in range(72)]
    outs = []
    for st in streams:
        with torch.cuda.stream(st):
            outs.append(usc.moe_unpermute(perm, si, rm, pr, padded_mode=False))
    torch.cuda.synchronize()
    for o in outs:
        assert_unpermute_equal(unpermute_numpy(o, inp), ref, inp)
