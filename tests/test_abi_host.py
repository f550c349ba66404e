"""The C-ABI library loads, exports every declared entry point, and rejects
bad arguments on the host (no GPU needed: each call below returns before
anything touches the CUDA runtime)."""
import ctypes
import os
import re
import subprocess

import pytest

from unpermute_stable_counting_gb300 import _build, _native

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_reorder.h")

OK, NULLPTR, INVALID, INNER, CUDA, WORKSPACE, UNSUPPORTED = 0, 161001, 161002, 561103, 561001, 561002, 561003
FAKE = ctypes.c_void_p(0x1000)  # never dereferenced: the calls return before any launch


@pytest.fixture(scope="module")
def L():
    _build.build_library()
    return _native.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b([A-Za-z_]\w*)\s*\(", text, flags=re.M))
                  - {"defined"})


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert set(names) == set(_native.SIGNATURES), names
    nm = subprocess.run(["nm", "-D", "--defined-only", _build.LIB_PATH], capture_output=True,
                        text=True, check=True).stdout
    exported = set(re.findall(r" T (\w+)$", nm, flags=re.M))
    for n in names:
        assert n in exported, n
        assert getattr(L, n) is not None


def test_status_strings_and_version(L):
    for code in (OK, NULLPTR, INVALID, INNER, CUDA, WORKSPACE, UNSUPPORTED):
        s = L.mr_status_string(code).decode()
        assert s and s != "unknown status"
    assert L.mr_status_string(12345).decode() == "unknown status"
    assert L.mr_version() >= 100


def _bws(L, E, shape, dt, ns, ln):
    ws = ctypes.c_uint64(0)
    arr = _native.int64_array(shape) if shape is not None else None
    st = L.ffnwb_batching_get_workspace_size(E, arr, dt, ns, ln, ctypes.byref(ws))
    return st, ws.value


@pytest.mark.parametrize("E,shape,dt,ns,ln,expect", [
    (8, (2, 8, 3, 128), 0, 0, 1, OK),
    (8192, (1024, 1, 64, 1), 2, 0, 0, OK),
    (1024, (256, 64, 9, 7168), 1, 0, 4, OK),
    (0, (2, 8, 3, 128), 0, 0, 1, INVALID),
    (8193, (2, 8, 3, 128), 0, 0, 1, INVALID),
    (8, (0, 8, 3, 128), 0, 0, 1, INVALID),
    (8, (1025, 8, 3, 128), 0, 0, 1, INVALID),
    (8, (2, 0, 3, 128), 0, 0, 1, INVALID),
    (8, (2, 8, 0, 128), 0, 0, 1, INVALID),
    (8, (2, 8, 65, 128), 0, 0, 1, INVALID),
    (8, (2, 8, 3, 0), 0, 0, 1, INVALID),
    (8, (2, 8, 3, 128), 3, 0, 1, INVALID),
    (8, (2, 8, 3, 128), -1, 0, 1, INVALID),
    (8, (2, 8, 3, 128), 0, 2, 1, INVALID),
    (8, (2, 8, 3, 128), 0, 1, 1, UNSUPPORTED),
    (8, (2, 8, 3, 128), 0, 0, 9, INVALID),
    (8, (2, 8, 3, 128), 0, 0, -1, INVALID),
    (8, (2, 8, 3, 128), 0, 0, 3, INVALID),   # 8 experts not divisible into 3 layers
    (8, None, 0, 0, 1, NULLPTR),
])
def test_batching_workspace_validation(L, E, shape, dt, ns, ln, expect):
    st, ws = _bws(L, E, shape, dt, ns, ln)
    assert st == expect
    if st == OK:
        assert ws > 0


def test_batching_workspace_null_out(L):
    arr = _native.int64_array((2, 8, 3, 128))
    assert L.ffnwb_batching_get_workspace_size(8, arr, 0, 0, 1, None) == NULLPTR


def _batching_call(L, **kw):
    a = dict(expertIds=FAKE, layerId=0, tokenData=FAKE, stride=256, scales=None, scaleStride=4,
             sess=FAKE, micro=FAKE, tok=None, E=8, shape=(2, 8, 3, 128), dt=0, ns=0, ln=1, y=FAKE,
             gl=FAKE, so=FAKE, mo=FAKE, to=FAKE, eo=FAKE, dyn=None, atn=FAKE, sidx=None,
             ws=FAKE, wsz=1 << 40, stream=None)
    a.update(kw)
    return L.ffnwb_batching(a["expertIds"], a["layerId"], a["tokenData"], a["stride"], a["scales"],
                            a["scaleStride"], a["sess"], a["micro"], a["tok"], a["E"],
                            _native.int64_array(a["shape"]), a["dt"], a["ns"], a["ln"], a["y"],
                            a["gl"], a["so"], a["mo"], a["to"], a["eo"], a["dyn"], a["atn"],
                            a["sidx"], a["ws"], a["wsz"], a["stream"])


@pytest.mark.parametrize("kw,expect", [
    (dict(expertIds=None), NULLPTR),
    (dict(tokenData=None), NULLPTR),
    (dict(sess=None), NULLPTR),
    (dict(micro=None), NULLPTR),
    (dict(y=None), NULLPTR),
    (dict(gl=None), NULLPTR),
    (dict(so=None), NULLPTR),
    (dict(mo=None), NULLPTR),
    (dict(to=None), NULLPTR),
    (dict(eo=None), NULLPTR),
    (dict(atn=None), NULLPTR),
    (dict(ws=None), NULLPTR),
    (dict(dt=2, stride=132, dyn=None), NULLPTR),         # INT8 needs dynamicScale
    (dict(layerId=1), INVALID),                           # one layer: layer id must be 0
    (dict(layerId=-1), INVALID),
    (dict(stride=255), INVALID),                          # row stride below H * 2 bytes
    (dict(dt=2, stride=130, dyn=FAKE), INVALID),          # INT8 interleaved: needs H + 4 bytes
    (dict(dt=2, stride=128, dyn=FAKE, scales=FAKE, scaleStride=2), INVALID),
    (dict(wsz=16), WORKSPACE),
    (dict(ns=1), UNSUPPORTED),
    (dict(E=0), INVALID),
])
def test_batching_execute_validation(L, kw, expect):
    assert _batching_call(L, **kw) == expect


def _uws(L, rows, H, dt, n, hp, pdt, T, Eu, padded, rs=None):
    ws = ctypes.c_uint64(0)
    arr = _native.int64_array(rs) if rs is not None else None
    st = L.moe_unpermute_get_workspace_size(rows, H, dt, n, hp, pdt, T, Eu, padded, arr, ctypes.byref(ws))
    return st, ws.value


@pytest.mark.parametrize("args,expect", [
    ((32768, 4096, 1, 32768, 1, 1, 4096, 64, 0), OK),          # top-k workload
    ((65536, 4096, 0, 65536, 1, 3, 16384, 128, 1), OK),        # padded workload (fp16 + fp32 probs)
    ((147456, 7168, 1, 147456, 1, 1, 16384, 9, 0), OK),        # round trip
    ((32, 16, 3, 32, 0, 3, 0, 0, 0, (4, 16)), OK),             # no probs: T from restoreShape
    ((32, 16, 3, 32, 0, 3, 0, 0, 1, (4, 16)), OK),
    ((32, 16, 2, 32, 1, 2, 4, 8, 0), INVALID),                 # int8 tokens are not allowed
    ((32, 16, 0, 32, 1, 1, 4, 8, 0), INVALID),                 # fp16 tokens with bf16 probs
    ((32, 16, 1, 32, 1, 3, 4, 8, 0), OK),                      # bf16 tokens with fp32 probs
    ((32, 16, 0, 32, 1, 3, 4, 8, 0), OK),                      # fp16 tokens with fp32 probs
    ((4 * 513, 8, 1, 4 * 513, 1, 1, 4, 8, 0), INNER),          # topK_num 513 > 512
    ((4 * 512, 8, 1, 4 * 512, 1, 1, 4, 8, 0), OK),             # topK_num 512
    ((32, 16, 1, 31, 1, 1, 4, 8, 0), INVALID),                 # not padded: n != T * topK
    ((32, 16, 1, 31, 1, 1, 4, 8, 1), INVALID),                 # padded: n != rows
    ((32, 16, 1, 32, 1, 1, 4, 5, 1), INNER),                   # padded: n not a multiple of experts
    ((32, 16, 1, 32, 1, 1, 4, 64, 1), INNER),                  # padded: capacity 0
    ((32, 16, 1, 32, 1, 1, 0, 8, 0), INNER),                   # probs shape with 0 tokens
    ((32, 0, 1, 32, 1, 1, 4, 8, 0), INVALID),
    ((32, 16, 1, 32, 1, 1, 4, 8, 2), INVALID),                 # paddedMode 2
    ((32, 16, 1, 32, 1, 1, 4, 8, 0, (5, 16)), INVALID),        # restoreShape disagrees with probs
    ((32, 16, 1, 32, 1, 1, 4, 8, 0, (4, 17)), INVALID),
    ((32, 16, 3, 32, 0, 3, 0, 0, 0), NULLPTR),                 # no probs and no restoreShape
])
def test_unpermute_workspace_validation(L, args, expect):
    st, ws = _uws(L, *args)
    assert st == expect
    if st == OK:
        assert ws > 0


def test_unpermute_workspace_null_out(L):
    assert L.moe_unpermute_get_workspace_size(32, 16, 1, 32, 1, 1, 4, 8, 0, None, None) == NULLPTR


def _unpermute_call(L, **kw):
    a = dict(perm=FAKE, si=FAKE, rmap=FAKE, probs=FAKE, rows=32, H=16, dt=1, n=32, pdt=1, T=4, Eu=8,
             padded=0, rs=None, out=FAKE, oi=FAKE, pt=FAKE, pp=FAKE, ws=FAKE, wsz=1 << 40, stream=None)
    a.update(kw)
    rs = _native.int64_array(a["rs"]) if a["rs"] is not None else None
    return L.moe_unpermute(a["perm"], a["si"], a["rmap"], a["probs"], a["rows"], a["H"], a["dt"],
                           a["n"], a["pdt"], a["T"], a["Eu"], a["padded"], rs, a["out"], a["oi"],
                           a["pt"], a["pp"], a["ws"], a["wsz"], a["stream"])


@pytest.mark.parametrize("kw,expect", [
    (dict(perm=None), NULLPTR),
    (dict(si=None), NULLPTR),
    (dict(out=None), NULLPTR),
    (dict(oi=None), NULLPTR),
    (dict(pt=None), NULLPTR),
    (dict(pp=None), NULLPTR),            # probs given: permuteProbs required
    (dict(ws=None), NULLPTR),
    (dict(rmap=None), INVALID),          # probs without routing map
    (dict(probs=None), INVALID),         # routing map without probs
    (dict(wsz=8), WORKSPACE),
    (dict(rows=4 * 600, n=4 * 600), INNER),
])
def test_unpermute_execute_validation(L, kw, expect):
    assert _unpermute_call(L, **kw) == expect


def test_profile_events_validation(L):
    assert L.mr_profile_set_events(None, 0) == OK
    assert L.mr_profile_set_events(None, 2) == INVALID
    assert L.mr_profile_set_events(None, 17) == INVALID
    assert L.mr_profile_set_events(None, -1) == INVALID


def _context_call(L, **kw):
    a = dict(ctx=ctypes.c_void_p(0x1000), E=8, shape=(2, 8, 3, 128), dt=0, ns=0, ln=1, timeout=1000,
             y=FAKE, gl=FAKE, so=FAKE, mo=FAKE, to=FAKE, eo=FAKE, dyn=None, atn=FAKE, status=None,
             ws=FAKE, wsz=1 << 40, stream=None)
    a.update(kw)
    return L.ffnwb_batching_context(a["ctx"], a["E"], _native.int64_array(a["shape"]), a["dt"], a["ns"],
                                    a["ln"], a["timeout"], a["y"], a["gl"], a["so"], a["mo"], a["to"],
                                    a["eo"], a["dyn"], a["atn"], a["status"], a["ws"], a["wsz"],
                                    a["stream"])


@pytest.mark.parametrize("kw,expect", [
    (dict(ctx=None), NULLPTR),
    (dict(y=None), NULLPTR),
    (dict(atn=None), NULLPTR),
    (dict(ws=None), NULLPTR),
    (dict(dt=2, dyn=None), NULLPTR),
    (dict(ctx=ctypes.c_void_p(0x1004)), INVALID),      # not 8-byte aligned
    (dict(timeout=-1), INVALID),
    (dict(timeout=60_000_001), INVALID),
    (dict(ns=2), INVALID),
    (dict(E=0), INVALID),
    (dict(wsz=8), WORKSPACE),
])
def test_context_execute_validation(L, kw, expect):
    assert _context_call(L, **kw) == expect


def test_context_workspace_size(L):
    ws = ctypes.c_uint64(0)
    shape = _native.int64_array((2, 8, 3, 128))
    assert L.ffnwb_batching_context_get_workspace_size(8, shape, 0, 1, 1, ctypes.byref(ws)) == OK
    ws_flat = ctypes.c_uint64(0)
    assert L.ffnwb_batching_get_workspace_size(8, shape, 0, 0, 1, ctypes.byref(ws_flat)) == OK
    assert ws.value > ws_flat.value
    assert L.ffnwb_batching_context_get_workspace_size(8, shape, 0, 2, 1, ctypes.byref(ws)) == INVALID
    assert L.ffnwb_batching_context_get_workspace_size(8, shape, 0, 0, 1, None) == NULLPTR


def _permute_call(L, **kw):
    a = dict(tok=FAKE, rmap=FAKE, T=16, H=32, dt=1, Eu=8, k=2, padded=0, cap=0, out=FAKE, si=FAKE,
             rows=None, ws=FAKE, wsz=1 << 40, stream=None)
    a.update(kw)
    return L.moe_permute(a["tok"], a["rmap"], a["T"], a["H"], a["dt"], a["Eu"], a["k"], a["padded"],
                         a["cap"], a["out"], a["si"], a["rows"], a["ws"], a["wsz"], a["stream"])


@pytest.mark.parametrize("kw,expect", [
    (dict(tok=None), NULLPTR),
    (dict(rmap=None), NULLPTR),
    (dict(out=None), NULLPTR),
    (dict(si=None), NULLPTR),
    (dict(ws=None), NULLPTR),
    (dict(dt=2), INVALID),                 # int8 tokens
    (dict(Eu=0), INVALID),
    (dict(Eu=8193), INVALID),
    (dict(k=0), INVALID),
    (dict(k=513), INNER),                  # topK_num > 512
    (dict(padded=1, cap=0), INVALID),
    (dict(padded=2), INVALID),
    (dict(T=0), INVALID),
    (dict(wsz=8), WORKSPACE),
])
def test_permute_execute_validation(L, kw, expect):
    assert _permute_call(L, **kw) == expect


def test_permute_workspace_size(L):
    ws = ctypes.c_uint64(0)
    assert L.moe_permute_get_workspace_size(4096, 4096, 1, 64, 8, 0, 0, ctypes.byref(ws)) == OK
    assert ws.value > 0
    assert L.moe_permute_get_workspace_size(16384, 4096, 0, 128, 0, 1, 512, ctypes.byref(ws)) == OK
    assert L.moe_permute_get_workspace_size(16, 32, 1, 8, 2, 0, 0, None) == NULLPTR


def _update_call(L, **kw):
    a = dict(ids=FAKE, idt=4, tab=FAKE, sc=None, sdt=3, thr=None, act=None, BS=8, K=4, E=16, F=3,
             rank=1, ws=4, mode=0, strides=None, out=FAKE, mask=None, stream=None)
    a.update(kw)
    return L.moe_update_expert(a["ids"], a["idt"], a["tab"], a["sc"], a["sdt"], a["thr"], a["act"],
                               a["BS"], a["K"], a["E"], a["F"], a["rank"], a["ws"], a["mode"],
                               a["strides"], a["out"], a["mask"], a["stream"])


@pytest.mark.parametrize("kw,expect", [
    (dict(ids=None), NULLPTR),
    (dict(tab=None), NULLPTR),
    (dict(out=None), NULLPTR),
    (dict(sc=FAKE), NULLPTR),                         # scales without threshold
    (dict(thr=FAKE), NULLPTR),                        # threshold without scales
    (dict(act=FAKE), NULLPTR),                        # activeMask without scales
    (dict(sc=FAKE, thr=FAKE), NULLPTR),               # pruning without a mask output
    (dict(sc=FAKE, thr=FAKE, mask=FAKE, sdt=2), INVALID),
    (dict(idt=3), INVALID),
    (dict(BS=0), INVALID),
    (dict(BS=513), INVALID),
    (dict(K=17, E=32), INVALID),
    (dict(K=5, E=4), INVALID),                        # K > moeExpertNum
    (dict(E=1025), INVALID),
    (dict(mode=2), INVALID),
    (dict(ws=1), INVALID),                            # by rank: worldSize >= 2
    (dict(ws=769, F=3), INVALID),
    (dict(rank=4), INVALID),                          # localRankId >= worldSize
    (dict(rank=-1), INVALID),
    (dict(F=1), INVALID),
    (dict(F=6), INVALID),                             # F > worldSize + 1
    (dict(mode=1, ws=0), INVALID),
    (dict(strides=_native.int64_array([4, 1, 3, 1, 4, 1, 1, 1, 4, 0, 4, 1])), INVALID),  # output stride 0
    (dict(strides=_native.int64_array([4, -1, 3, 1, 4, 1, 1, 1, 4, 1, 4, 1])), INVALID),
])
def test_update_expert_validation(L, kw, expect):
    assert _update_call(L, **kw) == expect


@pytest.mark.parametrize("flags,kw,expect", [
    (2, {}, INVALID),                                 # unknown option bit
    (0x80000000, {}, INVALID),
    (1, dict(wsz=16), WORKSPACE),                     # the option keeps the workspace size
    (1, dict(ns=1), UNSUPPORTED),
    (1, dict(y=None), NULLPTR),
])
def test_batching_ex_flags(L, flags, kw, expect):
    a = dict(expertIds=FAKE, layerId=0, tokenData=FAKE, stride=256, scales=None, scaleStride=4,
             sess=FAKE, micro=FAKE, tok=None, E=8, shape=(2, 8, 3, 128), dt=0, ns=0, ln=1, y=FAKE,
             gl=FAKE, so=FAKE, mo=FAKE, to=FAKE, eo=FAKE, dyn=None, atn=FAKE, sidx=None,
             ws=FAKE, wsz=1 << 40, stream=None)
    a.update(kw)
    st = L.ffnwb_batching_ex(a["expertIds"], a["layerId"], a["tokenData"], a["stride"], a["scales"],
                             a["scaleStride"], a["sess"], a["micro"], a["tok"], a["E"],
                             _native.int64_array(a["shape"]), a["dt"], a["ns"], a["ln"], a["y"],
                             a["gl"], a["so"], a["mo"], a["to"], a["eo"], a["dyn"], a["atn"],
                             a["sidx"], flags, a["ws"], a["wsz"], a["stream"])
    assert st == expect


@pytest.mark.parametrize("flags,kw,expect", [
    (4, {}, INVALID),
    (1, dict(wsz=8), WORKSPACE),
    (1, dict(ctx=None), NULLPTR),
])
def test_context_ex_flags(L, flags, kw, expect):
    a = dict(ctx=ctypes.c_void_p(0x1000), E=8, shape=(2, 8, 3, 128), dt=0, ns=0, ln=1, timeout=1000,
             y=FAKE, gl=FAKE, so=FAKE, mo=FAKE, to=FAKE, eo=FAKE, dyn=None, atn=FAKE, status=None,
             ws=FAKE, wsz=1 << 40, stream=None)
    a.update(kw)
    st = L.ffnwb_batching_context_ex(a["ctx"], a["E"], _native.int64_array(a["shape"]), a["dt"],
                                     a["ns"], a["ln"], a["timeout"], a["y"], a["gl"], a["so"], a["mo"],
                                     a["to"], a["eo"], a["dyn"], a["atn"], a["status"], flags, a["ws"],
                                     a["wsz"], a["stream"])
    assert st == expect


def _no_gpu():
    try:
        import torch
        return not torch.cuda.is_available()
    except Exception:
        return True


@pytest.mark.skipif(not _no_gpu(), reason="forces launch failures, which need a machine without a GPU")
def test_launch_failures_return_cuda_error(L):
    """Valid arguments on a machine without a GPU: the checks pass, the first
    CUDA call fails, and the call returns MR_ERR_CUDA (no kernel runs, so the
    placeholder pointers are never touched)."""
    CUDA = 561001
    assert _batching_call(L) == CUDA
    assert _context_call(L) == CUDA
    assert _permute_call(L) == CUDA
    assert _update_call(L) == CUDA
    assert _update_call(L, sc=FAKE, thr=FAKE, mask=FAKE) == CUDA
    # the not-padded unpermute first needs its auxiliary stream
    assert _unpermute_call(L) == CUDA
    assert _unpermute_call(L, padded=1) == CUDA
