"""Benchmark of the MoE expert-grouped token reorder on GB300.

One step = one pass of the whole hot path over one batch of synthetic input,
the full-scale round trip: FFN-worker batching of Y = 256*64*9 = 147456 slots
(expertNum 1024 over 4 layers, layer 2, H = 7168 bf16, Zipf(1.2) expert ids,
5% masked), then the not-padded unpermute with probs of its output y back to
16384 tokens x topK 9.

Prints ONE JSON line (rank 0). `value` is the effective HBM bandwidth of the
step (algorithmic bytes read + written / device time) over all ranks;
`tokens_per_s` the tokens the step processes per second. Inputs are larger
than L2 (2.1 GB of token rows per step), so no L2 flush is needed.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (the program the kernels are checked
against) on one host core: on the full workload when --warmup + --steps
full-size steps fit about REFERENCE_BUDGET_S (a 20-step run does), else on
a power-of-two fraction of its attention workers, which the line's
config.sample names.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as w  # noqa: E402

METRIC = "permute/unpermute effective HBM GB/s (% of ~8 TB/s peak) and tokens/s, 1 GB300"
WORKLOAD = ("full-scale round trip: batching A=256 BS=64 topK+1=9 (Y=147456) expertNum=1024 "
            "layerNum=4 layer_id=2 H=7168 bf16 Zipf(1.2) 5% masked, then not-padded unpermute "
            "with probs T=16384 topK=9 bf16")
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
FALLBACK_HBM_GBS = 6800.0
CSRC = os.path.join(ROOT, "unpermute_stable_counting_gb300", "csrc")


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-sample-attn", type=int, default=None,
                    help="attention workers (A) of each reference-arm step (default: the full "
                         "workload's 256 when --steps + --warmup oracle steps fit "
                         "REFERENCE_BUDGET_S, else the largest power-of-two fraction that does)")
    ap.add_argument("--small", action="store_true", help="a small case of the same workload (profiling)")
    ap.add_argument("--workload", choices=["roundtrip", "tiny", "topk", "int8", "padded", "context",
                                           "batching", "permute", "permute_padded", "update_expert", "decode_unpermute",
                                           "padded_slack", "batching_index", "large_map", "odd_h", "padded_lsd"],
                    default="roundtrip",
                    help="roundtrip (the bench line) or one of the other workloads, timed per call "
                         "with an L2 flush before each")
    ap.add_argument("--flush", choices=["write", "write-read"], default="write-read",
                    help="L2 flush before each call of --workload: a 512 MB write, optionally "
                         "followed by a 512 MB read that writes the dirty lines back before the "
                         "timed call")
    return ap.parse_args(argv)


# ---------------------------------------------------------------------------
# Workload and its algorithmic bytes
# ---------------------------------------------------------------------------

def workload_spec(small=False, attn=None):
    spec = dict(w.ROUNDTRIP_BATCHING)
    if small:
        spec["A"] = 32  # Y = 18432 slots, 264 MB of token rows: still larger than L2
    if attn is not None:
        spec["A"] = attn
    return spec


def make_host_inputs(spec):
    inp = w.make_batching(**spec)
    T, k = spec["A"] * spec["BS"], spec["K1"]
    El = spec["E"] // max(spec["layerNum"], 1)
    unmasked = (inp["expert_ids"] >= 0) & (inp["expert_ids"] < El)
    rmap, probs = w.make_roundtrip_probs(T=T, k=k, slot_unmasked=unmasked,
                                         probs_dtype=w.ROUNDTRIP_PROBS_DTYPE, seed=spec["seed"])
    return inp, rmap, probs, int(unmasked.sum())


def algorithmic_bytes(spec, U, V):
    """Bytes each step must read and write (inputs once, outputs once)."""
    Y = spec["A"] * spec["BS"] * spec["K1"]
    H, E = spec["H"], spec["E"]
    s = w.ELEM_BYTES[spec["dtype"]]
    T, k = spec["A"] * spec["BS"], spec["K1"]
    ps = w.ELEM_BYTES[w.ROUNDTRIP_PROBS_DTYPE]
    row = H * s
    # batching: keys, the U gathered rows, session/micro/token id lookups; y rows,
    # four int32 id outputs, the slot -> row map, group_list, actual_token_num
    b_read = Y * 4 + U * row + U * 12
    b_write = U * row + Y * 16 + Y * 4 + E * 16 + 8
    # unpermute: sortedIndices, the V contributing rows, routing map and probs;
    # the token outputs, outIndex, permuteTokenId, permuteProbs
    u_read = T * k * 4 + V * row + T * k * (1 + ps)
    u_write = T * row + T * k * (8 + ps)
    gather = U * (2 * row + 4)                    # batching row-gather kernel
    reduce_ = V * row + T * row + T * k * (4 + ps)  # unpermute gather-reduce kernel
    return dict(batching=b_read + b_write, unpermute=u_read + u_write, total=b_read + b_write + u_read + u_write,
                gather_kernel=gather, reduce_kernel=reduce_, tokens=T, slots=Y)


def sort_launches(n, key_range):
    """Kernels of the unpermute's index sort over n entries with key_range
    distinct keys, as the library plans it: one counting-sort pass (one
    block-local kernel up to 2048 entries, else rank, prefix and scatter) up to
    4096 keys; up to 2^22 keys that pass on the high bits plus the per-bucket
    fine sort; beyond, LSD passes of at most 12 bits (not padded)."""
    one_pass = 1 if n <= 2048 else 3
    if key_range <= 4096:
        return one_pass
    if key_range <= 1 << 22:
        return one_pass + 1
    bits = int(np.ceil(np.log2(key_range)))
    return 3 * ((bits + 11) // 12)


def masked_select_launches(T, Eu):
    """Kernels of the not-padded maskedSelect, as the library plans it (vector
    rows): none for a small map (T*Eu <= 16384, selected inside the reduce),
    one cooperative kernel up to 4096 tiles of 1024 entries, else three."""
    if T * Eu <= 16384:
        return 0
    return 1 if (T * Eu + 1023) // 1024 <= 4096 else 3


def launches_per_step(spec):
    Y = spec["A"] * spec["BS"] * spec["K1"]
    T = spec["A"] * spec["BS"]
    batching = 4  # rank, prefix, scatter, gather
    # maskedSelect (the routing map is [T, topK+1]), index sort, reduce
    unpermute = masked_select_launches(T, spec["K1"]) + sort_launches(Y, Y + 1) + 1
    return batching + unpermute


# ---------------------------------------------------------------------------
# Peaks, clocks, ncu traffic
# ---------------------------------------------------------------------------

def hbm_peak():
    try:
        with open(PEAKS_FILE) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def source_digest(files):
    """Digest of the kernel source files a profile was taken on."""
    h = hashlib.sha256()
    for name in sorted(files):
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel, units):
    """DRAM bytes (read + write) per launch from the committed ncu summary,
    scaled to `units` rows, or None if absent or if the kernel's source files
    changed since the counters were taken."""
    try:
        with open(TRAFFIC_FILE) as f:
            e = json.load(f)["kernels"][kernel]
        if e.get("source_digest") != source_digest(e["files"]):
            return None
        return float(e["dram_bytes_per_unit"]) * units
    except Exception:
        return None


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, local_rank):
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        ids = [v.strip() for v in vis.split(",") if v.strip()]
        self.index = ids[local_rank] if local_rank < len(ids) else str(local_rank)
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            p = [x.strip() for x in line.split(",")]
            if len(p) < 8:
                continue
            try:
                sm.append(float(p[0]))
                mx.append(float(p[1]))
            except ValueError:
                continue
            for n, v in zip(names, p[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# Distributed plumbing (replicas only: no data-path collective)
# ---------------------------------------------------------------------------

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Largest value over all ranks (the timing rule: the slowest rank)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_value(bytes_per_rank: float, world: int, max_seconds_per_step: float) -> float:
    """Whole-job effective GB/s: bytes all ranks moved / the slowest rank's time."""
    return bytes_per_rank * world / max_seconds_per_step / 1e9


# ---------------------------------------------------------------------------
# CPU oracle (baseline and reference arm)
# ---------------------------------------------------------------------------

def oracle_step(spec, inp, rmap, probs):
    import oracle
    T, k = spec["A"] * spec["BS"], spec["K1"]
    t0 = time.perf_counter()
    b = oracle.batching(inp)
    u = dict(permuted=b["y"], sortedIndices=b["sortedIndices"], routingMap=rmap, probs=probs,
             permutedRows=inp["Y"], H=inp["H"], tokenDtype=inp["tokenDtype"], n=T * k,
             probsDtype=w.ROUNDTRIP_PROBS_DTYPE, T=T, Eu=k, padded=0)
    oracle.unpermute(u)
    return time.perf_counter() - t0


def contributing_rows(spec, inp, probs):
    """V: slots whose row the unpermute reads (valid index and nonzero prob)."""
    El = spec["E"] // max(spec["layerNum"], 1)
    unmasked = (inp["expert_ids"] >= 0) & (inp["expert_ids"] < El)
    # the not-padded weight of slot i is the i-th maskedSelect value (expert-major order)
    T, k = spec["A"] * spec["BS"], spec["K1"]
    pv = probs.reshape(T, k).T[unmasked.reshape(T, k).T]
    nz = np.zeros(T * k, dtype=bool)
    nz[:pv.size] = (pv != 0)
    return int((unmasked & nz).sum())


CPU_SAMPLE_SECONDS = 10.0  # the bounded sample: whole steps until at least this much CPU time


def cpu_baseline(spec, inp, rmap, probs, ab):
    """The oracle, as it stands, on whole steps of the same inputs (rank 0),
    repeated until about CPU_SAMPLE_SECONDS of work; the value is the mean."""
    import oracle
    oracle.build()
    times = []
    while sum(times) < CPU_SAMPLE_SECONDS and len(times) < 100:
        times.append(oracle_step(spec, inp, rmap, probs))
    dt = sum(times) / len(times)
    return {"value": ab["total"] / dt / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "tokens_per_s": ab["tokens"] / dt, "seconds_per_step": dt, "steps": len(times),
            "sample": (f"{len(times)} steps of the same workload (A={spec['A']}, Y={ab['slots']} slots, "
                       f"{ab['tokens']} tokens, H={spec['H']}), {sum(times):.1f} s in total, on the "
                       f"single-threaded oracle, input generation excluded")}


REFERENCE_BUDGET_S = 150.0   # whole reference run: --warmup + --steps oracle steps
ORACLE_STEP_S_FULL = 1.9     # one oracle step of the full workload on a GB300 machine's Grace core


def reference_attn(args) -> int:
    """Attention workers of each reference-arm step: the full workload (256)
    when warmup + steps full-size oracle steps fit the budget, else the
    largest power-of-two fraction of it that does (at least 8)."""
    if args.cpu_sample_attn is not None:
        return args.cpu_sample_attn
    full = w.ROUNDTRIP_BATCHING["A"]
    n = max(1, args.steps + args.warmup)
    a = full
    while a > 8 and n * ORACLE_STEP_S_FULL * a / full > REFERENCE_BUDGET_S:
        a //= 2
    return a


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    spec = workload_spec(attn=reference_attn(args))
    inp, rmap, probs, U = make_host_inputs(spec)
    V = contributing_rows(spec, inp, probs)
    ab = algorithmic_bytes(spec, U, V)
    for _ in range(args.warmup):
        oracle_step(spec, inp, rmap, probs)
    times = [oracle_step(spec, inp, rmap, probs) for _ in range(args.steps)]
    total = sum(times)
    value = ab["total"] * args.steps / total / 1e9
    full = w.ROUNDTRIP_BATCHING["A"]
    if spec["A"] == full:
        sample = (f"each step: the full workload (A={full}, Y={ab['slots']} slots, {ab['tokens']} tokens, "
                  f"H=7168) on the single-threaded CPU oracle")
    else:
        sample = (f"A={spec['A']} of {full}: each step the round trip with {spec['A']} attention workers "
                  f"(Y={ab['slots']} slots, {ab['tokens']} tokens, H=7168) on the single-threaded CPU "
                  f"oracle, so that {args.warmup + args.steps} steps fit {REFERENCE_BUDGET_S:.0f} s")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": total / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": WORKLOAD, "sample": sample},
            "tokens_per_s": ab["tokens"] * args.steps / total,
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def run_ours(args):
    import torch

    import unpermute_stable_counting_gb300 as usc
    from unpermute_stable_counting_gb300 import _build

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    _build.build_library()

    spec = workload_spec(small=args.small)
    inp, rmap, probs, U = make_host_inputs(spec)
    V = contributing_rows(spec, inp, probs)
    ab = algorithmic_bytes(spec, U, V)
    Y, H, E = inp["Y"], inp["H"], inp["expertNum"]
    T, k = spec["A"] * spec["BS"], spec["K1"]
    shape = (inp["A"], inp["BS"], inp["K1"], H)
    pdt = w.ROUNDTRIP_PROBS_DTYPE

    # pinned host copies (e2e) and device-resident inputs
    def pinned(a):
        t = torch.from_numpy(np.ascontiguousarray(a))
        return t.pin_memory()

    h_ids, h_td = pinned(inp["expert_ids"]), pinned(inp["token_data"])
    h_sess, h_micro, h_tok = pinned(inp["session_in"]), pinned(inp["micro_in"]), pinned(inp["token_in"])
    h_rmap, h_probs = pinned(rmap), pinned(probs.view(np.int16))
    d = {n: t.to(dev) for n, t in dict(ids=h_ids, td=h_td, sess=h_sess, micro=h_micro, tok=h_tok,
                                       rmap=h_rmap, probs=h_probs).items()}
    d_td = d["td"].view(torch.bfloat16).view(Y, H)
    d_probs = d["probs"].view(torch.bfloat16).view(T, k)

    bout = usc.batching_outputs(Y, H, E, inp["tokenDtype"], dev, with_sorted_indices=True)
    uout = usc.unpermute_outputs(T, H, T * k, inp["tokenDtype"], pdt, dev)
    bws = torch.empty(usc.batching_workspace_size(E, shape, inp["tokenDtype"], inp["layerNum"]),
                      dtype=torch.uint8, device=dev)
    uws = torch.empty(usc.unpermute_workspace_size(Y, H, inp["tokenDtype"], T * k, True, pdt, T, k,
                                                   False), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(td=d_td, ids=d["ids"], sess=d["sess"], micro=d["micro"], tok=d["tok"], rm=d["rmap"],
             pr=d_probs):
        usc.ffnwb_batching(ids, td, sess, micro, expert_num=E, max_out_shape=shape,
                           token_dtype=inp["tokenDtype"], layer_num=inp["layerNum"],
                           layer_id=inp["layer_id"], token_ids=tok, with_sorted_indices=True,
                           out=bout, workspace=bws, stream=stream)
        usc.moe_unpermute(bout["y"], bout["sortedIndices"], rm, pr, padded_mode=False, out=uout,
                          workspace=uws, stream=stream)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    # ---- device-resident timing ------------------------------------------------
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    clocks = sampler.stop()
    if clocks is not None:
        clocks["window"] = "warm-up and timed steps"
    sec_step = e0.elapsed_time(e1) / 1e3 / args.steps
    sec_step = max_over_ranks(sec_step, world, dev)

    # ---- per-phase kernel times (library phase events on the launch stream) ----
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(10)]
    phase = {p: [] for p in range(5)}
    usc.profile_set_events(ev)
    try:
        for _ in range(args.steps):
            step()
            torch.cuda.synchronize()
            for p in range(5):
                phase[p].append(ev[2 * p].elapsed_time(ev[2 * p + 1]) / 1e3)
    finally:
        usc.profile_set_events(None)
    ph = {p: statistics.mean(v) for p, v in phase.items()}

    # ---- end to end through host buffers -----------------------------------
    # Every step copies its inputs from pinned host memory and reads its
    # results back, through the same public calls. The steps are pipelined the
    # way a serving loop would run them: two sets of device buffers, the
    # host->device copy of step i+1 on one stream while step i computes on
    # another and step i-1's results go back on a third (the host link's two
    # directions run at once). The timed region spans the first copy in to the
    # last copy out.
    e2e = None
    if not args.no_e2e:
        names_in = ("ids", "td", "sess", "micro", "tok", "rmap", "probs")
        hosts = dict(ids=h_ids, td=h_td, sess=h_sess, micro=h_micro, tok=h_tok, rmap=h_rmap,
                     probs=h_probs)
        dsets = [d, {n: torch.empty_like(d[n]) for n in names_in}]
        bouts = [bout, usc.batching_outputs(Y, H, E, inp["tokenDtype"], dev, with_sorted_indices=True)]
        uouts = [uout, usc.unpermute_outputs(T, H, T * k, inp["tokenDtype"], pdt, dev)]
        bnames = ("groupList", "actualTokenNum", "sessionIds", "microBatchIds", "tokenIds", "expertOffsets")
        def host_outputs():
            o = {("u", n): torch.empty(t.shape, dtype=t.dtype).pin_memory()
                 for n, t in uout.items() if t is not None}
            o.update({("b", n): torch.empty(bout[n].shape, dtype=bout[n].dtype).pin_memory()
                      for n in bnames})
            return o
        h_outs = [host_outputs(), host_outputs()]
        h2d = sum(hosts[n].numel() * hosts[n].element_size() for n in names_in)
        d2h = sum(t.numel() * t.element_size() for t in h_outs[0].values())
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_comp = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]
        for e in ev_comp + ev_out:
            e.record(stream)

        def e2e_step(i):
            j = i % 2
            dd, bo, uo = dsets[j], bouts[j], uouts[j]
            with torch.cuda.stream(s_in):
                s_in.wait_event(ev_comp[j])          # step i-2 no longer reads this set
                for n in names_in:
                    dd[n].copy_(hosts[n], non_blocking=True)
                ev_in[j].record(s_in)
            stream.wait_event(ev_in[j])
            stream.wait_event(ev_out[j])              # step i-2's results are home
            usc.ffnwb_batching(dd["ids"], dd["td"].view(torch.bfloat16).view(Y, H), dd["sess"], dd["micro"],
                               expert_num=E, max_out_shape=shape, token_dtype=inp["tokenDtype"],
                               layer_num=inp["layerNum"], layer_id=inp["layer_id"], token_ids=dd["tok"],
                               with_sorted_indices=True, out=bo, workspace=bws, stream=stream)
            usc.moe_unpermute(bo["y"], bo["sortedIndices"], dd["rmap"], dd["probs"].view(torch.bfloat16).view(T, k),
                              padded_mode=False, out=uo, workspace=uws, stream=stream)
            ev_comp[j].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_comp[j])
                for (kind, n), hh in h_outs[j].items():
                    hh.copy_((uo if kind == "u" else bo)[n], non_blocking=True)
                ev_out[j].record(s_out)

        for i in range(2):
            e2e_step(i)
        torch.cuda.synchronize()
        barrier()
        # enough steps that the pipeline's fill (the first copy in) and drain
        # (the last copy out) weigh little against the steady state
        n_e2e = max(4, min(args.steps, 30))
        e0.record(stream)
        s_in.wait_event(e0)
        s_out.wait_event(e0)
        for i in range(n_e2e):
            e2e_step(i)
        e1.record(s_out)
        torch.cuda.synchronize()
        e2e_sec = max_over_ranks(e0.elapsed_time(e1) / 1e3 / n_e2e, world, dev)
        e2e = {"value": aggregate_value(ab["total"], world, e2e_sec), "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_sec * 1e3,
               "steps": n_e2e, "pipeline": "double-buffered: copy in of step i+1, compute of step i "
                                          "and copy out of step i-1 on three streams"}
        del dsets, bouts, uouts

    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return 0

    peak, peak_kind = hbm_peak()
    gather_gbs = ab["gather_kernel"] / ph[1] / 1e9
    reduce_gbs = ab["reduce_kernel"] / ph[3] / 1e9
    # the round trip's rows are 16-byte aligned: the batching gathers them with the flat kernel
    gather_kernel = "batching_gather_flat_kernel"
    traffic = ncu_traffic(gather_kernel, U)
    value = aggregate_value(ab["total"], world, sec_step)
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": sec_step * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD if not args.small else WORKLOAD + " (A=32 small case)",
                   "l2": "inputs larger than L2 (2.1 GB of token rows per step); no flush",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "U_rows": U, "V_rows": V, "alg_bytes_per_step": ab["total"]},
        "tokens_per_s": ab["tokens"] * world / sec_step,
        "frac_of_hbm_peak": value / world / peak,
        "roofline": {"bound": "hbm", "kernel": gather_kernel, "achieved": gather_gbs,
                     "peak": peak, "unit": "GB/s", "frac": gather_gbs / peak,
                     "peak_source": f"{peak_kind} hbm_gbs", "traffic": traffic,
                     "alg_bytes_per_launch": ab["gather_kernel"]},
        "kernels": {
            "batching_index_ms": ph[0] * 1e3, "batching_gather_ms": ph[1] * 1e3,
            "batching_gather_gbs": gather_gbs,
            "unpermute_index_ms": ph[2] * 1e3, "unpermute_reduce_ms": ph[3] * 1e3,
            "unpermute_sort_ms_concurrent": ph[4] * 1e3,
            "unpermute_reduce_gbs": reduce_gbs, "unpermute_reduce_frac": reduce_gbs / peak,
            "batching_gbs": ab["batching"] / (ph[0] + ph[1]) / 1e9,
            "unpermute_gbs": ab["unpermute"] / (ph[2] + ph[3]) / 1e9},
        "gpu_launches": launches_per_step(spec) * args.steps,
        "clocks": clocks,
        "e2e": e2e,
    }
    if not args.no_cpu_baseline and world == 1:
        try:
            line["cpu_baseline"] = cpu_baseline(spec, inp, rmap, probs, ab)
        except Exception as ex:  # the oracle needs g++; report rather than fail the bench
            line["cpu_baseline"] = {"value": None, "error": str(ex)[:200]}
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


# ---------------------------------------------------------------------------
# The other workloads (supplementary timing, one call per iteration)
# ---------------------------------------------------------------------------

def run_workload(args):
    """Time one operation on one of the other workloads: each iteration
    flushes L2 (a 512 MB write) and is timed alone with CUDA events."""
    import torch

    import unpermute_stable_counting_gb300 as usc
    from unpermute_stable_counting_gb300 import _build
    _build.build_library()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    g = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    flush_read = torch.ones(128 << 20, dtype=torch.int32, device=dev) if args.flush == "write-read" else None
    name = args.workload
    if name in ("permute", "permute_padded"):
        # the permute that produces the top-k / padded unpermute inputs
        if name == "permute":
            u = w.make_unpermute_topk(**w.UNPERMUTE_TOPK)
            kw = dict(topk=u["n"] // u["T"])
        else:
            u = w.make_unpermute_padded(**w.UNPERMUTE_PADDED)
            kw = dict(padded_mode=True, capacity=u["n"] // u["Eu"])
        T, H, dt, Eu = u["T"], u["H"], u["tokenDtype"], u["Eu"]
        s = w.ELEM_BYTES[dt]
        x = w.normal_rows(T, H, dt, seed=5)
        tdt = {0: torch.float16, 1: torch.bfloat16, 3: torch.float32}
        xd = g(x.view(np.int16)).view(tdt[dt]) if dt != 3 else g(x)
        md = g(u["routingMap"])
        pairs = int(u["routingMap"].astype(np.int64).sum())
        rows = u["n"] if name == "permute_padded" else pairs
        alg = T * Eu + T * H * s + rows * H * s + u["n"] * 4
        units, unit_name = T, "tokens"
        ws = torch.empty(usc.permute_workspace_size(T, H, dt, Eu, kw.get("topk", 0),
                                                    kw.get("padded_mode", False), kw.get("capacity", 0)),
                         dtype=torch.uint8, device=dev)
        out = None

        def call():
            nonlocal out
            out = usc.moe_permute(xd, md, out=out, workspace=ws, **kw)
        phases = (0, 1)
    elif name == "update_expert":
        # MoeUpdateExpert at the page's maxima: remap + pruning of 512 x 16 ids
        u = w.make_update_expert(**w.UPDATE_EXPERT)
        BS, K = u["expert_ids"].shape
        ids, tab, thr, act = g(u["expert_ids"]), g(u["table"]), g(u["threshold"]), g(u["active"])
        sc = g(u["scales"].view(np.int16)).view(torch.bfloat16)
        # ids, two table words, a bf16 scale, the threshold and the active flag
        # read; an id and a mask byte written, per element
        alg = BS * K * (4 + 8 + 2 + 4 + 1) + BS + K * 4
        units, unit_name = BS, "tokens"
        out = None

        def call():
            nonlocal out
            out = usc.moe_update_expert(ids, tab, local_rank=3, world_size=u["world_size"], balance_mode=0,
                                        scales=sc, threshold=thr, active=act, out=out)
        phases = (0,)
    elif name in ("context", "batching", "batching_index"):
        # the round trip's batching alone, from flat arrays or from a
        # ScheduleContext (256 sessions x 4 micro-batches x 16 tokens x 9;
        # --small: 32 sessions, for profiling); batching_index: its slots and
        # keys with 16-byte rows
        spec = dict(w.ROUNDTRIP_BATCHING_INDEX if name == "batching_index" else w.ROUNDTRIP_BATCHING)
        if args.small:
            spec.update(A=32, session=32)
        inp = w.make_batching(**spec)
        n_sessions = spec["A"]
        Y, H, E, dt = inp["Y"], inp["H"], inp["expertNum"], inp["tokenDtype"]
        El = E // max(inp["layerNum"], 1)
        U = int(((inp["expert_ids"] >= 0) & (inp["expert_ids"] < El)).sum())
        row = H * 2
        alg = (Y * 4 + U * row + U * 12) + (U * row + Y * 16 + E * 16 + 8)
        units, unit_name = U, "slots"
        shape = (inp["A"], inp["BS"], inp["K1"], H)
        out = usc.batching_outputs(Y, H, E, dt, dev)
        td = g(inp["token_data"])
        if name == "context":
            info = w.make_token_info(sessions=n_sessions, micro=4, mbs=16, sel=9, expert_ids=inp["expert_ids"],
                                     layer_ids=inp["layer_id"], flags=1)
            info_d = g(info)
            ctx = w.pack_schedule_context(sessions=n_sessions, micro=4, mbs=16, sel=9, expert_num=El,
                                          info_ptr=info_d.data_ptr(), info_size=info.size,
                                          data_ptr=td.data_ptr(), data_size=td.numel())
            ctx_d = g(ctx)
            ws = torch.empty(usc.batching_context_workspace_size(E, shape, dt, inp["layerNum"], 1),
                             dtype=torch.uint8, device=dev)

            def call():
                usc.ffnwb_batching_context(ctx_d, expert_num=E, max_out_shape=shape, token_dtype=dt,
                                           layer_num=inp["layerNum"], need_schedule=1, out=out,
                                           workspace=ws)
        else:
            ids, sess, micro = g(inp["expert_ids"]), g(inp["session_in"]), g(inp["micro_in"])
            tok = g(inp["token_in"])
            ws = torch.empty(usc.batching_workspace_size(E, shape, dt, inp["layerNum"]), dtype=torch.uint8,
                             device=dev)

            def call():
                usc.ffnwb_batching(ids, td, sess, micro, expert_num=E, max_out_shape=shape, token_dtype=dt,
                                   layer_num=inp["layerNum"], layer_id=inp["layer_id"], token_ids=tok,
                                   out=out, workspace=ws)
        phases = (0, 1)
    elif name in ("tiny", "int8"):
        spec = dict(w.BATCHING_TINY if name == "tiny" else w.BATCHING_INT8_DECODE)
        inp = w.make_batching(**spec)
        Y, H, E, dt = inp["Y"], inp["H"], inp["expertNum"], inp["tokenDtype"]
        El = E // max(inp["layerNum"], 1)
        U = int(((inp["expert_ids"] >= 0) & (inp["expert_ids"] < El)).sum())
        s = 1 if dt == w.DT_INT8 else 2
        sc = 4 if dt == w.DT_INT8 else 0
        alg = (Y * 4 + U * (H * s + sc) + U * 12) + (U * (H * s + sc) + Y * 16 + E * 16 + 8)
        units, unit_name = U, "slots"
        args_d = dict(ids=g(inp["expert_ids"]), td=g(inp["token_data"]), sess=g(inp["session_in"]),
                      micro=g(inp["micro_in"]), tok=g(inp["token_in"]))
        shape = (inp["A"], inp["BS"], inp["K1"], H)
        out = usc.batching_outputs(Y, H, E, dt, dev)
        ws = torch.empty(usc.batching_workspace_size(E, shape, dt, inp["layerNum"]), dtype=torch.uint8,
                         device=dev)

        def call():
            usc.ffnwb_batching(args_d["ids"], args_d["td"], args_d["sess"], args_d["micro"], expert_num=E,
                               max_out_shape=shape, token_dtype=dt, layer_num=inp["layerNum"],
                               layer_id=inp["layer_id"], token_ids=args_d["tok"],
                               token_row_stride=inp["row_stride"], out=out, workspace=ws)
        phases = (0, 1)
    else:
        if name == "topk":
            u = w.make_unpermute_topk(**w.UNPERMUTE_TOPK)
        elif name == "decode_unpermute":
            u = w.make_unpermute_topk(**w.UNPERMUTE_DECODE)
        elif name == "padded_slack":
            u = w.make_unpermute_padded(**w.UNPERMUTE_PADDED_SLACK)
        elif name == "large_map":
            u = w.make_unpermute_topk(**w.UNPERMUTE_LARGE_MAP)
        elif name == "odd_h":
            u = w.make_unpermute_topk(**w.UNPERMUTE_ODD_H)
        elif name == "padded_lsd":
            u = w.make_unpermute_padded(**w.UNPERMUTE_PADDED_LSD)
        else:
            u = w.make_unpermute_padded(**w.UNPERMUTE_PADDED)
        T, H, n, dt, pdt, Eu = u["T"], u["H"], u["n"], u["tokenDtype"], u["probsDtype"], u["Eu"]
        s, ps = w.ELEM_BYTES[dt], w.ELEM_BYTES[pdt]
        si = u["sortedIndices"].astype(np.int64)
        if u["padded"]:
            # indices, prob lookups, the valid rows, the output, outIndex/permuteTokenId/permuteProbs
            V = int(((si >= 0) & (si < T)).sum())
            alg = n * (4 + ps) + V * H * s + T * H * s + n * (8 + ps)
        else:
            pr = u["probs"].reshape(T, Eu)
            pv = pr.T[(u["routingMap"] != 0).T]
            wgt = np.zeros(n, bool)
            wgt[:min(n, pv.size)] = pv[:n] != 0
            V = int((((si >= 0) & (si < u["permutedRows"])) & wgt).sum())
            alg = n * 4 + V * H * s + T * Eu * (1 + ps) + T * H * s + n * (8 + ps)
        units, unit_name = T, "tokens"
        tdt = {0: torch.float16, 1: torch.bfloat16, 3: torch.float32}
        fl = lambda a, d: (g(a) if d == 3 else g(np.ascontiguousarray(a).view(np.int16)).view(tdt[d]))
        perm, sidx, rm, pr_d = fl(u["permuted"], dt), g(u["sortedIndices"]), g(u["routingMap"]), fl(u["probs"], pdt)
        out = usc.unpermute_outputs(T, H, n, dt, pdt, dev)
        ws = torch.empty(usc.unpermute_workspace_size(u["permutedRows"], H, dt, n, True, pdt, T, Eu,
                                                      bool(u["padded"])), dtype=torch.uint8, device=dev)

        def call():
            usc.moe_unpermute(perm, sidx, rm, pr_d, padded_mode=bool(u["padded"]), out=out, workspace=ws)
        # index (probs; with padding also the sort), reduce, and the sort on the
        # auxiliary stream (not padded)
        phases = (2, 3) if u["padded"] else (2, 3, 4)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(10)]
    for _ in range(max(args.warmup, 3)):
        call()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def flush_l2():
        flush.fill_(1)
        if flush_read is not None:
            flush_read.sum()  # evicts the write's dirty lines, leaving clean ones

    # the call alone (its kernels chained by PDL, no events between them)
    tot = []
    for _ in range(args.steps):
        flush_l2()
        e0.record()
        call()
        e1.record()
        torch.cuda.synchronize()
        tot.append(e0.elapsed_time(e1) / 1e3)
    # then the library's phase events, in a pass of their own (an event between
    # two kernels ends their PDL overlap, so these phases sum to a little more)
    ph = {p: [] for p in phases}
    usc.profile_set_events(ev)
    try:
        for _ in range(max(args.steps // 4, 10)):
            flush_l2()
            call()
            torch.cuda.synchronize()
            for p in phases:
                ph[p].append(ev[2 * p].elapsed_time(ev[2 * p + 1]) / 1e3)
    finally:
        usc.profile_set_events(None)
    sec = statistics.median(tot)
    peak, _ = hbm_peak()
    line = {"workload": name, "value": alg / sec / 1e9, "unit": "GB/s", "us_per_call": sec * 1e6,
            "frac_of_hbm_peak": alg / sec / 1e9 / peak, f"{unit_name}_per_s": units / sec,
            "alg_bytes": alg, "phase_us": {str(p): statistics.median(v) * 1e6 for p, v in ph.items()},
            "l2": ("flushed before every call (512 MB write, then 512 MB read)" if flush_read is not None
                   else "flushed before every call (512 MB write)")}
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    if args.workload != "roundtrip":
        return run_workload(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
