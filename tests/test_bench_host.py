"""Host logic of bench.py, on the CPU: algorithmic byte counts, launch
counts, the max-over-ranks timing rule with two gloo ranks, and the
reference arm's JSON line."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

import bench
import workloads as w

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_algorithmic_bytes_by_hand():
    spec = dict(A=1, BS=2, K1=3, E=8, H=4, dtype=w.DT_BF16, layerNum=1)
    Y, T, k, row = 6, 2, 3, 8
    U, V = 5, 4
    ab = bench.algorithmic_bytes(spec, U, V)
    assert ab["batching"] == (Y * 4 + U * row + U * 12) + (U * row + Y * 16 + Y * 4 + 8 * 16 + 8)
    assert ab["unpermute"] == (T * k * 4 + V * row + T * k * 3) + (T * row + T * k * 10)
    assert ab["total"] == ab["batching"] + ab["unpermute"]
    assert ab["gather_kernel"] == U * (2 * row + 4)
    assert ab["tokens"] == T and ab["slots"] == Y


def test_roundtrip_workload_bytes_are_about_six_gigabytes():
    spec = bench.workload_spec()
    Y = spec["A"] * spec["BS"] * spec["K1"]
    U = int(0.95 * Y)
    ab = bench.algorithmic_bytes(spec, U, U)
    assert 3.9e9 < ab["batching"] < 4.2e9
    assert 2.1e9 < ab["unpermute"] < 2.4e9


def test_launch_count():
    spec = bench.workload_spec()
    # batching: rank, prefix, scatter, gather; unpermute: maskedSelect (one
    # cooperative kernel for the 16384 x 9 map), the index sort (147457 keys:
    # a coarse pass of 3 launches and the fine sort), reduce
    assert bench.masked_select_launches(64, 64) == 0
    assert bench.masked_select_launches(16384, 9) == 1
    assert bench.masked_select_launches(65536, 64) == 1
    assert bench.masked_select_launches(65600, 64) == 3
    assert bench.sort_launches(147456, 147457) == 4
    assert bench.sort_launches(3000, 4096) == 3
    assert bench.sort_launches(512, 4096) == 1
    assert bench.sort_launches(4096, 4097) == 4
    assert bench.sort_launches(1 << 22, (1 << 22) + 1) == 6       # 23 bits: two LSD passes
    assert bench.sort_launches(1 << 24, (1 << 24) + 1) == 9       # 25 bits: three
    assert bench.launches_per_step(spec) == 4 + 1 + 4 + 1


def test_contributing_rows_counts_valid_nonzero_slots():
    spec = dict(A=1, BS=2, K1=3, E=4, layerNum=1)
    inp = dict(expert_ids=np.array([0, 9, 1, 2, 3, 2**31 - 1], np.int32))
    probs = np.array([[1, 1, 1], [1, 1, 1]], np.uint16)
    # 4 unmasked slots (0, 2, 3, 4) give 4 maskedSelect values; slot i takes
    # the i-th value, so slot 4 gets the zero tail and is skipped
    assert bench.contributing_rows(spec, inp, probs) == 3


def _rank(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    t = bench.max_over_ranks(0.5 + rank, world)
    q.put((rank, t, bench.aggregate_value(1e9, world, t)))
    dist.barrier()
    dist.destroy_process_group()


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def test_max_over_ranks_gloo_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # both ranks see the slowest rank's time; value counts both ranks' bytes
    assert [r[1] for r in res] == [1.5, 1.5]
    assert all(abs(r[2] - 2e9 / 1.5 / 1e9) < 1e-9 for r in res)


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                        "--warmup", "0", "--cpu-sample-attn", "2"], cwd=ROOT, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_print_nothing():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                        "--warmup", "0", "--cpu-sample-attn", "2"], cwd=ROOT, capture_output=True,
                       text=True, timeout=600, env=env)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_reference_arm_size_follows_the_step_budget():
    """The reference arm times the full workload (A = 256) when the run's
    warmup + steps fit its time budget, else a power-of-two fraction."""
    sys.path.insert(0, ROOT)
    import bench
    full = bench.reference_attn(bench.parse_args(["--impl", "reference", "--steps", "20", "--warmup", "3"]))
    assert full == 256
    part = bench.reference_attn(bench.parse_args(["--impl", "reference", "--steps", "200", "--warmup", "10"]))
    assert part < 256 and 210 * bench.ORACLE_STEP_S_FULL * part / 256 <= bench.REFERENCE_BUDGET_S
    assert bench.reference_attn(bench.parse_args(["--cpu-sample-attn", "2"])) == 2


def test_other_path_workloads_reach_their_paths():
    """The recipes of the bench's other-path workloads have the shapes that
    take those paths: the batching kernel chain with short flat-gather rows,
    the three-kernel maskedSelect (more than 4M routing-map entries), the
    element-wise gather-reduce (rows that are not 16-byte vectors) and the
    LSD sort passes (more than 2^22 padded keys)."""
    b = w.ROUNDTRIP_BATCHING_INDEX
    Y = b["A"] * b["BS"] * b["K1"]
    assert Y > 32768 and b["H"] * 2 == 16 and Y * b["H"] * 2 // 16 >= 65536
    m = w.UNPERMUTE_LARGE_MAP
    assert m["T"] * m["Eu"] > (1 << 22)
    o = w.UNPERMUTE_ODD_H
    assert (o["H"] * w.ELEM_BYTES[o["dtype"]]) % 16 != 0
    pl = w.UNPERMUTE_PADDED_LSD
    assert pl["T"] + 1 > (1 << 22)
    src = open(bench.__file__).read()
    for name in ("batching_index", "large_map", "odd_h", "padded_lsd"):
        assert f'"{name}"' in src
