"""bench.py host logic without a GPU: the replica ranks' coordination over
gloo (world size 2: barrier, max and sum over ranks, only rank 0 prints) and
the oracle reference arm's JSON line."""
import json
import os
import socket
import subprocess
import sys

import pytest

from conftest import ROOT


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    d = bench.Dist()
    d.barrier()
    got = (d.max(10.0 * (rank + 1)), d.sum(rank + 1))
    d.barrier()
    d.close()
    q.put((rank, got))


def test_two_gloo_ranks_reduce_timings():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0] == (20.0, 3.0) and res[1] == (20.0, 3.0)


def _run_bench(args, env_extra=None, timeout=300):
    env = dict(os.environ)
    env.update(env_extra or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, capture_output=True,
                          text=True, timeout=timeout, env=env, cwd=ROOT)


def test_reference_arm_prints_one_json_line():
    r = _run_bench(["--impl", "reference", "--steps", "1", "--warmup", "1"])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    import bench
    assert d["cpu_baseline"]["kind"] == "oracle"
    # the oracle's attention is shared out over the host's cores (one thread
    # per core, at most one per sequence), and the CPU model is recorded
    assert d["cpu_baseline"]["cores"] == min(bench.host_cpu()[1], 128)
    assert d["cpu_baseline"]["host_cores"] == bench.host_cpu()[1] and d["cpu_baseline"]["cpu"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert d["metric"].startswith("paged decode-attention HBM GB/s")


def test_reference_arm_other_ranks_print_nothing():
    # under torchrun only rank 0 runs the oracle and prints; other ranks
    # return before doing any work
    import bench

    class Rank1:
        rank, world, local_rank = 1, 2, 1
    assert bench.run_reference(bench.parse_args(["--impl", "reference"]), Rank1()) is None


def test_traffic_record_round_trip(tmp_path):
    """--record-traffic reads ncu's raw page (metric names, a units row, one
    row per launch) and the bench reads the bytes back, only while the kernel
    sources are the ones the record names."""
    import bench
    raw = tmp_path / "raw.csv"
    raw.write_text('"ID","Kernel Name","dram__bytes_read.sum","dram__bytes_write.sum","gpu__time_duration.sum"\n'
                   '"","","Mbyte","Kbyte","usecond"\n'
                   '"0","void attn::paged_decode_kernel_mma_r128<64, 1, 4>(...)","188.27","3,619.5","39.21"\n')
    name = "test_traffic_tmp"
    out = bench.record_traffic(str(raw), name, "ncu ...")
    try:
        rec = json.load(open(out))
        assert rec["dram_bytes_read"] == 188270000 and rec["dram_bytes_write"] == 3619500
        assert rec["duration_ns"] == 39210
        assert bench.profile_traffic(name) == 188270000 + 3619500
        rec["kernel_sources_sha16"] = "0" * 16
        json.dump(rec, open(out, "w"))
        assert bench.profile_traffic(name) is None
    finally:
        os.remove(out)
