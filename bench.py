#!/usr/bin/env python
"""Benchmark of the paged KV-cache decode step on GB300.

One step = one decode step of one layer over the 128-sequence mixed-length
workload (64 x U[32,128], 38 x U[256,512], 26 x U[1024,2048] tokens; 12 heads
x 64, fp16; a pool of 4096 blocks of 16; shuffled frames): the scatter of each
sequence's new K/V token into its page slot and paged decode attention over
the grown contexts, as one fused call (pf_decode_step).  The same step as two
calls (pf_write_kv, then pf_paged_decode_attention) is timed too.  Inputs are
resident in HBM; the step rotates over pool replicas whose total size is over
three times the L2, so no step finds its pages in L2.

Printed (rank 0, one JSON line): value = algorithmic HBM bytes of the step /
step time (GB/s, whole job), decode tokens/s per layer, attention calls/s,
the same kernels on ordered frames, the gather leg, the roofline of the
attention kernel (CUDA events around every attention launch of the timed
region), an end-to-end number through the public API with host buffers, the
oracle timed on the host cores as a CPU baseline, SM clocks sampled during the
timed work, and the number of kernel launches timed.  Side legs, timed after
the main one: block copies and swaps, appends and prompts, grouped heads
(14/2 x 64) over pages of 1, 16, 64 and 256 tokens, the 13B-like shape (40 x
128 at 2048 tokens, batch 1..64, balanced vs no split) and a GPT-2-shaped
12-layer, 50-step decode loop (eager and replayed from a CUDA graph).

--impl reference times the fp64 CPU oracle on the same workload (the
reference arm of this project).  --gpus N under torchrun runs N independent
replicas (one per GPU, no collective on the data path); timings are the max
over ranks.
"""
import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth_inputs as si  # noqa: E402

METRIC = "paged decode-attention HBM GB/s (% of GB300 peak); decode tokens/s per layer"
SPEC_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
WORKLOAD_NAME = ("mixed-length: 1 layer, 12 heads x d_head 64 fp16, pool 4096 blocks of 16, 128 seqs "
                 "(64 x U[32,128], 38 x U[256,512], 26 x U[1024,2048] tokens, seed 42), shuffled frames (seed 7); "
                 "step = scatter of 128 new tokens + paged decode attention")


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20000)
    p.add_argument("--warmup", type=int, default=50)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--split", type=int, default=0, help="split_tokens (0 auto, -1 never)")
    p.add_argument("--cpu-budget-s", type=float, default=10.0, help="seconds of oracle work for cpu_baseline")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--main-only", action="store_true",
                   help="time the decode step legs only (no side legs): the command profiles are taken with")
    p.add_argument("--cpu-threads", type=int, default=0, help="host threads for the oracle (0: every core)")
    p.add_argument("--record-traffic", metavar="RAW_CSV",
                   help="write profiles/<--profile-name>.json from `ncu -i REP --page raw --csv` output, then exit")
    p.add_argument("--profile-name", default="attention_mixed_shuffled")
    p.add_argument("--profile-command", default="", help="the ncu command the capture came from (recorded)")
    p.add_argument("--prompt-only", action="store_true",
                   help="time only the prompt-attention legs on pools of their own (a small device footprint, "
                        "for profiling); prints one diagnostic JSON line, not the bench line")
    return p.parse_args(argv)


# ------------------------------------------------------------ distributed

class Dist:
    """Host-side coordination of replica ranks (gloo): a barrier and the max
    of a timing.  No collective touches the data path."""

    def __init__(self):
        self.rank = int(os.environ.get("RANK", "0"))
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            dist.init_process_group("gloo", rank=self.rank, world_size=self.world)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x):
        if not self.pg:
            return float(x)
        import torch
        t = torch.tensor([float(x)], dtype=torch.float64)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def sum(self, x):
        if not self.pg:
            return float(x)
        import torch
        t = torch.tensor([float(x)], dtype=torch.float64)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.SUM)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# ---------------------------------------------------------------- bytes

def attention_bytes(lens, n_q_heads, n_kv_heads, head_dim, block_size, out_bytes=2):
    """Algorithmic HBM bytes of one decode-attention call: every K and V byte
    of every context token once per kv-head, q, out, the used block-table
    entries and the lengths."""
    lens = np.asarray(lens, dtype=np.int64)
    kv = int(lens.sum()) * n_kv_heads * head_dim * 2 * 2
    qo = len(lens) * n_q_heads * head_dim * (2 + out_bytes)
    tables = int(((lens + block_size - 1) // block_size).sum()) * 4
    return kv + qo + tables + 4 * len(lens)


def write_bytes(n_tokens, n_kv_heads, head_dim):
    """Scatter: read and write K and V rows, plus seq/pos indices and one
    table entry per token."""
    return 2 * (n_tokens * n_kv_heads * head_dim * 2) * 2 + n_tokens * 12


def gather_bytes(lens, n_kv_heads, head_dim, block_size):
    lens = np.asarray(lens, dtype=np.int64)
    rows = int(lens.sum()) * n_kv_heads * head_dim * 2
    tables = int(((lens + block_size - 1) // block_size).sum()) * 4
    return 2 * rows * 2 + tables + 12 * len(lens)


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def read_tensor_peak():
    """Dense fp16 tensor TFLOP/s: the measured bf16 burst figure (fp16 and bf16
    have the same nominal dense rate), else the fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def profile_record(name):
    """The JSON record that `--record-traffic` wrote from an ncu capture of the
    decode kernel, or None if there is none or the kernel sources changed
    since it was taken."""
    path = os.path.join(ROOT, "profiles", name + ".json")
    try:
        with open(path) as f:
            rec = json.load(f)
        return rec if rec.get("kernel_sources_sha16") == kernel_sources_hash() else None
    except Exception:
        return None


def profile_traffic(name="attention_mixed_shuffled"):
    """DRAM bytes (read + write) of one launch of the decode kernel in that
    capture, or None."""
    rec = profile_record(name)
    return None if rec is None else int(rec["dram_bytes_read"]) + int(rec["dram_bytes_write"])


def profile_dram_summary():
    """Per layout: DRAM bytes and the GB/s they make over the captured
    launch's duration (ncu, one isolated launch: cold caches, serialised)."""
    out = {}
    for layout in ("shuffled", "ordered"):
        rec = profile_record("attention_mixed_" + layout)
        if rec and rec.get("duration_ns"):
            b = int(rec["dram_bytes_read"]) + int(rec["dram_bytes_write"])
            out[layout] = {"dram_bytes": b, "duration_us": rec["duration_ns"] / 1e3,
                           "dram_gbs": round(b / rec["duration_ns"], 1)}
    return out or None


_UNITS = {"byte": 1, "b": 1, "kbyte": 1e3, "kb": 1e3, "mbyte": 1e6, "mb": 1e6, "gbyte": 1e9, "gb": 1e9,
          "tbyte": 1e12, "tb": 1e12}
_NS = {"nsecond": 1, "ns": 1, "usecond": 1e3, "us": 1e3, "msecond": 1e6, "ms": 1e6, "second": 1e9, "s": 1e9}


def record_traffic(raw_csv, name, command):
    """Read `ncu -i REP --page raw --csv` output (a header row of metric names,
    a row of units, then one row per captured launch) and write the DRAM
    bytes of the first decode-kernel launch to profiles/<name>.json."""
    import csv
    rows = list(csv.reader(open(raw_csv)))
    head = next(i for i, r in enumerate(rows) if "dram__bytes_read.sum" in r)
    names, units, data = rows[head], rows[head + 1], rows[head + 2:]
    col = {n: i for i, n in enumerate(names)}
    launch = next(r for r in data if "paged_decode" in r[col["Kernel Name"]])

    def value(metric):
        i = col[metric]
        return int(round(float(launch[i].replace(",", "")) * _UNITS[units[i].strip().lower()]))

    rec = {"kernel": launch[col["Kernel Name"]], "dram_bytes_read": value("dram__bytes_read.sum"),
           "dram_bytes_write": value("dram__bytes_write.sum"),
           "duration_ns": None, "kernel_sources_sha16": kernel_sources_hash(), "command": command}
    if "gpu__time_duration.sum" in col:   # the raw page gives the duration in its own unit
        i = col["gpu__time_duration.sum"]
        scale = _NS[units[i].strip().lower()]
        rec["duration_ns"] = int(round(float(launch[i].replace(",", "")) * scale))
    out = os.path.join(ROOT, "profiles", name + ".json")
    with open(out, "w") as f:
        json.dump(rec, f, indent=1)
        f.write("\n")
    return out


def host_cpu():
    """(model name, logical cores this process may use) of the host."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if not model:
        try:
            for line in open("/proc/cpuinfo"):
                if line.lower().startswith(("model name", "cpu model", "hardware")):
                    model = line.split(":", 1)[1].strip()
                    break
        except Exception:
            pass
    try:
        cores = len(os.sched_getaffinity(0))
    except Exception:
        cores = os.cpu_count() or 1
    import platform
    return f"{model or 'unknown'} ({platform.machine()})", cores


def kernel_sources_hash():
    """Hash of the attention kernel's sources (the profile is only valid for them)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_cache_37_gb300", "csrc")
    for name in ("attention_kernel.cuh", "attention.cu", "attention_d64.cu", "device_common.cuh"):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


# --------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the GPU works."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            cmd = ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits", "-lms", "50"]
            if self.gpu_id:
                cmd += ["-i", self.gpu_id]
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------- workload

def workload():
    w = si.WORKLOADS["mixed"]
    lens = si.band_lengths(w["bands"])
    maxb = 2048 // w["block_size"]
    return w, lens, maxb


def oracle_step_timer(w, lens, bt, budget_s, max_steps=None, threads=0):
    """Run the fp64 oracle's decode step (scatter of the new tokens + paged
    attention) on host copies until budget_s has elapsed; returns (steps,
    seconds, threads).  The attention of a step is shared out over `threads`
    host threads (0: every core this process may use) by sequence, each
    thread calling the oracle on its own sequences (the C oracle runs
    without the interpreter lock); the oracle itself is unchanged."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    oracle.build()
    S = len(lens)
    H, D, B, N = w["n_kv_heads"], w["head_dim"], w["block_size"], w["n_blocks"]
    k = si.pool(1, N, B, H, D, si.SEED_VALUES)
    v = si.pool(1, N, B, H, D, si.SEED_VALUES + 1)
    q = si.fp16_normal((S, w["n_q_heads"], D), si.SEED_VALUES + 2)
    kn = si.fp16_normal((S, H, D), si.SEED_VALUES + 3)
    vn = si.fp16_normal((S, H, D), si.SEED_VALUES + 4)
    seq_idx = np.arange(S, dtype=np.int32)
    pos = (lens - 1).astype(np.int32)
    n = threads or host_cpu()[1]
    n = max(1, min(n, S))
    # longest first onto the least-loaded thread: equal token counts per thread
    load, parts = [0] * n, [[] for _ in range(n)]
    for s in np.argsort(-lens, kind="stable"):
        j = int(np.argmin(load))
        parts[j].append(int(s))
        load[j] += int(lens[s])
    shares = [(q[np.array(p_)], bt[np.array(p_)], lens[np.array(p_)]) for p_ in parts if p_]

    def attend(share):
        oracle.attention_paged(share[0], k, v, 0, share[1], share[2], w["scale"])

    steps, t0 = 0, time.perf_counter()
    with ThreadPoolExecutor(max_workers=len(shares)) as ex:
        while True:
            oracle.scatter(k, v, 0, kn, vn, bt, seq_idx, pos)
            list(ex.map(attend, shares))
            steps += 1
            el = time.perf_counter() - t0
            if el >= budget_s or (max_steps and steps >= max_steps):
                return steps, el, len(shares)


# ----------------------------------------------------------------- ours

def run_ours(args, dist):
    import torch
    import paged_kv_cache_37_gb300 as pkv

    pkv.build()
    lib = pkv.lib()
    device = torch.device("cuda", dist.local_rank)
    torch.cuda.set_device(device)
    props = torch.cuda.get_device_properties(device)
    w, lens, maxb = workload()
    S, Hq, Hkv, D, B, N = len(lens), w["n_q_heads"], w["n_kv_heads"], w["head_dim"], w["block_size"], w["n_blocks"]
    bt_shuf = si.block_tables(lens, B, N, si.SEED_SHUFFLE, max_blocks=maxb)
    bt_ord = si.block_tables(lens, B, N, 0, max_blocks=maxb)

    pool_pair = 2 * pkv.pf_pool_bytes(1, N, B, Hkv, D)
    l2 = getattr(props, "L2_cache_size", 128 << 20) or (128 << 20)
    R = max(3, -(-3 * l2 // pool_pair))
    gen = torch.Generator(device=device)
    reps = []
    for r in range(R):
        gen.manual_seed(si.SEED_VALUES + 10 * r)
        k = torch.randn((1, N, B, Hkv, D), generator=gen, device=device, dtype=torch.float32).half()
        v = torch.randn((1, N, B, Hkv, D), generator=gen, device=device, dtype=torch.float32).half()
        q = torch.randn((S, Hq, D), generator=gen, device=device, dtype=torch.float32).half()
        kn = torch.randn((S, Hkv, D), generator=gen, device=device, dtype=torch.float32).half()
        vn = torch.randn((S, Hkv, D), generator=gen, device=device, dtype=torch.float32).half()
        pool = pkv.pf_pool_create(k, v)
        ws = pkv.make_workspace(pool, S, Hq, maxb, args.split)
        out = torch.empty((S, Hq, D), dtype=torch.float16, device=device)
        reps.append(dict(k=k, v=v, q=q, kn=kn, vn=vn, pool=pool, ws=ws, out=out))
    to = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)
    lens_d = to(lens)
    seq_d = to(np.arange(S, dtype=np.int32))
    pos_d = to((lens - 1).astype(np.int32))
    tables = {"shuffled": to(bt_shuf), "ordered": to(bt_ord)}
    stream = torch.cuda.current_stream(device)
    sp = ctypes.c_void_p(stream.cuda_stream)
    P = lambda t: ctypes.c_void_p(t.data_ptr())

    def arg_sets(layout, overlap=True, split=None):
        split = args.split if split is None else split
        bt = tables[layout]
        key = "ws" if split == args.split else f"ws{split}"
        for r in reps:
            if key not in r:
                r[key] = pkv.make_workspace(r["pool"], S, Hq, maxb, split)
        ws_ = [(P(r[key]), r[key].numel()) for r in reps]
        wr = [(r["pool"].handle, 0, P(r["kn"]), P(r["vn"]), P(bt), S, maxb, P(seq_d), P(pos_d), S, sp) for r in reps]
        at = [(r["pool"].handle, 0, P(r["q"]), P(bt), maxb, P(lens_d), S, Hq, ctypes.c_float(w["scale"]),
               P(r["out"]), pkv.PF_F16, split, ws_[i][0], ws_[i][1], sp) for i, r in enumerate(reps)]
        # consecutive steps write neither the lengths nor the tables, so each
        # step's launch may overlap the previous step's kernel; a call timed
        # on its own (events around it) has nothing to overlap and does not ask
        flag = 0 if overlap is False else pkv.PF_STEP_OVERLAP_PREVIOUS
        fu = [(r["pool"].handle, 0, P(r["q"]), P(r["kn"]), P(r["vn"]), P(bt), maxb, P(lens_d), S, Hq,
               ctypes.c_float(w["scale"]), P(r["out"]), pkv.PF_F16, split, ws_[i][0], ws_[i][1],
               flag, sp)
              for i, r in enumerate(reps)]
        return wr, at, fu

    def check(rc):
        if rc:
            raise pkv.PagedKVError(rc, pkv.pf_last_error())

    def run_steps(layout, n, events=None, fused=True, split=None):
        wr, at, fu = arg_sets(layout, overlap=events is None, split=split)
        for i in range(n):
            r = i % R
            if events is not None:
                events[i][0].record(stream)
            if fused:
                check(lib.pf_decode_step(*fu[r]))
            else:
                check(lib.pf_write_kv(*wr[r]))
                if events is not None:
                    events[i][1].record(stream)
                check(lib.pf_paged_decode_attention(*at[r]))
            if events is not None:
                events[i][2].record(stream)

    def timed(layout, n, with_events=False, fused=True, split=None):
        evs = None
        if with_events:
            evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
        dist.barrier()
        torch.cuda.synchronize(device)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run_steps(layout, n, evs, fused, split)
        e1.record(stream)
        torch.cuda.synchronize(device)
        dist.barrier()
        total_ms = e0.elapsed_time(e1)
        per = None
        if evs:
            if fused:
                per = {"step_ms": statistics.mean(a.elapsed_time(c) for a, _, c in evs)}
            else:
                per = {"write_ms": statistics.mean(a.elapsed_time(b) for a, b, _ in evs),
                       "attn_ms": statistics.mean(b.elapsed_time(c) for _, b, c in evs)}
        return total_ms, per

    # kernels per step: the fused grid (cut pairs are merged inside it), plus
    # a merge grid for fixed chunks (split > 0); one of each per 1024 sequences
    attn_launches = (2 if args.split > 0 else 1) * -(-S // 1024)
    a_bytes = attention_bytes(lens, Hq, Hkv, D, B)
    w_bytes = write_bytes(S, Hkv, D)
    step_bytes = a_bytes + w_bytes
    K, W = args.steps, max(args.warmup, 3)

    gpu_uuid = None
    try:
        gpu_uuid = str(props.uuid)
        if gpu_uuid and not gpu_uuid.startswith("GPU-"):
            gpu_uuid = "GPU-" + gpu_uuid
    except Exception:
        pass
    sampler = ClockSampler(gpu_uuid)
    sampler.start()
    time.sleep(0.2)

    # warm-up (also encodes the TMA descriptors and sizes the grid)
    for fused in (True, False):
        run_steps("shuffled", W, fused=fused)
        run_steps("ordered", W, fused=fused)
    for layout in ("shuffled", "ordered"):   # the CUDA-core consumers (split_tokens -2)
        run_steps(layout, W, split=-2)
    torch.cuda.synchronize(device)
    pkv.pf_device_status(reset=True)

    # the contract's timed region: K fused steps, shuffled frames
    ms_main, _ = timed("shuffled", K)
    ms_main = dist.max(ms_main)
    # the same steps with CUDA events around every call (roofline)
    ms_ev, per = timed("shuffled", K, with_events=True)
    step_call_ms = dist.max(per["step_ms"])
    # ordered frames
    ms_ord, per_ord = timed("ordered", K, with_events=True)
    ms_ord = dist.max(ms_ord)
    step_ord_ms = dist.max(per_ord["step_ms"])
    # the unfused step: pf_write_kv, then pf_paged_decode_attention
    ms_unf, per_unf = timed("shuffled", K, with_events=True, fused=False)
    ms_unf = dist.max(ms_unf)
    attn_ms = dist.max(per_unf["attn_ms"])
    write_ms = dist.max(per_unf["write_ms"])
    # the same fused step on the CUDA-core consumers (balanced spans, fp32
    # warp-shuffle dot products and weights, no tensor cores), both layouts
    cc = {}
    for layout in ("shuffled", "ordered"):
        _, per_cc = timed(layout, K, with_events=True, split=-2)
        cc[layout] = dist.max(per_cc["step_ms"])
    ms_cc_b2b, _ = timed("shuffled", K, split=-2)
    ms_cc_b2b = dist.max(ms_cc_b2b)

    # side legs (skipped with --main-only, e.g. under a profiler)
    peak, peak_src = read_peaks()
    tc_peak, tc_src = read_tensor_peak()
    side = {}
    if not args.main_only:
        # gather leg: rebuild contiguous K/V for the whole batch
        off = si.cu_offsets(lens)
        T = int(off[-1])
        off_d = to(off[:-1])
        outs = [(torch.empty((T, Hkv, D), dtype=torch.float16, device=device),
                 torch.empty((T, Hkv, D), dtype=torch.float16, device=device)) for _ in range(R)]
        g_args = [(reps[r]["pool"].handle, 0, P(tables["shuffled"]), maxb, P(lens_d), P(off_d), S,
                   P(outs[r][0]), P(outs[r][1]), sp) for r in range(R)]
        for i in range(W):
            check(lib.pf_gather_kv(*g_args[i % R]))
        Kg = max(10, K // 10)
        dist.barrier()
        torch.cuda.synchronize(device)
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for i in range(Kg):
            check(lib.pf_gather_kv(*g_args[i % R]))
        g1.record(stream)
        torch.cuda.synchronize(device)
        gather_ms = dist.max(g0.elapsed_time(g1) / Kg)
        g_bytes = gather_bytes(lens, Hkv, D, B)
        del outs
        # the platform's own device copy of the same bytes (half read, half
        # written), two buffer pairs alternating: the measured copy peak comes
        # from a 4 GB copy, and a copy of this size ramps up and drains in a
        # visible share of its time
        half = g_bytes // 2 // 2
        cp_bufs = [(torch.empty(half, dtype=torch.float16, device=device),
                    torch.empty(half, dtype=torch.float16, device=device)) for _ in range(2)]
        for i in range(W):
            cp_bufs[i % 2][1].copy_(cp_bufs[i % 2][0])
        dist.barrier()
        torch.cuda.synchronize(device)
        g0.record(stream)
        for i in range(Kg):
            cp_bufs[i % 2][1].copy_(cp_bufs[i % 2][0])
        g1.record(stream)
        torch.cuda.synchronize(device)
        copy_same_ms = dist.max(g0.elapsed_time(g1) / Kg)
        del cp_bufs

        # whole-block legs: copy-on-write copies inside a pool (half the pool's
        # blocks onto the other half) and swapping the same blocks out to pinned
        # host memory and back in; bytes = every image read once and written once
        img = pkv.pf_block_image_bytes(reps[0]["pool"])
        nb = w["n_blocks"] // 2
        src_ids = to(np.arange(nb, dtype=np.int32))
        dst_ids = to(np.arange(nb, 2 * nb, dtype=np.int32))
        blk_bytes = 2 * nb * img
        swap_buf = torch.empty(nb * img, dtype=torch.uint8).pin_memory()

        def time_calls(fn, n):
            for i in range(3):
                fn(i)
            dist.barrier()
            torch.cuda.synchronize(device)
            b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            b0.record(stream)
            for i in range(n):
                fn(i)
            b1.record(stream)
            torch.cuda.synchronize(device)
            return dist.max(b0.elapsed_time(b1) / n)

        copy_ms = time_calls(lambda i: check(lib.pf_copy_blocks(reps[i % R]["pool"].handle, P(src_ids), P(dst_ids),
                                                                 nb, sp)), Kg)
        swap_out_ms = time_calls(lambda i: check(lib.pf_swap_out(reps[i % R]["pool"].handle, P(src_ids), nb,
                                                                  P(swap_buf), sp)), 10)
        swap_in_ms = time_calls(lambda i: check(lib.pf_swap_in(reps[i % R]["pool"].handle, P(swap_buf), P(dst_ids),
                                                                nb, sp)), 10)
        # the platform's own rate for the same bytes: copy-engine copies between
        # device memory and the same pinned buffer
        ce_dev = torch.empty(nb * img, dtype=torch.uint8, device=device)
        ce_d2h_ms = time_calls(lambda i: swap_buf.copy_(ce_dev, non_blocking=True), 10)
        ce_h2d_ms = time_calls(lambda i: ce_dev.copy_(swap_buf, non_blocking=True), 10)
        del swap_buf, ce_dev

        # multi-token append legs.  (1) 8 new tokens at the end of every sequence
        # of the workload (each sequence's K/V read once per kv-head: HBM-bound);
        # (2) whole prompts, 4 x 2048 tokens (causal attention over each prompt:
        # fp32 FMA-bound on the CUDA cores)
        n_app = 8
        cu_app = to(np.arange(S + 1, dtype=np.int32) * n_app)
        q_app = torch.randn((S * n_app, Hq, D), device=device).half()
        o_app = torch.empty_like(q_app)
        # the decode kernel takes it (8 tokens x 1 q-head = 8 rows per kv-head)
        app_ws = [pkv.make_prefill_workspace(reps[r]["pool"], S, Hq, maxb, n_app) for r in range(R)]
        app_args = [(reps[r]["pool"].handle, 0, P(q_app), P(tables["shuffled"]), maxb, P(lens_d), P(cu_app), S, n_app,
                     Hq, ctypes.c_float(w["scale"]), P(o_app), pkv.PF_F16, P(app_ws[r]), app_ws[r].numel(), sp)
                    for r in range(R)]
        app_ms = time_calls(lambda i: check(lib.pf_paged_prefill_attention(*app_args[i % R])), Kg)
        # the same append through the kernel that needs no workspace
        app2_args = [a_[:13] + (None, 0, sp) for a_ in app_args]
        app2_ms = time_calls(lambda i: check(lib.pf_paged_prefill_attention(*app2_args[i % R])), Kg)
        del app_ws
        app_bytes = attention_bytes(lens, Hq, Hkv, D, B) + (n_app - 1) * S * Hq * D * 2 * 2 + 4 * (S + 1)
        Lp, Sp = 2048, 4
        pr_lens = to(np.full(Sp, Lp, dtype=np.int32))
        pr_bt = to(np.arange(Sp * Lp // B, dtype=np.int32).reshape(Sp, Lp // B))
        pr_cu = to(np.arange(Sp + 1, dtype=np.int32) * Lp)
        q_pr = torch.randn((Sp * Lp, Hq, D), device=device).half()
        o_pr = torch.empty_like(q_pr)
        pr_args = (reps[0]["pool"].handle, 0, P(q_pr), P(pr_bt), Lp // B, P(pr_lens), P(pr_cu), Sp, Lp, Hq,
                   ctypes.c_float(w["scale"]), P(o_pr), pkv.PF_F16, None, 0, sp)
        pr_ms = time_calls(lambda i: check(lib.pf_paged_prefill_attention(*pr_args)), 50)
        pr_flops = 4.0 * Hq * D * Sp * Lp * (Lp + 1) / 2        # q.k and p.v over every causal pair
        del q_app, o_app, q_pr, o_pr
        # the same prompts with grouped heads at head_dim 128 (32 q-heads over
        # 8 kv-heads), on a pool of its own
        gq_Hq, gq_Hkv, gq_D = 32, 8, 128
        gq_nb = Sp * Lp // B
        gq_k = torch.randn((1, gq_nb, B, gq_Hkv, gq_D), device=device).half()
        gq_v = torch.randn((1, gq_nb, B, gq_Hkv, gq_D), device=device).half()
        gq_pool = pkv.pf_pool_create(gq_k, gq_v)
        gq_bt = to(np.random.default_rng(si.SEED_SHUFFLE).permutation(gq_nb).astype(np.int32).reshape(Sp, Lp // B))
        gq_q = torch.randn((Sp * Lp, gq_Hq, gq_D), device=device).half()
        gq_o = torch.empty_like(gq_q)
        gq_args = (gq_pool.handle, 0, P(gq_q), P(gq_bt), Lp // B, P(pr_lens), P(pr_cu), Sp, Lp, gq_Hq,
                   ctypes.c_float(1.0 / np.sqrt(gq_D)), P(gq_o), pkv.PF_F16, None, 0, sp)
        gq_ms = time_calls(lambda i: check(lib.pf_paged_prefill_attention(*gq_args)), 50)
        gq_flops = 4.0 * gq_Hq * gq_D * Sp * Lp * (Lp + 1) / 2
        del gq_k, gq_v, gq_pool, gq_q, gq_o

        # grouped heads: 14 q-heads over 2 kv-heads x 64, 256 sequences of
        # U[32, 4096] tokens (each K/V byte serves 7 q-heads), attention alone
        wg = si.WORKLOADS["gqa"]
        g_lens = si.uniform_lengths(wg["n_seqs"], wg["len_lo"], wg["len_hi"], seed=12)
        gHq, gHkv, gD, gB = wg["n_q_heads"], wg["n_kv_heads"], wg["head_dim"], 16
        gN = int(sum(-(-int(L_) // gB) for L_ in g_lens)) + 64
        g_maxb = -(-int(g_lens.max()) // gB)
        g_bt = to(si.block_tables(g_lens, gB, gN, si.SEED_SHUFFLE, max_blocks=g_maxb))
        g_lens_d = to(g_lens)
        g_reps = []
        for r in range(2):
            gk = torch.empty((1, gN, gB, gHkv, gD), dtype=torch.float16, device=device).normal_()
            gv = torch.empty_like(gk).normal_()
            gpool = pkv.pf_pool_create(gk, gv)
            gq = torch.empty((wg["n_seqs"], gHq, gD), dtype=torch.float16, device=device).normal_()
            g_reps.append((gk, gv, gpool, gq, torch.empty_like(gq), pkv.make_workspace(gpool, wg["n_seqs"], gHq, g_maxb)))
        g_args = [(gr[2].handle, 0, P(gr[3]), P(g_bt), g_maxb, P(g_lens_d), wg["n_seqs"], gHq, ctypes.c_float(wg["scale"]),
                   P(gr[4]), pkv.PF_F16, 0, P(gr[5]), gr[5].numel(), sp) for gr in g_reps]
        gqa_ms = time_calls(lambda i: check(lib.pf_paged_decode_attention(*g_args[i % 2])), Kg)
        gqa_bytes = attention_bytes(g_lens, gHq, gHkv, gD, gB)
        del g_reps
        # the same token counts stored in pages of 1, 64 and 256 tokens
        gqa_sweep = [{"block_size": gB, "ms": round(gqa_ms, 5), "gbs": round(gqa_bytes / (gqa_ms / 1e3) / 1e9, 1)}]
        for bs in (1, 64, 256):
            sN = int(sum(-(-int(L_) // bs) for L_ in g_lens)) + 64
            s_maxb = -(-int(g_lens.max()) // bs)
            s_bt = to(si.block_tables(g_lens, bs, sN, si.SEED_SHUFFLE, max_blocks=s_maxb))
            s_reps = []
            for r in range(2):
                sk = torch.empty((1, sN, bs, gHkv, gD), dtype=torch.float16, device=device).normal_()
                sv = torch.empty_like(sk).normal_()
                spool = pkv.pf_pool_create(sk, sv)
                s_reps.append((sk, sv, spool, pkv.make_workspace(spool, wg["n_seqs"], gHq, s_maxb),
                               torch.empty((wg["n_seqs"], gHq, gD), dtype=torch.float16, device=device)))
            gq0 = torch.empty((wg["n_seqs"], gHq, gD), dtype=torch.float16, device=device).normal_()
            s_args = [(sr[2].handle, 0, P(gq0), P(s_bt), s_maxb, P(g_lens_d), wg["n_seqs"], gHq,
                       ctypes.c_float(wg["scale"]), P(sr[4]), pkv.PF_F16, 0, P(sr[3]), sr[3].numel(), sp) for sr in s_reps]
            s_ms = time_calls(lambda i: check(lib.pf_paged_decode_attention(*s_args[i % 2])), max(10, Kg // 4))
            s_bytes = attention_bytes(g_lens, gHq, gHkv, gD, bs)
            gqa_sweep.append({"block_size": bs, "ms": round(s_ms, 5), "gbs": round(s_bytes / (s_ms / 1e3) / 1e9, 1)})
            del s_reps, gq0

        # 13B-like: 40 heads x 128, every sequence at 2048 tokens, batch 1 .. 64,
        # the balanced schedule (split_tokens 0) against no split (-1).  One pool
        # of 64 x 128 pages; a batch of S rotates over 64 / S disjoint table sets,
        # so no call finds its pages in L2.
        w13 = si.WORKLOADS["13b"]
        c13, H13, D13, B13 = w13["context_len"], w13["n_q_heads"], w13["head_dim"], w13["block_size"]
        pages13 = c13 // B13
        N13 = 64 * pages13
        k13 = torch.empty((1, N13, B13, H13, D13), dtype=torch.float16, device=device).normal_()
        v13 = torch.empty_like(k13).normal_()
        pool13 = pkv.pf_pool_create(k13, v13)
        bt13 = si.block_tables(np.full(64, c13, dtype=np.int32), B13, N13, si.SEED_SHUFFLE, max_blocks=pages13)
        split13 = []
        for S13 in w13["batches"]:
            sets = 64 // S13
            tabs = [to(np.ascontiguousarray(bt13[j * S13:(j + 1) * S13])) for j in range(sets)]
            l13 = to(np.full(S13, c13, dtype=np.int32))
            q13 = torch.empty((S13, H13, D13), dtype=torch.float16, device=device).normal_()
            o13 = torch.empty_like(q13)
            row = {"batch": S13}
            b13 = attention_bytes(np.full(S13, c13), H13, H13, D13, B13)
            for name_, spl in (("balanced", 0), ("no_split", -1)):
                ws13 = pkv.make_workspace(pool13, S13, H13, pages13, spl)
                a13 = [(pool13.handle, 0, P(q13), P(t_), pages13, P(l13), S13, H13, ctypes.c_float(w13["scale"]),
                        P(o13), pkv.PF_F16, spl, P(ws13), ws13.numel(), sp) for t_ in tabs]
                ms13 = time_calls(lambda i: check(lib.pf_paged_decode_attention(*a13[i % sets])), 20)
                row[name_ + "_us"] = round(ms13 * 1e3, 2)
                row[name_ + "_gbs"] = round(b13 / (ms13 / 1e3) / 1e9, 1)
            split13.append(row)
        del k13, v13, pool13

        # GPT-2-shaped decode loop: 12 layers x 12 heads x 64, 32 sequences with
        # prompts of U[16, 64] tokens, 50 decode steps of one fused call per
        # layer (launch-bound: ~9 MB per layer call).  Pages for the final
        # lengths are allocated up front; step i attends over prompt + i + 1.
        w2 = si.WORKLOADS["gpt2"]
        S2, L2n, H2, D2, B2 = w2["n_seqs"], w2["n_layers"], w2["n_q_heads"], w2["head_dim"], w2["block_size"]
        steps2 = w2["decode_steps"]
        pr2 = si.uniform_lengths(S2, w2["prompt_lo"], w2["prompt_hi"])
        N2 = S2 * w2["tokens_per_seq"] // B2
        maxb2 = w2["tokens_per_seq"] // B2
        bt2 = to(si.block_tables(pr2 + steps2, B2, N2, si.SEED_SHUFFLE, max_blocks=maxb2))
        lens2 = to(np.stack([pr2 + i + 1 for i in range(steps2)]).astype(np.int32))
        k2 = torch.empty((L2n, N2, B2, H2, D2), dtype=torch.float16, device=device).normal_()
        v2 = torch.empty_like(k2).normal_()
        pool2 = pkv.pf_pool_create(k2, v2)
        q2 = torch.empty((L2n, S2, H2, D2), dtype=torch.float16, device=device).normal_()
        kn2 = torch.empty((L2n, S2, H2, D2), dtype=torch.float16, device=device).normal_()
        o2 = torch.empty_like(q2)
        ws2 = pkv.make_workspace(pool2, S2, H2, maxb2, 0)
        args2 = [[(pool2.handle, l_, P(q2[l_]), P(kn2[l_]), P(kn2[l_]), P(bt2), maxb2, P(lens2[i]), S2, H2,
                   ctypes.c_float(w2["scale"]), P(o2[l_]), pkv.PF_F16, 0, P(ws2), ws2.numel(),
                   pkv.PF_STEP_OVERLAP_PREVIOUS, sp) for l_ in range(L2n)] for i in range(steps2)]

        def decode_loop(_):
            for i in range(steps2):
                for l_ in range(L2n):
                    check(lib.pf_decode_step(*args2[i][l_]))

        loop_ms = time_calls(decode_loop, 5)
        bytes2 = sum(attention_bytes(pr2 + i + 1, H2, H2, D2, B2) + write_bytes(S2, H2, D2) for i in range(steps2)) * L2n
        gpt2 = {"workload": "12 layers x 12 heads x 64, 32 sequences, prompts U[16,64], 50 decode steps, block 16, "
                            "pool of 512 tokens per sequence, shuffled frames",
                "ms_per_decode_step": round(loop_ms / steps2, 5),
                "us_per_layer_call": round(loop_ms / steps2 / L2n * 1e3, 2),
                "tokens_per_s_per_layer": round(S2 / (loop_ms / steps2 / L2n / 1e3), 1),
                "gbs": round(bytes2 / (loop_ms / 1e3) / 1e9, 1)}
        # the same 600 calls replayed from a CUDA graph (launch cost removed)
        try:
            gstream = torch.cuda.Stream(device)
            graph = torch.cuda.CUDAGraph()
            gsp = ctypes.c_void_p(gstream.cuda_stream)
            gargs = [[a_[:-1] + (gsp,) for a_ in row_] for row_ in args2]
            with torch.cuda.stream(gstream):
                decode_loop(0)   # warm on the capture stream
            torch.cuda.synchronize(device)
            with torch.cuda.graph(graph, stream=gstream):
                for i in range(steps2):
                    for l_ in range(L2n):
                        check(lib.pf_decode_step(*gargs[i][l_]))
            graph_ms = time_calls(lambda i: graph.replay(), 5)
            gpt2["graph_ms_per_decode_step"] = round(graph_ms / steps2, 5)
            gpt2["graph_tokens_per_s_per_layer"] = round(S2 / (graph_ms / steps2 / L2n / 1e3), 1)
            del graph
        except Exception as exc:   # capture is an optional view of the same work
            gpt2["graph_error"] = str(exc)[:200]
        del k2, v2, pool2

        side = {
            "block_copies": {"blocks": nb, "bytes": blk_bytes, "image_bytes": img,
                             "copy_gbs": round(blk_bytes / (copy_ms / 1e3) / 1e9, 1), "copy_ms": round(copy_ms, 5),
                             "copy_frac_of_measured_copy": round(blk_bytes / (copy_ms / 1e3) / 1e9 / peak, 4),
                             "swap_out_gbs": round(blk_bytes / 2 / (swap_out_ms / 1e3) / 1e9, 1),
                             "swap_in_gbs": round(blk_bytes / 2 / (swap_in_ms / 1e3) / 1e9, 1),
                             "copy_engine_d2h_gbs": round(blk_bytes / 2 / (ce_d2h_ms / 1e3) / 1e9, 1),
                             "copy_engine_h2d_gbs": round(blk_bytes / 2 / (ce_h2d_ms / 1e3) / 1e9, 1),
                             "swap_out_frac_of_copy_engine": round(ce_d2h_ms / swap_out_ms, 4),
                             "swap_in_frac_of_copy_engine": round(ce_h2d_ms / swap_in_ms, 4),
                             "swap_note": "GB/s of images moved between HBM and page-locked host memory; the "
                                          "copy engine's rate for the same bytes and buffer is the roofline"},
            "append_attention": {"new_tokens_per_seq": n_app, "ms": round(app_ms, 5), "bytes": app_bytes,
                                 "gbs": round(app_bytes / (app_ms / 1e3) / 1e9, 1),
                                 "frac_of_measured_copy": round(app_bytes / (app_ms / 1e3) / 1e9 / peak, 4),
                                 "kernel": "paged_decode_kernel_mma_r128<64,8,4> (8 rows per kv-head on tensor cores, "
                                           "workspace path)",
                                 "without_workspace_ms": round(app2_ms, 5),
                                 "without_workspace_gbs": round(app_bytes / (app2_ms / 1e3) / 1e9, 1)},
            "prompt_prefill": {"prompts": Sp, "tokens": Lp, "ms": round(pr_ms, 4), "flops": pr_flops,
                               "tflops": round(pr_flops / (pr_ms / 1e3) / 1e12, 2), "bound": "tensor",
                               "peak_tflops": tc_peak,
                               "frac": round(pr_flops / (pr_ms / 1e3) / 1e12 / tc_peak, 4),
                               "kernel": "prefill_tc_kernel<64> (tcgen05.mma, fp32 accumulators in tensor memory)",
                               "peak_note": f"{tc_src} dense bf16 burst TFLOP/s (MEASURED_PEAKS.json bf16_tflops; fp16 "
                                            "has the same nominal rate)"},
            "prompt_prefill_gqa128": {"prompts": Sp, "tokens": Lp, "q_heads": gq_Hq, "kv_heads": gq_Hkv,
                                      "head_dim": gq_D, "ms": round(gq_ms, 4), "flops": gq_flops,
                                      "tflops": round(gq_flops / (gq_ms / 1e3) / 1e12, 2), "bound": "tensor",
                                      "frac": round(gq_flops / (gq_ms / 1e3) / 1e12 / tc_peak, 4),
                                      "kernel": "prefill_tc_kernel<128>"},
            "gqa_attention": {"workload": "256 sequences of U[32,4096] tokens, 14 q-heads / 2 kv-heads x 64, "
                                          "block 16, shuffled frames", "kernel": "paged_decode_kernel_mma_r128<64,8,2> "
                                          "(7 rows per kv-head on tensor cores)", "ms": round(gqa_ms, 5), "bytes": gqa_bytes,
                              "gbs": round(gqa_bytes / (gqa_ms / 1e3) / 1e9, 1),
                              "frac_of_measured_copy": round(gqa_bytes / (gqa_ms / 1e3) / 1e9 / peak, 4)},
            "gqa_block_sizes": gqa_sweep,
            "split_13b": {"workload": "40 heads x 128, 2048 tokens per sequence, block 16, shuffled frames",
                          "rows": split13},
            "decode_loop_gpt2": gpt2,
            "gather": {"gbs": round(g_bytes / (gather_ms / 1e3) / 1e9, 1), "ms": round(gather_ms, 5),
                       "bytes": g_bytes, "frac_of_measured_copy": round(g_bytes / (gather_ms / 1e3) / 1e9 / peak, 4),
                       "copy_same_bytes_gbs": round(g_bytes / (copy_same_ms / 1e3) / 1e9, 1),
                       "frac_of_same_size_copy": round(copy_same_ms / gather_ms, 4),
                       "copy_note": "torch's device copy of the same bytes on this GPU; the measured copy peak "
                                    "is a 4 GB copy"},
        }
    clocks = sampler.stop()
    status = pkv.pf_device_status(reset=True)
    if status:
        raise RuntimeError(f"device status word {status} after the timed runs")

    # end to end through the public API: host buffers in pinned memory, the
    # step's inputs copied in and its output copied back inside the timed loop
    e2e = None
    if not args.no_e2e:
        # The step's inputs (q, the new K and V rows, tables, lengths) sit in
        # one pinned staging buffer and go over in one copy; the device-side
        # tensors are views of one buffer (each part 16-byte aligned).
        parts = {"q": reps[0]["q"].cpu(), "kn": reps[0]["kn"].cpu(), "vn": reps[0]["vn"].cpu(),
                 "bt": torch.from_numpy(bt_shuf), "lens": torch.from_numpy(lens)}
        offs, total = {}, 0
        for k_, v_ in parts.items():
            offs[k_] = total
            total += -(-v_.numel() * v_.element_size() // 16) * 16
        host_buf = torch.zeros(total, dtype=torch.uint8).pin_memory()
        dev_buf = torch.empty(total, dtype=torch.uint8, device=device)

        def view(buf, k_):
            v_ = parts[k_]
            nb = v_.numel() * v_.element_size()
            return buf[offs[k_]:offs[k_] + nb].view(v_.dtype).view(v_.shape)

        for k_ in parts:
            view(host_buf, k_).copy_(parts[k_])
        # two device input buffers: step i reads buffer i % 2 while the copy
        # stream brings step i + 1's inputs into the other one and reads step
        # i's output back as soon as it is done
        dev_bufs = [dev_buf, torch.empty(total, dtype=torch.uint8, device=device)]
        dev_in = [{k_: view(b_, k_) for k_ in parts} for b_ in dev_bufs]
        host_out = torch.empty((S, Hq, D), dtype=torch.float16).pin_memory()
        h2d = total
        d2h = host_out.numel() * host_out.element_size()
        Ke = max(10, min(K, 2000))
        copy_stream = torch.cuda.Stream(device)
        ev_in = [torch.cuda.Event() for _ in range(2)]     # inputs of buffer b are on the device
        ev_k = [torch.cuda.Event() for _ in range(2)]      # the step that read buffer b is done
        e_args = [[(r["pool"].handle, 0, P(di["q"]), P(di["kn"]), P(di["vn"]), P(di["bt"]), maxb, P(di["lens"]), S,
                    Hq, ctypes.c_float(w["scale"]), P(r["out"]), pkv.PF_F16, args.split, P(r["ws"]),
                    r["ws"].numel(), 0, sp) for di in dev_in] for r in reps]

        def stage_inputs(b):
            with torch.cuda.stream(copy_stream):
                dev_bufs[b].copy_(host_buf, non_blocking=True)
                ev_in[b].record(copy_stream)

        def e2e_step(i):
            b = i % 2
            r = i % R
            stream.wait_event(ev_in[b])
            check(lib.pf_decode_step(*e_args[r][b]))
            ev_k[b].record(stream)
            with torch.cuda.stream(copy_stream):
                copy_stream.wait_event(ev_k[1 - b])          # the previous step is done with the other buffer
                dev_bufs[1 - b].copy_(host_buf, non_blocking=True)
                ev_in[1 - b].record(copy_stream)
                copy_stream.wait_event(ev_k[b])              # this step's output
                host_out.copy_(reps[r]["out"], non_blocking=True)

        def e2e_run(n):
            for b in range(2):
                ev_k[b].record(stream)
            stage_inputs(0)
            for i in range(n):
                e2e_step(i)

        e2e_run(W)
        torch.cuda.synchronize(device)
        dist.barrier()
        t0 = time.perf_counter()
        e2e_run(Ke)
        torch.cuda.synchronize(device)
        el = dist.max(time.perf_counter() - t0)
        e2e = {"value": round(dist.sum(step_bytes) * Ke / el / 1e9, 2), "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": Ke,
               "ms_per_step": round(el * 1e3 / Ke, 4),
               "tokens_per_s_per_layer": round(dist.sum(S) * Ke / el, 1),
               "call": "pf_decode_step through the C ABI; each step's inputs copied in from one pinned buffer "
                       "and its output read back to pinned memory, on a copy stream overlapping the other steps"}

    step_s = ms_main / 1e3 / K
    call_s = step_call_ms / 1e3
    achieved = step_bytes / call_s / 1e9
    n = dist.world
    res = {
        "metric": METRIC,
        "value": round(dist.sum(step_bytes) / step_s / 1e9, 2),
        "unit": "GB/s",
        "n_gpus": n,
        "steps": K,
        "warmup": W,
        "ms_per_step": round(ms_main / K, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f16",
        "accumulate": "f32",
        "data": "synthetic",
        "config": {"workload": WORKLOAD_NAME, "split_tokens": args.split, "parallelism": f"replicas x{n}",
                   "l2": f"rotating {R} pool replicas ({R * pool_pair / 1e6:.0f} MB) > 3x L2 ({l2 / 1e6:.0f} MB)",
                   "step_bytes": step_bytes, "attention_bytes": a_bytes, "write_bytes": w_bytes,
                   "tokens_in_context": int(lens.sum()), "step_call": "pf_decode_step (fused scatter + attention, PF_STEP_OVERLAP_PREVIOUS)"},
        "tokens_per_s_per_layer": round(dist.sum(S) / step_s, 1),
        "attention_calls_per_s": round(n / call_s, 1),
        "pct_of_peak": {"step_vs_measured_copy": round(achieved / peak, 4),
                        "step_vs_8TBs_spec": round(achieved / SPEC_HBM_GBS, 4)},
        "per_call_ms": {"decode_step_fused": round(step_call_ms, 5),
                        "steps_back_to_back": round(ms_main / K, 5),
                        "steps_with_events": round(ms_ev / K, 5)},
        "unfused": {"ms_per_step": round(ms_unf / K, 5), "write_kv_ms": round(write_ms, 5),
                    "attention_ms": round(attn_ms, 5),
                    "attention_gbs": round(a_bytes / (attn_ms / 1e3) / 1e9, 1),
                    "attention_frac_of_measured_copy": round(a_bytes / (attn_ms / 1e3) / 1e9 / peak, 4)},
        "ordered": {"ms_per_step": round(ms_ord / K, 5), "decode_step_ms": round(step_ord_ms, 5),
                    "gbs": round(step_bytes / (step_ord_ms / 1e3) / 1e9, 1),
                    "shuffled_over_ordered_time": round(step_call_ms / step_ord_ms, 4)},
        "cuda_cores": {"split_tokens": -2,
                       "consumers": "warp-shuffle q.K over 8-lane groups, fp32 online softmax and weights, "
                                    "no tensor cores (paged_decode_kernel_r128<64,1,4>)",
                       "decode_step_ms": round(cc["shuffled"], 5),
                       "gbs": round(step_bytes / (cc["shuffled"] / 1e3) / 1e9, 1),
                       "frac_of_measured_copy": round(step_bytes / (cc["shuffled"] / 1e3) / 1e9 / peak, 4),
                       "ordered_decode_step_ms": round(cc["ordered"], 5),
                       "ordered_gbs": round(step_bytes / (cc["ordered"] / 1e3) / 1e9, 1),
                       "shuffled_over_ordered_time": round(cc["shuffled"] / cc["ordered"], 4),
                       "steps_back_to_back_ms": round(ms_cc_b2b / K, 5)},
        **side,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": profile_traffic(),
                     "ncu_dram": profile_dram_summary(),
                     "kernel": "pf_decode_step (paged_decode_kernel_mma_r128<64,1,4>: tensor-core consumers, fused write, "
                               "attention, in-kernel merge)",
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_src == "measured" else "fallback 6.8 TB/s"},
        "e2e": e2e,
        "gpu_launches": K * attn_launches,
        "clocks": clocks,
    }
    if dist.rank == 0:
        steps_cpu, el, nthr = oracle_step_timer(w, lens, bt_shuf, args.cpu_budget_s, threads=args.cpu_threads)
        model, ncores = host_cpu()
        res["cpu_baseline"] = {"value": round(step_bytes * steps_cpu / el / 1e9, 4), "unit": "GB/s", "cores": nthr,
                               "kind": "oracle", "cpu": model, "host_cores": ncores,
                               "sample": f"{steps_cpu} full decode steps of the same workload (scatter + fp64 "
                                         f"two-pass attention) in {el:.1f} s, the attention shared by sequence "
                                         f"over {nthr} threads"}
    return res


# ------------------------------------------------------------ reference

def run_reference(args, dist):
    """The reference arm: the fp64 CPU oracle on the same workload, metric and
    unit.  Each step is the full decode step; W + K steps are capped to keep
    the run within a few minutes (the cap and the sample are reported)."""
    if dist.rank != 0:
        return None
    w, lens, maxb = workload()
    bt = si.block_tables(lens, w["block_size"], w["n_blocks"], si.SEED_SHUFFLE, max_blocks=maxb)
    S = len(lens)
    step_bytes = (attention_bytes(lens, w["n_q_heads"], w["n_kv_heads"], w["head_dim"], w["block_size"]) +
                  write_bytes(S, w["n_kv_heads"], w["head_dim"]))
    # warm-up steps (untimed), then timed steps, both capped
    oracle_step_timer(w, lens, bt, 0.0, max_steps=max(1, min(args.warmup, 3)), threads=args.cpu_threads)
    k_cap = max(1, min(args.steps, 100))
    steps, el, nthr = oracle_step_timer(w, lens, bt, 1e9, max_steps=k_cap, threads=args.cpu_threads)
    value = step_bytes * steps / el / 1e9
    model, ncores = host_cpu()
    sample = (f"{steps} full decode steps (scatter + fp64 two-pass paged attention), the attention shared by "
              f"sequence over {nthr} threads")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": args.gpus,
        "steps": steps, "warmup": args.warmup, "ms_per_step": round(el * 1e3 / steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD_NAME, "split_tokens": args.split, "parallelism": f"host, {nthr} threads"},
        "tokens_per_s_per_layer": round(S * steps / el, 2),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": nthr, "kind": "oracle", "cpu": model,
                         "host_cores": ncores, "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_prompt_only(args):
    """The prompt legs alone: 4 prompts of 2048 tokens, 12 heads x 64 and 32
    q-heads over 8 kv-heads x 128, pages of 16 tokens in shuffled frames, each
    on a pool holding just those pages (a few tens of MB on the device)."""
    import numpy as np
    import torch
    import paged_kv_cache_37_gb300 as pkv
    pkv.lib()
    device = torch.device("cuda", 0)
    tc_peak, tc_src = read_tensor_peak()
    Sp, Lp, B = 4, 2048, 16
    to = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)
    lens = to(np.full(Sp, Lp, dtype=np.int32))
    cu = to(np.arange(Sp + 1, dtype=np.int32) * Lp)
    out = {"mode": "prompt_only", "prompts": Sp, "tokens": Lp, "block_size": B}
    for name, Hq, Hkv, D in (("prompt_prefill", 12, 12, 64), ("prompt_prefill_gqa128", 32, 8, 128)):
        nb = Sp * Lp // B
        gen = torch.Generator(device=device).manual_seed(si.SEED_VALUES)
        k = torch.randn((1, nb, B, Hkv, D), generator=gen, device=device).half()
        v = torch.randn((1, nb, B, Hkv, D), generator=gen, device=device).half()
        pool = pkv.pf_pool_create(k, v)
        bt = to(np.random.default_rng(si.SEED_SHUFFLE).permutation(nb).astype(np.int32).reshape(Sp, Lp // B))
        q = torch.randn((Sp * Lp, Hq, D), generator=gen, device=device).half()
        o = torch.empty_like(q)
        call = lambda: pkv.pf_paged_prefill_attention(pool, 0, q, bt, lens, cu, Lp, 1.0 / np.sqrt(D), o)
        for _ in range(max(args.warmup, 3)):
            call()
        torch.cuda.synchronize(device)
        n = max(1, min(args.steps, 200))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(n):
            call()
        e1.record()
        torch.cuda.synchronize(device)
        ms = e0.elapsed_time(e1) / n
        flops = 4.0 * Hq * D * Sp * Lp * (Lp + 1) / 2
        tf = flops / (ms / 1e3) / 1e12
        out[name] = {"q_heads": Hq, "kv_heads": Hkv, "head_dim": D, "calls": n, "ms": round(ms, 4),
                     "tflops": round(tf, 2), "frac": round(tf / tc_peak, 4), "peak_tflops": tc_peak,
                     "peak_source": tc_src}
        del k, v, pool, q, o
    if pkv.pf_device_status(reset=True) != 0:
        raise RuntimeError("device status flagged during the prompt legs")
    return out


def main(argv=None):
    args = parse_args(argv)
    if args.prompt_only:
        print(json.dumps(run_prompt_only(args)), flush=True)
        return
    if args.record_traffic:
        print(record_traffic(args.record_traffic, args.profile_name, args.profile_command))
        return
    dist = Dist()
    try:
        res = run_reference(args, dist) if args.impl == "reference" else run_ours(args, dist)
        if dist.rank == 0 and res is not None:
            print(json.dumps(res), flush=True)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
