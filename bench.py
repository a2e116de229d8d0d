#!/usr/bin/env python3
"""Benchmark of the FP8 paged decode step at the GLM-4.5 decode shape.

One step = the whole hot path over one batch: append one new BF16 K/V token
per sequence into the FP8 paged cache (quantise-on-append scatter), then
grouped-query paged FP8 decode attention over the updated cache.
Workload: B=16, S1=1, NQ=96, NKV=8, D=128, block_size=128, kv lengths
~U{1..4096} (seeded), s2_tile=512, PA_BSND cache; synthetic N(0,1) data.

Prints one JSON line (rank 0). Metric: achieved HBM GB/s over the step's
algorithmic bytes (valid tokens only), plus us/step. The step is timed on the
device with CUDA events over exactly --steps steps replayed from CUDA graphs;
the steps rotate over enough cache copies that their KV exceeds 3x the L2.

--gpus N: one rank per GPU, each a whole replica of the step (the path has no
exchange step); run as a plain script with N > 1 it starts N local ranks of
itself under torch.distributed.run.

--impl reference times the CPU oracle (the plain C restatement of the
pages) on a bounded sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import socket
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "FP8 paged decode attn: achieved HBM GB/s (% of peak), µs/step at GLM-4.5 shape"
UNIT = "GB/s"
WORKLOAD = ("glm45_decode_step: append 1 BF16 token/seq (quantise-on-append scatter) + FP8 "
            "paged GQA decode; B=16 S1=1 NQ=96 NKV=8 D=128 block_size=128 kv~U[1,4096] "
            "s2_tile=512 PA_BSND")
FALLBACK_HBM_GBS = 6800.0

# Programmatic stream serialisation between the step's kernels. The decode's
# inputs other than the KV cache (lengths, block table, q and its scales,
# v_scale) are never written by the append kernel before it, and the append
# writes only each sequence's newest cache position, so the decode may read
# everything else early (overlap_prologue=2; the newest blocks, key scales and
# its writes wait). The append's inputs (new K/V rows, slots, batches, v_scale)
# are never written by the previous step's decode, so its loads and encoding
# may overlap that decode (its stores wait).
OVERLAP_DECODE = 2
OVERLAP_APPEND = True

# DRAM traffic of one decode launch on this workload, from an ncu capture
# (dram__bytes_read.sum + dram__bytes_write.sum), valid only for the kernel
# sources it was taken with.
DECODE_TRAFFIC = {"sources_sha1": "913e24342602e851b8cd2947e066b3eae93f7761",
                  "bytes_per_launch": 57871104 + 116736}


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["glm45_step", "mla", "configs"], default="glm45_step",
                    help="glm45_step: the GLM-4.5 append + decode step (default); mla: the "
                         "MLA sparse FP8 decode at the DeepSeek-V3.2 page's b=64 case")
    ap.add_argument("--mla-format", choices=["page", "kvc0", "kvc1"], default="page",
                    help="MLA cache rows: the MLA page's packed row, or the KV compress "
                         "epilog's row for d=576 with quant mode 0 (BF16 group scales) or 1 "
                         "(E8M0 group scales)")
    ap.add_argument("--mla-batch", type=int, default=64,
                    help="sequences of the mla workload (64 = the page's case; smaller for "
                         "profiling captures)")
    ap.add_argument("--copies", type=int, default=0, help="cache copies to rotate (0 = auto)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--only", default="",
                    help="--workload configs: comma-separated configuration names to run")
    ap.add_argument("--ref-seconds", type=float, default=150.0,
                    help="--impl reference: wall time of the whole --steps + --warmup run")
    return ap.parse_args(argv)


# --------------------------------------------------------------------------
# ranks: one process per GPU, each a whole replica of the step (the path has no
# exchange step, so there is no data-path collective); the host joins the ranks
# only to start and stop the clock together and to take the slowest rank's time
# --------------------------------------------------------------------------

def dist_env(env=None):
    """(rank, world_size, local_rank) as torchrun exports them; 1 process by default."""
    env = os.environ if env is None else env
    rank = int(env.get("RANK", "0"))
    world = int(env.get("WORLD_SIZE", "1"))
    local = int(env.get("LOCAL_RANK", str(rank)))
    if world < 1 or not 0 <= rank < world or local < 0:
        raise ValueError("bad rank environment: RANK=%d WORLD_SIZE=%d LOCAL_RANK=%d"
                         % (rank, world, local))
    return rank, world, local


def free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def local_ranks_command(argv, nproc, port):
    """The command that runs this script as nproc local ranks (one per GPU)
    with the same arguments: torch.distributed.run on one node, rendezvous on
    127.0.0.1."""
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
            "--nproc-per-node=%d" % nproc, "--master-addr=127.0.0.1", "--master-port=%d" % port,
            os.path.abspath(__file__)] + list(argv)


def check_world(gpus, world):
    """--gpus N under a launcher must match the ranks it started."""
    if gpus != world:
        raise SystemExit("bench.py --gpus %d but the launcher started %d ranks" % (gpus, world))


def init_ranks(world, backend, device=None):
    """Join the process group (NCCL on GPUs; gloo for host-only use)."""
    if world > 1:
        import torch.distributed as dist
        if device is None:
            dist.init_process_group(backend)
        else:
            dist.init_process_group(backend, device_id=device)


def finish_ranks(world):
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device="cpu"):
    """The largest of every rank's x (each rank passes its own; all get the max)."""
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(world, bytes_per_step, steps, ms):
    """Whole-job GB/s: the bytes all ranks processed over the slowest rank's ms."""
    if ms <= 0:
        raise ValueError("non-positive time %r ms" % (ms,))
    return world * bytes_per_step * steps / (ms * 1e-3) / 1e9


def kernel_sources_sha1() -> str:
    h = hashlib.sha1()
    csrc = os.path.join(ROOT, "fp8_paged_kv_block_gb300", "csrc")
    for f in ("decode.cu", "common.cuh"):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def measured_hbm_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def workload():
    return workloads.glm()


def step_bytes(case, act_after):
    """Algorithmic bytes of one step: the decode over the updated lengths plus
    the append (BF16 K/V in, E4M3 codes and key scale out, slot and batch
    ids)."""
    import dataclasses
    dec = dataclasses.replace(case, act=act_after).algorithmic_bytes()
    app = case.B * case.NKV * (2 * case.D * 2 + 2 * case.D + 4) + case.B * 8
    return dec, app


# --------------------------------------------------------------------------
# clocks
# --------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,"
              "utilization.gpu")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) >= 10:
                    rows.append(p)
        os.unlink(self.path)
        busy = [r for r in rows if r[9].isdigit() and int(r[9]) > 0] or rows
        sm = [float(r[1]) for r in busy if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in busy for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows), "samples_busy": len(busy)}


# --------------------------------------------------------------------------
# CPU oracle baseline (also the reference arm)
# --------------------------------------------------------------------------

def oracle_sample(case, inp, budget_s: float, per_row_token_s: float):
    """Rows (whole (batch, kv head) units, in batch order) whose estimated
    oracle time fits ``budget_s``; at least one row."""
    rows, est, nbytes = [], 0.0, 0
    G = case.group
    for b in range(case.B):
        a = int(case.act[b])
        for n2 in range(case.NKV):
            unit_rows = [b * case.NQ + n2 * G + g for g in range(G)]
            t = per_row_token_s * a * G
            if rows and est + t > budget_s:
                return rows, nbytes
            rows.extend(unit_rows)
            est += t
            nbytes += a * (2 * case.D + 4) + G * (case.D + 4) + case.D * 4 + G * case.D * 2
    return rows, nbytes


def run_oracle_rows(case, inp, rows):
    import oracle
    return oracle.pa_decode(inp["q8"], inp["qs"], inp["kc"], inp["ksc"], inp["vc"], inp["vs"],
                            case.block_table, case.act, S1=case.S1, NKV=case.NKV,
                            layout=case.layout, s2_tile=case.s2_tile,
                            softmax_scale=case.softmax_scale, rows=np.asarray(rows))


def host_cpu() -> dict:
    """The host's CPU model (lscpu's model name, else the machine type) and its
    core count, recorded beside every oracle timing."""
    model = ""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.split(":", 1)[0].strip() == "Model name":
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return {"cpu_model": model or platform.machine(), "nproc": os.cpu_count() or 0}


def host_threads() -> int:
    """Cores this process may run on."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except (AttributeError, OSError):
        return max(1, os.cpu_count() or 1)


def deal_units(case, rows, threads):
    """Whole (batch, kv head) units of `rows` dealt round-robin to `threads`
    lists (empty lists dropped)."""
    G = case.group
    units = [rows[i:i + G] for i in range(0, len(rows), G)]
    chunks = [sum(units[k::threads], []) for k in range(threads)]
    return [c for c in chunks if c]


def calibrate_oracle(case, inp):
    """Seconds per (row x token) of the oracle on this host."""
    b = int(np.argmin(np.where(case.act >= 64, case.act, 1 << 30)))
    rows = [b * case.NQ]
    t0 = time.perf_counter()
    run_oracle_rows(case, inp, rows)
    return max((time.perf_counter() - t0) / max(int(case.act[b]), 1), 1e-9)


def cpu_baseline(case, budget_s: float):
    """The oracle on the host's cores: whole (batch, kv head) units dealt
    round-robin to one thread per core (the C oracle keeps no global state and
    ctypes releases the GIL during the call), the sample repeated until about
    budget_s of wall time has passed; the single-threaded rate is reported
    beside it."""
    from concurrent.futures import ThreadPoolExecutor
    from tests import _helpers as H
    inp = H.oracle_inputs(case)
    prt = calibrate_oracle(case, inp)
    rows, nbytes = oracle_sample(case, inp, budget_s / 2, prt)
    t0 = time.perf_counter()
    run_oracle_rows(case, inp, rows)
    dt1 = time.perf_counter() - t0
    threads = host_threads()
    # a sample about `threads` times larger for the threaded run (the whole
    # workload at most, then repeated)
    trows, tbytes = oracle_sample(case, inp, budget_s / 2 * threads, prt)
    chunks = deal_units(case, trows, threads)
    passes, t0 = 0, time.perf_counter()
    with ThreadPoolExecutor(max_workers=len(chunks)) as ex:
        while True:
            list(ex.map(lambda c: run_oracle_rows(case, inp, c), chunks))
            passes += 1
            if time.perf_counter() - t0 >= budget_s / 2:
                break
    dtn = time.perf_counter() - t0
    return {"value": passes * tbytes / dtn / 1e9, "unit": UNIT, "cores": len(chunks),
            "kind": "oracle",
            "sample": "%d of %d query rows (%d whole (batch, kv-head) units), decode only, "
                      "C oracle on %d threads (units dealt round-robin), %d pass(es) in %.1f s; "
                      "single-threaded %.4f GB/s on %d rows (%.1f s)"
                      % (len(trows), case.B * case.NQ, len(trows) // case.group, len(chunks),
                         passes, dtn,
                         nbytes / dt1 / 1e9, len(rows), dt1),
            "single_thread_value": nbytes / dt1 / 1e9, "seconds": dt1 + dtn,
            "sample_bytes": passes * tbytes}


def reference_arm(args, rank, world):
    if rank != 0:
        return
    case = workload()
    from tests import _helpers as H
    inp = H.oracle_inputs(case)
    prt = calibrate_oracle(case, inp)
    from concurrent.futures import ThreadPoolExecutor
    threads = host_threads()
    total_steps = args.steps + args.warmup
    # about --ref-seconds (150 s by default) of wall time over the whole run:
    # whole units in batch order while the busiest thread's estimated time per
    # step stays within that over the steps (at least one unit)
    wall = args.ref_seconds / max(total_steps, 1)
    G = case.group
    load = [0.0] * threads
    rows, nbytes = [], 0
    for b in range(case.B):
        a = int(case.act[b])
        for n2 in range(case.NKV):
            k = (len(rows) // G) % threads
            t = prt * a * G
            if rows and load[k] + t > wall:
                break
            load[k] += t
            rows.extend(b * case.NQ + n2 * G + g for g in range(G))
            nbytes += a * (2 * case.D + 4) + G * (case.D + 4) + case.D * 4 + G * case.D * 2
        else:
            continue
        break
    chunks = deal_units(case, rows, threads)
    with ThreadPoolExecutor(max_workers=len(chunks)) as ex:
        def one_step():
            list(ex.map(lambda c: run_oracle_rows(case, inp, c), chunks))
        for _ in range(args.warmup):
            one_step()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            one_step()
        dt = (time.perf_counter() - t0) / max(args.steps, 1)
    value = nbytes / dt / 1e9
    full = case.algorithmic_bytes()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": full / (value * 1e9) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3+f32",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample_rows": len(rows)},
        "cpu_baseline": {**host_cpu(), "value": value, "unit": UNIT, "cores": len(chunks),
                         "kind": "oracle",
                         "sample": "%d query rows (whole units, dealt round-robin to %d threads) "
                                   "per step, decode only; ms_per_step extrapolated to the full "
                                   "step by bytes" % (len(rows), len(chunks))},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------
# GPU arm
# --------------------------------------------------------------------------

def main(argv=None):
    argv = sys.argv[1:] if argv is None else list(argv)
    args = parse_args(argv)
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        # started without a launcher: start --gpus local ranks of this same
        # command and pass on their exit status (non-zero if any rank failed)
        sys.exit(subprocess.call(local_ranks_command(argv, args.gpus, free_port())))
    rank, world, local = dist_env()
    check_world(args.gpus, world)
    if args.workload == "configs":
        if args.impl == "reference":
            if rank == 0:
                print(json.dumps({"impl": "reference", "unavailable": "the configs sweep has no "
                                  "reference arm; the oracle is timed on the default workload"}))
            return
        configs_arm(args, rank, world, local)
        return
    if args.workload == "mla":
        if args.impl == "reference":
            mla_reference_arm(args, rank, world)
        else:
            mla_arm(args, rank, world, local)
        return
    if args.impl == "reference":
        reference_arm(args, rank, world)
        return

    import torch
    import fp8_paged_kv_block_gb300 as pa
    from fp8_paged_kv_block_gb300 import paged

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_ranks(world, "nccl", dev)
    pa.build()
    pa.lib()

    case = workload()
    knew, vnew, slot, act_after = workloads.step_tokens(case)
    dec_bytes, app_bytes = step_bytes(case, act_after)
    bytes_per_step = dec_bytes + app_bytes

    # ---- device inputs: queries, context cache, append inputs ----
    q8, qs = paged.quantize_queries(torch.from_numpy(case.q()).to(dev))
    k32, v32 = case.kv()
    base = paged.build_cache(torch.from_numpy(k32).to(dev), torch.from_numpy(v32).to(dev),
                             torch.from_numpy(case.cu_seqlens).to(dev),
                             torch.from_numpy(case.slots).to(dev),
                             torch.from_numpy(case.token_batch).to(dev), case.num_blocks,
                             case.layout)
    del k32, v32
    case.drop()
    cache_bytes = 2 * base.k_cache.numel() + 4 * base.k_scale.numel()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    copies = args.copies or max(3, math.ceil(3 * l2 / cache_bytes))
    caches = [base] + [paged.PagedFP8(base.k_cache.clone(), base.v_cache.clone(),
                                      base.k_scale.clone(), base.v_scale.clone(), base.layout)
                       for _ in range(copies - 1)]
    bt = torch.from_numpy(case.block_table).to(dev)
    act_d = torch.from_numpy(act_after).to(dev)
    slot_d = torch.from_numpy(slot).to(dev)
    tb_d = torch.arange(case.B, dtype=torch.int32, device=dev)
    kn_d, vn_d = knew.to(dev), vnew.to(dev)
    out = torch.empty((case.B * case.S1, case.NQ, case.D), dtype=torch.bfloat16, device=dev)
    ws = pa.DecodeWorkspace(case.B, case.S1, case.NQ, case.NKV, s2_tile=case.s2_tile, device=dev)

    def append(c):
        pa.cache_quant_scatter(kn_d, vn_d, c.k_cache, c.v_cache, slot_d, c.k_scale, c.v_scale,
                               tb_d, layout=case.layout, overlap_prologue=OVERLAP_APPEND)

    def attend(c, overlap=OVERLAP_DECODE):
        pa.decode(q8, qs, c.k_cache, c.k_scale, c.v_cache, c.v_scale, bt, act_d, out,
                  S1=case.S1, layout=case.layout, s2_tile=case.s2_tile,
                  softmax_scale=case.softmax_scale, workspace=ws, overlap_prologue=overlap)

    def step(i):
        c = caches[i % copies]
        append(c)
        attend(c)

    def capture(fn, n):
        s = torch.cuda.Stream(device=dev)
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            for i in range(min(n, copies)):
                fn(i)
        torch.cuda.current_stream().wait_stream(s)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(n):
                fn(i)
        return g

    cyc = copies * max(1, math.ceil(32 / copies))           # steps per replay
    g_step = capture(step, cyc)
    g_dec = capture(lambda i: attend(caches[i % copies]), cyc)
    # A run of n steps replays the cyc-step graph n // cyc times and one graph
    # of the remaining n % cyc steps (captured beforehand), so that every
    # kernel but the first of a replay overlaps its predecessor whatever n is.
    def with_tail(fn, full_graph, counts):
        tails = {n % cyc: capture(fn, n % cyc) for n in counts if n % cyc}
        return (full_graph, tails)

    counts = (max(args.warmup, 3), args.steps, cyc * 8)
    g_step = with_tail(step, g_step, counts)
    g_dec = with_tail(lambda i: attend(caches[i % copies]), g_dec, counts)
    # the same decode launches in plain stream order (no overlap of one launch
    # with the next), for reference
    g_dec0 = with_tail(lambda i: attend(caches[i % copies], 0),
                       capture(lambda i: attend(caches[i % copies], 0), cyc), counts)

    def run_steps(graphs, n):
        full_graph, tails = graphs
        for _ in range(n // cyc):
            full_graph.replay()
        if n % cyc:
            tails[n % cyc].replay()

    def timed(graphs, n):
        barrier(world)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        # keep the GPU busy (~0.1 ms spin) while the host submits the first
        # graph, so that the timed region holds device work only
        torch.cuda._sleep(200000)
        e0.record()
        run_steps(graphs, n)
        e1.record()
        torch.cuda.synchronize()
        barrier(world)
        return max_over_ranks(e0.elapsed_time(e1), world, dev)

    clocks = ClockSampler(local)
    # warm-up (untimed)
    run_steps(g_step, max(args.warmup, 3))
    run_steps(g_dec, max(args.warmup, 3))
    run_steps(g_dec0, max(args.warmup, 3))
    torch.cuda.synchronize()
    assert ws.error_flags() == 0, "decode kernel reported a wait timeout"

    def replay_dist(graphs, nrep):
        """Percentiles of us per step over nrep replays of the cyc-step graph,
        an event after each replay (this rank's)."""
        full_graph, _ = graphs
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(nrep + 1)]
        torch.cuda.synchronize()
        torch.cuda._sleep(200000)
        ev[0].record()
        for k in range(nrep):
            full_graph.replay()
            ev[k + 1].record()
        torch.cuda.synchronize()
        return percentiles([ev[k].elapsed_time(ev[k + 1]) * 1e3 / cyc for k in range(nrep)])

    clocks.start()
    t_start = time.perf_counter()
    ms_total = timed(g_step, args.steps)
    ms_dec = timed(g_dec, args.steps)
    ms_dec0 = timed(g_dec0, args.steps)
    nrep = max(10, args.steps // cyc)
    dist_step = replay_dist(g_step, nrep)
    dist_dec = replay_dist(g_dec, nrep)
    # keep the same work running until the clock sampler has seen ~1 s of it
    while time.perf_counter() - t_start < 1.0:
        run_steps(g_step, cyc * 8)
        torch.cuda.synchronize()

    # ---- end to end through the public API with host buffers ----
    # The step's inputs travel in one pinned host buffer (one host-to-device
    # copy per step); the output comes back with one device-to-host copy.
    # As a serving loop runs it: two device input buffers and two output
    # buffers alternate, the input copy of step i (its own stream) overlaps
    # the kernels of step i-1 and the output copy of step i (another stream)
    # those of step i+1; every step still copies its own inputs in and its
    # output back, and the timed region ends after the last output copy.
    host_parts = [q8.cpu(), qs.cpu(), knew, vnew, torch.from_numpy(slot), torch.from_numpy(act_after),
                  torch.from_numpy(case.block_table)]
    offs, total = [], 0
    for t in host_parts:
        offs.append(total)
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    h_pack = torch.empty(total, dtype=torch.uint8).pin_memory()
    for t, o in zip(host_parts, offs):
        n = t.numel() * t.element_size()
        h_pack[o:o + n].copy_(t.contiguous().view(-1).view(torch.uint8))
    NBUF = 2
    d_packs = [torch.empty(total, dtype=torch.uint8, device=dev) for _ in range(NBUF)]
    d_views = [[dp[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
                for t, o in zip(host_parts, offs)] for dp in d_packs]
    outs = [torch.empty_like(out) for _ in range(NBUF)]
    h_outs = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(NBUF)]
    h2d = total
    d2h = h_outs[0].numel() * h_outs[0].element_size()
    s_in = torch.cuda.Stream(device=dev)
    s_out = torch.cuda.Stream(device=dev)
    plans = {}   # (buffer, cache copy) -> the step's two library calls, prepared once

    def step_calls(k, c):
        if (k, c) not in plans:
            d_q8, d_qs, d_kn, d_vn, d_slot, d_act, d_bt = d_views[k]
            cc = caches[c]
            plans[(k, c)] = (
                pa.prepare_cache_quant_scatter(d_kn, d_vn, cc.k_cache, cc.v_cache, d_slot,
                                               cc.k_scale, cc.v_scale, tb_d, layout=case.layout,
                                               overlap_prologue=OVERLAP_APPEND),
                pa.prepare_decode(d_q8, d_qs, cc.k_cache, cc.k_scale, cc.v_cache, cc.v_scale,
                                  d_bt, d_act, outs[k], S1=case.S1, layout=case.layout,
                                  s2_tile=case.s2_tile, softmax_scale=case.softmax_scale,
                                  workspace=ws, overlap_prologue=OVERLAP_DECODE))
        return plans[(k, c)]

    def e2e_steps(i0, n):
        main = torch.cuda.current_stream()
        ev_in = [torch.cuda.Event() for _ in range(NBUF)]    # inputs of buffer k landed
        ev_used = [torch.cuda.Event() for _ in range(NBUF)]  # kernels done with buffer k
        ev_out = [torch.cuda.Event() for _ in range(NBUF)]   # output k copied to the host
        for k in range(NBUF):
            ev_used[k].record(main)
            ev_out[k].record(main)
        for i in range(i0, i0 + n):
            k = i % NBUF
            append, attend = step_calls(k, i % copies)
            # the append follows its input copy on the input stream: it writes
            # only each sequence's newest position, which the previous step's
            # decode does not read, so it may run beside that decode
            s_in.wait_event(ev_used[k])
            with torch.cuda.stream(s_in):
                d_packs[k].copy_(h_pack, non_blocking=True)
            append(s_in)
            ev_in[k].record(s_in)
            main.wait_event(ev_in[k])
            main.wait_event(ev_out[k])
            attend(main)
            ev_used[k].record(main)
            s_out.wait_event(ev_used[k])
            with torch.cuda.stream(s_out):
                h_outs[k].copy_(outs[k], non_blocking=True)
            ev_out[k].record(s_out)
        main.wait_stream(s_in)
        main.wait_stream(s_out)

    def e2e_graph(n):
        s = torch.cuda.Stream(device=dev)
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            e2e_steps(0, min(n, NBUF * copies))
        torch.cuda.current_stream().wait_stream(s)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            e2e_steps(0, n)
        return g

    # eager calls (one Python round trip per API call) ...
    e2e_steps(0, 3)
    torch.cuda.synchronize()
    n_e2e = args.steps
    barrier(world)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    e2e_steps(0, n_e2e)
    e1.record()
    torch.cuda.synchronize()
    ms_e2e_eager = e0.elapsed_time(e1)
    # ... and the same calls captured once in a CUDA graph (how a serving loop
    # issues its decode steps): every replayed step still copies its inputs in
    # from pinned host memory and its output back
    g_e2e = (e2e_graph(cyc), {n % cyc: e2e_graph(n % cyc) for n in counts if n % cyc})
    run_steps(g_e2e, max(args.warmup, 3))
    ms_e2e = timed(g_e2e, n_e2e)
    clk = clocks.stop()
    assert ws.error_flags() == 0, "decode kernel reported a wait timeout"
    ms_e2e_eager = max_over_ranks(ms_e2e_eager, world, dev)

    ms_step = ms_total / args.steps
    ms_dec_launch = ms_dec / args.steps
    value = whole_job_gbs(world, bytes_per_step, args.steps, ms_total)
    peak, peak_src = measured_hbm_peak()
    achieved = dec_bytes / (ms_dec_launch * 1e-3) / 1e9
    sha = kernel_sources_sha1()
    traffic = (DECODE_TRAFFIC["bytes_per_launch"]
               if DECODE_TRAFFIC["sources_sha1"] == sha else None)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(workload(), args.cpu_seconds)
        cpu = {k: cpu[k] for k in ("value", "unit", "cores", "kind", "sample")}
        cpu.update(host_cpu())

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "us_per_step": ms_step * 1e3, "us_per_step_dist": dist_step,
            "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "e4m3+f32", "data": "synthetic",
            "config": {
                "workload": WORKLOAD,
                "B": case.B, "kv_tokens": int(act_after.sum()), "bytes_per_step": bytes_per_step,
                "decode_bytes": dec_bytes, "append_bytes": app_bytes,
                "l2": "inputs larger than L2: %d cache copies rotated (%.0f MB > %.0f MB L2)"
                      % (copies, copies * cache_bytes / 1e6, l2 / 1e6),
                "timing": "CUDA graphs replayed on one stream, CUDA events over the K steps; "
                          "*_dist: percentiles over replays of a %d-step graph, an event after "
                          "each replay (rank 0)" % cyc,
                "parallelism": "replicas" if world > 1 else "single GPU",
                "launch": "programmatic dependent launch: the append's loads and encoding "
                          "overlap the previous decode (its stores wait for it); the decode's "
                          "prologue and its loads of cache blocks below each sequence's newest "
                          "position overlap the append (overlap_prologue=%d; the newest blocks, "
                          "key scales and all writes wait)" % OVERLAP_DECODE,
            },
            "gpu_launches": 2 * args.steps,
            "roofline": {"bound": "hbm", "kernel": "pa_fp8_decode", "achieved": achieved,
                         "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                         "traffic": traffic, "peak_source": peak_src,
                         "frac_of_8tbs_nominal": achieved / 8000.0,
                         "us_per_launch": ms_dec_launch * 1e3,
                         "us_per_launch_stream_order": ms_dec0 / args.steps * 1e3,
                         "us_per_launch_dist": dist_dec,
                         "algorithmic_bytes_per_launch": dec_bytes},
            "e2e": {"value": whole_job_gbs(world, bytes_per_step, n_e2e, ms_e2e), "unit": UNIT,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "us_per_step": ms_e2e / n_e2e * 1e3,
                    "issue": "the public-API calls of each step (pinned H2D copy of its "
                             "inputs, append, decode, D2H copy of its output; the two library "
                             "calls prepared once per buffer set) captured in a CUDA graph; two "
                             "input and two output buffers alternate; the copy and the append "
                             "run on an input stream beside the previous step's decode (the "
                             "append writes only the newest positions, which that decode does "
                             "not read), the output copy on an output stream, all ordered by "
                             "events",
                    "eager_us_per_step": ms_e2e_eager / n_e2e * 1e3},
            "clocks": clk,
            "cpu_baseline": cpu,
            "tokens_per_s": world * case.B * case.S1 * args.steps / (ms_total * 1e-3),
        }
        print(json.dumps(line), flush=True)
    finish_ranks(world)


# --------------------------------------------------------------------------
# Every decode configuration (--workload configs): one JSON line each
# --------------------------------------------------------------------------

def _page_config(i):
    b, s1, s2, nq, nkv = workloads.PAGE_CASES[i]
    return ("page%d" % i, lambda: workloads.page_case(i, s2_tile=0),
            "b=%d s1=%d s2=%d nq=%d nkv=%d, every sequence at its full s2 (a case of the GLM-4.5 "
            "paged FP8 page's test table) PA_BSND" % (b, s1, s2, nq, nkv))


CONFIGS = [  # (name, workload with s2_tile 0 = the library's automatic tile, description)
    ("tiny", lambda: workloads.tiny(s2_tile=0), "B=2 S1=1 NQ=4 NKV=1 kv {37,300} PA_BSND"),
    ("glm45", lambda: workloads.glm(s2_tile=0), "B=16 S1=1 NQ=96 NKV=8 kv~U[1,4096] PA_BSND"),
    ("long", lambda: workloads.long_ctx(s2_tile=0),
     "B=4 S1=1 NQ=96 NKV=8 kv~U[32768,131072], every 64th K row x8 before quantisation, PA_BSND"),
    ("ragged", lambda: workloads.ragged(s2_tile=0),
     "B=256 S1=2 NQ=96 NKV=8 kv~lognormal(median 1024, sigma 1) clipped to [1,16384] PA_BSND"),
    ("append", lambda: workloads.append(s2_tile=0),
     "64 new BF16 K/V rows (5% of slots -1) into contexts U[512,8192], NQ=96 NKV=8 BNBD, then "
     "decode over the updated cache"),
] + [_page_config(i) for i in range(len(workloads.PAGE_CASES))]


def percentiles(samples):
    """Median, 10th and 90th percentile of per-step samples."""
    a = np.asarray(samples, dtype=np.float64)
    return {"median": float(np.median(a)), "p10": float(np.percentile(a, 10)),
            "p90": float(np.percentile(a, 90)), "samples": int(a.size)}


def unit_rows(case, b, n2):
    """Flat output rows (b*S1 + s)*NQ + h of the (batch b, kv head n2) unit."""
    G = case.group
    return [(b * case.S1 + s) * case.NQ + n2 * G + g for s in range(case.S1) for g in range(G)]


def parity_units(case, act, budget_s, per_row_token_s, seed=0):
    """Whole (batch, kv head) units in a seeded random order while the
    oracle's estimated time stays within budget_s (at least one unit)."""
    units = [(b, n2) for b in range(case.B) for n2 in range(case.NKV)]
    order = np.random.default_rng(seed).permutation(len(units))
    pick, est = [], 0.0
    for k in order:
        b, n2 = units[int(k)]
        t = per_row_token_s * max(int(act[b]), 1) * case.S1 * case.group
        if pick and est + t > budget_s:
            break
        pick.append((b, n2))
        est += t
    return pick


class ConfigOracleLeg:
    """cpu_baseline leg of one configuration: the oracle's inputs for a
    sample of whole units (prepared while the case's K/V are in memory), then
    the oracle on those rows, timed on one host thread, and its outputs
    against the GPU's for the same rows (max / mean absolute error)."""

    def __init__(self, case, app, act_after, budget_s):
        from tests import _helpers as H
        self.case, self.app, self.act = case, app, act_after
        probe = H.oracle_inputs(case, batches=[int(np.argmin(case.act))])
        b = int(np.argmin(case.act))
        t0 = time.perf_counter()
        H.oracle_decode(case, probe, rows=np.asarray(unit_rows(case, b, 0)[:1]))
        prt = max((time.perf_counter() - t0) / max(int(case.act[b]), 1), 1e-9)
        del probe
        self.units = parity_units(case, act_after, budget_s, prt)
        batches = sorted({b for b, _ in self.units})
        self.inp = H.oracle_inputs(case, batches=batches)
        if app is not None:
            import oracle
            kn, vn = app.new_kv_f32()
            sel = np.asarray(batches)
            oracle.cache_quant_scatter(kn[sel], vn[sel], self.inp["kc"], self.inp["vc"],
                                       app.slot_mapping[sel].astype(np.int64), self.inp["ksc"],
                                       self.inp["vs"], sel.astype(np.int32), layout=case.layout)
        self.rows = np.asarray(sorted(r for b, n2 in self.units for r in unit_rows(case, b, n2)))

    def run(self, gpu_out_u16):
        from tests import _helpers as H
        import oracle
        dcase = dataclasses.replace(self.case, act=self.act)
        t0 = time.perf_counter()
        ref = H.oracle_decode(dcase, self.inp, rows=self.rows)
        dt = time.perf_counter() - t0
        g = oracle.bf16_to_float(gpu_out_u16).reshape(-1, self.case.D)[self.rows].astype(np.float64)
        r = oracle.bf16_to_float(ref).reshape(-1, self.case.D)[self.rows].astype(np.float64)
        err = np.abs(g - r)
        nbytes = sum(int(self.act[b]) * (2 * self.case.D + 4) + self.case.S1 * self.case.group
                     * (self.case.D * 3 + 4) + self.case.D * 4 for b, _ in self.units)
        cpu = {**host_cpu(), "value": nbytes / dt / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": "%d whole (batch, kv head) units = %d query rows, seeded random, "
                         "decode only, one thread, %.2f s" % (len(self.units), self.rows.size, dt)}
        acc = {"max_abs": float(err.max()), "mean_abs": float(err.mean()),
               "finite": bool(np.all(np.isfinite(g))), "rows": int(self.rows.size),
               "tol_max_abs": H.MAX_ABS_TOL, "tol_mean_abs": H.MEAN_ABS_TOL}
        acc["within_tol"] = bool(acc["finite"] and acc["max_abs"] <= H.MAX_ABS_TOL
                                 and acc["mean_abs"] <= H.MEAN_ABS_TOL)
        return cpu, acc


def configs_arm(args, rank, world, local):
    """Decode time per launch for each configuration at the library's
    automatic s2_tile (and the other built tiles beside it), inputs built on
    the device with the library's own kernels (as the parity tests build
    them); append + decode step for the append configuration; per-replay
    percentiles; the oracle on a sample of each configuration's rows (the
    cpu_baseline leg) with the error of the GPU's output on those rows."""
    import torch
    import fp8_paged_kv_block_gb300 as pa
    from fp8_paged_kv_block_gb300 import paged

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_ranks(world, "nccl", dev)
    pa.build()
    pa.lib()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    peak, peak_src = measured_hbm_peak()

    def timed(fn, n, reps):
        """(ms per call of fn(i), per-replay percentiles in us per call): a
        graph of reps calls replayed n // reps times, an event after each."""
        s = torch.cuda.Stream(device=dev)
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            for i in range(reps):
                fn(i)
        torch.cuda.current_stream().wait_stream(s)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(reps):
                fn(i)
        for _ in range(max(args.warmup, 3)):
            g.replay()
        nrep = max(3, n // reps)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(nrep + 1)]
        barrier(world)
        torch.cuda.synchronize()
        torch.cuda._sleep(200000)
        ev[0].record()
        for k in range(nrep):
            g.replay()
            ev[k + 1].record()
        torch.cuda.synchronize()
        barrier(world)
        ms = max_over_ranks(ev[0].elapsed_time(ev[-1]), world, dev) / (nrep * reps)
        dist = percentiles([ev[k].elapsed_time(ev[k + 1]) * 1e3 / reps for k in range(nrep)])
        if ws.error_flags():
            raise SystemExit("decode kernel reported a wait timeout (config %s)" % name)
        if rank == 0:
            print("  %s: %d x %d launches, %.2f us each" % (name, nrep, reps, ms * 1e3),
                  file=sys.stderr, flush=True)
        return ms, dist

    clocks = ClockSampler(local)
    clocks.start()
    lines = []
    for name, make, desc in CONFIGS:
        if args.only and name not in args.only.split(","):
            continue
        t_cfg = time.perf_counter()
        made = make()
        app = made if name == "append" else None
        case = app.ctx if app is not None else made
        act_after = app.act_after if app is not None else case.act
        tile = case.s2_tile or pa.auto_s2_tile(case.S1, case.NQ, case.NKV,
                                               case.max_blocks * case.BS)
        case = dataclasses.replace(case, s2_tile=tile)
        if app is not None:
            app = dataclasses.replace(app, ctx=case)
        dcase = dataclasses.replace(case, act=act_after)
        dec_bytes = dcase.algorithmic_bytes()
        q8, qs = paged.quantize_queries(torch.from_numpy(case.q()).to(dev))
        k32, v32 = case.kv()
        base = paged.build_cache(torch.from_numpy(k32).to(dev), torch.from_numpy(v32).to(dev),
                                 torch.from_numpy(case.cu_seqlens).to(dev),
                                 torch.from_numpy(case.slots).to(dev),
                                 torch.from_numpy(case.token_batch).to(dev), case.num_blocks,
                                 case.layout)
        del k32, v32
        leg = (ConfigOracleLeg(case, app, act_after, args.cpu_seconds / len(CONFIGS))
               if rank == 0 and not args.no_cpu_baseline else None)
        case.drop()
        cache_bytes = 2 * base.k_cache.numel() + 4 * base.k_scale.numel()
        copies = max(1, math.ceil(3 * l2 / cache_bytes))
        caches = [base] + [paged.PagedFP8(base.k_cache.clone(), base.v_cache.clone(),
                                          base.k_scale.clone(), base.v_scale.clone(), base.layout)
                           for _ in range(copies - 1)]
        bt = torch.from_numpy(case.block_table).to(dev)
        act_d = torch.from_numpy(act_after).to(dev)
        out = torch.empty((case.B * case.S1, case.NQ, case.D), dtype=torch.bfloat16, device=dev)
        ws = pa.DecodeWorkspace(case.B, case.S1, case.NQ, case.NKV, device=dev)

        def attend(i, overlap=OVERLAP_DECODE, s2_tile=tile):
            c = caches[i % copies]
            pa.decode(q8, qs, c.k_cache, c.k_scale, c.v_cache, c.v_scale, bt, act_d, out,
                      S1=case.S1, layout=case.layout, s2_tile=s2_tile,
                      softmax_scale=case.softmax_scale, workspace=ws, overlap_prologue=overlap)

        est_us = max(5.0, dec_bytes / (peak * 1e3) * 2.0)
        n = max(50, min(args.steps, int(100000 / est_us)))
        reps = copies * max(1, math.ceil(16 / copies))
        extra = {}
        if app is not None:
            kb, vb = app.new_kv_bf16()
            kn_d, vn_d = kb.to(dev), vb.to(dev)
            slot_d = torch.from_numpy(app.slot_mapping).to(dev)
            tb_d = torch.from_numpy(app.token_batch).to(dev)
            app_bytes = (app.T * case.NKV * (2 * case.D * 2 + 2 * case.D + 4) + app.T * 8)

            def append(i):
                c = caches[i % copies]
                pa.cache_quant_scatter(kn_d, vn_d, c.k_cache, c.v_cache, slot_d, c.k_scale,
                                       c.v_scale, tb_d, layout=case.layout,
                                       overlap_prologue=OVERLAP_APPEND)

            def step(i):
                append(i)
                attend(i)

            # the append first: every cache copy then holds the new token
            ms_app, dist_app = timed(append, n, reps)
            ms_step, dist_step = timed(step, n, reps)
            extra = {"append_us_per_launch": ms_app * 1e3, "append_us_dist": dist_app,
                     "append_bytes": app_bytes, "step_us": ms_step * 1e3,
                     "step_us_dist": dist_step,
                     "step_gbs": world * (dec_bytes + app_bytes) / (ms_step * 1e-3) / 1e9}
        ms_dec, dist_dec = timed(attend, n, reps)
        torch.cuda.synchronize()
        out_sel = host_u16(out)
        ms_dec0, _ = timed(lambda i: attend(i, 0), n, reps)
        alt = {}
        # (32-row units: 512 only; the 256-token tile is not run at this scale,
        # its launch on the ragged batch hung once and the cause is not found)
        for t in ((256, 512, 1024) if case.S1 * case.group <= 16 else (512,)):
            if t != tile:
                alt[str(t)] = timed(lambda i, t=t: attend(i, s2_tile=t), n, reps)[0] * 1e3
        alt[str(tile)] = ms_dec * 1e3
        assert ws.error_flags() == 0, "decode kernel reported a wait timeout"
        cpu, acc = leg.run(out_sel) if leg is not None else (None, None)
        gbs = dec_bytes / (ms_dec * 1e-3) / 1e9
        lines.append({
            "metric": METRIC, "value": world * gbs, "unit": UNIT, "n_gpus": world,
            "steps": n, "warmup": args.warmup, "ms_per_step": ms_dec,
            "us_per_step": ms_dec * 1e3, "us_per_step_dist": dist_dec,
            "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "e4m3+f32", "data": "synthetic",
            "config": {"workload": name + ": " + desc, "B": case.B, "S1": case.S1,
                       "NQ": case.NQ, "NKV": case.NKV, "s2_tile": tile,
                       "s2_tile_rule": "automatic (s2 = block table capacity %d)"
                                       % (case.max_blocks * case.BS),
                       "kv_tokens": int(act_after.sum()), "decode_bytes": dec_bytes,
                       "l2": ("inputs larger than L2: %d cache copies rotated (%.0f MB, L2 %.0f MB)"
                              % (copies, copies * cache_bytes / 1e6, l2 / 1e6)),
                       "timing": "CUDA graph of %d back-to-back decode launches "
                                 "(overlap_prologue=%d%s) replayed, CUDA events around each "
                                 "replay; dist = per-replay us per launch (rank 0)"
                                 % (reps, OVERLAP_DECODE,
                                    "" if case.S1 * case.group <= 16 else
                                    ", which the library runs in stream order at 32 rows")},
            "gpu_launches": n,
            "roofline": {"bound": "hbm", "kernel": "pa_fp8_decode", "achieved": gbs, "peak": peak,
                         "unit": "GB/s", "frac": gbs / peak, "traffic": None,
                         "peak_source": peak_src, "frac_of_8tbs_nominal": gbs / 8000.0,
                         "us_per_launch": ms_dec * 1e3,
                         "us_per_launch_stream_order": ms_dec0 * 1e3,
                         "us_per_launch_by_s2_tile": alt},
            "accuracy": acc,
            "cpu_baseline": cpu,
            "tokens_per_s": world * case.B * case.S1 / (ms_dec * 1e-3),
            **extra,
        })
        del caches, base, out, ws, leg
        torch.cuda.empty_cache()
        if rank == 0:
            print("config %s done in %.1f s" % (name, time.perf_counter() - t_cfg), file=sys.stderr,
                  flush=True)
    clk = clocks.stop()
    if rank == 0:
        for line in lines:
            line["clocks"] = clk
            print(json.dumps(line), flush=True)
    finish_ranks(world)


def host_u16(t):
    """A BF16 device tensor's bits as a host uint16 array."""
    import torch
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


# --------------------------------------------------------------------------
# MLA sparse FP8 decode (DeepSeek-V3.2 shape)
# --------------------------------------------------------------------------

MLA_METRIC = ("MLA sparse FP8 decode: achieved BF16 tensor TFLOP/s (% of peak), µs/step at the "
              "DeepSeek-V3.2 b=64 decode shape")
MLA_UNIT = "TFLOP/s"
MLA_WORKLOAD = ("%s: b=%d s_q=2 nq=128 n_kv=1 topk=2048 kv_lora_rank=512 "
                "qk_rope_dim=64 block_size=128 kv_act_seqs=65536 (all); 672-byte %s; s2_tile=128")
MLA_FORMATS = {  # --mla-format: (row format, KV compress quant mode, entry point, rows)
    "page": (workloads.MLA_FORMAT_PAGE, None, "mla_sparse_decode",
             "packed rows (E4M3 nope, BF16 rope, 4 FP32 group scales)"),
    "kvc0": (workloads.MLA_FORMAT_KVC_BF16, 0, "mla_sparse_decode_kvc",
             "KV compress epilog rows, quant mode 0 (BF16 rope, E4M3 nope, 8 BF16 group scales)"),
    "kvc1": (workloads.MLA_FORMAT_KVC_E8M0, 1, "mla_sparse_decode_kvc",
             "KV compress epilog rows, quant mode 1 (BF16 rope, E4M3 nope, 8 E8M0 group scales)"),
}


def mla_workload_name(args, B):
    _, _, entry, rows = MLA_FORMATS[args.mla_format]
    return MLA_WORKLOAD % (entry, B, rows)
MLA_VARIANTS = 2          # top-k selections rotated between steps (each ~172 MB of rows)
# DRAM traffic of one MLA decode launch on this workload from an ncu capture,
# valid only for the kernel source it was taken with.
# Captured on the 16-sequence case and scaled by the selected rows (x4): each
# row is read from DRAM once, so the traffic grows in proportion.
MLA_TRAFFIC = {"sources_sha1": "0d68231f9ece537b28bc832b8f9d4feb72772394", "format": "page",
               "bytes_per_launch": 4 * (54289152 + 336640)}


def mla_sources_sha1() -> str:
    with open(os.path.join(ROOT, "fp8_paged_kv_block_gb300", "csrc", "mla.cu"), "rb") as fh:
        return hashlib.sha1(fh.read()).hexdigest()


def measured_bf16_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), "measured (MEASURED_PEAKS.json bf16_tflops, burst)"
    except Exception:
        return 1900.0, "fallback"


def mla_host_cache(case, used, rb):
    """The full packed cache on the host with only the used rows drawn (the
    rest is never read and is never touched, so it costs no memory)."""
    host = np.zeros((case.num_blocks * case.BS, workloads.MLA_ROW_BYTES), dtype=np.uint8)
    host[used] = rb
    return host


def mla_oracle_sample(case, host, budget_s, row_format=workloads.MLA_FORMAT_PAGE, threads=1):
    """Time the oracle on whole query tokens (all heads), `threads` tokens at a
    time on as many threads (the C oracle keeps no global state and ctypes
    releases the GIL during the call), until about budget_s of wall time:
    (TFLOP/s, tokens, seconds, flops)."""
    from concurrent.futures import ThreadPoolExecutor
    import oracle
    qn, qr = case.q_bits()
    tk = case.topk_indices(0)
    cur = case.cur()
    NQ = case.NQ

    def one(t):
        rows = np.arange(int(t) * NQ, (int(t) + 1) * NQ, dtype=np.int64)
        oracle.mla_sparse_decode(qn, qr, host, tk, case.block_table, case.act, S1=case.S1,
                                 block_size=case.BS, s2_tile=case.s2_tile,
                                 softmax_scale=case.softmax_scale, rows=rows,
                                 row_format=row_format)
        b = int(t) // case.S1
        sel = tk[int(t), :int(cur[t])]
        nvalid = int(((sel >= 0) & (sel < case.act[b])).sum())
        return nvalid * 2 * NQ * (512 + 64 + 512)

    done, flops = 0, 0
    toks = np.random.default_rng(5).permutation(case.T)
    t0 = time.perf_counter()
    with ThreadPoolExecutor(max_workers=threads) as ex:
        for i in range(0, len(toks), threads):
            batch = toks[i:i + threads]
            flops += sum(ex.map(one, batch))
            done += len(batch)
            if time.perf_counter() - t0 >= budget_s:
                break
    dt = time.perf_counter() - t0
    return flops / dt / 1e12, done, dt, flops


def mla_reference_arm(args, rank, world):
    if rank != 0:
        return
    case = workloads.mla_page_b64(args.mla_batch)
    fmt = MLA_FORMATS[args.mla_format][0]
    used = case.rows_used((0,))
    host = mla_host_cache(case, used, case.row_bytes(used, fmt))
    total_steps = args.steps + args.warmup
    budget = max(args.cpu_seconds / max(total_steps, 1), 0.5)
    threads = host_threads()
    for _ in range(args.warmup):
        mla_oracle_sample(case, host, budget, fmt, threads)
    vals = []
    tok = 0
    for _ in range(args.steps):
        v, tok, _, _ = mla_oracle_sample(case, host, budget, fmt, threads)
        vals.append(v)
    value = statistics.median(vals) if vals else 0.0
    line = {
        "impl": "reference", "metric": MLA_METRIC, "value": value, "unit": MLA_UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": case.flops() / (value * 1e12) * 1e3 if value else None,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16+e4m3",
        "data": "synthetic", "config": {"workload": mla_workload_name(args, case.B),
                                        "sample_tokens": tok},
        "cpu_baseline": {**host_cpu(), "value": value, "unit": MLA_UNIT, "cores": threads,
                         "kind": "oracle",
                         "sample": "%d query tokens (all 128 heads) per step, %d at a time on "
                                   "%d threads; ms_per_step extrapolated to the 128-token decode "
                                   "by flops" % (tok, threads, threads)},
        "e2e": {"value": value, "unit": MLA_UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def mla_arm(args, rank, world, local):
    import torch
    import fp8_paged_kv_block_gb300 as pa

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_ranks(world, "nccl", dev)
    pa.build()
    pa.lib()

    case = workloads.mla_page_b64(args.mla_batch)
    fmt, quant_mode, entry, _ = MLA_FORMATS[args.mla_format]
    V = MLA_VARIANTS
    used = case.rows_used(range(V))
    rb = case.row_bytes(used, fmt)
    nrows = case.num_blocks * case.BS
    cache = torch.zeros((nrows, workloads.MLA_ROW_BYTES), dtype=torch.uint8, device=dev)
    cache[torch.from_numpy(used).to(dev)] = torch.from_numpy(rb).to(dev)
    qn_h, qr_h = case.q_bf16()
    qn, qr = qn_h.to(dev), qr_h.to(dev)
    tks = [torch.from_numpy(case.topk_indices(v)).to(dev) for v in range(V)]
    bt = torch.from_numpy(case.block_table).to(dev)
    act = torch.from_numpy(case.act).to(dev)
    out = torch.empty((case.T, case.NQ, 512), dtype=torch.bfloat16, device=dev)
    status = pa.MlaStatus(dev)
    flops_v = [case.flops(v) for v in range(V)]
    bytes_v = [case.algorithmic_bytes(v) for v in range(V)]

    def launch(i, q=(qn, qr), tk=None, o=out):
        if quant_mode is None:
            pa.mla_sparse_decode(q[0], q[1], cache, tks[i % V] if tk is None else tk, bt, act, o,
                                 S1=case.S1, status=status, block_size=case.BS,
                                 softmax_scale=case.softmax_scale)
        else:
            pa.mla_sparse_decode_kvc(q[0], q[1], cache, tks[i % V] if tk is None else tk, bt,
                                     act, o, quant_mode=quant_mode, S1=case.S1, status=status,
                                     block_size=case.BS, softmax_scale=case.softmax_scale)

    cyc = V * 6

    def capture(fn, n):
        s = torch.cuda.Stream(device=dev)
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            for i in range(min(n, V)):
                fn(i)
        torch.cuda.current_stream().wait_stream(s)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(n):
                fn(i)
        return g

    counts = (max(args.warmup, 3), args.steps)
    graphs = (capture(launch, cyc), {n % cyc: capture(launch, n % cyc) for n in counts if n % cyc})

    def run_steps(gr, n):
        full, tails = gr
        for _ in range(n // cyc):
            full.replay()
        if n % cyc:
            tails[n % cyc].replay()

    def timed(gr, n):
        barrier(world)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(200000)
        e0.record()
        run_steps(gr, n)
        e1.record()
        torch.cuda.synchronize()
        barrier(world)
        return max_over_ranks(e0.elapsed_time(e1), world, dev)

    run_steps(graphs, max(args.warmup, 3))
    torch.cuda.synchronize()
    assert status.value() == 0, "MLA decode kernel reported a wait timeout"
    clocks = ClockSampler(local)
    clocks.start()
    t_start = time.perf_counter()
    ms = timed(graphs, args.steps)
    while time.perf_counter() - t_start < 1.0:
        run_steps(graphs, cyc * 4)
        torch.cuda.synchronize()

    # ---- end to end: queries and selections in from pinned host memory, the
    # output back, every step; two device input sets and two outputs alternate
    # so that a step's copies (on their own streams, ordered by events)
    # overlap its neighbours' decode; captured in CUDA graphs ----
    h_q = [qn_h.pin_memory(), qr_h.pin_memory()]
    h_tk = [torch.from_numpy(case.topk_indices(v)).pin_memory() for v in range(V)]
    NBUF = 2
    d_qs = [[torch.empty_like(qn), torch.empty_like(qr)] for _ in range(NBUF)]
    d_tks = [torch.empty_like(tks[0]) for _ in range(NBUF)]
    d_outs = [torch.empty_like(out) for _ in range(NBUF)]
    h_outs = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(NBUF)]
    h2d = sum(t.numel() * t.element_size() for t in h_q) + h_tk[0].numel() * 4
    d2h = h_outs[0].numel() * h_outs[0].element_size()
    s_in = torch.cuda.Stream(device=dev)
    s_out = torch.cuda.Stream(device=dev)

    def e2e_steps(n):
        main = torch.cuda.current_stream()
        ev_in = [torch.cuda.Event() for _ in range(NBUF)]
        ev_used = [torch.cuda.Event() for _ in range(NBUF)]
        ev_out = [torch.cuda.Event() for _ in range(NBUF)]
        for k in range(NBUF):
            ev_used[k].record(main)
            ev_out[k].record(main)
        for i in range(n):
            k = i % NBUF
            s_in.wait_event(ev_used[k])
            with torch.cuda.stream(s_in):
                d_qs[k][0].copy_(h_q[0], non_blocking=True)
                d_qs[k][1].copy_(h_q[1], non_blocking=True)
                d_tks[k].copy_(h_tk[i % V], non_blocking=True)
            ev_in[k].record(s_in)
            main.wait_event(ev_in[k])
            main.wait_event(ev_out[k])
            launch(i, q=d_qs[k], tk=d_tks[k], o=d_outs[k])
            ev_used[k].record(main)
            s_out.wait_event(ev_used[k])
            with torch.cuda.stream(s_out):
                h_outs[k].copy_(d_outs[k], non_blocking=True)
            ev_out[k].record(s_out)
        main.wait_stream(s_in)
        main.wait_stream(s_out)

    def e2e_graph(n):
        s = torch.cuda.Stream(device=dev)
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            e2e_steps(min(n, NBUF * V))
        torch.cuda.current_stream().wait_stream(s)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            e2e_steps(n)
        return g

    g_e2e = (e2e_graph(cyc), {n % cyc: e2e_graph(n % cyc) for n in counts if n % cyc})
    run_steps(g_e2e, max(args.warmup, 3))
    n_e2e = args.steps
    ms_e2e = timed(g_e2e, n_e2e)
    clk = clocks.stop()
    torch.cuda.synchronize()
    assert status.value() == 0, "MLA decode kernel reported a wait timeout"

    flops_run = sum(flops_v[i % V] for i in range(args.steps))
    bytes_run = sum(bytes_v[i % V] for i in range(args.steps))
    us_launch = ms / args.steps * 1e3
    tflops = flops_run / (ms * 1e-3) / 1e12
    value = world * tflops
    peak, peak_src = measured_bf16_peak()
    hbm_peak, _ = measured_hbm_peak()
    gbs = bytes_run / (ms * 1e-3) / 1e9
    traffic = (MLA_TRAFFIC["bytes_per_launch"]
               if MLA_TRAFFIC["sources_sha1"] == mla_sources_sha1()
               and MLA_TRAFFIC["format"] == args.mla_format else None)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        host = mla_host_cache(case, used, rb)
        threads = host_threads()
        v, tok, dt, _ = mla_oracle_sample(case, host, args.cpu_seconds, fmt, threads)
        cpu = {**host_cpu(), "value": v, "unit": MLA_UNIT, "cores": threads, "kind": "oracle",
               "sample": "%d query tokens x 128 heads of the same workload (top-k selection 0), "
                         "C oracle, %d tokens at a time on %d threads, %.1f s"
                         % (tok, threads, threads, dt)}
    if rank == 0:
        line = {
            "metric": MLA_METRIC, "value": value, "unit": MLA_UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
            "us_per_step": us_launch, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16+e4m3", "data": "synthetic",
            "config": {
                "workload": mla_workload_name(args, case.B), "query_tokens": case.T,
                "keys_per_step": case.keys_read(0),
                "flops_per_step": flops_v[0], "bytes_per_step": bytes_v[0],
                "l2": "inputs larger than L2: %d top-k selections rotated (%.0f MB of rows each "
                      "> %.0f MB L2)" % (V, case.keys_read(0) * 656 / 1e6,
                                         torch.cuda.get_device_properties(dev).L2_cache_size / 1e6),
                "timing": "CUDA graphs replayed on one stream, CUDA events over the K steps",
                "parallelism": "replicas" if world > 1 else "single GPU",
            },
            "gpu_launches": args.steps,
            "roofline": {"bound": "tensor", "kernel": "pa_" + entry, "achieved": tflops,
                         "peak": peak, "unit": "TFLOP/s", "frac": tflops / peak,
                         "traffic": traffic, "peak_source": peak_src,
                         "us_per_launch": us_launch,
                         "algorithmic_flops_per_launch": flops_v[0],
                         "hbm": {"achieved_gbs": gbs, "peak_gbs": hbm_peak, "frac": gbs / hbm_peak,
                                 "algorithmic_bytes_per_launch": bytes_v[0]}},
            "e2e": {"value": world * flops_run / (ms_e2e * 1e-3) / 1e12, "unit": MLA_UNIT,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "us_per_step": ms_e2e / n_e2e * 1e3,
                    "issue": "pinned H2D copies of the queries and the step's top-k selection, "
                             "the decode, the D2H copy of the output, every step; two buffer "
                             "sets alternate so that a step's copies (own streams, ordered by "
                             "events) overlap its neighbours' decode; CUDA graphs"},
            "clocks": clk,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    finish_ranks(world)


if __name__ == "__main__":
    main()
