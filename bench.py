"""CSA2 decode benchmark: query-tok/s at 1M context, batch 32 (4 KV-source groups
x 10 layers per step), with the Indexer's and the attention's HBM bandwidth
against the measured roofline.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--config 3]

One step = one decode token for each of the B sequences through the whole
path of every layer: per group a Compressor append on the KV-source layer, a
window append on the 9 layers that share its compressed cache, one Indexer
scan over all compressed positions, one two-level selection, and 10 sparse
attention calls (one per layer, each with its own query and window).
Inputs are resident in HBM before timing; the per-step caches (4.8 GB of
index keys + 19 GB of compressed KV) are far larger than L2.

Prints one JSON line (rank 0). --impl reference times the CPU oracle (fp64 C)
on a bounded sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import faulthandler
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "CSA2 decode query-tok/s at 1M ctx, batch 32; indexer+attn HBM GB/s vs roofline"
UNIT = "query-tok/s"



_T0 = time.time()
_TRACE = None  # pinned launch-trace record (csa2_trace_attach), read after an error


def max_over_ranks(x, dist=None, device="cpu"):
    """The largest value of x over the ranks of the process group (x itself
    without one): the whole-job time of weakly scaled replicas is the slowest
    rank's."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def phase(msg):
    """Progress marker on stderr (the JSON line stays the only stdout output)."""
    print("[bench %7.1fs] %s" % (time.time() - _T0, msg), file=sys.stderr, flush=True)

def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# DRAM bytes per scanned position of k_index_scores_tc, from one ncu capture of
# the decode workload B=32, T=131072 (151.42 MB read + 4.22 MB written over
# 2,097,152 positions, the first timed launch). The figure belongs to that build
# of the kernel: it is reported only while the kernel source hashes to the same
# value.
INDEX_TRAFFIC_PER_POS = (151421696 + 4223744) / 2097152
INDEX_TRAFFIC_SRC_SHA256 = "b79582b21d45d77acce63abc8f633a4075edcb2c09e9f3a4be3abd1caa7edfc1"


def index_traffic(positions: float):
    import hashlib
    src = os.path.join(ROOT, "csa2_compressed_sparse_02_gb300", "csrc", "index_scores.cu")
    try:
        with open(src, "rb") as f:
            if hashlib.sha256(f.read()).hexdigest() != INDEX_TRAFFIC_SRC_SHA256:
                return None
    except OSError:
        return None
    return INDEX_TRAFFIC_PER_POS * positions


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock/throttle samples every 200 ms while running."""

    Q = ("index,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid=None):
        self.uuid = uuid
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.p = None

    def __enter__(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", "--query-gpu=" + self.Q, "--format=csv,noheader,nounits",
                                       "-lms", "200"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.p = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.p is not None:
            self.p.terminate()
            try:
                self.p.wait(timeout=5)
            except Exception:
                self.p.kill()

    def summary(self):
        self.f.flush()
        rows = []
        with open(self.f.name) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 10:
                    rows.append(parts)
        os.unlink(self.f.name)
        mine = [r for r in rows if self.uuid and self.uuid in r[1]]
        rows = mine or rows
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        mx = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[6 + i] == "Active"})
        loaded = [x for x in sm if x > 0.5 * (max(mx) if mx else 1)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ----------------------------------------------------------------------------- CPU oracle
def oracle_units(cfg, units, threads):
    """Run the oracle on `units` (group, seq) decode units of step 0 with `threads`
    threads; returns (unit seconds list, cores used). Inputs are regenerated before
    the timed oracle calls; each unit times only its own oracle arithmetic."""
    from concurrent.futures import ThreadPoolExecutor

    import numpy as np

    from csa2_compressed_sparse_02_gb300 import inputs as I
    from oracle import oracle as orc
    from oracle import reference

    def one(gs):
        g, s = gs
        T = cfg.first_lengths()[s]
        n_c = T // 2
        qv, qs, w = I.host_index_q(cfg, g, s, 0)
        kv, ks = I.host_index_keys(cfg, g, s, n_c)
        t0 = time.perf_counter()
        scores, _ = orc.index_scores(qv, qs, w, kv, ks)
        orc.block_max(scores, 8)
        idx, n_sel = orc.select(scores, 8, 2048, 512)
        sel = [int(j) for j in idx[:n_sel]]
        comp = reference.compressed_rows(cfg, cfg.layer(g, 0), s, sel)
        for r in range(cfg.readers):
            reference.attention(cfg, g, r, s, 0, sel, comp)
        return time.perf_counter() - t0

    with ThreadPoolExecutor(max_workers=threads) as ex:
        secs = list(ex.map(one, units))
    return secs, threads


def cpu_threads():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cpu_baseline(cfg, budget_units=None):
    threads = cpu_threads()  # every host core this process may run on
    n = budget_units or threads
    units = [(i % cfg.groups, (7 * i) % cfg.B) for i in range(n)]
    secs, cores = oracle_units(cfg, units, threads)
    per_unit = statistics.mean(secs)
    units_per_step = cfg.B * cfg.groups
    # `cores` units run concurrently, one per core
    value = cfg.B * cores / (per_unit * units_per_step)
    return {"value": value, "unit": UNIT, "cores": cores, "nproc": os.cpu_count(), "kind": "oracle",
            "sample": "%d (group, sequence) units of step 0 (Indexer over all %d compressed "
                      "positions, selection, compressed rows of the 512 selected, %d attention "
                      "layers), %d in parallel; mean %.2f s per unit; scaled to %d units per step"
                      % (n, cfg.first_lengths()[0] // 2, cfg.readers, cores, per_unit,
                         units_per_step)}


def run_reference(args, cfg, rank):
    if rank != 0:
        return
    threads = cpu_threads()  # every host core this process may run on, as the GPU arm's baseline
    per = []
    for _ in range(args.warmup):
        oracle_units(cfg, [(0, 0)], 1)
    t_all = []
    for k in range(args.steps):
        units = [((k + i) % cfg.groups, (7 * (k + i)) % cfg.B) for i in range(threads)]
        t0 = time.perf_counter()
        secs, _ = oracle_units(cfg, units, threads)
        t_all.append(time.perf_counter() - t0)
        per += secs
    per_unit = statistics.mean(per)
    value = cfg.B * threads / (per_unit * cfg.B * cfg.groups)
    ms_per_step = 1000.0 * per_unit * cfg.B * cfg.groups / threads
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 0,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": cfg.workload, "B": cfg.B,
                                            "T": cfg.first_lengths()[0]},
            "ms_per_step_extrapolated": True,
            "extrapolation": "each timed step runs %d (group, sequence) units of the %d a step "
                             "has, one per core; ms_per_step and value scale the mean unit time "
                             "to the whole step" % (threads, cfg.B * cfg.groups),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "nproc": os.cpu_count(),
                             "kind": "oracle",
                             "sample": "per step %d (group, sequence) units in parallel; "
                                       "scaled to %d units per step" % (threads, cfg.B * cfg.groups)},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- GPU
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", type=int, default=3)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the FP4 MMA rate, prefill chunk and ragged-run keys")
    ap.add_argument("--nvtx", action="store_true", help="mark the timed steps with an NVTX range")
    ap.add_argument("--eager", action="store_true", help="launch kernels one by one (no CUDA graph)")
    ap.add_argument("--whole-unit-attn", action="store_true",
                    help="fused attention in whole (layer, sequence) units, round robin, instead "
                         "of even (unit, tile) ranges per CTA")
    ap.add_argument("--chunk", type=int, default=0,
                    help="configuration 4 only: queries in the prefill chunk (default 8192)")
    args = ap.parse_args()
    faulthandler.enable()  # a crash prints every thread's Python stack to stderr
    args.warmup = max(3, args.warmup)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    from csa2_compressed_sparse_02_gb300.inputs import CONFIGS, PREFILL
    if args.config == PREFILL.number:
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "the reference arm times the "
                              "decode step; the prefill chunk is a secondary measurement"}))
            return
        prefill_main(args)
        return
    cfg = CONFIGS[args.config]
    if args.impl == "reference":
        run_reference(args, cfg, rank)
        return

    import torch
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)

    def barrier():
        if dist is not None:
            dist.barrier()

    from csa2_compressed_sparse_02_gb300 import workloads

    K, Wm = args.steps, args.warmup
    e2e_steps = 0 if args.no_e2e else K
    global _TRACE
    from csa2_compressed_sparse_02_gb300 import api as _api
    _TRACE = _api.trace_attach()
    phase("filling configuration %d" % args.config)
    split_steps = min(K, 10)  # the separate pass that times every call
    run = workloads.DecodeRun(cfg, n_steps=Wm + 2 + K + split_steps + e2e_steps + 5, out_slots=2,
                              split_attention=not args.whole_unit_attn)
    stream = torch.cuda.current_stream()

    # ---------------- warm-up, then one CUDA graph per prepared step
    for _ in range(Wm):
        run.step()
    torch.cuda.synchronize()
    mode = "eager"
    if not args.eager:
        phase("warm-up done; capturing graphs")
        # Timed graphs carry one pair of events, around group 0's Indexer launch (the
        # roofline's live launch time): every event in a graph orders the kernels
        # around it fully, and events around all 16 calls cost ~0.11 ms per step.
        # The per-call split comes from a second set, replayed after the timed region.
        full = run.capture_set(with_timers=True)
        if full is not None and run.capture(with_timers=True, timer_cats=("index",),
                                            timer_groups=(0,)):
            mode = "cuda-graph"
            for _ in range(2):
                run.step_graph()
            torch.cuda.synchronize()
    advance = run.step_graph if mode == "cuda-graph" else None
    phase("%s ready; timed steps" % mode)
    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    scan_bytes, eager_timers, slots = [], {}, []
    with ClockSampler(uuid) as clk:
        barrier()
        torch.cuda.synchronize()
        if args.nvtx:
            torch.cuda.nvtx.range_push("timed")
        start.record(stream)
        for _ in range(K):
            scan_bytes.append(run.scan_bytes())
            slots.append(run.step_done % run.n_prep)
            if advance:
                advance()
            else:
                run.step(timers=eager_timers)
        end.record(stream)
        if args.nvtx:
            torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize()
        barrier()
    clocks = clk.summary()
    elapsed = max_over_ranks(start.elapsed_time(end) / 1000.0, dist, dev)
    assert int(run.dev_status.item()) == 0, "device status %d" % int(run.dev_status.item())
    step_s = elapsed / K
    value = world * cfg.B * K / elapsed

    # Indexer launch time from the events of the timed steps (group 0's launch of
    # every step; the graph of a slot keeps the events of its last replay)
    if mode == "cuda-graph":
        idx_evs = [ev for k in dict.fromkeys(slots) for ev in run.graph_timers[k].get("index", [])]
    else:
        idx_evs = eager_timers["index"]
    scan_s = statistics.mean(a.elapsed_time(b) for a, b in idx_evs) / 1000.0
    # per-call split: a separate pass with events around every call (graph mode), or
    # the timed steps' own events (eager)
    split_ms = None
    if mode == "cuda-graph":
        graphs_all, timers_all = full
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        used = []
        s0.record(stream)
        for _ in range(split_steps):
            k = run.step_done % run.n_prep
            graphs_all[k].replay()
            run.step_done += 1
            used.append(k)
        s1.record(stream)
        torch.cuda.synchronize()
        split_ms = s0.elapsed_time(s1) / split_steps
        timers = {}
        for k in dict.fromkeys(used):
            for cat, evs in timers_all[k].items():
                timers.setdefault(cat, []).extend(evs)
        steps_covered = len(set(used))
    else:
        timers, steps_covered = eager_timers, K
    breakdown = {cat: sum(a.elapsed_time(b) for a, b in evs) / steps_covered
                 for cat, evs in timers.items()}  # ms per step spent in each call category
    scan_b = statistics.mean(scan_bytes)
    hbm_peak, peak_kind = peaks()
    achieved = scan_b / scan_s / 1e9
    attn_b = run.attn_bytes_per_call() * cfg.readers * cfg.groups
    step_alg_bytes = scan_b * cfg.groups + attn_b

    # ---------------- end to end through the public API with host buffers
    e2e = None
    if e2e_steps:
        phase("timed steps done; end-to-end steps")
        e2e = run_e2e(run, e2e_steps, stream, barrier, lambda x: max_over_ranks(x, dist, dev), world)

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": Wm, "ms_per_step": 1000.0 * step_s, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "nvfp4/e4m3/bf16 in, fp32 accumulate",
        "data": "synthetic (seeded counter-based generator; N(0,1)-shaped latents, "
                "uniform E2M1 index codes, 16 planted keys/seq)",
        "config": {"workload": cfg.workload, "B": cfg.B, "T": cfg.first_lengths()[0],
                   "groups": cfg.groups, "layers_per_group": cfg.readers,
                   "l2": "inputs larger than L2: %.2f GB of index keys streamed per step, "
                         "%.1f GB compressed cache" % (scan_b / 76.5 * 72 * cfg.groups / 1e9,
                                                       scan_b / 76.5 * 288 * cfg.groups / 1e9),
                   "parallelism": "replicas x%d (sequences sharded, no collective)" % world,
                   "attention_schedule": "whole units round robin" if args.whole_unit_attn
                   else "even (unit, tile) ranges per CTA, cut units merged"},
        "roofline": {"kernel": "index_scores (Indexer scan, fused block max)", "bound": "hbm",
                     "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "traffic": index_traffic(scan_b / 76.5),
                     "traffic_source": "ncu dram bytes of a B=32 T=131072 launch, scaled per position",
                     "peak_source": peak_kind, "launch_ms": 1000.0 * scan_s,
                     "bytes_per_launch": scan_b},
        "path_hbm": {"algorithmic_bytes_per_step": step_alg_bytes,
                     "achieved_gbs": step_alg_bytes / step_s / 1e9,
                     "frac": step_alg_bytes / step_s / 1e9 / hbm_peak},
        "gpu_launches": run.launches_per_step() * K,
        "launch_mode": mode,
        "ms_per_step_by_call": breakdown,
        "by_call_source": ("separate pass of %d steps with events around every call (%.3f ms "
                           "per step there)" % (split_steps, split_ms)) if split_ms else
                          "events around every call of the timed (eager) steps",
        "clocks": clocks,
    }
    if e2e:
        line["e2e"] = e2e
    if rank == 0 and not args.no_extras:
        # secondary workloads, after the timed region: the FP4 tensor rate, the
        # prefill chunk (configuration 4) and the ragged 16-step run (configuration 5)
        del run
        torch.cuda.empty_cache()
        phase("FP4 MMA rate")
        line["fp4_peak"] = fp4_peak(torch)
        phase("prefill chunk (configuration 4)")
        line["prefill"] = prefill_summary(torch, line["fp4_peak"]["tflops"])
        phase("ragged decode, 16 steps (configuration 5)")
        line["config5"] = config5_summary(torch)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        phase("oracle baseline on the host cores")
        line["cpu_baseline"] = cpu_baseline(cfg)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def prefill_main(args):
    """Configuration 4: one prefill chunk (8,192 queries on a 262,144-token context):
    window and Compressor append, per-query Indexer, selection and attention. A
    secondary line: prefill tokens per second, with the per-call split."""
    import dataclasses

    import torch
    from csa2_compressed_sparse_02_gb300 import workloads
    from csa2_compressed_sparse_02_gb300.inputs import PREFILL
    cfg = dataclasses.replace(PREFILL, chunk=args.chunk) if args.chunk > 0 else PREFILL
    run = workloads.PrefillRun(cfg)
    for _ in range(args.warmup):
        run.reset()
        run.run()
    torch.cuda.synchronize()
    K = max(1, min(args.steps, 10))
    timers = {}
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
    except Exception:
        pass
    with ClockSampler(uuid) as clk:
        torch.cuda.synchronize()
        start.record()
        for _ in range(K):
            run.reset()
            run.run(timers)
        end.record()
        torch.cuda.synchronize()
    assert int(run.dev_status.item()) == 0, "device status %d" % int(run.dev_status.item())
    el = start.elapsed_time(end) / 1000.0 / K
    n = cfg.chunk
    print(json.dumps({
        "metric": "CSA2 prefill tokens/s, chunk of %d queries on a %d-token context" % (n, cfg.T0),
        "value": n / el, "unit": "tok/s", "n_gpus": 1, "steps": K, "warmup": args.warmup,
        "ms_per_step": 1000.0 * el, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "nvfp4/e4m3/bf16 in, fp32 accumulate",
        "data": "synthetic (seeded counter-based generator)",
        "config": {"workload": cfg.workload if cfg is PREFILL else
                   "prefill chunk of %d queries on a %d-token context, NVFP4" % (n, cfg.T0),
                   "T0": cfg.T0, "chunk": n},
        "ms_per_step_by_call": {c: sum(a.elapsed_time(b) for a, b in evs) / K
                                for c, evs in timers.items()},
        "clocks": clk.summary(), "gpu_launches": None}), flush=True)


def fp4_peak(torch, iters=20000, launches=4):
    """The block-scaled FP4 MMA rate (csa2_fp4_mma_peak: the prefill Indexer's
    instruction, M = N = 128, K = 64, one CTA per SM), timed with CUDA events."""
    from csa2_compressed_sparse_02_gb300 import api
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.fp4_mma_peak(sms, 1000, st)  # warm-up
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(launches):
        api.fp4_mma_peak(sms, iters, st)
    b.record()
    torch.cuda.synchronize()
    assert int(st.item()) == 0, "fp4_mma_peak status %d" % int(st.item())
    flops = launches * sms * iters * 2.0 * 128 * 128 * 128
    tflops = flops / (a.elapsed_time(b) / 1e3) / 1e12
    return {"tflops": tflops, "shape": "tcgen05.mma.kind::mxf4nvf4.block_scale.scale_vec::4X, "
            "M=128 N=128 K=64, operands in shared memory, one CTA per SM, back to back",
            "ctas": sms, "iters": iters, "source": "measured in this run"}


def prefill_summary(torch, peak_tflops, chunks=3):
    """Configuration 4 (8,192 prefill queries on a 262,144-token context), timed
    after the decode line: chunk tokens/s, the per-call split, and the Indexer's
    FP4 contraction rate against the measured FP4 MMA rate."""
    from csa2_compressed_sparse_02_gb300 import workloads
    from csa2_compressed_sparse_02_gb300.inputs import DI, HI, PREFILL
    run = workloads.PrefillRun(PREFILL)
    for _ in range(2):
        run.reset()
        run.run()
    torch.cuda.synchronize()
    timers = {}
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(chunks):
        run.reset()
        run.run(timers)
    b.record()
    torch.cuda.synchronize()
    assert int(run.dev_status.item()) == 0, "device status %d" % int(run.dev_status.item())
    per_chunk = a.elapsed_time(b) / 1e3 / chunks
    split = {c: sum(x.elapsed_time(y) for x, y in evs) / chunks for c, evs in timers.items()}
    # FP4 contraction of the Indexer: 32 heads x 128 dims per visible compressed position
    n = PREFILL.chunk
    visible = sum((PREFILL.T0 + i + 1) // PREFILL.ratio for i in range(n))
    idx_flop = 2.0 * HI * DI * visible
    idx_tflops = idx_flop / (split["index"] / 1e3) / 1e12
    out = {"workload": PREFILL.workload, "value": n / per_chunk, "unit": "tok/s",
           "ms_per_chunk": 1e3 * per_chunk, "ms_per_chunk_by_call": split,
           "indexer": {"flop_per_chunk": idx_flop, "tflops": idx_tflops,
                       "fp4_peak_tflops": peak_tflops,
                       "frac": idx_tflops / peak_tflops if peak_tflops else None,
                       "peak_source": "fp4_peak of this line (measured)"}}
    del run
    torch.cuda.empty_cache()
    return out


def config5_summary(torch, warmup=3, steps=16):
    """Configuration 5 (32 sequences, context lengths log-uniform in [4,096,
    1,048,576], ragged caches, 1 index source + 5 readers): 16 consecutive decode
    steps as CUDA graphs, query-tok/s."""
    from csa2_compressed_sparse_02_gb300 import workloads
    from csa2_compressed_sparse_02_gb300.inputs import CONFIGS
    cfg = CONFIGS[5]
    run = workloads.DecodeRun(cfg, n_steps=warmup + 2 + steps)
    for _ in range(warmup):
        run.step()
    torch.cuda.synchronize()
    graphs = run.capture()
    if graphs:
        for _ in range(2):
            run.step_graph()
    else:
        for _ in range(2):
            run.step()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(steps):
        run.step_graph() if graphs else run.step()
    b.record()
    torch.cuda.synchronize()
    assert int(run.dev_status.item()) == 0, "device status %d" % int(run.dev_status.item())
    el = a.elapsed_time(b) / 1e3
    lens = cfg.first_lengths()
    out = {"workload": cfg.workload, "value": cfg.B * steps / el, "unit": UNIT,
           "ms_per_step": 1e3 * el / steps, "steps": steps,
           "launch_mode": "cuda-graph" if graphs else "eager",
           "context_tokens": {"min": min(lens), "max": max(lens), "mean": sum(lens) / len(lens)}}
    del run
    torch.cuda.empty_cache()
    return out


def run_e2e(run, K, stream, barrier, over_ranks=lambda x: x, world=1):
    """Same steps through the public API with every step's inputs copied from pinned
    host memory and its attention outputs copied back, inside the timed region
    (DecodeRun.pipelined_steps: the copies overlap the neighbouring steps' compute;
    the region ends when the last step's outputs have reached the host)."""
    import torch
    for _ in range(3):
        run.step_graph() if getattr(run, "graphs", None) else run.step(stream)
    torch.cuda.synchronize()
    slots = sorted({(run.step_done + i) % run.n_prep for i in range(K)})
    host_in = {k: run.host_input_pairs(k) for k in slots}
    host_out = torch.empty(run.outputs_of_slot(0).shape, dtype=run.outputs_of_slot(0).dtype,
                           pin_memory=True)
    h2d = sum(h.numel() * h.element_size() for h, _ in host_in[slots[0]])
    d2h = host_out.numel() * host_out.element_size()
    torch.cuda.synchronize()
    # the link as this process sees it: one slot's copies alone, each way
    link = {}
    for name, fn in (("h2d_gbs", lambda: [d.copy_(h, non_blocking=True) for h, d in host_in[slots[0]]]),
                     ("d2h_gbs", lambda: host_out.copy_(run.outputs_of_slot(0), non_blocking=True))):
        fn()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(3):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        link[name] = 3 * (h2d if name == "h2d_gbs" else d2h) / (a.elapsed_time(b) / 1e3) / 1e9
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    start.record(stream)
    t_host = time.perf_counter()
    run.pipelined_steps(K, host_in, lambda i: host_out, stream)
    t_host = time.perf_counter() - t_host
    end.record(stream)
    torch.cuda.synchronize()
    barrier()
    el = over_ranks(start.elapsed_time(end) / 1000.0)
    phase("end-to-end: %.3f ms per step (host enqueue %.3f ms per step); copies alone "
          "%.0f GB/s in, %.0f GB/s out" % (1e3 * el / K, 1e3 * t_host / K, link["h2d_gbs"],
                                           link["d2h_gbs"]))
    return {"value": world * run.cfg.B * K / el, "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "link_gbs": link,
            "overlap": "inputs of step i+1 and outputs of step i copied on side streams "
                       "while step i (resp. i+1) computes; one contiguous copy each way per step"}


if __name__ == "__main__":
    try:
        main()
    except Exception:
        if _TRACE is not None:  # which kernel launch was running when the error came
            from csa2_compressed_sparse_02_gb300 import api as _api
            print("[bench] " + _api.trace_read(_TRACE), file=sys.stderr, flush=True)
        raise
