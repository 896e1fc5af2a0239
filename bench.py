"""Benchmark: CSA/HCA compressor gated-softmax pooling, forward + backward, per THD pack.

One step = csa_compressor_fwd + csa_compressor_bwd (the whole hot path) on one
synthetic pack resident in HBM. Metric: fwd+bwd time and achieved HBM GB/s, where the
bytes are the algorithmic ones (each consumed kv/score element read once, out/dout,
the full dKV/dScore writes, ape and dAPE; workspace traffic is not counted).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

Two timed passes of K steps each, both reported; `value` is the lower throughput:
  * flushed: before every step (outside the events) L2 is flushed, then one fwd+bwd is
    timed with events on its boundaries;
  * steady: K back-to-back fwd+bwd steps between two events, rotating over enough full
    buffer sets (inputs and outputs) that their total exceeds twice the L2 size, with no
    flush, so every step also pays the write-back of the previous step's gradients.
N > 1 runs one replica of the pack per GPU (the pooling has no cross-pack exchange):
under torch.distributed.run, or, when started without it, by relaunching itself under
it with N processes. Timing is the max over ranks, and the value is the bytes of all
ranks over that time. Rank 0 prints one JSON line.
--impl reference times the fp64 CPU oracle on all host cores instead (rank 0 only).

KPool configs (``--config kpool_*``, the DSA indexer's key pooling): one step is one
csa_kpool_fwd call (default FP32 mode; the key-dtype compression mode is timed beside
it); the same two passes, e2e, clocks, roofline and CPU baseline.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import thd_synth as ts  # noqa: E402

METRIC = "fwd+bwd µs and achieved HBM GB/s (% of GB300 roofline) per THD pack"
KPOOL_METRIC = "KPool forward µs and achieved HBM GB/s (% of GB300 roofline) per THD key pack"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 256 << 20
# The pages' own fwd + bwd times for the packs they measure (forward kernel after
# vectorisation + backward region, nsys kernel time, on B200 -- another machine: context,
# not the target). vs_baseline = our GB/s / (the same algorithmic bytes / that time).
PAGE_FWD_BWD_US = {"1x8192_d128": 4.5 + 12.8, "3x8192_d128": 10.0 + 22.2,
                   "1x8192_d512": 12.4 + 22.8, "3x8192_d512": 35.0 + 66.0}
# DRAM bytes per call of the roofline's kernel, from one ncu capture of the current
# kernel (the summaries are kept with the profiles): its DRAM reads (dram__bytes_read.sum)
# plus the bytes it writes into L2 (lts__t_sectors_srcunit_tex_op_write.sum x 32, all of
# which reach DRAM, also the part still dirty in L2 when the kernel ends), plus, for the
# compressor's backward call, the dAPE partials the reduction kernel reads (row groups x
# ratio x coff*d x 4 bytes). Re-measured whenever a kernel changes.
ROOFLINE_TRAFFIC = {"3x8192_d512": 108.2688e6 + 3223553 * 32 + 152 * 4 * 1024 * 4,
                    "long_r128_d512": 137.305344e6 + 4349953 * 32 + 19 * 128 * 512 * 4,
                    "kpool_64x8192_d128_p4": 268.466176e6 + 1048576 * 32}


# ----------------------------------------------------------------------------------
# Algorithmic bytes
# ----------------------------------------------------------------------------------

def consumed_slots(pack) -> int:
    lens = np.diff(pack.cu_seqlens.astype(np.int64))
    n = lens // pack.ratio
    if pack.coff == 2:
        return int(np.sum(np.where(n >= 1, pack.d * pack.ratio * (2 * n - 1), 0)))
    return int(np.sum(pack.d * pack.ratio * n))


def algorithmic_bytes(pack):
    ncons = consumed_slots(pack)
    rc = pack.ratio * pack.C
    reads = 2 * 2 * ncons + 4 * rc + 4 * (pack.S + 1)
    fwd = reads + 2 * pack.total_comp * pack.d
    bwd = reads + 2 * pack.total_comp * pack.d + 2 * 2 * pack.capacity * pack.C + 4 * rc
    return fwd, bwd


def workload_name(pack) -> str:
    lens = np.diff(pack.cu_seqlens)
    return (f"{pack.name}: THD pack S={pack.S} tokens={int(lens.sum())} capacity={pack.capacity} "
            f"ratio={pack.ratio} coff={pack.coff} d={pack.d} total_comp={pack.total_comp}")


def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            return float(json.load(fh)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ----------------------------------------------------------------------------------
# Multi-rank aggregation (replicas: one pack per GPU, no data-path collective)
# ----------------------------------------------------------------------------------

def max_over_ranks(values, device="cpu"):
    """Element-wise max of `values` over all ranks (identity without a process group)."""
    import torch
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def whole_job_gbs(world: int, bytes_per_rank_step: int, ms_per_step: float) -> float:
    """Bytes all ranks moved per step over the slowest rank's step time, in GB/s."""
    return world * bytes_per_rank_step / (ms_per_step * 1e-3) / 1e9


# ----------------------------------------------------------------------------------
# Clocks during the timed region
# ----------------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id: str):
        self.proc = None
        self.gpu_id = gpu_id
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_id}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
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
            out, _ = self.proc.communicate()
        rows = [r.split(",") for r in out.strip().splitlines() if r.count(",") >= 8]
        if not rows:
            return None
        mhz = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        maxm = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        reasons = sorted({n for r in rows for n, v in zip(self.NAMES, r[5:9])
                          if v.strip().lower() == "active"})
        return {"sm_mhz": statistics.median(mhz) if mhz else None,
                "sm_max_mhz": max(maxm) if maxm else None, "reasons": reasons,
                "samples": len(rows)}


# ----------------------------------------------------------------------------------
# Our arm
# ----------------------------------------------------------------------------------

def run_ours(args, rank, world, local_rank):
    import torch
    import gated_pooling_gb300 as gp

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    gp.load()
    pack = ts.make_pack(args.config)
    fwd_b, bwd_b = algorithmic_bytes(pack)
    S, r, coff, d, cap, TC, C = (pack.S, pack.ratio, pack.coff, pack.d, pack.capacity,
                                 pack.total_comp, pack.C)
    wsb = gp.csa_compressor_bwd_workspace_bytes(S, r, coff, d, cap, TC)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream

    def buffer_set(inputs):
        return {"in": inputs,
                "out": torch.empty((TC, d), dtype=torch.bfloat16, device=dev),
                "dkv": torch.empty((cap, C), dtype=torch.bfloat16, device=dev),
                "dsc": torch.empty((cap, C), dtype=torch.bfloat16, device=dev),
                "dape": torch.empty((r, C), dtype=torch.float32, device=dev),
                "ws": torch.empty(max(wsb, 16), dtype=torch.uint8, device=dev)}

    def set_bytes(bs):
        ts_ = list(bs["in"].values()) + [bs[k] for k in ("out", "dkv", "dsc", "dape", "ws")]
        return sum(x.numel() * x.element_size() for x in ts_)

    # the steady pass rotates over enough full buffer sets (inputs and outputs) that their
    # total is more than twice the L2 size: no step finds its data in L2
    base = buffer_set(ts.to_torch(pack, dev))
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or (132 << 20))
    # (at most 64 sets: a pack small enough to need more is launch-bound anyway, and its
    # steady pass then runs from L2, which the config line states)
    n_sets = min(max(args.rotate, -(-2 * l2 // set_bytes(base))), max(args.rotate, 64))
    sets = [base] + [buffer_set({k: v.clone() for k, v in base["in"].items()})
                     for _ in range(n_sets - 1)]
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_rd = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def flush_l2():
        # write a buffer larger than L2, then read another one: L2 ends up holding clean
        # lines of neither input, so the timed kernels pay no write-back of the flush
        flush.zero_()
        flush_rd.sum()

    def fwd(bs, e=err, strm=sp):
        t = bs["in"]
        gp.csa_compressor_fwd(t["kv"], t["score"], t["ape"], t["cu_seqlens"], S, r, coff, d,
                              cap, bs["out"], TC, e, stream=strm)

    def bwd(bs, e=err, strm=sp):
        t = bs["in"]
        gp.csa_compressor_bwd(t["kv"], t["score"], t["ape"], t["cu_seqlens"], t["dout"], S, r,
                              coff, d, cap, TC, bs["dkv"], bs["dsc"], bs["dape"], 0, bs["ws"],
                              wsb, e, stream=strm)

    for k in range(max(args.warmup, n_sets)):
        flush_l2()
        fwd(sets[k % n_sets])
        bwd(sets[k % n_sets])
    torch.cuda.synchronize()
    if int(err.item()) != 0:
        raise RuntimeError(f"device error {int(err.item())}")

    def new_events(n):
        return [torch.cuda.Event(enable_timing=True) for _ in range(n)]

    props = torch.cuda.get_device_properties(dev)
    gpu_id = str(getattr(props, "uuid", local_rank))
    if gpu_id and not gpu_id.startswith("GPU-") and "-" in gpu_id:
        gpu_id = "GPU-" + gpu_id  # nvidia-smi spells device UUIDs with this prefix
    sampler = ClockSampler(gpu_id)
    if rank == 0:
        sampler.start()

    def bracket():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    # pass 1, flushed: the K timed steps with L2 flushed before each (outside the events),
    # events on each step's boundaries only, so the backward's launch may overlap the
    # forward's tail as it does when a user issues the two calls back to back
    sev = [new_events(2) for _ in range(args.steps)]
    bracket()
    for k in range(args.steps):
        flush_l2()
        sev[k][0].record(stream)
        fwd(base)
        bwd(base)
        sev[k][1].record(stream)
    bracket()
    # pass 2, steady: K back-to-back steps over the rotated buffer sets, no flush
    st0, st1 = new_events(2)
    bracket()
    st0.record(stream)
    for k in range(args.steps):
        fwd(sets[k % n_sets])
        bwd(sets[k % n_sets])
    st1.record(stream)
    bracket()
    # the per-call split (and the roofline's backward-call time): K back-to-back forward
    # calls, then K back-to-back backward calls, over the rotated sets, events at the ends
    # only (an event between two calls would keep the second from launching early, which
    # back-to-back calls do)
    def steady_only(call):
        a, b = new_events(2)
        bracket()
        a.record(stream)
        for k in range(args.steps):
            call(sets[k % n_sets])
        b.record(stream)
        bracket()
        return a.elapsed_time(b)

    fwd_pass_ms = steady_only(fwd)
    bwd_pass_ms = steady_only(bwd)
    clocks = sampler.stop() if rank == 0 else None
    if int(err.item()) != 0:
        raise RuntimeError(f"device error {int(err.item())}")
    step_ms = [sev[k][0].elapsed_time(sev[k][1]) for k in range(args.steps)]
    total_ms, steady_total, fwd_total, bwd_total = max_over_ranks(
        [sum(step_ms), st0.elapsed_time(st1), fwd_pass_ms, bwd_pass_ms], device=dev)
    flushed_ms = total_ms / args.steps
    steady_ms = steady_total / args.steps
    ms_step = max(flushed_ms, steady_ms)  # the lower throughput is the headline
    fwd_us = fwd_total / args.steps * 1e3
    bwd_us = bwd_total / args.steps * 1e3
    value = whole_job_gbs(world, fwd_b + bwd_b, ms_step)

    # context: the same two calls captured once in a CUDA graph and replayed
    graph_us = None
    if not args.no_graph:
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                fwd(base, strm=None)
                bwd(base, strm=None)
        stream.wait_stream(side)
        gev = [new_events(2) for _ in range(min(args.steps, 200))]
        for a, b in gev:
            flush_l2()
            a.record(stream)
            g.replay()
            b.record(stream)
        torch.cuda.synchronize()
        graph_us = round(1e3 * sum(a.elapsed_time(b) for a, b in gev) / len(gev), 2)

    # end to end through the public API with host buffers (copies inside the region)
    e2e = run_e2e(args, pack, base["in"], dev, fwd_b + bwd_b, wsb) if rank == 0 else None
    if world > 1:
        torch.distributed.barrier()
    if rank != 0:
        return None

    peak, peak_kind = measured_hbm_peak()
    bwd_gbs = bwd_b / (bwd_us * 1e-6) / 1e9
    vs_baseline, baseline = None, None
    if args.config in PAGE_FWD_BWD_US:
        page_gbs = (fwd_b + bwd_b) / (PAGE_FWD_BWD_US[args.config] * 1e-6) / 1e9
        vs_baseline = round(value / page_gbs, 3)
        baseline = {"value": round(page_gbs, 1), "unit": "GB/s",
                    "source": f"the pages' fwd + bwd kernel times ({PAGE_FWD_BWD_US[args.config]:.1f} "
                              "us, nsys, B200: another machine, context only) over the same "
                              "algorithmic bytes"}
    per_gpu = lambda ms: (fwd_b + bwd_b) / (ms * 1e-3) / 1e9
    res = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": vs_baseline, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": workload_name(pack), "ratio": r, "coff": coff, "d": d, "S": S,
                   "capacity": cap, "total_comp": TC,
                   "l2": (f"value = the slower of two passes: (flushed) L2 flushed before every "
                          f"step outside the timed events ({L2_FLUSH_BYTES >> 20} MiB write, then "
                          f"a {L2_FLUSH_BYTES >> 20} MiB read); (steady) back-to-back steps "
                          f"rotating over {n_sets} full buffer sets of "
                          f"{set_bytes(base) / 1e6:.1f} MB "
                          + (f"(> 2x the {l2 >> 20} MiB L2)" if n_sets * set_bytes(base) > 2 * l2
                             else f"(together smaller than the {l2 >> 20} MiB L2: this pass "
                                  f"runs from L2)")
                          + ", no flush; per-call times from steady passes of one call kind"),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "flushed": {"us_per_step": round(flushed_ms * 1e3, 2),
                    "gbs_per_gpu": round(per_gpu(flushed_ms), 1)},
        "steady": {"us_per_step": round(steady_ms * 1e3, 2),
                   "gbs_per_gpu": round(per_gpu(steady_ms), 1), "buffer_sets": n_sets,
                   "set_bytes": set_bytes(base)},
        "fwd_us": round(fwd_us, 2), "bwd_us": round(bwd_us, 2),
        "fwd_plus_bwd_calls_us": round(fwd_us + bwd_us, 2),
        "graph_fwd_bwd_us": graph_us,
        "fwd_bytes": fwd_b, "bwd_bytes": bwd_b,
        "flushed_step_us_median": round(1e3 * float(np.median(step_ms)), 2),
        "flushed_step_us_min": round(1e3 * min(step_ms), 2),
        "fwd_gbs": round(fwd_b / (fwd_us * 1e-6) / 1e9, 1), "bwd_gbs": round(bwd_gbs, 1),
        "frac_of_measured_hbm": round(value / world / peak, 4),
        "frac_of_8tbs": round(value / world / NOMINAL_HBM_GBS, 4),
        "roofline": {"bound": "hbm", "kernel": "csa_compressor_bwd (pooling backward + dAPE reduction)",
                     "achieved": round(bwd_gbs, 1), "peak": peak, "peak_kind": peak_kind,
                     "unit": "GB/s", "frac": round(bwd_gbs / peak, 4),
                     "traffic": ROOFLINE_TRAFFIC.get(args.config)},
        "e2e": e2e, "clocks": clocks,
        # our kernels per timed pass: forward, pooling backward, dAPE reduction per step
        "gpu_launches": 3 * args.steps,
        "baseline": baseline,
    }
    if world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(pack, budget_s=args.cpu_seconds)
    return res


def run_e2e(args, pack, t, dev, alg_bytes, wsb):
    """The same metric through the public API with the data on the host: every step copies
    its inputs from pinned host memory to the device, runs both calls and copies every
    output back. Steps are pipelined the way a caller streaming packs would run them: two
    sets of device buffers, host-to-device copies on one stream, the calls on a second,
    device-to-host copies on a third, ordered by events, so that one step's input copy
    overlaps the previous step's output copy. The region runs from the first input copy to
    the last output copy."""
    import torch
    import gated_pooling_gb300 as gp

    S, r, coff, d, cap, TC, C = (pack.S, pack.ratio, pack.coff, pack.d, pack.capacity,
                                 pack.total_comp, pack.C)
    host = {k: v.cpu().pin_memory() for k, v in t.items()}
    h_out = torch.empty((TC, d), dtype=torch.bfloat16).pin_memory()
    h_dkv = torch.empty((cap, C), dtype=torch.bfloat16).pin_memory()
    h_dsc = torch.empty((cap, C), dtype=torch.bfloat16).pin_memory()
    h_dape = torch.empty((r, C), dtype=torch.float32).pin_memory()
    slots = []
    for _ in range(2):
        slots.append({
            "in": {k: torch.empty_like(v) for k, v in t.items()},
            "out": torch.empty((TC, d), dtype=torch.bfloat16, device=dev),
            "dkv": torch.empty((cap, C), dtype=torch.bfloat16, device=dev),
            "dsc": torch.empty((cap, C), dtype=torch.bfloat16, device=dev),
            "dape": torch.empty((r, C), dtype=torch.float32, device=dev),
            "ws": torch.empty(max(wsb, 16), dtype=torch.uint8, device=dev),
            "h2d_done": torch.cuda.Event(), "comp_done": torch.cuda.Event(),
            "d2h_done": torch.cuda.Event(),
        })
    s_h2d, s_comp, s_d2h = (torch.cuda.Stream(dev) for _ in range(3))
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = sum(x.numel() * x.element_size() for x in (h_out, h_dkv, h_dsc, h_dape))

    def step(k):
        sl = slots[k % 2]
        with torch.cuda.stream(s_h2d):
            if k >= 2:
                s_h2d.wait_event(sl["comp_done"])  # step k-2's calls have read these inputs
            for name, buf in sl["in"].items():
                buf.copy_(host[name], non_blocking=True)
            sl["h2d_done"].record(s_h2d)
        with torch.cuda.stream(s_comp):
            s_comp.wait_event(sl["h2d_done"])
            if k >= 2:
                s_comp.wait_event(sl["d2h_done"])  # step k-2's outputs have left
            x = sl["in"]
            sp = s_comp.cuda_stream
            gp.csa_compressor_fwd(x["kv"], x["score"], x["ape"], x["cu_seqlens"], S, r, coff, d,
                                  cap, sl["out"], TC, None, stream=sp)
            gp.csa_compressor_bwd(x["kv"], x["score"], x["ape"], x["cu_seqlens"], x["dout"], S,
                                  r, coff, d, cap, TC, sl["dkv"], sl["dsc"], sl["dape"], 0,
                                  sl["ws"], wsb, None, stream=sp)
            sl["comp_done"].record(s_comp)
        with torch.cuda.stream(s_d2h):
            s_d2h.wait_event(sl["comp_done"])
            h_out.copy_(sl["out"], non_blocking=True)
            h_dkv.copy_(sl["dkv"], non_blocking=True)
            h_dsc.copy_(sl["dsc"], non_blocking=True)
            h_dape.copy_(sl["dape"], non_blocking=True)
            sl["d2h_done"].record(s_d2h)

    for k in range(4):
        step(k)
    torch.cuda.synchronize()
    n = args.e2e_steps
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s_h2d)
    for k in range(n):
        step(k)
    s_d2h.wait_stream(s_h2d)
    b.record(s_d2h)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / n
    return {"value": round(alg_bytes / (ms * 1e-3) / 1e9, 1), "unit": "GB/s",
            "ms_per_step": round(ms, 4), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "pipelined": "two buffer sets; input copy, calls and output copy on three streams"}


# ----------------------------------------------------------------------------------
# KPool arm
# ----------------------------------------------------------------------------------

def kpool_bytes(pack) -> int:
    """Algorithmic bytes of one KPool forward: every pooled key and gate element read once
    (2 + 2 bytes), one bf16 output row per pool, cu_seqlens and the leads."""
    pooled = pack.total_pools * pack.pool * pack.d
    lead = 0 if pack.lead is None else 4 * pack.S
    return 4 * pooled + 2 * pack.total_pools * pack.d + 4 * (pack.S + 1) + lead


def kpool_workload_name(pack) -> str:
    lens = np.diff(pack.cu_seqlens)
    return (f"{pack.name}: THD key pack S={pack.S} keys={int(lens.sum())} capacity={pack.capacity} "
            f"pool={pack.pool} d={pack.d} pools={pack.total_pools} "
            f"leads={'none' if pack.lead is None else 'per segment'}")


def run_ours_kpool(args, rank, world, local_rank):
    import torch
    import gated_pooling_gb300 as gp

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    gp.load()
    pack = ts.make_kpool(args.config)
    nbytes = kpool_bytes(pack)
    TC, d = pack.total_pools, pack.d
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream

    def buffer_set(inputs):
        return {"in": inputs, "out": torch.empty((TC, d), dtype=torch.bfloat16, device=dev)}

    def set_bytes(bs):
        return sum(x.numel() * x.element_size() for x in list(bs["in"].values()) + [bs["out"]])

    base = buffer_set(ts.kpool_to_torch(pack, dev))
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or (132 << 20))
    n_sets = min(max(args.rotate, -(-2 * l2 // set_bytes(base))), max(args.rotate, 64))
    sets = [base] + [buffer_set({k: v.clone() for k, v in base["in"].items()})
                     for _ in range(n_sets - 1)]
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_rd = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def flush_l2():
        flush.zero_()
        flush_rd.sum()

    def call(bs, compress=0):
        t = bs["in"]
        gp.csa_kpool_fwd(t["key"], t["gate"], t["cu_seqlens"], t.get("lead"), pack.S, pack.pool,
                         d, pack.capacity, bs["out"], TC, compress, err, stream=sp)

    for k in range(max(args.warmup, n_sets)):
        flush_l2()
        call(sets[k % n_sets])
        call(sets[k % n_sets], 1)
    torch.cuda.synchronize()
    if int(err.item()) != 0:
        raise RuntimeError(f"device error {int(err.item())}")

    def new_events(n):
        return [torch.cuda.Event(enable_timing=True) for _ in range(n)]

    props = torch.cuda.get_device_properties(dev)
    gpu_id = str(getattr(props, "uuid", local_rank))
    if gpu_id and not gpu_id.startswith("GPU-") and "-" in gpu_id:
        gpu_id = "GPU-" + gpu_id
    sampler = ClockSampler(gpu_id)
    if rank == 0:
        sampler.start()

    def bracket():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    sev = [new_events(2) for _ in range(args.steps)]
    bracket()
    for k in range(args.steps):
        flush_l2()
        sev[k][0].record(stream)
        call(base)
        sev[k][1].record(stream)
    bracket()

    def steady(compress):
        a, b = new_events(2)
        bracket()
        a.record(stream)
        for k in range(args.steps):
            call(sets[k % n_sets], compress)
        b.record(stream)
        bracket()
        return a.elapsed_time(b)

    steady_total = steady(0)
    steady_c_total = steady(1)
    clocks = sampler.stop() if rank == 0 else None
    if int(err.item()) != 0:
        raise RuntimeError(f"device error {int(err.item())}")
    step_ms = [sev[k][0].elapsed_time(sev[k][1]) for k in range(args.steps)]
    total_ms, st_ms, stc_ms = max_over_ranks([sum(step_ms), steady_total, steady_c_total],
                                             device=dev)
    flushed_ms = total_ms / args.steps
    steady_ms = st_ms / args.steps
    compress_ms = stc_ms / args.steps
    ms_step = max(flushed_ms, steady_ms)
    value = whole_job_gbs(world, nbytes, ms_step)
    e2e = run_kpool_e2e(args, pack, base["in"], dev, nbytes) if rank == 0 else None
    if world > 1:
        torch.distributed.barrier()
    if rank != 0:
        return None
    peak, peak_kind = measured_hbm_peak()
    call_gbs = nbytes / (steady_ms * 1e-3) / 1e9
    per_gpu = lambda ms: nbytes / (ms * 1e-3) / 1e9
    res = {
        "metric": KPOOL_METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": kpool_workload_name(pack), "pool": pack.pool, "d": d,
                   "S": pack.S, "capacity": pack.capacity, "pools": TC, "mode": "fp32 weighted sum",
                   "l2": (f"value = the slower of two passes: (flushed) L2 flushed before every "
                          f"call outside the timed events; (steady) back-to-back calls rotating "
                          f"over {n_sets} buffer sets of {set_bytes(base) / 1e6:.1f} MB "
                          + (f"(> 2x the {l2 >> 20} MiB L2)" if n_sets * set_bytes(base) > 2 * l2
                             else f"(together smaller than the {l2 >> 20} MiB L2)") + ", no flush"),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "flushed": {"us_per_step": round(flushed_ms * 1e3, 2),
                    "gbs_per_gpu": round(per_gpu(flushed_ms), 1)},
        "steady": {"us_per_step": round(steady_ms * 1e3, 2),
                   "gbs_per_gpu": round(per_gpu(steady_ms), 1), "buffer_sets": n_sets,
                   "set_bytes": set_bytes(base)},
        "compress_us": round(compress_ms * 1e3, 2),
        "compress_gbs": round(per_gpu(compress_ms), 1),
        "bytes": nbytes,
        "frac_of_measured_hbm": round(value / world / peak, 4),
        "frac_of_8tbs": round(value / world / NOMINAL_HBM_GBS, 4),
        "roofline": {"bound": "hbm", "kernel": "csa_kpool_fwd (one pooling kernel)",
                     "achieved": round(call_gbs, 1), "peak": peak, "peak_kind": peak_kind,
                     "unit": "GB/s", "frac": round(call_gbs / peak, 4),
                     "traffic": ROOFLINE_TRAFFIC.get(args.config)},
        "e2e": e2e, "clocks": clocks,
        "gpu_launches": args.steps,
    }
    if world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = kpool_cpu_baseline(pack, budget_s=args.cpu_seconds)
    return res


def run_kpool_e2e(args, pack, t, dev, alg_bytes):
    """KPool through the public API with host buffers: each step copies the keys, gates,
    cu_seqlens and leads in from pinned host memory, pools, and copies the pooled keys back;
    pipelined over two device buffer sets on three streams like the compressor's e2e."""
    import torch
    import gated_pooling_gb300 as gp

    TC, d = pack.total_pools, pack.d
    host = {k: v.cpu().pin_memory() for k, v in t.items()}
    h_out = torch.empty((TC, d), dtype=torch.bfloat16).pin_memory()
    slots = [{"in": {k: torch.empty_like(v) for k, v in t.items()},
              "out": torch.empty((TC, d), dtype=torch.bfloat16, device=dev),
              "h2d_done": torch.cuda.Event(), "comp_done": torch.cuda.Event(),
              "d2h_done": torch.cuda.Event()} for _ in range(2)]
    s_h2d, s_comp, s_d2h = (torch.cuda.Stream(dev) for _ in range(3))
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = h_out.numel() * h_out.element_size()

    def step(k):
        sl = slots[k % 2]
        with torch.cuda.stream(s_h2d):
            if k >= 2:
                s_h2d.wait_event(sl["comp_done"])
            for name, buf in sl["in"].items():
                buf.copy_(host[name], non_blocking=True)
            sl["h2d_done"].record(s_h2d)
        with torch.cuda.stream(s_comp):
            s_comp.wait_event(sl["h2d_done"])
            if k >= 2:
                s_comp.wait_event(sl["d2h_done"])
            x = sl["in"]
            gp.csa_kpool_fwd(x["key"], x["gate"], x["cu_seqlens"], x.get("lead"), pack.S,
                             pack.pool, d, pack.capacity, sl["out"], TC, 0, None,
                             stream=s_comp.cuda_stream)
            sl["comp_done"].record(s_comp)
        with torch.cuda.stream(s_d2h):
            s_d2h.wait_event(sl["comp_done"])
            h_out.copy_(sl["out"], non_blocking=True)
            sl["d2h_done"].record(s_d2h)

    for k in range(4):
        step(k)
    torch.cuda.synchronize()
    n = args.e2e_steps
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s_h2d)
    for k in range(n):
        step(k)
    s_d2h.wait_stream(s_h2d)
    b.record(s_d2h)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / n
    return {"value": round(alg_bytes / (ms * 1e-3) / 1e9, 1), "unit": "GB/s",
            "ms_per_step": round(ms, 4), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "pipelined": "two buffer sets; input copy, call and output copy on three streams"}


def kpool_oracle_seconds(pack, threads: int) -> float:
    import oracle
    t0 = time.perf_counter()
    oracle.kpool_fwd_pack(pack, nthreads=threads)
    return time.perf_counter() - t0


def kpool_cpu_baseline(pack, budget_s=12.0):
    """The KPool oracle as it stands, on all host cores (std::thread over pool ranges) on
    the whole pack; `value` is that figure."""
    import oracle
    cores = oracle.hardware_threads()
    times = []
    t_end = time.perf_counter() + budget_s
    while not times or (time.perf_counter() < t_end and len(times) < 10):
        times.append(kpool_oracle_seconds(pack, cores))
    sec = statistics.median(times)
    return {"value": round(kpool_bytes(pack) / sec / 1e9, 4), "unit": "GB/s", "cores": cores,
            "kind": "oracle",
            "sample": f"the whole pack, FP32 mode on {cores} host threads (pool ranges), "
                      f"x{len(times)}, median {sec:.3f} s per call"}


def run_reference_kpool(args, rank):
    if rank != 0:
        return None
    import oracle
    oracle.build()
    cores = oracle.hardware_threads()
    pack = ts.make_kpool(args.config)
    for _ in range(args.warmup):
        kpool_oracle_seconds(pack, cores)
    times = [kpool_oracle_seconds(pack, cores) for _ in range(args.steps)]
    ms = 1e3 * sum(times) / len(times)
    value = kpool_bytes(pack) / (ms * 1e-3) / 1e9
    desc = f"fp64 KPool oracle on {cores} host threads (pool ranges), the whole pack per step"
    return {"impl": "reference", "metric": KPOOL_METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": kpool_workload_name(pack), "pool": pack.pool, "d": pack.d,
                       "S": pack.S, "capacity": pack.capacity, "pools": pack.total_pools,
                       "mode": "fp32 weighted sum"},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores,
                             "kind": "oracle", "sample": desc},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


# ----------------------------------------------------------------------------------
# CPU oracle (baseline leg and the reference arm)
# ----------------------------------------------------------------------------------

def sample_pack(pack, tokens: int):
    """The first `tokens` tokens (a multiple of ratio) of the pack's first segment, as a
    one-segment pack with the same ratio, coff, d and value streams."""
    tokens = max(pack.ratio, min(tokens, int(pack.cu_seqlens[1]) - int(pack.cu_seqlens[0])))
    tokens -= tokens % pack.ratio
    c0 = int(pack.cu_seqlens[0])
    n = tokens // pack.ratio
    return ts.Pack(pack.name + f"[sample {tokens} tokens]", pack.ratio, pack.coff, pack.d, tokens,
                   np.array([0, tokens], np.int32), pack.kv[c0:c0 + tokens],
                   pack.score[c0:c0 + tokens], pack.ape, pack.dout[:n])


def oracle_step_seconds(sp, threads: int = 1):
    """One fwd + bwd pass of the oracle: the single-thread entry points, or the
    multi-thread drivers over `threads` host threads."""
    import oracle
    t0 = time.perf_counter()
    if threads == 1:
        oracle.fwd_pack(sp)
        oracle.bwd_pack(sp)
    else:
        oracle.fwd_threads(sp, threads)
        oracle.bwd_threads(sp, threads)
    return time.perf_counter() - t0


def cpu_baseline(pack, budget_s=12.0):
    """The oracle as it stands, timed on this host: on all cores (std::thread over output
    rows) on the whole pack, and single-threaded on a bounded sample (the first 8192
    tokens of segment 0). `value` is the all-core figure."""
    import oracle
    cores = oracle.hardware_threads()
    fb, bb = algorithmic_bytes(pack)
    times = []
    t_end = time.perf_counter() + budget_s / 2
    while not times or (time.perf_counter() < t_end and len(times) < 10):
        times.append(oracle_step_seconds(pack, cores))
    sec_mt = statistics.median(times)
    sp = sample_pack(pack, min(int(pack.cu_seqlens[1]) - int(pack.cu_seqlens[0]), 8192))
    sfb, sbb = algorithmic_bytes(sp)
    stimes = []
    t_end = time.perf_counter() + budget_s / 2
    while not stimes or (time.perf_counter() < t_end and len(stimes) < 10):
        stimes.append(oracle_step_seconds(sp))
    sec_st = statistics.median(stimes)
    return {"value": round((fb + bb) / sec_mt / 1e9, 4), "unit": "GB/s", "cores": cores,
            "kind": "oracle",
            "sample": f"the whole pack, fwd+bwd on {cores} host threads (output-row ranges), "
                      f"x{len(times)}, median {sec_mt:.3f} s per pass",
            "sec_per_pass": round(sec_mt, 4),
            "single_thread": {"value": round((sfb + sbb) / sec_st / 1e9, 4), "unit": "GB/s",
                              "cores": 1,
                              "sample": f"first {sp.capacity} tokens of segment 0 "
                                        f"({sp.total_comp} output rows), x{len(stimes)}, "
                                        f"median {sec_st:.3f} s per pass"}}


def run_reference(args, rank):
    if rank != 0:
        return None
    import oracle
    oracle.build()
    cores = oracle.hardware_threads()
    pack = ts.make_pack(args.config)
    # each step is the whole pack on all host cores when that keeps the run within about
    # two minutes, else the first tokens of segment 0 that do
    budget = 120.0 / max(1, args.steps + args.warmup)
    probe = sample_pack(pack, 256 * pack.ratio)
    per_tok = oracle_step_seconds(probe, cores) / probe.capacity
    if per_tok * pack.capacity <= budget:
        sp, desc_sample = pack, "the whole pack"
    else:
        full = int(pack.cu_seqlens[1]) - int(pack.cu_seqlens[0])
        sp = sample_pack(pack, int(max(pack.ratio, min(full, budget / max(per_tok, 1e-9)))))
        desc_sample = f"the first {sp.capacity} tokens of segment 0 ({sp.total_comp} output rows)"
    fb, bb = algorithmic_bytes(sp)
    for _ in range(args.warmup):
        oracle_step_seconds(sp, cores)
    times = [oracle_step_seconds(sp, cores) for _ in range(args.steps)]
    ms = 1e3 * sum(times) / len(times)
    value = (fb + bb) / (ms * 1e-3) / 1e9
    desc = f"fp64 oracle on {cores} host threads (output-row ranges), {desc_sample} per step"
    return {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload_name(pack), "ratio": pack.ratio, "coff": pack.coff,
                       "d": pack.d, "S": pack.S, "capacity": pack.capacity,
                       "total_comp": pack.total_comp},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores,
                             "kind": "oracle", "sample": desc},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


# ----------------------------------------------------------------------------------
# Launch
# ----------------------------------------------------------------------------------

def replica_command(script, argv, nproc: int, port: int):
    """The command that runs `script argv` as `nproc` ranks of one node under
    torch.distributed.run, rendezvous on 127.0.0.1:`port`."""
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
            f"--nproc-per-node={nproc}", "--master-addr", "127.0.0.1",
            f"--master-port={port}", script, *argv]


def free_port() -> int:
    import socket
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", default=ts.HEADLINE, choices=sorted(ts.SPECS) + sorted(ts.KPOOL_SPECS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--rotate", type=int, default=3,
                    help="minimum buffer sets the steady pass rotates over")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.rotate < 3:
        ap.error("--rotate must be at least 3")

    if "WORLD_SIZE" not in os.environ and args.gpus > 1 and args.impl == "ours":
        # one replica per GPU: relaunch under torch.distributed.run with N ranks
        cmd = replica_command(os.path.abspath(__file__), sys.argv[1:], args.gpus, free_port())
        sys.exit(subprocess.call(cmd))

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    kpool = args.config in ts.KPOOL_SPECS
    if args.impl == "reference":
        res = run_reference_kpool(args, rank) if kpool else run_reference(args, rank)
    else:
        if world > 1:
            import torch
            torch.cuda.set_device(local_rank)
            torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
        res = (run_ours_kpool if kpool else run_ours)(args, rank, world, local_rank)
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
