#!/usr/bin/env python
"""Throughput of the Polestar calibration + commit path on GB300.

One *step* is one denoising step of the seeded synthetic trajectory: a
``polestar_calibrate_step`` over every layer of every sequence (block entry:
full/partial forward, K-means, NVFP4, proxy baseline; within-block: patch,
proxy KL, top-k, sparse update packets) followed by ``polestar_commit``.  The
timed steps continue the trajectory after the warm-up, so they contain the
trajectory's own mix of block entries and within-block steps.

Metric: calibration steps/s (``value``); window tokens/s, per-class kernel
time, the roofline of the dominant kernel and the CPU oracle's throughput are
reported alongside.  Inputs (x0, logits, mask) of every step are resident in
HBM before the timed region; the per-step working set (the 32-layer weights,
14 GB) is far larger than L2, so no L2 flush is needed between steps.

Multi-GPU (torchrun): every rank runs an independent replica on its own
sequences (weak scaling, no collective on the data path); the JSON line
reports the whole-job aggregate over max-over-ranks time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

# the largest workload that fits one GPU: LLaDA-8B shape, batch 32, prompt 1024,
# generation 1024 (the stress configuration: the sparse refresh fires every step)
DEFAULT_WORKLOAD = "llada8b_p1024_g1024_b32"
# the other full-size workloads, measured after the headline (their own lines in
# "other_workloads"; fewer steps each)
DEFAULT_ALSO = "llada8b_p512_g256_b1,llada8b_p512_g512_b8,dream7b_p512_g256_b4"
# DRAM bytes (read + write) per launch of a kernel class, taken from one Nsight
# Compute capture of the current kernels (dram__bytes_read.sum +
# dram__bytes_write.sum, mean over the class's launches in the captured step),
# keyed by workload and class; an entry is removed whenever those kernels change,
# and the line then reports traffic null.
NCU_TRAFFIC_PER_LAUNCH = {}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
_T0 = time.perf_counter()


def log(msg):
    """Progress on stderr (the JSON line alone goes to stdout)."""
    print(f"[bench {time.perf_counter() - _T0:7.1f} s] {msg}", file=sys.stderr, flush=True)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        d["_source"] = "measured"
        return d
    d = dict(FALLBACK_PEAKS)
    d["_source"] = "fallback"
    return d


# ------------------------------------------------------------------ distributed
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(ws, backend):
    import torch.distributed as dist
    if ws > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return dist


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, ws: int, device=None) -> float:
    """Max of a host scalar over ranks (identity for one rank)."""
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_line(per_rank_units: float, ws: int, seconds_max: float) -> float:
    """Whole-job throughput: units of every rank over the slowest rank's time."""
    return per_rank_units * ws / seconds_max


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clk_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------ workload
def make_inputs(w, n_steps, device):
    """Trajectory inputs of the first n_steps steps, drawn on `device`."""
    import torch
    from drift_aware_kv_gb300 import synth
    tr = synth.Trajectory(w, device=device)
    dt = synth.torch_dtype(w)
    steps = []
    for _ in range(n_steps):
        st = tr.next_step()
        if st is None:
            break
        steps.append(dict(
            x0=st["x0"].to(dt), logits=st["logits"], masked=st["masked"].to(torch.uint8),
            n_unmasked=st["n_unmasked"], block_index=st["block_index"], block_entry=st["block_entry"]))
    return steps


# classes whose roofline the line reports, with their bound: projections are
# tensor-bound at batch >= 8 and at block entries, HBM-bound (weight stream)
# below; everything else moves bytes
def class_roofline(name, s, w, peaks):
    if s["launches"] == 0 or s["ms"] <= 0:
        return None
    if s["bytes"] <= 0 and s["flops"] <= 0:
        return {"bound": None, "frac": None, "avg_launch_us": s["ms"] * 1e3 / s["launches"],
                "launches": s["launches"], "note": "no algorithmic byte or flop model for this class"}
    # the roof that bounds the class: its flops at the tensor peak against its
    # algorithmic bytes at the copy rate, whichever takes longer
    tf_peak = peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops"))
    tensor = s["flops"] / (tf_peak * 1e12) > s["bytes"] / (peaks["hbm_gbs"] * 1e9)
    if tensor:
        peak = peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops"))
        achieved = s["flops"] / (s["ms"] / 1e3) / 1e12
        r = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
             "peak_source": peaks["_source"] + " bf16 sustained"}
    else:
        peak = peaks["hbm_gbs"]
        achieved = s["bytes"] / (s["ms"] / 1e3) / 1e9
        r = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
             "peak_source": peaks["_source"] + " copy"}
    r["traffic"] = NCU_TRAFFIC_PER_LAUNCH.get((w.name, name))
    r["algorithmic_bytes_per_launch"] = s["bytes"] / s["launches"]
    r["algorithmic_flops_per_launch"] = s["flops"] / s["launches"]
    r["avg_launch_us"] = s["ms"] * 1e3 / s["launches"]
    r["launches"] = s["launches"]
    if s["flops"] > 0:
        r["tflops"] = s["flops"] / (s["ms"] / 1e3) / 1e12
    if s["bytes"] > 0:
        r["gbs"] = s["bytes"] / (s["ms"] / 1e3) / 1e9
    return r


def run_workload(args, w, peaks, ws, rank, local, n_warmup, n_timed, full):
    """Warm-up + timed steps of one workload.  full: also the calibration-
    overhead region and the end-to-end region (the headline workload)."""
    import torch
    from drift_aware_kv_gb300 import polestar as P
    from drift_aware_kv_gb300 import synth

    dev = torch.device("cuda", local)
    log(f"{w.name}: weights")
    W = synth.make_weights(w, dev)
    total = n_warmup + n_timed
    log(f"{w.name}: inputs of {total} steps")
    steps = make_inputs(w.replace(seed=w.seed + rank), total, dev)
    if len(steps) < total:
        raise SystemExit(f"{w.name}: trajectory has only {len(steps)} steps < warmup + steps = {total}")
    torch.cuda.synchronize(dev)
    stream = torch.cuda.current_stream(dev)
    # the NVFP4 store's host traffic runs on a side stream of its own
    offload = args.host_store
    side = torch.cuda.Stream(dev) if offload else None
    cm = torch.zeros(w.batch, 2 * w.block, dtype=torch.uint8, device=dev)
    timed = steps[n_warmup:]

    def region(profile: bool, no_refresh: bool = False):
        """Fresh context: warm-up steps, then the timed steps.  The headline
        region runs without per-kernel events (they would serialise the
        programmatic dependent launches); the profiled region repeats the same
        steps with CUDA events around every launch for the per-class times.
        no_refresh: the same steps with the tau_upd trigger out of reach (no
        sparse refresh inside a block), for the calibration overhead."""
        wr = w.replace(tau_upd=10 ** 6) if no_refresh else w
        ps = P.Polestar(wr, W, stream=stream, side_stream=side, host_offload=offload)
        fired = []

        def do_step(st):
            o = ps.calibrate_step(st["x0"], st["n_unmasked"], st["block_index"], st["block_entry"])
            fired.append(not st["block_entry"] and all(o.fire[s] for s in range(w.batch)))
            ps.commit(st["logits"], st["masked"], cm)

        for st in steps[:n_warmup]:
            do_step(st)
        torch.cuda.synchronize(dev)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(timed) + 1)]
        if profile:
            ps.profile_begin(32 * w.n_layers * len(timed) + 256)
        clk = ClockSampler(local)
        launches0 = ps.launch_count()
        barrier(ws)
        torch.cuda.synchronize(dev)
        clk.start()
        t0 = time.perf_counter()
        ev[0].record(stream)
        issue_first = None
        for i, st in enumerate(timed):
            do_step(st)
            ev[i + 1].record(stream)
            if issue_first is None:
                # host time to enqueue one step into an empty queue (later
                # steps' enqueue times are bounded by the GPU once it fills)
                issue_first = time.perf_counter() - t0
        torch.cuda.synchronize(dev)
        wall = time.perf_counter() - t0
        barrier(ws)
        clocks = clk.stop()
        stats = ps.profile_end() if profile else None
        launches = ps.launch_count() - launches0
        step_ms = [ev[i].elapsed_time(ev[i + 1]) for i in range(len(timed))]
        total_ms = ev[0].elapsed_time(ev[-1])
        ps.close()
        return dict(stats=stats, launches=launches, step_ms=step_ms, total_ms=total_ms, wall=wall,
                    clocks=clocks, issue_first=issue_first, fired=fired[n_warmup:])

    log(f"{w.name}: timed region")
    main = region(profile=False)
    log(f"{w.name}: profiled region")
    prof = region(profile=True)
    overhead = None
    if full:
        # calibration overhead (the pages' App. D.10 measure): within-block steps
        # in which every sequence refreshed, against the same steps without refresh
        log(f"{w.name}: same steps without refresh")
        base = region(profile=False, no_refresh=True)
        log(f"{w.name}: same steps without refresh, profiled")
        base_prof = region(profile=True, no_refresh=True)
        fired_idx = [i for i, f in enumerate(main["fired"]) if f]
        if fired_idx:
            t_fire = statistics.mean(main["step_ms"][i] for i in fired_idx)
            t_base = statistics.mean(base["step_ms"][i] for i in fired_idx)
            # the same difference with every launch bracketed by events (the
            # launches then run one after another, as without any overlap)
            s_fire = statistics.mean(prof["step_ms"][i] for i in fired_idx)
            s_base = statistics.mean(base_prof["step_ms"][i] for i in fired_idx)
            per_layer = (t_fire - t_base) / w.n_layers
            serial = (s_fire - s_base) / w.n_layers
            overhead = {"ms_per_layer": per_layer, "steps": len(fired_idx),
                        "step_ms_refreshing": t_fire, "step_ms_same_steps_no_refresh": t_base,
                        "ms_per_layer_serialized": serial,
                        "overlap_fraction": (1.0 - per_layer / serial) if serial > 0 else None,
                        "what": "per-layer added time of a within-block step in which every sequence runs the "
                                "sparse refresh (patch, centroid update, proxy attention + KL, top-k, update "
                                "packets), against the same step with the trigger off; 'serialized' is the same "
                                "difference with every launch bracketed by CUDA events (no launch overlaps the "
                                "next), and overlap_fraction = 1 - ms_per_layer / ms_per_layer_serialized"}
    stats = prof["stats"]
    step_ms, total_ms, wall, clocks = main["step_ms"], main["total_ms"], main["wall"], main["clocks"]
    total_s = max_over_ranks(total_ms / 1e3, ws, dev)
    n_entry = sum(1 for st in timed if st["block_entry"])
    n_within = len(timed) - n_entry
    entry_ms = [m for m, st in zip(step_ms, timed) if st["block_entry"]]
    within_ms = [m for m, st in zip(step_ms, timed) if not st["block_entry"]]

    # ---- e2e: host buffers through polestar_step_host, copies in the timed region
    e2e = None
    if full and not args.no_e2e:
        # the first e2e_steps timed steps again, from pinned host buffers, after
        # the same warm-up (the last three warm-up steps also through the host path)
        n_e = min(args.e2e_steps, len(timed))
        ew = min(n_warmup, 3)
        log(f"{w.name}: host copies of {ew + n_e} steps' inputs")
        host = []
        for st in steps[n_warmup - ew: n_warmup + n_e]:
            host.append(dict(x0=st["x0"].cpu(), logits=st["logits"].cpu(), masked=st["masked"].cpu(),
                             n_unmasked=st["n_unmasked"], block_index=st["block_index"],
                             block_entry=st["block_entry"]))
        # two pinned staging sets, reused alternately as a serving loop reuses
        # its staging buffers: each step's inputs are written into one before
        # the step (untimed: that is the inputs' arrival in pinned memory), and
        # each call of polestar_step_host is timed from the host (it returns
        # with the result copied back and the stream synchronised).  Fresh
        # pinned buffers per step (17 GB at batch 32) made the copies 2-25x
        # slower on some GB300 machines, differently from machine to machine.
        stage = [{k: torch.empty_like(host[0][k]).pin_memory() for k in ("x0", "logits", "masked")}
                 for _ in range(2)]
        ps2 = P.Polestar(w, W, stream=stream, side_stream=side, host_offload=offload)
        cmh = torch.zeros(w.batch, 2 * w.block, dtype=torch.uint8).pin_memory()
        for st in steps[:n_warmup - ew]:
            ps2.calibrate_step(st["x0"], st["n_unmasked"], st["block_index"], st["block_entry"])
            ps2.commit(st["logits"], st["masked"], cm)

        def host_step(i, st):
            sb = stage[i % 2]
            for k in ("x0", "logits", "masked"):
                sb[k].copy_(st[k])
            t = time.perf_counter()
            ps2.step_host(sb["x0"], st["n_unmasked"], st["block_index"], st["block_entry"], sb["logits"],
                          sb["masked"], cmh)
            return time.perf_counter() - t

        for i, st in enumerate(host[:ew]):
            host_step(i, st)
        log(f"{w.name}: end-to-end region")
        barrier(ws)
        e2e_s = max_over_ranks(sum(host_step(ew + i, st) for i, st in enumerate(host[ew:])), ws, dev)
        ps2.close()
        h2d = host[0]["x0"].numel() * host[0]["x0"].element_size() + \
            host[0]["logits"].numel() * 4 + host[0]["masked"].numel()
        n_e_entry = sum(1 for st in host[ew:] if st["block_entry"])
        dev_ms = sum(step_ms[:n_e])
        e2e = {"value": aggregate_line(n_e, ws, e2e_s), "unit": "steps/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(cmh.numel()),
               "steps": n_e, "block_entries": n_e_entry,
               "device_value_same_steps": 1e3 * n_e / dev_ms if dev_ms > 0 else None,
               "what": f"the first {n_e} timed steps, each one call of polestar_step_host timed from the host "
                       "(x0, logits and mask copied in from pinned staging buffers, commit mask copied out, "
                       "stream synchronised); two staging sets reused alternately, each filled with its "
                       "step's inputs before the call"}
        del host, stage

    closed = None
    if full and not args.no_closed_loop:
        log(f"{w.name}: closed-loop region")
        closed = closed_loop_region(w, W, dev, stream, ws, args.closed_loop_steps)

    rooflines = {k: class_roofline(k, v, w, peaks) for k, v in stats.items()}
    rooflines = {k: v for k, v in rooflines.items() if v is not None}
    dom = max(stats, key=lambda k: stats[k]["ms"])
    roof = dict(rooflines[dom])
    roof["kernel"] = dom
    roof["traffic_unit"] = "bytes per launch (ncu dram__bytes_read.sum + dram__bytes_write.sum)"
    roof["measured_in"] = "profiled timed region (same steps, CUDA events around each launch)"

    nw_mean = statistics.mean(len(synth.window_positions(w, st["block_index"])) for st in timed)
    value = aggregate_line(len(timed), ws, total_s)
    return {
        "value": value, "ms_per_step": total_ms / len(timed), "steps": len(timed), "warmup": n_warmup,
        "config": {"workload": w.name, "model": "LLaDA-8B-shaped" if "llada" in w.name else "Dream-7B-shaped",
                   "layers": w.n_layers, "d_model": w.d_model, "batch": w.batch, "seq_len": w.seq_len,
                   "block": w.block, "window": w.prefix_win + w.suffix_win, "K": w.K, "topk": w.topk,
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
                   "nvfp4_store": "pinned host, 2-layer device ring" if offload else "device",
                   "l2": "per-step working set (weights) >> L2; no flush needed",
                   "timed_block_entries": n_entry, "timed_within_block_steps": n_within,
                   "attention_kernel": {0: "library choice", 1: "pipelined mma.sync", 2: "tcgen05"}[args.attn_impl]},
        "window_tokens_per_s": value * w.batch * nw_mean,
        "block_entry_ms": statistics.mean(entry_ms) if entry_ms else None,
        "within_block_ms": statistics.mean(within_ms) if within_ms else None,
        "within_block_steps_per_s": 1e3 / statistics.mean(within_ms) if within_ms else None,
        "kernel_ms_profiled_region": {k: round(v["ms"], 3) for k, v in stats.items()},
        "profiled_region_ms_per_step": prof["total_ms"] / len(timed),
        "kernel_launches": {k: v["launches"] for k, v in stats.items()},
        "calibration_overhead": overhead,
        "closed_loop": closed,
        "roofline": roof, "rooflines": rooflines, "clocks": clocks, "e2e": e2e,
        "gpu_launches": int(main["launches"]), "wall_s": wall,
        "host_issue_ms_first_step": main["issue_first"] * 1e3,
        "first_step_block_entry": bool(timed[0]["block_entry"]),
    }


def closed_loop_region(w, W, dev, stream, ws, n_timed, n_warmup=3):
    """Closed-loop decoding (Algorithm 1 in full) on the same weights: every step
    embeds the current tokens, calibrates, runs the final norm + LM head over
    the 2B gate rows, gates and writes the greedy tokens (the host reads the
    committed counts back every step).  A seeded prompt, random-init token
    embedding and LM head of the workload's vocabulary; with these weights the
    masked rows predict alike, so most commits come from the progress rule and
    tokens per forward stays near 1.  Times the steps after the warm-up with
    CUDA events, then the same number of further steps with per-launch events
    for the classes."""
    import torch
    from drift_aware_kv_gb300 import polestar as P
    from drift_aware_kv_gb300 import synth
    from drift_aware_kv_gb300.decode import Generator

    ps = P.Polestar(w, W, stream=stream)
    dw = synth.make_decode_weights(w, dev)
    gen = Generator(ps, dw)
    tok, msk = synth.make_prompt(w, dev)
    tok = tok.to(torch.int32)
    msk = msk.to(torch.uint8)
    it = gen.steps(tok, msk)
    for _ in range(n_warmup):
        next(it)
    torch.cuda.synchronize(dev)
    barrier(ws)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    n = committed = entries = 0
    for blk, entry, counts, left in it:
        n += 1
        committed += sum(counts)
        entries += int(entry)
        if n == n_timed:
            break
    e1.record(stream)
    torch.cuda.synchronize(dev)
    total_s = max_over_ranks(e0.elapsed_time(e1) / 1e3, ws, dev)
    ps.profile_begin(40 * w.n_layers * n_timed + 256)
    m = 0
    for _ in it:
        m += 1
        if m == n_timed:
            break
    stats = ps.profile_end()
    ps.close()
    del gen, dw
    torch.cuda.empty_cache()
    return {"steps_per_s": aggregate_line(n, ws, total_s), "ms_per_step": total_s * 1e3 / max(n, 1), "steps": n,
            "block_entries": entries, "tokens_committed": committed,
            "tokens_per_forward": committed / w.batch / max(n, 1), "vocab": w.vocab,
            "kernel_ms_profiled_steps": {k: round(v["ms"], 3) for k, v in stats.items()},
            "what": "embed + calibrate + final norm and LM head over the 2B gate rows + commit + progress rule "
                    "and greedy tokens, per step, committed counts read back each step; random-init weights "
                    "(tokens per forward near 1: the progress rule commits most tokens)"}


def run_device(args, w, peaks, ws, rank, local):
    import torch
    from drift_aware_kv_gb300 import synth
    from drift_aware_kv_gb300.build import build

    torch.cuda.set_device(local)
    if rank == 0 or ws == 1:
        build()
    barrier(ws)
    if args.attn_impl:
        from drift_aware_kv_gb300 import polestar as P
        P.attention_impl(args.attn_impl)
    out = run_workload(args, w, peaks, ws, rank, local, args.warmup, args.steps, full=True)
    out.update({"metric": "calibration steps/s", "unit": "steps/s", "n_gpus": ws, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
                "data": "synthetic (seeded trajectory drawn on the GPU, random-init N(0,0.02) weights)"})
    others = {}
    for name in [n for n in args.also.split(",") if n and n != w.name]:
        torch.cuda.empty_cache()
        wo = synth.WORKLOADS[name]
        r = run_workload(args, wo, peaks, ws, rank, local, 3, args.also_steps, full=False)
        others[name] = {k: r[k] for k in ("value", "ms_per_step", "steps", "warmup", "window_tokens_per_s",
                                          "block_entry_ms", "within_block_ms", "within_block_steps_per_s",
                                          "kernel_ms_profiled_region", "roofline", "rooflines", "clocks",
                                          "gpu_launches")}
        others[name]["config"] = r["config"]
    out["other_workloads"] = others
    return out


# ------------------------------------------------------------------ CPU oracle
def oracle_sample_workload(w, n_layers_sample):
    """The bounded sample the CPU oracle runs: sequence 0 of the workload (its own
    seeded drift schedule) on the first n_layers_sample layers.  Every other knob
    of the workload stays as it is."""
    return w.replace(batch=1, n_layers=min(n_layers_sample, w.n_layers))


def oracle_sample(w, n_layers_sample, n_steps, warmup=0):
    """Time the unmodified CPU oracle over the first warmup + n_steps trajectory
    steps of the sample workload; returns the seconds of each timed step (what
    was run, unscaled) and whether it was a block entry."""
    from drift_aware_kv_gb300 import synth
    from oracle import polestar_oracle as O
    ws = oracle_sample_workload(w, n_layers_sample)
    W = O.weights_to_numpy(synth.make_weights(ws, "cpu"))
    orc = O.PolestarOracle(ws, W)
    tr = synth.Trajectory(ws)
    dt = synth.torch_dtype(ws)
    times, kinds = [], []
    for i in range(warmup + n_steps):
        st = tr.next_step()
        if st is None:
            break
        x0 = st["x0"].to(dt).double().numpy()
        lg = st["logits"].numpy()
        mk = st["masked"].numpy()
        t0 = time.perf_counter()
        orc.calibrate_step(x0, st["n_unmasked"], st["block_index"], st["block_entry"])
        orc.commit(lg, mk)
        dtm = time.perf_counter() - t0
        if i >= warmup:
            times.append(dtm)
            kinds.append(bool(st["block_entry"]))
    return times, kinds


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        info = threadpool_info()
        return max([i.get("num_threads", 1) for i in info] or [1])
    except Exception:
        return os.cpu_count() or 1


def oracle_pieces(w, seed=0):
    """The oracle's separate pieces timed once each at the workload's full sizes
    (one problem: one layer of one sequence): spherical K-means + anchors of the
    window rows, residual NVFP4 of those rows, proxy KL drift over all heads and
    keys, the confidence of the 2B logit rows, and the commit threshold."""
    import numpy as np
    from oracle import polestar_oracle as O
    g = np.random.default_rng(seed)
    nw, d, K, H, N = w.prefix_win + w.suffix_win, w.d_model, w.K, w.n_heads, w.seq_len
    Hw = O.to_f32(g.standard_normal((nw, d)))
    out = {}
    t0 = time.perf_counter()
    labels, z, s_, A, _ = O.spherical_kmeans(Hw, K, w.kmeans_iters, O.kmeans_init(w.seed, 0, 0, 0, nw, K))
    out["kmeans_ms"] = 1e3 * (time.perf_counter() - t0)
    t0 = time.perf_counter()
    O.nvfp4_encode(O.to_f32(Hw - A[labels]))
    out["nvfp4_encode_ms"] = 1e3 * (time.perf_counter() - t0)
    sc, sp = g.standard_normal((K, H, N)), g.standard_normal((K, H, N))
    t0 = time.perf_counter()
    O.kl_div(sc, O.logsumexp(sc), sp, O.logsumexp(sp)).mean(axis=1)
    out["proxy_kl_ms"] = 1e3 * (time.perf_counter() - t0)
    lg = g.standard_normal((2 * w.block, w.vocab)).astype(np.float32)
    t0 = time.perf_counter()
    c = O.confidence(lg)
    O.drift_threshold(c, w.tau_s, w.alpha)
    out["confidence_gate_ms"] = 1e3 * (time.perf_counter() - t0)
    out["sizes"] = f"{nw} x {d} window rows, K = {K}; KL over {K} x {H} x {N}; {2 * w.block} x {w.vocab} logits"
    return out


CPU_SAMPLE_LAYERS = 1


def cpu_baseline(w, n_entry, n_within, budget_steps=3):
    """The oracle on a bounded sample (sequence 0, first layer, the first
    budget_steps trajectory steps: a block entry and within-block steps), plus
    its separate pieces at full size.  `value` converts the sample's measured
    per-step seconds to whole-workload steps/s -- every layer of every sequence,
    with the timed GPU steps' mix of block entries and within-block steps -- by
    plain multiplication (the oracle runs sequences and layers one after the
    other); that conversion is an estimate and is labelled so."""
    try:
        oracle_pieces(w)  # first touch of the large arrays, thread pools
        pieces = oracle_pieces(w)
    except Exception as e:  # an auxiliary figure never stops the bench line
        pieces = {"error": repr(e)}
    t0 = time.perf_counter()
    times, kinds = oracle_sample(w, CPU_SAMPLE_LAYERS, budget_steps)
    wall = time.perf_counter() - t0
    te = [t for t, k in zip(times, kinds) if k]
    tw = [t for t, k in zip(times, kinds) if not k]
    te_m = statistics.mean(te) if te else None
    tw_m = statistics.mean(tw) if tw else None
    scale = w.batch * w.n_layers / min(CPU_SAMPLE_LAYERS, w.n_layers)
    n = n_entry + n_within
    est = scale * ((n_entry * (te_m or 0)) + (n_within * (tw_m or te_m or 0))) / max(1, n)
    return {"value": 1.0 / est if est > 0 else None, "unit": "steps/s", "cores": blas_threads(),
            "kind": "oracle",
            "value_is": (f"estimate: the sample's measured seconds per step x {scale:g} (batch {w.batch} x "
                         f"{w.n_layers} layers / {min(CPU_SAMPLE_LAYERS, w.n_layers)} sampled), weighted "
                         f"{n_entry} entry : {n_within} within-block like the timed GPU steps"),
            "sample": (f"sequence 0 of {w.name}, layer 0 only, first {len(times)} trajectory steps "
                       f"(numpy float64 on the host's BLAS threads)"),
            "sample_s_per_step": {"block_entry": te_m, "within_block": tw_m},
            "sample_wall_s": wall, "pieces_full_size": pieces}


def run_reference(args, w):
    """Reference arm: the CPU oracle as it stands, timed step by step.  Each step
    is a bounded sample of the workload -- one trajectory step of sequence 0 on
    the first layer -- and `value` is those sample steps per second, exactly as
    timed.  The whole-workload equivalent (every layer of every sequence) is a
    separately named estimate."""
    t0 = time.perf_counter()
    times, kinds = oracle_sample(w, CPU_SAMPLE_LAYERS, args.steps, warmup=args.warmup)
    wall = time.perf_counter() - t0
    total = sum(times)
    value = len(times) / total
    scale = w.batch * w.n_layers / min(CPU_SAMPLE_LAYERS, w.n_layers)
    sample = (f"each step: one trajectory step (calibrate + commit) of sequence 0 of {w.name} on layer 0 "
              f"only; {sum(kinds)} of the {len(times)} timed steps are block entries")
    cb = {"value": value, "unit": "steps/s", "cores": blas_threads(), "kind": "oracle", "sample": sample}
    return {"impl": "reference", "metric": "calibration steps/s", "value": value, "unit": "steps/s",
            "n_gpus": 1, "steps": len(times), "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": w.name, "sample": sample}, "cpu_baseline": cb,
            "whole_step_estimate": {"steps_per_s": value / scale,
                                    "is": f"estimate: sample steps/s / {scale:g} (batch x layers / sampled layers)"},
            "wall_s": wall,
            "e2e": {"value": value, "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=16)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", default="polestar", choices=["polestar", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--also", default=DEFAULT_ALSO,
                    help="comma-separated further workloads measured after the headline ('' for none)")
    ap.add_argument("--also-steps", type=int, default=8, help="timed steps of each further workload")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=8,
                    help="timed steps replayed end to end from pinned host buffers (1.6 GB each at batch 32)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-closed-loop", action="store_true")
    ap.add_argument("--closed-loop-steps", type=int, default=8, help="timed closed-loop decoding steps")
    ap.add_argument("--attn-impl", type=int, default=0, choices=[0, 1, 2],
                    help="attention kernel: 0 the library's choice, 1 pipelined mma.sync, 2 tcgen05 (comparison runs)")
    ap.add_argument("--host-store", action="store_true",
                    help="keep the NVFP4 residual store in pinned host memory (2-layer device ring) instead of "
                         "device memory")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    from drift_aware_kv_gb300 import synth
    w = synth.WORKLOADS[args.workload]
    ws, rank, local = dist_env()
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, w)), flush=True)
        return
    init_dist(ws, "nccl")
    peaks = load_peaks()
    out = run_device(args, w, peaks, ws, rank, local)
    if rank == 0:
        if not args.no_cpu_baseline:
            log("cpu baseline (oracle sample)")
            out["cpu_baseline"] = cpu_baseline(w, out["config"]["timed_block_entries"],
                                               out["config"]["timed_within_block_steps"])
        log("done")
        print(json.dumps(out), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
