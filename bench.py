"""Benchmark of the paged KV-cache hot path on GB300.

One step = one pass of the whole path over one batch of the page-shaped workload
(48 layer tensors [147456, 2, 16, 1, 128] bf16, 8 prompts x 576 blocks):
  kv_slot_mapping (73728 new tokens) -> kv_reshape_and_cache (48 layers) ->
  kv_build_xfer_list (4608 blocks) -> kv_pack_blocks (1.81 GB staged) ->
  kv_unpack_blocks (into the receiver's 147456-block cache at other block ids).
value = algorithmic bytes of the step (payload read + written, index arrays) / step time,
in GB/s, summed over ranks.  Inputs are larger than L2 (the step moves ~11 GB).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Under torchrun each rank runs an independent replica on its own GPU (weak scaling).
--impl reference times the CPU oracle (the plain C statement of the same step) on the
host cores on a bounded sample of the same workload.

Other modes: --stage host (staging in pinned host memory), --sw-window N (the
sliding-window clip before the builder), --layers / --num-blocks (reduced cases for
profiling captures), and two profiling drivers that print one JSON line of their own:
--write-only (the new-token write alone: the two calls and kv_write_tokens) and
--hash-only (kv_block_hashes alone).
"""
from __future__ import annotations

import argparse
import datetime
import gc
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_cache_81_gb300 import workloads as W  # noqa: E402

FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 512 << 20  # larger than the 129 MB L2
FLUSH_BELOW_BYTES = 1 << 30  # steps moving less than this are timed with an L2 flush before each step
NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e nominal bandwidth (context; the roofline uses the measured copy peak)
PG_TIMEOUT_S = 300  # process-group timeout under torchrun
KERNEL_NAMES = ("slot_mapping", "reshape_and_cache", "build_xfer_list", "pack", "unpack")
COPY_SOURCES = ("paged_kv_cache_81_gb300/csrc/kv_copy.cu", "paged_kv_cache_81_gb300/csrc/kv_copy.cuh",
                "paged_kv_cache_81_gb300/csrc/kv_bulk.cu", "paged_kv_cache_81_gb300/csrc/kv_async.cuh",
                "paged_kv_cache_81_gb300/csrc/kv_common.cuh")
WRITE_SOURCES = ("paged_kv_cache_81_gb300/csrc/kv_write.cu", "paged_kv_cache_81_gb300/csrc/kv_common.cuh")
# the sources whose change makes a kernel's DRAM-traffic record stale
KERNEL_SOURCES = {"pack": COPY_SOURCES, "unpack": COPY_SOURCES, "reshape_and_cache": WRITE_SOURCES}
COPY_KERNELS = ("reshape_and_cache", "pack", "unpack")  # the bandwidth-bound kernels of a step
# the other presets, measured at full size after the headline step (one after another)
EXTRA_WORKLOADS = ("tiny", "mid", "mla", "asym_remap", "page_shaped_kv_first")
EXTRA_TIMED_S = 0.5  # each extra workload's timed region lasts about this long


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="page_shaped", choices=sorted(W.PRESETS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the context measurements after the timed steps (write path, prior art, prefix hash)")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the other presets' full-size runs after the headline step")
    ap.add_argument("--workloads", default=",".join(EXTRA_WORKLOADS),
                    help="comma-separated presets measured at full size after the headline step")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="CPU work budget of the oracle baseline")
    ap.add_argument("--stage", default="device", choices=["device", "host"],
                    help="staging buffer in HBM, or in pinned host memory (pack/unpack over the host link)")
    ap.add_argument("--sw-window", type=int, default=0,
                    help="clip every request's block lists to the last N tokens before the xfer_list (0 = off)")
    ap.add_argument("--layers", type=int, default=None, help="override the layer count (profiling captures)")
    ap.add_argument("--num-blocks", type=int, default=None, help="override blocks per tensor (profiling captures)")
    ap.add_argument("--e2e-copy-streams", type=int, default=1,
                    help="host->device streams the e2e leg splits each step's new rows over")
    ap.add_argument("--write-only", action="store_true",
                    help="only the new-token write (slot_mapping + reshape_and_cache, kv_write_tokens); no receiver "
                         "or staging buffer (profiling captures)")
    ap.add_argument("--hash-only", action="store_true",
                    help="run only the prefix-hash measurement (kv_block_hashes), e.g. to profile its kernels")
    return ap.parse_args()


def workload(args) -> W.Workload:
    """The named preset, optionally shrunk for a profiler capture (same lists, smaller cache)."""
    from dataclasses import replace
    wl = W.PRESETS[args.workload]
    if args.layers:
        wl = replace(wl, n_layers=args.layers)
    if args.num_blocks:
        wl = replace(wl, src=replace(wl.src, num_blocks=args.num_blocks),
                     dst=replace(wl.dst, num_blocks=args.num_blocks))
    if args.layers or args.num_blocks:
        wl = replace(wl, name=f"{wl.name}[layers={wl.n_layers},num_blocks={wl.src.num_blocks}]")
    return wl


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def source_hash(paths) -> str:
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str, kernel: str):
    """DRAM bytes (read + write) per full-size launch of `kernel` from the committed ncu record of
    this workload (profiles/<workload>_dram.json), or None when the record is missing, holds no
    entry for the kernel, or the kernel's sources changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", f"{workload}_dram.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    entry = rec.get("kernels", {}).get(kernel)
    sources = KERNEL_SOURCES.get(kernel)
    if not entry or not sources or entry.get("source_hash") != source_hash(sources):
        return None
    return int(entry["bytes_per_launch_full"])


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        self.t0 = time.time()

    def mark(self):
        return time.time()

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t_begin, t_end):
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) >= 9:
                        rows.append(parts)
        except Exception:
            pass
        finally:
            if self.path and os.path.exists(self.path):
                os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1])]
        reasons = set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in rows:
            for name, v in zip(names, r[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": num(rows[0][2]),
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": max((num(r[3]) or 0.0) for r in rows)}


def reduce_max(x: float, device) -> float:
    """The maximum of x over all ranks (x itself without an initialised process group)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def config_dict(wl: W.Workload, case: W.Case, step=None) -> dict:
    d = {"workload": wl.name, "layers": wl.n_layers, "tensors": wl.n_tensors, "layout": wl.src.layout,
         "num_blocks": wl.src.num_blocks, "block_size": wl.src.block_size, "row_bytes": wl.src.row_bytes,
         "requests": case.n_reqs, "blocks_listed": case.n_blocks, "new_tokens": case.n_tokens,
         "payload_dtype": "bf16 (moved as opaque 16-byte vectors)",
         "l2": "inputs larger than L2: no flush (each step moves several GB through a 129 MB L2)"}
    if step is not None and step.bytes().total < FLUSH_BELOW_BYTES:
        d["l2"] = (f"flushed: a {L2_FLUSH_BYTES >> 20} MB write between timed steps (the step moves less than "
                   f"{FLUSH_BELOW_BYTES >> 20} MB); each step is timed by its own events, the flush outside them")
    if not wl.equal_geometry:
        d.update(dst_block_size=wl.dst.block_size, slice_bytes=wl.moved_slice, slice_off=wl.slice_off)
    if step is not None:
        d["max_run_blocks"] = step.max_run_blocks
        if step.sw_window:
            d.update(sw_window=step.sw_window, blocks_sent=step.n_listed)
    return d


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def run_ours(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        # a rank that dies makes the others' next collective fail within this bound instead of hanging
        dist.init_process_group("nccl", timeout=datetime.timedelta(seconds=PG_TIMEOUT_S))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from paged_kv_cache_81_gb300 import build
    build.build()
    from paged_kv_cache_81_gb300 import pagedkv as K

    wl = workload(args)
    case = W.make_case(wl)
    seed = wl.seed * 7919 + rank
    step = make_step(wl, case, dev, seed, host_stage=args.stage == "host", sw_window=args.sw_window or None)
    stream = torch.cuda.current_stream(dev)
    K.kv_get_last_error(clear=True)

    def barrier():
        if world > 1:
            dist.barrier()

    # the step as a user issues it (step.run(), no event inside): value and ms_per_step
    t = run_timed(step, dev, stream, args.steps, args.warmup, barrier=barrier, gpu_index=local, instrument=False)
    elapsed_ms = reduce_max(t["elapsed_ms"], dev)
    b = step.bytes()
    ms_per_step = elapsed_ms / args.steps
    value = world * b.total * args.steps / (elapsed_ms * 1e-3) / 1e9
    # then the same number of steps with every call bracketed by events: each kernel's duration
    ti = run_timed(step, dev, stream, args.steps, 0, barrier=barrier, gpu_index=local, instrument=True)

    peak, peak_kind = peaks()
    kernels, per_bytes, per_kernel_ms = kernel_stats(step, ti["per_kernel_all"], peak)
    roofline = roofline_entry(wl.name, per_bytes, per_kernel_ms, peak, peak_kind)

    extras = not args.no_extras
    write_path = measure_write_path(step, dev) if extras and step.n_tokens else None
    prior_art = measure_prior_art(step, dev, stream) if extras and args.stage == "device" and not args.sw_window \
        else None
    prefix_hash = measure_prefix_hash(case, dev, stream) if extras and case.req_tokens is not None else None
    single = measure_single_request(step, dev) if extras and args.stage == "device" and not args.sw_window else None

    host_link = None
    if args.stage == "host":
        # the bound of pack/unpack with host staging: device<->pinned copies of the staging size
        host_link = measure_host_link(step.stage, dev, stream)
        payload = per_bytes["pack"] // 2
        host_link["pack_gbs"] = round(payload / (per_kernel_ms["pack"] * 1e-3) / 1e9, 1)
        host_link["pack_frac_of_d2h"] = round(host_link["pack_gbs"] / host_link["d2h_gbs"], 4)
        if per_bytes["unpack"]:
            host_link["unpack_gbs"] = round(payload / (per_kernel_ms["unpack"] * 1e-3) / 1e9, 1)
            host_link["unpack_frac_of_h2d"] = round(host_link["unpack_gbs"] / host_link["h2d_gbs"], 4)

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, wl, case, step, dev, stream, K, world, barrier)

    line = {
        "metric": "KV pack/unpack GB/s moved and % of HBM peak; reshape_and_cache tokens/s",
        "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "u8", "data": f"synthetic (seeded random cache contents and block lists of the {wl.name} workload)",
        "config": config_dict(wl, case, step),
        "roofline": roofline,
        "kernels": kernels,
        "schedule": "build_xfer_list on a second stream beside slot_mapping + reshape_and_cache; pack, then "
                    "unpack, after both",
        "gpu_launches": args.steps * step.launches_per_step,
        "clocks": t["clocks"],
        "kernel_timing": {"steps": args.steps, "ms_per_step": round(reduce_max(ti["elapsed_ms"], dev) / args.steps, 4),
                          "clocks": ti["clocks"],
                          "how": "value and ms_per_step time K steps issued as step.run() with no event inside a step; "
                                 "kernels and roofline come from K more steps with CUDA events around every call on "
                                 "the stream it runs on (the events themselves lengthen that step)"},
        "e2e": e2e,
    }
    if write_path is not None:
        line["write_path"] = write_path
    if prior_art is not None:
        line["prior_art"] = prior_art
    if prefix_hash is not None:
        line["prefix_hash"] = prefix_hash
    if single is not None:
        line["single_request"] = single
    if host_link is not None:
        line["host_link"] = host_link
        line["config"]["stage"] = "pinned host memory"
    if extras and world == 1 and not args.no_workloads:
        # the other presets at full size, one after another: the headline step's buffers go first
        del step
        gc.collect()
        torch.cuda.empty_cache()
        names = [n for n in args.workloads.split(",") if n and n != wl.name]
        unknown = [n for n in names if n not in W.PRESETS]
        if unknown:
            raise SystemExit(f"unknown workloads {unknown}")
        line["workloads"] = measure_workloads(names, dev, stream, peak, peak_kind, local)
    if rank == 0 and not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(wl, case, args.cpu_seconds)
        if extras:
            line["cpu_baseline_all_cores"] = cpu_baseline_all_cores(wl, case, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def make_step(wl: W.Workload, case: W.Case, dev, seed: int, **kw):
    """The workload's caches (seeded random bits on the device), new token rows and TransferStep."""
    from paged_kv_cache_81_gb300.step import TransferStep

    src = W.device_cache(wl.src, wl.n_tensors, dev, seed=seed)
    dst = W.device_cache(wl.dst, wl.n_tensors, dev, seed=seed + 1) if wl.kind != "mla" else None
    new = W.new_token_rows(wl.src, wl.n_tensors, case.n_tokens, dev, seed=seed + 2)
    return TransferStep(wl, case, src, dst, new, device=dev, **kw)


def run_timed(step, dev, stream, steps: int, warmup: int, barrier=lambda: None, gpu_index: int = 0,
              instrument: bool = True) -> dict:
    """W untimed warm-up steps, then exactly K timed steps between CUDA events on `stream`, with a
    synchronize (and the barrier) on both sides and nvidia-smi clocks sampled meanwhile.

    instrument=False issues every step as step.run(), the call a user makes, with no event inside
    it; this pass gives the step time.  instrument=True brackets every call of a step with its own
    events (the builder on the step's second stream, issued first beside slot_mapping and
    reshape_and_cache; the rest on `stream`); this pass gives each kernel's duration.  The events
    cost the step time too (about 20 us of a 1.6 ms page-shaped step).  A step that moves less than
    FLUSH_BELOW_BYTES gets an L2-flushing write before it, outside its events, and the elapsed time
    is then the sum of the steps' own start-to-end brackets."""
    import torch
    from paged_kv_cache_81_gb300 import pagedkv as K

    side = step.side_stream()

    def slot_mapping():
        if step.n_tokens:
            K.kv_slot_mapping(step.block_table, step.token_req, step.token_pos, step.src.block_size, step.slot)

    def reshape_and_cache():
        if step.n_tokens:
            K.kv_reshape_and_cache(step.src, step.new_kv, step.slot)

    def timed_step(e):
        """One step.run(), bracketed: e[0] start, e[1] slot, e[2] reshape, e[3] joined, e[4] pack,
        e[5] unpack on `stream`; e[6], e[7] around the builder on the side stream."""
        e[0].record(stream)
        side.wait_stream(stream)
        e[6].record(side)
        step.build(side)
        e[7].record(side)
        slot_mapping()
        e[1].record(stream)
        reshape_and_cache()
        e[2].record(stream)
        stream.wait_stream(side)
        e[3].record(stream)
        step.pack(stream)
        e[4].record(stream)
        step.unpack(stream)
        e[5].record(stream)

    brackets = {"slot_mapping": (0, 1), "reshape_and_cache": (1, 2), "build_xfer_list": (6, 7), "pack": (3, 4),
                "unpack": (4, 5)}

    for _ in range(max(3, warmup)):
        step.run()
    torch.cuda.synchronize(dev)
    err = K.kv_get_last_error(clear=True)
    if err:
        raise RuntimeError(f"device error word {err:#x} after warm-up")

    sampler = ClockSampler(gpu_index)
    sampler.start()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(8)] for _ in range(steps)]
    barrier()
    torch.cuda.synchronize(dev)
    t_wall0 = time.time()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    flush = step.bytes().total < FLUSH_BELOW_BYTES
    flush_buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev) if flush else None
    start.record(stream)
    for s in range(steps):
        if flush:
            flush_buf.fill_(s & 0xFF)  # evicts the previous step's data from L2, outside the step's events
        if instrument:
            timed_step(ev[s])
        elif flush:
            ev[s][0].record(stream)
            step.run(stream)
            ev[s][5].record(stream)
        else:
            step.run(stream)
    end.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    t_wall1 = time.time()
    sampler.stop()
    clocks = sampler.summary(t_wall0, t_wall1)
    if flush:  # the sum of the steps' own durations, without the flushes between them
        elapsed_ms = sum(ev[s][0].elapsed_time(ev[s][5]) for s in range(steps))
    else:
        elapsed_ms = start.elapsed_time(end)
    per_kernel_all = {name: [ev[s][a].elapsed_time(ev[s][b]) for s in range(steps)]
                      for name, (a, b) in brackets.items()} if instrument else None
    err = K.kv_get_last_error(clear=True)
    if err:
        raise RuntimeError(f"device error word {err:#x} in the timed region")
    return {"elapsed_ms": elapsed_ms, "per_kernel_all": per_kernel_all, "clocks": clocks}


def kernel_stats(step, per_kernel_all: dict, peak: float):
    """Per-call entries (mean, median and best of the timed steps; algorithmic bytes; GB/s and the
    fractions of the measured and the nominal HBM bandwidth) of one timed run."""
    b = step.bytes()
    per_bytes = {"slot_mapping": b.slot_mapping, "reshape_and_cache": b.reshape_and_cache,
                 "build_xfer_list": b.build_xfer_list, "pack": b.pack, "unpack": b.unpack}
    per_kernel_ms = {name: statistics.mean(v) for name, v in per_kernel_all.items()}
    kernels = {}
    for name in KERNEL_NAMES:
        if per_bytes[name] == 0:
            continue
        ms = per_kernel_ms[name]
        gbs = per_bytes[name] / (ms * 1e-3) / 1e9
        kernels[name] = {"ms": round(ms, 4), "ms_median": round(statistics.median(per_kernel_all[name]), 4),
                         "ms_best": round(min(per_kernel_all[name]), 4), "bytes": per_bytes[name],
                         "gbs": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4),
                         "frac_of_nominal": round(gbs / NOMINAL_HBM_GBS, 4)}
    if step.n_tokens:
        kernels["reshape_and_cache"]["tokens_per_s"] = round(step.n_tokens / (per_kernel_ms["reshape_and_cache"] * 1e-3), 1)
    return kernels, per_bytes, per_kernel_ms


def roofline_entry(workload: str, per_bytes: dict, per_kernel_ms: dict, peak: float, peak_kind: str) -> dict:
    """The roofline of the step's bound kernel: of the bandwidth-bound calls (reshape_and_cache,
    pack, unpack) the one with the largest mean duration in this run, which is also the one
    furthest below the HBM peak when they move the same bytes."""
    cands = [k for k in COPY_KERNELS if per_bytes.get(k)]
    dominant = max(cands, key=lambda k: per_kernel_ms[k])
    achieved = per_bytes[dominant] / (per_kernel_ms[dominant] * 1e-3) / 1e9
    return {"bound": "hbm", "kernel": dominant, "achieved": round(achieved, 1), "peak": peak,
            "peak_kind": f"of {peak_kind} (MEASURED_PEAKS.json hbm_gbs, copy read+write)"
            if peak_kind == "measured" else "of fallback", "unit": "GB/s",
            "frac": round(achieved / peak, 4), "traffic": ncu_traffic(workload, dominant),
            "nominal_gbs": NOMINAL_HBM_GBS, "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
            "algorithmic_bytes_per_launch": per_bytes[dominant],
            "choice": "the slowest of reshape_and_cache, pack and unpack (largest mean duration)"}


def measure_workloads(names, dev, stream, peak: float, peak_kind: str, gpu_index: int) -> dict:
    """Every other preset at full size, one after another, each on freshly allocated caches that are
    freed before the next: the whole step timed for about EXTRA_TIMED_S (at least 5 steps, after 3
    warm-up steps), with per-call events and clocks as for the headline step."""
    import torch

    out = {}
    for name in names:
        wl = W.PRESETS[name]
        case = W.make_case(wl)
        step = make_step(wl, case, dev, wl.seed * 7919)
        probe = run_timed(step, dev, stream, 3, 3, gpu_index=gpu_index, instrument=False)  # sizes the timed run
        per_step_ms = max(probe["elapsed_ms"] / 3, 1e-3)
        steps = int(min(200, max(5, EXTRA_TIMED_S * 1e3 // per_step_ms)))
        t = run_timed(step, dev, stream, steps, 0, gpu_index=gpu_index, instrument=False)
        ti = run_timed(step, dev, stream, steps, 0, gpu_index=gpu_index, instrument=True)
        kernels, per_bytes, per_kernel_ms = kernel_stats(step, ti["per_kernel_all"], peak)
        entry = {"config": config_dict(wl, case, step), "steps": steps,
                 "ms_per_step": round(t["elapsed_ms"] / steps, 4),
                 "value": round(step.bytes().total * steps / (t["elapsed_ms"] * 1e-3) / 1e9, 1), "unit": "GB/s",
                 "roofline": roofline_entry(wl.name, per_bytes, per_kernel_ms, peak, peak_kind),
                 "kernels": kernels, "clocks": t["clocks"],
                 "device_time": "value: the steps issued as step.run() between two CUDA events; kernels: as many "
                                "steps again with CUDA events around each call on the stream it runs on"}
        if wl.kind == "mla" and step.n_tokens:
            # the decode write is launch-bound: besides its events inside the eager steps above,
            # its device time per write issued back to back from a CUDA graph
            back_to_back = measure_write_device({"two_calls": step.write_tokens, "write_tokens": step.write_tokens_call,
                                                 "fused": step.write_tokens_fused}, dev)
            entry["decode_write"] = {"tokens": step.n_tokens, "tensors": len(step.src.tensors),
                                     "eager_us_slot_mapping": round(kernels["slot_mapping"]["ms"] * 1e3, 2),
                                     "eager_us_reshape_and_cache": round(kernels["reshape_and_cache"]["ms"] * 1e3, 2),
                                     "device_us_per_write_back_to_back": back_to_back,
                                     "tokens_per_s_back_to_back": round(step.n_tokens / (back_to_back["write_tokens"]
                                                                                         * 1e-6), 1)}
        out[name] = entry
        del step
        gc.collect()
        torch.cuda.empty_cache()
    return out


def measure_prior_art(step, dev, stream, reps: int = 5):
    """The pages' own mechanism on the same GPU, for context: the NCCL connector gathers one
    tensor per (request, layer) with torch advanced indexing, layer[block_ids] (layer[:, block_ids]
    for kv-first), and the receiver scatters it with layer[block_ids] = tensor.  Whole-row
    workloads only (no head slice, same block size)."""
    import torch

    wl, case = step.wl, step.case
    if wl.moved_slice != wl.src.row_bytes or (step.dst is not None and not step.equal):
        return None
    kv_first = wl.src.layout == "kv_first"
    src_lists = [torch.from_numpy(case.src_ids[case.req_offsets[r]:case.req_offsets[r + 1]].astype("int64")).to(dev)
                 for r in range(case.n_reqs)]
    dst_lists = [torch.from_numpy(case.dst_ids[case.dst_req_offsets[r]:case.dst_req_offsets[r + 1]].astype("int64"))
                 .to(dev) for r in range(case.n_reqs)]

    def gather():
        return [[(layer[:, ids] if kv_first else layer[ids]) for ids in src_lists] for layer in step.src.tensors]

    def scatter(parts):
        for layer, per_req in zip(step.dst.tensors, parts):
            for ids, t in zip(dst_lists, per_req):
                if kv_first:
                    layer[:, ids] = t
                else:
                    layer[ids] = t

    parts = gather()
    if step.dst is not None:
        scatter(parts)
    torch.cuda.synchronize(dev)
    a, b, c = (torch.cuda.Event(enable_timing=True) for _ in range(3))
    g_ms = s_ms = 0.0
    for _ in range(reps):
        parts = None  # free the previous gather first (MLA's per-request tensors total ~38 GB)
        a.record(stream)
        parts = gather()
        b.record(stream)
        if step.dst is not None:
            scatter(parts)
        c.record(stream)
        torch.cuda.synchronize(dev)
        g_ms += a.elapsed_time(b)
        s_ms += b.elapsed_time(c)
    payload = step.bytes().pack  # read + written, as for kv_pack_blocks
    out = {"kind": "torch advanced indexing per (request, layer): layer[block_ids] gather, "
                   "layer[block_ids] = tensor scatter",
           "torch_calls_per_step": len(step.src.tensors) * case.n_reqs * (2 if step.dst is not None else 1),
           "gather_gbs": round(payload / (g_ms / reps * 1e-3) / 1e9, 1)}
    if step.dst is not None:
        out["scatter_gbs"] = round(payload / (s_ms / reps * 1e-3) / 1e9, 1)
    return out


def measure_prefix_hash(case, dev, stream, reps: int = 20) -> dict:
    """kv_block_hashes over the batch's token ids (seeded synthetic ids, the case's request lengths)."""
    import torch
    from paged_kv_cache_81_gb300 import pagedkv as K

    rng = np.random.default_rng(case.wl.seed + 7)
    lens = case.req_tokens.astype(np.int64)
    off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    toks = torch.from_numpy(rng.integers(0, 128000, size=int(off[-1])).astype(np.int32)).to(dev)
    off_d = torch.from_numpy(off).to(dev)
    bs = case.wl.src.block_size
    ws = torch.empty(max(16, K.kv_block_hashes_workspace_bytes(toks.shape[0], bs)), dtype=torch.uint8, device=dev)
    o, h = K.kv_block_hashes(off_d, toks, bs, 81, workspace=ws)
    torch.cuda.synchronize(dev)

    def timed(workspace):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        K.kv_block_hashes(off_d, toks, bs, 81, o, h, workspace=workspace)
        a.record(stream)
        for _ in range(reps):
            K.kv_block_hashes(off_d, toks, bs, 81, o, h, workspace=workspace)
        b.record(stream)
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b) / reps * 1e3

    tables_only = ws[: max(16, (toks.shape[0] // bs) * 2048)]
    us, two_kernel_us, chain_us = timed(ws), timed(tables_only), timed(None)
    n_hashes = int(sum(int(l) // bs for l in lens))
    return {"requests": int(lens.shape[0]), "tokens": int(off[-1]), "hashes": n_hashes, "us": round(us, 2),
            "hashes_per_s": round(n_hashes / (us * 1e-6), 1), "two_kernel_us": round(two_kernel_us, 2),
            "chain_us": round(chain_us, 2),
            "note": "us: the full workspace (tables and walk in one cooperative launch when the walk is the longer "
                    "part, else as two_kernel_us); two_kernel_us: a workspace of the tables alone (table kernel, then "
                    "the walk); chain_us: no workspace, one thread per request"}


def measure_single_request(step, dev, blocks: int = 64, iters: int = 200):
    """Latency of moving one request: build + pack + unpack of its first `blocks` blocks in every
    tensor of the same caches (wall clock per transfer, issued call by call and from a CUDA graph)."""
    import torch
    from paged_kv_cache_81_gb300.step import TransferStep

    wl, case = step.wl, step.case
    n = min(blocks, int(case.req_offsets[1] - case.req_offsets[0]))
    if n <= 0 or step.dst is None:
        return None
    one = W.Case(wl, np.array([0, n], np.int32), case.src_ids[:n].copy(), np.array([0, n], np.int32),
                 case.dst_ids[:n].copy() if step.equal else case.dst_ids[:case.dst_req_offsets[1]].copy(),
                 req_tokens=None)
    if not step.equal:  # the receiver's list of the first request, as many blocks as the staged tokens need
        one.dst_req_offsets = np.array([0, one.dst_ids.shape[0]], np.int32)
    small = TransferStep(wl, one, step.src.tensors, step.dst.tensors, device=dev)

    def transfer():
        small.build()
        small.pack()
        small.unpack()

    def wall(fn):
        for _ in range(5):
            fn()
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for _ in range(iters):
            fn()
        torch.cuda.synchronize(dev)
        return (time.perf_counter() - t0) / iters * 1e6

    eager = wall(transfer)
    graph = small.capture(transfer)
    replay = wall(graph.replay)
    del graph
    return {"blocks": n, "tensors": len(step.src.tensors), "bytes_moved": small.bytes().pack + small.bytes().unpack,
            "eager_us": round(eager, 2), "graph_us": round(replay, 2)}


def measure_write_path(step, dev, iters: int = 200) -> dict:
    """Wall-clock cost of the new-token write issued call by call from Python and replayed from a
    CUDA graph, in three forms: kv_slot_mapping + kv_reshape_and_cache; kv_write_tokens with
    slot_out; kv_write_tokens without slot_out (both one fused launch that looks the slots up in
    the row copy).  Plus each form's device time per write issued back to back from a graph."""
    import torch

    def timed(fn):
        for _ in range(5):
            fn()
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for _ in range(iters):
            fn()
        torch.cuda.synchronize(dev)
        return (time.perf_counter() - t0) / iters * 1e6

    forms = {"": step.write_tokens, "write_tokens_": step.write_tokens_call, "fused_": step.write_tokens_fused}
    out = {"tokens": step.n_tokens, "tensors": len(step.src.tensors)}
    for prefix, fn in forms.items():
        out[f"{prefix}eager_us_per_step"] = round(timed(fn), 2)
        graph = step.capture(fn)
        out[f"{prefix}graph_us_per_step"] = round(timed(graph.replay), 2)
        del graph
    out["device_us_per_write_back_to_back"] = measure_write_device(
        {"two_calls": step.write_tokens, "write_tokens": step.write_tokens_call, "fused": step.write_tokens_fused}, dev)
    return out


def measure_write_device(fns: dict, dev, per_graph: int = 20, replays: int = 10) -> dict:
    """Device time of one new-token write issued back to back: `per_graph` writes captured in one
    CUDA graph, the graph replayed `replays` times between CUDA events on the replaying stream."""
    import torch

    cur = torch.cuda.current_stream(dev)
    side = torch.cuda.Stream(dev)
    out = {}
    for name, fn in fns.items():
        fn()
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        side.wait_stream(cur)
        with torch.cuda.graph(g, stream=side):
            for _ in range(per_graph):
                fn()
        cur.wait_stream(side)
        for _ in range(3):
            g.replay()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(cur)
        for _ in range(replays):
            g.replay()
        b.record(cur)
        torch.cuda.synchronize(dev)
        out[name] = round(a.elapsed_time(b) * 1e3 / (replays * per_graph), 2)
        del g
    return out


def measure_host_link(host_buf, dev, stream, reps: int = 5) -> dict:
    """Device->host and host->device copy bandwidth (one direction's bytes) of a pinned buffer."""
    import torch

    d = torch.empty(host_buf.numel(), dtype=torch.uint8, device=dev)
    out = {}
    for name, (dst, src) in (("d2h_gbs", (host_buf, d)), ("h2d_gbs", (d, host_buf))):
        dst.copy_(src, non_blocking=True)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            dst.copy_(src, non_blocking=True)
        b.record(stream)
        torch.cuda.synchronize(dev)
        out[name] = round(host_buf.numel() * reps / (a.elapsed_time(b) * 1e-3) / 1e9, 1)
    del d
    return out


def run_e2e(args, wl, case, step, dev, stream, K, world, barrier):
    """The same step through the public API from pinned host buffers.

    Every step copies its inputs host->device (the new K/V rows of all layers and the token
    and block lists) and reads its run count back device->host.  All input copies go on a
    second stream into one of two buffer sets, so the copies of step k+1 run while step k
    computes; events order each buffer set's reuse after the step that read it.  The device
    error word is read once at the end (4 bytes)."""
    import torch

    comp = stream
    copy_stream = torch.cuda.Stream(dev)
    n_split = max(1, int(getattr(args, "e2e_copy_streams", 1)))
    row_streams = [copy_stream] + [torch.cuda.Stream(dev) for _ in range(n_split - 1)]
    row_done = [[torch.cuda.Event() for _ in row_streams] for _ in range(2)]
    names = ["req_offsets", "src_ids", "dst_req_offsets", "dst_ids"]
    if step.n_tokens:
        names += ["block_table", "token_req", "token_pos"]
    if step.sw_window:
        names += ["req_tokens"]
    host = {n: getattr(step, n).cpu().pin_memory() for n in names}
    sets = [{n: getattr(step, n) for n in names}, {n: getattr(step, n).clone() for n in names}]
    host_rows = None
    if step.n_tokens:
        big = step.new_kv[0]._base  # all tensors' new rows share one device buffer
        rows = [big, torch.empty_like(big)]
        for k in range(2):
            sets[k]["_rows"] = rows[k]
            sets[k]["_views"] = [rows[k][i] for i in range(rows[k].shape[0])]
        host_rows = torch.empty(big.shape, dtype=big.dtype, pin_memory=True)
        host_rows.copy_(big)
    steps = max(1, min(args.steps, 100))
    n_runs_host = torch.empty(steps, dtype=torch.int32, pin_memory=True)
    copied = [torch.cuda.Event() for _ in range(2)]
    freed = [torch.cuda.Event() for _ in range(2)]
    # per-step copy brackets on the copy stream: the rate the link delivers while the steps run
    c_begin = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    c_end = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    timing = {"on": False}
    h2d = sum(h.numel() * h.element_size() for h in host.values()) + (
        host_rows.numel() * host_rows.element_size() if host_rows is not None else 0)
    d2h = 4

    def issue_copy(k):
        b = k % 2
        if k >= 2:
            copy_stream.wait_event(freed[b])  # step k-2 is done with this buffer set
        if timing["on"]:
            c_begin[k].record(copy_stream)
        with torch.cuda.stream(copy_stream):
            for n in names:
                sets[b][n].copy_(host[n], non_blocking=True)
        if host_rows is not None:
            # the new rows, split over the copy streams (equal byte ranges of the one buffer)
            src_flat, dst_flat = host_rows.view(-1), sets[b]["_rows"].view(-1)
            edges = [src_flat.numel() * i // len(row_streams) for i in range(len(row_streams) + 1)]
            for i, rs in enumerate(row_streams):
                if rs is not copy_stream:
                    rs.wait_stream(copy_stream)
                with torch.cuda.stream(rs):
                    dst_flat[edges[i]:edges[i + 1]].copy_(src_flat[edges[i]:edges[i + 1]], non_blocking=True)
                if rs is not copy_stream:
                    row_done[b][i].record(rs)
                    copy_stream.wait_event(row_done[b][i])
        if timing["on"]:
            c_end[k].record(copy_stream)
        copied[b].record(copy_stream)

    def run_step(k):
        b = k % 2
        comp.wait_event(copied[b])
        for n in names:
            setattr(step, n, sets[b][n])
        if host_rows is not None:
            step.new_kv = sets[b]["_views"]
        step.run()
        freed[b].record(comp)
        n_runs_host[k:k + 1].copy_(step.xfer.n_runs, non_blocking=True)

    def run(n):
        issue_copy(0)
        if n > 1:
            issue_copy(1)
        for k in range(n):
            run_step(k)
            if k + 2 < n:
                issue_copy(k + 2)

    run(min(3, steps))
    torch.cuda.synchronize(dev)
    barrier()
    torch.cuda.synchronize(dev)
    timing["on"] = True
    t0 = time.perf_counter()
    run(steps)
    err = K.kv_get_last_error(clear=False)  # 4-byte read of the device error word; synchronises
    barrier()
    secs = time.perf_counter() - t0
    timing["on"] = False
    copy_ms = sum(c_begin[k].elapsed_time(c_end[k]) for k in range(steps))
    if err:
        raise RuntimeError(f"device error word {err:#x} in the end-to-end run")
    for n in names:  # leave the step on its original buffers
        setattr(step, n, sets[0][n])
    if host_rows is not None:
        step.new_kv = sets[0]["_views"]
    secs = reduce_max(secs, dev)
    value = world * step.bytes().total * steps / secs / 1e9
    out = {"value": round(value, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "steps": steps, "ms_per_step": round(secs / steps * 1e3, 4),
           "pipelined": "input copies of step k+1 (second stream, double-buffered) overlap step k",
           "copy_streams": len(row_streams)}
    if host_rows is not None:
        # this machine's host->device link, measured on the same pinned buffer: the bound of the leg
        link = measure_host_link(host_rows.view(torch.uint8).reshape(-1), dev, comp, reps=3)["h2d_gbs"]
        out["h2d_link_gbs"] = link
        out["link_bound_ms_per_step"] = round(h2d / (link * 1e9) * 1e3, 4)
    # what the copies achieved inside the timed run (the link is shared with the host's other work)
    out["h2d_gbs_during_run"] = round(h2d * steps / (copy_ms * 1e-3) / 1e9, 1)
    out["copy_ms_per_step_during_run"] = round(copy_ms / steps, 4)
    return out


# ---------------------------------------------------------------------------
# the oracle on the host cores: CPU baseline and the reference arm
# ---------------------------------------------------------------------------
class OracleSample:
    """A bounded sample of the workload for the CPU oracle: `layers` layer tensors of the
    full-size geometry (same block lists, same new tokens), on the host."""

    def __init__(self, wl: W.Workload, case: W.Case, layers: int = 1):
        import oracle

        self.oracle = oracle
        self.wl, self.case = wl, case
        self.nt = min(wl.n_tensors, layers * wl.src.tensors_per_layer)
        g = wl.src
        st = g.byte_strides()
        shape = (g.tensor_bytes,)
        self.src = [np.ones(shape, dtype=np.uint8) for _ in range(self.nt)]  # touched, so no page faults are timed
        self.src_cache = oracle.Cache(self.src, g.num_blocks, g.block_size, g.n_planes, st["block_stride"],
                                      st["plane_stride"], st["token_stride"], g.row_bytes)
        self.has_dst = wl.kind != "mla"
        if self.has_dst:
            d = wl.dst
            ds = d.byte_strides()
            self.dst = [np.ones((d.tensor_bytes,), dtype=np.uint8) for _ in range(self.nt)]
            self.dst_cache = oracle.Cache(self.dst, d.num_blocks, d.block_size, d.n_planes, ds["block_stride"],
                                          ds["plane_stride"], ds["token_stride"], d.row_bytes)
        T = case.n_tokens
        self.rows = [np.full((T, g.row_bytes), k, dtype=np.uint8) for k in range(self.nt * g.n_planes)] if T else []
        # algorithmic bytes of one sampled step (same accounting as the GPU step, scaled to the sample)
        payload = self.nt * case.n_blocks * g.n_planes * g.block_size * wl.moved_slice
        self.bytes = (T * 20 if T else 0) + (self.nt * g.n_planes * T * g.row_bytes * 2 + T * 8 if T else 0) + \
            case.n_blocks * 4 * (2 if (wl.equal_geometry and self.has_dst) else 1) + 2 * payload + \
            (2 * payload if self.has_dst else 0)

    def step(self):
        o, wl, case = self.oracle, self.wl, self.case
        if case.n_tokens:
            slot, _ = o.slot_mapping(case.block_table, case.token_req, case.token_pos, wl.src.block_size)
            o.reshape_and_cache(self.src_cache, self.rows, slot)
        equal = wl.equal_geometry and self.has_dst
        o.build_xfer_list(case.req_offsets, case.src_ids, case.dst_ids if equal else None, 0)
        stage = o.pack(self.src_cache, case.req_offsets, case.src_ids, wl.slice_off, wl.moved_slice)
        if self.has_dst:
            o.unpack(self.dst_cache, stage, case.req_offsets, case.dst_req_offsets, case.dst_ids,
                     wl.src.block_size, wl.moved_slice, wl.dst_slice_off)


def cpu_baseline(wl, case, seconds: float) -> dict:
    s = OracleSample(wl, case, layers=1)
    s.step()  # warm
    n, t0 = 0, time.perf_counter()
    while True:
        s.step()
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return {"value": round(s.bytes * n / el / 1e9, 3), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{n} steps of one layer ({s.nt} of {wl.n_tensors} tensors) of the {wl.name} step, "
                      f"single-threaded C oracle, {el:.1f} s; host has {os.cpu_count()} cores"}


def cpu_baseline_all_cores(wl, case, seconds: float) -> dict:
    """The same oracle step on every host core at once: one thread per core, each with its own
    one-layer sample (its own caches and staging), as a multi-layer step would spread layers.
    The C oracle runs outside the GIL (ctypes releases it), so the threads run in parallel.
    The thread count is capped so that the samples take at most half of the free host memory."""
    import threading

    probe = OracleSample(wl, case, layers=1)
    per_sample = sum(a.nbytes for a in probe.src) + sum(a.nbytes for a in getattr(probe, "dst", [])) + \
        sum(a.nbytes for a in probe.rows) + probe.nt * case.n_blocks * wl.src.n_planes * wl.src.block_size * \
        wl.moved_slice
    del probe
    try:
        free = os.sysconf("SC_AVPHYS_PAGES") * os.sysconf("SC_PAGE_SIZE")
    except (ValueError, OSError):
        free = 0
    cores = os.cpu_count() or 1
    threads = max(1, min(cores, int(free * 0.5 // max(per_sample, 1)))) if free else 1
    samples = [None] * threads
    counts = [0] * threads
    ready = threading.Barrier(threads + 1)
    go = threading.Event()
    stop = threading.Event()
    errors = []

    def worker(k):
        try:
            samples[k] = OracleSample(wl, case, layers=1)
            samples[k].step()  # warm
        except BaseException as e:  # reported below; the barrier must still be reached
            errors.append(e)
        ready.wait()
        go.wait()
        while samples[k] is not None and not stop.is_set():
            samples[k].step()
            counts[k] += 1

    ts = [threading.Thread(target=worker, args=(k,), daemon=True) for k in range(threads)]
    for t in ts:
        t.start()
    ready.wait()
    if errors:
        stop.set()
        go.set()
        raise errors[0]
    t0 = time.perf_counter()
    go.set()
    time.sleep(seconds)
    stop.set()
    for t in ts:
        t.join()
    el = time.perf_counter() - t0
    step_bytes = samples[0].bytes
    n = sum(counts)
    return {"value": round(step_bytes * n / el / 1e9, 3), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{threads} threads, each repeating one layer ({samples[0].nt} of {wl.n_tensors} tensors) "
                      f"of the {wl.name} step with its own caches; {n} steps in {el:.1f} s; host has {cores} cores"}


def run_reference(args):
    if int(os.environ.get("RANK", "0")) != 0:
        return  # under torchrun only rank 0 runs the CPU oracle
    wl = workload(args)
    case = W.make_case(wl)
    s = OracleSample(wl, case, layers=1)
    for _ in range(max(1, args.warmup)):
        s.step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        s.step()
    secs = time.perf_counter() - t0
    value = s.bytes * args.steps / secs / 1e9
    line = {
        "impl": "reference",
        "metric": "KV pack/unpack GB/s moved and % of HBM peak; reshape_and_cache tokens/s",
        "value": round(value, 3), "unit": "GB/s", "n_gpus": 0, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(secs / args.steps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "u8", "data": "synthetic",
        "config": config_dict(wl, case),
        "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"each step is one layer ({s.nt} of {wl.n_tensors} tensors) of the {wl.name} "
                                   f"step on the single-threaded C oracle; host has {os.cpu_count()} cores"},
        "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_hash_only(args):
    """Only the prefix-hash measurement of the workload's batch (no caches are allocated): the
    driver for profiling the hash kernels."""
    import torch
    from paged_kv_cache_81_gb300 import build
    build.build()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    wl = workload(args)
    case = W.make_case(wl)
    if case.req_tokens is None:
        raise SystemExit(f"workload {wl.name} has no token batch to hash")
    print(json.dumps({"workload": wl.name, "prefix_hash": measure_prefix_hash(case, dev, torch.cuda.current_stream(dev),
                                                                             reps=args.steps)}), flush=True)


def run_write_only(args):
    """Only the new-token write of the workload: the source cache and the new rows are allocated,
    no receiver cache or staging buffer.  The driver for profiling the write kernels: it issues
    `--steps` eager rounds of slot_mapping + reshape_and_cache and of kv_write_tokens without
    slot_out (the fused kernel), then (unless --no-extras) times each from CUDA graphs."""
    import torch
    from paged_kv_cache_81_gb300 import build
    build.build()
    from paged_kv_cache_81_gb300 import pagedkv as K
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    wl = workload(args)
    case = W.make_case(wl)
    if not case.n_tokens:
        raise SystemExit(f"workload {wl.name} writes no new tokens")
    seed = wl.seed * 7919
    cache = K.PagedCache.from_tensors(W.device_cache(wl.src, wl.n_tensors, dev, seed=seed), wl.src.layout)
    new = W.new_token_rows(wl.src, wl.n_tensors, case.n_tokens, dev, seed=seed + 2)
    table, req, pos = (torch.from_numpy(a).to(dev) for a in (case.block_table, case.token_req, case.token_pos))
    slot = torch.empty(case.n_tokens, dtype=torch.int64, device=dev)
    bs = wl.src.block_size

    def two_calls():
        K.kv_slot_mapping(table, req, pos, bs, slot)
        K.kv_reshape_and_cache(cache, new, slot)

    def fused():
        K.kv_write_tokens(cache, new, table, req, pos, None)

    K.kv_get_last_error(clear=True)
    for _ in range(args.steps):
        two_calls()
        fused()
    torch.cuda.synchronize(dev)
    err = K.kv_get_last_error()
    if err:
        raise SystemExit(f"device error word {err:#x}")
    line = {"workload": wl.name, "tokens": case.n_tokens, "tensors": wl.n_tensors,
            "bytes_per_write": 2 * case.n_tokens * wl.src.n_planes * wl.src.row_bytes * wl.n_tensors}
    if not args.no_extras:
        line["device_us_per_write_back_to_back"] = measure_write_device(
            {"two_calls": two_calls, "fused": fused}, dev)
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.hash_only:
        run_hash_only(args)
    elif args.write_only:
        run_write_only(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
