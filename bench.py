"""Benchmark: one paged decode step on GB300.

A step is one pass of the whole hot path over one batch: the copy-on-write
block copies the pool asked for, the KV write of each sequence's new token
through the slot mapping, and paged decode attention over the updated cache
(stream-K pieces + the log-sum-exp merge where a sequence spans several
CTAs). By default the KV write is fused into the decode launch
(pa_append_decode).

Headline workload (default): the largest single-GPU configuration, a
Llama-3-70B-class long-context layer: 32 sequences, 64 query / 8 KV heads,
head dim 128, bf16, block size 16, context lengths uniform in [8192, 32768]
(+1 appended token), physical blocks shuffled across a pool 1.25x the need.
Synthetic seeded data, q/K/V ~ N(0, 1). Its K/V (2.7 GB per step) is 20x
the 129 MB L2, and two pool copies rotate, so every step streams from HBM.

Timing. W untimed warm-up steps and a sustained untimed loop under the
clock sampler, then K steps timed by one pair of CUDA events with nothing
in between (value, ms_per_step). A separate pass after it brackets single
launches of the step's decode call with events (roofline.achieved): an
event next to a launch serialises it with its neighbours, so that pass is
kept out of the timed loop.

Metric: algorithmic bytes per step / step time (GB/s), with the fraction of
the measured HBM peak (and of the 8 TB/s nominal) and steps/s alongside.
Algorithmic bytes: every cached K/V byte of every sequence once (GQA
packing), q in and out, block-table entries and lengths, plus the KV
write's bytes.

``other_workloads`` carries the other configurations (the tiny one, the
8B-class layer at 64 and 256 sequences, the 70B-class batch of 8, the
shared-prefix + copy-on-write batch) and the variants (block sizes 8 and
32, the 8-bit cache, several new tokens per sequence), each with its plain
step loop and its bracketed launch.

``--impl reference`` times the float64 CPU oracle (the reference arm) on a
bounded sample of the headline workload.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "paged decode attention KV HBM GB/s (% of GB300 peak) and decode steps/s"
UNIT = "GB/s"
L2_BYTES = 129 * 1024 * 1024
NOMINAL_HBM_GBS = 8000.0  # GB300 HBM3e, nominal

# name -> (recipe factory, description)
WORKLOADS = {
    "tiny_b4": (lambda: workloads.tiny(),
                "4 seqs {1,5,17,33}+1, 4 q / 1 KV head, head_dim 64, bf16, block 16, 16-block pool"),
    "llama8b_layer_b64": (lambda: workloads.llama8b_layer(),
                          "64 seqs, 32 q / 8 KV heads, head_dim 128, bf16, block 16, "
                          "L~U[128,2048]+1, shuffled 1.25x pool"),
    "llama8b_high_concurrency_b256": (lambda: workloads.llama8b_high_concurrency(),
                                      "256 seqs, 32/8 heads, head_dim 128, bf16, block 16, "
                                      "L~lognormal(median 800, sigma 1) clipped [16,4096]+1"),
    "llama70b_long_b8": (lambda: workloads.llama70b_long(batch=8),
                         "8 seqs, 64/8 heads, head_dim 128, bf16, block 16, L~U[8192,32768]+1"),
    "llama70b_long_b32": (lambda: workloads.llama70b_long(batch=32),
                          "32 seqs, 64 q / 8 KV heads, head_dim 128, bf16, block 16, "
                          "L~U[8192,32768]+1 appended token, shuffled 1.25x pool"),
    "shared_prefix_cow_b512": (lambda: workloads.shared_prefix(),
                               "512 seqs over one 1024-token shared prefix + U[16,512] suffixes, "
                               "32 copy-on-write appends, 32/8 heads, head_dim 128, bf16"),
    "llama8b_layer_b64_bs8": (lambda: workloads.llama8b_layer(block_size=8),
                              "the 64-sequence 8B-class layer at block size 8"),
    "llama8b_layer_b64_bs32": (lambda: workloads.llama8b_layer(block_size=32),
                               "the 64-sequence 8B-class layer at block size 32"),
    "llama70b_long_b8_bs32": (lambda: workloads.llama70b_long(batch=8, block_size=32),
                              "the 70B-class batch of 8 at block size 32"),
}
HEADLINE = "llama70b_long_b32"
# BASELINE configs these workloads stand for
CONFIG_OF = {"tiny_b4": 1, "llama8b_layer_b64": 2, "llama8b_high_concurrency_b256": 3,
             "llama70b_long_b8": 4, "llama70b_long_b32": 4, "shared_prefix_cow_b512": 5}


# ----------------------------------------------------------------------------- bytes

def decode_bytes(lens, num_q_heads: int, num_kv_heads: int, head_dim: int, block_size: int = 16,
                 kv_elem_bytes: int = 2) -> int:
    """Algorithmic bytes of one decode: K+V of every cached token once per KV
    head, q in and out, table entries, lengths."""
    lens = np.asarray(lens, dtype=np.int64)
    B = len(lens)
    kv = int(lens.sum()) * num_kv_heads * head_dim * kv_elem_bytes * 2
    qo = B * num_q_heads * head_dim * 2 * 2
    tables = int(((lens + block_size - 1) // block_size).sum()) * 4 + 4 * B
    return kv + qo + tables


def decode_bytes_fp8(lens, num_q_heads: int, num_kv_heads: int, head_dim: int,
                     block_size: int = 16) -> int:
    """Algorithmic bytes of one decode over the 8-bit cache: one byte per K/V
    element, bf16 q in and out, table entries, lengths."""
    return decode_bytes(lens, num_q_heads, num_kv_heads, head_dim, block_size, kv_elem_bytes=1)


def append_bytes(num_tokens: int, num_kv_heads: int, head_dim: int, cache_elem_bytes: int = 2) -> int:
    """KV write: read the new bf16 K/V rows, write them into the cache, read the slots."""
    return num_tokens * num_kv_heads * head_dim * 2 * (2 + cache_elem_bytes) + 8 * num_tokens


def cow_bytes(num_pairs: int, num_kv_heads: int, head_dim: int, block_size: int = 16,
              elem_bytes: int = 2) -> int:
    """Block copy: read and write a whole block of K and of V per pair."""
    return num_pairs * 2 * num_kv_heads * block_size * head_dim * elem_bytes * 2


def profiled_traffic(summary: str = "pa_decode_tc_llama70b_b32.md"):
    """DRAM bytes (read + write) of one decode launch from a committed ncu
    summary, or None when the kernel sources have changed since that capture
    (the summary records a sha256 prefix of each source file)."""
    import hashlib
    import re

    path = summary if os.path.isabs(summary) else os.path.join(ROOT, "profiles", summary)
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"traffic_bytes_per_launch:\s*(\d+)", text)
    h = re.search(r"source_sha256_prefix:\s*(.+)", text)
    if not m or not h:
        return None
    csrc = os.path.join(ROOT, "paged_kv_cache_92_gb300", "csrc")
    for item in h.group(1).split():
        name, want = item.split("=")
        with open(os.path.join(csrc, name), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest()[:len(want)] != want:
                return None
    return int(m.group(1))


def max_over_ranks(x: float, device, world: int) -> float:
    """The largest of every rank's x (all ranks call this; one rank returns x)."""
    if world <= 1:
        return float(x)
    import torch

    t = torch.tensor([float(x)], device=device, dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(step_bytes: int, steps: int, elapsed_ms: float, world: int) -> float:
    """Whole-job throughput of N replicas: every rank processes step_bytes per
    step, and the job takes the slowest rank's time."""
    return world * step_bytes * steps / (elapsed_ms * 1e-3) / 1e9


def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "source": "fallback"}


def host_threads() -> int:
    """Host threads the oracle runs on: OMP_NUM_THREADS when set, else every core."""
    try:
        n = int(os.environ.get("OMP_NUM_THREADS", "0"))
    except ValueError:
        n = 0
    return n if n > 0 else (os.cpu_count() or 1)


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return "unknown"


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while the GPU is loaded."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 50):
        self.proc = None
        self.path = None
        try:
            import tempfile

            fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", f"-lms={period_ms}"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r) if v == "Active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------------------- step plans

class StepPlan:
    """Pre-marshalled C-ABI calls for one step on one KV-pool copy: the
    copy-on-write copies (if any), then the KV write and the decode (one
    pa_append_decode call when fused). ``run(ev)`` brackets the decode call
    with the event pair ``ev``."""

    def __init__(self, lib, dec_params, ws_ptr, ws_bytes, stream, rc_args=None, cow_args=None,
                 append=None, fp8=False):
        self.lib = lib
        self.dec = dec_params
        self.ws_ptr, self.ws_bytes = ws_ptr, ws_bytes
        self.rc_args = rc_args
        self.cow_args = cow_args
        self.stream = stream
        self.append = append
        self.fp8 = fp8

    def run(self, ev_dec=None):
        lib = self.lib
        if self.cow_args is not None:
            copy = lib.pa_copy_blocks_fp8 if self.fp8 else lib.pa_copy_blocks
            st = copy(*self.cow_args, self.stream)
            if st:
                raise RuntimeError(f"copy_blocks failed: {st}: {lib.pa_last_error()}")
        if self.append is None and self.rc_args is not None:
            st = lib.pa_reshape_and_cache(*self.rc_args, self.stream)
            if st:
                raise RuntimeError(f"pa_reshape_and_cache failed: {st}")
        if ev_dec is not None:
            ev_dec[0].record()
        if self.append is None:
            st = lib.pa_decode(ctypes.byref(self.dec), self.ws_ptr, self.ws_bytes, self.stream)
        else:
            st = lib.pa_append_decode(ctypes.byref(self.dec), ctypes.byref(self.append),
                                      self.ws_ptr, self.ws_bytes, self.stream)
        if st:
            raise RuntimeError(f"decode failed: {st}: {lib.pa_last_error()}")
        if ev_dec is not None:
            ev_dec[1].record()


def setup_workload(r: workloads.Recipe, device, n_copies: int):
    import paged_kv_cache_92_gb300 as pk

    pool = pk.Pool(r.num_blocks, r.block_size, free_order=r.free_order)
    seqs = workloads.drive_prefill(pool, r)
    slots, cows = workloads.drive_step_append(pool, seqs, r)
    tables = workloads.tables_of(pool, seqs)
    lens = (r.lens0 + r.append).astype(np.int32)
    pool.close()
    q, kn, vn, kc, vc = workloads.step_tensors(r, str(device))
    copies = [(kc, vc)] + [(kc.clone(), vc.clone()) for _ in range(n_copies - 1)]
    return dict(tables=tables, lens=lens, slots=slots, cows=cows, q=q, kn=kn, vn=vn,
                copies=copies)


def n_copies_for(r: workloads.Recipe) -> int:
    """Pool copies to rotate: enough that consecutive steps never find their
    K/V in L2 (at least two, more while a copy is below 3x L2)."""
    kv = 2 * r.num_blocks * r.num_kv_heads * r.block_size * r.head_dim * 2
    return max(2, min(4, math.ceil(3 * L2_BYTES / max(kv, 1))))


def count_launches(variant: int, fused: bool, max_len: int, num_cow: int, fp8: bool = False,
                   query_len: int = 1) -> int:
    """Kernels one step launches: copy-on-write copy (if any pairs), the KV
    write (unless fused into the tensor-core decode), the 8-bit query split /
    multi-token query permute (when needed), the decode, the merge (always for
    the tensor-core kernel; for the CUDA-core kernel only when a sequence
    spans several 512-token partitions)."""
    n = 1 if num_cow else 0
    if variant == 0:
        n += (0 if fused else 1) + 2 + (1 if fp8 or query_len > 1 else 0)
    else:
        n += 1 + 1 + (1 if max_len > 512 else 0)
    return n


def make_plans(pk, W, device, partition_tokens=0, variant=0, overlap=True, fused=True):
    import torch

    lib = pk.load()
    stream = torch.cuda.current_stream().cuda_stream or None
    tables_d = torch.from_numpy(W["tables"]).to(device)
    lens_d = torch.from_numpy(W["lens"]).to(device)
    slots_d = torch.from_numpy(W["slots"]).to(device)
    cows_d = torch.from_numpy(W["cows"]).to(device) if len(W["cows"]) else None
    out = torch.empty_like(W["q"])
    keep = [tables_d, lens_d, slots_d, cows_d, out]
    plans = []
    ws = None
    for kc, vc in W["copies"]:
        p = pk.make_decode_params(W["q"], out, kc, vc, tables_d, lens_d,
                                  max_context_len=int(W["lens"].max()),
                                  partition_tokens=partition_tokens, variant=variant,
                                  overlap_prologue=overlap)
        need = pk.pa_decode_workspace_size(p)
        if ws is None and need:
            ws = torch.empty(need, dtype=torch.uint8, device=device)
            keep.append(ws)
        NB, Hkv, BS, D = kc.shape
        rc_args = (W["kn"].data_ptr(), W["vn"].data_ptr(), kc.data_ptr(), vc.data_ptr(),
                   slots_d.data_ptr(), W["kn"].shape[0], Hkv, D, BS, NB)
        cow_args = None
        if cows_d is not None:
            cow_args = (kc.data_ptr(), vc.data_ptr(), cows_d.data_ptr(), cows_d.shape[0], Hkv, D,
                        BS, NB)
        app = pk.make_append_params(W["kn"], W["vn"], slots_d, kc, vc) if fused else None
        plans.append(StepPlan(lib, p, ws.data_ptr() if ws is not None else None,
                              ws.numel() if ws is not None else 0, stream, rc_args=rc_args,
                              cow_args=cow_args, append=app))
    return plans, out, keep


# ----------------------------------------------------------------------------- timing

def time_loop(plans, steps: int, stream) -> float:
    """Milliseconds per step of ``steps`` back-to-back steps (rotating over the
    plans), one event pair around the whole loop and nothing in between."""
    import torch

    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record(stream)
    for k in range(steps):
        plans[k % len(plans)].run()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / steps


def time_launches(plans, n: int) -> float:
    """Mean milliseconds of the decode call (decode kernel + merge, with the
    fused KV write) bracketed by an event pair, over n steps."""
    import torch

    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n)]
    torch.cuda.synchronize()
    for k in range(n):
        plans[k % len(plans)].run(evs[k])
    torch.cuda.synchronize()
    return statistics.mean(a.elapsed_time(b) for a, b in evs)


# columns of one other_workloads row (a compact table: the bench line must fit
# the few thousand characters a log tail keeps)
ROW_COLS = ["config", "seqs", "step_bytes", "step_us", "step_gbs", "step_frac", "launch_us",
            "launch_frac"]


def entry(step_bytes: int, step_ms: float, launch_bytes: int, launch_ms: float, peak: float,
          config=None, seqs=None, hbm_fraction: bool = True) -> list:
    """One secondary workload's row (ROW_COLS): the plain step loop
    (``step_*``) and the bracketed decode call (``launch_*``; its bytes are the
    step's less any copy-on-write copies), GB/s of algorithmic bytes and
    fractions of the measured HBM peak (None where the bytes are logical, not
    HBM: the shared prefix is read from L2)."""
    sg = step_bytes / (step_ms * 1e-3) / 1e9
    lg = launch_bytes / (launch_ms * 1e-3) / 1e9
    return [config, seqs, int(step_bytes), round(step_ms * 1e3, 2), round(sg, 1),
            round(sg / peak, 4) if hbm_fraction else None,
            round(launch_ms * 1e3, 2), round(lg / peak, 4) if hbm_fraction else None]


# ----------------------------------------------------------------------------- our arm

def run_ours(args, rank: int, world: int) -> dict:
    import torch

    import paged_kv_cache_92_gb300 as pk

    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    pk.load()
    name = args.workload
    r = WORKLOADS[name][0]()
    W = setup_workload(r, device, n_copies=n_copies_for(r))
    fused = not args.separate_append
    plans, out, keep = make_plans(pk, W, device, variant=args.variant,
                                  overlap=not args.no_overlap, fused=fused)
    lens = W["lens"]
    H, D, BS = r.num_kv_heads, r.head_dim, r.block_size
    dec_b = decode_bytes(lens, r.num_q_heads, H, D, BS)
    app_b = append_bytes(len(W["slots"]), H, D)
    step_b = dec_b + app_b + cow_bytes(len(W["cows"]), H, D, BS)
    # bytes of the bracketed launch: the decode, plus the KV write when it is fused in
    roof_b = dec_b + (app_b if fused else 0)
    pool_copy_bytes = 2 * W["copies"][0][0].numel() * 2
    launches_per_step = count_launches(args.variant, fused, int(lens.max()), len(W["cows"]))

    stream = torch.cuda.current_stream()
    # warm-up (untimed), then a sustained untimed loop under the clock sampler
    for i in range(args.warmup):
        plans[i % len(plans)].run()
    torch.cuda.synchronize()
    sampler = ClockSampler(local_rank)
    t_sustain = time.time()
    i = 0
    while time.time() - t_sustain < args.sustain_s:
        for _ in range(16):
            plans[i % len(plans)].run()
            i += 1
        torch.cuda.synchronize()

    # the timed region: K plain steps, one event pair around them
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    start.record(stream)
    for k in range(args.steps):
        plans[k % len(plans)].run()
    stop.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    if world > 1:
        torch.distributed.barrier()
    elapsed_ms = max_over_ranks(start.elapsed_time(stop), device, world)
    ms_per_step = elapsed_ms / args.steps
    value = whole_job_gbs(step_b, args.steps, elapsed_ms, world)

    # the launch pass (after the timed region): the decode call bracketed by events
    n_launch = max(args.launch_samples, 2 * len(plans))
    dec_avg_ms = time_launches(plans, n_launch)
    peaks = measured_peaks()
    achieved = roof_b / (dec_avg_ms * 1e-3) / 1e9

    # end to end through the public API: pinned host inputs -> device, step,
    # result -> pinned host, every step
    e2e = run_e2e(pk, W, r, device, max(args.steps, args.e2e_steps), args.warmup, step_b,
                  args.variant)

    traffic = profiled_traffic(f"pa_decode_tc_{PROFILE_OF.get(name, name)}.md") \
        if args.variant == 0 and fused else None
    res = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) q/K/V and context lengths; no weights needed)",
        "pct_of_peak": round(100 * value / world / peaks["hbm_gbs"], 2),
        "pct_of_nominal_8tbs": round(100 * value / world / NOMINAL_HBM_GBS, 2),
        "steps_per_s": round(1000.0 / ms_per_step, 1),
        "config": {
            "workload": f"{name}: {WORKLOADS[name][1]}",
            "baseline_config": CONFIG_OF.get(name),
            "num_seqs": r.num_seqs, "num_q_heads": r.num_q_heads, "num_kv_heads": H,
            "head_dim": D, "block_size": BS, "total_context_tokens": int(lens.sum()),
            "algorithmic_bytes_per_step": step_b, "decode_bytes_per_step": dec_b,
            "l2": f"inputs larger than L2: {len(W['copies'])} rotating KV pool copies of "
                  f"{pool_copy_bytes / 1e6:.0f} MB each (L2 129 MB)",
            "timed_region": "plain step loop, one event pair around all steps",
            "parallelism": "replicas only" if world > 1 else "single GPU",
        },
        "roofline": {
            "bound": "hbm",
            "kernel": (("pa_append_decode: " if fused else "pa_decode: ")
                       + ("tensor-core" if args.variant == 0 else "CUDA-core")
                       + (" decode kernel with the KV write fused in" if fused else
                          " decode kernel") + " + split-K merge"),
            "bytes_per_launch": roof_b,
            "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": round(achieved / peaks["hbm_gbs"], 4),
            "frac_of_nominal_8tbs": round(achieved / NOMINAL_HBM_GBS, 4),
            "traffic": traffic,
            "peak_source": f"{peaks['source']} hbm_gbs (copy, burst)",
            "avg_launch_ms": round(dec_avg_ms, 5), "timed_launches": n_launch,
            "launch_timing": "separate pass after the timed region, each launch bracketed by "
                             "CUDA events on the launching stream",
        },
        "clocks": clocks,
        "gpu_launches": launches_per_step * args.steps,
        "e2e": e2e,
    }
    del plans, keep, W
    torch.cuda.empty_cache()
    other = None
    if not args.no_workloads:
        other = {"cols": ROW_COLS}
        other.update(measure_bf16_workloads(pk, device, variant=args.variant,
                                            overlap=not args.no_overlap, fused=fused,
                                            skip=(name,)))
        if args.variant == 0:
            other.update(measure_fp8_workloads(pk, device))
            other.update(measure_multi_workloads(pk, device))
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(name, budget_s=args.cpu_baseline_s)
    if other is not None:
        res["other_workloads"] = other  # last: the end of the line survives a log's tail
    return res


# ncu summaries by workload (profiles/pa_decode_tc_<suffix>.md)
PROFILE_OF = {"llama70b_long_b32": "llama70b_b32", "llama8b_layer_b64": "llama8b_b64",
              "shared_prefix_cow_b512": "shared_prefix_b512"}


def measure_bf16_workloads(pk, device, variant: int = 0, overlap: bool = True, fused: bool = True,
                           steps: int = 200, launches: int = 100, warmup: int = 10, only=None,
                           skip=()) -> dict:
    """The bf16 workloads other than the headline, measured after the main
    timed region. The shared-prefix batch re-reads its 64 shared blocks within
    a step from L2 by design, so its GB/s counts logical bytes and carries no
    HBM fraction (``dram_*`` from its ncu summary instead, when current)."""
    import torch

    out = {}
    peak = measured_peaks()["hbm_gbs"]
    stream = torch.cuda.current_stream()
    for name, (make, desc) in WORKLOADS.items():
        if name in skip or (only is not None and name != only):
            continue
        r = make()
        W = setup_workload(r, device, n_copies=n_copies_for(r))
        plans, _, keep = make_plans(pk, W, device, variant=variant, overlap=overlap, fused=fused)
        lens = W["lens"]
        H, D, BS = r.num_kv_heads, r.head_dim, r.block_size
        dec_b = decode_bytes(lens, r.num_q_heads, H, D, BS)
        app_b = append_bytes(len(W["slots"]), H, D)
        step_b = dec_b + app_b + cow_bytes(len(W["cows"]), H, D, BS)
        for i in range(warmup):
            plans[i % len(plans)].run()
        step_ms = time_loop(plans, steps, stream)
        launch_ms = time_launches(plans, launches)
        shared = name == "shared_prefix_cow_b512"
        out[name] = entry(step_b, step_ms, dec_b + (app_b if fused else 0), launch_ms, peak,
                          config=CONFIG_OF.get(name), seqs=r.num_seqs, hbm_fraction=not shared)
        if shared:
            # logical K/V bytes (the 64 shared blocks hit L2); the true DRAM
            # fraction from the launch's ncu DRAM bytes, while that summary is current
            dram = profiled_traffic(f"pa_decode_tc_{PROFILE_OF[name]}.md") if fused else None
            out["shared_prefix_dram_frac"] = (round(dram / (launch_ms * 1e-3) / 1e9 / peak, 4)
                                              if dram else None)
        del plans, keep, W
        torch.cuda.empty_cache()
    return out


def measure_fp8_workloads(pk, device, steps: int = 200, launches: int = 100, warmup: int = 10,
                          only=None) -> dict:
    """The same workloads on the 8-bit (E4M3) cache: each bf16 pool copy is
    quantised into an E4M3 pool (per-KV-head scales 0.05 for K and V) through
    pa_reshape_and_cache_fp8, then the step (quantising KV write in the
    decode's preparation launch) is timed like the bf16 runs; the launch is
    the pa_append_decode call (query split + write, decode, merge)."""
    import torch

    lib = pk.load()
    out = {}
    recipes = [("llama8b_layer_b64_fp8_e4m3", workloads.llama8b_layer()),
               ("llama8b_high_concurrency_b256_fp8_e4m3", workloads.llama8b_high_concurrency()),
               ("llama70b_long_b8_fp8_e4m3", workloads.llama70b_long(batch=8)),
               ("llama70b_long_b32_fp8_e4m3", workloads.llama70b_long(batch=32)),
               ("llama8b_layer_b64_bs32_fp8_e4m3", workloads.llama8b_layer(block_size=32))]
    peak = measured_peaks()["hbm_gbs"]
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream or None
    for name, r in recipes:
        if only is not None and name != only:
            continue
        W = setup_workload(r, device, n_copies=2)
        H, D = r.num_kv_heads, r.head_dim
        ks = torch.full((H,), 0.05, dtype=torch.float32, device=device)
        vs = torch.full((H,), 0.05, dtype=torch.float32, device=device)
        tables_d = torch.from_numpy(W["tables"]).to(device)
        lens_d = torch.from_numpy(W["lens"]).to(device)
        slots_d = torch.from_numpy(W["slots"]).to(device)
        cows_d = torch.from_numpy(W["cows"]).to(device) if len(W["cows"]) else None
        outb = torch.empty_like(W["q"])
        keep, plans = [ks, vs, tables_d, lens_d, slots_d, cows_d, outb], []
        copies = W.pop("copies")
        while copies:
            kc, vc = copies.pop(0)
            NB, BS = kc.shape[0], kc.shape[2]
            k8 = torch.empty((NB, H, BS, D), dtype=torch.uint8, device=device)
            v8 = torch.empty((NB, H, BS // 16, D, 16), dtype=torch.uint8, device=device)
            rows = torch.arange(NB * BS, dtype=torch.int64, device=device)
            pk.pa_reshape_and_cache_fp8(kc.permute(0, 2, 1, 3).reshape(NB * BS, H, D).contiguous(),
                                        vc.permute(0, 2, 1, 3).reshape(NB * BS, H, D).contiguous(),
                                        k8, v8, rows, ks, vs)
            del kc, vc, rows
            torch.cuda.empty_cache()
            p = pk.make_decode_params(W["q"], outb, k8, v8, tables_d, lens_d,
                                      max_context_len=int(W["lens"].max()), k_scale=ks, v_scale=vs,
                                      overlap_prologue=True)
            ws = torch.empty(pk.pa_decode_workspace_size(p), dtype=torch.uint8, device=device)
            app = pk.make_append_params(W["kn"], W["vn"], slots_d, k8, v8)
            cow_args = None if cows_d is None else (k8.data_ptr(), v8.data_ptr(),
                                                     cows_d.data_ptr(), cows_d.shape[0], H, D,
                                                     BS, NB)
            plans.append(StepPlan(lib, p, ws.data_ptr(), ws.numel(), sh, cow_args=cow_args,
                                  append=app, fp8=True))
            keep += [k8, v8, ws]
        lens = W["lens"]
        dec_b = decode_bytes_fp8(lens, r.num_q_heads, H, D, r.block_size)
        app_b = append_bytes(len(W["slots"]), H, D, cache_elem_bytes=1)
        step_b = dec_b + app_b + cow_bytes(len(W["cows"]), H, D, r.block_size, elem_bytes=1)
        for i in range(warmup):
            plans[i % len(plans)].run()
        step_ms = time_loop(plans, steps, stream)
        launch_ms = time_launches(plans, launches)
        out[name] = entry(step_b, step_ms, dec_b + app_b, launch_ms, peak, seqs=r.num_seqs)
        del plans, keep, W
        torch.cuda.empty_cache()
    return out


def measure_multi_workloads(pk, device, steps: int = 200, launches: int = 100, warmup: int = 10,
                            only=None) -> dict:
    """Q new tokens per sequence (query_len Q, causal among them), the KV write
    of all of them fused into the decode: the bf16 caches of the workloads
    above, each sequence's last Q tokens being the new ones. Algorithmic
    bytes: the decode's (K/V once per KV head, tables) with Q rows of q and
    out per sequence, plus the new tokens' K/V written."""
    import torch

    lib = pk.load()
    out = {}
    cases = [("llama8b_layer_b64_q2", workloads.llama8b_layer(), 2),
             ("llama8b_layer_b64_q4", workloads.llama8b_layer(), 4),
             # more tokens than one column group holds: groups of 4 (G 4) or 2 (G 8)
             ("llama8b_layer_b64_q8", workloads.llama8b_layer(), 8),
             ("llama8b_layer_b64_q16", workloads.llama8b_layer(), 16),
             ("llama8b_layer_b64_q64", workloads.llama8b_layer(), 64),
             ("llama70b_long_b8_q8", workloads.llama70b_long(batch=8), 8),
             ("llama8b_high_concurrency_b256_q4", workloads.llama8b_high_concurrency(), 4),
             ("llama70b_long_b8_q2", workloads.llama70b_long(batch=8), 2),
             ("llama8b_layer_b64_bs32_q8", workloads.llama8b_layer(block_size=32), 8)]
    peak = measured_peaks()["hbm_gbs"]
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream or None
    for name, r, Q in cases:
        if only is not None and name != only:
            continue
        W = setup_workload(r, device, n_copies=2)
        H, D, Hq = r.num_kv_heads, r.head_dim, r.num_q_heads
        lens, tables = W["lens"], W["tables"]
        B = len(lens)
        pos = (lens[:, None] - Q + np.arange(Q)[None, :]).reshape(-1)
        seq = np.repeat(np.arange(B), Q)
        bs = r.block_size
        slots = (tables[seq, pos // bs].astype(np.int64) * bs + pos % bs).astype(np.int64)
        g = torch.Generator(device="cpu").manual_seed(7)
        q = torch.randn(B, Q, Hq, D, generator=g).to(torch.bfloat16).to(device)
        kn = torch.randn(B * Q, H, D, generator=g).to(torch.bfloat16).to(device)
        vn = torch.randn(B * Q, H, D, generator=g).to(torch.bfloat16).to(device)
        tables_d = torch.from_numpy(tables).to(device)
        lens_d = torch.from_numpy(lens).to(device)
        slots_d = torch.from_numpy(slots).to(device)
        o = torch.empty_like(q)
        keep, plans = [q, kn, vn, tables_d, lens_d, slots_d, o], []
        for kc, vc in W["copies"]:
            p = pk.make_decode_params(q, o, kc, vc, tables_d, lens_d,
                                      max_context_len=int(lens.max()), overlap_prologue=True)
            a = pk.make_append_params(kn, vn, slots_d, kc, vc)
            ws = torch.empty(pk.pa_decode_workspace_size(p), dtype=torch.uint8, device=device)
            plans.append(StepPlan(lib, p, ws.data_ptr(), ws.numel(), sh, append=a))
            keep.append(ws)
        dec_b = decode_bytes(lens, Hq, H, D) + B * (Q - 1) * Hq * D * 2 * 2
        step_b = dec_b + append_bytes(B * Q, H, D)
        for i in range(warmup):
            plans[i % len(plans)].run()
        step_ms = time_loop(plans, steps, stream)
        launch_ms = time_launches(plans, launches)
        out[name] = entry(step_b, step_ms, step_b, launch_ms, peak, seqs=B)
        del plans, keep, W
        torch.cuda.empty_cache()
    return out


def run_e2e(pk, W, r, device, steps: int, warmup: int, step_b: int, variant: int = 0) -> dict:
    """The same step end to end through ``pa_step_host``: each step is one C
    call that copies the packed inputs (q, new K/V, slots, tables, lengths,
    copy-on-write pairs) from pinned host memory to the device, runs the
    step, returns the output to pinned host memory and synchronises. Both
    buffers are pinned, so a kernel reads the inputs over the host link and
    the decode writes the output rows into host memory (no DMA copies)."""
    import torch

    lib = pk.load()
    B, Hq, D = W["q"].shape
    params = []
    host_in = None
    for kc, vc in W["copies"]:
        p = pk.make_step_host_params(kc, vc, B, Hq, W["tables"].shape[1], int(W["lens"].max()),
                                     num_cow_pairs=len(W["cows"]), variant=variant)
        if host_in is None:
            host_in = pk.pack_step_inputs(p, W["q"].cpu(), W["kn"].cpu(), W["vn"].cpu(),
                                          W["slots"], W["tables"], W["lens"],
                                          W["cows"] if len(W["cows"]) else None)
        params.append(p)
    host_out = torch.empty((B, Hq, D), dtype=torch.bfloat16).pin_memory()
    for p in params:
        p.host_in, p.host_out = host_in.data_ptr(), host_out.data_ptr()
    ws = torch.empty(pk.pa_step_host_workspace_size(params[0]), dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream().cuda_stream or None
    refs = [ctypes.byref(p) for p in params]

    def step(i):
        st = lib.pa_step_host(refs[i % len(refs)], ws.data_ptr(), ws.numel(), stream)
        if st:
            raise RuntimeError(f"pa_step_host failed: {st}: {lib.pa_last_error()}")

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    marks = [0.0] * (steps + 1)
    marks[0] = time.perf_counter()
    for i in range(steps):
        step(i)  # returns once the output is in host memory
        marks[i + 1] = time.perf_counter()
    dt = marks[-1] - marks[0]
    per_step = sorted(marks[i + 1] - marks[i] for i in range(steps))
    return {"value": round(step_b * steps / dt / 1e9, 2), "unit": UNIT,
            "h2d_bytes_per_step": int(host_in.numel()), "d2h_bytes_per_step": int(host_out.numel() * 2),
            "steps": steps, "ms_per_step": round(dt / steps * 1e3, 4),
            "ms_per_step_median": round(per_step[steps // 2] * 1e3, 4),
            "ms_per_step_max": round(per_step[-1] * 1e3, 4),
            "api": "pa_step_host (one C call per step: a kernel stages the packed inputs from "
                   "pinned host memory over the host link, copy-on-write, fused KV write + decode "
                   "+ merge writing the output rows into pinned host memory, stream sync)"}


# ----------------------------------------------------------------------------- CPU oracle

def _oracle_sample_inputs(r: workloads.Recipe):
    """Host layout and contents for the oracle (its own pool model)."""
    import oracle

    model = oracle.PoolModel(r.num_blocks, r.block_size, free_order=r.free_order)
    seqs = workloads.drive_prefill(model, r)
    workloads.drive_step_append(model, seqs, r)
    tables = workloads.tables_of(model, seqs)
    lens = (r.lens0 + r.append).astype(np.int32)
    q, kn, vn, kc, vc = workloads.step_tensors(r, "cpu")
    return tables, lens, q, kc, vc


# sequences of each workload in the oracle's bounded sample
CPU_SAMPLE_SEQS = {"llama70b_long_b32": 4, "llama70b_long_b8": 4, "llama8b_layer_b64": 16,
                   "llama8b_high_concurrency_b256": 16}


def time_oracle(r: workloads.Recipe, inputs, threads: int, budget_s: float):
    """The float64 oracle on ``threads`` host threads over the sample's
    (sequence, query head) units, cycling through the sample, until the time
    budget is spent (at least one call). Returns (GB/s, units done, seconds)."""
    import oracle

    tables, lens, qb, kb, vb = inputs
    B, Hq = len(lens), r.num_q_heads
    # a call's units: whole sequences when every thread gets work, else a
    # thread's worth of query heads
    per_call = Hq if threads > 1 else max(1, Hq // 8)
    oracle.set_num_threads(threads)
    done_bytes, n_units, k = 0, 0, 0
    per_unit = [decode_bytes(lens[b:b + 1], Hq, r.num_kv_heads, r.head_dim, r.block_size) / Hq
                for b in range(B)]
    t0 = time.perf_counter()
    while n_units == 0 or time.perf_counter() - t0 < budget_s:
        b, h0 = (k * per_call) // Hq % B, (k * per_call) % Hq
        units = [(b, h) for h in range(h0, min(Hq, h0 + per_call))]
        oracle.paged_decode(qb, kb, vb, tables, lens, units=units)
        done_bytes += per_unit[b] * len(units)
        n_units += len(units)
        k += 1
    dt = time.perf_counter() - t0
    return done_bytes / dt / 1e9, n_units, dt


def cpu_baseline(headline: str, budget_s: float = 2.5) -> dict:
    """The float64 C oracle on this host's cores: the headline workload and
    the 8B-class layer (64 and 256 sequences) and the 70B-class batch of 8,
    each at all host threads and at one thread. Each runs on a bounded sample
    of its workload (its first few sequences, same lengths and geometry, on a
    pool of their own) for about ``budget_s`` seconds. GB/s of algorithmic
    decode bytes."""
    import oracle

    nproc = host_threads()
    names = [headline] + [n for n in ("llama8b_layer_b64", "llama8b_high_concurrency_b256",
                                      "llama70b_long_b8") if n != headline]
    per = {}
    head = None
    for name in names:
        r = WORKLOADS[name][0]()
        k = min(r.num_seqs, CPU_SAMPLE_SEQS.get(name, 8))
        sub = workloads.subset(r, list(range(k)))
        tables, lens, q, kc, vc = _oracle_sample_inputs(sub)
        inputs = (tables, lens, oracle.bf16_bits(q), oracle.bf16_bits(kc), oracle.bf16_bits(vc))
        res = [CONFIG_OF.get(name), k]
        for threads in (nproc, 1):
            gbs, n_units, dt = time_oracle(sub, inputs, threads, budget_s)
            res.append(round(gbs, 4))
            if name == headline and threads == nproc:
                head = (gbs, n_units, dt, k)
        per[name] = res
        del inputs, q, kc, vc
    oracle.set_num_threads(nproc)
    gbs, n_units, dt, k = head
    return {"value": round(gbs, 4), "unit": UNIT, "cores": nproc, "kind": "oracle",
            "cpu_model": cpu_model(),
            "sample": f"float64 C oracle (OpenMP over (sequence, query head) units) on the first "
                      f"{k} sequences of {headline} (same lengths and geometry, own pool): "
                      f"{n_units} units in {dt:.1f} s on {nproc} threads",
            "per_config_cols": ["config", "sample_seqs", f"gbs_{nproc}_threads", "gbs_1_thread"],
            "per_config": per}


def run_reference(args) -> dict:
    import oracle

    name = args.workload
    r = WORKLOADS[name][0]()
    k = min(r.num_seqs, CPU_SAMPLE_SEQS.get(name, 8))
    sub = workloads.subset(r, list(range(k)))
    tables, lens, q, kc, vc = _oracle_sample_inputs(sub)
    qb, kb, vb = oracle.bf16_bits(q), oracle.bf16_bits(kc), oracle.bf16_bits(vc)
    oracle.set_num_threads(host_threads())
    Hq = r.num_q_heads

    def step(i):  # one whole sequence (all query heads) per step
        b = i % k
        oracle.paged_decode(qb, kb, vb, tables, lens, units=[(b, h) for h in range(Hq)])
        return decode_bytes(lens[b:b + 1], Hq, r.num_kv_heads, r.head_dim, r.block_size)

    for i in range(args.warmup):
        step(i)
    total = 0
    t0 = time.perf_counter()
    for i in range(args.steps):
        total += step(args.warmup + i)
    dt = time.perf_counter() - t0
    value = total / dt / 1e9
    sample = (f"each step: float64 C oracle decode of one whole sequence (all {Hq} query heads) "
              f"of {name}, cycling through its first {k} sequences (same lengths and geometry, "
              f"own pool)")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3 / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) q/K/V and context lengths)",
        "config": {"workload": f"{name} (sampled): {WORKLOADS[name][1]}",
                   "num_seqs": r.num_seqs, "num_q_heads": Hq, "num_kv_heads": r.num_kv_heads,
                   "head_dim": r.head_dim, "block_size": r.block_size},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample, "cpu_model": cpu_model()},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


# ----------------------------------------------------------------------------- main

def run_case(args) -> int:
    """One secondary workload alone, on cuda:0."""
    import torch

    import paged_kv_cache_92_gb300 as pk

    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    pk.load()
    kw = dict(steps=args.steps, warmup=args.warmup, only=args.case)
    res = measure_bf16_workloads(pk, device, variant=args.variant, **kw)
    if args.variant == 0:
        res.update(measure_fp8_workloads(pk, device, **kw))
        res.update(measure_multi_workloads(pk, device, **kw))
    if not res:
        print(json.dumps({"case": args.case, "error": "no such workload"}))
        return 2
    print(json.dumps({"case": args.case, **dict(zip(ROW_COLS, res[args.case]))}))
    return 0


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=HEADLINE,
                    help="the workload of the headline line (default: the largest "
                         "single-GPU configuration)")
    ap.add_argument("--e2e-steps", type=int, default=200,
                    help="end-to-end steps (at least --steps): one host hiccup in a short loop "
                         "would otherwise move the mean")
    ap.add_argument("--sustain-s", type=float, default=1.0,
                    help="untimed loaded seconds before the timed region (clock sampling)")
    ap.add_argument("--launch-samples", type=int, default=50,
                    help="bracketed decode calls in the launch pass after the timed region")
    ap.add_argument("--cpu-baseline-s", type=float, default=2.5,
                    help="seconds of oracle work per (workload, thread count) sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the measurements on the other workload shapes")
    ap.add_argument("--separate-append", action="store_true",
                    help="launch the KV write as its own kernel instead of fusing it into the "
                         "decode (pa_reshape_and_cache + pa_decode)")
    ap.add_argument("--no-overlap", action="store_true",
                    help="launch the decode in plain stream order instead of overlapping its "
                         "set-up with the previous kernel")
    ap.add_argument("--variant", type=int, default=0, choices=[0, 1],
                    help="decode kernel: 0 tensor-core (default), 1 CUDA-core")
    ap.add_argument("--case", default=None,
                    help="run only this entry of other_workloads (e.g. "
                         "llama8b_layer_b64_fp8_e4m3) for --steps steps after --warmup, and "
                         "print its figures (for profiling one kernel; not the bench line)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args)))
        return 0

    if args.case is not None:
        return run_case(args)
    if world > 1:
        import torch

        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        torch.distributed.init_process_group("nccl")
    res = run_ours(args, rank, world)
    if rank == 0:
        print(json.dumps(res))
    if world > 1:
        import torch

        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
