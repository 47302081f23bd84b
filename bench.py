#!/usr/bin/env python3
"""Benchmark: CP prefill causal TFLOP/s on one GB300 (both ring schedules).

One step = one layer's CP prefill with Pass-KV followed by the same layer with
Pass-Q, on the 128K-token workload (batch 1, 16 q heads, 1 kv head, head_dim
128, 16 CP chunks of 8192, causal, bf16).  value = causal-effective FLOPs of
the step / device time.  Inputs are resident in HBM before the timed region;
Q and O (512 MiB each) are larger than L2, so no L2 flush is inserted.

Also reported: ms per layer of each schedule at 128K and at 1M tokens, the
roofline of the dominant kernel (live CUDA-event timing of every launch), the
end-to-end number through the host-buffer entry point, and the fp64 CPU
oracle timed on a bounded sample of rows (baseline only).

--impl reference times that oracle as the reference arm (CPU, rank 0 only).
Multi-GPU: "replicas only" -- each rank runs the whole step on its own GPU
with no data-path collective (weak scaling); value sums all ranks' FLOPs over
the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "CP prefill causal TFLOP/s & % of GB300 BF16 peak; ms/layer at 128K and 1M tokens"
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}

# DRAM bytes (read + write) per tensor FLOP of each instance of the prefill
# attention kernel (profiler kind) from one ncu capture, and the kernel source
# it was taken from; the roofline's traffic is null whenever the source
# differs from the capture or a timed launch has no record.
TRAFFIC_RECORD = {
    "attn_tc": {"sha": "4247d6041a1fae0a", "bytes_per_flop": 52.07e6 / 5.498e11,
                "capture": "profiles/attn_pair_32k_step.md"},
    "attn_tc_onchip": {"sha": "4247d6041a1fae0a", "bytes_per_flop": 1.7117e9 / 7.0369e13,
                       "capture": "profiles/attn_pair_onchip_128k_passkv.md"},
}
ATTN_KINDS = ("attn_tc", "attn_tc_onchip")


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        out = {}
        for key in ("bf16_tflops", "bf16_tflops_sustained", "hbm_gbs"):
            val = d.get(key)
            if isinstance(val, dict):
                val = val.get("value")
            if val is not None:
                out[key] = float(val)
        if "bf16_tflops" in out:
            return out, "measured"
    except (OSError, ValueError):
        pass
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_sha():
    p = os.path.join(ROOT, "context_ring_attention_cpattn_gb300", "csrc", "attn_pair.cu")
    with open(p, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
              "clocks_event_reasons.sw_power_cap"]

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) != len(self.FIELDS):
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
                power.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[3:]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "power_w_median": statistics.median(power), "samples": len(sm),
                "reasons": sorted(reasons)}


def dist_setup():
    import torch

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------- oracle legs
def oracle_sample(w, n_rows, seed=7):
    """Time the fp64 oracle on n_rows seeded query rows of workload w (host cores)."""
    import numpy as np

    import oracle
    from context_ring_attention_cpattn_gb300.workloads import make_qkv

    rng = np.random.default_rng(seed)
    rows = np.sort(rng.choice(w.sq, size=n_rows, replace=False))
    q, k, v = make_qkv(w, device="cpu")
    qs = q[:, rows].float().numpy()
    kh, vh = k.float().numpy(), v.float().numpy()
    threads = oracle.default_threads()
    oracle.build()
    t0 = time.perf_counter()
    oracle.attention(qs, kh, vh, q_pos=w.q_base + rows, causal=w.causal, threads=threads)
    dt = time.perf_counter() - t0
    pos = w.q_base + rows
    vis = np.minimum(pos + 1, w.skv).clip(min=0).sum() if w.causal else n_rows * w.skv
    flops = 4.0 * w.head_dim * w.hq * w.batch * float(vis)
    return flops, dt, threads, rows


def run_reference(args, w):
    world, rank, _ = int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")), 0
    if rank != 0:
        return 0
    n_rows = args.ref_rows
    for _ in range(args.warmup):
        oracle_sample(w, n_rows)
    tot_f, tot_t, threads = 0.0, 0.0, 1
    for s in range(args.steps):
        f, dt, threads, _ = oracle_sample(w, n_rows, seed=100 + s)
        tot_f += f
        tot_t += dt
    value = tot_f / tot_t / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * tot_t / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "hq": w.hq, "hkv": w.hkv,
                   "head_dim": w.head_dim, "seq_len": w.sq, "n_chunks": w.n_chunks},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": f"{n_rows} seeded query rows x {w.hq} heads of the {w.name} "
                                   f"workload per step, full causal key range"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------- GPU arm
def time_modes(B, w, q, k, v, outs, wss, steps, warmup, world, modes, profile_cap=0, launch=0):
    """Warm up, then time `steps` steps, each running the given schedules in
    order.  Returns the elapsed ms (max over ranks), per-schedule ms lists and
    profile records."""
    import torch

    def one(mode):
        o, lse = outs[mode]
        B.prefill(q, k, v, w.n_chunks, mode, q_base=w.q_base, causal=w.causal, out=o, lse=lse,
                  workspace=wss[mode], launch=launch)

    for _ in range(warmup):
        for m in modes:
            one(m)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(modes) + 1)]
          for _ in range(steps)]
    if profile_cap:
        B.profile_begin(profile_cap)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for s in range(steps):
        ev[s][0].record(stream)
        for x, m in enumerate(modes):
            one(m)
            ev[s][x + 1].record(stream)
    end.record(stream)
    end.synchronize()
    recs = B.profile_end(profile_cap) if profile_cap else []
    torch.cuda.synchronize()
    barrier(world)
    elapsed = start.elapsed_time(end)
    per_mode = {m: [ev[s][x].elapsed_time(ev[s][x + 1]) for s in range(steps)]
                for x, m in enumerate(modes)}
    return max_over_ranks(elapsed, world), per_mode, recs


def time_merge2(B, w, hbm_peak, peak_src, reps=5):
    """Pairwise in-place LSE merge (cpattn_merge) of two fp32 partials of the
    workload's shape; algorithmic bytes = read both sides + write one."""
    import torch

    shape = (w.batch, w.sq, w.hq, w.head_dim)
    g = torch.Generator(device="cuda")
    g.manual_seed(11)
    oa = torch.randn(shape, generator=g, device="cuda")
    ob = torch.randn(shape, generator=g, device="cuda")
    la = torch.randn((w.batch, w.hq, w.sq), generator=g, device="cuda")
    lb = torch.randn((w.batch, w.hq, w.sq), generator=g, device="cuda")
    for _ in range(2):
        B.merge_(oa, la, ob, lb)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        B.merge_(oa, la, ob, lb)
    e1.record()
    e1.synchronize()
    ms = e0.elapsed_time(e1) / reps
    nbytes = 3.0 * w.batch * w.sq * w.hq * (w.head_dim * 4 + 4)
    gbs = nbytes / (ms * 1e-3) / 1e9
    del oa, ob, la, lb
    torch.cuda.empty_cache()
    return {"bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s", "frac": gbs / hbm_peak,
            "frac_of_8TBs": gbs / 8000.0, "ms": ms, "bytes_per_launch": nbytes,
            "shape": "fp32 [%d, %d, %d, %d] both sides" % shape, "peak_source": f"{peak_src} HBM copy"}


def time_decode(B, steps, hbm_peak, peak_src, name="decode-128k-b8"):
    """Pass-Q decode (cpattn_decode) of one token per sequence against a
    CP-sharded cache: HBM-bound; algorithmic bytes = visible K and V + Q + O,
    plus the fp32 partials written and re-read by the merge."""
    import torch

    from context_ring_attention_cpattn_gb300.workloads import WORKLOADS, make_qkv

    w = WORKLOADS[name]
    q, k, v = make_qkv(w, device="cuda")
    out = torch.empty_like(q)
    lse = torch.empty((w.batch, w.hq, w.sq), dtype=torch.float32, device="cuda")
    need = B.decode_workspace_size(q, k, w.n_chunks, w.q_base, w.causal)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")

    def run():
        B.decode(q, k, v, w.n_chunks, q_base=w.q_base, causal=w.causal, out=out, lse=lse,
                 workspace=ws)

    for _ in range(5):
        run()
    torch.cuda.synchronize()
    n = max(20, steps * 4)
    # Flush L2 between calls so each one streams the cache from HBM (K/V are
    # 512 MiB in total, larger than L2, but the tail of one call is still
    # resident at the start of the next): write 256 MiB, then read another
    # 256 MiB so that the written lines are back in HBM before the timed call
    # starts (their write-back would otherwise compete with the call).
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    clean = torch.ones(256 << 20, dtype=torch.uint8, device="cuda")
    B.profile_begin(4 * n)
    evs = []
    for _ in range(n):
        flush.zero_()
        clean.max()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        run()
        e1.record()
        evs.append((e0, e1))
    torch.cuda.synchronize()
    recs = B.profile_end(4 * n)
    ms = statistics.median(a.elapsed_time(b) for a, b in evs)
    vis = min(w.q_base + w.sq, w.skv)
    kv_bytes = 2.0 * w.batch * vis * w.hkv * w.head_dim * 2
    part_bytes = need  # fp32 partials: written once, read once
    qo_bytes = 2.0 * w.batch * w.sq * w.hq * w.head_dim * 2
    total = kv_bytes + 2.0 * part_bytes + qo_bytes
    attn = [r for r in recs if r[0] == "attn_tc"]
    attn_ms = statistics.median(r[1] for r in attn) if attn else None
    del q, k, v, out, ws, flush, clean
    torch.cuda.empty_cache()
    return {"workload": name, "ms_per_call": ms, "tokens_per_s": w.batch * w.sq / (ms * 1e-3),
            "achieved": total / (ms * 1e-3) / 1e9, "unit": "GB/s", "peak": hbm_peak,
            "frac": total / (ms * 1e-3) / 1e9 / hbm_peak, "bytes_per_call": total,
            "attn_kernel": {"ms": attn_ms, "kv_GBs": (kv_bytes / (attn_ms * 1e-3) / 1e9) if attn_ms else None,
                            "frac": (kv_bytes / (attn_ms * 1e-3) / 1e9 / hbm_peak) if attn_ms else None},
            "l2": "256 MiB written, then 256 MiB read, between calls (L2 flush)", "peak_source": f"{peak_src} HBM copy"}


def make_buffers(B, w, q, k, modes, launch=0):
    import torch

    outs, wss = {}, {}
    for mode in modes:
        outs[mode] = (torch.empty_like(q),
                      torch.empty((w.batch, w.hq, w.sq), dtype=torch.float32, device=q.device))
        n = B.workspace_size(q, k, w.n_chunks, mode, w.q_base, w.causal, launch=launch)
        wss[mode] = torch.empty(max(n, 256), dtype=torch.uint8, device=q.device)
    return outs, wss


def custom_workload(base, args):
    """The named workload with any command-line shape overrides applied."""
    import dataclasses

    fields = {"sq": args.seq, "skv": args.kv_seq if args.kv_seq is not None else args.seq,
              "n_chunks": args.chunks, "hq": args.hq, "hkv": args.hkv, "head_dim": args.head_dim,
              "dtype": args.dtype, "batch": args.batch, "q_base": args.q_base}
    fields = {k: v for k, v in fields.items() if v is not None}
    if args.no_causal:
        fields["causal"] = False
    if not fields:
        return base
    w = dataclasses.replace(base, **fields)
    tag = ",".join(f"{k}={v}" for k, v in sorted(fields.items()))
    return dataclasses.replace(w, name=f"{base.name}[{tag}]")


def seeds_of(args):
    return (args.seed, args.seed + 1, args.seed + 2)


LAUNCH_NAMES = {0: "one launch per ring step", 1: "persistent CTAs per ring step",
                2: "one persistent launch for all ring steps",
                4: "one persistent launch for all ring steps, on-chip Pass-KV accumulator"}


def launch_modes(B, w, q, k, modes, launch):
    """The launch mode each schedule resolves to (AUTO depends on the schedule)."""
    names = {B.PASS_KV: "pass_kv", B.PASS_Q: "pass_q"}
    pre = "auto: " if launch == B.LAUNCH_AUTO else ""
    return {names[m]: pre + LAUNCH_NAMES[B.launch_mode(q, k, w.n_chunks, m, w.q_base, w.causal,
                                                        launch=launch)] for m in modes}


def time_workload(B, name, steps, warmup, world, modes, launch, peaks):
    """ms per layer (median) of each schedule on a named workload, with its
    causal-effective TFLOP/s and fraction of the bf16 peaks."""
    import torch

    from context_ring_attention_cpattn_gb300.workloads import WORKLOADS, make_qkv

    w = WORKLOADS[name]
    q, k, v = make_qkv(w, device="cuda")
    outs, wss = make_buffers(B, w, q, k, modes, launch)
    _, pm, _ = time_modes(B, w, q, k, v, outs, wss, steps, warmup, world, modes, launch=launch)
    names = {B.PASS_KV: "pass_kv", B.PASS_Q: "pass_q"}
    f = w.causal_flops()
    out = {"flops_per_layer": f, "steps": steps, "warmup": warmup,
           "launch_mode": launch_modes(B, w, q, k, modes, launch), "dtype": w.dtype}
    for m in modes:
        ms = statistics.median(pm[m])
        tf = f / (ms * 1e-3) / 1e12
        out[names[m]] = {"ms_per_layer": ms, "tflops": tf,
                         "frac_of_bf16_burst": tf / peaks["bf16_tflops"],
                         "frac_of_bf16_sustained": tf / peaks.get("bf16_tflops_sustained",
                                                                  peaks["bf16_tflops"])}
    del q, k, v, outs, wss
    torch.cuda.empty_cache()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="128k")
    ap.add_argument("--skip-1m", action="store_true", help="do not time the 1M-token layer")
    ap.add_argument("--skip-e2e", action="store_true")
    ap.add_argument("--skip-decode", action="store_true", help="do not time the decode leg")
    ap.add_argument("--launch", type=int, default=None, choices=[0, 1, 2, 3, 4],
                    help="ring launch mode: 0 per step, 1 persistent per step, 2 one launch, "
                         "3 auto (the library default), 4 one launch with an on-chip Pass-KV "
                         "accumulator")
    ap.add_argument("--schedules", default="both", choices=["both", "kv", "q"],
                    help="ring schedules in one step (default: Pass-KV then Pass-Q)")
    ap.add_argument("--cpu-rows", type=int, default=2048,
                    help="oracle rows for cpu_baseline (0 skips it)")
    ap.add_argument("--ref-rows", type=int, default=256, help="oracle rows per reference step")
    ap.add_argument("--skip-per-workload", action="store_true",
                    help="do not time the other configurations (tiny, Llama-3-8B, partial 32K, 1M)")
    # Shape overrides of the main workload (any of them makes a custom workload).
    ov = ap.add_argument_group("workload overrides")
    ov.add_argument("--seq", type=int, help="query rows")
    ov.add_argument("--kv-seq", type=int, help="key/value rows (default: --seq)")
    ov.add_argument("--chunks", type=int, help="CP chunks (ranks)")
    ov.add_argument("--hq", type=int, help="query heads")
    ov.add_argument("--hkv", type=int, help="key/value heads")
    ov.add_argument("--head-dim", type=int, choices=[64, 128])
    ov.add_argument("--dtype", choices=["bf16", "fp32"])
    ov.add_argument("--batch", type=int)
    ov.add_argument("--q-base", type=int, help="absolute position of query row 0")
    ov.add_argument("--no-causal", action="store_true")
    ov.add_argument("--seed", type=int, default=1, help="Q/K/V seeds are seed, seed+1, seed+2")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        print("note: warmup raised to 3 (timing rule)", file=sys.stderr)
        args.warmup = 3

    from context_ring_attention_cpattn_gb300.workloads import WORKLOADS

    w = custom_workload(WORKLOADS[args.workload], args)
    if args.impl == "reference":
        return run_reference(args, w)

    import torch

    world, rank, local = dist_setup()
    from context_ring_attention_cpattn_gb300 import binding as B
    from context_ring_attention_cpattn_gb300 import build as pkg_build
    from context_ring_attention_cpattn_gb300.workloads import make_qkv

    if rank == 0 or world == 1:
        pkg_build.build()
    barrier(world)
    B.lib()

    modes = {"both": (B.PASS_KV, B.PASS_Q), "kv": (B.PASS_KV,), "q": (B.PASS_Q,)}[args.schedules]
    names = {B.PASS_KV: "pass_kv", B.PASS_Q: "pass_q"}
    launch = B.LAUNCH_AUTO if args.launch is None else args.launch
    q, k, v = make_qkv(w, device="cuda", seeds=seeds_of(args))
    outs, wss = make_buffers(B, w, q, k, modes, launch)
    flops_layer = w.causal_flops()
    flops_step = len(modes) * flops_layer
    launches_per_step = 0
    for mode in modes:
        plan = B.prefill_plan(w.sq, w.skv, w.n_chunks, mode, w.q_base, w.causal)
        launches_per_step += len({e[0] for e in plan}) + 1
    cap = (launches_per_step + 4) * args.steps

    clocks = ClockSampler(local)
    clocks.start()
    elapsed, per_mode, recs = time_modes(B, w, q, k, v, outs, wss, args.steps, args.warmup, world,
                                         modes, profile_cap=cap, launch=launch)
    clk = clocks.stop()
    # A kernel-side wait that gave up leaves garbage output: such a run is no
    # measurement.
    dev_status = B.device_status(clear=True)
    if dev_status != 0:
        print(f"bench: device status {dev_status} after the timed region", file=sys.stderr)
    ms_step = elapsed / args.steps
    value = world * flops_step * args.steps / (elapsed * 1e-3) / 1e12

    peaks, peak_src = load_peaks()
    tc = [r for r in recs if r[0] in ATTN_KINDS]
    tc_ms = sum(r[1] for r in tc)
    tc_flops = sum(r[2] for r in tc)
    achieved = tc_flops / (tc_ms * 1e-3) / 1e12 if tc_ms > 0 else None
    peak = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])
    traffic = None
    sha = kernel_sha()
    if tc and all(TRAFFIC_RECORD.get(r[0], {}).get("sha") == sha for r in tc):
        traffic = sum(TRAFFIC_RECORD[r[0]]["bytes_per_flop"] * r[2] for r in tc) / len(tc)
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": (achieved / peak) if achieved else None, "traffic": traffic,
                "kernel": "attn_pair_kernel (tcgen05 cta_group::2 partial attention; "
                          "per-step and on-chip instances)",
                "peak_source": f"{peak_src} bf16 dense, sustained",
                "launches_timed": len(tc), "avg_launch_ms": tc_ms / len(tc) if tc else None,
                "share_of_step": tc_ms / elapsed if elapsed else None}
    # The same figures per kernel instance (the step mixes Pass-KV's on-chip
    # launch with Pass-Q's per-step launches at 128K).
    by_inst = {}
    for kind in ATTN_KINDS:
        rk = [r for r in tc if r[0] == kind]
        ms_k = sum(r[1] for r in rk)
        if rk and ms_k > 0:
            ach = sum(r[2] for r in rk) / (ms_k * 1e-3) / 1e12
            by_inst[kind] = {"launches": len(rk), "achieved": ach, "frac": ach / peak,
                             "share_of_step": ms_k / elapsed if elapsed else None,
                             "capture": TRAFFIC_RECORD.get(kind, {}).get("capture")}
    roofline["by_instance"] = by_inst

    ms_layer = {names[m]: statistics.median(per_mode[m]) for m in modes}
    # Load balance of the ring this single GPU emulates: on N GPUs each ring
    # step lasts as long as its busiest rank.  Projected N-GPU time = measured
    # single-GPU time x critical / total (communication not included).
    ring = {}
    for assign, aname in ((B.ASSIGN_CONTIGUOUS, "contiguous"), (B.ASSIGN_ZIGZAG, "zigzag")):
        ring[aname] = {}
        for m in modes:
            try:
                crit, tot, _ = B.critical_path(w.sq, w.skv, w.n_chunks, m, w.q_base, w.causal, assign)
            except B.CpattnError:
                continue
            ring[aname][names[m]] = {
                "balance": tot / (w.n_chunks * crit),
                "projected_ms_per_layer_on_n_ranks": ms_layer[names[m]] * crit / tot}
    hbm_peak = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    mn = [r for r in recs if r[0] == "mergeN"]
    merge_roofline = {}
    if mn:
        gbs = sum(r[2] for r in mn) / (sum(r[1] for r in mn) * 1e-3) / 1e9
        merge_roofline["mergeN"] = {
            "bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s",
            "frac": gbs / hbm_peak, "frac_of_8TBs": gbs / 8000.0, "launches_timed": len(mn),
            "bytes_per_launch": sum(r[2] for r in mn) / len(mn),
            "peak_source": f"{peak_src} HBM copy"}
    merge_roofline["merge2"] = time_merge2(B, w, hbm_peak, peak_src)
    decode = None if args.skip_decode else time_decode(B, args.steps, hbm_peak, peak_src)
    cfg = {"workload": w.name, "batch": w.batch, "hq": w.hq, "hkv": w.hkv, "head_dim": w.head_dim,
           "seq_len": w.sq, "n_chunks": w.n_chunks, "causal": w.causal,
           "launch_mode": launch_modes(B, w, q, k, modes, launch),
           "step": " + ".join({"pass_kv": "Pass-KV prefill", "pass_q": "Pass-Q prefill"}[names[m]]
                               for m in modes) + " of one layer",
           "flops_per_layer": flops_layer, "ms_per_layer": ms_layer,
           "tflops_per_schedule": {k_: flops_layer / (v_ * 1e-3) / 1e12 for k_, v_ in ms_layer.items()},
           "pct_of_bf16_peak": 100.0 * value / world / peaks["bf16_tflops"],
           "peak_bf16_tflops": peaks["bf16_tflops"], "peak_source": peak_src,
           "l2": "inputs larger than L2: Q and O are 512 MiB each (K/V 32 MiB each stay L2-resident, as on a CP rank)",
           "parallelism": f"replicas x{world}", "cp_ring_projection": ring}
    mode_c, kvb, qb = B.choose_mode_ex(q, k, w.n_chunks, w.q_base, w.causal)
    cfg["schedule_choice"] = {"model_picks": names[mode_c], "pass_kv_ring_bytes": kvb,
                              "pass_q_ring_bytes": qb,
                              "model": "cpattn_prefill_choose_mode_ex (masked ring hops)"}
    if len(modes) == 2:
        cfg["schedule_choice"]["faster_on_one_gpu"] = min(ms_layer, key=ms_layer.get)

    # ---- the other configurations: ms per layer of each schedule (median),
    # 3 warm-ups each; the 1M layer is timed 5 times.
    if not args.skip_per_workload:
        del outs, wss
        torch.cuda.empty_cache()
        per = {}
        for name in ("tiny", "llama3-8b", "partial-32k", "128k", "1m"):
            if name == "1m" and args.skip_1m:
                continue
            if name == w.name:
                per[name] = {"flops_per_layer": flops_layer, "steps": args.steps,
                             "warmup": args.warmup, "launch_mode": cfg["launch_mode"],
                             "dtype": w.dtype, "see": "the main workload above"}
                for m in modes:
                    tf = flops_layer / (ms_layer[names[m]] * 1e-3) / 1e12
                    per[name][names[m]] = {
                        "ms_per_layer": ms_layer[names[m]], "tflops": tf,
                        "frac_of_bf16_burst": tf / peaks["bf16_tflops"],
                        "frac_of_bf16_sustained": tf / peaks.get("bf16_tflops_sustained",
                                                                 peaks["bf16_tflops"])}
                continue
            steps_w = 5 if name == "1m" else max(10, args.steps)
            per[name] = time_workload(B, name, steps_w, 3, world, modes, launch, peaks)
        cfg["per_workload"] = per
        if len(modes) == 2 and "partial-32k" in per:
            wp = WORKLOADS["partial-32k"]
            qp, kp, _ = make_qkv(wp, device="cuda")
            mode_p, kvp, qbp = B.choose_mode_ex(qp, kp, wp.n_chunks, wp.q_base, wp.causal)
            msp = {names[m]: per["partial-32k"][names[m]]["ms_per_layer"] for m in modes}
            cfg["schedule_choice_partial_32k"] = {
                "model_picks": names[mode_p], "pass_kv_ring_bytes": kvp, "pass_q_ring_bytes": qbp,
                "ms_per_layer": msp, "faster_on_one_gpu": min(msp, key=msp.get)}
            del qp, kp
        if "1m" in per:
            cfg["ms_per_layer_1m"] = {names[m]: per["1m"][names[m]]["ms_per_layer"] for m in modes}
        outs, wss = make_buffers(B, w, q, k, modes, launch)

    # ---- end to end through the host-buffer entry point
    e2e = None
    if not args.skip_e2e:
        qh, kh, vh = (t.cpu().pin_memory() for t in (q, k, v))
        oh = torch.empty_like(qh).pin_memory()
        lh = torch.empty((w.batch, w.hq, w.sq), dtype=torch.float32).pin_memory()
        need = max(B.host_scratch_size(qh, kh, w.n_chunks, m, w.q_base, w.causal)
                   for m in modes)
        del outs, wss
        torch.cuda.empty_cache()
        scratch = torch.empty(need, dtype=torch.uint8, device="cuda")

        per_call = {names[m]: [] for m in modes}

        def host_step():
            # Each call returns with its stream synchronised: wall time per call.
            for m in modes:
                t = time.perf_counter()
                B.prefill_host(qh, kh, vh, w.n_chunks, m, oh, lh, scratch, q_base=w.q_base,
                               causal=w.causal)
                per_call[names[m]].append(1e3 * (time.perf_counter() - t))

        for _ in range(args.warmup):
            host_step()
        for m in modes:
            per_call[names[m]].clear()
        barrier(world)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            host_step()
        t_e2e = max_over_ranks(time.perf_counter() - t0, world)
        in_bytes = sum(t.numel() * t.element_size() for t in (qh, kh, vh))
        out_bytes = oh.numel() * oh.element_size() + lh.numel() * 4
        e2e = {"value": world * flops_step * args.steps / t_e2e / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": len(modes) * in_bytes,
               "d2h_bytes_per_step": len(modes) * out_bytes,
               "ms_per_step": 1e3 * t_e2e / args.steps,
               "ms_per_call": {k: statistics.median(x) for k, x in per_call.items() if x},
               "path": "cpattn_prefill_host (pinned host buffers; copies inside the timed region)"}
        del scratch

    # ---- CPU baseline: the oracle on a bounded sample (rank 0 only)
    cpu_baseline = None
    if rank == 0 and args.cpu_rows > 0:
        f, dt, threads, rows = oracle_sample(w, args.cpu_rows)
        cpu_baseline = {"value": f / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                        "sample": f"{args.cpu_rows} seeded query rows x {w.hq} heads of the {w.name} "
                                  f"workload (full causal key range each), fp64, {dt:.1f} s"}

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                "data": "synthetic (seeded i.i.d. N(0,1) Q/K/V, bf16)", "config": cfg,
                "roofline": roofline, "merge_roofline": merge_roofline, "decode": decode,
                "cpu_baseline": cpu_baseline, "e2e": e2e,
                "gpu_launches": len(recs), "device_status": dev_status, "clocks": clk}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
