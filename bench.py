"""Benchmark of the differential-attention hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one pass of the prefill hot path on the 3B-layer workload (B 4, N 4096, 12 heads,
d 128, dv 256, causal, bf16): lambda formed from its four vectors in the kernel's prologue, the
fused DiffAttn prefill, RMSNorm and the (1 - lambda_init) scale. `value` is TFLOP/s counted at
1536 MMA flops per causal query-key pair (4d for the two score maps + 4dv for the two value
products), summed over ranks (weak scaling: every rank runs its own batch).

The JSON line carries, in this order: the primary keys (with the roofline of the prefill kernel,
the clocks of its timed loop and an end-to-end figure through host buffers beside the bare copy
bound of the same bytes), one compact block per secondary workload, the float64 oracle timed on
the host cores, a `headline` summary, and last the decode workload (B 64, cache 32768, 12 heads:
HBM GB/s) with the clocks of its own timed loop.

Roofline peaks: MEASURED_PEAKS.json's burst bf16 figure for a timed loop under a second, its
sustained figure for longer loops, its copy bandwidth for HBM-bound kernels; the nominal dense
figures of the part (2.25 PFLOP/s bf16, 8 TB/s) are reported beside them as `frac_nominal`.

`--impl reference` times the float64 CPU oracle (the only reference implementation that exists
for this method) on bounded samples of the same workload, on rank 0 only.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time
import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

PREFILL = dict(B=4, N=4096, H=12, d=128, dv=256, layer=12)
DECODE = dict(B=64, L=32768, H=12, d=128, dv=256, layer=12)
V2 = dict(B=2, N=8192, Hq=64, Hkv=8, d=128)
V2_DECODE = dict(B=64, L=32768, Hq=64, Hkv=8, d=128)
GDA = dict(B=4, N=4096, Hs=12, Hn=3, d=128, dv=256, layer=12)       # 4 signal heads per noise head
GDA_DECODE = dict(B=64, L=32768, Hs=12, Hn=3, d=128, dv=256, layer=12)
LONG = dict(B=1, N=65536, H=12, d=128, dv=256, layer=24)
PREFILL_WORKLOAD = ("prefill_3b: B4 N4096 H12 d128 dv256 causal, lambda (layer 12, formed in the "
                    "kernel) + DiffAttn + RMSNorm + (1 - lambda_init)")
FLOPS_PER_PAIR = 1536        # 4d + 4dv MMA flops per causal (query, key) pair, V1
FLOPS_PER_PAIR_DEF = 1024    # 4d + 2dv: the definition (A1 - lambda A2) V
V2_FLOPS_PER_PAIR = 8 * 128  # per (query, key) pair of one differential pair: 2 heads x (QK + PV)
# backward per causal pair: S1, S2 recomputed (4d), dW = dO V^T (2dv), dV (2dv), dK1+dK2 (4d),
# dQ1+dQ2 (4d) = 2560, i.e. 2.5x the definition's forward count; the kernels issue 4352 (the
# delta pass 2d + 2dv, and dW once per map)
BWD_FLOPS_PER_PAIR = 4 * 128 + 2 * 256 + 2 * 256 + 4 * 128 + 4 * 128
BWD_ISSUED_FLOPS_PER_PAIR = (2 * 128 + 2 * 256) + 2 * (2 * 128 + 2 * 256 + 2 * 128 + 2 * 128) \
    + (4 * 128 + 2 * 256)

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# nominal dense figures of the part, reported beside the measured fractions
NOMINAL = {"bf16_tflops": 2250.0, "hbm_gbs": 8000.0}
# a timed loop this long or longer (seconds-long: the power cap has settled) is read against the
# sustained bf16 peak; shorter loops against the burst peak
SUSTAINED_AFTER_MS = 2000.0


def causal_pairs(N: int) -> int:
    return N * (N + 1) // 2


def prefill_flops(cfg=PREFILL, per_pair=FLOPS_PER_PAIR) -> float:
    return float(cfg["B"] * cfg["H"] * causal_pairs(cfg["N"]) * per_pair)


def decode_bytes(cfg=DECODE) -> float:
    return float(cfg["B"] * cfg["L"] * cfg["H"] * (2 * cfg["d"] + cfg["dv"]) * 2)


def gda_decode_bytes(cfg=GDA_DECODE) -> float:
    # each cached row once: K of the signal and noise heads, V of the signal heads
    return float(cfg["B"] * cfg["L"] * ((cfg["Hs"] + cfg["Hn"]) * cfg["d"] + cfg["Hs"] * cfg["dv"]) * 2)


def v2_decode_bytes(cfg=V2_DECODE) -> float:
    return float(cfg["B"] * cfg["L"] * cfg["Hkv"] * 2 * cfg["d"] * 2)


def varlen_lengths():
    """A seeded mix of 16 sequence lengths from 1 to 4096 tokens (16,384 in total): the packed
    stand-in for a batch of documents of different lengths."""
    rng = np.random.default_rng(12)
    lens = np.maximum(1, np.round(rng.pareto(1.2, 16) * 300)).astype(int)
    lens = np.minimum(lens, 4096)
    lens[0], lens[-1] = 4096, 1
    rest = 16384 - lens.sum()
    lens[1] = max(1, lens[1] + rest)
    return [int(x) for x in np.minimum(lens, 4096)]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def source_sha(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "differential_attention_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(summary: str, sha: str):
    """dram bytes per launch from a committed ncu summary, or None if absent or stale."""
    path = os.path.join(ROOT, "profiles", summary)
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_sha = re.search(r"kernel_source_sha256:\s*([0-9a-f]+)", text)
    m_b = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not m_sha or not m_b or m_sha.group(1) != sha:
        return None
    return float(m_b.group(1))


def dist_barrier():
    """Synchronise the device, then all ranks (no-op in a single process)."""
    import torch
    import torch.distributed as dist
    if torch.cuda.is_available() and torch.cuda.is_initialized():
        torch.cuda.synchronize()
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.barrier()


def dist_max(x: float, device=None) -> float:
    """Maximum of `x` over all ranks (the timing rule: the slowest rank sets the job's time)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    dev = device if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = []
        for ln in (self.out or "").splitlines():
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), smax=float(parts[2]), power=float(parts[3]),
                                 hw=parts[5], hwt=parts[6], swt=parts[7], pcap=parts[8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        loaded = [r for r in rows if r["power"] > 200.0] or rows
        reasons = set()
        for r in loaded:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in loaded),
                "sm_max_mhz": max(r["smax"] for r in rows), "reasons": sorted(reasons),
                "samples": len(loaded), "power_w_max": max(r["power"] for r in rows)}


# ---------------------------------------------------------------------------------------------
# CPU baseline: the float64 oracle on a bounded sample of the workload
# ---------------------------------------------------------------------------------------------
def oracle_sample(budget_s: float, seed: int = 0):
    """Time the oracle on whole heads of the 3B-layer prefill (every causal row of a head, heads
    and sequences in order) until `budget_s` of CPU time is used. Returns (TFLOP/s at 1536
    flops/pair, cores, description, pairs, seconds)."""
    import numpy as np
    import torch
    from oracle import diffattn_ref as ref
    from synth import make_prefill_inputs

    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    torch.set_num_threads(cores)
    N, d, H = PREFILL["N"], PREFILL["d"], PREFILL["H"]
    li = ref.lambda_init(PREFILL["layer"])
    rows_done, pairs, t_used, heads = 0, 0, 0.0, 0
    block = 256
    for b in range(PREFILL["B"]):  # sequences of the workload, one at a time
        if t_used >= budget_s:
            break
        inp = make_prefill_inputs(1, N, H, d, PREFILL["dv"], seed=seed + b, layer=PREFILL["layer"])
        lam = float(ref.lambda_full(*inp.lam_vectors, layer=PREFILL["layer"])[0])
        q, k, v = (ref._f64(t) for t in (inp.q, inp.k, inp.v))
        for h in range(H):
            if t_used >= budget_s:
                break
            qh, kh, vh = q[:, :, h:h + 1], k[:, :, h:h + 1], v[:, :, h:h + 1]
            for hi in range(N, 0, -block):
                if t_used >= budget_s:
                    break
                rows = np.arange(max(0, hi - block), hi)
                t0 = time.perf_counter()
                ref.diffattn_fwd(qh, kh, vh, [lam], li, rows=rows)
                t_used += time.perf_counter() - t0
                rows_done += rows.shape[0]
                pairs += int(np.sum(rows + 1))
            heads += 1
    tflops = pairs * FLOPS_PER_PAIR / t_used / 1e12
    desc = (f"oracle (numpy float64, {cores} threads) on {rows_done} causal query rows "
            f"({heads} (sequence, head) pairs, longest rows first) of the 3B-layer prefill: "
            f"{pairs} query-key pairs in {t_used:.1f} s")
    return tflops, cores, desc, pairs, t_used


def run_reference(args, rank: int, world: int):
    if rank != 0:
        return
    # each step times a bounded sample; the whole run stays within ~2 minutes
    per_step = max(0.05, min(5.0, 120.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample(per_step * 0.25)
    vals, times, pairs_total = [], [], 0
    cores, desc = None, None
    for _ in range(args.steps):
        v, cores, desc, pairs, t = oracle_sample(per_step)
        vals.append(v)
        times.append(t)
        pairs_total += pairs
    value = pairs_total * FLOPS_PER_PAIR / sum(times) / 1e12
    line = {
        "impl": "reference", "metric": "DiffAttn fwd TFLOP/s (% dense BF16 TC peak); decode HBM GB/s (% peak)",
        "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * sum(times) / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": PREFILL_WORKLOAD, "global_batch": PREFILL["B"],
                   "seq_len": PREFILL["N"], "parallelism": "none (host cores)",
                   "flops_per_pair": FLOPS_PER_PAIR},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"per step: {desc}"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------------------------
# our path
# ---------------------------------------------------------------------------------------------
class Timer:
    """Warm-up, then `n` calls of `fn` on the current stream, each bracketed by CUDA events.

    Returns the mean per-call time (ms), the whole timed region (ms, from its own events) and,
    when `clocks` is set, the clocks nvidia-smi saw while the loop ran."""

    def __init__(self, torch, dev, barrier, warmup):
        self.torch, self.dev, self.barrier, self.warmup = torch, dev, barrier, warmup
        self.stream = torch.cuda.current_stream()

    def ev(self):
        return self.torch.cuda.Event(enable_timing=True)

    def __call__(self, fn, n, clocks=False, status=None):
        for _ in range(self.warmup):
            fn()
        if status:
            status()
        evs = [(self.ev(), self.ev()) for _ in range(n)]
        t0, t1 = self.ev(), self.ev()

        def loop():
            self.barrier()
            t0.record(self.stream)
            for a, b in evs:
                a.record(self.stream)
                fn()
                b.record(self.stream)
            t1.record(self.stream)
            self.barrier()

        clk = None
        if clocks:
            with ClockSampler(self.dev.index) as sampler:
                loop()
            clk = sampler.summary()
        else:
            loop()
        if status:
            status()
        return {"ms": statistics.mean(a.elapsed_time(b) for a, b in evs),
                "total_ms": t0.elapsed_time(t1), "n": n, "clocks": clk}


def tensor_peak(peaks, peak_src, total_ms, scale=1.0, what="bf16"):
    """The measured bf16 peak that applies to a loop of `total_ms`: the burst figure for a loop
    well under a second (the kernel does not reach the power cap), the sustained one otherwise."""
    if total_ms < SUSTAINED_AFTER_MS:
        key, kind = "bf16_tflops", "burst"
    else:
        key, kind = "bf16_tflops_sustained", "sustained"
    p = peaks.get(key, FALLBACK_PEAKS[key]) * scale
    src = f"{key} of {peak_src} ({kind}: the timed loop ran {total_ms:.0f} ms)"
    if scale != 1.0:
        src = f"{scale} x " + src + f"; {what}"
    return p, src


def tensor_roof(flops, t, peaks, peak_src, scale=1.0, what="bf16", nominal_scale=1.0):
    achieved = flops / (t["ms"] * 1e-3) / 1e12
    peak, src = tensor_peak(peaks, peak_src, t["total_ms"], scale, what)
    nominal = NOMINAL["bf16_tflops"] * nominal_scale
    return {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
            "frac": achieved / peak, "peak_source": src,
            "frac_nominal": achieved / nominal, "nominal_peak": nominal}


def hbm_roof(nbytes, t, peaks, peak_src):
    achieved = nbytes / (t["ms"] * 1e-3) / 1e9
    peak = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak, "peak_source": f"hbm_gbs of {peak_src} (copy, read+write)",
            "frac_nominal": achieved / NOMINAL["hbm_gbs"], "nominal_peak": NOMINAL["hbm_gbs"]}


def compact(value, unit, t, roof, workload, world, **extra):
    """A secondary workload's block: its figure, time, roofline fractions and a short name."""
    blk = {"value": world * value, "unit": unit, "ms": round(t["ms"], 4), "calls": t["n"],
           "frac": round(roof["frac"], 4), "frac_nominal": round(roof["frac_nominal"], 4),
           "peak": f'{roof["peak"]:.1f} {roof["unit"]} ({roof["peak_source"].split(" (")[0]})',
           "workload": workload}
    blk.update(extra)
    return blk


def run_ours(args, rank: int, world: int, local_rank: int):
    import torch
    import differential_attention_gb300 as da
    from synth import (make_decode_inputs, make_dout, make_gda_decode_inputs, make_gda_inputs,
                       make_lambda_vectors, make_prefill_inputs, make_v2_decode_inputs,
                       make_v2_inputs, to_fp8_e4m3)

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    da.build()
    peaks, peak_src = load_peaks()
    stream = torch.cuda.current_stream()

    def barrier():
        dist_barrier()

    def max_over_ranks(x: float) -> float:
        return dist_max(x, dev)

    timer = Timer(torch, dev, barrier, args.warmup)
    status = da.diffattn_device_status
    want = lambda name: args.only in ("all", name)

    line = {"metric": "DiffAttn fwd TFLOP/s (% dense BF16 TC peak); decode HBM GB/s (% peak)",
            "value": None, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": None, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic"}
    extra = {}      # secondary workloads, printed after the primary keys
    decode_blk = None

    # ======================= prefill: the step that `value` measures =======================
    if want("prefill"):
        c = PREFILL
        inp = make_prefill_inputs(c["B"], c["N"], c["H"], c["d"], c["dv"], seed=1000 + rank,
                                  layer=c["layer"], device=dev)
        # one lambda per layer, shared by every head ([P3]), formed inside the prefill kernel
        lv = tuple(t.to(dev).contiguous() for t in make_lambda_vectors(c["d"], seed=1001 + rank))
        out = torch.empty((c["B"], c["N"], c["H"], c["dv"]), dtype=torch.bfloat16, device=dev)

        def step():
            da.diffattn_fwd_fused_lambda(inp.q, inp.k, inp.v, *lv, layer=c["layer"], out=out)

        t = timer(step, args.steps, clocks=True, status=status)
        ms_per_step = max_over_ranks(t["total_ms"]) / args.steps
        flops = prefill_flops()
        roof = tensor_roof(flops, t, peaks, peak_src)
        sha = source_sha(["prefill_exact.cu", "ptx.cuh"])
        roof.update({"traffic": profiled_traffic("prefill_exact_3b.md", sha),
                     "kernel": "prefill_exact_kernel<128,256,false> (lambda in the prologue)",
                     "kernel_ms": t["ms"], "flops_per_launch": flops,
                     "flops_per_pair": FLOPS_PER_PAIR,
                     "definition_count_tflops":
                         flops / FLOPS_PER_PAIR * FLOPS_PER_PAIR_DEF / (t["ms"] * 1e-3) / 1e12})
        line.update({
            "value": world * flops / (ms_per_step * 1e-3) / 1e12,
            "ms_per_step": ms_per_step,
            "config": {"workload": PREFILL_WORKLOAD,
                       "global_batch": PREFILL["B"] * world, "seq_len": PREFILL["N"],
                       "parallelism": f"replicas x{world} (independent batches, no collective)",
                       "l2": "inputs larger than L2 (q, k, v = 302 MB per rank)",
                       "flops_per_pair": FLOPS_PER_PAIR},
            "roofline": roof,
            "gpu_launches": args.steps,
            "clocks": t["clocks"],
        })

        # ---------------- end to end through host buffers ----------------
        e2e_steps = max(3, min(20, args.steps))
        hq, hk, hv = (x.cpu().pin_memory() for x in (inp.q, inp.k, inp.v))
        hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        hws = torch.empty(da.diffattn_fwd_host_workspace_size(c["B"], c["N"], c["H"], c["d"], c["dv"]),
                          dtype=torch.uint8, device=dev)

        def e2e_step():
            da.diffattn_fwd_host(hq, hk, hv, hout, *lv, layer=c["layer"], workspace=hws)

        te = timer(e2e_step, e2e_steps)
        e2e_ms = max_over_ranks(te["total_ms"]) / e2e_steps

        # the copy bound: the same pinned buffers moved with one plain cudaMemcpyAsync per tensor
        # and no kernel; host-to-device on one stream, device-to-host on another, concurrently
        # (the least any pipeline over this host link can take), and all four on one stream
        dq, dk, dvv = (torch.empty_like(x) for x in (inp.q, inp.k, inp.v))
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

        def copies_overlapped():
            s_in.wait_stream(stream)
            s_out.wait_stream(stream)
            with torch.cuda.stream(s_in):
                for d_, h_ in ((dq, hq), (dk, hk), (dvv, hv)):
                    d_.copy_(h_, non_blocking=True)
            with torch.cuda.stream(s_out):
                hout.copy_(out, non_blocking=True)
            stream.wait_stream(s_in)
            stream.wait_stream(s_out)

        def copies_serial():
            for d_, h_ in ((dq, hq), (dk, hk), (dvv, hv)):
                d_.copy_(h_, non_blocking=True)
            hout.copy_(out, non_blocking=True)

        tco = timer(copies_overlapped, e2e_steps)
        tcs = timer(copies_serial, e2e_steps)
        copy_ms = max_over_ranks(tco["total_ms"]) / e2e_steps
        copy_serial_ms = max_over_ranks(tcs["total_ms"]) / e2e_steps
        h2d, d2h = 3 * inp.q.numel() * 2, out.numel() * 2
        line["e2e"] = {"value": world * flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                       "ms_per_step": e2e_ms,
                       "copy_bound_ms": copy_ms, "copy_serial_ms": copy_serial_ms,
                       "e2e_over_copy_bound": e2e_ms / copy_ms,
                       "link_gbs": (h2d + d2h) / (copy_ms * 1e-3) / 1e9,
                       "via": "diffattn_fwd_host: pinned host q, k, v copied in, each "
                              "sequence's copies overlapped with the prefill of the others; the "
                              "prefill stores its output rows into the pinned host out over the "
                              "link (d2h bytes); copy_bound_ms: the same bytes, plain copies "
                              "only, H2D and D2H on two streams at once"}
        del hq, hk, hv, hout, hws, dq, dk, dvv

        # the single-pass kernel (one flash pass per map on a 2-CTA cluster, opt-in), same inputs
        lam_h = da.diffattn_lambda(*(x.expand(c["H"], -1).contiguous() for x in lv), layer=c["layer"])
        li = da.diffattn_lambda_init(c["layer"])
        ts = timer(lambda: da.diffattn_fwd(inp.q, inp.k, inp.v, lam_h, li, single_pass=True,
                                           out=out), max(5, min(50, args.steps)), status=status)
        td = timer(lambda: da.diffattn_fwd(inp.q, inp.k, inp.v, lam_h, li, out=out),
                   max(5, min(50, args.steps)), status=status)
        rs, rd = tensor_roof(flops, ts, peaks, peak_src), tensor_roof(flops, td, peaks, peak_src)
        extra["prefill_single_pass"] = compact(
            rs["achieved"], "TFLOP/s", ts, rs,
            "prefill_3b, DIFFATTN_SINGLE_PASS: prefill_tc_kernel (a flash pass per map, 2-CTA "
            "cluster)", world, default_two_pass_ms=round(td["ms"], 4))
        del inp, out
        torch.cuda.empty_cache()

    # ======================= long-context prefill =======================
    if want("long"):
        c = LONG
        inp = make_prefill_inputs(c["B"], c["N"], c["H"], c["d"], c["dv"], seed=4000 + rank,
                                  layer=c["layer"], device=dev, needle=True)
        lv = tuple(x.to(dev).contiguous() for x in make_lambda_vectors(c["d"], seed=4001 + rank))
        out = torch.empty((c["B"], c["N"], c["H"], c["dv"]), dtype=torch.bfloat16, device=dev)
        t = timer(lambda: da.diffattn_fwd_fused_lambda(inp.q, inp.k, inp.v, *lv, layer=c["layer"],
                                                       out=out),
                  max(3, min(10, args.steps)), status=status)
        lflops = prefill_flops(c)
        r = tensor_roof(lflops, t, peaks, peak_src)
        extra["prefill_64k"] = compact(r["achieved"], "TFLOP/s", t, r,
                                       "B1 N65536 H12 causal, layer 24, one needle key per head", world)
        del inp, out
        torch.cuda.empty_cache()

    # ======================= V2 =======================
    if want("v2"):
        vc = V2
        vinp = make_v2_inputs(vc["B"], vc["N"], vc["Hq"], vc["Hkv"], vc["d"], seed=3000 + rank,
                              device=dev)
        vout = torch.empty((vc["B"], vc["N"], vc["Hq"] // 2, vc["d"]), dtype=torch.bfloat16,
                           device=dev)
        t = timer(lambda: da.diffattn_v2_fwd(vinp.q, vinp.k, vinp.v, vinp.lam_logit, out=vout),
                  max(5, min(30, args.steps)), status=status)
        tx = timer(lambda: da.diffattn_v2_fwd(vinp.q, vinp.k, vinp.v, vinp.lam_logit, out=vout,
                                              exact=True), 5, status=status)
        vflops = float(vc["B"] * (vc["Hq"] // 2) * causal_pairs(vc["N"]) * V2_FLOPS_PER_PAIR)
        r = tensor_roof(vflops, t, peaks, peak_src)
        extra["v2"] = compact(r["achieved"], "TFLOP/s", t, r,
                              "B2 N8192 Hq64 (32 pairs) Hkv8 d128 causal, v2_pair_kernel", world,
                              exact_two_pass_ms=round(tx["ms"], 4),
                              traffic=profiled_traffic("v2_pair_gqa.md",
                                                       source_sha(["prefill_v2.cu", "ptx.cuh"])))
        del vinp, vout
        torch.cuda.empty_cache()

    # ======================= prefill with fp8 scores =======================
    if want("fp8"):
        c = PREFILL
        inp = make_prefill_inputs(c["B"], c["N"], c["H"], c["d"], c["dv"], seed=9000 + rank,
                                  layer=c["layer"], device=dev)
        q8, qs = to_fp8_e4m3(inp.q)
        k8, ks = to_fp8_e4m3(inp.k)
        lam = torch.full((c["H"],), 0.6, dtype=torch.float32, device=dev)
        li = da.diffattn_lambda_init(c["layer"])
        out = torch.empty((c["B"], c["N"], c["H"], c["dv"]), dtype=torch.bfloat16, device=dev)
        t = timer(lambda: da.diffattn_fwd_fp8(q8, k8, inp.v, lam, qs, ks, li, out=out),
                  max(5, min(200, args.steps)), status=status)
        # 1024 of the 1536 flops per pair are score products at the fp8 rate (2x bf16 by the
        # nominal ratio), 512 the bf16 product with V: blended peak 1.5x bf16
        r = tensor_roof(prefill_flops(), t, peaks, peak_src, scale=1.5,
                        what="scores at the fp8 rate (2x bf16, nominal ratio), V product at bf16",
                        nominal_scale=1.5)
        extra["prefill_fp8"] = compact(r["achieved"], "TFLOP/s", t, r,
                                       "prefill_3b with fp8 e4m3 q, k (per-tensor scales)", world,
                                       peak_note="blended: 1.5 x bf16")
        del inp, q8, k8, out
        torch.cuda.empty_cache()

    # ======================= variable-length prefill (packed sequences) =======================
    if want("varlen"):
        c = PREFILL
        lens = varlen_lengths()
        total = int(sum(lens))
        inp = make_prefill_inputs(1, total, c["H"], c["d"], c["dv"], seed=8000 + rank,
                                  layer=c["layer"], device=dev)
        cu = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32, device=dev)
        lam = torch.full((c["H"],), 0.6, dtype=torch.float32, device=dev)
        li = da.diffattn_lambda_init(c["layer"])
        out = torch.empty((total, c["H"], c["dv"]), dtype=torch.bfloat16, device=dev)
        q, k, v = inp.q[0], inp.k[0], inp.v[0]
        n_steps = max(5, min(50, args.steps))
        t = timer(lambda: da.diffattn_fwd_varlen(q, k, v, cu, lam, li, max_seqlen=max(lens),
                                                 out=out), n_steps, status=status)
        vflops = float(sum(c["H"] * causal_pairs(n) * FLOPS_PER_PAIR for n in lens))
        r = tensor_roof(vflops, t, peaks, peak_src)
        extra["varlen"] = compact(r["achieved"], "TFLOP/s", t, r,
                                  f"{len(lens)} packed sequences, {min(lens)}..{max(lens)} tokens "
                                  f"({total}), causal, H12", world)
        del inp, out, q, k, v
        torch.cuda.empty_cache()

        # the last 1024-token chunk of each prefill_3b prompt against its 4096 keys
        Lq, Lk = 1024, c["N"]
        kin = make_prefill_inputs(c["B"], Lk, c["H"], c["d"], c["dv"], seed=8100 + rank,
                                  layer=c["layer"], device=dev)
        k, v = kin.k.reshape(-1, c["H"], 2 * c["d"]), kin.v.reshape(-1, c["H"], c["dv"])
        q = kin.q[:, Lk - Lq:].reshape(-1, c["H"], 2 * c["d"]).contiguous()
        cu_q = torch.arange(c["B"] + 1, dtype=torch.int32, device=dev) * Lq
        cu_k = torch.arange(c["B"] + 1, dtype=torch.int32, device=dev) * Lk
        out = torch.empty((c["B"] * Lq, c["H"], c["dv"]), dtype=torch.bfloat16, device=dev)
        t = timer(lambda: da.diffattn_fwd_varlen_qk(q, k, v, cu_q, cu_k, lam, li, max_seqlen_q=Lq,
                                                    max_seqlen_k=Lk, out=out),
                  n_steps, status=status)
        pairs = Lq * (Lk - Lq) + Lq * (Lq + 1) // 2  # query at position p sees p + 1 keys
        cflops = float(c["B"] * c["H"] * pairs * FLOPS_PER_PAIR)
        r = tensor_roof(cflops, t, peaks, peak_src)
        extra["varlen_qk"] = compact(r["achieved"], "TFLOP/s", t, r,
                                     f"last {Lq}-query chunk of B{c['B']} prompts over {Lk} keys",
                                     world)

        # the same chunk with the prompts' keys in a pool of 256-token pages in a random order
        ps = 256
        mp = Lk // ps
        k_pool = kin.k.reshape(c["B"] * mp, ps, c["H"], 2 * c["d"])
        v_pool = kin.v.reshape(c["B"] * mp, ps, c["H"], c["dv"])
        gp = torch.Generator(device="cpu")
        gp.manual_seed(8200 + rank)
        table = torch.randperm(c["B"] * mp, generator=gp).to(torch.int32).view(c["B"], mp).to(dev)
        # the pool's pages in table order hold the prompts' keys: page table[b, i] <- (b, i)
        k_pool = k_pool[torch.argsort(table.flatten())].contiguous()
        v_pool = v_pool[torch.argsort(table.flatten())].contiguous()
        sk = torch.full((c["B"],), Lk, dtype=torch.int32, device=dev)
        t = timer(lambda: da.diffattn_fwd_paged(q, k_pool, v_pool, cu_q, sk, table, lam, li,
                                                max_seqlen_q=Lq, max_seqlen_k=Lk, out=out),
                  n_steps, status=status)
        r = tensor_roof(cflops, t, peaks, peak_src)
        extra["paged_prefill"] = compact(r["achieved"], "TFLOP/s", t, r,
                                         f"the varlen_qk chunk, keys in shuffled {ps}-token pages",
                                         world)
        del kin, out, q, k, v, k_pool, v_pool, table
        torch.cuda.empty_cache()

    # ======================= training step: forward (saving statistics) + backward ==========
    if want("backward"):
        c = PREFILL
        inp = make_prefill_inputs(c["B"], c["N"], c["H"], c["d"], c["dv"], seed=7000 + rank,
                                  layer=c["layer"], device=dev)
        dy = make_dout(c["B"], c["N"], c["H"], c["dv"], seed=7007 + rank, device=dev)
        lam = torch.linspace(0.5, 0.9, c["H"], dtype=torch.float32, device=dev)
        li = da.diffattn_lambda_init(c["layer"])
        w = torch.ones(c["dv"], dtype=torch.float32, device=dev)
        ws = torch.empty(da.diffattn_bwd_workspace_size(c["B"], c["N"], c["H"], c["d"], c["dv"]),
                         dtype=torch.uint8, device=dev)
        saved = {}
        grads = dict(dq=torch.empty_like(inp.q), dk=torch.empty_like(inp.k),
                     dv=torch.empty_like(inp.v),
                     dlam=torch.empty(c["H"], dtype=torch.float32, device=dev),
                     dw=torch.empty(c["dv"], dtype=torch.float32, device=dev))

        def fwd():
            saved["out"], saved["o_pre"], saved["stats"] = da.diffattn_fwd_train(
                inp.q, inp.k, inp.v, lam, li, norm_weight=w)

        def bwd():
            da.diffattn_bwd(inp.q, inp.k, inp.v, saved["o_pre"], saved["stats"], dy, lam, li,
                            norm_weight=w, workspace=ws, grads=grads)

        n_steps = max(3, min(20, args.steps))
        tf_ = timer(fwd, n_steps, status=status)
        tb = timer(bwd, n_steps, status=status)
        pairs = c["B"] * c["H"] * causal_pairs(c["N"])
        bflops = float(pairs * BWD_FLOPS_PER_PAIR)
        r = tensor_roof(bflops, tb, peaks, peak_src)
        extra["backward"] = compact(
            r["achieved"], "TFLOP/s", tb, r,
            "prefill_3b training: every gradient (2560 flops per causal pair)", world,
            fwd_train_ms=round(tf_["ms"], 4),
            traffic=profiled_traffic("backward_dkdq_3b.md", source_sha(["backward.cu", "ptx.cuh"])))
        del inp, dy, saved, grads, ws
        torch.cuda.empty_cache()

        # the backward over the packed-sequence workload (16 sequences of mixed length)
        lens = varlen_lengths()
        total = int(sum(lens))
        pin = make_prefill_inputs(1, total, c["H"], c["d"], c["dv"], seed=7100 + rank,
                                  layer=c["layer"], device=dev)
        q, k, v = pin.q[0], pin.k[0], pin.v[0]
        dyp = make_dout(1, total, c["H"], c["dv"], seed=7107 + rank, device=dev)[0]
        cu = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32, device=dev)
        mx = max(lens)
        _, o_pre, stats = da.diffattn_fwd_train_varlen(q, k, v, cu, lam, li, max_seqlen=mx,
                                                       norm_weight=w)
        ws = torch.empty(da.diffattn_bwd_varlen_workspace_size(len(lens), mx, total, c["H"],
                                                               c["d"], c["dv"]),
                         dtype=torch.uint8, device=dev)
        grads = dict(dq=torch.empty_like(q), dk=torch.empty_like(k), dv=torch.empty_like(v),
                     dlam=torch.empty(c["H"], dtype=torch.float32, device=dev),
                     dw=torch.empty(c["dv"], dtype=torch.float32, device=dev))
        t = timer(lambda: da.diffattn_bwd_varlen(q, k, v, o_pre, stats, dyp, cu, lam, li,
                                                 max_seqlen=mx, norm_weight=w, workspace=ws,
                                                 grads=grads), n_steps, status=status)
        vflops = float(sum(c["H"] * causal_pairs(n) * BWD_FLOPS_PER_PAIR for n in lens))
        r = tensor_roof(vflops, t, peaks, peak_src)
        extra["backward_varlen"] = compact(r["achieved"], "TFLOP/s", t, r,
                                           f"backward over the {len(lens)} packed sequences", world)
        del pin, q, k, v, dyp, o_pre, stats, ws, grads
        torch.cuda.empty_cache()

    # ======================= grouped: signal heads sharing noise heads =======================
    if want("gda"):
        gc = GDA
        ginp = make_gda_inputs(gc["B"], gc["N"], gc["Hs"], gc["Hn"], gc["d"], gc["dv"],
                               seed=5000 + rank, device=dev)
        gout = torch.empty((gc["B"], gc["N"], gc["Hs"], gc["dv"]), dtype=torch.bfloat16, device=dev)
        li_g = da.diffattn_lambda_init(gc["layer"])
        gws = torch.empty(da.diffattn_gda_fwd_workspace_size(gc["B"], gc["N"], gc["Hs"], gc["Hn"]),
                          dtype=torch.uint8, device=dev)
        t = timer(lambda: da.diffattn_gda_fwd(ginp.q, ginp.k, ginp.v, ginp.lam, gc["Hs"], li_g,
                                              workspace=gws, out=gout),
                  max(5, min(50, args.steps)), status=status)
        t1 = timer(lambda: da.diffattn_gda_fwd(ginp.q, ginp.k, ginp.v, ginp.lam, gc["Hs"], li_g,
                                               noise_pass=False, out=gout),
                   max(5, min(50, args.steps)), status=status)
        pairs = float(gc["B"] * gc["Hs"] * causal_pairs(gc["N"]))
        G = gc["Hs"] // gc["Hn"]
        # the method's own MMA work per (signal head, causal pair): its map's scores (2d), the
        # noise map's scores once per group (2d / G) and both maps' products with V (4dv)
        method_per_pair = 2 * gc["d"] + 2 * gc["d"] / G + 4 * gc["dv"]
        # issued by the two launches: the noise pass's scores once per noise head (2d / G), the
        # signal heads' first pass over their own map (2d), the second pass's two maps (4d) and
        # the product with V (2dv)
        issued_per_pair = 2 * gc["d"] / G + 2 * gc["d"] + 4 * gc["d"] + 2 * gc["dv"]
        r = tensor_roof(pairs * method_per_pair, t, peaks, peak_src)
        issued = pairs * issued_per_pair / (t["ms"] * 1e-3) / 1e12
        extra["gda_prefill"] = compact(r["achieved"], "TFLOP/s", t, r,
                                       "prefill_3b with 12 signal heads over 3 noise heads", world,
                                       flops_per_pair=method_per_pair,
                                       issued_tflops=round(issued, 1),
                                       issued_flops_per_pair=issued_per_pair,
                                       one_launch_ms=round(t1["ms"], 4))

        # the same heads with fp8 e4m3 q and k (one launch: each signal head forms its noise map)
        q8, qs = to_fp8_e4m3(ginp.q)
        k8, ks = to_fp8_e4m3(ginp.k)
        t8 = timer(lambda: da.diffattn_gda_fwd_fp8(q8, k8, ginp.v, ginp.lam, gc["Hs"], qs, ks, li_g,
                                                   out=gout),
                   max(5, min(50, args.steps)), status=status)
        # issued per (signal head, pair), as on the prefill_fp8 line: both maps' scores in both
        # passes at the fp8 rate, the product with V at bf16 (1536 flops, blended peak 1.5x bf16)
        r = tensor_roof(pairs * FLOPS_PER_PAIR, t8, peaks, peak_src, scale=1.5,
                        what="scores at the fp8 rate (2x bf16, nominal ratio), V product at bf16",
                        nominal_scale=1.5)
        extra["gda_prefill_fp8"] = compact(r["achieved"], "TFLOP/s", t8, r,
                                           "gda_prefill with fp8 e4m3 q and k (one launch)", world,
                                           flops_per_pair=FLOPS_PER_PAIR)
        del ginp, gout, q8, k8
        torch.cuda.empty_cache()

        # the last 1024-token chunk of each prompt against its 4096 keys, keys packed with offsets
        # of their own, then in a pool of shuffled 256-token pages
        Lq, Lk = 1024, gc["N"]
        cin = make_gda_inputs(gc["B"], Lk, gc["Hs"], gc["Hn"], gc["d"], gc["dv"], seed=5050 + rank,
                              device=dev)
        heads = gc["Hs"] + gc["Hn"]
        ck, cv = cin.k.reshape(-1, heads, gc["d"]), cin.v.reshape(-1, gc["Hs"], gc["dv"])
        cq = cin.q[:, Lk - Lq:].reshape(-1, heads, gc["d"]).contiguous()
        ccu_q = torch.arange(gc["B"] + 1, dtype=torch.int32, device=dev) * Lq
        ccu_k = torch.arange(gc["B"] + 1, dtype=torch.int32, device=dev) * Lk
        cout = torch.empty((gc["B"] * Lq, gc["Hs"], gc["dv"]), dtype=torch.bfloat16, device=dev)
        cws = torch.empty(da.diffattn_gda_fwd_workspace_size(gc["B"], Lq, gc["Hs"], gc["Hn"]),
                          dtype=torch.uint8, device=dev)
        t = timer(lambda: da.diffattn_gda_fwd_varlen_qk(cq, ck, cv, ccu_q, ccu_k, cin.lam, gc["Hs"],
                                                        li_g, max_seqlen_q=Lq, max_seqlen_k=Lk,
                                                        workspace=cws, out=cout),
                  max(5, min(50, args.steps)), status=status)
        cpairs = float(gc["B"] * gc["Hs"] * (Lq * (Lk - Lq) + Lq * (Lq + 1) // 2))
        r = tensor_roof(cpairs * method_per_pair, t, peaks, peak_src)
        extra["gda_chunk"] = compact(r["achieved"], "TFLOP/s", t, r,
                                     f"last {Lq}-query chunk of B{gc['B']} prompts over {Lk} keys, "
                                     f"12 signal heads over 3 noise heads", world,
                                     flops_per_pair=method_per_pair)
        cps = 256
        cmp_ = Lk // cps
        cgp = torch.Generator(device="cpu")
        cgp.manual_seed(5060 + rank)
        ctable = torch.randperm(gc["B"] * cmp_, generator=cgp).to(torch.int32).view(gc["B"], cmp_).to(dev)
        corder = torch.argsort(ctable.flatten())
        ck_pool = cin.k.reshape(gc["B"] * cmp_, cps, heads, gc["d"])[corder].contiguous()
        cv_pool = cin.v.reshape(gc["B"] * cmp_, cps, gc["Hs"], gc["dv"])[corder].contiguous()
        csk = torch.full((gc["B"],), Lk, dtype=torch.int32, device=dev)
        t = timer(lambda: da.diffattn_gda_fwd_paged(cq, ck_pool, cv_pool, ccu_q, csk, ctable,
                                                    cin.lam, gc["Hs"], li_g, max_seqlen_q=Lq,
                                                    max_seqlen_k=Lk, workspace=cws, out=cout),
                  max(5, min(50, args.steps)), status=status)
        r = tensor_roof(cpairs * method_per_pair, t, peaks, peak_src)
        extra["gda_chunk_paged"] = compact(r["achieved"], "TFLOP/s", t, r,
                                           f"the gda_chunk line, keys in shuffled {cps}-token pages",
                                           world, flops_per_pair=method_per_pair)
        del cin, ck, cv, cq, cout, cws, ck_pool, cv_pool, ctable
        torch.cuda.empty_cache()

        # the same heads over the packed sequences of the varlen line
        lens = varlen_lengths()
        total = int(sum(lens))
        vin = make_gda_inputs(1, total, gc["Hs"], gc["Hn"], gc["d"], gc["dv"], seed=5100 + rank,
                              device=dev)
        cu = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32, device=dev)
        vout = torch.empty((total, gc["Hs"], gc["dv"]), dtype=torch.bfloat16, device=dev)
        vws = torch.empty(da.diffattn_gda_fwd_workspace_size(len(lens), max(lens), gc["Hs"],
                                                             gc["Hn"]),
                          dtype=torch.uint8, device=dev)
        q, k, v = vin.q[0], vin.k[0], vin.v[0]
        t = timer(lambda: da.diffattn_gda_fwd_varlen(q, k, v, cu, vin.lam, gc["Hs"], li_g,
                                                     max_seqlen=max(lens), workspace=vws,
                                                     out=vout),
                  max(5, min(50, args.steps)), status=status)
        vpairs = float(sum(gc["Hs"] * causal_pairs(n) for n in lens))
        r = tensor_roof(vpairs * method_per_pair, t, peaks, peak_src)
        extra["gda_varlen"] = compact(r["achieved"], "TFLOP/s", t, r,
                                      f"{len(lens)} packed sequences ({total} tokens), 12 signal "
                                      f"heads over 3 noise heads", world,
                                      flops_per_pair=method_per_pair)
        del vin, vout, vws, q, k, v
        torch.cuda.empty_cache()

        gd = dict(GDA_DECODE, B=args.decode_batch)
        gdi = make_gda_decode_inputs(gd["B"], gd["L"], gd["Hs"], gd["Hn"], gd["d"], gd["dv"],
                                     seed=5100 + rank, device=dev)
        gws = torch.empty(da.diffattn_decode_workspace_size(gd["B"], gd["L"], gd["Hs"]),
                          dtype=torch.uint8, device=dev)
        gdout = torch.empty((gd["B"], gd["Hs"], gd["dv"]), dtype=torch.bfloat16, device=dev)
        t = timer(lambda: da.diffattn_gda_decode(gdi.q, gdi.k_cache, gdi.v_cache, gdi.lam,
                                                 gd["Hs"], li_g, workspace=gws, out=gdout),
                  max(5, min(50, args.steps)), status=status)
        gdbytes = gda_decode_bytes(gd)
        r = hbm_roof(gdbytes, t, peaks, peak_src)
        extra["gda_decode"] = compact(r["achieved"], "GB/s", t, r,
                                      f"decode_32k with 12 signal heads over 3 noise heads, B{gd['B']}",
                                      world, traffic=profiled_traffic(
                                          "gda_decode_32k.md", source_sha(["decode.cu", "ptx.cuh"])))

        # the same cache as pools of 64-token pages, each sequence's pages scattered over them
        gps = 64
        gmp = gd["L"] // gps
        gk_pool = gdi.k_cache.view(gd["B"] * gmp, gps, gd["Hs"] + gd["Hn"], gd["d"])
        gv_pool = gdi.v_cache.view(gd["B"] * gmp, gps, gd["Hs"], gd["dv"])
        ggp = torch.Generator(device="cpu")
        ggp.manual_seed(5200 + rank)
        gtable = torch.randperm(gd["B"] * gmp, generator=ggp).to(torch.int32).view(gd["B"], gmp).to(dev)
        t = timer(lambda: da.diffattn_gda_decode_paged(gdi.q, gk_pool, gv_pool, gtable, gdi.seqlens,
                                                       gdi.lam, gd["Hs"], li_g, workspace=gws,
                                                       out=gdout),
                  max(5, min(50, args.steps)), status=status)
        r = hbm_roof(gdbytes, t, peaks, peak_src)
        extra["gda_decode_paged"] = compact(r["achieved"], "GB/s", t, r,
                                            f"gda_decode_32k in shuffled {gps}-token pages", world)
        del gdi, gws, gdout, gk_pool, gv_pool, gtable
        torch.cuda.empty_cache()

        # training on the grouped prefill: forward saving statistics, then every gradient
        ginp = make_gda_inputs(gc["B"], gc["N"], gc["Hs"], gc["Hn"], gc["d"], gc["dv"],
                               seed=5000 + rank, device=dev)
        gws = torch.empty(da.diffattn_gda_fwd_workspace_size(gc["B"], gc["N"], gc["Hs"], gc["Hn"]),
                          dtype=torch.uint8, device=dev)
        gdy = make_dout(gc["B"], gc["N"], gc["Hs"], gc["dv"], seed=5300 + rank, device=dev)
        gw = torch.ones(gc["dv"], dtype=torch.float32, device=dev)
        gbws = torch.empty(da.diffattn_gda_bwd_workspace_size(gc["B"], gc["N"], gc["Hs"], gc["Hn"]),
                           dtype=torch.uint8, device=dev)
        ggrads = dict(dq=torch.empty_like(ginp.q), dk=torch.empty_like(ginp.k),
                      dv=torch.empty_like(ginp.v),
                      dlam=torch.empty(gc["Hs"], dtype=torch.float32, device=dev),
                      dw=torch.empty(gc["dv"], dtype=torch.float32, device=dev))
        gsaved = {}

        def gfwd():
            gsaved["out"], gsaved["o_pre"], gsaved["stats"] = da.diffattn_gda_fwd_train(
                ginp.q, ginp.k, ginp.v, ginp.lam, gc["Hs"], li_g, norm_weight=gw, workspace=gws)

        def gbwd():
            da.diffattn_gda_bwd(ginp.q, ginp.k, ginp.v, gsaved["o_pre"], gsaved["stats"], gdy,
                                ginp.lam, gc["Hs"], li_g, norm_weight=gw, workspace=gbws,
                                grads=ggrads)

        n_steps = max(3, min(20, args.steps))
        tf_ = timer(gfwd, n_steps, status=status)
        tb = timer(gbwd, n_steps, status=status)
        # per (signal head, causal pair): the V1 count with the noise map's scores formed once per
        # group (2d / G instead of 2d)
        gbwd_per_pair = BWD_FLOPS_PER_PAIR - 2 * gc["d"] + 2 * gc["d"] / G
        gpairs = float(gc["B"] * gc["Hs"] * causal_pairs(gc["N"]))
        r = tensor_roof(gpairs * gbwd_per_pair, tb, peaks, peak_src)
        extra["gda_backward"] = compact(r["achieved"], "TFLOP/s", tb, r,
                                        "gda_prefill training: every gradient", world,
                                        flops_per_pair=gbwd_per_pair,
                                        fwd_train_ms=round(tf_["ms"], 4))
        del ginp, gws, gdy, gbws, ggrads, gsaved
        torch.cuda.empty_cache()

        # the grouped backward over the packed sequences of the varlen line
        lens = varlen_lengths()
        total, mx = int(sum(lens)), max(lens)
        vin = make_gda_inputs(1, total, gc["Hs"], gc["Hn"], gc["d"], gc["dv"], seed=5400 + rank,
                              device=dev)
        q, k, v = vin.q[0], vin.k[0], vin.v[0]
        vdy = make_dout(1, total, gc["Hs"], gc["dv"], seed=5407 + rank, device=dev)[0]
        cu = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32, device=dev)
        _, o_pre, stats = da.diffattn_gda_fwd_train_varlen(q, k, v, cu, vin.lam, gc["Hs"], li_g,
                                                           max_seqlen=mx, norm_weight=gw)
        vbws = torch.empty(da.diffattn_gda_bwd_varlen_workspace_size(len(lens), mx, total,
                                                                     gc["Hs"], gc["Hn"]),
                           dtype=torch.uint8, device=dev)
        vgrads = dict(dq=torch.empty_like(q), dk=torch.empty_like(k), dv=torch.empty_like(v),
                      dlam=torch.empty(gc["Hs"], dtype=torch.float32, device=dev),
                      dw=torch.empty(gc["dv"], dtype=torch.float32, device=dev))
        t = timer(lambda: da.diffattn_gda_bwd_varlen(q, k, v, o_pre, stats, vdy, cu, vin.lam,
                                                     gc["Hs"], li_g, max_seqlen=mx,
                                                     norm_weight=gw, workspace=vbws,
                                                     grads=vgrads), n_steps, status=status)
        vpairs = float(sum(gc["Hs"] * causal_pairs(n) for n in lens))
        r = tensor_roof(vpairs * gbwd_per_pair, t, peaks, peak_src)
        extra["gda_backward_varlen"] = compact(r["achieved"], "TFLOP/s", t, r,
                                               f"grouped backward over the {len(lens)} packed "
                                               f"sequences", world, flops_per_pair=gbwd_per_pair)
        del vin, q, k, v, vdy, o_pre, stats, vbws, vgrads, gw
        torch.cuda.empty_cache()

    # ======================= V2 decode =======================
    if want("v2_decode"):
        c = dict(V2_DECODE, B=args.decode_batch)
        vd = make_v2_decode_inputs(c["B"], c["L"], c["Hq"], c["Hkv"], c["d"], seed=5000 + rank,
                                   device=dev)
        ws = torch.empty(da.diffattn_v2_decode_workspace_size(c["B"], c["L"], c["Hq"], c["Hkv"],
                                                              c["d"]), dtype=torch.uint8, device=dev)
        vdout = torch.empty((c["B"], c["Hq"] // 2, c["d"]), dtype=torch.bfloat16, device=dev)
        n_steps = max(5, min(50, args.steps))
        t = timer(lambda: da.diffattn_v2_decode(vd.q, vd.k_cache, vd.v_cache, vd.lam_logit,
                                                workspace=ws, out=vdout), n_steps, status=status)
        nbytes = v2_decode_bytes(c)
        r = hbm_roof(nbytes, t, peaks, peak_src)
        extra["v2_decode"] = compact(r["achieved"], "GB/s", t, r,
                                     f"B{c['B']} cache 32768, Hq64 over Hkv8, d128", world,
                                     traffic=profiled_traffic(
                                         "v2_decode_32k.md", source_sha(["decode_v2_tc.cu", "ptx.cuh"])))

        # fp8 e4m3 q and K cache (per-tensor scales), V bf16: 3/4 of the bytes for every key
        q8, qds = to_fp8_e4m3(vd.q)
        k8, kds = to_fp8_e4m3(vd.k_cache)
        t8 = timer(lambda: da.diffattn_v2_decode_fp8(q8, k8, vd.v_cache, vd.lam_logit, qds, kds,
                                                     workspace=ws, out=vdout), n_steps, status=status)
        r8 = hbm_roof(nbytes * 3 / 4, t8, peaks, peak_src)
        extra["v2_decode_fp8"] = compact(r8["achieved"], "GB/s", t8, r8,
                                         "v2_decode_32k, fp8 e4m3 q and K cache, bf16 V", world,
                                         speedup_vs_bf16_cache=round(t["ms"] / t8["ms"], 3))
        del q8, k8

        # the same cache as pools of pages placed in a random order
        for ps in (64, 16):
            mp = c["L"] // ps
            k_pool = vd.k_cache.view(c["B"] * mp, ps, c["Hkv"], c["d"])
            v_pool = vd.v_cache.view(c["B"] * mp, ps, c["Hkv"], c["d"])
            gp = torch.Generator(device="cpu")
            gp.manual_seed(5100 + ps + rank)
            table = torch.randperm(c["B"] * mp, generator=gp).to(torch.int32).view(c["B"], mp).to(dev)
            tp = timer(lambda: da.diffattn_v2_decode_paged(vd.q, k_pool, v_pool, table, vd.seqlens,
                                                           vd.lam_logit, workspace=ws, out=vdout),
                       n_steps, status=status)
            rp = hbm_roof(nbytes, tp, peaks, peak_src)
            extra[f"v2_decode_paged_{ps}"] = compact(rp["achieved"], "GB/s", tp, rp,
                                                     f"v2_decode_32k in shuffled {ps}-token pages",
                                                     world)
            del k_pool, v_pool, table
        del vd, ws, vdout
        torch.cuda.empty_cache()

    # ======================= decode (config of the metric's second half) =======================
    if want("decode"):
        dcfg = dict(DECODE, B=args.decode_batch)
        dinp = make_decode_inputs(dcfg["B"], dcfg["L"], dcfg["H"], dcfg["d"], dcfg["dv"],
                                  seed=2000 + rank, device=dev)
        ws = torch.empty(da.diffattn_decode_workspace_size(dcfg["B"], dcfg["L"], dcfg["H"]),
                         dtype=torch.uint8, device=dev)
        dout = torch.empty((dcfg["B"], dcfg["H"], dcfg["dv"]), dtype=torch.bfloat16, device=dev)
        li_dec = da.diffattn_lambda_init(dcfg["layer"])
        dbytes = decode_bytes(dcfg)

        # the same cache as a pool of 64-token pages, each sequence's pages scattered over it
        ps = 64
        mp = dcfg["L"] // ps
        k_pool = dinp.k_cache.view(dcfg["B"] * mp, ps, dcfg["H"], 2 * dcfg["d"])
        v_pool = dinp.v_cache.view(dcfg["B"] * mp, ps, dcfg["H"], dcfg["dv"])
        gp = torch.Generator(device="cpu")
        gp.manual_seed(2100 + rank)
        table = torch.randperm(dcfg["B"] * mp, generator=gp).to(torch.int32).view(dcfg["B"], mp).to(dev)
        tp = timer(lambda: da.diffattn_decode_paged(dinp.q, k_pool, v_pool, table, dinp.seqlens,
                                                    dinp.lam, li_dec, workspace=ws, out=dout),
                   max(5, min(50, args.steps)), status=status)
        rp = hbm_roof(dbytes, tp, peaks, peak_src)
        extra["decode_paged"] = compact(rp["achieved"], "GB/s", tp, rp,
                                        "decode_32k in shuffled 64-token pages", world)

        # the headline decode loop: long enough (>= ~0.7 s) for its own clock record; the 25.8 GB
        # cache is 200x the L2, so every call streams it from HBM
        n_dec = max(5, min(200, 10 * args.steps))
        t = timer(lambda: da.diffattn_decode(dinp.q, dinp.k_cache, dinp.v_cache, dinp.lam, li_dec,
                                             workspace=ws, out=dout), n_dec, clocks=True,
                  status=status)
        dms = max_over_ranks(t["ms"])
        t["ms"] = dms
        r = hbm_roof(dbytes, t, peaks, peak_src)
        r.update({"traffic": profiled_traffic("decode_32k.md", source_sha(["decode.cu", "ptx.cuh"])),
                  "bytes_per_launch": dbytes})
        decode_blk = {
            "metric": "decode HBM GB/s", "value": world * r["achieved"], "unit": "GB/s",
            "ms_per_call": dms, "calls": n_dec,
            "workload": f"decode_32k: B{dcfg['B']} x 1 query, cache 32768, H12, d128, dv256, bf16 "
                        "(25.8 GB, read once per call)",
            "frac": r["frac"], "frac_nominal": r["frac_nominal"],
            "roofline": r, "clocks": t["clocks"], "gpu_launches": 2 * n_dec}
        del dinp, ws, dout, k_pool, v_pool, table
        torch.cuda.empty_cache()

    # ======================= CPU baseline (rank 0, N = 1 only) =======================
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and args.only == "all":
        v, cores, desc, _, _ = oracle_sample(args.cpu_seconds)
        cpu = {"value": v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": desc}

    # the secondary workloads first, then the CPU baseline, the headline figures, and the
    # decode block last (the end of the line is what a truncated log keeps)
    line.update(extra)
    line["cpu_baseline"] = cpu
    head = {}
    if line.get("roofline"):
        head.update({"prefill_3b_tflops": round(line["roofline"]["achieved"], 1),
                     "prefill_frac": round(line["roofline"]["frac"], 4),
                     "prefill_frac_nominal": round(line["roofline"]["frac_nominal"], 4)})
    if decode_blk:
        head.update({"decode_32k_gbs": round(decode_blk["value"], 1),
                     "decode_frac": round(decode_blk["frac"], 4),
                     "decode_frac_nominal": round(decode_blk["frac_nominal"], 4)})
    line["headline"] = head
    line["decode"] = decode_blk
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", choices=["all", "prefill", "decode", "v2", "v2_decode", "long", "backward", "varlen", "fp8", "gda"], default="all",
                    help="profiling aid: run one workload (the JSON line then lacks the others)")
    ap.add_argument("--decode-batch", type=int, default=DECODE["B"],
                    help="profiling aid: a smaller decode batch for captures that save device memory")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and args.impl == "ours":
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local_rank)
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
