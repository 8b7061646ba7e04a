"""Benchmark of the differential-attention hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one pass of the prefill hot path on the 3B-layer workload (B 4, N 4096, 12 heads,
d 128, dv 256, causal, bf16): the lambda kernel (exp reparameterisation) followed by the fused
DiffAttn prefill with RMSNorm and (1 - lambda_init) epilogue. `value` is TFLOP/s counted at 1536
MMA flops per causal query-key pair (4d for the two score maps + 4dv for the two value products),
summed over ranks (weak scaling: every rank runs its own batch). The same JSON line carries the
decode workload (B 64, cache 32768, 12 heads: HBM GB/s) and the V2 GQA workload as secondary
objects, the roofline of the dominant kernel, the clocks seen during the timed region, an
end-to-end number through host buffers, and the float64 oracle timed on the host cores.

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
def run_ours(args, rank: int, world: int, local_rank: int):
    import torch
    import torch.distributed as dist
    import differential_attention_gb300 as da
    from synth import (make_decode_inputs, make_dout, make_gda_decode_inputs, make_gda_inputs,
                       make_lambda_vectors, make_prefill_inputs, make_v2_decode_inputs,
                       make_v2_inputs, to_fp8_e4m3)

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    da.build()
    peaks, peak_src = load_peaks()
    stream = torch.cuda.current_stream()
    peak_tf = peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
    hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])

    def barrier():
        dist_barrier()

    def max_over_ranks(x: float) -> float:
        return dist_max(x, dev)

    def ev():
        return torch.cuda.Event(enable_timing=True)

    line = {"metric": "DiffAttn fwd TFLOP/s (% dense BF16 TC peak); decode HBM GB/s (% peak)",
            "value": None, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": None, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic"}

    # ======================= prefill: the step that `value` measures =======================
    if args.only in ("all", "prefill"):
        c = PREFILL
        inp = make_prefill_inputs(c["B"], c["N"], c["H"], c["d"], c["dv"], seed=1000 + rank,
                                  layer=c["layer"], device=dev)
        # one lambda per layer, shared by every head ([P3]), formed inside the prefill kernel
        lv = tuple(t.to(dev).contiguous() for t in make_lambda_vectors(c["d"], seed=1001 + rank))
        out = torch.empty((c["B"], c["N"], c["H"], c["dv"]), dtype=torch.bfloat16, device=dev)

        def step(q, k, v):
            da.diffattn_fwd_fused_lambda(q, k, v, *lv, layer=c["layer"], out=out)

        for _ in range(args.warmup):
            step(inp.q, inp.k, inp.v)
        da.diffattn_device_status()
        kev = [(ev(), ev()) for _ in range(args.steps)]
        with ClockSampler(dev.index) as clk:
            barrier()
            t_start, t_end = ev(), ev()
            t_start.record(stream)
            for i in range(args.steps):
                kev[i][0].record(stream)
                step(inp.q, inp.k, inp.v)
                kev[i][1].record(stream)
            t_end.record(stream)
            barrier()
        da.diffattn_device_status()
        total_ms = max_over_ranks(t_start.elapsed_time(t_end))
        ms_per_step = total_ms / args.steps
        kernel_ms = statistics.mean(a.elapsed_time(b) for a, b in kev)
        flops = prefill_flops()
        achieved = flops / (kernel_ms * 1e-3) / 1e12
        sha = source_sha(["prefill_exact.cu", "ptx.cuh"])
        line.update({
            "value": world * flops / (ms_per_step * 1e-3) / 1e12,
            "ms_per_step": ms_per_step,
            "config": {"workload": PREFILL_WORKLOAD,
                       "global_batch": PREFILL["B"] * world, "seq_len": PREFILL["N"],
                       "parallelism": f"replicas x{world} (independent batches, no collective)",
                       "l2": "inputs larger than L2 (q, k, v = 302 MB per rank)",
                       "flops_per_pair": FLOPS_PER_PAIR},
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak_tf,
                         "unit": "TFLOP/s", "frac": achieved / peak_tf,
                         "traffic": profiled_traffic("prefill_exact_3b.md", sha),
                         "kernel": "prefill_exact_kernel<128,256,false>", "kernel_ms": kernel_ms,
                         "flops_per_launch": flops,
                         "peak_source": f"bf16_tflops_sustained of {peak_src} (kernel run back to back)",
                         "definition_count_tflops":
                             flops / FLOPS_PER_PAIR * FLOPS_PER_PAIR_DEF / (kernel_ms * 1e-3) / 1e12},
            "gpu_launches": args.steps,
            "clocks": clk.summary(),
        })

        # ---------------- end to end through host buffers ----------------
        e2e_steps = max(3, min(20, args.steps))
        hq, hk, hv = (t.cpu().pin_memory() for t in (inp.q, inp.k, inp.v))
        hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        hws = torch.empty(da.diffattn_fwd_host_workspace_size(c["B"], c["N"], c["H"], c["d"], c["dv"]),
                          dtype=torch.uint8, device=dev)

        def e2e_step():
            da.diffattn_fwd_host(hq, hk, hv, hout, *lv, layer=c["layer"], workspace=hws)

        e2e_step()
        barrier()
        e0, e1 = ev(), ev()
        e0.record(stream)
        for _ in range(e2e_steps):
            e2e_step()
        e1.record(stream)
        barrier()
        e2e_ms = max_over_ranks(e0.elapsed_time(e1)) / e2e_steps
        line["e2e"] = {"value": world * flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                       "h2d_bytes_per_step": 3 * inp.q.numel() * 2,
                       "d2h_bytes_per_step": out.numel() * 2, "ms_per_step": e2e_ms,
                       "via": "diffattn_fwd_host: pinned host q, k, v in and out, copies of "
                              "each sequence overlapped with the prefill of the others"}
        del inp, out, hq, hk, hv, hout, hws
        torch.cuda.empty_cache()

    # ======================= decode =======================
    if args.only in ("all", "decode"):
        dcfg = dict(DECODE, B=args.decode_batch)
        dinp = make_decode_inputs(dcfg["B"], dcfg["L"], dcfg["H"], dcfg["d"], dcfg["dv"],
                                  seed=2000 + rank, device=dev)
        ws = torch.empty(da.diffattn_decode_workspace_size(dcfg["B"], dcfg["L"], dcfg["H"]),
                         dtype=torch.uint8, device=dev)
        dout = torch.empty((dcfg["B"], dcfg["H"], dcfg["dv"]), dtype=torch.bfloat16, device=dev)
        li_dec = da.diffattn_lambda_init(dcfg["layer"])

        def dec():
            da.diffattn_decode(dinp.q, dinp.k_cache, dinp.v_cache, dinp.lam, li_dec, workspace=ws,
                               out=dout)

        for _ in range(args.warmup):
            dec()
        barrier()
        dsteps = max(5, min(50, args.steps))
        dev_ev = [(ev(), ev()) for _ in range(dsteps)]
        for i in range(dsteps):
            dev_ev[i][0].record(stream)
            dec()
            dev_ev[i][1].record(stream)
        barrier()
        da.diffattn_device_status()
        dms = statistics.mean(a.elapsed_time(b) for a, b in dev_ev)
        dbytes = decode_bytes(dcfg)
        dgbs = dbytes / (dms * 1e-3) / 1e9
        dsha = source_sha(["decode.cu", "ptx.cuh"])
        line["decode"] = {
            "metric": "decode HBM GB/s", "value": world * dgbs, "unit": "GB/s", "ms_per_call": dms,
            "workload": f"decode_32k: B{dcfg['B']}, one query per sequence, cache 32768, H12, "
                        "d128, dv256, bf16 (cache 25.8 GB at B64, larger than L2)",
            "roofline": {"bound": "hbm", "achieved": dgbs, "peak": hbm, "unit": "GB/s",
                         "frac": dgbs / hbm, "traffic": profiled_traffic("decode_32k.md", dsha),
                         "bytes_per_launch": dbytes,
                         "peak_source": f"hbm_gbs of {peak_src} (copy, read+write)",
                         "timed": "diffattn_decode call (split kernel + combine kernel)"},
            "gpu_launches": 2 * dsteps}

        # the same cache as a pool of 64-token pages, each sequence's pages scattered over it
        ps = 64
        mp = dcfg["L"] // ps
        k_pool = dinp.k_cache.view(dcfg["B"] * mp, ps, dcfg["H"], 2 * dcfg["d"])
        v_pool = dinp.v_cache.view(dcfg["B"] * mp, ps, dcfg["H"], dcfg["dv"])
        gp = torch.Generator(device="cpu")
        gp.manual_seed(2100 + rank)
        table = torch.randperm(dcfg["B"] * mp, generator=gp).to(torch.int32).view(dcfg["B"], mp).to(dev)

        def dec_paged():
            da.diffattn_decode_paged(dinp.q, k_pool, v_pool, table, dinp.seqlens, dinp.lam, li_dec,
                                     workspace=ws, out=dout)

        for _ in range(args.warmup):
            dec_paged()
        barrier()
        pev = [(ev(), ev()) for _ in range(dsteps)]
        for i in range(dsteps):
            pev[i][0].record(stream)
            dec_paged()
            pev[i][1].record(stream)
        barrier()
        da.diffattn_device_status()
        pms = statistics.mean(a.elapsed_time(b) for a, b in pev)
        pgbs = dbytes / (pms * 1e-3) / 1e9
        line["decode_paged"] = {
            "metric": "decode HBM GB/s", "value": world * pgbs, "unit": "GB/s", "ms_per_call": pms,
            "workload": f"decode_32k over a paged cache: B{dcfg['B']}, cache 32768 in 64-token pages "
                        "placed in a random order in the pool, H12, d128, dv256, bf16",
            "roofline": {"bound": "hbm", "achieved": pgbs, "peak": hbm, "unit": "GB/s",
                         "frac": pgbs / hbm, "bytes_per_launch": dbytes,
                         "peak_source": f"hbm_gbs of {peak_src} (copy, read+write)",
                         "timed": "diffattn_decode_paged call (split kernel + combine kernel)"},
            "gpu_launches": 2 * dsteps}
        del dinp, ws, dout, k_pool, v_pool, table
        torch.cuda.empty_cache()

    # ======================= long-context prefill =======================
    if args.only in ("all", "long"):
        c = LONG
        inp = make_prefill_inputs(c["B"], c["N"], c["H"], c["d"], c["dv"], seed=4000 + rank,
                                  layer=c["layer"], device=dev, needle=True)
        lv = tuple(t.to(dev).contiguous() for t in make_lambda_vectors(c["d"], seed=4001 + rank))
        out = torch.empty((c["B"], c["N"], c["H"], c["dv"]), dtype=torch.bfloat16, device=dev)

        def lstep():
            da.diffattn_fwd_fused_lambda(inp.q, inp.k, inp.v, *lv, layer=c["layer"], out=out)

        for _ in range(args.warmup):
            lstep()
        barrier()
        lsteps = max(3, min(10, args.steps))
        l_ev = [(ev(), ev()) for _ in range(lsteps)]
        for i in range(lsteps):
            l_ev[i][0].record(stream)
            lstep()
            l_ev[i][1].record(stream)
        barrier()
        da.diffattn_device_status()
        lms = statistics.mean(a.elapsed_time(b) for a, b in l_ev)
        lflops = prefill_flops(c)
        ltf = lflops / (lms * 1e-3) / 1e12
        line["prefill_64k"] = {
            "metric": "DiffAttn fwd TFLOP/s", "value": world * ltf, "unit": "TFLOP/s",
            "ms_per_call": lms,
            "workload": "prefill_64k: B1 N65536 H12 d128 dv256 causal, layer 24, one needle key per head",
            "roofline": {"bound": "tensor", "achieved": ltf, "peak": peak_tf, "unit": "TFLOP/s",
                         "frac": ltf / peak_tf, "flops_per_launch": lflops}}
        del inp, out
        torch.cuda.empty_cache()

    # ======================= V2 =======================
    if args.only in ("all", "v2"):
        vc = V2
        vinp = make_v2_inputs(vc["B"], vc["N"], vc["Hq"], vc["Hkv"], vc["d"], seed=3000 + rank,
                              device=dev)
        vout = torch.empty((vc["B"], vc["N"], vc["Hq"] // 2, vc["d"]), dtype=torch.bfloat16,
                           device=dev)

        def v2():
            da.diffattn_v2_fwd(vinp.q, vinp.k, vinp.v, vinp.lam_logit, out=vout)

        for _ in range(args.warmup):
            v2()
        barrier()
        vsteps = max(5, min(30, args.steps))
        v_ev = [(ev(), ev()) for _ in range(vsteps)]
        for i in range(vsteps):
            v_ev[i][0].record(stream)
            v2()
            v_ev[i][1].record(stream)
        barrier()
        da.diffattn_device_status()
        vms = statistics.mean(a.elapsed_time(b) for a, b in v_ev)
        # the exact two-pass path (DIFFATTN_EXACT) on the same inputs, for context
        x_ev = [(ev(), ev()) for _ in range(5)]
        for a, b_ in x_ev:
            a.record(stream)
            da.diffattn_v2_fwd(vinp.q, vinp.k, vinp.v, vinp.lam_logit, out=vout, exact=True)
            b_.record(stream)
        barrier()
        da.diffattn_device_status()
        xms = statistics.mean(a.elapsed_time(b_) for a, b_ in x_ev)
        vflops = float(vc["B"] * (vc["Hq"] // 2) * causal_pairs(vc["N"]) * V2_FLOPS_PER_PAIR)
        vtf = vflops / (vms * 1e-3) / 1e12
        line["v2"] = {"metric": "V2 fwd TFLOP/s", "value": world * vtf, "unit": "TFLOP/s",
                      "ms_per_call": vms,
                      "workload": "v2_gqa: B2 N8192 Hq64 (32 pairs) Hkv8 d128 causal",
                      "kernel": "v2_pair_kernel<128,2> (both heads of a pair in one CTA, one "
                                "flash pass per head)",
                      "exact_two_pass_ms": xms,
                      "roofline": {"bound": "tensor", "achieved": vtf, "peak": peak_tf,
                                   "unit": "TFLOP/s", "frac": vtf / peak_tf,
                                   "flops_per_launch": vflops,
                                   "traffic": profiled_traffic(
                                       "v2_pair_gqa.md",
                                       source_sha(["prefill_v2.cu", "ptx.cuh"]))}}
        del vinp, vout
        torch.cuda.empty_cache()

    # ======================= prefill with fp8 scores =======================
    if args.only in ("all", "fp8"):
        c = PREFILL
        inp = make_prefill_inputs(c["B"], c["N"], c["H"], c["d"], c["dv"], seed=9000 + rank,
                                  layer=c["layer"], device=dev)
        q8, qs = to_fp8_e4m3(inp.q)
        k8, ks = to_fp8_e4m3(inp.k)
        lam = torch.full((c["H"],), 0.6, dtype=torch.float32, device=dev)
        li = da.diffattn_lambda_init(c["layer"])
        out = torch.empty((c["B"], c["N"], c["H"], c["dv"]), dtype=torch.bfloat16, device=dev)

        def f8step():
            da.diffattn_fwd_fp8(q8, k8, inp.v, lam, qs, ks, li, out=out)

        for _ in range(args.warmup):
            f8step()
        barrier()
        n_steps = max(5, min(200, args.steps))
        evs = [(ev(), ev()) for _ in range(n_steps)]
        for i in range(n_steps):
            evs[i][0].record(stream)
            f8step()
            evs[i][1].record(stream)
        barrier()
        da.diffattn_device_status()
        ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
        f8flops = prefill_flops()
        f8tf = f8flops / (ms * 1e-3) / 1e12
        # 1024 of the 1536 flops per pair are score products on the fp8 tensor cores (twice the
        # bf16 rate by the nominal ratio), 512 the bf16 product with V: blended peak 1.5x bf16
        blend = 1.5 * peak_tf
        line["prefill_fp8"] = {
            "metric": "DiffAttn fwd TFLOP/s", "value": world * f8tf, "unit": "TFLOP/s",
            "ms_per_call": ms,
            "workload": "prefill_3b (B4 N4096 H12 d128 dv256 causal) with fp8 e4m3 q and k "
                        "(per-tensor absmax scale), bf16 v and output",
            "roofline": {"bound": "tensor", "achieved": f8tf, "peak": blend, "unit": "TFLOP/s",
                         "frac": f8tf / blend, "flops_per_launch": f8flops,
                         "peak_source": "1.5 x bf16_tflops_sustained: scores at the fp8 rate "
                                        "(2x bf16, nominal ratio), the V product at the bf16 rate"},
            "gpu_launches": n_steps}
        del inp, q8, k8, out
        torch.cuda.empty_cache()

    # ======================= variable-length prefill (packed sequences) =======================
    if args.only in ("all", "varlen"):
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

        def vstep():
            da.diffattn_fwd_varlen(q, k, v, cu, lam, li, max_seqlen=max(lens), out=out)

        for _ in range(args.warmup):
            vstep()
        barrier()
        n_steps = max(5, min(50, args.steps))
        evs = [(ev(), ev()) for _ in range(n_steps)]
        for i in range(n_steps):
            evs[i][0].record(stream)
            vstep()
            evs[i][1].record(stream)
        barrier()
        da.diffattn_device_status()
        ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
        vflops = float(sum(c["H"] * causal_pairs(n) * FLOPS_PER_PAIR for n in lens))
        vtf = vflops / (ms * 1e-3) / 1e12
        line["varlen"] = {
            "metric": "DiffAttn fwd TFLOP/s", "value": world * vtf, "unit": "TFLOP/s",
            "ms_per_call": ms,
            "workload": f"prefill_3b shapes over {len(lens)} packed sequences of mixed length "
                        f"(seeded, {min(lens)}..{max(lens)} tokens, {total} in total), causal, H12",
            "roofline": {"bound": "tensor", "achieved": vtf, "peak": peak_tf, "unit": "TFLOP/s",
                         "frac": vtf / peak_tf, "flops_per_launch": vflops},
            "gpu_launches": n_steps}
        del inp, out, q, k, v
        torch.cuda.empty_cache()

        # the last 1024-token chunk of each prefill_3b prompt against its 4096 keys (queries and
        # keys with offsets of their own)
        Lq, Lk = 1024, c["N"]
        kin = make_prefill_inputs(c["B"], Lk, c["H"], c["d"], c["dv"], seed=8100 + rank,
                                  layer=c["layer"], device=dev)
        k, v = kin.k.reshape(-1, c["H"], 2 * c["d"]), kin.v.reshape(-1, c["H"], c["dv"])
        q = kin.q[:, Lk - Lq:].reshape(-1, c["H"], 2 * c["d"]).contiguous()
        cu_q = torch.arange(c["B"] + 1, dtype=torch.int32, device=dev) * Lq
        cu_k = torch.arange(c["B"] + 1, dtype=torch.int32, device=dev) * Lk
        out = torch.empty((c["B"] * Lq, c["H"], c["dv"]), dtype=torch.bfloat16, device=dev)

        def cstep():
            da.diffattn_fwd_varlen_qk(q, k, v, cu_q, cu_k, lam, li, max_seqlen_q=Lq,
                                      max_seqlen_k=Lk, out=out)

        for _ in range(args.warmup):
            cstep()
        barrier()
        evs = [(ev(), ev()) for _ in range(n_steps)]
        for i in range(n_steps):
            evs[i][0].record(stream)
            cstep()
            evs[i][1].record(stream)
        barrier()
        da.diffattn_device_status()
        ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
        pairs = Lq * (Lk - Lq) + Lq * (Lq + 1) // 2  # query at position p sees p + 1 keys
        cflops = float(c["B"] * c["H"] * pairs * FLOPS_PER_PAIR)
        ctf = cflops / (ms * 1e-3) / 1e12
        line["varlen_qk"] = {
            "metric": "DiffAttn fwd TFLOP/s", "value": world * ctf, "unit": "TFLOP/s",
            "ms_per_call": ms,
            "workload": f"prefill_3b prompts computed as a last chunk: B{c['B']}, {Lq} queries "
                        f"against {Lk} keys each, causal, H12, d128, dv256",
            "roofline": {"bound": "tensor", "achieved": ctf, "peak": peak_tf, "unit": "TFLOP/s",
                         "frac": ctf / peak_tf, "flops_per_launch": cflops},
            "gpu_launches": n_steps}

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

        def pstep():
            da.diffattn_fwd_paged(q, k_pool, v_pool, cu_q, sk, table, lam, li, max_seqlen_q=Lq,
                                  max_seqlen_k=Lk, out=out)

        for _ in range(args.warmup):
            pstep()
        barrier()
        evs = [(ev(), ev()) for _ in range(n_steps)]
        for i in range(n_steps):
            evs[i][0].record(stream)
            pstep()
            evs[i][1].record(stream)
        barrier()
        da.diffattn_device_status()
        ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
        ptf = cflops / (ms * 1e-3) / 1e12
        line["paged_prefill"] = {
            "metric": "DiffAttn fwd TFLOP/s", "value": world * ptf, "unit": "TFLOP/s",
            "ms_per_call": ms,
            "workload": f"the varlen_qk chunk with the keys in {ps}-token pages placed in a random "
                        "order in the pool",
            "roofline": {"bound": "tensor", "achieved": ptf, "peak": peak_tf, "unit": "TFLOP/s",
                         "frac": ptf / peak_tf, "flops_per_launch": cflops},
            "gpu_launches": n_steps}
        del kin, out, q, k, v, k_pool, v_pool, table
        torch.cuda.empty_cache()

    # ======================= training step: forward (saving statistics) + backward ==========
    if args.only in ("all", "backward"):
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

        for _ in range(args.warmup):
            fwd()
            bwd()
        barrier()
        n_steps = max(3, min(20, args.steps))
        ev_f = [(ev(), ev()) for _ in range(n_steps)]
        ev_b = [(ev(), ev()) for _ in range(n_steps)]
        for i in range(n_steps):
            ev_f[i][0].record(stream)
            fwd()
            ev_f[i][1].record(stream)
            ev_b[i][0].record(stream)
            bwd()
            ev_b[i][1].record(stream)
        barrier()
        da.diffattn_device_status()
        fms = statistics.mean(a.elapsed_time(b) for a, b in ev_f)
        bms = statistics.mean(a.elapsed_time(b) for a, b in ev_b)
        pairs = c["B"] * c["H"] * causal_pairs(c["N"])
        bflops = float(pairs * BWD_FLOPS_PER_PAIR)
        btf = bflops / (bms * 1e-3) / 1e12
        line["backward"] = {
            "metric": "DiffAttn bwd TFLOP/s", "value": world * btf, "unit": "TFLOP/s",
            "ms_per_call": bms, "fwd_train_ms": fms,
            "workload": "prefill_3b training step: B4 N4096 H12 d128 dv256 causal, norm + scale; "
                        "forward with saved statistics, then every gradient",
            "roofline": {"bound": "tensor", "achieved": btf, "peak": peak_tf, "unit": "TFLOP/s",
                         "frac": btf / peak_tf, "flops_per_launch": bflops,
                         "flops_per_pair": BWD_FLOPS_PER_PAIR,
                         "issued_flops_per_pair": BWD_ISSUED_FLOPS_PER_PAIR,
                         "traffic": profiled_traffic("backward_dkdq_3b.md",
                                                     source_sha(["backward.cu", "ptx.cuh"])),
                         "traffic_kernel": "bwd_dkdq_kernel (the largest of the five)"},
            "gpu_launches": 5 * n_steps}
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

        def bwd_packed():
            da.diffattn_bwd_varlen(q, k, v, o_pre, stats, dyp, cu, lam, li, max_seqlen=mx,
                                   norm_weight=w, workspace=ws, grads=grads)

        for _ in range(args.warmup):
            bwd_packed()
        barrier()
        evs = [(ev(), ev()) for _ in range(n_steps)]
        for i in range(n_steps):
            evs[i][0].record(stream)
            bwd_packed()
            evs[i][1].record(stream)
        barrier()
        da.diffattn_device_status()
        ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
        vflops = float(sum(c["H"] * causal_pairs(n) * BWD_FLOPS_PER_PAIR for n in lens))
        vtf = vflops / (ms * 1e-3) / 1e12
        line["backward_varlen"] = {
            "metric": "DiffAttn bwd TFLOP/s", "value": world * vtf, "unit": "TFLOP/s",
            "ms_per_call": ms,
            "workload": f"backward over {len(lens)} packed sequences of mixed length ({min(lens)}.."
                        f"{max(lens)} tokens, {total} in total), causal, H12, norm + scale",
            "roofline": {"bound": "tensor", "achieved": vtf, "peak": peak_tf, "unit": "TFLOP/s",
                         "frac": vtf / peak_tf, "flops_per_launch": vflops},
            "gpu_launches": 5 * n_steps}
        del pin, q, k, v, dyp, o_pre, stats, ws, grads
        torch.cuda.empty_cache()

    # ======================= V2 decode =======================
    if args.only in ("all", "v2_decode"):
        c = dict(V2_DECODE, B=args.decode_batch)
        vd = make_v2_decode_inputs(c["B"], c["L"], c["Hq"], c["Hkv"], c["d"], seed=5000 + rank,
                                   device=dev)
        ws = torch.empty(da.diffattn_v2_decode_workspace_size(c["B"], c["L"], c["Hq"], c["Hkv"],
                                                              c["d"]), dtype=torch.uint8, device=dev)
        vdout = torch.empty((c["B"], c["Hq"] // 2, c["d"]), dtype=torch.bfloat16, device=dev)

        def v2dec():
            da.diffattn_v2_decode(vd.q, vd.k_cache, vd.v_cache, vd.lam_logit, workspace=ws,
                                  out=vdout)

        for _ in range(args.warmup):
            v2dec()
        barrier()
        n_steps = max(5, min(50, args.steps))
        evs = [(ev(), ev()) for _ in range(n_steps)]
        for i in range(n_steps):
            evs[i][0].record(stream)
            v2dec()
            evs[i][1].record(stream)
        barrier()
        da.diffattn_device_status()
        ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
        nbytes = v2_decode_bytes(c)
        gbs = nbytes / (ms * 1e-3) / 1e9
        line["v2_decode"] = {
            "metric": "V2 decode HBM GB/s", "value": world * gbs, "unit": "GB/s", "ms_per_call": ms,
            "workload": f"v2_decode_32k: B{c['B']}, one query per sequence, cache 32768, Hq64 "
                        "(32 pairs) over Hkv8, d128, bf16 (cache 8.6 GB at B64, larger than L2)",
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s",
                         "frac": gbs / hbm,
                         "traffic": profiled_traffic("v2_decode_32k.md",
                                                     source_sha(["decode_v2_tc.cu", "ptx.cuh"])),
                         "bytes_per_launch": nbytes,
                         "peak_source": f"hbm_gbs of {peak_src} (copy, read+write)",
                         "timed": "diffattn_v2_decode call (split kernel + combine kernel)"},
            "gpu_launches": 2 * n_steps}

        # fp8 e4m3 q and K cache (per-tensor scales), V bf16: 3/4 of the bytes for every key
        q8, qds = to_fp8_e4m3(vd.q)
        k8, kds = to_fp8_e4m3(vd.k_cache)

        def v2dec8():
            da.diffattn_v2_decode_fp8(q8, k8, vd.v_cache, vd.lam_logit, qds, kds, workspace=ws,
                                      out=vdout)

        for _ in range(args.warmup):
            v2dec8()
        barrier()
        evs = [(ev(), ev()) for _ in range(n_steps)]
        for i in range(n_steps):
            evs[i][0].record(stream)
            v2dec8()
            evs[i][1].record(stream)
        barrier()
        da.diffattn_device_status()
        ms8 = statistics.mean(a.elapsed_time(b) for a, b in evs)
        nbytes8 = nbytes * 3 / 4
        gbs8 = nbytes8 / (ms8 * 1e-3) / 1e9
        line["v2_decode_fp8"] = {
            "metric": "V2 decode HBM GB/s", "value": world * gbs8, "unit": "GB/s",
            "ms_per_call": ms8, "speedup_vs_bf16_cache": ms / ms8,
            "workload": f"v2_decode_32k with fp8 e4m3 q and K cache (per-tensor scales), bf16 V",
            "roofline": {"bound": "hbm", "achieved": gbs8, "peak": hbm, "unit": "GB/s",
                         "frac": gbs8 / hbm, "bytes_per_launch": nbytes8,
                         "peak_source": f"hbm_gbs of {peak_src} (copy, read+write)",
                         "timed": "diffattn_v2_decode_fp8 call (split kernel + combine kernel)"},
            "gpu_launches": 2 * n_steps}
        del q8, k8

        # the same cache as pools of pages placed in a random order: 64-token pages (one TMA box
        # per 64 keys) and 16-token pages (the smallest box the tensor-core kernel takes)
        paged = {}
        for ps in (64, 16):
            mp = c["L"] // ps
            k_pool = vd.k_cache.view(c["B"] * mp, ps, c["Hkv"], c["d"])
            v_pool = vd.v_cache.view(c["B"] * mp, ps, c["Hkv"], c["d"])
            gp = torch.Generator(device="cpu")
            gp.manual_seed(5100 + ps + rank)
            table = torch.randperm(c["B"] * mp, generator=gp).to(torch.int32).view(c["B"], mp).to(dev)

            def v2dec_paged():
                da.diffattn_v2_decode_paged(vd.q, k_pool, v_pool, table, vd.seqlens, vd.lam_logit,
                                            workspace=ws, out=vdout)

            for _ in range(args.warmup):
                v2dec_paged()
            barrier()
            evs = [(ev(), ev()) for _ in range(n_steps)]
            for i in range(n_steps):
                evs[i][0].record(stream)
                v2dec_paged()
                evs[i][1].record(stream)
            barrier()
            da.diffattn_device_status()
            pms = statistics.mean(a.elapsed_time(b) for a, b in evs)
            pgbs = nbytes / (pms * 1e-3) / 1e9
            paged[f"page_{ps}"] = {"value": world * pgbs, "ms_per_call": pms, "frac": pgbs / hbm}
            del k_pool, v_pool, table
        line["v2_decode_paged"] = {
            "metric": "V2 decode HBM GB/s", "unit": "GB/s",
            "value": paged["page_64"]["value"], "ms_per_call": paged["page_64"]["ms_per_call"],
            "workload": f"v2_decode_32k over a paged cache: B{c['B']}, cache 32768 in pages placed "
                        "in a random order in the pool, Hq64 over Hkv8, d128, bf16",
            "page_sizes": paged,
            "roofline": {"bound": "hbm", "achieved": paged["page_64"]["value"] / world, "peak": hbm,
                         "unit": "GB/s", "frac": paged["page_64"]["frac"],
                         "bytes_per_launch": nbytes,
                         "peak_source": f"hbm_gbs of {peak_src} (copy, read+write)",
                         "timed": "diffattn_v2_decode_paged call, 64-token pages (split kernel + "
                                  "combine kernel)"},
            "gpu_launches": 2 * n_steps * len(paged)}
        del vd, ws, vdout
        torch.cuda.empty_cache()

    # ======================= grouped: signal heads sharing noise heads =======================
    if args.only in ("all", "gda"):
        gc = GDA
        ginp = make_gda_inputs(gc["B"], gc["N"], gc["Hs"], gc["Hn"], gc["d"], gc["dv"],
                               seed=5000 + rank, device=dev)
        gout = torch.empty((gc["B"], gc["N"], gc["Hs"], gc["dv"]), dtype=torch.bfloat16, device=dev)
        li_g = da.diffattn_lambda_init(gc["layer"])

        def gda():
            da.diffattn_gda_fwd(ginp.q, ginp.k, ginp.v, ginp.lam, gc["Hs"], li_g, out=gout)

        for _ in range(args.warmup):
            gda()
        barrier()
        gsteps = max(5, min(50, args.steps))
        g_ev = [(ev(), ev()) for _ in range(gsteps)]
        for i in range(gsteps):
            g_ev[i][0].record(stream)
            gda()
            g_ev[i][1].record(stream)
        barrier()
        da.diffattn_device_status()
        gms = statistics.mean(a.elapsed_time(b) for a, b in g_ev)
        gflops = float(gc["B"] * gc["Hs"] * causal_pairs(gc["N"]) * FLOPS_PER_PAIR)
        gtf = gflops / (gms * 1e-3) / 1e12
        line["gda_prefill"] = {
            "metric": "DiffAttn fwd TFLOP/s", "value": world * gtf, "unit": "TFLOP/s",
            "ms_per_call": gms,
            "workload": "gda_prefill_3b: B4 N4096, 12 signal heads over 3 noise heads (4 per noise "
                        "head), d128 dv256 causal, RMSNorm + scale",
            "roofline": {"bound": "tensor", "achieved": gtf, "peak": peak_tf, "unit": "TFLOP/s",
                         "frac": gtf / peak_tf, "flops_per_launch": gflops,
                         "flops_per_pair": FLOPS_PER_PAIR,
                         "note": "MMA flops issued: each signal head's CTA recomputes its noise map"},
            "gpu_launches": gsteps}
        del ginp, gout
        torch.cuda.empty_cache()

        gd = dict(GDA_DECODE, B=args.decode_batch)
        gdi = make_gda_decode_inputs(gd["B"], gd["L"], gd["Hs"], gd["Hn"], gd["d"], gd["dv"],
                                     seed=5100 + rank, device=dev)
        gws = torch.empty(da.diffattn_decode_workspace_size(gd["B"], gd["L"], gd["Hs"]),
                          dtype=torch.uint8, device=dev)
        gdout = torch.empty((gd["B"], gd["Hs"], gd["dv"]), dtype=torch.bfloat16, device=dev)

        def gdec():
            da.diffattn_gda_decode(gdi.q, gdi.k_cache, gdi.v_cache, gdi.lam, gd["Hs"], li_g,
                                   workspace=gws, out=gdout)

        for _ in range(args.warmup):
            gdec()
        barrier()
        gdsteps = max(5, min(50, args.steps))
        gd_ev = [(ev(), ev()) for _ in range(gdsteps)]
        for i in range(gdsteps):
            gd_ev[i][0].record(stream)
            gdec()
            gd_ev[i][1].record(stream)
        barrier()
        da.diffattn_device_status()
        gdms = statistics.mean(a.elapsed_time(b) for a, b in gd_ev)
        gdbytes = gda_decode_bytes(gd)
        dsha_g = source_sha(["decode.cu", "ptx.cuh"])
        gdgbs = gdbytes / (gdms * 1e-3) / 1e9
        line["gda_decode"] = {
            "metric": "decode HBM GB/s", "value": world * gdgbs, "unit": "GB/s", "ms_per_call": gdms,
            "workload": f"gda_decode_32k: B{gd['B']}, one query per sequence, cache 32768, 12 "
                        "signal heads over 3 noise heads, d128, dv256, bf16 (cache 20.9 GB at B64)",
            "roofline": {"bound": "hbm", "achieved": gdgbs, "peak": hbm, "unit": "GB/s",
                         "frac": gdgbs / hbm, "bytes_per_launch": gdbytes,
                         "traffic": profiled_traffic("gda_decode_32k.md", dsha_g),
                         "peak_source": f"hbm_gbs of {peak_src} (copy, read+write)",
                         "timed": "diffattn_gda_decode call (group kernel + combine kernel); a "
                                  "noise row serves the 4 signal heads of its group from L1"},
            "gpu_launches": 2 * gdsteps}
        del gdi, gws, gdout
        torch.cuda.empty_cache()

    # ======================= CPU baseline (rank 0, N = 1 only) =======================
    line["cpu_baseline"] = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and args.only == "all":
        v, cores, desc, _, _ = oracle_sample(args.cpu_seconds)
        line["cpu_baseline"] = {"value": v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                                "sample": desc}
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
