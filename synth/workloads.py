"""Seeded synthetic workloads for differential attention.

Every generator here only draws random numbers (torch generators, so one call gives the same values
each time on a given device) and rounds them to the storage dtype. The shapes follow the 3B-layer
shape table of "Differential Transformer: softmax can't say zero, so it subtracts" (section "Half
the heads, same parameters": hidden 3072, 12 differential heads, d = 128, value width 256) and the
V2 layout of "Differential Transformer V2" (query heads doubled, KV heads unchanged, GQA groups
contiguous).

Tensor layouts (all row-major, last dimension contiguous):
  prefill   q [B, N, H, 2d] = [Q1 | Q2],  k [B, N, H, 2d] = [K1 | K2],  v [B, N, H, dv]
  decode    q [B, H, 2d],  k_cache [B, L, H, 2d],  v_cache [B, L, H, dv],  seqlens [B] int32
  V2        q [B, N, Hq, d] (pair p = heads 2p, 2p+1),  k, v [B, N, Hkv, d],  lam_logit [B, N, Hq/2]
  grouped   q, k [B, N, Hs + Hn, d] (Hs signal heads' Q1/K1, then Hn noise heads' Q2/K2),
            v [B, N, Hs, dv], lam [Hs]; decode q [B, Hs + Hn, d], caches [B, L, Hs + Hn, d] and
            [B, L, Hs, dv]
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

# The five workloads, by what they are. Sizes are the full sizes; tests scale them down.
WORKLOADS = {
    "tiny_fp32": dict(B=1, N=128, H=1, d=64, dv=128, causal=False, dtype="fp32", lam=0.8, norm=False),
    "prefill_3b": dict(B=4, N=4096, H=12, d=128, dv=256, causal=True, dtype="bf16", layer=12, norm=True),
    "prefill_64k": dict(B=1, N=65536, H=12, d=128, dv=256, causal=True, dtype="bf16", layer=24, norm=True,
                        needle=True),
    "decode_32k": dict(B=64, L=32768, H=12, d=128, dv=256, dtype="bf16", layer=12, norm=True),
    "v2_gqa": dict(B=2, N=8192, Hq=64, Hkv=8, d=128, causal=True, dtype="bf16"),
    "v2_decode_32k": dict(B=64, L=32768, Hq=64, Hkv=8, d=128, dtype="bf16"),
    # grouped: the 12 heads of prefill_3b / decode_32k as signal heads over 3 noise heads (4 per
    # noise head, the ratio "What other people found" reports for Grouped Differential Attention)
    "gda_prefill_3b": dict(B=4, N=4096, Hs=12, Hn=3, d=128, dv=256, causal=True, dtype="bf16",
                           layer=12, norm=True),
    "gda_decode_32k": dict(B=64, L=32768, Hs=12, Hn=3, d=128, dv=256, dtype="bf16", layer=12,
                           norm=True),
}

NORM_EPS = 1e-5


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(int(seed))
    return g


def bf16_round(x: torch.Tensor) -> torch.Tensor:
    """Round to bfloat16 (nearest-even) and keep the bf16 tensor."""
    return x.to(torch.bfloat16)


def _randn(shape, g: torch.Generator, device, std: float = 1.0) -> torch.Tensor:
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x


def make_lambda_vectors(dim: int, seed: int, n_sets: int = 1, std: float = 0.1, device="cpu"):
    """The four lambda vectors lq1, lk1, lq2, lk2, each [n_sets, dim], drawn i.i.d. N(0, std^2).

    std = 0.1 is the initialisation given in section "lambda, re-parameterised" of "Differential
    Transformer: softmax can't say zero, so it subtracts" (vectors drawn from N(0, 0.1^2)).
    """
    g = _gen(seed, device)
    return tuple(_randn((n_sets, dim), g, device, std) for _ in range(4))


@dataclass
class PrefillInputs:
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    lam_vectors: tuple | None = None  # (lq1, lk1, lq2, lk2), each [1, d] fp32
    lam_fixed: float | None = None    # a fixed lambda (tiny workload)
    layer: int | None = None
    causal: bool = True
    norm: bool = True
    eps: float = NORM_EPS
    needle: dict = field(default_factory=dict)


def make_tiny_inputs(seed: int = 0, device="cpu") -> PrefillInputs:
    """Tiny fp32 case: Q1, Q2, K1, K2 [128, 64] and V [128, 128], i.i.d. N(0, 1), seed 0.

    Returned in the prefill layout with B = H = 1, drawn in the order Q1, Q2, K1, K2, V.
    """
    cfg = WORKLOADS["tiny_fp32"]
    n, d, dv = cfg["N"], cfg["d"], cfg["dv"]
    g = _gen(seed, device)
    q1, q2, k1, k2 = (_randn((n, d), g, device) for _ in range(4))
    v = _randn((n, dv), g, device)
    q = torch.cat([q1, q2], dim=-1).reshape(1, n, 1, 2 * d).contiguous()
    k = torch.cat([k1, k2], dim=-1).reshape(1, n, 1, 2 * d).contiguous()
    v = v.reshape(1, n, 1, dv).contiguous()
    return PrefillInputs(q=q, k=k, v=v, lam_fixed=cfg["lam"], causal=False, norm=False)


def make_prefill_inputs(B: int, N: int, H: int, d: int, dv: int, seed: int, layer: int = 12,
                        causal: bool = True, device="cpu", needle: bool = False,
                        dtype=torch.bfloat16) -> PrefillInputs:
    """Prefill inputs: q, k, v ~ N(0, 1)/sqrt(d), rounded to `dtype`; lambda vectors ~ N(0, 0.1^2).

    With `needle`, each head of each batch gets one key j* < N-1 (seeded) whose map-1 logit against
    the last query is raised by D = ln(N - 1): K1[j*] += (D * sqrt(d) / |q1_last|^2) * q1_last,
    computed in fp32 on the already-rounded q before k is rounded. D = ln(n - 1) is the gap at
    which a lone needle keeps half of a softmax row ("Why softmax can't say zero").
    """
    g = _gen(seed, device)
    std = 1.0 / math.sqrt(d)
    q = _randn((B, N, H, 2 * d), g, device, std).to(dtype)
    k32 = _randn((B, N, H, 2 * d), g, device, std)
    v = _randn((B, N, H, dv), g, device, std).to(dtype)
    info = {}
    if needle:
        D = math.log(N - 1)
        gi = _gen(seed + 7919, "cpu")
        js = torch.randint(0, N - 1, (B, H), generator=gi)
        q1_last = q[:, N - 1, :, :d].float()                    # [B, H, d]
        coef = D * math.sqrt(d) / (q1_last * q1_last).sum(-1)   # [B, H]
        for b in range(B):
            for h in range(H):
                j = int(js[b, h])
                k32[b, j, h, :d] += coef[b, h] * q1_last[b, h]
        info = dict(D=D, positions=js)
    k = k32.to(dtype)
    del k32
    lv = make_lambda_vectors(d, seed + 1, device="cpu")
    return PrefillInputs(q=q, k=k, v=v, lam_vectors=lv, layer=layer, causal=causal, norm=True,
                         needle=info)


@dataclass
class DecodeInputs:
    q: torch.Tensor
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    seqlens: torch.Tensor
    lam: torch.Tensor        # [H] fp32
    layer: int = 12
    eps: float = NORM_EPS


def make_decode_inputs(B: int, L: int, H: int, d: int, dv: int, seed: int, layer: int = 12,
                       device="cpu", ragged: bool = False, dtype=torch.bfloat16) -> DecodeInputs:
    """Decode inputs: cache ~ N(0, 1), q ~ N(0, 1)/sqrt(d), lambda[h] ~ U[0.2, 0.8].

    The cache is drawn one batch row at a time so peak host/device memory stays at one row of
    fp32. With `ragged`, seqlens[b] is drawn uniformly in [1, L]; otherwise every row holds L keys.
    """
    g = _gen(seed, device)
    q = _randn((B, H, 2 * d), g, device, 1.0 / math.sqrt(d)).to(dtype)
    k_cache = torch.empty((B, L, H, 2 * d), dtype=dtype, device=device)
    v_cache = torch.empty((B, L, H, dv), dtype=dtype, device=device)
    for b in range(B):
        k_cache[b].copy_(_randn((L, H, 2 * d), g, device))
        v_cache[b].copy_(_randn((L, H, dv), g, device))
    gh = _gen(seed + 1, "cpu")
    lam = (0.2 + 0.6 * torch.rand((H,), generator=gh, dtype=torch.float32)).to(device)
    if ragged:
        seqlens = torch.randint(1, L + 1, (B,), generator=gh, dtype=torch.int32)
    else:
        seqlens = torch.full((B,), L, dtype=torch.int32)
    return DecodeInputs(q=q, k_cache=k_cache, v_cache=v_cache, seqlens=seqlens.to(device), lam=lam,
                        layer=layer)


@dataclass
class V2Inputs:
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    lam_logit: torch.Tensor  # [B, N, Hq/2] fp32, sigmoid is applied by the operator
    causal: bool = True


def make_v2_inputs(B: int, N: int, Hq: int, Hkv: int, d: int, seed: int, causal: bool = True,
                   device="cpu", dtype=torch.bfloat16) -> V2Inputs:
    """V2 inputs: q [B,N,Hq,d], k, v [B,N,Hkv,d] ~ N(0, 1)/sqrt(d); lambda logits ~ N(0, 1)."""
    g = _gen(seed, device)
    std = 1.0 / math.sqrt(d)
    q = _randn((B, N, Hq, d), g, device, std).to(dtype)
    k = _randn((B, N, Hkv, d), g, device, std).to(dtype)
    v = _randn((B, N, Hkv, d), g, device, std).to(dtype)
    lam_logit = _randn((B, N, Hq // 2), g, device)
    return V2Inputs(q=q, k=k, v=v, lam_logit=lam_logit, causal=causal)


@dataclass
class V2DecodeInputs:
    q: torch.Tensor          # [B, Hq, d]
    k_cache: torch.Tensor    # [B, L, Hkv, d]
    v_cache: torch.Tensor    # [B, L, Hkv, d]
    seqlens: torch.Tensor    # [B] int32
    lam_logit: torch.Tensor  # [B, Hq/2] fp32, sigmoid is applied by the operator


def make_v2_decode_inputs(B: int, L: int, Hq: int, Hkv: int, d: int, seed: int, device="cpu",
                          ragged: bool = False, dtype=torch.bfloat16) -> V2DecodeInputs:
    """V2 decode inputs: cache ~ N(0, 1), q ~ N(0, 1)/sqrt(d), lambda logits ~ N(0, 1); the cache
    is drawn one batch row at a time. With `ragged`, seqlens[b] ~ U{1..L}, else L everywhere."""
    g = _gen(seed, device)
    q = _randn((B, Hq, d), g, device, 1.0 / math.sqrt(d)).to(dtype)
    k_cache = torch.empty((B, L, Hkv, d), dtype=dtype, device=device)
    v_cache = torch.empty((B, L, Hkv, d), dtype=dtype, device=device)
    for b in range(B):
        k_cache[b].copy_(_randn((L, Hkv, d), g, device))
        v_cache[b].copy_(_randn((L, Hkv, d), g, device))
    gh = _gen(seed + 1, "cpu")
    lam_logit = torch.randn((B, Hq // 2), generator=gh, dtype=torch.float32)
    if ragged:
        seqlens = torch.randint(1, L + 1, (B,), generator=gh, dtype=torch.int32)
    else:
        seqlens = torch.full((B,), L, dtype=torch.int32)
    return V2DecodeInputs(q=q, k_cache=k_cache, v_cache=v_cache, seqlens=seqlens.to(device),
                          lam_logit=lam_logit.to(device))


def make_dout(B: int, N: int, H: int, dv: int, seed: int, device="cpu", dtype=torch.bfloat16):
    """Upstream gradient dL/dout for the backward: N(0, 1) per element."""
    return _randn((B, N, H, dv), _gen(seed, device), device).to(dtype)


def page_cache(k_cache: torch.Tensor, v_cache: torch.Tensor, page_size: int, seed: int,
               spare_pages: int = 0):
    """Cut a contiguous cache [B, L, H, *] (L a multiple of page_size) into pages, place them in a
    pool in a seeded random order (with `spare_pages` unused pages of noise), and return
    (k_pool, v_pool, block_table int32 [B, L / page_size])."""
    B, L, H, wk = k_cache.shape
    wv = v_cache.shape[-1]
    mp = L // page_size
    n = B * mp + spare_pages
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    slot = torch.randperm(n, generator=g)[:B * mp]  # pool slot of logical page (b, p)
    k_pool = torch.randn((n, page_size, H, wk), generator=g).to(k_cache.dtype).to(k_cache.device)
    v_pool = torch.randn((n, page_size, H, wv), generator=g).to(v_cache.dtype).to(v_cache.device)
    slot_d = slot.to(k_cache.device)
    k_pool[slot_d] = k_cache.reshape(B * mp, page_size, H, wk)
    v_pool[slot_d] = v_cache.reshape(B * mp, page_size, H, wv)
    return k_pool, v_pool, slot.reshape(B, mp).to(torch.int32).to(k_cache.device)


def to_fp8_e4m3(x: torch.Tensor):
    """Per-tensor absmax cast to fp8 e4m3: returns (x8, descale) with x ~= x8 * descale (the
    largest magnitude maps to 448, the format's largest finite value)."""
    amax = float(x.float().abs().max())
    descale = amax / 448.0 if amax > 0 else 1.0
    return (x.float() / descale).to(torch.float8_e4m3fn), descale


@dataclass
class GroupedInputs:
    q: torch.Tensor          # [B, N, Hs + Hn, d]
    k: torch.Tensor          # [B, N, Hs + Hn, d]
    v: torch.Tensor          # [B, N, Hs, dv]
    lam: torch.Tensor        # [Hs] fp32
    n_signal: int
    layer: int = 12


def make_gda_inputs(B: int, N: int, Hs: int, Hn: int, d: int, dv: int, seed: int, layer: int = 12,
                    device="cpu", dtype=torch.bfloat16) -> GroupedInputs:
    """Grouped prefill inputs: q, k, v ~ N(0, 1)/sqrt(d) as for the ungrouped prefill, with the
    signal and noise heads along one head axis; lambda[h] ~ U[0.2, 0.8]."""
    g = _gen(seed, device)
    std = 1.0 / math.sqrt(d)
    q = _randn((B, N, Hs + Hn, d), g, device, std).to(dtype)
    k = _randn((B, N, Hs + Hn, d), g, device, std).to(dtype)
    v = _randn((B, N, Hs, dv), g, device, std).to(dtype)
    gh = _gen(seed + 1, "cpu")
    lam = (0.2 + 0.6 * torch.rand((Hs,), generator=gh, dtype=torch.float32)).to(device)
    return GroupedInputs(q=q, k=k, v=v, lam=lam, n_signal=Hs, layer=layer)


@dataclass
class GroupedDecodeInputs:
    q: torch.Tensor          # [B, Hs + Hn, d]
    k_cache: torch.Tensor    # [B, L, Hs + Hn, d]
    v_cache: torch.Tensor    # [B, L, Hs, dv]
    seqlens: torch.Tensor    # [B] int32
    lam: torch.Tensor        # [Hs] fp32
    n_signal: int
    layer: int = 12


def make_gda_decode_inputs(B: int, L: int, Hs: int, Hn: int, d: int, dv: int, seed: int,
                           layer: int = 12, device="cpu", ragged: bool = False,
                           dtype=torch.bfloat16) -> GroupedDecodeInputs:
    """Grouped decode inputs, drawn as make_decode_inputs draws the ungrouped ones: cache
    ~ N(0, 1) one batch row at a time, q ~ N(0, 1)/sqrt(d), lambda[h] ~ U[0.2, 0.8]."""
    g = _gen(seed, device)
    q = _randn((B, Hs + Hn, d), g, device, 1.0 / math.sqrt(d)).to(dtype)
    k_cache = torch.empty((B, L, Hs + Hn, d), dtype=dtype, device=device)
    v_cache = torch.empty((B, L, Hs, dv), dtype=dtype, device=device)
    for b in range(B):
        k_cache[b].copy_(_randn((L, Hs + Hn, d), g, device))
        v_cache[b].copy_(_randn((L, Hs, dv), g, device))
    gh = _gen(seed + 1, "cpu")
    lam = (0.2 + 0.6 * torch.rand((Hs,), generator=gh, dtype=torch.float32)).to(device)
    if ragged:
        seqlens = torch.randint(1, L + 1, (B,), generator=gh, dtype=torch.int32)
    else:
        seqlens = torch.full((B,), L, dtype=torch.int32)
    return GroupedDecodeInputs(q=q, k_cache=k_cache, v_cache=v_cache, seqlens=seqlens.to(device),
                               lam=lam, n_signal=Hs, layer=layer)
