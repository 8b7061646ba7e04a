"""GPU parity at the full workload sizes, in the launch configurations bench.py times.

Inputs are drawn on the device (seeded CUDA generator) and the kernels run on the whole problem.
The float64 oracle then recomputes the outputs from the same inputs, copied to the host:

* the 3B-layer prefill (B4 N4096 H12) and the 32K-token decode (B64 H12) are checked in full:
  every row of every (sequence, head), every sequence of the decode batch, each (sequence, head)
  against the bf16 bar on its own;
* the 64K-token prefill and the V2 shapes are checked on sampled rows (the first rows, the last
  row and seeded random rows of every head), since the oracle would need minutes per head there.

The operator checked is the one page "Differential Transformer: softmax can't say zero, so it
subtracts" defines in "The mechanism, exactly", followed by the per-head norm and the
(1 - lambda_init) scale of "The row no longer sums to one". Tolerances are those of the small
cases (tests/gpu_util.py).
"""
import numpy as np
import pytest
import torch

import differential_attention_gb300 as da
from oracle import diffattn_ref as ref
from synth import (make_decode_inputs, make_dout, make_lambda_vectors, make_prefill_inputs,
                   make_v2_decode_inputs, make_v2_inputs)
from tests.gpu_util import assert_bf16, assert_grad

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    da.build()
    da.lib()
    yield
    torch.cuda.empty_cache()


def _rows(N, n_first, n_rand, seed):
    rng = np.random.default_rng(seed)
    rand = rng.choice(np.arange(n_first, N - 1), size=min(n_rand, max(0, N - 1 - n_first)), replace=False)
    return np.unique(np.concatenate([np.arange(min(n_first, N)), [N - 1], rand]))


def _prefill_case(B, N, H, layer, seed, needle, n_first, n_rand):
    inp = make_prefill_inputs(B, N, H, 128, 256, seed=seed, layer=layer, device=DEV, needle=needle)
    lv = make_lambda_vectors(128, seed=seed + 1)
    lv_h = tuple(t.to(DEV).expand(H, -1).contiguous() for t in lv)
    lam_h = da.diffattn_lambda(*lv_h, layer=layer)
    li = da.diffattn_lambda_init(layer)
    out = da.diffattn_fwd(inp.q, inp.k, inp.v, lam_h, li)
    da.diffattn_device_status()
    lam = float(ref.lambda_full(*lv, layer=layer)[0])
    rows = _rows(N, n_first, n_rand, seed)
    got, want = [], []
    for b in range(B):
        for h in range(H):
            q = inp.q[b:b + 1, :, h:h + 1].cpu()
            k = inp.k[b:b + 1, :, h:h + 1].cpu()
            v = inp.v[b:b + 1, :, h:h + 1].cpu()
            want.append(ref.diffattn_fwd(q, k, v, [lam], ref.lambda_init(layer), rows=rows)[0, :, 0])
            got.append(out[b, torch.as_tensor(rows, device=DEV), h].float().cpu().numpy())
    return np.stack(got), np.stack(want), lam


def _host64(t):
    """float64 numpy copy of a device tensor: the bf16 values exactly, converted on the host."""
    return t.cpu().to(torch.float64).numpy()


def test_prefill_3b_full():
    """B4 N4096 H12 d128 dv256 causal, lambda from the layer-12 vectors, RMSNorm + scale: every
    row of all 48 (sequence, head) pairs against the oracle, each pair within the bf16 bar."""
    B, N, H, layer = 4, 4096, 12, 12
    inp = make_prefill_inputs(B, N, H, 128, 256, seed=1000, layer=layer, device=DEV)
    lv = make_lambda_vectors(128, seed=1001)
    lv_h = tuple(t.to(DEV).expand(H, -1).contiguous() for t in lv)
    lam_h = da.diffattn_lambda(*lv_h, layer=layer)
    li = da.diffattn_lambda_init(layer)
    out = da.diffattn_fwd(inp.q, inp.k, inp.v, lam_h, li)
    da.diffattn_device_status()
    lam = float(ref.lambda_full(*lv, layer=layer)[0])
    q, k, v, got = (t.cpu() for t in (inp.q, inp.k, inp.v, out))
    del inp, out
    torch.cuda.empty_cache()
    worst_rel, worst_abs = 0.0, 0.0
    for b in range(B):
        for h in range(H):
            sl = lambda t: t[b:b + 1, :, h:h + 1].to(torch.float64).numpy()
            want = ref.diffattn_fwd(sl(q), sl(k), sl(v), [lam], ref.lambda_init(layer))
            max_abs, rel = assert_bf16(sl(got), want)
            worst_rel, worst_abs = max(worst_rel, rel), max(worst_abs, max_abs)
    print(f"prefill_3b, all {B * H * N} rows: worst rel L2 {worst_rel:.2e}, worst max abs {worst_abs:.2e}")


def test_prefill_64k_full_with_needle():
    """B1 N65536 H12 causal, layer 24, one needle key per head raised by ln(N-1) against the last
    query: the last row (needle row), the first rows and random rows of every head."""
    got, want, lam = _prefill_case(1, 65536, 12, 24, seed=2024, needle=True, n_first=32, n_rand=64)
    assert_bf16(got, want)


def test_fwd_host_3b_bit_equal():
    """The end-to-end entry point at the 3B-layer shape (pinned host buffers, each sequence in
    1024-row pieces computed as they land): bit-equal to the device-side fused-lambda prefill,
    which the full check above ties to the oracle."""
    B, N, H, layer = 4, 4096, 12, 12
    inp = make_prefill_inputs(B, N, H, 128, 256, seed=1100, layer=layer, device=DEV)
    lv = tuple(t.to(DEV).contiguous() for t in make_lambda_vectors(128, seed=1101))
    want = da.diffattn_fwd_fused_lambda(inp.q, inp.k, inp.v, *lv, layer=layer).cpu()
    hq, hk, hv = (t.cpu().pin_memory() for t in (inp.q, inp.k, inp.v))
    hout = torch.zeros((B, N, H, 256), dtype=torch.bfloat16).pin_memory()
    da.diffattn_fwd_host(hq, hk, hv, hout, *lv, layer=layer)
    torch.cuda.synchronize()
    da.diffattn_device_status()
    assert torch.equal(hout, want)
    del inp
    torch.cuda.empty_cache()


def test_decode_32k_full():
    """B64, cache 32768, H12: all 64 sequences (every head) against the oracle, one sequence's
    cache (0.4 GB of bf16) at a time, each (sequence, head) within the bf16 bar."""
    inp = make_decode_inputs(64, 32768, 12, 128, 256, seed=2000, device=DEV)
    li = da.diffattn_lambda_init(12)
    out = da.diffattn_decode(inp.q, inp.k_cache, inp.v_cache, inp.lam, li).cpu()
    da.diffattn_device_status()
    q, lam, seqlens = _host64(inp.q), _host64(inp.lam), inp.seqlens.cpu().numpy()
    worst_rel = 0.0
    for b in range(64):
        want = ref.diffattn_decode(q[b:b + 1], _host64(inp.k_cache[b:b + 1]),
                                   _host64(inp.v_cache[b:b + 1]), seqlens[b:b + 1], lam,
                                   ref.lambda_init(12))
        for h in range(12):
            _, rel = assert_bf16(out[b, h], want[0, h])
            worst_rel = max(worst_rel, rel)
    print(f"decode_32k, all 64 sequences x 12 heads: worst rel L2 {worst_rel:.2e}")
    del inp
    torch.cuda.empty_cache()


def test_v2_gqa_full():
    """B2 N8192, 32 pairs over 8 KV heads, causal: sampled rows of every pair."""
    inp = make_v2_inputs(2, 8192, 64, 8, 128, seed=3000, device=DEV)
    out = da.diffattn_v2_fwd(inp.q, inp.k, inp.v, inp.lam_logit)
    da.diffattn_device_status()
    rows = _rows(8192, 32, 64, 3000)
    got, want = [], []
    for b in range(2):
        for p in range(32):
            g = ref.v2_kv_head(p, 64, 8)
            q = inp.q[b:b + 1, :, 2 * p:2 * p + 2].cpu()
            k = inp.k[b:b + 1, :, g:g + 1].cpu()
            v = inp.v[b:b + 1, :, g:g + 1].cpu()
            lam = inp.lam_logit[b:b + 1, :, p:p + 1].cpu()
            want.append(ref.diffattn_v2_fwd(q, k, v, lam, rows=rows)[0, :, 0])
            got.append(out[b, torch.as_tensor(rows, device=DEV), p].float().cpu().numpy())
    assert_bf16(np.stack(got), np.stack(want))


def test_v2_decode_32k_full():
    """B64, cache 32768, 64 query heads over 8 KV heads: all pairs of 3 sampled sequences."""
    inp = make_v2_decode_inputs(64, 32768, 64, 8, 128, seed=4000, device=DEV)
    out = da.diffattn_v2_decode(inp.q, inp.k_cache, inp.v_cache, inp.lam_logit)
    da.diffattn_device_status()
    sample = [0, 29, 63]
    want = ref.diffattn_v2_decode(inp.q[sample].cpu(), inp.k_cache[sample].cpu(),
                                  inp.v_cache[sample].cpu(), inp.seqlens[sample].cpu(),
                                  inp.lam_logit[sample].cpu())
    assert_bf16(out[sample], want)
    del inp
    torch.cuda.empty_cache()


def test_bwd_3b_full():
    """Backward at B4 N4096 H12 (the bench's training launch): every gradient of head 5 in all
    four sequences (so dlambda[5] is complete) and of head 0 in sequence 1."""
    B, N, H = 4, 4096, 12
    inp = make_prefill_inputs(B, N, H, 128, 256, seed=6000, layer=12, device=DEV)
    dy = make_dout(B, N, H, 256, seed=6007, device=DEV)
    lam = torch.linspace(0.5, 0.9, H, dtype=torch.float32, device=DEV)
    li = da.diffattn_lambda_init(12)
    _, o_pre, stats = da.diffattn_fwd_train(inp.q, inp.k, inp.v, lam, li)
    g = da.diffattn_bwd(inp.q, inp.k, inp.v, o_pre, stats, dy, lam, li)
    da.diffattn_device_status()
    lam_h = lam.cpu().numpy()
    dl5 = 0.0
    for b, h in [(0, 5), (1, 5), (2, 5), (3, 5), (1, 0)]:
        sl = lambda t: t[b:b + 1, :, h:h + 1].cpu()
        want = ref.diffattn_bwd(sl(inp.q), sl(inp.k), sl(inp.v), lam_h[h:h + 1], ref.lambda_init(12),
                                sl(dy))
        for name in ("dq", "dk", "dv"):
            assert_grad(g[name][b:b + 1, :, h:h + 1], want[name], name=f"{name} b{b} h{h}")
        if h == 5:
            dl5 += want["dlam"][0]
    assert_grad(g["dlam"][5:6], np.array([dl5]), rel_tol=1e-2, name="dlam[5]")
    del inp, dy, o_pre, stats, g
    torch.cuda.empty_cache()
