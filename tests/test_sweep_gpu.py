"""Seeded randomized sweep: every entry point on a spread of small shapes (lengths from 1 up to
several tiles with ragged tails, several batch rows and heads, causal or not, with and without
the norm and the fixed rescale) against the float64 oracle. Each case draws its own shape from a
fixed seed, so a failure names a reproducible case."""
import numpy as np
import pytest
import torch

import differential_attention_gb300 as da
from oracle import diffattn_ref as ref
from synth import (make_decode_inputs, make_dout, make_prefill_inputs, make_v2_decode_inputs,
                   make_v2_inputs, page_cache, to_fp8_e4m3)
from tests.gpu_util import assert_bf16, assert_grad

pytestmark = pytest.mark.gpu

DEV = "cuda"
N_CASES = 10


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    da.build()
    da.lib()
    yield
    da.diffattn_device_status()


def _shape(seed, nmax=700):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 4))
    N = int(rng.choice([1, 2, 63, 127, 128, 129, 255, int(rng.integers(3, nmax))]))
    H = int(rng.integers(1, 4))
    causal = bool(rng.integers(0, 2))
    norm = bool(rng.integers(0, 2))
    scale = bool(rng.integers(0, 2))
    lam = rng.uniform(0.0, 1.1, H)
    return rng, B, N, H, causal, norm, scale, lam


@pytest.mark.parametrize("case", range(N_CASES))
def test_sweep_prefill(case):
    rng, B, N, H, causal, norm, scale, lam = _shape(1000 + case)
    inp = make_prefill_inputs(B, N, H, 128, 256, seed=1000 + case, causal=causal)
    li = ref.lambda_init(int(rng.integers(1, 30)))
    w = torch.tensor(rng.uniform(0.5, 1.5, 256), dtype=torch.float32)
    got = da.diffattn_fwd(inp.q.to(DEV), inp.k.to(DEV), inp.v.to(DEV),
                          torch.tensor(lam, dtype=torch.float32, device=DEV), li,
                          norm_weight=w.to(DEV), causal=causal, norm=norm, scale=scale)
    want = ref.diffattn_fwd(inp.q, inp.k, inp.v, lam, li, norm_weight=w, causal=causal, norm=norm,
                            apply_scale=scale)
    assert_bf16(got, want)


@pytest.mark.parametrize("case", range(N_CASES))
def test_sweep_fp8_and_varlen(case):
    rng, B, N, H, causal, norm, scale, lam = _shape(1100 + case)
    inp = make_prefill_inputs(B, N, H, 128, 256, seed=1100 + case, causal=causal)
    li = ref.lambda_init(12)
    lam_t = torch.tensor(lam, dtype=torch.float32, device=DEV)
    q8, qs = to_fp8_e4m3(inp.q)
    k8, ks = to_fp8_e4m3(inp.k)
    got = da.diffattn_fwd_fp8(q8.to(DEV), k8.to(DEV), inp.v.to(DEV), lam_t, qs, ks, li,
                              causal=causal, norm=norm, scale=scale)
    want = ref.diffattn_fwd(q8.float() * qs, k8.float() * ks, inp.v, lam, li, causal=causal,
                            norm=norm, apply_scale=scale)
    assert_bf16(got, want)
    # the same tokens as one packed batch of B sequences of different lengths
    lens = [int(x) for x in rng.integers(0, N + 1, B)]
    lens[0] = max(1, lens[0])
    total = B * N
    qp, kp, vp = (t.reshape(total, H, -1) for t in (inp.q, inp.k, inp.v))
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    got = da.diffattn_fwd_varlen(qp.to(DEV), kp.to(DEV), vp.to(DEV), cu.to(DEV), lam_t, li,
                                 causal=causal, norm=norm, scale=scale)
    want = ref.diffattn_fwd_varlen(qp, kp, vp, cu, lam, li, causal=causal, norm=norm,
                                   apply_scale=scale)
    assert_bf16(got[:sum(lens)], want[:sum(lens)])


@pytest.mark.parametrize("case", range(N_CASES))
def test_sweep_decodes(case):
    rng, B, L, H, _, norm, scale, lam = _shape(1200 + case, nmax=2000)
    inp = make_decode_inputs(B, L, H, 128, 256, seed=1200 + case, ragged=True)
    li = ref.lambda_init(12)
    got = da.diffattn_decode(inp.q.to(DEV), inp.k_cache.to(DEV), inp.v_cache.to(DEV),
                             inp.lam.to(DEV), li, seqlens=inp.seqlens.to(DEV), norm=norm, scale=scale)
    want = ref.diffattn_decode(inp.q, inp.k_cache, inp.v_cache, inp.seqlens, inp.lam, li,
                               norm=norm, apply_scale=scale)
    assert_bf16(got, want)
    ps = int(rng.choice([1, 7, 16, 64]))
    Lp = (L + ps - 1) // ps * ps
    kc = torch.zeros((B, Lp, H, 256), dtype=torch.bfloat16)
    vc = torch.zeros((B, Lp, H, 256), dtype=torch.bfloat16)
    kc[:, :L], vc[:, :L] = inp.k_cache, inp.v_cache
    k_pool, v_pool, table = page_cache(kc, vc, ps, seed=1250 + case, spare_pages=2)
    gotp = da.diffattn_decode_paged(inp.q.to(DEV), k_pool.to(DEV), v_pool.to(DEV), table.to(DEV),
                                    inp.seqlens.to(DEV), inp.lam.to(DEV), li, norm=norm, scale=scale)
    assert_bf16(gotp, want)
    G = int(rng.choice([2, 4, 8]))
    Hkv = int(rng.integers(1, 3))
    v2 = make_v2_decode_inputs(B, L, G * Hkv, Hkv, 128, seed=1260 + case, ragged=True)
    for cc in (False, True):
        got2 = da.diffattn_v2_decode(v2.q.to(DEV), v2.k_cache.to(DEV), v2.v_cache.to(DEV),
                                     v2.lam_logit.to(DEV), seqlens=v2.seqlens.to(DEV), cuda_cores=cc)
        assert_bf16(got2, ref.diffattn_v2_decode(v2.q, v2.k_cache, v2.v_cache, v2.seqlens,
                                                 v2.lam_logit))


@pytest.mark.parametrize("case", range(N_CASES))
def test_sweep_v2_prefill(case):
    rng, B, N, _, causal, _, _, _ = _shape(1300 + case)
    Hkv = int(rng.integers(1, 3))
    Hq = Hkv * int(rng.choice([2, 4]))
    d = int(rng.choice([64, 128]))
    inp = make_v2_inputs(B, N, Hq, Hkv, d, seed=1300 + case, causal=causal)
    got = da.diffattn_v2_fwd(inp.q.to(DEV), inp.k.to(DEV), inp.v.to(DEV), inp.lam_logit.to(DEV),
                             causal=causal)
    assert_bf16(got, ref.diffattn_v2_fwd(inp.q, inp.k, inp.v, inp.lam_logit, causal=causal))


@pytest.mark.parametrize("case", range(6))
def test_sweep_backward(case):
    rng, B, N, H, causal, norm, scale, lam = _shape(1400 + case, nmax=450)
    N = max(N, 2)  # one visible key makes dlambda a pure cancellation (see test_backward_gpu)
    inp = make_prefill_inputs(B, N, H, 128, 256, seed=1400 + case, causal=causal)
    dy = make_dout(B, N, H, 256, seed=1407 + case)
    li = ref.lambda_init(12)
    w = torch.tensor(rng.uniform(0.5, 1.5, 256), dtype=torch.float32)
    lam_t = torch.tensor(lam, dtype=torch.float32, device=DEV)
    q, k, v = inp.q.to(DEV), inp.k.to(DEV), inp.v.to(DEV)
    wd = w.to(DEV) if norm else None
    _, o_pre, stats = da.diffattn_fwd_train(q, k, v, lam_t, li, norm_weight=wd, causal=causal,
                                            norm=norm, scale=scale)
    g = da.diffattn_bwd(q, k, v, o_pre, stats, dy.to(DEV), lam_t, li, norm_weight=wd,
                        causal=causal, norm=norm, scale=scale)
    want = ref.diffattn_bwd(inp.q, inp.k, inp.v, lam, li, dy, norm_weight=w if norm else None,
                            norm=norm, apply_scale=scale, causal=causal)
    for name in ("dq", "dk", "dv"):
        assert_grad(g[name], want[name], name=name)


@pytest.mark.parametrize("case", range(8))
def test_sweep_packed_chunks(case):
    """Packed sequences whose queries are the last Lq of Lk positions (V1 and V2), random
    lengths including Lq = 0, Lq = 1 and Lq = Lk."""
    rng = np.random.default_rng(1500 + case)
    B = int(rng.integers(1, 5))
    lens_k = [int(rng.integers(1, 600)) for _ in range(B)]
    lens_q = [int(rng.choice([0, 1, lk, int(rng.integers(0, lk + 1))])) for lk in lens_k]
    lens_q[0] = max(1, lens_q[0])
    causal = bool(rng.integers(0, 2))
    tq, tk = sum(lens_q), sum(lens_k)
    cu_q = torch.tensor(np.concatenate([[0], np.cumsum(lens_q)]), dtype=torch.int32)
    cu_k = torch.tensor(np.concatenate([[0], np.cumsum(lens_k)]), dtype=torch.int32)
    H = int(rng.integers(1, 3))
    kv = make_prefill_inputs(1, tk, H, 128, 256, seed=1500 + case, causal=causal)
    q = make_prefill_inputs(1, tq, H, 128, 256, seed=1550 + case).q[0]
    lam = rng.uniform(0.0, 1.1, H)
    li = ref.lambda_init(12)
    got = da.diffattn_fwd_varlen_qk(q.to(DEV), kv.k[0].to(DEV), kv.v[0].to(DEV), cu_q.to(DEV),
                                    cu_k.to(DEV), torch.tensor(lam, dtype=torch.float32, device=DEV),
                                    li, causal=causal)
    assert_bf16(got, ref.diffattn_fwd_varlen_qk(q, kv.k[0], kv.v[0], cu_q, cu_k, lam, li,
                                                causal=causal))
    Hkv = int(rng.integers(1, 3))
    Hq = Hkv * int(rng.choice([2, 4]))
    v2 = make_v2_inputs(1, tk, Hq, Hkv, 128, seed=1570 + case, causal=causal)
    v2q = make_v2_inputs(1, tq, Hq, Hkv, 128, seed=1590 + case)
    got2 = da.diffattn_v2_fwd_varlen(v2q.q[0].to(DEV), v2.k[0].to(DEV), v2.v[0].to(DEV),
                                     v2q.lam_logit[0].to(DEV), cu_q.to(DEV), cu_k.to(DEV),
                                     causal=causal)
    assert_bf16(got2, ref.diffattn_v2_fwd_varlen(v2q.q[0], v2.k[0], v2.v[0], v2q.lam_logit[0],
                                                 cu_q, cu_k, causal=causal))


@pytest.mark.parametrize("case", range(6))
def test_sweep_paged_prefill(case):
    """Packed queries against keys in a shuffled page pool (V1 and V2), random lengths and page
    sizes of 128 or 256 tokens."""
    rng = np.random.default_rng(1600 + case)
    B = int(rng.integers(1, 4))
    ps = int(rng.choice([128, 256]))
    lens_k = [int(rng.integers(1, 700)) for _ in range(B)]
    lens_q = [max(1, int(rng.integers(0, lk + 1))) for lk in lens_k]
    causal = bool(rng.integers(0, 2))
    mp = (max(lens_k) + ps - 1) // ps + int(rng.integers(0, 2))
    cu_q = torch.tensor(np.concatenate([[0], np.cumsum(lens_q)]), dtype=torch.int32)
    sk = torch.tensor(lens_k, dtype=torch.int32)
    H = int(rng.integers(1, 3))
    kin = make_prefill_inputs(B, mp * ps, H, 128, 256, seed=1600 + case)
    k_pool, v_pool, table = page_cache(kin.k, kin.v, ps, seed=1610 + case, spare_pages=2)
    q = make_prefill_inputs(1, sum(lens_q), H, 128, 256, seed=1620 + case).q[0]
    lam = rng.uniform(0.0, 1.1, H)
    li = ref.lambda_init(12)
    got = da.diffattn_fwd_paged(q.to(DEV), k_pool.to(DEV), v_pool.to(DEV), cu_q.to(DEV),
                                sk.to(DEV), table.to(DEV),
                                torch.tensor(lam, dtype=torch.float32, device=DEV), li,
                                causal=causal)
    assert_bf16(got, ref.diffattn_fwd_paged(q, k_pool, v_pool, cu_q, sk, table, lam, li,
                                            causal=causal))
    Hkv = int(rng.integers(1, 3))
    Hq = Hkv * int(rng.choice([2, 4]))
    g = torch.Generator().manual_seed(1630 + case)
    kc = (torch.randn((B, mp * ps, Hkv, 128), generator=g) / 128 ** 0.5).to(torch.bfloat16)
    vc = (torch.randn((B, mp * ps, Hkv, 128), generator=g) / 128 ** 0.5).to(torch.bfloat16)
    k2, v2, t2 = page_cache(kc, vc, ps, seed=1640 + case, spare_pages=1)
    q2 = (torch.randn((sum(lens_q), Hq, 128), generator=g) / 128 ** 0.5).to(torch.bfloat16)
    lg = torch.randn((sum(lens_q), Hq // 2), generator=g, dtype=torch.float32)
    got2 = da.diffattn_v2_fwd_paged(q2.to(DEV), k2.to(DEV), v2.to(DEV), lg.to(DEV), cu_q.to(DEV),
                                    sk.to(DEV), t2.to(DEV), causal=causal)
    assert_bf16(got2, ref.diffattn_v2_fwd_paged(q2, k2, v2, lg, cu_q, sk, t2, causal=causal))
