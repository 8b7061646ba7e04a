"""GPU parity at full size for the bench lines beyond the five base workloads: fp8 scores, the
packed, chunked and paged prefills, the grouped packed and fp8 prefills, the paged and fp8
decodes, the packed backward and the grouped backward (batched and packed). Each runs in the
launch configuration bench.py times. Inputs are drawn on the device; the float64 oracle
recomputes sampled outputs. Where two entry points run the same arithmetic on the same data
(paged against contiguous caches) the outputs must also be bit-identical."""
import numpy as np
import pytest
import torch

import differential_attention_gb300 as da
from bench import varlen_lengths
from oracle import diffattn_ref as ref
from synth import (make_decode_inputs, make_dout, make_gda_inputs, make_prefill_inputs,
                   make_v2_decode_inputs, to_fp8_e4m3)
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
    rand = rng.choice(np.arange(n_first, N - 1), size=min(n_rand, max(0, N - 1 - n_first)),
                      replace=False)
    return np.unique(np.concatenate([np.arange(min(n_first, N)), [N - 1], rand]))


def _shuffled_pages(k_cache, v_cache, ps, seed):
    """The bench's paged layout: the contiguous cache viewed as pages, the pages moved to a
    seeded random order in the pool, and the block table that finds them there."""
    B, L = k_cache.shape[:2]
    mp = L // ps
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    table = torch.randperm(B * mp, generator=g).to(torch.int32).view(B, mp).to(k_cache.device)
    order = torch.argsort(table.flatten())
    k_pool = k_cache.reshape(B * mp, ps, *k_cache.shape[2:])[order].contiguous()
    v_pool = v_cache.reshape(B * mp, ps, *v_cache.shape[2:])[order].contiguous()
    return k_pool, v_pool, table


def test_prefill_fp8_full():
    """prefill_3b with fp8 e4m3 q, k (per-tensor absmax scales): sampled rows of every head of
    two sequences against the oracle on the dequantized values."""
    B, N, H = 4, 4096, 12
    inp = make_prefill_inputs(B, N, H, 128, 256, seed=9000, layer=12, device=DEV)
    q8, qs = to_fp8_e4m3(inp.q)
    k8, ks = to_fp8_e4m3(inp.k)
    lam = torch.full((H,), 0.6, dtype=torch.float32, device=DEV)
    li = da.diffattn_lambda_init(12)
    out = da.diffattn_fwd_fp8(q8, k8, inp.v, lam, qs, ks, li)
    da.diffattn_device_status()
    rows = _rows(N, 32, 64, 9000)
    got, want = [], []
    for b in (0, 3):
        for h in range(H):
            q = q8[b:b + 1, :, h:h + 1].cpu().double() * qs
            k = k8[b:b + 1, :, h:h + 1].cpu().double() * ks
            v = inp.v[b:b + 1, :, h:h + 1].cpu()
            want.append(ref.diffattn_fwd(q, k, v, [0.6], ref.lambda_init(12), rows=rows)[0, :, 0])
            got.append(out[b, torch.as_tensor(rows, device=DEV), h].float().cpu().numpy())
    assert_bf16(np.stack(got), np.stack(want))


def test_varlen_full():
    """The bench's 16 packed sequences (1..4096 tokens, 16384 in all): sampled rows of every head
    of five sequences (the longest, the one-token one and three between) against each sequence's
    own prefill in the oracle."""
    H = 12
    lens = varlen_lengths()
    total = int(sum(lens))
    inp = make_prefill_inputs(1, total, H, 128, 256, seed=8000, layer=12, device=DEV)
    cu = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32, device=DEV)
    lam = torch.full((H,), 0.6, dtype=torch.float32, device=DEV)
    li = da.diffattn_lambda_init(12)
    out = da.diffattn_fwd_varlen(inp.q[0], inp.k[0], inp.v[0], cu, lam, li, max_seqlen=max(lens))
    da.diffattn_device_status()
    offs = np.concatenate([[0], np.cumsum(lens)])
    got, want = [], []
    for s in (0, 1, 5, 9, 15):
        s0, n = int(offs[s]), int(lens[s])
        rows = _rows(n, 16, 32, 8000 + s)
        sl = lambda t: t[:, s0:s0 + n].cpu()
        w = ref.diffattn_fwd(sl(inp.q), sl(inp.k), sl(inp.v), [0.6] * H, ref.lambda_init(12),
                             rows=rows)[0]
        want.append(w.reshape(-1, 256))
        got.append(out[torch.as_tensor(s0 + rows, device=DEV)].float().cpu().numpy().reshape(-1, 256))
    assert_bf16(np.concatenate(got), np.concatenate(want))


def test_gda_varlen_full():
    """The bench's grouped packed line: the 16 packed sequences with 12 signal heads over 3 noise
    heads, both launches (noise statistics once per noise head, into a workspace). Sampled rows of
    every signal head of five sequences against each sequence's own grouped prefill in the
    oracle."""
    Hs, Hn = 12, 3
    lens = varlen_lengths()
    total = int(sum(lens))
    inp = make_gda_inputs(1, total, Hs, Hn, 128, 256, seed=5100, device=DEV)
    cu = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32, device=DEV)
    li = da.diffattn_lambda_init(12)
    ws = torch.empty(da.diffattn_gda_fwd_workspace_size(len(lens), max(lens), Hs, Hn),
                     dtype=torch.uint8, device=DEV)
    out = da.diffattn_gda_fwd_varlen(inp.q[0], inp.k[0], inp.v[0], cu, inp.lam, Hs, li,
                                     max_seqlen=max(lens), workspace=ws)
    da.diffattn_device_status()
    offs = np.concatenate([[0], np.cumsum(lens)])
    lam = inp.lam.cpu().numpy()
    got, want = [], []
    for s in (0, 1, 5, 9, 15):
        s0, n = int(offs[s]), int(lens[s])
        rows = _rows(n, 16, 32, 5100 + s)
        sl = lambda t: t[:, s0:s0 + n].cpu()
        w = ref.diffattn_gda_fwd(sl(inp.q), sl(inp.k), sl(inp.v), lam, li, Hs, rows=rows)[0]
        want.append(w.reshape(-1, 256))
        got.append(out[torch.as_tensor(s0 + rows, device=DEV)].float().cpu().numpy().reshape(-1, 256))
    assert_bf16(np.concatenate(got), np.concatenate(want))


def test_gda_fp8_full():
    """The bench's grouped fp8 line (B4 N4096, 12 signal heads over 3 noise heads, fp8 e4m3 q and
    k with per-tensor scales): sampled rows of every signal head of two sequences against the
    oracle's grouped prefill on the dequantized values."""
    B, N, Hs, Hn = 4, 4096, 12, 3
    inp = make_gda_inputs(B, N, Hs, Hn, 128, 256, seed=5000, device=DEV)
    q8, qs = to_fp8_e4m3(inp.q)
    k8, ks = to_fp8_e4m3(inp.k)
    li = da.diffattn_lambda_init(12)
    out = da.diffattn_gda_fwd_fp8(q8, k8, inp.v, inp.lam, Hs, qs, ks, li)
    da.diffattn_device_status()
    rows = _rows(N, 32, 64, 5001)
    lam = inp.lam.cpu().numpy()
    got, want = [], []
    for b in (1, 2):
        for h in range(Hs):
            sel = [h, Hs + h // (Hs // Hn)]
            q = q8[b:b + 1, :, sel].cpu().double() * qs
            k = k8[b:b + 1, :, sel].cpu().double() * ks
            v = inp.v[b:b + 1, :, h:h + 1].cpu()
            want.append(ref.diffattn_gda_fwd(q, k, v, lam[h:h + 1], li, 1, rows=rows)[0, :, 0])
            got.append(out[b, torch.as_tensor(rows, device=DEV), h].float().cpu().numpy())
    assert_bf16(np.stack(got), np.stack(want))
    del inp, q8, k8, out
    torch.cuda.empty_cache()


def test_gda_chunk_and_paged_full():
    """The bench's grouped chunk lines: the last 1024 rows of four 4096-token prompts (12 signal
    over 3 noise heads) against all their keys, keys packed and in shuffled 256-token pages:
    bit-identical to each other and to those rows of the whole prompts' grouped prefill; sampled
    rows against the oracle."""
    B, Lq, Lk, Hs, Hn = 4, 1024, 4096, 12, 3
    cin = make_gda_inputs(B, Lk, Hs, Hn, 128, 256, seed=5050, device=DEV)
    li = da.diffattn_lambda_init(12)
    heads = Hs + Hn
    k, v = cin.k.reshape(-1, heads, 128), cin.v.reshape(-1, Hs, 256)
    q = cin.q[:, Lk - Lq:].reshape(-1, heads, 128).contiguous()
    cu_q = torch.arange(B + 1, dtype=torch.int32, device=DEV) * Lq
    cu_k = torch.arange(B + 1, dtype=torch.int32, device=DEV) * Lk
    out = da.diffattn_gda_fwd_varlen_qk(q, k, v, cu_q, cu_k, cin.lam, Hs, li, max_seqlen_q=Lq,
                                        max_seqlen_k=Lk)
    k_pool, v_pool, table = _shuffled_pages(cin.k, cin.v, 256, 5060)
    sk = torch.full((B,), Lk, dtype=torch.int32, device=DEV)
    pout = da.diffattn_gda_fwd_paged(q, k_pool, v_pool, cu_q, sk, table, cin.lam, Hs, li,
                                     max_seqlen_q=Lq, max_seqlen_k=Lk)
    whole = da.diffattn_gda_fwd(cin.q, cin.k, cin.v, cin.lam, Hs, li)
    da.diffattn_device_status()
    assert torch.equal(out, pout)
    assert torch.equal(out, whole[:, Lk - Lq:].reshape(-1, Hs, 256))
    rows = _rows(Lq, 16, 32, 5050)
    lam = cin.lam.cpu().numpy()
    got, want = [], []
    for b in (0, 3):
        sl = lambda t: t[b:b + 1].cpu()
        w = ref.diffattn_gda_fwd(sl(cin.q), sl(cin.k), sl(cin.v), lam, ref.lambda_init(12), Hs,
                                 rows=Lk - Lq + rows)[0]
        want.append(w.reshape(-1, 256))
        got.append(out[torch.as_tensor(b * Lq + rows, device=DEV)].float().cpu().numpy().reshape(-1, 256))
    assert_bf16(np.concatenate(got), np.concatenate(want))
    del cin, k_pool, v_pool, whole
    torch.cuda.empty_cache()


def test_varlen_qk_and_paged_full():
    """The last 1024 rows of four 4096-token prompts against all their keys (queries at the end of
    their keys), contiguous and in shuffled 256-token pages: the two are bit-identical, and
    sampled rows match the oracle's whole-prompt prefill at those positions."""
    B, Lq, Lk, H = 4, 1024, 4096, 12
    kin = make_prefill_inputs(B, Lk, H, 128, 256, seed=8100, layer=12, device=DEV)
    k, v = kin.k.reshape(-1, H, 256), kin.v.reshape(-1, H, 256)
    q = kin.q[:, Lk - Lq:].reshape(-1, H, 256).contiguous()
    cu_q = torch.arange(B + 1, dtype=torch.int32, device=DEV) * Lq
    cu_k = torch.arange(B + 1, dtype=torch.int32, device=DEV) * Lk
    lam = torch.full((H,), 0.6, dtype=torch.float32, device=DEV)
    li = da.diffattn_lambda_init(12)
    out = da.diffattn_fwd_varlen_qk(q, k, v, cu_q, cu_k, lam, li, max_seqlen_q=Lq, max_seqlen_k=Lk)
    k_pool, v_pool, table = _shuffled_pages(kin.k, kin.v, 256, 8200)
    sk = torch.full((B,), Lk, dtype=torch.int32, device=DEV)
    pout = da.diffattn_fwd_paged(q, k_pool, v_pool, cu_q, sk, table, lam, li, max_seqlen_q=Lq,
                                 max_seqlen_k=Lk)
    da.diffattn_device_status()
    assert torch.equal(out, pout)
    rows = _rows(Lq, 16, 48, 8100)
    got, want = [], []
    for b in (0, 2):
        for h in (0, 7, 11):
            sl = lambda t: t[b:b + 1, :, h:h + 1].cpu()
            want.append(ref.diffattn_fwd(sl(kin.q), sl(kin.k), sl(kin.v), [0.6],
                                         ref.lambda_init(12), rows=Lk - Lq + rows)[0, :, 0])
            got.append(out[torch.as_tensor(b * Lq + rows, device=DEV), h].float().cpu().numpy())
    assert_bf16(np.stack(got), np.stack(want))
    del kin, k_pool, v_pool
    torch.cuda.empty_cache()


def test_decode_paged_full():
    """decode_32k (B64, cache 32768, H12) in shuffled 64-token pages: bit-identical to the
    contiguous decode of the same cache; every head of 3 sampled sequences against the oracle."""
    inp = make_decode_inputs(64, 32768, 12, 128, 256, seed=2000, device=DEV)
    li = da.diffattn_lambda_init(12)
    flat = da.diffattn_decode(inp.q, inp.k_cache, inp.v_cache, inp.lam, li)
    k_pool, v_pool, table = _shuffled_pages(inp.k_cache, inp.v_cache, 64, 2100)
    k_cache_cpu = {s: inp.k_cache[s].cpu() for s in (3, 40, 63)}
    v_cache_cpu = {s: inp.v_cache[s].cpu() for s in (3, 40, 63)}
    del inp.k_cache, inp.v_cache
    torch.cuda.empty_cache()
    paged = da.diffattn_decode_paged(inp.q, k_pool, v_pool, table, inp.seqlens, inp.lam, li)
    da.diffattn_device_status()
    assert torch.equal(flat, paged)
    sample = [3, 40, 63]
    want = ref.diffattn_decode(inp.q[sample].cpu(), torch.stack([k_cache_cpu[s] for s in sample]),
                               torch.stack([v_cache_cpu[s] for s in sample]),
                               inp.seqlens[sample].cpu(), inp.lam.cpu(), ref.lambda_init(12))
    assert_bf16(paged[sample], want)
    del k_pool, v_pool
    torch.cuda.empty_cache()


def test_v2_decode_fp8_and_paged_full():
    """v2_decode_32k (B64, cache 32768, 64 query heads over 8 KV heads): with fp8 q and K cache
    against the oracle on the dequantized values; in shuffled pages of 64 and of 16 tokens
    bit-identical to the contiguous bf16 decode, which is checked against the oracle."""
    inp = make_v2_decode_inputs(64, 32768, 64, 8, 128, seed=4000, device=DEV)
    sample = [0, 29, 63]
    flat = da.diffattn_v2_decode(inp.q, inp.k_cache, inp.v_cache, inp.lam_logit)
    want = ref.diffattn_v2_decode(inp.q[sample].cpu(), inp.k_cache[sample].cpu(),
                                  inp.v_cache[sample].cpu(), inp.seqlens[sample].cpu(),
                                  inp.lam_logit[sample].cpu())
    assert_bf16(flat[sample], want)
    q8, qs = to_fp8_e4m3(inp.q)
    k8, ks = to_fp8_e4m3(inp.k_cache)
    out8 = da.diffattn_v2_decode_fp8(q8, k8, inp.v_cache, inp.lam_logit, qs, ks)
    da.diffattn_device_status()
    want8 = ref.diffattn_v2_decode(q8[sample].cpu().double() * qs,
                                   k8[sample].cpu().double() * ks, inp.v_cache[sample].cpu(),
                                   inp.seqlens[sample].cpu(), inp.lam_logit[sample].cpu())
    assert_bf16(out8[sample], want8)
    del q8, k8
    torch.cuda.empty_cache()
    for ps in (64, 16):
        k_pool, v_pool, table = _shuffled_pages(inp.k_cache, inp.v_cache, ps, 4100 + ps)
        paged = da.diffattn_v2_decode_paged(inp.q, k_pool, v_pool, table, inp.seqlens,
                                            inp.lam_logit)
        da.diffattn_device_status()
        assert torch.equal(paged, flat), f"page size {ps}"
        del k_pool, v_pool, table
        torch.cuda.empty_cache()
    del inp
    torch.cuda.empty_cache()


def test_bwd_varlen_full():
    """The bench's packed backward (16 sequences, 1..4096 tokens): every gradient of head 3 in the
    longest sequence and of all heads in the shortest multi-token and a mid-length sequence
    against the oracle's per-sequence backward."""
    H = 12
    lens = varlen_lengths()
    total = int(sum(lens))
    inp = make_prefill_inputs(1, total, H, 128, 256, seed=7100, layer=12, device=DEV)
    q, k, v = inp.q[0], inp.k[0], inp.v[0]
    dy = make_dout(1, total, H, 256, seed=7107, device=DEV)[0]
    cu = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32, device=DEV)
    lam = torch.linspace(0.5, 0.9, H, dtype=torch.float32, device=DEV)
    li = da.diffattn_lambda_init(12)
    mx = max(lens)
    _, o_pre, stats = da.diffattn_fwd_train_varlen(q, k, v, cu, lam, li, max_seqlen=mx)
    g = da.diffattn_bwd_varlen(q, k, v, o_pre, stats, dy, cu, lam, li, max_seqlen=mx)
    da.diffattn_device_status()
    offs = np.concatenate([[0], np.cumsum(lens)])
    lam_h = lam.cpu().numpy()
    mid = int(np.argsort(lens)[len(lens) // 2])
    short = min((n, s) for s, n in enumerate(lens) if n >= 2)[1]
    cases = [(0, [3]), (mid, list(range(H))), (short, list(range(H)))]
    for s, heads in cases:
        s0, n = int(offs[s]), int(lens[s])
        for h in heads:
            sl = lambda t: t[None, s0:s0 + n, h:h + 1].cpu()
            want = ref.diffattn_bwd(sl(q), sl(k), sl(v), lam_h[h:h + 1], ref.lambda_init(12),
                                    sl(dy))
            for name in ("dq", "dk", "dv"):
                assert_grad(g[name][None, s0:s0 + n, h:h + 1], want[name],
                            name=f"{name} seq{s} h{h}")
    del inp, dy, o_pre, stats, g
    torch.cuda.empty_cache()


def _group_heads(grp, Hs, G):
    """Signal heads of noise group grp, and those heads followed by its noise head."""
    sig = list(range(grp * G, grp * G + G))
    return sig, sig + [Hs + grp]


def test_gda_bwd_3b_full():
    """The bench's grouped training line (B4 N4096, 12 signal heads over 3 noise heads, noise
    statistics through the workspace): every gradient of one group (signal heads 4-7 and noise
    head 13) in sequence 2 against the oracle's grouped backward."""
    B, N, Hs, Hn = 4, 4096, 12, 3
    G = Hs // Hn
    inp = make_gda_inputs(B, N, Hs, Hn, 128, 256, seed=5000, device=DEV)
    dy = make_dout(B, N, Hs, 256, seed=5300, device=DEV)
    li = da.diffattn_lambda_init(12)
    w = torch.ones(256, dtype=torch.float32, device=DEV)
    ws = torch.empty(da.diffattn_gda_fwd_workspace_size(B, N, Hs, Hn), dtype=torch.uint8,
                     device=DEV)
    _, o_pre, stats = da.diffattn_gda_fwd_train(inp.q, inp.k, inp.v, inp.lam, Hs, li,
                                                norm_weight=w, workspace=ws)
    g = da.diffattn_gda_bwd(inp.q, inp.k, inp.v, o_pre, stats, dy, inp.lam, Hs, li, norm_weight=w)
    da.diffattn_device_status()
    b = 2
    sig, heads = _group_heads(1, Hs, G)
    sl = lambda t, hs: t[b:b + 1][:, :, hs].cpu()
    want = ref.diffattn_gda_bwd(sl(inp.q, heads), sl(inp.k, heads), sl(inp.v, sig),
                                inp.lam.cpu().numpy()[sig], li, G, sl(dy, sig),
                                norm_weight=np.ones(256))
    for name, hs in (("dq", heads), ("dk", heads), ("dv", sig)):
        for j, h in enumerate(hs):
            assert_grad(g[name][b:b + 1, :, h:h + 1], want[name][:, :, j:j + 1],
                        name=f"{name} b{b} h{h}")
    del inp, dy, ws, o_pre, stats, g
    torch.cuda.empty_cache()


def test_gda_bwd_varlen_full():
    """The bench's grouped packed backward (the 16 packed sequences, 12 signal heads over 3 noise
    heads): every gradient of one group in a 2497-token sequence and of every group in the
    shortest multi-token sequence against the oracle's grouped backward of that sequence."""
    Hs, Hn = 12, 3
    G = Hs // Hn
    lens = varlen_lengths()
    total = int(sum(lens))
    inp = make_gda_inputs(1, total, Hs, Hn, 128, 256, seed=5400, device=DEV)
    q, k, v = inp.q[0], inp.k[0], inp.v[0]
    dy = make_dout(1, total, Hs, 256, seed=5407, device=DEV)[0]
    cu = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32, device=DEV)
    li = da.diffattn_lambda_init(12)
    mx = max(lens)
    _, o_pre, stats = da.diffattn_gda_fwd_train_varlen(q, k, v, cu, inp.lam, Hs, li, max_seqlen=mx)
    g = da.diffattn_gda_bwd_varlen(q, k, v, o_pre, stats, dy, cu, inp.lam, Hs, li, max_seqlen=mx)
    da.diffattn_device_status()
    offs = np.concatenate([[0], np.cumsum(lens)])
    lam = inp.lam.cpu().numpy()
    long_s = lens.index(2497)
    short = min((n, s) for s, n in enumerate(lens) if n >= 2)[1]
    for s, groups in ((long_s, [2]), (short, range(Hn))):
        s0, n = int(offs[s]), int(lens[s])
        for grp in groups:
            sig, heads = _group_heads(grp, Hs, G)
            sl = lambda t, hs: t[None, s0:s0 + n][:, :, hs].cpu()
            want = ref.diffattn_gda_bwd(sl(q, heads), sl(k, heads), sl(v, sig), lam[sig], li, G,
                                        sl(dy, sig))
            for name, hs in (("dq", heads), ("dk", heads), ("dv", sig)):
                for j, h in enumerate(hs):
                    assert_grad(g[name][None, s0:s0 + n, h:h + 1], want[name][:, :, j:j + 1],
                                name=f"{name} seq{s} h{h}")
    del inp, dy, o_pre, stats, g
    torch.cuda.empty_cache()
