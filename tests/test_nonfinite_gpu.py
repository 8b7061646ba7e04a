"""Non-finite inputs propagate and stay where they belong: a NaN reaches exactly the outputs whose
definition contains it and no other. The oracle reading is "propagate; values are not inspected".
What both sides fix uniquely is which rows become NaN; every other row must be bit-identical to
the clean run (each output row depends only on its own query and the keys it may see)."""
import pytest
import torch

import differential_attention_gb300 as da
from synth import make_decode_inputs, make_prefill_inputs

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    da.build()
    da.lib()
    yield
    da.diffattn_device_status()


def _run(q, k, v, lam, causal=True):
    out = da.diffattn_fwd(q, k, v, lam, 0.5, causal=causal)
    torch.cuda.synchronize()
    return out


def _nan_rows(out):
    """[B, N, H] mask: the row is NaN in every channel."""
    return torch.isnan(out.float()).all(dim=-1)


@pytest.mark.parametrize("causal", [True, False])
def test_nan_query_row_reaches_only_its_row(causal):
    B, N, H = 2, 300, 3
    inp = make_prefill_inputs(B, N, H, 128, 256, seed=301)
    q, k, v = inp.q.to(DEV), inp.k.to(DEV), inp.v.to(DEV)
    lam = torch.tensor([0.3, 0.6, 0.9], dtype=torch.float32, device=DEV)
    clean = _run(q, k, v, lam, causal)
    bad = q.clone()
    bad[1, 137, 2, 5] = float("nan")                 # map 1 of head 2, query row 137
    bad[0, 10, 0, 128 + 7] = float("nan")            # map 2 of head 0, query row 10
    out = _run(bad, k, v, lam, causal)
    want = torch.zeros((B, N, H), dtype=torch.bool, device=DEV)
    want[1, 137, 2] = True
    want[0, 10, 0] = True
    assert torch.equal(_nan_rows(out), want)
    assert torch.equal(out[~want], clean[~want])
    da.diffattn_device_status()


def test_nan_key_reaches_the_rows_that_see_it():
    """Causal: a NaN in key row j of one head turns rows j .. N-1 of that head to NaN; the rows
    before j (which may not see it, inside its tile or not) and every other head are bit-identical
    to the clean run."""
    B, N, H, j = 1, 400, 2, 201
    inp = make_prefill_inputs(B, N, H, 128, 256, seed=303)
    q, k, v = inp.q.to(DEV), inp.k.to(DEV), inp.v.to(DEV)
    lam = torch.tensor([0.4, 0.7], dtype=torch.float32, device=DEV)
    clean = _run(q, k, v, lam)
    bad = k.clone()
    bad[0, j, 1, 3] = float("nan")                   # K1 of head 1
    out = _run(q, bad, v, lam)
    want = torch.zeros((B, N, H), dtype=torch.bool, device=DEV)
    want[0, j:, 1] = True
    assert torch.equal(_nan_rows(out), want)
    assert torch.equal(out[~want], clean[~want])


def test_nan_in_decode_cache_reaches_only_its_sequence_and_head():
    inp = make_decode_inputs(3, 700, 3, 128, 256, seed=305)
    q, kc, vc, lam = (t.to(DEV) for t in (inp.q, inp.k_cache, inp.v_cache, inp.lam))
    clean = da.diffattn_decode(q, kc, vc, lam, 0.5)
    bad = kc.clone()
    bad[2, 350, 1, 200] = float("nan")               # K2 of head 1, sequence 2
    out = da.diffattn_decode(q, bad, vc, lam, 0.5)
    torch.cuda.synchronize()
    nan = torch.isnan(out.float()).all(dim=-1)
    want = torch.zeros((3, 3), dtype=torch.bool, device=DEV)
    want[2, 1] = True
    assert torch.equal(nan, want)
    assert torch.equal(out[~want], clean[~want])
    da.diffattn_device_status()


# ------------------------------------------------------------------------------------------
# Keys no query may see never reach an output, even when their values are not finite: cache rows
# past a sequence's length in its last page, and rows of a packed buffer that belong to no
# sequence, are outside the operator's definition (the oracle never reads them). Their scores
# are masked, and their V rows must not enter the product either (0 * NaN is NaN).
# ------------------------------------------------------------------------------------------
def _page_pool(Lk, ps, Hkv, width, seed):
    """One sequence of Lk keys in a shuffled pool of pages of ps rows (plus a spare page)."""
    g = torch.Generator().manual_seed(seed)
    mp = (max(Lk) + ps - 1) // ps
    n = len(Lk) * mp + 1
    k_pool = (torch.randn((n, ps, Hkv, width[0]), generator=g) / 128 ** 0.5).to(torch.bfloat16)
    v_pool = (torch.randn((n, ps, Hkv, width[1]), generator=g) / 128 ** 0.5).to(torch.bfloat16)
    table = torch.randperm(n, generator=g)[:len(Lk) * mp].reshape(len(Lk), mp).to(torch.int32)
    return k_pool, v_pool, table


def _poison_past_end(k_pool, v_pool, table, Lk, ps):
    """NaN in every pool row a sequence's table reaches but its keys do not (rows Lk .. of its
    last used page, and its unused table pages)."""
    kp, vp = k_pool.clone(), v_pool.clone()
    for b, L in enumerate(Lk):
        for pi in range(table.shape[1]):
            lo = max(0, L - pi * ps)
            if lo < ps:
                kp[table[b, pi], lo:] = float("nan")
                vp[table[b, pi], lo:] = float("nan")
    return kp, vp


@pytest.mark.parametrize("exact", [False, True])
def test_v2_paged_prefill_ignores_rows_past_the_keys(exact):
    ps, Hq, Hkv = 128, 8, 2
    Lq, Lk = [200, 5], [600, 130]
    k_pool, v_pool, table = _page_pool(Lk, ps, Hkv, (128, 128), seed=311)
    g = torch.Generator().manual_seed(312)
    q = (torch.randn((sum(Lq), Hq, 128), generator=g) / 128 ** 0.5).to(torch.bfloat16).to(DEV)
    lg = torch.randn((sum(Lq), Hq // 2), generator=g, dtype=torch.float32).to(DEV)
    cu_q = torch.tensor([0, Lq[0], sum(Lq)], dtype=torch.int32, device=DEV)
    sk = torch.tensor(Lk, dtype=torch.int32, device=DEV)
    run = lambda kp, vp: da.diffattn_v2_fwd_paged(q, kp.to(DEV), vp.to(DEV), lg, cu_q, sk,
                                                   table.to(DEV), exact=exact)
    clean = run(k_pool, v_pool)
    bad = run(*_poison_past_end(k_pool, v_pool, table, Lk, ps))
    torch.cuda.synchronize()
    assert not torch.isnan(bad.float()).any()
    assert torch.equal(bad, clean)
    da.diffattn_device_status()


def test_v1_paged_prefill_ignores_rows_past_the_keys():
    ps, H = 128, 2
    Lq, Lk = [300, 1], [700, 200]
    k_pool, v_pool, table = _page_pool(Lk, ps, H, (256, 256), seed=313)
    q = make_prefill_inputs(1, sum(Lq), H, 128, 256, seed=314).q[0].to(DEV)
    cu_q = torch.tensor([0, Lq[0], sum(Lq)], dtype=torch.int32, device=DEV)
    sk = torch.tensor(Lk, dtype=torch.int32, device=DEV)
    lam = torch.tensor([0.45, 0.8], dtype=torch.float32, device=DEV)
    run = lambda kp, vp: da.diffattn_fwd_paged(q, kp.to(DEV), vp.to(DEV), cu_q, sk, table.to(DEV),
                                               lam, 0.5)
    clean = run(k_pool, v_pool)
    bad = run(*_poison_past_end(k_pool, v_pool, table, Lk, ps))
    torch.cuda.synchronize()
    assert not torch.isnan(bad.float()).any()
    assert torch.equal(bad, clean)
    da.diffattn_device_status()


@pytest.mark.parametrize("exact", [False, True])
def test_packed_prefills_ignore_rows_in_no_sequence(exact):
    """Padding rows after the last packed sequence (NaN keys and values) change nothing, for the
    V2 prefill and (exact=True) the V1 prefill with keys of their own."""
    g = torch.Generator().manual_seed(315)
    lens_q, lens_k, pad = [100, 70], [300, 70], 50
    tq, tk = sum(lens_q), sum(lens_k) + pad
    cu_q = torch.tensor([0, lens_q[0], tq], dtype=torch.int32, device=DEV)
    cu_k = torch.tensor([0, lens_k[0], tk - pad], dtype=torch.int32, device=DEV)
    q2 = (torch.randn((tq, 8, 128), generator=g) / 128 ** 0.5).to(torch.bfloat16).to(DEV)
    k2 = (torch.randn((tk, 2, 128), generator=g) / 128 ** 0.5).to(torch.bfloat16).to(DEV)
    v2 = (torch.randn((tk, 2, 128), generator=g) / 128 ** 0.5).to(torch.bfloat16).to(DEV)
    lg = torch.randn((tq, 4), generator=g, dtype=torch.float32).to(DEV)
    k2b, v2b = k2.clone(), v2.clone()
    k2b[tk - pad:] = float("nan")
    v2b[tk - pad:] = float("nan")
    run2 = lambda k, v: da.diffattn_v2_fwd_varlen(q2, k, v, lg, cu_q, cu_k, exact=exact)
    clean, bad = run2(k2, v2), run2(k2b, v2b)
    torch.cuda.synchronize()
    assert not torch.isnan(bad.float()).any()
    assert torch.equal(bad, clean)
    if exact:
        q1 = (torch.randn((tq, 2, 256), generator=g) / 128 ** 0.5).to(torch.bfloat16).to(DEV)
        k1 = (torch.randn((tk, 2, 256), generator=g) / 128 ** 0.5).to(torch.bfloat16).to(DEV)
        v1 = (torch.randn((tk, 2, 256), generator=g) / 128 ** 0.5).to(torch.bfloat16).to(DEV)
        k1b, v1b = k1.clone(), v1.clone()
        k1b[tk - pad:] = float("nan")
        v1b[tk - pad:] = float("nan")
        lam = torch.tensor([0.3, 0.7], dtype=torch.float32, device=DEV)
        run1 = lambda k, v: da.diffattn_fwd_varlen_qk(q1, k, v, cu_q, cu_k, lam, 0.5)
        c1, b1 = run1(k1, v1), run1(k1b, v1b)
        torch.cuda.synchronize()
        assert not torch.isnan(b1.float()).any()
        assert torch.equal(b1, c1)
    da.diffattn_device_status()
