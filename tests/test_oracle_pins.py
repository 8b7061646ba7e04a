"""Pins for the float64 oracle (CPU only).

Each pin ties an oracle function to something other than the oracle itself: a number printed on
the pages (fixtures under tests/golden/, each citing its page and section), a closed form, a
library routine that the method reduces to in a special case, or pure-Python brute force on tiny
inputs. `test_planted_mistakes_are_caught` plants plausible mistakes in the oracle (on the CPU)
and checks that at least one pin fails for each.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import diffattn_ref as ref

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _sdpa(q, k, v, causal):
    """torch's scaled_dot_product_attention in float64 on the CPU (library routine)."""
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float64))
    return F.scaled_dot_product_attention(t(q)[None], t(k)[None], t(v)[None], is_causal=causal)[0].numpy()


def _cummean(v):
    return np.cumsum(v, axis=0) / np.arange(1, v.shape[0] + 1)[:, None]


# ------------------------------------------------------------------------------------------
# pins (plain functions so the planted-mistake test can run them against a mutated oracle)
# ------------------------------------------------------------------------------------------

def pin_lambda_init_table():
    g = _golden("lambda_init_table.json")
    for l, li, om in zip(g["layers"], g["lambda_init"], g["one_minus_init"]):
        assert round(ref.lambda_init(l), 2) == pytest.approx(li, abs=1e-9), l
        assert round(1.0 - ref.lambda_init(l), 2) == pytest.approx(om, abs=1e-9), l


def pin_lambda_init_shape():
    assert ref.lambda_init(1) == pytest.approx(0.2, abs=1e-15)
    vals = [ref.lambda_init(l) for l in range(1, 60)]
    assert all(b > a for a, b in zip(vals, vals[1:]))
    assert vals[-1] == pytest.approx(0.8, abs=1e-6) and vals[-1] < 0.8


def pin_lambda_closed_forms():
    dim = 16
    z = np.zeros((1, dim))
    for l in (1, 5, 12):
        assert ref.lambda_full(z, z, z, z, l)[0] == pytest.approx(ref.lambda_init(l), abs=1e-15)
    # dot1 = ln 3 and dot2 = ln 2 -> lambda = 3 - 2 + lambda_init; swapping the sets -> 2 - 3.
    a = np.zeros((1, dim)); a[0, 3] = math.log(3.0)
    b = np.zeros((1, dim)); b[0, 3] = 1.0
    c = np.zeros((1, dim)); c[0, 7] = 0.5
    e = np.zeros((1, dim)); e[0, 7] = 2 * math.log(2.0)
    li = ref.lambda_init(12)
    assert ref.lambda_full(a, b, c, e, 12)[0] == pytest.approx(1.0 + li, abs=1e-12)
    assert ref.lambda_full(c, e, a, b, 12)[0] == pytest.approx(-1.0 + li, abs=1e-12)


def pin_lambda_spread():
    g = _golden("lambda_spread.json")
    rng = np.random.default_rng(12345)
    # 100,000 initialisations (standard error of the spread ~3.6e-4), drawn in chunks of 10,000
    # to keep the working set small
    lam = np.concatenate([
        ref.lambda_full(*[rng.standard_normal((10_000, g["dim"])) * g["vector_std"]
                          for _ in range(4)], layer=12)
        for _ in range(10)])
    assert np.std(lam) == pytest.approx(g["lambda_std"], abs=2e-3)
    assert np.mean(lam) == pytest.approx(ref.lambda_init(12), abs=3e-3)


def pin_softmax_floor():
    g = _golden("softmax_floor.json")
    d = 4
    for n, Dp in zip(g["n"], g["D_half"]):
        D = math.log(n - 1)
        assert round(D, 2) == pytest.approx(Dp, abs=1e-9)
        # One head, lambda = 0: query 0 sees key 0 at logit D and n-1 keys at logit 0.
        q = np.zeros((1, d)); q[0, 0] = D * math.sqrt(d)
        k = np.zeros((n, d)); k[0, 0] = 1.0
        v = np.zeros((n, 2)); v[0, 0] = 1.0; v[1:, 1] = 1.0
        o = ref.diff_attn_head(q, k, q, k, v, 0.0, causal=False)
        assert o[0, 0] == pytest.approx(g["share_at_D_half"], abs=1e-12)
        assert o[0, 1] == pytest.approx(1.0 - g["share_at_D_half"], abs=1e-12)


def pin_toy_needle_table():
    g = _golden("toy_needle_table.json")
    lam, gap, sigma, seeds = g["lam"], g["gap"], g["sigma"], g["seeds"]

    def draws(n, rho, seed_ids):
        z1 = np.empty((len(seed_ids), n)); z2 = np.empty((len(seed_ids), n))
        for i, s in enumerate(seed_ids):
            c, e = np.random.default_rng(s).standard_normal((2, n))
            z1[i] = sigma * c
            z1[i, 0] += gap
            z2[i] = sigma * (rho * c + math.sqrt(1 - rho * rho) * e)
        return z1, z2

    def per_seed(n, rho):
        """Needle share |w_0| / sum |w| and needle weight w_0 of each seed's row, without and with
        the subtraction. Rows are independent, so they are drawn and weighted 50 seeds at a time:
        the same values as one pass over all seeds, in a working set that stays in cache."""
        out = {k: [] for k in ("share_single", "share_diff", "w_single", "w_diff")}
        for s0 in range(0, seeds, 50):
            z1, z2 = draws(n, rho, range(s0, min(seeds, s0 + 50)))
            for tag, lam_ in (("single", 0.0), ("diff", lam)):
                w = ref.diff_weights(z1, z2, lam_)
                out["share_" + tag].append(np.abs(w[:, 0]) / np.abs(w).sum(axis=1))
                out["w_" + tag].append(w[:, 0])
        return {k: float(np.mean(np.concatenate(v))) for k, v in out.items()}

    for row in g["rho_sweep_n32"]:
        m = per_seed(32, row["rho"])
        assert round(m["share_single"], 3) == pytest.approx(row["single"], abs=1e-9)
        assert round(m["share_diff"], 3) == pytest.approx(row["diff"], abs=1e-9)
        assert round(m["w_single"], 3) == pytest.approx(row["w_single"], abs=1e-9)
        assert round(m["w_diff"], 3) == pytest.approx(row["w_diff"], abs=1e-9)
    for row in g["n_sweep_rho09"]:
        m = per_seed(row["n"], 0.9)
        assert round(m["share_single"], 3) == pytest.approx(row["single"], abs=1e-9)
        assert round(m["share_diff"], 3) == pytest.approx(row["diff"], abs=1e-9)


def pin_worked_example():
    g = _golden("worked_example_rowsum.json")
    n, d, lam = g["n"], g["d"], g["lam"]
    torch.manual_seed(g["seed"])
    q1, k1, q2, k2 = torch.randn(4, n, d)
    _v = torch.randn(n, 2 * d)  # drawn to keep the generator sequence of the example
    S1 = ref.scores(ref._f64(q1), ref._f64(k1), np.arange(n), causal=False)
    S2 = ref.scores(ref._f64(q2), ref._f64(k2), np.arange(n), causal=False)
    W = ref.diff_weights(S1, S2, lam)
    assert f"{W.sum(axis=-1)[0]:.2f}" == g["printed_row_sum"]
    assert int((W < 0).sum()) == g["printed_negative"] and W.size == g["printed_total"]


def pin_row_sums():
    rng = np.random.default_rng(3)
    n, d = 37, 8
    for lam in (0.0, 0.2, 0.8, 1.3):
        for causal in (False, True):
            S1 = ref.scores(rng.standard_normal((n, d)), rng.standard_normal((n, d)), np.arange(n), causal)
            S2 = ref.scores(rng.standard_normal((n, d)), rng.standard_normal((n, d)), np.arange(n), causal)
            W = ref.diff_weights(S1, S2, lam)
            assert np.allclose(W.sum(-1), 1.0 - lam, atol=1e-12)
            if causal:
                assert np.all(W[np.triu_indices(n, 1)] == 0.0)


def pin_lambda_zero_is_softmax_attention():
    rng = np.random.default_rng(4)
    for causal in (False, True):
        n, d, dv = 29, 16, 32
        q1, k1, q2, k2 = (rng.standard_normal((n, d)) for _ in range(4))
        v = rng.standard_normal((n, dv))
        o = ref.diff_attn_head(q1, k1, q2, k2, v, 0.0, causal)
        assert np.allclose(o, _sdpa(q1, k1, v, causal), atol=1e-12, rtol=0)


def pin_equal_maps_scale_attention():
    rng = np.random.default_rng(5)
    for causal in (False, True):
        n, d, dv = 31, 8, 16
        q, k = rng.standard_normal((n, d)), rng.standard_normal((n, d))
        v = rng.standard_normal((n, dv))
        lam = 0.71
        o = ref.diff_attn_head(q, k, q, k, v, lam, causal)
        assert np.allclose(o, (1 - lam) * _sdpa(q, k, v, causal), atol=1e-12, rtol=0)


def pin_brute_force_tiny():
    rng = np.random.default_rng(6)
    n, d, dv, lam = 5, 3, 4, 0.6
    q1, k1, q2, k2 = (rng.standard_normal((n, d)).tolist() for _ in range(4))
    v = rng.standard_normal((n, dv)).tolist()
    for causal in (False, True):
        expect = []
        for i in range(n):
            keys = [j for j in range(n) if (not causal or j <= i)]
            maps = []
            for Q, K in ((q1, k1), (q2, k2)):
                logits = [sum(Q[i][t] * K[j][t] for t in range(d)) / math.sqrt(d) for j in keys]
                mx = max(logits)
                ex = [math.exp(x - mx) for x in logits]
                tot = sum(ex)
                maps.append([x / tot for x in ex])
            w = [maps[0][a] - lam * maps[1][a] for a in range(len(keys))]
            expect.append([sum(w[a] * v[j][c] for a, j in enumerate(keys)) for c in range(dv)])
        got = ref.diff_attn_head(np.array(q1), np.array(k1), np.array(q2), np.array(k2), np.array(v),
                                 lam, causal)
        assert np.allclose(got, np.array(expect), atol=1e-13, rtol=0)


def pin_norm_and_scale():
    rng = np.random.default_rng(7)
    dv, eps = 256, 1e-5
    O = rng.standard_normal((9, dv)) * np.array([1e-4, 1e-3, 3e-3, 1e-2, 0.1, 1, 3, 10, 100])[:, None]
    w = rng.standard_normal(dv)
    lib = F.rms_norm(torch.from_numpy(O), (dv,), torch.from_numpy(w), eps).numpy()
    assert np.allclose(ref.subln(O, w, eps), lib, atol=1e-13, rtol=1e-12)
    li = ref.lambda_init(12)
    # constant row c: every channel becomes |c| / sqrt(c^2 + eps) * (1 - lambda_init), signed
    for c in (1e-4, 3e-3, 0.5, -2.0):
        Y = ref.head_epilogue(np.full((1, dv), c), None, eps, li, norm=True, apply_scale=True)
        assert np.allclose(Y, np.sign(c) * abs(c) / math.sqrt(c * c + eps) * (1 - li), atol=1e-14, rtol=1e-12)
    Y0 = ref.head_epilogue(np.zeros((1, dv)), None, eps, li, norm=True, apply_scale=True)
    assert np.all(Y0 == 0.0)


def pin_fwd_layout():
    """q [B,N,H,2d] = [Q1|Q2]: with Q2 = K2 = 0 map 2 is uniform over the visible keys, so each
    head's output is SDPA(Q1, K1, V) - lambda_h * running-mean(V), then RMSNorm and the scale."""
    rng = np.random.default_rng(8)
    B, N, H, d, dv, eps = 2, 19, 3, 4, 8, 1e-5
    q = rng.standard_normal((B, N, H, 2 * d)); k = rng.standard_normal((B, N, H, 2 * d))
    q[..., d:] = 0.0; k[..., d:] = 0.0
    v = rng.standard_normal((B, N, H, dv))
    lam = np.array([0.3, 0.55, 0.9])
    w = rng.standard_normal(dv)
    li = ref.lambda_init(7)
    out = ref.diffattn_fwd(q, k, v, lam, li, norm_weight=w, eps=eps, causal=True)
    for b in range(B):
        for h in range(H):
            O = _sdpa(q[b, :, h, :d], k[b, :, h, :d], v[b, :, h], True) - lam[h] * _cummean(v[b, :, h])
            Y = F.rms_norm(torch.from_numpy(O), (dv,), torch.from_numpy(w), eps).numpy() * (1 - li)
            assert np.allclose(out[b, :, h], Y, atol=1e-12, rtol=1e-10), (b, h)
    rows = np.array([0, 5, 18])
    sub = ref.diffattn_fwd(q, k, v, lam, li, norm_weight=w, eps=eps, causal=True, rows=rows)
    assert np.array_equal(sub, out[:, rows])


def pin_decode_is_last_prefill_row():
    rng = np.random.default_rng(9)
    B, L, H, d, dv = 3, 23, 2, 4, 8
    kc = rng.standard_normal((B, L, H, 2 * d)); vc = rng.standard_normal((B, L, H, dv))
    q = rng.standard_normal((B, H, 2 * d))
    lam = np.array([0.4, 0.8]); li = ref.lambda_init(12); seqlens = np.array([23, 1, 11])
    out = ref.diffattn_decode(q, kc, vc, seqlens, lam, li)
    for b in range(B):
        Lb = seqlens[b]
        qp = rng.standard_normal((1, Lb, H, 2 * d)); qp[0, Lb - 1] = q[b]
        full = ref.diffattn_fwd(qp, kc[b:b + 1, :Lb], vc[b:b + 1, :Lb], lam, li, causal=True,
                                rows=np.array([Lb - 1]))
        assert np.allclose(out[b], full[0, 0], atol=1e-12, rtol=1e-12), b


def pin_v2():
    rng = np.random.default_rng(10)
    B, N, Hq, Hkv, d = 1, 17, 8, 2, 8
    q = rng.standard_normal((B, N, Hq, d)); k = rng.standard_normal((B, N, Hkv, d))
    v = rng.standard_normal((B, N, Hkv, d))
    # Query heads of one GQA group are contiguous: Hq/Hkv = 4 query heads per KV head, so pairs
    # 0 and 1 (heads 0..3) use KV head 0 and pairs 2 and 3 (heads 4..7) use KV head 1.
    expected_group = {0: 0, 1: 0, 2: 1, 3: 1}
    off = np.full((B, N, Hq // 2), -700.0)  # sigmoid -> 0: plain attention of head 2p
    out = ref.diffattn_v2_fwd(q, k, v, off, causal=True)
    for p, g in expected_group.items():
        assert np.allclose(out[0, :, p], _sdpa(q[0, :, 2 * p], k[0, :, g], v[0, :, g], True), atol=1e-12)
    q2 = q.copy(); q2[:, :, 1::2] = q2[:, :, 0::2]
    logit = rng.standard_normal((B, N, Hq // 2))
    out2 = ref.diffattn_v2_fwd(q2, k, v, logit, causal=False)
    sig = 1 / (1 + np.exp(-logit))
    for p, g in expected_group.items():
        a = _sdpa(q2[0, :, 2 * p], k[0, :, g], v[0, :, g], False)
        assert np.allclose(out2[0, :, p], (1 - sig[0, :, p])[:, None] * a, atol=1e-12)


def pin_v2_decode_is_last_prefill_row():
    rng = np.random.default_rng(11)
    B, L, Hq, Hkv, d = 3, 19, 8, 2, 8
    kc = rng.standard_normal((B, L, Hkv, d)); vc = rng.standard_normal((B, L, Hkv, d))
    q = rng.standard_normal((B, Hq, d)); logit = rng.standard_normal((B, Hq // 2))
    seqlens = np.array([19, 1, 7])
    out = ref.diffattn_v2_decode(q, kc, vc, seqlens, logit)
    for b in range(B):
        Lb = seqlens[b]
        qp = rng.standard_normal((1, Lb, Hq, d)); qp[0, Lb - 1] = q[b]
        lp = rng.standard_normal((1, Lb, Hq // 2)); lp[0, Lb - 1] = logit[b]
        full = ref.diffattn_v2_fwd(qp, kc[b:b + 1, :Lb], vc[b:b + 1, :Lb], lp, causal=True,
                                   rows=np.array([Lb - 1]))
        assert np.allclose(out[b], full[0, 0], atol=1e-12, rtol=1e-12), b


def _bwd_case(rng, B, N, H, d, dv):
    q = rng.standard_normal((B, N, H, 2 * d))
    k = rng.standard_normal((B, N, H, 2 * d))
    v = rng.standard_normal((B, N, H, dv))
    dy = rng.standard_normal((B, N, H, dv))
    lam = rng.uniform(0.1, 1.1, H)
    w = rng.uniform(0.5, 1.5, dv)
    return q, k, v, dy, lam, w


def pin_bwd_finite_differences():
    """The backward against central differences of the (separately pinned) forward: for each
    input, the directional derivative of L = sum(dy * fwd) along a random direction equals the
    inner product of the returned gradient with that direction."""
    rng = np.random.default_rng(7)
    eps = 1e-6
    for causal in (True, False):
        for norm in (True, False):
            q, k, v, dy, lam, w = _bwd_case(rng, 2, 7, 2, 3, 5)
            li = 0.35
            g = ref.diffattn_bwd(q, k, v, lam, li, dy, norm_weight=w, eps=1e-5, norm=norm,
                                 causal=causal)
            args = dict(q=q, k=k, v=v, lam=lam, w=w)

            def L(a):
                return float(np.sum(dy * ref.diffattn_fwd(a["q"], a["k"], a["v"], a["lam"], li,
                                                          norm_weight=a["w"], eps=1e-5, norm=norm,
                                                          causal=causal)))
            for name, key in (("dq", "q"), ("dk", "k"), ("dv", "v"), ("dlam", "lam"), ("dw", "w")):
                D = rng.standard_normal(np.shape(args[key]))
                hi, lo = dict(args), dict(args)
                hi[key] = args[key] + eps * D
                lo[key] = args[key] - eps * D
                fd = (L(hi) - L(lo)) / (2 * eps)
                an = float(np.sum(g[name] * D))
                assert an == pytest.approx(fd, rel=1e-6, abs=1e-8), (name, causal, norm, an, fd)


def pin_bwd_autograd():
    """The backward against torch autograd (float64) of an independent torch expression of the
    forward."""
    rng = np.random.default_rng(11)
    B, N, H, d, dv = 1, 9, 3, 4, 8
    q, k, v, dy, lam, w = _bwd_case(rng, B, N, H, d, dv)
    li, eps = 0.6, 1e-5
    t = lambda a: torch.tensor(a, dtype=torch.float64, requires_grad=True)
    tq, tk, tv, tl, tw = t(q), t(k), t(v), t(lam), t(w)
    S1 = torch.einsum("bnhd,bmhd->bhnm", tq[..., :d], tk[..., :d]) / math.sqrt(d)
    S2 = torch.einsum("bnhd,bmhd->bhnm", tq[..., d:], tk[..., d:]) / math.sqrt(d)
    mask = torch.ones(N, N, dtype=torch.bool).tril()
    S1, S2 = S1.masked_fill(~mask, float("-inf")), S2.masked_fill(~mask, float("-inf"))
    Wt = torch.softmax(S1, -1) - tl[None, :, None, None] * torch.softmax(S2, -1)
    O = torch.einsum("bhnm,bmhe->bnhe", Wt, tv)
    Y = O * torch.rsqrt((O * O).mean(-1, keepdim=True) + eps) * tw * (1 - li)
    (Y * torch.tensor(dy)).sum().backward()
    g = ref.diffattn_bwd(q, k, v, lam, li, dy, norm_weight=w, eps=eps)
    for name, tt in (("dq", tq), ("dk", tk), ("dv", tv), ("dlam", tl), ("dw", tw)):
        assert np.allclose(g[name], tt.grad.numpy(), rtol=1e-10, atol=1e-12), name


def pin_lambda_bwd():
    """Gradients of the lambda re-parameterisation against central differences."""
    rng = np.random.default_rng(5)
    vecs = [rng.standard_normal((3, 8)) * 0.3 for _ in range(4)]
    dl = rng.standard_normal(3)
    grads = ref.lambda_full_bwd(*vecs, dl)
    eps = 1e-6
    for i in range(4):
        D = rng.standard_normal(vecs[i].shape)
        hi = [x + eps * D if j == i else x for j, x in enumerate(vecs)]
        lo = [x - eps * D if j == i else x for j, x in enumerate(vecs)]
        fd = (np.sum(dl * ref.lambda_full(*hi, 12)) - np.sum(dl * ref.lambda_full(*lo, 12))) / (2 * eps)
        assert float(np.sum(grads[i] * D)) == pytest.approx(fd, rel=1e-6), i


def pin_paged_decode():
    """Paged decode equals contiguous decode when the pool is the contiguous cache cut into pages
    (identity table), and is unchanged when the pool's pages are shuffled and the table follows."""
    rng = np.random.default_rng(17)
    B, L, H, d, dv, ps = 3, 20, 2, 4, 8, 6
    max_pages = (L + ps - 1) // ps
    q = rng.standard_normal((B, H, 2 * d))
    kc = rng.standard_normal((B, max_pages * ps, H, 2 * d))
    vc = rng.standard_normal((B, max_pages * ps, H, dv))
    seqlens = np.array([20, 1, 13])
    lam = np.array([0.3, 0.7])
    want = ref.diffattn_decode(q, kc, vc, seqlens, lam, 0.4)
    k_pool = kc.reshape(B * max_pages, ps, H, 2 * d)
    v_pool = vc.reshape(B * max_pages, ps, H, dv)
    table = np.arange(B * max_pages).reshape(B, max_pages)
    got = ref.diffattn_decode_paged(q, k_pool, v_pool, table, seqlens, lam, 0.4)
    assert np.allclose(got, want, rtol=1e-12, atol=1e-12)
    perm = rng.permutation(B * max_pages)          # new slot of each old page
    k_sh = np.empty_like(k_pool); v_sh = np.empty_like(v_pool)
    k_sh[perm], v_sh[perm] = k_pool, v_pool
    got2 = ref.diffattn_decode_paged(q, k_sh, v_sh, perm[table], seqlens, lam, 0.4)
    assert np.allclose(got2, want, rtol=1e-12, atol=1e-12)


def pin_v2_paged_decode():
    """Paged V2 decode equals contiguous V2 decode over the same keys: identity table, then a
    shuffled pool with the table following it; table entries past a sequence's pages are unused."""
    rng = np.random.default_rng(23)
    B, Hq, Hkv, d, ps = 3, 8, 2, 4, 4
    max_pages = 5
    q = rng.standard_normal((B, Hq, d))
    kc = rng.standard_normal((B, max_pages * ps, Hkv, d))
    vc = rng.standard_normal((B, max_pages * ps, Hkv, d))
    seqlens = np.array([17, 3, 20])
    lam = rng.standard_normal((B, Hq // 2))
    want = ref.diffattn_v2_decode(q, kc, vc, seqlens, lam)
    k_pool = kc.reshape(B * max_pages, ps, Hkv, d)
    v_pool = vc.reshape(B * max_pages, ps, Hkv, d)
    table = np.arange(B * max_pages).reshape(B, max_pages)
    got = ref.diffattn_v2_decode_paged(q, k_pool, v_pool, table, seqlens, lam)
    assert np.allclose(got, want, rtol=1e-12, atol=1e-12)
    perm = rng.permutation(B * max_pages)
    k_sh = np.empty_like(k_pool); v_sh = np.empty_like(v_pool)
    k_sh[perm], v_sh[perm] = k_pool, v_pool
    t2 = perm[table]
    t2[1, 1:] = -1                                   # sequence 1 holds 3 keys: one page
    got2 = ref.diffattn_v2_decode_paged(q, k_sh, v_sh, t2, seqlens, lam)
    assert np.allclose(got2, want, rtol=1e-12, atol=1e-12)


def pin_varlen():
    """Packed sequences: with equal lengths the result is the batched prefill's; and each sequence
    sees only itself (changing another sequence's tokens leaves its rows unchanged)."""
    rng = np.random.default_rng(19)
    B, N, H, d, dv = 3, 7, 2, 4, 8
    q = rng.standard_normal((B, N, H, 2 * d)); k = rng.standard_normal((B, N, H, 2 * d))
    v = rng.standard_normal((B, N, H, dv)); lam = np.array([0.2, 0.9])
    cu = np.arange(B + 1) * N
    got = ref.diffattn_fwd_varlen(q.reshape(B * N, H, 2 * d), k.reshape(B * N, H, 2 * d),
                                  v.reshape(B * N, H, dv), cu, lam, 0.3)
    want = ref.diffattn_fwd(q, k, v, lam, 0.3).reshape(B * N, H, dv)
    assert np.allclose(got, want, rtol=1e-12, atol=1e-12)
    cu2 = np.array([0, 5, 5, 12, 20])
    T = 21
    q2, k2, v2 = (rng.standard_normal((T, H, w)) for w in (2 * d, 2 * d, dv))
    a = ref.diffattn_fwd_varlen(q2, k2, v2, cu2, lam, 0.3)
    k3 = k2.copy(); k3[5:12] += rng.standard_normal(k3[5:12].shape); v3 = v2.copy(); v3[12:20] -= 2.0
    b = ref.diffattn_fwd_varlen(q2, k3, v3, cu2, lam, 0.3)
    assert np.allclose(a[0:5], b[0:5]) and not np.allclose(a[5:12], b[5:12])
    assert np.allclose(a[5:12], ref.diffattn_fwd(q2[None, 5:12], k2[None, 5:12], v2[None, 5:12], lam, 0.3)[0])
    assert np.all(a[20] == 0)


def pin_varlen_qk():
    """Queries as the last Lq of Lk positions: they equal those rows of the full prefill (the
    earlier queries do not matter), Lq = Lk is the packed prefill, and Lq = 1 is the decode of
    the last position over all Lk keys."""
    rng = np.random.default_rng(29)
    H, d, dv = 2, 4, 8
    Lks, Lqs = [9, 5, 12, 7], [4, 5, 1, 0]
    lam = np.array([0.35, 0.8])
    k = rng.standard_normal((sum(Lks), H, 2 * d)); v = rng.standard_normal((sum(Lks), H, dv))
    qf = rng.standard_normal((sum(Lks), H, 2 * d))          # a query for every key position
    cu_k = np.concatenate([[0], np.cumsum(Lks)])
    # the last Lq query rows of each sequence, packed
    q = np.concatenate([qf[cu_k[i + 1] - Lqs[i]:cu_k[i + 1]] for i in range(4)])
    cu_q = np.concatenate([[0], np.cumsum(Lqs)])
    got = ref.diffattn_fwd_varlen_qk(q, k, v, cu_q, cu_k, lam, 0.3)
    full = ref.diffattn_fwd_varlen(qf, k, v, cu_k, lam, 0.3)
    want = np.concatenate([full[cu_k[i + 1] - Lqs[i]:cu_k[i + 1]] for i in range(4)])
    assert np.allclose(got, want, rtol=1e-12, atol=1e-12)
    # Lq = 1 (sequence 2): the decode of its last position over its 12 keys
    s0 = cu_k[2]
    dec = ref.diffattn_decode(q[None, cu_q[2], :, :], k[None, s0:s0 + 12], v[None, s0:s0 + 12],
                              np.array([12]), lam, 0.3)
    assert np.allclose(got[cu_q[2]], dec[0], rtol=1e-12, atol=1e-12)
    # non-causal: every query row sees all of its sequence's keys, whatever its position
    nc = ref.diffattn_fwd_varlen_qk(q, k, v, cu_q, cu_k, lam, 0.3, causal=False)
    full_nc = ref.diffattn_fwd_varlen(qf, k, v, cu_k, lam, 0.3, causal=False)
    want_nc = np.concatenate([full_nc[cu_k[i + 1] - Lqs[i]:cu_k[i + 1]] for i in range(4)])
    assert np.allclose(nc, want_nc, rtol=1e-12, atol=1e-12)


def pin_v2_varlen():
    """V2 over packed sequences: with shared offsets each sequence equals the batched V2 prefill
    of that sequence alone; with keys of their own, the queries equal the last rows of the full
    sequence's V2 prefill."""
    rng = np.random.default_rng(31)
    Hq, Hkv, d = 8, 2, 4
    lens = [6, 1, 9]
    T = sum(lens)
    q = rng.standard_normal((T, Hq, d)); k = rng.standard_normal((T, Hkv, d))
    v = rng.standard_normal((T, Hkv, d)); lam = rng.standard_normal((T, Hq // 2))
    cu = np.concatenate([[0], np.cumsum(lens)])
    got = ref.diffattn_v2_fwd_varlen(q, k, v, lam, cu)
    for i in range(3):
        a, b = cu[i], cu[i + 1]
        one = ref.diffattn_v2_fwd(q[None, a:b], k[None, a:b], v[None, a:b], lam[None, a:b])[0]
        assert np.allclose(got[a:b], one, rtol=1e-12, atol=1e-12)
    # sequence 2 (9 positions) with only its last 4 queries
    a, b = cu[2], cu[3]
    cu_q, cu_k = np.array([0, 4]), np.array([0, 9])
    part = ref.diffattn_v2_fwd_varlen(q[b - 4:b], k[a:b], v[a:b], lam[b - 4:b], cu_q, cu_k)
    assert np.allclose(part, got[b - 4:b], rtol=1e-12, atol=1e-12)


def pin_paged_prefill():
    """Prefill over pages: with the pool holding each sequence's keys in order (identity table)
    it is the packed prefill over those keys, and shuffling the pool's pages with the table
    following them changes nothing; V2 likewise."""
    rng = np.random.default_rng(37)
    H, d, dv, ps = 2, 4, 8, 3
    Lk, Lq = [7, 3], [2, 3]
    mp = 3
    kc = rng.standard_normal((2, mp * ps, H, 2 * d)); vc = rng.standard_normal((2, mp * ps, H, dv))
    q = rng.standard_normal((sum(Lq), H, 2 * d)); lam = np.array([0.4, 0.9])
    cu_q = np.concatenate([[0], np.cumsum(Lq)])
    k_pool = kc.reshape(2 * mp, ps, H, 2 * d); v_pool = vc.reshape(2 * mp, ps, H, dv)
    table = np.arange(2 * mp).reshape(2, mp)
    got = ref.diffattn_fwd_paged(q, k_pool, v_pool, cu_q, np.array(Lk), table, lam, 0.2)
    kp = np.concatenate([kc[0, :7], kc[1, :3]]); vp = np.concatenate([vc[0, :7], vc[1, :3]])
    want = ref.diffattn_fwd_varlen_qk(q, kp, vp, cu_q, np.array([0, 7, 10]), lam, 0.2)
    assert np.allclose(got, want, rtol=1e-12, atol=1e-12)
    perm = rng.permutation(2 * mp)
    k_sh = np.empty_like(k_pool); v_sh = np.empty_like(v_pool)
    k_sh[perm], v_sh[perm] = k_pool, v_pool
    got2 = ref.diffattn_fwd_paged(q, k_sh, v_sh, cu_q, np.array(Lk), perm[table], lam, 0.2)
    assert np.allclose(got2, want, rtol=1e-12, atol=1e-12)
    Hq, Hkv = 4, 2
    q2 = rng.standard_normal((sum(Lq), Hq, d)); lg = rng.standard_normal((sum(Lq), Hq // 2))
    k2 = rng.standard_normal((2 * mp, ps, Hkv, d)); v2 = rng.standard_normal((2 * mp, ps, Hkv, d))
    a = ref.diffattn_v2_fwd_paged(q2, k2, v2, lg, cu_q, np.array(Lk), table)
    flat_k, flat_v = k2.reshape(2 * mp * ps, Hkv, d), v2.reshape(2 * mp * ps, Hkv, d)
    rows = np.concatenate([np.arange(7), mp * ps + np.arange(3)])
    b = ref.diffattn_v2_fwd_varlen(q2, flat_k[rows], flat_v[rows], lg, cu_q, np.array([0, 7, 10]))
    assert np.allclose(a, b, rtol=1e-12, atol=1e-12)


def pin_bwd_varlen():
    """Packed backward: with equal lengths it is the batched backward; the per-sequence dlam
    partial sums add up to the whole."""
    rng = np.random.default_rng(41)
    B, N, H, d, dv = 2, 5, 2, 4, 8
    q = rng.standard_normal((B, N, H, 2 * d)); k = rng.standard_normal((B, N, H, 2 * d))
    v = rng.standard_normal((B, N, H, dv)); dy = rng.standard_normal((B, N, H, dv))
    lam = np.array([0.3, 0.7]); w = rng.uniform(0.5, 1.5, dv)
    want = ref.diffattn_bwd(q, k, v, lam, 0.2, dy, norm_weight=w)
    cu = np.array([0, N, 2 * N])
    got = ref.diffattn_bwd_varlen(q.reshape(B * N, H, -1), k.reshape(B * N, H, -1),
                                  v.reshape(B * N, H, -1), cu, lam, 0.2, dy.reshape(B * N, H, -1),
                                  norm_weight=w)
    for name in ("dq", "dk", "dv"):
        assert np.allclose(got[name], want[name].reshape(B * N, H, -1), rtol=1e-12, atol=1e-12)
    assert np.allclose(got["dlam"], want["dlam"], rtol=1e-12, atol=1e-12)
    assert np.allclose(got["dw"], want["dw"], rtol=1e-12, atol=1e-12)


def pin_gda():
    """Grouped prefill: with one noise head per signal head it is the ungrouped operator; with G
    signal heads per noise head it is the ungrouped operator whose Q2, K2 of head h are copies of
    noise head floor(h / G) (repetition over contiguous groups); a noise head reaches exactly the
    signal heads of its own group."""
    rng = np.random.default_rng(43)
    B, N, d, dv, li = 2, 9, 4, 8, 0.35
    w = rng.uniform(0.5, 1.5, dv)
    for Hs, Hn in ((3, 3), (6, 2), (4, 1)):
        G = Hs // Hn
        q = rng.standard_normal((B, N, Hs + Hn, d)); k = rng.standard_normal((B, N, Hs + Hn, d))
        v = rng.standard_normal((B, N, Hs, dv)); lam = rng.uniform(0.1, 0.9, Hs)
        rep = np.repeat(np.arange(Hs, Hs + Hn), G)            # noise head of each signal head
        q_v1 = np.concatenate([q[:, :, :Hs], q[:, :, rep]], axis=-1)
        k_v1 = np.concatenate([k[:, :, :Hs], k[:, :, rep]], axis=-1)
        for causal in (False, True):
            want = ref.diffattn_fwd(q_v1, k_v1, v, lam, li, norm_weight=w, causal=causal)
            got = ref.diffattn_gda_fwd(q, k, v, lam, li, Hs, norm_weight=w, causal=causal)
            assert np.allclose(got, want, rtol=1e-12, atol=1e-12)
        if Hn > 1:
            base = ref.diffattn_gda_fwd(q, k, v, lam, li, Hs, norm=False, apply_scale=False)
            q2 = q.copy(); q2[:, :, Hs + 1] += 1.0               # move noise head 1 only
            moved = ref.diffattn_gda_fwd(q2, k, v, lam, li, Hs, norm=False, apply_scale=False)
            same = np.all(np.isclose(moved, base, rtol=0, atol=0), axis=(0, 1, 3))
            assert same.tolist() == [h // G != 1 for h in range(Hs)]


def pin_gda_bwd():
    """Grouped backward: with one noise head per signal head it is the ungrouped backward on the
    halves stored as heads; every gradient matches central differences of the grouped forward's
    loss <dy, Y> (a noise head's gradient collects its whole group)."""
    rng = np.random.default_rng(37)
    B, N, H, d, dv = 1, 5, 2, 3, 4
    q1, q2, k1, k2 = (rng.standard_normal((B, N, H, d)) for _ in range(4))
    v = rng.standard_normal((B, N, H, dv)); dy = rng.standard_normal((B, N, H, dv))
    lam = np.array([0.3, 0.8]); w = np.linspace(0.5, 1.5, dv)
    g = ref.diffattn_gda_bwd(np.concatenate([q1, q2], 2), np.concatenate([k1, k2], 2), v, lam,
                             0.4, H, dy, norm_weight=w)
    u = ref.diffattn_bwd(np.concatenate([q1, q2], 3), np.concatenate([k1, k2], 3), v, lam, 0.4, dy,
                         norm_weight=w)
    assert np.allclose(g["dq"][:, :, :H], u["dq"][..., :d]) and np.allclose(g["dq"][:, :, H:], u["dq"][..., d:])
    assert np.allclose(g["dk"][:, :, :H], u["dk"][..., :d]) and np.allclose(g["dk"][:, :, H:], u["dk"][..., d:])
    assert np.allclose(g["dv"], u["dv"]) and np.allclose(g["dlam"], u["dlam"]) and np.allclose(g["dw"], u["dw"])
    # grouped: 3 signal heads over 1 noise head, central differences
    Hs, Hn = 3, 1
    q = rng.standard_normal((1, 4, Hs + Hn, d)); k = rng.standard_normal((1, 4, Hs + Hn, d))
    v = rng.standard_normal((1, 4, Hs, dv)); dy = rng.standard_normal((1, 4, Hs, dv))
    lam = np.array([0.2, 0.5, 0.9])
    grads = ref.diffattn_gda_bwd(q, k, v, lam, 0.4, Hs, dy, norm_weight=w)
    loss = lambda q_, k_, v_, lam_, w_: float(np.sum(dy * ref.diffattn_gda_fwd(
        q_, k_, v_, lam_, 0.4, Hs, norm_weight=w_)))
    h = 1e-6
    for name, x in (("dq", q), ("dk", k), ("dv", v)):
        for idx in [(0, 3, Hs, 1), (0, 2, 0, 2), (0, 1, 2, 0)] if name != "dv" else [(0, 3, 1, 2), (0, 0, 2, 3)]:
            xp = x.copy(); xm = x.copy(); xp[idx] += h; xm[idx] -= h
            args_p = [q, k, v]; args_m = [q, k, v]
            pos = ("dq", "dk", "dv").index(name)
            args_p[pos] = xp; args_m[pos] = xm
            fd = (loss(*args_p, lam, w) - loss(*args_m, lam, w)) / (2 * h)
            assert abs(fd - grads[name][idx]) < 1e-6 * max(1.0, abs(fd)), (name, idx)
    for i in range(Hs):
        lp = lam.copy(); lm = lam.copy(); lp[i] += h; lm[i] -= h
        fd = (loss(q, k, v, lp, w) - loss(q, k, v, lm, w)) / (2 * h)
        assert abs(fd - grads["dlam"][i]) < 1e-6 * max(1.0, abs(fd))
    for c in (0, 3):
        wp = w.copy(); wm = w.copy(); wp[c] += h; wm[c] -= h
        fd = (loss(q, k, v, lam, wp) - loss(q, k, v, lam, wm)) / (2 * h)
        assert abs(fd - grads["dw"][c]) < 1e-6 * max(1.0, abs(fd))


def pin_gda_varlen():
    """Packed grouped prefill: with equal lengths it is the batched grouped prefill; with one noise
    head per signal head it is the ungrouped packed prefill on the halves stored as heads; each
    sequence sees only itself."""
    rng = np.random.default_rng(23)
    B, N, Hs, Hn, d, dv = 2, 6, 4, 2, 4, 8
    q = rng.standard_normal((B, N, Hs + Hn, d)); k = rng.standard_normal((B, N, Hs + Hn, d))
    v = rng.standard_normal((B, N, Hs, dv)); lam = np.array([0.1, 0.5, 0.9, 0.3])
    cu = np.arange(B + 1) * N
    got = ref.diffattn_gda_fwd_varlen(q.reshape(B * N, Hs + Hn, d), k.reshape(B * N, Hs + Hn, d),
                                      v.reshape(B * N, Hs, dv), cu, lam, 0.2, Hs)
    want = ref.diffattn_gda_fwd(q, k, v, lam, 0.2, Hs).reshape(B * N, Hs, dv)
    assert np.allclose(got, want, rtol=1e-12, atol=1e-12)
    # n_noise = n_signal on packed rows: the ungrouped packed operator with [Q1 | Q2] halves
    cu2 = np.array([0, 3, 3, 9, 10]); T = 11; H = 3
    q1, q2, k1, k2 = (rng.standard_normal((T, H, d)) for _ in range(4))
    vv = rng.standard_normal((T, H, dv)); lam3 = np.array([0.7, 0.2, 0.4])
    g = ref.diffattn_gda_fwd_varlen(np.concatenate([q1, q2], 1), np.concatenate([k1, k2], 1), vv,
                                    cu2, lam3, 0.3, H)
    u = ref.diffattn_fwd_varlen(np.concatenate([q1, q2], 2), np.concatenate([k1, k2], 2), vv, cu2,
                                lam3, 0.3)
    assert np.allclose(g, u, rtol=1e-12, atol=1e-12) and np.all(g[10] == 0)
    # independence: another sequence's noise keys do not reach this one
    qq = np.concatenate([q1, q2], 1)[:, :H + 1]; kk = np.concatenate([k1, k2], 1)[:, :H + 1]
    a = ref.diffattn_gda_fwd_varlen(qq, kk, vv, cu2, lam3, 0.3, H)
    kk2 = kk.copy(); kk2[3:9, H] += rng.standard_normal((6, d))  # (a shared shift would cancel)
    b = ref.diffattn_gda_fwd_varlen(qq, kk2, vv, cu2, lam3, 0.3, H)
    assert np.allclose(a[:3], b[:3]) and np.allclose(a[9], b[9]) and not np.allclose(a[3:9], b[3:9])


def pin_gda_bwd_varlen():
    """Packed grouped backward: with equal lengths it is the batched grouped backward; with one
    noise head per signal head it is the ungrouped packed backward on the halves stored as heads;
    rows in no sequence get zero gradients and a sequence's gradients see only itself."""
    rng = np.random.default_rng(47)
    B, N, Hs, Hn, d, dv = 2, 5, 4, 2, 3, 4
    q = rng.standard_normal((B, N, Hs + Hn, d)); k = rng.standard_normal((B, N, Hs + Hn, d))
    v = rng.standard_normal((B, N, Hs, dv)); dy = rng.standard_normal((B, N, Hs, dv))
    lam = np.array([0.2, 0.6, 0.9, 0.4]); w = rng.uniform(0.5, 1.5, dv)
    want = ref.diffattn_gda_bwd(q, k, v, lam, 0.3, Hs, dy, norm_weight=w)
    got = ref.diffattn_gda_bwd_varlen(q.reshape(B * N, Hs + Hn, d), k.reshape(B * N, Hs + Hn, d),
                                      v.reshape(B * N, Hs, dv), np.arange(B + 1) * N, lam, 0.3, Hs,
                                      dy.reshape(B * N, Hs, dv), norm_weight=w)
    for name in ("dq", "dk", "dv"):
        assert np.allclose(got[name], want[name].reshape(B * N, *want[name].shape[2:]), rtol=1e-12,
                           atol=1e-12), name
    assert np.allclose(got["dlam"], want["dlam"]) and np.allclose(got["dw"], want["dw"])
    # n_noise = n_signal: the ungrouped packed backward on [Q1 | Q2], an empty sequence, a tail
    cu = np.array([0, 3, 3, 8]); T, H = 9, 2
    q1, q2, k1, k2 = (rng.standard_normal((T, H, d)) for _ in range(4))
    vv = rng.standard_normal((T, H, dv)); dd = rng.standard_normal((T, H, dv))
    lam2 = np.array([0.5, 0.8])
    g = ref.diffattn_gda_bwd_varlen(np.concatenate([q1, q2], 1), np.concatenate([k1, k2], 1), vv,
                                    cu, lam2, 0.3, H, dd, norm_weight=w)
    u = ref.diffattn_bwd_varlen(np.concatenate([q1, q2], 2), np.concatenate([k1, k2], 2), vv, cu,
                                lam2, 0.3, dd, norm_weight=w)
    assert np.allclose(g["dq"][:, :H], u["dq"][..., :d]) and np.allclose(g["dq"][:, H:], u["dq"][..., d:])
    assert np.allclose(g["dk"][:, :H], u["dk"][..., :d]) and np.allclose(g["dk"][:, H:], u["dk"][..., d:])
    assert np.allclose(g["dv"], u["dv"]) and np.allclose(g["dlam"], u["dlam"]) and np.allclose(g["dw"], u["dw"])
    assert not g["dq"][8].any() and not g["dk"][8].any() and not g["dv"][8].any()
    # a sequence's gradients do not depend on another sequence's rows
    k3 = np.concatenate([k1, k2], 1).copy(); k3[3:8] += rng.standard_normal((5, 2 * H, d))
    g3 = ref.diffattn_gda_bwd_varlen(np.concatenate([q1, q2], 1), k3, vv, cu, lam2, 0.3, H, dd,
                                     norm_weight=w)
    assert np.allclose(g3["dq"][:3], g["dq"][:3]) and np.allclose(g3["dk"][:3], g["dk"][:3])
    assert not np.allclose(g3["dq"][3:8], g["dq"][3:8])


def pin_gda_varlen_qk_and_paged():
    """Grouped prefill with queries at the end of their keys: with Lq = Lk it is the packed grouped
    prefill; each query row equals that row of the whole sequence's grouped prefill; with one noise
    head per signal head it is the ungrouped form on the halves stored as heads; paged keys
    through any table give the same result."""
    rng = np.random.default_rng(31)
    Hs, Hn, d, dv = 4, 2, 4, 8
    lam = np.array([0.3, 0.5, 0.7, 0.9])
    lk = [9, 1, 6]; lq = [3, 1, 6]
    cu_k = np.concatenate([[0], np.cumsum(lk)]); cu_q = np.concatenate([[0], np.cumsum(lq)])
    k = rng.standard_normal((cu_k[-1], Hs + Hn, d)); v = rng.standard_normal((cu_k[-1], Hs, dv))
    qk = rng.standard_normal((cu_k[-1], Hs + Hn, d))   # queries at every key position
    q = np.concatenate([qk[cu_k[b + 1] - lq[b]:cu_k[b + 1]] for b in range(3)])
    for causal in (True, False):
        got = ref.diffattn_gda_fwd_varlen_qk(q, k, v, cu_q, cu_k, lam, 0.4, Hs, causal=causal)
        whole = ref.diffattn_gda_fwd_varlen(qk, k, v, cu_k, lam, 0.4, Hs, causal=causal)
        want = np.concatenate([whole[cu_k[b + 1] - lq[b]:cu_k[b + 1]] for b in range(3)])
        assert np.allclose(got, want, rtol=1e-12, atol=1e-12)
    same = ref.diffattn_gda_fwd_varlen_qk(qk, k, v, cu_k, cu_k, lam, 0.4, Hs)
    assert np.allclose(same, ref.diffattn_gda_fwd_varlen(qk, k, v, cu_k, lam, 0.4, Hs),
                       rtol=1e-12, atol=1e-12)
    # one noise head per signal head: the ungrouped chunked form on [Q1 | Q2] halves
    H = 3
    q1, q2 = rng.standard_normal((cu_q[-1], H, d)), rng.standard_normal((cu_q[-1], H, d))
    k1, k2 = rng.standard_normal((cu_k[-1], H, d)), rng.standard_normal((cu_k[-1], H, d))
    vv = rng.standard_normal((cu_k[-1], H, dv)); lam3 = np.array([0.2, 0.6, 0.8])
    g = ref.diffattn_gda_fwd_varlen_qk(np.concatenate([q1, q2], 1), np.concatenate([k1, k2], 1),
                                       vv, cu_q, cu_k, lam3, 0.3, H)
    u = ref.diffattn_fwd_varlen_qk(np.concatenate([q1, q2], 2), np.concatenate([k1, k2], 2), vv,
                                   cu_q, cu_k, lam3, 0.3)
    assert np.allclose(g, u, rtol=1e-12, atol=1e-12)
    # paged: pages of 4 keys, shuffled in the pool
    ps = 4
    mp = max((n + ps - 1) // ps for n in lk)
    pool_k = np.zeros((3 * mp, ps, Hs + Hn, d)); pool_v = np.zeros((3 * mp, ps, Hs, dv))
    perm = rng.permutation(3 * mp); table = perm.reshape(3, mp)
    for b in range(3):
        for j in range(lk[b]):
            pool_k[table[b, j // ps], j % ps] = k[cu_k[b] + j]
            pool_v[table[b, j // ps], j % ps] = v[cu_k[b] + j]
    paged = ref.diffattn_gda_fwd_paged(q, pool_k, pool_v, cu_q, np.array(lk), table, lam, 0.4, Hs)
    assert np.allclose(paged, ref.diffattn_gda_fwd_varlen_qk(q, k, v, cu_q, cu_k, lam, 0.4, Hs),
                       rtol=1e-12, atol=1e-12)


def pin_gda_decode_paged():
    """Paged grouped decode equals the contiguous grouped decode over the same keys: identity
    table, then the pool's pages shuffled with the table following; ragged lengths."""
    rng = np.random.default_rng(29)
    B, L, Hs, Hn, d, dv, ps = 3, 17, 4, 2, 4, 8, 5
    max_pages = (L + ps - 1) // ps
    q = rng.standard_normal((B, Hs + Hn, d))
    kc = rng.standard_normal((B, max_pages * ps, Hs + Hn, d))
    vc = rng.standard_normal((B, max_pages * ps, Hs, dv))
    seqlens = np.array([17, 1, 9])
    lam = np.array([0.2, 0.5, 0.7, 0.9])
    want = ref.diffattn_gda_decode(q, kc, vc, seqlens, lam, 0.4, Hs)
    k_pool = kc.reshape(B * max_pages, ps, Hs + Hn, d)
    v_pool = vc.reshape(B * max_pages, ps, Hs, dv)
    table = np.arange(B * max_pages).reshape(B, max_pages)
    got = ref.diffattn_gda_decode_paged(q, k_pool, v_pool, table, seqlens, lam, 0.4, Hs)
    assert np.allclose(got, want, rtol=1e-12, atol=1e-12)
    perm = rng.permutation(B * max_pages)
    k_sh = np.empty_like(k_pool); v_sh = np.empty_like(v_pool)
    k_sh[perm], v_sh[perm] = k_pool, v_pool
    got2 = ref.diffattn_gda_decode_paged(q, k_sh, v_sh, perm[table], seqlens, lam, 0.4, Hs)
    assert np.allclose(got2, want, rtol=1e-12, atol=1e-12)
    # keys past a sequence's length (rows 1.. of the one-key sequence's page) do not reach it;
    # a key inside it (row 0 of sequence 0's first page) does
    k_sh2 = k_sh.copy(); k_sh2[perm[table[1, 0]], 1:] += rng.standard_normal((ps - 1, Hs + Hn, d))
    got3 = ref.diffattn_gda_decode_paged(q, k_sh2, v_sh, perm[table], seqlens, lam, 0.4, Hs)
    assert np.allclose(got3, want, rtol=1e-12, atol=1e-12)
    k_sh3 = k_sh.copy(); k_sh3[perm[table[0, 0]], 0] += rng.standard_normal((Hs + Hn, d))
    got4 = ref.diffattn_gda_decode_paged(q, k_sh3, v_sh, perm[table], seqlens, lam, 0.4, Hs)
    assert not np.allclose(got4[0], want[0]) and np.allclose(got4[1:], want[1:])


def pin_gda_decode_is_last_prefill_row():
    """Grouped decode equals the last row of a causal grouped prefill over the same keys."""
    rng = np.random.default_rng(47)
    B, L, Hs, Hn, d, dv = 2, 11, 4, 2, 4, 8
    q = rng.standard_normal((B, L, Hs + Hn, d)); k = rng.standard_normal((B, L, Hs + Hn, d))
    v = rng.standard_normal((B, L, Hs, dv)); lam = rng.uniform(0.1, 0.9, Hs)
    full = ref.diffattn_gda_fwd(q, k, v, lam, 0.4, Hs, causal=True)
    got = ref.diffattn_gda_decode(q[:, -1], k, v, np.array([L, L]), lam, 0.4, Hs)
    assert np.allclose(got, full[:, -1], rtol=1e-12, atol=1e-12)
    short = ref.diffattn_gda_decode(q[:, 5], k, v, np.array([6, 6]), lam, 0.4, Hs)
    assert np.allclose(short, full[:, 5], rtol=1e-12, atol=1e-12)


PINS = [pin_lambda_init_table, pin_lambda_init_shape, pin_lambda_closed_forms, pin_lambda_spread,
        pin_softmax_floor, pin_toy_needle_table, pin_worked_example, pin_row_sums,
        pin_lambda_zero_is_softmax_attention, pin_equal_maps_scale_attention, pin_brute_force_tiny,
        pin_norm_and_scale, pin_fwd_layout, pin_decode_is_last_prefill_row, pin_v2,
        pin_v2_decode_is_last_prefill_row, pin_bwd_finite_differences, pin_bwd_autograd,
        pin_lambda_bwd, pin_paged_decode, pin_v2_paged_decode, pin_varlen, pin_varlen_qk,
        pin_v2_varlen, pin_paged_prefill, pin_bwd_varlen, pin_gda, pin_gda_bwd, pin_gda_bwd_varlen, pin_gda_varlen,
        pin_gda_varlen_qk_and_paged, pin_gda_decode_paged, pin_gda_decode_is_last_prefill_row]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin()


# ------------------------------------------------------------------------------------------
# planted mistakes: each must make at least one pin fail
# ------------------------------------------------------------------------------------------

def _mutants():
    orig = {n: getattr(ref, n) for n in ("lambda_init", "lambda_full", "scores", "diff_weights",
                                         "subln", "head_epilogue", "v2_kv_head", "softmax_rows",
                                         "diff_attn_head_bwd", "lambda_full_bwd",
                                         "gda_noise_head")}

    def bwd_dlam_sign(*a):
        g = orig["diff_attn_head_bwd"](*a)
        return g[:5] + (-g[5],)

    def lambda_bwd_swapped(lq1, lk1, lq2, lk2, dlam):
        g = orig["lambda_full_bwd"](lq1, lk1, lq2, lk2, dlam)
        return g[1], g[0], g[2], g[3]

    def scores_wrong_scale(Q, K, row_ids, causal):
        return orig["scores"](Q, K, row_ids, causal) * math.sqrt(Q.shape[-1]) / math.sqrt(2 * Q.shape[-1])

    def scores_transposed(Q, K, row_ids, causal):
        S = (K @ Q.T) if Q.shape[0] == K.shape[0] else (Q @ K.T)
        S = S / math.sqrt(Q.shape[-1])
        if causal:
            S = np.where(np.arange(K.shape[0])[None, :] > row_ids[:, None], -np.inf, S)
        return S

    def scores_mask_off_by_one(Q, K, row_ids, causal):
        S = (Q @ K.T) / math.sqrt(Q.shape[-1])
        if causal:
            S = np.where(np.arange(K.shape[0])[None, :] >= row_ids[:, None], -np.inf, S)
            S[:, 0] = np.where(row_ids == 0, 0.0, S[:, 0])
        return S

    return {
        "lambda_init sign": ("lambda_init", lambda l: 0.8 - 0.6 * math.exp(0.3 * (l - 1))),
        "lambda_init index base": ("lambda_init", lambda l: 0.8 - 0.6 * math.exp(-0.3 * l)),
        "lambda_full plus": ("lambda_full", lambda a, b, c, d, layer: orig["lambda_full"](a, b, c, d, layer)
                             + 2 * np.exp(np.sum(ref._f64(c) * ref._f64(d), axis=-1))),
        "scale sqrt(2d)": ("scores", scores_wrong_scale),
        "scores transposed": ("scores", scores_transposed),
        "mask off by one": ("scores", scores_mask_off_by_one),
        "diff plus": ("diff_weights", lambda S1, S2, lam: ref.softmax_rows(S1) + lam * ref.softmax_rows(S2)),
        "softmax wrong axis": ("softmax_rows", lambda S: np.exp(S) / np.sum(np.exp(S), axis=0, keepdims=True)),
        "norm without eps": ("subln", lambda O, w, eps: ref._f64(O) / np.sqrt(np.mean(ref._f64(O) ** 2, -1, keepdims=True)) * (1.0 if w is None else ref._f64(w))),
        "scale 1+lambda_init": ("head_epilogue", lambda O, w, eps, li, norm, apply_scale:
                                orig["head_epilogue"](O, w, eps, li, norm, False) * ((1 + li) if apply_scale else 1)),
        "v2 wrong group": ("v2_kv_head", lambda p, Hq, Hkv: p // (Hq // Hkv)),
        "softmax bwd without row term": ("softmax_rows_bwd", lambda A, dA: A * dA),
        "norm bwd without projection": ("subln_bwd", lambda O, w, eps, dY: (
            ref._f64(dY) * (1.0 if w is None else ref._f64(w))
            / np.sqrt(np.mean(ref._f64(O) ** 2, -1, keepdims=True) + eps),
            np.zeros(np.shape(O)[-1]))),
        "dlam sign": ("diff_attn_head_bwd", bwd_dlam_sign),
        "lambda bwd q/k swapped": ("lambda_full_bwd", lambda_bwd_swapped),
        "varlen: one sequence": ("varlen_segments", lambda cu: [(0, int(np.asarray(cu)[-1]))]),
        "gda noise heads interleaved": ("gda_noise_head", lambda h, hs, hn: h % hn),
        "queries at the first positions": ("query_positions", lambda Lq, Lk: np.arange(Lq)),
        "paged row: page and offset swapped": ("paged_rows", lambda table, sl, ps, b: (
            np.asarray(ref._f64(table)).astype(np.int64)[b, np.arange(int(np.asarray(ref._f64(sl))[b])) % ps]
            * ps + np.arange(int(np.asarray(ref._f64(sl))[b])) // ps)),
    }


# The two statistical pins (thousands of draws) run last: a mistake is caught as soon as one pin
# fails, so most mutants never reach them.
_SLOW_PINS = (pin_toy_needle_table, pin_lambda_spread)
PINS_CHEAP_FIRST = [p for p in PINS if p not in _SLOW_PINS] + list(_SLOW_PINS)


@pytest.mark.parametrize("name", list(_mutants().keys()))
def test_planted_mistakes_are_caught(name, monkeypatch):
    attr, fn = _mutants()[name]
    monkeypatch.setattr(ref, attr, fn)
    caught_by = None
    for pin in PINS_CHEAP_FIRST:
        try:
            with np.errstate(all="ignore"):
                pin()
        except (AssertionError, FloatingPointError, ValueError, IndexError):
            caught_by = pin.__name__
            break
    assert caught_by, f"planted mistake '{name}' passed every pin"
