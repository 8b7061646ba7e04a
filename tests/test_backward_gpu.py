"""GPU parity of the training path (forward with saved statistics, then the backward) against
the float64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import differential_attention_gb300 as da
from oracle import diffattn_ref as ref
from synth import make_dout, make_prefill_inputs
from tests.gpu_util import assert_bf16, assert_grad

pytestmark = pytest.mark.gpu

DEV = "cuda"
LAYER = 12


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    da.build()
    da.lib()
    yield
    da.diffattn_device_status()


def _case(B, N, H, seed, causal):
    inp = make_prefill_inputs(B, N, H, 128, 256, seed=seed, layer=LAYER, causal=causal)
    dy = make_dout(B, N, H, 256, seed=seed + 7)
    lam = np.linspace(0.3, 0.9, H)
    w = torch.linspace(0.8, 1.2, 256, dtype=torch.float32)
    return inp, dy, lam, w


def _log2_sum_exp(Q, K, causal):
    """Per row, log2 sum_j exp(s_ij) with s = Q K^T / sqrt(d) from the oracle's scores."""
    S = ref.scores(ref._f64(Q), ref._f64(K), np.arange(Q.shape[0]), causal)
    m = np.max(S, axis=-1, keepdims=True)
    return (m[:, 0] + np.log(np.sum(np.exp(S - m), axis=-1))) / np.log(2.0)


def _dlam_term_scale(inp, dy, lam, li, w, norm, scale, causal):
    """Per head, sum over rows of |dO_i| |O2_i| (oracle pieces): the size of the terms whose sum is
    -dlambda. dlambda can cancel far below it (with one visible key the norm's gradient is
    orthogonal to O = (1 - lambda) V_0), and the kernel's error follows the terms: each is formed
    from dO rounded to bf16."""
    B, N, H, two_d = inp.q.shape
    d = two_d // 2
    out = np.zeros(H)
    s = (1.0 - li) if scale else 1.0
    for b in range(B):
        for h in range(H):
            O = ref.diff_attn_head(inp.q[b, :, h, :d], inp.k[b, :, h, :d], inp.q[b, :, h, d:],
                                   inp.k[b, :, h, d:], inp.v[b, :, h], float(lam[h]), causal)
            dys = ref._f64(dy[b, :, h]) * s
            dO = ref.subln_bwd(O, w, 1e-5, dys)[0] if norm else dys
            O2 = ref.attention_head(inp.q[b, :, h, d:], inp.k[b, :, h, d:], inp.v[b, :, h], causal)
            out[h] += float(np.sum(np.linalg.norm(dO, axis=-1) * np.linalg.norm(O2, axis=-1)))
    return out


def _assert_dlam(got, want, term_scale):
    g = got.double().cpu().numpy()
    bound = 1e-2 * np.abs(want) + 2.0 ** -8 * term_scale
    assert np.all(np.abs(g - want) <= bound), (g, want, bound)


@pytest.mark.parametrize("B,N,H,causal", [(1, 300, 2, True), (1, 200, 1, False)])
def test_fwd_train_outputs(B, N, H, causal):
    inp, _, lam, w = _case(B, N, H, 201 + N, causal)
    li = ref.lambda_init(LAYER)
    q, k, v = inp.q.to(DEV), inp.k.to(DEV), inp.v.to(DEV)
    lam_t = torch.tensor(lam, dtype=torch.float32, device=DEV)
    out, o_pre, stats = da.diffattn_fwd_train(q, k, v, lam_t, li, norm_weight=w.to(DEV), causal=causal)
    plain = da.diffattn_fwd(q, k, v, lam_t, li, norm_weight=w.to(DEV), causal=causal)
    assert torch.equal(out, plain)  # the training outputs do not change the forward's result
    for b in range(B):
        for h in range(H):
            d = 128
            O = ref.diff_attn_head(inp.q[b, :, h, :d], inp.k[b, :, h, :d], inp.q[b, :, h, d:],
                                   inp.k[b, :, h, d:], inp.v[b, :, h], float(lam[h]), causal)
            assert_bf16(o_pre[b, :, h], O)
            for mp in range(2):
                want = _log2_sum_exp(inp.q[b, :, h, mp * d:(mp + 1) * d],
                                     inp.k[b, :, h, mp * d:(mp + 1) * d], causal)
                got = stats[b, h, mp, :N].double().cpu().numpy()
                assert np.max(np.abs(got - want)) < 2e-3, (b, h, mp)


@pytest.mark.parametrize("B,N,H,causal,norm,scale", [
    (1, 128, 2, True, True, True),
    (2, 300, 2, True, True, True),
    (1, 257, 1, False, True, True),
    (1, 200, 2, True, False, False),
    (1, 1, 1, True, False, True),
    (1, 2, 1, True, True, True),
    (1, 640, 1, True, True, True),
])
def test_bwd_small(B, N, H, causal, norm, scale):
    """Every gradient against the oracle: ragged tails, one-row and multi-tile sequences,
    causal and not, with and without the norm and the fixed rescale. (With one key and the norm,
    dlambda is a pure cancellation -- O = (1 - lambda) V_0 and the norm's gradient is orthogonal
    to O -- so the one-row case runs without the norm.)"""
    inp, dy, lam, w = _case(B, N, H, 301 + N, causal)
    li = ref.lambda_init(LAYER)
    q, k, v = inp.q.to(DEV), inp.k.to(DEV), inp.v.to(DEV)
    lam_t = torch.tensor(lam, dtype=torch.float32, device=DEV)
    wd = w.to(DEV) if norm else None
    _, o_pre, stats = da.diffattn_fwd_train(q, k, v, lam_t, li, norm_weight=wd, causal=causal,
                                            norm=norm, scale=scale)
    g = da.diffattn_bwd(q, k, v, o_pre, stats, dy.to(DEV), lam_t, li, norm_weight=wd,
                        causal=causal, norm=norm, scale=scale)
    want = ref.diffattn_bwd(inp.q, inp.k, inp.v, lam, li, dy, norm_weight=w if norm else None,
                            norm=norm, apply_scale=scale, causal=causal)
    for name in ("dq", "dk", "dv"):
        assert_grad(g[name], want[name], name=name)
    _assert_dlam(g["dlam"], want["dlam"],
                 _dlam_term_scale(inp, dy, lam, li, w if norm else None, norm, scale, causal))
    if norm:
        assert_grad(g["dw"], want["dw"], rel_tol=1e-2, name="dw")
    else:
        assert torch.count_nonzero(g["dw"]) == 0


def test_bwd_lambda_zero_and_equal_maps():
    """Special cases with a known structure: lambda = 0 gives dK2 = dQ2 = 0."""
    B, N, H = 1, 256, 1
    inp, dy, _, w = _case(B, N, H, 401, True)
    li = ref.lambda_init(LAYER)
    q, k, v = inp.q.to(DEV), inp.k.to(DEV), inp.v.to(DEV)
    lam_t = torch.zeros(H, dtype=torch.float32, device=DEV)
    _, o_pre, stats = da.diffattn_fwd_train(q, k, v, lam_t, li, norm_weight=w.to(DEV))
    g = da.diffattn_bwd(q, k, v, o_pre, stats, dy.to(DEV), lam_t, li, norm_weight=w.to(DEV))
    assert torch.count_nonzero(g["dq"][..., 128:]) == 0
    assert torch.count_nonzero(g["dk"][..., 128:]) == 0
    want = ref.diffattn_bwd(inp.q, inp.k, inp.v, np.zeros(H), li, dy, norm_weight=w)
    for name in ("dq", "dk", "dv"):
        assert_grad(g[name], want[name], name=name)


@pytest.mark.parametrize("lens,causal,norm", [([300, 0, 129, 5, 640], True, True),
                                              ([128, 257], False, True),
                                              ([200, 2, 77], True, False)])
def test_train_varlen(lens, causal, norm):
    """Training over packed sequences: the forward equals the packed prefill (bit-equal) and every
    gradient matches the oracle's per-sequence backward; rows in no sequence stay zero."""
    H = 2
    total = sum(lens) + 3
    inp, dy, lam, w = _case(1, total, H, 401 + len(lens), causal)
    q, k, v, dyp = inp.q[0], inp.k[0], inp.v[0], dy[0]
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    li = ref.lambda_init(LAYER)
    lam_t = torch.tensor(lam, dtype=torch.float32, device=DEV)
    wd = w.to(DEV) if norm else None
    qd, kd, vd, cud = q.to(DEV), k.to(DEV), v.to(DEV), cu.to(DEV)
    out, o_pre, stats = da.diffattn_fwd_train_varlen(qd, kd, vd, cud, lam_t, li, norm_weight=wd,
                                                     causal=causal, norm=norm)
    plain = da.diffattn_fwd_varlen(qd, kd, vd, cud, lam_t, li, norm_weight=wd, causal=causal,
                                   norm=norm)
    n = sum(lens)
    assert torch.equal(out[:n], plain[:n])
    g = da.diffattn_bwd_varlen(qd, kd, vd, o_pre, stats, dyp.to(DEV), cud, lam_t, li,
                               norm_weight=wd, causal=causal, norm=norm)
    want = ref.diffattn_bwd_varlen(q, k, v, cu, lam, li, dyp, norm_weight=w if norm else None,
                                   norm=norm, causal=causal)
    for name in ("dq", "dk", "dv"):
        assert_grad(g[name][:n], want[name][:n], name=name)
        assert torch.count_nonzero(g[name][n:]) == 0
    terms = np.zeros(H)
    for s0, s1 in zip(cu[:-1].tolist(), cu[1:].tolist()):
        if s1 > s0:
            one = type(inp)(**{**inp.__dict__, "q": inp.q[:, s0:s1], "k": inp.k[:, s0:s1],
                               "v": inp.v[:, s0:s1]})
            terms += _dlam_term_scale(one, dy[:, s0:s1], lam, li, w if norm else None, norm,
                                      True, causal)
    _assert_dlam(g["dlam"], want["dlam"], terms)
    if norm:
        assert_grad(g["dw"], want["dw"], rel_tol=1e-2, name="dw")
    da.diffattn_device_status()


def test_train_varlen_bad_offsets_are_reported():
    """A sequence running past the packed length (and longer than max_seqlen) is skipped by the
    forward and every backward kernel, and reported."""
    inp, dy, lam, w = _case(1, 256, 1, 451, True)
    cu = torch.tensor([0, 128, 400], dtype=torch.int32, device=DEV)  # 400 > total
    lam_t = torch.tensor(lam[:1], dtype=torch.float32, device=DEV)
    q, k, v = inp.q[0].to(DEV), inp.k[0].to(DEV), inp.v[0].to(DEV)
    out, o_pre, stats = da.diffattn_fwd_train_varlen(q, k, v, cu, lam_t, 0.5, max_seqlen=256)
    with pytest.raises(da.DiffAttnError) as e:
        da.diffattn_device_status()
    assert e.value.status == -9
    da.diffattn_bwd_varlen(q, k, v, o_pre, stats, dy[0].to(DEV), cu, lam_t, 0.5, max_seqlen=256)
    with pytest.raises(da.DiffAttnError) as e:
        da.diffattn_device_status()
    assert e.value.status == -9
    da.diffattn_device_status()



@pytest.mark.parametrize("n_sets,per_set", [(1, 12), (4, 1)])
def test_lambda_bwd(n_sets, per_set):
    """The vectors' gradients from dlambda against the oracle's chain rule (one lambda per layer
    fed by every head's dlambda, and one per head)."""
    g = torch.Generator().manual_seed(461 + n_sets)
    vecs = [torch.randn((n_sets, 128), generator=g) * 0.1 for _ in range(4)]
    dl = torch.randn((n_sets * per_set,), generator=g)
    got = da.diffattn_lambda_bwd(*(t.to(DEV) for t in vecs), dl.to(DEV))
    want = ref.lambda_full_bwd(*vecs, dl.numpy().reshape(n_sets, per_set).sum(axis=1))
    for a, b in zip(got, want):
        np.testing.assert_allclose(a.double().cpu().numpy(), b, rtol=1e-5, atol=1e-6)
