"""GPU parity of grouped training (the forward saving its statistics, then the backward) against
the float64 oracle, through the C ABI. Signal head h's gradients are those of the ungrouped
operator with map 2 in noise head n_signal + h / G; a noise head's dQ2 and dK2 collect its
group's contributions."""
import numpy as np
import pytest
import torch

import differential_attention_gb300 as da
from oracle import diffattn_ref as ref
from synth import make_dout, make_gda_inputs
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
    da.diffattn_device_status()


def _w():
    return torch.linspace(0.8, 1.2, 256, dtype=torch.float32)


def _log2_sum_exp(Q, K, causal):
    S = ref.scores(ref._f64(Q), ref._f64(K), np.arange(Q.shape[0]), causal)
    m = np.max(S, axis=-1, keepdims=True)
    return (m[:, 0] + np.log(np.sum(np.exp(S - m), axis=-1))) / np.log(2.0)


def _dlam_term_scale(inp, dy, li, w, norm, scale, causal):
    """Per signal head, sum over rows of |dO_i| |O2_i| (oracle pieces): the size of the terms
    whose sum is -dlambda, which can cancel far below them."""
    B, N, heads, d = inp.q.shape
    Hs = inp.n_signal
    lam = inp.lam.cpu().numpy()
    out = np.zeros(Hs)
    s = (1.0 - li) if scale else 1.0
    for b in range(B):
        for h in range(Hs):
            g = Hs + ref.gda_noise_head(h, Hs, heads - Hs)
            O = ref.diff_attn_head(inp.q[b, :, h], inp.k[b, :, h], inp.q[b, :, g], inp.k[b, :, g],
                                   inp.v[b, :, h], float(lam[h]), causal)
            dys = ref._f64(dy[b, :, h]) * s
            dO = ref.subln_bwd(O, w, 1e-5, dys)[0] if norm else dys
            O2 = ref.attention_head(inp.q[b, :, g], inp.k[b, :, g], inp.v[b, :, h], causal)
            out[h] += float(np.sum(np.linalg.norm(dO, axis=-1) * np.linalg.norm(O2, axis=-1)))
    return out


@pytest.mark.parametrize("noise_pass", [True, False])
def test_gda_fwd_train_outputs(noise_pass):
    """The training forward's output is the grouped prefill's (bit-equal, same launch form); o_pre
    and each map's row statistic match the oracle (map 2's from the noise head)."""
    B, N, Hs, Hn, causal = 1, 300, 6, 2, True
    inp = make_gda_inputs(B, N, Hs, Hn, 128, 256, seed=71)
    li = ref.lambda_init(inp.layer)
    q, k, v, lam = inp.q.to(DEV), inp.k.to(DEV), inp.v.to(DEV), inp.lam.to(DEV)
    out, o_pre, stats = da.diffattn_gda_fwd_train(q, k, v, lam, Hs, li, norm_weight=_w().to(DEV),
                                                  noise_pass=noise_pass)
    plain = da.diffattn_gda_fwd(q, k, v, lam, Hs, li, norm_weight=_w().to(DEV),
                                noise_pass=noise_pass)
    torch.cuda.synchronize()
    da.diffattn_device_status()
    assert torch.equal(out, plain)
    lam_np = inp.lam.numpy()
    for h in range(Hs):
        g = Hs + ref.gda_noise_head(h, Hs, Hn)
        O = ref.diff_attn_head(inp.q[0, :, h], inp.k[0, :, h], inp.q[0, :, g], inp.k[0, :, g],
                               inp.v[0, :, h], float(lam_np[h]), causal)
        assert_bf16(o_pre[0, :, h], O)
        for mp, hh in ((0, h), (1, g)):
            want = _log2_sum_exp(inp.q[0, :, hh], inp.k[0, :, hh], causal)
            got = stats[0, h, mp, :N].double().cpu().numpy()
            assert np.max(np.abs(got - want)) < 2e-3, (h, mp)


# (B, N, Hs, Hn, causal, norm, scale): group sizes 1 to 4, ragged tails, one-row sequences
GDA_BWD_CASES = [(1, 300, 4, 1, True, True, True), (2, 200, 6, 2, True, True, True),
                 (1, 257, 3, 3, False, True, True), (1, 130, 12, 3, True, False, False),
                 (1, 1, 2, 1, True, False, True), (1, 640, 4, 2, True, True, True)]


@pytest.mark.parametrize("B,N,Hs,Hn,causal,norm,scale", GDA_BWD_CASES)
def test_gda_bwd(B, N, Hs, Hn, causal, norm, scale):
    """Every gradient against the oracle's grouped backward."""
    inp = make_gda_inputs(B, N, Hs, Hn, 128, 256, seed=73 + N + Hs)
    dy = make_dout(B, N, Hs, 256, seed=79 + N)
    li = ref.lambda_init(inp.layer)
    w = _w()
    q, k, v, lam = inp.q.to(DEV), inp.k.to(DEV), inp.v.to(DEV), inp.lam.to(DEV)
    wd = w.to(DEV) if norm else None
    _, o_pre, stats = da.diffattn_gda_fwd_train(q, k, v, lam, Hs, li, norm_weight=wd,
                                                causal=causal, norm=norm, scale=scale)
    g = da.diffattn_gda_bwd(q, k, v, o_pre, stats, dy.to(DEV), lam, Hs, li, norm_weight=wd,
                            causal=causal, norm=norm, scale=scale)
    torch.cuda.synchronize()
    da.diffattn_device_status()
    want = ref.diffattn_gda_bwd(inp.q, inp.k, inp.v, inp.lam, li, Hs, dy,
                                norm_weight=w if norm else None, norm=norm, apply_scale=scale,
                                causal=causal)
    for name in ("dq", "dk", "dv"):
        assert_grad(g[name], want[name], name=name)
    term = _dlam_term_scale(inp, dy, li, w if norm else None, norm, scale, causal)
    gl = g["dlam"].double().cpu().numpy()
    assert np.all(np.abs(gl - want["dlam"]) <= 1e-2 * np.abs(want["dlam"]) + 2.0 ** -8 * term)
    if norm:
        assert_grad(g["dw"], want["dw"], rel_tol=1e-2, name="dw")
    else:
        assert torch.count_nonzero(g["dw"]) == 0


def test_gda_bwd_is_ungrouped_with_one_signal_head_per_noise_head():
    """With n_noise = n_signal every noise head has one contribution: the grouped backward does
    the ungrouped one's arithmetic on the [Q1 | Q2] layout (the noise dK's single fp32 addition
    onto zero is exact). dK, dV, dlambda and the norm weight's gradient are reduced in a fixed
    order and are bit-equal; dQ's fp32 accumulator takes one reduction per key tile in whatever
    order the CTAs finish, so over several key tiles it agrees to the last bf16 bit only."""
    B, H = 1, 3
    for N in (128, 384):
        inp = make_gda_inputs(B, N, H, H, 128, 256, seed=83 + N)
        dy = make_dout(B, N, H, 256, seed=89).to(DEV)
        q, k, v, lam = inp.q.to(DEV), inp.k.to(DEV), inp.v.to(DEV), inp.lam.to(DEV)
        w = _w().to(DEV)
        _, o_pre, stats = da.diffattn_gda_fwd_train(q, k, v, lam, H, 0.5, norm_weight=w)
        g = da.diffattn_gda_bwd(q, k, v, o_pre, stats, dy, lam, H, 0.5, norm_weight=w)
        qu = torch.cat([q[:, :, :H], q[:, :, H:]], dim=3).contiguous()
        ku = torch.cat([k[:, :, :H], k[:, :, H:]], dim=3).contiguous()
        _, o_pre_u, stats_u = da.diffattn_fwd_train(qu, ku, v, lam, 0.5, norm_weight=w)
        u = da.diffattn_bwd(qu, ku, v, o_pre_u, stats_u, dy, lam, 0.5, norm_weight=w)
        torch.cuda.synchronize()
        da.diffattn_device_status()
        assert torch.equal(o_pre, o_pre_u) and torch.equal(stats, stats_u)
        dk_u = torch.cat([u["dk"][..., :128], u["dk"][..., 128:]], dim=2)
        assert torch.equal(g["dk"], dk_u), N
        for name in ("dv", "dlam", "dw"):
            assert torch.equal(g[name], u[name]), (name, N)
        dq_u = torch.cat([u["dq"][..., :128], u["dq"][..., 128:]], dim=2).float()
        dq = g["dq"].float()
        if N <= 128:
            assert torch.equal(dq, dq_u)
        else:
            ulp = 2.0 ** -7 * dq_u.abs() + 1e-3 * dq_u.abs().max()
            assert bool(((dq - dq_u).abs() <= ulp).all())


# packed sequences: (lengths, n_signal, n_noise, causal, norm); empty and one-token sequences,
# ragged and multi-tile ones, and three rows after the last sequence that belong to none
GDA_VARLEN_CASES = [([300, 0, 129, 5, 640], 4, 2, True, True), ([128, 257], 3, 3, False, True),
                    ([200, 1, 77], 6, 2, True, False)]


@pytest.mark.parametrize("lens,Hs,Hn,causal,norm", GDA_VARLEN_CASES)
def test_gda_train_varlen(lens, Hs, Hn, causal, norm):
    """Grouped training over packed sequences: the forward equals the packed grouped prefill
    (bit-equal) and every gradient matches the oracle's per-sequence grouped backward; rows in no
    sequence stay zero."""
    n = sum(lens)
    total = n + 3
    inp = make_gda_inputs(1, total, Hs, Hn, 128, 256, seed=91 + len(lens) + Hs)
    dy = make_dout(1, total, Hs, 256, seed=97 + len(lens))
    q, k, v, dyp = inp.q[0], inp.k[0], inp.v[0], dy[0]
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    li = ref.lambda_init(inp.layer)
    w = _w()
    wd = w.to(DEV) if norm else None
    qd, kd, vd, cud, lam = q.to(DEV), k.to(DEV), v.to(DEV), cu.to(DEV), inp.lam.to(DEV)
    out, o_pre, stats = da.diffattn_gda_fwd_train_varlen(qd, kd, vd, cud, lam, Hs, li,
                                                         norm_weight=wd, causal=causal, norm=norm)
    plain = da.diffattn_gda_fwd_varlen(qd, kd, vd, cud, lam, Hs, li, norm_weight=wd,
                                       causal=causal, norm=norm)
    assert torch.equal(out[:n], plain[:n])
    g = da.diffattn_gda_bwd_varlen(qd, kd, vd, o_pre, stats, dyp.to(DEV), cud, lam, Hs, li,
                                   norm_weight=wd, causal=causal, norm=norm)
    torch.cuda.synchronize()
    da.diffattn_device_status()
    want = ref.diffattn_gda_bwd_varlen(q, k, v, cu, inp.lam, li, Hs, dyp,
                                       norm_weight=w if norm else None, norm=norm, causal=causal)
    for name in ("dq", "dk", "dv"):
        assert_grad(g[name][:n], want[name][:n], name=name)
        assert torch.count_nonzero(g[name][n:]) == 0
    terms = np.zeros(Hs)
    for s0, s1 in zip(cu[:-1].tolist(), cu[1:].tolist()):
        if s1 > s0:
            one = type(inp)(**{**inp.__dict__, "q": inp.q[:, s0:s1], "k": inp.k[:, s0:s1],
                               "v": inp.v[:, s0:s1]})
            terms += _dlam_term_scale(one, dy[:, s0:s1], li, w if norm else None, norm, True,
                                      causal)
    gl = g["dlam"].double().cpu().numpy()
    assert np.all(np.abs(gl - want["dlam"]) <= 1e-2 * np.abs(want["dlam"]) + 2.0 ** -8 * terms)
    if norm:
        assert_grad(g["dw"], want["dw"], rel_tol=1e-2, name="dw")


def test_gda_bwd_varlen_one_sequence_is_the_batched_backward():
    """One packed sequence filling the batch: the signal heads' dK, dV, dlambda and the norm
    weight's gradient are bit-equal to the batched grouped backward's (fixed-order sums); dQ and
    the noise heads' dK agree to the last bf16 bit (their fp32 sums, over key tiles and over the
    group's signal heads, land in any order)."""
    N, Hs, Hn = 384, 6, 2
    inp = make_gda_inputs(1, N, Hs, Hn, 128, 256, seed=103, device=DEV)
    dy = make_dout(1, N, Hs, 256, seed=107).to(DEV)
    w = _w().to(DEV)
    cu = torch.tensor([0, N], dtype=torch.int32, device=DEV)
    _, o_pre, stats = da.diffattn_gda_fwd_train(inp.q, inp.k, inp.v, inp.lam, Hs, 0.4, norm_weight=w)
    g = da.diffattn_gda_bwd(inp.q, inp.k, inp.v, o_pre, stats, dy, inp.lam, Hs, 0.4, norm_weight=w)
    _, o_pre_p, stats_p = da.diffattn_gda_fwd_train_varlen(inp.q[0], inp.k[0], inp.v[0], cu,
                                                           inp.lam, Hs, 0.4, norm_weight=w)
    p = da.diffattn_gda_bwd_varlen(inp.q[0], inp.k[0], inp.v[0], o_pre_p, stats_p, dy[0], cu,
                                   inp.lam, Hs, 0.4, norm_weight=w)
    torch.cuda.synchronize()
    da.diffattn_device_status()
    assert torch.equal(o_pre[0], o_pre_p) and torch.equal(stats, stats_p)
    assert torch.equal(g["dk"][0, :, :Hs], p["dk"][:, :Hs]) and torch.equal(g["dv"][0], p["dv"])
    assert torch.equal(g["dlam"], p["dlam"]) and torch.equal(g["dw"], p["dw"])
    for a, b in ((g["dq"][0], p["dq"]), (g["dk"][0, :, Hs:], p["dk"][:, Hs:])):
        a, b = a.float(), b.float()
        assert bool(((a - b).abs() <= 2.0 ** -7 * b.abs() + 1e-3 * b.abs().max()).all())


def test_gda_train_varlen_bad_offsets_are_reported():
    """A sequence running past the packed length is skipped by the grouped training forward and
    every backward kernel, and reported."""
    inp = make_gda_inputs(1, 256, 4, 2, 128, 256, seed=109, device=DEV)
    dy = make_dout(1, 256, 4, 256, seed=113).to(DEV)
    cu = torch.tensor([0, 128, 400], dtype=torch.int32, device=DEV)  # 400 > total
    q, k, v = inp.q[0], inp.k[0], inp.v[0]
    out, o_pre, stats = da.diffattn_gda_fwd_train_varlen(q, k, v, cu, inp.lam, 4, 0.5,
                                                         max_seqlen=256)
    with pytest.raises(da.DiffAttnError) as e:
        da.diffattn_device_status()
    assert e.value.status == -9
    da.diffattn_gda_bwd_varlen(q, k, v, o_pre, stats, dy[0], cu, inp.lam, 4, 0.5, max_seqlen=256)
    with pytest.raises(da.DiffAttnError) as e:
        da.diffattn_device_status()
    assert e.value.status == -9
    da.diffattn_device_status()
