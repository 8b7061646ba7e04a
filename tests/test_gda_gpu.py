"""GPU parity of grouped differential attention (several signal heads subtracting one shared
noise head's map): prefill and decode, called through the C ABI, against the float64 oracle on
identical seeded inputs; small cases on every output element, the full-size workloads on sampled
rows (prefill) and sampled sequences (decode), in the launch configurations bench.py times."""
import numpy as np
import pytest
import torch

import differential_attention_gb300 as da
from oracle import diffattn_ref as ref
from synth import make_gda_decode_inputs, make_gda_inputs, to_fp8_e4m3
from tests.gpu_util import assert_bf16, assert_fp32

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
    torch.cuda.empty_cache()


def _w(dv):
    return torch.linspace(0.5, 1.5, dv, dtype=torch.float32)


# (B, N, Hs, Hn, d, causal): group sizes 1 (ungrouped), 2, 3, 4 and 12, ragged tails, one token
GDA_CASES = [
    (1, 1, 2, 1, 128, True),
    (2, 77, 12, 3, 128, True),
    (2, 300, 4, 1, 128, True),
    (1, 645, 6, 2, 128, True),
    (2, 129, 3, 3, 128, False),
    (1, 384, 12, 4, 128, False),
    (2, 200, 4, 2, 64, True),
    (1, 333, 6, 3, 64, False),
]


@pytest.mark.parametrize("noise_pass", [True, False])
@pytest.mark.parametrize("B,N,Hs,Hn,d,causal", GDA_CASES)
def test_gda_fwd_small(B, N, Hs, Hn, d, causal, noise_pass):
    """Both forms against the oracle: the noise maps' statistics computed once per noise head
    (two launches, d = 128) or by every signal head (one launch)."""
    inp = make_gda_inputs(B, N, Hs, Hn, d, 2 * d, seed=101 + N + Hs)
    li = ref.lambda_init(inp.layer)
    w = _w(2 * d)
    got = da.diffattn_gda_fwd(inp.q.to(DEV), inp.k.to(DEV), inp.v.to(DEV), inp.lam.to(DEV), Hs,
                              li, norm_weight=w.to(DEV), causal=causal, noise_pass=noise_pass)
    want = ref.diffattn_gda_fwd(inp.q, inp.k, inp.v, inp.lam, li, Hs, norm_weight=w, causal=causal)
    assert_bf16(got, want)
    da.diffattn_device_status()


def test_gda_noise_pass_is_bit_equal_to_one_launch():
    """A noise map's row statistic is computed with the same arithmetic, in the same order,
    whether its own launch forms it once per noise head or every signal head forms it again: the
    two forms give bit-identical outputs (ragged tail, 3 signal heads per noise head)."""
    inp = make_gda_inputs(2, 700, 6, 2, 128, 256, seed=23, device=DEV)
    ws = torch.full((da.diffattn_gda_fwd_workspace_size(2, 700, 6, 2),), 255, dtype=torch.uint8,
                    device=DEV)  # stale contents must not matter
    a = da.diffattn_gda_fwd(inp.q, inp.k, inp.v, inp.lam, 6, 0.7, workspace=ws)
    b = da.diffattn_gda_fwd(inp.q, inp.k, inp.v, inp.lam, 6, 0.7, noise_pass=False)
    torch.cuda.synchronize()
    da.diffattn_device_status()
    assert torch.equal(a, b)


# (sequence lengths, Hs, Hn, d, causal): empty and one-token sequences, ragged tails, several tiles
GDA_VARLEN_CASES = [
    ([300, 1, 129, 0, 640], 6, 2, 128, True),
    ([128, 256], 4, 1, 128, False),
    ([5, 77, 200], 12, 3, 128, True),
    ([200, 0, 331], 6, 3, 64, True),
]


@pytest.mark.parametrize("noise_pass", [True, False])
@pytest.mark.parametrize("lens,Hs,Hn,d,causal", GDA_VARLEN_CASES)
def test_gda_fwd_varlen(lens, Hs, Hn, d, causal, noise_pass):
    """Packed grouped prefill against the oracle; rows in no sequence untouched; one sequence
    bit-equal to the batched grouped prefill of that sequence alone (same form)."""
    total = sum(lens) + 3
    inp = make_gda_inputs(1, total, Hs, Hn, d, 2 * d, seed=211 + len(lens) + Hs)
    q, k, v = inp.q[0], inp.k[0], inp.v[0]
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    li = ref.lambda_init(inp.layer)
    w = _w(2 * d)
    ws = None
    if noise_pass:  # stale workspace contents must not matter
        ws = torch.full((max(1, da.diffattn_gda_fwd_workspace_size(len(lens), max(lens), Hs, Hn,
                                                                   d, 2 * d)),),
                        255, dtype=torch.uint8, device=DEV)
    got = da.diffattn_gda_fwd_varlen(q.to(DEV), k.to(DEV), v.to(DEV), cu.to(DEV), inp.lam.to(DEV),
                                     Hs, li, norm_weight=w.to(DEV), causal=causal,
                                     noise_pass=noise_pass, workspace=ws)
    want = ref.diffattn_gda_fwd_varlen(q, k, v, cu, inp.lam, li, Hs, norm_weight=w, causal=causal)
    n_in = sum(lens)
    assert_bf16(got[:n_in], want[:n_in])
    assert torch.count_nonzero(got[n_in:]) == 0
    i = min(2, len(lens) - 1)
    s0, n = int(cu[i]), lens[i]
    one = da.diffattn_gda_fwd(q[None, s0:s0 + n].contiguous().to(DEV),
                              k[None, s0:s0 + n].contiguous().to(DEV),
                              v[None, s0:s0 + n].contiguous().to(DEV), inp.lam.to(DEV), Hs, li,
                              norm_weight=w.to(DEV), causal=causal, noise_pass=noise_pass)
    torch.cuda.synchronize()
    da.diffattn_device_status()
    assert torch.equal(got[s0:s0 + n], one[0])


def test_gda_fwd_varlen_bad_offsets_are_reported():
    """A sequence past the packed length is skipped by the kernels' own check (both launches of
    the two-launch form) and reported as DIFFATTN_ERR_INDEX."""
    inp = make_gda_inputs(1, 256, 4, 2, 128, 256, seed=227)
    cu = torch.tensor([0, 128, 400], dtype=torch.int32, device=DEV)  # 400 > total
    da.diffattn_gda_fwd_varlen(inp.q[0].to(DEV), inp.k[0].to(DEV), inp.v[0].to(DEV), cu,
                               inp.lam.to(DEV), 4, 0.5, max_seqlen=256)
    with pytest.raises(da.DiffAttnError) as e:
        da.diffattn_device_status()
    assert e.value.status == -9  # DIFFATTN_ERR_INDEX
    da.diffattn_device_status()


# (query lengths, key lengths, Hs, Hn, causal): a chunk far into a long prefix, decode-like one-row
# chunks, an empty sequence, whole prompts (Lq = Lk)
GDA_QK_CASES = [([300, 1, 100, 0, 640], [300, 700, 357, 90, 640], 6, 2, True),
                ([128, 77], [1000, 77], 12, 3, True),
                ([50, 200], [260, 200], 4, 1, False)]


def _gda_qk_inputs(lq, lk, Hs, Hn, seed):
    g = torch.Generator().manual_seed(seed)
    tq, tk = sum(lq), sum(lk)
    q = (torch.randn((tq, Hs + Hn, 128), generator=g) / 128 ** 0.5).to(torch.bfloat16)
    k = (torch.randn((tk, Hs + Hn, 128), generator=g) / 128 ** 0.5).to(torch.bfloat16)
    v = (torch.randn((tk, Hs, 256), generator=g) / 128 ** 0.5).to(torch.bfloat16)
    lam = 0.2 + 0.6 * torch.rand((Hs,), generator=g)
    cu_q = torch.tensor(np.concatenate([[0], np.cumsum(lq)]), dtype=torch.int32)
    cu_k = torch.tensor(np.concatenate([[0], np.cumsum(lk)]), dtype=torch.int32)
    return q, k, v, lam, cu_q, cu_k


def _pool(k, v, lk, ps, seed):
    """Each sequence's keys cut into pages of ps tokens, the pages shuffled in pools."""
    B = len(lk)
    mp = max(1, max((n + ps - 1) // ps for n in lk))
    g = torch.Generator().manual_seed(seed)
    table = torch.randperm(B * mp, generator=g).to(torch.int32).view(B, mp)
    kp = torch.zeros((B * mp, ps) + tuple(k.shape[1:]), dtype=k.dtype)
    vp = torch.zeros((B * mp, ps) + tuple(v.shape[1:]), dtype=v.dtype)
    off = 0
    for b, n in enumerate(lk):
        for j0 in range(0, n, ps):
            j1 = min(n, j0 + ps)
            kp[table[b, j0 // ps], :j1 - j0] = k[off + j0:off + j1]
            vp[table[b, j0 // ps], :j1 - j0] = v[off + j0:off + j1]
        off += n
    return kp, vp, table


@pytest.mark.parametrize("noise_pass", [True, False])
@pytest.mark.parametrize("lq,lk,Hs,Hn,causal", GDA_QK_CASES)
def test_gda_fwd_varlen_qk_and_paged(lq, lk, Hs, Hn, causal, noise_pass):
    """Grouped prefill with queries at the end of their keys against the oracle, keys packed with
    offsets of their own and in shuffled 128-token pages: the two bit-equal."""
    q, k, v, lam, cu_q, cu_k = _gda_qk_inputs(lq, lk, Hs, Hn, seed=53 + sum(lq))
    w = _w(256)
    li = 0.6
    got = da.diffattn_gda_fwd_varlen_qk(q.to(DEV), k.to(DEV), v.to(DEV), cu_q.to(DEV),
                                        cu_k.to(DEV), lam.to(DEV), Hs, li, norm_weight=w.to(DEV),
                                        causal=causal, noise_pass=noise_pass)
    want = ref.diffattn_gda_fwd_varlen_qk(q, k, v, cu_q, cu_k, lam, li, Hs, norm_weight=w,
                                          causal=causal)
    assert_bf16(got, want)
    kp, vp, table = _pool(k, v, lk, 128, seed=59 + sum(lk))
    paged = da.diffattn_gda_fwd_paged(q.to(DEV), kp.to(DEV), vp.to(DEV), cu_q.to(DEV),
                                      torch.tensor(lk, dtype=torch.int32, device=DEV),
                                      table.to(DEV), lam.to(DEV), Hs, li, norm_weight=w.to(DEV),
                                      causal=causal, noise_pass=noise_pass)
    torch.cuda.synchronize()
    da.diffattn_device_status()
    assert torch.equal(got, paged)


def test_gda_fwd_varlen_qk_chunk_equals_whole_prompt_rows():
    """The last 388 rows of two 900-token prompts (from row 512: the chunk's query tiles then
    fall on the whole prompt's tile boundaries) as a chunk over all 900 keys: bit-equal to those
    rows of the grouped prefill of the whole prompts (same tiles, same arithmetic)."""
    inp = make_gda_inputs(2, 900, 6, 2, 128, 256, seed=61, device=DEV)
    whole = da.diffattn_gda_fwd(inp.q, inp.k, inp.v, inp.lam, 6, 0.5)
    q = inp.q[:, 512:].reshape(-1, 8, 128).contiguous()
    k, v = inp.k.reshape(-1, 8, 128), inp.v.reshape(-1, 6, 256)
    cu_q = torch.tensor([0, 388, 776], dtype=torch.int32, device=DEV)
    cu_k = torch.tensor([0, 900, 1800], dtype=torch.int32, device=DEV)
    chunk = da.diffattn_gda_fwd_varlen_qk(q, k, v, cu_q, cu_k, inp.lam, 6, 0.5)
    torch.cuda.synchronize()
    da.diffattn_device_status()
    assert torch.equal(chunk, whole[:, 512:].reshape(-1, 6, 256))


def test_gda_fwd_no_norm_no_scale():
    inp = make_gda_inputs(1, 200, 6, 2, 128, 256, seed=7)
    got = da.diffattn_gda_fwd(inp.q.to(DEV), inp.k.to(DEV), inp.v.to(DEV), inp.lam.to(DEV), 6,
                              0.3, norm=False, scale=False)
    want = ref.diffattn_gda_fwd(inp.q, inp.k, inp.v, inp.lam, 0.3, 6, norm=False, apply_scale=False)
    assert_bf16(got, want, abs_tol=3e-2)


@pytest.mark.parametrize("dtype,cuda_cores", [("bf16", True), ("fp32", False)])
def test_gda_fwd_cuda_core_path(dtype, cuda_cores):
    inp = make_gda_inputs(2, 150, 4, 2, 64, 128, seed=9,
                          dtype=torch.float32 if dtype == "fp32" else torch.bfloat16)
    li = 0.45
    got = da.diffattn_gda_fwd(inp.q.to(DEV), inp.k.to(DEV), inp.v.to(DEV), inp.lam.to(DEV), 4, li,
                              cuda_cores=cuda_cores)
    want = ref.diffattn_gda_fwd(inp.q, inp.k, inp.v, inp.lam, li, 4)
    (assert_fp32 if dtype == "fp32" else assert_bf16)(got, want)


def test_gda_fwd_single_pass():
    inp = make_gda_inputs(1, 300, 4, 2, 128, 256, seed=13)
    lam = torch.full((4,), 0.5, dtype=torch.float32)
    got = da.diffattn_gda_fwd(inp.q.to(DEV), inp.k.to(DEV), inp.v.to(DEV), lam.to(DEV), 4, 0.6,
                              single_pass=True)
    want = ref.diffattn_gda_fwd(inp.q, inp.k, inp.v, lam, 0.6, 4)
    assert_bf16(got, want)


def test_gda_fwd_is_ungrouped_kernel_on_repeated_noise_heads():
    """The grouped instantiation does the same arithmetic as the ungrouped one on a [Q1|Q2]
    layout whose Q2/K2 repeat each noise head over its group: the outputs are bit-identical."""
    B, N, Hs, Hn, d = 2, 260, 6, 2, 128
    inp = make_gda_inputs(B, N, Hs, Hn, d, 2 * d, seed=17, device=DEV)
    rep = torch.arange(Hs, Hs + Hn, device=DEV).repeat_interleave(Hs // Hn)
    q1 = torch.cat([inp.q[:, :, :Hs], inp.q[:, :, rep]], dim=-1).contiguous()
    k1 = torch.cat([inp.k[:, :, :Hs], inp.k[:, :, rep]], dim=-1).contiguous()
    a = da.diffattn_gda_fwd(inp.q, inp.k, inp.v, inp.lam, Hs, 0.7, noise_pass=False)
    b = da.diffattn_fwd(q1, k1, inp.v, inp.lam, 0.7)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


# fp8 scores: (B, N, Hs, Hn, causal): one token, group sizes 1 to 4, ragged tails, full attention
GDA_FP8_CASES = [(1, 1, 2, 1, True), (2, 300, 12, 3, True), (1, 645, 6, 2, True),
                 (2, 129, 4, 4, False)]


@pytest.mark.parametrize("B,N,Hs,Hn,causal", GDA_FP8_CASES)
def test_gda_fwd_fp8(B, N, Hs, Hn, causal):
    """fp8 e4m3 q and k with per-tensor descale factors: the oracle runs the grouped prefill on
    exactly the dequantised fp8 values, so the bar is the bf16 prefill's."""
    inp = make_gda_inputs(B, N, Hs, Hn, 128, 256, seed=401 + N + Hs)
    q8, qs = to_fp8_e4m3(inp.q)
    k8, ks = to_fp8_e4m3(inp.k)
    li = ref.lambda_init(inp.layer)
    w = _w(256)
    got = da.diffattn_gda_fwd_fp8(q8.to(DEV), k8.to(DEV), inp.v.to(DEV), inp.lam.to(DEV), Hs, qs,
                                  ks, li, norm_weight=w.to(DEV), causal=causal)
    want = ref.diffattn_gda_fwd(q8.float() * qs, k8.float() * ks, inp.v, inp.lam, li, Hs,
                                norm_weight=w, causal=causal)
    assert_bf16(got, want)
    da.diffattn_device_status()


def test_gda_fwd_fp8_is_ungrouped_fp8_on_repeated_noise_heads():
    """The grouped fp8 instantiation does the ungrouped fp8 prefill's arithmetic on a [Q1|Q2]
    layout whose Q2/K2 repeat each noise head over its group: the outputs are bit-identical."""
    B, N, Hs, Hn = 2, 260, 6, 2
    inp = make_gda_inputs(B, N, Hs, Hn, 128, 256, seed=19, device=DEV)
    q8, qs = to_fp8_e4m3(inp.q)
    k8, ks = to_fp8_e4m3(inp.k)
    rep = torch.arange(Hs, Hs + Hn, device=DEV).repeat_interleave(Hs // Hn)

    def halves(t8):  # [Q1 of head h | Q2 of its noise head] per signal head, through byte views
        u = t8.view(torch.uint8)
        return torch.cat([u[:, :, :Hs], u[:, :, rep]], dim=-1).contiguous().view(torch.float8_e4m3fn)

    a = da.diffattn_gda_fwd_fp8(q8, k8, inp.v, inp.lam, Hs, qs, ks, 0.7)
    b = da.diffattn_fwd_fp8(halves(q8), halves(k8), inp.v, inp.lam, qs, ks, 0.7)
    torch.cuda.synchronize()
    da.diffattn_device_status()
    assert torch.equal(a, b)


def test_gda_fwd_guard_band():
    """Nothing is written outside the output tensor."""
    inp = make_gda_inputs(1, 150, 4, 2, 128, 256, seed=19)
    n = 150 * 4 * 256
    buf = torch.full((n + 2 * 4096,), 7.0, dtype=torch.bfloat16, device=DEV)
    out = buf[4096:4096 + n].view(1, 150, 4, 256)
    da.diffattn_gda_fwd(inp.q.to(DEV), inp.k.to(DEV), inp.v.to(DEV), inp.lam.to(DEV), 4, 0.5,
                        out=out)
    torch.cuda.synchronize()
    assert torch.all(buf[:4096] == 7.0) and torch.all(buf[4096 + n:] == 7.0)


# (B, L, Hs, Hn, ragged)
GDA_DECODE_CASES = [(2, 1, 2, 2, False), (3, 700, 4, 1, True), (2, 5000, 12, 3, False),
                    (4, 3001, 6, 2, True)]


@pytest.mark.parametrize("B,L,Hs,Hn,ragged", GDA_DECODE_CASES)
def test_gda_decode_small(B, L, Hs, Hn, ragged):
    inp = make_gda_decode_inputs(B, L, Hs, Hn, 128, 256, seed=23 + L, ragged=ragged)
    li = ref.lambda_init(inp.layer)
    w = torch.linspace(0.8, 1.2, 256, dtype=torch.float32)
    got = da.diffattn_gda_decode(inp.q.to(DEV), inp.k_cache.to(DEV), inp.v_cache.to(DEV),
                                 inp.lam.to(DEV), Hs, li, seqlens=inp.seqlens.to(DEV),
                                 norm_weight=w.to(DEV))
    want = ref.diffattn_gda_decode(inp.q, inp.k_cache, inp.v_cache, inp.seqlens, inp.lam, li, Hs,
                                   norm_weight=w)
    assert_bf16(got, want)
    da.diffattn_device_status()


def _paged(k_cache, v_cache, ps, seed):
    """The caches cut into pages of ps tokens (the last page padded), the pages moved to a seeded
    random order in the pools, and the block table that finds them there."""
    B, L = k_cache.shape[:2]
    mp = (L + ps - 1) // ps
    pad = mp * ps - L
    if pad:
        k_cache = torch.cat([k_cache, torch.zeros_like(k_cache[:, :pad])], 1)
        v_cache = torch.cat([v_cache, torch.zeros_like(v_cache[:, :pad])], 1)
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    table = torch.randperm(B * mp, generator=g).to(torch.int32).view(B, mp)
    order = torch.argsort(table.flatten())
    k_pool = k_cache.reshape(B * mp, ps, *k_cache.shape[2:])[order].contiguous()
    v_pool = v_cache.reshape(B * mp, ps, *v_cache.shape[2:])[order].contiguous()
    return k_pool, v_pool, table


# (B, L, Hs, Hn, page size, ragged): pages of 16 to 256 tokens, group sizes 1 to 4, a last page
# partly used, one-key sequences
GDA_DECODE_PAGED_CASES = [(2, 300, 4, 1, 16, True), (3, 1000, 12, 3, 64, True),
                          (2, 777, 6, 2, 256, False), (4, 129, 3, 3, 128, True)]


@pytest.mark.parametrize("B,L,Hs,Hn,ps,ragged", GDA_DECODE_PAGED_CASES)
def test_gda_decode_paged(B, L, Hs, Hn, ps, ragged):
    """Grouped decode over shuffled pages: against the oracle's paged composition, and bit-equal
    to the contiguous grouped decode on the same keys."""
    inp = make_gda_decode_inputs(B, L, Hs, Hn, 128, 256, seed=41 + L, ragged=ragged)
    li = ref.lambda_init(inp.layer)
    w = torch.linspace(0.8, 1.2, 256, dtype=torch.float32)
    k_pool, v_pool, table = _paged(inp.k_cache, inp.v_cache, ps, seed=43 + ps)
    got = da.diffattn_gda_decode_paged(inp.q.to(DEV), k_pool.to(DEV), v_pool.to(DEV),
                                       table.to(DEV), inp.seqlens.to(DEV), inp.lam.to(DEV), Hs,
                                       li, norm_weight=w.to(DEV))
    want = ref.diffattn_gda_decode_paged(inp.q, k_pool, v_pool, table, inp.seqlens, inp.lam, li,
                                         Hs, norm_weight=w)
    assert_bf16(got, want)
    contiguous = da.diffattn_gda_decode(inp.q.to(DEV), inp.k_cache.to(DEV), inp.v_cache.to(DEV),
                                        inp.lam.to(DEV), Hs, li, seqlens=inp.seqlens.to(DEV),
                                        norm_weight=w.to(DEV))
    torch.cuda.synchronize()
    da.diffattn_device_status()
    assert torch.equal(got, contiguous)


def test_gda_decode_paged_bad_page_is_reported():
    """A used block-table entry outside the pool reads page 0 instead (nothing faults) and the host
    sees DIFFATTN_ERR_INDEX; entries past a sequence's keys are not read."""
    inp = make_gda_decode_inputs(2, 256, 4, 2, 128, 256, seed=47)
    k_pool, v_pool, table = _paged(inp.k_cache, inp.v_cache, 64, seed=48)
    seqlens = torch.tensor([256, 60], dtype=torch.int32)
    ok_table = table.clone()
    ok_table[1, 1:] = 10_000  # past sequence 1's 60 keys: never read
    da.diffattn_gda_decode_paged(inp.q.to(DEV), k_pool.to(DEV), v_pool.to(DEV), ok_table.to(DEV),
                                 seqlens.to(DEV), inp.lam.to(DEV), 4, 0.5)
    torch.cuda.synchronize()
    da.diffattn_device_status()  # nothing flagged
    bad = table.clone()
    bad[0, 2] = 10_000  # keys 128..191 of sequence 0
    da.diffattn_gda_decode_paged(inp.q.to(DEV), k_pool.to(DEV), v_pool.to(DEV), bad.to(DEV),
                                 seqlens.to(DEV), inp.lam.to(DEV), 4, 0.5)
    with pytest.raises(da.DiffAttnError) as e:
        da.diffattn_device_status()
    assert e.value.status == -9  # DIFFATTN_ERR_INDEX
    da.diffattn_device_status()


def test_gda_decode_matches_prefill_last_row():
    inp = make_gda_inputs(1, 384, 6, 2, 128, 256, seed=29, device=DEV)
    pre = da.diffattn_gda_fwd(inp.q, inp.k, inp.v, inp.lam, 6, 0.5)
    dec = da.diffattn_gda_decode(inp.q[:, -1].contiguous(), inp.k, inp.v, inp.lam, 6, 0.5)
    got = dec.float().cpu().numpy()
    want = pre[:, -1].float().cpu().numpy()
    assert np.max(np.abs(got - want)) < 4e-2
    assert np.linalg.norm(got - want) / np.linalg.norm(want) < 2e-2


def _rows(N, n_first, n_rand, seed):
    rng = np.random.default_rng(seed)
    rand = rng.choice(np.arange(n_first, N - 1), size=n_rand, replace=False)
    return np.unique(np.concatenate([np.arange(n_first), [N - 1], rand]))


def test_gda_prefill_3b_full():
    """B4 N4096, 12 signal heads over 3 noise heads, causal, RMSNorm + scale: sampled rows of
    every signal head."""
    B, N, Hs, Hn = 4, 4096, 12, 3
    inp = make_gda_inputs(B, N, Hs, Hn, 128, 256, seed=5000, device=DEV)
    li = ref.lambda_init(inp.layer)
    out = da.diffattn_gda_fwd(inp.q, inp.k, inp.v, inp.lam, Hs, li)
    da.diffattn_device_status()
    rows = _rows(N, 64, 128, 5000)
    lam = inp.lam.cpu().numpy()
    got, want = [], []
    for b in range(B):
        for h in range(Hs):
            g = Hs + ref.gda_noise_head(h, Hs, Hn)
            sel = [h, g]
            q = inp.q[b:b + 1, :, sel].cpu()
            k = inp.k[b:b + 1, :, sel].cpu()
            v = inp.v[b:b + 1, :, h:h + 1].cpu()
            want.append(ref.diffattn_gda_fwd(q, k, v, lam[h:h + 1], li, 1, rows=rows)[0, :, 0])
            got.append(out[b, torch.as_tensor(rows, device=DEV), h].float().cpu().numpy())
    assert_bf16(np.stack(got), np.stack(want))


def test_gda_decode_32k_full():
    """B64, cache 32768, 12 signal heads over 3 noise heads: every head of 4 sampled sequences."""
    inp = make_gda_decode_inputs(64, 32768, 12, 3, 128, 256, seed=5100, device=DEV)
    li = ref.lambda_init(inp.layer)
    out = da.diffattn_gda_decode(inp.q, inp.k_cache, inp.v_cache, inp.lam, 12, li)
    da.diffattn_device_status()
    sample = [0, 21, 50, 63]
    want = ref.diffattn_gda_decode(inp.q[sample].cpu(), inp.k_cache[sample].cpu(),
                                   inp.v_cache[sample].cpu(), inp.seqlens[sample].cpu(),
                                   inp.lam.cpu(), li, 12)
    assert_bf16(out[sample], want)
    del inp
    torch.cuda.empty_cache()


def test_gda_decode_paged_32k_full():
    """The same grouped decode over shuffled 64-token pages (the bench's paged layout): bit-equal
    to the contiguous call for every sequence and head, and 2 sampled sequences against the
    oracle's paged composition."""
    inp = make_gda_decode_inputs(64, 32768, 12, 3, 128, 256, seed=5300, device=DEV, ragged=True)
    li = ref.lambda_init(inp.layer)
    flat = da.diffattn_gda_decode(inp.q, inp.k_cache, inp.v_cache, inp.lam, 12, li,
                                  seqlens=inp.seqlens)
    k_pool, v_pool, table = _paged(inp.k_cache, inp.v_cache, 64, seed=5301)
    del inp.k_cache, inp.v_cache
    torch.cuda.empty_cache()
    table = table.to(DEV)
    paged = da.diffattn_gda_decode_paged(inp.q, k_pool, v_pool, table, inp.seqlens, inp.lam, 12, li)
    torch.cuda.synchronize()
    da.diffattn_device_status()
    assert torch.equal(flat, paged)
    sample = [5, 44]
    pages = sorted({int(x) for s_ in sample for x in table[s_].cpu().tolist()})
    remap = {pg: i for i, pg in enumerate(pages)}
    sub_table = torch.tensor([[remap[int(x)] for x in table[s_].cpu().tolist()] for s_ in sample],
                             dtype=torch.int32)
    idx = torch.tensor(pages, device=DEV)
    want = ref.diffattn_gda_decode_paged(inp.q[sample].cpu(), k_pool[idx].cpu(), v_pool[idx].cpu(),
                                         sub_table, inp.seqlens[sample].cpu(), inp.lam.cpu(), li, 12)
    assert_bf16(paged[sample], want)
    del k_pool, v_pool
    torch.cuda.empty_cache()
