"""C-ABI checks that need no GPU: the library loads, exports every symbol that include/diffattn.h
declares, and rejects bad arguments with the documented status codes before touching a device.
Pointers passed here are never dereferenced (validation is pure arithmetic on the host)."""
import ctypes
import math
import os
import re

import pytest

import differential_attention_gb300 as da
from oracle import diffattn_ref as ref

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "diffattn.h")


@pytest.fixture(scope="module")
def L():
    da.build()
    return da.lib()


def declared_symbols():
    text = open(HEADER).read()
    return re.findall(r"DIFFATTN_API\s+[\w\s\*]+?\b(diffattn_\w+)\s*\(", text)


def test_header_declares_the_entry_points():
    names = set(declared_symbols())
    for n in ("diffattn_lambda", "diffattn_fwd", "diffattn_decode", "diffattn_v2_fwd",
              "diffattn_decode_workspace_size", "diffattn_last_error_string"):
        assert n in names


def test_every_declared_symbol_is_exported(L):
    for name in declared_symbols():
        assert hasattr(L, name), name


def test_only_declared_symbols_are_exported():
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", da.LIB_PATH], capture_output=True, text=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    ours = {s for s in exported if s.startswith("diffattn_")}
    assert ours == set(declared_symbols())


def test_version(L):
    assert da.diffattn_version() >= 10000


def test_lambda_init_host_function_matches_oracle(L):
    for layer in (1, 2, 4, 8, 12, 16, 24, 28, 100):
        assert da.diffattn_lambda_init(layer) == pytest.approx(ref.lambda_init(layer), rel=1e-6, abs=1e-7)
    assert math.isnan(da.diffattn_lambda_init(0))


FAKE = ctypes.c_void_p(0x10000)     # 16-byte aligned, never dereferenced
ODD = ctypes.c_void_p(0x10008)      # 8-byte aligned only


def _fwd(L, q=FAKE, k=FAKE, v=FAKE, out=FAKE, lam=FAKE, B=1, N=16, H=1, d=128, dv=256, flags=7,
         dtype=0, eps=1e-5):
    return L.diffattn_fwd(q, k, v, out, lam, 0.5, None, eps, B, N, H, d, dv, flags, dtype, None)


def test_fwd_validation(L):
    assert _fwd(L, q=None) == -1
    assert _fwd(L, flags=64) == -1
    assert _fwd(L, eps=0.0) == -1
    assert _fwd(L, dtype=7) == -3
    assert _fwd(L, N=0) == -2
    assert _fwd(L, d=96, dv=192) == -2
    assert _fwd(L, d=128, dv=128) == -2
    assert _fwd(L, q=ODD) == -4
    assert "aligned" in L.diffattn_last_error_string().decode()


def test_decode_validation(L):
    n = ctypes.c_size_t(0)
    assert L.diffattn_decode_workspace_size(64, 32768, 12, 128, 256, ctypes.byref(n)) == 0
    need = n.value
    assert need > 0 and need % 16 == 0
    assert L.diffattn_decode_workspace_size(1, 0, 1, 128, 256, ctypes.byref(n)) == -2
    assert L.diffattn_decode_workspace_size(1, 10, 1, 64, 128, ctypes.byref(n)) == -2

    def dec(ws=FAKE, ws_bytes=need, d=128, dv=256, dtype=0, q=FAKE, flags=6):
        return L.diffattn_decode(q, FAKE, FAKE, None, FAKE, FAKE, 0.5, None, 1e-5, 64, 32768, 12,
                                 d, dv, flags, dtype, ws, ws_bytes, None)

    assert dec(q=None) == -1
    assert dec(flags=16) == -1
    assert dec(dtype=1) == -3
    assert dec(d=64, dv=128) == -2
    assert dec(ws=None) == -8
    assert dec(ws_bytes=need - 1) == -8
    assert dec(ws=ctypes.c_void_p(0x10010)) == -8  # not 256-byte aligned


def test_decode_split_counts(L):
    """The split arithmetic of diffattn_decode and of its no-allocation variant (host only).
    The no-allocation call keeps diffattn_decode's slices whenever B x H x splits partial
    records (2064 bytes each) fit in its 16 MiB scratch, and otherwise cuts the cache into
    fewer, longer slices of whole 32-key CTA rounds that still cover every key."""
    max_units = (16 << 20) // 2064
    assert max_units == 8128
    # few (sequence, head) pairs: both calls split alike
    assert da.diffattn_decode_split_count(3, 3001, 2) == da.diffattn_decode_split_count(3, 3001, 2, True)
    # 768 pairs: 10 splits fit; the 3000-key cache and the 32K-token decode both need lowering
    for lmax in (3000, 32768):
        ws_s, _ = da.diffattn_decode_split_count(64, lmax, 12)
        na_s, _ = da.diffattn_decode_split_count(64, lmax, 12, True)
        assert ws_s > 10 and na_s <= 10 and na_s < ws_s, (lmax, ws_s, na_s)
    for B, lmax, H in [(1, 1, 1), (1, 31, 1), (2, 257, 3), (3, 3001, 2), (16, 8192, 12),
                       (64, 3000, 12), (64, 32768, 12), (8128, 100000, 1), (127, 65536, 64),
                       (1000, 5, 8), (7, 1 << 20, 5)]:
        ws_s, ws_c = da.diffattn_decode_split_count(B, lmax, H)
        na_s, na_c = da.diffattn_decode_split_count(B, lmax, H, True)
        for s, c in ((ws_s, ws_c), (na_s, na_c)):
            assert c % 32 == 0 and s * c >= lmax and (s - 1) * c < lmax, (B, lmax, H, s, c)
        assert na_s * B * H <= max_units and na_s <= ws_s
        if ws_s * B * H <= max_units:
            assert (na_s, na_c) == (ws_s, ws_c)
    s, c = ctypes.c_int(0), ctypes.c_int(0)
    assert L.diffattn_decode_split_count(8129, 16, 1, 1, ctypes.byref(s), ctypes.byref(c)) == -2
    assert L.diffattn_decode_split_count(8129, 16, 1, 0, ctypes.byref(s), ctypes.byref(c)) == 0
    assert L.diffattn_decode_split_count(0, 16, 1, 0, ctypes.byref(s), ctypes.byref(c)) == -2
    assert L.diffattn_decode_split_count(1, 16, 1, 0, None, ctypes.byref(c)) == -1


def test_v2_validation(L):
    def v2(Hq=64, Hkv=8, d=128, dtype=0, flags=1, q=FAKE):
        return L.diffattn_v2_fwd(q, FAKE, FAKE, FAKE, FAKE, 2, 64, Hq, Hkv, d, flags, dtype, None)

    assert v2(q=None) == -1
    assert v2(flags=2) == -1
    assert v2(flags=1 | 32 | 16) == -1  # DIFFATTN_EXACT with DIFFATTN_SINGLE_PASS
    assert v2(flags=1 | 32 | 8) == -1   # DIFFATTN_EXACT with DIFFATTN_CUDA_CORES
    assert v2(flags=64) == -1
    assert v2(Hq=63) == -2
    assert v2(Hq=64, Hkv=64) == -2   # Hq/Hkv = 1: a pair would straddle two GQA groups
    assert v2(Hq=48, Hkv=16) == -2   # Hq/Hkv = 3
    assert v2(Hq=64, Hkv=7) == -2
    assert v2(d=96) == -2
    assert v2(dtype=5) == -3


def test_lambda_validation(L):
    assert L.diffattn_lambda(None, FAKE, FAKE, FAKE, 128, 1, 12, FAKE, None) == -1
    assert L.diffattn_lambda(FAKE, FAKE, FAKE, FAKE, 128, 1, 0, FAKE, None) == -1
    assert L.diffattn_lambda(FAKE, FAKE, FAKE, FAKE, 0, 1, 12, FAKE, None) == -2
    assert L.diffattn_lambda(FAKE, FAKE, FAKE, FAKE, 128, 0, 12, FAKE, None) == -2


def test_binding_requires_cuda_tensors():
    import torch
    q = torch.zeros(1, 8, 1, 256, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        da.diffattn_fwd(q, q, q, torch.zeros(1), 0.5)


def test_v2_decode_validation(L):
    n = ctypes.c_size_t(0)
    assert L.diffattn_v2_decode_workspace_size(64, 32768, 64, 8, 128, ctypes.byref(n)) == 0
    need = n.value
    assert L.diffattn_v2_decode_workspace_size(1, 16, 6, 1, 128, ctypes.byref(n)) == -2  # group 6

    def v2d(q=FAKE, Hq=64, Hkv=8, d=128, dtype=0, flags=0, ws=FAKE, ws_bytes=need):
        return L.diffattn_v2_decode(q, FAKE, FAKE, None, FAKE, FAKE, 64, 32768, Hq, Hkv, d, flags,
                                    dtype, ws, ws_bytes, None)

    assert v2d(q=None) == -1
    assert v2d(flags=2) == -1
    assert v2d(Hq=24, Hkv=8) == -2
    assert v2d(d=64) == -2
    assert v2d(dtype=1) == -3
    assert v2d(q=ODD) == -4
    assert v2d(ws_bytes=need - 1) == -8


def test_v2_decode_paged_validation(L):
    n = ctypes.c_size_t(0)
    assert L.diffattn_v2_decode_workspace_size(8, 64 * 256, 16, 2, 128, ctypes.byref(n)) == 0
    need = n.value

    def v2p(table=FAKE, seqlens=FAKE, num_pages=100, page_size=64, max_pages=256, Hq=16,
            flags=0, dtype=0, ws_bytes=need):
        return L.diffattn_v2_decode_paged(FAKE, FAKE, FAKE, table, seqlens, FAKE, FAKE, 8, Hq, 2,
                                          128, num_pages, page_size, max_pages, flags, dtype, FAKE,
                                          ws_bytes, None)

    assert v2p(table=None) == -1
    assert v2p(seqlens=None) == -1  # required for a paged cache
    assert v2p(flags=2) == -1
    assert v2p(page_size=0) == -2
    assert v2p(max_pages=1 << 20, page_size=4096) == -2  # 2^32 keys
    assert v2p(num_pages=1 << 20, page_size=4096) == -2  # pool rows past 2^31
    assert v2p(Hq=12) == -2  # group of 6
    assert v2p(dtype=1) == -3
    assert v2p(ws_bytes=need - 1) == -8


def test_lambda_bwd_validation(L):
    args = [FAKE] * 5
    assert L.diffattn_lambda_bwd(*args, 128, 1, 12, FAKE, FAKE, FAKE, None, None) == -1
    assert L.diffattn_lambda_bwd(*args, 0, 1, 12, FAKE, FAKE, FAKE, FAKE, None) == -2
    assert L.diffattn_lambda_bwd(*args, 128, 1, 0, FAKE, FAKE, FAKE, FAKE, None) == -2
    assert L.diffattn_lambda_bwd(ctypes.c_void_p(0x10002), *args[1:], 128, 1, 12, FAKE, FAKE,
                                 FAKE, FAKE, None) == -4


def test_v2_decode_fp8_validation(L):
    n = ctypes.c_size_t(0)
    assert L.diffattn_v2_decode_workspace_size(4, 1024, 16, 2, 128, ctypes.byref(n)) == 0

    def dec(qd=0.5, kd=0.5, Hq=16, ws=n.value, flags=0):
        return L.diffattn_v2_decode_fp8(FAKE, FAKE, FAKE, None, FAKE, FAKE, qd, kd, 4, 1024, Hq, 2,
                                        128, flags, FAKE, ws, None)
    assert dec(qd=0.0) == -1
    assert dec(kd=float("inf")) == -1
    assert dec(flags=8) == -1          # no CUDA-core form
    assert dec(Hq=12) == -2
    assert dec(ws=n.value - 1) == -8


def test_training_varlen_validation(L):
    n = ctypes.c_size_t(0)
    assert L.diffattn_bwd_varlen_workspace_size(2, 300, 200, 2, 128, 256, ctypes.byref(n)) == -2
    assert L.diffattn_bwd_varlen_workspace_size(2, 300, 600, 2, 128, 256, ctypes.byref(n)) == 0
    assert L.diffattn_fwd_train_varlen(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, 16, 32, FAKE, 0.5,
                                       None, 1e-5, 2, 2, 128, 256, 7, 0, None) == -1
    assert L.diffattn_fwd_train_varlen(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 64, 32, FAKE, 0.5,
                                       None, 1e-5, 2, 2, 128, 256, 7, 0, None) == -2
    assert L.diffattn_bwd_varlen(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 16, 32, FAKE, 0.5, None,
                                 1e-5, FAKE, FAKE, FAKE, FAKE, None, 2, 2, 128, 256, 7, 0, FAKE,
                                 0, None) == -8


def test_training_validation(L):
    def train(q=FAKE, stats=FAKE, d=128, dv=256, flags=7, dtype=0):
        return L.diffattn_fwd_train(q, FAKE, FAKE, FAKE, FAKE, stats, FAKE, 0.5, None, 1e-5, 1, 16,
                                    1, d, dv, flags, dtype, None)

    assert train(q=None) == -1
    assert train(flags=8) == -1          # DIFFATTN_CUDA_CORES has no training path
    assert train(d=64, dv=128) == -2
    assert train(dtype=1) == -3
    assert train(stats=ODD) == -4
    n = ctypes.c_size_t(0)
    assert L.diffattn_bwd_workspace_size(4, 4096, 12, 128, 256, ctypes.byref(n)) == 0
    need = n.value

    def bwd(q=FAKE, dlam=FAKE, ws=FAKE, ws_bytes=need, N=4096):
        return L.diffattn_bwd(q, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0.5, None, 1e-5, FAKE, FAKE,
                              FAKE, dlam, None, 4, N, 12, 128, 256, 7, 0, ws, ws_bytes, None)

    assert bwd(q=None) == -1
    assert bwd(dlam=None) == -1
    assert bwd(N=0) == -2
    assert bwd(q=ODD) == -4
    assert bwd(ws_bytes=need - 1) == -8


def test_fused_lambda_varlen_fp8_strided_validation(L):
    def fused(layer=12, dim=128, sets=1, H=2, flags=7):
        return L.diffattn_fwd_fused_lambda(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, dim, sets,
                                           layer, None, 1e-5, 1, 16, H, 128, 256, flags, 0, None)

    assert fused(layer=0) == -1
    assert fused(dim=0) == -2
    assert fused(sets=3, H=2) == -2      # one lambda set per head, or one for all
    assert fused(flags=8) == -1

    def varlen(maxlen=16, total=32, cu=FAKE):
        return L.diffattn_fwd_varlen(FAKE, FAKE, FAKE, FAKE, cu, maxlen, total, FAKE, 0.5, None,
                                     1e-5, 2, 1, 128, 256, 7, 0, None)

    def varlen_qk(mq=16, mk=32, tq=32, tk=64, cu=FAKE):
        return L.diffattn_fwd_varlen_qk(FAKE, FAKE, FAKE, FAKE, cu, FAKE, mq, mk, tq, tk, FAKE,
                                        0.5, None, 1e-5, 2, 2, 128, 256, 7, 0, None)
    assert varlen_qk(cu=None) == -1
    assert varlen_qk(mq=64, mk=32) == -2   # more queries than keys
    assert varlen_qk(tq=64, tk=32) == -2
    assert varlen_qk(mk=128, tk=64) == -2
    assert varlen_qk(cu=ctypes.c_void_p(0x10002)) == -4
    def paged(ps=128, mq=16, mk=300, tq=32, pages=8, maxp=4, d=128):
        return L.diffattn_fwd_paged(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, mq, mk, tq, pages,
                                    ps, maxp, FAKE, 0.5, None, 1e-5, 2, 2, d, 2 * d, 7, 0, None)
    assert paged(ps=64) == -2              # a tile of 128 keys must lie in one page
    assert paged(mk=8, mq=16) == -2        # fewer keys than queries
    assert paged(mk=600) == -2             # more keys than the table can name (4 x 128)
    assert paged(d=64) == -2
    assert L.diffattn_v2_fwd_paged(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, 16, 32, 32, 8,
                                   128, 4, 2, 8, 2, 128, 1, 0, None) == -1
    def v2var(cu=FAKE, Hq=8, Hkv=2, flags=1):
        return L.diffattn_v2_fwd_varlen(FAKE, FAKE, FAKE, FAKE, FAKE, cu, None, 16, 16, 32, 32, 2,
                                        Hq, Hkv, 128, flags, 0, None)
    assert v2var(cu=None) == -1
    assert v2var(flags=4) == -1            # only DIFFATTN_CAUSAL
    assert v2var(Hq=6, Hkv=2) == -2        # a pair split across GQA groups
    assert varlen(cu=None) == -1
    assert varlen(maxlen=64, total=32) == -2
    assert varlen(cu=ctypes.c_void_p(0x10002)) == -4

    def fp8(qd=1.0, d=128):
        return L.diffattn_fwd_fp8(FAKE, FAKE, FAKE, FAKE, qd, 1.0, FAKE, 0.5, None, 1e-5, 1, 16, 1,
                                  d, 2 * d, 7, None)

    assert fp8(qd=0.0) == -1
    assert fp8(qd=float("inf")) == -1
    assert fp8(d=64) == -2

    def gda_fp8(qd=1.0, d=128, ns=12, nn=3, flags=7, lam=FAKE, v=FAKE):
        return L.diffattn_gda_fwd_fp8(FAKE, FAKE, v, FAKE, qd, 1.0, lam, 0.5, None, 1e-5, 2, 16,
                                      ns, nn, d, 2 * d, flags, None)

    assert gda_fp8(lam=None) == -1
    assert gda_fp8(qd=-1.0) == -1
    assert gda_fp8(qd=float("nan")) == -1
    assert gda_fp8(flags=7 | 16) == -1       # only CAUSAL | NORM | SCALE
    assert gda_fp8(d=64) == -2
    assert gda_fp8(ns=12, nn=5) == -2        # signal heads not a multiple of noise heads
    assert gda_fp8(v=ctypes.c_void_p(0x10008)) == -4

    def strided(st):
        arr = (ctypes.c_longlong * 12)(*st)
        return L.diffattn_fwd_strided(FAKE, FAKE, FAKE, FAKE, arr, FAKE, 0.5, None, 1e-5, 1, 16, 1,
                                      128, 256, 7, 0, None)

    dense = [16 * 256, 256, 256] * 4
    assert strided([s if i != 4 else 260 for i, s in enumerate(dense)]) == -4  # not 16-byte
    assert strided([s if i != 0 else 0 for i, s in enumerate(dense)]) == -4
    assert L.diffattn_fwd_strided(FAKE, FAKE, FAKE, FAKE, None, FAKE, 0.5, None, 1e-5, 1, 16, 1, 128,
                                  256, 7, 0, None) == -1


def test_paged_and_host_validation(L):
    n = ctypes.c_size_t(0)
    assert L.diffattn_decode_workspace_size(2, 64 * 16, 2, 128, 256, ctypes.byref(n)) == 0
    need = n.value

    def paged(table=FAKE, ps=16, mp=64, npages=200, ws_bytes=need):
        return L.diffattn_decode_paged(FAKE, FAKE, FAKE, table, FAKE, FAKE, FAKE, 0.5, None, 1e-5, 2,
                                       2, 128, 256, npages, ps, mp, 6, 0, FAKE, ws_bytes, None)

    assert paged(table=None) == -1
    assert paged(ps=0) == -2
    assert paged(table=ctypes.c_void_p(0x10002)) == -4
    assert paged(ws_bytes=need - 1) == -8
    assert L.diffattn_fwd_host_workspace_size(4, 4096, 12, 128, 256, ctypes.byref(n)) == 0
    hneed = n.value

    def host(q=FAKE, layer=12, ws_bytes=hneed):
        return L.diffattn_fwd_host(q, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 128, 1, layer, None,
                                   1e-5, 4, 4096, 12, 128, 256, 7, FAKE, ws_bytes, None)

    assert host(q=None) == -1
    assert host(layer=0) == -1
    assert host(ws_bytes=hneed - 1) == -8


def test_gda_validation(L):
    def fwd(ns=12, nn=3, d=128, dv=256, flags=7, dtype=0, q=FAKE, N=16, ws=None, ws_bytes=0):
        return L.diffattn_gda_fwd(q, FAKE, FAKE, FAKE, FAKE, 0.5, None, 1e-5, 1, N, ns, nn, d, dv,
                                  flags, dtype, ws, ws_bytes, None)

    n = ctypes.c_size_t(0)
    assert L.diffattn_gda_fwd_workspace_size(4, 4096, 12, 3, 128, 256, ctypes.byref(n)) == 0
    assert n.value == 4 * 3 * 4096 * 4                   # one fp32 statistic per noise row
    assert L.diffattn_gda_fwd_workspace_size(1, 130, 12, 3, 128, 256, ctypes.byref(n)) == 0
    assert n.value == 3 * 256 * 4                         # rows padded to the 128-row tile
    assert L.diffattn_gda_fwd_workspace_size(1, 130, 12, 3, 64, 128, ctypes.byref(n)) == 0
    assert n.value == 0                                   # d = 64: one launch, no workspace
    assert L.diffattn_gda_fwd_workspace_size(1, 130, 12, 5, 128, 256, ctypes.byref(n)) == -2
    assert fwd(ws=ctypes.c_void_p(0x10000), ws_bytes=3 * 128 * 4 - 4) == -8
    assert fwd(ws=ctypes.c_void_p(0x10010), ws_bytes=1 << 20) == -8   # not 256-byte aligned

    assert fwd(q=None) == -1
    assert fwd(flags=64) == -1
    assert fwd(dtype=7) == -3
    assert fwd(N=0) == -2
    assert fwd(nn=0) == -2
    assert fwd(ns=12, nn=5) == -2          # not a whole number of signal heads per noise head
    assert "multiple" in L.diffattn_last_error_string().decode()
    assert fwd(d=96, dv=192) == -2
    assert fwd(q=ODD) == -4

    def fwd_var(ns=12, nn=3, d=128, flags=7, dtype=0, cu=FAKE, maxlen=300, total=1000, ws=None,
                ws_bytes=0):
        return L.diffattn_gda_fwd_varlen(FAKE, FAKE, FAKE, FAKE, cu, maxlen, total, FAKE, 0.5,
                                         None, 1e-5, 4, ns, nn, d, 2 * d, flags, dtype, ws,
                                         ws_bytes, None)

    assert fwd_var(cu=None) == -1
    assert fwd_var(flags=7 | 8) == -1          # the CUDA-core and single-pass forms: batched only
    assert fwd_var(dtype=1) == -3
    assert fwd_var(maxlen=2000) == -2          # longer than the packed axis
    assert fwd_var(ns=12, nn=5) == -2
    assert fwd_var(d=96) == -2
    assert fwd_var(cu=ctypes.c_void_p(0x10002)) == -4
    # the workspace holds B sequences of max_seqlen rows: 4 * 3 * 384 fp32 here
    assert fwd_var(ws=ctypes.c_void_p(0x10000), ws_bytes=4 * 3 * 384 * 4 - 4) == -8
    assert fwd_var(ws=ctypes.c_void_p(0x10010), ws_bytes=1 << 20) == -8

    def fwd_qk(mq=16, mk=32, tq=32, tk=64, cu=FAKE, d=128, ws=None, ws_bytes=0):
        return L.diffattn_gda_fwd_varlen_qk(FAKE, FAKE, FAKE, FAKE, cu, FAKE, mq, mk, tq, tk, FAKE,
                                            0.5, None, 1e-5, 2, 12, 3, d, 2 * d, 7, 0, ws,
                                            ws_bytes, None)

    assert fwd_qk(cu=None) == -1
    assert fwd_qk(mq=64, mk=32) == -2          # more queries than keys
    assert fwd_qk(mk=128, tk=64) == -2
    assert fwd_qk(d=64) == -2                  # d = 128 only
    assert fwd_qk(cu=ctypes.c_void_p(0x10002)) == -4
    assert fwd_qk(ws=ctypes.c_void_p(0x10000), ws_bytes=4) == -8

    def fwd_pg(ps=128, mq=16, mk=300, tq=32, pages=8, maxp=4, table=FAKE):
        return L.diffattn_gda_fwd_paged(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, table, mq, mk, tq,
                                        pages, ps, maxp, FAKE, 0.5, None, 1e-5, 2, 12, 3, 128, 256,
                                        7, 0, None, 0, None)

    assert fwd_pg(table=None) == -1
    assert fwd_pg(ps=64) == -2                 # a tile of 128 keys must lie in one page
    assert fwd_pg(mk=600) == -2                # more keys than max_pages * page_size

    n = ctypes.c_size_t(0)
    assert L.diffattn_decode_workspace_size(8, 4096, 12, 128, 256, ctypes.byref(n)) == 0
    need = n.value

    def dec(ns=12, nn=3, d=128, dv=256, dtype=0, ws=FAKE, ws_bytes=need, flags=6):
        return L.diffattn_gda_decode(FAKE, FAKE, FAKE, None, FAKE, FAKE, 0.5, None, 1e-5, 8, 4096,
                                     ns, nn, d, dv, flags, dtype, ws, ws_bytes, None)

    assert dec(flags=16) == -1
    assert dec(dtype=1) == -3
    assert dec(ns=12, nn=8) == -2
    assert dec(d=64, dv=128) == -2
    assert dec(ws_bytes=need - 1) == -8
    assert dec(ws=ctypes.c_void_p(0x10010)) == -8

    # paged: the workspace is sized for max_pages * page_size keys (32 pages of 128 here)
    def decp(ns=12, nn=3, d=128, ps=128, mp=32, table=FAKE, seqlens=FAKE, ws_bytes=need, flags=6):
        return L.diffattn_gda_decode_paged(FAKE, FAKE, FAKE, table, seqlens, FAKE, FAKE, 0.5, None,
                                           1e-5, 8, ns, nn, d, 2 * d, 500, ps, mp, flags, 0, FAKE,
                                           ws_bytes, None)

    assert decp(table=None) == -1
    assert decp(seqlens=None) == -1
    assert decp(flags=16) == -1
    assert decp(ns=12, nn=5) == -2
    assert decp(d=64) == -2
    assert decp(ps=0) == -2
    assert decp(table=ctypes.c_void_p(0x10002)) == -4
    assert decp(ws_bytes=need - 1) == -8


def test_gda_training_validation(L):
    def train(q=FAKE, stats=FAKE, ns=12, nn=3, d=128, dv=256, flags=7, dtype=0, ws=None,
              ws_bytes=0):
        return L.diffattn_gda_fwd_train(q, FAKE, FAKE, FAKE, FAKE, stats, FAKE, 0.5, None, 1e-5, 1,
                                        300, ns, nn, d, dv, flags, dtype, ws, ws_bytes, None)

    assert train(q=None) == -1
    assert train(stats=None) == -1
    assert train(flags=8) == -1              # DIFFATTN_CUDA_CORES has no training path
    assert train(ns=12, nn=5) == -2          # not a whole number of signal heads per noise head
    assert train(d=64, dv=128) == -2
    assert train(dtype=1) == -3
    assert train(stats=ODD) == -4
    assert train(ws=ctypes.c_void_p(0x10000), ws_bytes=3 * 384 * 4 - 4) == -8
    n = ctypes.c_size_t(0)
    assert L.diffattn_gda_bwd_workspace_size(4, 4096, 12, 3, 128, 256, ctypes.byref(n)) == 0
    need = n.value
    m = ctypes.c_size_t(0)
    assert L.diffattn_bwd_workspace_size(4, 4096, 12, 128, 256, ctypes.byref(m)) == 0
    # the ungrouped backward's workspace for the signal heads, plus the noise heads' fp32 dK sums
    assert need >= m.value + 4 * 4096 * 3 * 128 * 4
    assert L.diffattn_gda_bwd_workspace_size(4, 4096, 12, 5, 128, 256, ctypes.byref(n)) == -2

    def bwd(q=FAKE, dk=FAKE, ns=12, nn=3, ws=FAKE, ws_bytes=need, N=4096, dtype=0):
        return L.diffattn_gda_bwd(q, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0.5, None, 1e-5, FAKE, dk,
                                  FAKE, FAKE, None, 4, N, ns, nn, 128, 256, 7, dtype, ws, ws_bytes,
                                  None)

    assert bwd(q=None) == -1
    assert bwd(dk=None) == -1
    assert bwd(N=0) == -2
    assert bwd(ns=12, nn=0) == -2
    assert bwd(dtype=1) == -3
    assert bwd(q=ODD) == -4
    assert bwd(ws_bytes=need - 1) == -8

    # packed sequences
    def train_v(cu=FAKE, stats=FAKE, ns=12, nn=3, mx=300, total=1000, dtype=0):
        return L.diffattn_gda_fwd_train_varlen(FAKE, FAKE, FAKE, FAKE, FAKE, stats, cu, mx, total,
                                               FAKE, 0.5, None, 1e-5, 4, ns, nn, 128, 256, 7,
                                               dtype, None, 0, None)

    assert train_v(cu=None) == -1
    assert train_v(stats=None) == -1
    assert train_v(ns=12, nn=5) == -2
    assert train_v(mx=2000) == -2            # longer than the packed axis
    assert train_v(dtype=1) == -3
    assert train_v(cu=ctypes.c_void_p(0x10002)) == -4
    assert L.diffattn_gda_bwd_varlen_workspace_size(4, 300, 1000, 12, 3, 128, 256,
                                                    ctypes.byref(n)) == 0
    need_v = n.value
    assert L.diffattn_gda_bwd_varlen_workspace_size(4, 300, 200, 12, 3, 128, 256,
                                                    ctypes.byref(n)) == -2

    def bwd_v(cu=FAKE, ns=12, nn=3, ws_bytes=need_v, total=1000):
        return L.diffattn_gda_bwd_varlen(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, cu, 300, total, FAKE,
                                         0.5, None, 1e-5, FAKE, FAKE, FAKE, FAKE, None, 4, ns, nn,
                                         128, 256, 7, 0, FAKE, ws_bytes, None)

    assert bwd_v(cu=None) == -1
    assert bwd_v(ns=12, nn=5) == -2
    assert bwd_v(total=200) == -2
    assert bwd_v(ws_bytes=need_v - 1) == -8


def test_v2_decode_fp8_paged_validation(L):
    n = ctypes.c_size_t(0)
    assert L.diffattn_v2_decode_workspace_size(4, 4096, 16, 2, 128, ctypes.byref(n)) == 0
    need = n.value

    def dec(ps=128, mp=32, qd=1.0, flags=0, d=128, table=FAKE, ws_bytes=need):
        return L.diffattn_v2_decode_fp8_paged(FAKE, FAKE, FAKE, table, FAKE, FAKE, FAKE, qd, 1.0,
                                              4, 16, 2, d, 200, ps, mp, flags, FAKE, ws_bytes, None)

    assert dec(table=None) == -1
    assert dec(flags=16) == -1
    assert dec(qd=0.0) == -1
    assert dec(ps=64, mp=64) == -7          # fp8 pages must be whole 128-key tiles
    assert "multiple of 128" in L.diffattn_last_error_string().decode()
    assert dec(d=64) == -2
    assert dec(ws_bytes=need - 1) == -8


def test_binding_constants_match_the_header():
    """Every flag, dtype and status value the binding passes or compares equals the header's."""
    hdr = open(os.path.join(os.path.dirname(__file__), "..", "include", "diffattn.h")).read()
    defines = {m.group(1): int(m.group(2))
               for m in re.finditer(r"#define (DIFFATTN_[A-Z_0-9]+) (\d+)\b", hdr)}
    enums = {m.group(1): int(m.group(2))
             for m in re.finditer(r"\b(DIFFATTN_[A-Z_0-9]+) = (-?\d+)", hdr)}
    for name in ("DIFFATTN_CAUSAL", "DIFFATTN_NORM", "DIFFATTN_SCALE", "DIFFATTN_CUDA_CORES",
                 "DIFFATTN_SINGLE_PASS", "DIFFATTN_EXACT"):
        assert getattr(da, name) == defines[name], name
    for name in ("DIFFATTN_OK", "DIFFATTN_BF16", "DIFFATTN_FP32"):
        assert getattr(da, name) == enums[name], name
    flags = [defines[n] for n in defines if n not in ("DIFFATTN_H_",) and n in dir(da)]
    assert len(set(flags)) == len(flags)  # distinct bits
