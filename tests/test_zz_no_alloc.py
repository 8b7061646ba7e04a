"""The decode entry point that allocates nothing (diffattn_decode_noalloc).

It exists for callers that cannot allocate device memory where they decode: a plugin inside a
host runtime that owns all device buffers and offers no allocator, or a latency-bound decode loop
that may not call cudaMalloc / cudaFree. Its split partials live in a scratch array built into the
library, shared by all calls on a device. These tests call it through the C ABI twice in a row
(different shapes, so the second call runs over what the first left in the shared array) and
compare each result with diffattn_decode (which takes a caller workspace) on the same inputs,
within the bf16 tolerance the other parity tests use. The file is named to be collected last.
"""
import ctypes

import pytest
import torch

import differential_attention_gb300 as da
from synth import make_decode_inputs
from tests.gpu_util import assert_bf16

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    da.build()
    da.lib()


def _both(inp, li, w):
    kw = dict(seqlens=inp.seqlens.to(DEV), norm_weight=w)
    args = (inp.q.to(DEV), inp.k_cache.to(DEV), inp.v_cache.to(DEV), inp.lam.to(DEV), li)
    with_ws = da.diffattn_decode(*args, **kw)
    no_alloc = da.diffattn_decode_noalloc(*args, **kw)
    return with_ws, no_alloc


def test_noalloc_matches_workspace_decode_two_calls():
    w = torch.linspace(0.9, 1.1, 256, dtype=torch.float32, device=DEV)
    # first call: ragged lengths, few (sequence, head) pairs -> same split count as diffattn_decode
    a = make_decode_inputs(3, 3001, 2, 128, 256, seed=501, ragged=True)
    # second call: 192 (sequence, head) pairs over 8192 keys -> fewer splits than diffattn_decode,
    # run over the partials the first call left in the shared array
    b = make_decode_inputs(16, 8192, 12, 128, 256, seed=502, ragged=False)
    li = da.diffattn_lambda_init(12)
    ra, na = _both(a, li, w)
    rb, nb = _both(b, li, w)
    torch.cuda.synchronize()
    assert_bf16(na, ra)
    assert_bf16(nb, rb)
    da.diffattn_device_status()


def test_noalloc_rejects_too_many_pairs():
    L = da.lib()
    fake = ctypes.c_void_p(0x10000)
    # B * H = 8129 > 16 MiB / (516 floats * 4 B) = 8128
    rc = L.diffattn_decode_noalloc(fake, fake, fake, None, fake, fake, 0.5, None, 1e-5, 8129, 16,
                                   1, 128, 256, 6, 0, None)
    assert rc == -2
    assert "scratch" in L.diffattn_last_error_string().decode()
