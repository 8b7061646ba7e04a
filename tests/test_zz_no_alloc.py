"""The decode entry point that allocates nothing (diffattn_decode_noalloc).

It exists for callers that cannot allocate device memory where they decode: a plugin inside a
host runtime that owns all device buffers and offers no allocator, or a latency-bound decode loop
that may not call cudaMalloc / cudaFree (both can synchronise the device). Its split partials
live in a scratch array built into the library, shared by all calls on a device.

The test calls it through the C ABI twice in a row, on shapes that take both of its branches:

1. 3 sequences x 2 heads over up to 3001 keys: the partials of diffattn_decode's split count fit
   in the scratch, so both entry points run the same kernels on the same slices, and their
   outputs must be bit-identical;
2. 64 sequences x 12 heads over up to 3000 keys: 12 slices per (sequence, head) would not fit,
   so the no-allocation call cuts the cache into fewer, longer slices (the split counts are
   read from diffattn_decode_split_count), runs over what the first call left in the array,
   and must agree with diffattn_decode within the bf16 tolerance of the other parity tests.

Both results are also checked against the float64 oracle. The file is named to be collected
last, and the test passes alone in a fresh process as well as after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import differential_attention_gb300 as da
from oracle import diffattn_ref as ref
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


def _oracle(inp, w, layer):
    """The float64 oracle's decode, one sequence's cache copied to the host at a time."""
    host = lambda t: t.cpu().to(torch.float64).numpy()
    q, lam, seqlens, w = host(inp.q), host(inp.lam), inp.seqlens.cpu().numpy(), host(w)
    B = q.shape[0]
    return np.concatenate([
        ref.diffattn_decode(q[b:b + 1], host(inp.k_cache[b:b + 1]), host(inp.v_cache[b:b + 1]),
                            seqlens[b:b + 1], lam, ref.lambda_init(layer), norm_weight=w)
        for b in range(B)])


def test_noalloc_matches_workspace_decode_two_calls():
    layer = 12
    w = torch.linspace(0.9, 1.1, 256, dtype=torch.float32, device=DEV)
    li = da.diffattn_lambda_init(layer)

    # first call: the split count is kept -> bit-identical to diffattn_decode
    a = make_decode_inputs(3, 3001, 2, 128, 256, seed=501, ragged=True)
    assert da.diffattn_decode_split_count(3, 3001, 2) == da.diffattn_decode_split_count(3, 3001, 2, True)
    ra, na = _both(a, li, w)

    # second call: the split count is lowered (12 -> at most 10 slices per (sequence, head))
    b = make_decode_inputs(64, 3000, 12, 128, 256, seed=502, ragged=True, device=DEV)
    ws_splits, _ = da.diffattn_decode_split_count(64, 3000, 12)
    na_splits, _ = da.diffattn_decode_split_count(64, 3000, 12, True)
    assert na_splits < ws_splits, (na_splits, ws_splits)
    rb, nb = _both(b, li, w)
    torch.cuda.synchronize()
    da.diffattn_device_status()

    assert torch.equal(na, ra)
    assert_bf16(nb, rb)
    assert_bf16(na, _oracle(a, w, layer))
    assert_bf16(nb, _oracle(b, w, layer))


def test_noalloc_rejects_too_many_pairs():
    L = da.lib()
    fake = ctypes.c_void_p(0x10000)
    # B * H = 8129 > 16 MiB / (516 floats * 4 B) = 8128
    rc = L.diffattn_decode_noalloc(fake, fake, fake, None, fake, fake, 0.5, None, 1e-5, 8129, 16,
                                   1, 128, 256, 6, 0, None)
    assert rc == -2
    assert "scratch" in L.diffattn_last_error_string().decode()
