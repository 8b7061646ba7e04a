"""Canaries: every output (and workspace) a call writes sits between guard bands that must come
back untouched, for the entry points beyond the prefill (whose guard test is in
test_parity_gpu.py): decode, V2 prefill and decode, the grouped decode, and the backward's
gradients. Shapes are ragged so that partial tiles and split tails write at the edges."""
import pytest
import torch

import differential_attention_gb300 as da
from synth import (make_decode_inputs, make_dout, make_gda_decode_inputs, make_prefill_inputs,
                   make_v2_decode_inputs, make_v2_inputs)

pytestmark = pytest.mark.gpu

DEV = "cuda"
G = 4096  # guard elements on each side


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    da.build()
    da.lib()
    yield
    da.diffattn_device_status()


class Guarded:
    """A tensor of `shape` inside a buffer with G guard elements on each side, filled with a
    canary value."""

    def __init__(self, shape, dtype, canary=7.0):
        n = 1
        for s in shape:
            n *= s
        self.n, self.canary = n, canary
        self.buf = torch.full((n + 2 * G,), canary, dtype=dtype, device=DEV)
        self.t = self.buf[G:G + n].view(*shape)

    def intact(self):
        torch.cuda.synchronize()
        return bool(torch.all(self.buf[:G] == self.canary)) and bool(
            torch.all(self.buf[G + self.n:] == self.canary))


def test_decode_guard():
    inp = make_decode_inputs(3, 701, 2, 128, 256, seed=401, ragged=True)
    out = Guarded((3, 2, 256), torch.bfloat16)
    ws = Guarded((da.diffattn_decode_workspace_size(3, 701, 2),), torch.uint8, canary=0x5A)
    da.diffattn_decode(inp.q.to(DEV), inp.k_cache.to(DEV), inp.v_cache.to(DEV), inp.lam.to(DEV),
                       0.5, seqlens=inp.seqlens.to(DEV), workspace=ws.t, out=out.t)
    assert out.intact() and ws.intact()


def test_v2_prefill_and_decode_guard():
    inp = make_v2_inputs(1, 333, 8, 2, 128, seed=403)
    out = Guarded((1, 333, 4, 128), torch.bfloat16)
    da.diffattn_v2_fwd(inp.q.to(DEV), inp.k.to(DEV), inp.v.to(DEV), inp.lam_logit.to(DEV),
                       out=out.t)
    assert out.intact()
    dinp = make_v2_decode_inputs(3, 517, 16, 2, 128, seed=405, ragged=True)
    dout = Guarded((3, 8, 128), torch.bfloat16)
    ws = Guarded((da.diffattn_v2_decode_workspace_size(3, 517, 16, 2, 128),), torch.uint8,
                 canary=0x5A)
    da.diffattn_v2_decode(dinp.q.to(DEV), dinp.k_cache.to(DEV), dinp.v_cache.to(DEV),
                          dinp.lam_logit.to(DEV), seqlens=dinp.seqlens.to(DEV), workspace=ws.t,
                          out=dout.t)
    assert dout.intact() and ws.intact()


def test_gda_decode_guard():
    inp = make_gda_decode_inputs(2, 901, 6, 2, 128, 256, seed=407, ragged=True)
    out = Guarded((2, 6, 256), torch.bfloat16)
    ws = Guarded((da.diffattn_decode_workspace_size(2, 901, 6),), torch.uint8, canary=0x5A)
    da.diffattn_gda_decode(inp.q.to(DEV), inp.k_cache.to(DEV), inp.v_cache.to(DEV),
                           inp.lam.to(DEV), 6, 0.5, seqlens=inp.seqlens.to(DEV), workspace=ws.t,
                           out=out.t)
    assert out.intact() and ws.intact()


def test_backward_guard():
    B, N, H = 1, 333, 2
    inp = make_prefill_inputs(B, N, H, 128, 256, seed=409)
    q, k, v = inp.q.to(DEV), inp.k.to(DEV), inp.v.to(DEV)
    dy = make_dout(B, N, H, 256, seed=411).to(DEV)
    lam = torch.tensor([0.4, 0.7], dtype=torch.float32, device=DEV)
    _, o_pre, stats = da.diffattn_fwd_train(q, k, v, lam, 0.5)
    g = {name: Guarded(shape, dt) for name, shape, dt in (
        ("dq", q.shape, torch.bfloat16), ("dk", k.shape, torch.bfloat16),
        ("dv", v.shape, torch.bfloat16), ("dlam", (H,), torch.float32),
        ("dw", (256,), torch.float32))}
    w = torch.ones(256, dtype=torch.float32, device=DEV)
    ws = Guarded((da.diffattn_bwd_workspace_size(B, N, H, 128, 256),), torch.uint8, canary=0x5A)
    da.diffattn_bwd(q, k, v, o_pre, stats, dy, lam, 0.5, norm_weight=w, workspace=ws.t,
                    grads={name: x.t for name, x in g.items()})
    for name, x in g.items():
        assert x.intact(), name
    assert ws.intact()
