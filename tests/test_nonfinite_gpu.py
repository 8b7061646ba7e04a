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
