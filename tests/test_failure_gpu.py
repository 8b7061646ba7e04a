"""Failure detection on the GPU without a GPU fault: a kernel's bounded wait runs out (it waits
on a barrier that nothing arrives on), the kernel returns, the host reads ERR_TIMEOUT from the
device status word once, and the context stays usable for normal work."""
import numpy as np
import pytest
import torch

import differential_attention_gb300 as da
from oracle import diffattn_ref as ref
from synth import make_prefill_inputs
from tests.gpu_util import assert_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    da.build()


def test_bounded_wait_reports_timeout_and_context_survives():
    da.diffattn_device_status()  # start clean
    da.diffattn_selftest_wait_timeout(50)
    with pytest.raises(da.DiffAttnError) as exc:
        da.diffattn_device_status()
    assert exc.value.status == -6
    da.diffattn_device_status()  # the flag was cleared by the read
    inp = make_prefill_inputs(1, 200, 2, 128, 256, seed=7)
    lam = np.array([0.5, 0.7])
    got = da.diffattn_fwd(inp.q.cuda(), inp.k.cuda(), inp.v.cuda(),
                          torch.tensor(lam, dtype=torch.float32, device="cuda"), 0.4)
    assert_bf16(got, ref.diffattn_fwd(inp.q, inp.k, inp.v, lam, 0.4))
    da.diffattn_device_status()


def test_selftest_rejects_bad_limit():
    with pytest.raises(da.DiffAttnError):
        da.diffattn_selftest_wait_timeout(0)
