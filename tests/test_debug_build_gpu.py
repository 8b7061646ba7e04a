"""The bounds-checking debug build of the library, run under the small-case parity suite.

libdiffattn_debug.so is the same source compiled with -DDIFFATTN_DEBUG: every kernel checks the
tile coordinates of its TMA copies and every row it gathers or stores against the extent of its
tensor, and reports a failed check through diffattn_device_status (DIFFATTN_ERR_INDEX) instead of
touching memory outside the tensor. It stands in for a memory sanitizer. This test builds it and
runs the small-case GPU suites -- every entry point on small, ragged and edge-case shapes
(test_parity_gpu.py), the backward (test_backward_gpu.py), the grouped form and its training
path (test_gda_gpu.py, test_gda_train_gpu.py), non-finite inputs and guard bands around every output and workspace -- in a child process that
loads the debug build; each test checks against the float64 oracle and calls
diffattn_device_status, and all must pass with no check failing.
"""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_parity_suite_under_the_debug_build():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    env = dict(os.environ, DIFFATTN_DEBUG_BUILD="1")
    build = subprocess.run([sys.executable, "-c", "import differential_attention_gb300 as da; "
                            "print(da.build())"], cwd=ROOT, env=env, capture_output=True, text=True,
                           timeout=1200)
    assert build.returncode == 0, build.stdout[-2000:] + build.stderr[-4000:]
    assert build.stdout.strip().endswith("libdiffattn_debug.so")
    suites = ["tests/test_parity_gpu.py", "tests/test_backward_gpu.py", "tests/test_gda_gpu.py",
              "tests/test_gda_train_gpu.py", "tests/test_nonfinite_gpu.py",
              "tests/test_guard_gpu.py"]
    run = subprocess.run([sys.executable, "-m", "pytest", *suites, "-m", "gpu", "-x", "-q", "-p",
                          "no:cacheprovider"], cwd=ROOT, env=env, capture_output=True, text=True,
                         timeout=1800)
    assert run.returncode == 0, run.stdout[-4000:] + run.stderr[-2000:]
    summary = [ln for ln in run.stdout.splitlines() if " passed" in ln]
    assert summary, run.stdout[-2000:]
    print("debug build:", build.stdout.strip(), "|", summary[-1])
    n_passed = int(summary[-1].split(" passed")[0].split()[-1])
    assert n_passed >= 150, summary[-1]
