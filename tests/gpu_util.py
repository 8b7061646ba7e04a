"""Shared helpers for the GPU parity tests: tolerances and comparison against the oracle."""
import numpy as np
import torch

# Tolerances: fp32 I/O max |err| <= 1e-4; bf16 I/O (fp32 accumulation) relative L2 <= 1e-2 and
# max |err| <= 3e-2, measured on the final (normed, scaled) output against the float64 oracle.
FP32_MAX_ABS = 1e-4
BF16_REL_L2 = 1e-2
BF16_MAX_ABS = 3e-2


def to64(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        return t.detach().float().cpu().double().numpy()
    return np.asarray(t, dtype=np.float64)


def errors(got, want):
    g, w = to64(got), to64(want)
    assert g.shape == w.shape, (g.shape, w.shape)
    assert np.all(np.isfinite(g)), "non-finite output"
    diff = g - w
    max_abs = float(np.max(np.abs(diff))) if diff.size else 0.0
    den = float(np.linalg.norm(w))
    rel = float(np.linalg.norm(diff) / den) if den > 0 else float(np.linalg.norm(diff))
    return max_abs, rel


def assert_fp32(got, want):
    max_abs, rel = errors(got, want)
    assert max_abs <= FP32_MAX_ABS, f"max abs {max_abs:.3e} > {FP32_MAX_ABS}"
    return max_abs, rel


def assert_bf16(got, want, rel_tol=BF16_REL_L2, abs_tol=BF16_MAX_ABS):
    max_abs, rel = errors(got, want)
    assert rel <= rel_tol and max_abs <= abs_tol, f"rel L2 {rel:.3e} (<= {rel_tol}), max abs {max_abs:.3e} (<= {abs_tol})"
    return max_abs, rel


# Gradients (backward of the bf16 prefill): P, dS, W and dO are rounded to bf16 before each
# product (relative 2^-9 each) and every product accumulates in fp32, so a gradient carries a few
# bf16 roundings of relative error: relative L2 <= 2e-2 per tensor, and no element off by more
# than 5e-2 of the tensor's largest magnitude.
GRAD_REL_L2 = 2e-2
GRAD_MAX_REL = 5e-2


# Where the exact gradient is identically zero (one visible key: the softmax is constant), the
# kernel's dW - delta differs from 0 by the bf16 rounding of dO, so the bar is absolute.
GRAD_ZERO_ABS = 1e-3


def assert_grad(got, want, rel_tol=GRAD_REL_L2, max_rel=GRAD_MAX_REL, name=""):
    g, w = to64(got), to64(want)
    max_abs, rel = errors(g, w)
    scale = float(np.max(np.abs(w))) if w.size else 0.0
    if scale == 0.0:
        assert max_abs <= GRAD_ZERO_ABS, f"{name}: exact gradient is 0, max abs {max_abs:.3e}"
        return max_abs, rel
    assert rel <= rel_tol and max_abs <= max_rel * max(scale, 1e-30), (
        f"{name}: rel L2 {rel:.3e} (<= {rel_tol}), max abs {max_abs:.3e} "
        f"(<= {max_rel} x {scale:.3e})")
    return max_abs, rel
