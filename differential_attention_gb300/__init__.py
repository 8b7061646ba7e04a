"""Differential attention on GB300 (sm_103a): Python binding of libdiffattn.so.

Every function here has the name of the C entry point it calls (include/diffattn.h) and only
marshals arguments: torch tensors supply device memory and the current CUDA stream, and all of the
operator's arithmetic runs in the library's CUDA kernels. There is no CPU or PyTorch fallback; if
the library has not been built, every call raises.

Layouts (dense, row-major):
    diffattn_fwd     q, k [B, N, H, 2d] ([Q1|Q2], [K1|K2]), v [B, N, H, 2d]  -> [B, N, H, 2d]
    diffattn_decode  q [B, H, 2d], k_cache, v_cache [B, L, H, 2d]            -> [B, H, 2d]
    diffattn_v2_fwd  q [B, N, Hq, d], k, v [B, N, Hkv, d], lam [B, N, Hq/2]  -> [B, N, Hq/2, d]
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
# DIFFATTN_DEBUG_BUILD=1 selects the bounds-checking debug build of the same library
# (libdiffattn_debug.so: every kernel checks its tile coordinates and row indices and reports a
# failure through diffattn_device_status); the default is the release build.
DEBUG_BUILD = os.environ.get("DIFFATTN_DEBUG_BUILD", "0") == "1"
LIB_PATH = os.path.join(_PKG, "libdiffattn_debug.so" if DEBUG_BUILD else "libdiffattn.so")

DIFFATTN_OK = 0
DIFFATTN_BF16 = 0
DIFFATTN_FP32 = 1
DIFFATTN_CAUSAL = 1
DIFFATTN_NORM = 2
DIFFATTN_SCALE = 4
DIFFATTN_CUDA_CORES = 8
DIFFATTN_SINGLE_PASS = 16
DIFFATTN_EXACT = 32

STATUS_NAMES = {0: "OK", -1: "ERR_ARG", -2: "ERR_SHAPE", -3: "ERR_DTYPE", -4: "ERR_ALIGN",
                -5: "ERR_CUDA", -6: "ERR_TIMEOUT", -7: "ERR_UNSUPPORTED", -8: "ERR_WORKSPACE",
                -9: "ERR_INDEX"}


class DiffAttnError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


_lib = None

_SIGNATURES = {
    "diffattn_version": (ctypes.c_int, []),
    "diffattn_last_error_string": (ctypes.c_char_p, []),
    "diffattn_device_status": (ctypes.c_int, [ctypes.c_void_p]),
    "diffattn_lambda_init": (ctypes.c_float, [ctypes.c_int]),
    "diffattn_selftest_wait_timeout": (ctypes.c_int, [ctypes.c_int, ctypes.c_void_p]),
    "diffattn_lambda": (ctypes.c_int, [ctypes.c_void_p] * 4 + [ctypes.c_int] * 3
                        + [ctypes.c_void_p, ctypes.c_void_p]),
    "diffattn_lambda_bwd": (ctypes.c_int, [ctypes.c_void_p] * 5 + [ctypes.c_int] * 3
                            + [ctypes.c_void_p] * 5),
    "diffattn_fwd": (ctypes.c_int, [ctypes.c_void_p] * 5 + [ctypes.c_float, ctypes.c_void_p,
                                                             ctypes.c_float] + [ctypes.c_int] * 7
                     + [ctypes.c_void_p]),
    "diffattn_decode_workspace_size": (ctypes.c_int, [ctypes.c_int] * 5
                                       + [ctypes.POINTER(ctypes.c_size_t)]),
    "diffattn_decode": (ctypes.c_int, [ctypes.c_void_p] * 6 + [ctypes.c_float, ctypes.c_void_p,
                                                               ctypes.c_float] + [ctypes.c_int] * 7
                        + [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "diffattn_decode_noalloc": (ctypes.c_int, [ctypes.c_void_p] * 6
                                + [ctypes.c_float, ctypes.c_void_p, ctypes.c_float]
                                + [ctypes.c_int] * 7 + [ctypes.c_void_p]),
    "diffattn_decode_split_count": (ctypes.c_int, [ctypes.c_int] * 4
                                    + [ctypes.POINTER(ctypes.c_int)] * 2),
    "diffattn_v2_fwd": (ctypes.c_int, [ctypes.c_void_p] * 5 + [ctypes.c_int] * 7
                        + [ctypes.c_void_p]),
    "diffattn_v2_decode_workspace_size": (ctypes.c_int, [ctypes.c_int] * 5
                                          + [ctypes.POINTER(ctypes.c_size_t)]),
    "diffattn_decode_paged": (ctypes.c_int, [ctypes.c_void_p] * 7 + [ctypes.c_float, ctypes.c_void_p,
                                                                      ctypes.c_float]
                              + [ctypes.c_int] * 9 + [ctypes.c_void_p, ctypes.c_size_t,
                                                      ctypes.c_void_p]),
    "diffattn_fwd_host_workspace_size": (ctypes.c_int, [ctypes.c_int] * 5
                                         + [ctypes.POINTER(ctypes.c_size_t)]),
    "diffattn_fwd_host": (ctypes.c_int, [ctypes.c_void_p] * 8 + [ctypes.c_int] * 3
                          + [ctypes.c_void_p, ctypes.c_float] + [ctypes.c_int] * 6
                          + [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "diffattn_fwd_strided": (ctypes.c_int, [ctypes.c_void_p] * 4 + [ctypes.POINTER(ctypes.c_longlong)]
                             + [ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p, ctypes.c_float]
                             + [ctypes.c_int] * 7 + [ctypes.c_void_p]),
    "diffattn_fwd_fp8": (ctypes.c_int, [ctypes.c_void_p] * 4 + [ctypes.c_float] * 2
                         + [ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p, ctypes.c_float]
                         + [ctypes.c_int] * 6 + [ctypes.c_void_p]),
    "diffattn_fwd_varlen": (ctypes.c_int, [ctypes.c_void_p] * 5 + [ctypes.c_int] * 2
                            + [ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p, ctypes.c_float]
                            + [ctypes.c_int] * 6 + [ctypes.c_void_p]),
    "diffattn_fwd_varlen_qk": (ctypes.c_int, [ctypes.c_void_p] * 6 + [ctypes.c_int] * 4
                               + [ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p, ctypes.c_float]
                               + [ctypes.c_int] * 6 + [ctypes.c_void_p]),
    "diffattn_v2_fwd_varlen": (ctypes.c_int, [ctypes.c_void_p] * 7 + [ctypes.c_int] * 10
                               + [ctypes.c_void_p]),
    "diffattn_fwd_paged": (ctypes.c_int, [ctypes.c_void_p] * 7 + [ctypes.c_int] * 6
                           + [ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p, ctypes.c_float]
                           + [ctypes.c_int] * 6 + [ctypes.c_void_p]),
    "diffattn_v2_fwd_paged": (ctypes.c_int, [ctypes.c_void_p] * 8 + [ctypes.c_int] * 12
                              + [ctypes.c_void_p]),
    "diffattn_fwd_fused_lambda": (ctypes.c_int, [ctypes.c_void_p] * 8 + [ctypes.c_int] * 3
                                  + [ctypes.c_void_p, ctypes.c_float] + [ctypes.c_int] * 7
                                  + [ctypes.c_void_p]),
    "diffattn_fwd_train": (ctypes.c_int, [ctypes.c_void_p] * 7 + [ctypes.c_float, ctypes.c_void_p,
                                                                   ctypes.c_float]
                           + [ctypes.c_int] * 7 + [ctypes.c_void_p]),
    "diffattn_bwd_workspace_size": (ctypes.c_int, [ctypes.c_int] * 5
                                    + [ctypes.POINTER(ctypes.c_size_t)]),
    "diffattn_bwd": (ctypes.c_int, [ctypes.c_void_p] * 7 + [ctypes.c_float, ctypes.c_void_p,
                                                             ctypes.c_float]
                     + [ctypes.c_void_p] * 5 + [ctypes.c_int] * 7
                     + [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "diffattn_fwd_train_varlen": (ctypes.c_int, [ctypes.c_void_p] * 7 + [ctypes.c_int] * 2
                                  + [ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p,
                                     ctypes.c_float]
                                  + [ctypes.c_int] * 6 + [ctypes.c_void_p]),
    "diffattn_bwd_varlen_workspace_size": (ctypes.c_int, [ctypes.c_int] * 6
                                           + [ctypes.POINTER(ctypes.c_size_t)]),
    "diffattn_bwd_varlen": (ctypes.c_int, [ctypes.c_void_p] * 7 + [ctypes.c_int] * 2
                            + [ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p, ctypes.c_float]
                            + [ctypes.c_void_p] * 5 + [ctypes.c_int] * 6
                            + [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "diffattn_v2_decode": (ctypes.c_int, [ctypes.c_void_p] * 6 + [ctypes.c_int] * 7
                           + [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "diffattn_v2_decode_fp8": (ctypes.c_int, [ctypes.c_void_p] * 6 + [ctypes.c_float] * 2
                               + [ctypes.c_int] * 6
                               + [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "diffattn_v2_decode_paged": (ctypes.c_int, [ctypes.c_void_p] * 7 + [ctypes.c_int] * 9
                                 + [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "diffattn_v2_decode_fp8_paged": (ctypes.c_int, [ctypes.c_void_p] * 7 + [ctypes.c_float] * 2
                                     + [ctypes.c_int] * 8
                                     + [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "diffattn_gda_fwd_workspace_size": (ctypes.c_int, [ctypes.c_int] * 6
                                        + [ctypes.POINTER(ctypes.c_size_t)]),
    "diffattn_gda_fwd": (ctypes.c_int, [ctypes.c_void_p] * 5 + [ctypes.c_float, ctypes.c_void_p,
                                                                 ctypes.c_float] + [ctypes.c_int] * 8
                         + [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "diffattn_gda_fwd_fp8": (ctypes.c_int, [ctypes.c_void_p] * 4 + [ctypes.c_float] * 2
                             + [ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p, ctypes.c_float]
                             + [ctypes.c_int] * 7 + [ctypes.c_void_p]),
    "diffattn_gda_fwd_varlen": (ctypes.c_int, [ctypes.c_void_p] * 5 + [ctypes.c_int] * 2
                                + [ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p,
                                   ctypes.c_float] + [ctypes.c_int] * 7
                                + [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "diffattn_gda_decode_paged": (ctypes.c_int, [ctypes.c_void_p] * 7
                                  + [ctypes.c_float, ctypes.c_void_p, ctypes.c_float]
                                  + [ctypes.c_int] * 10
                                  + [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "diffattn_gda_fwd_varlen_qk": (ctypes.c_int, [ctypes.c_void_p] * 6 + [ctypes.c_int] * 4
                                   + [ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p,
                                      ctypes.c_float] + [ctypes.c_int] * 7
                                   + [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "diffattn_gda_fwd_paged": (ctypes.c_int, [ctypes.c_void_p] * 7 + [ctypes.c_int] * 6
                               + [ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p, ctypes.c_float]
                               + [ctypes.c_int] * 7
                               + [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "diffattn_gda_fwd_train": (ctypes.c_int, [ctypes.c_void_p] * 7 + [ctypes.c_float, ctypes.c_void_p,
                                                                       ctypes.c_float]
                               + [ctypes.c_int] * 8
                               + [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "diffattn_gda_bwd_workspace_size": (ctypes.c_int, [ctypes.c_int] * 6
                                        + [ctypes.POINTER(ctypes.c_size_t)]),
    "diffattn_gda_bwd": (ctypes.c_int, [ctypes.c_void_p] * 7 + [ctypes.c_float, ctypes.c_void_p,
                                                                 ctypes.c_float]
                         + [ctypes.c_void_p] * 5 + [ctypes.c_int] * 8
                         + [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "diffattn_gda_fwd_train_varlen": (ctypes.c_int, [ctypes.c_void_p] * 7 + [ctypes.c_int] * 2
                                      + [ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p,
                                         ctypes.c_float] + [ctypes.c_int] * 7
                                      + [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "diffattn_gda_bwd_varlen_workspace_size": (ctypes.c_int, [ctypes.c_int] * 7
                                               + [ctypes.POINTER(ctypes.c_size_t)]),
    "diffattn_gda_bwd_varlen": (ctypes.c_int, [ctypes.c_void_p] * 7 + [ctypes.c_int] * 2
                                + [ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p,
                                   ctypes.c_float] + [ctypes.c_void_p] * 5 + [ctypes.c_int] * 7
                                + [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "diffattn_gda_decode": (ctypes.c_int, [ctypes.c_void_p] * 6 + [ctypes.c_float, ctypes.c_void_p,
                                                                    ctypes.c_float]
                            + [ctypes.c_int] * 8 + [ctypes.c_void_p, ctypes.c_size_t,
                                                     ctypes.c_void_p]),
}


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it has not been built with `build()`)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m differential_attention_gb300.builder`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype, fn.argtypes = res, args
        _lib = L
    return _lib


def build(force: bool = False) -> str:
    """Compile libdiffattn.so (libdiffattn_debug.so with DIFFATTN_DEBUG_BUILD=1) for sm_103a if it
    is missing or stale (see builder.py)."""
    from .builder import build_library
    return build_library(force=force, debug=DEBUG_BUILD)


def _check(rc: int):
    if rc != DIFFATTN_OK:
        msg = lib().diffattn_last_error_string().decode(errors="replace")
        raise DiffAttnError(rc, msg)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dev(name, t, dtype=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t


def _code(dtype):
    if dtype == torch.bfloat16:
        return DIFFATTN_BF16
    if dtype == torch.float32:
        return DIFFATTN_FP32
    raise ValueError(f"unsupported dtype {dtype}")


def diffattn_version() -> int:
    return lib().diffattn_version()


def diffattn_device_status(stream=None) -> None:
    """Synchronise `stream` and raise DiffAttnError if a kernel's bounded wait ran out."""
    _check(lib().diffattn_device_status(_stream(stream)))


def diffattn_selftest_wait_timeout(limit_ms: int = 50, stream=None) -> None:
    """Launch the diagnostic kernel whose bounded wait runs out after `limit_ms`; the next
    diffattn_device_status() then raises DiffAttnError with ERR_TIMEOUT (once)."""
    _check(lib().diffattn_selftest_wait_timeout(int(limit_ms), _stream(stream)))


def diffattn_lambda_init(layer: int) -> float:
    return float(lib().diffattn_lambda_init(int(layer)))


def diffattn_lambda(lq1, lk1, lq2, lk2, layer: int, out=None, stream=None):
    """lambda = exp(lq1.lk1) - exp(lq2.lk2) + lambda_init(layer) per row of the [n_sets, dim]
    fp32 vectors; returns a device fp32 tensor [n_sets]."""
    for n, t in (("lq1", lq1), ("lk1", lk1), ("lq2", lq2), ("lk2", lk2)):
        _dev(n, t, torch.float32)
    if not (lq1.shape == lk1.shape == lq2.shape == lk2.shape) or lq1.dim() != 2:
        raise ValueError("lambda vectors must all be [n_sets, dim]")
    n_sets, dim = lq1.shape
    if out is None:
        out = torch.empty(n_sets, dtype=torch.float32, device=lq1.device)
    _dev("out", out, torch.float32)
    _check(lib().diffattn_lambda(_ptr(lq1), _ptr(lk1), _ptr(lq2), _ptr(lk2), dim, n_sets,
                                 int(layer), _ptr(out), _stream(stream)))
    return out


def diffattn_lambda_bwd(lq1, lk1, lq2, lk2, dlam, stream=None):
    """Gradients of lambda with respect to its [n_sets, dim] vectors given dlam (fp32,
    [n_sets * per_set]: each set sums per_set consecutive entries, e.g. the per-head dlambda of
    diffattn_bwd for one lambda per layer). Returns (dlq1, dlk1, dlq2, dlk2)."""
    for n, t in (("lq1", lq1), ("lk1", lk1), ("lq2", lq2), ("lk2", lk2), ("dlam", dlam)):
        _dev(n, t, torch.float32)
    if not (lq1.shape == lk1.shape == lq2.shape == lk2.shape) or lq1.dim() != 2:
        raise ValueError("lambda vectors must all be [n_sets, dim]")
    n_sets, dim = lq1.shape
    if dlam.numel() % n_sets != 0:
        raise ValueError("dlam must hold a whole number of entries per set")
    grads = tuple(torch.empty_like(lq1) for _ in range(4))
    _check(lib().diffattn_lambda_bwd(_ptr(lq1), _ptr(lk1), _ptr(lq2), _ptr(lk2), _ptr(dlam), dim,
                                     n_sets, dlam.numel() // n_sets, *(_ptr(g) for g in grads),
                                     _stream(stream)))
    return grads


def diffattn_fwd(q, k, v, lam, lambda_init: float = 0.0, norm_weight=None, eps: float = 1e-5,
                 causal: bool = True, norm: bool = True, scale: bool = True,
                 cuda_cores: bool = False, single_pass: bool = False, out=None, stream=None):
    """Differential-attention prefill; see include/diffattn.h for the exact semantics."""
    _dev("q", q)
    B, N, H, two_d = q.shape
    d, dv = two_d // 2, v.shape[-1]
    _dev("k", k, q.dtype)
    _dev("v", v, q.dtype)
    if k.shape != q.shape or v.shape[:3] != (B, N, H):
        raise ValueError("k must match q, and v must be [B, N, H, dv]")
    _dev("lam", lam, torch.float32)
    if lam.numel() != H:
        raise ValueError("lam must hold one value per head")
    if norm_weight is not None:
        _dev("norm_weight", norm_weight, torch.float32)
    if out is None:
        out = torch.empty((B, N, H, dv), dtype=q.dtype, device=q.device)
    _dev("out", out, q.dtype)
    flags = ((DIFFATTN_CAUSAL if causal else 0) | (DIFFATTN_NORM if norm else 0)
             | (DIFFATTN_SCALE if scale else 0) | (DIFFATTN_CUDA_CORES if cuda_cores else 0)
             | (DIFFATTN_SINGLE_PASS if single_pass else 0))
    _check(lib().diffattn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lam), float(lambda_init),
                              _ptr(norm_weight), float(eps), B, N, H, d, dv, flags,
                              _code(q.dtype), _stream(stream)))
    return out


def diffattn_decode_workspace_size(B: int, Lmax: int, H: int, d: int = 128, dv: int = 256) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().diffattn_decode_workspace_size(B, Lmax, H, d, dv, ctypes.byref(n)))
    return int(n.value)


def diffattn_decode(q, k_cache, v_cache, lam, lambda_init: float = 0.0, seqlens=None,
                    norm_weight=None, eps: float = 1e-5, norm: bool = True, scale: bool = True,
                    workspace=None, out=None, stream=None):
    """Split-KV decode of one query per sequence against its cache."""
    _dev("q", q, torch.bfloat16)
    B, H, two_d = q.shape
    d = two_d // 2
    _dev("k_cache", k_cache, torch.bfloat16)
    _dev("v_cache", v_cache, torch.bfloat16)
    Lmax, dv = k_cache.shape[1], v_cache.shape[-1]
    if k_cache.shape != (B, Lmax, H, two_d) or v_cache.shape[:3] != (B, Lmax, H):
        raise ValueError("caches must be [B, Lmax, H, 2d] and [B, Lmax, H, dv]")
    _dev("lam", lam, torch.float32)
    if seqlens is not None:
        _dev("seqlens", seqlens, torch.int32)
    if norm_weight is not None:
        _dev("norm_weight", norm_weight, torch.float32)
    need = diffattn_decode_workspace_size(B, Lmax, H, d, dv)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    _dev("workspace", workspace)
    if out is None:
        out = torch.empty((B, H, dv), dtype=torch.bfloat16, device=q.device)
    _dev("out", out, torch.bfloat16)
    flags = (DIFFATTN_NORM if norm else 0) | (DIFFATTN_SCALE if scale else 0)
    _check(lib().diffattn_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(seqlens), _ptr(out),
                                 _ptr(lam), float(lambda_init), _ptr(norm_weight), float(eps), B,
                                 Lmax, H, d, dv, flags, DIFFATTN_BF16, _ptr(workspace),
                                 workspace.numel() * workspace.element_size(), _stream(stream)))
    return out


def diffattn_decode_noalloc(q, k_cache, v_cache, lam, lambda_init: float = 0.0, seqlens=None,
                            norm_weight=None, eps: float = 1e-5, norm: bool = True,
                            scale: bool = True, out=None, stream=None):
    """diffattn_decode for callers that cannot allocate device memory where they decode: the
    split partials go to a scratch array built into the library instead of a workspace. `out`
    must be given by such a caller (otherwise one is allocated here for convenience)."""
    _dev("q", q, torch.bfloat16)
    B, H, two_d = q.shape
    _dev("k_cache", k_cache, torch.bfloat16)
    _dev("v_cache", v_cache, torch.bfloat16)
    Lmax, dv = k_cache.shape[1], v_cache.shape[-1]
    if k_cache.shape != (B, Lmax, H, two_d) or v_cache.shape[:3] != (B, Lmax, H):
        raise ValueError("caches must be [B, Lmax, H, 2d] and [B, Lmax, H, dv]")
    _dev("lam", lam, torch.float32)
    if seqlens is not None:
        _dev("seqlens", seqlens, torch.int32)
    if norm_weight is not None:
        _dev("norm_weight", norm_weight, torch.float32)
    if out is None:
        out = torch.empty((B, H, dv), dtype=torch.bfloat16, device=q.device)
    _dev("out", out, torch.bfloat16)
    flags = (DIFFATTN_NORM if norm else 0) | (DIFFATTN_SCALE if scale else 0)
    _check(lib().diffattn_decode_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(seqlens),
                                         _ptr(out), _ptr(lam), float(lambda_init),
                                         _ptr(norm_weight), float(eps), B, Lmax, H, two_d // 2,
                                         dv, flags, DIFFATTN_BF16, _stream(stream)))
    return out


def diffattn_decode_split_count(B: int, Lmax: int, H: int, noalloc: bool = False):
    """(splits, keys per split) of diffattn_decode (noalloc False) or diffattn_decode_noalloc
    (noalloc True) for B sequences x H heads over Lmax cached keys. Host arithmetic only."""
    s, c = ctypes.c_int(0), ctypes.c_int(0)
    _check(lib().diffattn_decode_split_count(int(B), int(Lmax), int(H), int(bool(noalloc)),
                                             ctypes.byref(s), ctypes.byref(c)))
    return int(s.value), int(c.value)


def diffattn_v2_fwd(q, k, v, lam_logit, causal: bool = True, cuda_cores: bool = False,
                    single_pass: bool = False, exact: bool = False, out=None, stream=None):
    """DIFF V2 pair prefill: attn[2p] - sigmoid(lam_logit) * attn[2p+1] over shared GQA KV.

    By default one flash pass per head (both heads of a pair in one CTA); `exact` takes the
    two-pass kernel that rounds the difference of the maps once; `cuda_cores` the CUDA-core path.
    `single_pass` names the default."""
    _dev("q", q)
    B, N, Hq, d = q.shape
    _dev("k", k, q.dtype)
    _dev("v", v, q.dtype)
    Hkv = k.shape[2]
    if k.shape != (B, N, Hkv, d) or v.shape != k.shape:
        raise ValueError("k and v must be [B, N, Hkv, d]")
    _dev("lam_logit", lam_logit, torch.float32)
    if lam_logit.shape != (B, N, Hq // 2):
        raise ValueError("lam_logit must be [B, N, Hq/2]")
    if out is None:
        out = torch.empty((B, N, Hq // 2, d), dtype=q.dtype, device=q.device)
    _dev("out", out, q.dtype)
    flags = ((DIFFATTN_CAUSAL if causal else 0) | (DIFFATTN_CUDA_CORES if cuda_cores else 0)
             | (DIFFATTN_SINGLE_PASS if single_pass else 0) | (DIFFATTN_EXACT if exact else 0))
    _check(lib().diffattn_v2_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(lam_logit), _ptr(out), B, N, Hq,
                                 Hkv, d, flags, _code(q.dtype), _stream(stream)))
    return out


def diffattn_v2_decode_workspace_size(B: int, Lmax: int, Hq: int, Hkv: int, d: int) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().diffattn_v2_decode_workspace_size(B, Lmax, Hq, Hkv, d, ctypes.byref(n)))
    return n.value


def diffattn_v2_decode(q, k_cache, v_cache, lam_logit, seqlens=None, cuda_cores: bool = False,
                       workspace=None, out=None, stream=None):
    """DIFF V2 decode: one query token per sequence, attn[2p] - sigmoid(lam_logit) * attn[2p+1]
    over the shared GQA cache; q [B, Hq, d], caches [B, Lmax, Hkv, d], lam_logit [B, Hq/2]."""
    _dev("q", q, torch.bfloat16)
    B, Hq, d = q.shape
    _dev("k_cache", k_cache, torch.bfloat16)
    _dev("v_cache", v_cache, torch.bfloat16)
    Lmax, Hkv = k_cache.shape[1], k_cache.shape[2]
    if k_cache.shape != (B, Lmax, Hkv, d) or v_cache.shape != k_cache.shape:
        raise ValueError("caches must both be [B, Lmax, Hkv, d]")
    _dev("lam_logit", lam_logit, torch.float32)
    if lam_logit.shape != (B, Hq // 2):
        raise ValueError("lam_logit must be [B, Hq/2]")
    if seqlens is not None:
        _dev("seqlens", seqlens, torch.int32)
    need = diffattn_v2_decode_workspace_size(B, Lmax, Hq, Hkv, d)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    _dev("workspace", workspace)
    if out is None:
        out = torch.empty((B, Hq // 2, d), dtype=torch.bfloat16, device=q.device)
    _dev("out", out, torch.bfloat16)
    _check(lib().diffattn_v2_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(seqlens),
                                    _ptr(lam_logit), _ptr(out), B, Lmax, Hq, Hkv, d,
                                    DIFFATTN_CUDA_CORES if cuda_cores else 0,
                                    DIFFATTN_BF16, _ptr(workspace),
                                    workspace.numel() * workspace.element_size(), _stream(stream)))
    return out


def diffattn_v2_decode_fp8(q8, k_cache8, v_cache, lam_logit, q_descale: float, k_descale: float,
                           seqlens=None, workspace=None, out=None, stream=None):
    """DIFF V2 decode with fp8 e4m3 q [B, Hq, d] and K cache [B, Lmax, Hkv, d] (real values
    q8 * q_descale, k8 * k_descale) and a bf16 V cache."""
    _dev("q8", q8, torch.float8_e4m3fn)
    B, Hq, d = q8.shape
    _dev("k_cache8", k_cache8, torch.float8_e4m3fn)
    _dev("v_cache", v_cache, torch.bfloat16)
    Lmax, Hkv = k_cache8.shape[1], k_cache8.shape[2]
    if k_cache8.shape != (B, Lmax, Hkv, d) or v_cache.shape != k_cache8.shape:
        raise ValueError("caches must both be [B, Lmax, Hkv, d]")
    _dev("lam_logit", lam_logit, torch.float32)
    if lam_logit.shape != (B, Hq // 2):
        raise ValueError("lam_logit must be [B, Hq/2]")
    if seqlens is not None:
        _dev("seqlens", seqlens, torch.int32)
    if workspace is None:
        workspace = torch.empty(diffattn_v2_decode_workspace_size(B, Lmax, Hq, Hkv, d),
                                dtype=torch.uint8, device=q8.device)
    _dev("workspace", workspace)
    if out is None:
        out = torch.empty((B, Hq // 2, d), dtype=torch.bfloat16, device=q8.device)
    _dev("out", out, torch.bfloat16)
    _check(lib().diffattn_v2_decode_fp8(_ptr(q8), _ptr(k_cache8), _ptr(v_cache), _ptr(seqlens),
                                        _ptr(lam_logit), _ptr(out), float(q_descale),
                                        float(k_descale), B, Lmax, Hq, Hkv, d, 0, _ptr(workspace),
                                        workspace.numel() * workspace.element_size(),
                                        _stream(stream)))
    return out


def diffattn_v2_decode_paged(q, k_pool, v_pool, block_table, seqlens, lam_logit,
                             cuda_cores: bool = False, workspace=None, out=None, stream=None):
    """DIFF V2 decode over a paged cache: pools [num_pages, page_size, Hkv, d], block_table
    [B, max_pages] int32, seqlens [B] int32; q [B, Hq, d], lam_logit [B, Hq/2]."""
    _dev("q", q, torch.bfloat16)
    B, Hq, d = q.shape
    _dev("k_pool", k_pool, torch.bfloat16)
    _dev("v_pool", v_pool, torch.bfloat16)
    num_pages, page_size, Hkv = k_pool.shape[0], k_pool.shape[1], k_pool.shape[2]
    if k_pool.shape != (num_pages, page_size, Hkv, d) or v_pool.shape != k_pool.shape:
        raise ValueError("pools must both be [num_pages, page_size, Hkv, d]")
    _dev("block_table", block_table, torch.int32)
    _dev("seqlens", seqlens, torch.int32)
    if block_table.dim() != 2 or block_table.shape[0] != B or seqlens.shape != (B,):
        raise ValueError("block_table must be [B, max_pages] and seqlens [B]")
    max_pages = block_table.shape[1]
    _dev("lam_logit", lam_logit, torch.float32)
    if lam_logit.shape != (B, Hq // 2):
        raise ValueError("lam_logit must be [B, Hq/2]")
    if workspace is None:
        need = diffattn_v2_decode_workspace_size(B, max_pages * page_size, Hq, Hkv, d)
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    _dev("workspace", workspace)
    if out is None:
        out = torch.empty((B, Hq // 2, d), dtype=torch.bfloat16, device=q.device)
    _dev("out", out, torch.bfloat16)
    _check(lib().diffattn_v2_decode_paged(_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_table),
                                          _ptr(seqlens), _ptr(lam_logit), _ptr(out), B, Hq, Hkv,
                                          d, num_pages, page_size, max_pages,
                                          DIFFATTN_CUDA_CORES if cuda_cores else 0, DIFFATTN_BF16,
                                          _ptr(workspace),
                                          workspace.numel() * workspace.element_size(),
                                          _stream(stream)))
    return out


def _train_flags(causal, norm, scale):
    return ((DIFFATTN_CAUSAL if causal else 0) | (DIFFATTN_NORM if norm else 0)
            | (DIFFATTN_SCALE if scale else 0))


def diffattn_fwd_train(q, k, v, lam, lambda_init: float = 0.0, norm_weight=None, eps: float = 1e-5,
                       causal: bool = True, norm: bool = True, scale: bool = True, stream=None):
    """Forward for training: returns (out, o_pre, stats); o_pre is the head output before the
    norm and scale, stats [B, H, 2, Npad] the per-row base-2 log-sum-exp of each map."""
    _dev("q", q, torch.bfloat16)
    B, N, H, two_d = q.shape
    d = two_d // 2
    _dev("k", k, torch.bfloat16)
    _dev("v", v, torch.bfloat16)
    dv = v.shape[-1]
    _dev("lam", lam, torch.float32)
    if norm_weight is not None:
        _dev("norm_weight", norm_weight, torch.float32)
    out = torch.empty((B, N, H, dv), dtype=torch.bfloat16, device=q.device)
    o_pre = torch.empty_like(out)
    npad = (N + 127) // 128 * 128
    stats = torch.empty((B, H, 2, npad), dtype=torch.float32, device=q.device)
    _check(lib().diffattn_fwd_train(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(o_pre), _ptr(stats),
                                    _ptr(lam), float(lambda_init), _ptr(norm_weight), float(eps),
                                    B, N, H, d, dv, _train_flags(causal, norm, scale),
                                    DIFFATTN_BF16, _stream(stream)))
    return out, o_pre, stats


def diffattn_bwd_workspace_size(B: int, N: int, H: int, d: int, dv: int) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().diffattn_bwd_workspace_size(B, N, H, d, dv, ctypes.byref(n)))
    return n.value


def diffattn_bwd(q, k, v, o_pre, stats, dout, lam, lambda_init: float = 0.0, norm_weight=None,
                 eps: float = 1e-5, causal: bool = True, norm: bool = True, scale: bool = True,
                 workspace=None, grads=None, stream=None):
    """Backward of the V1 prefill. Returns dict(dq, dk, dv, dlam, dw) (dw None without a norm
    weight tensor to differentiate)."""
    _dev("q", q, torch.bfloat16)
    B, N, H, two_d = q.shape
    d = two_d // 2
    dv = v.shape[-1]
    for name, t in (("k", k), ("v", v), ("o_pre", o_pre), ("dout", dout)):
        _dev(name, t, torch.bfloat16)
    _dev("stats", stats, torch.float32)
    _dev("lam", lam, torch.float32)
    if norm_weight is not None:
        _dev("norm_weight", norm_weight, torch.float32)
    if workspace is None:
        workspace = torch.empty(diffattn_bwd_workspace_size(B, N, H, d, dv), dtype=torch.uint8,
                                device=q.device)
    if grads is None:
        grads = dict(dq=torch.empty_like(q), dk=torch.empty_like(k), dv=torch.empty_like(v),
                     dlam=torch.empty((H,), dtype=torch.float32, device=q.device),
                     dw=torch.empty((dv,), dtype=torch.float32, device=q.device))
    _check(lib().diffattn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o_pre), _ptr(stats), _ptr(dout),
                              _ptr(lam), float(lambda_init), _ptr(norm_weight), float(eps),
                              _ptr(grads["dq"]), _ptr(grads["dk"]), _ptr(grads["dv"]),
                              _ptr(grads["dlam"]), _ptr(grads.get("dw")), B, N, H, d, dv,
                              _train_flags(causal, norm, scale), DIFFATTN_BF16, _ptr(workspace),
                              workspace.numel() * workspace.element_size(), _stream(stream)))
    return grads


def _max_seqlen(cu_seqlens, max_seqlen):
    B = cu_seqlens.numel() - 1
    if max_seqlen is None:
        max_seqlen = int((cu_seqlens[1:] - cu_seqlens[:-1]).max().item()) if B > 0 else 1
    return B, max(1, int(max_seqlen))


def diffattn_fwd_train_varlen(q, k, v, cu_seqlens, lam, lambda_init: float = 0.0, max_seqlen=None,
                              norm_weight=None, eps: float = 1e-5, causal: bool = True,
                              norm: bool = True, scale: bool = True, stream=None):
    """Training forward over packed sequences (q, k [total, H, 2d], v [total, H, dv]): returns
    (out, o_pre, stats) with stats [B, H, 2, Npad], Npad the longest sequence rounded up to 128."""
    _dev("q", q, torch.bfloat16)
    total, H, two_d = q.shape
    d = two_d // 2
    _dev("k", k, torch.bfloat16)
    _dev("v", v, torch.bfloat16)
    dv = v.shape[-1]
    _dev("cu_seqlens", cu_seqlens, torch.int32)
    B, N = _max_seqlen(cu_seqlens, max_seqlen)
    _dev("lam", lam, torch.float32)
    if norm_weight is not None:
        _dev("norm_weight", norm_weight, torch.float32)
    out = torch.zeros((total, H, dv), dtype=torch.bfloat16, device=q.device)
    o_pre = torch.zeros_like(out)
    stats = torch.zeros((B, H, 2, (N + 127) // 128 * 128), dtype=torch.float32, device=q.device)
    _check(lib().diffattn_fwd_train_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(o_pre),
                                           _ptr(stats), _ptr(cu_seqlens), N, total, _ptr(lam),
                                           float(lambda_init), _ptr(norm_weight), float(eps), B, H,
                                           d, dv, _train_flags(causal, norm, scale), DIFFATTN_BF16,
                                           _stream(stream)))
    return out, o_pre, stats


def diffattn_bwd_varlen_workspace_size(B: int, max_seqlen: int, total: int, H: int, d: int,
                                       dv: int) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().diffattn_bwd_varlen_workspace_size(B, max_seqlen, total, H, d, dv,
                                                    ctypes.byref(n)))
    return n.value


def diffattn_bwd_varlen(q, k, v, o_pre, stats, dout, cu_seqlens, lam, lambda_init: float = 0.0,
                        max_seqlen=None, norm_weight=None, eps: float = 1e-5, causal: bool = True,
                        norm: bool = True, scale: bool = True, workspace=None, grads=None,
                        stream=None):
    """Backward over packed sequences, from the tensors of diffattn_fwd_train_varlen. Returns
    dict(dq, dk, dv, dlam, dw); rows in no sequence stay zero in the returned tensors."""
    _dev("q", q, torch.bfloat16)
    total, H, two_d = q.shape
    d = two_d // 2
    dv = v.shape[-1]
    for name, t in (("k", k), ("v", v), ("o_pre", o_pre), ("dout", dout)):
        _dev(name, t, torch.bfloat16)
    _dev("stats", stats, torch.float32)
    _dev("cu_seqlens", cu_seqlens, torch.int32)
    B, N = _max_seqlen(cu_seqlens, max_seqlen)
    _dev("lam", lam, torch.float32)
    if norm_weight is not None:
        _dev("norm_weight", norm_weight, torch.float32)
    if workspace is None:
        workspace = torch.empty(diffattn_bwd_varlen_workspace_size(B, N, total, H, d, dv),
                                dtype=torch.uint8, device=q.device)
    if grads is None:
        grads = dict(dq=torch.zeros_like(q), dk=torch.zeros_like(k), dv=torch.zeros_like(v),
                     dlam=torch.empty((H,), dtype=torch.float32, device=q.device),
                     dw=torch.empty((dv,), dtype=torch.float32, device=q.device))
    _check(lib().diffattn_bwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o_pre), _ptr(stats),
                                     _ptr(dout), _ptr(cu_seqlens), N, total, _ptr(lam),
                                     float(lambda_init), _ptr(norm_weight), float(eps),
                                     _ptr(grads["dq"]), _ptr(grads["dk"]), _ptr(grads["dv"]),
                                     _ptr(grads["dlam"]), _ptr(grads.get("dw")), B, H, d, dv,
                                     _train_flags(causal, norm, scale), DIFFATTN_BF16,
                                     _ptr(workspace), workspace.numel() * workspace.element_size(),
                                     _stream(stream)))
    return grads


def diffattn_fwd_fused_lambda(q, k, v, lq1, lk1, lq2, lk2, layer: int, norm_weight=None,
                              eps: float = 1e-5, causal: bool = True, norm: bool = True,
                              scale: bool = True, out=None, stream=None):
    """Prefill with lambda formed in the kernel from the four re-parameterisation vectors
    ([1, dim] for one lambda per layer, or [H, dim]) and the 1-indexed layer."""
    _dev("q", q, torch.bfloat16)
    B, N, H, two_d = q.shape
    d = two_d // 2
    _dev("k", k, torch.bfloat16)
    _dev("v", v, torch.bfloat16)
    dv = v.shape[-1]
    vecs = [lq1, lk1, lq2, lk2]
    for i, t in enumerate(vecs):
        _dev(f"lambda vector {i}", t, torch.float32)
    sets, dim = vecs[0].shape
    if any(t.shape != (sets, dim) for t in vecs):
        raise ValueError("the four lambda vectors must share one shape [sets, dim]")
    if norm_weight is not None:
        _dev("norm_weight", norm_weight, torch.float32)
    if out is None:
        out = torch.empty((B, N, H, dv), dtype=torch.bfloat16, device=q.device)
    _dev("out", out, torch.bfloat16)
    _check(lib().diffattn_fwd_fused_lambda(_ptr(q), _ptr(k), _ptr(v), _ptr(out), *[_ptr(t) for t in vecs],
                                           dim, sets, int(layer), _ptr(norm_weight), float(eps), B, N,
                                           H, d, dv, _train_flags(causal, norm, scale), DIFFATTN_BF16,
                                           _stream(stream)))
    return out


def diffattn_decode_paged(q, k_pool, v_pool, block_table, seqlens, lam, lambda_init: float = 0.0,
                          norm_weight=None, eps: float = 1e-5, norm: bool = True,
                          scale: bool = True, workspace=None, out=None, stream=None):
    """Decode over a paged cache: pools [num_pages, page_size, H, 2d] / [.., dv], block_table
    [B, max_pages] int32, seqlens [B] int32."""
    _dev("q", q, torch.bfloat16)
    B, H, two_d = q.shape
    d = two_d // 2
    _dev("k_pool", k_pool, torch.bfloat16)
    _dev("v_pool", v_pool, torch.bfloat16)
    num_pages, page_size = k_pool.shape[0], k_pool.shape[1]
    dv = v_pool.shape[-1]
    if k_pool.shape != (num_pages, page_size, H, two_d) or v_pool.shape[:3] != (num_pages, page_size, H):
        raise ValueError("pools must be [num_pages, page_size, H, 2d] and [num_pages, page_size, H, dv]")
    _dev("block_table", block_table, torch.int32)
    _dev("seqlens", seqlens, torch.int32)
    max_pages = block_table.shape[1]
    _dev("lam", lam, torch.float32)
    if norm_weight is not None:
        _dev("norm_weight", norm_weight, torch.float32)
    if workspace is None:
        workspace = torch.empty(diffattn_decode_workspace_size(B, max_pages * page_size, H, d, dv),
                                dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty((B, H, dv), dtype=torch.bfloat16, device=q.device)
    _dev("out", out, torch.bfloat16)
    flags = (DIFFATTN_NORM if norm else 0) | (DIFFATTN_SCALE if scale else 0)
    _check(lib().diffattn_decode_paged(_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_table),
                                       _ptr(seqlens), _ptr(out), _ptr(lam), float(lambda_init),
                                       _ptr(norm_weight), float(eps), B, H, d, dv, num_pages,
                                       page_size, max_pages, flags, DIFFATTN_BF16, _ptr(workspace),
                                       workspace.numel() * workspace.element_size(), _stream(stream)))
    return out


def diffattn_fwd_varlen(q, k, v, cu_seqlens, lam, lambda_init: float = 0.0, max_seqlen=None,
                        norm_weight=None, eps: float = 1e-5, causal: bool = True, norm: bool = True,
                        scale: bool = True, out=None, stream=None):
    """Prefill over packed sequences: q, k [total, H, 2d], v [total, H, dv], cu_seqlens int32
    [B + 1] on the device. `max_seqlen` (the longest sequence) is read from cu_seqlens if not
    given (one device-to-host copy)."""
    _dev("q", q, torch.bfloat16)
    total, H, two_d = q.shape
    d = two_d // 2
    _dev("k", k, torch.bfloat16)
    _dev("v", v, torch.bfloat16)
    dv = v.shape[-1]
    _dev("cu_seqlens", cu_seqlens, torch.int32)
    B = cu_seqlens.numel() - 1
    if max_seqlen is None:
        max_seqlen = int((cu_seqlens[1:] - cu_seqlens[:-1]).max().item()) if B > 0 else 1
    _dev("lam", lam, torch.float32)
    if norm_weight is not None:
        _dev("norm_weight", norm_weight, torch.float32)
    if out is None:
        out = torch.zeros((total, H, dv), dtype=torch.bfloat16, device=q.device)
    _dev("out", out, torch.bfloat16)
    _check(lib().diffattn_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(cu_seqlens),
                                     max(1, int(max_seqlen)), total, _ptr(lam), float(lambda_init),
                                     _ptr(norm_weight), float(eps), B, H, d, dv,
                                     _train_flags(causal, norm, scale), DIFFATTN_BF16,
                                     _stream(stream)))
    return out


def diffattn_fwd_varlen_qk(q, k, v, cu_seqlens_q, cu_seqlens_k, lam, lambda_init: float = 0.0,
                           max_seqlen_q=None, max_seqlen_k=None, norm_weight=None,
                           eps: float = 1e-5, causal: bool = True, norm: bool = True,
                           scale: bool = True, out=None, stream=None):
    """Packed prefill where each sequence's Lq queries (q, out [total_q, H, *]) are the last Lq of
    its Lk keys (k, v [total_k, H, *]); cu_seqlens_q and cu_seqlens_k are int32 [B + 1] on the
    device. Missing maxima are read from the offsets (one device-to-host copy each)."""
    _dev("q", q, torch.bfloat16)
    total_q, H, two_d = q.shape
    d = two_d // 2
    _dev("k", k, torch.bfloat16)
    _dev("v", v, torch.bfloat16)
    total_k, dv = k.shape[0], v.shape[-1]
    if k.shape != (total_k, H, two_d) or v.shape[:2] != (total_k, H):
        raise ValueError("k must be [total_k, H, 2d] and v [total_k, H, dv]")
    _dev("cu_seqlens_q", cu_seqlens_q, torch.int32)
    _dev("cu_seqlens_k", cu_seqlens_k, torch.int32)
    B = cu_seqlens_q.numel() - 1
    if cu_seqlens_k.numel() != B + 1:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must both have B + 1 entries")
    if max_seqlen_q is None:
        max_seqlen_q = int((cu_seqlens_q[1:] - cu_seqlens_q[:-1]).max().item()) if B > 0 else 1
    if max_seqlen_k is None:
        max_seqlen_k = int((cu_seqlens_k[1:] - cu_seqlens_k[:-1]).max().item()) if B > 0 else 1
    _dev("lam", lam, torch.float32)
    if norm_weight is not None:
        _dev("norm_weight", norm_weight, torch.float32)
    if out is None:
        out = torch.zeros((total_q, H, dv), dtype=torch.bfloat16, device=q.device)
    _dev("out", out, torch.bfloat16)
    _check(lib().diffattn_fwd_varlen_qk(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(cu_seqlens_q),
                                        _ptr(cu_seqlens_k), max(1, int(max_seqlen_q)),
                                        max(1, int(max_seqlen_k)), total_q, total_k, _ptr(lam),
                                        float(lambda_init), _ptr(norm_weight), float(eps), B, H, d,
                                        dv, _train_flags(causal, norm, scale), DIFFATTN_BF16,
                                        _stream(stream)))
    return out


def diffattn_v2_fwd_varlen(q, k, v, lam_logit, cu_seqlens_q, cu_seqlens_k=None, max_seqlen_q=None,
                           max_seqlen_k=None, causal: bool = True, exact: bool = False, out=None,
                           stream=None):
    """DIFF V2 over packed sequences: q [total_q, Hq, d], k, v [total_k, Hkv, d], lam_logit
    [total_q, Hq/2]; cu_seqlens_k None means the keys share the queries' offsets. `exact` as for
    diffattn_v2_fwd."""
    _dev("q", q, torch.bfloat16)
    total_q, Hq, d = q.shape
    _dev("k", k, torch.bfloat16)
    _dev("v", v, torch.bfloat16)
    total_k, Hkv = k.shape[0], k.shape[1]
    if k.shape != (total_k, Hkv, d) or v.shape != k.shape:
        raise ValueError("k and v must both be [total_k, Hkv, d]")
    _dev("lam_logit", lam_logit, torch.float32)
    if lam_logit.shape != (total_q, Hq // 2):
        raise ValueError("lam_logit must be [total_q, Hq/2]")
    _dev("cu_seqlens_q", cu_seqlens_q, torch.int32)
    B = cu_seqlens_q.numel() - 1
    if max_seqlen_q is None:
        max_seqlen_q = int((cu_seqlens_q[1:] - cu_seqlens_q[:-1]).max().item()) if B > 0 else 1
    if cu_seqlens_k is not None:
        _dev("cu_seqlens_k", cu_seqlens_k, torch.int32)
        if cu_seqlens_k.numel() != B + 1:
            raise ValueError("cu_seqlens_q and cu_seqlens_k must both have B + 1 entries")
        if max_seqlen_k is None:
            max_seqlen_k = int((cu_seqlens_k[1:] - cu_seqlens_k[:-1]).max().item()) if B > 0 else 1
    else:
        max_seqlen_k = max_seqlen_q
    if out is None:
        out = torch.zeros((total_q, Hq // 2, d), dtype=torch.bfloat16, device=q.device)
    _dev("out", out, torch.bfloat16)
    _check(lib().diffattn_v2_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(lam_logit), _ptr(out),
                                        _ptr(cu_seqlens_q), _ptr(cu_seqlens_k),
                                        max(1, int(max_seqlen_q)), max(1, int(max_seqlen_k)),
                                        total_q, total_k, B, Hq, Hkv, d,
                                        (DIFFATTN_CAUSAL if causal else 0) | (DIFFATTN_EXACT if exact else 0),
                                        DIFFATTN_BF16,
                                        _stream(stream)))
    return out


def _paged_args(q, k_pool, v_pool, cu_seqlens_q, seqlens_k, block_table, max_seqlen_q,
                max_seqlen_k):
    _dev("k_pool", k_pool, torch.bfloat16)
    _dev("v_pool", v_pool, torch.bfloat16)
    _dev("cu_seqlens_q", cu_seqlens_q, torch.int32)
    _dev("seqlens_k", seqlens_k, torch.int32)
    _dev("block_table", block_table, torch.int32)
    B = cu_seqlens_q.numel() - 1
    if seqlens_k.shape != (B,) or block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("seqlens_k must be [B] and block_table [B, max_pages]")
    if max_seqlen_q is None:
        max_seqlen_q = int((cu_seqlens_q[1:] - cu_seqlens_q[:-1]).max().item()) if B > 0 else 1
    if max_seqlen_k is None:
        max_seqlen_k = int(seqlens_k.max().item()) if B > 0 else 1
    return B, max(1, int(max_seqlen_q)), max(1, int(max_seqlen_k))


def diffattn_fwd_paged(q, k_pool, v_pool, cu_seqlens_q, seqlens_k, block_table, lam,
                       lambda_init: float = 0.0, max_seqlen_q=None, max_seqlen_k=None,
                       norm_weight=None, eps: float = 1e-5, causal: bool = True,
                       norm: bool = True, scale: bool = True, out=None, stream=None):
    """Packed queries q [total_q, H, 2d] against keys in a page pool: k_pool [num_pages,
    page_size, H, 2d], v_pool [.., H, dv]; sequence b has seqlens_k[b] keys through
    block_table[b] and its queries are the last of those positions."""
    _dev("q", q, torch.bfloat16)
    total_q, H, two_d = q.shape
    d = two_d // 2
    B, mq, mk = _paged_args(q, k_pool, v_pool, cu_seqlens_q, seqlens_k, block_table,
                            max_seqlen_q, max_seqlen_k)
    num_pages, page_size, dv = k_pool.shape[0], k_pool.shape[1], v_pool.shape[-1]
    if k_pool.shape != (num_pages, page_size, H, two_d) or v_pool.shape[:3] != (num_pages, page_size, H):
        raise ValueError("pools must be [num_pages, page_size, H, 2d] and [num_pages, page_size, H, dv]")
    _dev("lam", lam, torch.float32)
    if norm_weight is not None:
        _dev("norm_weight", norm_weight, torch.float32)
    if out is None:
        out = torch.zeros((total_q, H, dv), dtype=torch.bfloat16, device=q.device)
    _dev("out", out, torch.bfloat16)
    _check(lib().diffattn_fwd_paged(_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(out),
                                    _ptr(cu_seqlens_q), _ptr(seqlens_k), _ptr(block_table), mq, mk,
                                    total_q, num_pages, page_size, block_table.shape[1], _ptr(lam),
                                    float(lambda_init), _ptr(norm_weight), float(eps), B, H, d, dv,
                                    _train_flags(causal, norm, scale), DIFFATTN_BF16,
                                    _stream(stream)))
    return out


def diffattn_v2_fwd_paged(q, k_pool, v_pool, lam_logit, cu_seqlens_q, seqlens_k, block_table,
                          max_seqlen_q=None, max_seqlen_k=None, causal: bool = True,
                          exact: bool = False, out=None,
                          stream=None):
    """DIFF V2 with packed queries q [total_q, Hq, d] against keys in a page pool: k_pool,
    v_pool [num_pages, page_size, Hkv, d]; lam_logit [total_q, Hq/2]."""
    _dev("q", q, torch.bfloat16)
    total_q, Hq, d = q.shape
    B, mq, mk = _paged_args(q, k_pool, v_pool, cu_seqlens_q, seqlens_k, block_table,
                            max_seqlen_q, max_seqlen_k)
    num_pages, page_size, Hkv = k_pool.shape[0], k_pool.shape[1], k_pool.shape[2]
    if k_pool.shape != (num_pages, page_size, Hkv, d) or v_pool.shape != k_pool.shape:
        raise ValueError("pools must both be [num_pages, page_size, Hkv, d]")
    _dev("lam_logit", lam_logit, torch.float32)
    if lam_logit.shape != (total_q, Hq // 2):
        raise ValueError("lam_logit must be [total_q, Hq/2]")
    if out is None:
        out = torch.zeros((total_q, Hq // 2, d), dtype=torch.bfloat16, device=q.device)
    _dev("out", out, torch.bfloat16)
    _check(lib().diffattn_v2_fwd_paged(_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(lam_logit),
                                       _ptr(out), _ptr(cu_seqlens_q), _ptr(seqlens_k),
                                       _ptr(block_table), mq, mk, total_q, num_pages, page_size,
                                       block_table.shape[1], B, Hq, Hkv, d,
                                       (DIFFATTN_CAUSAL if causal else 0) | (DIFFATTN_EXACT if exact else 0),
                                       DIFFATTN_BF16,
                                       _stream(stream)))
    return out


def diffattn_fwd_fp8(q8, k8, v, lam, q_descale: float, k_descale: float, lambda_init: float = 0.0,
                     norm_weight=None, eps: float = 1e-5, causal: bool = True, norm: bool = True,
                     scale: bool = True, out=None, stream=None):
    """Prefill with fp8 e4m3 q and k (real values q8 * q_descale, k8 * k_descale) and bf16 v:
    the score products run on the fp8 tensor cores."""
    _dev("q8", q8, torch.float8_e4m3fn)
    B, N, H, two_d = q8.shape
    d = two_d // 2
    _dev("k8", k8, torch.float8_e4m3fn)
    _dev("v", v, torch.bfloat16)
    dv = v.shape[-1]
    _dev("lam", lam, torch.float32)
    if norm_weight is not None:
        _dev("norm_weight", norm_weight, torch.float32)
    if out is None:
        out = torch.empty((B, N, H, dv), dtype=torch.bfloat16, device=v.device)
    _dev("out", out, torch.bfloat16)
    _check(lib().diffattn_fwd_fp8(_ptr(q8), _ptr(k8), _ptr(v), _ptr(out), float(q_descale),
                                  float(k_descale), _ptr(lam), float(lambda_init),
                                  _ptr(norm_weight), float(eps), B, N, H, d, dv,
                                  _train_flags(causal, norm, scale), _stream(stream)))
    return out


def _strided(name, t, dtype=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != 4 or t.stride(-1) != 1:
        raise ValueError(f"{name} must be 4-D [B, N, H, width] with a contiguous last dimension")
    return list(t.stride()[:3])


def diffattn_fwd_strided(q, k, v, lam, lambda_init: float = 0.0, norm_weight=None,
                         eps: float = 1e-5, causal: bool = True, norm: bool = True,
                         scale: bool = True, cuda_cores: bool = False, out=None, stream=None):
    """diffattn_fwd over strided views (e.g. q, k, v = qkv[:, :, 0], qkv[:, :, 1], qkv[:, :, 2]
    of a fused [B, N, 3, H, 2d] projection); `out` may be a strided view too."""
    B, N, H, two_d = q.shape
    d = two_d // 2
    dv = v.shape[-1]
    st = _strided("q", q) + _strided("k", k, q.dtype) + _strided("v", v, q.dtype)
    if out is None:
        out = torch.empty((B, N, H, dv), dtype=q.dtype, device=q.device)
    st += _strided("out", out, q.dtype)
    _dev("lam", lam, torch.float32)
    if norm_weight is not None:
        _dev("norm_weight", norm_weight, torch.float32)
    arr = (ctypes.c_longlong * 12)(*st)
    flags = ((DIFFATTN_CAUSAL if causal else 0) | (DIFFATTN_NORM if norm else 0)
             | (DIFFATTN_SCALE if scale else 0) | (DIFFATTN_CUDA_CORES if cuda_cores else 0))
    _check(lib().diffattn_fwd_strided(_ptr(q), _ptr(k), _ptr(v), _ptr(out), arr, _ptr(lam),
                                      float(lambda_init), _ptr(norm_weight), float(eps), B, N, H,
                                      d, dv, flags, _code(q.dtype), _stream(stream)))
    return out


def diffattn_fwd_host_workspace_size(B: int, N: int, H: int, d: int, dv: int) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().diffattn_fwd_host_workspace_size(B, N, H, d, dv, ctypes.byref(n)))
    return n.value


def diffattn_fwd_host(q, k, v, out, lq1, lk1, lq2, lk2, layer: int, norm_weight=None,
                      eps: float = 1e-5, causal: bool = True, norm: bool = True, scale: bool = True,
                      workspace=None, stream=None):
    """The layer's forward with q, k, v and out in page-locked host memory; copies in and out are
    pipelined against the prefill of other chunks. Returns `out` (filled when the stream is done)."""
    for name, t in (("q", q), ("k", k), ("v", v), ("out", out)):
        if not isinstance(t, torch.Tensor) or t.is_cuda or not t.is_contiguous() or t.dtype != torch.bfloat16:
            raise ValueError(f"{name} must be a contiguous bf16 host tensor")
    B, N, H, two_d = q.shape
    d = two_d // 2
    dv = v.shape[-1]
    vecs = [lq1, lk1, lq2, lk2]
    for i, t in enumerate(vecs):
        _dev(f"lambda vector {i}", t, torch.float32)
    sets, dim = vecs[0].shape
    if norm_weight is not None:
        _dev("norm_weight", norm_weight, torch.float32)
    if workspace is None:
        workspace = torch.empty(diffattn_fwd_host_workspace_size(B, N, H, d, dv), dtype=torch.uint8,
                                device=lq1.device)
    _check(lib().diffattn_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(out), *[_ptr(t) for t in vecs],
                                   dim, sets, int(layer), _ptr(norm_weight), float(eps), B, N, H, d,
                                   dv, _train_flags(causal, norm, scale), _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), _stream(stream)))
    return out


def diffattn_gda_fwd_workspace_size(B: int, N: int, n_signal: int, n_noise: int, d: int = 128,
                                    dv: int = 256) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().diffattn_gda_fwd_workspace_size(B, N, n_signal, n_noise, d, dv, ctypes.byref(n)))
    return int(n.value)


def diffattn_gda_fwd_fp8(q8, k8, v, lam, n_signal: int, q_descale: float, k_descale: float,
                         lambda_init: float = 0.0, norm_weight=None, eps: float = 1e-5,
                         causal: bool = True, norm: bool = True, scale: bool = True, out=None,
                         stream=None):
    """Grouped prefill with fp8 e4m3 q and k (real values q8 * q_descale, k8 * k_descale; the head
    split of diffattn_gda_fwd) and bf16 v [B, N, n_signal, dv]: the score products run on the fp8
    tensor cores."""
    _dev("q8", q8, torch.float8_e4m3fn)
    B, N, heads, d = q8.shape
    n_noise = heads - int(n_signal)
    _dev("k8", k8, torch.float8_e4m3fn)
    _dev("v", v, torch.bfloat16)
    if k8.shape != q8.shape or v.shape[:3] != (B, N, n_signal):
        raise ValueError("k8 must match q8, and v must be [B, N, n_signal, dv]")
    dv = v.shape[-1]
    _dev("lam", lam, torch.float32)
    if norm_weight is not None:
        _dev("norm_weight", norm_weight, torch.float32)
    if out is None:
        out = torch.empty((B, N, int(n_signal), dv), dtype=torch.bfloat16, device=v.device)
    _dev("out", out, torch.bfloat16)
    _check(lib().diffattn_gda_fwd_fp8(_ptr(q8), _ptr(k8), _ptr(v), _ptr(out), float(q_descale),
                                      float(k_descale), _ptr(lam), float(lambda_init),
                                      _ptr(norm_weight), float(eps), B, N, int(n_signal), n_noise,
                                      d, dv, _train_flags(causal, norm, scale), _stream(stream)))
    return out


def diffattn_gda_fwd(q, k, v, lam, n_signal: int, lambda_init: float = 0.0, norm_weight=None,
                     eps: float = 1e-5, causal: bool = True, norm: bool = True, scale: bool = True,
                     cuda_cores: bool = False, single_pass: bool = False, noise_pass: bool = True,
                     workspace=None, out=None, stream=None):
    """Grouped differential-attention prefill: q, k [B, N, n_signal + n_noise, d] (signal heads'
    Q1/K1 first, then the noise heads' Q2/K2), v [B, N, n_signal, dv], lam [n_signal]; signal
    head h subtracts noise head h // (n_signal / n_noise). With `noise_pass` (the default) the
    noise maps' row statistics are computed once per noise head into `workspace` (allocated here
    if not given); without it each signal head recomputes them. See include/diffattn.h."""
    _dev("q", q)
    B, N, heads, d = q.shape
    n_noise = heads - int(n_signal)
    dv = v.shape[-1]
    _dev("k", k, q.dtype)
    _dev("v", v, q.dtype)
    if k.shape != q.shape or v.shape[:3] != (B, N, n_signal):
        raise ValueError("k must match q, and v must be [B, N, n_signal, dv]")
    _dev("lam", lam, torch.float32)
    if lam.numel() != n_signal:
        raise ValueError("lam must hold one value per signal head")
    if norm_weight is not None:
        _dev("norm_weight", norm_weight, torch.float32)
    if out is None:
        out = torch.empty((B, N, n_signal, dv), dtype=q.dtype, device=q.device)
    _dev("out", out, q.dtype)
    flags = ((DIFFATTN_CAUSAL if causal else 0) | (DIFFATTN_NORM if norm else 0)
             | (DIFFATTN_SCALE if scale else 0) | (DIFFATTN_CUDA_CORES if cuda_cores else 0)
             | (DIFFATTN_SINGLE_PASS if single_pass else 0))
    ws_bytes = 0
    if noise_pass:
        need = diffattn_gda_fwd_workspace_size(B, N, int(n_signal), n_noise, d, dv)
        if workspace is None and need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
        if workspace is not None:
            _dev("workspace", workspace)
            ws_bytes = workspace.numel() * workspace.element_size()
    else:
        workspace = None
    _check(lib().diffattn_gda_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lam),
                                  float(lambda_init), _ptr(norm_weight), float(eps), B, N,
                                  int(n_signal), n_noise, d, dv, flags, _code(q.dtype),
                                  _ptr(workspace), ws_bytes, _stream(stream)))
    return out


def diffattn_gda_fwd_varlen(q, k, v, cu_seqlens, lam, n_signal: int, lambda_init: float = 0.0,
                            max_seqlen=None, norm_weight=None, eps: float = 1e-5,
                            causal: bool = True, norm: bool = True, scale: bool = True,
                            noise_pass: bool = True, workspace=None, out=None, stream=None):
    """Grouped prefill over packed sequences: q, k [total, n_signal + n_noise, d], v
    [total, n_signal, dv], cu_seqlens int32 [B + 1] on the device. `max_seqlen` is read from
    cu_seqlens if not given (one device-to-host copy); the workspace is sized for B sequences of
    max_seqlen rows."""
    _dev("q", q, torch.bfloat16)
    total, heads, d = q.shape
    n_noise = heads - int(n_signal)
    dv = v.shape[-1]
    _dev("k", k, torch.bfloat16)
    _dev("v", v, torch.bfloat16)
    if k.shape != q.shape or v.shape[:2] != (total, n_signal):
        raise ValueError("k must match q, and v must be [total, n_signal, dv]")
    _dev("cu_seqlens", cu_seqlens, torch.int32)
    B = cu_seqlens.numel() - 1
    if max_seqlen is None:
        max_seqlen = int((cu_seqlens[1:] - cu_seqlens[:-1]).max().item()) if B > 0 else 1
    max_seqlen = max(1, int(max_seqlen))
    _dev("lam", lam, torch.float32)
    if lam.numel() != n_signal:
        raise ValueError("lam must hold one value per signal head")
    if norm_weight is not None:
        _dev("norm_weight", norm_weight, torch.float32)
    if out is None:
        out = torch.zeros((total, n_signal, dv), dtype=torch.bfloat16, device=q.device)
    _dev("out", out, torch.bfloat16)
    ws_bytes = 0
    if noise_pass:
        need = diffattn_gda_fwd_workspace_size(max(1, B), max_seqlen, int(n_signal), n_noise, d, dv)
        if workspace is None and need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
        if workspace is not None:
            _dev("workspace", workspace)
            ws_bytes = workspace.numel() * workspace.element_size()
    else:
        workspace = None
    _check(lib().diffattn_gda_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(cu_seqlens),
                                         max_seqlen, total, _ptr(lam), float(lambda_init),
                                         _ptr(norm_weight), float(eps), B, int(n_signal), n_noise,
                                         d, dv, _train_flags(causal, norm, scale), DIFFATTN_BF16,
                                         _ptr(workspace), ws_bytes, _stream(stream)))
    return out


def _gda_ws(noise_pass, workspace, B, max_seqlen, n_signal, n_noise, d, dv, device):
    """The two-launch form's workspace (allocated here if not given), or none."""
    if not noise_pass:
        return None, 0
    need = diffattn_gda_fwd_workspace_size(max(1, B), max_seqlen, int(n_signal), n_noise, d, dv)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=device)
    if workspace is None:
        return None, 0
    _dev("workspace", workspace)
    return workspace, workspace.numel() * workspace.element_size()


def diffattn_gda_fwd_varlen_qk(q, k, v, cu_seqlens_q, cu_seqlens_k, lam, n_signal: int,
                               lambda_init: float = 0.0, max_seqlen_q=None, max_seqlen_k=None,
                               norm_weight=None, eps: float = 1e-5, causal: bool = True,
                               norm: bool = True, scale: bool = True, noise_pass: bool = True,
                               workspace=None, out=None, stream=None):
    """Grouped prefill with each sequence's queries at the end of its keys: q [total_q,
    n_signal + n_noise, d], k [total_k, n_signal + n_noise, d], v [total_k, n_signal, dv],
    cu_seqlens_q / cu_seqlens_k int32 [B + 1] on the device."""
    _dev("q", q, torch.bfloat16)
    total_q, heads, d = q.shape
    n_noise = heads - int(n_signal)
    _dev("k", k, torch.bfloat16)
    _dev("v", v, torch.bfloat16)
    total_k, dv = k.shape[0], v.shape[-1]
    if k.shape != (total_k, heads, d) or v.shape[:2] != (total_k, n_signal):
        raise ValueError("k must be [total_k, n_signal + n_noise, d] and v [total_k, n_signal, dv]")
    _dev("cu_seqlens_q", cu_seqlens_q, torch.int32)
    _dev("cu_seqlens_k", cu_seqlens_k, torch.int32)
    B = cu_seqlens_q.numel() - 1
    if max_seqlen_q is None:
        max_seqlen_q = int((cu_seqlens_q[1:] - cu_seqlens_q[:-1]).max().item()) if B > 0 else 1
    if max_seqlen_k is None:
        max_seqlen_k = int((cu_seqlens_k[1:] - cu_seqlens_k[:-1]).max().item()) if B > 0 else 1
    mq, mk = max(1, int(max_seqlen_q)), max(1, int(max_seqlen_k))
    _dev("lam", lam, torch.float32)
    if norm_weight is not None:
        _dev("norm_weight", norm_weight, torch.float32)
    if out is None:
        out = torch.zeros((total_q, int(n_signal), dv), dtype=torch.bfloat16, device=q.device)
    _dev("out", out, torch.bfloat16)
    workspace, ws_bytes = _gda_ws(noise_pass, workspace, B, mq, n_signal, n_noise, d, dv, q.device)
    _check(lib().diffattn_gda_fwd_varlen_qk(_ptr(q), _ptr(k), _ptr(v), _ptr(out),
                                            _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), mq, mk,
                                            total_q, total_k, _ptr(lam), float(lambda_init),
                                            _ptr(norm_weight), float(eps), B, int(n_signal),
                                            n_noise, d, dv, _train_flags(causal, norm, scale),
                                            DIFFATTN_BF16, _ptr(workspace), ws_bytes,
                                            _stream(stream)))
    return out


def diffattn_gda_fwd_paged(q, k_pool, v_pool, cu_seqlens_q, seqlens_k, block_table, lam,
                           n_signal: int, lambda_init: float = 0.0, max_seqlen_q=None,
                           max_seqlen_k=None, norm_weight=None, eps: float = 1e-5,
                           causal: bool = True, norm: bool = True, scale: bool = True,
                           noise_pass: bool = True, workspace=None, out=None, stream=None):
    """Grouped prefill of packed queries q [total_q, n_signal + n_noise, d] against keys in page
    pools k_pool [num_pages, page_size, n_signal + n_noise, d], v_pool [.., n_signal, dv];
    sequence b has seqlens_k[b] keys through block_table[b] and its queries are the last of those
    positions."""
    _dev("q", q, torch.bfloat16)
    total_q, heads, d = q.shape
    n_noise = heads - int(n_signal)
    B, mq, mk = _paged_args(q, k_pool, v_pool, cu_seqlens_q, seqlens_k, block_table,
                            max_seqlen_q, max_seqlen_k)
    num_pages, page_size, dv = k_pool.shape[0], k_pool.shape[1], v_pool.shape[-1]
    if (k_pool.shape != (num_pages, page_size, heads, d)
            or v_pool.shape[:3] != (num_pages, page_size, n_signal)):
        raise ValueError("pools must be [num_pages, page_size, n_signal + n_noise, d] and "
                         "[num_pages, page_size, n_signal, dv]")
    _dev("lam", lam, torch.float32)
    if norm_weight is not None:
        _dev("norm_weight", norm_weight, torch.float32)
    if out is None:
        out = torch.zeros((total_q, int(n_signal), dv), dtype=torch.bfloat16, device=q.device)
    _dev("out", out, torch.bfloat16)
    workspace, ws_bytes = _gda_ws(noise_pass, workspace, B, mq, n_signal, n_noise, d, dv, q.device)
    _check(lib().diffattn_gda_fwd_paged(_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(out),
                                        _ptr(cu_seqlens_q), _ptr(seqlens_k), _ptr(block_table), mq,
                                        mk, total_q, num_pages, page_size, block_table.shape[1],
                                        _ptr(lam), float(lambda_init), _ptr(norm_weight),
                                        float(eps), B, int(n_signal), n_noise, d, dv,
                                        _train_flags(causal, norm, scale), DIFFATTN_BF16,
                                        _ptr(workspace), ws_bytes, _stream(stream)))
    return out


def diffattn_gda_fwd_train(q, k, v, lam, n_signal: int, lambda_init: float = 0.0,
                           norm_weight=None, eps: float = 1e-5, causal: bool = True,
                           norm: bool = True, scale: bool = True, noise_pass: bool = True,
                           workspace=None, stream=None):
    """Grouped forward for training: returns (out, o_pre, stats); o_pre [B, N, n_signal, dv] is
    each signal head's output before the norm and scale, stats [B, n_signal, 2, Npad] the per-row
    base-2 log-sum-exp of each map."""
    _dev("q", q, torch.bfloat16)
    B, N, heads, d = q.shape
    n_noise = heads - int(n_signal)
    _dev("k", k, torch.bfloat16)
    _dev("v", v, torch.bfloat16)
    dv = v.shape[-1]
    _dev("lam", lam, torch.float32)
    if norm_weight is not None:
        _dev("norm_weight", norm_weight, torch.float32)
    out = torch.empty((B, N, int(n_signal), dv), dtype=torch.bfloat16, device=q.device)
    o_pre = torch.empty_like(out)
    npad = (N + 127) // 128 * 128
    stats = torch.empty((B, int(n_signal), 2, npad), dtype=torch.float32, device=q.device)
    workspace, ws_bytes = _gda_ws(noise_pass, workspace, B, N, n_signal, n_noise, d, dv, q.device)
    _check(lib().diffattn_gda_fwd_train(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(o_pre),
                                        _ptr(stats), _ptr(lam), float(lambda_init),
                                        _ptr(norm_weight), float(eps), B, N, int(n_signal),
                                        n_noise, d, dv, _train_flags(causal, norm, scale),
                                        DIFFATTN_BF16, _ptr(workspace), ws_bytes, _stream(stream)))
    return out, o_pre, stats


def diffattn_gda_bwd_workspace_size(B: int, N: int, n_signal: int, n_noise: int, d: int = 128,
                                    dv: int = 256) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().diffattn_gda_bwd_workspace_size(B, N, n_signal, n_noise, d, dv, ctypes.byref(n)))
    return n.value


def diffattn_gda_bwd(q, k, v, o_pre, stats, dout, lam, n_signal: int, lambda_init: float = 0.0,
                     norm_weight=None, eps: float = 1e-5, causal: bool = True, norm: bool = True,
                     scale: bool = True, workspace=None, grads=None, stream=None):
    """Backward of the grouped prefill. Returns dict(dq, dk [B, N, n_signal + n_noise, d], dv,
    dlam [n_signal], dw)."""
    _dev("q", q, torch.bfloat16)
    B, N, heads, d = q.shape
    n_noise = heads - int(n_signal)
    dv = v.shape[-1]
    for name, t in (("k", k), ("v", v), ("o_pre", o_pre), ("dout", dout)):
        _dev(name, t, torch.bfloat16)
    _dev("stats", stats, torch.float32)
    _dev("lam", lam, torch.float32)
    if norm_weight is not None:
        _dev("norm_weight", norm_weight, torch.float32)
    if workspace is None:
        workspace = torch.empty(diffattn_gda_bwd_workspace_size(B, N, int(n_signal), n_noise, d, dv),
                                dtype=torch.uint8, device=q.device)
    if grads is None:
        grads = dict(dq=torch.empty_like(q), dk=torch.empty_like(k), dv=torch.empty_like(v),
                     dlam=torch.empty((int(n_signal),), dtype=torch.float32, device=q.device),
                     dw=torch.empty((dv,), dtype=torch.float32, device=q.device))
    _check(lib().diffattn_gda_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o_pre), _ptr(stats), _ptr(dout),
                                  _ptr(lam), float(lambda_init), _ptr(norm_weight), float(eps),
                                  _ptr(grads["dq"]), _ptr(grads["dk"]), _ptr(grads["dv"]),
                                  _ptr(grads["dlam"]), _ptr(grads.get("dw")), B, N, int(n_signal),
                                  n_noise, d, dv, _train_flags(causal, norm, scale), DIFFATTN_BF16,
                                  _ptr(workspace), workspace.numel() * workspace.element_size(),
                                  _stream(stream)))
    return grads


def diffattn_gda_fwd_train_varlen(q, k, v, cu_seqlens, lam, n_signal: int, lambda_init: float = 0.0,
                                  max_seqlen=None, norm_weight=None, eps: float = 1e-5,
                                  causal: bool = True, norm: bool = True, scale: bool = True,
                                  noise_pass: bool = True, workspace=None, stream=None):
    """Grouped training forward over packed sequences (q, k [total, n_signal + n_noise, d],
    v [total, n_signal, dv]): returns (out, o_pre, stats) with stats [B, n_signal, 2, Npad],
    Npad the longest sequence rounded up to 128."""
    _dev("q", q, torch.bfloat16)
    total, heads, d = q.shape
    n_noise = heads - int(n_signal)
    _dev("k", k, torch.bfloat16)
    _dev("v", v, torch.bfloat16)
    dv = v.shape[-1]
    _dev("cu_seqlens", cu_seqlens, torch.int32)
    B, N = _max_seqlen(cu_seqlens, max_seqlen)
    _dev("lam", lam, torch.float32)
    if norm_weight is not None:
        _dev("norm_weight", norm_weight, torch.float32)
    out = torch.zeros((total, int(n_signal), dv), dtype=torch.bfloat16, device=q.device)
    o_pre = torch.zeros_like(out)
    stats = torch.zeros((B, int(n_signal), 2, (N + 127) // 128 * 128), dtype=torch.float32,
                        device=q.device)
    workspace, ws_bytes = _gda_ws(noise_pass, workspace, B, N, n_signal, n_noise, d, dv, q.device)
    _check(lib().diffattn_gda_fwd_train_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(o_pre),
                                               _ptr(stats), _ptr(cu_seqlens), N, total, _ptr(lam),
                                               float(lambda_init), _ptr(norm_weight), float(eps), B,
                                               int(n_signal), n_noise, d, dv,
                                               _train_flags(causal, norm, scale), DIFFATTN_BF16,
                                               _ptr(workspace), ws_bytes, _stream(stream)))
    return out, o_pre, stats


def diffattn_gda_bwd_varlen_workspace_size(B: int, max_seqlen: int, total: int, n_signal: int,
                                           n_noise: int, d: int = 128, dv: int = 256) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().diffattn_gda_bwd_varlen_workspace_size(B, max_seqlen, total, n_signal, n_noise,
                                                        d, dv, ctypes.byref(n)))
    return n.value


def diffattn_gda_bwd_varlen(q, k, v, o_pre, stats, dout, cu_seqlens, lam, n_signal: int,
                            lambda_init: float = 0.0, max_seqlen=None, norm_weight=None,
                            eps: float = 1e-5, causal: bool = True, norm: bool = True,
                            scale: bool = True, workspace=None, grads=None, stream=None):
    """Grouped backward over packed sequences, from the tensors of diffattn_gda_fwd_train_varlen.
    Returns dict(dq, dk [total, n_signal + n_noise, d], dv, dlam [n_signal], dw); rows in no
    sequence stay zero in the returned tensors."""
    _dev("q", q, torch.bfloat16)
    total, heads, d = q.shape
    n_noise = heads - int(n_signal)
    dv = v.shape[-1]
    for name, t in (("k", k), ("v", v), ("o_pre", o_pre), ("dout", dout)):
        _dev(name, t, torch.bfloat16)
    _dev("stats", stats, torch.float32)
    _dev("cu_seqlens", cu_seqlens, torch.int32)
    B, N = _max_seqlen(cu_seqlens, max_seqlen)
    _dev("lam", lam, torch.float32)
    if norm_weight is not None:
        _dev("norm_weight", norm_weight, torch.float32)
    if workspace is None:
        workspace = torch.empty(diffattn_gda_bwd_varlen_workspace_size(B, N, total, int(n_signal),
                                                                       n_noise, d, dv),
                                dtype=torch.uint8, device=q.device)
    if grads is None:
        grads = dict(dq=torch.zeros_like(q), dk=torch.zeros_like(k), dv=torch.zeros_like(v),
                     dlam=torch.empty((int(n_signal),), dtype=torch.float32, device=q.device),
                     dw=torch.empty((dv,), dtype=torch.float32, device=q.device))
    _check(lib().diffattn_gda_bwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o_pre), _ptr(stats),
                                         _ptr(dout), _ptr(cu_seqlens), N, total, _ptr(lam),
                                         float(lambda_init), _ptr(norm_weight), float(eps),
                                         _ptr(grads["dq"]), _ptr(grads["dk"]), _ptr(grads["dv"]),
                                         _ptr(grads["dlam"]), _ptr(grads.get("dw")), B,
                                         int(n_signal), n_noise, d, dv,
                                         _train_flags(causal, norm, scale), DIFFATTN_BF16,
                                         _ptr(workspace), workspace.numel() * workspace.element_size(),
                                         _stream(stream)))
    return grads


def diffattn_gda_decode(q, k_cache, v_cache, lam, n_signal: int, lambda_init: float = 0.0,
                        seqlens=None, norm_weight=None, eps: float = 1e-5, norm: bool = True,
                        scale: bool = True, workspace=None, out=None, stream=None):
    """Grouped decode: q [B, n_signal + n_noise, d], k_cache [B, Lmax, n_signal + n_noise, d],
    v_cache [B, Lmax, n_signal, dv], lam [n_signal]; returns [B, n_signal, dv]."""
    _dev("q", q, torch.bfloat16)
    B, heads, d = q.shape
    n_noise = heads - int(n_signal)
    _dev("k_cache", k_cache, torch.bfloat16)
    _dev("v_cache", v_cache, torch.bfloat16)
    Lmax, dv = k_cache.shape[1], v_cache.shape[-1]
    if k_cache.shape != (B, Lmax, heads, d) or v_cache.shape[:3] != (B, Lmax, n_signal):
        raise ValueError("caches must be [B, Lmax, n_signal + n_noise, d] and "
                         "[B, Lmax, n_signal, dv]")
    _dev("lam", lam, torch.float32)
    if seqlens is not None:
        _dev("seqlens", seqlens, torch.int32)
    if norm_weight is not None:
        _dev("norm_weight", norm_weight, torch.float32)
    need = diffattn_decode_workspace_size(B, Lmax, int(n_signal), d, dv)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    _dev("workspace", workspace)
    if out is None:
        out = torch.empty((B, n_signal, dv), dtype=torch.bfloat16, device=q.device)
    _dev("out", out, torch.bfloat16)
    flags = (DIFFATTN_NORM if norm else 0) | (DIFFATTN_SCALE if scale else 0)
    _check(lib().diffattn_gda_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(seqlens),
                                     _ptr(out), _ptr(lam), float(lambda_init), _ptr(norm_weight),
                                     float(eps), B, Lmax, int(n_signal), n_noise, d, dv, flags,
                                     DIFFATTN_BF16, _ptr(workspace),
                                     workspace.numel() * workspace.element_size(), _stream(stream)))
    return out


def diffattn_gda_decode_paged(q, k_pool, v_pool, block_table, seqlens, lam, n_signal: int,
                              lambda_init: float = 0.0, norm_weight=None, eps: float = 1e-5,
                              norm: bool = True, scale: bool = True, workspace=None, out=None,
                              stream=None):
    """Grouped decode over a paged cache: q [B, n_signal + n_noise, d], pools
    [num_pages, page_size, n_signal + n_noise, d] and [num_pages, page_size, n_signal, dv],
    block_table [B, max_pages] int32, seqlens [B] int32; returns [B, n_signal, dv]."""
    _dev("q", q, torch.bfloat16)
    B, heads, d = q.shape
    n_noise = heads - int(n_signal)
    _dev("k_pool", k_pool, torch.bfloat16)
    _dev("v_pool", v_pool, torch.bfloat16)
    num_pages, page_size = k_pool.shape[0], k_pool.shape[1]
    dv = v_pool.shape[-1]
    if (k_pool.shape != (num_pages, page_size, heads, d)
            or v_pool.shape[:3] != (num_pages, page_size, n_signal)):
        raise ValueError("pools must be [num_pages, page_size, n_signal + n_noise, d] and "
                         "[num_pages, page_size, n_signal, dv]")
    _dev("block_table", block_table, torch.int32)
    _dev("seqlens", seqlens, torch.int32)
    max_pages = block_table.shape[1]
    _dev("lam", lam, torch.float32)
    if norm_weight is not None:
        _dev("norm_weight", norm_weight, torch.float32)
    if workspace is None:
        workspace = torch.empty(diffattn_decode_workspace_size(B, max_pages * page_size,
                                                               int(n_signal), d, dv),
                                dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty((B, int(n_signal), dv), dtype=torch.bfloat16, device=q.device)
    _dev("out", out, torch.bfloat16)
    flags = (DIFFATTN_NORM if norm else 0) | (DIFFATTN_SCALE if scale else 0)
    _check(lib().diffattn_gda_decode_paged(_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_table),
                                           _ptr(seqlens), _ptr(out), _ptr(lam), float(lambda_init),
                                           _ptr(norm_weight), float(eps), B, int(n_signal), n_noise,
                                           d, dv, num_pages, page_size, max_pages, flags,
                                           DIFFATTN_BF16, _ptr(workspace),
                                           workspace.numel() * workspace.element_size(),
                                           _stream(stream)))
    return out


def diffattn_v2_decode_fp8_paged(q8, k_pool8, v_pool, block_table, seqlens, lam_logit,
                                 q_descale: float, k_descale: float, workspace=None, out=None,
                                 stream=None):
    """DIFF V2 decode with fp8 e4m3 q [B, Hq, d] and K pool [num_pages, page_size, Hkv, d] (real
    values q8 * q_descale, k8 * k_descale), a bf16 V pool, block_table [B, max_pages] and seqlens
    [B] int32; page_size a multiple of 128."""
    _dev("q8", q8, torch.float8_e4m3fn)
    B, Hq, d = q8.shape
    _dev("k_pool8", k_pool8, torch.float8_e4m3fn)
    _dev("v_pool", v_pool, torch.bfloat16)
    num_pages, page_size, Hkv = k_pool8.shape[0], k_pool8.shape[1], k_pool8.shape[2]
    if k_pool8.shape != (num_pages, page_size, Hkv, d) or v_pool.shape != k_pool8.shape:
        raise ValueError("pools must both be [num_pages, page_size, Hkv, d]")
    _dev("block_table", block_table, torch.int32)
    _dev("seqlens", seqlens, torch.int32)
    if block_table.dim() != 2 or block_table.shape[0] != B or seqlens.shape != (B,):
        raise ValueError("block_table must be [B, max_pages] and seqlens [B]")
    max_pages = block_table.shape[1]
    _dev("lam_logit", lam_logit, torch.float32)
    if lam_logit.shape != (B, Hq // 2):
        raise ValueError("lam_logit must be [B, Hq/2]")
    if workspace is None:
        workspace = torch.empty(diffattn_v2_decode_workspace_size(B, max_pages * page_size, Hq,
                                                                  Hkv, d),
                                dtype=torch.uint8, device=q8.device)
    _dev("workspace", workspace)
    if out is None:
        out = torch.empty((B, Hq // 2, d), dtype=torch.bfloat16, device=q8.device)
    _dev("out", out, torch.bfloat16)
    _check(lib().diffattn_v2_decode_fp8_paged(
        _ptr(q8), _ptr(k_pool8), _ptr(v_pool), _ptr(block_table), _ptr(seqlens), _ptr(lam_logit),
        _ptr(out), float(q_descale), float(k_descale), B, Hq, Hkv, d, num_pages, page_size,
        max_pages, 0, _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)))
    return out
