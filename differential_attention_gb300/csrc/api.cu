// api.cu -- the extern "C" entry points declared in include/diffattn.h: argument validation,
// error reporting and dispatch to the kernels. No arithmetic of the operator happens here.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <string>

#include "diffattn.h"
#include "internal.h"

namespace {

thread_local std::string t_err;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_err = buf;
  return code;
}

int ok() {
  t_err.clear();
  return DIFFATTN_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int cuda_fail(cudaError_t e, const char* what) {
  return fail(DIFFATTN_ERR_CUDA, "%s: %s (%d)", what, cudaGetErrorString(e), static_cast<int>(e));
}

// The kernels are built for sm_103a only.
int check_device() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  int major = 0, minor = 0;
  e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
  if (major != 10 || minor != 3)
    return fail(DIFFATTN_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a",
                dev, major, minor);
  return DIFFATTN_OK;
}

constexpr int kPrefillFlags =
    DIFFATTN_CAUSAL | DIFFATTN_NORM | DIFFATTN_SCALE | DIFFATTN_CUDA_CORES | DIFFATTN_SINGLE_PASS;

}  // namespace

constexpr int DEV_BAD_INDEX_BIT = 2;  // the kernels' DEV_BAD_INDEX status bit
constexpr int DEV_BOUNDS_BIT = 4;     // DEV_BOUNDS: a debug-build bounds check failed

extern "C" {

DIFFATTN_API int diffattn_version(void) { return 1 * 10000 + 0 * 100 + 0; }

DIFFATTN_API const char* diffattn_last_error_string(void) { return t_err.c_str(); }

DIFFATTN_API int diffattn_device_status(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int v = 0, w = 0, x = 0, y = 0, z = 0;
  e = da::status_prefill_tc(&v);
  if (e == cudaSuccess) e = da::status_prefill_exact(&w);
  int pv = 0;
  if (e == cudaSuccess) e = da::status_prefill_v2(&pv);
  w |= pv;
  if (e == cudaSuccess) e = da::status_simt(&x);
  if (e == cudaSuccess) e = da::status_v2_decode_tc(&y);
  if (e == cudaSuccess) e = da::status_backward(&z);
  int dd = 0;
  if (e == cudaSuccess) e = da::status_decode(&dd);
  if (e != cudaSuccess) return cuda_fail(e, "reading the device status word");
  v |= w | x | y | z | dd;
  if (v & DEV_BOUNDS_BIT)
    return fail(DIFFATTN_ERR_INDEX,
                "a debug-build bounds check failed: a tile coordinate or row index was outside "
                "its tensor (status %d)", v);
  if (v & DEV_BAD_INDEX_BIT)
    return fail(DIFFATTN_ERR_INDEX, "a block-table entry was outside [0, num_pages) (status %d)", v);
  if (v != 0) return fail(DIFFATTN_ERR_TIMEOUT, "a bounded wait inside a kernel ran out (status %d)", v);
  return ok();
}

DIFFATTN_API int diffattn_selftest_wait_timeout(int limit_ms, void* stream) {
  if (limit_ms < 1 || limit_ms > 2000)
    return fail(DIFFATTN_ERR_ARG, "diffattn_selftest_wait_timeout: limit_ms must be in [1, 2000]");
  int rc = check_device();
  if (rc) return rc;
  cudaError_t e = da::launch_wait_timeout(limit_ms, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "diffattn_selftest_wait_timeout launch");
  return ok();
}

DIFFATTN_API float diffattn_lambda_init(int layer) {
  if (layer < 1) return NAN;
  return static_cast<float>(0.8 - 0.6 * std::exp(-0.3 * (layer - 1)));
}

DIFFATTN_API int diffattn_lambda(const float* lq1, const float* lk1, const float* lq2,
                                 const float* lk2, int dim, int n_sets, int layer,
                                 float* lambda_out, void* stream) {
  if (!lq1 || !lk1 || !lq2 || !lk2 || !lambda_out)
    return fail(DIFFATTN_ERR_ARG, "diffattn_lambda: null pointer");
  if (layer < 1) return fail(DIFFATTN_ERR_ARG, "diffattn_lambda: layer must be >= 1 (got %d)", layer);
  if (dim < 1 || dim > 4096 || n_sets < 1)
    return fail(DIFFATTN_ERR_SHAPE, "diffattn_lambda: need 1 <= dim <= 4096 and n_sets >= 1");
  if (!aligned(lq1, 4) || !aligned(lk1, 4) || !aligned(lq2, 4) || !aligned(lk2, 4) ||
      !aligned(lambda_out, 4))
    return fail(DIFFATTN_ERR_ALIGN, "diffattn_lambda: fp32 pointers must be 4-byte aligned");
  int rc = check_device();
  if (rc) return rc;
  cudaError_t e = da::launch_lambda(lq1, lk1, lq2, lk2, dim, n_sets, diffattn_lambda_init(layer),
                                    lambda_out, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "diffattn_lambda launch");
  return ok();
}

DIFFATTN_API int diffattn_lambda_bwd(const float* lq1, const float* lk1, const float* lq2,
                                     const float* lk2, const float* dlambda, int dim, int n_sets,
                                     int per_set, float* dlq1, float* dlk1, float* dlq2,
                                     float* dlk2, void* stream) {
  const char* fn = "diffattn_lambda_bwd";
  if (!lq1 || !lk1 || !lq2 || !lk2 || !dlambda || !dlq1 || !dlk1 || !dlq2 || !dlk2)
    return fail(DIFFATTN_ERR_ARG, "%s: null pointer", fn);
  if (dim < 1 || dim > 4096 || n_sets < 1 || per_set < 1 ||
      static_cast<long long>(n_sets) * per_set > (1LL << 24))
    return fail(DIFFATTN_ERR_SHAPE, "%s: need 1 <= dim <= 4096, n_sets >= 1 and per_set >= 1", fn);
  for (const void* ptr : {static_cast<const void*>(lq1), static_cast<const void*>(lk1),
                          static_cast<const void*>(lq2), static_cast<const void*>(lk2),
                          static_cast<const void*>(dlambda), static_cast<const void*>(dlq1),
                          static_cast<const void*>(dlk1), static_cast<const void*>(dlq2),
                          static_cast<const void*>(dlk2)})
    if (!aligned(ptr, 4)) return fail(DIFFATTN_ERR_ALIGN, "%s: fp32 pointers must be 4-byte aligned", fn);
  int rc = check_device();
  if (rc) return rc;
  cudaError_t e = da::launch_lambda_bwd(lq1, lk1, lq2, lk2, dlambda, dim, n_sets, per_set, dlq1,
                                        dlk1, dlq2, dlk2, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "diffattn_lambda_bwd launch");
  return ok();
}

static int run_prefill(da::Problem& p, int dtype, const char* name, cudaStream_t s) {
  da::fill_dense_strides(p);
  const bool simt = (p.flags & DIFFATTN_CUDA_CORES) || dtype == DIFFATTN_FP32;
  if ((p.flags & DIFFATTN_SINGLE_PASS) && !simt && !da::dense_strides(p))
    return fail(DIFFATTN_ERR_UNSUPPORTED, "%s: DIFFATTN_SINGLE_PASS needs dense tensors", name);
  if (simt) {
    cudaError_t e = da::launch_prefill_simt(p, dtype == DIFFATTN_BF16, s);
    if (e != cudaSuccess) return cuda_fail(e, name);
    return ok();
  }
  char err[256] = {0};
  cudaError_t e = (p.flags & DIFFATTN_SINGLE_PASS) ? da::launch_prefill_tc(p, s, err, sizeof(err))
                                                   : da::launch_prefill_exact(p, s, err, sizeof(err));
  if (e == cudaErrorNotSupported)
    return fail(DIFFATTN_ERR_SHAPE, "%s: no tensor-core kernel for dqk=%d dv=%d", name, p.dqk, p.dv);
  if (err[0]) return fail(DIFFATTN_ERR_CUDA, "%s: %s", name, err);
  if (e != cudaSuccess) return cuda_fail(e, name);
  return ok();
}

// V2 pair prefill: one flash pass per head, both heads of a pair in one CTA
static int run_v2_pair(da::Problem& p, const char* name, cudaStream_t s) {
  char err[256] = {0};
  cudaError_t e = da::launch_prefill_v2(p, s, err, sizeof(err));
  if (e == cudaErrorNotSupported)
    return fail(DIFFATTN_ERR_SHAPE, "%s: no V2 pair kernel for d=%d", name, p.dqk);
  if (err[0]) return fail(DIFFATTN_ERR_CUDA, "%s: %s", name, err);
  if (e != cudaSuccess) return cuda_fail(e, name);
  return ok();
}

DIFFATTN_API int diffattn_fwd(const void* q, const void* k, const void* v, void* out,
                              const float* lambda, float lambda_init, const float* norm_weight,
                              float eps, int B, int N, int H, int d, int dv, int flags, int dtype,
                              void* stream) {
  if (!q || !k || !v || !out || !lambda) return fail(DIFFATTN_ERR_ARG, "diffattn_fwd: null pointer");
  if (flags & ~kPrefillFlags) return fail(DIFFATTN_ERR_ARG, "diffattn_fwd: unknown flag bits 0x%x", flags);
  if ((flags & DIFFATTN_NORM) && !(eps > 0.f))
    return fail(DIFFATTN_ERR_ARG, "diffattn_fwd: eps must be > 0 with DIFFATTN_NORM");
  if (dtype != DIFFATTN_BF16 && dtype != DIFFATTN_FP32)
    return fail(DIFFATTN_ERR_DTYPE, "diffattn_fwd: dtype must be DIFFATTN_BF16 or DIFFATTN_FP32");
  if (B < 1 || N < 1 || H < 1) return fail(DIFFATTN_ERR_SHAPE, "diffattn_fwd: B, N, H must be >= 1");
  if (!(d == 64 || d == 128) || dv != 2 * d)
    return fail(DIFFATTN_ERR_SHAPE, "diffattn_fwd: need d in {64, 128} and dv = 2d (got d=%d dv=%d)", d, dv);
  const long long tiles = (static_cast<long long>(N) + 127) / 128 * B * H;
  if (tiles * 2 > 0x7fffffffLL || static_cast<long long>(N) * H > (1LL << 30))
    return fail(DIFFATTN_ERR_SHAPE, "diffattn_fwd: problem too large for one launch");
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
      !aligned(lambda, 4) || (norm_weight && !aligned(norm_weight, 16)))
    return fail(DIFFATTN_ERR_ALIGN, "diffattn_fwd: tensors must be 16-byte aligned");
  int rc = check_device();
  if (rc) return rc;
  da::Problem p{};
  p.q = q;
  p.k = k;
  p.v = v;
  p.out = out;
  p.B = B;
  p.N = N;
  p.units = H;
  p.dqk = d;
  p.dv = dv;
  p.mode = da::MODE_V1;
  p.q_heads = H;
  p.kv_heads = H;
  p.q_cols = 2 * d;
  p.k_cols = 2 * d;
  p.group = 1;
  p.lambda = lambda;
  p.lam_logit = nullptr;
  p.norm_w = norm_weight;
  p.eps = eps;
  p.lambda_init = lambda_init;
  p.flags = flags;
  p.scale = 1.0f / std::sqrt(static_cast<float>(d));
  return run_prefill(p, dtype, "diffattn_fwd", static_cast<cudaStream_t>(stream));
}

DIFFATTN_API int diffattn_decode_workspace_size(int B, int Lmax, int H, int d, int dv,
                                                size_t* bytes) {
  if (!bytes) return fail(DIFFATTN_ERR_ARG, "diffattn_decode_workspace_size: null pointer");
  if (B < 1 || Lmax < 1 || H < 1 || d != 128 || dv != 256)
    return fail(DIFFATTN_ERR_SHAPE, "diffattn_decode_workspace_size: need B, Lmax, H >= 1, d = 128, dv = 256");
  *bytes = da::decode_workspace_bytes(B, Lmax, H, dv);
  return ok();
}

DIFFATTN_API int diffattn_decode(const void* q, const void* k_cache, const void* v_cache,
                                 const int* seqlens, void* out, const float* lambda,
                                 float lambda_init, const float* norm_weight, float eps, int B,
                                 int Lmax, int H, int d, int dv, int flags, int dtype,
                                 void* workspace, size_t ws_bytes, void* stream) {
  if (!q || !k_cache || !v_cache || !out || !lambda)
    return fail(DIFFATTN_ERR_ARG, "diffattn_decode: null pointer");
  if (flags & ~(DIFFATTN_CAUSAL | DIFFATTN_NORM | DIFFATTN_SCALE))
    return fail(DIFFATTN_ERR_ARG, "diffattn_decode: unknown flag bits 0x%x", flags);
  if ((flags & DIFFATTN_NORM) && !(eps > 0.f))
    return fail(DIFFATTN_ERR_ARG, "diffattn_decode: eps must be > 0 with DIFFATTN_NORM");
  if (dtype != DIFFATTN_BF16) return fail(DIFFATTN_ERR_DTYPE, "diffattn_decode: dtype must be DIFFATTN_BF16");
  if (B < 1 || Lmax < 1 || H < 1 || B > 65535 || H > 65535)
    return fail(DIFFATTN_ERR_SHAPE, "diffattn_decode: need 1 <= B, H <= 65535 and Lmax >= 1");
  if (d != 128 || dv != 256)
    return fail(DIFFATTN_ERR_SHAPE, "diffattn_decode: need d = 128 and dv = 256 (got d=%d dv=%d)", d, dv);
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
      !aligned(lambda, 4) || (seqlens && !aligned(seqlens, 4)) ||
      (norm_weight && !aligned(norm_weight, 16)))
    return fail(DIFFATTN_ERR_ALIGN, "diffattn_decode: tensors must be 16-byte aligned");
  const size_t need = da::decode_workspace_bytes(B, Lmax, H, dv);
  if (!workspace || ws_bytes < need || !aligned(workspace, 256))
    return fail(DIFFATTN_ERR_WORKSPACE, "diffattn_decode: need a 256-byte aligned workspace of %zu bytes", need);
  int rc = check_device();
  if (rc) return rc;
  da::DecodeArgs a{};
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.seqlens = seqlens;
  a.out = out;
  a.lambda = lambda;
  a.lambda_init = lambda_init;
  a.norm_w = norm_weight;
  a.eps = eps;
  a.flags = flags;
  a.B = B;
  a.Lmax = Lmax;
  a.H = H;
  a.d = d;
  a.dv = dv;
  a.ws = static_cast<float*>(workspace);
  cudaError_t e = da::launch_decode(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "diffattn_decode launch");
  return ok();
}

DIFFATTN_API int diffattn_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                         const int* seqlens, void* out, const float* lambda,
                                         float lambda_init, const float* norm_weight, float eps,
                                         int B, int Lmax, int H, int d, int dv, int flags,
                                         int dtype, void* stream) {
  static_assert(da::kNoAllocScratchBytes == DIFFATTN_DECODE_NOALLOC_SCRATCH_BYTES, "scratch size");
  if (!q || !k_cache || !v_cache || !out || !lambda)
    return fail(DIFFATTN_ERR_ARG, "diffattn_decode_noalloc: null pointer");
  if (flags & ~(DIFFATTN_CAUSAL | DIFFATTN_NORM | DIFFATTN_SCALE))
    return fail(DIFFATTN_ERR_ARG, "diffattn_decode_noalloc: unknown flag bits 0x%x", flags);
  if ((flags & DIFFATTN_NORM) && !(eps > 0.f))
    return fail(DIFFATTN_ERR_ARG, "diffattn_decode_noalloc: eps must be > 0 with DIFFATTN_NORM");
  if (dtype != DIFFATTN_BF16)
    return fail(DIFFATTN_ERR_DTYPE, "diffattn_decode_noalloc: dtype must be DIFFATTN_BF16");
  if (B < 1 || Lmax < 1 || H < 1 || B > 65535 || H > 65535)
    return fail(DIFFATTN_ERR_SHAPE, "diffattn_decode_noalloc: need 1 <= B, H <= 65535 and Lmax >= 1");
  if (d != 128 || dv != 256)
    return fail(DIFFATTN_ERR_SHAPE, "diffattn_decode_noalloc: need d = 128 and dv = 256 (got d=%d dv=%d)", d, dv);
  const long long units = static_cast<long long>(B) * H;
  if (units > da::decode_noalloc_max_units())
    return fail(DIFFATTN_ERR_SHAPE,
                "diffattn_decode_noalloc: B*H = %lld exceeds the %lld (sequence, head) pairs whose "
                "partials fit in the built-in %zu-byte scratch; use diffattn_decode with a workspace",
                units, da::decode_noalloc_max_units(), da::kNoAllocScratchBytes);
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
      !aligned(lambda, 4) || (seqlens && !aligned(seqlens, 4)) ||
      (norm_weight && !aligned(norm_weight, 16)))
    return fail(DIFFATTN_ERR_ALIGN, "diffattn_decode_noalloc: tensors must be 16-byte aligned");
  int rc = check_device();
  if (rc) return rc;
  da::DecodeArgs a{};
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.seqlens = seqlens;
  a.out = out;
  a.lambda = lambda;
  a.lambda_init = lambda_init;
  a.norm_w = norm_weight;
  a.eps = eps;
  a.flags = flags;
  a.B = B;
  a.Lmax = Lmax;
  a.H = H;
  a.d = d;
  a.dv = dv;
  a.ws = nullptr;
  cudaError_t e = da::launch_decode_noalloc(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "diffattn_decode_noalloc");
  return ok();
}

DIFFATTN_API int diffattn_decode_split_count(int B, int Lmax, int H, int noalloc, int* splits,
                                             int* chunk_keys) {
  if (!splits || !chunk_keys) return fail(DIFFATTN_ERR_ARG, "diffattn_decode_split_count: null pointer");
  if (B < 1 || Lmax < 1 || H < 1)
    return fail(DIFFATTN_ERR_SHAPE, "diffattn_decode_split_count: need B, Lmax, H >= 1");
  int chunk = 0;
  if (noalloc) {
    if (static_cast<long long>(B) * H > da::decode_noalloc_max_units())
      return fail(DIFFATTN_ERR_SHAPE, "diffattn_decode_split_count: B*H = %lld exceeds the "
                  "no-allocation scratch limit of %lld", static_cast<long long>(B) * H,
                  da::decode_noalloc_max_units());
    *splits = da::decode_noalloc_splits(B, Lmax, H, &chunk);
  } else {
    *splits = da::decode_splits(B, Lmax, H, &chunk);
  }
  *chunk_keys = chunk;
  return ok();
}

DIFFATTN_API int diffattn_v2_fwd(const void* q, const void* k, const void* v,
                                 const float* lam_logit, void* out, int B, int N, int Hq, int Hkv,
                                 int d, int flags, int dtype, void* stream) {
  if (!q || !k || !v || !lam_logit || !out) return fail(DIFFATTN_ERR_ARG, "diffattn_v2_fwd: null pointer");
  constexpr int kV2Flags =
      DIFFATTN_CAUSAL | DIFFATTN_CUDA_CORES | DIFFATTN_SINGLE_PASS | DIFFATTN_EXACT;
  if (flags & ~kV2Flags) return fail(DIFFATTN_ERR_ARG, "diffattn_v2_fwd: unknown flag bits 0x%x", flags);
  if ((flags & DIFFATTN_EXACT) && (flags & (DIFFATTN_CUDA_CORES | DIFFATTN_SINGLE_PASS)))
    return fail(DIFFATTN_ERR_ARG, "diffattn_v2_fwd: DIFFATTN_EXACT excludes the other path flags");
  if (dtype != DIFFATTN_BF16 && dtype != DIFFATTN_FP32)
    return fail(DIFFATTN_ERR_DTYPE, "diffattn_v2_fwd: dtype must be DIFFATTN_BF16 or DIFFATTN_FP32");
  if (B < 1 || N < 1 || Hq < 2 || Hkv < 1)
    return fail(DIFFATTN_ERR_SHAPE, "diffattn_v2_fwd: B, N, Hkv must be >= 1 and Hq >= 2");
  if (Hq % 2 != 0 || Hq % Hkv != 0 || (Hq / Hkv) % 2 != 0)
    return fail(DIFFATTN_ERR_SHAPE,
                "diffattn_v2_fwd: need Hq even, Hq %% Hkv == 0 and Hq/Hkv even (a pair in one GQA group); "
                "got Hq=%d Hkv=%d", Hq, Hkv);
  if (!(d == 64 || d == 128)) return fail(DIFFATTN_ERR_SHAPE, "diffattn_v2_fwd: need d in {64, 128}");
  const long long tiles = (static_cast<long long>(N) + 127) / 128 * B * (Hq / 2);
  if (tiles * 2 > 0x7fffffffLL || static_cast<long long>(N) * Hq > (1LL << 30))
    return fail(DIFFATTN_ERR_SHAPE, "diffattn_v2_fwd: problem too large for one launch");
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
      !aligned(lam_logit, 4))
    return fail(DIFFATTN_ERR_ALIGN, "diffattn_v2_fwd: tensors must be 16-byte aligned");
  int rc = check_device();
  if (rc) return rc;
  da::Problem p{};
  p.q = q;
  p.k = k;
  p.v = v;
  p.out = out;
  p.B = B;
  p.N = N;
  p.units = Hq / 2;
  p.dqk = d;
  p.dv = d;
  p.mode = da::MODE_V2;
  p.q_heads = Hq;
  p.kv_heads = Hkv;
  p.q_cols = d;
  p.k_cols = d;
  p.group = Hq / Hkv;
  p.lambda = nullptr;
  p.lam_logit = lam_logit;
  p.norm_w = nullptr;
  p.eps = 0.f;
  p.lambda_init = 0.f;
  p.scale = 1.0f / std::sqrt(static_cast<float>(d));
  if (dtype == DIFFATTN_BF16 && !(flags & (DIFFATTN_CUDA_CORES | DIFFATTN_EXACT))) {
    p.flags = flags & DIFFATTN_CAUSAL;
    return run_v2_pair(p, "diffattn_v2_fwd", static_cast<cudaStream_t>(stream));
  }
  p.flags = flags & (DIFFATTN_CAUSAL | DIFFATTN_CUDA_CORES);
  return run_prefill(p, dtype, "diffattn_v2_fwd", static_cast<cudaStream_t>(stream));
}

}  // extern "C"

namespace {
int check_v2_decode_shape(const char* fn, int B, int Lmax, int Hq, int Hkv, int d) {
  if (B < 1 || Lmax < 1 || Hq < 2 || Hkv < 1 || B > 65535 || Hkv > 65535)
    return fail(DIFFATTN_ERR_SHAPE, "%s: need 1 <= B, Hkv <= 65535, Lmax >= 1 and Hq >= 2", fn);
  if (Hq % Hkv != 0 || !(Hq / Hkv == 2 || Hq / Hkv == 4 || Hq / Hkv == 8))
    return fail(DIFFATTN_ERR_SHAPE, "%s: need Hq / Hkv in {2, 4, 8} (got Hq=%d Hkv=%d)", fn, Hq, Hkv);
  if (d != 128) return fail(DIFFATTN_ERR_SHAPE, "%s: need d = 128 (got %d)", fn, d);
  if (static_cast<long long>(Hq / 2) > 65535)
    return fail(DIFFATTN_ERR_SHAPE, "%s: Hq / 2 must be <= 65535", fn);
  return DIFFATTN_OK;
}
}  // namespace

DIFFATTN_API int diffattn_v2_decode_workspace_size(int B, int Lmax, int Hq, int Hkv, int d,
                                                   size_t* bytes) {
  if (!bytes) return fail(DIFFATTN_ERR_ARG, "diffattn_v2_decode_workspace_size: null pointer");
  int rc = check_v2_decode_shape("diffattn_v2_decode_workspace_size", B, Lmax, Hq, Hkv, d);
  if (rc) return rc;
  *bytes = da::v2_decode_workspace_bytes(B, Lmax, Hq, Hkv);
  return ok();
}

DIFFATTN_API int diffattn_v2_decode(const void* q, const void* k_cache, const void* v_cache,
                                    const int* seqlens, const float* lam_logit, void* out, int B,
                                    int Lmax, int Hq, int Hkv, int d, int flags, int dtype,
                                    void* workspace, size_t ws_bytes, void* stream) {
  if (!q || !k_cache || !v_cache || !lam_logit || !out)
    return fail(DIFFATTN_ERR_ARG, "diffattn_v2_decode: null pointer");
  if (flags & ~(DIFFATTN_CAUSAL | DIFFATTN_CUDA_CORES))
    return fail(DIFFATTN_ERR_ARG, "diffattn_v2_decode: unknown flag bits 0x%x", flags);
  if (dtype != DIFFATTN_BF16) return fail(DIFFATTN_ERR_DTYPE, "diffattn_v2_decode: dtype must be DIFFATTN_BF16");
  int rc = check_v2_decode_shape("diffattn_v2_decode", B, Lmax, Hq, Hkv, d);
  if (rc) return rc;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
      !aligned(lam_logit, 4) || (seqlens && !aligned(seqlens, 4)))
    return fail(DIFFATTN_ERR_ALIGN, "diffattn_v2_decode: tensors must be 16-byte aligned");
  const size_t need = da::v2_decode_workspace_bytes(B, Lmax, Hq, Hkv);
  if (!workspace || ws_bytes < need || !aligned(workspace, 256))
    return fail(DIFFATTN_ERR_WORKSPACE, "diffattn_v2_decode: need a 256-byte aligned workspace of %zu bytes", need);
  rc = check_device();
  if (rc) return rc;
  da::V2DecodeArgs a{};
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.seqlens = seqlens;
  a.lam_logit = lam_logit;
  a.out = out;
  a.B = B;
  a.Lmax = Lmax;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.ws = static_cast<float*>(workspace);
  char err[256] = {0};
  cudaError_t e = (flags & DIFFATTN_CUDA_CORES)
                      ? da::launch_v2_decode(a, static_cast<cudaStream_t>(stream))
                      : da::launch_v2_decode_tc(a, static_cast<cudaStream_t>(stream), err, sizeof(err));
  if (e == cudaErrorNotSupported) return fail(DIFFATTN_ERR_UNSUPPORTED, "diffattn_v2_decode: unsupported group size");
  if (e == cudaErrorInvalidValue && err[0]) return fail(DIFFATTN_ERR_CUDA, "diffattn_v2_decode: %s", err);
  if (e != cudaSuccess) return cuda_fail(e, "diffattn_v2_decode launch");
  return ok();
}

DIFFATTN_API int diffattn_v2_decode_paged(const void* q, const void* k_pool, const void* v_pool,
                                          const int* block_table, const int* seqlens,
                                          const float* lam_logit, void* out, int B, int Hq,
                                          int Hkv, int d, int num_pages, int page_size,
                                          int max_pages, int flags, int dtype, void* workspace,
                                          size_t ws_bytes, void* stream) {
  if (!q || !k_pool || !v_pool || !block_table || !seqlens || !lam_logit || !out)
    return fail(DIFFATTN_ERR_ARG, "diffattn_v2_decode_paged: null pointer");
  if (flags & ~(DIFFATTN_CAUSAL | DIFFATTN_CUDA_CORES))
    return fail(DIFFATTN_ERR_ARG, "diffattn_v2_decode_paged: unknown flag bits 0x%x", flags);
  if (dtype != DIFFATTN_BF16)
    return fail(DIFFATTN_ERR_DTYPE, "diffattn_v2_decode_paged: dtype must be DIFFATTN_BF16");
  if (num_pages < 1 || page_size < 1 || max_pages < 1)
    return fail(DIFFATTN_ERR_SHAPE, "diffattn_v2_decode_paged: need num_pages, page_size, max_pages >= 1");
  const long long lmax = static_cast<long long>(max_pages) * page_size;
  if (lmax > (1LL << 30) || static_cast<long long>(num_pages) * page_size > 0x7fffffffLL)
    return fail(DIFFATTN_ERR_SHAPE, "diffattn_v2_decode_paged: need max_pages * page_size <= 2^30 and num_pages * page_size < 2^31");
  const int Lmax = static_cast<int>(lmax);
  int rc = check_v2_decode_shape("diffattn_v2_decode_paged", B, Lmax, Hq, Hkv, d);
  if (rc) return rc;
  if (!aligned(q, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(out, 16) ||
      !aligned(lam_logit, 4) || !aligned(seqlens, 4) || !aligned(block_table, 4))
    return fail(DIFFATTN_ERR_ALIGN, "diffattn_v2_decode_paged: tensors must be 16-byte aligned");
  const size_t need = da::v2_decode_workspace_bytes(B, Lmax, Hq, Hkv);
  if (!workspace || ws_bytes < need || !aligned(workspace, 256))
    return fail(DIFFATTN_ERR_WORKSPACE, "diffattn_v2_decode_paged: need a 256-byte aligned workspace of %zu bytes", need);
  rc = check_device();
  if (rc) return rc;
  da::V2DecodeArgs a{};
  a.q = q;
  a.k_cache = k_pool;
  a.v_cache = v_pool;
  a.seqlens = seqlens;
  a.lam_logit = lam_logit;
  a.out = out;
  a.B = B;
  a.Lmax = Lmax;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.ws = static_cast<float*>(workspace);
  a.block_table = block_table;
  a.page_size = page_size;
  a.max_pages = max_pages;
  a.num_pages = num_pages;
  char err[256] = {0};
  cudaError_t e = (flags & DIFFATTN_CUDA_CORES)
                      ? da::launch_v2_decode(a, static_cast<cudaStream_t>(stream))
                      : da::launch_v2_decode_tc(a, static_cast<cudaStream_t>(stream), err, sizeof(err));
  if (e == cudaErrorNotSupported) return fail(DIFFATTN_ERR_UNSUPPORTED, "diffattn_v2_decode_paged: unsupported shape");
  if (e == cudaErrorInvalidValue && err[0]) return fail(DIFFATTN_ERR_CUDA, "diffattn_v2_decode_paged: %s", err);
  if (e != cudaSuccess) return cuda_fail(e, "diffattn_v2_decode_paged launch");
  return ok();
}

DIFFATTN_API int diffattn_v2_decode_fp8(const void* q8, const void* k_cache8, const void* v_cache,
                                        const int* seqlens, const float* lam_logit, void* out,
                                        float q_descale, float k_descale, int B, int Lmax, int Hq,
                                        int Hkv, int d, int flags, void* workspace,
                                        size_t ws_bytes, void* stream) {
  const char* fn = "diffattn_v2_decode_fp8";
  if (!q8 || !k_cache8 || !v_cache || !lam_logit || !out)
    return fail(DIFFATTN_ERR_ARG, "%s: null pointer", fn);
  if (flags & ~DIFFATTN_CAUSAL) return fail(DIFFATTN_ERR_ARG, "%s: unknown flag bits 0x%x", fn, flags);
  if (!(q_descale > 0.f) || !(k_descale > 0.f) || !std::isfinite(q_descale * k_descale))
    return fail(DIFFATTN_ERR_ARG, "%s: descales must be finite and > 0", fn);
  int rc = check_v2_decode_shape(fn, B, Lmax, Hq, Hkv, d);
  if (rc) return rc;
  if (!aligned(q8, 16) || !aligned(k_cache8, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
      !aligned(lam_logit, 4) || (seqlens && !aligned(seqlens, 4)))
    return fail(DIFFATTN_ERR_ALIGN, "%s: tensors must be 16-byte aligned", fn);
  const size_t need = da::v2_decode_workspace_bytes(B, Lmax, Hq, Hkv);
  if (!workspace || ws_bytes < need || !aligned(workspace, 256))
    return fail(DIFFATTN_ERR_WORKSPACE, "%s: need a 256-byte aligned workspace of %zu bytes", fn, need);
  rc = check_device();
  if (rc) return rc;
  da::V2DecodeArgs a{};
  a.q = q8;
  a.k_cache = k_cache8;
  a.v_cache = v_cache;
  a.seqlens = seqlens;
  a.lam_logit = lam_logit;
  a.out = out;
  a.B = B;
  a.Lmax = Lmax;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.ws = static_cast<float*>(workspace);
  a.k8 = true;
  a.qk_descale = q_descale * k_descale;
  char err[256] = {0};
  cudaError_t e = da::launch_v2_decode_tc(a, static_cast<cudaStream_t>(stream), err, sizeof(err));
  if (e == cudaErrorNotSupported) return fail(DIFFATTN_ERR_UNSUPPORTED, "%s: unsupported shape", fn);
  if (e == cudaErrorInvalidValue && err[0]) return fail(DIFFATTN_ERR_CUDA, "%s: %s", fn, err);
  if (e != cudaSuccess) return cuda_fail(e, fn);
  return ok();
}

DIFFATTN_API int diffattn_v2_decode_fp8_paged(const void* q8, const void* k_pool8,
                                              const void* v_pool, const int* block_table,
                                              const int* seqlens, const float* lam_logit,
                                              void* out, float q_descale, float k_descale, int B,
                                              int Hq, int Hkv, int d, int num_pages, int page_size,
                                              int max_pages, int flags, void* workspace,
                                              size_t ws_bytes, void* stream) {
  const char* fn = "diffattn_v2_decode_fp8_paged";
  if (!q8 || !k_pool8 || !v_pool || !block_table || !seqlens || !lam_logit || !out)
    return fail(DIFFATTN_ERR_ARG, "%s: null pointer", fn);
  if (flags & ~DIFFATTN_CAUSAL) return fail(DIFFATTN_ERR_ARG, "%s: unknown flag bits 0x%x", fn, flags);
  if (!(q_descale > 0.f) || !(k_descale > 0.f) || !std::isfinite(q_descale * k_descale))
    return fail(DIFFATTN_ERR_ARG, "%s: descales must be finite and > 0", fn);
  if (num_pages < 1 || page_size < 1 || max_pages < 1)
    return fail(DIFFATTN_ERR_SHAPE, "%s: need num_pages, page_size, max_pages >= 1", fn);
  if (page_size % 128 != 0)
    return fail(DIFFATTN_ERR_UNSUPPORTED, "%s: fp8 pages must hold a multiple of 128 tokens (got %d)", fn, page_size);
  const long long lmax = static_cast<long long>(max_pages) * page_size;
  if (lmax > (1LL << 30) || static_cast<long long>(num_pages) * page_size > 0x7fffffffLL)
    return fail(DIFFATTN_ERR_SHAPE, "%s: need max_pages * page_size <= 2^30 and num_pages * page_size < 2^31", fn);
  const int Lmax = static_cast<int>(lmax);
  int rc = check_v2_decode_shape(fn, B, Lmax, Hq, Hkv, d);
  if (rc) return rc;
  if (!aligned(q8, 16) || !aligned(k_pool8, 16) || !aligned(v_pool, 16) || !aligned(out, 16) ||
      !aligned(lam_logit, 4) || !aligned(seqlens, 4) || !aligned(block_table, 4))
    return fail(DIFFATTN_ERR_ALIGN, "%s: tensors must be 16-byte aligned", fn);
  const size_t need = da::v2_decode_workspace_bytes(B, Lmax, Hq, Hkv);
  if (!workspace || ws_bytes < need || !aligned(workspace, 256))
    return fail(DIFFATTN_ERR_WORKSPACE, "%s: need a 256-byte aligned workspace of %zu bytes", fn, need);
  rc = check_device();
  if (rc) return rc;
  da::V2DecodeArgs a{};
  a.q = q8;
  a.k_cache = k_pool8;
  a.v_cache = v_pool;
  a.seqlens = seqlens;
  a.lam_logit = lam_logit;
  a.out = out;
  a.B = B;
  a.Lmax = Lmax;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.ws = static_cast<float*>(workspace);
  a.block_table = block_table;
  a.page_size = page_size;
  a.max_pages = max_pages;
  a.num_pages = num_pages;
  a.k8 = true;
  a.qk_descale = q_descale * k_descale;
  char err[256] = {0};
  cudaError_t e = da::launch_v2_decode_tc(a, static_cast<cudaStream_t>(stream), err, sizeof(err));
  if (e == cudaErrorNotSupported) return fail(DIFFATTN_ERR_UNSUPPORTED, "%s: unsupported shape", fn);
  if (e == cudaErrorInvalidValue && err[0]) return fail(DIFFATTN_ERR_CUDA, "%s: %s", fn, err);
  if (e != cudaSuccess) return cuda_fail(e, fn);
  return ok();
}

namespace {
int check_train_shape(const char* fn, int B, int N, int H, int d, int dv, int dtype) {
  if (dtype != DIFFATTN_BF16) return fail(DIFFATTN_ERR_DTYPE, "%s: dtype must be DIFFATTN_BF16", fn);
  if (B < 1 || N < 1 || H < 1) return fail(DIFFATTN_ERR_SHAPE, "%s: B, N, H must be >= 1", fn);
  if (d != 128 || dv != 256)
    return fail(DIFFATTN_ERR_SHAPE, "%s: need d = 128 and dv = 256 (got d=%d dv=%d)", fn, d, dv);
  const long long tiles = (static_cast<long long>(N) + 127) / 128 * B * H;
  if (tiles * 2 > 0x7fffffffLL || static_cast<long long>(N) * H > (1LL << 30))
    return fail(DIFFATTN_ERR_SHAPE, "%s: problem too large for one launch", fn);
  return DIFFATTN_OK;
}
}  // namespace

namespace {
// the training forward, batched (cu null: [B, N, H, *]) or packed (cu [B + 1], N the longest
// sequence, `total` rows)
int fwd_train_impl(const char* fn, const void* q, const void* k, const void* v, void* out,
                   void* o_pre, float* stats, const float* lambda, float lambda_init,
                   const float* norm_weight, float eps, int B, int N, int H, int d, int dv,
                   int flags, int dtype, const int* cu, int total, void* stream) {
  if (!q || !k || !v || !out || !o_pre || !stats || !lambda)
    return fail(DIFFATTN_ERR_ARG, "%s: null pointer", fn);
  constexpr int kTrainFlags = DIFFATTN_CAUSAL | DIFFATTN_NORM | DIFFATTN_SCALE;
  if (flags & ~kTrainFlags) return fail(DIFFATTN_ERR_ARG, "%s: unknown flag bits 0x%x", fn, flags);
  if ((flags & DIFFATTN_NORM) && !(eps > 0.f))
    return fail(DIFFATTN_ERR_ARG, "%s: eps must be > 0 with DIFFATTN_NORM", fn);
  int rc = check_train_shape(fn, B, N, H, d, dv, dtype);
  if (rc) return rc;
  if (cu && (total < N || static_cast<long long>(total) * H > (1LL << 30)))
    return fail(DIFFATTN_ERR_SHAPE, "%s: need max_seqlen <= total and total * H <= 2^30", fn);
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
      !aligned(o_pre, 16) || !aligned(stats, 16) || !aligned(lambda, 4) ||
      (norm_weight && !aligned(norm_weight, 16)) || (cu && !aligned(cu, 4)))
    return fail(DIFFATTN_ERR_ALIGN, "%s: tensors must be 16-byte aligned", fn);
  rc = check_device();
  if (rc) return rc;
  da::Problem p{};
  p.q = q;
  p.k = k;
  p.v = v;
  p.out = out;
  p.B = B;
  p.N = N;
  p.units = H;
  p.dqk = d;
  p.dv = dv;
  p.mode = da::MODE_V1;
  p.q_heads = H;
  p.kv_heads = H;
  p.q_cols = 2 * d;
  p.k_cols = 2 * d;
  p.group = 1;
  p.lambda = lambda;
  p.norm_w = norm_weight;
  p.eps = eps;
  p.lambda_init = lambda_init;
  p.flags = flags;
  p.scale = 1.0f / std::sqrt(static_cast<float>(d));
  p.stats = stats;
  p.o_pre = o_pre;
  p.n_pad = (N + 127) / 128 * 128;
  p.cu_seqlens = cu;
  p.total = total;
  return run_prefill(p, dtype, fn, static_cast<cudaStream_t>(stream));
}
}  // namespace

DIFFATTN_API int diffattn_fwd_train(const void* q, const void* k, const void* v, void* out,
                                    void* o_pre, float* stats, const float* lambda,
                                    float lambda_init, const float* norm_weight, float eps, int B,
                                    int N, int H, int d, int dv, int flags, int dtype,
                                    void* stream) {
  return fwd_train_impl("diffattn_fwd_train", q, k, v, out, o_pre, stats, lambda, lambda_init,
                        norm_weight, eps, B, N, H, d, dv, flags, dtype, nullptr, 0, stream);
}

DIFFATTN_API int diffattn_fwd_train_varlen(const void* q, const void* k, const void* v,
                                           void* out, void* o_pre, float* stats,
                                           const int* cu_seqlens, int max_seqlen, int total,
                                           const float* lambda, float lambda_init,
                                           const float* norm_weight, float eps, int B, int H,
                                           int d, int dv, int flags, int dtype, void* stream) {
  if (!cu_seqlens) return fail(DIFFATTN_ERR_ARG, "diffattn_fwd_train_varlen: null pointer");
  return fwd_train_impl("diffattn_fwd_train_varlen", q, k, v, out, o_pre, stats, lambda,
                        lambda_init, norm_weight, eps, B, max_seqlen, H, d, dv, flags, dtype,
                        cu_seqlens, total, stream);
}

DIFFATTN_API int diffattn_bwd_workspace_size(int B, int N, int H, int d, int dv, size_t* bytes) {
  if (!bytes) return fail(DIFFATTN_ERR_ARG, "diffattn_bwd_workspace_size: null pointer");
  int rc = check_train_shape("diffattn_bwd_workspace_size", B, N, H, d, dv, DIFFATTN_BF16);
  if (rc) return rc;
  *bytes = da::backward_workspace_bytes(B, N, H, static_cast<long long>(B) * N);
  return ok();
}

namespace {
// the backward, batched (cu null) or packed (cu [B + 1], N the longest sequence, `total` rows)
int bwd_impl(const char* fn, const void* q, const void* k, const void* v, const void* o_pre,
             const float* stats, const void* dout, const float* lambda, float lambda_init,
             const float* norm_weight, float eps, void* dq, void* dk, void* dv, float* dlambda,
             float* dnorm_weight, int B, int N, int H, int d, int dv_width, int flags, int dtype,
             const int* cu, int total, void* workspace, size_t ws_bytes, void* stream,
             int n_noise = 0) {
  if (!q || !k || !v || !o_pre || !stats || !dout || !lambda || !dq || !dk || !dv || !dlambda)
    return fail(DIFFATTN_ERR_ARG, "%s: null pointer", fn);
  constexpr int kTrainFlags = DIFFATTN_CAUSAL | DIFFATTN_NORM | DIFFATTN_SCALE;
  if (flags & ~kTrainFlags) return fail(DIFFATTN_ERR_ARG, "%s: unknown flag bits 0x%x", fn, flags);
  if ((flags & DIFFATTN_NORM) && !(eps > 0.f))
    return fail(DIFFATTN_ERR_ARG, "%s: eps must be > 0 with DIFFATTN_NORM", fn);
  int rc = check_train_shape(fn, B, N, H, d, dv_width, dtype);
  if (rc) return rc;
  if (cu && (total < N || static_cast<long long>(total) * H > (1LL << 30)))
    return fail(DIFFATTN_ERR_SHAPE, "%s: need max_seqlen <= total and total * H <= 2^30", fn);
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o_pre, 16) ||
      !aligned(stats, 16) || !aligned(dout, 16) || !aligned(dq, 16) || !aligned(dk, 16) ||
      !aligned(dv, 16) || !aligned(lambda, 4) || !aligned(dlambda, 4) ||
      (norm_weight && !aligned(norm_weight, 16)) || (dnorm_weight && !aligned(dnorm_weight, 4)) ||
      (cu && !aligned(cu, 4)))
    return fail(DIFFATTN_ERR_ALIGN, "%s: tensors must be 16-byte aligned", fn);
  const long long rows = cu ? total : static_cast<long long>(B) * N;
  const size_t need = da::backward_workspace_bytes(B, N, H, rows, n_noise > 0);
  if (!workspace || ws_bytes < need || !aligned(workspace, 256))
    return fail(DIFFATTN_ERR_WORKSPACE, "%s: need a 256-byte aligned workspace of %zu bytes", fn, need);
  rc = check_device();
  if (rc) return rc;
  da::BackwardArgs a{};
  a.q = q;
  a.k = k;
  a.v = v;
  a.o_pre = o_pre;
  a.stats = stats;
  a.dout = dout;
  a.lambda = lambda;
  a.lambda_init = lambda_init;
  a.norm_w = norm_weight;
  a.eps = eps;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.dlambda = dlambda;
  a.dnorm_w = dnorm_weight;
  a.B = B;
  a.N = N;
  a.H = H;
  a.flags = flags;
  a.workspace = workspace;
  a.cu_seqlens = cu;
  a.total = total;
  a.n_noise = n_noise;
  char err[256] = {0};
  cudaError_t e = da::launch_backward(a, static_cast<cudaStream_t>(stream), err, sizeof(err));
  if (err[0]) return fail(DIFFATTN_ERR_CUDA, "%s: %s", fn, err);
  if (e != cudaSuccess) return cuda_fail(e, fn);
  return ok();
}
}  // namespace

DIFFATTN_API int diffattn_bwd(const void* q, const void* k, const void* v, const void* o_pre,
                              const float* stats, const void* dout, const float* lambda,
                              float lambda_init, const float* norm_weight, float eps, void* dq,
                              void* dk, void* dv, float* dlambda, float* dnorm_weight, int B,
                              int N, int H, int d, int dv_width, int flags, int dtype,
                              void* workspace, size_t ws_bytes, void* stream) {
  return bwd_impl("diffattn_bwd", q, k, v, o_pre, stats, dout, lambda, lambda_init, norm_weight,
                  eps, dq, dk, dv, dlambda, dnorm_weight, B, N, H, d, dv_width, flags, dtype,
                  nullptr, 0, workspace, ws_bytes, stream);
}

DIFFATTN_API int diffattn_bwd_varlen_workspace_size(int B, int max_seqlen, int total, int H,
                                                   int d, int dv, size_t* bytes) {
  if (!bytes) return fail(DIFFATTN_ERR_ARG, "diffattn_bwd_varlen_workspace_size: null pointer");
  int rc = check_train_shape("diffattn_bwd_varlen_workspace_size", B, max_seqlen, H, d, dv,
                             DIFFATTN_BF16);
  if (rc) return rc;
  if (total < max_seqlen)
    return fail(DIFFATTN_ERR_SHAPE, "diffattn_bwd_varlen_workspace_size: need max_seqlen <= total");
  *bytes = da::backward_workspace_bytes(B, max_seqlen, H, total);
  return ok();
}

DIFFATTN_API int diffattn_bwd_varlen(const void* q, const void* k, const void* v,
                                     const void* o_pre, const float* stats, const void* dout,
                                     const int* cu_seqlens, int max_seqlen, int total,
                                     const float* lambda, float lambda_init,
                                     const float* norm_weight, float eps, void* dq, void* dk,
                                     void* dv, float* dlambda, float* dnorm_weight, int B, int H,
                                     int d, int dv_width, int flags, int dtype, void* workspace,
                                     size_t ws_bytes, void* stream) {
  if (!cu_seqlens) return fail(DIFFATTN_ERR_ARG, "diffattn_bwd_varlen: null pointer");
  return bwd_impl("diffattn_bwd_varlen", q, k, v, o_pre, stats, dout, lambda, lambda_init,
                  norm_weight, eps, dq, dk, dv, dlambda, dnorm_weight, B, max_seqlen, H, d,
                  dv_width, flags, dtype, cu_seqlens, total, workspace, ws_bytes, stream);
}

DIFFATTN_API int diffattn_fwd_fused_lambda(const void* q, const void* k, const void* v, void* out,
                                           const float* lq1, const float* lk1, const float* lq2,
                                           const float* lk2, int lambda_dim, int lambda_sets,
                                           int layer, const float* norm_weight, float eps, int B,
                                           int N, int H, int d, int dv, int flags, int dtype,
                                           void* stream) {
  if (!q || !k || !v || !out || !lq1 || !lk1 || !lq2 || !lk2)
    return fail(DIFFATTN_ERR_ARG, "diffattn_fwd_fused_lambda: null pointer");
  constexpr int kFusedFlags = DIFFATTN_CAUSAL | DIFFATTN_NORM | DIFFATTN_SCALE;
  if (flags & ~kFusedFlags)
    return fail(DIFFATTN_ERR_ARG, "diffattn_fwd_fused_lambda: unknown flag bits 0x%x", flags);
  if ((flags & DIFFATTN_NORM) && !(eps > 0.f))
    return fail(DIFFATTN_ERR_ARG, "diffattn_fwd_fused_lambda: eps must be > 0 with DIFFATTN_NORM");
  if (dtype != DIFFATTN_BF16)
    return fail(DIFFATTN_ERR_DTYPE, "diffattn_fwd_fused_lambda: dtype must be DIFFATTN_BF16");
  if (layer < 1) return fail(DIFFATTN_ERR_ARG, "diffattn_fwd_fused_lambda: layer must be >= 1");
  if (lambda_dim < 1 || lambda_dim > 4096 || !(lambda_sets == 1 || lambda_sets == H))
    return fail(DIFFATTN_ERR_SHAPE, "diffattn_fwd_fused_lambda: need 1 <= lambda_dim <= 4096 and lambda_sets in {1, H}");
  if (B < 1 || N < 1 || H < 1) return fail(DIFFATTN_ERR_SHAPE, "diffattn_fwd_fused_lambda: B, N, H must be >= 1");
  if (!(d == 64 || d == 128) || dv != 2 * d)
    return fail(DIFFATTN_ERR_SHAPE, "diffattn_fwd_fused_lambda: need d in {64, 128} and dv = 2d");
  const long long tiles = (static_cast<long long>(N) + 127) / 128 * B * H;
  if (tiles * 2 > 0x7fffffffLL || static_cast<long long>(N) * H > (1LL << 30))
    return fail(DIFFATTN_ERR_SHAPE, "diffattn_fwd_fused_lambda: problem too large for one launch");
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
      !aligned(lq1, 4) || !aligned(lk1, 4) || !aligned(lq2, 4) || !aligned(lk2, 4) ||
      (norm_weight && !aligned(norm_weight, 16)))
    return fail(DIFFATTN_ERR_ALIGN, "diffattn_fwd_fused_lambda: tensors must be 16-byte aligned");
  int rc = check_device();
  if (rc) return rc;
  da::Problem p{};
  p.q = q;
  p.k = k;
  p.v = v;
  p.out = out;
  p.B = B;
  p.N = N;
  p.units = H;
  p.dqk = d;
  p.dv = dv;
  p.mode = da::MODE_V1;
  p.q_heads = H;
  p.kv_heads = H;
  p.q_cols = 2 * d;
  p.k_cols = 2 * d;
  p.group = 1;
  p.norm_w = norm_weight;
  p.eps = eps;
  p.lambda_init = diffattn_lambda_init(layer);
  p.flags = flags;
  p.scale = 1.0f / std::sqrt(static_cast<float>(d));
  p.lam_vec[0] = lq1;
  p.lam_vec[1] = lk1;
  p.lam_vec[2] = lq2;
  p.lam_vec[3] = lk2;
  p.lam_dim = lambda_dim;
  p.lam_sets = lambda_sets;
  return run_prefill(p, dtype, "diffattn_fwd_fused_lambda", static_cast<cudaStream_t>(stream));
}

DIFFATTN_API int diffattn_decode_paged(const void* q, const void* k_pool, const void* v_pool,
                                       const int* block_table, const int* seqlens, void* out,
                                       const float* lambda, float lambda_init,
                                       const float* norm_weight, float eps, int B, int H, int d,
                                       int dv, int num_pages, int page_size, int max_pages,
                                       int flags, int dtype, void* workspace, size_t ws_bytes,
                                       void* stream) {
  if (!q || !k_pool || !v_pool || !block_table || !seqlens || !out || !lambda)
    return fail(DIFFATTN_ERR_ARG, "diffattn_decode_paged: null pointer");
  if (flags & ~(DIFFATTN_CAUSAL | DIFFATTN_NORM | DIFFATTN_SCALE))
    return fail(DIFFATTN_ERR_ARG, "diffattn_decode_paged: unknown flag bits 0x%x", flags);
  if ((flags & DIFFATTN_NORM) && !(eps > 0.f))
    return fail(DIFFATTN_ERR_ARG, "diffattn_decode_paged: eps must be > 0 with DIFFATTN_NORM");
  if (dtype != DIFFATTN_BF16) return fail(DIFFATTN_ERR_DTYPE, "diffattn_decode_paged: dtype must be DIFFATTN_BF16");
  if (B < 1 || H < 1 || B > 65535 || H > 65535 || num_pages < 1 || page_size < 1 || max_pages < 1)
    return fail(DIFFATTN_ERR_SHAPE, "diffattn_decode_paged: need 1 <= B, H <= 65535 and num_pages, page_size, max_pages >= 1");
  const long long lmax = static_cast<long long>(max_pages) * page_size;
  if (lmax > 0x7fffffffLL || static_cast<long long>(num_pages) * page_size > (1LL << 40))
    return fail(DIFFATTN_ERR_SHAPE, "diffattn_decode_paged: max_pages * page_size too large");
  if (d != 128 || dv != 256)
    return fail(DIFFATTN_ERR_SHAPE, "diffattn_decode_paged: need d = 128 and dv = 256 (got d=%d dv=%d)", d, dv);
  if (!aligned(q, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(out, 16) ||
      !aligned(lambda, 4) || !aligned(seqlens, 4) || !aligned(block_table, 4) ||
      (norm_weight && !aligned(norm_weight, 16)))
    return fail(DIFFATTN_ERR_ALIGN, "diffattn_decode_paged: tensors must be 16-byte aligned");
  const int Lmax = static_cast<int>(lmax);
  const size_t need = da::decode_workspace_bytes(B, Lmax, H, dv);
  if (!workspace || ws_bytes < need || !aligned(workspace, 256))
    return fail(DIFFATTN_ERR_WORKSPACE, "diffattn_decode_paged: need a 256-byte aligned workspace of %zu bytes", need);
  int rc = check_device();
  if (rc) return rc;
  da::DecodeArgs a{};
  a.q = q;
  a.k_cache = k_pool;
  a.v_cache = v_pool;
  a.seqlens = seqlens;
  a.out = out;
  a.lambda = lambda;
  a.lambda_init = lambda_init;
  a.norm_w = norm_weight;
  a.eps = eps;
  a.flags = flags;
  a.B = B;
  a.Lmax = Lmax;
  a.H = H;
  a.d = d;
  a.dv = dv;
  a.ws = static_cast<float*>(workspace);
  a.block_table = block_table;
  a.page_size = page_size;
  a.max_pages = max_pages;
  a.num_pages = num_pages;
  cudaError_t e = da::launch_decode(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "diffattn_decode_paged launch");
  return ok();
}

DIFFATTN_API int diffattn_fwd_varlen(const void* q, const void* k, const void* v, void* out,
                                     const int* cu_seqlens, int max_seqlen, int total,
                                     const float* lambda, float lambda_init,
                                     const float* norm_weight, float eps, int B, int H, int d,
                                     int dv, int flags, int dtype, void* stream) {
  if (!q || !k || !v || !out || !cu_seqlens || !lambda)
    return fail(DIFFATTN_ERR_ARG, "diffattn_fwd_varlen: null pointer");
  constexpr int kVarFlags = DIFFATTN_CAUSAL | DIFFATTN_NORM | DIFFATTN_SCALE;
  if (flags & ~kVarFlags) return fail(DIFFATTN_ERR_ARG, "diffattn_fwd_varlen: unknown flag bits 0x%x", flags);
  if ((flags & DIFFATTN_NORM) && !(eps > 0.f))
    return fail(DIFFATTN_ERR_ARG, "diffattn_fwd_varlen: eps must be > 0 with DIFFATTN_NORM");
  if (dtype != DIFFATTN_BF16) return fail(DIFFATTN_ERR_DTYPE, "diffattn_fwd_varlen: dtype must be DIFFATTN_BF16");
  if (B < 1 || H < 1 || max_seqlen < 1 || total < 1 || max_seqlen > total)
    return fail(DIFFATTN_ERR_SHAPE, "diffattn_fwd_varlen: need B, H >= 1 and 1 <= max_seqlen <= total");
  if (!(d == 64 || d == 128) || dv != 2 * d)
    return fail(DIFFATTN_ERR_SHAPE, "diffattn_fwd_varlen: need d in {64, 128} and dv = 2d");
  const long long tiles = (static_cast<long long>(max_seqlen) + 127) / 128 * B * H;
  if (tiles * 2 > 0x7fffffffLL || static_cast<long long>(total) * H > (1LL << 30))
    return fail(DIFFATTN_ERR_SHAPE, "diffattn_fwd_varlen: problem too large for one launch");
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
      !aligned(lambda, 4) || !aligned(cu_seqlens, 4) || (norm_weight && !aligned(norm_weight, 16)))
    return fail(DIFFATTN_ERR_ALIGN, "diffattn_fwd_varlen: tensors must be 16-byte aligned");
  int rc = check_device();
  if (rc) return rc;
  da::Problem p{};
  p.q = q;
  p.k = k;
  p.v = v;
  p.out = out;
  p.B = B;
  p.N = max_seqlen;
  p.units = H;
  p.dqk = d;
  p.dv = dv;
  p.mode = da::MODE_V1;
  p.q_heads = H;
  p.kv_heads = H;
  p.q_cols = 2 * d;
  p.k_cols = 2 * d;
  p.group = 1;
  p.lambda = lambda;
  p.norm_w = norm_weight;
  p.eps = eps;
  p.lambda_init = lambda_init;
  p.flags = flags;
  p.scale = 1.0f / std::sqrt(static_cast<float>(d));
  p.cu_seqlens = cu_seqlens;
  p.total = total;
  return run_prefill(p, dtype, "diffattn_fwd_varlen", static_cast<cudaStream_t>(stream));
}

DIFFATTN_API int diffattn_fwd_varlen_qk(const void* q, const void* k, const void* v, void* out,
                                        const int* cu_seqlens_q, const int* cu_seqlens_k,
                                        int max_seqlen_q, int max_seqlen_k, int total_q,
                                        int total_k, const float* lambda, float lambda_init,
                                        const float* norm_weight, float eps, int B, int H, int d,
                                        int dv, int flags, int dtype, void* stream) {
  const char* fn = "diffattn_fwd_varlen_qk";
  if (!q || !k || !v || !out || !cu_seqlens_q || !cu_seqlens_k || !lambda)
    return fail(DIFFATTN_ERR_ARG, "%s: null pointer", fn);
  constexpr int kVarFlags = DIFFATTN_CAUSAL | DIFFATTN_NORM | DIFFATTN_SCALE;
  if (flags & ~kVarFlags) return fail(DIFFATTN_ERR_ARG, "%s: unknown flag bits 0x%x", fn, flags);
  if ((flags & DIFFATTN_NORM) && !(eps > 0.f))
    return fail(DIFFATTN_ERR_ARG, "%s: eps must be > 0 with DIFFATTN_NORM", fn);
  if (dtype != DIFFATTN_BF16) return fail(DIFFATTN_ERR_DTYPE, "%s: dtype must be DIFFATTN_BF16", fn);
  if (B < 1 || H < 1 || max_seqlen_q < 1 || total_q < 1 || max_seqlen_q > total_q ||
      max_seqlen_k < max_seqlen_q || total_k < total_q || max_seqlen_k > total_k)
    return fail(DIFFATTN_ERR_SHAPE, "%s: need B, H >= 1, 1 <= max_seqlen_q <= total_q, "
                "max_seqlen_q <= max_seqlen_k <= total_k and total_q <= total_k", fn);
  if (!(d == 64 || d == 128) || dv != 2 * d)
    return fail(DIFFATTN_ERR_SHAPE, "%s: need d in {64, 128} and dv = 2d", fn);
  const long long tiles = (static_cast<long long>(max_seqlen_q) + 127) / 128 * B * H;
  if (tiles * 2 > 0x7fffffffLL || static_cast<long long>(total_k) * H > (1LL << 30))
    return fail(DIFFATTN_ERR_SHAPE, "%s: problem too large for one launch", fn);
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
      !aligned(lambda, 4) || !aligned(cu_seqlens_q, 4) || !aligned(cu_seqlens_k, 4) ||
      (norm_weight && !aligned(norm_weight, 16)))
    return fail(DIFFATTN_ERR_ALIGN, "%s: tensors must be 16-byte aligned", fn);
  int rc = check_device();
  if (rc) return rc;
  da::Problem p{};
  p.q = q;
  p.k = k;
  p.v = v;
  p.out = out;
  p.B = B;
  p.N = max_seqlen_q;
  p.units = H;
  p.dqk = d;
  p.dv = dv;
  p.mode = da::MODE_V1;
  p.q_heads = H;
  p.kv_heads = H;
  p.q_cols = 2 * d;
  p.k_cols = 2 * d;
  p.group = 1;
  p.lambda = lambda;
  p.norm_w = norm_weight;
  p.eps = eps;
  p.lambda_init = lambda_init;
  p.flags = flags;
  p.scale = 1.0f / std::sqrt(static_cast<float>(d));
  p.cu_seqlens = cu_seqlens_q;
  p.total = total_q;
  p.cu_seqlens_k = cu_seqlens_k;
  p.total_k = total_k;
  p.max_seqlen_k = max_seqlen_k;
  return run_prefill(p, dtype, fn, static_cast<cudaStream_t>(stream));
}

DIFFATTN_API int diffattn_v2_fwd_varlen(const void* q, const void* k, const void* v,
                                        const float* lam_logit, void* out,
                                        const int* cu_seqlens_q, const int* cu_seqlens_k,
                                        int max_seqlen_q, int max_seqlen_k, int total_q,
                                        int total_k, int B, int Hq, int Hkv, int d, int flags,
                                        int dtype, void* stream) {
  const char* fn = "diffattn_v2_fwd_varlen";
  if (!q || !k || !v || !lam_logit || !out || !cu_seqlens_q)
    return fail(DIFFATTN_ERR_ARG, "%s: null pointer", fn);
  if (flags & ~(DIFFATTN_CAUSAL | DIFFATTN_EXACT))
    return fail(DIFFATTN_ERR_ARG, "%s: unknown flag bits 0x%x", fn, flags);
  if (dtype != DIFFATTN_BF16) return fail(DIFFATTN_ERR_DTYPE, "%s: dtype must be DIFFATTN_BF16", fn);
  if (!cu_seqlens_k) {  // the keys share the query offsets
    max_seqlen_k = max_seqlen_q;
    total_k = total_q;
  }
  if (B < 1 || Hq < 2 || Hkv < 1 || max_seqlen_q < 1 || total_q < 1 || max_seqlen_q > total_q ||
      max_seqlen_k < max_seqlen_q || total_k < total_q || max_seqlen_k > total_k)
    return fail(DIFFATTN_ERR_SHAPE, "%s: need B, Hkv >= 1, Hq >= 2, 1 <= max_seqlen_q <= total_q, "
                "max_seqlen_q <= max_seqlen_k <= total_k and total_q <= total_k", fn);
  if (Hq % 2 != 0 || Hq % Hkv != 0 || (Hq / Hkv) % 2 != 0)
    return fail(DIFFATTN_ERR_SHAPE, "%s: need Hq even, Hq %% Hkv == 0 and Hq/Hkv even (got Hq=%d Hkv=%d)",
                fn, Hq, Hkv);
  if (!(d == 64 || d == 128)) return fail(DIFFATTN_ERR_SHAPE, "%s: need d in {64, 128}", fn);
  const long long tiles = (static_cast<long long>(max_seqlen_q) + 127) / 128 * B * (Hq / 2);
  if (tiles * 2 > 0x7fffffffLL || static_cast<long long>(total_k) * Hq > (1LL << 30))
    return fail(DIFFATTN_ERR_SHAPE, "%s: problem too large for one launch", fn);
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
      !aligned(lam_logit, 4) || !aligned(cu_seqlens_q, 4) || (cu_seqlens_k && !aligned(cu_seqlens_k, 4)))
    return fail(DIFFATTN_ERR_ALIGN, "%s: tensors must be 16-byte aligned", fn);
  int rc = check_device();
  if (rc) return rc;
  da::Problem p{};
  p.q = q;
  p.k = k;
  p.v = v;
  p.out = out;
  p.B = B;
  p.N = max_seqlen_q;
  p.units = Hq / 2;
  p.dqk = d;
  p.dv = d;
  p.mode = da::MODE_V2;
  p.q_heads = Hq;
  p.kv_heads = Hkv;
  p.q_cols = d;
  p.k_cols = d;
  p.group = Hq / Hkv;
  p.lam_logit = lam_logit;
  p.flags = flags & DIFFATTN_CAUSAL;
  p.scale = 1.0f / std::sqrt(static_cast<float>(d));
  p.cu_seqlens = cu_seqlens_q;
  p.total = total_q;
  p.cu_seqlens_k = cu_seqlens_k;
  p.total_k = total_k;
  p.max_seqlen_k = max_seqlen_k;
  if (!(flags & DIFFATTN_EXACT)) return run_v2_pair(p, fn, static_cast<cudaStream_t>(stream));
  return run_prefill(p, dtype, fn, static_cast<cudaStream_t>(stream));
}

namespace {
// shape rules shared by the two paged prefills
int check_paged_prefill(const char* fn, int B, int max_seqlen_q, int max_seqlen_k, int total_q,
                        int num_pages, int page_size, int max_pages) {
  if (B < 1 || max_seqlen_q < 1 || total_q < 1 || max_seqlen_q > total_q ||
      max_seqlen_k < max_seqlen_q || num_pages < 1 || max_pages < 1)
    return fail(DIFFATTN_ERR_SHAPE, "%s: need B >= 1, 1 <= max_seqlen_q <= total_q, "
                "max_seqlen_q <= max_seqlen_k, num_pages >= 1 and max_pages >= 1", fn);
  if (page_size < 128 || page_size % 128 != 0)
    return fail(DIFFATTN_ERR_SHAPE, "%s: page_size must be a multiple of 128 (got %d)", fn, page_size);
  if (static_cast<long long>(num_pages) * page_size > 0x7fffffffLL ||
      static_cast<long long>(max_pages) * page_size > (1LL << 30) ||
      static_cast<long long>(max_seqlen_k) > static_cast<long long>(max_pages) * page_size)
    return fail(DIFFATTN_ERR_SHAPE, "%s: need num_pages * page_size < 2^31 and "
                "max_seqlen_k <= max_pages * page_size <= 2^30", fn);
  return DIFFATTN_OK;
}
}  // namespace

DIFFATTN_API int diffattn_fwd_paged(const void* q, const void* k_pool, const void* v_pool,
                                    void* out, const int* cu_seqlens_q, const int* seqlens_k,
                                    const int* block_table, int max_seqlen_q, int max_seqlen_k,
                                    int total_q, int num_pages, int page_size, int max_pages,
                                    const float* lambda, float lambda_init,
                                    const float* norm_weight, float eps, int B, int H, int d,
                                    int dv, int flags, int dtype, void* stream) {
  const char* fn = "diffattn_fwd_paged";
  if (!q || !k_pool || !v_pool || !out || !cu_seqlens_q || !seqlens_k || !block_table || !lambda)
    return fail(DIFFATTN_ERR_ARG, "%s: null pointer", fn);
  constexpr int kFlags = DIFFATTN_CAUSAL | DIFFATTN_NORM | DIFFATTN_SCALE;
  if (flags & ~kFlags) return fail(DIFFATTN_ERR_ARG, "%s: unknown flag bits 0x%x", fn, flags);
  if ((flags & DIFFATTN_NORM) && !(eps > 0.f))
    return fail(DIFFATTN_ERR_ARG, "%s: eps must be > 0 with DIFFATTN_NORM", fn);
  if (dtype != DIFFATTN_BF16) return fail(DIFFATTN_ERR_DTYPE, "%s: dtype must be DIFFATTN_BF16", fn);
  int rc = check_paged_prefill(fn, B, max_seqlen_q, max_seqlen_k, total_q, num_pages, page_size,
                               max_pages);
  if (rc) return rc;
  if (H < 1) return fail(DIFFATTN_ERR_SHAPE, "%s: H must be >= 1", fn);
  if (d != 128 || dv != 256)
    return fail(DIFFATTN_ERR_SHAPE, "%s: need d = 128 and dv = 256 (got d=%d dv=%d)", fn, d, dv);
  const long long tiles = (static_cast<long long>(max_seqlen_q) + 127) / 128 * B * H;
  if (tiles * 2 > 0x7fffffffLL || static_cast<long long>(num_pages) * page_size * H > (1LL << 34))
    return fail(DIFFATTN_ERR_SHAPE, "%s: problem too large for one launch", fn);
  if (!aligned(q, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(out, 16) ||
      !aligned(lambda, 4) || !aligned(cu_seqlens_q, 4) || !aligned(seqlens_k, 4) ||
      !aligned(block_table, 4) || (norm_weight && !aligned(norm_weight, 16)))
    return fail(DIFFATTN_ERR_ALIGN, "%s: tensors must be 16-byte aligned", fn);
  rc = check_device();
  if (rc) return rc;
  da::Problem p{};
  p.q = q;
  p.k = k_pool;
  p.v = v_pool;
  p.out = out;
  p.B = B;
  p.N = max_seqlen_q;
  p.units = H;
  p.dqk = d;
  p.dv = dv;
  p.mode = da::MODE_V1;
  p.q_heads = H;
  p.kv_heads = H;
  p.q_cols = 2 * d;
  p.k_cols = 2 * d;
  p.group = 1;
  p.lambda = lambda;
  p.norm_w = norm_weight;
  p.eps = eps;
  p.lambda_init = lambda_init;
  p.flags = flags;
  p.scale = 1.0f / std::sqrt(static_cast<float>(d));
  p.cu_seqlens = cu_seqlens_q;
  p.total = total_q;
  p.max_seqlen_k = max_seqlen_k;
  p.seqlens_k = seqlens_k;
  p.block_table = block_table;
  p.page_size = page_size;
  p.max_pages = max_pages;
  p.num_pages = num_pages;
  return run_prefill(p, dtype, fn, static_cast<cudaStream_t>(stream));
}

DIFFATTN_API int diffattn_v2_fwd_paged(const void* q, const void* k_pool, const void* v_pool,
                                       const float* lam_logit, void* out,
                                       const int* cu_seqlens_q, const int* seqlens_k,
                                       const int* block_table, int max_seqlen_q, int max_seqlen_k,
                                       int total_q, int num_pages, int page_size, int max_pages,
                                       int B, int Hq, int Hkv, int d, int flags, int dtype,
                                       void* stream) {
  const char* fn = "diffattn_v2_fwd_paged";
  if (!q || !k_pool || !v_pool || !lam_logit || !out || !cu_seqlens_q || !seqlens_k || !block_table)
    return fail(DIFFATTN_ERR_ARG, "%s: null pointer", fn);
  if (flags & ~(DIFFATTN_CAUSAL | DIFFATTN_EXACT))
    return fail(DIFFATTN_ERR_ARG, "%s: unknown flag bits 0x%x", fn, flags);
  if (dtype != DIFFATTN_BF16) return fail(DIFFATTN_ERR_DTYPE, "%s: dtype must be DIFFATTN_BF16", fn);
  int rc = check_paged_prefill(fn, B, max_seqlen_q, max_seqlen_k, total_q, num_pages, page_size,
                               max_pages);
  if (rc) return rc;
  if (Hq < 2 || Hkv < 1 || Hq % 2 != 0 || Hq % Hkv != 0 || (Hq / Hkv) % 2 != 0)
    return fail(DIFFATTN_ERR_SHAPE, "%s: need Hq even, Hq %% Hkv == 0 and Hq/Hkv even (got Hq=%d Hkv=%d)",
                fn, Hq, Hkv);
  if (d != 128) return fail(DIFFATTN_ERR_SHAPE, "%s: need d = 128 (got %d)", fn, d);
  const long long tiles = (static_cast<long long>(max_seqlen_q) + 127) / 128 * B * (Hq / 2);
  if (tiles * 2 > 0x7fffffffLL)
    return fail(DIFFATTN_ERR_SHAPE, "%s: problem too large for one launch", fn);
  if (!aligned(q, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(out, 16) ||
      !aligned(lam_logit, 4) || !aligned(cu_seqlens_q, 4) || !aligned(seqlens_k, 4) ||
      !aligned(block_table, 4))
    return fail(DIFFATTN_ERR_ALIGN, "%s: tensors must be 16-byte aligned", fn);
  rc = check_device();
  if (rc) return rc;
  da::Problem p{};
  p.q = q;
  p.k = k_pool;
  p.v = v_pool;
  p.out = out;
  p.B = B;
  p.N = max_seqlen_q;
  p.units = Hq / 2;
  p.dqk = d;
  p.dv = d;
  p.mode = da::MODE_V2;
  p.q_heads = Hq;
  p.kv_heads = Hkv;
  p.q_cols = d;
  p.k_cols = d;
  p.group = Hq / Hkv;
  p.lam_logit = lam_logit;
  p.flags = flags & DIFFATTN_CAUSAL;
  p.scale = 1.0f / std::sqrt(static_cast<float>(d));
  p.cu_seqlens = cu_seqlens_q;
  p.total = total_q;
  p.max_seqlen_k = max_seqlen_k;
  p.seqlens_k = seqlens_k;
  p.block_table = block_table;
  p.page_size = page_size;
  p.max_pages = max_pages;
  p.num_pages = num_pages;
  if (!(flags & DIFFATTN_EXACT)) return run_v2_pair(p, fn, static_cast<cudaStream_t>(stream));
  return run_prefill(p, dtype, fn, static_cast<cudaStream_t>(stream));
}

DIFFATTN_API int diffattn_fwd_fp8(const void* q, const void* k, const void* v, void* out,
                                  float q_descale, float k_descale, const float* lambda,
                                  float lambda_init, const float* norm_weight, float eps, int B,
                                  int N, int H, int d, int dv, int flags, void* stream) {
  if (!q || !k || !v || !out || !lambda) return fail(DIFFATTN_ERR_ARG, "diffattn_fwd_fp8: null pointer");
  constexpr int kF8Flags = DIFFATTN_CAUSAL | DIFFATTN_NORM | DIFFATTN_SCALE;
  if (flags & ~kF8Flags) return fail(DIFFATTN_ERR_ARG, "diffattn_fwd_fp8: unknown flag bits 0x%x", flags);
  if ((flags & DIFFATTN_NORM) && !(eps > 0.f))
    return fail(DIFFATTN_ERR_ARG, "diffattn_fwd_fp8: eps must be > 0 with DIFFATTN_NORM");
  if (!(q_descale > 0.f) || !(k_descale > 0.f) || !std::isfinite(q_descale) || !std::isfinite(k_descale))
    return fail(DIFFATTN_ERR_ARG, "diffattn_fwd_fp8: descale factors must be finite and > 0");
  if (B < 1 || N < 1 || H < 1) return fail(DIFFATTN_ERR_SHAPE, "diffattn_fwd_fp8: B, N, H must be >= 1");
  if (d != 128 || dv != 256)
    return fail(DIFFATTN_ERR_SHAPE, "diffattn_fwd_fp8: need d = 128 and dv = 256 (got d=%d dv=%d)", d, dv);
  const long long tiles = (static_cast<long long>(N) + 127) / 128 * B * H;
  if (tiles * 2 > 0x7fffffffLL || static_cast<long long>(N) * H > (1LL << 30))
    return fail(DIFFATTN_ERR_SHAPE, "diffattn_fwd_fp8: problem too large for one launch");
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
      !aligned(lambda, 4) || (norm_weight && !aligned(norm_weight, 16)))
    return fail(DIFFATTN_ERR_ALIGN, "diffattn_fwd_fp8: tensors must be 16-byte aligned");
  int rc = check_device();
  if (rc) return rc;
  da::Problem p{};
  p.q = q;
  p.k = k;
  p.v = v;
  p.out = out;
  p.B = B;
  p.N = N;
  p.units = H;
  p.dqk = d;
  p.dv = dv;
  p.mode = da::MODE_V1;
  p.q_heads = H;
  p.kv_heads = H;
  p.q_cols = 2 * d;
  p.k_cols = 2 * d;
  p.group = 1;
  p.lambda = lambda;
  p.norm_w = norm_weight;
  p.eps = eps;
  p.lambda_init = lambda_init;
  p.flags = flags;
  p.scale = q_descale * k_descale / std::sqrt(static_cast<float>(d));
  p.qk_fp8 = true;
  return run_prefill(p, DIFFATTN_BF16, "diffattn_fwd_fp8", static_cast<cudaStream_t>(stream));
}

DIFFATTN_API int diffattn_fwd_strided(const void* q, const void* k, const void* v, void* out,
                                      const long long* strides, const float* lambda,
                                      float lambda_init, const float* norm_weight, float eps,
                                      int B, int N, int H, int d, int dv, int flags, int dtype,
                                      void* stream) {
  if (!strides) return fail(DIFFATTN_ERR_ARG, "diffattn_fwd_strided: null strides");
  if (!q || !k || !v || !out || !lambda) return fail(DIFFATTN_ERR_ARG, "diffattn_fwd_strided: null pointer");
  if (flags & ~kPrefillFlags) return fail(DIFFATTN_ERR_ARG, "diffattn_fwd_strided: unknown flag bits 0x%x", flags);
  if ((flags & DIFFATTN_NORM) && !(eps > 0.f))
    return fail(DIFFATTN_ERR_ARG, "diffattn_fwd_strided: eps must be > 0 with DIFFATTN_NORM");
  if (dtype != DIFFATTN_BF16 && dtype != DIFFATTN_FP32)
    return fail(DIFFATTN_ERR_DTYPE, "diffattn_fwd_strided: dtype must be DIFFATTN_BF16 or DIFFATTN_FP32");
  if (B < 1 || N < 1 || H < 1) return fail(DIFFATTN_ERR_SHAPE, "diffattn_fwd_strided: B, N, H must be >= 1");
  if (!(d == 64 || d == 128) || dv != 2 * d)
    return fail(DIFFATTN_ERR_SHAPE, "diffattn_fwd_strided: need d in {64, 128} and dv = 2d");
  const long long tiles = (static_cast<long long>(N) + 127) / 128 * B * H;
  if (tiles * 2 > 0x7fffffffLL || static_cast<long long>(N) * H > (1LL << 30))
    return fail(DIFFATTN_ERR_SHAPE, "diffattn_fwd_strided: problem too large for one launch");
  // strides: positive, and multiples of 16 bytes (the tensor-map rule) for bf16
  const long long align_elems = dtype == DIFFATTN_BF16 ? 8 : 4;
  for (int i = 0; i < 12; ++i)
    if (strides[i] < 1 || strides[i] % align_elems != 0 || strides[i] > (1LL << 36))
      return fail(DIFFATTN_ERR_ALIGN, "diffattn_fwd_strided: stride %d (%lld) must be a positive multiple of 16 bytes", i, strides[i]);
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
      !aligned(lambda, 4) || (norm_weight && !aligned(norm_weight, 16)))
    return fail(DIFFATTN_ERR_ALIGN, "diffattn_fwd_strided: tensors must be 16-byte aligned");
  int rc = check_device();
  if (rc) return rc;
  da::Problem p{};
  p.q = q;
  p.k = k;
  p.v = v;
  p.out = out;
  p.B = B;
  p.N = N;
  p.units = H;
  p.dqk = d;
  p.dv = dv;
  p.mode = da::MODE_V1;
  p.q_heads = H;
  p.kv_heads = H;
  p.q_cols = 2 * d;
  p.k_cols = 2 * d;
  p.group = 1;
  p.lambda = lambda;
  p.norm_w = norm_weight;
  p.eps = eps;
  p.lambda_init = lambda_init;
  p.flags = flags;
  p.scale = 1.0f / std::sqrt(static_cast<float>(d));
  for (int i = 0; i < 3; ++i) {
    p.qs[i] = strides[i];
    p.ks[i] = strides[3 + i];
    p.vs[i] = strides[6 + i];
    p.os[i] = strides[9 + i];
  }
  return run_prefill(p, dtype, "diffattn_fwd_strided", static_cast<cudaStream_t>(stream));
}

namespace {
// one chunk of diffattn_fwd_host: the fused-lambda exact prefill on device slot buffers
cudaError_t host_chunk_prefill(const da::HostPipeArgs& a, const void* q, const void* k,
                               const void* v, void* out, int nb, cudaStream_t s, void* ctx) {
  da::Problem p{};
  p.q = q;
  p.k = k;
  p.v = v;
  p.out = out;
  p.B = nb;
  p.N = a.N;
  p.units = a.H;
  p.dqk = a.d;
  p.dv = a.dv;
  p.mode = da::MODE_V1;
  p.q_heads = a.H;
  p.kv_heads = a.H;
  p.q_cols = 2 * a.d;
  p.k_cols = 2 * a.d;
  p.group = 1;
  p.norm_w = a.norm_w;
  p.eps = a.eps;
  p.lambda_init = diffattn_lambda_init(a.layer);
  p.flags = a.flags;
  p.scale = 1.0f / std::sqrt(static_cast<float>(a.d));
  for (int i = 0; i < 4; ++i) p.lam_vec[i] = a.lam_vec[i];
  p.lam_dim = a.lam_dim;
  p.lam_sets = a.lam_sets;
  da::fill_dense_strides(p);
  char* err = static_cast<char*>(ctx);
  return da::launch_prefill_exact(p, s, err, 256);
}

// one piece of diffattn_fwd_host: `rows` queries at the end of `keys` keys of one sequence (the
// key-offset form of the exact prefill, lambda formed in the kernel)
cudaError_t host_piece_prefill(const da::HostPipeArgs& a, const void* q, const void* k,
                               const void* v, void* out, int rows, int keys, const int* cu_q,
                               const int* cu_k, cudaStream_t s, void* ctx) {
  da::Problem p{};
  p.q = q;
  p.k = k;
  p.v = v;
  p.out = out;
  p.B = 1;
  p.N = rows;
  p.units = a.H;
  p.dqk = a.d;
  p.dv = a.dv;
  p.mode = da::MODE_V1;
  p.q_heads = a.H;
  p.kv_heads = a.H;
  p.q_cols = 2 * a.d;
  p.k_cols = 2 * a.d;
  p.group = 1;
  p.norm_w = a.norm_w;
  p.eps = a.eps;
  p.lambda_init = diffattn_lambda_init(a.layer);
  p.flags = a.flags;
  p.scale = 1.0f / std::sqrt(static_cast<float>(a.d));
  for (int i = 0; i < 4; ++i) p.lam_vec[i] = a.lam_vec[i];
  p.lam_dim = a.lam_dim;
  p.lam_sets = a.lam_sets;
  p.cu_seqlens = cu_q;
  p.total = rows;
  p.cu_seqlens_k = cu_k;
  p.total_k = keys;
  p.max_seqlen_k = keys;
  da::fill_dense_strides(p);
  char* err = static_cast<char*>(ctx);
  return da::launch_prefill_exact(p, s, err, 256);
}
}  // namespace

DIFFATTN_API int diffattn_fwd_host_workspace_size(int B, int N, int H, int d, int dv, size_t* bytes) {
  if (!bytes) return fail(DIFFATTN_ERR_ARG, "diffattn_fwd_host_workspace_size: null pointer");
  if (B < 1 || N < 1 || H < 1 || !(d == 64 || d == 128) || dv != 2 * d)
    return fail(DIFFATTN_ERR_SHAPE, "diffattn_fwd_host_workspace_size: need B, N, H >= 1, d in {64, 128}, dv = 2d");
  *bytes = da::host_workspace_bytes(B, N, H, d, dv);
  return ok();
}

DIFFATTN_API int diffattn_fwd_host(const void* q_host, const void* k_host, const void* v_host,
                                   void* out_host, const float* lq1, const float* lk1,
                                   const float* lq2, const float* lk2, int lambda_dim,
                                   int lambda_sets, int layer, const float* norm_weight,
                                   float eps, int B, int N, int H, int d, int dv, int flags,
                                   void* workspace, size_t ws_bytes, void* stream) {
  if (!q_host || !k_host || !v_host || !out_host || !lq1 || !lk1 || !lq2 || !lk2)
    return fail(DIFFATTN_ERR_ARG, "diffattn_fwd_host: null pointer");
  constexpr int kHostFlags = DIFFATTN_CAUSAL | DIFFATTN_NORM | DIFFATTN_SCALE;
  if (flags & ~kHostFlags) return fail(DIFFATTN_ERR_ARG, "diffattn_fwd_host: unknown flag bits 0x%x", flags);
  if ((flags & DIFFATTN_NORM) && !(eps > 0.f))
    return fail(DIFFATTN_ERR_ARG, "diffattn_fwd_host: eps must be > 0 with DIFFATTN_NORM");
  if (layer < 1) return fail(DIFFATTN_ERR_ARG, "diffattn_fwd_host: layer must be >= 1");
  if (lambda_dim < 1 || lambda_dim > 4096 || !(lambda_sets == 1 || lambda_sets == H))
    return fail(DIFFATTN_ERR_SHAPE, "diffattn_fwd_host: need 1 <= lambda_dim <= 4096 and lambda_sets in {1, H}");
  if (B < 1 || N < 1 || H < 1) return fail(DIFFATTN_ERR_SHAPE, "diffattn_fwd_host: B, N, H must be >= 1");
  if (!(d == 64 || d == 128) || dv != 2 * d)
    return fail(DIFFATTN_ERR_SHAPE, "diffattn_fwd_host: need d in {64, 128} and dv = 2d");
  if (static_cast<long long>(N) * H > (1LL << 30))
    return fail(DIFFATTN_ERR_SHAPE, "diffattn_fwd_host: problem too large for one launch");
  if (!aligned(lq1, 4) || !aligned(lk1, 4) || !aligned(lq2, 4) || !aligned(lk2, 4) ||
      (norm_weight && !aligned(norm_weight, 16)))
    return fail(DIFFATTN_ERR_ALIGN, "diffattn_fwd_host: tensors must be aligned");
  const size_t need = da::host_workspace_bytes(B, N, H, d, dv);
  if (!workspace || ws_bytes < need || !aligned(workspace, 256))
    return fail(DIFFATTN_ERR_WORKSPACE, "diffattn_fwd_host: need a 256-byte aligned workspace of %zu bytes", need);
  int rc = check_device();
  if (rc) return rc;
  da::HostPipeArgs a{};
  a.q = q_host;
  a.k = k_host;
  a.v = v_host;
  a.out = out_host;
  a.B = B;
  a.N = N;
  a.H = H;
  a.d = d;
  a.dv = dv;
  a.workspace = workspace;
  a.lam_vec[0] = lq1;
  a.lam_vec[1] = lk1;
  a.lam_vec[2] = lq2;
  a.lam_vec[3] = lk2;
  a.lam_dim = lambda_dim;
  a.lam_sets = lambda_sets;
  a.layer = layer;
  a.norm_w = norm_weight;
  a.eps = eps;
  a.flags = flags;
  char err[256] = {0};
  cudaError_t e = da::launch_host_pipeline(a, static_cast<cudaStream_t>(stream), host_chunk_prefill,
                                           host_piece_prefill, err);
  if (err[0]) return fail(DIFFATTN_ERR_CUDA, "diffattn_fwd_host: %s", err);
  if (e != cudaSuccess) return cuda_fail(e, "diffattn_fwd_host");
  return ok();
}

// ---------------------------------------------------------------------------------------------
// grouped differential attention: n_signal heads, each subtracting the map of one of n_noise
// shared noise heads (contiguous groups of G = n_signal / n_noise)
// ---------------------------------------------------------------------------------------------
static int check_groups(const char* fn, int n_signal, int n_noise) {
  if (n_signal < 1 || n_noise < 1 || n_signal % n_noise != 0 || n_signal > 65535)
    return fail(DIFFATTN_ERR_SHAPE, "%s: need n_signal a multiple of n_noise >= 1 (got %d, %d)", fn,
                n_signal, n_noise);
  return 0;
}

DIFFATTN_API int diffattn_gda_fwd_workspace_size(int B, int N, int n_signal, int n_noise, int d,
                                                 int dv, size_t* bytes) {
  const char* fn = "diffattn_gda_fwd_workspace_size";
  if (!bytes) return fail(DIFFATTN_ERR_ARG, "%s: null pointer", fn);
  if (B < 1 || N < 1) return fail(DIFFATTN_ERR_SHAPE, "%s: B, N must be >= 1", fn);
  if (int rc = check_groups(fn, n_signal, n_noise)) return rc;
  if (!(d == 64 || d == 128) || dv != 2 * d)
    return fail(DIFFATTN_ERR_SHAPE, "%s: need d in {64, 128} and dv = 2d", fn);
  // one fp32 row statistic per (sequence, noise head, row padded to the 128-row tile); d = 64
  // runs in one launch and needs none
  *bytes = d == 128 ? static_cast<size_t>(B) * n_noise * ((N + 127) / 128 * 128) * sizeof(float)
                    : 0;
  return ok();
}

DIFFATTN_API int diffattn_gda_fwd(const void* q, const void* k, const void* v, void* out,
                                  const float* lambda, float lambda_init, const float* norm_weight,
                                  float eps, int B, int N, int n_signal, int n_noise, int d, int dv,
                                  int flags, int dtype, void* workspace, size_t ws_bytes,
                                  void* stream) {
  const char* fn = "diffattn_gda_fwd";
  if (!q || !k || !v || !out || !lambda) return fail(DIFFATTN_ERR_ARG, "%s: null pointer", fn);
  if (flags & ~kPrefillFlags) return fail(DIFFATTN_ERR_ARG, "%s: unknown flag bits 0x%x", fn, flags);
  if ((flags & DIFFATTN_NORM) && !(eps > 0.f))
    return fail(DIFFATTN_ERR_ARG, "%s: eps must be > 0 with DIFFATTN_NORM", fn);
  if (dtype != DIFFATTN_BF16 && dtype != DIFFATTN_FP32)
    return fail(DIFFATTN_ERR_DTYPE, "%s: dtype must be DIFFATTN_BF16 or DIFFATTN_FP32", fn);
  if (B < 1 || N < 1) return fail(DIFFATTN_ERR_SHAPE, "%s: B, N must be >= 1", fn);
  if (int rc = check_groups(fn, n_signal, n_noise)) return rc;
  if (!(d == 64 || d == 128) || dv != 2 * d)
    return fail(DIFFATTN_ERR_SHAPE, "%s: need d in {64, 128} and dv = 2d (got d=%d dv=%d)", fn, d, dv);
  const int heads = n_signal + n_noise;
  const long long tiles = (static_cast<long long>(N) + 127) / 128 * B * n_signal;
  if (tiles * 2 > 0x7fffffffLL || static_cast<long long>(N) * heads > (1LL << 30))
    return fail(DIFFATTN_ERR_SHAPE, "%s: problem too large for one launch", fn);
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
      !aligned(lambda, 4) || (norm_weight && !aligned(norm_weight, 16)))
    return fail(DIFFATTN_ERR_ALIGN, "%s: tensors must be 16-byte aligned", fn);
  // a workspace selects the two-launch form (tensor-core path, d = 128)
  const bool simt = (flags & DIFFATTN_CUDA_CORES) || dtype == DIFFATTN_FP32;
  const bool two_launch = workspace && d == 128 && !simt && !(flags & DIFFATTN_SINGLE_PASS);
  if (two_launch) {
    size_t need = 0;
    diffattn_gda_fwd_workspace_size(B, N, n_signal, n_noise, d, dv, &need);
    if (ws_bytes < need || !aligned(workspace, 256))
      return fail(DIFFATTN_ERR_WORKSPACE, "%s: need a 256-byte aligned workspace of %zu bytes", fn,
                  need);
  }
  int rc = check_device();
  if (rc) return rc;
  da::Problem p{};
  p.q = q;
  p.k = k;
  p.v = v;
  p.out = out;
  p.B = B;
  p.N = N;
  p.units = n_signal;
  p.dqk = d;
  p.dv = dv;
  p.mode = da::MODE_GDA;
  p.q_heads = heads;
  p.kv_heads = heads;
  p.q_cols = d;
  p.k_cols = d;
  p.group = n_signal / n_noise;
  p.lambda = lambda;
  p.lam_logit = nullptr;
  p.norm_w = norm_weight;
  p.eps = eps;
  p.lambda_init = lambda_init;
  p.flags = flags;
  p.scale = 1.0f / std::sqrt(static_cast<float>(d));
  if (two_launch) p.gda_noise = static_cast<float*>(workspace);
  return run_prefill(p, dtype, fn, static_cast<cudaStream_t>(stream));
}

DIFFATTN_API int diffattn_gda_fwd_fp8(const void* q, const void* k, const void* v, void* out,
                                      float q_descale, float k_descale, const float* lambda,
                                      float lambda_init, const float* norm_weight, float eps,
                                      int B, int N, int n_signal, int n_noise, int d, int dv,
                                      int flags, void* stream) {
  const char* fn = "diffattn_gda_fwd_fp8";
  if (!q || !k || !v || !out || !lambda) return fail(DIFFATTN_ERR_ARG, "%s: null pointer", fn);
  constexpr int kF8Flags = DIFFATTN_CAUSAL | DIFFATTN_NORM | DIFFATTN_SCALE;
  if (flags & ~kF8Flags) return fail(DIFFATTN_ERR_ARG, "%s: unknown flag bits 0x%x", fn, flags);
  if ((flags & DIFFATTN_NORM) && !(eps > 0.f))
    return fail(DIFFATTN_ERR_ARG, "%s: eps must be > 0 with DIFFATTN_NORM", fn);
  if (!(q_descale > 0.f) || !(k_descale > 0.f) || !std::isfinite(q_descale) ||
      !std::isfinite(k_descale))
    return fail(DIFFATTN_ERR_ARG, "%s: descale factors must be finite and > 0", fn);
  if (B < 1 || N < 1) return fail(DIFFATTN_ERR_SHAPE, "%s: B, N must be >= 1", fn);
  if (int rc = check_groups(fn, n_signal, n_noise)) return rc;
  if (d != 128 || dv != 256)
    return fail(DIFFATTN_ERR_SHAPE, "%s: need d = 128 and dv = 256 (got d=%d dv=%d)", fn, d, dv);
  const int heads = n_signal + n_noise;
  const long long tiles = (static_cast<long long>(N) + 127) / 128 * B * n_signal;
  if (tiles * 2 > 0x7fffffffLL || static_cast<long long>(N) * heads > (1LL << 30))
    return fail(DIFFATTN_ERR_SHAPE, "%s: problem too large for one launch", fn);
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
      !aligned(lambda, 4) || (norm_weight && !aligned(norm_weight, 16)))
    return fail(DIFFATTN_ERR_ALIGN, "%s: tensors must be 16-byte aligned", fn);
  int rc = check_device();
  if (rc) return rc;
  da::Problem p{};
  p.q = q;
  p.k = k;
  p.v = v;
  p.out = out;
  p.B = B;
  p.N = N;
  p.units = n_signal;
  p.dqk = d;
  p.dv = dv;
  p.mode = da::MODE_GDA;
  p.q_heads = heads;
  p.kv_heads = heads;
  p.q_cols = d;
  p.k_cols = d;
  p.group = n_signal / n_noise;
  p.lambda = lambda;
  p.lam_logit = nullptr;
  p.norm_w = norm_weight;
  p.eps = eps;
  p.lambda_init = lambda_init;
  p.flags = flags;
  p.scale = q_descale * k_descale / std::sqrt(static_cast<float>(d));
  p.qk_fp8 = true;
  return run_prefill(p, DIFFATTN_BF16, fn, static_cast<cudaStream_t>(stream));
}

DIFFATTN_API int diffattn_gda_fwd_train(const void* q, const void* k, const void* v, void* out,
                                        void* o_pre, float* stats, const float* lambda,
                                        float lambda_init, const float* norm_weight, float eps,
                                        int B, int N, int n_signal, int n_noise, int d, int dv,
                                        int flags, int dtype, void* workspace, size_t ws_bytes,
                                        void* stream) {
  const char* fn = "diffattn_gda_fwd_train";
  if (!q || !k || !v || !out || !o_pre || !stats || !lambda)
    return fail(DIFFATTN_ERR_ARG, "%s: null pointer", fn);
  constexpr int kTrainFlags = DIFFATTN_CAUSAL | DIFFATTN_NORM | DIFFATTN_SCALE;
  if (flags & ~kTrainFlags) return fail(DIFFATTN_ERR_ARG, "%s: unknown flag bits 0x%x", fn, flags);
  if ((flags & DIFFATTN_NORM) && !(eps > 0.f))
    return fail(DIFFATTN_ERR_ARG, "%s: eps must be > 0 with DIFFATTN_NORM", fn);
  if (int rc = check_groups(fn, n_signal, n_noise)) return rc;
  if (int rc = check_train_shape(fn, B, N, n_signal + n_noise, d, dv, dtype)) return rc;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
      !aligned(o_pre, 16) || !aligned(stats, 16) || !aligned(lambda, 4) ||
      (norm_weight && !aligned(norm_weight, 16)))
    return fail(DIFFATTN_ERR_ALIGN, "%s: tensors must be 16-byte aligned", fn);
  if (workspace) {
    size_t need = 0;
    diffattn_gda_fwd_workspace_size(B, N, n_signal, n_noise, d, dv, &need);
    if (ws_bytes < need || !aligned(workspace, 256))
      return fail(DIFFATTN_ERR_WORKSPACE, "%s: need a 256-byte aligned workspace of %zu bytes", fn,
                  need);
  }
  int rc = check_device();
  if (rc) return rc;
  da::Problem p{};
  p.q = q;
  p.k = k;
  p.v = v;
  p.out = out;
  p.B = B;
  p.N = N;
  p.units = n_signal;
  p.dqk = d;
  p.dv = dv;
  p.mode = da::MODE_GDA;
  p.q_heads = n_signal + n_noise;
  p.kv_heads = n_signal + n_noise;
  p.q_cols = d;
  p.k_cols = d;
  p.group = n_signal / n_noise;
  p.lambda = lambda;
  p.lam_logit = nullptr;
  p.norm_w = norm_weight;
  p.eps = eps;
  p.lambda_init = lambda_init;
  p.flags = flags;
  p.scale = 1.0f / std::sqrt(static_cast<float>(d));
  p.stats = stats;
  p.o_pre = o_pre;
  p.n_pad = (N + 127) / 128 * 128;
  if (workspace) p.gda_noise = static_cast<float*>(workspace);
  return run_prefill(p, dtype, fn, static_cast<cudaStream_t>(stream));
}

DIFFATTN_API int diffattn_gda_bwd_workspace_size(int B, int N, int n_signal, int n_noise, int d,
                                                 int dv, size_t* bytes) {
  const char* fn = "diffattn_gda_bwd_workspace_size";
  if (!bytes) return fail(DIFFATTN_ERR_ARG, "%s: null pointer", fn);
  if (int rc = check_groups(fn, n_signal, n_noise)) return rc;
  if (int rc = check_train_shape(fn, B, N, n_signal + n_noise, d, dv, DIFFATTN_BF16)) return rc;
  *bytes = da::backward_workspace_bytes(B, N, n_signal, static_cast<long long>(B) * N, true);
  return ok();
}

DIFFATTN_API int diffattn_gda_bwd(const void* q, const void* k, const void* v, const void* o_pre,
                                  const float* stats, const void* dout, const float* lambda,
                                  float lambda_init, const float* norm_weight, float eps, void* dq,
                                  void* dk, void* dv, float* dlambda, float* dnorm_weight, int B,
                                  int N, int n_signal, int n_noise, int d, int dv_width, int flags,
                                  int dtype, void* workspace, size_t ws_bytes, void* stream) {
  const char* fn = "diffattn_gda_bwd";
  if (int rc = check_groups(fn, n_signal, n_noise)) return rc;
  if (int rc = check_train_shape(fn, B, N, n_signal + n_noise, d, dv_width, dtype)) return rc;
  return bwd_impl(fn, q, k, v, o_pre, stats, dout, lambda, lambda_init, norm_weight, eps, dq, dk,
                  dv, dlambda, dnorm_weight, B, N, n_signal, d, dv_width, flags, dtype, nullptr, 0,
                  workspace, ws_bytes, stream, n_noise);
}

DIFFATTN_API int diffattn_gda_fwd_train_varlen(const void* q, const void* k, const void* v,
                                               void* out, void* o_pre, float* stats,
                                               const int* cu_seqlens, int max_seqlen, int total,
                                               const float* lambda, float lambda_init,
                                               const float* norm_weight, float eps, int B,
                                               int n_signal, int n_noise, int d, int dv, int flags,
                                               int dtype, void* workspace, size_t ws_bytes,
                                               void* stream) {
  const char* fn = "diffattn_gda_fwd_train_varlen";
  if (!q || !k || !v || !out || !o_pre || !stats || !cu_seqlens || !lambda)
    return fail(DIFFATTN_ERR_ARG, "%s: null pointer", fn);
  constexpr int kTrainFlags = DIFFATTN_CAUSAL | DIFFATTN_NORM | DIFFATTN_SCALE;
  if (flags & ~kTrainFlags) return fail(DIFFATTN_ERR_ARG, "%s: unknown flag bits 0x%x", fn, flags);
  if ((flags & DIFFATTN_NORM) && !(eps > 0.f))
    return fail(DIFFATTN_ERR_ARG, "%s: eps must be > 0 with DIFFATTN_NORM", fn);
  if (int rc = check_groups(fn, n_signal, n_noise)) return rc;
  const int heads = n_signal + n_noise;
  if (int rc = check_train_shape(fn, B, max_seqlen, heads, d, dv, dtype)) return rc;
  if (total < max_seqlen || static_cast<long long>(total) * heads > (1LL << 30))
    return fail(DIFFATTN_ERR_SHAPE, "%s: need max_seqlen <= total and total * heads <= 2^30", fn);
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
      !aligned(o_pre, 16) || !aligned(stats, 16) || !aligned(lambda, 4) ||
      !aligned(cu_seqlens, 4) || (norm_weight && !aligned(norm_weight, 16)))
    return fail(DIFFATTN_ERR_ALIGN, "%s: tensors must be 16-byte aligned", fn);
  if (workspace) {  // the noise maps' statistics of B sequences of up to max_seqlen rows
    size_t need = 0;
    diffattn_gda_fwd_workspace_size(B, max_seqlen, n_signal, n_noise, d, dv, &need);
    if (ws_bytes < need || !aligned(workspace, 256))
      return fail(DIFFATTN_ERR_WORKSPACE, "%s: need a 256-byte aligned workspace of %zu bytes", fn,
                  need);
  }
  int rc = check_device();
  if (rc) return rc;
  da::Problem p{};
  p.q = q;
  p.k = k;
  p.v = v;
  p.out = out;
  p.B = B;
  p.N = max_seqlen;
  p.units = n_signal;
  p.dqk = d;
  p.dv = dv;
  p.mode = da::MODE_GDA;
  p.q_heads = heads;
  p.kv_heads = heads;
  p.q_cols = d;
  p.k_cols = d;
  p.group = n_signal / n_noise;
  p.lambda = lambda;
  p.lam_logit = nullptr;
  p.norm_w = norm_weight;
  p.eps = eps;
  p.lambda_init = lambda_init;
  p.flags = flags;
  p.scale = 1.0f / std::sqrt(static_cast<float>(d));
  p.stats = stats;
  p.o_pre = o_pre;
  p.n_pad = (max_seqlen + 127) / 128 * 128;
  p.cu_seqlens = cu_seqlens;
  p.total = total;
  if (workspace) p.gda_noise = static_cast<float*>(workspace);
  return run_prefill(p, dtype, fn, static_cast<cudaStream_t>(stream));
}

DIFFATTN_API int diffattn_gda_bwd_varlen_workspace_size(int B, int max_seqlen, int total,
                                                        int n_signal, int n_noise, int d, int dv,
                                                        size_t* bytes) {
  const char* fn = "diffattn_gda_bwd_varlen_workspace_size";
  if (!bytes) return fail(DIFFATTN_ERR_ARG, "%s: null pointer", fn);
  if (int rc = check_groups(fn, n_signal, n_noise)) return rc;
  if (int rc = check_train_shape(fn, B, max_seqlen, n_signal + n_noise, d, dv, DIFFATTN_BF16))
    return rc;
  if (total < max_seqlen) return fail(DIFFATTN_ERR_SHAPE, "%s: need max_seqlen <= total", fn);
  *bytes = da::backward_workspace_bytes(B, max_seqlen, n_signal, total, true);
  return ok();
}

DIFFATTN_API int diffattn_gda_bwd_varlen(const void* q, const void* k, const void* v,
                                         const void* o_pre, const float* stats, const void* dout,
                                         const int* cu_seqlens, int max_seqlen, int total,
                                         const float* lambda, float lambda_init,
                                         const float* norm_weight, float eps, void* dq, void* dk,
                                         void* dv, float* dlambda, float* dnorm_weight, int B,
                                         int n_signal, int n_noise, int d, int dv_width, int flags,
                                         int dtype, void* workspace, size_t ws_bytes,
                                         void* stream) {
  const char* fn = "diffattn_gda_bwd_varlen";
  if (!cu_seqlens) return fail(DIFFATTN_ERR_ARG, "%s: null pointer", fn);
  if (int rc = check_groups(fn, n_signal, n_noise)) return rc;
  const int heads = n_signal + n_noise;
  if (int rc = check_train_shape(fn, B, max_seqlen, heads, d, dv_width, dtype)) return rc;
  if (total < max_seqlen || static_cast<long long>(total) * heads > (1LL << 30))
    return fail(DIFFATTN_ERR_SHAPE, "%s: need max_seqlen <= total and total * heads <= 2^30", fn);
  return bwd_impl(fn, q, k, v, o_pre, stats, dout, lambda, lambda_init, norm_weight, eps, dq, dk,
                  dv, dlambda, dnorm_weight, B, max_seqlen, n_signal, d, dv_width, flags, dtype,
                  cu_seqlens, total, workspace, ws_bytes, stream, n_noise);
}

DIFFATTN_API int diffattn_gda_fwd_varlen(const void* q, const void* k, const void* v, void* out,
                                         const int* cu_seqlens, int max_seqlen, int total,
                                         const float* lambda, float lambda_init,
                                         const float* norm_weight, float eps, int B, int n_signal,
                                         int n_noise, int d, int dv, int flags, int dtype,
                                         void* workspace, size_t ws_bytes, void* stream) {
  const char* fn = "diffattn_gda_fwd_varlen";
  if (!q || !k || !v || !out || !cu_seqlens || !lambda)
    return fail(DIFFATTN_ERR_ARG, "%s: null pointer", fn);
  constexpr int kVarFlags = DIFFATTN_CAUSAL | DIFFATTN_NORM | DIFFATTN_SCALE;
  if (flags & ~kVarFlags) return fail(DIFFATTN_ERR_ARG, "%s: unknown flag bits 0x%x", fn, flags);
  if ((flags & DIFFATTN_NORM) && !(eps > 0.f))
    return fail(DIFFATTN_ERR_ARG, "%s: eps must be > 0 with DIFFATTN_NORM", fn);
  if (dtype != DIFFATTN_BF16) return fail(DIFFATTN_ERR_DTYPE, "%s: dtype must be DIFFATTN_BF16", fn);
  if (B < 1 || max_seqlen < 1 || total < 1 || max_seqlen > total)
    return fail(DIFFATTN_ERR_SHAPE, "%s: need B >= 1 and 1 <= max_seqlen <= total", fn);
  if (int rc = check_groups(fn, n_signal, n_noise)) return rc;
  if (!(d == 64 || d == 128) || dv != 2 * d)
    return fail(DIFFATTN_ERR_SHAPE, "%s: need d in {64, 128} and dv = 2d (got d=%d dv=%d)", fn, d, dv);
  const int heads = n_signal + n_noise;
  const long long tiles = (static_cast<long long>(max_seqlen) + 127) / 128 * B * n_signal;
  if (tiles * 2 > 0x7fffffffLL || static_cast<long long>(total) * heads > (1LL << 30))
    return fail(DIFFATTN_ERR_SHAPE, "%s: problem too large for one launch", fn);
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
      !aligned(lambda, 4) || !aligned(cu_seqlens, 4) || (norm_weight && !aligned(norm_weight, 16)))
    return fail(DIFFATTN_ERR_ALIGN, "%s: tensors must be 16-byte aligned", fn);
  // the workspace holds the statistics of B sequences of up to max_seqlen rows
  const bool two_launch = workspace && d == 128;
  if (two_launch) {
    size_t need = 0;
    diffattn_gda_fwd_workspace_size(B, max_seqlen, n_signal, n_noise, d, dv, &need);
    if (ws_bytes < need || !aligned(workspace, 256))
      return fail(DIFFATTN_ERR_WORKSPACE, "%s: need a 256-byte aligned workspace of %zu bytes", fn,
                  need);
  }
  int rc = check_device();
  if (rc) return rc;
  da::Problem p{};
  p.q = q;
  p.k = k;
  p.v = v;
  p.out = out;
  p.B = B;
  p.N = max_seqlen;
  p.units = n_signal;
  p.dqk = d;
  p.dv = dv;
  p.mode = da::MODE_GDA;
  p.q_heads = heads;
  p.kv_heads = heads;
  p.q_cols = d;
  p.k_cols = d;
  p.group = n_signal / n_noise;
  p.lambda = lambda;
  p.lam_logit = nullptr;
  p.norm_w = norm_weight;
  p.eps = eps;
  p.lambda_init = lambda_init;
  p.flags = flags;
  p.scale = 1.0f / std::sqrt(static_cast<float>(d));
  p.cu_seqlens = cu_seqlens;
  p.total = total;
  if (two_launch) p.gda_noise = static_cast<float*>(workspace);
  return run_prefill(p, dtype, fn, static_cast<cudaStream_t>(stream));
}

// grouped prefill with queries at the end of their keys: the keys packed with offsets of their
// own (koff) or in page pools (paged); the remaining arguments as diffattn_gda_fwd_varlen
static int gda_prefill_qk(const char* fn, const void* q, const void* k, const void* v, void* out,
                          const int* cu_q, const int* cu_k, const int* seqlens_k,
                          const int* block_table, int max_q, int max_k, int total_q, int total_k,
                          int num_pages, int page_size, int max_pages, const float* lambda,
                          float lambda_init, const float* norm_weight, float eps, int B,
                          int n_signal, int n_noise, int d, int dv, int flags, int dtype,
                          void* workspace, size_t ws_bytes, void* stream) {
  constexpr int kFlags = DIFFATTN_CAUSAL | DIFFATTN_NORM | DIFFATTN_SCALE;
  if (flags & ~kFlags) return fail(DIFFATTN_ERR_ARG, "%s: unknown flag bits 0x%x", fn, flags);
  if ((flags & DIFFATTN_NORM) && !(eps > 0.f))
    return fail(DIFFATTN_ERR_ARG, "%s: eps must be > 0 with DIFFATTN_NORM", fn);
  if (dtype != DIFFATTN_BF16) return fail(DIFFATTN_ERR_DTYPE, "%s: dtype must be DIFFATTN_BF16", fn);
  if (int rc = check_groups(fn, n_signal, n_noise)) return rc;
  if (d != 128 || dv != 256)
    return fail(DIFFATTN_ERR_SHAPE, "%s: need d = 128 and dv = 256 (got d=%d dv=%d)", fn, d, dv);
  const int heads = n_signal + n_noise;
  const long long tiles = (static_cast<long long>(max_q) + 127) / 128 * B * n_signal;
  const long long krows = block_table ? static_cast<long long>(num_pages) * page_size : total_k;
  if (tiles * 2 > 0x7fffffffLL || krows * heads > (1LL << 34) ||
      static_cast<long long>(total_q) * heads > (1LL << 30))
    return fail(DIFFATTN_ERR_SHAPE, "%s: problem too large for one launch", fn);
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
      !aligned(lambda, 4) || !aligned(cu_q, 4) || (cu_k && !aligned(cu_k, 4)) ||
      (seqlens_k && !aligned(seqlens_k, 4)) || (block_table && !aligned(block_table, 4)) ||
      (norm_weight && !aligned(norm_weight, 16)))
    return fail(DIFFATTN_ERR_ALIGN, "%s: tensors must be 16-byte aligned", fn);
  if (workspace) {  // the two-launch form: statistics of B sequences of up to max_q query rows
    size_t need = 0;
    diffattn_gda_fwd_workspace_size(B, max_q, n_signal, n_noise, d, dv, &need);
    if (ws_bytes < need || !aligned(workspace, 256))
      return fail(DIFFATTN_ERR_WORKSPACE, "%s: need a 256-byte aligned workspace of %zu bytes", fn,
                  need);
  }
  int rc = check_device();
  if (rc) return rc;
  da::Problem p{};
  p.q = q;
  p.k = k;
  p.v = v;
  p.out = out;
  p.B = B;
  p.N = max_q;
  p.units = n_signal;
  p.dqk = d;
  p.dv = dv;
  p.mode = da::MODE_GDA;
  p.q_heads = heads;
  p.kv_heads = heads;
  p.q_cols = d;
  p.k_cols = d;
  p.group = n_signal / n_noise;
  p.lambda = lambda;
  p.lam_logit = nullptr;
  p.norm_w = norm_weight;
  p.eps = eps;
  p.lambda_init = lambda_init;
  p.flags = flags;
  p.scale = 1.0f / std::sqrt(static_cast<float>(d));
  p.cu_seqlens = cu_q;
  p.total = total_q;
  p.max_seqlen_k = max_k;
  if (block_table) {
    p.seqlens_k = seqlens_k;
    p.block_table = block_table;
    p.page_size = page_size;
    p.max_pages = max_pages;
    p.num_pages = num_pages;
  } else {
    p.cu_seqlens_k = cu_k;
    p.total_k = total_k;
  }
  if (workspace) p.gda_noise = static_cast<float*>(workspace);
  return run_prefill(p, dtype, fn, static_cast<cudaStream_t>(stream));
}

DIFFATTN_API int diffattn_gda_fwd_varlen_qk(const void* q, const void* k, const void* v, void* out,
                                            const int* cu_seqlens_q, const int* cu_seqlens_k,
                                            int max_seqlen_q, int max_seqlen_k, int total_q,
                                            int total_k, const float* lambda, float lambda_init,
                                            const float* norm_weight, float eps, int B,
                                            int n_signal, int n_noise, int d, int dv, int flags,
                                            int dtype, void* workspace, size_t ws_bytes,
                                            void* stream) {
  const char* fn = "diffattn_gda_fwd_varlen_qk";
  if (!q || !k || !v || !out || !cu_seqlens_q || !cu_seqlens_k || !lambda)
    return fail(DIFFATTN_ERR_ARG, "%s: null pointer", fn);
  if (B < 1 || max_seqlen_q < 1 || total_q < 1 || max_seqlen_q > total_q ||
      max_seqlen_k < max_seqlen_q || max_seqlen_k > total_k)
    return fail(DIFFATTN_ERR_SHAPE, "%s: need B >= 1, 1 <= max_seqlen_q <= total_q and "
                "max_seqlen_q <= max_seqlen_k <= total_k", fn);
  return gda_prefill_qk(fn, q, k, v, out, cu_seqlens_q, cu_seqlens_k, nullptr, nullptr,
                        max_seqlen_q, max_seqlen_k, total_q, total_k, 0, 0, 0, lambda, lambda_init,
                        norm_weight, eps, B, n_signal, n_noise, d, dv, flags, dtype, workspace,
                        ws_bytes, stream);
}

DIFFATTN_API int diffattn_gda_fwd_paged(const void* q, const void* k_pool, const void* v_pool,
                                        void* out, const int* cu_seqlens_q, const int* seqlens_k,
                                        const int* block_table, int max_seqlen_q, int max_seqlen_k,
                                        int total_q, int num_pages, int page_size, int max_pages,
                                        const float* lambda, float lambda_init,
                                        const float* norm_weight, float eps, int B, int n_signal,
                                        int n_noise, int d, int dv, int flags, int dtype,
                                        void* workspace, size_t ws_bytes, void* stream) {
  const char* fn = "diffattn_gda_fwd_paged";
  if (!q || !k_pool || !v_pool || !out || !cu_seqlens_q || !seqlens_k || !block_table || !lambda)
    return fail(DIFFATTN_ERR_ARG, "%s: null pointer", fn);
  if (int rc = check_paged_prefill(fn, B, max_seqlen_q, max_seqlen_k, total_q, num_pages,
                                   page_size, max_pages))
    return rc;
  return gda_prefill_qk(fn, q, k_pool, v_pool, out, cu_seqlens_q, nullptr, seqlens_k,
                        block_table, max_seqlen_q, max_seqlen_k, total_q, 0, num_pages, page_size,
                        max_pages, lambda, lambda_init, norm_weight, eps, B, n_signal, n_noise, d,
                        dv, flags, dtype, workspace, ws_bytes, stream);
}

DIFFATTN_API int diffattn_gda_decode(const void* q, const void* k_cache, const void* v_cache,
                                     const int* seqlens, void* out, const float* lambda,
                                     float lambda_init, const float* norm_weight, float eps, int B,
                                     int Lmax, int n_signal, int n_noise, int d, int dv, int flags,
                                     int dtype, void* workspace, size_t ws_bytes, void* stream) {
  const char* fn = "diffattn_gda_decode";
  if (!q || !k_cache || !v_cache || !out || !lambda) return fail(DIFFATTN_ERR_ARG, "%s: null pointer", fn);
  if (flags & ~(DIFFATTN_CAUSAL | DIFFATTN_NORM | DIFFATTN_SCALE))
    return fail(DIFFATTN_ERR_ARG, "%s: unknown flag bits 0x%x", fn, flags);
  if ((flags & DIFFATTN_NORM) && !(eps > 0.f))
    return fail(DIFFATTN_ERR_ARG, "%s: eps must be > 0 with DIFFATTN_NORM", fn);
  if (dtype != DIFFATTN_BF16) return fail(DIFFATTN_ERR_DTYPE, "%s: dtype must be DIFFATTN_BF16", fn);
  if (B < 1 || Lmax < 1 || B > 65535)
    return fail(DIFFATTN_ERR_SHAPE, "%s: need 1 <= B <= 65535 and Lmax >= 1", fn);
  if (int rc = check_groups(fn, n_signal, n_noise)) return rc;
  if (d != 128 || dv != 256)
    return fail(DIFFATTN_ERR_SHAPE, "%s: need d = 128 and dv = 256 (got d=%d dv=%d)", fn, d, dv);
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
      !aligned(lambda, 4) || (seqlens && !aligned(seqlens, 4)) ||
      (norm_weight && !aligned(norm_weight, 16)))
    return fail(DIFFATTN_ERR_ALIGN, "%s: tensors must be 16-byte aligned", fn);
  const size_t need = da::decode_workspace_bytes(B, Lmax, n_signal, dv);
  if (!workspace || ws_bytes < need || !aligned(workspace, 256))
    return fail(DIFFATTN_ERR_WORKSPACE, "%s: need a 256-byte aligned workspace of %zu bytes", fn, need);
  int rc = check_device();
  if (rc) return rc;
  da::DecodeArgs a{};
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.seqlens = seqlens;
  a.out = out;
  a.lambda = lambda;
  a.lambda_init = lambda_init;
  a.norm_w = norm_weight;
  a.eps = eps;
  a.flags = flags;
  a.B = B;
  a.Lmax = Lmax;
  a.H = n_signal;
  a.d = d;
  a.dv = dv;
  a.ws = static_cast<float*>(workspace);
  a.noise_group = n_signal / n_noise;
  cudaError_t e = da::launch_decode(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, fn);
  return ok();
}

DIFFATTN_API int diffattn_gda_decode_paged(const void* q, const void* k_pool, const void* v_pool,
                                           const int* block_table, const int* seqlens, void* out,
                                           const float* lambda, float lambda_init,
                                           const float* norm_weight, float eps, int B,
                                           int n_signal, int n_noise, int d, int dv, int num_pages,
                                           int page_size, int max_pages, int flags, int dtype,
                                           void* workspace, size_t ws_bytes, void* stream) {
  const char* fn = "diffattn_gda_decode_paged";
  if (!q || !k_pool || !v_pool || !block_table || !seqlens || !out || !lambda)
    return fail(DIFFATTN_ERR_ARG, "%s: null pointer", fn);
  if (flags & ~(DIFFATTN_CAUSAL | DIFFATTN_NORM | DIFFATTN_SCALE))
    return fail(DIFFATTN_ERR_ARG, "%s: unknown flag bits 0x%x", fn, flags);
  if ((flags & DIFFATTN_NORM) && !(eps > 0.f))
    return fail(DIFFATTN_ERR_ARG, "%s: eps must be > 0 with DIFFATTN_NORM", fn);
  if (dtype != DIFFATTN_BF16) return fail(DIFFATTN_ERR_DTYPE, "%s: dtype must be DIFFATTN_BF16", fn);
  if (B < 1 || B > 65535 || num_pages < 1 || page_size < 1 || max_pages < 1)
    return fail(DIFFATTN_ERR_SHAPE, "%s: need 1 <= B <= 65535 and num_pages, page_size, max_pages >= 1", fn);
  if (int rc = check_groups(fn, n_signal, n_noise)) return rc;
  const long long lmax = static_cast<long long>(max_pages) * page_size;
  if (lmax > 0x7fffffffLL || static_cast<long long>(num_pages) * page_size > (1LL << 40))
    return fail(DIFFATTN_ERR_SHAPE, "%s: max_pages * page_size too large", fn);
  if (d != 128 || dv != 256)
    return fail(DIFFATTN_ERR_SHAPE, "%s: need d = 128 and dv = 256 (got d=%d dv=%d)", fn, d, dv);
  if (!aligned(q, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(out, 16) ||
      !aligned(lambda, 4) || !aligned(seqlens, 4) || !aligned(block_table, 4) ||
      (norm_weight && !aligned(norm_weight, 16)))
    return fail(DIFFATTN_ERR_ALIGN, "%s: tensors must be 16-byte aligned", fn);
  const int Lmax = static_cast<int>(lmax);
  const size_t need = da::decode_workspace_bytes(B, Lmax, n_signal, dv);
  if (!workspace || ws_bytes < need || !aligned(workspace, 256))
    return fail(DIFFATTN_ERR_WORKSPACE, "%s: need a 256-byte aligned workspace of %zu bytes", fn, need);
  int rc = check_device();
  if (rc) return rc;
  da::DecodeArgs a{};
  a.q = q;
  a.k_cache = k_pool;
  a.v_cache = v_pool;
  a.seqlens = seqlens;
  a.out = out;
  a.lambda = lambda;
  a.lambda_init = lambda_init;
  a.norm_w = norm_weight;
  a.eps = eps;
  a.flags = flags;
  a.B = B;
  a.Lmax = Lmax;
  a.H = n_signal;
  a.d = d;
  a.dv = dv;
  a.ws = static_cast<float*>(workspace);
  a.noise_group = n_signal / n_noise;
  a.block_table = block_table;
  a.page_size = page_size;
  a.max_pages = max_pages;
  a.num_pages = num_pages;
  cudaError_t e = da::launch_decode(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, fn);
  return ok();
}
