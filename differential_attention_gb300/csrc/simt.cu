// simt.cu -- CUDA-core kernels: lambda, and the fp32 prefill path (also serves bf16 on request).
//
// lambda: page "Differential Transformer: softmax can't say zero, so it subtracts", section
// "lambda, re-parameterised": lambda = exp(lq1 . lk1) - exp(lq2 . lk2) + lambda_init.
//
// Prefill (same page, section "The mechanism, exactly"): one warp per query row computes the
// two softmax maps with exact row statistics (pass 1: running max and sum per map; pass 2: the
// signed weights w_j = e^{s1_j - m1}/l1 - lambda e^{s2_j - m2}/l2) and accumulates w V, then
// applies the per-head RMSNorm and the (1 - lambda_init) scale ("The row no longer sums to
// one"). All arithmetic is fp32 with accurate expf, which is what the fp32 I/O path needs.
#include <cuda_bf16.h>

#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace da {

// ------------------------------------------------------------------------------------------
// lambda
// ------------------------------------------------------------------------------------------
// (lq1 . lk1, lq2 . lk2) of set `set`, reduced over the block; every thread gets both.
__device__ __forceinline__ float2 lambda_dots(const float* __restrict__ lq1,
                                              const float* __restrict__ lk1,
                                              const float* __restrict__ lq2,
                                              const float* __restrict__ lk2, int dim, int set) {
  const size_t base = static_cast<size_t>(set) * dim;
  float d1 = 0.f, d2 = 0.f;
  for (int i = threadIdx.x; i < dim; i += blockDim.x) {
    d1 = fmaf(lq1[base + i], lk1[base + i], d1);
    d2 = fmaf(lq2[base + i], lk2[base + i], d2);
  }
  __shared__ float red[2][32];
  for (int o = 16; o > 0; o >>= 1) {
    d1 += __shfl_xor_sync(0xffffffffu, d1, o);
    d2 += __shfl_xor_sync(0xffffffffu, d2, o);
  }
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) {
    red[0][w] = d1;
    red[1][w] = d2;
  }
  __syncthreads();
  float a = 0.f, b = 0.f;
  for (int i = 0; i < (int)(blockDim.x >> 5); ++i) {  // the same fixed order in every thread
    a += red[0][i];
    b += red[1][i];
  }
  return make_float2(a, b);
}

__global__ void lambda_kernel(const float* __restrict__ lq1, const float* __restrict__ lk1,
                              const float* __restrict__ lq2, const float* __restrict__ lk2,
                              int dim, float lambda_init, float* __restrict__ out) {
  const float2 d = lambda_dots(lq1, lk1, lq2, lk2, dim, blockIdx.x);
  if (threadIdx.x == 0) out[blockIdx.x] = expf(d.x) - expf(d.y) + lambda_init;
}

// Gradients of lambda = exp(lq1 . lk1) - exp(lq2 . lk2) + lambda_init with respect to the four
// vectors of each set, given g = the sum of dlambda over the set's `per_set` consecutive entries:
// dlq1 = g e1 lk1, dlk1 = g e1 lq1, dlq2 = -g e2 lk2, dlk2 = -g e2 lq2 (e_m = exp(lq_m . lk_m)).
__global__ void lambda_bwd_kernel(const float* __restrict__ lq1, const float* __restrict__ lk1,
                                  const float* __restrict__ lq2, const float* __restrict__ lk2,
                                  const float* __restrict__ dlam, int dim, int per_set,
                                  float* __restrict__ dlq1, float* __restrict__ dlk1,
                                  float* __restrict__ dlq2, float* __restrict__ dlk2) {
  const int set = blockIdx.x;
  const float2 d = lambda_dots(lq1, lk1, lq2, lk2, dim, set);
  float g = 0.f;
  for (int i = 0; i < per_set; ++i) g += dlam[static_cast<size_t>(set) * per_set + i];
  const float g1 = g * expf(d.x), g2 = -g * expf(d.y);
  const size_t base = static_cast<size_t>(set) * dim;
  for (int i = threadIdx.x; i < dim; i += blockDim.x) {
    dlq1[base + i] = g1 * lk1[base + i];
    dlk1[base + i] = g1 * lq1[base + i];
    dlq2[base + i] = g2 * lk2[base + i];
    dlk2[base + i] = g2 * lq2[base + i];
  }
}

// ------------------------------------------------------------------------------------------
// diagnostics: a bounded wait that is certain to run out
// ------------------------------------------------------------------------------------------
__global__ void wait_timeout_kernel(unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_barrier_init();
  }
  __syncthreads();
  // Nothing ever arrives on `bar`: the wait runs for limit_ns, flags DEV_TIMEOUT and returns.
  if (threadIdx.x == 0) mbar_wait_limit(smem_u32(&bar), 0, nullptr, limit_ns);
}

cudaError_t launch_wait_timeout(int limit_ms, cudaStream_t s) {
  wait_timeout_kernel<<<1, 32, 0, s>>>(static_cast<unsigned long long>(limit_ms) * 1000000ull);
  return cudaGetLastError();
}

cudaError_t status_simt(int* v) { return read_clear_status(v); }

cudaError_t launch_lambda(const float* lq1, const float* lk1, const float* lq2, const float* lk2,
                          int dim, int n_sets, float lambda_init, float* out, cudaStream_t s) {
  lambda_kernel<<<n_sets, 128, 0, s>>>(lq1, lk1, lq2, lk2, dim, lambda_init, out);
  return cudaGetLastError();
}

cudaError_t launch_lambda_bwd(const float* lq1, const float* lk1, const float* lq2,
                              const float* lk2, const float* dlam, int dim, int n_sets,
                              int per_set, float* dlq1, float* dlk1, float* dlq2, float* dlk2,
                              cudaStream_t s) {
  lambda_bwd_kernel<<<n_sets, 128, 0, s>>>(lq1, lk1, lq2, lk2, dlam, dim, per_set, dlq1, dlk1,
                                           dlq2, dlk2);
  return cudaGetLastError();
}

// ------------------------------------------------------------------------------------------
// CUDA-core prefill
// ------------------------------------------------------------------------------------------
template <typename T>
__device__ __forceinline__ float ldf(const T* p);
template <>
__device__ __forceinline__ float ldf<float>(const float* p) {
  return *p;
}
template <>
__device__ __forceinline__ float ldf<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}
template <typename T>
__device__ __forceinline__ T from_f(float x);
template <>
__device__ __forceinline__ float from_f<float>(float x) {
  return x;
}
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

constexpr int kSimtRows = 4;     // query rows (warps) per block
constexpr int kSimtMaxD = 128;   // max query/key width of one map
constexpr int kSimtMaxDv = 256;  // max value width

// Merge two (max, sum-of-exp) pairs.
__device__ __forceinline__ void merge_ml(float& m, float& l, float m2, float l2) {
  const float M = fmaxf(m, m2);
  if (M == -INFINITY) return;
  l = l * expf(m - M) + l2 * expf(m2 - M);
  m = M;
}

template <typename T>
__global__ void __launch_bounds__(kSimtRows * 32)
    prefill_simt_kernel(const Problem p) {
  __shared__ float sq[kSimtRows][2][kSimtMaxD];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i = blockIdx.x * kSimtRows + warp;
  const int u = blockIdx.y, b = blockIdx.z;
  if (i >= p.N) return;  // no block-level barrier below

  const T* q = static_cast<const T*>(p.q);
  const T* k = static_cast<const T*>(p.k);
  const T* v = static_cast<const T*>(p.v);
  const int d = p.dqk, dv = p.dv;
  for (int r = 0; r < 2; ++r) {
    const T* qr = q + elem_off(p.qs, b, i, q_head_of(p, u, r)) + q_col_of(p, r);
    for (int c = lane; c < d; c += 32) sq[warp][r][c] = ldf(qr + c);
  }
  __syncwarp();

  const int kvh = kv_head_of(p, u);  // V head
  const int kh0 = k_head_of(p, u, 0), kh1 = k_head_of(p, u, 1);
  const int kend = (p.flags & 1) ? (i + 1) : p.N;
  auto krow = [&](int j, int r) {
    return k + elem_off(p.ks, b, j, r ? kh1 : kh0) + k_col_of(p, r);
  };
  auto score = [&](int j, int r) {
    const T* kr = krow(j, r);
    float acc = 0.f;
    for (int c = 0; c < d; ++c) acc = fmaf(sq[warp][r][c], ldf(kr + c), acc);
    return acc * p.scale;
  };

  // pass 1: exact row statistics of both maps
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
  for (int j = lane; j < kend; j += 32) {
    for (int r = 0; r < 2; ++r) {
      const float s = score(j, r);
      if (s > m[r]) {
        l[r] = l[r] * expf(m[r] - s) + 1.f;
        m[r] = s;
      } else {
        l[r] += expf(s - m[r]);
      }
    }
  }
  for (int o = 16; o > 0; o >>= 1) {
    for (int r = 0; r < 2; ++r) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m[r], o);
      const float l2 = __shfl_xor_sync(0xffffffffu, l[r], o);
      merge_ml(m[r], l[r], m2, l2);
    }
  }

  float lam;
  if (p.mode != MODE_V2) {
    lam = p.lambda[u];
  } else {
    const float x = p.lam_logit[(static_cast<size_t>(b) * p.N + i) * p.units + u];
    lam = 1.f / (1.f + expf(-x));
  }
  const float inv_l1 = 1.f / l[0], lam_l2 = lam / l[1];

  // pass 2: signed weights times V
  constexpr int kMaxC = kSimtMaxDv / 32;
  float acc[kMaxC];
#pragma unroll
  for (int c = 0; c < kMaxC; ++c) acc[c] = 0.f;
  const int ncol = dv / 32;
  for (int j0 = 0; j0 < kend; j0 += 32) {
    const int j = j0 + lane;
    float w = 0.f;
    if (j < kend) w = expf(score(j, 0) - m[0]) * inv_l1 - expf(score(j, 1) - m[1]) * lam_l2;
    const int cnt = min(32, kend - j0);
    for (int jj = 0; jj < cnt; ++jj) {
      const float wj = __shfl_sync(0xffffffffu, w, jj);
      const T* vr = v + elem_off(p.vs, b, j0 + jj, kvh);
#pragma unroll
      for (int c = 0; c < kMaxC; ++c)
        if (c < ncol) acc[c] = fmaf(wj, ldf(vr + lane + 32 * c), acc[c]);
    }
  }

  // epilogue: RMSNorm over dv channels, then (1 - lambda_init)
  if (p.flags & 2) {
    float ss = 0.f;
#pragma unroll
    for (int c = 0; c < kMaxC; ++c)
      if (c < ncol) ss = fmaf(acc[c], acc[c], ss);
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float rstd = 1.f / sqrtf(ss / static_cast<float>(dv) + p.eps);
#pragma unroll
    for (int c = 0; c < kMaxC; ++c)
      if (c < ncol) acc[c] *= rstd * (p.norm_w ? p.norm_w[lane + 32 * c] : 1.f);
  }
  const float sc = (p.flags & 4) ? (1.f - p.lambda_init) : 1.f;
  T* out = static_cast<T*>(p.out);
  const size_t oo = elem_off(p.os, b, i, u);
#pragma unroll
  for (int c = 0; c < kMaxC; ++c)
    if (c < ncol) out[oo + lane + 32 * c] = from_f<T>(acc[c] * sc);
}

cudaError_t launch_prefill_simt(const Problem& p, bool is_bf16, cudaStream_t s) {
  dim3 grid((p.N + kSimtRows - 1) / kSimtRows, p.units, p.B);
  if (is_bf16)
    prefill_simt_kernel<__nv_bfloat16><<<grid, kSimtRows * 32, 0, s>>>(p);
  else
    prefill_simt_kernel<float><<<grid, kSimtRows * 32, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace da
