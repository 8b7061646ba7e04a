// decode.cu -- split-KV differential-attention decode over a bf16 KV cache.
//
// One query per sequence attends to its cached keys with both maps (page "Differential
// Transformer: softmax can't say zero, so it subtracts", section "The mechanism, exactly"). Page
// "Differential Transformer V2" notes that V1 decoding with stock kernels loads the value cache
// twice; here every cached K1|K2 row and V row is streamed from HBM exactly once and serves both
// maps.
//
// Stage 1 (decode_split_kernel, grid splits x H x B): a CTA owns one contiguous slice of one
// (b, h) cache. Each warp walks keys in groups of kG: lane t loads 16 bytes of the K row
// (columns 8t..8t+7: K1 for lanes 0-15, K2 for lanes 16-31) and 16 bytes of the V row, the score
// of each map is reduced over its 16 lanes, and both maps keep their own running max / sum and a
// 256-wide fp32 accumulator (8 columns per lane), rescaled once per group. The CTA's warps are
// merged in shared memory and one partial (m1, l1, m2, l2, o1[256], o2[256]) goes to the
// workspace.
// Stage 2 (decode_combine_kernel, grid H x B): thread c merges the partials of channel c, forms
// o1/l1 - lambda * o2/l2, and applies the per-head RMSNorm and the (1 - lambda_init) scale.
#include <cuda_bf16.h>

#include <cmath>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace da {

constexpr int kDecWarps = 8;
constexpr int kDecThreads = kDecWarps * 32;
constexpr int kG = 4;                  // keys per warp per group
constexpr int kDecWidth = 256;         // 2d = dv = 256
constexpr int kRec = 4 + 2 * kDecWidth; // floats per partial record
constexpr float kLog2e = 1.4426950408889634f;

int decode_splits(int B, int Lmax, int H, int* chunk_out) {
  // Aim for ~64 CTAs per SM-equivalent of the 152-SM part so the last wave is a small fraction.
  const long long units = static_cast<long long>(B) * H;
  long long target = (64LL * 152 + units - 1) / units;
  if (target < 1) target = 1;
  const int step = kDecWarps * kG;  // keys one CTA round covers
  long long chunk = (Lmax + target - 1) / target;
  if (chunk < 256) chunk = 256;
  chunk = (chunk + step - 1) / step * step;
  const int splits = static_cast<int>((Lmax + chunk - 1) / chunk);
  if (chunk_out) *chunk_out = static_cast<int>(chunk);
  return splits;
}

size_t decode_workspace_bytes(int B, int Lmax, int H, int dv) {
  (void)dv;
  const int S = decode_splits(B, Lmax, H, nullptr);
  return static_cast<size_t>(B) * H * S * kRec * sizeof(float);
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

struct DecSplitParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* kc;
  const __nv_bfloat16* vc;
  const int* seqlens;
  float* ws;
  int Lmax, H, splits, chunk;
  float scale_log2;
};

__global__ void __launch_bounds__(kDecThreads) decode_split_kernel(const DecSplitParams p) {
  const int s = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int L = p.seqlens ? p.seqlens[b] : p.Lmax;
  L = L < 1 ? 1 : (L > p.Lmax ? p.Lmax : L);
  const int k0 = s * p.chunk;
  const int k1 = min(k0 + p.chunk, L);

  float qf[8];
  {
    const uint4 qu = *reinterpret_cast<const uint4*>(p.q + (static_cast<size_t>(b) * p.H + h) *
                                                              kDecWidth + 8 * lane);
    bf16x8_to_f32(qu, qf);
#pragma unroll
    for (int i = 0; i < 8; ++i) qf[i] *= p.scale_log2;
  }

  float m1 = -INFINITY, l1 = 0.f, m2 = -INFINITY, l2 = 0.f;
  float o1[8], o2[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) o1[i] = o2[i] = 0.f;

  const size_t row_stride = static_cast<size_t>(p.H) * kDecWidth;  // elements between keys
  const __nv_bfloat16* kbase =
      p.kc + (static_cast<size_t>(b) * p.Lmax * p.H + h) * kDecWidth + 8 * lane;
  const __nv_bfloat16* vbase =
      p.vc + (static_cast<size_t>(b) * p.Lmax * p.H + h) * kDecWidth + 8 * lane;

  for (int g0 = k0 + warp * kG; g0 < k1; g0 += kDecWarps * kG) {
    uint4 ku[kG], vu[kG];
#pragma unroll
    for (int e = 0; e < kG; ++e) {
      const int j = min(g0 + e, k1 - 1);  // clamp keeps the load in bounds; masked below
      ku[e] = ldg_stream(kbase + static_cast<size_t>(j) * row_stride);
      vu[e] = ldg_stream(vbase + static_cast<size_t>(j) * row_stride);
    }
    float sc[kG];
#pragma unroll
    for (int e = 0; e < kG; ++e) {
      float kf[8];
      bf16x8_to_f32(ku[e], kf);
      float acc = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) acc = fmaf(qf[i], kf[i], acc);
      sc[e] = acc;
    }
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) {
#pragma unroll
      for (int e = 0; e < kG; ++e) sc[e] += __shfl_xor_sync(0xffffffffu, sc[e], o);
    }
    float s1[kG], s2[kG];
#pragma unroll
    for (int e = 0; e < kG; ++e) {
      const float other = __shfl_xor_sync(0xffffffffu, sc[e], 16);
      const bool valid = (g0 + e) < k1;
      s1[e] = valid ? (lane < 16 ? sc[e] : other) : -INFINITY;
      s2[e] = valid ? (lane < 16 ? other : sc[e]) : -INFINITY;
    }
    float gm1 = s1[0], gm2 = s2[0];
#pragma unroll
    for (int e = 1; e < kG; ++e) {
      gm1 = fmaxf(gm1, s1[e]);
      gm2 = fmaxf(gm2, s2[e]);
    }
    const float n1 = fmaxf(m1, gm1), n2 = fmaxf(m2, gm2);  // finite: key g0 is valid
    const float c1 = ex2_approx(m1 - n1), c2 = ex2_approx(m2 - n2);
    l1 *= c1;
    l2 *= c2;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      o1[i] *= c1;
      o2[i] *= c2;
    }
#pragma unroll
    for (int e = 0; e < kG; ++e) {
      const float p1 = ex2_approx(s1[e] - n1), p2 = ex2_approx(s2[e] - n2);
      l1 += p1;
      l2 += p2;
      float vf[8];
      bf16x8_to_f32(vu[e], vf);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        o1[i] = fmaf(p1, vf[i], o1[i]);
        o2[i] = fmaf(p2, vf[i], o2[i]);
      }
    }
    m1 = n1;
    m2 = n2;
  }

  // merge the CTA's warps
  __shared__ float s_o[kDecWarps][2][kDecWidth];
  __shared__ float s_ml[kDecWarps][4];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    s_o[warp][0][8 * lane + i] = o1[i];
    s_o[warp][1][8 * lane + i] = o2[i];
  }
  if (lane == 0) {
    s_ml[warp][0] = m1;
    s_ml[warp][1] = l1;
    s_ml[warp][2] = m2;
    s_ml[warp][3] = l2;
  }
  __syncthreads();
  const int c = threadIdx.x;  // channel
  float* rec = p.ws + ((static_cast<size_t>(b) * p.H + h) * p.splits + s) * kRec;
  float M[2] = {-INFINITY, -INFINITY};
#pragma unroll
  for (int w = 0; w < kDecWarps; ++w) {
    M[0] = fmaxf(M[0], s_ml[w][0]);
    M[1] = fmaxf(M[1], s_ml[w][2]);
  }
  float oa[2] = {0.f, 0.f}, la[2] = {0.f, 0.f};
#pragma unroll
  for (int w = 0; w < kDecWarps; ++w) {
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const float mw = s_ml[w][2 * r];
      if (mw != -INFINITY) {
        const float f = ex2_approx(mw - M[r]);
        la[r] = fmaf(s_ml[w][2 * r + 1], f, la[r]);
        oa[r] = fmaf(s_o[w][r][c], f, oa[r]);
      }
    }
  }
  rec[4 + c] = oa[0];
  rec[4 + kDecWidth + c] = oa[1];
  if (c == 0) {
    rec[0] = M[0];
    rec[1] = la[0];
    rec[2] = M[1];
    rec[3] = la[1];
  }
}

struct DecCombineParams {
  const float* ws;
  const float* lambda;
  const float* norm_w;
  __nv_bfloat16* out;
  float lambda_init, eps;
  int flags, H, splits;
};

__global__ void __launch_bounds__(kDecWidth) decode_combine_kernel(const DecCombineParams p) {
  const int h = blockIdx.x, b = blockIdx.y, c = threadIdx.x;
  const float* recs = p.ws + (static_cast<size_t>(b) * p.H + h) * p.splits * kRec;
  float M[2] = {-INFINITY, -INFINITY};
  for (int s = 0; s < p.splits; ++s) {
    M[0] = fmaxf(M[0], recs[s * kRec + 0]);
    M[1] = fmaxf(M[1], recs[s * kRec + 2]);
  }
  float o[2] = {0.f, 0.f}, l[2] = {0.f, 0.f};
  for (int s = 0; s < p.splits; ++s) {
    const float* r = recs + s * kRec;
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      const float ms = r[2 * m];
      if (ms != -INFINITY) {
        const float f = ex2_approx(ms - M[m]);
        l[m] = fmaf(r[2 * m + 1], f, l[m]);
        o[m] = fmaf(r[4 + m * kDecWidth + c], f, o[m]);
      }
    }
  }
  float y = o[0] / l[0] - p.lambda[h] * (o[1] / l[1]);
  if (p.flags & 2) {
    __shared__ float red[kDecWidth / 32];
    float ss = y * y;
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if ((c & 31) == 0) red[c >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int i = 0; i < kDecWidth / 32; ++i) tot += red[i];
    y *= (1.f / sqrtf(tot / static_cast<float>(kDecWidth) + p.eps)) * (p.norm_w ? p.norm_w[c] : 1.f);
  }
  if (p.flags & 4) y *= (1.f - p.lambda_init);
  p.out[(static_cast<size_t>(b) * p.H + h) * kDecWidth + c] = __float2bfloat16_rn(y);
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t st) {
  int chunk = 0;
  const int S = decode_splits(a.B, a.Lmax, a.H, &chunk);
  DecSplitParams sp;
  sp.q = static_cast<const __nv_bfloat16*>(a.q);
  sp.kc = static_cast<const __nv_bfloat16*>(a.k_cache);
  sp.vc = static_cast<const __nv_bfloat16*>(a.v_cache);
  sp.seqlens = a.seqlens;
  sp.ws = a.ws;
  sp.Lmax = a.Lmax;
  sp.H = a.H;
  sp.splits = S;
  sp.chunk = chunk;
  sp.scale_log2 = kLog2e / sqrtf(static_cast<float>(a.d));
  decode_split_kernel<<<dim3(S, a.H, a.B), kDecThreads, 0, st>>>(sp);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  DecCombineParams cp;
  cp.ws = a.ws;
  cp.lambda = a.lambda;
  cp.norm_w = a.norm_w;
  cp.out = static_cast<__nv_bfloat16*>(a.out);
  cp.lambda_init = a.lambda_init;
  cp.eps = a.eps;
  cp.flags = a.flags;
  cp.H = a.H;
  cp.splits = S;
  decode_combine_kernel<<<dim3(a.H, a.B), kDecWidth, 0, st>>>(cp);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------------------------
// Decode without a caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they decode: a plugin running
// inside a host runtime that owns every device buffer and offers no allocator, or a decode loop
// with a hard latency budget where cudaMalloc / cudaFree (which may synchronise the device) are
// not allowed. For them the split partials go to a fixed scratch array that is part of this
// library's device image: every GPU that loads the library holds kNoAllocScratchBytes of it
// until the process exits.
//
// The array is shared by every call on a device and keeps the previous call's contents. Nothing
// in it needs clearing: the split kernel writes every record (empty splits included) before the
// combine kernel of the same call reads it. Two such calls that run at the same time on one
// device (different streams, or graphs replayed concurrently) overwrite each other's partials:
// the caller must keep them ordered.
//
// Host code may not use the array's name as a device address (on the host it names a host-side
// stand-in). The device address is looked up once per device with cudaGetSymbolAddress, with that
// device current, on the first call made on it; make that first call before any stream capture.
// ---------------------------------------------------------------------------------------------
static __device__ __align__(256) float g_decode_scratch[kNoAllocScratchBytes / sizeof(float)];

namespace {
constexpr int kMaxDevices = 128;
std::mutex g_scratch_mu;
float* g_scratch_addr[kMaxDevices] = {};
}  // namespace

cudaError_t decode_scratch_address(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = static_cast<float*>(p);
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

long long decode_noalloc_max_units() {
  return static_cast<long long>(kNoAllocScratchBytes / (kRec * sizeof(float)));
}

// Same kernels as launch_decode, with the split count lowered (if needed) so that the partials
// of all B x H x splits records fit in the scratch array.
cudaError_t launch_decode_noalloc(const DecodeArgs& a, cudaStream_t st) {
  const long long units = static_cast<long long>(a.B) * a.H;
  if (units > decode_noalloc_max_units()) return cudaErrorInvalidValue;
  float* scratch = nullptr;
  cudaError_t e = decode_scratch_address(&scratch);
  if (e != cudaSuccess) return e;
  int chunk = 0;
  int S = decode_splits(a.B, a.Lmax, a.H, &chunk);
  const long long fit = decode_noalloc_max_units() / units;
  if (S > fit) {
    const int step = kDecWarps * kG;
    long long c = (a.Lmax + fit - 1) / fit;
    c = (c + step - 1) / step * step;
    chunk = static_cast<int>(c);
    S = static_cast<int>((a.Lmax + c - 1) / c);
  }
  DecSplitParams sp;
  sp.q = static_cast<const __nv_bfloat16*>(a.q);
  sp.kc = static_cast<const __nv_bfloat16*>(a.k_cache);
  sp.vc = static_cast<const __nv_bfloat16*>(a.v_cache);
  sp.seqlens = a.seqlens;
  sp.ws = scratch;
  sp.Lmax = a.Lmax;
  sp.H = a.H;
  sp.splits = S;
  sp.chunk = chunk;
  sp.scale_log2 = kLog2e / sqrtf(static_cast<float>(a.d));
  decode_split_kernel<<<dim3(S, a.H, a.B), kDecThreads, 0, st>>>(sp);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  DecCombineParams cp;
  cp.ws = scratch;
  cp.lambda = a.lambda;
  cp.norm_w = a.norm_w;
  cp.out = static_cast<__nv_bfloat16*>(a.out);
  cp.lambda_init = a.lambda_init;
  cp.eps = a.eps;
  cp.flags = a.flags;
  cp.H = a.H;
  cp.splits = S;
  decode_combine_kernel<<<dim3(a.H, a.B), kDecWidth, 0, st>>>(cp);
  return cudaGetLastError();
}

}  // namespace da
