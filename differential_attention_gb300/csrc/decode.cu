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
// Grouped form (decode_group_kernel; H signal heads sharing H / G noise heads, q [B, H + H/G, 128],
// K cache [B, L, H + H/G, 128], V cache [B, L, H, 256]): lanes 0-15 read signal head h's K1 row,
// lanes 16-31 noise head H + h/G's K2 row; a CTA covers several heads of one noise group.
#include <cuda_bf16.h>

#include <cmath>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>

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
  const int* block_table;  // paged: [B, max_pages]
  int page_size, max_pages, num_pages;
  uint32_t ps_magic, ps_shift;  // j / page_size = (umulhi(j, magic) + j) >> shift, j < 2^31
  int group;                    // grouped form: signal heads per noise head
  int hpc;                      // grouped form: signal heads per CTA (a divisor of group)
};

// Pool row of key j of sequence b in a paged cache [num_pages, page_size, heads, w]. A page id
// outside [0, num_pages) flags DEV_BAD_INDEX and reads page 0 instead (the call's result is then
// invalid, nothing faults).
__device__ __forceinline__ size_t paged_row(const int* table, int max_pages, int page_size,
                                            int num_pages, uint32_t magic, uint32_t shift, int b,
                                            int j) {
  const uint32_t uj = static_cast<uint32_t>(j);
  const uint32_t pi = (__umulhi(uj, magic) + uj) >> shift;  // j / page_size
  int pg = __ldg(table + static_cast<size_t>(b) * max_pages + pi);
  if (pg < 0 || pg >= num_pages) {
    flag_device_error(DEV_BAD_INDEX);
    pg = 0;
  }
  return static_cast<size_t>(pg) * page_size + (uj - pi * static_cast<uint32_t>(page_size));
}

// Row (key j of sequence b) of a contiguous [B, Lmax, H, w] cache, or of a paged pool.
template <bool kPaged>
__device__ __forceinline__ size_t cache_row(const DecSplitParams& p, int b, int j) {
  size_t r;
  if constexpr (kPaged)
    r = paged_row(p.block_table, p.max_pages, p.page_size, p.num_pages, p.ps_magic, p.ps_shift, b,
                  j);
  else
    r = static_cast<size_t>(b) * p.Lmax + j;
  // debug builds: the row inside the cache (the grid's z extent is the batch)
  if (!dbg_index_ok(static_cast<long long>(r),
                    kPaged ? 1LL * p.num_pages * p.page_size : 1LL * gridDim.z * p.Lmax))
    r = 0;
  return r;
}

template <bool kPaged>
__global__ void __launch_bounds__(kDecThreads, kPaged ? 3 : 4) decode_split_kernel(const DecSplitParams p) {
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
  const __nv_bfloat16* kbase = p.kc + static_cast<size_t>(h) * kDecWidth + 8 * lane;
  const __nv_bfloat16* vbase = p.vc + static_cast<size_t>(h) * kDecWidth + 8 * lane;

  for (int g0 = k0 + warp * kG; g0 < k1; g0 += kDecWarps * kG) {
    uint4 ku[kG], vu[kG];
#pragma unroll
    for (int e = 0; e < kG; ++e) {
      const int j = min(g0 + e, k1 - 1);  // clamp keeps the load in bounds; masked below
      const size_t row = cache_row<kPaged>(p, b, j) * row_stride;
      ku[e] = ldg_stream(kbase + row);
      vu[e] = ldg_stream(vbase + row);
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

// Grouped decode: one CTA per (split, block of `hpc` signal heads of one noise group, sequence),
// kGroupWarps warps per head splitting the keys. Lanes 0-15 stream the head's K1 half row past L1;
// lanes 16-31 read the noise head's K2 half row through L1, where the block's other heads find it,
// so a noise row enters the SM once per block instead of once per head. The math per warp is that
// of decode_split_kernel; the partials go to the same records. kPaged: the caches are page pools
// [num_pages, page_size, heads, w] addressed through the block table, key by key.
constexpr int kGroupWarps = 2;

__device__ __forceinline__ uint4 ldg_l1(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

template <bool kPaged>
__device__ __forceinline__ void decode_group_body(const DecSplitParams& p) {
  const int s = blockIdx.x, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = warp / kGroupWarps, wi = warp % kGroupWarps;
  const int h = blockIdx.y * p.hpc + r;                    // this warp's signal head
  const int heads = p.H + p.H / p.group;                   // heads of q and of the K cache
  const int kh = lane < 16 ? h : p.H + h / p.group;        // K1 of h, or K2 of its noise head
  constexpr int kHalf = kDecWidth / 2;
  int L = p.seqlens ? p.seqlens[b] : p.Lmax;
  L = L < 1 ? 1 : (L > p.Lmax ? p.Lmax : L);
  const int k0 = s * p.chunk;
  const int k1 = min(k0 + p.chunk, L);

  float qf[8];
  {
    const uint4 qu = *reinterpret_cast<const uint4*>(
        p.q + (static_cast<size_t>(b) * heads + kh) * kHalf + 8 * (lane & 15));
    bf16x8_to_f32(qu, qf);
#pragma unroll
    for (int i = 0; i < 8; ++i) qf[i] *= p.scale_log2;
  }

  float m1 = -INFINITY, l1 = 0.f, m2 = -INFINITY, l2 = 0.f;
  float o1[8], o2[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) o1[i] = o2[i] = 0.f;

  const size_t k_stride = static_cast<size_t>(heads) * kHalf;   // elements between keys
  const size_t v_stride = static_cast<size_t>(p.H) * kDecWidth;
  // contiguous caches: sequence b's rows start at b * Lmax; page pools: rows come from the table
  const size_t row0 = kPaged ? 0 : static_cast<size_t>(b) * p.Lmax;
  const __nv_bfloat16* kbase = p.kc + row0 * k_stride + static_cast<size_t>(kh) * kHalf +
                               8 * (lane & 15);
  const __nv_bfloat16* vbase = p.vc + row0 * v_stride + static_cast<size_t>(h) * kDecWidth + 8 * lane;
  const bool noise_lane = lane >= 16;

  for (int g0 = k0 + wi * kG; g0 < k1; g0 += kGroupWarps * kG) {
    uint4 ku[kG], vu[kG];
    // paged: the pool row of key g0 from one table lookup; the group's other keys follow it in
    // the same page unless the group crosses a page boundary (then each key looks its page up)
    size_t prow0 = 0;
    bool one_page = false;
    if constexpr (kPaged) {
      const uint32_t uj = static_cast<uint32_t>(g0);
      const uint32_t pi = (__umulhi(uj, p.ps_magic) + uj) >> p.ps_shift;  // g0 / page_size
      const uint32_t off = uj - pi * static_cast<uint32_t>(p.page_size);
      one_page = off + kG <= static_cast<uint32_t>(p.page_size);
      if (one_page) {
        int pg = __ldg(p.block_table + static_cast<size_t>(b) * p.max_pages + pi);
        if (pg < 0 || pg >= p.num_pages) {
          flag_device_error(DEV_BAD_INDEX);
          pg = 0;
        }
        prow0 = static_cast<size_t>(pg) * p.page_size + off;
      }
    }
#pragma unroll
    for (int e = 0; e < kG; ++e) {
      size_t j = static_cast<size_t>(min(g0 + e, k1 - 1));  // clamped in bounds; masked below
      if constexpr (kPaged) {
        // the key's row in the pool (j - g0 < kG stays inside g0's page on the one-page path)
        j = one_page ? prow0 + (j - static_cast<size_t>(g0)) : cache_row<true>(p, b, static_cast<int>(j));
        if (!dbg_index_ok(static_cast<long long>(j), 1LL * p.num_pages * p.page_size)) j = 0;
      } else {
        if (!dbg_index_ok(static_cast<long long>(j), p.Lmax)) j = 0;
      }
      ku[e] = noise_lane ? ldg_l1(kbase + j * k_stride) : ldg_stream(kbase + j * k_stride);
      vu[e] = ldg_stream(vbase + j * v_stride);
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

  // merge each head's warps
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
  for (int idx = threadIdx.x; idx < p.hpc * kDecWidth; idx += blockDim.x) {
    const int rr = idx / kDecWidth, c = idx % kDecWidth;
    const int w0 = rr * kGroupWarps;
    float* rec = p.ws + ((static_cast<size_t>(b) * p.H + blockIdx.y * p.hpc + rr) * p.splits + s) * kRec;
    float M[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int w = 0; w < kGroupWarps; ++w) {
      M[0] = fmaxf(M[0], s_ml[w0 + w][0]);
      M[1] = fmaxf(M[1], s_ml[w0 + w][2]);
    }
    float oa[2] = {0.f, 0.f}, la[2] = {0.f, 0.f};
#pragma unroll
    for (int w = 0; w < kGroupWarps; ++w) {
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        const float mw = s_ml[w0 + w][2 * m];
        if (mw != -INFINITY) {
          const float f = ex2_approx(mw - M[m]);
          la[m] = fmaf(s_ml[w0 + w][2 * m + 1], f, la[m]);
          oa[m] = fmaf(s_o[w0 + w][m][c], f, oa[m]);
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
}

// The contiguous form keeps the register budget the compiler picks for it (80); the paged form,
// with its table lookups, is held to three CTAs per SM.
__global__ void __launch_bounds__(kDecThreads) decode_group_kernel(const DecSplitParams p) {
  decode_group_body<false>(p);
}
__global__ void __launch_bounds__(kDecThreads, 3) decode_group_paged_kernel(const DecSplitParams p) {
  decode_group_body<true>(p);
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

cudaError_t status_decode(int* v) { return read_clear_status(v); }

void page_magic(int page_size, uint32_t* magic, uint32_t* shift) {
  // division by the invariant page size d (Granlund and Montgomery, "Division by invariant
  // integers using multiplication", 1994): l = ceil(log2 d), m = 2^32 (2^l - d) / d + 1
  uint32_t l = 0;
  while ((1ull << l) < static_cast<unsigned long long>(page_size)) ++l;
  const unsigned long long d = static_cast<unsigned long long>(page_size);
  *magic = static_cast<uint32_t>(((1ull << 32) * ((1ull << l) - d)) / d + 1);
  *shift = l;
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
  sp.block_table = a.block_table;
  sp.page_size = a.page_size;
  sp.max_pages = a.max_pages;
  sp.num_pages = a.num_pages;
  sp.ps_magic = sp.ps_shift = 0;
  if (a.block_table) page_magic(a.page_size, &sp.ps_magic, &sp.ps_shift);
  sp.group = a.noise_group;
  sp.hpc = 1;
  if (a.noise_group) {
    // signal heads per CTA: the largest divisor of the group that fits the CTA's warps
    const int max_hpc = kDecWarps / kGroupWarps;
    for (int d = 1; d <= max_hpc; ++d)
      if (a.noise_group % d == 0) sp.hpc = d;
    const dim3 grid(S, a.H / sp.hpc, a.B);
    if (a.block_table)
      decode_group_paged_kernel<<<grid, kGroupWarps * 32 * sp.hpc, 0, st>>>(sp);
    else
      decode_group_kernel<<<grid, kGroupWarps * 32 * sp.hpc, 0, st>>>(sp);
  } else if (a.block_table)
    decode_split_kernel<true><<<dim3(S, a.H, a.B), kDecThreads, 0, st>>>(sp);
  else
    decode_split_kernel<false><<<dim3(S, a.H, a.B), kDecThreads, 0, st>>>(sp);
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
// device (on different streams, say) overwrite each other's partials: the caller must keep them
// ordered.
//
// Host code may not use the array's name as a device address (on the host it names a host-side
// stand-in). The device address is looked up with cudaGetSymbolAddress, with that device current,
// on the first call made on it (and again on the first call after its context was recreated);
// make that first call before any stream capture.
// ---------------------------------------------------------------------------------------------
static __device__ __align__(256) float g_decode_scratch[kNoAllocScratchBytes / sizeof(float)];

namespace {
constexpr int kMaxDevices = 128;
std::mutex g_scratch_mu;
// The array's device address is a property of the context the module was loaded into, so the
// cache remembers the context it was looked up in: after the primary context of a device is torn
// down and recreated (cudaDeviceReset in this process), the next call looks it up again.
struct ScratchSlot {
  CUcontext ctx = nullptr;
  float* addr = nullptr;
};
ScratchSlot g_scratch_slot[kMaxDevices];

PFN_cuCtxGetCurrent_v4000 ctx_get_current_entry() {
  static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult res;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &res) ==
            cudaSuccess &&
        res == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
  });
  return fn;
}
}  // namespace

cudaError_t decode_scratch_address(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  auto get_ctx = ctx_get_current_entry();
  if (!get_ctx) return cudaErrorNotSupported;
  CUcontext ctx = nullptr;
  if (get_ctx(&ctx) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  if (ctx == nullptr) {
    // no context current on this thread yet: cudaSetDevice makes the device's primary one current
    e = cudaSetDevice(dev);
    if (e != cudaSuccess) return e;
    if (get_ctx(&ctx) != CUDA_SUCCESS || ctx == nullptr) return cudaErrorDeviceUninitialized;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  ScratchSlot& slot = g_scratch_slot[dev];
  if (slot.addr == nullptr || slot.ctx != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) return e;
    slot.ctx = ctx;
    slot.addr = static_cast<float*>(p);
  }
  *out = slot.addr;
  return cudaSuccess;
}

long long decode_noalloc_max_units() {
  return static_cast<long long>(kNoAllocScratchBytes / (kRec * sizeof(float)));
}

// The split count of diffattn_decode, lowered when B x H x splits records would not fit in the
// scratch array: the chunk grows to ceil(Lmax / fit) keys, rounded up to whole CTA rounds, so
// that splits = ceil(Lmax / chunk) <= fit. Requires B * H <= decode_noalloc_max_units().
int decode_noalloc_splits(int B, int Lmax, int H, int* chunk_out) {
  int chunk = 0;
  int S = decode_splits(B, Lmax, H, &chunk);
  const long long units = static_cast<long long>(B) * H;
  const long long fit = decode_noalloc_max_units() / units;
  if (S > fit) {
    const int step = kDecWarps * kG;
    long long c = (Lmax + fit - 1) / fit;
    c = (c + step - 1) / step * step;
    chunk = static_cast<int>(c);
    S = static_cast<int>((Lmax + c - 1) / c);
  }
  if (chunk_out) *chunk_out = chunk;
  return S;
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
  const int S = decode_noalloc_splits(a.B, a.Lmax, a.H, &chunk);
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
  sp.block_table = nullptr;
  sp.group = 0;
  decode_split_kernel<false><<<dim3(S, a.H, a.B), kDecThreads, 0, st>>>(sp);
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

// =============================================================================================
// DIFF V2 decode (page "Differential Transformer: softmax can't say zero, so it subtracts",
// section "DIFF V2: what the authors changed"; page "Differential Transformer V2": the KV
// cache is that of a baseline Transformer, so decoding reads it as a baseline would).
//
// One query token per sequence; the G = Hq / Hkv query heads of a GQA group share one KV head,
// and query heads (2p, 2p+1) form differential pair p. Stage 1 (v2dec_split_kernel, grid
// splits x Hkv x B): a CTA streams one slice of one KV head's cache once for all G query heads.
// Each half-warp walks its own keys, kV2Keys at a time: lane t' (0..15) loads 16 bytes (8 dims)
// of each K and V row, forms the G partial dot products, and a butterfly reduce-scatter over the
// 16 lanes leaves head h's score in lanes 2h, 2h+1 (for G = 8), which keep that head's running
// max and sum; the rescale factors and probabilities are broadcast back for the 8 x G fp32
// output accumulators. Half-warps and warps are merged in shared memory; one record per
// (b, kv head, split) holds, per query head, (m, l, o[d]). Stage 2 (v2dec_combine_kernel, grid
// pairs x B): thread c merges the splits for channel c of both heads of its pair and writes
// o_a / l_a - sigmoid(lam) * o_b / l_b.
// =============================================================================================
namespace {
constexpr int kV2D = 128;          // head dim
constexpr int kV2Keys = 4;         // keys per half-warp per step
constexpr int kV2Warps = 8;

// Sum each of the G values of v over the 16 lanes of the half-warp; afterwards lane t' holds the
// total of value (t' >> sh) & (G - 1) for the shift sh = log2(16 / G) (lanes 2h, 2h+1 for G = 8).
template <int G>
__device__ __forceinline__ float reduce_scatter16(float (&v)[G], int lane) {
  // rounds over lane bits 3, 2, ... while more than one value is left
  int cnt = G;
#pragma unroll
  for (int bit = 8; bit >= 1; bit >>= 1) {
    if (cnt > 1) {
      const bool up = (lane & bit) != 0;
      const int half = cnt >> 1;
#pragma unroll
      for (int i = 0; i < G / 2; ++i) {
        if (i < half) {
          const float send = up ? v[i] : v[i + half];
          const float keep = up ? v[i + half] : v[i];
          v[i] = keep + __shfl_xor_sync(0xffffffffu, send, bit);
        }
      }
      cnt = half;
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], bit);
    }
  }
  return v[0];
}

template <int G>
struct V2DecParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* kc;
  const __nv_bfloat16* vc;
  const int* seqlens;
  float* ws;
  int Lmax, Hq, Hkv, splits, chunk;
  float scale_log2;
  const int* block_table;  // paged: [B, max_pages]
  int page_size, max_pages, num_pages;
  uint32_t ps_magic, ps_shift;
};

template <int G, bool kPaged>
__global__ void __launch_bounds__(kV2Warps * 32) v2dec_split_kernel(const V2DecParams<G> p) {
  constexpr int kRec = G * (2 + kV2D);  // floats per record: per head m, l, o[128]
  const int s = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hl = lane & 15, half = lane >> 4;
  constexpr int kSh = (G == 8) ? 1 : (G == 4) ? 2 : 3;  // head of lane: (hl >> kSh) & (G-1)
  const int my_head = (hl >> kSh) & (G - 1);
  int L = p.seqlens ? p.seqlens[b] : p.Lmax;
  L = L < 1 ? 1 : (L > p.Lmax ? p.Lmax : L);
  const int k0 = s * p.chunk, k1 = min(k0 + p.chunk, L);

  float qf[G][8];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const uint4 qu = *reinterpret_cast<const uint4*>(
        p.q + (static_cast<size_t>(b) * p.Hq + g * G + h) * kV2D + 8 * hl);
    bf16x8_to_f32(qu, qf[h]);
#pragma unroll
    for (int i = 0; i < 8; ++i) qf[h][i] *= p.scale_log2;
  }
  float m = -INFINITY, l = 0.f;  // running stats of head my_head (this lane pair)
  float o[G][8];
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int i = 0; i < 8; ++i) o[h][i] = 0.f;

  const size_t row = static_cast<size_t>(p.Hkv) * kV2D;  // elements between keys
  const __nv_bfloat16* kb = p.kc + static_cast<size_t>(g) * kV2D + 8 * hl;
  const __nv_bfloat16* vb = p.vc + static_cast<size_t>(g) * kV2D + 8 * hl;
  auto rowof = [&](int j) -> size_t {
    size_t r;
    if constexpr (kPaged)
      r = paged_row(p.block_table, p.max_pages, p.page_size, p.num_pages, p.ps_magic, p.ps_shift,
                    b, j);
    else
      r = static_cast<size_t>(b) * p.Lmax + j;
    // debug builds: the row inside the cache (the grid's z extent is the batch)
    if (!dbg_index_ok(static_cast<long long>(r),
                      kPaged ? 1LL * p.num_pages * p.page_size : 1LL * gridDim.z * p.Lmax))
      r = 0;
    return r;
  };
  constexpr int kStride = kV2Warps * 2 * kV2Keys;  // keys per CTA step
  // The loop bound is warp-uniform so that every shuffle below has all 32 lanes; a half-warp
  // whose keys all lie past k1 takes part with masked scores and leaves its state unchanged.
  for (int jw = k0 + warp * 2 * kV2Keys; jw < k1; jw += kStride) {
    const int j0 = jw + half * kV2Keys;
    uint4 ku[kV2Keys], vu[kV2Keys];
#pragma unroll
    for (int e = 0; e < kV2Keys; ++e) {
      const int j = min(j0 + e, k1 - 1);  // clamped in bounds; masked below
      const size_t rj = rowof(j) * row;
      ku[e] = ldg_stream(kb + rj);
      vu[e] = ldg_stream(vb + rj);
    }
    float sc[kV2Keys];
#pragma unroll
    for (int e = 0; e < kV2Keys; ++e) {
      float kf[8];
      bf16x8_to_f32(ku[e], kf);
      float part[G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float a = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) a = fmaf(qf[h][i], kf[i], a);
        part[h] = a;
      }
      const float r = reduce_scatter16<G>(part, hl);
      sc[e] = (j0 + e < k1) ? r : -INFINITY;
    }
    float mx = sc[0];
#pragma unroll
    for (int e = 1; e < kV2Keys; ++e) mx = fmaxf(mx, sc[e]);
    const float mn = fmaxf(m, mx);
    const float ms = (mn == -INFINITY) ? 0.f : mn;  // no key seen yet: keep the state at zero
    const float corr = ex2_approx(m - ms);
    float pe[kV2Keys];
    float ps = 0.f;
#pragma unroll
    for (int e = 0; e < kV2Keys; ++e) {
      pe[e] = ex2_approx(sc[e] - ms);
      ps += pe[e];
    }
    l = l * corr + ps;
    m = mn;
    // every head's correction and probabilities, broadcast to the whole half-warp
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float ch = __shfl_sync(0xffffffffu, corr, (lane & 16) | (h << kSh));
#pragma unroll
      for (int i = 0; i < 8; ++i) o[h][i] *= ch;
    }
#pragma unroll
    for (int e = 0; e < kV2Keys; ++e) {
      float vf[8];
      bf16x8_to_f32(vu[e], vf);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float ph = __shfl_sync(0xffffffffu, pe[e], (lane & 16) | (h << kSh));
#pragma unroll
        for (int i = 0; i < 8; ++i) o[h][i] = fmaf(ph, vf[i], o[h][i]);
      }
    }
  }

  // merge the two half-warps of this warp in registers (lane t and t ^ 16 hold the same dims)
  {
    const float m_o = __shfl_xor_sync(0xffffffffu, m, 16);
    const float l_o = __shfl_xor_sync(0xffffffffu, l, 16);
    const float M = fmaxf(m, m_o);
    const float Ms = (M == -INFINITY) ? 0.f : M;
    const float f_me = ex2_approx(m - Ms), f_ot = ex2_approx(m_o - Ms);
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const int src = h << kSh;
      const float a = __shfl_sync(0xffffffffu, f_me, (lane & 16) | src);
      const float c = __shfl_sync(0xffffffffu, f_ot, (lane & 16) | src);
#pragma unroll
      for (int i = 0; i < 8; ++i) o[h][i] = o[h][i] * a + __shfl_xor_sync(0xffffffffu, o[h][i], 16) * c;
    }
    l = l * f_me + l_o * f_ot;
    m = M;
  }
  // then the warps, in shared memory
  __shared__ float s_o[kV2Warps][G][kV2D];
  __shared__ float s_ml[kV2Warps][G][2];
  if (half == 0) {
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int i = 0; i < 8; ++i) s_o[warp][h][8 * hl + i] = o[h][i];
    if ((hl & ((1 << kSh) - 1)) == 0) {
      s_ml[warp][my_head][0] = m;
      s_ml[warp][my_head][1] = l;
    }
  }
  __syncthreads();
  float* rec = p.ws + ((static_cast<size_t>(b) * p.Hkv + g) * p.splits + s) * kRec;
  for (int idx = threadIdx.x; idx < G * kV2D; idx += kV2Warps * 32) {
    const int h = idx / kV2D, c = idx % kV2D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kV2Warps; ++w) M = fmaxf(M, s_ml[w][h][0]);
    float oa = 0.f, la = 0.f;
#pragma unroll
    for (int w = 0; w < kV2Warps; ++w) {
      const float mw = s_ml[w][h][0];
      if (mw != -INFINITY) {
        const float f = ex2_approx(mw - M);
        la = fmaf(s_ml[w][h][1], f, la);
        oa = fmaf(s_o[w][h][c], f, oa);
      }
    }
    rec[h * (2 + kV2D) + 2 + c] = oa;
    if (c == 0) {
      rec[h * (2 + kV2D) + 0] = M;
      rec[h * (2 + kV2D) + 1] = la;
    }
  }
}

struct V2CombineParams {
  const float* ws;
  const float* lam_logit;
  __nv_bfloat16* out;
  int Hq, Hkv, G, splits;
};

__global__ void __launch_bounds__(kV2D) v2dec_combine_kernel(const V2CombineParams p) {
  const int pair = blockIdx.x, b = blockIdx.y, c = threadIdx.x;
  const int P = p.Hq / 2;
  const int ha = 2 * pair, g = ha / p.G;
  const int rec_len = p.G * (2 + kV2D);
  const float* recs = p.ws + (static_cast<size_t>(b) * p.Hkv + g) * p.splits * rec_len;
  float res[2];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int h = (ha + k) - g * p.G;
    float M = -INFINITY;
    for (int s = 0; s < p.splits; ++s) M = fmaxf(M, recs[s * rec_len + h * (2 + kV2D)]);
    float o = 0.f, l = 0.f;
    for (int s = 0; s < p.splits; ++s) {
      const float* r = recs + s * rec_len + h * (2 + kV2D);
      if (r[0] != -INFINITY) {
        const float f = ex2_approx(r[0] - M);
        l = fmaf(r[1], f, l);
        o = fmaf(r[2 + c], f, o);
      }
    }
    res[k] = o / l;
  }
  const float z = p.lam_logit[static_cast<size_t>(b) * P + pair];
  const float lam = 1.f / (1.f + expf(-z));
  p.out[(static_cast<size_t>(b) * P + pair) * kV2D + c] = __float2bfloat16_rn(res[0] - lam * res[1]);
}

template <int G>
cudaError_t launch_v2dec(const V2DecodeArgs& a, cudaStream_t st, int S, int chunk) {
  V2DecParams<G> sp;
  sp.q = static_cast<const __nv_bfloat16*>(a.q);
  sp.kc = static_cast<const __nv_bfloat16*>(a.k_cache);
  sp.vc = static_cast<const __nv_bfloat16*>(a.v_cache);
  sp.seqlens = a.seqlens;
  sp.ws = a.ws;
  sp.Lmax = a.Lmax;
  sp.Hq = a.Hq;
  sp.Hkv = a.Hkv;
  sp.splits = S;
  sp.chunk = chunk;
  sp.scale_log2 = kLog2e / sqrtf(static_cast<float>(kV2D));
  sp.block_table = a.block_table;
  sp.page_size = a.page_size;
  sp.max_pages = a.max_pages;
  sp.num_pages = a.num_pages;
  sp.ps_magic = sp.ps_shift = 0;
  if (a.block_table) {
    page_magic(a.page_size, &sp.ps_magic, &sp.ps_shift);
    v2dec_split_kernel<G, true><<<dim3(S, a.Hkv, a.B), kV2Warps * 32, 0, st>>>(sp);
  } else {
    v2dec_split_kernel<G, false><<<dim3(S, a.Hkv, a.B), kV2Warps * 32, 0, st>>>(sp);
  }
  return cudaGetLastError();
}
}  // namespace

int v2_decode_splits(int B, int Lmax, int Hkv, int* chunk_out) {
  const long long units = static_cast<long long>(B) * Hkv;
  long long target = (16LL * 152 + units - 1) / units;
  if (target < 1) target = 1;
  const int step = kV2Warps * 2 * kV2Keys;
  long long chunk = (Lmax + target - 1) / target;
  if (chunk < 512) chunk = 512;
  chunk = (chunk + step - 1) / step * step;
  const int splits = static_cast<int>((Lmax + chunk - 1) / chunk);
  if (chunk_out) *chunk_out = static_cast<int>(chunk);
  return splits;
}

size_t v2_decode_workspace_bytes(int B, int Lmax, int Hq, int Hkv) {
  // room for the records of either split kernel (CUDA cores or tensor cores)
  const int S1 = v2_decode_splits(B, Lmax, Hkv, nullptr);
  const int S2 = v2_decode_tc_splits(B, Lmax, Hkv, nullptr);
  const int S = S1 > S2 ? S1 : S2;
  const int G = Hq / Hkv;
  return static_cast<size_t>(B) * Hkv * S * G * (2 + kV2D) * sizeof(float);
}

cudaError_t launch_v2_combine(const V2DecodeArgs& a, int splits, cudaStream_t st) {
  V2CombineParams cp;
  cp.ws = a.ws;
  cp.lam_logit = a.lam_logit;
  cp.out = static_cast<__nv_bfloat16*>(a.out);
  cp.Hq = a.Hq;
  cp.Hkv = a.Hkv;
  cp.G = a.Hq / a.Hkv;
  cp.splits = splits;
  v2dec_combine_kernel<<<dim3(a.Hq / 2, a.B), kV2D, 0, st>>>(cp);
  return cudaGetLastError();
}

cudaError_t launch_v2_decode(const V2DecodeArgs& a, cudaStream_t st) {
  int chunk = 0;
  const int S = v2_decode_splits(a.B, a.Lmax, a.Hkv, &chunk);
  const int G = a.Hq / a.Hkv;
  cudaError_t e;
  if (G == 2)
    e = launch_v2dec<2>(a, st, S, chunk);
  else if (G == 4)
    e = launch_v2dec<4>(a, st, S, chunk);
  else if (G == 8)
    e = launch_v2dec<8>(a, st, S, chunk);
  else
    return cudaErrorNotSupported;
  if (e != cudaSuccess) return e;
  return launch_v2_combine(a, S, st);
}

}  // namespace da
