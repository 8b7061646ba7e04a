// prefill_exact.cu -- differential-attention prefill on the sm_103a tensor cores that forms the
// signed weights A1 - lambda A2 in fp32 before they are rounded for the tensor-core product.
//
// Operator (page "Differential Transformer: softmax can't say zero, so it subtracts", section
// "The mechanism, exactly"): out = (softmax(Q1 K1^T/sqrt d) - lambda softmax(Q2 K2^T/sqrt d)) V,
// then the per-head RMSNorm over dv channels and the (1 - lambda_init) scale ("The row no longer
// sums to one"). V2 ("DIFF V2: what the authors changed"): query heads 2p and 2p+1 share one GQA
// K/V head, lambda = sigmoid(logit) per token and pair, no norm.
//
// Why two passes. A row of A1 - lambda A2 sums to 1 - lambda, so when the two maps are close the
// product (A1 - lambda A2) V is a small difference of two large, nearly equal terms. Rounding
// each map's probabilities to bf16 before multiplying by V (one flash pass per map) leaves an
// error of about 2^-9 of each term, i.e. ~2^-9 / |1 - lambda| of the result. This kernel first
// finds each map's exact row max and row sum (pass 1: QK^T only), then (pass 2) recomputes the
// scores, forms D = 2^(s1 - b1) - lambda 2^(s2 - b2) with b = max + log2(sum) in fp32, rounds D
// (already small) to bf16 and runs a single D V product. Both passes together issue the same
// MMA work as the single-pass form (4d + 4dv flops per query-key pair).
//
// Structure: one CTA per 128-row query tile of one unit, 64-key tiles. TMA stages Q1|Q2 once and
// a ring of K tiles (each K tile is streamed twice, once per pass) and V tiles (pass 2 only).
// tcgen05.mma writes S1 and S2 (64 columns each, double-buffered) into tensor memory; four
// softmax warps (one thread per query row) read them, and in pass 2 write D as packed bf16 over
// the S1 columns; a second tcgen05.mma (A = D from tensor memory, B = V from shared memory)
// accumulates O (128 x dv fp32, columns 256..) in tensor memory. Epilogue: RMSNorm and scale
// straight out of tensor memory. Warp 0 = TMA producer, warp 1 = MMA issuer / TMEM owner,
// warps 4-7 = softmax and epilogue. Every wait is bounded.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <cmath>
#include <cstdio>

#include "internal.h"
#include "ptx.cuh"

namespace da {
namespace exact {

constexpr int BM = 128;
constexpr int BN = 64;
constexpr int kThreads = 256;
constexpr int kSoftmaxWarp0 = 4;
constexpr int kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;

template <int DQK, int DV, bool SHARED_K>
struct Cfg {
  static constexpr int kQChunk = BM * 128;                 // 128 rows x 64 bf16
  static constexpr int kKChunk = BN * 128;                 // 64 rows x 64 bf16
  static constexpr int kQMapBytes = BM * DQK * 2;          // one map's Q tile
  static constexpr int kKMapBytes = BN * DQK * 2;          // one map's K tile
  static constexpr int kQBytes = 2 * kQMapBytes;
  static constexpr int kKBytes = (SHARED_K ? 1 : 2) * kKMapBytes;  // one K stage
  static constexpr int kVBytes = BN * DV * 2;              // one V stage
  static constexpr int NSK = (DQK == 128 && DV == 256) ? 3 : 4;
  static constexpr int NSV = (DQK == 128 && DV == 256) ? 2 : 4;
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + kQBytes;
  static constexpr int kVOff = kKOff + NSK * kKBytes;
  static constexpr int kEnd = kVOff + NSV * kVBytes;
  static constexpr int kDynSmem = kEnd + 1024;
  static constexpr int kOCol = 256;
  static_assert(kOCol + DV <= kTmemCols, "TMEM budget");
  static_assert(kDynSmem <= 232448 - 1024, "shared memory budget");
};

struct Barriers {
  uint64_t q_full;
  uint64_t k_full[4], k_empty[4], v_full[4], v_empty[4];
  uint64_t s_full[2], s_done[2];
  uint64_t o_full;
  uint64_t teardown;
};

struct KParams {
  Problem p;
  int n_qt;
  float scale_log2;
};

template <int DQK, int DV, bool SHARED_K>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_exact_kernel(const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const KParams kp) {
  using C = Cfg<DQK, DV, SHARED_K>;
  constexpr int NSK = C::NSK, NSV = C::NSV;
  extern __shared__ uint8_t smem_raw[];
  __shared__ Barriers bars;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const Problem& P = kp.p;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sQ = smem_u32(smem + C::kQOff);
  const uint32_t sK = smem_u32(smem + C::kKOff);
  const uint32_t sV = smem_u32(smem + C::kVOff);

  // ---- work item: longest causal tiles first ----
  const int BU = P.B * P.units;
  const bool causal = (P.flags & 1) != 0;
  const int item = blockIdx.x;
  const int qt = causal ? (kp.n_qt - 1 - item / BU) : (item / BU);
  const int bu = item % BU;
  const int b = bu / P.units, u = bu % P.units;
  const int n_kv_all = (P.N + BN - 1) / BN;
  const int n = causal ? min((qt * BM + BM + BN - 1) / BN, n_kv_all) : n_kv_all;
  const int T = 2 * n;  // tiles over both passes

  auto bar = [](uint64_t& x) { return smem_u32(&x); };

  if (threadIdx.x == 0) {
    mbar_init(bar(bars.q_full), 1);
    for (int s = 0; s < 4; ++s) {
      mbar_init(bar(bars.k_full[s]), 1);
      mbar_init(bar(bars.k_empty[s]), 1);
      mbar_init(bar(bars.v_full[s]), 1);
      mbar_init(bar(bars.v_empty[s]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(bars.s_full[i]), 1);
      mbar_init(bar(bars.s_done[i]), 128);
    }
    mbar_init(bar(bars.o_full), 1);
    mbar_init(bar(bars.teardown), 1);
    abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  volatile int* abrt = &abort_flag;

  if (warp == 0) {
    // ================================ TMA producer ================================
    if (lane == 0) {
      const int kvh = kv_head_of(P, u);
      mbar_arrive_expect_tx(bar(bars.q_full), C::kQBytes);
      for (int r = 0; r < 2; ++r)
        for (int c = 0; c < DQK / 64; ++c)
          tma_load_4d(sQ + r * C::kQMapBytes + c * C::kQChunk, &tm_q, bar(bars.q_full),
                      q_col_of(P, r) + 64 * c, q_head_of(P, u, r), qt * BM, b);
      int k_issued = 0, v_issued = 0;
      bool ok = true;
      for (int t = 0; t < T && ok; ++t) {
        const int j = t < n ? t : t - n;
        const int s = t % NSK;
        if (!(ok = mbar_wait(bar(bars.k_empty[s]), ((t / NSK) & 1) ^ 1, abrt))) break;
        mbar_arrive_expect_tx(bar(bars.k_full[s]), C::kKBytes);
        for (int r = 0; r < (SHARED_K ? 1 : 2); ++r)
          for (int c = 0; c < DQK / 64; ++c)
            tma_load_4d(sK + s * C::kKBytes + r * C::kKMapBytes + c * C::kKChunk, &tm_k,
                        bar(bars.k_full[s]), k_col_of(P, r) + 64 * c, kvh, j * BN, b);
        k_issued = t + 1;
        if (t >= n) {
          const int jv = t - n, sv = jv % NSV;
          if (!(ok = mbar_wait(bar(bars.v_empty[sv]), ((jv / NSV) & 1) ^ 1, abrt))) break;
          mbar_arrive_expect_tx(bar(bars.v_full[sv]), C::kVBytes);
          for (int c = 0; c < DV / 64; ++c)
            tma_load_4d(sV + sv * C::kVBytes + c * C::kKChunk, &tm_v, bar(bars.v_full[sv]),
                        64 * c, kvh, jv * BN, b);
          v_issued = jv + 1;
        }
      }
      // make sure no copy of ours is still landing in shared memory
      mbar_wait(bar(bars.q_full), 0, nullptr);
      for (int t = max(0, k_issued - NSK); t < k_issued; ++t)
        mbar_wait(bar(bars.k_full[t % NSK]), (t / NSK) & 1, nullptr);
      for (int jv = max(0, v_issued - NSV); jv < v_issued; ++jv)
        mbar_wait(bar(bars.v_full[jv % NSV]), (jv / NSV) & 1, nullptr);
    }
  } else if (warp == 1) {
    // ================================ MMA issuer ==================================
    if (lane == 0) {
      constexpr uint32_t idesc_s = umma_idesc_bf16(BM, BN, 0, 0);
      constexpr uint32_t idesc_o = umma_idesc_bf16(BM, DV, 0, 1);
      bool ok = mbar_wait(bar(bars.q_full), 0, abrt);
      tc_fence_after();
      for (int t = 0; ok && t <= T; ++t) {
        if (t < T) {
          const int buf = t & 1, s = t % NSK;
          // S buffer `buf` was last used by tile t-2: its scores must have been read (pass 1)
          // or replaced by D and handed over (pass 2; that D's product was issued already).
          if (t >= 2 && !(ok = mbar_wait(bar(bars.s_done[buf]), ((t - 2) >> 1) & 1, abrt))) break;
          if (!(ok = mbar_wait(bar(bars.k_full[s]), (t / NSK) & 1, abrt))) break;
          tc_fence_after();
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const uint32_t d_s = tmem + buf * 128 + r * 64;
            const uint32_t kbase = sK + s * C::kKBytes + (SHARED_K ? 0 : r * C::kKMapBytes);
#pragma unroll
            for (int kk = 0; kk < DQK / 16; ++kk) {
              const uint64_t ad = umma_smem_desc(
                  sQ + r * C::kQMapBytes + (kk >> 2) * C::kQChunk + (kk & 3) * 32, 16, 1024);
              const uint64_t bd =
                  umma_smem_desc(kbase + (kk >> 2) * C::kKChunk + (kk & 3) * 32, 16, 1024);
              mma_bf16_ss(d_s, ad, bd, idesc_s, kk > 0 ? 1u : 0u);
            }
          }
          tc_commit(bar(bars.k_empty[s]));
          tc_commit(bar(bars.s_full[buf]));
        }
        const int tp = t - 1;
        if (tp >= n) {
          const int bp = tp & 1, jv = tp - n, sv = jv % NSV;
          if (!(ok = mbar_wait(bar(bars.s_done[bp]), (tp >> 1) & 1, abrt))) break;
          if (!(ok = mbar_wait(bar(bars.v_full[sv]), (jv / NSV) & 1, abrt))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk) {
            const uint32_t a_t = tmem + bp * 128 + kk * 8;  // D: 16 bf16 keys per 8 columns
            const uint64_t bd = umma_smem_desc(sV + sv * C::kVBytes + kk * 2048, C::kKChunk, 1024);
            mma_bf16_ts(tmem + C::kOCol, a_t, bd, idesc_o, (jv > 0 || kk > 0) ? 1u : 0u);
          }
          tc_commit(bar(bars.v_empty[sv]));
          if (tp == T - 1) tc_commit(bar(bars.o_full));
        }
      }
      tc_commit(bar(bars.teardown));
      mbar_wait(bar(bars.teardown), 0, nullptr);
    }
  } else if (warp >= kSoftmaxWarp0) {
    // ============================ softmax and epilogue ============================
    const int r = 32 * (warp & 3) + lane;
    const int row = qt * BM + r;
    const uint32_t tl = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const float sl2 = kp.scale_log2;
    const int lim = causal ? min(row + 1, P.N) : P.N;  // keys [0, lim) are visible
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
    float bias[2] = {0.f, 0.f}, lam = 0.f;
    bool ok = true;

    for (int t = 0; t < T; ++t) {
      const int buf = t & 1;
      const bool pass2 = t >= n;
      const int key0 = (pass2 ? t - n : t) * BN;
      ok = mbar_wait(bar(bars.s_full[buf]), (t >> 1) & 1, abrt);
      if (__any_sync(0xffffffffu, !ok)) { ok = false; break; }
      tc_fence_after();
      uint32_t sr[2][64];
      tmem_ld32(tmem + tl + buf * 128 + 0, *reinterpret_cast<uint32_t(*)[32]>(&sr[0][0]));
      tmem_ld32(tmem + tl + buf * 128 + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[0][32]));
      tmem_ld32(tmem + tl + buf * 128 + 64, *reinterpret_cast<uint32_t(*)[32]>(&sr[1][0]));
      tmem_ld32(tmem + tl + buf * 128 + 96, *reinterpret_cast<uint32_t(*)[32]>(&sr[1][32]));
      tmem_wait_ld();
      if (key0 + BN > lim) {
#pragma unroll
        for (int i = 0; i < BN; ++i)
          if (key0 + i >= lim) {
            sr[0][i] = __float_as_uint(-INFINITY);
            sr[1][i] = __float_as_uint(-INFINITY);
          }
      }
      __syncwarp();
      if (!pass2) {
        // ---- pass 1: exact row max and row sum of each map (online over key tiles) ----
        tc_fence_before();
        mbar_arrive(bar(bars.s_done[buf]));  // scores are in registers: the buffer is free
#pragma unroll
        for (int mp = 0; mp < 2; ++mp) {
          float mx[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) mx[i] = __uint_as_float(sr[mp][i]);
#pragma unroll
          for (int i = 4; i < BN; ++i) mx[i & 3] = fmaxf(mx[i & 3], __uint_as_float(sr[mp][i]));
          const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * sl2;
          const float mn = fmaxf(m[mp], mt);
          const float nb = (mn == -INFINITY) ? 0.f : -mn;
          float la[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int i = 0; i < BN; ++i)
            la[i & 3] += ex2_approx(fmaf(__uint_as_float(sr[mp][i]), sl2, nb));
          l[mp] = l[mp] * ex2_approx(m[mp] + nb) + ((la[0] + la[1]) + (la[2] + la[3]));
          m[mp] = mn;
        }
        if (t == n - 1) {
          // p / l = 2^(x - (m + log2 l)); lambda of this row
          bias[0] = -(m[0] + __log2f(l[0]));
          bias[1] = -(m[1] + __log2f(l[1]));
          if (P.mode == MODE_V1) {
            lam = P.lambda[u];
          } else if (row < P.N) {
            const float z = P.lam_logit[(static_cast<size_t>(b) * P.N + row) * P.units + u];
            lam = 1.f / (1.f + expf(-z));
          }
        }
      } else {
        // ---- pass 2: D = A1 - lambda A2 in fp32, rounded once to bf16 ----
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float a0 = ex2_approx(fmaf(__uint_as_float(sr[0][2 * i]), sl2, bias[0]));
          const float a1 = ex2_approx(fmaf(__uint_as_float(sr[0][2 * i + 1]), sl2, bias[0]));
          const float c0 = ex2_approx(fmaf(__uint_as_float(sr[1][2 * i]), sl2, bias[1]));
          const float c1 = ex2_approx(fmaf(__uint_as_float(sr[1][2 * i + 1]), sl2, bias[1]));
          pk[i] = pack_bf16x2(fmaf(-lam, c0, a0), fmaf(-lam, c1, a1));
        }
        tmem_st32(tmem + tl + buf * 128, pk);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(bars.s_done[buf]));
      }
    }
    if (ok) {
      ok = mbar_wait(bar(bars.o_full), 0, abrt);
      ok = !__any_sync(0xffffffffu, !ok);
    }
    tc_fence_after();
    // ------------------------------- epilogue -------------------------------------
    if (ok) {
      float scale = 1.f;
      if (P.flags & 2) {
        float ss = 0.f;
#pragma unroll 1
        for (int c = 0; c < DV / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tmem + tl + C::kOCol + 32 * c, o);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) ss = fmaf(__uint_as_float(o[i]), __uint_as_float(o[i]), ss);
        }
        scale = 1.f / sqrtf(ss / static_cast<float>(DV) + P.eps);
      }
      if (P.flags & 4) scale *= (1.f - P.lambda_init);
      __nv_bfloat16* out = static_cast<__nv_bfloat16*>(P.out) +
                           ((static_cast<size_t>(b) * P.N + row) * P.units + u) * DV;
      const float* w = (P.flags & 2) ? P.norm_w : nullptr;
#pragma unroll 1
      for (int c = 0; c < DV / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tmem + tl + C::kOCol + 32 * c, o);
        tmem_wait_ld();
        if (row < P.N) {
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            uint4 pkt;
            uint32_t* pw = reinterpret_cast<uint32_t*>(&pkt);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int e = 8 * g + 2 * i;
              const float w0 = w ? w[32 * c + e] : 1.f;
              const float w1 = w ? w[32 * c + e + 1] : 1.f;
              pw[i] = pack_bf16x2(__uint_as_float(o[e]) * scale * w0,
                                  __uint_as_float(o[e + 1]) * scale * w1);
            }
            *reinterpret_cast<uint4*>(out + 32 * c + 8 * g) = pkt;
          }
        }
      }
    }
  }

  // ---- teardown ----
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 4-D bf16 map over [B, N, heads, cols] with a 64-col x 1 x rows x 1 box, 128-byte swizzle,
// zero fill out of bounds.
static bool make_map(CUtensorMap* m, const void* base, int cols, int heads, int N, int B,
                     int box_rows, char* err, size_t err_len) {
  auto fn = get_encode_fn();
  if (!fn) {
    snprintf(err, err_len, "cuTensorMapEncodeTiled entry point unavailable");
    return false;
  }
  cuuint64_t dims[4] = {(cuuint64_t)cols, (cuuint64_t)heads, (cuuint64_t)N, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)cols * 2, (cuuint64_t)cols * heads * 2,
                           (cuuint64_t)cols * heads * 2 * (cuuint64_t)N};
  cuuint32_t box[4] = {64, 1, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(err, err_len, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
    return false;
  }
  return true;
}

template <int DQK, int DV, bool SHARED_K>
static cudaError_t launch_cfg(const Problem& p, cudaStream_t s, char* err, size_t err_len) {
  using C = Cfg<DQK, DV, SHARED_K>;
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, p.q, p.q_cols, p.q_heads, p.N, p.B, BM, err, err_len) ||
      !make_map(&mk, p.k, p.k_cols, p.kv_heads, p.N, p.B, BN, err, err_len) ||
      !make_map(&mv, p.v, DV, p.kv_heads, p.N, p.B, BN, err, err_len))
    return cudaErrorInvalidValue;
  auto kern = prefill_exact_kernel<DQK, DV, SHARED_K>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kDynSmem);
  if (e != cudaSuccess) return e;
  KParams kp;
  kp.p = p;
  kp.n_qt = (p.N + BM - 1) / BM;
  kp.scale_log2 = kLog2e * p.scale;
  const long long items = static_cast<long long>(kp.n_qt) * p.B * p.units;
  if (items == 0) return cudaSuccess;
  kern<<<dim3(static_cast<unsigned>(items)), kThreads, C::kDynSmem, s>>>(mq, mk, mv, kp);
  return cudaGetLastError();
}

}  // namespace exact

cudaError_t status_prefill_exact(int* v) { return read_clear_status(v); }

cudaError_t launch_prefill_exact(const Problem& p, cudaStream_t s, char* err, size_t err_len) {
  if (p.mode == MODE_V1) {
    if (p.dqk == 128 && p.dv == 256) return exact::launch_cfg<128, 256, false>(p, s, err, err_len);
    if (p.dqk == 64 && p.dv == 128) return exact::launch_cfg<64, 128, false>(p, s, err, err_len);
  } else {
    if (p.dqk == 128 && p.dv == 128) return exact::launch_cfg<128, 128, true>(p, s, err, err_len);
    if (p.dqk == 64 && p.dv == 64) return exact::launch_cfg<64, 64, true>(p, s, err, err_len);
  }
  return cudaErrorNotSupported;
}

}  // namespace da
