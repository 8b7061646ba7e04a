// prefill_tc.cu -- fused differential-attention prefill on the sm_103a tensor cores.
//
// Operator (page "Differential Transformer: softmax can't say zero, so it subtracts", section
// "The mechanism, exactly"): out = (softmax(Q1 K1^T/sqrt d) - lambda softmax(Q2 K2^T/sqrt d)) V,
// then a per-head RMSNorm over the dv channels and a (1 - lambda_init) scale (section "The row no
// longer sums to one"). The V2 variant (section "DIFF V2: what the authors changed") subtracts
// two query heads of one GQA group with a per-token sigmoid lambda and no norm.
//
// Design. A cluster of two CTAs owns one 128-row query tile of one unit (head or V2 pair):
// CTA rank r computes map r as a flash-attention pass -- TMA stages Q_r, K_r and the shared V
// tile into 128B-swizzled shared memory, tcgen05.mma writes the 128x128 score tile into tensor
// memory (double-buffered), four softmax warps (one thread per query row) keep the map's own
// running max and sum, write P as bf16 back into the score columns, and a second tcgen05.mma
// (A = P from tensor memory, B = V from shared memory) accumulates O_r (128 x dv fp32) in tensor
// memory. Per CTA: S buffers 2 x 128 columns + O dv <= 256 columns = all 512 TMEM columns,
// which is why the two maps live on two SMs. Both CTAs stream the same V tile; the second read
// is served by L2, so HBM sees V once. The epilogue exchanges half of each O row through
// distributed shared memory: rank 0 ends with columns [0, dv/2) and rank 1 with [dv/2, dv) of
// O1/l1 - lambda O2/l2; the two halves' sums of squares are exchanged for the RMSNorm.
//
// Warp roles (256 threads): warp 0 = TMA producer, warp 1 = MMA issuer and TMEM owner,
// warps 4-7 = softmax / correction / epilogue (row = 32 * (warp % 4) + lane, matching the TMEM
// lane quarter each warp may access). Every mbarrier wait is bounded (ptx.cuh); on a timeout the
// kernel flags the device status word and unwinds without trapping.
#include <cuda.h>
#include <cuda_bf16.h>

#include <cmath>
#include <cstdio>

#include "internal.h"
#include "ptx.cuh"

namespace da {
namespace tc {

constexpr int BM = 128;
constexpr int BN = 128;
constexpr int kThreads = 256;
constexpr int kSoftmaxWarp0 = 4;
constexpr int kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: stale max allowed while p <= 2^8

template <int DQK, int DV, int NS>
struct Cfg {
  static constexpr int kChunkBytes = 128 * 128;          // one 128-row x 64-col bf16 box
  static constexpr int kQBytes = BM * DQK * 2;
  static constexpr int kKBytes = BN * DQK * 2;
  static constexpr int kVBytes = BN * DV * 2;
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + kQBytes;
  static constexpr int kVOff = kKOff + NS * kKBytes;
  static constexpr int kEnd = kVOff + NS * kVBytes;
  static constexpr int kXStride = DV / 2 + 4;            // floats per exchange-buffer row
  static constexpr int kXBytes = BM * kXStride * 4;
  static constexpr int kDynSmem = kEnd + 1024;           // + slack for 1024 B alignment
  static constexpr int kSCol = 0;                        // S buffers at columns 0 and 128
  static constexpr int kOCol = 256;                      // O at columns 256 .. 256 + DV
  static_assert(DQK % 64 == 0 && DV % 64 == 0, "64-column TMA boxes");
  static_assert(kXBytes <= NS * kVBytes, "exchange buffer reuses the V stages");
  static_assert(kOCol + DV <= kTmemCols, "TMEM budget");
  static_assert(kDynSmem <= 232448 - 1024, "shared memory budget");
};

struct Barriers {
  uint64_t q_full;
  uint64_t k_full[4], k_empty[4], v_full[4], v_empty[4];
  uint64_t s_full[2], p_full[2];
  uint64_t o_done;
  uint64_t teardown;
  uint64_t can_write, data_ready, ss_ready;  // cluster exchange (arrived by the peer CTA)
};

struct KParams {
  Problem p;
  int n_qt;         // query tiles per unit
  float scale_log2; // log2(e) / sqrt(dqk)
};

template <int DQK, int DV, int NS>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const KParams kp) {
  using C = Cfg<DQK, DV, NS>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ Barriers bars;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  __shared__ float ss_peer[BM];

  const Problem& P = kp.p;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sQ = smem_u32(smem + C::kQOff);
  const uint32_t sK = smem_u32(smem + C::kKOff);
  const uint32_t sV = smem_u32(smem + C::kVOff);
  float* xbuf = reinterpret_cast<float*>(smem + C::kVOff);

  // ---- work item: longest causal tiles first ----
  const int cluster_id = blockIdx.x >> 1;
  const int BU = P.B * P.units;
  const bool causal = (P.flags & 1) != 0;
  const int qt = causal ? (kp.n_qt - 1 - cluster_id / BU) : (cluster_id / BU);
  const int bu = cluster_id % BU;
  const int b = bu / P.units, u = bu % P.units;
  const int n_kv_all = (P.N + BN - 1) / BN;
  const int n_kv = causal ? min(qt + 1, n_kv_all) : n_kv_all;

  auto bar = [](uint64_t& x) { return smem_u32(&x); };

  if (threadIdx.x == 0) {
    mbar_init(bar(bars.q_full), 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(bar(bars.k_full[s]), 1);
      mbar_init(bar(bars.k_empty[s]), 1);
      mbar_init(bar(bars.v_full[s]), 1);
      mbar_init(bar(bars.v_empty[s]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(bars.s_full[i]), 1);
      mbar_init(bar(bars.p_full[i]), 128);
    }
    mbar_init(bar(bars.o_done), 1);
    mbar_init(bar(bars.teardown), 1);
    mbar_init(bar(bars.can_write), 128);
    mbar_init(bar(bars.data_ready), 128);
    mbar_init(bar(bars.ss_ready), 128);
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
  cluster_sync_all();  // barrier inits visible cluster-wide, TMEM address published
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  volatile int* abrt = &abort_flag;

  if (warp == 0) {
    // ================================ TMA producer ================================
    if (lane == 0) {
      const int qh = q_head_of(P, u, rank), qc = q_col_of(P, rank);
      const int kvh = kv_head_of(P, u), kc = k_col_of(P, rank);  // V head; K column
      const int kh = k_head_of(P, u, rank);                        // K head of this CTA's map
      // extents of the three tensor maps (the host builds them with these dimensions)
      const Ext4 eq{P.q_cols, P.q_heads, P.N, P.B, 2}, ek{P.k_cols, P.kv_heads, P.N, P.B, 2};
      const Ext4 ev{DV, v_heads(P), P.N, P.B, 2};
      mbar_arrive_expect_tx(bar(bars.q_full), C::kQBytes);
      for (int c = 0; c < DQK / 64; ++c)
        tma_load_4d_chk(sQ + c * C::kChunkBytes, &tm_q, bar(bars.q_full), qc + 64 * c, qh, qt * BM,
                        b, eq);
      int issued = 0;
      for (int j = 0; j < n_kv; ++j) {
        const int s = j % NS;
        const uint32_t ph = (j / NS) & 1;
        if (!mbar_wait(bar(bars.k_empty[s]), ph ^ 1, abrt)) break;
        mbar_arrive_expect_tx(bar(bars.k_full[s]), C::kKBytes);
        for (int c = 0; c < DQK / 64; ++c)
          tma_load_4d_chk(sK + s * C::kKBytes + c * C::kChunkBytes, &tm_k, bar(bars.k_full[s]),
                          kc + 64 * c, kh, j * BN, b, ek);
        if (!mbar_wait(bar(bars.v_empty[s]), ph ^ 1, abrt)) {
          issued = 2 * j + 1;
          break;
        }
        mbar_arrive_expect_tx(bar(bars.v_full[s]), C::kVBytes);
        for (int c = 0; c < DV / 64; ++c)
          tma_load_4d_chk(sV + s * C::kVBytes + c * C::kChunkBytes, &tm_v, bar(bars.v_full[s]),
                          64 * c, kvh, j * BN, b, ev);
        issued = 2 * j + 2;
      }
      // Before leaving, make sure no copy of ours is still landing in shared memory.
      mbar_wait(bar(bars.q_full), 0, nullptr);
      for (int t = issued - 1; t >= 0 && t >= issued - 2 * NS; --t) {
        const int j = t >> 1, s = j % NS;
        const uint32_t ph = (j / NS) & 1;
        mbar_wait((t & 1) ? bar(bars.v_full[s]) : bar(bars.k_full[s]), ph, nullptr);
      }
    }
  } else if (warp == 1) {
    // ================================ MMA issuer ==================================
    if (lane == 0) {
      constexpr uint32_t idesc_s = umma_idesc_bf16(BM, BN, 0, 0);
      constexpr uint32_t idesc_o = umma_idesc_bf16(BM, DV, 0, 1);
      // Descriptors are built once; each k-step adds a constant offset.
      const uint64_t dq0 = umma_smem_desc(sQ, 16, 1024);
      const uint64_t dk0 = umma_smem_desc(sK, 16, 1024);
      const uint64_t dv0 = umma_smem_desc(sV, C::kChunkBytes, 1024);
      bool ok = mbar_wait(bar(bars.q_full), 0, abrt);
      tc_fence_after();
      for (int j = 0; ok && j <= n_kv; ++j) {
        if (j < n_kv) {
          const int s = j % NS, buf = j & 1;
          if (!(ok = mbar_wait(bar(bars.k_full[s]), (j / NS) & 1, abrt))) break;
          tc_fence_after();
          const uint32_t d_s = tmem + C::kSCol + buf * BN;
#pragma unroll
          for (int kk = 0; kk < DQK / 16; ++kk) {
            const uint32_t off = (kk >> 2) * C::kChunkBytes + (kk & 3) * 32;
            mma_bf16_ss(d_s, desc_add(dq0, off), desc_add(dk0, s * C::kKBytes + off), idesc_s,
                        kk > 0 ? 1u : 0u);
          }
          tc_commit(bar(bars.k_empty[s]));
          tc_commit(bar(bars.s_full[buf]));
        }
        if (j >= 1) {
          const int jp = j - 1, sp = jp % NS, bp = jp & 1;
          if (!(ok = mbar_wait(bar(bars.p_full[bp]), (jp >> 1) & 1, abrt))) break;
          if (!(ok = mbar_wait(bar(bars.v_full[sp]), (jp / NS) & 1, abrt))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk) {
            const uint32_t a_t = tmem + C::kSCol + bp * BN + kk * 8;  // 16 bf16 keys = 8 cols
            mma_bf16_ts(tmem + C::kOCol, a_t, desc_add(dv0, sp * C::kVBytes + kk * 2048), idesc_o,
                        (jp > 0 || kk > 0) ? 1u : 0u);
          }
          tc_commit(bar(bars.v_empty[sp]));
          tc_commit(bar(bars.o_done));
        }
      }
      // Wait for every MMA we issued before TMEM can be released.
      tc_commit(bar(bars.teardown));
      mbar_wait(bar(bars.teardown), 0, nullptr);
    }
  } else if (warp >= kSoftmaxWarp0) {
    // ======================== softmax / correction / epilogue =====================
    const int r = 32 * (warp & 3) + lane;            // row within the tile
    const int row = qt * BM + r;                     // query position
    const uint32_t tl = static_cast<uint32_t>(32 * (warp & 3)) << 16;  // TMEM lane quarter
    const float sl2 = kp.scale_log2;
    float m = -INFINITY, l = 0.f;
    bool ok = true;

    for (int j = 0; j < n_kv; ++j) {
      const int buf = j & 1;
      ok = mbar_wait(bar(bars.s_full[buf]), (j >> 1) & 1, abrt);
      if (__any_sync(0xffffffffu, !ok)) { ok = false; break; }
      tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tmem + tl + C::kSCol + buf * BN + 32 * c, sr[c]);
      tmem_wait_ld();
      // raw scores; masked keys become -inf
      const int key0 = j * BN;
      const int lim = causal ? min(row + 1, P.N) : P.N;  // keys [0, lim) are visible
      if (key0 + BN > lim) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (key0 + 32 * c + i >= lim) sr[c][i] = __float_as_uint(-INFINITY);
      }
      __syncwarp();
      float mx[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mx[i] = __uint_as_float(sr[0][i]);
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int i = 0; i < 32; ++i)
          mx[i & 7] = fmaxf(mx[i & 7], __uint_as_float(sr[c][i]));
#pragma unroll
      for (int i = 0; i < 4; ++i) mx[i] = fmaxf(mx[i], mx[i + 4]);
      const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * sl2;
      if (j == 0) {
        m = mt;
      } else {
        const bool need = mt > m + kRescaleThreshold;
        if (__any_sync(0xffffffffu, need)) {
          // O holds tiles 0 .. j-1 scaled by the old max: wait for PV(j-1), then rescale O.
          const float mn = need ? mt : m;
          const float f = ex2_approx(m - mn);
          l *= f;
          m = mn;
          ok = mbar_wait(bar(bars.o_done), (j - 1) & 1, abrt);
          if (__any_sync(0xffffffffu, !ok)) { ok = false; break; }
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < DV / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tmem + tl + C::kOCol + 32 * c, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * f);
            tmem_st32(tmem + tl + C::kOCol + 32 * c, o);
          }
          tmem_wait_st();
        }
      }
      // P = 2^(s * scale_log2 - m) in bf16, written over the first 64 columns of this S buffer
      const float nmo = (m == -INFINITY) ? 0.f : -m;
      float lacc[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint32_t pk[8];
        float la = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int e = 16 * c + 2 * i;
          const float p0 = ex2_approx(fmaf(__uint_as_float(sr[e >> 5][e & 31]), sl2, nmo));
          const float p1 = ex2_approx(fmaf(__uint_as_float(sr[(e + 1) >> 5][(e + 1) & 31]), sl2, nmo));
          la += p0 + p1;
          pk[i] = pack_bf16x2(p0, p1);
        }
        lacc[c] = la;
        tmem_st8(tmem + tl + C::kSCol + buf * BN + 8 * c, pk);
      }
      l += ((lacc[0] + lacc[1]) + (lacc[2] + lacc[3])) + ((lacc[4] + lacc[5]) + (lacc[6] + lacc[7]));
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(bars.p_full[buf]));
    }
    if (ok) {
      ok = mbar_wait(bar(bars.o_done), (n_kv - 1) & 1, abrt);
      ok = !__any_sync(0xffffffffu, !ok);
    }
    tc_fence_after();

    // ------------------------------- epilogue -------------------------------------
    float f;
    if (P.mode != MODE_V2) {
      f = (rank == 0 ? 1.f : P.lambda[u]) / l;
    } else {
      float lam = 0.f;
      if (row < P.N) {
        const float z = P.lam_logit[(static_cast<size_t>(b) * P.N + row) * P.units + u];
        lam = 1.f / (1.f + expf(-z));
      }
      f = (rank == 0 ? 1.f : lam) / l;
    }
    constexpr int H2 = DV / 2;
    const int send0 = rank == 0 ? H2 : 0;
    const int keep0 = rank == 0 ? 0 : H2;
    float* xrow = xbuf + r * C::kXStride;
    const uint32_t xrow_peer = mapa_shared(smem_u32(xrow), peer);

    // 1) tell the peer it may write into our (now idle) V stages; wait for its permission.
    mbar_arrive_remote(mapa_shared(bar(bars.can_write), peer));
    bool w_ok = mbar_wait<true>(bar(bars.can_write), 0, nullptr);
    ok = ok && !__any_sync(0xffffffffu, !w_ok);
    // 2) send our scaled half of the row.
    if (ok) {
#pragma unroll 1
      for (int c = 0; c < H2 / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tmem + tl + C::kOCol + send0 + 32 * c, o);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; i += 4)
          st_cluster_v4(xrow_peer + (32 * c + i) * 4, __uint_as_float(o[i]) * f,
                        __uint_as_float(o[i + 1]) * f, __uint_as_float(o[i + 2]) * f,
                        __uint_as_float(o[i + 3]) * f);
      }
    }
    mbar_arrive_remote(mapa_shared(bar(bars.data_ready), peer));
    bool d_ok = mbar_wait<true>(bar(bars.data_ready), 0, nullptr);
    ok = ok && !__any_sync(0xffffffffu, !d_ok);
    // 3) combine with the peer's half: y = O1/l1 - lambda O2/l2 on our columns.
    float ss = 0.f;
    if (ok) {
#pragma unroll 1
      for (int c = 0; c < H2 / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tmem + tl + C::kOCol + keep0 + 32 * c, o);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          float4 pv = *reinterpret_cast<float4*>(xrow + 32 * c + i);
          float4 y;
          const float a0 = __uint_as_float(o[i]) * f, a1 = __uint_as_float(o[i + 1]) * f;
          const float a2 = __uint_as_float(o[i + 2]) * f, a3 = __uint_as_float(o[i + 3]) * f;
          if (rank == 0) {
            y = make_float4(a0 - pv.x, a1 - pv.y, a2 - pv.z, a3 - pv.w);
          } else {
            y = make_float4(pv.x - a0, pv.y - a1, pv.z - a2, pv.w - a3);
          }
          ss += y.x * y.x + y.y * y.y + y.z * y.z + y.w * y.w;
          *reinterpret_cast<float4*>(xrow + 32 * c + i) = y;
        }
      }
    }
    // 4) RMSNorm over all dv channels: exchange the halves' sums of squares.
    float scale = 1.f;
    if (P.flags & 2) {
      if (ok) st_cluster_f32(mapa_shared(smem_u32(&ss_peer[r]), peer), ss);
      mbar_arrive_remote(mapa_shared(bar(bars.ss_ready), peer));
      bool s_ok = mbar_wait<true>(bar(bars.ss_ready), 0, nullptr);
      ok = ok && !__any_sync(0xffffffffu, !s_ok);
      const float tot = ss + ss_peer[r];
      scale = 1.f / sqrtf(tot / static_cast<float>(DV) + P.eps);
    }
    if (P.flags & 4) scale *= (1.f - P.lambda_init);
    // 5) store our half of the row.
    if (ok && row < P.N) {
      __nv_bfloat16* out = static_cast<__nv_bfloat16*>(P.out) +
                           ((static_cast<size_t>(b) * P.N + row) * P.units + u) * DV + keep0;
      const float* w = P.norm_w ? P.norm_w + keep0 : nullptr;
#pragma unroll 4
      for (int c = 0; c < H2; c += 8) {
        const float4 y0 = *reinterpret_cast<const float4*>(xrow + c);
        const float4 y1 = *reinterpret_cast<const float4*>(xrow + c + 4);
        float g[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
        uint4 pkt;
        uint32_t* pw = reinterpret_cast<uint32_t*>(&pkt);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float w0 = (w && (P.flags & 2)) ? w[c + 2 * i] : 1.f;
          const float w1 = (w && (P.flags & 2)) ? w[c + 2 * i + 1] : 1.f;
          pw[i] = pack_bf16x2(g[2 * i] * scale * w0, g[2 * i + 1] * scale * w1);
        }
        *reinterpret_cast<uint4*>(out + c) = pkt;
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
// 4-D bf16 map over [B, N, heads, cols] (cols innermost) with a 64-col x 1 x 128-row x 1 box,
// 128-byte swizzle, zero fill out of bounds.
static bool make_map(CUtensorMap* m, const void* base, int cols, int heads, int N, int B,
                     char* err, size_t err_len) {
  cuuint64_t dims[4] = {(cuuint64_t)cols, (cuuint64_t)heads, (cuuint64_t)N, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)cols * 2, (cuuint64_t)cols * heads * 2,
                           (cuuint64_t)cols * heads * 2 * (cuuint64_t)N};
  cuuint32_t box[4] = {64, 1, 128, 1};
  return encode_tmap_4d(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, dims, strides, box, err, err_len);
}

template <int DQK, int DV, int NS>
static cudaError_t launch_cfg(const Problem& p, cudaStream_t s, char* err, size_t err_len) {
  using C = Cfg<DQK, DV, NS>;
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, p.q, p.q_cols, p.q_heads, p.N, p.B, err, err_len) ||
      !make_map(&mk, p.k, p.k_cols, p.kv_heads, p.N, p.B, err, err_len) ||
      !make_map(&mv, p.v, DV, v_heads(p), p.N, p.B, err, err_len))
    return cudaErrorInvalidValue;
  auto kern = prefill_tc_kernel<DQK, DV, NS>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kDynSmem);
  if (e != cudaSuccess) return e;
  KParams kp;
  kp.p = p;
  kp.n_qt = (p.N + BM - 1) / BM;
  kp.scale_log2 = kLog2e * p.scale;
  const long long clusters = static_cast<long long>(kp.n_qt) * p.B * p.units;
  if (clusters == 0) return cudaSuccess;
  kern<<<dim3(static_cast<unsigned>(2 * clusters)), kThreads, C::kDynSmem, s>>>(mq, mk, mv, kp);
  return cudaGetLastError();
}

}  // namespace tc

cudaError_t status_prefill_tc(int* v) { return read_clear_status(v); }

cudaError_t launch_prefill_tc(const Problem& p, cudaStream_t s, char* err, size_t err_len) {
  if (p.dqk == 128 && p.dv == 256) return tc::launch_cfg<128, 256, 2>(p, s, err, err_len);
  if (p.dqk == 128 && p.dv == 128) return tc::launch_cfg<128, 128, 3>(p, s, err, err_len);
  if (p.dqk == 64 && p.dv == 128) return tc::launch_cfg<64, 128, 4>(p, s, err, err_len);
  if (p.dqk == 64 && p.dv == 64) return tc::launch_cfg<64, 64, 4>(p, s, err, err_len);
  return cudaErrorNotSupported;
}

}  // namespace da
