// backward.cu -- gradients of the V1 prefill (page "Differential Transformer: softmax can't say
// zero, so it subtracts", section "The mechanism, exactly" gives the forward; the backward is its
// chain rule taken step by step in reverse).
//
// Per head, with c = 1/sqrt(d), A_m = softmax(c Q_m K_m^T) (causal), W = A1 - lam A2, O = W V and
// Y = RMSNorm(O) * w * (1 - lambda_init):
//   dO from dY through the norm;  dW = dO V^T;  dV = W^T dO;  dlam = -sum(A2 * dW)
//   dS_m = coef_m * A_m * (dW - delta_m),  coef_1 = 1, coef_2 = -lam,
//   delta_m[i] = sum_j A_m[i,j] dW[i,j] = dO_i . (A_m V)_i
//   dQ_m = c dS_m K_m,  dK_m = c dS_m^T Q_m.
// The forward for training saves, per row and map, b_m = log2 sum_j 2^(c log2(e) s_ij), so that
// A_m = 2^(c log2(e) s - b_m) is recomputed exactly without a running max.
//
// Kernels, in launch order:
//   bwd_pre_kernel    CUDA cores: norm backward -> dO (bf16), D = dO . O, norm-weight partials;
//                     zeroes the fp32 dQ accumulator.
//   bwd_delta_kernel  tcgen05, query-major: O2 = A2 V -> delta_2 = dO . O2,
//                     delta_1 = D + lam delta_2 (because O = O1 - lam O2), and -sum delta_2 per CTA.
//   bwd_dkdq_kernel   tcgen05, key-major, one map per CTA: S = Q K^T, dW = dO V^T per inner
//                     tile, dS in shared memory, dK += dS^T Q (TMEM), dQ partial = dS K (TMEM)
//                     added to the fp32 accumulator with TMA tensor reductions.
//   bwd_dv_kernel     tcgen05, key-major: S1, S2 per inner tile -> W in shared memory,
//                     dV += W^T dO.
//   bwd_finish_kernel dQ fp32 -> bf16; dlam and norm-weight sums (fixed order: deterministic).
// TMEM is 512 columns per SM; each tensor-core kernel fills it exactly:
//   delta: S double-buffered (2 x 128) + O2 (256);  dkdq: S^T, dW^T, dK, dQ (4 x 128);
//   dv: S1^T, S2^T (2 x 128) + dV (256).
// Every wait is bounded (2 s); a timeout flags DEV_TIMEOUT in this file's status word and the
// roles unwind without hanging.
//
// Grouped form (GR instantiations, page "Differential Transformer: softmax can't say zero, so it
// subtracts", section "What other people found"): q, k are [B, N, Hs + Hn, d] with map 2 of
// signal head h in noise head Hs + h / G; the tile kernels read map 2's Q and K there. dQ goes to
// an fp32 accumulator of q's layout as before; a noise head's dK2 collects the contributions of
// the G signal heads of its group through fp32 reductions into dkacc [tokens, Hn, d], converted
// by bwd_gda_dk_kernel.
#include <cuda.h>

#include <cstdio>

#include "internal.h"
#include "ptx.cuh"

namespace da {
namespace bwd {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kD = 128;    // width of one query/key half
constexpr int kDV = 256;   // value width
constexpr int kT = 128;    // rows per tile (queries or keys)
constexpr int kBox = kT * 128;  // one 64-column box of a 128-row tile: 16 KB

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}
// bulk_load of n floats at element offset `off` of an fp32 array of `total` elements. Debug
// builds check the range; a failed check loads from offset 0, so the barrier still completes.
__device__ __forceinline__ void bulk_load_f32(uint32_t dst, const float* base, size_t off,
                                              size_t total, uint32_t n, uint32_t bar) {
  if constexpr (kDebugChecks) {
    if (off + n > total) {
      flag_device_error(DEV_BOUNDS);
      off = 0;
    }
  }
  bulk_load(dst, base + off, n * 4, bar);
}
__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b),
               "f"(c), "f"(d)
               : "memory");
}
// Add a shared-memory tile into global memory through a tensor map (fp32 add in L2).
__device__ __forceinline__ void tma_reduce_add_4d(const void* tmap, uint32_t smem_src, int c0,
                                                  int c1, int c2, int c3) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.4d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(tmap)),
      "r"(smem_src), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read_le1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ bool bar_and(uint32_t id, uint32_t count, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\tsetp.ne.u32 pi, %1, 0;\n\t"
      "barrier.red.and.pred po, %2, %3, pi;\n\tselp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}
__device__ __forceinline__ uint64_t f2mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Launch order for L2 reuse: work units (a head, or a head and map) are taken in groups of
// `group`; inside a group, tile rank 0 (the longest causal tile) of every unit first, then rank 1,
// and so on. Returns the unit and the tile rank of item `idx`.
__device__ __forceinline__ void grouped_item(int idx, int n_units, int n_tiles, int group,
                                             int& unit, int& rank) {
  const int g0 = (idx / (group * n_tiles)) * group;
  const int gsize = min(group, n_units - g0);
  const int r = idx - g0 * n_tiles;
  rank = r / gsize;
  unit = g0 + r % gsize;
}

struct Args {
  const __nv_bfloat16* q;   // [B, N, H, 2d]
  const __nv_bfloat16* k;   // [B, N, H, 2d]
  const __nv_bfloat16* v;   // [B, N, H, dv]
  const __nv_bfloat16* o_pre;  // [B, N, H, dv]
  const __nv_bfloat16* dy;     // [B, N, H, dv]
  const float* stats;          // [B, H, 2, Npad]
  const float* lambda;         // [H]
  const float* norm_w;         // [dv] or null
  __nv_bfloat16* dq;           // [B, N, H, 2d]
  __nv_bfloat16* dk;           // [B, N, H, 2d]
  __nv_bfloat16* dv;           // [B, N, H, dv]
  float* dlambda;              // [H]
  float* dnorm_w;              // [dv] or null
  // workspace
  __nv_bfloat16* dO;           // [B, N, H, dv]
  float* delta;                // [B, H, 2, Npad]: D (after pre) then delta_1; delta_2
  float* dqacc;                // [B, N, H, 2d]
  float* dw_part;              // [pre blocks, dv]
  float* dl_part;              // [B, H, n_qt]
  int B, N, H, Npad, n_t;
  int pre_blocks;
  int grp_delta, grp_dkdq, grp_dv;  // L2 groups (units per group) of the three tile kernels
  float eps, scale_out;        // scale_out = (1 - lambda_init) with DIFFATTN_SCALE, else 1
  bool norm, causal;
  float c_log2;                // log2(e) / sqrt(d)
  float c;                     // 1 / sqrt(d)
  // packed sequences (null: batched): sequence b is rows cu[b] .. cu[b+1]-1 of [total, H, *];
  // N is then the longest sequence, and stats, delta, dl_part keep their per-sequence layout
  const int* cu;
  int total;
  // grouped form: G signal heads per noise head (0: the ungrouped layout), heads of q and k
  // (Hs + Hn), and the noise heads' fp32 dK accumulator [tokens, Hn, d]
  int group, hqk;
  float* dkacc;
};

// Head and first column of map m's Q or K for unit h: [Q1 | Q2] of head h, or (grouped) head h
// for map 1 and noise head H + h / G for map 2, each d wide.
template <bool GR>
__device__ __forceinline__ int qk_head(const Args& a, int h, int m) {
  if constexpr (GR) return m ? a.H + h / a.group : h;
  else return h;
}
template <bool GR>
__device__ __forceinline__ int qk_col(int m) {
  return GR ? 0 : m * kD;
}

// Rows of sequence b: [s0, s0 + len) of the token axis (batched: b N .. b N + N - 1), and the
// TMA coordinates (row, batch) of its first row. False for offsets outside the packed tensor
// or longer than N: the caller reports DEV_BAD_INDEX and skips the sequence. A tile that reaches
// past the sequence's end reads (and, for dQ, adds zeros into) the next sequence's rows, which
// every mask treats as past the end.
struct SeqRows {
  int s0, len, trow, tb;
};
__device__ __forceinline__ bool seq_rows(const Args& a, int b, SeqRows& s) {
  if (!a.cu) {
    s.s0 = b * a.N;
    s.len = a.N;
    s.trow = 0;
    s.tb = b;
    return true;
  }
  s.s0 = a.cu[b];
  s.len = a.cu[b + 1] - s.s0;
  s.trow = s.s0;
  s.tb = 0;
  return s.s0 >= 0 && s.len >= 0 && s.len <= a.N && s.s0 <= a.total - s.len;
}

// Extent of the tensor maps over [B, N, H, cols] (packed: one batch row of `total` tokens), for
// the debug-build checks of tile coordinates.
__device__ __forceinline__ Ext4 map_ext(const Args& a, int cols, int elt) {
  return Ext4{cols, a.H, a.cu ? a.total : a.N, a.cu ? 1 : a.B, elt};
}
// Extent of the q and k maps (and of the dQ accumulator, elt 4)
template <bool GR>
__device__ __forceinline__ Ext4 qk_ext(const Args& a, int elt) {
  return GR ? Ext4{kD, a.hqk, a.cu ? a.total : a.N, a.cu ? 1 : a.B, elt} : map_ext(a, 2 * kD, elt);
}

// =============================================================================================
// bwd_pre_kernel: one warp per (b, n, h) row, lane = 8 channels. Without the norm dO = s dY;
// with it (r = (mean(O^2) + eps)^-1/2, Yhat = O r, g = s dY w): dO = r (g - Yhat mean(g Yhat)),
// dw += s dY Yhat. D = dO . O uses dO as rounded to bf16 (the value the MMAs see).
// =============================================================================================
constexpr int kPreWarps = 8;

__global__ void __launch_bounds__(kPreWarps * 32) bwd_pre_kernel(const Args a) {
  __shared__ float sdw[kPreWarps][kDV];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // packed: rows past the last sequence belong to none and are skipped
  const long long rows = a.cu ? static_cast<long long>(min(max(a.cu[a.B], 0), a.total)) * a.H
                              : static_cast<long long>(a.B) * a.N * a.H;
  float wl[8], dwl[8];
  float4 w0 = make_float4(1.f, 1.f, 1.f, 1.f), w1 = w0;
  if (a.norm_w) {
    w0 = reinterpret_cast<const float4*>(a.norm_w + 8 * lane)[0];
    w1 = reinterpret_cast<const float4*>(a.norm_w + 8 * lane)[1];
  }
  wl[0] = w0.x; wl[1] = w0.y; wl[2] = w0.z; wl[3] = w0.w;
  wl[4] = w1.x; wl[5] = w1.y; wl[6] = w1.z; wl[7] = w1.w;
#pragma unroll
  for (int i = 0; i < 8; ++i) dwl[i] = 0.f;
  const float s = a.scale_out;
  for (long long r = static_cast<long long>(blockIdx.x) * kPreWarps + warp; r < rows;
       r += static_cast<long long>(gridDim.x) * kPreWarps) {
    const size_t off = static_cast<size_t>(r) * kDV + 8 * lane;
    float o[8], dy[8], g[8];
    bf16x8_to_f32(*reinterpret_cast<const uint4*>(a.o_pre + off), o);
    bf16x8_to_f32(*reinterpret_cast<const uint4*>(a.dy + off), dy);
    float dO[8];
    if (a.norm) {
      float ss = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) ss = fmaf(o[i], o[i], ss);
      const float rs = rsqrtf(warp_sum(ss) / kDV + a.eps);
      float gy = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        g[i] = s * dy[i] * wl[i];
        gy = fmaf(g[i], o[i] * rs, gy);
        dwl[i] = fmaf(s * dy[i], o[i] * rs, dwl[i]);
      }
      const float mg = warp_sum(gy) / kDV;
#pragma unroll
      for (int i = 0; i < 8; ++i) dO[i] = rs * (g[i] - o[i] * rs * mg);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) dO[i] = s * dy[i];
    }
    uint4 pk;
    pk.x = pack_bf16x2(dO[0], dO[1]);
    pk.y = pack_bf16x2(dO[2], dO[3]);
    pk.z = pack_bf16x2(dO[4], dO[5]);
    pk.w = pack_bf16x2(dO[6], dO[7]);
    *reinterpret_cast<uint4*>(a.dO + off) = pk;
    float dr[8];
    bf16x8_to_f32(pk, dr);
    float Dp = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) Dp = fmaf(dr[i], o[i], Dp);
    const float D = warp_sum(Dp);
    const int h = static_cast<int>(r % a.H);
    const long long bn = r / a.H;
    int n, b;
    if (a.cu) {  // the sequence holding token bn: the last b with cu[b] <= bn
      int lo = 0, hi = a.B - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.cu[mid] <= bn) lo = mid; else hi = mid - 1;
      }
      b = lo;
      n = static_cast<int>(bn - a.cu[b]);
    } else {
      n = static_cast<int>(bn % a.N);
      b = static_cast<int>(bn / a.N);
    }
    if (lane == 0 && n < a.Npad) a.delta[(static_cast<size_t>(b) * a.H + h) * 2 * a.Npad + n] = D;
    float4* zq = reinterpret_cast<float4*>(a.dqacc + static_cast<size_t>(r) * (2 * kD) + 8 * lane);
    zq[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    zq[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    // grouped: the noise heads' dK accumulator, d floats per row (its rows [tokens, Hn] lie
    // inside the tokens x Hs rows zeroed here)
    if (a.dkacc)
      reinterpret_cast<float4*>(a.dkacc + static_cast<size_t>(r) * kD)[lane] =
          make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) sdw[warp][8 * lane + i] = dwl[i];
  __syncthreads();
  for (int cidx = threadIdx.x; cidx < kDV; cidx += blockDim.x) {
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < kPreWarps; ++w) t += sdw[w][cidx];
    a.dw_part[static_cast<size_t>(blockIdx.x) * kDV + cidx] = t;
  }
}

// =============================================================================================
// bwd_delta_kernel: one CTA per (query tile, b, h). Warp 0 TMA, warp 1 MMA + TMEM, warps 2-5:
// thread r = query row r. S2 = Q2 K2^T (double-buffered TMEM), P2 = 2^(c' s - b2) to shared
// memory (K-major), O2 += P2 V (TMEM). Then delta_2 = dO . O2, delta_1 = D + lam delta_2.
// Loads stream through a ring of 32 KB slots in the order the MMA issuer uses them:
// K2_0, then per tile t >= 1: K2_t, V_{t-1} keys 0-63, V_{t-1} keys 64-127; finally V_{n-1}.
// =============================================================================================
namespace dl {
constexpr int kThreads = 192;
constexpr int kSlot = 32 * 1024;
constexpr int kNSlot = 5;
constexpr int kQOff = 0;                         // Q2 tile, 32 KB
constexpr int kPOff = kQOff + 2 * kBox;          // P buffer, 32 KB
constexpr int kRingOff = kPOff + 2 * kBox;       // ring
constexpr int kCtrlOff = kRingOff + kNSlot * kSlot;
constexpr int kVHalfBox = 64 * 128;              // one 64-column box of 64 keys: 8 KB
struct Ctrl {
  uint64_t q_full, slot_full[kNSlot], slot_empty[kNSlot], s_full[2], s_free[2], p_full, p_empty,
      o_full, teardown;
  uint32_t tmem_slot;
  int abort_flag;
  float red[4];
};
constexpr int kDynSmem = kCtrlOff + static_cast<int>(sizeof(Ctrl));
}  // namespace dl

template <bool GR>
__global__ void __launch_bounds__(dl::kThreads, 1)
    bwd_delta_kernel(const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_vh, const Args a) {
  using namespace dl;
  extern __shared__ __align__(1024) uint8_t smem[];
  Ctrl& cs = *reinterpret_cast<Ctrl*>(smem + kCtrlOff);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sQ = smem_u32(smem + kQOff), sP = smem_u32(smem + kPOff);
  const uint32_t sRing = smem_u32(smem + kRingOff);
  auto bar = [](uint64_t& x) { return smem_u32(&x); };
  if ((smem_u32(smem) & 1023u) != 0) {  // the swizzled layouts need 1 KB alignment
    if (threadIdx.x == 0) flag_device_error(DEV_TIMEOUT);
    return;
  }

  int bh, rank;
  grouped_item(static_cast<int>(blockIdx.x), a.B * a.H, a.n_t, a.grp_delta, bh, rank);
  const int qt = a.causal ? a.n_t - 1 - rank : rank;
  const int b = bh / a.H, h = bh % a.H;
  SeqRows sq;
  const bool seq_ok = seq_rows(a, b, sq);
  const int nts = (sq.len + kT - 1) / kT;  // this sequence's tiles
  if (!seq_ok || qt >= nts) {  // nothing to do (packed): this tile's share of dlambda is 0
    if (threadIdx.x == 0) {
      if (!seq_ok && qt == 0) flag_device_error(DEV_BAD_INDEX);
      a.dl_part[static_cast<size_t>(bh) * a.n_t + qt] = 0.f;
    }
    return;
  }
  const int n = a.causal ? qt + 1 : nts;  // key tiles
  auto k_idx = [](int t) { return t + 2 * max(0, t - 1); };

  if (threadIdx.x == 0) {
    mbar_init(bar(cs.q_full), 1);
    for (int i = 0; i < kNSlot; ++i) {
      mbar_init(bar(cs.slot_full[i]), 1);
      mbar_init(bar(cs.slot_empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(cs.s_full[i]), 1);
      mbar_init(bar(cs.s_free[i]), 128);
    }
    mbar_init(bar(cs.p_full), 128);
    mbar_init(bar(cs.p_empty), 1);
    mbar_init(bar(cs.o_full), 1);
    mbar_init(bar(cs.teardown), 1);
    cs.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&cs.tmem_slot), 512);
    tmem_relinquish();
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = cs.tmem_slot;
  volatile int* abrt = &cs.abort_flag;

  if (warp == 0) {
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_vh);
      mbar_arrive_expect_tx(bar(cs.q_full), 2 * kBox);
      for (int c = 0; c < 2; ++c)
        tma_load_4d_chk(sQ + c * kBox, &tm_q, bar(cs.q_full), qk_col<GR>(1) + 64 * c,
                        qk_head<GR>(a, h, 1), sq.trow + qt * kT, sq.tb, qk_ext<GR>(a, 2));
      int issued = 0;
      bool ok = true;
      auto acquire = [&](int idx, uint32_t bytes) -> int {
        const int s = idx % kNSlot;
        if (!mbar_wait(bar(cs.slot_empty[s]), ((idx / kNSlot) & 1) ^ 1, abrt)) return -1;
        mbar_arrive_expect_tx(bar(cs.slot_full[s]), bytes);
        return s;
      };
      for (int t = 0; t <= n && ok; ++t) {
        int idx = k_idx(t);
        if (t < n) {
          const int s = acquire(idx, 2 * kBox);
          if (s < 0) { ok = false; break; }
          for (int c = 0; c < 2; ++c)
            tma_load_4d_chk(sRing + s * kSlot + c * kBox, &tm_k, bar(cs.slot_full[s]),
                            qk_col<GR>(1) + 64 * c, qk_head<GR>(a, h, 1), sq.trow + t * kT, sq.tb,
                            qk_ext<GR>(a, 2));
          issued = ++idx;
        }
        if (t >= 1) {
          for (int hf = 0; hf < 2 && ok; ++hf) {
            const int s = acquire(idx, 4 * kVHalfBox);
            if (s < 0) { ok = false; break; }
            for (int c = 0; c < 4; ++c)
              tma_load_4d_chk(sRing + s * kSlot + c * kVHalfBox, &tm_vh, bar(cs.slot_full[s]), 64 * c,
                          h, sq.trow + (t - 1) * kT + 64 * hf, sq.tb, map_ext(a, kDV, 2));
            issued = ++idx;
          }
        }
      }
      mbar_wait(bar(cs.q_full), 0, nullptr);
      for (int i = max(0, issued - kNSlot); i < issued; ++i)
        mbar_wait(bar(cs.slot_full[i % kNSlot]), (i / kNSlot) & 1, nullptr);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc_s = umma_idesc_bf16(kT, kT, 0, 0);
      constexpr uint32_t idesc_o = umma_idesc_bf16(kT, kDV, 0, 1);
      const uint64_t dq0 = umma_smem_desc(sQ, 16, 1024);
      const uint64_t dr0 = umma_smem_desc(sRing, 16, 1024);
      const uint64_t dvh0 = umma_smem_desc(sRing, kVHalfBox, 1024);
      const uint64_t dp0 = umma_smem_desc(sP, 16, 1024);
      bool ok = mbar_wait(bar(cs.q_full), 0, abrt);
      tc_fence_after();
      for (int t = 0; ok && t <= n; ++t) {
        int idx = k_idx(t);
        if (t < n) {
          const int buf = t & 1;
          if (t >= 2 && !(ok = mbar_wait(bar(cs.s_free[buf]), ((t >> 1) - 1) & 1, abrt))) break;
          const int s = idx % kNSlot;
          if (!(ok = mbar_wait(bar(cs.slot_full[s]), (idx / kNSlot) & 1, abrt))) break;
          tc_fence_after();
          const uint64_t kd = desc_add(dr0, s * kSlot);
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk) {
            const uint32_t off = (kk >> 2) * kBox + (kk & 3) * 32;
            mma_bf16_ss(tmem + buf * kT, desc_add(dq0, off), desc_add(kd, off), idesc_s,
                        kk > 0 ? 1u : 0u);
          }
          tc_commit(bar(cs.slot_empty[s]));
          tc_commit(bar(cs.s_full[buf]));
          ++idx;
        }
        if (t >= 1) {
          const int jv = t - 1;
          if (!(ok = mbar_wait(bar(cs.p_full), jv & 1, abrt))) break;
          for (int hf = 0; hf < 2; ++hf) {
            const int s = (idx + hf) % kNSlot;
            if (!(ok = mbar_wait(bar(cs.slot_full[s]), ((idx + hf) / kNSlot) & 1, abrt))) break;
            tc_fence_after();
            const uint64_t vd = desc_add(dvh0, s * kSlot);
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4) {
              const int kk = 4 * hf + k4;
              mma_bf16_ss(tmem + 2 * kT, desc_add(dp0, (kk >> 2) * kBox + (kk & 3) * 32),
                          desc_add(vd, k4 * 2048), idesc_o, (jv > 0 || kk > 0) ? 1u : 0u);
            }
            tc_commit(bar(cs.slot_empty[s]));
          }
          if (!ok) break;
          tc_commit(bar(cs.p_empty));
          if (t == n) tc_commit(bar(cs.o_full));
        }
      }
      tc_commit(bar(cs.teardown));
      mbar_wait(bar(cs.teardown), 0, nullptr);
    }
  } else {
    // ---- softmax rows: thread r = query row ----
    const int q4 = warp & 3;
    const int r = 32 * q4 + lane;
    const int row = qt * kT + r;
    const uint32_t tl = static_cast<uint32_t>(32 * q4) << 16;
    const size_t st_base = static_cast<size_t>(b * a.H + h) * 2 * a.Npad;
    const float b2 = row < sq.len ? a.stats[st_base + a.Npad + row] : 0.f;
    const int lim = a.causal ? min(row + 1, sq.len) : sq.len;  // keys [0, lim) visible
    const uint32_t p_row = sP + r * 128;
    bool ok = true;
    for (int t = 0; t < n; ++t) {
      const int buf = t & 1;
      ok = ok && mbar_wait(bar(cs.s_full[buf]), (t >> 1) & 1, abrt);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tmem + tl + buf * kT + 32 * c, sr[c]);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(bar(cs.s_free[buf]));
      const int key0 = t * kT;
      uint32_t pk[kT / 2];
      // the mask is tested outside the unrolled loops: only the tile that reaches the row's
      // last visible key takes the masked copy
      if (key0 + kT <= lim) {
#pragma unroll
        for (int i = 0; i < kT / 2; ++i) {
          const float x0 = fmaf(__uint_as_float(sr[i >> 4][(2 * i) & 31]), a.c_log2, -b2);
          const float x1 = fmaf(__uint_as_float(sr[i >> 4][(2 * i + 1) & 31]), a.c_log2, -b2);
          pk[i] = pack_bf16x2(ex2_approx(x0), ex2_approx(x1));
        }
      } else {
#pragma unroll
        for (int i = 0; i < kT / 2; ++i) {
          const float x0 = fmaf(__uint_as_float(sr[i >> 4][(2 * i) & 31]), a.c_log2, -b2);
          const float x1 = fmaf(__uint_as_float(sr[i >> 4][(2 * i + 1) & 31]), a.c_log2, -b2);
          const float p0 = (key0 + 2 * i < lim) ? ex2_approx(x0) : 0.f;
          const float p1 = (key0 + 2 * i + 1 < lim) ? ex2_approx(x1) : 0.f;
          pk[i] = pack_bf16x2(p0, p1);
        }
      }
      if (t > 0) {
        ok = mbar_wait(bar(cs.p_empty), (t - 1) & 1, abrt);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
      }
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int blk = u >> 3, uu = u & 7;
        st_shared_v4(p_row + blk * kBox + ((uu ^ (r & 7)) << 4), pk[4 * u], pk[4 * u + 1],
                     pk[4 * u + 2], pk[4 * u + 3]);
      }
      fence_proxy_async_smem();
      mbar_arrive(bar(cs.p_full));
    }
    if (ok) {
      ok = mbar_wait(bar(cs.o_full), 0, abrt);
      ok = __all_sync(0xffffffffu, ok);
    }
    float d2 = 0.f;
    if (ok) {
      tc_fence_after();
      const __nv_bfloat16* dorow =
          a.dO + ((static_cast<size_t>(sq.s0) + min(row, sq.len - 1)) * a.H + h) * kDV;
#pragma unroll 1
      for (int c = 0; c < kDV / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tmem + tl + 2 * kT + 32 * c, o);
        tmem_wait_ld();
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          float f[8];
          bf16x8_to_f32(*reinterpret_cast<const uint4*>(dorow + 32 * c + 8 * g), f);
#pragma unroll
          for (int i = 0; i < 8; ++i) d2 = fmaf(f[i], __uint_as_float(o[8 * g + i]), d2);
        }
      }
      if (row < sq.len) {
        const float lam = a.lambda[h];
        float* dl = a.delta + st_base;
        dl[row] = dl[row] + lam * d2;  // D = dO . O = delta_1 - lam delta_2
        dl[a.Npad + row] = d2;
      } else {
        d2 = 0.f;
      }
    }
    const float ws = warp_sum(-d2);
    if (lane == 0) cs.red[q4] = ws;
    if (bar_and(1, 128, ok) && r == 0)
      a.dl_part[static_cast<size_t>(bh) * a.n_t + qt] = cs.red[0] + cs.red[1] + cs.red[2] + cs.red[3];
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// =============================================================================================
// bwd_dkdq_kernel: one CTA per (key tile j, b, h, map m); key-major over the CTAs, but each
// inner tile is computed query-major: S = Q K^T and dW = dO V^T have the 128 queries on the TMEM
// lanes, so a query's b and delta are per-thread constants. Warps 0 (TMA), 1 (MMA, TMEM),
// 2-9: two warpgroups, thread r = query row r, key columns [64 w, 64 w + 64); 10-13: the dQ
// warpgroup (thread r = query row r, all 128 d-columns), which moves each tile's dQ partial
// through a staging ring of two 32-column boxes and adds it into the fp32 accumulator with TMA
// tensor reductions, off the path of every operand.
// TMEM: S cols 0-127, dK 256-383, and two buffers P0 (128-255) and P1 (384-511): tile t's dW
// goes to P(t & 1), and once the dS warps have read it, tile t's dQ partial overwrites it; so
// dW_{t+1} needs only dQ_{t-1} drained and runs while the dS warps work on tile t.
// Shared memory: K_m,j (32 KB) stays; V_j has one half-slot (32 KB: dv columns [0, 128) or
// [128, 256)), refilled once per inner tile: tile t's dW runs over the half left in the slot
// by tile t - 1 first, then over the other half (so halves alternate 0,1 | 1,0 | 0,1 ...).
// Q_m,i (32 KB + its b and delta rows) and dO_i (64 KB) have one slot each; the dS tile (32 KB,
// [query][key]) is read MN-major as dS^T for dK and K-major for dQ; the dQ staging ring (32 KB).
// MMA issue order per inner tile t: dW_{t+1} over the resident V half | dK_t | dW_{t+1} over the
// other half | dQ_t | S_{t+1}: the first half runs while the dS warps work on tile t, the V
// half-load runs under dK_t, and the next Q load under the second half and dQ_t.
// =============================================================================================
namespace kq {
constexpr int kThreads = 448;  // TMA, MMA, 8 dS warps, 4 dQ warps
constexpr int kKOff = 0;
constexpr int kVOff = kKOff + 2 * kBox;
constexpr int kQOff = kVOff + 2 * kBox;
constexpr int kDOOff = kQOff + 2 * kBox;
constexpr int kDSOff = kDOOff + 4 * kBox;
constexpr int kSTOff = kDSOff + 2 * kBox;   // dQ staging: two boxes of 32 fp32 columns
constexpr int kBDOff = kSTOff + 2 * kBox;   // b[128], delta[128]
constexpr int kCtrlOff = kBDOff + 2 * kT * 4;
struct Ctrl {
  uint64_t k_full, v_full, v_empty, q_full, q_empty, do_full, do_empty, s_full, s_free, ds_full,
      ds_empty, dq_full, dq_free, dk_full, teardown;
  uint32_t tmem_slot;
  int abort_flag;
};
constexpr int kDynSmem = kCtrlOff + static_cast<int>(sizeof(Ctrl));
static_assert(kDynSmem <= 232448, "dK/dQ kernel exceeds 227 KB of shared memory");
// TMEM column of buffer P(t & 1), which holds dW_t and then the dQ partial of tile t
__device__ __forceinline__ uint32_t pbuf(int t) { return static_cast<uint32_t>(kT + 2 * kT * (t & 1)); }
}  // namespace kq

template <bool GR>
__global__ void __launch_bounds__(kq::kThreads, 1)
    bwd_dkdq_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_dqacc, const Args a) {
  using namespace kq;
  extern __shared__ __align__(1024) uint8_t smem[];
  Ctrl& cs = *reinterpret_cast<Ctrl*>(smem + kCtrlOff);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sK = smem_u32(smem + kKOff), sV = smem_u32(smem + kVOff);
  const uint32_t sQ = smem_u32(smem + kQOff), sDO = smem_u32(smem + kDOOff);
  const uint32_t sDS = smem_u32(smem + kDSOff), sST = smem_u32(smem + kSTOff);
  const uint32_t sBD = smem_u32(smem + kBDOff);
  const float* bd = reinterpret_cast<const float*>(smem + kBDOff);
  auto bar = [](uint64_t& x) { return smem_u32(&x); };
  if ((smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) flag_device_error(DEV_TIMEOUT);
    return;
  }

  int unit, j;
  grouped_item(static_cast<int>(blockIdx.x), a.B * a.H * 2, a.n_t, a.grp_dkdq, unit, j);
  const int m = unit & 1, bh = unit >> 1;  // both maps of a head run side by side (shared dO)
  const int b = bh / a.H, h = bh % a.H;
  SeqRows sq;
  const bool seq_ok = seq_rows(a, b, sq);
  const int nts = (sq.len + kT - 1) / kT;  // this sequence's tiles
  if (!seq_ok || j >= nts) {  // (packed) no keys of this sequence in this tile
    if (!seq_ok && j == 0 && m == 0 && threadIdx.x == 0) flag_device_error(DEV_BAD_INDEX);
    return;
  }
  const int i0 = a.causal ? j : 0;
  const int T = nts - i0;  // inner (query) tiles

  if (threadIdx.x == 0) {
    mbar_init(bar(cs.k_full), 1);
    mbar_init(bar(cs.v_full), 1);
    mbar_init(bar(cs.v_empty), 1);
    mbar_init(bar(cs.q_full), 1);
    mbar_init(bar(cs.q_empty), 1);
    mbar_init(bar(cs.do_full), 1);
    mbar_init(bar(cs.do_empty), 1);
    mbar_init(bar(cs.s_full), 1);
    mbar_init(bar(cs.s_free), 256);
    mbar_init(bar(cs.ds_full), 256);
    mbar_init(bar(cs.ds_empty), 1);
    mbar_init(bar(cs.dq_full), 1);
    mbar_init(bar(cs.dq_free), 128);
    mbar_init(bar(cs.dk_full), 1);
    mbar_init(bar(cs.teardown), 1);
    cs.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&cs.tmem_slot), 512);
    tmem_relinquish();
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = cs.tmem_slot;
  volatile int* abrt = &cs.abort_flag;
  const size_t st_base = static_cast<size_t>(b * a.H + h) * 2 * a.Npad + static_cast<size_t>(m) * a.Npad;

  if (warp == 0) {
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      prefetch_tmap(&tm_do);
      // V half-load n carries dv columns [128 (n & 1), +128): load 0 with K, then load t + 1
      // (tile t's second half) once tile t's first half has been read
      auto load_v = [&](int n) {
        mbar_arrive_expect_tx(bar(cs.v_full), 2 * kBox);
        for (int c = 0; c < 2; ++c)
          tma_load_4d_chk(sV + c * kBox, &tm_v, bar(cs.v_full), 128 * (n & 1) + 64 * c, h,
                          sq.trow + j * kT, sq.tb, map_ext(a, kDV, 2));
      };
      mbar_arrive_expect_tx(bar(cs.k_full), 2 * kBox);
      for (int c = 0; c < 2; ++c)
        tma_load_4d_chk(sK + c * kBox, &tm_k, bar(cs.k_full), qk_col<GR>(m) + 64 * c,
                        qk_head<GR>(a, h, m), sq.trow + j * kT, sq.tb, qk_ext<GR>(a, 2));
      load_v(0);
      bool ok = true;
      int nv = 1, ndo = 0, nq = 0;  // loads issued: V halves, dO tiles, Q tiles
      for (int t = 0; t < T && ok; ++t) {
        const int i = i0 + t;
        if (!(ok = mbar_wait(bar(cs.do_empty), (t & 1) ^ 1, abrt))) break;
        ++ndo;
        mbar_arrive_expect_tx(bar(cs.do_full), 4 * kBox);
        for (int c = 0; c < 4; ++c)
          tma_load_4d_chk(sDO + c * kBox, &tm_do, bar(cs.do_full), 64 * c, h, sq.trow + i * kT, sq.tb, map_ext(a, kDV, 2));
        // in the order the MMA issuer frees the slots: tile t's first dW half frees the V slot
        // before dK_{t-1} frees the Q slot
        if (!(ok = mbar_wait(bar(cs.v_empty), (nv & 1) ^ 1, abrt))) break;
        load_v(nv++);
        if (!(ok = mbar_wait(bar(cs.q_empty), (t & 1) ^ 1, abrt))) break;
        ++nq;
        mbar_arrive_expect_tx(bar(cs.q_full), 2 * kBox + 2 * kT * 4);
        for (int c = 0; c < 2; ++c)
          tma_load_4d_chk(sQ + c * kBox, &tm_q, bar(cs.q_full), qk_col<GR>(m) + 64 * c,
                          qk_head<GR>(a, h, m), sq.trow + i * kT, sq.tb, qk_ext<GR>(a, 2));
        const size_t nst = static_cast<size_t>(a.B) * a.H * 2 * a.Npad;
        bulk_load_f32(sBD, a.stats, st_base + static_cast<size_t>(i) * kT, nst, kT, bar(cs.q_full));
        bulk_load_f32(sBD + kT * 4, a.delta, st_base + static_cast<size_t>(i) * kT, nst, kT,
                      bar(cs.q_full));
      }
      // nothing of ours may still be landing at exit
      mbar_wait(bar(cs.k_full), 0, nullptr);
      mbar_wait(bar(cs.v_full), (nv - 1) & 1, nullptr);
      if (ndo > 0) mbar_wait(bar(cs.do_full), (ndo - 1) & 1, nullptr);
      if (nq > 0) mbar_wait(bar(cs.q_full), (nq - 1) & 1, nullptr);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc_kk = umma_idesc_bf16(kT, kT, 0, 0);  // S, dW (queries x keys)
      constexpr uint32_t idesc_dk = umma_idesc_bf16(kT, kD, 1, 1);  // dS^T (MN) x Q (MN)
      constexpr uint32_t idesc_dq = umma_idesc_bf16(kT, kD, 0, 1);  // dS (K-major) x K (MN)
      const uint64_t dK0 = umma_smem_desc(sK, 16, 1024);
      const uint64_t dKmn = umma_smem_desc(sK, kBox, 1024);
      const uint64_t dV0 = umma_smem_desc(sV, 16, 1024);
      const uint64_t dQ0 = umma_smem_desc(sQ, 16, 1024);
      const uint64_t dQmn = umma_smem_desc(sQ, kBox, 1024);
      const uint64_t dDO0 = umma_smem_desc(sDO, 16, 1024);
      const uint64_t dDS0 = umma_smem_desc(sDS, 16, 1024);
      const uint64_t dDSmn = umma_smem_desc(sDS, kBox, 1024);
      int nv = 0;  // V half-loads waited for
      // dW_t goes to TMEM buffer P(t & 1) (columns 128 + 256 (t & 1)), over the V half in the
      // slot (dv columns [128 hf, +128)): 8 K-steps from dO's boxes 2 hf, 2 hf + 1
      auto dw_half = [&](int t, int hf) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * kBox + (kk & 3) * 32;
          mma_bf16_ss(tmem + pbuf(t), desc_add(dDO0, 2 * hf * kBox + off), desc_add(dV0, off),
                      idesc_kk, (hf == (t & 1) && kk == 0) ? 0u : 1u);
        }
      };
      auto wait_v = [&]() -> bool {
        const bool r = mbar_wait(bar(cs.v_full), nv & 1, abrt);
        ++nv;
        tc_fence_after();
        return r;
      };
      // dW_t: first over the V half left in the slot (hf = t & 1), then over the other half once
      // it has loaded. P(t & 1) last held dQ_{t-2}, which the dQ warps must have read.
      auto dw_first = [&](int t) -> bool {
        if (!mbar_wait(bar(cs.do_full), t & 1, abrt)) return false;
        if (t >= 2 && !mbar_wait(bar(cs.dq_free), t & 1, abrt)) return false;
        if (t == 0 && !wait_v()) return false;
        tc_fence_after();
        dw_half(t, t & 1);
        tc_commit(bar(cs.v_empty));  // the slot may take the other half
        return true;
      };
      auto dw_second = [&](int t) -> bool {
        if (!wait_v()) return false;
        dw_half(t, (t & 1) ^ 1);
        tc_commit(bar(cs.do_empty));  // dO_t read: the slot may take dO_{t+1}
        return true;
      };
      // S_t (columns 0-127, free once the dS warps hold S_{t-1}); its commit also covers dW_t
      auto issue_s = [&](int t) -> bool {
        if (t > 0 && !mbar_wait(bar(cs.s_free), (t - 1) & 1, abrt)) return false;
        if (!mbar_wait(bar(cs.q_full), t & 1, abrt)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kBox + (kk & 3) * 32;
          mma_bf16_ss(tmem, desc_add(dQ0, off), desc_add(dK0, off), idesc_kk, kk > 0 ? 1u : 0u);
        }
        tc_commit(bar(cs.s_full));  // S_t and dW_t
        return true;
      };
      bool ok = mbar_wait(bar(cs.k_full), 0, abrt);
      tc_fence_after();
      if (ok && T > 0) ok = dw_first(0) && dw_second(0) && issue_s(0);
      for (int t = 0; ok && t < T; ++t) {
        const bool nxt = t + 1 < T;
        // dW_{t+1}'s first half runs while the dS warps work on tile t; its second half waits
        // for the other V half, whose load runs under dK_t
        if (nxt && !(ok = dw_first(t + 1))) break;
        if (!(ok = mbar_wait(bar(cs.ds_full), t & 1, abrt))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kT / 16; ++kk)  // dK += dS^T Q  (K = queries)
          mma_bf16_ss(tmem + 2 * kT, desc_add(dDSmn, kk * 2048), desc_add(dQmn, kk * 2048),
                      idesc_dk, (t > 0 || kk > 0) ? 1u : 0u);
        tc_commit(bar(cs.q_empty));
        if (nxt && !(ok = dw_second(t + 1))) break;
#pragma unroll
        for (int kk = 0; kk < kT / 16; ++kk)  // dQ partial = dS K into P(t & 1)  (K = keys)
          mma_bf16_ss(tmem + pbuf(t), desc_add(dDS0, (kk >> 2) * kBox + (kk & 3) * 32),
                      desc_add(dKmn, kk * 2048), idesc_dq, kk > 0 ? 1u : 0u);
        tc_commit(bar(cs.dq_full));
        tc_commit(bar(cs.ds_empty));
        if (nxt && !(ok = issue_s(t + 1))) break;
      }
      tc_commit(bar(cs.dk_full));
      tc_commit(bar(cs.teardown));
      mbar_wait(bar(cs.teardown), 0, nullptr);
    }
  } else if (warp < 2 + 8) {
    // ---- dS warpgroups: thread r = query row r of the inner tile, key columns
    // [64 wg, 64 wg + 64); the row's b and delta are per-thread constants ----
    const int wg = (warp - 2) >> 2;
    const int q4 = warp & 3;
    const int r = 32 * q4 + lane;
    const int key = j * kT + r;  // for the dK readout (TMEM lane = key row there)
    const uint32_t tl = static_cast<uint32_t>(32 * q4) << 16;
    const float lam = a.lambda[h];
    const float coef = (m == 0 ? 1.f : -lam) * a.c;
    const uint64_t c2 = f2pack(a.c_log2, a.c_log2), coef2 = f2pack(coef, coef);
    const uint32_t ds_row = sDS + wg * kBox + r * 128;
    bool ok = true;
    for (int t = 0; t < T; ++t) {
      const int i = i0 + t;
      ok = ok && mbar_wait(bar(cs.s_full), t & 1, abrt);
      ok = ok && mbar_wait(bar(cs.q_full), t & 1, abrt);  // b and delta of this tile
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const int qq = i * kT + r;
      const float nb = -bd[r], nd = -bd[kT + r] * coef;
      const uint64_t nb2 = f2pack(nb, nb), nd2 = f2pack(nd, nd);
      // masks only where the tile reaches past N or crosses the diagonal
      const bool edge = (j + 1) * kT > sq.len || (i + 1) * kT > sq.len || (a.causal && i == j);
      uint32_t pk[32];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t sv[32], wv[32];
        tmem_ld32(tmem + tl + 64 * wg + 32 * hh, sv);
        tmem_ld32(tmem + tl + pbuf(t) + 64 * wg + 32 * hh, wv);
        tmem_wait_ld();
        if (hh == 1) {
          tc_fence_before();
          mbar_arrive(bar(cs.s_free));  // S is in registers
        }
        // dS for a pair of keys; the mask is tested outside the unrolled loops (only tiles that
        // reach past N or cross the diagonal take the masked copy)
        auto ds_pair = [&](int e, float& y0, float& y1) {
          float x0, x1;
          f2unpack(f2fma(f2pack(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), c2, nb2), x0, x1);
          const uint64_t g = f2fma(f2pack(__uint_as_float(wv[e]), __uint_as_float(wv[e + 1])), coef2, nd2);
          f2unpack(f2mul(f2pack(ex2_approx(x0), ex2_approx(x1)), g), y0, y1);
        };
        if (!edge) {
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            float y0, y1;
            ds_pair(e, y0, y1);
            pk[16 * hh + (e >> 1)] = pack_bf16x2(y0, y1);
          }
        } else {
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            float y0, y1;
            ds_pair(e, y0, y1);
            const int kk0 = j * kT + 64 * wg + 32 * hh + e;
            const bool v0 = kk0 < sq.len && qq < sq.len && (!a.causal || qq >= kk0);
            const bool v1 = kk0 + 1 < sq.len && qq < sq.len && (!a.causal || qq >= kk0 + 1);
            pk[16 * hh + (e >> 1)] = pack_bf16x2(v0 ? y0 : 0.f, v1 ? y1 : 0.f);
          }
        }
      }
      if (t > 0) {
        ok = mbar_wait(bar(cs.ds_empty), (t - 1) & 1, abrt);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u)
        st_shared_v4(ds_row + ((u ^ (r & 7)) << 4), pk[4 * u], pk[4 * u + 1], pk[4 * u + 2],
                     pk[4 * u + 3]);
      fence_proxy_async_smem();
      tc_fence_before();  // dW_t has been read: dQ_t may overwrite P(t & 1)
      mbar_arrive(bar(cs.ds_full));
    }
    if (ok) {
      ok = mbar_wait(bar(cs.dk_full), 0, abrt);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok) {
      tc_fence_after();
      uint32_t o[2][32];
      tmem_ld32(tmem + tl + 2 * kT + 64 * wg, o[0]);
      tmem_ld32(tmem + tl + 2 * kT + 64 * wg + 32, o[1]);
      tmem_wait_ld();
      if (GR && m == 1 && key < sq.len) {
        // grouped, map 2: this signal head's share of its noise head's dK2, added in fp32
        float* dst = a.dkacc +
                     ((static_cast<size_t>(sq.s0) + key) * (a.hqk - a.H) + h / a.group) * kD +
                     64 * wg;
        if (dbg_index_ok(static_cast<long long>((static_cast<size_t>(sq.s0) + key) *
                                                    (a.hqk - a.H) + h / a.group),
                         (a.cu ? 1LL * a.total : 1LL * a.B * a.N) * (a.hqk - a.H))) {
#pragma unroll
          for (int hh = 0; hh < 2; ++hh)
#pragma unroll
            for (int g = 0; g < 8; ++g)
              red_add_v4(dst + 32 * hh + 4 * g, __uint_as_float(o[hh][4 * g]),
                         __uint_as_float(o[hh][4 * g + 1]), __uint_as_float(o[hh][4 * g + 2]),
                         __uint_as_float(o[hh][4 * g + 3]));
        }
      } else if (key < sq.len) {
        __nv_bfloat16* dst = a.dk + ((static_cast<size_t>(sq.s0) + key) * (GR ? a.hqk : a.H) +
                                     qk_head<GR>(a, h, m)) * (GR ? kD : 2 * kD) +
                             qk_col<GR>(m) + 64 * wg;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            uint4 pkt;
            pkt.x = pack_bf16x2(__uint_as_float(o[hh][8 * g]), __uint_as_float(o[hh][8 * g + 1]));
            pkt.y = pack_bf16x2(__uint_as_float(o[hh][8 * g + 2]), __uint_as_float(o[hh][8 * g + 3]));
            pkt.z = pack_bf16x2(__uint_as_float(o[hh][8 * g + 4]), __uint_as_float(o[hh][8 * g + 5]));
            pkt.w = pack_bf16x2(__uint_as_float(o[hh][8 * g + 6]), __uint_as_float(o[hh][8 * g + 7]));
            *reinterpret_cast<uint4*>(dst + 32 * hh + 8 * g) = pkt;
          }
      }
    }
  } else {
    // ---- dQ warpgroup: thread r = query row r of the inner tile. Each tile's dQ partial
    // (TMEM buffer P(t & 1)) is read two 32-column boxes at a time into registers, so the buffer
    // is free for dW_{t+2} after two loads; each pair goes into a staging ring of two 128B-swizzled
    // boxes and is added into the fp32 accumulator by TMA tensor reductions. Thread 0 issues the
    // reductions and waits until they have read the ring before it is restaged. ----
    const int q4 = warp & 3;
    const int r = 32 * q4 + lane;
    const uint32_t tl = static_cast<uint32_t>(32 * q4) << 16;
    const Ext4 eacc = qk_ext<GR>(a, 4);
    const int qh = qk_head<GR>(a, h, m), qc = qk_col<GR>(m);
    bool ok = true;
    for (int t = 0; t < T; ++t) {
      bool g = ok && mbar_wait(bar(cs.dq_full), t & 1, abrt);
      g = __all_sync(0xffffffffu, g);
      if (!(ok = bar_and(2, 128, g))) break;
      tc_fence_after();
      const int i = i0 + t;
#pragma unroll 1
      for (int pr = 0; pr < 2; ++pr) {
        uint32_t o[2][32];
        tmem_ld32(tmem + tl + pbuf(t) + 64 * pr, o[0]);
        tmem_ld32(tmem + tl + pbuf(t) + 64 * pr + 32, o[1]);
        tmem_wait_ld();
        if (pr == 1) {
          tc_fence_before();
          mbar_arrive(bar(cs.dq_free));
          // the ring: thread 0 waits for the first pair's reductions to have read it
          if (r == 0) bulk_wait_read();
          named_barrier_sync(2, 128);
        }
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          const uint32_t row = sST + x * kBox + r * 128;
#pragma unroll
          for (int u = 0; u < 8; ++u)
            st_shared_v4(row + ((u ^ (r & 7)) << 4), o[x][4 * u], o[x][4 * u + 1], o[x][4 * u + 2],
                         o[x][4 * u + 3]);
        }
        fence_proxy_async_smem();
        named_barrier_sync(2, 128);
        if (r == 0) {
          for (int x = 0; x < 2; ++x) {
            const int c = 2 * pr + x;
            if (!kDebugChecks ||
                (dbg_index_ok(sq.trow + i * kT, eacc.z) && dbg_index_ok(sq.tb, eacc.w) &&
                 dbg_index_ok(qh, eacc.y) && dbg_index_ok(qc + 32 * c, eacc.x)))
              tma_reduce_add_4d(&tm_dqacc, sST + x * kBox, qc + 32 * c, qh, sq.trow + i * kT,
                                sq.tb);
          }
          bulk_commit();
          // before the next tile restages the ring (ordered by the barrier that opens it)
          if (pr == 1) bulk_wait_read();
        }
      }
    }
    if (r == 0) bulk_wait_all();
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// =============================================================================================
// bwd_dv_kernel: one CTA per (key tile j, b, h); key-major over the CTAs, each inner tile
// query-major like the dK/dQ kernel. Warps 0 (TMA), 1 (MMA, TMEM), 2-9: two warpgroups, thread
// r = query row r, key columns [64 wg, 64 wg + 64).
// TMEM: S1 cols 0-127, S2 128-255, dV 256-511. Shared memory: K1_j, K2_j (64 KB) stay;
// Q1_i | Q2_i (64 KB, with b1, b2) and dO_i (64 KB) one slot each; the W tile ([query][key],
// 32 KB), read MN-major as W^T for dV.
// MMA order per inner tile: S_{t+1} (as soon as the Q slot refills) before dV_t.
// Loads: each map's half of the Q slot has its own barriers, so Q1 of tile t + 1 loads as soon as
// S1_t is done (while S2_t and dV_{t-1} run), and the producer issues tile t + 1's Q before tile
// t's dO (which waits for dV_{t-1}): each Q load has about 2200 cycles of lead instead of 1400.
// =============================================================================================
namespace vv {
constexpr int kThreads = 320;
constexpr int kKOff = 0;                    // K1 (2 boxes) then K2 (2 boxes)
constexpr int kQOff = kKOff + 4 * kBox;     // Q1 then Q2
constexpr int kDOOff = kQOff + 4 * kBox;
constexpr int kWOff = kDOOff + 4 * kBox;
constexpr int kBOff = kWOff + 2 * kBox;     // two buffers of b1[128], b2[128]
constexpr int kCtrlOff = kBOff + 2 * 2 * kT * 4;
struct Ctrl {
  uint64_t kv_full, q_full[2], q_empty[2], do_full, do_empty, s_full, s_free, w_full, w_empty,
      dv_full, teardown, b_full[2], b_empty[2];
  uint32_t tmem_slot;
  int abort_flag;
};
constexpr int kDynSmem = kCtrlOff + static_cast<int>(sizeof(Ctrl));
}  // namespace vv

template <bool GR>
__global__ void __launch_bounds__(vv::kThreads, 1)
    bwd_dv_kernel(const __grid_constant__ CUtensorMap tm_q,
                  const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_do, const Args a) {
  using namespace vv;
  extern __shared__ __align__(1024) uint8_t smem[];
  Ctrl& cs = *reinterpret_cast<Ctrl*>(smem + kCtrlOff);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t sK = smem_u32(smem + kKOff), sQ = smem_u32(smem + kQOff);
  const uint32_t sDO = smem_u32(smem + kDOOff), sW = smem_u32(smem + kWOff);
  const uint32_t sB = smem_u32(smem + kBOff);
  const float* bbase = reinterpret_cast<const float*>(smem + kBOff);
  auto bar = [](uint64_t& x) { return smem_u32(&x); };
  if ((smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) flag_device_error(DEV_TIMEOUT);
    return;
  }

  int bh, j;
  grouped_item(static_cast<int>(blockIdx.x), a.B * a.H, a.n_t, a.grp_dv, bh, j);
  const int b = bh / a.H, h = bh % a.H;
  SeqRows sq;
  const bool seq_ok = seq_rows(a, b, sq);
  const int nts = (sq.len + kT - 1) / kT;  // this sequence's tiles
  if (!seq_ok || j >= nts) {  // (packed) no keys of this sequence in this tile
    if (!seq_ok && j == 0 && threadIdx.x == 0) flag_device_error(DEV_BAD_INDEX);
    return;
  }
  const int i0 = a.causal ? j : 0;
  const int T = nts - i0;

  if (threadIdx.x == 0) {
    mbar_init(bar(cs.kv_full), 1);
    for (int mp = 0; mp < 2; ++mp) {
      mbar_init(bar(cs.q_full[mp]), 1);
      mbar_init(bar(cs.q_empty[mp]), 1);
    }
    mbar_init(bar(cs.do_full), 1);
    mbar_init(bar(cs.do_empty), 1);
    mbar_init(bar(cs.s_full), 1);
    mbar_init(bar(cs.s_free), 256);
    mbar_init(bar(cs.w_full), 256);
    mbar_init(bar(cs.w_empty), 1);
    mbar_init(bar(cs.dv_full), 1);
    mbar_init(bar(cs.teardown), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(cs.b_full[i]), 1);
      mbar_init(bar(cs.b_empty[i]), 256);
    }
    cs.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&cs.tmem_slot), 512);
    tmem_relinquish();
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = cs.tmem_slot;
  volatile int* abrt = &cs.abort_flag;
  const size_t st_base = static_cast<size_t>(b * a.H + h) * 2 * a.Npad;

  if (warp == 0) {
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_do);
      mbar_arrive_expect_tx(bar(cs.kv_full), 4 * kBox);
      for (int c = 0; c < 4; ++c)
        tma_load_4d_chk(sK + c * kBox, &tm_k, bar(cs.kv_full), qk_col<GR>(c >> 1) + 64 * (c & 1),
                        qk_head<GR>(a, h, c >> 1), sq.trow + j * kT, sq.tb, qk_ext<GR>(a, 2));
      // Q of inner tile t: map mp's half once S_mp of tile t - 1 has read it; b1, b2 (the
      // softmax's row statistics) into buffer t & 1 once the softmax has read tile t - 2's, on a
      // barrier of that buffer's own (the Q barriers run up to two tiles ahead of the softmax,
      // which a parity wait could not tell apart)
      int nq[2] = {0, 0}, nd = 0, nb = 0;  // Q halves, dO tiles and statistics issued
      auto load_q = [&](int t) -> bool {
        const int i = i0 + t;
        for (int mp = 0; mp < 2; ++mp) {
          if (!mbar_wait(bar(cs.q_empty[mp]), (t & 1) ^ 1, abrt)) return false;
          mbar_arrive_expect_tx(bar(cs.q_full[mp]), 2 * kBox);
          for (int c = 0; c < 2; ++c)
            tma_load_4d_chk(sQ + (2 * mp + c) * kBox, &tm_q, bar(cs.q_full[mp]),
                            qk_col<GR>(mp) + 64 * c, qk_head<GR>(a, h, mp), sq.trow + i * kT,
                            sq.tb, qk_ext<GR>(a, 2));
          ++nq[mp];
        }
        if (!mbar_wait(bar(cs.b_empty[t & 1]), ((t >> 1) & 1) ^ 1, abrt)) return false;
        mbar_arrive_expect_tx(bar(cs.b_full[t & 1]), 2 * kT * 4);
        const uint32_t sb = sB + (t & 1) * 2 * kT * 4;
        const size_t nst = static_cast<size_t>(a.B) * a.H * 2 * a.Npad;
        bulk_load_f32(sb, a.stats, st_base + static_cast<size_t>(i) * kT, nst, kT,
                      bar(cs.b_full[t & 1]));
        bulk_load_f32(sb + kT * 4, a.stats, st_base + a.Npad + static_cast<size_t>(i) * kT, nst, kT,
                      bar(cs.b_full[t & 1]));
        ++nb;
        return true;
      };
      bool ok = T > 0 && load_q(0);
      for (int t = 0; t < T && ok; ++t) {
        // tile t + 1's Q first: its slots free up before tile t's dO slot does
        if (t + 1 < T && !(ok = load_q(t + 1))) break;
        if (!(ok = mbar_wait(bar(cs.do_empty), (t & 1) ^ 1, abrt))) break;
        mbar_arrive_expect_tx(bar(cs.do_full), 4 * kBox);
        for (int c = 0; c < 4; ++c)
          tma_load_4d_chk(sDO + c * kBox, &tm_do, bar(cs.do_full), 64 * c, h,
                          sq.trow + (i0 + t) * kT, sq.tb, map_ext(a, kDV, 2));
        ++nd;
      }
      // nothing of ours may still be landing at exit: wait for each barrier's last armed phase
      mbar_wait(bar(cs.kv_full), 0, nullptr);
      for (int mp = 0; mp < 2; ++mp)
        if (nq[mp] > 0) mbar_wait(bar(cs.q_full[mp]), (nq[mp] - 1) & 1, nullptr);
      if (nd > 0) mbar_wait(bar(cs.do_full), (nd - 1) & 1, nullptr);
      for (int k = max(0, nb - 2); k < nb; ++k)
        mbar_wait(bar(cs.b_full[k & 1]), (k >> 1) & 1, nullptr);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc_s = umma_idesc_bf16(kT, kT, 0, 0);   // S_m = Q_m K_m^T
      constexpr uint32_t idesc_v = umma_idesc_bf16(kT, kDV, 1, 1);  // W^T (MN) x dO (MN)
      const uint64_t dK0 = umma_smem_desc(sK, 16, 1024);
      const uint64_t dQ0 = umma_smem_desc(sQ, 16, 1024);
      const uint64_t dDOmn = umma_smem_desc(sDO, kBox, 1024);
      const uint64_t dWmn = umma_smem_desc(sW, kBox, 1024);
      auto issue_s = [&](int t) -> bool {
        if (t > 0 && !mbar_wait(bar(cs.s_free), (t - 1) & 1, abrt)) return false;
#pragma unroll
        for (int mp = 0; mp < 2; ++mp) {
          if (!mbar_wait(bar(cs.q_full[mp]), t & 1, abrt)) return false;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk) {
            const uint32_t off = mp * 2 * kBox + (kk >> 2) * kBox + (kk & 3) * 32;
            mma_bf16_ss(tmem + mp * kT, desc_add(dQ0, off), desc_add(dK0, off), idesc_s,
                        kk > 0 ? 1u : 0u);
          }
          tc_commit(bar(cs.q_empty[mp]));  // this map's half of the slot may take the next tile
        }
        tc_commit(bar(cs.s_full));
        return true;
      };
      bool ok = mbar_wait(bar(cs.kv_full), 0, abrt);
      tc_fence_after();
      if (ok && T > 0) ok = issue_s(0);
      for (int t = 0; ok && t < T; ++t) {
        if (t + 1 < T && !(ok = issue_s(t + 1))) break;
        if (!(ok = mbar_wait(bar(cs.w_full), t & 1, abrt))) break;
        if (!(ok = mbar_wait(bar(cs.do_full), t & 1, abrt))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kT / 16; ++kk)  // dV += W^T dO  (K = queries)
          mma_bf16_ss(tmem + 2 * kT, desc_add(dWmn, kk * 2048), desc_add(dDOmn, kk * 2048),
                      idesc_v, (t > 0 || kk > 0) ? 1u : 0u);
        tc_commit(bar(cs.w_empty));
        tc_commit(bar(cs.do_empty));
      }
      tc_commit(bar(cs.dv_full));
      tc_commit(bar(cs.teardown));
      mbar_wait(bar(cs.teardown), 0, nullptr);
    }
  } else {
    // thread r = query row r of the inner tile (key columns [64 wg, 64 wg + 64)): the row's b1
    // and b2 are per-thread constants; for the dV readout, TMEM lane r = key row r
    const int wg = (warp - 2) >> 2;
    const int q4 = warp & 3;
    const int r = 32 * q4 + lane;
    const int key = j * kT + r;
    const uint32_t tl = static_cast<uint32_t>(32 * q4) << 16;
    const float lam = a.lambda[h];
    const uint64_t c2 = f2pack(a.c_log2, a.c_log2), nlam2 = f2pack(-lam, -lam);
    const uint32_t w_row = sW + wg * kBox + r * 128;
    bool ok = true;
    for (int t = 0; t < T; ++t) {
      const int i = i0 + t;
      ok = ok && mbar_wait(bar(cs.s_full), t & 1, abrt);
      ok = ok && mbar_wait(bar(cs.b_full[t & 1]), (t >> 1) & 1, abrt);  // b1, b2 of this tile
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const float* bb = bbase + (t & 1) * 2 * kT;
      const float nb1 = -bb[r], nb2 = -bb[kT + r];
      mbar_arrive(bar(cs.b_empty[t & 1]));  // this buffer of b1, b2 may be refilled (tile t + 2)
      const uint64_t nb1_2 = f2pack(nb1, nb1), nb2_2 = f2pack(nb2, nb2);
      const int qq = i * kT + r;
      const bool edge = (j + 1) * kT > sq.len || (i + 1) * kT > sq.len || (a.causal && i == j);
      uint32_t pk[32];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t s1[32], s2[32];
        tmem_ld32(tmem + tl + 64 * wg + 32 * hh, s1);
        tmem_ld32(tmem + tl + kT + 64 * wg + 32 * hh, s2);
        tmem_wait_ld();
        if (hh == 1) {
          tc_fence_before();
          mbar_arrive(bar(cs.s_free));  // both score tiles are in registers
        }
        // W for a pair of keys; the mask is tested outside the unrolled loops (only tiles that
        // reach past N or cross the diagonal take the masked copy)
        auto w_pair = [&](int e, float& w0, float& w1) {
          float x0, x1, y0, y1;
          f2unpack(f2fma(f2pack(__uint_as_float(s1[e]), __uint_as_float(s1[e + 1])), c2, nb1_2), x0, x1);
          f2unpack(f2fma(f2pack(__uint_as_float(s2[e]), __uint_as_float(s2[e + 1])), c2, nb2_2), y0, y1);
          f2unpack(f2fma(f2pack(ex2_approx(y0), ex2_approx(y1)), nlam2,
                         f2pack(ex2_approx(x0), ex2_approx(x1))),
                   w0, w1);
        };
        if (!edge) {
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            float w0, w1;
            w_pair(e, w0, w1);
            pk[16 * hh + (e >> 1)] = pack_bf16x2(w0, w1);
          }
        } else {
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            float w0, w1;
            w_pair(e, w0, w1);
            const int kk0 = j * kT + 64 * wg + 32 * hh + e;
            const bool v0 = kk0 < sq.len && qq < sq.len && (!a.causal || qq >= kk0);
            const bool v1 = kk0 + 1 < sq.len && qq < sq.len && (!a.causal || qq >= kk0 + 1);
            pk[16 * hh + (e >> 1)] = pack_bf16x2(v0 ? w0 : 0.f, v1 ? w1 : 0.f);
          }
        }
      }
      if (t > 0) {
        ok = mbar_wait(bar(cs.w_empty), (t - 1) & 1, abrt);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u)
        st_shared_v4(w_row + ((u ^ (r & 7)) << 4), pk[4 * u], pk[4 * u + 1], pk[4 * u + 2],
                     pk[4 * u + 3]);
      fence_proxy_async_smem();
      mbar_arrive(bar(cs.w_full));
    }
    if (ok) {
      ok = mbar_wait(bar(cs.dv_full), 0, abrt);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok) {
      tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t o[32];
        tmem_ld32(tmem + tl + 2 * kT + 128 * wg + 32 * c, o);
        tmem_wait_ld();
        if (key < sq.len) {
          __nv_bfloat16* dst = a.dv + ((static_cast<size_t>(sq.s0) + key) * a.H + h) * kDV +
                               128 * wg + 32 * c;
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            uint4 pkt;
            pkt.x = pack_bf16x2(__uint_as_float(o[8 * g]), __uint_as_float(o[8 * g + 1]));
            pkt.y = pack_bf16x2(__uint_as_float(o[8 * g + 2]), __uint_as_float(o[8 * g + 3]));
            pkt.z = pack_bf16x2(__uint_as_float(o[8 * g + 4]), __uint_as_float(o[8 * g + 5]));
            pkt.w = pack_bf16x2(__uint_as_float(o[8 * g + 6]), __uint_as_float(o[8 * g + 7]));
            *reinterpret_cast<uint4*>(dst + 8 * g) = pkt;
          }
        }
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// =============================================================================================
// bwd_finish_kernel: blocks [0, nq) convert dQ (two 8-element groups per thread and step, both
// groups' loads issued first); block nq sums dlam; blocks nq + 1 .. nq + 8 sum the norm-weight
// partials, 32 channels each: warp w adds partials w, w + 8, ... (lane = channel), then the eight
// warp sums are added in warp order. Every sum has a fixed order: the result is deterministic.
// =============================================================================================
constexpr int kFinishSumBlocks = kDV / 32;

// Grouped form: the noise heads' dK (fp32 sums over each group's signal heads) to bf16 at heads
// Hs .. Hs + Hn - 1 of dk [tokens, Hs + Hn, d]; one thread per 8 channels.
__global__ void __launch_bounds__(256) bwd_gda_dk_kernel(const Args a, long long tokens) {
  // packed: rows past the last sequence belong to none and are not written
  if (a.cu) tokens = min(tokens, static_cast<long long>(min(max(a.cu[a.B], 0), a.total)));
  const int hn = a.hqk - a.H;
  const long long n8 = tokens * hn * (kD / 8);
  for (long long e = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; e < n8;
       e += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long row = e / (kD / 8);             // token * Hn + g
    const int c8 = static_cast<int>(e % (kD / 8));
    const long long t = row / hn;
    const int g = static_cast<int>(row % hn);
    const float4 x = reinterpret_cast<const float4*>(a.dkacc)[2 * e];
    const float4 y = reinterpret_cast<const float4*>(a.dkacc)[2 * e + 1];
    uint4 pk;
    pk.x = pack_bf16x2(x.x, x.y);
    pk.y = pack_bf16x2(x.z, x.w);
    pk.z = pack_bf16x2(y.x, y.y);
    pk.w = pack_bf16x2(y.z, y.w);
    reinterpret_cast<uint4*>(a.dk + (static_cast<size_t>(t) * a.hqk + a.H + g) * kD)[c8] = pk;
  }
}

__global__ void __launch_bounds__(256) bwd_finish_kernel(const Args a, long long n8, int nq) {
  if (static_cast<int>(blockIdx.x) < nq) {
    // packed: rows past the last sequence belong to none and are not written
    if (a.cu)
      n8 = min(n8, static_cast<long long>(min(max(a.cu[a.B], 0), a.total)) *
                       (a.group ? a.hqk * kD : a.H * 2 * kD) / 8);
    const long long stride = static_cast<long long>(nq) * 256;
    const float4* src = reinterpret_cast<const float4*>(a.dqacc);
    for (long long e = static_cast<long long>(blockIdx.x) * 256 + threadIdx.x; e < n8;
         e += 2 * stride) {
      const long long e2 = e + stride;
      const bool two = e2 < n8;
      const float4 x = src[2 * e], y = src[2 * e + 1];
      float4 x2 = x, y2 = y;
      if (two) {
        x2 = src[2 * e2];
        y2 = src[2 * e2 + 1];
      }
      uint4 pk;
      pk.x = pack_bf16x2(x.x, x.y);
      pk.y = pack_bf16x2(x.z, x.w);
      pk.z = pack_bf16x2(y.x, y.y);
      pk.w = pack_bf16x2(y.z, y.w);
      reinterpret_cast<uint4*>(a.dq)[e] = pk;
      if (two) {
        pk.x = pack_bf16x2(x2.x, x2.y);
        pk.y = pack_bf16x2(x2.z, x2.w);
        pk.z = pack_bf16x2(y2.x, y2.y);
        pk.w = pack_bf16x2(y2.z, y2.w);
        reinterpret_cast<uint4*>(a.dq)[e2] = pk;
      }
    }
    return;
  }
  if (static_cast<int>(blockIdx.x) == nq) {
    for (int h = threadIdx.x; h < a.H; h += blockDim.x) {
      float s = 0.f;
      for (int b = 0; b < a.B; ++b)
        for (int t = 0; t < a.n_t; ++t) s += a.dl_part[(static_cast<size_t>(b) * a.H + h) * a.n_t + t];
      a.dlambda[h] = s;
    }
    return;
  }
  if (!a.dnorm_w) return;
  __shared__ float part[8][32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = (static_cast<int>(blockIdx.x) - nq - 1) * 32 + lane;
  float s = 0.f;
  for (int k = warp; k < a.pre_blocks; k += 8) s += a.dw_part[static_cast<size_t>(k) * kDV + c];
  part[warp][lane] = s;
  __syncthreads();
  if (warp == 0) {
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) t += part[w][lane];
    a.dnorm_w[c] = a.norm ? t : 0.f;
  }
}

// ---------------------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------------------
// 4-D bf16 map over [B, N, H, cols], box 64 x 1 x rows x 1, 128-byte swizzle, zero fill.
static bool make_map(CUtensorMap* m, const void* base, int cols, int H, int N, int B, int rows,
                     char* err, size_t err_len) {
  cuuint64_t dims[4] = {(cuuint64_t)cols, (cuuint64_t)H, (cuuint64_t)N, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)cols * 2, (cuuint64_t)cols * H * 2,
                           (cuuint64_t)cols * H * 2 * (cuuint64_t)N};
  cuuint32_t box[4] = {64, 1, (cuuint32_t)rows, 1};
  return encode_tmap_4d(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, dims, strides, box, err, err_len);
}

// 4-D fp32 map over the dQ accumulator [B, N, H, 2d], box 32 x 1 x 128 x 1 (128-byte rows),
// 128-byte swizzle: the target of the dK/dQ kernel's tensor reductions.
static bool make_map_f32(CUtensorMap* m, void* base, int cols, int H, int N, int B, char* err,
                         size_t err_len) {
  cuuint64_t dims[4] = {(cuuint64_t)cols, (cuuint64_t)H, (cuuint64_t)N, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)cols * 4, (cuuint64_t)cols * H * 4,
                           (cuuint64_t)cols * H * 4 * (cuuint64_t)N};
  cuuint32_t box[4] = {32, 1, (cuuint32_t)kT, 1};
  return encode_tmap_4d(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, base, dims, strides, box, err, err_len);
}

static size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct WsLayout {
  size_t dO, delta, dqacc, dw_part, dl_part, dkacc, total;
  int pre_blocks;
};
// tokens: B N (batched) or the packed length; grouped: plus the noise heads' dK accumulator
// (sized for tokens x H rows of d floats, H the signal heads: Hn <= H)
static WsLayout ws_layout(int B, int N, int H, long long tokens, bool grouped = false) {
  WsLayout w;
  const int Npad = (N + kT - 1) / kT * kT;
  const int n_t = Npad / kT;
  const long long rows = tokens * H;
  long long blocks = (rows + kPreWarps - 1) / kPreWarps;
  w.pre_blocks = static_cast<int>(blocks < 8 * 152 ? blocks : 8 * 152);
  size_t off = 0;
  w.dO = off;
  off = align256(off + static_cast<size_t>(rows) * kDV * 2);
  w.delta = off;
  off = align256(off + static_cast<size_t>(B) * H * 2 * Npad * 4);
  w.dqacc = off;
  off = align256(off + static_cast<size_t>(rows) * 2 * kD * 4);
  w.dw_part = off;
  off = align256(off + static_cast<size_t>(w.pre_blocks) * kDV * 4);
  w.dl_part = off;
  off = align256(off + static_cast<size_t>(B) * H * n_t * 4);
  w.dkacc = off;
  if (grouped) off = align256(off + static_cast<size_t>(rows) * kD * 4);
  w.total = off;
  return w;
}

}  // namespace bwd

size_t backward_workspace_bytes(int B, int N, int H, long long rows, bool grouped) {
  return bwd::ws_layout(B, N, H, rows, grouped).total;
}

cudaError_t status_backward(int* v) { return read_clear_status(v); }

cudaError_t launch_backward(const BackwardArgs& x, cudaStream_t st, char* err, size_t err_len) {
  using namespace bwd;
  const bool packed = x.cu_seqlens != nullptr;
  const long long tokens = packed ? x.total : static_cast<long long>(x.B) * x.N;
  const bool grouped = x.n_noise > 0;
  const WsLayout L = ws_layout(x.B, x.N, x.H, tokens, grouped);
  uint8_t* ws = static_cast<uint8_t*>(x.workspace);
  Args a{};
  a.q = static_cast<const __nv_bfloat16*>(x.q);
  a.k = static_cast<const __nv_bfloat16*>(x.k);
  a.v = static_cast<const __nv_bfloat16*>(x.v);
  a.o_pre = static_cast<const __nv_bfloat16*>(x.o_pre);
  a.dy = static_cast<const __nv_bfloat16*>(x.dout);
  a.stats = x.stats;
  a.lambda = x.lambda;
  a.norm_w = x.norm_w;
  a.dq = static_cast<__nv_bfloat16*>(x.dq);
  a.dk = static_cast<__nv_bfloat16*>(x.dk);
  a.dv = static_cast<__nv_bfloat16*>(x.dv);
  a.dlambda = x.dlambda;
  a.dnorm_w = x.dnorm_w;
  a.dO = reinterpret_cast<__nv_bfloat16*>(ws + L.dO);
  a.delta = reinterpret_cast<float*>(ws + L.delta);
  a.dqacc = reinterpret_cast<float*>(ws + L.dqacc);
  a.dw_part = reinterpret_cast<float*>(ws + L.dw_part);
  a.dl_part = reinterpret_cast<float*>(ws + L.dl_part);
  a.B = x.B;
  a.N = x.N;
  a.H = x.H;
  a.Npad = (x.N + kT - 1) / kT * kT;
  a.n_t = a.Npad / kT;
  a.pre_blocks = L.pre_blocks;
  a.eps = x.eps;
  a.scale_out = (x.flags & 4) ? (1.f - x.lambda_init) : 1.f;
  a.norm = (x.flags & 2) != 0;
  a.causal = (x.flags & 1) != 0;
  a.c = 1.f / sqrtf(static_cast<float>(kD));
  a.c_log2 = kLog2e * a.c;
  a.cu = x.cu_seqlens;
  a.total = x.total;
  a.group = grouped ? x.H / x.n_noise : 0;
  a.hqk = grouped ? x.H + x.n_noise : x.H;
  a.dkacc = grouped ? reinterpret_cast<float*>(ws + L.dkacc) : nullptr;
  {
    // bytes each unit keeps re-reading (or, for dQ, accumulating) while its tiles run; a group
    // keeps about 24 MB of them in the 126 MB L2 (swept at the 3B-layer size over 12-96 MB:
    // 24 MB was fastest, 0.8 % ahead of 48 MB, and 96 MB 1.2 % behind it)
    const double n = static_cast<double>(x.N);
    auto grp = [&](double unit_bytes, int n_units) {
      long long g = static_cast<long long>(24.0 * 1024 * 1024 / (unit_bytes > 1 ? unit_bytes : 1));
      return static_cast<int>(g < 1 ? 1 : (g > n_units ? n_units : g));
    };
    a.grp_delta = grp(n * (kD + kDV) * 2, x.B * x.H);                 // K2, V
    a.grp_dkdq = 2 * grp(2 * n * (kD * 2 + kDV * 2 + kD * 4), x.B * x.H);  // Q_m, dO, dQ_m; x2 maps
    a.grp_dv = grp(n * (2 * kD + kDV) * 2, x.B * x.H);               // Q1|Q2, dO
    if (a.grp_dkdq > 2 * x.B * x.H) a.grp_dkdq = 2 * x.B * x.H;
  }

  // packed: the token axis as one batch row of `total`
  const int mN = packed ? x.total : x.N, mB = packed ? 1 : x.B;
  CUtensorMap mq, mk, mv, mvh, mdo, mdq;
  // q, k (and the dQ accumulator): [Q1 | Q2] per head, or (grouped) d-wide heads Hs + Hn
  const int qk_cols = grouped ? kD : 2 * kD;
  if (!make_map_f32(&mdq, a.dqacc, qk_cols, a.hqk, mN, mB, err, err_len) ||
      !make_map(&mq, x.q, qk_cols, a.hqk, mN, mB, kT, err, err_len) ||
      !make_map(&mk, x.k, qk_cols, a.hqk, mN, mB, kT, err, err_len) ||
      !make_map(&mv, x.v, kDV, x.H, mN, mB, kT, err, err_len) ||
      !make_map(&mvh, x.v, kDV, x.H, mN, mB, kT / 2, err, err_len) ||
      !make_map(&mdo, a.dO, kDV, x.H, mN, mB, kT, err, err_len))
    return cudaErrorInvalidValue;

  bwd_pre_kernel<<<L.pre_blocks, kPreWarps * 32, 0, st>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  const int items = a.n_t * x.B * x.H;
  auto delta_k = grouped ? bwd_delta_kernel<true> : bwd_delta_kernel<false>;
  auto dkdq_k = grouped ? bwd_dkdq_kernel<true> : bwd_dkdq_kernel<false>;
  auto dv_k = grouped ? bwd_dv_kernel<true> : bwd_dv_kernel<false>;
  e = cudaFuncSetAttribute(delta_k, cudaFuncAttributeMaxDynamicSharedMemorySize, dl::kDynSmem);
  if (e != cudaSuccess) return e;
  delta_k<<<items, dl::kThreads, dl::kDynSmem, st>>>(mq, mk, mvh, a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  e = cudaFuncSetAttribute(dkdq_k, cudaFuncAttributeMaxDynamicSharedMemorySize, kq::kDynSmem);
  if (e != cudaSuccess) return e;
  dkdq_k<<<2 * items, kq::kThreads, kq::kDynSmem, st>>>(mq, mk, mv, mdo, mdq, a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  e = cudaFuncSetAttribute(dv_k, cudaFuncAttributeMaxDynamicSharedMemorySize, vv::kDynSmem);
  if (e != cudaSuccess) return e;
  dv_k<<<items, vv::kThreads, vv::kDynSmem, st>>>(mq, mk, mdo, a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  if (grouped) {  // the noise heads' dK from their fp32 sums
    bwd_gda_dk_kernel<<<8 * 152, 256, 0, st>>>(a, tokens);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }

  const long long n8 = tokens * a.hqk * qk_cols / 8;
  long long nq = (n8 + 255) / 256;
  if (nq > 8 * 152) nq = 8 * 152;  // eight 256-thread blocks per SM: a full SM of threads
  bwd_finish_kernel<<<static_cast<int>(nq) + 1 + kFinishSumBlocks, 256, 0, st>>>(
      a, n8, static_cast<int>(nq));
  return cudaGetLastError();
}

}  // namespace da
