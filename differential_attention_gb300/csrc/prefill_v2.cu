// prefill_v2.cu -- DIFF V2 pair prefill on the sm_103a tensor cores, both heads of a pair in one
// CTA.
//
// Operator (page "Differential Transformer: softmax can't say zero, so it subtracts", section
// "DIFF V2: what the authors changed"; page "Differential Transformer V2"): query heads 2p and
// 2p+1 of one GQA group attend over their shared K/V head with plain softmax attention each, and
// out[p] = attn[2p] - sigmoid(lam[t, p]) * attn[2p+1], with no per-head norm. Each head is a stock
// attention (the pages run it as two flash-attention calls), so each map's probabilities are
// rounded to bf16 before the product with V, as there; the subtraction is taken in fp32 from the
// two normalised head outputs.
//
// Design. One CTA owns one 128-row query tile of one pair (b, p). Tensor memory holds all four
// accumulators of the pair: S_a, S_b (128 x 128 fp32 scores, columns 0 and 128) and O_a, O_b
// (128 x D fp32, columns 256 and 256 + D). Per 128-key tile the MMA issuer runs
//   S_a = Q_a K^T, S_b = Q_b K^T   (A, B from shared memory, K-major)
//   O_a += P_a V,  O_b += P_b V    (A = P from tensor memory, B = V from shared memory, MN-major)
// where P_h (bf16) is written by the softmax threads over the first 64 columns of S_h. S_h of the
// next tile may only start once O_h's product (which reads P_h from those columns) has completed,
// so the issue order is
//   PV_a(j), [PV_a(j) done] S_a(j+1), PV_b(j), [PV_b(j) done] S_b(j+1), PV_a(j+1), ...
// and while the softmax of one head runs, the tensor pipe works on the other head's products: the
// two heads ping-pong. (Issuing S_a, S_b, PV_a, PV_b per tile instead lets head a's softmax stall
// the pipe: measured 18 % slower at the 8192-token GQA shape.) The online softmax keeps a stale row
// maximum: O_h is rescaled in tensor memory only when a tile's maximum exceeds the running one by
// more than 2^8.
//
// Warp roles (320 threads): warp 0 = TMA producer (Q_a and Q_b once, then K and V tiles through
// rings of NS slots), warp 1 = MMA issuer and TMEM owner, warps 2-5 = softmax of head a, warps
// 6-9 = softmax of head b (row = 32 * (warp % 4) + lane, the TMEM lane quarter each warp may
// access). The epilogue splits the output columns between the two warpgroups. Every mbarrier
// wait is bounded (ptx.cuh); on a timeout the kernel flags the device status word and unwinds
// without trapping.
#include <cuda.h>
#include <cuda_bf16.h>

#include <cmath>
#include <cstdio>

#include "internal.h"
#include "ptx.cuh"

namespace da {
namespace v2p {

constexpr int BM = 128;
constexpr int BN = 128;
constexpr int kThreads = 320;
constexpr int kSoftmaxWarp0 = 2;
constexpr int kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: stale max allowed while p <= 2^8

template <int D, int NS>
struct Cfg {
  static constexpr int kChunkBytes = 128 * 128;  // one 128-row x 64-col bf16 box
  static constexpr int kQBytes = BM * D * 2;     // one head's query tile
  static constexpr int kKBytes = BN * D * 2;
  static constexpr int kVBytes = BN * D * 2;
  static constexpr int kQOff = 0;                // Q_a, then Q_b
  static constexpr int kKOff = kQOff + 2 * kQBytes;
  static constexpr int kVOff = kKOff + NS * kKBytes;
  static constexpr int kEnd = kVOff + NS * kVBytes;
  static constexpr int kDynSmem = kEnd + 1024;   // + slack for 1024 B alignment
  static constexpr int kOCol = 256;              // O_a at 256, O_b at 256 + D
  static_assert(D % 64 == 0, "64-column TMA boxes");
  static_assert(kOCol + 2 * D <= kTmemCols, "TMEM budget");
  static_assert(kDynSmem <= 232448 - 1024, "shared memory budget");
};

struct Barriers {
  uint64_t q_full;
  uint64_t k_full[4], k_empty[4], v_full[4], v_empty[4];
  uint64_t s_full[2], p_full[2], pv_done[2];  // per head
  uint64_t teardown;
};

struct KParams {
  Problem p;
  int n_qt;          // query tiles per sequence
  int group;         // (batch, pair) units per launch-order group (their K/V share L2)
  float scale_log2;  // log2(e) / sqrt(D)
};

// Where the queries and keys are (KMODE): batched [B, N] (kDense); packed along the token axis
// with cu_seqlens, keys at the queries' rows (kPacked) or with offsets of their own
// (kKeysOffset); or packed queries against keys in a page pool through a block table
// (kKeysPaged; page size a multiple of 128, so a key tile lies in one page). A compile-time
// choice, so that the batched kernel carries none of the packed form's live values.
enum : int { kDense = 0, kPacked = 1, kKeysOffset = 2, kKeysPaged = 3 };

template <int D, int NS, int KMODE>
__global__ void __launch_bounds__(kThreads, 1)
    v2_pair_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const KParams kp) {
  using C = Cfg<D, NS>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ Barriers bars;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  __shared__ float row_factor[2][BM];  // epilogue: 1/l_a and sigmoid(lam)/l_b per row

  const Problem& P = kp.p;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sQ = smem_u32(smem + C::kQOff);
  const uint32_t sK = smem_u32(smem + C::kKOff);
  const uint32_t sV = smem_u32(smem + C::kVOff);

  // ---- work item: (batch, pair) units in groups whose K/V fit in L2 together; inside a group
  // the query tiles go longest-first (causal) across the group's units ----
  const int BU = P.B * P.units;
  const bool causal = (P.flags & 1) != 0;
  const int item = blockIdx.x;
  const int g0 = (item / (kp.group * kp.n_qt)) * kp.group;
  const int gsize = min(kp.group, BU - g0);
  const int r_in = item - g0 * kp.n_qt;
  const int qt = causal ? (kp.n_qt - 1 - r_in / gsize) : (r_in / gsize);
  const int bu = g0 + r_in % gsize;
  const int b = bu / P.units, u = bu % P.units;
  // this sequence's query rows: [seq0, seq0 + SN) of the (packed) token axis, TMA batch
  // coordinate tb; its keys: SNk rows from kseq0 (or through the block table). With keys of
  // their own the queries are the sequence's last SN positions: query i sees keys [0, qoff + i].
  int seq0 = 0, SN = P.N, tb = b;
  if constexpr (KMODE != kDense) {
    seq0 = P.cu_seqlens[b];
    SN = P.cu_seqlens[b + 1] - seq0;
    tb = 0;
    // offsets are device data: a sequence outside [0, total) or longer than the stated maximum
    // is reported (DEV_BAD_INDEX) and skipped, so no store leaves the output
    if (seq0 < 0 || SN < 0 || SN > P.N || seq0 > P.total - SN) {
      if (threadIdx.x == 0 && qt == 0) flag_device_error(DEV_BAD_INDEX);
      return;
    }
    if (qt * BM >= SN) return;  // a tile past this sequence's end: nothing to do (uniform)
  }
  int kseq0 = seq0, SNk = SN;
  if constexpr (KMODE == kKeysOffset) {
    kseq0 = P.cu_seqlens_k[b];
    SNk = P.cu_seqlens_k[b + 1] - kseq0;
    if (kseq0 < 0 || SNk < SN || kseq0 > P.total_k - SNk) {
      if (threadIdx.x == 0 && qt == 0) flag_device_error(DEV_BAD_INDEX);
      return;
    }
  } else if constexpr (KMODE == kKeysPaged) {
    kseq0 = 0;
    SNk = P.seqlens_k[b];
    if (SNk < SN || SNk > P.max_pages * P.page_size) {
      if (threadIdx.x == 0 && qt == 0) flag_device_error(DEV_BAD_INDEX);
      return;
    }
  }
  const int qoff = KMODE >= kKeysOffset ? SNk - SN : 0;
  const int n_kv_all = (SNk + BN - 1) / BN;
  // causal: the tile's last query row sees keys up to qoff + (qt + 1) BM - 1
  const int n_kv = !causal ? n_kv_all
                           : KMODE >= kKeysOffset ? min((qoff + (qt + 1) * BM + BN - 1) / BN, n_kv_all)
                                                  : min(qt + 1, n_kv_all);  // BM == BN
  // first output row of the tile on the (packed or batched) token axis
  const size_t orow_tile =
      (KMODE != kDense ? static_cast<size_t>(seq0) : static_cast<size_t>(b) * P.N) +
      static_cast<size_t>(qt) * BM;

  auto bar = [](uint64_t& x) { return smem_u32(&x); };

  if (threadIdx.x == 0) {
    mbar_init(bar(bars.q_full), 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(bar(bars.k_full[s]), 1);
      mbar_init(bar(bars.k_empty[s]), 1);
      mbar_init(bar(bars.v_full[s]), 1);
      mbar_init(bar(bars.v_empty[s]), 1);
    }
    for (int h = 0; h < 2; ++h) {
      mbar_init(bar(bars.s_full[h]), 1);
      mbar_init(bar(bars.p_full[h]), 128);
      mbar_init(bar(bars.pv_done[h]), 1);
    }
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
  __syncthreads();  // barrier inits visible, TMEM address published
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  volatile int* abrt = &abort_flag;

  if (warp == 0) {
    // ================================ TMA producer ================================
    if (lane == 0) {
      const int kvh = kv_head_of(P, u);
      // extents of the three tensor maps (the host builds them with these dimensions)
      const int mN = KMODE != kDense ? P.total : P.N, mB = KMODE != kDense ? 1 : P.B;
      const int mNk = KMODE == kKeysPaged    ? P.num_pages * P.page_size
                      : KMODE == kKeysOffset ? P.total_k
                                             : mN;
      const Ext4 eq{D, P.q_heads, mN, mB, 2}, ekv{D, P.kv_heads, mNk, mB, 2};
      mbar_arrive_expect_tx(bar(bars.q_full), 2 * C::kQBytes);
      for (int h = 0; h < 2; ++h)
        for (int c = 0; c < D / 64; ++c)
          tma_load_4d_chk(sQ + h * C::kQBytes + c * C::kChunkBytes, &tm_q, bar(bars.q_full),
                          64 * c, 2 * u + h, seq0 + qt * BM, tb, eq);
      // token-axis row of the sequence's key r: packed or batched rows, or (paged) the pool row
      // through the block table. A page id outside the pool reads page 0 and, where the key is
      // in use, flags DEV_BAD_INDEX.
      auto key_row = [&](int r) -> int {
        if constexpr (KMODE == kKeysPaged) {
          const int pi = r / P.page_size;
          int pg = 0;
          if (pi < P.max_pages) {
            pg = P.block_table[static_cast<size_t>(b) * P.max_pages + pi];
            if (pg < 0 || pg >= P.num_pages) {
              if (r < SNk) flag_device_error(DEV_BAD_INDEX);
              pg = 0;
            }
          }
          return pg * P.page_size + (r - pi * P.page_size);
        } else {
          return kseq0 + r;
        }
      };
      int issued = 0;
      for (int j = 0; j < n_kv; ++j) {
        const int s = j % NS;
        const uint32_t ph = (j / NS) & 1;
        const int krow = key_row(j * BN);  // (paged: the table read overlaps the slot wait)
        if (!mbar_wait(bar(bars.k_empty[s]), ph ^ 1, abrt)) break;
        mbar_arrive_expect_tx(bar(bars.k_full[s]), C::kKBytes);
        for (int c = 0; c < D / 64; ++c)
          tma_load_4d_chk(sK + s * C::kKBytes + c * C::kChunkBytes, &tm_k, bar(bars.k_full[s]),
                          64 * c, kvh, krow, tb, ekv);
        if (!mbar_wait(bar(bars.v_empty[s]), ph ^ 1, abrt)) {
          issued = 2 * j + 1;
          break;
        }
        mbar_arrive_expect_tx(bar(bars.v_full[s]), C::kVBytes);
        for (int c = 0; c < D / 64; ++c)
          tma_load_4d_chk(sV + s * C::kVBytes + c * C::kChunkBytes, &tm_v, bar(bars.v_full[s]),
                          64 * c, kvh, krow, tb, ekv);
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
      constexpr uint32_t idesc_o = umma_idesc_bf16(BM, D, 0, 1);
      // Descriptors are built once; each k-step adds a constant offset.
      const uint64_t dq0 = umma_smem_desc(sQ, 16, 1024);
      const uint64_t dk0 = umma_smem_desc(sK, 16, 1024);
      const uint64_t dv0 = umma_smem_desc(sV, C::kChunkBytes, 1024);
      bool ok = mbar_wait(bar(bars.q_full), 0, abrt);
      tc_fence_after();
      // S_h(t) = Q_h K_t^T into S_h's columns
      auto issue_s = [&](int h, int t) {
        const int s = t % NS;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * C::kChunkBytes + (kk & 3) * 32;
          mma_bf16_ss(tmem + h * BN, desc_add(dq0, h * C::kQBytes + off),
                      desc_add(dk0, s * C::kKBytes + off), idesc_s, kk > 0 ? 1u : 0u);
        }
        tc_commit(bar(bars.s_full[h]));
      };
      if (ok) ok = mbar_wait(bar(bars.k_full[0]), 0, abrt);
      if (ok) {
        tc_fence_after();
        issue_s(0, 0);
        issue_s(1, 0);
        tc_commit(bar(bars.k_empty[0]));
      }
      for (int j = 0; ok && j < n_kv; ++j) {
        const int s = j % NS;
        if (!(ok = mbar_wait(bar(bars.v_full[s]), (j / NS) & 1, abrt))) break;
        for (int h = 0; h < 2 && ok; ++h) {
          if (!(ok = mbar_wait(bar(bars.p_full[h]), j & 1, abrt))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk) {
            const uint32_t a_t = tmem + h * BN + kk * 8;
            mma_bf16_ts(tmem + C::kOCol + h * D, a_t, desc_add(dv0, s * C::kVBytes + kk * 2048),
                        idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
          }
          tc_commit(bar(bars.pv_done[h]));
          if (h == 1) tc_commit(bar(bars.v_empty[s]));
          if (j + 1 < n_kv) {
            const int s1 = (j + 1) % NS;
            if (h == 0 && !(ok = mbar_wait(bar(bars.k_full[s1]), ((j + 1) / NS) & 1, abrt))) break;
            if (!(ok = mbar_wait(bar(bars.pv_done[h]), j & 1, abrt))) break;
            tc_fence_after();
            issue_s(h, j + 1);
            if (h == 1) tc_commit(bar(bars.k_empty[s1]));
          }
        }
      }
      // Wait for every MMA we issued before TMEM can be released.
      tc_commit(bar(bars.teardown));
      mbar_wait(bar(bars.teardown), 0, nullptr);
    }
  } else {
    // =========================== softmax / correction / epilogue ===========================
    const int h = (warp - kSoftmaxWarp0) >> 2;       // head of the pair: 0 = 2p, 1 = 2p + 1
    const int r = 32 * (warp & 3) + lane;            // row within the tile
    const int row = qt * BM + r;                     // query position
    const uint32_t tl = static_cast<uint32_t>(32 * (warp & 3)) << 16;  // TMEM lane quarter
    const uint32_t t_s = tmem + tl + h * BN;
    const uint32_t t_o = tmem + tl + C::kOCol + h * D;
    const float sl2 = kp.scale_log2;
    const int lim = causal ? min(qoff + row + 1, SNk) : SNk;  // keys [0, lim) are visible
    float m = -INFINITY, l = 0.f;
    bool ok = true;

    for (int j = 0; j < n_kv; ++j) {
      ok = mbar_wait(bar(bars.s_full[h]), j & 1, abrt);
      if (__any_sync(0xffffffffu, !ok)) { ok = false; break; }
      tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(t_s + 32 * c, sr[c]);
      tmem_wait_ld();
      const int key0 = j * BN;
      if (key0 + BN > lim) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (key0 + 32 * c + i >= lim) sr[c][i] = __float_as_uint(-INFINITY);
      }
      __syncwarp();  // lim differs per lane: reconverge before the warp-wide tcgen05 ops below
      float mx[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mx[i] = __uint_as_float(sr[0][i]);
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int i = (c == 0 ? 8 : 0); i < 32; i += 2)
          mx[i & 7] = fmax3(mx[i & 7], __uint_as_float(sr[c][i]), __uint_as_float(sr[c][i + 1]));
#pragma unroll
      for (int i = 0; i < 4; ++i) mx[i] = fmaxf(mx[i], mx[i + 4]);
      const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * sl2;
      if (j == 0) {
        m = mt;
      } else {
        const bool need = mt > m + kRescaleThreshold;
        if (__any_sync(0xffffffffu, need)) {
          // O_h holds tiles 0 .. j-1 scaled by the old max: wait for their product, rescale.
          const float mn = need ? mt : m;
          const float f = ex2_approx(m - mn);
          l *= f;
          m = mn;
          ok = mbar_wait(bar(bars.pv_done[h]), (j - 1) & 1, abrt);
          if (__any_sync(0xffffffffu, !ok)) { ok = false; break; }
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < D / 16; ++c) {
            uint32_t o[16];
            tmem_ld16(t_o + 16 * c, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * f);
            tmem_st16(t_o + 16 * c, o);
          }
          tmem_wait_st();
        }
      }
      // P = 2^(s * scale_log2 - m) in bf16, written over the first 64 columns of S_h
      const float nm = (m == -INFINITY) ? 0.f : -m;
      const uint64_t c2 = f2pack(sl2, sl2), nm2 = f2pack(nm, nm);
      uint64_t lsum = f2pack(0.f, 0.f);
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint32_t pk[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int e = 16 * c + 2 * i;
          const uint64_t x = f2fma(f2pack(__uint_as_float(sr[e >> 5][e & 31]),
                                          __uint_as_float(sr[e >> 5][(e & 31) + 1])),
                                   c2, nm2);
          float x0, x1;
          f2unpack(x, x0, x1);
          const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
          lsum = f2add(lsum, f2pack(p0, p1));
          pk[i] = pack_bf16x2(p0, p1);
        }
        tmem_st8(t_s + 8 * c, pk);
      }
      float l0, l1;
      f2unpack(lsum, l0, l1);
      l += l0 + l1;
      if constexpr (KMODE != kDense) {
        // Packed or paged keys: the tile's rows past the sequence's keys hold other data (the next
        // sequence, padding, unused page rows) that may not be finite. Their P is 0, but 0 * NaN
        // would still reach O, so head a's threads zero those V rows before releasing P_a (both
        // heads' products are issued after that). Batched tiles past N are zero-filled by TMA.
        if (h == 0 && key0 + BN > SNk) {
          const int s = j % NS;
          ok = mbar_wait(bar(bars.v_full[s]), (j / NS) & 1, abrt);
          if (__any_sync(0xffffffffu, !ok)) { ok = false; break; }
          if (key0 + r >= SNk) {
#pragma unroll
            for (int c = 0; c < D / 64; ++c) {
              const uint32_t vrow = sV + s * C::kVBytes + c * C::kChunkBytes + r * 128;
#pragma unroll
              for (int q = 0; q < 8; ++q) st_shared_v4(vrow + 16 * q, 0u, 0u, 0u, 0u);
            }
          }
          fence_proxy_async_smem();
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(bars.p_full[h]));
    }
    if (ok) {
      ok = mbar_wait(bar(bars.pv_done[h]), (n_kv - 1) & 1, abrt);
      ok = !__any_sync(0xffffffffu, !ok);
    }
    tc_fence_after();

    // ------------------------------- epilogue -------------------------------------
    // out = O_a / l_a - sigmoid(lam) * O_b / l_b; warpgroup h stores columns [h D/2, (h+1) D/2)
    if (h == 0) {
      row_factor[0][r] = 1.f / l;
    } else {
      float lam = 0.f;
      if (row < SN) {
        const float z = P.lam_logit[(orow_tile + r) * P.units + u];
        lam = 1.f / (1.f + expf(-z));
      }
      row_factor[1][r] = lam / l;
    }
    __syncwarp();
    named_barrier_sync(1, 256);
    const float fa = row_factor[0][r], fb = row_factor[1][r];
    // `ok` is uniform per warp; the row test is not, so the tensor-memory loads (warp-wide
    // .sync.aligned instructions) stay outside it and only the stores are predicated.
    if (ok) {
      // The warp's 32 rows x D/2 columns go through shared memory (the K ring, idle once the
      // last score product is done), so that each store instruction writes whole 128-byte row
      // pieces instead of 32 scattered 16-byte ones.
      constexpr int H2 = D / 2;
      constexpr int RB = H2 * 2;          // bytes of one row's slice
      constexpr int PIECES = RB / 16;     // 16-byte pieces per slice
      constexpr int RPI = 32 / PIECES;    // rows per store instruction
      static_assert(256 * RB <= NS * C::kKBytes, "staging fits in the K ring");
      const int col0 = h * H2;
      uint8_t* stage = smem + C::kKOff + (warp - kSoftmaxWarp0) * 32 * RB;
      const bool live = row < SN;
#pragma unroll 1
      for (int c = 0; c < H2; c += 32) {
        uint32_t oa[32], ob[32];
        tmem_ld32(tmem + tl + C::kOCol + col0 + c, oa);
        tmem_ld32(tmem + tl + C::kOCol + D + col0 + c, ob);
        tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4 pkt;
          uint32_t* pw = reinterpret_cast<uint32_t*>(&pkt);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int e = 8 * q + 2 * i;
            pw[i] = pack_bf16x2(__uint_as_float(oa[e]) * fa - __uint_as_float(ob[e]) * fb,
                                __uint_as_float(oa[e + 1]) * fa - __uint_as_float(ob[e + 1]) * fb);
          }
          const int piece = (c + 8 * q) / 8;
          *reinterpret_cast<uint4*>(stage + lane * RB + ((piece ^ (lane & (PIECES - 1))) * 16)) = pkt;
        }
      }
      __syncwarp();
      const size_t orow0 = (orow_tile + 32 * (warp & 3)) * P.units + u;
      __nv_bfloat16* out0 = static_cast<__nv_bfloat16*>(P.out) + col0;
#pragma unroll
      for (int it = 0; it < PIECES; ++it) {
        const int rr = it * RPI + lane / PIECES;   // row (lane of the warp) this lane stores
        const int pc = lane % PIECES;
        const uint4 v = *reinterpret_cast<const uint4*>(stage + rr * RB + ((pc ^ (rr & (PIECES - 1))) * 16));
        if (qt * BM + 32 * (warp & 3) + rr < SN &&
            dbg_index_ok(static_cast<long long>(orow_tile) + 32 * (warp & 3) + rr,
                         KMODE != kDense ? P.total : 1LL * P.B * P.N))
          *reinterpret_cast<uint4*>(out0 + (orow0 + static_cast<size_t>(rr) * P.units) * D + pc * 8) = v;
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
// 4-D bf16 map over a dense [B, N, heads, D] tensor with a 64-col x 1 x 128-row x 1 box,
// 128-byte swizzle, zero fill out of bounds.
static bool make_map(CUtensorMap* m, const void* base, int cols, int heads, int N, int B,
                     char* err, size_t err_len) {
  cuuint64_t dims[4] = {(cuuint64_t)cols, (cuuint64_t)heads, (cuuint64_t)N, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)cols * 2, (cuuint64_t)cols * heads * 2,
                           (cuuint64_t)cols * heads * 2 * (cuuint64_t)N};
  cuuint32_t box[4] = {64, 1, 128, 1};
  return encode_tmap_4d(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, dims, strides, box, err, err_len);
}

template <int D, int NS, int KMODE>
static cudaError_t launch_cfg(const Problem& p, cudaStream_t s, char* err, size_t err_len) {
  using C = Cfg<D, NS>;
  CUtensorMap mq, mk, mv;
  // packed sequences: one batch row of `total` tokens; otherwise [B, N]
  const int mN = KMODE != kDense ? p.total : p.N, mB = KMODE != kDense ? 1 : p.B;
  // keys with offsets of their own, or the page pools as one [num_pages * page_size] axis
  const int mNk = KMODE == kKeysPaged    ? p.num_pages * p.page_size
                  : KMODE == kKeysOffset ? p.total_k
                                         : mN;
  if (!make_map(&mq, p.q, D, p.q_heads, mN, mB, err, err_len) ||
      !make_map(&mk, p.k, D, p.kv_heads, mNk, mB, err, err_len) ||
      !make_map(&mv, p.v, D, p.kv_heads, mNk, mB, err, err_len))
    return cudaErrorInvalidValue;
  auto kern = v2_pair_kernel<D, NS, KMODE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kDynSmem);
  if (e != cudaSuccess) return e;
  KParams kp;
  kp.p = p;
  kp.n_qt = (p.N + BM - 1) / BM;
  kp.scale_log2 = kLog2e * p.scale;
  {
    // K/V bytes per (batch, pair) unit (the group / 2 pairs of a KV head share them); keep a
    // launch-order group's K/V within 32 MB of L2. Measured at the 8192-token GQA shape: with
    // 32 MB DRAM reads equal q + k + v (338 MB), with 64 MB (the whole K/V of the launch) the
    // streamed queries and outputs evict K/V tiles that later query tiles read again (594 MB)
    const int nk = (p.cu_seqlens_k || p.block_table) ? p.max_seqlen_k : p.N;
    const double kv_bytes = static_cast<double>(nk) * D * 2.0 * 2.0 / (p.group / 2);
    long long g = static_cast<long long>((32.0 * 1024 * 1024) / (kv_bytes > 1 ? kv_bytes : 1));
    const long long bu = static_cast<long long>(p.B) * p.units;
    kp.group = static_cast<int>(g < 1 ? 1 : (g > bu ? bu : g));
  }
  const long long items = static_cast<long long>(kp.n_qt) * p.B * p.units;
  if (items == 0) return cudaSuccess;
  kern<<<dim3(static_cast<unsigned>(items)), kThreads, C::kDynSmem, s>>>(mq, mk, mv, kp);
  return cudaGetLastError();
}

}  // namespace v2p

cudaError_t status_prefill_v2(int* v) { return read_clear_status(v); }

// V2 pair prefill, bf16 tensors: q [B, N, Hq, D], k and v [B, N, Hkv, D] (or packed along the
// token axis with cu_seqlens, keys with offsets of their own or in a page pool), D = 64 or 128.
cudaError_t launch_prefill_v2(const Problem& p, cudaStream_t s, char* err, size_t err_len) {
  if (p.mode != MODE_V2 || p.dqk != p.dv || p.group < 2 || p.group % 2 != 0)
    return cudaErrorNotSupported;
  using namespace v2p;
  const int mode = !p.cu_seqlens ? kDense
                   : p.block_table ? kKeysPaged
                   : p.cu_seqlens_k ? kKeysOffset
                                    : kPacked;
  if (p.dqk == 128) {
    switch (mode) {
      case kDense: return launch_cfg<128, 2, kDense>(p, s, err, err_len);
      case kPacked: return launch_cfg<128, 2, kPacked>(p, s, err, err_len);
      case kKeysOffset: return launch_cfg<128, 2, kKeysOffset>(p, s, err, err_len);
      default: return launch_cfg<128, 2, kKeysPaged>(p, s, err, err_len);
    }
  }
  if (p.dqk == 64) {
    switch (mode) {
      case kDense: return launch_cfg<64, 4, kDense>(p, s, err, err_len);
      case kPacked: return launch_cfg<64, 4, kPacked>(p, s, err, err_len);
      case kKeysOffset: return launch_cfg<64, 4, kKeysOffset>(p, s, err, err_len);
      default: break;
    }
  }
  return cudaErrorNotSupported;
}

}  // namespace da
