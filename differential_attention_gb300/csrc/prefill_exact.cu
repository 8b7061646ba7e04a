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
// (already small) to bf16 once and runs a single D V product. Both passes together issue the
// same MMA work as the single-pass form (4d + 4dv flops per query-key pair).
//
// Structure: one CTA per 128-row query tile of one unit, 128-key tiles (a tcgen05.mma with
// M = 128 has a fixed cost of ~95 cycles, so score MMAs use N = 128 and value MMAs N = dv).
//   pass 1: S1, S2 (128 fp32 columns each) double-buffered over all 512 TMEM columns;
//   pass 2: S1, S2 single-buffered in columns 0..255, O (128 x dv fp32) in columns 256..;
//           D goes to shared memory (128B-swizzled K-major), so the next score MMA overlaps the
//           D computation; the value MMA reads D and V from shared memory.
// TMA stages Q1|Q2 once and a ring of K tiles (one load per map; each K tile is streamed twice,
// once per pass) and V half tiles (pass 2 only), issued in exactly the order the MMA issuer
// consumes them so that no load waits behind a slot of another kind. Four softmax warpgroups (one
// thread per query row each) split every tile's 128 keys; their partial row statistics merge
// once at the pass boundary. Epilogue: RMSNorm and scale straight out of tensor memory, each
// warpgroup taking a quarter of the columns. Warp 0 = TMA producer, warp 1 = MMA issuer and TMEM
// owner, warps 2-17 = softmax and epilogue. Every wait is bounded.
#include <cuda.h>
#include <cuda_bf16.h>

#include <cmath>
#include <cstdio>

#include "internal.h"
#include "ptx.cuh"

namespace da {
namespace exact {

constexpr int BM = 128;
constexpr int BN = 128;
constexpr int kSoftmaxWarp0 = 2;  // warp 0 TMA, warp 1 MMA, warps 2..17 softmax
constexpr int kNumWG = 4;         // softmax warpgroups; each takes 32 keys of every tile
constexpr int kSoftmaxThreads = 128 * kNumWG;
constexpr int kThreads = 32 * kSoftmaxWarp0 + kSoftmaxThreads;
constexpr int KW = 128 / kNumWG;  // keys per warpgroup per tile
constexpr int kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kSmemLimit = 232448;  // bytes of shared memory one CTA may use

// QK8: q and k hold fp8 e4m3 (v stays bf16); the score products run as kind::f8f6f4.
template <int DQK, int DV, bool SHARED_K, bool QK8 = false>
struct Cfg {
  static constexpr int kChunk = 128 * 128;              // 128 rows x 128 bytes (one TMA box)
  static constexpr int kQKElt = QK8 ? 1 : 2;            // bytes per q/k element
  static constexpr int kQKBoxCols = 128 / kQKElt;       // q/k elements per 128-byte box row
  static constexpr int kQKBoxes = DQK * kQKElt / 128;   // boxes per map's Q or K tile
  static constexpr int kQKSteps = DQK * kQKElt / 32;    // score MMA k-steps (32 bytes each)
  static constexpr int kQMapBytes = BM * DQK * kQKElt;  // one map's Q tile
  static constexpr int kKMapBytes = BN * DQK * kQKElt;  // one map's K tile
  static constexpr int kQBytes = 2 * kQMapBytes;
  // K loads per key tile: one per map, or one for both (shared K in V2; both fp8 maps in a slot)
  static constexpr int kKLoads = (SHARED_K || QK8) ? 1 : 2;
  static constexpr int kKLoadBytes = QK8 ? 2 * kKMapBytes : kKMapBytes;
  static constexpr int kVHalfChunk = (BN / 2) * 128;    // 64 keys x 64 bf16
  static constexpr int kVHalfBytes = (BN / 2) * DV * 2; // half of a V tile (one load)
  static constexpr int kDBytes = BM * BN * 2;           // D tile (bf16)
  static constexpr int kSlot = kKLoadBytes > kVHalfBytes ? kKLoadBytes : kVHalfBytes;
  static constexpr int kRingBudget = kSmemLimit - 2048 - 1024 - kQBytes - kDBytes;
  static constexpr int NSLOT = (kRingBudget / kSlot) > 8 ? 8 : (kRingBudget / kSlot);
  static constexpr int kQOff = 0;
  static constexpr int kDOff = kQOff + kQBytes;
  static constexpr int kSlotOff = kDOff + kDBytes;
  static constexpr int kEnd = kSlotOff + NSLOT * kSlot;
  static constexpr int kDynSmem = kEnd + 1024;          // + slack for 1024 B alignment
  static constexpr int kOCol = 256;
  static_assert(NSLOT >= kKLoads + 2, "each load of a key tile needs its own slot");
  static_assert(kOCol + DV <= kTmemCols, "TMEM budget");
  static_assert(kDynSmem + 2048 <= kSmemLimit, "shared memory budget (dynamic + static)");
};

struct Barriers {
  uint64_t q_full;
  uint64_t slot_full[8], slot_empty[8];
  uint64_t s_full[2], s_free[2];  // scores in TMEM buffer b ready / read by both warpgroups
  uint64_t d_full, d_empty;       // D tile in shared memory written / consumed
  uint64_t o_full;
  uint64_t teardown;
};

struct KParams {
  Problem p;
  int n_qt;
  int group;  // (batch, unit) pairs whose K/V share L2 in one launch-order group
  float scale_log2;
};

// Where a sequence's keys are (KMODE).
enum : int {
  kKeysShared = 0,  // at the queries' rows (batched, or packed with cu_seqlens)
  kKeysOffset = 1,  // packed with offsets of their own (cu_seqlens_k)
  kKeysPaged = 2,   // in a page pool through a block table (page size a multiple of 128)
};

// SHARED_K: the V2 operator (both maps read one K tile); without it, V1 (launch_prefill_exact
// picks the instantiation by mode). KMODE: where the keys are. GROUPED: the grouped form (map 1's
// Q and K in the unit's noise head). The key modes and the grouped form are instantiations of
// their own: their extra live values made the default variants spill at their 96-register
// budget.
template <int DQK, int DV, bool SHARED_K, bool QK8, int KMODE, bool GROUPED = false>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_exact_kernel(const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const KParams kp) {
  using C = Cfg<DQK, DV, SHARED_K, QK8>;
  constexpr int NSLOT = C::NSLOT;
  extern __shared__ uint8_t smem_raw[];
  __shared__ Barriers bars;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const Problem& P = kp.p;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sQ = smem_u32(smem + C::kQOff);
  const uint32_t sD = smem_u32(smem + C::kDOff);
  const uint32_t sSlot = smem_u32(smem + C::kSlotOff);
  // The D buffer doubles as scratch for the warpgroups' statistics merge (pass boundary) and
  // the sums of squares (epilogue): D is not in use at either point.
  float* scratch = reinterpret_cast<float*>(smem + C::kDOff);

  // Launch order: (batch, unit) pairs are taken in groups whose K/V fit in L2 together; inside a
  // group the query tiles go longest-first (causal) across the group's pairs.
  // grouped form in two launches: phase 1 runs one CTA per (noise head, query tile) -- unit u is
  // then the first signal head of the noise head's group -- and phase 2 the signal heads
  const int gphase = GROUPED ? P.gda_phase : 0;
  const int gunits = gphase == 1 ? P.units / P.group : P.units;
  const int BU = P.B * gunits;
  const bool causal = (P.flags & 1) != 0;
  const int item = blockIdx.x;
  const int g0 = (item / (kp.group * kp.n_qt)) * kp.group;
  const int gsize = min(kp.group, BU - g0);
  const int r_in = item - g0 * kp.n_qt;
  const int qt = causal ? (kp.n_qt - 1 - r_in / gsize) : (r_in / gsize);
  const int bu = g0 + r_in % gsize;
  const int b = bu / gunits, u = gphase == 1 ? (bu % gunits) * P.group : bu % gunits;
  // this sequence's query rows: [seq0, seq0 + SN) of the (packed) token axis, its key rows
  // [kseq0, kseq0 + SNk); TMA batch coordinate tb. With keys of their own (cu_seqlens_k) the
  // queries are the sequence's last SN positions: query row i sees keys [0, qoff + i], with
  // qoff = SNk - SN.
  int seq0 = 0, SN = P.N, tb = b;
  if (P.cu_seqlens) {
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
    // keys outside k, or fewer keys than queries: reported and skipped like the query offsets
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
  const int qoff = KMODE != kKeysShared ? SNk - SN : 0;
  const int n_kv_all = (SNk + BN - 1) / BN;
  // causal: the tile's last query row sees keys up to qoff + (qt + 1) BM - 1
  const int n = !causal ? n_kv_all
                        : KMODE != kKeysShared ? min((qoff + (qt + 1) * BM + BN - 1) / BN, n_kv_all)
                               : min(qt + 1, n_kv_all);  // BM == BN
  // W1: pass 1 runs over 256-key tiles (one N = 256 score MMA per map and k-step instead of two
  // N = 128 ones: a tcgen05.mma's cost grows far less than its N). Only S1 and S2 live in pass 1,
  // so each map's 256 score columns take half of tensor memory, single-buffered. The shared-K
  // (V2), fp8 and d = 64 forms keep 128-key tiles in both passes (a 256-row chunk of K is one
  // 32 KB ring slot at d = 128).
  constexpr bool W1 = !SHARED_K && !QK8 && DQK == 128;
  static_assert(!W1 || C::kSlot >= 2 * C::kChunk, "a 256-row K chunk fills one ring slot");
  const int n1 = W1 ? (n + 1) / 2 : n;  // pass-1 tiles (the last one 128 keys wide when n is odd)
  const int T = gphase == 1 ? n1 : n1 + n;  // tiles over both passes (phase 1: pass 1 only)
  // maps in pass 1: both, or (grouped phases, W1 only) map 2 alone (phase 1) or map 1 alone
  // (phase 2)
  const int p1maps = gphase ? 1 : 2, p1map0 = gphase == 1 ? 1 : 0;

  // Ring order of the loads = the order in which the MMA issuer consumes them. Iteration t < n1
  // of the issuer uses the K loads of pass-1 tile t: with W1 one per map and 64-column chunk
  // (each a slot of 256 key rows), else one per map (or one shared K). Iteration t >= n1 uses
  // the K loads of pass-2 tile t - n1 (one per map, both chunks of 128 rows), then for t > n1
  // the two V halves of pass-2 tile jv = t - 1 - n1. base(t) = index of iteration t's first load.
  constexpr int KL = C::kKLoads;
  const int KL1 = W1 ? 2 * p1maps : KL;
  auto base = [n1, KL1](int t) {
    return t <= n1 ? KL1 * t : KL1 * n1 + KL + (KL + 2) * (t - n1 - 1);
  };
  auto k_load = [&](int t, int r) { return base(t) + r; };
  auto v_load = [&](int jv, int h) {
    const int t = n1 + 1 + jv;
    return base(t) + (t < T ? KL : 0) + h;
  };
  // TMEM score buffer of tile t and its use count on that buffer (barrier phase index). With W1
  // buffer 0 holds map 1's scores (pass 1) and both maps' (pass 2), buffer 1 map 2's (pass 1):
  // each is used once per tile, so the use count of either is t.
  auto sbuf = [n1](int t) { return (!W1 && t < n1) ? (t & 1) : 0; };
  auto suse = [n1](int t) { return W1 ? t : t < n1 ? (t >> 1) : ((n1 + 1) >> 1) + (t - n1); };

  auto bar = [](uint64_t& x) { return smem_u32(&x); };

  if (threadIdx.x == 0) {
    mbar_init(bar(bars.q_full), 1);
    for (int s = 0; s < 8; ++s) {
      mbar_init(bar(bars.slot_full[s]), 1);
      mbar_init(bar(bars.slot_empty[s]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(bars.s_full[i]), 1);
      mbar_init(bar(bars.s_free[i]), kSoftmaxThreads);
    }
    mbar_init(bar(bars.d_full), kSoftmaxThreads);
    mbar_init(bar(bars.d_empty), 1);
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
      const int kvh = kv_head_of(P, u);  // V (and the K of both maps but in the grouped form)
      // extents of the three tensor maps (the host builds them with these dimensions)
      const int mN = P.cu_seqlens ? P.total : P.N, mB = P.cu_seqlens ? 1 : P.B;
      const int mNk = KMODE == kKeysPaged    ? P.num_pages * P.page_size
                      : KMODE == kKeysOffset ? P.total_k
                                             : mN;
      const Ext4 eq{P.q_cols, P.q_heads, mN, mB, C::kQKElt};
      const Ext4 ek{P.k_cols, P.kv_heads, mNk, mB, C::kQKElt};
      const Ext4 ev{DV, v_heads(P), mNk, mB, 2};
      mbar_arrive_expect_tx(bar(bars.q_full), C::kQBytes);
      for (int r = 0; r < 2; ++r)
        for (int c = 0; c < C::kQKBoxes; ++c)
          tma_load_4d_chk(sQ + r * C::kQMapBytes + c * C::kChunk, &tm_q, bar(bars.q_full),
                          q_col_of(P, r) + C::kQKBoxCols * c,
                          GROUPED ? grouped_head(P, u, r) : (P.mode == MODE_V1 ? u : 2 * u + r),
                          seq0 + qt * BM, tb, eq);
      int issued = 0;  // loads issued into the ring
      auto acquire = [&](int idx, uint32_t bytes) -> int {
        const int slot = idx % NSLOT;
        if (!mbar_wait(bar(bars.slot_empty[slot]), ((idx / NSLOT) & 1) ^ 1, abrt)) return -1;
        mbar_arrive_expect_tx(bar(bars.slot_full[slot]), bytes);
        return slot;
      };
      // token-axis row of the sequence's key r: packed or batched rows, or (paged) the pool row
      // through the block table. A page id outside the pool reads page 0 and, where the key is
      // in use, flags DEV_BAD_INDEX; tiles start at multiples of 64 keys, inside one page.
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
      bool ok = true;
      for (int t = 0; t <= T && ok; ++t) {
        if (W1 && t < n1) {
          // pass-1 tile t: keys [256 t, 256 t + 256), one slot per map and 64-column chunk,
          // holding its 256 rows as two 128-row boxes (one when the tile is 128 keys wide)
          const int halves = 2 * t + 1 < n ? 2 : 1;
          const int krow0 = key_row(2 * t * BN);
          const int krow1 = halves == 2 ? key_row((2 * t + 1) * BN) : 0;
          for (int q = 0; q < KL1 && ok; ++q) {
            const int mp = p1maps == 2 ? (q >> 1) : p1map0, c = q & 1;
            const int ks = acquire(k_load(t, q), halves * C::kChunk);
            if (ks < 0) {
              ok = false;
              break;
            }
            for (int hh = 0; hh < halves; ++hh)
              tma_load_4d_chk(sSlot + ks * C::kSlot + hh * C::kChunk, &tm_k,
                              bar(bars.slot_full[ks]), k_col_of(P, mp) + C::kQKBoxCols * c,
                              GROUPED ? grouped_head(P, u, mp) : kvh, hh ? krow1 : krow0, tb, ek);
            issued = k_load(t, q) + 1;
          }
        } else if (t < T) {
          const int j = t < n1 ? t : t - n1;
          const int krow = key_row(j * BN);  // (paged: the table read overlaps the slot wait)
          for (int r = 0; r < KL && ok; ++r) {
            const int ks = acquire(k_load(t, r), C::kKLoadBytes);
            if (ks < 0) {
              ok = false;
              break;
            }
            for (int mp = QK8 ? 0 : r; mp <= (QK8 ? 1 : r); ++mp)  // maps in this load
              for (int c = 0; c < C::kQKBoxes; ++c)
                tma_load_4d_chk(
                    sSlot + ks * C::kSlot + (QK8 ? mp * C::kKMapBytes : 0) + c * C::kChunk, &tm_k,
                    bar(bars.slot_full[ks]), k_col_of(P, mp) + C::kQKBoxCols * c,
                    GROUPED ? grouped_head(P, u, mp) : kvh, krow, tb, ek);
            issued = k_load(t, r) + 1;
          }
        }
        if (ok && t >= n1 + 1) {
          const int jv = t - n1 - 1;
          for (int h = 0; h < 2 && ok; ++h) {
            const int vrow = key_row(jv * BN + 64 * h);
            const int vs = acquire(v_load(jv, h), C::kVHalfBytes);
            if (vs < 0) {
              ok = false;
              break;
            }
            for (int c = 0; c < DV / 64; ++c)
              tma_load_4d_chk(sSlot + vs * C::kSlot + c * C::kVHalfChunk, &tm_v,
                              bar(bars.slot_full[vs]), 64 * c, kvh, vrow, tb, ev);
            issued = v_load(jv, h) + 1;
          }
        }
      }
      // make sure no copy of ours is still landing in shared memory
      mbar_wait(bar(bars.q_full), 0, nullptr);
      for (int i = max(0, issued - NSLOT); i < issued; ++i)
        mbar_wait(bar(bars.slot_full[i % NSLOT]), (i / NSLOT) & 1, nullptr);
    }
  } else if (warp == 1) {
    // ================================ MMA issuer ==================================
    if (lane == 0) {
      constexpr uint32_t idesc_s = QK8 ? umma_idesc_e4m3(BM, BN) : umma_idesc_bf16(BM, BN, 0, 0);
      constexpr uint32_t idesc_o = umma_idesc_bf16(BM, DV, 0, 1);
      // Descriptors are built once; each k-step adds a constant offset.
      const uint64_t dq0 = umma_smem_desc(sQ, 16, 1024);
      const uint64_t dslot0 = umma_smem_desc(sSlot, 16, 1024);
      const uint64_t dv0 = umma_smem_desc(sSlot, C::kVHalfChunk, 1024);  // V: MN-major, LBO = chunk
      const uint64_t dd0 = umma_smem_desc(sD, 16, 1024);
      bool ok = mbar_wait(bar(bars.q_full), 0, abrt);
      tc_fence_after();
      for (int t = 0; ok && t <= T; ++t) {
        if (W1 && t < n1) {
          // pass-1 tile t: S_r (128 x 256, or 128 x 128 for a last tile of 128 keys) into
          // columns 256 r; each 64-column chunk's slot is released as soon as its four k-steps
          // are done, so the next tile's load overlaps the rest of this tile's products
          constexpr uint32_t idesc_w = umma_idesc_bf16(BM, 2 * BN, 0, 0);
          const uint32_t idesc = 2 * t + 1 < n ? idesc_w : idesc_s;
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            if (p1maps == 1 && r != p1map0) continue;
            if (t > 0 && !(ok = mbar_wait(bar(bars.s_free[r]), (t - 1) & 1, abrt))) break;
            const uint64_t qd = desc_add(dq0, r * C::kQMapBytes);
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              const int ki = k_load(t, (p1maps == 2 ? 2 * r : 0) + c), s = ki % NSLOT;
              if (!(ok = mbar_wait(bar(bars.slot_full[s]), (ki / NSLOT) & 1, abrt))) break;
              tc_fence_after();
              const uint64_t kd = desc_add(dslot0, s * C::kSlot);
#pragma unroll
              for (int k4 = 0; k4 < 4; ++k4)
                mma_bf16_ss(tmem + r * 256, desc_add(qd, c * C::kChunk + k4 * 32),
                            desc_add(kd, k4 * 32), idesc, (c > 0 || k4 > 0) ? 1u : 0u);
              tc_commit(bar(bars.slot_empty[s]));
            }
            if (!ok) break;
            tc_commit(bar(bars.s_full[r]));
          }
          if (!ok) break;
        } else if (t < T) {
          const int buf = sbuf(t);
          // The buffer's previous scores must have been read by both warpgroups: tile t-2 in
          // pass 1 (two buffers), tile t-1 in pass 2 (one buffer; reading t-1 implies t-2; with
          // W1 the last pass-1 tile's map-1 scores, which held these columns).
          const int prev = t < n1 ? t - 2 : t - 1;
          if (prev >= 0 &&
              !(ok = mbar_wait(bar(bars.s_free[sbuf(prev)]), suse(prev) & 1, abrt)))
            break;
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const int ki = k_load(t, (SHARED_K || QK8) ? 0 : r), s = ki % NSLOT;
            if (r < KL) {
              if (!(ok = mbar_wait(bar(bars.slot_full[s]), (ki / NSLOT) & 1, abrt))) break;
              tc_fence_after();
            }
            const uint32_t d_s = tmem + buf * 256 + r * 128;
            const uint64_t qd = desc_add(dq0, r * C::kQMapBytes);
            const uint64_t kd = desc_add(dslot0, s * C::kSlot + (QK8 ? r * C::kKMapBytes : 0));
#pragma unroll
            for (int kk = 0; kk < C::kQKSteps; ++kk) {
              const uint32_t off = (kk >> 2) * C::kChunk + (kk & 3) * 32;
              if constexpr (QK8)
                mma_e4m3_ss(d_s, desc_add(qd, off), desc_add(kd, off), idesc_s, kk > 0 ? 1u : 0u);
              else
                mma_bf16_ss(d_s, desc_add(qd, off), desc_add(kd, off), idesc_s, kk > 0 ? 1u : 0u);
            }
            if (r == 1 || (!SHARED_K && !QK8)) tc_commit(bar(bars.slot_empty[s]));
          }
          if (!ok) break;
          tc_commit(bar(bars.s_full[buf]));
        }
        const int tp = t - 1;
        if (tp >= n1) {
          const int jv = tp - n1;
          // O's columns held map 2's scores in the last pass-1 tile (W1): read by now
          if (W1 && jv == 0 && p1maps == 2 &&
              !(ok = mbar_wait(bar(bars.s_free[1]), (n1 - 1) & 1, abrt)))
            break;
          if (!(ok = mbar_wait(bar(bars.d_full), jv & 1, abrt))) break;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int vi = v_load(jv, h), sv = vi % NSLOT;
            if (!(ok = mbar_wait(bar(bars.slot_full[sv]), (vi / NSLOT) & 1, abrt))) break;
            tc_fence_after();
            const uint64_t vd = desc_add(dv0, sv * C::kSlot);
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4) {
              // A = D (128 rows x 16 keys, K-major), B = V half (16 keys x dv, MN-major)
              const int kk = 4 * h + k4;
              const uint64_t ad = desc_add(dd0, (kk >> 2) * C::kChunk + (kk & 3) * 32);
              mma_bf16_ss(tmem + C::kOCol, ad, desc_add(vd, k4 * 2048), idesc_o,
                          (jv > 0 || kk > 0) ? 1u : 0u);
            }
            tc_commit(bar(bars.slot_empty[sv]));
          }
          if (!ok) break;
          tc_commit(bar(bars.d_empty));
          if (tp == T - 1) tc_commit(bar(bars.o_full));
        }
      }
      tc_commit(bar(bars.teardown));
      mbar_wait(bar(bars.teardown), 0, nullptr);
    }
  } else if (warp >= kSoftmaxWarp0) {
    // ============================ softmax and epilogue ============================
    // Warpgroup wg (warps 2+4wg .. 5+4wg, which cover the four TMEM lane quarters) handles keys
    // [32 wg, 32 wg + 32) of every tile, both maps, for its query row.
    const int wg = (warp - kSoftmaxWarp0) >> 2;
    const int r = 32 * (warp & 3) + lane;
    const int row = qt * BM + r;
    const uint32_t tl = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const float sl2 = kp.scale_log2;
    const int lim = causal ? min(qoff + row + 1, SNk) : SNk;  // keys [0, lim) are visible
    // output row on the token axis: packed (seq0 + row) or batched (b * N + row); `oaddr` is
    // the row's element offset in the (possibly strided) output
    const size_t orow = P.cu_seqlens ? static_cast<size_t>(seq0) + row
                                     : static_cast<size_t>(b) * P.N + row;
    const size_t oaddr = P.cu_seqlens ? elem_off(P.os, 0, seq0 + row, u) : elem_off(P.os, b, row, u);
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
    float bias[2] = {0.f, 0.f}, lam = 0.f;
    bool ok = true, merged = false;
    // lambda from its vectors: computed now, while the first tiles are still in flight
    const float lam_fused =
        (P.mode == MODE_V1 && P.lam_vec[0]) ? lambda_from_vectors_warp(P, u) : 0.f;

    // Merge the warpgroups' partial row statistics (once, at the pass boundary). The D buffer
    // is free then: no D has been written yet.
    auto merge = [&]() {
      float* st = scratch + (wg * 4) * BM;
      st[0 * BM + r] = m[0];
      st[1 * BM + r] = l[0];
      st[2 * BM + r] = m[1];
      st[3 * BM + r] = l[1];
      named_barrier_sync(1, kSoftmaxThreads);
#pragma unroll
      for (int mp = 0; mp < 2; ++mp) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kNumWG; ++w) M = fmaxf(M, scratch[(w * 4 + 2 * mp) * BM + r]);
        float L = 0.f;
#pragma unroll
        for (int w = 0; w < kNumWG; ++w) {
          const float mw = scratch[(w * 4 + 2 * mp) * BM + r];
          if (mw != -INFINITY) L += scratch[(w * 4 + 2 * mp + 1) * BM + r] * ex2_approx(mw - M);
        }
        bias[mp] = -(M + __log2f(L));
      }
      // grouped, phase 2: the noise map's statistic comes from phase 1 (rows past N: unused)
      if (gphase == 2)
        bias[1] = -P.gda_noise[(static_cast<size_t>(b) * (P.units / P.group) + u / P.group) *
                                   P.n_pad + row];
      if (GROUPED || P.mode == MODE_V1) {
        lam = P.lam_vec[0] ? lam_fused : P.lambda[u];
      } else if (row < (SHARED_K ? SN : P.N)) {
        // V2: the sigmoid of this token's logit for pair u (packed sequences: token seq0 + row;
        // the select exists only in the V2 instantiations, as changes here shifted the V1 code)
        size_t t = static_cast<size_t>(b) * P.N + row;
        if constexpr (SHARED_K) {
          if (P.cu_seqlens) t = orow;
        }
        const float z = P.lam_logit[t * P.units + u];
        lam = 1.f / (1.f + expf(-z));
      }
      named_barrier_sync(1, kSoftmaxThreads);  // all have read the scratch before D overwrites it
      merged = true;
    };

    // This thread's part of the D tile: row r, keys 32 wg .. 32 wg + 31 = 16-byte units
    // 4 (wg & 1) .. +3 of 64-key chunk wg / 2, in the 128B-swizzled K-major layout (unit u of a
    // row lands at u ^ (r % 8) within the row's 128 bytes).
    const uint32_t d_row = sD + (wg >> 1) * C::kChunk + r * 128;
    const int u0 = (wg & 1) * 4;

    // Pass-1 statistics over 32 scores v of one map: their sum of 2^(s c - ref), and their
    // maximum (times c).
    auto sum32 = [&](const uint32_t (&v)[KW], float ref) -> float {
      const uint64_t scale2 = f2pack(sl2, sl2), off2 = f2pack(-ref, -ref);
      uint64_t acc[2] = {f2pack(0.f, 0.f), f2pack(0.f, 0.f)};
#pragma unroll
      for (int i = 0; i < KW; i += 2) {
        float x0, x1;
        f2unpack(f2fma(f2pack(__uint_as_float(v[i]), __uint_as_float(v[i + 1])), scale2, off2),
                 x0, x1);
        acc[(i >> 1) & 1] = f2add(acc[(i >> 1) & 1], f2pack(ex2_approx(x0), ex2_approx(x1)));
      }
      float a0, a1, a2, a3;
      f2unpack(acc[0], a0, a1);
      f2unpack(acc[1], a2, a3);
      return (a0 + a1) + (a2 + a3);
    };
    auto max32 = [&](const uint32_t (&v)[KW]) -> float {
      float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int i = 0; i < KW; i += 2)
        mx[(i >> 1) & 3] = fmax3(mx[(i >> 1) & 3], __uint_as_float(v[i]), __uint_as_float(v[i + 1]));
      return fmax3(fmaxf(mx[0], mx[1]), mx[2], mx[3]) * sl2;
    };

    for (int t = 0; t < T; ++t) {
      if (W1 && t < n1) {
        // ---- pass 1 over 256-key tile t: keys [64 wg, 64 wg + 64) of each map, map by map ----
        // (statistics as in the 128-key form below: a sum against the reference point m, the
        // maximum only on a row's first tile with a visible key or when the sum passes 2^64)
        const int wkey0 = 2 * t * BN + 2 * KW * wg;
#pragma unroll
        for (int mp = 0; mp < 2; ++mp) {
          if (p1maps == 1 && mp != p1map0) continue;
          ok = mbar_wait(bar(bars.s_full[mp]), t & 1, abrt);
          if (__any_sync(0xffffffffu, !ok)) {
            ok = false;
            break;
          }
          tc_fence_after();
          uint32_t sw[2][KW];
          const uint32_t sb = tmem + tl + mp * 256 + 2 * KW * wg;
          tmem_ld32(sb, sw[0]);
          tmem_ld32(sb + KW, sw[1]);
          tmem_wait_ld();
          tc_fence_before();
          mbar_arrive(bar(bars.s_free[mp]));  // this map's scores are in registers
          if (wkey0 + 2 * KW > lim) {
#pragma unroll
            for (int i = 0; i < KW; ++i) {
              if (wkey0 + i >= lim) sw[0][i] = __float_as_uint(-INFINITY);
              if (wkey0 + KW + i >= lim) sw[1][i] = __float_as_uint(-INFINITY);
            }
          }
          __syncwarp();
          float sum = 0.f;
          bool redo = m[mp] == -INFINITY;
          if (!redo) {
            sum = sum32(sw[0], m[mp]) + sum32(sw[1], m[mp]);
            redo = sum > 0x1p64f;  // also true for +inf; a NaN score keeps its NaN
          }
          if (redo) {
            const float mn = fmaxf(m[mp], fmaxf(max32(sw[0]), max32(sw[1])));
            if (mn == -INFINITY) continue;  // every key so far is masked for this row
            sum = sum32(sw[0], mn) + sum32(sw[1], mn);
            l[mp] = l[mp] * ex2_approx(m[mp] - mn);
            m[mp] = mn;
          }
          l[mp] += sum;
        }
        if (!ok) break;
        continue;
      }
      const bool pass2 = t >= n1;
      if (pass2 && !merged) merge();
      const int buf = sbuf(t);
      const int key0 = (pass2 ? t - n1 : t) * BN + KW * wg;
      ok = mbar_wait(bar(bars.s_full[buf]), suse(t) & 1, abrt);
      if (__any_sync(0xffffffffu, !ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[2][KW];
      const uint32_t sb = tmem + tl + buf * 256 + KW * wg;
      tmem_ld32(sb, sr[0]);
      tmem_ld32(sb + 128, sr[1]);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(bar(bars.s_free[buf]));  // scores are in registers: the buffer is free
      if (key0 + KW > lim) {
#pragma unroll
        for (int i = 0; i < KW; ++i)
          if (key0 + i >= lim) {
            sr[0][i] = __float_as_uint(-INFINITY);
            sr[1][i] = __float_as_uint(-INFINITY);
          }
      }
      __syncwarp();
      if (!pass2) {
        // ---- pass 1: exact row max and row sum of each map (online over key tiles) ----
        // The sum is taken against the running maximum m (any reference point gives the same
        // statistics: b = m + log2 l); the tile's own maximum is found only on a row's first
        // tile with a visible key, or when a score so far above m overflows the sum.
        auto tile_sum = [&](int mp, float ref) -> float { return sum32(sr[mp], ref); };
        auto tile_max = [&](int mp) -> float { return max32(sr[mp]); };
#pragma unroll
        for (int mp = 0; mp < 2; ++mp) {
          float sum = 0.f;
          bool redo = m[mp] == -INFINITY;
          if (!redo) {
            sum = tile_sum(mp, m[mp]);
            redo = sum > 0x1p64f;  // also true for +inf; a NaN score keeps its NaN
          }
          if (redo) {
            const float mn = fmaxf(m[mp], tile_max(mp));
            if (mn == -INFINITY) continue;  // every key so far is masked for this row
            sum = tile_sum(mp, mn);
            l[mp] = l[mp] * ex2_approx(m[mp] - mn);
            m[mp] = mn;
          }
          l[mp] += sum;
        }
      } else {
        // ---- pass 2: D = A1 - lambda A2 in fp32, rounded once to bf16, into shared memory ----
        const int jv = t - n1;
        const uint64_t scale2 = f2pack(sl2, sl2), bias2 = f2pack(bias[0], bias[1]);
        const uint64_t nlam2 = f2pack(-lam, -lam);
        uint32_t pk[KW / 2];
#pragma unroll
        for (int i = 0; i < KW / 2; ++i) {
          float x1a, x2a, x1b, x2b;  // (map 1, map 2) of keys 2i and 2i+1
          f2unpack(f2fma(f2pack(__uint_as_float(sr[0][2 * i]), __uint_as_float(sr[1][2 * i])),
                         scale2, bias2),
                   x1a, x2a);
          f2unpack(f2fma(f2pack(__uint_as_float(sr[0][2 * i + 1]),
                                __uint_as_float(sr[1][2 * i + 1])),
                         scale2, bias2),
                   x1b, x2b);
          float da, db;
          f2unpack(f2fma(nlam2, f2pack(ex2_approx(x2a), ex2_approx(x2b)),
                         f2pack(ex2_approx(x1a), ex2_approx(x1b))),
                   da, db);
          pk[i] = pack_bf16x2(da, db);
        }
        // the previous D must have been consumed by its value MMA
        if (jv > 0) {
          ok = mbar_wait(bar(bars.d_empty), (jv - 1) & 1, abrt);
          if (__any_sync(0xffffffffu, !ok)) {
            ok = false;
            break;
          }
        }
#pragma unroll
        for (int uu = 0; uu < KW / 8; ++uu)
          st_shared_v4(d_row + (((u0 + uu) ^ (r & 7)) << 4), pk[4 * uu], pk[4 * uu + 1],
                       pk[4 * uu + 2], pk[4 * uu + 3]);
        // Packed or paged keys: the tile's rows past the sequence's keys hold other data (the next
        // sequence, padding, unused page rows) that may not be finite. Their D is 0, but 0 * NaN
        // would still reach O, so those V rows are zeroed before D is released to the V product.
        // Batched tiles past N are zero-filled by TMA.
        const int vkey0 = jv * BN;
        if ((KMODE != kKeysShared || P.cu_seqlens) && vkey0 + BN > SNk) {
          for (int h = 0; h < 2 && ok; ++h) {
            const int idx = v_load(jv, h);
            ok = mbar_wait(bar(bars.slot_full[idx % NSLOT]), (idx / NSLOT) & 1, abrt);
          }
          if (__any_sync(0xffffffffu, !ok)) {
            ok = false;
            break;
          }
          // thread (wg, r): key r of the tile (V half r / 64, row r % 64), 64-column chunks
          // wg, wg + 4, ... of that row
          if (vkey0 + r >= SNk) {
            const int vs = v_load(jv, r >> 6) % NSLOT;
            for (int c = wg; c < DV / 64; c += kNumWG) {
              const uint32_t vrow = sSlot + vs * C::kSlot + c * C::kVHalfChunk + (r & 63) * 128;
#pragma unroll
              for (int q = 0; q < 8; ++q) st_shared_v4(vrow + 16 * q, 0u, 0u, 0u, 0u);
            }
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(bar(bars.d_full));
      }
    }
    if (!merged) merge();
    if (gphase == 1) {
      // grouped, phase 1: the noise map's row statistic is this launch's only output
      if (ok && wg == 0 && row < P.N)
        P.gda_noise[(static_cast<size_t>(b) * (P.units / P.group) + u / P.group) * P.n_pad + row] =
            -bias[1];
      ok = false;  // no epilogue
    }
    if (ok) {
      ok = mbar_wait(bar(bars.o_full), 0, abrt);
      ok = !__any_sync(0xffffffffu, !ok);
    }
    tc_fence_after();
    // ------------------------------- epilogue -------------------------------------
    // Warpgroup wg owns columns [wg * dv/4, (wg+1) * dv/4) of each row; the RMSNorm sum of
    // squares is combined across the warpgroups (scratch = D buffer, idle after o_full).
    constexpr int HC = DV / kNumWG;
    constexpr int CW = HC >= 32 ? 32 : 16;
    const int c0 = wg * HC;
    auto ld_o = [&](int c, uint32_t (&o)[CW]) {
      if constexpr (CW == 32)
        tmem_ld32(tmem + tl + C::kOCol + c0 + CW * c, o);
      else
        tmem_ld16(tmem + tl + C::kOCol + c0 + CW * c, o);
      tmem_wait_ld();
    };
    float ss = 0.f;
    if (ok && (P.flags & 2)) {
#pragma unroll 1
      for (int c = 0; c < HC / CW; ++c) {
        uint32_t o[CW];
        ld_o(c, o);
#pragma unroll
        for (int i = 0; i < CW; ++i) ss = fmaf(__uint_as_float(o[i]), __uint_as_float(o[i]), ss);
      }
    }
    float scale = 1.f;
    if (P.flags & 2) {
      scratch[wg * BM + r] = ss;
      named_barrier_sync(1, kSoftmaxThreads);
      float tot = 0.f;
#pragma unroll
      for (int w = 0; w < kNumWG; ++w) tot += scratch[w * BM + r];
      scale = 1.f / sqrtf(tot / static_cast<float>(DV) + P.eps);
    }
    if (P.flags & 4) scale *= (1.f - P.lambda_init);
    if (ok) {
      // The warp's 32 rows x HC columns go through shared memory (the load ring, idle once the
      // last product is done), so that each store instruction writes whole 128-byte row pieces
      // instead of 32 scattered 16-byte ones.
      constexpr int RB = HC * 2;          // bytes of one row's slice
      constexpr int PIECES = RB / 16;     // 16-byte pieces per slice (8 at dv 256, 4 at dv 128)
      constexpr int RPI = 32 / PIECES;    // rows per store instruction
      static_assert(kSoftmaxThreads * RB <= C::NSLOT * C::kSlot, "staging fits in the ring");
      uint8_t* stage = smem + C::kSlotOff + (warp - kSoftmaxWarp0) * 32 * RB;
      const bool live = row < SN;
      const float* w = (P.flags & 2) && P.norm_w ? P.norm_w + c0 : nullptr;
#pragma unroll 1
      for (int c = 0; c < HC / CW; ++c) {
        uint32_t o[CW];
        ld_o(c, o);
#pragma unroll
        for (int g = 0; g < CW / 8; ++g) {
          uint4 pkt;
          uint32_t* pw = reinterpret_cast<uint32_t*>(&pkt);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int e = 8 * g + 2 * i;
            const float w0 = w ? w[CW * c + e] : 1.f;
            const float w1 = w ? w[CW * c + e + 1] : 1.f;
            pw[i] = pack_bf16x2(__uint_as_float(o[e]) * scale * w0,
                                __uint_as_float(o[e + 1]) * scale * w1);
          }
          const int piece = (CW * c + 8 * g) / 8;
          *reinterpret_cast<uint4*>(stage + lane * RB + ((piece ^ (lane & (PIECES - 1))) * 16)) = pkt;
        }
        if (live && dbg_index_ok(static_cast<long long>(orow),
                                 P.cu_seqlens ? P.total : 1LL * P.B * P.N)) {
          if (P.o_pre) {  // training: the head output before the norm and scale
            __nv_bfloat16* op = static_cast<__nv_bfloat16*>(P.o_pre) +
                                (orow * P.units + u) * DV + c0;
#pragma unroll
            for (int g = 0; g < CW / 8; ++g) {
              uint4 pkt;
              uint32_t* pw = reinterpret_cast<uint32_t*>(&pkt);
#pragma unroll
              for (int i = 0; i < 4; ++i)
                pw[i] = pack_bf16x2(__uint_as_float(o[8 * g + 2 * i]),
                                    __uint_as_float(o[8 * g + 2 * i + 1]));
              *reinterpret_cast<uint4*>(op + CW * c + 8 * g) = pkt;
            }
          }
        }
      }
      __syncwarp();
      __nv_bfloat16* out0 = static_cast<__nv_bfloat16*>(P.out) + c0;
#pragma unroll
      for (int it = 0; it < PIECES; ++it) {
        const int rr = it * RPI + lane / PIECES;   // row (lane of the warp) this lane stores
        const int pc = lane % PIECES;
        const size_t addr = __shfl_sync(0xffffffffu, static_cast<unsigned long long>(oaddr), rr);
        bool rlive = __shfl_sync(0xffffffffu, live ? 1 : 0, rr) != 0;
        if constexpr (kDebugChecks) {  // (every lane takes the shuffle)
          const long long rrow = static_cast<long long>(
              __shfl_sync(0xffffffffu, static_cast<unsigned long long>(orow), rr));
          if (rlive) rlive = dbg_index_ok(rrow, P.cu_seqlens ? P.total : 1LL * P.B * P.N);
        }
        const uint4 v = *reinterpret_cast<const uint4*>(stage + rr * RB + ((pc ^ (rr & (PIECES - 1))) * 16));
        if (rlive) *reinterpret_cast<uint4*>(out0 + addr + pc * 8) = v;
      }
      if (P.stats && wg == 0 && row < P.N) {
        float* st = P.stats + (static_cast<size_t>(b) * P.units + u) * 2 * P.n_pad + row;
        st[0] = -bias[0];
        st[P.n_pad] = -bias[1];
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
// 4-D bf16 map over [B, N, heads, cols] with a 64-col x 1 x box_rows x 1 box, 128-byte swizzle,
// zero fill out of bounds.
static bool make_map(CUtensorMap* m, const void* base, int cols, int heads, int N, int B,
                     const long long (&st)[3], int box_rows, char* err, size_t err_len,
                     int elt = 2) {
  cuuint64_t dims[4] = {(cuuint64_t)cols, (cuuint64_t)heads, (cuuint64_t)N, (cuuint64_t)B};
  // element strides (batch, token, head) -> byte strides of dims 1..3 (head, token, batch)
  cuuint64_t strides[3] = {(cuuint64_t)st[2] * elt, (cuuint64_t)st[1] * elt,
                           (cuuint64_t)st[0] * elt};
  cuuint32_t box[4] = {(cuuint32_t)(128 / elt), 1, (cuuint32_t)box_rows, 1};  // 128-byte rows
  const CUtensorMapDataType type = elt == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  return encode_tmap_4d(m, type, base, dims, strides, box, err, err_len);
}

template <int DQK, int DV, bool SHARED_K, bool QK8 = false, int KMODE = kKeysShared,
          bool GROUPED = false>
static cudaError_t launch_cfg(const Problem& p, cudaStream_t s, char* err, size_t err_len) {
  using C = Cfg<DQK, DV, SHARED_K, QK8>;
  CUtensorMap mq, mk, mv;
  // packed sequences: one batch row of `total` tokens; otherwise [B, N]
  const int mN = p.cu_seqlens ? p.total : p.N, mB = p.cu_seqlens ? 1 : p.B;
  // keys with offsets of their own, or the page pools as one [num_pages * page_size] axis
  const int mNk = KMODE == kKeysPaged    ? p.num_pages * p.page_size
                  : KMODE == kKeysOffset ? p.total_k
                                         : mN;
  if (!make_map(&mq, p.q, p.q_cols, p.q_heads, mN, mB, p.qs, BM, err, err_len, C::kQKElt) ||
      !make_map(&mk, p.k, p.k_cols, p.kv_heads, mNk, mB, p.ks, BN, err, err_len, C::kQKElt) ||
      !make_map(&mv, p.v, DV, v_heads(p), mNk, mB, p.vs, BN / 2, err, err_len))
    return cudaErrorInvalidValue;
  auto kern = prefill_exact_kernel<DQK, DV, SHARED_K, QK8, KMODE, GROUPED>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kDynSmem);
  if (e != cudaSuccess) return e;
  KParams kp;
  kp.p = p;
  kp.n_qt = (p.N + BM - 1) / BM;
  kp.scale_log2 = kLog2e * p.scale;
  {
    // K/V bytes one (batch, unit) pair streams; keep a group's K/V within 32 MB of L2. Measured
    // at the 3B-layer shape: with 32 MB DRAM reads equal q + k + v (303 MB), with 64 MB the
    // streamed queries and outputs evict K/V tiles that later query tiles read again (408 MB)
    const int nk = (p.cu_seqlens_k || p.block_table) ? p.max_seqlen_k : p.N;
    const double kv_bytes = static_cast<double>(nk) * (p.k_cols * C::kQKElt + DV * 2.0);
    long long g = static_cast<long long>((32.0 * 1024 * 1024) / (kv_bytes > 1 ? kv_bytes : 1));
    const long long bu = static_cast<long long>(p.B) * p.units;
    kp.group = static_cast<int>(g < 1 ? 1 : (g > bu ? bu : g));
  }
  // grouped phase 1: one CTA per (noise head, query tile)
  const int gunits = (GROUPED && p.gda_phase == 1) ? p.units / p.group : p.units;
  const long long items = static_cast<long long>(kp.n_qt) * p.B * gunits;
  if (items == 0) return cudaSuccess;
  kern<<<dim3(static_cast<unsigned>(items)), kThreads, C::kDynSmem, s>>>(mq, mk, mv, kp);
  return cudaGetLastError();
}

}  // namespace exact

cudaError_t status_prefill_exact(int* v) { return read_clear_status(v); }

cudaError_t launch_prefill_exact(const Problem& p, cudaStream_t s, char* err, size_t err_len) {
  if (p.mode == MODE_GDA) {  // grouped: batched, packed, keys of their own or paged
    if (p.qk_fp8) {  // fp8 scores: batched, one launch (each signal head forms its noise map)
      if (p.dqk != 128 || p.dv != 256 || p.cu_seqlens) return cudaErrorNotSupported;
      Problem q = p;
      q.gda_phase = 0;
      return exact::launch_cfg<128, 256, false, true, exact::kKeysShared, true>(q, s, err, err_len);
    }
    const bool koff = p.cu_seqlens && p.cu_seqlens_k;
    const bool paged = p.cu_seqlens && p.block_table;
    if (p.dqk == 128 && p.dv == 256) {
      auto launch = [&](const Problem& q) {
        return paged  ? exact::launch_cfg<128, 256, false, false, exact::kKeysPaged, true>(q, s, err, err_len)
               : koff ? exact::launch_cfg<128, 256, false, false, exact::kKeysOffset, true>(q, s, err, err_len)
                      : exact::launch_cfg<128, 256, false, false, exact::kKeysShared, true>(q, s, err, err_len);
      };
      if (!p.gda_noise) {
        Problem q = p;
        q.gda_phase = 0;
        return launch(q);
      }
      // two launches: the noise maps' statistics once per noise head, then the signal heads
      Problem q = p;
      q.n_pad = (p.N + exact::BM - 1) / exact::BM * exact::BM;
      q.gda_phase = 1;
      cudaError_t e = launch(q);
      if (e != cudaSuccess) return e;
      q.gda_phase = 2;
      return launch(q);
    }
    if (koff || paged) return cudaErrorNotSupported;
    if (p.dqk == 64 && p.dv == 128) {  // (one launch: the two-launch form needs d = 128)
      Problem q = p;
      q.gda_phase = 0;
      return exact::launch_cfg<64, 128, false, false, exact::kKeysShared, true>(q, s, err, err_len);
    }
  } else if (p.mode == MODE_V1) {
    if (p.qk_fp8) {
      if (p.dqk == 128 && p.dv == 256) return exact::launch_cfg<128, 256, false, true>(p, s, err, err_len);
      return cudaErrorNotSupported;
    }
    const bool koff = p.cu_seqlens && p.cu_seqlens_k;
    const bool paged = p.cu_seqlens && p.block_table;
    if (p.dqk == 128 && p.dv == 256)
      return paged  ? exact::launch_cfg<128, 256, false, false, exact::kKeysPaged>(p, s, err, err_len)
             : koff ? exact::launch_cfg<128, 256, false, false, exact::kKeysOffset>(p, s, err, err_len)
                    : exact::launch_cfg<128, 256, false>(p, s, err, err_len);
    if (p.dqk == 64 && p.dv == 128 && !paged)
      return koff ? exact::launch_cfg<64, 128, false, false, exact::kKeysOffset>(p, s, err, err_len)
                  : exact::launch_cfg<64, 128, false>(p, s, err, err_len);
  } else {
    const bool koff = p.cu_seqlens && p.cu_seqlens_k;
    const bool paged = p.cu_seqlens && p.block_table;
    if (p.dqk == 128 && p.dv == 128)
      return paged  ? exact::launch_cfg<128, 128, true, false, exact::kKeysPaged>(p, s, err, err_len)
             : koff ? exact::launch_cfg<128, 128, true, false, exact::kKeysOffset>(p, s, err, err_len)
                    : exact::launch_cfg<128, 128, true>(p, s, err, err_len);
    if (p.dqk == 64 && p.dv == 64 && !paged)
      return koff ? exact::launch_cfg<64, 64, true, false, exact::kKeysOffset>(p, s, err, err_len)
                  : exact::launch_cfg<64, 64, true>(p, s, err, err_len);
  }
  return cudaErrorNotSupported;
}

}  // namespace da
