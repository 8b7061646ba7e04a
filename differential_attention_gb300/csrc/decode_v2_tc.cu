// decode_v2_tc.cu -- DIFF V2 decode on the tensor cores (page "Differential Transformer:
// softmax can't say zero, so it subtracts", section "DIFF V2: what the authors changed"; page
// "Differential Transformer V2": decoding reads an unchanged baseline KV cache).
//
// The G = Hq / Hkv query heads of a GQA group share one KV head, so for one cache tile of 128
// keys the scores of all G heads are one skinny matrix product, and so is the output update:
//   S^T[128 keys x 16] = K_tile[128 x 128] . Q^T[128 x 16]      (heads padded to N = 16)
//   O^T[128 dims x 16] = V_tile^T[128 x 128 keys] . P^T[128 keys x 16]
// Both run as tcgen05.mma kind::f16 (M = 128, N = 16, bf16 operands, fp32 accumulators in TMEM).
// K_tile and Q are K-major 128-byte-swizzled tiles straight from TMA; V_tile^T is the same TMA
// tile read MN-major; P^T is written K-major by the softmax threads. Columns G..15 of S and O
// are computed from whatever the unused rows hold and are never read.
//
// Work: one item = (sequence b, KV head g, split s of the cache); a persistent grid of one CTA
// per SM takes items round-robin. Warp roles:
//   warp 0     TMA producer: Q of each item (G rows), then K and V tiles into a 3-stage ring
//              (for a paged cache with pages smaller than a tile: Q only)
//   warps 6-13 paged cache with pages smaller than a tile: gather K and V rows into the ring
//   warp 1     TMEM owner and MMA issuer: S_t, then O_{t-1} (so S_{t+1} overlaps softmax_t)
//   warps 2-5  softmax: thread r owns key r of the tile for S and dim r of the head for O;
//              per-head running max (exact, no lazy rescale), probabilities to P^T in bf16,
//              per-thread partial sums; the fp32 output accumulates in registers as
//              o = o * corr_t + O_t. At the end of an item they write one record per query head
//              (m, l, o[128]) in the layout the split-merge kernel of decode.cu reads.
// Keys past the item's end inside the last tile get probability 0; their V rows are zeroed in
// shared memory before the product, so cache contents beyond seqlens[b] are never used.
// Paged cache, page size a multiple of 128: a tile lies in one page and is one TMA box per
// 64-dim half, as for a contiguous cache. Other page sizes: TMA's cost per box makes one box per
// page slow for small pages, so gather warps copy the tile themselves: each looks up the pool
// rows of its 32 keys through the block table, then copies the rows with 16-byte cp.async into
// the same 128-byte-swizzled layout TMA would write.
// A page id outside the pool reads page 0 and, where the key is in use, flags DEV_BAD_INDEX.
// Every wait is bounded; a timeout flags DEV_TIMEOUT and all roles unwind without hanging.
#include <cuda.h>

#include <cstdio>

#include "internal.h"
#include "ptx.cuh"

namespace da {
namespace v2tc {

constexpr float kLog2e = 1.4426950408889634f;  // log2(e): scores are kept in base-2 units
constexpr int kD = 128;                    // head dim
constexpr int kTile = 128;                 // keys per tile
constexpr int kN = 16;                     // MMA N (query heads, padded)
constexpr int kStages = 3;                 // K/V ring depth
constexpr int kChunk = kTile * 128;        // one 64-dim box of a K or V tile: 16 KB
constexpr int kKV = 2 * kChunk;            // one K or V tile: 32 KB
constexpr int kQSlot = 2 * kN * 128;       // Q slot: two 64-dim boxes of 16 rows: 4 KB
constexpr int kPBuf = 2 * kN * 128;        // P^T buffer: two 64-key blocks of 16 rows: 4 KB
constexpr int kKOff = 0;
constexpr int kVOff = kKOff + kStages * kKV;
constexpr int kQOff = kVOff + kStages * kKV;
constexpr int kPOff = kQOff + 2 * kQSlot;
constexpr int kSmemUsed = kPOff + 2 * kPBuf;
constexpr int kDynSmem = kSmemUsed + 1024;  // + alignment slack
constexpr int kThreads = 448;
constexpr int kSoftmaxThreads = 128;
constexpr int kGatherWarp0 = 6;            // warps 6-13 gather K, V from a paged cache:
constexpr int kGatherWarps = 4;            // two teams of four warps, tiles taken in turn
constexpr int kGatherTeams = 2;
constexpr uint32_t kTmemCols = 64;         // S[2] at cols 0, 16; O[2] at cols 32, 48
constexpr int kRecStride = 2 + kD;         // floats per query head in a record
static_assert(kDynSmem <= 227 * 1024, "shared memory budget");

struct Barriers {
  uint64_t k_full[kStages], v_full[kStages], kv_empty[kStages];
  uint64_t q_full[2], q_empty[2];
  uint64_t s_full[2], s_empty[2], p_full[2], o_full[2], o_empty[2];
  uint64_t teardown;
};

struct Params {
  const int* seqlens;
  float* ws;
  int B, Lmax, Hq, Hkv, splits, chunk, n_items;
  float scale_log2;
  const int* block_table;  // paged: [B, max_pages]; null for a contiguous cache
  int page_size, max_pages, num_pages, box_rows;
  int gather;                       // paged, page size not a multiple of 128: warp 0 gathers
  const uint8_t* kpool;             // gather: pool bases and the bytes between keys (Hkv * 256)
  const uint8_t* vpool;
  size_t key_bytes;
  uint32_t ps_magic, ps_shift;      // j / page_size = (umulhi(j, magic) + j) >> shift
};

// Extents of the q, K and V tensor maps (the host builds them with these dimensions), for the
// debug-build checks of tile coordinates: q [B][Hq][128]; caches [B or 1][rows][Hkv][128].
__device__ __forceinline__ Ext4 q_ext(const Params& p, int elt) { return Ext4{kD, p.Hq, p.B, 1, elt}; }
__device__ __forceinline__ Ext4 kv_ext(const Params& p, int elt) {
  const bool paged = p.block_table != nullptr;
  return Ext4{kD, p.Hkv, paged ? p.num_pages * p.page_size : p.Lmax, paged ? 1 : p.B, elt};
}

__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
}
__device__ __forceinline__ float warp_max(float x) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}
// Barrier over `count` threads that also ANDs a predicate across them: every softmax thread
// passes the same sequence of these, failed or not, so a timeout seen by some threads ends the
// loop for all of them together.
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
__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

struct Item {
  int b, g, s, k0, k1, nt;
};
__device__ __forceinline__ Item item_of(const Params& p, int i) {
  Item it;
  it.s = i % p.splits;
  const int bg = i / p.splits;
  it.g = bg % p.Hkv;
  it.b = bg / p.Hkv;
  int L = p.seqlens ? p.seqlens[it.b] : p.Lmax;
  L = L < 1 ? 1 : (L > p.Lmax ? p.Lmax : L);
  it.k0 = it.s * p.chunk;
  it.k1 = min(it.k0 + p.chunk, L);
  it.nt = it.k1 > it.k0 ? (it.k1 - it.k0 + kTile - 1) / kTile : 0;
  return it;
}

// Pool row of key j of item `it` (paged cache). An entry past the block table's end reads page
// 0; so does one outside the pool, which flags DEV_BAD_INDEX when the key is in use.
__device__ __forceinline__ int page_row(const Params& p, const Item& it, int j) {
  const uint32_t uj = static_cast<uint32_t>(j);
  const uint32_t pi = (__umulhi(uj, p.ps_magic) + uj) >> p.ps_shift;
  int pg = 0;
  if (pi < static_cast<uint32_t>(p.max_pages)) {
    pg = __ldg(p.block_table + static_cast<size_t>(it.b) * p.max_pages + pi);
    if (pg < 0 || pg >= p.num_pages) {
      if (j < it.k1) flag_device_error(DEV_BAD_INDEX);
      pg = 0;
    }
  }
  return pg * p.page_size + static_cast<int>(uj - pi * static_cast<uint32_t>(p.page_size));
}

// K8: q and the K cache in fp8 e4m3 (scales folded into scale_log2). A K row or a Q row of 128
// elements is then one 128-byte swizzle atom: one TMA box a tile (the first 16 KB of the tile's
// 32 KB stage) and four kind::f8f6f4 k-steps for the scores; V and the output product are bf16.
template <int G, bool K8>
__global__ void __launch_bounds__(kThreads, 1)
    v2dec_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const Params p) {
  static_assert(G == 2 || G == 4 || G == 8, "group size");
  extern __shared__ uint8_t smem_raw[];
  __shared__ Barriers bars;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  __shared__ float red[2][4][8];
  __shared__ float lred[4][8];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sK = smem_u32(smem + kKOff), sV = smem_u32(smem + kVOff);
  const uint32_t sQ = smem_u32(smem + kQOff), sP = smem_u32(smem + kPOff);
  auto bar = [](uint64_t& x) { return smem_u32(&x); };

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(bar(bars.k_full[i]), p.gather ? kGatherWarps : 1);
      mbar_init(bar(bars.v_full[i]), p.gather ? kGatherWarps : 1);
      mbar_init(bar(bars.kv_empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(bars.q_full[i]), 1);
      mbar_init(bar(bars.q_empty[i]), 1);
      mbar_init(bar(bars.s_full[i]), 1);
      mbar_init(bar(bars.s_empty[i]), kSoftmaxThreads);
      mbar_init(bar(bars.p_full[i]), kSoftmaxThreads);
      mbar_init(bar(bars.o_full[i]), 1);
      mbar_init(bar(bars.o_empty[i]), kSoftmaxThreads);
    }
    mbar_init(bar(bars.teardown), 1);
    abort_flag = 0;
    fence_barrier_init();
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
  // Q rows G..15 and P^T rows G..15 are never written again: zero them so that the padded
  // columns of S and O are defined
  for (int i = threadIdx.x; i < (2 * kQSlot + 2 * kPBuf) / 16; i += kThreads)
    st_shared_v4(sQ + 16 * i, 0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  volatile int* abrt = &abort_flag;

  if (warp == 0 && p.gather) {
    // ======================= Q producer (the gather warps load K, V) =======================
    if (lane == 0) {
      int qi = 0;
      for (int i = blockIdx.x; i < p.n_items; i += gridDim.x) {
        const Item it = item_of(p, i);
        if (it.nt == 0) continue;
        const int qs = qi & 1;
        if (!mbar_wait(bar(bars.q_empty[qs]), ((qi >> 1) & 1) ^ 1, abrt)) break;
        mbar_arrive_expect_tx(bar(bars.q_full[qs]), (K8 ? 1 : 2) * G * 128);
        for (int c = 0; c < (K8 ? 1 : 2); ++c)
          tma_load_4d_chk(sQ + qs * kQSlot + c * (kN * 128), &tm_q, bar(bars.q_full[qs]), 64 * c,
                      it.g * G, it.b, 0, q_ext(p, K8 ? 1 : 2));
        ++qi;
      }
      for (int j = max(0, qi - 2); j < qi; ++j)
        mbar_wait(bar(bars.q_full[j & 1]), (j >> 1) & 1, nullptr);
    }
  } else if (warp >= kGatherWarp0) {
    // ====================== gathering producers (paged cache only) =======================
    // Tiles alternate between the two teams, so two tiles are in flight. Warp w of a team
    // copies keys 32w .. 32w + 31 of its tiles: lane l looks up the pool row of key 32w + l, then
    // each instruction copies two keys' 256-byte head rows (lanes 0-15 one key, lanes 16-31 the
    // next, 16 bytes a lane). A warp waits for its own copies, fences them for the tensor cores'
    // proxy and arrives on the tile's barrier (four arrivals complete it).
    if (p.gather) {
      const int gw = (warp - kGatherWarp0) % kGatherWarps;
      const int team = (warp - kGatherWarp0) / kGatherWarps;
      int n = 0;
      bool ok = true;
      const int kh = lane >> 4;
      const uint32_t ch = lane & 15;
      const uint32_t cdst = (ch >> 3) * kChunk, jc = ch & 7;
      for (int i = blockIdx.x; ok && i < p.n_items; i += gridDim.x) {
        const Item it = item_of(p, i);
        if (it.nt == 0) continue;
        const uint8_t* kg = p.kpool + static_cast<size_t>(it.g) * (2 * kD) + ch * 16;
        const uint8_t* vg = p.vpool + static_cast<size_t>(it.g) * (2 * kD) + ch * 16;
        for (int t = 0; t < it.nt; ++t, ++n) {
          if (n % kGatherTeams != team) continue;  // the other team's tile
          const int st = n % kStages;
          int row = page_row(p, it, it.k0 + t * kTile + 32 * gw + lane);
          if (!dbg_index_ok(row, 1LL * p.num_pages * p.page_size)) row = 0;
          // every lane waits: with lane 0 waiting alone and the others parked at a shuffle, the
          // warp resumed late enough to halve the throughput
          const bool w = mbar_wait(bar(bars.kv_empty[st]), ((n / kStages) & 1) ^ 1, abrt);
          if (!(ok = __all_sync(0xffffffffu, w))) break;
          const uint32_t dk = sK + st * kKV + cdst, dv = sV + st * kKV + cdst;
#pragma unroll
          for (int kk = 0; kk < 16; ++kk) {
            const int rl = 2 * kk + kh, r = 32 * gw + rl;
            const int rr = __shfl_sync(0xffffffffu, row, rl);
            cp_async16(dk + r * 128 + ((jc ^ (r & 7)) << 4),
                       kg + static_cast<size_t>(rr) * p.key_bytes);
          }
          cp_async_commit();
#pragma unroll
          for (int kk = 0; kk < 16; ++kk) {
            const int rl = 2 * kk + kh, r = 32 * gw + rl;
            const int rr = __shfl_sync(0xffffffffu, row, rl);
            cp_async16(dv + r * 128 + ((jc ^ (r & 7)) << 4),
                       vg + static_cast<size_t>(rr) * p.key_bytes);
          }
          cp_async_commit();
          cp_async_wait<0>();  // our part of the tile has landed: hand it over
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(bar(bars.k_full[st]));
            mbar_arrive(bar(bars.v_full[st]));
          }
        }
      }
      cp_async_wait<0>();  // nothing of ours may still be landing when the CTA exits
    }
  } else if (warp == 0) {
    // ================================ TMA producer ================================
    if (lane == 0) {
      int n = 0, qi = 0;
      bool ok = true;
      for (int i = blockIdx.x; ok && i < p.n_items; i += gridDim.x) {
        const Item it = item_of(p, i);
        if (it.nt == 0) continue;
        const int qs = qi & 1;
        if (!(ok = mbar_wait(bar(bars.q_empty[qs]), ((qi >> 1) & 1) ^ 1, abrt))) break;
        mbar_arrive_expect_tx(bar(bars.q_full[qs]), (K8 ? 1 : 2) * G * 128);
        for (int c = 0; c < (K8 ? 1 : 2); ++c)
          tma_load_4d_chk(sQ + qs * kQSlot + c * (kN * 128), &tm_q, bar(bars.q_full[qs]), 64 * c,
                      it.g * G, it.b, 0, q_ext(p, K8 ? 1 : 2));
        ++qi;
        for (int t = 0; t < it.nt; ++t, ++n) {
          const int st = n % kStages;
          const int key = it.k0 + t * kTile;
          // paged, page size a multiple of 128: the tile is rows row0 .. row0 + 127 of one page
          const int row0 = p.block_table ? page_row(p, it, key) : 0;
          if (!(ok = mbar_wait(bar(bars.kv_empty[st]), ((n / kStages) & 1) ^ 1, abrt))) break;
          mbar_arrive_expect_tx(bar(bars.k_full[st]), K8 ? kChunk : kKV);
          if (p.block_table) {
            for (int c = 0; c < (K8 ? 1 : 2); ++c)
              tma_load_4d_chk(sK + st * kKV + c * kChunk, &tm_k, bar(bars.k_full[st]), 64 * c, it.g,
                          row0, 0, kv_ext(p, K8 ? 1 : 2));
            mbar_arrive_expect_tx(bar(bars.v_full[st]), kKV);
            for (int c = 0; c < 2; ++c)
              tma_load_4d_chk(sV + st * kKV + c * kChunk, &tm_v, bar(bars.v_full[st]), 64 * c, it.g,
                          row0, 0, kv_ext(p, 2));
          } else {
            for (int c = 0; c < (K8 ? 1 : 2); ++c)
              tma_load_4d_chk(sK + st * kKV + c * kChunk, &tm_k, bar(bars.k_full[st]), 64 * c, it.g,
                          key, it.b, kv_ext(p, K8 ? 1 : 2));
            mbar_arrive_expect_tx(bar(bars.v_full[st]), kKV);
            for (int c = 0; c < 2; ++c)
              tma_load_4d_chk(sV + st * kKV + c * kChunk, &tm_v, bar(bars.v_full[st]), 64 * c, it.g,
                          key, it.b, kv_ext(p, 2));
          }
        }
      }
      // no copy of ours may still be landing when the CTA exits
      for (int j = max(0, qi - 2); j < qi; ++j)
        mbar_wait(bar(bars.q_full[j & 1]), (j >> 1) & 1, nullptr);
      for (int j = max(0, n - kStages); j < n; ++j) {
        mbar_wait(bar(bars.k_full[j % kStages]), (j / kStages) & 1, nullptr);
        mbar_wait(bar(bars.v_full[j % kStages]), (j / kStages) & 1, nullptr);
      }
    }
  } else if (warp == 1) {
    // ================================ MMA issuer ==================================
    if (lane == 0) {
      constexpr uint32_t idesc_s = K8 ? umma_idesc_e4m3(kTile, kN)   // A = K, B = Q: K-major
                                      : umma_idesc_bf16(kTile, kN, 0, 0);
      constexpr uint32_t idesc_o = umma_idesc_bf16(kD, kN, 1, 0);     // A = V^T MN-major
      const uint64_t dk0 = umma_smem_desc(sK, 16, 1024);
      const uint64_t dv0 = umma_smem_desc(sV, kChunk, 1024);  // LBO = stride of 64-dim boxes
      const uint64_t dq0 = umma_smem_desc(sQ, 16, 1024);
      const uint64_t dp0 = umma_smem_desc(sP, 16, 1024);
      int n = 0, qi = 0;
      bool ok = true;
      for (int i = blockIdx.x; ok && i < p.n_items; i += gridDim.x) {
        const Item it = item_of(p, i);
        if (it.nt == 0) continue;
        const int qs = qi & 1;
        if (!(ok = mbar_wait(bar(bars.q_full[qs]), (qi >> 1) & 1, abrt))) break;
        tc_fence_after();
        for (int t = 0; t <= it.nt; ++t) {
          if (t < it.nt) {
            const int nn = n + t, st = nn % kStages, sb = nn & 1;
            if (!(ok = mbar_wait(bar(bars.s_empty[sb]), ((nn >> 1) & 1) ^ 1, abrt))) break;
            if (!(ok = mbar_wait(bar(bars.k_full[st]), (nn / kStages) & 1, abrt))) break;
            tc_fence_after();
            const uint64_t kd = desc_add(dk0, st * kKV), qd = desc_add(dq0, qs * kQSlot);
            if constexpr (K8) {
#pragma unroll
              for (int k = 0; k < 4; ++k)  // 32 fp8 elements (32 bytes) a k-step
                mma_e4m3_ss(tmem + sb * kN, desc_add(kd, k * 32), desc_add(qd, k * 32), idesc_s,
                            k > 0 ? 1u : 0u);
            } else {
#pragma unroll
              for (int k = 0; k < kD / 16; ++k) {
                mma_bf16_ss(tmem + sb * kN, desc_add(kd, (k >> 2) * kChunk + (k & 3) * 32),
                            desc_add(qd, (k >> 2) * (kN * 128) + (k & 3) * 32), idesc_s,
                            k > 0 ? 1u : 0u);
              }
            }
            tc_commit(bar(bars.s_full[sb]));
            if (t == it.nt - 1) tc_commit(bar(bars.q_empty[qs]));
          }
          if (t >= 1) {
            const int pn = n + t - 1, st = pn % kStages, pb = pn & 1;
            if (!(ok = mbar_wait(bar(bars.p_full[pb]), (pn >> 1) & 1, abrt))) break;
            if (!(ok = mbar_wait(bar(bars.v_full[st]), (pn / kStages) & 1, abrt))) break;
            if (!(ok = mbar_wait(bar(bars.o_empty[pb]), ((pn >> 1) & 1) ^ 1, abrt))) break;
            tc_fence_after();
            const uint64_t vd = desc_add(dv0, st * kKV), pd = desc_add(dp0, pb * kPBuf);
#pragma unroll
            for (int k = 0; k < kTile / 16; ++k) {
              mma_bf16_ss(tmem + 2 * kN + pb * kN, desc_add(vd, k * 2048),
                          desc_add(pd, (k >> 2) * (kN * 128) + (k & 3) * 32), idesc_o,
                          k > 0 ? 1u : 0u);
            }
            tc_commit(bar(bars.o_full[pb]));
            tc_commit(bar(bars.kv_empty[st]));
          }
        }
        n += it.nt;
        ++qi;
      }
      tc_commit(bar(bars.teardown));
      mbar_wait(bar(bars.teardown), 0, nullptr);
    }
  } else {
    // ============================ softmax and output (warps 2-5) =================
    const int q4 = warp & 3;  // TMEM lane quarter this warp may access
    const int r = 32 * q4 + lane;
    const uint32_t tl = static_cast<uint32_t>(32 * q4) << 16;
    const float sl2 = p.scale_log2;
    // byte offset of P^T element (head h, key r) in a K-major 128-byte-swizzled buffer
    const uint32_t p_key = (r >> 6) * (kN * 128) + ((((r & 63) >> 3)) << 4) + (r & 7) * 2;
    int n = 0;
    bool ok = true;
    for (int i = blockIdx.x; ok && i < p.n_items; i += gridDim.x) {
      const Item it = item_of(p, i);
      float* rec = p.ws + ((static_cast<size_t>(it.b) * p.Hkv + it.g) * p.splits + it.s) *
                              (static_cast<size_t>(G) * kRecStride);
      if (it.nt == 0) {  // split past this sequence's end: an empty record
#pragma unroll
        for (int h = 0; h < G; ++h) {
          rec[h * kRecStride + 2 + r] = 0.f;
          if (r == 0) {
            rec[h * kRecStride] = -INFINITY;
            rec[h * kRecStride + 1] = 0.f;
          }
        }
        continue;
      }
      float m[G], ls[G], o[G], cprev[G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        m[h] = -INFINITY;
        ls[h] = 0.f;
        o[h] = 0.f;
        cprev[h] = 0.f;
      }
      for (int t = 0; t <= it.nt; ++t) {
        float corr[G];
        if (t < it.nt) {
          const int nn = n + t, sb = nn & 1, st = nn % kStages;
          const int key = it.k0 + t * kTile + r;
          const bool valid = key < it.k1;
          float x[G];
          bool good = ok && mbar_wait(bar(bars.s_full[sb]), (nn >> 1) & 1, abrt);
          good = __all_sync(0xffffffffu, good);
          if (good) {
            tc_fence_after();
            uint32_t sv[8];
            tmem_ld8(tmem + tl + sb * kN, sv);
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(bar(bars.s_empty[sb]));
#pragma unroll
            for (int h = 0; h < G; ++h) {
              x[h] = valid ? __uint_as_float(sv[h]) * sl2 : -INFINITY;
              const float wm = warp_max(x[h]);
              if (lane == 0) red[nn & 1][q4][h] = wm;
            }
            // last tile with keys past the item's end: zero their V rows so that cache contents
            // there (never initialised, possibly not finite) cannot reach the product
            if (it.k0 + (t + 1) * kTile > it.k1) {
              good = mbar_wait(bar(bars.v_full[st]), (nn / kStages) & 1, abrt);
              good = __all_sync(0xffffffffu, good);
              if (good && !valid) {
#pragma unroll
                for (int c = 0; c < 2; ++c)
#pragma unroll
                  for (int j = 0; j < 8; ++j)
                    st_shared_v4(sV + st * kKV + c * kChunk + r * 128 + 16 * j, 0u, 0u, 0u, 0u);
              }
            }
          }
          if (!(ok = bar_and(1, kSoftmaxThreads, good))) break;
#pragma unroll
          for (int h = 0; h < G; ++h) {
            const float tmax = fmaxf(fmaxf(red[nn & 1][0][h], red[nn & 1][1][h]),
                                     fmaxf(red[nn & 1][2][h], red[nn & 1][3][h]));
            const float mn = fmaxf(m[h], tmax);  // finite: every tile holds a valid key
            corr[h] = ex2_approx(m[h] - mn);
            const float pr = ex2_approx(x[h] - mn);
            ls[h] = fmaf(ls[h], corr[h], pr);
            m[h] = mn;
            const uint32_t a = sP + (nn & 1) * kPBuf + (h >> 3) * 1024 + (h & 7) * 128 +
                               (p_key ^ ((h & 7) << 4));
            st_shared_u16(a, __bfloat16_as_ushort(__float2bfloat16_rn(pr)));
          }
          fence_proxy_async_smem();
          mbar_arrive(bar(bars.p_full[nn & 1]));
        }
        if (t >= 1 && ok) {
          const int pn = n + t - 1, pb = pn & 1;
          bool good = mbar_wait(bar(bars.o_full[pb]), (pn >> 1) & 1, abrt);
          good = __all_sync(0xffffffffu, good);
          if (good) {
            tc_fence_after();
            uint32_t ov[8];
            tmem_ld8(tmem + tl + 2 * kN + pb * kN, ov);
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(bar(bars.o_empty[pb]));
#pragma unroll
            for (int h = 0; h < G; ++h) o[h] = fmaf(o[h], cprev[h], __uint_as_float(ov[h]));
          } else {
            ok = false;  // the next bar_and (tile or epilogue) ends the loop for everyone
          }
        }
        if (t < it.nt) {
#pragma unroll
          for (int h = 0; h < G; ++h) cprev[h] = corr[h];
        }
      }
      // ---- item epilogue: total sums, then the record ----
      bool good = ok;
      if (good) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float s = warp_sum(ls[h]);
          if (lane == 0) lred[q4][h] = s;
        }
      }
      if (!(ok = bar_and(1, kSoftmaxThreads, good))) break;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        rec[h * kRecStride + 2 + r] = o[h];
        if (r == h) {
          rec[h * kRecStride] = m[h];
          rec[h * kRecStride + 1] = lred[0][h] + lred[1][h] + lred[2][h] + lred[3][h];
        }
      }
      // lred is rewritten only after the next item's first tile barrier
      n += it.nt;
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
// 4-D bf16 map over a row-major [d3][d2][d1][128] tensor, box 64 x box1 x box2 x 1, 128-byte
// swizzle, zero fill out of bounds.
static bool make_map(CUtensorMap* m, const void* base, uint64_t d1, uint64_t d2, uint64_t d3,
                     uint32_t box1, uint32_t box2, char* err, size_t err_len) {
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(kD), d1, d2, d3};
  cuuint64_t strides[3] = {kD * 2ull, kD * 2ull * d1, kD * 2ull * d1 * d2};
  cuuint32_t box[4] = {64, box1, box2, 1};
  return encode_tmap_4d(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, dims, strides, box, err, err_len);
}

// The same map over fp8 (one byte an element): box 128 x box1 x box2 x 1, 128-byte rows.
static bool make_map8(CUtensorMap* m, const void* base, uint64_t d1, uint64_t d2, uint64_t d3,
                      uint32_t box1, uint32_t box2, char* err, size_t err_len) {
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(kD), d1, d2, d3};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(kD), kD * 1ull * d1, kD * 1ull * d1 * d2};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(kD), box1, box2, 1};
  return encode_tmap_4d(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, dims, strides, box, err, err_len);
}

static int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
    n = 152;
  return n;
}

template <int G, bool K8>
static cudaError_t launch_g(const V2DecodeArgs& a, int splits, int chunk, cudaStream_t st,
                            char* err, size_t err_len) {
  CUtensorMap mq, mk, mv;
  const bool paged = a.block_table != nullptr;
  const bool gather = paged && a.page_size % kTile != 0;
  // paged: the pools as one [num_pages * page_size, Hkv, 128] cache (the maps are not used when
  // warp 0 gathers)
  const uint64_t rows = paged ? static_cast<uint64_t>(a.num_pages) * a.page_size : a.Lmax;
  const uint32_t box_rows = gather ? 1u : kTile;
  const bool qk_ok =
      K8 ? make_map8(&mq, a.q, a.Hq, a.B, 1, G, 1, err, err_len) &&
               make_map8(&mk, a.k_cache, a.Hkv, rows, paged ? 1 : a.B, 1, box_rows, err, err_len)
         : make_map(&mq, a.q, a.Hq, a.B, 1, G, 1, err, err_len) &&
               make_map(&mk, a.k_cache, a.Hkv, rows, paged ? 1 : a.B, 1, box_rows, err, err_len);
  if (!qk_ok || !make_map(&mv, a.v_cache, a.Hkv, rows, paged ? 1 : a.B, 1, box_rows, err, err_len))
    return cudaErrorInvalidValue;
  auto kern = v2dec_tc_kernel<G, K8>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kDynSmem);
  if (e != cudaSuccess) return e;
  Params p;
  p.seqlens = a.seqlens;
  p.ws = a.ws;
  p.B = a.B;
  p.Lmax = a.Lmax;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.splits = splits;
  p.chunk = chunk;
  p.n_items = a.B * a.Hkv * splits;
  p.scale_log2 = kLog2e / sqrtf(static_cast<float>(kD)) * (K8 ? a.qk_descale : 1.f);
  p.block_table = a.block_table;
  p.page_size = a.page_size;
  p.max_pages = a.max_pages;
  p.num_pages = a.num_pages;
  p.box_rows = static_cast<int>(box_rows);
  p.gather = gather ? 1 : 0;
  p.kpool = static_cast<const uint8_t*>(a.k_cache);
  p.vpool = static_cast<const uint8_t*>(a.v_cache);
  p.key_bytes = static_cast<size_t>(a.Hkv) * kD * 2;
  p.ps_magic = p.ps_shift = 0;
  if (paged) page_magic(a.page_size, &p.ps_magic, &p.ps_shift);
  const int grid = min(p.n_items, sm_count());
  kern<<<grid, kThreads, kDynSmem, st>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

}  // namespace v2tc

int v2_decode_tc_splits(int B, int Lmax, int Hkv, int* chunk_out) {
  // About 32 items per SM, each a whole number of 128-key tiles between 2 and 16 tiles.
  const long long units = static_cast<long long>(B) * Hkv;
  const long long want = (32LL * 152 + units - 1) / units;
  long long chunk = (Lmax + want - 1) / want;
  chunk = (chunk + v2tc::kTile - 1) / v2tc::kTile * v2tc::kTile;
  if (chunk < 2 * v2tc::kTile) chunk = 2 * v2tc::kTile;
  if (chunk > 16 * v2tc::kTile) chunk = 16 * v2tc::kTile;
  if (chunk_out) *chunk_out = static_cast<int>(chunk);
  return static_cast<int>((Lmax + chunk - 1) / chunk);
}

cudaError_t status_v2_decode_tc(int* v) { return read_clear_status(v); }

cudaError_t launch_v2_decode_tc(const V2DecodeArgs& a, cudaStream_t st, char* err,
                                size_t err_len) {
  int chunk = 0;
  const int S = v2_decode_tc_splits(a.B, a.Lmax, a.Hkv, &chunk);
  const int G = a.Hq / a.Hkv;
  if (a.block_table && static_cast<long long>(a.num_pages) * a.page_size > 0x7fffffffLL)
    return cudaErrorNotSupported;
  // fp8 K rows are gathered by no warp: pages of fp8 K must be whole tiles
  if (a.k8 && a.block_table && a.page_size % v2tc::kTile != 0) return cudaErrorNotSupported;
  cudaError_t e;
  if (G == 8)
    e = a.k8 ? v2tc::launch_g<8, true>(a, S, chunk, st, err, err_len)
             : v2tc::launch_g<8, false>(a, S, chunk, st, err, err_len);
  else if (G == 4)
    e = a.k8 ? v2tc::launch_g<4, true>(a, S, chunk, st, err, err_len)
             : v2tc::launch_g<4, false>(a, S, chunk, st, err, err_len);
  else if (G == 2)
    e = a.k8 ? v2tc::launch_g<2, true>(a, S, chunk, st, err, err_len)
             : v2tc::launch_g<2, false>(a, S, chunk, st, err, err_len);
  else
    return cudaErrorNotSupported;
  if (e != cudaSuccess) return e;
  return launch_v2_combine(a, S, st);
}

}  // namespace da
