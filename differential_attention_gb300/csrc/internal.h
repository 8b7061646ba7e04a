// internal.h -- declarations shared by the library's translation units (not part of the ABI).
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace da {

enum Mode : int { MODE_V1 = 0, MODE_V2 = 1, MODE_GDA = 2 };

// One prefill problem, in the terms both prefill kernels (tensor-core and CUDA-core) use.
// A "unit" is one differential head (V1) or one pair of query heads (V2); each unit has two maps
// r = 0, 1 whose queries/keys are located by the helpers below.
//   V1: q [B,N,H,2d], k [B,N,H,2d], v [B,N,H,dv]; map r uses columns [r*d, r*d + d) of head h.
//   V2: q [B,N,Hq,d], k/v [B,N,Hkv,d]; map r uses query head 2p + r and KV head 2p / (Hq/Hkv).
//   GDA (grouped: Hs signal heads, Hn noise heads): q, k [B,N,Hs+Hn,d], v [B,N,Hs,dv]; map 0
//        uses head h of q and k, map 1 the noise head Hs + h / (Hs/Hn); V, lambda and the norm
//        are those of signal head h, as in V1.
struct Problem {
  const void* q;
  const void* k;
  const void* v;
  void* out;
  int B, N;
  int units;        // V1: H;  V2: Hq / 2;  GDA: Hs
  int dqk, dv;      // query/key width of one map, value width
  int mode;
  int q_heads;      // heads in the q tensor (V1: H, V2: Hq, GDA: Hs + Hn)
  int kv_heads;     // heads in the k (and, but for GDA, v) tensors (V1: H, V2: Hkv, GDA: Hs + Hn)
  int q_cols;       // elements per (token, head) row of q (V1: 2d, V2 and GDA: d)
  int k_cols;       // same for k
  int group;        // V2: Hq / Hkv (query heads per KV head); GDA: Hs / Hn; V1: 1
  const float* lambda;     // V1: [H]
  const float* lam_logit;  // V2: [B, N, Hq/2]
  const float* norm_w;     // [dv] or null (weight 1)
  float eps;
  float lambda_init;
  int flags;
  float scale;             // 1 / sqrt(dqk)
  // forward for training (V1, exact path): per row and map the base-2 log-sum-exp of the scaled
  // scores, [B, H, 2, n_pad]; and the head output before the norm and scale, [B, N, H, dv]
  float* stats;
  void* o_pre;
  int n_pad;
  // lambda formed inside the kernel (V1, exact path) from the re-parameterisation vectors
  // lq1, lk1, lq2, lk2 [lam_sets, lam_dim] (lam_sets 1: one lambda for every head); null: read
  // `lambda`. lambda_init is then that of the layer.
  const float* lam_vec[4];
  int lam_dim, lam_sets;
  // variable-length prefill (V1, exact path): sequences packed along the token axis of
  // q/k/v/out [total, H, *]; sequence b holds rows cu_seqlens[b] .. cu_seqlens[b+1]-1. N is then
  // the longest sequence (it sizes the grid) and `total` the packed length.
  const int* cu_seqlens;
  int total;
  // q and k in fp8 e4m3 (V1, exact path): the score products run as kind::f8f6f4; `scale`
  // then also carries the per-tensor dequantisation factors
  bool qk_fp8;
  // element strides (batch, token, head) of q, k, v and out; the last dimension is contiguous.
  // All zero: the dense layout (filled in by fill_dense_strides).
  long long qs[3], ks[3], vs[3], os[3];
  // keys with offsets of their own (null: the keys share cu_seqlens): sequence b's keys are rows
  // cu_seqlens_k[b] .. cu_seqlens_k[b+1]-1 of k/v [total_k, H, *], and its Lq queries are the
  // last Lq of its Lk >= Lq positions (causal: query i sees keys 0 .. Lk - Lq + i). Last in the
  // struct, so that adding them moved no other field of the kernels' parameters.
  const int* cu_seqlens_k;
  int total_k, max_seqlen_k;
  // paged keys (with cu_seqlens for the queries): sequence b has seqlens_k[b] keys, key r at row
  // r % page_size of page block_table[b * max_pages + r / page_size] of the pools k/v
  // [num_pages, page_size, H, *]; its queries are the last of those positions, as above
  const int* seqlens_k;
  const int* block_table;
  int page_size, max_pages, num_pages;
  // grouped form in two launches (exact path, d = 128): phase 1 computes each noise map's row
  // statistic (base-2 log-sum-exp of the scaled scores) once per noise head into gda_noise
  // [B, Hn, n_pad]; phase 2 runs the signal heads, whose first pass covers their own map only and
  // reads the noise map's statistic from gda_noise. Phase 0: one launch, each signal head's CTA
  // recomputing its noise map's statistics.
  int gda_phase;
  float* gda_noise;
};

// heads in the v tensor (and the output's units are Problem::units)
__host__ __device__ inline int v_heads(const Problem& p) {
  return p.mode == MODE_GDA ? p.units : p.kv_heads;
}

__host__ inline void fill_dense_strides(Problem& p) {
  if (p.qs[2] != 0) return;
  auto dense = [&](long long (&s)[3], int heads, int cols) {
    s[2] = cols;
    s[1] = static_cast<long long>(heads) * cols;
    s[0] = s[1] * p.N;
  };
  dense(p.qs, p.q_heads, p.q_cols);
  dense(p.ks, p.kv_heads, p.k_cols);
  dense(p.vs, v_heads(p), p.dv);
  dense(p.os, p.units, p.dv);
}
__host__ inline bool dense_strides(const Problem& p) {
  Problem d = p;
  d.qs[2] = 0;
  fill_dense_strides(d);
  for (int i = 0; i < 3; ++i)
    if (d.qs[i] != p.qs[i] || d.ks[i] != p.ks[i] || d.vs[i] != p.vs[i] || d.os[i] != p.os[i])
      return false;
  return true;
}
__host__ __device__ inline size_t elem_off(const long long (&s)[3], long long b, long long n,
                                           long long h) {
  return static_cast<size_t>(b * s[0] + n * s[1] + h * s[2]);
}

// TMA tensor map of 4 dimensions with 128-byte swizzle, 256-byte L2 promotion and zero fill out
// of bounds (tmap.cu); dims innermost first, byte strides of dims 1..3.
bool encode_tmap_4d(CUtensorMap* m, CUtensorMapDataType type, const void* base,
                    const cuuint64_t (&dims)[4], const cuuint64_t (&byte_strides)[3],
                    const cuuint32_t (&box)[4], char* err, size_t err_len);

// lambda = exp(lq1 . lk1) - exp(lq2 . lk2) + lambda_init for head u, from Problem::lam_vec.
// Called by a whole warp (lanes split the dot products); every lane gets the value.
__device__ inline float lambda_from_vectors_warp(const Problem& p, int u) {
  const int lane = threadIdx.x & 31;
  const int set = p.lam_sets == 1 ? 0 : u;
  const float* a = p.lam_vec[0] + static_cast<size_t>(set) * p.lam_dim;
  const float* b = p.lam_vec[1] + static_cast<size_t>(set) * p.lam_dim;
  const float* c = p.lam_vec[2] + static_cast<size_t>(set) * p.lam_dim;
  const float* d = p.lam_vec[3] + static_cast<size_t>(set) * p.lam_dim;
  float d1 = 0.f, d2 = 0.f;
  for (int i = lane; i < p.lam_dim; i += 32) {
    d1 = fmaf(__ldg(a + i), __ldg(b + i), d1);
    d2 = fmaf(__ldg(c + i), __ldg(d + i), d2);
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    d1 += __shfl_xor_sync(0xffffffffu, d1, o);
    d2 += __shfl_xor_sync(0xffffffffu, d2, o);
  }
  return expf(d1) - expf(d2) + p.lambda_init;
}

// grouped form: the Q and K head of map r of signal head u (map 1 in noise head u / group)
__host__ __device__ inline int grouped_head(const Problem& p, int u, int r) {
  return r == 0 ? u : p.units + u / p.group;
}
__host__ __device__ inline int q_head_of(const Problem& p, int u, int r) {
  return p.mode == MODE_V1 ? u : p.mode == MODE_V2 ? 2 * u + r : grouped_head(p, u, r);
}
__host__ __device__ inline int q_col_of(const Problem& p, int r) {
  return p.mode == MODE_V1 ? r * p.dqk : 0;
}
// the V head of unit u (and the K head of both maps in V1 and V2)
__host__ __device__ inline int kv_head_of(const Problem& p, int u) {
  return p.mode == MODE_V2 ? (2 * u) / p.group : u;
}
// the K head of map r of unit u
__host__ __device__ inline int k_head_of(const Problem& p, int u, int r) {
  return p.mode == MODE_GDA ? grouped_head(p, u, r) : kv_head_of(p, u);
}
__host__ __device__ inline int k_col_of(const Problem& p, int r) {
  return p.mode == MODE_V1 ? r * p.dqk : 0;
}

// Launchers. Each returns cudaSuccess or the launch error; `is_bf16` selects the storage type.
cudaError_t launch_lambda(const float* lq1, const float* lk1, const float* lq2, const float* lk2,
                          int dim, int n_sets, float lambda_init, float* out, cudaStream_t s);
cudaError_t launch_lambda_bwd(const float* lq1, const float* lk1, const float* lq2,
                              const float* lk2, const float* dlam, int dim, int n_sets,
                              int per_set, float* dlq1, float* dlk1, float* dlq2, float* dlk2,
                              cudaStream_t s);
cudaError_t launch_prefill_simt(const Problem& p, bool is_bf16, cudaStream_t s);
// Tensor-core prefill (bf16). Returns cudaErrorNotSupported for shapes it does not cover.
cudaError_t launch_prefill_tc(const Problem& p, cudaStream_t s, char* err, size_t err_len);
// DIFF V2 pair prefill, one flash pass per head, both heads of a pair in one CTA (dense bf16).
cudaError_t launch_prefill_v2(const Problem& p, cudaStream_t s, char* err, size_t err_len);
cudaError_t status_prefill_v2(int* v);

struct DecodeArgs {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int* seqlens;
  void* out;
  const float* lambda;
  float lambda_init;
  const float* norm_w;
  float eps;
  int flags;
  int B, Lmax, H, d, dv;
  float* ws;
  // paged cache (block_table non-null): k_cache / v_cache are pools [num_pages, page_size, H, *]
  // and key j of sequence b lives in page block_table[b * max_pages + j / page_size];
  // Lmax = max_pages * page_size
  const int* block_table;
  int page_size, max_pages, num_pages;
  // grouped form: H signal heads, signal head h subtracting noise head H + h / noise_group of
  // q [B, H + H/G, d] and the K cache [.., H + H/G, d]; 0: the V1 layout
  int noise_group;
};
int decode_splits(int B, int Lmax, int H, int* chunk_out);
size_t decode_workspace_bytes(int B, int Lmax, int H, int dv);
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s);  // contiguous or paged
cudaError_t status_decode(int* v);

// DIFF V2 decode: Hq query heads (pairs 2p, 2p+1) over an [B, Lmax, Hkv, 128] cache.
struct V2DecodeArgs {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int* seqlens;
  const float* lam_logit;
  void* out;
  int B, Lmax, Hq, Hkv;
  float* ws;
  // paged cache (block_table non-null): pools [num_pages, page_size, Hkv, 128], key j of sequence
  // b in page block_table[b * max_pages + j / page_size]; Lmax = max_pages * page_size
  const int* block_table;
  int page_size, max_pages, num_pages;
  // q and k_cache in fp8 e4m3: scores times qk_descale (the product of the two scales)
  bool k8;
  float qk_descale;
};
// j / page_size = (umulhi(j, magic) + j) >> shift for 0 <= j < 2^31 (division by an invariant
// integer, Granlund and Montgomery 1994)
void page_magic(int page_size, uint32_t* magic, uint32_t* shift);
int v2_decode_splits(int B, int Lmax, int Hkv, int* chunk_out);      // CUDA-core split kernel
int v2_decode_tc_splits(int B, int Lmax, int Hkv, int* chunk_out);   // tensor-core split kernel
size_t v2_decode_workspace_bytes(int B, int Lmax, int Hq, int Hkv);  // enough for either
cudaError_t launch_v2_decode(const V2DecodeArgs& a, cudaStream_t s);  // CUDA cores
cudaError_t launch_v2_decode_tc(const V2DecodeArgs& a, cudaStream_t s, char* err, size_t err_len);
cudaError_t launch_v2_combine(const V2DecodeArgs& a, int splits, cudaStream_t s);
cudaError_t status_v2_decode_tc(int* v);

// Prefill from host buffers with the copies pipelined against compute (host_pipeline.cu).
struct HostPipeArgs {
  const void* q;  // host [B, N, H, 2d]
  const void* k;  // host [B, N, H, 2d]
  const void* v;  // host [B, N, H, dv]
  void* out;      // host [B, N, H, dv]
  int B, N, H, d, dv;
  void* workspace;  // device, host_workspace_bytes()
  const float* lam_vec[4];
  int lam_dim, lam_sets, layer;
  const float* norm_w;
  float eps;
  int flags;
};
int host_chunk_sequences(int B, int N, int H);
int host_piece_rows(int N, int flags);  // rows per piece of the piecewise pipeline, 0: chunks
size_t host_workspace_bytes(int B, int N, int H, int d, int dv);
cudaError_t launch_host_pipeline(const HostPipeArgs& a, cudaStream_t stream,
                                 cudaError_t (*run)(const HostPipeArgs&, const void*, const void*,
                                                    const void*, void*, int, cudaStream_t, void*),
                                 cudaError_t (*run_piece)(const HostPipeArgs&, const void*,
                                                          const void*, const void*, void*, int,
                                                          int, const int*, const int*,
                                                          cudaStream_t, void*),
                                 void* ctx);

// Backward of the V1 prefill (d = 128, dv = 256, bf16).
struct BackwardArgs {
  const void* q;
  const void* k;
  const void* v;
  const void* o_pre;
  const float* stats;
  const void* dout;
  const float* lambda;
  float lambda_init;
  const float* norm_w;
  float eps;
  void* dq;
  void* dk;
  void* dv;
  float* dlambda;
  float* dnorm_w;
  int B, N, H, flags;
  void* workspace;
  // packed sequences (null: batched [B, N, H, *]): rows cu_seqlens[b] .. cu_seqlens[b+1]-1 of
  // [total, H, *]; N is then the longest sequence
  const int* cu_seqlens;
  int total;
  // grouped form (0: ungrouped): H is then the number of signal heads, q and k are
  // [B, N, H + n_noise, d] and v, out [B, N, H, dv]
  int n_noise;
};
// rows: B N (batched) or `total` (packed); N the (longest) sequence length; grouped: with room
// for the noise heads' dK accumulator
size_t backward_workspace_bytes(int B, int N, int H, long long rows, bool grouped = false);
cudaError_t launch_backward(const BackwardArgs& a, cudaStream_t s, char* err, size_t err_len);
cudaError_t status_backward(int* v);

// Decode whose split partials live in a fixed device array of this size (no workspace argument).
constexpr size_t kNoAllocScratchBytes = static_cast<size_t>(16) << 20;
long long decode_noalloc_max_units();  // largest B * H whose partials fit (one split each)
int decode_noalloc_splits(int B, int Lmax, int H, int* chunk_out);  // splits the no-alloc call runs
cudaError_t launch_decode_noalloc(const DecodeArgs& a, cudaStream_t s);

// Two-pass tensor-core prefill (A1 - lambda A2 formed in fp32 before rounding).
cudaError_t launch_prefill_exact(const Problem& p, cudaStream_t s, char* err, size_t err_len);

// Read and clear the device status word of a tensor-core prefill translation unit.
cudaError_t status_prefill_tc(int* v);
cudaError_t status_prefill_exact(int* v);
cudaError_t status_simt(int* v);

// Diagnostics: one kernel whose bounded wait (on a barrier nothing arrives on) runs out after
// limit_ms and sets the device status word of the CUDA-core translation unit.
cudaError_t launch_wait_timeout(int limit_ms, cudaStream_t s);

}  // namespace da
