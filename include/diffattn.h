/*
 * diffattn.h -- C ABI of the GB300 (sm_103a) differential-attention library (libdiffattn.so).
 *
 * The operator (page "Differential Transformer: softmax can't say zero, so it subtracts",
 * section "The mechanism, exactly", DiffAttn equation and the quoted MultiheadDiffAttn.forward):
 *
 *   DiffAttn = ( softmax(Q1 K1^T / sqrt(d)) - lambda * softmax(Q2 K2^T / sqrt(d)) ) V
 *
 * with V of width dv = 2d shared by both maps, followed per head by an RMSNorm over the dv
 * channels and a fixed multiply by (1 - lambda_init) (same page, section "The row no longer sums
 * to one"; page "Differential Transformer: Noise-Canceling Attention by Subtraction", section
 * "Making lambda learnable and stable").
 *
 * Conventions shared by every entry point
 *   - Pointers named "device" are caller-owned CUDA device memory; the library never allocates
 *     and never frees them. Host pointers are named "host".
 *   - Tensors are dense row-major with the layout given at each call (last dimension contiguous,
 *     no padding between rows). Every tensor pointer must be 16-byte aligned.
 *   - `stream` is a cudaStream_t (CUstream) passed as void*; NULL means the legacy default stream.
 *     Calls are asynchronous on that stream: a return of DIFFATTN_OK means the work was enqueued.
 *   - Every call returns 0 (DIFFATTN_OK) or a negative diffattn_status. Argument checks happen
 *     before anything is enqueued; on error nothing is launched and diffattn_last_error_string()
 *     (thread-local) describes the failure. Input values are not inspected: NaN/Inf propagate.
 *   - Kernels never trap. Every wait inside a kernel is bounded; a wait that runs out sets a
 *     device error flag and the kernel returns early, leaving the output undefined. Read the flag
 *     with diffattn_device_status().
 */
#ifndef DIFFATTN_H_
#define DIFFATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DIFFATTN_API __attribute__((visibility("default")))

typedef enum {
  DIFFATTN_OK = 0,
  DIFFATTN_ERR_ARG = -1,         /* null pointer, bad scalar or flag */
  DIFFATTN_ERR_SHAPE = -2,       /* unsupported or inconsistent sizes */
  DIFFATTN_ERR_DTYPE = -3,       /* dtype not supported by this entry point */
  DIFFATTN_ERR_ALIGN = -4,       /* a pointer is not 16-byte aligned */
  DIFFATTN_ERR_CUDA = -5,        /* a CUDA runtime/driver call failed (message has the code) */
  DIFFATTN_ERR_TIMEOUT = -6,     /* a kernel's bounded wait ran out (see diffattn_device_status) */
  DIFFATTN_ERR_UNSUPPORTED = -7, /* device is not sm_103 / sm_100 family */
  DIFFATTN_ERR_WORKSPACE = -8,   /* workspace missing or smaller than *_workspace_size */
  DIFFATTN_ERR_INDEX = -9        /* a device-side index (a block-table entry) was out of range */
} diffattn_status;

typedef enum { DIFFATTN_BF16 = 0, DIFFATTN_FP32 = 1 } diffattn_dtype;

/* flags */
#define DIFFATTN_CAUSAL 1 /* key j visible to query i iff j <= i (prefill, Nq = Nk, top-left) */
#define DIFFATTN_NORM 2   /* per-head RMSNorm over the dv channels: o / sqrt(mean(o^2) + eps) * w */
#define DIFFATTN_SCALE 4  /* multiply the (normed) head output by (1 - lambda_init) */
#define DIFFATTN_CUDA_CORES 8 /* prefill only: take the CUDA-core path (fp32 math, exact row
                                 statistics per map) instead of the tensor cores; for cross-checks */
#define DIFFATTN_SINGLE_PASS 16 /* prefill only: one flash pass per map on the tensor cores, each
   map's probabilities rounded to bf16 before the product with V (the numerics of running a flash
   kernel once per map and subtracting). Fewer exponentials, but when the two maps are close its
   error relative to the output grows like 2^-9 / |1 - lambda|. The default tensor-core path finds
   each map's exact row statistics first and rounds A1 - lambda A2 once, after the subtraction.
   For diffattn_v2_fwd, one pass per head is the default (see there). */
#define DIFFATTN_EXACT 32 /* V2 prefills (diffattn_v2_fwd, _varlen, _paged) only: find each head's
   exact row statistics first and round attn[2p] - sigmoid(lam) * attn[2p+1] once, after the
   subtraction (the V1 default path), instead of one flash pass per head. */

/* Library version (major * 10000 + minor * 100 + patch). */
DIFFATTN_API int diffattn_version(void);

/* Thread-local description of the last error returned on this thread ("" if none). The string is
 * owned by the library and valid until the next call on the same thread. */
DIFFATTN_API const char* diffattn_last_error_string(void);

/* Synchronises `stream`, then reads and clears the device error flags that kernels set.
 * Returns DIFFATTN_OK, DIFFATTN_ERR_TIMEOUT (a bounded wait ran out since the last call),
 * DIFFATTN_ERR_INDEX (device-side offsets were out of range: a paged decode met a block-table
 * entry outside [0, num_pages), and read page 0 instead; or a varlen prefill met a sequence
 * outside [0, total), and skipped it; that call's output is invalid), or DIFFATTN_ERR_CUDA.
 * In the debug build of the library (libdiffattn_debug.so, compiled with -DDIFFATTN_DEBUG) every
 * kernel also checks each tile coordinate of its TMA copies and each row it gathers or stores
 * against the extent of its tensor; a failed check clamps the copy into the tensor (or skips the
 * load or store) and is reported here as DIFFATTN_ERR_INDEX. The release library has no such
 * checks. */
DIFFATTN_API int diffattn_device_status(void* stream);

/* Diagnostics (not part of the method): launch one kernel whose bounded wait is certain to run
 * out -- it waits on a barrier that nothing arrives on -- after `limit_ms` (1..2000). The kernel
 * then sets the device status word and returns; it neither faults nor traps, and the context
 * stays usable. The next diffattn_device_status() reports DIFFATTN_ERR_TIMEOUT (once). Use it to
 * check that failure detection reaches the host. Errors: ERR_ARG, ERR_UNSUPPORTED, ERR_CUDA. */
DIFFATTN_API int diffattn_selftest_wait_timeout(int limit_ms, void* stream);

/* ------------------------------------------------------------------------------------------
 * lambda
 * Page "Differential Transformer: softmax can't say zero, so it subtracts", section "lambda,
 * re-parameterised": lambda = exp(lq1 . lk1) - exp(lq2 . lk2) + lambda_init, with
 * lambda_init(l) = 0.8 - 0.6 * exp(-0.3 * (l - 1)) for the 1-indexed layer l (also page
 * "Differential Transformer: Noise-Canceling Attention by Subtraction", section "Making lambda
 * learnable and stable").
 * ------------------------------------------------------------------------------------------ */

/* lambda_init for 1-indexed layer `layer` (>= 1). Host function; returns NaN for layer < 1. */
DIFFATTN_API float diffattn_lambda_init(int layer);

/* lambda for `n_sets` independent sets of four vectors.
 *   lq1, lk1, lq2, lk2 : device fp32 [n_sets, dim] each
 *   lambda_out         : device fp32 [n_sets]
 * The dot products and exponentials are taken in fp32. One set per layer (shared by every head)
 * is the page's reading; pass n_sets = H for one lambda per head.
 * Errors: ERR_ARG (null pointer, layer < 1), ERR_SHAPE (dim < 1 or > 4096, n_sets < 1). */
DIFFATTN_API int diffattn_lambda(const float* lq1, const float* lk1, const float* lq2,
                                 const float* lk2, int dim, int n_sets, int layer,
                                 float* lambda_out, void* stream);

/* Gradients of lambda with respect to its four vectors (training; the chain rule through the
 * re-parameterisation): for set s, g = dlambda[s * per_set] + ... + dlambda[s * per_set +
 * per_set - 1], e_m = exp(lq_m . lk_m), and
 *   dlq1 = g e1 lk1,  dlk1 = g e1 lq1,  dlq2 = -g e2 lk2,  dlk2 = -g e2 lq2.
 * per_set = H sums the per-head dlambda of diffattn_bwd into one lambda per layer; per_set = 1
 * with n_sets = H is one lambda per head.
 *   lq1 .. lk2 : device fp32 [n_sets, dim];  dlambda : device fp32 [n_sets * per_set]
 *   dlq1 .. dlk2 : device fp32 [n_sets, dim] (overwritten)
 * Errors: ERR_ARG, ERR_SHAPE, ERR_ALIGN, ERR_CUDA. */
DIFFATTN_API int diffattn_lambda_bwd(const float* lq1, const float* lk1, const float* lq2,
                                     const float* lk2, const float* dlambda, int dim, int n_sets,
                                     int per_set, float* dlq1, float* dlk1, float* dlq2,
                                     float* dlk2, void* stream);

/* ------------------------------------------------------------------------------------------
 * Prefill: DiffAttn over N tokens (causal or full), then the per-head epilogue.
 *   q      : device [B, N, H, 2d]  = [Q1 | Q2] per head
 *   k      : device [B, N, H, 2d]  = [K1 | K2] per head
 *   v      : device [B, N, H, dv]  (dv = 2d: one V shared by both maps)
 *   out    : device [B, N, H, dv]  (same dtype as the inputs)
 *   lambda : device fp32 [H]       (broadcast one value to all heads for one lambda per layer)
 *   lambda_init : used only with DIFFATTN_SCALE
 *   norm_weight : device fp32 [dv], or NULL for weight 1 (used only with DIFFATTN_NORM)
 *   eps    : RMSNorm epsilon (> 0 with DIFFATTN_NORM)
 *   flags  : DIFFATTN_CAUSAL | DIFFATTN_NORM | DIFFATTN_SCALE, optionally DIFFATTN_CUDA_CORES
 *            or DIFFATTN_SINGLE_PASS
 *   dtype  : DIFFATTN_BF16 (tensor-core path, fp32 accumulation and softmax) or DIFFATTN_FP32
 *            (CUDA-core fp32 path)
 * Supported: d in {64, 128}, dv = 2d, N >= 1, B, H >= 1. The 1/sqrt(d) scale uses d = width of
 * one query/key half.
 * Errors: ERR_ARG, ERR_SHAPE, ERR_DTYPE, ERR_ALIGN, ERR_UNSUPPORTED, ERR_CUDA.
 * ------------------------------------------------------------------------------------------ */
DIFFATTN_API int diffattn_fwd(const void* q, const void* k, const void* v, void* out,
                              const float* lambda, float lambda_init, const float* norm_weight,
                              float eps, int B, int N, int H, int d, int dv, int flags, int dtype,
                              void* stream);

/* ------------------------------------------------------------------------------------------
 * Decode: one query per sequence against its KV cache, split over the cache length and merged.
 * Page "Differential Transformer V2": V1 decoding with stock kernels loads the value cache twice;
 * this call reads every cached K and V element once for both maps.
 *   q       : device [B, H, 2d]          = [Q1 | Q2]
 *   k_cache : device [B, Lmax, H, 2d]    = [K1 | K2]
 *   v_cache : device [B, Lmax, H, dv]
 *   seqlens : device int32 [B], 1 <= seqlens[b] <= Lmax (keys 0 .. seqlens[b]-1 are attended,
 *             no mask inside that range), or NULL for Lmax everywhere. Values are not checked on
 *             the host; an entry outside [1, Lmax] is clamped into it on the device.
 *   out     : device [B, H, dv]
 *   lambda  : device fp32 [H];  lambda_init, norm_weight, eps, flags: as for diffattn_fwd
 *             (DIFFATTN_CAUSAL is ignored)
 *   workspace, ws_bytes : device scratch of at least diffattn_decode_workspace_size() bytes,
 *             256-byte aligned; contents need not be initialised. It must not be shared with a
 *             call that can run at the same time.
 * Supported: dtype DIFFATTN_BF16, d = 128, dv = 256.
 * Errors: as diffattn_fwd, plus ERR_WORKSPACE.
 * ------------------------------------------------------------------------------------------ */
DIFFATTN_API int diffattn_decode_workspace_size(int B, int Lmax, int H, int d, int dv,
                                                size_t* bytes);
DIFFATTN_API int diffattn_decode(const void* q, const void* k_cache, const void* v_cache,
                                 const int* seqlens, void* out, const float* lambda,
                                 float lambda_init, const float* norm_weight, float eps, int B,
                                 int Lmax, int H, int d, int dv, int flags, int dtype,
                                 void* workspace, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------------------------
 * Decode that allocates nothing (the paper has no counterpart: this is a deployment aid).
 * For callers that cannot allocate device memory where they decode -- a plugin inside a host
 * runtime that owns every device buffer and hands out no allocator, or a latency-bound decode
 * loop that may not call cudaMalloc / cudaFree because they can synchronise the device. The
 * arguments and the result are those of diffattn_decode without workspace / ws_bytes; the split
 * partials go to a scratch array built into the library (DIFFATTN_DECODE_NOALLOC_SCRATCH_BYTES,
 * held on every GPU that loads the library until the process exits).
 *   Limit: B * H <= DIFFATTN_DECODE_NOALLOC_SCRATCH_BYTES / 2064 (= 8128); larger calls return
 *   DIFFATTN_ERR_SHAPE. Where B * H * (diffattn_decode's split count) records of 2064 bytes
 *   would not fit, the cache is cut into fewer, longer slices (diffattn_decode_split_count
 *   reports both counts); the result then agrees with diffattn_decode to rounding. Otherwise
 *   both calls run the same kernels on the same slices and agree bit for bit.
 *   The first call on each device looks up the array's device address (cudaGetSymbolAddress,
 *   with that device current); make that first call before any stream capture. The address
 *   belongs to the device's current context: a call made after that context was destroyed and
 *   recreated in this process (cudaDeviceReset) looks it up again.
 *   All calls on a device share the array: calls that can run at the same time (on other
 *   streams) race on it, so keep them ordered. No call depends on what an earlier call left
 *   there. It calls no allocator (cudaMalloc, cudaFree or any library that allocates).
 * ------------------------------------------------------------------------------------------ */
#define DIFFATTN_DECODE_NOALLOC_SCRATCH_BYTES (16u << 20)
DIFFATTN_API int diffattn_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                         const int* seqlens, void* out, const float* lambda,
                                         float lambda_init, const float* norm_weight, float eps,
                                         int B, int Lmax, int H, int d, int dv, int flags,
                                         int dtype, void* stream);

/* ------------------------------------------------------------------------------------------
 * How many slices of the cache a decode of B sequences x H heads over Lmax keys is split into:
 * by diffattn_decode (noalloc = 0) or by diffattn_decode_noalloc (noalloc = 1). Host-only
 * arithmetic (no device is touched), so a caller can tell whether the two calls will agree bit
 * for bit (equal counts) or to rounding (the no-allocation call lowered its count).
 *   splits, chunk_keys : host int out-parameters: the slice count and keys per slice.
 * Errors: ERR_ARG (null pointer), ERR_SHAPE (B, Lmax or H < 1, or noalloc = 1 with B * H above
 * the no-allocation limit).
 * ------------------------------------------------------------------------------------------ */
DIFFATTN_API int diffattn_decode_split_count(int B, int Lmax, int H, int noalloc, int* splits,
                                             int* chunk_keys);

/* ------------------------------------------------------------------------------------------
 * DIFF V2 prefill (page "Differential Transformer: softmax can't say zero, so it subtracts",
 * section "DIFF V2: what the authors changed"; page "Differential Transformer V2"): softmax
 * attention of 2h query heads over GQA KV heads, then out_p = attn[2p] - sigmoid(lam) * attn[2p+1]
 * per token and pair; no per-head norm and no lambda_init.
 *   q         : device [B, N, Hq, d]; pair p = query heads (2p, 2p+1)
 *   k, v      : device [B, N, Hkv, d]; query heads of one GQA group are contiguous, so pair p
 *               reads KV head floor(2p / (Hq / Hkv))
 *   lam_logit : device fp32 [B, N, Hq/2], the value before the sigmoid
 *   out       : device [B, N, Hq/2, d]
 *   flags     : DIFFATTN_CAUSAL or 0, optionally one of DIFFATTN_CUDA_CORES, DIFFATTN_EXACT
 * Numerics: by default each head of a pair is one flash pass on the tensor cores, as the pages run
 * it (two stock attention calls): its probabilities are rounded to bf16 before the product with V,
 * the two normalised head outputs are subtracted in fp32. DIFFATTN_EXACT takes the two-pass kernel
 * that rounds the difference of the maps once instead; DIFFATTN_SINGLE_PASS is the default here.
 * Supported: dtype DIFFATTN_BF16, d in {64, 128}, Hq even, Hq % Hkv == 0 and (Hq / Hkv) even (the
 * two heads of a pair must sit in one GQA group). The scale is 1/sqrt(d).
 * Errors: ERR_ARG, ERR_SHAPE, ERR_DTYPE, ERR_ALIGN, ERR_UNSUPPORTED, ERR_CUDA.
 * ------------------------------------------------------------------------------------------ */
/* ------------------------------------------------------------------------------------------
 * Decode over a paged KV cache: diffattn_decode with the cache held in fixed-size pages of a
 * shared pool (the pages give no cache layout; this is the usual serving layout, and the method
 * is unchanged: key j of sequence b is row j % page_size of page block_table[b][j / page_size]).
 *   k_pool : device [num_pages, page_size, H, 2d] = [K1 | K2]
 *   v_pool : device [num_pages, page_size, H, dv]
 *   block_table : device int32 [B, max_pages]; entries for keys < seqlens[b] must be in
 *            [0, num_pages) (checked on the device: see DIFFATTN_ERR_INDEX); the rest are not read
 *   seqlens : device int32 [B], required, in [1, max_pages * page_size] (clamped on the device)
 *   other arguments and the workspace: as diffattn_decode, with
 *   diffattn_decode_workspace_size(B, max_pages * page_size, H, d, dv)
 * Supported: dtype DIFFATTN_BF16, d = 128, dv = 256, page_size >= 1.
 * Errors: as diffattn_decode.
 * ------------------------------------------------------------------------------------------ */
DIFFATTN_API int diffattn_decode_paged(const void* q, const void* k_pool, const void* v_pool,
                                       const int* block_table, const int* seqlens, void* out,
                                       const float* lambda, float lambda_init,
                                       const float* norm_weight, float eps, int B, int H, int d,
                                       int dv, int num_pages, int page_size, int max_pages,
                                       int flags, int dtype, void* workspace, size_t ws_bytes,
                                       void* stream);

DIFFATTN_API int diffattn_v2_fwd(const void* q, const void* k, const void* v,
                                 const float* lam_logit, void* out, int B, int N, int Hq, int Hkv,
                                 int d, int flags, int dtype, void* stream);

/* ------------------------------------------------------------------------------------------
 * DIFF V2 decode (page "Differential Transformer: softmax can't say zero, so it subtracts",
 * section "DIFF V2: what the authors changed"; page "Differential Transformer V2": the KV cache
 * is a baseline Transformer's, so decoding reads it as a baseline does). One query token per
 * sequence: softmax attention of each of the Hq query heads over its GQA KV head's cached keys
 * 0 .. seqlens[b]-1, then out_p = attn[2p] - sigmoid(lam_logit[b, p]) * attn[2p+1]. Every cached
 * K and V element is read once for all Hq / Hkv query heads of its group.
 *   q         : device [B, Hq, d]; pair p = query heads (2p, 2p+1)
 *   k_cache, v_cache : device [B, Lmax, Hkv, d]; query head h reads KV head h / (Hq / Hkv)
 *   seqlens   : device int32 [B] in [1, Lmax], or NULL for Lmax everywhere (clamped on the
 *               device as for diffattn_decode)
 *   lam_logit : device fp32 [B, Hq/2], the value before the sigmoid
 *   out       : device [B, Hq/2, d]
 *   flags     : 0 runs the tensor-core kernel; DIFFATTN_CUDA_CORES the CUDA-core one (same
 *               result up to rounding order); DIFFATTN_CAUSAL is accepted and ignored
 *   workspace, ws_bytes : device scratch of at least diffattn_v2_decode_workspace_size() bytes,
 *               256-byte aligned, not shared with a call that can run at the same time.
 * Supported: dtype DIFFATTN_BF16, d = 128, Hq / Hkv in {2, 4, 8}. The scale is 1/sqrt(d).
 * Errors: ERR_ARG, ERR_SHAPE, ERR_DTYPE, ERR_ALIGN, ERR_WORKSPACE, ERR_UNSUPPORTED, ERR_CUDA.
 * ------------------------------------------------------------------------------------------ */
DIFFATTN_API int diffattn_v2_decode_workspace_size(int B, int Lmax, int Hq, int Hkv, int d,
                                                   size_t* bytes);
DIFFATTN_API int diffattn_v2_decode(const void* q, const void* k_cache, const void* v_cache,
                                    const int* seqlens, const float* lam_logit, void* out, int B,
                                    int Lmax, int Hq, int Hkv, int d, int flags, int dtype,
                                    void* workspace, size_t ws_bytes, void* stream);

/* DIFF V2 decode with q and the K cache in fp8 e4m3 (page "Differential Transformer: softmax
 * can't say zero, so it subtracts", on quantized attention logits): the scores come from
 * fp8 x fp8 tensor-core products, scaled by q_descale * k_descale / sqrt(d); V stays bf16. A
 * cached key then costs 3/4 of the bf16 cache's bytes.
 *   q8 : device e4m3 [B, Hq, d] (q ~ q8 * q_descale);  k_cache8 : device e4m3 [B, Lmax, Hkv, d]
 *   (k ~ k_cache8 * k_descale);  v_cache : device bf16 [B, Lmax, Hkv, d]
 *   q_descale, k_descale : per-tensor scales, finite and > 0
 * Other arguments (the workspace included) as diffattn_v2_decode; flags: 0 or DIFFATTN_CAUSAL
 * (ignored). Errors: ERR_ARG, ERR_SHAPE, ERR_ALIGN, ERR_WORKSPACE, ERR_UNSUPPORTED, ERR_CUDA. */
DIFFATTN_API int diffattn_v2_decode_fp8(const void* q8, const void* k_cache8, const void* v_cache,
                                        const int* seqlens, const float* lam_logit, void* out,
                                        float q_descale, float k_descale, int B, int Lmax, int Hq,
                                        int Hkv, int d, int flags, void* workspace,
                                        size_t ws_bytes, void* stream);

/* DIFF V2 decode with fp8 e4m3 q and K over a paged cache: the result of diffattn_v2_decode_fp8
 * where key j of sequence b sits at row j % page_size of page block_table[b * max_pages +
 * j / page_size], as in diffattn_v2_decode_paged.
 *   q8 : device e4m3 [B, Hq, d];  k_pool8 : device e4m3 [num_pages, page_size, Hkv, d];
 *   v_pool : device bf16 [num_pages, page_size, Hkv, d]
 *   block_table, seqlens (required), workspace : as for diffattn_v2_decode_paged
 *   q_descale, k_descale, lam_logit, out, flags : as for diffattn_v2_decode_fp8
 * Supported: page_size a multiple of 128 (each 128-key tile is one TMA box of a page; other page
 * sizes: ERR_UNSUPPORTED). A used block-table entry outside [0, num_pages) reads page 0 and makes
 * the next diffattn_device_status() report DIFFATTN_ERR_INDEX.
 * Errors: ERR_ARG, ERR_SHAPE, ERR_ALIGN, ERR_WORKSPACE, ERR_UNSUPPORTED, ERR_CUDA. */
DIFFATTN_API int diffattn_v2_decode_fp8_paged(const void* q8, const void* k_pool8,
                                              const void* v_pool, const int* block_table,
                                              const int* seqlens, const float* lam_logit,
                                              void* out, float q_descale, float k_descale, int B,
                                              int Hq, int Hkv, int d, int num_pages, int page_size,
                                              int max_pages, int flags, void* workspace,
                                              size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------------------------
 * DIFF V2 decode over a paged KV cache: the result of diffattn_v2_decode where key j of
 * sequence b sits at row j % page_size of page block_table[b * max_pages + j / page_size].
 *   k_pool, v_pool : device [num_pages, page_size, Hkv, d]
 *   block_table    : device int32 [B, max_pages]; only entries for keys < seqlens[b] are used
 *   seqlens        : device int32 [B] (required), clamped to [1, max_pages * page_size]
 *   q, lam_logit, out, flags : as for diffattn_v2_decode
 *   workspace, ws_bytes : at least diffattn_v2_decode_workspace_size(B, max_pages * page_size,
 *                    Hq, Hkv, d) bytes, 256-byte aligned.
 * Any page size >= 1 (multiples of 128 read each tile of 128 keys as TMA boxes, others gather
 * the keys' rows one by one). A used block-table entry outside [0, num_pages) reads page 0
 * instead and makes the next diffattn_device_status() report DIFFATTN_ERR_INDEX; that call's
 * output is then invalid.
 * Errors: ERR_ARG, ERR_SHAPE (max_pages * page_size > 2^30 or num_pages * page_size >= 2^31),
 * ERR_DTYPE, ERR_ALIGN, ERR_WORKSPACE, ERR_UNSUPPORTED, ERR_CUDA.
 * ------------------------------------------------------------------------------------------ */
DIFFATTN_API int diffattn_v2_decode_paged(const void* q, const void* k_pool, const void* v_pool,
                                          const int* block_table, const int* seqlens,
                                          const float* lam_logit, void* out, int B, int Hq,
                                          int Hkv, int d, int num_pages, int page_size,
                                          int max_pages, int flags, int dtype, void* workspace,
                                          size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------------------------
 * Prefill straight from host memory (not part of the method; the serving path around it): the
 * layer's forward of diffattn_fwd_fused_lambda with q, k, v and out in host memory. The batch is
 * cut into chunks of whole sequences that pass through two slots of `workspace` in turn; the
 * copies in and out run on two library-owned streams and overlap the prefill of the previous or
 * next chunk, which runs on `stream`.
 *   q_host, k_host : host [B, N, H, 2d] bf16;  v_host, out_host : host [B, N, H, dv] bf16.
 *                    Page-locked (cudaHostAlloc / cudaHostRegister) memory is needed for the
 *                    copies to overlap; all four must stay valid until `stream` completes. A
 *                    page-locked out_host that is mapped into the device's address space (the
 *                    default for cudaHostAlloc on unified-address systems) is written by the
 *                    prefill's own stores over the host link, with no output copy; any other
 *                    out_host is filled by copies from the workspace.
 *   lq1 .. lk2, lambda_dim, lambda_sets, layer, norm_weight, eps, flags :
 *                    device data and meaning as diffattn_fwd_fused_lambda
 *   workspace, ws_bytes : device, >= diffattn_fwd_host_workspace_size(), 256-byte aligned, not
 *                    shared with a call that can run at the same time
 * The call returns once everything is enqueued; `stream` then completes after the last output
 * row has been written. Calls on one device serialise on the library's copy streams.
 * Supported: d in {64, 128}, dv = 2d. Errors: as diffattn_fwd_fused_lambda, plus ERR_WORKSPACE.
 * ------------------------------------------------------------------------------------------ */
DIFFATTN_API int diffattn_fwd_host_workspace_size(int B, int N, int H, int d, int dv,
                                                  size_t* bytes);
DIFFATTN_API int diffattn_fwd_host(const void* q_host, const void* k_host, const void* v_host,
                                   void* out_host, const float* lq1, const float* lk1,
                                   const float* lq2, const float* lk2, int lambda_dim,
                                   int lambda_sets, int layer, const float* norm_weight,
                                   float eps, int B, int N, int H, int d, int dv, int flags,
                                   void* workspace, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------------------------
 * Prefill over strided tensors: diffattn_fwd where q, k, v and out may be views, e.g. slices of
 * one fused projection output [B, N, 3, H, 2d]. The last dimension of each tensor is
 * contiguous; the others are given as element strides:
 *   strides : host int64 [12] = {q: batch, token, head,  k: batch, token, head,
 *                                v: batch, token, head,  out: batch, token, head}
 *             each a positive multiple of 16 bytes (8 bf16 or 4 fp32 elements)
 * Other arguments as diffattn_fwd. DIFFATTN_SINGLE_PASS needs the dense layout (ERR_UNSUPPORTED
 * otherwise); the default tensor-core path and the CUDA-core path take any strides. Elements of
 * `out` outside the addressed rows and columns are not written.
 * Errors: as diffattn_fwd.
 * ------------------------------------------------------------------------------------------ */
DIFFATTN_API int diffattn_fwd_strided(const void* q, const void* k, const void* v, void* out,
                                      const long long* strides, const float* lambda,
                                      float lambda_init, const float* norm_weight, float eps,
                                      int B, int N, int H, int d, int dv, int flags, int dtype,
                                      void* stream);

/* ------------------------------------------------------------------------------------------
 * Variable-length prefill: diffattn_fwd over sequences of different lengths packed along the
 * token axis (no padding), each attending only to itself (causally with DIFFATTN_CAUSAL). The
 * pages give no batching scheme; the operator per sequence is that of diffattn_fwd.
 *   q, k   : device [total, H, 2d];  v, out : device [total, H, dv]
 *   cu_seqlens : device int32 [B + 1], cu_seqlens[0] = 0, non-decreasing, cu_seqlens[B] <= total;
 *            sequence b is rows cu_seqlens[b] .. cu_seqlens[b+1]-1 (empty sequences allowed).
 *            Checked on the device: a sequence outside [0, total) or longer than max_seqlen is
 *            skipped and reported by diffattn_device_status() as DIFFATTN_ERR_INDEX.
 *   max_seqlen : the longest sequence (sizes the grid)
 *   lambda, lambda_init, norm_weight, eps, flags : as diffattn_fwd
 * Rows of `out` that belong to no sequence are not written.
 * Supported: dtype DIFFATTN_BF16 (tensor-core exact path), d in {64, 128}, dv = 2d.
 * Errors: as diffattn_fwd.
 * ------------------------------------------------------------------------------------------ */
DIFFATTN_API int diffattn_fwd_varlen(const void* q, const void* k, const void* v, void* out,
                                     const int* cu_seqlens, int max_seqlen, int total,
                                     const float* lambda, float lambda_init,
                                     const float* norm_weight, float eps, int B, int H, int d,
                                     int dv, int flags, int dtype, void* stream);

/* ------------------------------------------------------------------------------------------
 * Variable-length prefill with queries and keys of their own lengths: sequence b has Lk keys
 * (rows cu_seqlens_k[b] .. cu_seqlens_k[b+1]-1 of k and v) and Lq <= Lk queries (rows
 * cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 of q and out), which are its last Lq positions. With
 * DIFFATTN_CAUSAL, query i of the sequence sees keys 0 .. Lk - Lq + i (the causal mask aligned
 * at the end). This covers a prompt computed in chunks against the keys cached so far, and
 * several new tokens at once over a cache. With Lq = Lk it is diffattn_fwd_varlen; with Lq = 1
 * the decode of the sequence's last query. The pages give no batching scheme; the operator per
 * query row is that of diffattn_fwd (P3 "The mechanism, exactly").
 *   q      : device [total_q, H, 2d];  out : device [total_q, H, dv]
 *   k      : device [total_k, H, 2d];  v   : device [total_k, H, dv]
 *   cu_seqlens_q, cu_seqlens_k : device int32 [B + 1] each, non-decreasing from 0. Checked on
 *            the device: a sequence outside its tensor, with Lq > max_seqlen_q, or with Lk < Lq is
 *            skipped and reported by diffattn_device_status() as DIFFATTN_ERR_INDEX.
 *   max_seqlen_q, max_seqlen_k : the longest query and key runs (max_seqlen_q sizes the grid)
 *   lambda, lambda_init, norm_weight, eps, flags : as diffattn_fwd
 * Rows of `out` that belong to no sequence are not written.
 * Supported: dtype DIFFATTN_BF16 (tensor-core exact path), d in {64, 128}, dv = 2d.
 * Errors: ERR_ARG, ERR_SHAPE (also max_seqlen_q > max_seqlen_k or total_q > total_k), ERR_DTYPE,
 * ERR_ALIGN, ERR_CUDA.
 * ------------------------------------------------------------------------------------------ */
DIFFATTN_API int diffattn_fwd_varlen_qk(const void* q, const void* k, const void* v, void* out,
                                        const int* cu_seqlens_q, const int* cu_seqlens_k,
                                        int max_seqlen_q, int max_seqlen_k, int total_q,
                                        int total_k, const float* lambda, float lambda_init,
                                        const float* norm_weight, float eps, int B, int H, int d,
                                        int dv, int flags, int dtype, void* stream);

/* ------------------------------------------------------------------------------------------
 * DIFF V2 over packed sequences (page "Differential Transformer: softmax can't say zero, so it
 * subtracts", section "DIFF V2: what the authors changed"): diffattn_v2_fwd per sequence, the
 * sequences packed along the token axis, optionally with keys of their own lengths as for
 * diffattn_fwd_varlen_qk (a sequence's Lq queries are its last Lq of Lk positions).
 *   q : device [total_q, Hq, d];  k, v : device [total_k, Hkv, d]
 *   lam_logit : device fp32 [total_q, Hq/2] (per token and pair, before the sigmoid)
 *   out : device [total_q, Hq/2, d]
 *   cu_seqlens_q : device int32 [B + 1];  cu_seqlens_k : device int32 [B + 1], or NULL for keys
 *            at the queries' offsets (max_seqlen_k and total_k are then ignored). Checked on the
 *            device as for diffattn_fwd_varlen_qk (DIFFATTN_ERR_INDEX).
 *   flags : DIFFATTN_CAUSAL or 0, optionally DIFFATTN_EXACT (numerics as for diffattn_v2_fwd:
 *            one flash pass per head by default)
 * Rows of `out` that belong to no sequence are not written. Supported: dtype DIFFATTN_BF16,
 * d in {64, 128}, Hq/Hkv even.
 * Errors: ERR_ARG, ERR_SHAPE, ERR_DTYPE, ERR_ALIGN, ERR_CUDA.
 * ------------------------------------------------------------------------------------------ */
DIFFATTN_API int diffattn_v2_fwd_varlen(const void* q, const void* k, const void* v,
                                        const float* lam_logit, void* out,
                                        const int* cu_seqlens_q, const int* cu_seqlens_k,
                                        int max_seqlen_q, int max_seqlen_k, int total_q,
                                        int total_k, int B, int Hq, int Hkv, int d, int flags,
                                        int dtype, void* stream);

/* ------------------------------------------------------------------------------------------
 * Prefill over a paged KV cache: diffattn_fwd_varlen_qk (V1) and diffattn_v2_fwd_varlen (V2)
 * with each sequence's keys in pages of a pool, as a serving engine holds them: a prompt chunk,
 * or several new tokens, against the keys cached so far. The pages give no cache layout; the
 * operator per query row is unchanged.
 *   q, out : packed queries as for diffattn_fwd_varlen_qk / diffattn_v2_fwd_varlen
 *            (cu_seqlens_q, device int32 [B + 1]); sequence b's Lq queries are the last Lq of
 *            its Lk = seqlens_k[b] key positions
 *   k_pool, v_pool : device [num_pages, page_size, H, 2d] and [.., H, dv] (V1), or
 *            [num_pages, page_size, Hkv, d] both (V2)
 *   seqlens_k   : device int32 [B]; block_table : device int32 [B, max_pages]: key r of
 *            sequence b is row r % page_size of page block_table[b * max_pages + r / page_size]
 *   max_seqlen_q, max_seqlen_k : the longest query run (sizes the grid) and key run
 *   page_size   : a multiple of 128 (a tile of 128 keys lies in one page)
 * Checked on the device: a sequence with Lk < Lq or Lk > max_pages * page_size is skipped, and a
 * used block-table entry outside [0, num_pages) reads page 0; both are reported by
 * diffattn_device_status() as DIFFATTN_ERR_INDEX. Entries past a sequence's keys are not read.
 * Other arguments (flags included: DIFFATTN_EXACT for V2) as the packed calls. Supported: dtype
 * DIFFATTN_BF16, d = 128 (V1: dv = 256).
 * Errors: ERR_ARG, ERR_SHAPE, ERR_DTYPE, ERR_ALIGN, ERR_CUDA.
 * ------------------------------------------------------------------------------------------ */
DIFFATTN_API int diffattn_fwd_paged(const void* q, const void* k_pool, const void* v_pool,
                                    void* out, const int* cu_seqlens_q, const int* seqlens_k,
                                    const int* block_table, int max_seqlen_q, int max_seqlen_k,
                                    int total_q, int num_pages, int page_size, int max_pages,
                                    const float* lambda, float lambda_init,
                                    const float* norm_weight, float eps, int B, int H, int d,
                                    int dv, int flags, int dtype, void* stream);
DIFFATTN_API int diffattn_v2_fwd_paged(const void* q, const void* k_pool, const void* v_pool,
                                       const float* lam_logit, void* out,
                                       const int* cu_seqlens_q, const int* seqlens_k,
                                       const int* block_table, int max_seqlen_q, int max_seqlen_k,
                                       int total_q, int num_pages, int page_size, int max_pages,
                                       int B, int Hq, int Hkv, int d, int flags, int dtype,
                                       void* stream);

/* ------------------------------------------------------------------------------------------
 * Prefill with fp8 scores (page "Differential Transformer: softmax can't say zero, so it
 * subtracts", on the attention logits quantized to low bit widths: DIFF's logits are several
 * times smaller relative to their spread, so low-bit score products cost it little).
 * diffattn_fwd where q and k hold fp8 e4m3 values with one dequantisation factor each:
 *   q, k : device fp8 e4m3 [B, N, H, 2d] = [Q1 | Q2], [K1 | K2]; the real values are
 *          q * q_descale and k * k_descale (per tensor, finite, > 0)
 *   v, out : device bf16 as for diffattn_fwd
 * The score products Q_m K_m^T run on the fp8 tensor cores (tcgen05 kind::f8f6f4, fp32
 * accumulation); the two softmaxes, the subtraction, the product with V (bf16), the norm and the
 * scale are those of diffattn_fwd.
 * Supported: d = 128, dv = 256; flags DIFFATTN_CAUSAL | DIFFATTN_NORM | DIFFATTN_SCALE.
 * Errors: as diffattn_fwd.
 * ------------------------------------------------------------------------------------------ */
DIFFATTN_API int diffattn_fwd_fp8(const void* q, const void* k, const void* v, void* out,
                                  float q_descale, float k_descale, const float* lambda,
                                  float lambda_init, const float* norm_weight, float eps, int B,
                                  int N, int H, int d, int dv, int flags, void* stream);

/* ------------------------------------------------------------------------------------------
 * Prefill with lambda formed inside the kernel (pages "Differential Transformer: Noise-
 * Canceling Attention by Subtraction", section "Making lambda learnable and stable", and
 * "Differential Transformer: softmax can't say zero, so it subtracts", section "lambda,
 * re-parameterised"): diffattn_fwd, but instead of lambda[H] it takes the four
 * re-parameterisation vectors and the layer, and each CTA computes
 *   lambda = exp(lq1 . lk1) - exp(lq2 . lk2) + lambda_init(layer),
 *   lambda_init(layer) = 0.8 - 0.6 exp(-0.3 (layer - 1))   (layer 1-indexed)
 * in fp32 before its subtraction pass, so a layer's step is one launch.
 *   lq1, lk1, lq2, lk2 : device fp32 [lambda_sets, lambda_dim]; lambda_sets = 1 (one lambda for
 *                        every head) or H (one per head); 1 <= lambda_dim <= 4096
 *   layer              : >= 1; also sets the (1 - lambda_init) scale of DIFFATTN_SCALE
 * Supported: dtype DIFFATTN_BF16 (tensor-core exact path), d in {64, 128}, dv = 2d; flags
 * DIFFATTN_CAUSAL | DIFFATTN_NORM | DIFFATTN_SCALE.
 * Errors: as diffattn_fwd.
 * ------------------------------------------------------------------------------------------ */
DIFFATTN_API int diffattn_fwd_fused_lambda(const void* q, const void* k, const void* v, void* out,
                                           const float* lq1, const float* lk1, const float* lq2,
                                           const float* lk2, int lambda_dim, int lambda_sets,
                                           int layer, const float* norm_weight, float eps, int B,
                                           int N, int H, int d, int dv, int flags, int dtype,
                                           void* stream);

/* ------------------------------------------------------------------------------------------
 * Training: forward that keeps what the backward needs, and the backward of the V1 prefill
 * (page "Differential Transformer: softmax can't say zero, so it subtracts", section "The
 * mechanism, exactly" defines the forward; the gradients are its chain rule).
 *
 * diffattn_fwd_train: diffattn_fwd (tensor-core exact path) plus two outputs:
 *   o_pre : device bf16 [B, N, H, dv], the head output (A1 - lambda A2) V before the norm/scale
 *   stats : device fp32 [B, H, 2, Npad], Npad = N rounded up to a multiple of 128: for each row
 *           and map m, b_m = log2 sum_j 2^(log2(e) s_ij / sqrt(d)) over the visible keys, so that
 *           A_m = 2^(log2(e) s / sqrt(d) - b_m). Entries past N are not written.
 *   flags : DIFFATTN_CAUSAL | DIFFATTN_NORM | DIFFATTN_SCALE
 * Supported: dtype DIFFATTN_BF16, d = 128, dv = 256.
 *
 * diffattn_bwd: given dout = dL/dout [B, N, H, dv] (bf16) and the tensors of a diffattn_fwd_train
 * call with the same arguments, writes
 *   dq, dk : device bf16 [B, N, H, 2d] = [dQ1 | dQ2], [dK1 | dK2]
 *   dv     : device bf16 [B, N, H, dv]
 *   dlambda: device fp32 [H], dL/dlambda[h] (summed over batch and rows; overwritten)
 *   dnorm_weight : device fp32 [dv] or NULL, dL/dw of the norm weight (summed over every row and
 *           head; zeros without DIFFATTN_NORM)
 *   workspace, ws_bytes : at least diffattn_bwd_workspace_size() bytes, 256-byte aligned, not
 *           shared with a call that can run at the same time (contents need not be initialised).
 * lambda_init, norm_weight, eps and flags must be those of the forward. The result is
 * deterministic except for the order of the fp32 additions that build dq.
 * Errors: ERR_ARG, ERR_SHAPE, ERR_DTYPE, ERR_ALIGN, ERR_WORKSPACE, ERR_CUDA.
 * ------------------------------------------------------------------------------------------ */
DIFFATTN_API int diffattn_fwd_train(const void* q, const void* k, const void* v, void* out,
                                    void* o_pre, float* stats, const float* lambda,
                                    float lambda_init, const float* norm_weight, float eps, int B,
                                    int N, int H, int d, int dv, int flags, int dtype,
                                    void* stream);
DIFFATTN_API int diffattn_bwd_workspace_size(int B, int N, int H, int d, int dv, size_t* bytes);
DIFFATTN_API int diffattn_bwd(const void* q, const void* k, const void* v, const void* o_pre,
                              const float* stats, const void* dout, const float* lambda,
                              float lambda_init, const float* norm_weight, float eps, void* dq,
                              void* dk, void* dv, float* dlambda, float* dnorm_weight, int B,
                              int N, int H, int d, int dv_width, int flags, int dtype,
                              void* workspace, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------------------------
 * Training over packed sequences: diffattn_fwd_train and diffattn_bwd for sequences of
 * different lengths packed along the token axis, each attending only to itself, as
 * diffattn_fwd_varlen does for the forward.
 *   q, k : device [total, H, 2d];  v, out, o_pre, dout : device [total, H, dv];
 *   dq, dk : device [total, H, 2d];  dv : device [total, H, dv]
 *   cu_seqlens : device int32 [B + 1], non-decreasing from 0: sequence b is rows
 *            cu_seqlens[b] .. cu_seqlens[b+1]-1. Checked on the device: a sequence outside
 *            [0, total) or longer than max_seqlen is skipped and reported by
 *            diffattn_device_status() as DIFFATTN_ERR_INDEX.
 *   stats : device fp32 [B, H, 2, Npad], Npad = max_seqlen rounded up to a multiple of 128;
 *            row i of sequence b at index i (entries past the sequence's length mean nothing)
 *   workspace, ws_bytes : at least diffattn_bwd_varlen_workspace_size() bytes
 * Rows that belong to no sequence are not written. dlambda and dnorm_weight sum over every
 * sequence. Other arguments, support and errors as diffattn_fwd_train and diffattn_bwd.
 * ------------------------------------------------------------------------------------------ */
DIFFATTN_API int diffattn_fwd_train_varlen(const void* q, const void* k, const void* v,
                                           void* out, void* o_pre, float* stats,
                                           const int* cu_seqlens, int max_seqlen, int total,
                                           const float* lambda, float lambda_init,
                                           const float* norm_weight, float eps, int B, int H,
                                           int d, int dv, int flags, int dtype, void* stream);
DIFFATTN_API int diffattn_bwd_varlen_workspace_size(int B, int max_seqlen, int total, int H,
                                                   int d, int dv, size_t* bytes);
DIFFATTN_API int diffattn_bwd_varlen(const void* q, const void* k, const void* v,
                                     const void* o_pre, const float* stats, const void* dout,
                                     const int* cu_seqlens, int max_seqlen, int total,
                                     const float* lambda, float lambda_init,
                                     const float* norm_weight, float eps, void* dq, void* dk,
                                     void* dv, float* dlambda, float* dnorm_weight, int B, int H,
                                     int d, int dv_width, int flags, int dtype, void* workspace,
                                     size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------------------------
 * Grouped differential attention (page "Differential Transformer: softmax can't say zero, so it
 * subtracts", section "What other people found": the Grouped Differential Attention result, 3
 * or 4 signal heads per noise head). n_signal heads keep their own Q1, K1, V, lambda and norm;
 * they are split in n_noise contiguous groups of G = n_signal / n_noise, and signal head h
 * subtracts the map of noise head h / G:
 *   out_h = epilogue((softmax(Q1_h K1_h^T / sqrt d) - lambda[h] softmax(Q2_g K2_g^T / sqrt d)) V_h)
 * with g = h / G and the epilogue of diffattn_fwd. n_noise = n_signal is diffattn_fwd with the
 * halves of q and k stored as heads of their own.
 *   q      : device [B, N, n_signal + n_noise, d]: heads 0 .. n_signal-1 hold Q1 of the signal
 *            heads, heads n_signal .. n_signal+n_noise-1 Q2 of the noise heads
 *   k      : device [B, N, n_signal + n_noise, d], the same split for K1 and K2
 *   v, out : device [B, N, n_signal, dv]
 *   lambda : device fp32 [n_signal]
 *   lambda_init, norm_weight, eps, flags, dtype : as for diffattn_fwd
 *   workspace, ws_bytes : device scratch of diffattn_gda_fwd_workspace_size() bytes, 256-byte
 *            aligned, contents need not be initialised; or NULL. With a workspace (tensor-core
 *            path, d = 128) the call runs two launches: the first computes each noise map's row
 *            statistic (its exact softmax normaliser) once per noise head into the workspace;
 *            the second runs the signal heads, whose first pass then covers their own map only.
 *            With NULL each signal head's CTA recomputes its group's noise map statistics (two
 *            maps per head, as in diffattn_fwd); the result is the same up to rounding. The
 *            workspace must not be shared with a call that can run at the same time.
 * Supported: d in {64, 128}, dv = 2d, n_signal a multiple of n_noise. The noise heads' K is read
 * from HBM once per group and from L2 by the group's other heads.
 * Errors: ERR_ARG, ERR_SHAPE, ERR_DTYPE, ERR_ALIGN, ERR_WORKSPACE, ERR_UNSUPPORTED, ERR_CUDA.
 * ------------------------------------------------------------------------------------------ */
DIFFATTN_API int diffattn_gda_fwd_workspace_size(int B, int N, int n_signal, int n_noise, int d,
                                                 int dv, size_t* bytes);
DIFFATTN_API int diffattn_gda_fwd(const void* q, const void* k, const void* v, void* out,
                                  const float* lambda, float lambda_init, const float* norm_weight,
                                  float eps, int B, int N, int n_signal, int n_noise, int d, int dv,
                                  int flags, int dtype, void* workspace, size_t ws_bytes,
                                  void* stream);

/* Grouped prefill with fp8 scores: diffattn_gda_fwd where q and k hold fp8 e4m3 values with one
 * dequantisation factor each (page "Differential Transformer: softmax can't say zero, so it
 * subtracts": section "What other people found" for the grouped form, and its note on attention
 * logits quantized to low bit widths for the fp8 score products).
 *   q, k   : device fp8 e4m3 [B, N, n_signal + n_noise, d], the head split of diffattn_gda_fwd;
 *            the real values are q * q_descale and k * k_descale (per tensor, finite, > 0)
 *   v, out : device bf16 [B, N, n_signal, dv]
 *   lambda, lambda_init, norm_weight, eps : as for diffattn_gda_fwd
 * The score products run on the fp8 tensor cores (tcgen05 kind::f8f6f4, fp32 accumulation); the
 * softmaxes, the subtraction, the product with V (bf16), the norm and the scale are those of
 * diffattn_gda_fwd. One launch: each signal head's CTA forms its noise map's statistics itself.
 * n_noise = n_signal is diffattn_fwd_fp8 with the halves of q and k stored as heads of their own.
 * Supported: d = 128, dv = 256, n_signal a multiple of n_noise; flags DIFFATTN_CAUSAL |
 * DIFFATTN_NORM | DIFFATTN_SCALE.
 * Errors: ERR_ARG (null pointer, unknown flag, eps, descale factors), ERR_SHAPE, ERR_ALIGN,
 * ERR_CUDA.
 */
DIFFATTN_API int diffattn_gda_fwd_fp8(const void* q, const void* k, const void* v, void* out,
                                      float q_descale, float k_descale, const float* lambda,
                                      float lambda_init, const float* norm_weight, float eps,
                                      int B, int N, int n_signal, int n_noise, int d, int dv,
                                      int flags, void* stream);

/* Grouped prefill over packed sequences: diffattn_gda_fwd on sequences of different lengths
 * packed along the token axis (no padding), each attending only to itself, as
 * diffattn_fwd_varlen does for the ungrouped operator.
 *   q, k   : device [total, n_signal + n_noise, d] (the head split of diffattn_gda_fwd)
 *   v, out : device [total, n_signal, dv]
 *   cu_seqlens, max_seqlen, total : as diffattn_fwd_varlen (offsets checked on the device)
 *   workspace, ws_bytes : as diffattn_gda_fwd, of diffattn_gda_fwd_workspace_size(B,
 *            max_seqlen, ...) bytes (entry (b, g, i): row i of sequence b's noise map g), or NULL
 * Rows of `out` that belong to no sequence are not written.
 * Supported: dtype DIFFATTN_BF16 (tensor-core exact path), flags CAUSAL | NORM | SCALE, d in
 * {64, 128}, dv = 2d, n_signal a multiple of n_noise.
 * Errors: as diffattn_gda_fwd.
 */
DIFFATTN_API int diffattn_gda_fwd_varlen(const void* q, const void* k, const void* v, void* out,
                                         const int* cu_seqlens, int max_seqlen, int total,
                                         const float* lambda, float lambda_init,
                                         const float* norm_weight, float eps, int B, int n_signal,
                                         int n_noise, int d, int dv, int flags, int dtype,
                                         void* workspace, size_t ws_bytes, void* stream);

/* Grouped training: the forward saving what the backward needs, and the backward (gradients of
 * every input of diffattn_gda_fwd, the chain rule of its operator: signal head h's gradients are
 * those of the ungrouped operator with map 2 taken from noise head n_signal + h / G, and a
 * noise head's dQ2 and dK2 sum the contributions of the G signal heads of its group).
 *   diffattn_gda_fwd_train: diffattn_gda_fwd plus
 *     o_pre : device bf16 [B, N, n_signal, dv], each signal head's output before the norm
 *     stats : device fp32 [B, n_signal, 2, Npad] (Npad = N rounded up to 128): per row and map the
 *             base-2 log-sum-exp of the scaled scores (map 2's is its noise head's)
 *     workspace, ws_bytes : as diffattn_gda_fwd (NULL: one launch)
 *   diffattn_gda_bwd: dout [B, N, n_signal, dv] the gradient of out; writes
 *     dq, dk : device bf16 [B, N, n_signal + n_noise, d] (q's layout)
 *     dv     : device bf16 [B, N, n_signal, dv]
 *     dlambda : device fp32 [n_signal];  dnorm_weight : device fp32 [dv] or NULL
 *     workspace, ws_bytes : at least diffattn_gda_bwd_workspace_size() bytes, 256-byte aligned
 *   The noise heads' dK2 is summed in fp32 through atomic additions, so its last bits can
 *   differ from run to run; every other output is deterministic.
 * Supported: batched, d = 128, dv = 256, dtype DIFFATTN_BF16, flags CAUSAL | NORM | SCALE,
 * n_signal a multiple of n_noise.
 * Errors: ERR_ARG, ERR_SHAPE, ERR_DTYPE, ERR_ALIGN, ERR_WORKSPACE, ERR_CUDA.
 */
DIFFATTN_API int diffattn_gda_fwd_train(const void* q, const void* k, const void* v, void* out,
                                        void* o_pre, float* stats, const float* lambda,
                                        float lambda_init, const float* norm_weight, float eps,
                                        int B, int N, int n_signal, int n_noise, int d, int dv,
                                        int flags, int dtype, void* workspace, size_t ws_bytes,
                                        void* stream);
DIFFATTN_API int diffattn_gda_bwd_workspace_size(int B, int N, int n_signal, int n_noise, int d,
                                                 int dv, size_t* bytes);
DIFFATTN_API int diffattn_gda_bwd(const void* q, const void* k, const void* v, const void* o_pre,
                                  const float* stats, const void* dout, const float* lambda,
                                  float lambda_init, const float* norm_weight, float eps, void* dq,
                                  void* dk, void* dv, float* dlambda, float* dnorm_weight, int B,
                                  int N, int n_signal, int n_noise, int d, int dv_width, int flags,
                                  int dtype, void* workspace, size_t ws_bytes, void* stream);

/* Grouped training over packed sequences: diffattn_gda_fwd_train and diffattn_gda_bwd with the
 * packed layout of diffattn_gda_fwd_varlen (page "Differential Transformer: softmax can't say
 * zero, so it subtracts", section "What other people found", with the batching of
 * diffattn_fwd_train_varlen / diffattn_bwd_varlen). Each sequence's gradients are those of its
 * own grouped forward; dlambda and dnorm_weight sum over the sequences.
 *   q, k, dq, dk : device bf16 [total, n_signal + n_noise, d]; v, dv, out, o_pre, dout : device
 *                  bf16 [total, n_signal, dv]; sequence b is rows cu_seqlens[b] ..
 *                  cu_seqlens[b+1] - 1 (device int32 [B + 1], non-decreasing, cu[B] <= total,
 *                  checked on the device)
 *   stats        : device fp32 [B, n_signal, 2, Npad], Npad = max_seqlen rounded up to 128
 *   max_seqlen   : the longest sequence (an upper bound)
 *   workspace    : forward, as diffattn_gda_fwd_varlen (or NULL); backward, at least
 *                  diffattn_gda_bwd_varlen_workspace_size(B, max_seqlen, total, ...) bytes,
 *                  256-byte aligned
 * Rows of out, o_pre, dq, dk and dv that belong to no sequence are not written.
 * Supported: dtype DIFFATTN_BF16, flags CAUSAL | NORM | SCALE, d = 128, dv = 256, n_signal a
 * multiple of n_noise.
 * Errors: as diffattn_gda_fwd_train / diffattn_gda_bwd; ERR_SHAPE if max_seqlen > total or total *
 * (n_signal + n_noise) > 2^30; bad offsets are reported through diffattn_device_status. */
DIFFATTN_API int diffattn_gda_fwd_train_varlen(const void* q, const void* k, const void* v,
                                               void* out, void* o_pre, float* stats,
                                               const int* cu_seqlens, int max_seqlen, int total,
                                               const float* lambda, float lambda_init,
                                               const float* norm_weight, float eps, int B,
                                               int n_signal, int n_noise, int d, int dv, int flags,
                                               int dtype, void* workspace, size_t ws_bytes,
                                               void* stream);
DIFFATTN_API int diffattn_gda_bwd_varlen_workspace_size(int B, int max_seqlen, int total,
                                                        int n_signal, int n_noise, int d, int dv,
                                                        size_t* bytes);
DIFFATTN_API int diffattn_gda_bwd_varlen(const void* q, const void* k, const void* v,
                                         const void* o_pre, const float* stats, const void* dout,
                                         const int* cu_seqlens, int max_seqlen, int total,
                                         const float* lambda, float lambda_init,
                                         const float* norm_weight, float eps, void* dq, void* dk,
                                         void* dv, float* dlambda, float* dnorm_weight, int B,
                                         int n_signal, int n_noise, int d, int dv_width, int flags,
                                         int dtype, void* workspace, size_t ws_bytes,
                                         void* stream);

/* Grouped prefill with each sequence's queries at the end of its keys (chunked prompts, new tokens
 * over a cache): diffattn_gda_fwd's operator with the key layout of diffattn_fwd_varlen_qk
 * (keys packed with offsets of their own) or of diffattn_fwd_paged (keys in page pools).
 *   q, out : device [total_q, n_signal + n_noise, d] and [total_q, n_signal, dv], packed by
 *            cu_seqlens_q as in diffattn_gda_fwd_varlen
 *   k, v   : device [total_k, n_signal + n_noise, d] and [total_k, n_signal, dv] with
 *            cu_seqlens_k (varlen_qk); or pools k_pool [num_pages, page_size, n_signal + n_noise, d]
 *            and v_pool [num_pages, page_size, n_signal, dv] with seqlens_k and block_table
 *            (paged; page_size a multiple of 128)
 *   the offsets, lengths and table are checked on the device as for the ungrouped forms
 *   workspace, ws_bytes : as diffattn_gda_fwd, of diffattn_gda_fwd_workspace_size(B,
 *            max_seqlen_q, ...) bytes, or NULL (each signal head then forms its noise map's
 *            statistics itself)
 * Rows of `out` that belong to no sequence are not written.
 * Supported: dtype DIFFATTN_BF16, flags CAUSAL | NORM | SCALE, d = 128, dv = 256, n_signal a
 * multiple of n_noise.
 * Errors: as diffattn_gda_fwd; ERR_SHAPE as diffattn_fwd_varlen_qk / diffattn_fwd_paged.
 */
DIFFATTN_API int diffattn_gda_fwd_varlen_qk(const void* q, const void* k, const void* v, void* out,
                                            const int* cu_seqlens_q, const int* cu_seqlens_k,
                                            int max_seqlen_q, int max_seqlen_k, int total_q,
                                            int total_k, const float* lambda, float lambda_init,
                                            const float* norm_weight, float eps, int B,
                                            int n_signal, int n_noise, int d, int dv, int flags,
                                            int dtype, void* workspace, size_t ws_bytes,
                                            void* stream);
DIFFATTN_API int diffattn_gda_fwd_paged(const void* q, const void* k_pool, const void* v_pool,
                                        void* out, const int* cu_seqlens_q, const int* seqlens_k,
                                        const int* block_table, int max_seqlen_q, int max_seqlen_k,
                                        int total_q, int num_pages, int page_size, int max_pages,
                                        const float* lambda, float lambda_init,
                                        const float* norm_weight, float eps, int B, int n_signal,
                                        int n_noise, int d, int dv, int flags, int dtype,
                                        void* workspace, size_t ws_bytes, void* stream);

/* Grouped decode: one query token per sequence over its cached keys 0 .. seqlens[b]-1, with the
 * head split of diffattn_gda_fwd.
 *   q       : device bf16 [B, n_signal + n_noise, d]
 *   k_cache : device bf16 [B, Lmax, n_signal + n_noise, d]
 *   v_cache : device bf16 [B, Lmax, n_signal, dv];  out : device bf16 [B, n_signal, dv]
 *   seqlens, lambda ([n_signal]), lambda_init, norm_weight, eps, flags : as for diffattn_decode
 *   workspace, ws_bytes : at least diffattn_decode_workspace_size(B, Lmax, n_signal, d, dv)
 *                         bytes, 256-byte aligned
 * Supported: d = 128, dv = 256, n_signal a multiple of n_noise. Every cached K1, K2 and V row is
 * streamed once per head that reads it: a noise row serves the G heads of its group, the
 * repeats mostly from L2.
 * Errors: ERR_ARG, ERR_SHAPE, ERR_DTYPE, ERR_ALIGN, ERR_WORKSPACE, ERR_CUDA. */
DIFFATTN_API int diffattn_gda_decode(const void* q, const void* k_cache, const void* v_cache,
                                     const int* seqlens, void* out, const float* lambda,
                                     float lambda_init, const float* norm_weight, float eps, int B,
                                     int Lmax, int n_signal, int n_noise, int d, int dv, int flags,
                                     int dtype, void* workspace, size_t ws_bytes, void* stream);

/* Grouped decode over a paged KV cache: diffattn_gda_decode with the caches held in fixed-size
 * pages of shared pools, addressed as in diffattn_decode_paged (key j of sequence b is row
 * j % page_size of page block_table[b][j / page_size]).
 *   k_pool : device bf16 [num_pages, page_size, n_signal + n_noise, d] (the head split of
 *            diffattn_gda_fwd)
 *   v_pool : device bf16 [num_pages, page_size, n_signal, dv]
 *   block_table, seqlens, num_pages, page_size, max_pages : as for diffattn_decode_paged (any
 *            page size; a used table entry outside [0, num_pages) reads page 0 instead and is
 *            reported by diffattn_device_status() as DIFFATTN_ERR_INDEX)
 *   other arguments as diffattn_gda_decode; workspace of at least
 *   diffattn_decode_workspace_size(B, max_pages * page_size, n_signal, d, dv) bytes
 * Supported: d = 128, dv = 256, n_signal a multiple of n_noise.
 * Errors: ERR_ARG, ERR_SHAPE, ERR_DTYPE, ERR_ALIGN, ERR_WORKSPACE, ERR_CUDA. */
DIFFATTN_API int diffattn_gda_decode_paged(const void* q, const void* k_pool, const void* v_pool,
                                           const int* block_table, const int* seqlens, void* out,
                                           const float* lambda, float lambda_init,
                                           const float* norm_weight, float eps, int B,
                                           int n_signal, int n_noise, int d, int dv, int num_pages,
                                           int page_size, int max_pages, int flags, int dtype,
                                           void* workspace, size_t ws_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DIFFATTN_H_ */
