"""Float64 CPU oracle for differential attention.

TEST INFRASTRUCTURE ONLY. This module is imported by `tests/`, by `__graft_entry__.smoke()` and by
`bench.py`'s CPU-baseline leg, and by nothing else: the library's product path never calls it and
shares no code with it (no kernels, headers, helpers or constants). Inputs come from `synth/`.

It is the plain definition of the operator written out in float64 with numpy, one step per
equation, blocked over query rows only so that memory stays O(rows_per_block x N). No other
blocking, fusion or reordering is done: every score is formed, every softmax row is normalised,
the two maps are subtracted and the difference is multiplied by V, in that order.

Sources (page title, section):
  [P1] "Differential Transformer: Noise-Canceling Attention by Subtraction" -- "The mechanism",
       "Making lambda learnable and stable".
  [P3] "Differential Transformer: softmax can't say zero, so it subtracts" -- "The mechanism,
       exactly" (DiffAttn equation and the quoted MultiheadDiffAttn.forward), "lambda,
       re-parameterised", "The row no longer sums to one", "DIFF V2: what the authors changed".
  [P5] "Differential Transformer V2" -- GQA pairing of the subtracted heads.

Readings taken where the pages are silent or disagree:
  * the 1/sqrt(d) scale uses d = width of one query/key half (P1 `d**0.5`, P3 Q_i in R^{N x d});
  * lambda is one float per head (P1 says per head, P3 says one per layer shared by every head; a
    per-head array covers both); it is computed and used in full precision, no clipping;
  * the per-head norm is an RMSNorm over all dv channels of the head, y = o / sqrt(mean(o^2) + eps)
    * w, then times (1 - lambda_init) (P3 quotes `subln` then `* (1 - lambda_init)`); the
    GroupNorm "+ lambda_init" form on the Japanese page is treated as garbled;
  * causal prefill with Nq = Nk: key j is visible to query i iff j <= i; when a sequence's Lq
    queries are the last of its Lk key positions (the packed and paged forms), the query at
    position p sees keys 0 .. p, so the mask is aligned at the end; decode attends to every
    cached key of its row;
  * V2 pairs heads (2p, 2p+1), uses KV head floor(2p / (Hq/Hkv)), lambda = sigmoid(logit) per
    token and pair, no per-head norm, and the default 1/sqrt(d) scale.
  * grouped differential attention (the pages give only "3 or 4 signal heads per noise head"):
    Hs signal heads and Hn noise heads, Hs a multiple of Hn; signal head h keeps its own Q1, K1,
    V, lambda and norm, and subtracts the map of noise head floor(h / (Hs/Hn)), the noise heads
    split in contiguous groups as the query heads of a GQA group are. With Hn = Hs it is the
    ungrouped operator.

Parity pins: every function here is pinned by `tests/test_oracle_pins.py` (worked examples printed
on the pages, closed forms, library routines for special cases, brute force on tiny inputs).
"""
from __future__ import annotations

import math

import numpy as np

ROW_BLOCK = 256


def _f64(x) -> np.ndarray:
    """float64 copy of a numpy array or a (CPU) torch tensor, without importing torch."""
    if hasattr(x, "detach"):
        x = x.detach().cpu().float().numpy()
    return np.asarray(x, dtype=np.float64)


# --------------------------------------------------------------------------------------------
# lambda  ([P1] "Making lambda learnable and stable"; [P3] "lambda, re-parameterised")
# --------------------------------------------------------------------------------------------

def lambda_init(layer: int) -> float:
    """lambda_init(l) = 0.8 - 0.6 * exp(-0.3 * (l - 1)), with l the 1-indexed layer."""
    return 0.8 - 0.6 * math.exp(-0.3 * (layer - 1))


def lambda_full(lq1, lk1, lq2, lk2, layer: int) -> np.ndarray:
    """lambda = exp(lq1 . lk1) - exp(lq2 . lk2) + lambda_init(layer), one value per row (head set).

    Vectors are [n_sets, dim] (or [dim]); the dot products run over the last axis.
    """
    lq1, lk1, lq2, lk2 = (_f64(t) for t in (lq1, lk1, lq2, lk2))
    dot1 = np.sum(lq1 * lk1, axis=-1)
    dot2 = np.sum(lq2 * lk2, axis=-1)
    return np.exp(dot1) - np.exp(dot2) + lambda_init(layer)


# --------------------------------------------------------------------------------------------
# the two maps and their difference  ([P3] "The mechanism, exactly"; [P1] "The mechanism")
# --------------------------------------------------------------------------------------------

def softmax_rows(S: np.ndarray) -> np.ndarray:
    """Row-wise softmax exp(S - rowmax) / sum. -inf entries get weight 0."""
    m = np.max(S, axis=-1, keepdims=True)
    e = np.exp(S - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def scores(Q: np.ndarray, K: np.ndarray, row_ids: np.ndarray | None, causal: bool) -> np.ndarray:
    """S = Q K^T / sqrt(d) with d = Q's width; causal sets S[i, j] = -inf for key j > query i.

    `row_ids` are the absolute query positions of Q's rows (needed for the causal mask).
    """
    d = Q.shape[-1]
    S = (Q @ K.T) / math.sqrt(d)
    if causal:
        cols = np.arange(K.shape[0])[None, :]
        S = np.where(cols > row_ids[:, None], -np.inf, S)
    return S


def diff_weights(S1: np.ndarray, S2: np.ndarray, lam: float) -> np.ndarray:
    """W = softmax(S1) - lam * softmax(S2): the signed weights of one differential head."""
    return softmax_rows(S1) - lam * softmax_rows(S2)


def diff_attn_head(q1, k1, q2, k2, v, lam: float, causal: bool, rows=None) -> np.ndarray:
    """DiffAttn for one head: (softmax(Q1 K1^T/sqrt d) - lam softmax(Q2 K2^T/sqrt d)) V.

    q1, q2 [Nq, d]; k1, k2 [Nk, d]; v [Nk, dv]. Returns the rows listed in `rows` (default all),
    [len(rows), dv], computed ROW_BLOCK query rows at a time.
    """
    q1, k1, q2, k2, v = (_f64(t) for t in (q1, k1, q2, k2, v))
    rows = np.arange(q1.shape[0]) if rows is None else np.asarray(rows)
    out = np.empty((rows.shape[0], v.shape[1]), dtype=np.float64)
    for s in range(0, rows.shape[0], ROW_BLOCK):
        r = rows[s:s + ROW_BLOCK]
        S1 = scores(q1[r], k1, r, causal)
        S2 = scores(q2[r], k2, r, causal)
        out[s:s + ROW_BLOCK] = diff_weights(S1, S2, lam) @ v
    return out


# --------------------------------------------------------------------------------------------
# per-head norm and fixed rescale  ([P3] "The row no longer sums to one"; [P1] items 1-2)
# --------------------------------------------------------------------------------------------

def subln(O: np.ndarray, weight, eps: float) -> np.ndarray:
    """RMSNorm over the last axis: O / sqrt(mean(O^2) + eps) * weight."""
    O = _f64(O)
    rms = np.sqrt(np.mean(O * O, axis=-1, keepdims=True) + eps)
    w = 1.0 if weight is None else _f64(weight)
    return O / rms * w


def head_epilogue(O, weight, eps: float, lam_init: float, norm: bool, apply_scale: bool):
    """subln (when `norm`) then multiply by (1 - lambda_init) (when `apply_scale`)."""
    Y = subln(O, weight, eps) if norm else _f64(O)
    if apply_scale:
        Y = Y * (1.0 - lam_init)
    return Y


# --------------------------------------------------------------------------------------------
# the three operator entry points
# --------------------------------------------------------------------------------------------

def diffattn_fwd(q, k, v, lam, lam_init: float, norm_weight=None, eps: float = 1e-5,
                 norm: bool = True, apply_scale: bool = True, causal: bool = True, rows=None):
    """Prefill over the layout q [B,N,H,2d] = [Q1|Q2], k [B,N,H,2d] = [K1|K2], v [B,N,H,dv].

    lam: one value per head ([H]) or a scalar. Returns float64 [B, len(rows), H, dv].
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, N, H, two_d = q.shape
    d = two_d // 2
    lam = np.broadcast_to(_f64(lam), (H,))
    rows = np.arange(N) if rows is None else np.asarray(rows)
    out = np.empty((B, rows.shape[0], H, v.shape[-1]), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            O = diff_attn_head(q[b, :, h, :d], k[b, :, h, :d], q[b, :, h, d:], k[b, :, h, d:],
                               v[b, :, h, :], float(lam[h]), causal, rows)
            out[b, :, h, :] = head_epilogue(O, norm_weight, eps, lam_init, norm, apply_scale)
    return out


def diffattn_decode(q, k_cache, v_cache, seqlens, lam, lam_init: float, norm_weight=None,
                    eps: float = 1e-5, norm: bool = True, apply_scale: bool = True):
    """One query per sequence over its cached keys 0 .. seqlens[b]-1 (no mask inside that range).

    q [B,H,2d], k_cache [B,L,H,2d], v_cache [B,L,H,dv], seqlens [B]. Returns float64 [B,H,dv].
    """
    q = _f64(q)
    B, H, two_d = q.shape
    d = two_d // 2
    lam = np.broadcast_to(_f64(lam), (H,))
    seqlens = np.asarray(_f64(seqlens)).astype(np.int64)
    out = np.empty((B, H, v_cache.shape[-1]), dtype=np.float64)
    for b in range(B):
        L = int(seqlens[b])
        kb = _f64(k_cache[b, :L])
        vb = _f64(v_cache[b, :L])
        for h in range(H):
            O = diff_attn_head(q[b, h:h + 1, :d], kb[:, h, :d], q[b, h:h + 1, d:], kb[:, h, d:],
                               vb[:, h, :], float(lam[h]), causal=False)
            out[b, h, :] = head_epilogue(O, norm_weight, eps, lam_init, norm, apply_scale)[0]
    return out


def sigmoid(x):
    x = _f64(x)
    return 1.0 / (1.0 + np.exp(-x))


def attention_head(q, k, v, causal: bool, rows=None) -> np.ndarray:
    """Plain softmax attention softmax(q k^T / sqrt d) v for one head, blocked over rows."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    rows = np.arange(q.shape[0]) if rows is None else np.asarray(rows)
    out = np.empty((rows.shape[0], v.shape[1]), dtype=np.float64)
    for s in range(0, rows.shape[0], ROW_BLOCK):
        r = rows[s:s + ROW_BLOCK]
        out[s:s + ROW_BLOCK] = softmax_rows(scores(q[r], k, r, causal)) @ v
    return out


def v2_kv_head(p: int, Hq: int, Hkv: int) -> int:
    """KV head shared by pair p: query heads of one GQA group are contiguous ([P5]), so query head
    2p belongs to group floor(2p / (Hq / Hkv)); heads 2p and 2p+1 fall in the same group whenever
    Hq / Hkv is even."""
    return (2 * p) // (Hq // Hkv)


def diffattn_v2_fwd(q, k, v, lam_logit, causal: bool = True, rows=None):
    """DIFF V2 ([P3] "DIFF V2: what the authors changed"): attention over 2h query heads sharing
    GQA KV heads, then out_p = attn[2p] - sigmoid(lam[t, p]) * attn[2p+1]; no norm, no lambda_init.

    q [B,N,Hq,d], k, v [B,N,Hkv,d], lam_logit [B,N,Hq/2]. Returns float64 [B, len(rows), Hq/2, d].
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, N, Hq, d = q.shape
    Hkv = k.shape[2]
    P = Hq // 2
    rows = np.arange(N) if rows is None else np.asarray(rows)
    sig = sigmoid(lam_logit)
    out = np.empty((B, rows.shape[0], P, v.shape[-1]), dtype=np.float64)
    for b in range(B):
        for p in range(P):
            g = v2_kv_head(p, Hq, Hkv)
            a1 = attention_head(q[b, :, 2 * p], k[b, :, g], v[b, :, g], causal, rows)
            a2 = attention_head(q[b, :, 2 * p + 1], k[b, :, g], v[b, :, g], causal, rows)
            out[b, :, p, :] = a1 - sig[b, rows, p][:, None] * a2
    return out


def diffattn_v2_decode(q, k_cache, v_cache, seqlens, lam_logit):
    """DIFF V2 decode: one query token per sequence over its cached keys 0 .. seqlens[b]-1 (no
    mask inside that range); out_p = attn[2p] - sigmoid(lam[b, p]) * attn[2p+1], the two query
    heads of pair p sharing the GQA KV head floor(2p / (Hq / Hkv)) ([P3] "DIFF V2: what the
    authors changed"; [P5] on V2 decoding over an unchanged KV cache).

    q [B,Hq,d], k_cache, v_cache [B,L,Hkv,d], seqlens [B], lam_logit [B,Hq/2].
    Returns float64 [B, Hq/2, d].
    """
    q = _f64(q)
    B, Hq, d = q.shape
    Hkv = k_cache.shape[2]
    P = Hq // 2
    seqlens = np.asarray(_f64(seqlens)).astype(np.int64)
    sig = sigmoid(lam_logit)
    out = np.empty((B, P, v_cache.shape[-1]), dtype=np.float64)
    for b in range(B):
        L = int(seqlens[b])
        kb, vb = _f64(k_cache[b, :L]), _f64(v_cache[b, :L])
        for p in range(P):
            g = v2_kv_head(p, Hq, Hkv)
            a1 = attention_head(q[b, 2 * p:2 * p + 1], kb[:, g], vb[:, g], causal=False)
            a2 = attention_head(q[b, 2 * p + 1:2 * p + 2], kb[:, g], vb[:, g], causal=False)
            out[b, p, :] = (a1 - sig[b, p] * a2)[0]
    return out


# --------------------------------------------------------------------------------------------
# backward of the V1 prefill: the gradients a training step needs  ([P3] "The mechanism,
# exactly" gives the forward; its gradients follow by the chain rule, step by step in reverse)
# --------------------------------------------------------------------------------------------

def subln_bwd(O, weight, eps: float, dY):
    """Gradients of Y = O / sqrt(mean(O^2) + eps) * w (over the last axis) given dY.

    With r = (mean(O^2) + eps)^(-1/2) and Yhat = O r: dO = r (g - Yhat mean(g Yhat)), g = dY w;
    dw = sum over rows of dY Yhat. Returns (dO, dw).
    """
    O, dY = _f64(O), _f64(dY)
    r = 1.0 / np.sqrt(np.mean(O * O, axis=-1, keepdims=True) + eps)
    Yhat = O * r
    w = 1.0 if weight is None else _f64(weight)
    g = dY * w
    dO = r * (g - Yhat * np.mean(g * Yhat, axis=-1, keepdims=True))
    dw = np.sum(dY * Yhat, axis=0)
    return dO, dw


def softmax_rows_bwd(A: np.ndarray, dA: np.ndarray) -> np.ndarray:
    """dS for A = softmax(S) along rows: A * (dA - rowsum(dA * A)). Masked entries (A = 0) get 0."""
    return A * (dA - np.sum(dA * A, axis=-1, keepdims=True))


def diff_attn_head_bwd(q1, k1, q2, k2, v, lam: float, causal: bool, dO):
    """Gradients of O = (softmax(S1) - lam softmax(S2)) V with S_m = Q_m K_m^T / sqrt(d).

    Reverse order of the forward: dW = dO V^T and dV = W^T dO; dA1 = dW, dA2 = -lam dW and
    dlam = -sum(A2 * dW); each softmax backward; then dQ_m = dS_m K_m / sqrt(d) and
    dK_m = dS_m^T Q_m / sqrt(d). Returns (dq1, dk1, dq2, dk2, dv, dlam).
    """
    q1, k1, q2, k2, v, dO = (_f64(t) for t in (q1, k1, q2, k2, v, dO))
    rows = np.arange(q1.shape[0])
    c = 1.0 / math.sqrt(q1.shape[-1])
    A1 = softmax_rows(scores(q1, k1, rows, causal))
    A2 = softmax_rows(scores(q2, k2, rows, causal))
    W = A1 - lam * A2
    dW = dO @ v.T
    dv = W.T @ dO
    dlam = -float(np.sum(A2 * dW))
    dS1 = softmax_rows_bwd(A1, dW)
    dS2 = softmax_rows_bwd(A2, -lam * dW)
    return (dS1 @ k1 * c, dS1.T @ q1 * c, dS2 @ k2 * c, dS2.T @ q2 * c, dv, dlam)


def diffattn_bwd(q, k, v, lam, lam_init: float, dy, norm_weight=None, eps: float = 1e-5,
                 norm: bool = True, apply_scale: bool = True, causal: bool = True, heads=None):
    """Backward of `diffattn_fwd` for the upstream gradient dy [B,N,H,dv].

    Returns dict(dq [B,N,H,2d] = [dQ1|dQ2], dk [B,N,H,2d] = [dK1|dK2], dv [B,N,H,dv],
    dlam [H], dw [dv]) in float64; dw is the gradient of the per-channel norm weight (summed over
    every row and head; zeros without the norm). `heads` restricts the work to a list of
    (b, h) pairs (others stay zero) -- dlam and dw then sum over those pairs only.
    """
    q, k, v, dy = _f64(q), _f64(k), _f64(v), _f64(dy)
    B, N, H, two_d = q.shape
    d = two_d // 2
    dvw = v.shape[-1]
    lam = np.broadcast_to(_f64(lam), (H,))
    s = (1.0 - lam_init) if apply_scale else 1.0
    out = dict(dq=np.zeros_like(q), dk=np.zeros_like(k), dv=np.zeros_like(v),
               dlam=np.zeros(H), dw=np.zeros(dvw))
    pairs = [(b, h) for b in range(B) for h in range(H)] if heads is None else heads
    for b, h in pairs:
        q1, q2 = q[b, :, h, :d], q[b, :, h, d:]
        k1, k2 = k[b, :, h, :d], k[b, :, h, d:]
        O = diff_attn_head(q1, k1, q2, k2, v[b, :, h, :], float(lam[h]), causal)
        dYs = dy[b, :, h, :] * s
        if norm:
            dO, dwh = subln_bwd(O, norm_weight, eps, dYs)
            out["dw"] += dwh
        else:
            dO = dYs
        dq1, dk1, dq2, dk2, dvh, dl = diff_attn_head_bwd(q1, k1, q2, k2, v[b, :, h, :],
                                                          float(lam[h]), causal, dO)
        out["dq"][b, :, h, :d], out["dq"][b, :, h, d:] = dq1, dq2
        out["dk"][b, :, h, :d], out["dk"][b, :, h, d:] = dk1, dk2
        out["dv"][b, :, h, :] = dvh
        out["dlam"][h] += dl
    return out


def lambda_full_bwd(lq1, lk1, lq2, lk2, dlam):
    """Gradients of lambda = exp(lq1 . lk1) - exp(lq2 . lk2) + lambda_init w.r.t. the four
    vectors ([n_sets, dim]) given dlam [n_sets]. Returns (dlq1, dlk1, dlq2, dlk2)."""
    lq1, lk1, lq2, lk2 = (_f64(t) for t in (lq1, lk1, lq2, lk2))
    g = _f64(dlam)[..., None]
    e1 = np.exp(np.sum(lq1 * lk1, axis=-1, keepdims=True))
    e2 = np.exp(np.sum(lq2 * lk2, axis=-1, keepdims=True))
    return g * e1 * lk1, g * e1 * lq1, -g * e2 * lk2, -g * e2 * lq2


# --------------------------------------------------------------------------------------------
# decode over a paged cache (a serving layout; the method is unchanged)
# --------------------------------------------------------------------------------------------

def paged_rows(block_table, seqlens, page_size: int, b: int) -> np.ndarray:
    """Pool row of every key of sequence b: key j is row j % page_size of page
    block_table[b, j // page_size], i.e. pool row block_table[b, j // page_size] * page_size +
    j % page_size."""
    L = int(np.asarray(_f64(seqlens)).astype(np.int64)[b])
    table = np.asarray(_f64(block_table)).astype(np.int64)
    j = np.arange(L)
    return table[b, j // page_size] * page_size + j % page_size


def diffattn_decode_paged(q, k_pool, v_pool, block_table, seqlens, lam, lam_init: float,
                          norm_weight=None, eps: float = 1e-5, norm: bool = True,
                          apply_scale: bool = True):
    """`diffattn_decode` over a cache held in pages: k_pool [num_pages, page_size, H, 2d],
    v_pool [num_pages, page_size, H, dv], block_table [B, max_pages], seqlens [B]. Each sequence's
    keys are gathered from the pool in order, then decoded as a contiguous cache."""
    num_pages, page_size, H, w = k_pool.shape
    kp = _f64(k_pool).reshape(num_pages * page_size, H, w)
    vp = _f64(v_pool).reshape(num_pages * page_size, H, v_pool.shape[-1])
    B = q.shape[0]
    sl = np.asarray(_f64(seqlens)).astype(np.int64)
    L = int(sl.max())
    kc = np.zeros((B, L, H, w))
    vc = np.zeros((B, L, H, vp.shape[-1]))
    for b in range(B):
        rows = paged_rows(block_table, seqlens, page_size, b)
        kc[b, :rows.size] = kp[rows]
        vc[b, :rows.size] = vp[rows]
    return diffattn_decode(q, kc, vc, sl, lam, lam_init, norm_weight, eps, norm, apply_scale)


def diffattn_v2_decode_paged(q, k_pool, v_pool, block_table, seqlens, lam_logit):
    """`diffattn_v2_decode` over a cache held in pages: k_pool, v_pool [num_pages, page_size,
    Hkv, d], block_table [B, max_pages], seqlens [B]. Each sequence's keys are gathered from the
    pool in order, then decoded as a contiguous cache."""
    num_pages, page_size, Hkv, w = k_pool.shape
    kp = _f64(k_pool).reshape(num_pages * page_size, Hkv, w)
    vp = _f64(v_pool).reshape(num_pages * page_size, Hkv, v_pool.shape[-1])
    B = q.shape[0]
    sl = np.asarray(_f64(seqlens)).astype(np.int64)
    L = int(sl.max())
    kc = np.zeros((B, L, Hkv, w))
    vc = np.zeros((B, L, Hkv, vp.shape[-1]))
    for b in range(B):
        rows = paged_rows(block_table, seqlens, page_size, b)
        kc[b, :rows.size] = kp[rows]
        vc[b, :rows.size] = vp[rows]
    return diffattn_v2_decode(q, kc, vc, sl, lam_logit)


def diffattn_gda_decode_paged(q, k_pool, v_pool, block_table, seqlens, lam, lam_init: float,
                              n_signal: int, norm_weight=None, eps: float = 1e-5,
                              norm: bool = True, apply_scale: bool = True):
    """`diffattn_gda_decode` over a cache held in pages: k_pool [num_pages, page_size, Hs + Hn, d],
    v_pool [num_pages, page_size, Hs, dv], block_table [B, max_pages], seqlens [B]. Each
    sequence's keys are gathered from the pool in order, then decoded as a contiguous cache."""
    num_pages, page_size, heads, w = k_pool.shape
    kp = _f64(k_pool).reshape(num_pages * page_size, heads, w)
    vp = _f64(v_pool).reshape(num_pages * page_size, v_pool.shape[2], v_pool.shape[-1])
    B = q.shape[0]
    sl = np.asarray(_f64(seqlens)).astype(np.int64)
    L = int(sl.max())
    kc = np.zeros((B, L, heads, w))
    vc = np.zeros((B, L, vp.shape[1], vp.shape[-1]))
    for b in range(B):
        rows = paged_rows(block_table, seqlens, page_size, b)
        kc[b, :rows.size] = kp[rows]
        vc[b, :rows.size] = vp[rows]
    return diffattn_gda_decode(q, kc, vc, sl, lam, lam_init, n_signal, norm_weight, eps, norm,
                               apply_scale)


# --------------------------------------------------------------------------------------------
# variable-length prefill (packed sequences; the operator per sequence is unchanged)
# --------------------------------------------------------------------------------------------

def varlen_segments(cu_seqlens) -> list:
    """(start, end) rows of each packed sequence from the offsets cu_seqlens [B + 1]."""
    cu = np.asarray(_f64(cu_seqlens)).astype(np.int64)
    return [(int(cu[i]), int(cu[i + 1])) for i in range(cu.size - 1)]


def diffattn_fwd_varlen(q, k, v, cu_seqlens, lam, lam_init: float, norm_weight=None,
                        eps: float = 1e-5, norm: bool = True, apply_scale: bool = True,
                        causal: bool = True):
    """`diffattn_fwd` applied to each sequence of a packed batch on its own: q, k [total, H, 2d],
    v [total, H, dv]; sequence b is rows cu_seqlens[b] .. cu_seqlens[b+1]-1. Returns float64
    [total, H, dv]; rows in no sequence are 0."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    out = np.zeros((q.shape[0], q.shape[1], v.shape[-1]))
    for s0, s1 in varlen_segments(cu_seqlens):
        if s1 > s0:
            out[s0:s1] = diffattn_fwd(q[None, s0:s1], k[None, s0:s1], v[None, s0:s1], lam, lam_init,
                                      norm_weight, eps, norm, apply_scale, causal)[0]
    return out


# --------------------------------------------------------------------------------------------
# queries and keys of their own lengths (a prompt in chunks, several new tokens over a cache);
# the operator per query row is unchanged ([P3] "The mechanism, exactly")
# --------------------------------------------------------------------------------------------

def query_positions(Lq: int, Lk: int) -> np.ndarray:
    """Positions of a sequence's Lq queries among its Lk keys: they are the last Lq."""
    return np.arange(Lq) + (Lk - Lq)


def diffattn_fwd_varlen_qk(q, k, v, cu_seqlens_q, cu_seqlens_k, lam, lam_init: float,
                           norm_weight=None, eps: float = 1e-5, norm: bool = True,
                           apply_scale: bool = True, causal: bool = True):
    """Packed prefill where sequence b has keys k, v rows cu_seqlens_k[b] .. cu_seqlens_k[b+1]-1
    and queries q rows cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1, its last Lq positions; the query
    at position p sees keys 0 .. p (causal) or all Lk keys. q, k [*, H, 2d] = [Q1|Q2], [K1|K2];
    v [*, H, dv]. Returns float64 [total_q, H, dv]; rows in no sequence are 0."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    H, two_d = q.shape[1], q.shape[2]
    d = two_d // 2
    lam = np.broadcast_to(_f64(lam), (H,))
    out = np.zeros((q.shape[0], H, v.shape[-1]))
    for (q0, q1), (k0, k1) in zip(varlen_segments(cu_seqlens_q), varlen_segments(cu_seqlens_k)):
        if q1 == q0:
            continue
        pos = query_positions(q1 - q0, k1 - k0)
        for h in range(H):
            for s in range(0, q1 - q0, ROW_BLOCK):
                r = slice(q0 + s, min(q1, q0 + s + ROW_BLOCK))
                p = pos[s:s + ROW_BLOCK]
                S1 = scores(q[r, h, :d], k[k0:k1, h, :d], p, causal)
                S2 = scores(q[r, h, d:], k[k0:k1, h, d:], p, causal)
                O = diff_weights(S1, S2, float(lam[h])) @ v[k0:k1, h, :]
                out[r, h, :] = head_epilogue(O, norm_weight, eps, lam_init, norm, apply_scale)
    return out


def diffattn_v2_fwd_varlen(q, k, v, lam_logit, cu_seqlens_q, cu_seqlens_k=None,
                           causal: bool = True):
    """`diffattn_v2_fwd` per packed sequence: q [total_q, Hq, d], k, v [total_k, Hkv, d],
    lam_logit [total_q, Hq/2]; sequence b's queries are rows cu_seqlens_q[b] .. of q, its keys
    rows cu_seqlens_k[b] .. of k and v (cu_seqlens_q when None), the queries being its last Lq
    positions. Returns float64 [total_q, Hq/2, d]; rows in no sequence are 0."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    Hq, d = q.shape[1], q.shape[2]
    Hkv = k.shape[1]
    sig = sigmoid(lam_logit)
    out = np.zeros((q.shape[0], Hq // 2, v.shape[-1]))
    cu_k = cu_seqlens_q if cu_seqlens_k is None else cu_seqlens_k
    for (q0, q1), (k0, k1) in zip(varlen_segments(cu_seqlens_q), varlen_segments(cu_k)):
        if q1 == q0:
            continue
        pos = query_positions(q1 - q0, k1 - k0)
        for p in range(Hq // 2):
            g = v2_kv_head(p, Hq, Hkv)
            kg, vg = k[k0:k1, g], v[k0:k1, g]
            for s in range(0, q1 - q0, ROW_BLOCK):
                r = slice(q0 + s, min(q1, q0 + s + ROW_BLOCK))
                ps = pos[s:s + ROW_BLOCK]
                a1 = softmax_rows(scores(q[r, 2 * p], kg, ps, causal)) @ vg
                a2 = softmax_rows(scores(q[r, 2 * p + 1], kg, ps, causal)) @ vg
                out[r, p, :] = a1 - sig[r, p][:, None] * a2
    return out


def gather_pages(pool, block_table, seqlens_k):
    """Each sequence's keys read from a page pool [num_pages, page_size, ...] in order, packed one
    sequence after another: returns (rows [sum(seqlens_k), ...], offsets [B + 1])."""
    num_pages, page_size = pool.shape[0], pool.shape[1]
    flat = _f64(pool).reshape((num_pages * page_size,) + tuple(pool.shape[2:]))
    B = int(np.asarray(_f64(seqlens_k)).size)
    rows = [paged_rows(block_table, seqlens_k, page_size, b) for b in range(B)]
    cu = np.concatenate([[0], np.cumsum([r.size for r in rows])]).astype(np.int64)
    idx = np.concatenate(rows).astype(np.int64) if B else np.zeros(0, dtype=np.int64)
    return flat[idx], cu


def diffattn_fwd_paged(q, k_pool, v_pool, cu_seqlens_q, seqlens_k, block_table, lam,
                       lam_init: float, norm_weight=None, eps: float = 1e-5, norm: bool = True,
                       apply_scale: bool = True, causal: bool = True):
    """`diffattn_fwd_varlen_qk` with each sequence's keys read from page pools k_pool
    [num_pages, page_size, H, 2d], v_pool [.., H, dv] through block_table [B, max_pages]."""
    k, cu_k = gather_pages(k_pool, block_table, seqlens_k)
    v, _ = gather_pages(v_pool, block_table, seqlens_k)
    return diffattn_fwd_varlen_qk(q, k, v, cu_seqlens_q, cu_k, lam, lam_init, norm_weight, eps,
                                  norm, apply_scale, causal)


def diffattn_v2_fwd_paged(q, k_pool, v_pool, lam_logit, cu_seqlens_q, seqlens_k, block_table,
                          causal: bool = True):
    """`diffattn_v2_fwd_varlen` with each sequence's keys read from page pools k_pool, v_pool
    [num_pages, page_size, Hkv, d] through block_table [B, max_pages]."""
    k, cu_k = gather_pages(k_pool, block_table, seqlens_k)
    v, _ = gather_pages(v_pool, block_table, seqlens_k)
    return diffattn_v2_fwd_varlen(q, k, v, lam_logit, cu_seqlens_q, cu_k, causal)


def diffattn_bwd_varlen(q, k, v, cu_seqlens, lam, lam_init: float, dy, norm_weight=None,
                        eps: float = 1e-5, norm: bool = True, apply_scale: bool = True,
                        causal: bool = True):
    """`diffattn_bwd` over packed sequences (q, k [total, H, 2d], v, dy [total, H, dv]): each
    sequence's gradients are those of its own forward; dlam and dw sum over the sequences. Rows in
    no sequence get zero gradients."""
    q, k, v, dy = _f64(q), _f64(k), _f64(v), _f64(dy)
    H = q.shape[1]
    out = dict(dq=np.zeros_like(q), dk=np.zeros_like(k), dv=np.zeros_like(v),
               dlam=np.zeros(H), dw=np.zeros(v.shape[-1]))
    for s0, s1 in varlen_segments(cu_seqlens):
        if s1 == s0:
            continue
        g = diffattn_bwd(q[None, s0:s1], k[None, s0:s1], v[None, s0:s1], lam, lam_init,
                         dy[None, s0:s1], norm_weight, eps, norm, apply_scale, causal)
        for name in ("dq", "dk", "dv"):
            out[name][s0:s1] = g[name][0]
        out["dlam"] += g["dlam"]
        out["dw"] += g["dw"]
    return out


# --------------------------------------------------------------------------------------------
# grouped differential attention: several signal heads subtract one shared noise head
# ([P3] "What other people found": the Grouped Differential Attention result, 3 or 4 signal
# heads per noise head against 1:1)
# --------------------------------------------------------------------------------------------

def gda_noise_head(h: int, n_signal: int, n_noise: int) -> int:
    """Noise head whose map signal head h subtracts: signal heads are split into n_noise
    contiguous groups of G = n_signal / n_noise, as the query heads of a GQA group are, so head h
    takes noise head floor(h / G)."""
    return h // (n_signal // n_noise)


def diffattn_gda_fwd(q, k, v, lam, lam_init: float, n_signal: int, norm_weight=None,
                     eps: float = 1e-5, norm: bool = True, apply_scale: bool = True,
                     causal: bool = True, rows=None):
    """Grouped prefill: signal head h computes (softmax(Q1_h K1_h^T/sqrt d) - lam[h]
    softmax(Q2_g K2_g^T/sqrt d)) V_h with g = gda_noise_head(h), then the per-head norm and the
    (1 - lambda_init) scale of the ungrouped operator.

    q, k [B, N, Hs + Hn, d]: heads 0 .. Hs-1 hold the signal heads' Q1 (K1), heads Hs .. Hs+Hn-1
    the noise heads' Q2 (K2). v [B, N, Hs, dv]. lam [Hs] or a scalar.
    Returns float64 [B, len(rows), Hs, dv].
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, N, heads, d = q.shape
    Hs = n_signal
    Hn = heads - Hs
    lam = np.broadcast_to(_f64(lam), (Hs,))
    rows = np.arange(N) if rows is None else np.asarray(rows)
    out = np.empty((B, rows.shape[0], Hs, v.shape[-1]), dtype=np.float64)
    for b in range(B):
        for h in range(Hs):
            g = Hs + gda_noise_head(h, Hs, Hn)
            O = diff_attn_head(q[b, :, h], k[b, :, h], q[b, :, g], k[b, :, g], v[b, :, h],
                               float(lam[h]), causal, rows)
            out[b, :, h, :] = head_epilogue(O, norm_weight, eps, lam_init, norm, apply_scale)
    return out


def diffattn_gda_fwd_varlen(q, k, v, cu_seqlens, lam, lam_init: float, n_signal: int,
                            norm_weight=None, eps: float = 1e-5, norm: bool = True,
                            apply_scale: bool = True, causal: bool = True):
    """`diffattn_gda_fwd` applied to each sequence of a packed batch on its own: q, k
    [total, Hs + Hn, d], v [total, Hs, dv]; sequence b is rows cu_seqlens[b] .. cu_seqlens[b+1]-1.
    Returns float64 [total, Hs, dv]; rows in no sequence are 0."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    out = np.zeros((q.shape[0], n_signal, v.shape[-1]))
    for s0, s1 in varlen_segments(cu_seqlens):
        if s1 > s0:
            out[s0:s1] = diffattn_gda_fwd(q[None, s0:s1], k[None, s0:s1], v[None, s0:s1], lam,
                                          lam_init, n_signal, norm_weight, eps, norm, apply_scale,
                                          causal)[0]
    return out


def diffattn_gda_fwd_varlen_qk(q, k, v, cu_seqlens_q, cu_seqlens_k, lam, lam_init: float,
                               n_signal: int, norm_weight=None, eps: float = 1e-5,
                               norm: bool = True, apply_scale: bool = True, causal: bool = True):
    """`diffattn_gda_fwd` where sequence b has keys k, v rows cu_seqlens_k[b] .. and queries q
    rows cu_seqlens_q[b] .., its last Lq positions (as in `diffattn_fwd_varlen_qk`). q, k
    [*, Hs + Hn, d], v [*, Hs, dv]. Each sequence's queries are placed at their positions among
    Lk and the grouped prefill is taken on those rows only. Returns float64 [total_q, Hs, dv];
    rows in no sequence are 0."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    out = np.zeros((q.shape[0], n_signal, v.shape[-1]))
    for (q0, q1), (k0, k1) in zip(varlen_segments(cu_seqlens_q), varlen_segments(cu_seqlens_k)):
        if q1 == q0:
            continue
        pos = query_positions(q1 - q0, k1 - k0)
        q_full = np.zeros((1, k1 - k0) + q.shape[1:])
        q_full[0, pos] = q[q0:q1]
        out[q0:q1] = diffattn_gda_fwd(q_full, k[None, k0:k1], v[None, k0:k1], lam, lam_init,
                                      n_signal, norm_weight, eps, norm, apply_scale, causal,
                                      rows=pos)[0]
    return out


def diffattn_gda_fwd_paged(q, k_pool, v_pool, cu_seqlens_q, seqlens_k, block_table, lam,
                           lam_init: float, n_signal: int, norm_weight=None, eps: float = 1e-5,
                           norm: bool = True, apply_scale: bool = True, causal: bool = True):
    """`diffattn_gda_fwd_varlen_qk` with each sequence's keys read from page pools k_pool
    [num_pages, page_size, Hs + Hn, d], v_pool [.., Hs, dv] through block_table [B, max_pages]."""
    k, cu_k = gather_pages(k_pool, block_table, seqlens_k)
    v, _ = gather_pages(v_pool, block_table, seqlens_k)
    return diffattn_gda_fwd_varlen_qk(q, k, v, cu_seqlens_q, cu_k, lam, lam_init, n_signal,
                                      norm_weight, eps, norm, apply_scale, causal)


def diffattn_gda_bwd(q, k, v, lam, lam_init: float, n_signal: int, dy, norm_weight=None,
                     eps: float = 1e-5, norm: bool = True, apply_scale: bool = True,
                     causal: bool = True):
    """Backward of `diffattn_gda_fwd` for the upstream gradient dy [B, N, Hs, dv]. Signal head h's
    operator is the ungrouped one with map 2 taken from noise head g = Hs + gda_noise_head(h), so
    its gradients are those of `diff_attn_head_bwd`; a noise head's dQ2 and dK2 are the sums of
    the contributions of the signal heads of its group.

    Returns dict(dq [B,N,Hs+Hn,d], dk [B,N,Hs+Hn,d], dv [B,N,Hs,dv], dlam [Hs], dw [dv]) in
    float64 (dw: the norm weight's gradient, zeros without the norm)."""
    q, k, v, dy = _f64(q), _f64(k), _f64(v), _f64(dy)
    B, N, heads, d = q.shape
    Hs = n_signal
    Hn = heads - Hs
    lam = np.broadcast_to(_f64(lam), (Hs,))
    s = (1.0 - lam_init) if apply_scale else 1.0
    out = dict(dq=np.zeros_like(q), dk=np.zeros_like(k), dv=np.zeros_like(v),
               dlam=np.zeros(Hs), dw=np.zeros(v.shape[-1]))
    for b in range(B):
        for h in range(Hs):
            g = Hs + gda_noise_head(h, Hs, Hn)
            q1, k1, q2, k2 = q[b, :, h], k[b, :, h], q[b, :, g], k[b, :, g]
            O = diff_attn_head(q1, k1, q2, k2, v[b, :, h], float(lam[h]), causal)
            dYs = dy[b, :, h] * s
            if norm:
                dO, dwh = subln_bwd(O, norm_weight, eps, dYs)
                out["dw"] += dwh
            else:
                dO = dYs
            dq1, dk1, dq2, dk2, dvh, dl = diff_attn_head_bwd(q1, k1, q2, k2, v[b, :, h],
                                                              float(lam[h]), causal, dO)
            out["dq"][b, :, h] += dq1
            out["dk"][b, :, h] += dk1
            out["dq"][b, :, g] += dq2
            out["dk"][b, :, g] += dk2
            out["dv"][b, :, h] = dvh
            out["dlam"][h] += dl
    return out


def diffattn_gda_bwd_varlen(q, k, v, cu_seqlens, lam, lam_init: float, n_signal: int, dy,
                            norm_weight=None, eps: float = 1e-5, norm: bool = True,
                            apply_scale: bool = True, causal: bool = True):
    """`diffattn_gda_bwd` over packed sequences (q, k [total, Hs + Hn, d], v, dy [total, Hs, dv]):
    each sequence's gradients are those of its own grouped forward; dlam and dw sum over the
    sequences. Rows in no sequence get zero gradients."""
    q, k, v, dy = _f64(q), _f64(k), _f64(v), _f64(dy)
    out = dict(dq=np.zeros_like(q), dk=np.zeros_like(k), dv=np.zeros_like(v),
               dlam=np.zeros(n_signal), dw=np.zeros(v.shape[-1]))
    for s0, s1 in varlen_segments(cu_seqlens):
        if s1 == s0:
            continue
        g = diffattn_gda_bwd(q[None, s0:s1], k[None, s0:s1], v[None, s0:s1], lam, lam_init,
                             n_signal, dy[None, s0:s1], norm_weight, eps, norm, apply_scale,
                             causal)
        for name in ("dq", "dk", "dv"):
            out[name][s0:s1] = g[name][0]
        out["dlam"] += g["dlam"]
        out["dw"] += g["dw"]
    return out


def diffattn_gda_decode(q, k_cache, v_cache, seqlens, lam, lam_init: float, n_signal: int,
                        norm_weight=None, eps: float = 1e-5, norm: bool = True,
                        apply_scale: bool = True):
    """Grouped decode: one query per sequence over its cached keys 0 .. seqlens[b]-1 (no mask
    inside that range). q [B, Hs + Hn, d], k_cache [B, L, Hs + Hn, d] (signal heads first, as in
    `diffattn_gda_fwd`), v_cache [B, L, Hs, dv]. Returns float64 [B, Hs, dv]."""
    q = _f64(q)
    B, heads, d = q.shape
    Hs = n_signal
    Hn = heads - Hs
    lam = np.broadcast_to(_f64(lam), (Hs,))
    seqlens = np.asarray(_f64(seqlens)).astype(np.int64)
    out = np.empty((B, Hs, v_cache.shape[-1]), dtype=np.float64)
    for b in range(B):
        L = int(seqlens[b])
        kb, vb = _f64(k_cache[b, :L]), _f64(v_cache[b, :L])
        for h in range(Hs):
            g = Hs + gda_noise_head(h, Hs, Hn)
            O = diff_attn_head(q[b, h:h + 1], kb[:, h], q[b, g:g + 1], kb[:, g], vb[:, h],
                               float(lam[h]), causal=False)
            out[b, h, :] = head_epilogue(O, norm_weight, eps, lam_init, norm, apply_scale)[0]
    return out
