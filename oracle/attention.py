"""Float64 oracle: paged (BSR) attention and the attention-state merge.

Test infrastructure only (see the package docstring).  Plain, slow and direct:
every step is the definition, written with numpy primitives.

What is computed (page "FlashInfer：面向 LLM 推理服务的高效可定制注意力引擎"):
  * The KV-cache is a block-sparse-row matrix whose non-zero blocks are the
    physical pages a request reads (核心机制 1 "统一 KV-Cache 存储", paper
    §3.1.1, Figure 2).  Request i owns pages kv_indices[kv_indptr[i]:kv_indptr[i+1]];
    every page is full except the last, which holds last_page_len[i] tokens.
  * Queries and outputs are ragged, padding-free tensors packed by qo_indptr
    (术语与记号 "ragged 张量", paper §3.1.1).
  * The canonical output of attention is the state (O, LSE): the output vector
    and the log-sum-exp of the scores; a merge operator on states is
    associative and commutative, which is what lets the KV be split into chunks
    (术语与记号 "Attention State 与 ⊕", paper §2.2).
  * Grouped-query heads: query head h reads KV head floor(h / g), g = H_qo / H_kv
    (术语与记号 "GQA 头组融合", paper Appendix A).

Readings where the pages are silent (each listed in the design notes):
  * LSE uses the natural logarithm and includes the softmax scale:
    LSE = log sum_j exp(scale * q.k_j).
  * The merge of (O_a, s_a) and (O_b, s_b) is the unique one consistent with
    that definition: s = log(e^s_a + e^s_b), O = e^(s_a - s) O_a + e^(s_b - s) O_b;
    its identity is (0, -inf).
  * A row with no visible keys has O = 0 and LSE = -inf (the identity state).
  * Causal masks are aligned to the end of each request's KV: query token t
    (0-based within its request) sees keys j <= l_kv - l_q + t.
  * Page layout "HND" is [pages, H_kv, page_size, D]; "NHD" is [pages, page_size, H_kv, D].

Attention variants (问题背景 挑战二 names sliding-window masks and Grok's logit
soft-cap among the variants a serving library must carry; 核心机制 5, paper
§3.2.3, treats them as logits transforms and masks of one template):
  * Sliding window, read with causal masks: query token t, aligned at position
    p = l_kv - l_q + t, sees keys p - window_left .. p (window_left + 1 keys).
  * Logit soft-cap: the scaled logit x = scale * q.k becomes cap * tanh(x / cap)
    before the softmax, so every logit lies in (-cap, cap).

FP8 KV (核心机制 8 / paper App. F lists FP8 KV-cache support; reading): pages may
hold e4m3 codes with one scale per tensor, K = k_scale * e4m3(K code) and
likewise V.  e4m3 is the 8-bit float with 1 sign bit, 4 exponent bits (bias 7)
and 3 mantissa bits: exponent field 0 encodes subnormals m/8 * 2^-6, field 15
with mantissa 7 encodes NaN, there are no infinities, and the largest finite
value is 1.75 * 2^8 = 448.
"""
from __future__ import annotations

import numpy as np

NEG_INF = -np.inf


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> exact float64 values (bf16 is the top half of an f32)."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def e4m3_to_f64(codes: np.ndarray) -> np.ndarray:
    """e4m3 codes (uint8) -> float64: sign * (1 + m/8) * 2^(e - 7), or sign * (m/8) * 2^-6 when e = 0."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


def request_lengths(qo_indptr, kv_indptr, last_page_len, page_size):
    """Per-request query length l_q and KV length l_kv (BSR block row i, paper §3.1.1).

    l_kv = (pages - 1) * page_size + last_page_len when the request has pages, else 0.
    """
    qo = np.asarray(qo_indptr, dtype=np.int64)
    kv = np.asarray(kv_indptr, dtype=np.int64)
    last = np.asarray(last_page_len, dtype=np.int64)
    l_q = qo[1:] - qo[:-1]
    n_pages = kv[1:] - kv[:-1]
    l_kv = np.where(n_pages > 0, (n_pages - 1) * page_size + last, 0)
    return l_q, l_kv


def gather_kv(pages: np.ndarray, kv_indptr, kv_indices, l_kv: int, page_size: int, i: int, kv_head: int,
              layout: str = "HND") -> np.ndarray:
    """Rows 0..l_kv-1 of request i's KV for one KV head, as float64 [l_kv, D].

    Walks the request's page list in order; token p lives in page
    kv_indices[kv_indptr[i] + p // page_size] at row p % page_size.
    """
    base = int(kv_indptr[i])
    p = np.arange(l_kv, dtype=np.int64)
    page = np.asarray(kv_indices, dtype=np.int64)[base + p // page_size]
    r = p % page_size
    if layout == "HND":
        rows = pages[page, kv_head, r]
    elif layout == "NHD":
        rows = pages[page, r, kv_head]
    else:
        raise ValueError(layout)
    if pages.dtype == np.uint16:
        return bf16_to_f64(rows)
    if pages.dtype == np.uint8:
        return e4m3_to_f64(rows)
    return np.asarray(rows, dtype=np.float64)


def visible_counts(l_q: int, l_kv: int, causal: bool) -> np.ndarray:
    """Number of keys each query token of a request sees (keys 0..count-1)."""
    t = np.arange(l_q, dtype=np.int64)
    if not causal:
        return np.full(l_q, l_kv, dtype=np.int64)
    return np.clip(l_kv - l_q + t + 1, 0, l_kv)


def window_starts(l_q: int, l_kv: int, window_left: int) -> np.ndarray:
    """First key each query token sees under a sliding window (0 without one): max(0, p - window_left)."""
    t = np.arange(l_q, dtype=np.int64)
    if window_left < 0:
        return np.zeros(l_q, dtype=np.int64)
    return np.maximum(0, l_kv - l_q + t - window_left)


def attention_state(q_rows: np.ndarray, k: np.ndarray, v: np.ndarray, n_visible, scale: float, first=0,
                    soft_cap: float = 0.0):
    """State (O, LSE) of each query row over keys first[r] .. n_visible[r]-1, in float64.

    s_j = scale * q . k_j (then cap * tanh(s_j / cap) when soft_cap > 0) ;  M = max_j s_j ;
    LSE = M + log sum_j exp(s_j - M) ;  O = sum_j exp(s_j - LSE) v_j .
    A row with no visible key gets (0, -inf).
    """
    q_rows = np.asarray(q_rows, dtype=np.float64)
    n_rows, d = q_rows.shape
    o = np.zeros((n_rows, v.shape[1] if v.ndim == 2 else d), dtype=np.float64)
    lse = np.full(n_rows, NEG_INF, dtype=np.float64)
    n_visible = np.broadcast_to(np.asarray(n_visible, dtype=np.int64), (n_rows,))
    first = np.broadcast_to(np.asarray(first, dtype=np.int64), (n_rows,))
    if k.shape[0] == 0:
        return o, lse
    s = scale * (q_rows @ k.T)
    if soft_cap > 0:
        s = soft_cap * np.tanh(s / soft_cap)
    for r in range(n_rows):
        lo, n = int(first[r]), int(n_visible[r])
        if n <= lo:
            continue
        sr = s[r, lo:n]
        m = sr.max()
        w = np.exp(sr - m)
        z = w.sum()
        lse[r] = m + np.log(z)
        o[r] = (w @ v[lo:n]) / z
    return o, lse


def batch_attention(b, layout: str = "HND", requests=None, scale: float | None = None, window_left: int = -1,
                    soft_cap: float = 0.0, k_scale: float = 1.0, v_scale: float = 1.0):
    """O [total_q, H_qo, D] and LSE [total_q, H_qo] (float64) for a paged batch.

    `b` carries the library's input arrays (see serving_attention_plan_gb300.workloads.PagedBatch).
    Rows of requests not in `requests` (when given) are left as (0, -inf).  A sliding window
    (window_left >= 0) needs a causal batch.
    """
    if window_left >= 0 and not b.causal:
        raise ValueError("the sliding window is read with causal masks")
    d = b.head_dim
    scale = 1.0 / np.sqrt(d) if scale is None else scale
    g = b.num_qo_heads // b.num_kv_heads
    l_q, l_kv = request_lengths(b.qo_indptr, b.kv_indptr, b.last_page_len, b.page_size)
    total_q = int(b.qo_indptr[-1])
    o = np.zeros((total_q, b.num_qo_heads, d), dtype=np.float64)
    lse = np.full((total_q, b.num_qo_heads), NEG_INF, dtype=np.float64)
    reqs = range(len(l_q)) if requests is None else requests
    for i in reqs:
        q0, nq, nk = int(b.qo_indptr[i]), int(l_q[i]), int(l_kv[i])
        if nq == 0:
            continue
        vis = visible_counts(nq, nk, b.causal)
        lo = window_starts(nq, nk, window_left)
        for hk in range(b.num_kv_heads):
            k = k_scale * gather_kv(b.k_pages, b.kv_indptr, b.kv_indices, nk, b.page_size, i, hk, layout)
            v = v_scale * gather_kv(b.v_pages, b.kv_indptr, b.kv_indices, nk, b.page_size, i, hk, layout)
            for h in range(hk * g, (hk + 1) * g):
                qr = bf16_to_f64(b.q[q0:q0 + nq, h])
                oo, ll = attention_state(qr, k, v, vis, scale, lo, soft_cap)
                o[q0:q0 + nq, h] = oo
                lse[q0:q0 + nq, h] = ll
    return o, lse


def attention_rows(b, i: int, h: int, tokens, layout: str = "HND", scale: float | None = None,
                   window_left: int = -1, soft_cap: float = 0.0, k_scale: float = 1.0, v_scale: float = 1.0):
    """State of selected query tokens (0-based within request i) of query head h."""
    if window_left >= 0 and not b.causal:
        raise ValueError("the sliding window is read with causal masks")
    d = b.head_dim
    scale = 1.0 / np.sqrt(d) if scale is None else scale
    g = b.num_qo_heads // b.num_kv_heads
    l_q, l_kv = request_lengths(b.qo_indptr, b.kv_indptr, b.last_page_len, b.page_size)
    nq, nk = int(l_q[i]), int(l_kv[i])
    tokens = np.asarray(tokens, dtype=np.int64)
    vis = visible_counts(nq, nk, b.causal)[tokens]
    lo = window_starts(nq, nk, window_left)[tokens]
    k = k_scale * gather_kv(b.k_pages, b.kv_indptr, b.kv_indices, nk, b.page_size, i, h // g, layout)
    v = v_scale * gather_kv(b.v_pages, b.kv_indptr, b.kv_indices, nk, b.page_size, i, h // g, layout)
    qr = bf16_to_f64(b.q[int(b.qo_indptr[i]) + tokens, h])
    return attention_state(qr, k, v, vis, scale, lo, soft_cap)


def merge_states(o_a, lse_a, o_b, lse_b):
    """(O_a, s_a) merged with (O_b, s_b): s = log(e^s_a + e^s_b), O = e^(s_a-s) O_a + e^(s_b-s) O_b.

    Evaluated with m = max(s_a, s_b) so no exponent overflows; two empty states
    (s = -inf) merge to the empty state (0, -inf).
    """
    o_a = np.asarray(o_a, dtype=np.float64)
    o_b = np.asarray(o_b, dtype=np.float64)
    lse_a = np.asarray(lse_a, dtype=np.float64)
    lse_b = np.asarray(lse_b, dtype=np.float64)
    m = np.maximum(lse_a, lse_b)
    both_empty = np.isneginf(m)
    m_safe = np.where(both_empty, 0.0, m)
    wa = np.where(np.isneginf(lse_a), 0.0, np.exp(lse_a - m_safe))
    wb = np.where(np.isneginf(lse_b), 0.0, np.exp(lse_b - m_safe))
    z = wa + wb
    z_safe = np.where(both_empty, 1.0, z)
    lse = np.where(both_empty, NEG_INF, m_safe + np.log(z_safe))
    o = (wa[..., None] * o_a + wb[..., None] * o_b) / z_safe[..., None]
    o = np.where(both_empty[..., None], 0.0, o)
    return o, lse
