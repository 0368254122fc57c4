"""Seeded synthetic inputs for paged serving attention.

This module only draws random numbers and lays them out as a block-sparse-row
(BSR) paged KV-cache plus ragged queries.  It holds none of the attention
arithmetic: the CPU oracle and the CUDA library both consume what it returns.

Layouts (the ones the library's C ABI takes):
  q        uint16 bf16 bits, [total_q, H_qo, D]   ragged rows packed by qo_indptr
  k_pages  uint16 bf16 bits, [P, H_kv, page_size, D]   ("HND" page layout)
  v_pages  same as k_pages
  qo_indptr [B+1], kv_indptr [B+1], kv_indices [nnz], last_page_len [B]: int32

The BSR view follows "FlashInfer: Efficient and Customizable Attention Engine
for LLM Inference Serving" (MLSys 2025), section 3.1.1 and Figure 2: each
request's KV is a list of pages (the non-zero blocks of one block row), the
last page possibly partly filled.  Section 3.1.2 / Figure 3 (composable formats)
motivates the shared-prefix workload, whose two sub-matrices share one page pool.

Recipe per workload (seed = workload index): draw lengths, then the page
permutation, then Q, then the K pool, then the V pool, all from
numpy.random.default_rng(seed); samples are float32 standard normals (times a
scale) rounded to bf16 with round-to-nearest-even.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

HEAD_DIM = 128


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); return the uint16 bit patterns.

    Inputs are finite normal samples, so the NaN/overflow corner of the rounding
    never arises here.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def _bf16_normals(rng: np.random.Generator, shape, scale: float) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if scale != 1.0:
        x *= np.float32(scale)
    return f32_to_bf16_bits(x)


@dataclass
class PagedBatch:
    """One batch in the library's input format (all arrays host-side numpy)."""

    name: str
    num_qo_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    causal: bool
    qo_indptr: np.ndarray
    kv_indptr: np.ndarray
    kv_indices: np.ndarray
    last_page_len: np.ndarray
    q: np.ndarray
    k_pages: np.ndarray
    v_pages: np.ndarray
    meta: dict = field(default_factory=dict)

    @property
    def batch_size(self) -> int:
        return int(self.qo_indptr.shape[0] - 1)

    @property
    def num_pages(self) -> int:
        return int(self.k_pages.shape[0])

    @property
    def total_q(self) -> int:
        return int(self.qo_indptr[-1])


@dataclass
class SharedPrefixBatch:
    """Composable-format workload: one shared prefix block row plus per-request suffixes.

    `prefix` has a single block row holding all requests' query tokens (Br = number
    of requests); `suffix` has one block row per request (Br = 1); `flat` is the same
    attention as one plain paged batch (prefix pages followed by each request's own
    pages).  All three share q and the page pool; no KV data is duplicated.
    """

    prefix: PagedBatch
    suffix: PagedBatch
    flat: PagedBatch


def _pages_from_lengths(lengths: np.ndarray, page_size: int):
    n_pages = (lengths + page_size - 1) // page_size
    kv_indptr = np.zeros(lengths.shape[0] + 1, dtype=np.int64)
    kv_indptr[1:] = np.cumsum(n_pages)
    last = np.where(n_pages > 0, lengths - (n_pages - 1) * page_size, 0)
    return kv_indptr.astype(np.int32), last.astype(np.int32), int(kv_indptr[-1])


def make_paged_batch(
    rng: np.random.Generator,
    name: str,
    q_lens,
    kv_lens,
    num_qo_heads: int,
    num_kv_heads: int,
    page_size: int,
    causal: bool,
    pool_pages: int | None = None,
    scale: float = 1.0,
    head_dim: int = HEAD_DIM,
    with_data: bool = True,
) -> PagedBatch:
    """Build a paged batch from given lengths: page permutation, then Q, K pool, V pool.

    Pages of all requests are a random permutation of the pool (or, with
    `pool_pages` larger than needed, a random subset of it in random order).
    With with_data=False only the index arrays are drawn (q/k/v are empty);
    they are identical to the full draw's, since they come first.
    """
    q_lens = np.asarray(q_lens, dtype=np.int64)
    kv_lens = np.asarray(kv_lens, dtype=np.int64)
    kv_indptr, last, nnz = _pages_from_lengths(kv_lens, page_size)
    pool = nnz if pool_pages is None else int(pool_pages)
    if pool < nnz:
        raise ValueError("page pool smaller than the pages the batch needs")
    perm = rng.permutation(pool)[:nnz].astype(np.int32)
    qo_indptr = np.zeros(q_lens.shape[0] + 1, dtype=np.int32)
    qo_indptr[1:] = np.cumsum(q_lens)
    total_q = int(qo_indptr[-1])
    if with_data:
        q = _bf16_normals(rng, (total_q, num_qo_heads, head_dim), scale)
        k = _bf16_normals(rng, (pool, num_kv_heads, page_size, head_dim), scale)
        v = _bf16_normals(rng, (pool, num_kv_heads, page_size, head_dim), scale)
    else:
        q = np.zeros((0, num_qo_heads, head_dim), np.uint16)
        k = np.zeros((pool, num_kv_heads, page_size, 0), np.uint16)
        v = k
    return PagedBatch(
        name=name,
        num_qo_heads=num_qo_heads,
        num_kv_heads=num_kv_heads,
        head_dim=head_dim,
        page_size=page_size,
        causal=causal,
        qo_indptr=qo_indptr,
        kv_indptr=kv_indptr,
        kv_indices=perm,
        last_page_len=last,
        q=q,
        k_pages=k,
        v_pages=v,
    )


# ---------------------------------------------------------------------------
# The five named workloads
# ---------------------------------------------------------------------------

WORKLOADS = (
    "tiny_decode",          # B=4, 8/2 heads, page 16, KV {37,128,255,512}
    "llama3_8b_decode",     # B=128, 32/8 heads, page 16, KV ~ U[1,4096]
    "skewed_long_decode",   # B=64, 64/8 heads, page 1, 1 x 131072 + 63 x U[256,1024]
    "ragged_causal_prefill",  # B=16, 32/8 heads, page 16, q = kv ~ U[128,4096], causal
    "shared_prefix_decode",   # 64 x (8192 shared prefix + U[256,1024] own suffix)
)


def tiny_decode(with_data: bool = True) -> PagedBatch:
    rng = np.random.default_rng(0)
    kv = np.array([37, 128, 255, 512], dtype=np.int64)
    return make_paged_batch(rng, "tiny_decode", np.ones(4, np.int64), kv, 8, 2, 16, False, pool_pages=128,
                            with_data=with_data)


def llama3_8b_decode(batch: int = 128, max_kv: int = 4096, with_data: bool = True) -> PagedBatch:
    rng = np.random.default_rng(1)
    kv = rng.integers(1, max_kv + 1, size=batch)
    return make_paged_batch(rng, "llama3_8b_decode", np.ones(batch, np.int64), kv, 32, 8, 16, False,
                            with_data=with_data)


def skewed_long_decode(long_len: int = 131072, n_short: int = 63, with_data: bool = True) -> PagedBatch:
    rng = np.random.default_rng(2)
    short = rng.integers(256, 1025, size=n_short)
    kv = np.concatenate([[long_len], short]).astype(np.int64)
    return make_paged_batch(rng, "skewed_long_decode", np.ones(kv.shape[0], np.int64), kv, 64, 8, 1, False,
                            with_data=with_data)


def ragged_causal_prefill(batch: int = 16, lo: int = 128, hi: int = 4096, with_data: bool = True) -> PagedBatch:
    rng = np.random.default_rng(3)
    lens = rng.integers(lo, hi + 1, size=batch)
    return make_paged_batch(rng, "ragged_causal_prefill", lens, lens, 32, 8, 16, True, scale=0.5,
                            with_data=with_data)


def shared_prefix_decode(n_req: int = 64, prefix_len: int = 8192, lo: int = 256, hi: int = 1024) -> SharedPrefixBatch:
    """64 one-token requests sharing a page-aligned prefix, each with its own suffix pages."""
    page_size, hq, hk = 16, 32, 8
    if prefix_len % page_size:
        raise ValueError("the shared prefix must fill whole pages")
    rng = np.random.default_rng(4)
    suf = rng.integers(lo, hi + 1, size=n_req).astype(np.int64)
    pre_pages = prefix_len // page_size
    s_indptr, s_last, s_nnz = _pages_from_lengths(suf, page_size)
    pool = pre_pages + s_nnz
    perm = rng.permutation(pool).astype(np.int32)
    q = _bf16_normals(rng, (n_req, hq, HEAD_DIM), 1.0)
    k = _bf16_normals(rng, (pool, hk, page_size, HEAD_DIM), 1.0)
    v = _bf16_normals(rng, (pool, hk, page_size, HEAD_DIM), 1.0)
    pre_idx = perm[:pre_pages]
    suf_idx = perm[pre_pages:]
    ones = np.arange(n_req + 1, dtype=np.int32)
    prefix = PagedBatch(
        "shared_prefix_decode/prefix", hq, hk, HEAD_DIM, page_size, False,
        qo_indptr=np.array([0, n_req], np.int32),
        kv_indptr=np.array([0, pre_pages], np.int32),
        kv_indices=pre_idx.copy(),
        last_page_len=np.array([page_size], np.int32),
        q=q, k_pages=k, v_pages=v,
    )
    suffix = PagedBatch(
        "shared_prefix_decode/suffix", hq, hk, HEAD_DIM, page_size, False,
        qo_indptr=ones.copy(), kv_indptr=s_indptr, kv_indices=suf_idx.copy(), last_page_len=s_last,
        q=q, k_pages=k, v_pages=v,
    )
    flat_lists = [np.concatenate([pre_idx, suf_idx[s_indptr[i]:s_indptr[i + 1]]]) for i in range(n_req)]
    f_indptr = np.zeros(n_req + 1, np.int32)
    f_indptr[1:] = np.cumsum([len(x) for x in flat_lists])
    flat = PagedBatch(
        "shared_prefix_decode/flat", hq, hk, HEAD_DIM, page_size, False,
        qo_indptr=ones.copy(), kv_indptr=f_indptr,
        kv_indices=np.concatenate(flat_lists).astype(np.int32), last_page_len=s_last.copy(),
        q=q, k_pages=k, v_pages=v,
    )
    meta = {"prefix_len": prefix_len, "suffix_lens": suf}
    prefix.meta, suffix.meta, flat.meta = dict(meta), dict(meta), dict(meta)
    return SharedPrefixBatch(prefix, suffix, flat)


# ---------------------------------------------------------------------------
# FP8 (e4m3) pages
# ---------------------------------------------------------------------------

def _e4m3_table() -> np.ndarray:
    """Values of the 127 non-negative finite e4m3 codes (1 sign, 4 exponent bits with bias 7,
    3 mantissa bits; exponent 0 holds subnormals; code 0x7F is NaN)."""
    vals = []
    for code in range(0x7F):
        e, m = code >> 3, code & 7
        vals.append(m / 8.0 * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7))
    return np.array(vals)


def to_e4m3(x: np.ndarray) -> np.ndarray:
    """float -> e4m3 codes, round to nearest (ties to the even code), saturating at +-448."""
    table = _e4m3_table()
    a = np.minimum(np.abs(np.asarray(x, dtype=np.float64)), table[-1])
    hi = np.clip(np.searchsorted(table, a), 1, len(table) - 1)
    lo = hi - 1
    d_lo, d_hi = a - table[lo], table[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    code = np.where(a == 0, 0, code).astype(np.uint8)
    return (code | np.where(np.signbit(np.asarray(x, dtype=np.float64)) & (code != 0), 0x80, 0)).astype(np.uint8)


def as_e4m3(b: PagedBatch, k_scale: float, v_scale: float) -> PagedBatch:
    """The batch with its K/V pages quantised to e4m3 codes of K / k_scale and V / v_scale."""
    import dataclasses
    bf = lambda bits: (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)
    return dataclasses.replace(b, k_pages=to_e4m3(bf(b.k_pages) / k_scale), v_pages=to_e4m3(bf(b.v_pages) / v_scale),
                               meta=dict(b.meta, k_scale=k_scale, v_scale=v_scale))


# ---------------------------------------------------------------------------
# Kernel-level length distributions (batch 16; constant / uniform / Zipf)
# ---------------------------------------------------------------------------

KERNEL_DISTS = ("constant", "uniform", "zipf")
KERNEL_DIST_WORKLOADS = tuple(f"kernel_{d}_{m}" for m in ("decode", "prefill") for d in KERNEL_DISTS)


def kernel_dist_lengths(rng: np.random.Generator, dist: str, batch: int = 16) -> np.ndarray:
    """constant: 1024; uniform: U[512, 1024]; zipf: 512 * k, k ~ Zipf(2.5), capped at 16384 (mean ~1000)."""
    if dist == "constant":
        return np.full(batch, 1024, np.int64)
    if dist == "uniform":
        return rng.integers(512, 1025, size=batch).astype(np.int64)
    if dist == "zipf":
        return np.minimum(512 * rng.zipf(2.5, size=batch), 16384).astype(np.int64)
    raise ValueError(dist)


def kernel_dist(dist: str, mode: str, batch: int = 16, with_data: bool = True) -> PagedBatch:
    """Batch 16, 32/8 heads, page 16: decode (one query token) or causal prefill (q = kv) over the lengths."""
    seed = 10 + KERNEL_DIST_WORKLOADS.index(f"kernel_{dist}_{mode}")
    rng = np.random.default_rng(seed)
    lens = kernel_dist_lengths(rng, dist, batch)
    if mode == "decode":
        return make_paged_batch(rng, f"kernel_{dist}_decode", np.ones(batch, np.int64), lens, 32, 8, 16, False,
                                with_data=with_data)
    if mode == "prefill":
        return make_paged_batch(rng, f"kernel_{dist}_prefill", lens, lens, 32, 8, 16, True, scale=0.5,
                                with_data=with_data)
    raise ValueError(mode)


def by_name(name: str):
    if name.startswith("kernel_"):
        _, dist, mode = name.split("_")
        return kernel_dist(dist, mode)
    return {
        "tiny_decode": tiny_decode,
        "llama3_8b_decode": llama3_8b_decode,
        "skewed_long_decode": skewed_long_decode,
        "ragged_causal_prefill": ragged_causal_prefill,
        "shared_prefix_decode": shared_prefix_decode,
    }[name]()


def random_small_batch(
    seed: int,
    batch: int,
    num_qo_heads: int,
    num_kv_heads: int,
    page_size: int,
    causal: bool,
    q_len_range=(1, 1),
    kv_len_range=(0, 64),
    extra_pages: int = 3,
    head_dim: int = HEAD_DIM,
    scale: float = 1.0,
) -> PagedBatch:
    """Small ragged batch for parity tests: lengths drawn first, then as in make_paged_batch."""
    rng = np.random.default_rng(seed)
    ql = rng.integers(q_len_range[0], q_len_range[1] + 1, size=batch)
    kl = rng.integers(kv_len_range[0], kv_len_range[1] + 1, size=batch)
    n_pages = int(((kl + page_size - 1) // page_size).sum())
    return make_paged_batch(
        rng, f"random_small_{seed}", ql, kl, num_qo_heads, num_kv_heads, page_size, causal,
        pool_pages=n_pages + extra_pages, scale=scale, head_dim=head_dim,
    )
