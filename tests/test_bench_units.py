"""The benchmark's work units on CPU: the bytes and flops that every reported rate divides by.

Counted here by brute force from the definitions: a query token t of a request with l_q queries
and l_kv keys sees key j when j <= l_kv - l_q + t (causal; every key otherwise), and with a window
w also j >= l_kv - l_q + t - w (page "FlashInfer：面向 LLM 推理服务的高效可定制注意力引擎",
术语与记号 and 问题背景 挑战二).  Each visible (query row, key) pair costs 2 * 128 multiply-adds in
Q K^T and 2 * 128 in P V; each KV token moves its K and V rows once per KV head.
"""
import numpy as np
import pytest

import bench
from serving_attention_plan_gb300 import workloads as W


def brute_pairs(b, window_left=-1):
    qo = b.qo_indptr.astype(np.int64)
    n_p = np.diff(b.kv_indptr.astype(np.int64))
    total = 0
    for i in range(b.batch_size):
        l_q = int(qo[i + 1] - qo[i])
        l_kv = int((n_p[i] - 1) * b.page_size + b.last_page_len[i]) if n_p[i] > 0 else 0
        for t in range(l_q):
            for j in range(l_kv):
                p = l_kv - l_q + t
                if b.causal and j > p:
                    continue
                if window_left >= 0 and j < p - window_left:
                    continue
                total += 1
    return total


@pytest.mark.parametrize("seed,causal,q_range,window", [
    (0, False, (1, 1), -1),
    (1, True, (1, 3), -1),
    (2, True, (5, 40), -1),       # prefill-shaped rows, some with l_q > l_kv
    (3, True, (5, 40), 7),        # sliding window
    (4, True, (1, 1), 0),         # window 0: each row sees one key
])
def test_visible_pairs_and_flops_match_brute_force(seed, causal, q_range, window):
    b = W.random_small_batch(seed, batch=6, num_qo_heads=8, num_kv_heads=2, page_size=4, causal=causal,
                             q_len_range=q_range, kv_len_range=(0, 37))
    pairs = brute_pairs(b, window)
    assert bench.visible_pairs(b, window) == pairs
    assert bench.flops(b, window) == 4 * 128 * pairs * b.num_qo_heads


def test_kv_bytes_and_algorithmic_bytes():
    b = W.random_small_batch(7, batch=5, num_qo_heads=8, num_kv_heads=2, page_size=16, causal=False,
                             kv_len_range=(1, 100))
    n_p = np.diff(b.kv_indptr.astype(np.int64))
    tokens = int(sum((n - 1) * 16 + int(last) for n, last in zip(n_p, b.last_page_len) if n > 0))
    assert bench.kv_bytes(b) == tokens * 2 * 128 * 2 * 2          # K and V rows, bf16
    rows = b.total_q * 8
    assert bench.algorithmic_bytes(b) == bench.kv_bytes(b) + rows * 128 * 2 * 2 + rows * 4 + int(n_p.sum()) * 4
    b8 = W.as_e4m3(b, 0.5, 0.5)
    assert bench.kv_bytes(b8) * 2 == bench.kv_bytes(b)             # one byte per e4m3 code
