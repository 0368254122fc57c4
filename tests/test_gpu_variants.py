"""GPU parity of the attention variants against the float64 oracle: sliding window (causal), logit
soft-cap and the NHD page layout, on both paths.  Source: page "FlashInfer：面向 LLM 推理服务的
高效可定制注意力引擎", 问题背景 挑战二 (paper §1: sliding-window masks, logit soft-cap) and
核心机制 5 (paper §3.2-3.2.3: masks, logits transforms and the KV layout as template inputs)."""
import dataclasses

import numpy as np
import pytest

from oracle import attention as A
from serving_attention_plan_gb300 import workloads as W

from .gpu_helpers import alloc_out, assert_close, to_device, torch_mod

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from serving_attention_plan_gb300 import build
    build.build()
    assert torch_mod().cuda.is_available()


def as_nhd(b):
    """The same pages stored [pages, page_size, H_kv, D]."""
    return dataclasses.replace(b, k_pages=np.ascontiguousarray(b.k_pages.transpose(0, 2, 1, 3)),
                               v_pages=np.ascontiguousarray(b.v_pages.transpose(0, 2, 1, 3)))


def run_variant(b, window, cap, layout, num_sms=0):
    from serving_attention_plan_gb300 import binding as B
    torch = torch_mod()
    ws = B.Workspace(b.batch_size, max(b.total_q, 1), max(int(b.kv_indptr[-1]), 1), b.num_qo_heads,
                     b.num_kv_heads, b.head_dim, num_sms)
    ws.set_variant(window, cap, layout)
    q, k, v = to_device(b)
    o, lse = alloc_out(b)
    ws.plan(b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, b.page_size, b.causal)
    ws.run(q, k, v, o, lse)
    torch.cuda.synchronize()
    assert ws.get_error() == 0
    return o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64), ws


CASES = [
    # (hq, hk, page, q range, kv range, causal, window, soft-cap, layout, SM budget)
    (32, 8, 16, (1, 1), (1, 900), True, 64, 0.0, "HND", 5),        # decode g=4, window, split rows
    (64, 8, 16, (1, 1), (1, 900), True, 200, 30.0, "NHD", 0),      # decode g=8: window + cap + NHD
    (8, 2, 1, (1, 1), (1, 500), False, -1, 5.0, "NHD", 3),         # decode, page 1, cap, NHD
    (32, 8, 128, (1, 1), (1, 1500), False, -1, 0.0, "NHD", 0),     # decode, NHD page 128: boxes inside a page
    (16, 16, 8, (1, 2), (2, 600), True, -1, 0.0, "NHD", 4),        # decode g = 1, 16 KV heads, NHD page 8
    (8, 8, 5, (1, 2), (2, 300), True, 17, 10.0, "HND", 2),         # bulk loader, CUDA-core consumer
    (16, 4, 12, (1, 1), (1, 700), True, 100, 0.0, "HND", 4),       # bulk loader, R = 4, window
    (8, 2, 16, (20, 200), (200, 1500), True, 128, 0.0, "HND", 4),  # tensor cores, window, split rows
    (32, 8, 16, (50, 300), (300, 900), True, -1, 2.0, "NHD", 0),   # tensor cores, cap near the logits
    (16, 4, 32, (30, 100), (100, 600), True, 40, 5.0, "NHD", 2),   # tensor cores: all three, page 32
    (8, 8, 128, (17, 130), (10, 600), False, -1, 0.0, "NHD", 1),   # tensor cores, NHD page 128
    (12, 4, 8, (10, 90), (90, 400), True, 0, 0.0, "HND", 2),       # window 0: one key per row; g = 3
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_variant_parity(case):
    hq, hk, ps, qr, kr, causal, window, cap, layout, n_sms = CASES[case]
    b = W.random_small_batch(4000 + case, batch=6, num_qo_heads=hq, num_kv_heads=hk, page_size=ps, causal=causal,
                             q_len_range=qr, kv_len_range=kr, extra_pages=3, scale=1.5 if cap else 0.5)
    bb = as_nhd(b) if layout == "NHD" else b
    o, lse, ws = run_variant(bb, window, cap, layout, n_sms)
    assert ws.info()[1] == (0 if qr[1] * hq // hk <= 8 else 1)
    ro, rl = A.batch_attention(bb, layout=layout, window_left=window, soft_cap=cap)
    assert_close(o, lse, ro, rl)


def test_variant_reruns_bit_identical():
    b = as_nhd(W.random_small_batch(4100, batch=3, num_qo_heads=8, num_kv_heads=2, page_size=16, causal=True,
                                    q_len_range=(40, 90), kv_len_range=(3000, 6000), scale=1.5))
    o1, l1, ws = run_variant(b, 2000, 4.0, "NHD", 16)
    assert ws.info()[7] > 0          # windowed rows still long enough to be split
    o2, l2, _ = run_variant(b, 2000, 4.0, "NHD", 16)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    ro, rl = A.batch_attention(b, layout="NHD", window_left=2000, soft_cap=4.0)
    assert_close(o1, l1, ro, rl)


def test_variant_arguments_checked():
    from serving_attention_plan_gb300 import binding as B
    ws = B.Workspace(4, 4, 64, 8, 2)
    for bad in [dict(window_left=-2), dict(logits_soft_cap=-1.0), dict(logits_soft_cap=float("nan"))]:
        with pytest.raises(B.FiError) as ei:
            ws.set_variant(**bad)
        assert ei.value.status == 1
    b = W.random_small_batch(4101, batch=2, num_qo_heads=8, num_kv_heads=2, page_size=16, causal=False,
                             kv_len_range=(16, 64))
    ws.set_variant(window_left=8)
    with pytest.raises(B.FiError) as ei:          # the window is read with causal masks
        ws.plan(b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, 16, False)
    assert ei.value.status == 3
    b5 = W.random_small_batch(4102, batch=2, num_qo_heads=8, num_kv_heads=2, page_size=5, causal=False,
                              kv_len_range=(16, 64))
    ws5 = B.Workspace(4, 4, 64, 8, 2)
    ws5.set_variant(kv_layout="NHD")
    with pytest.raises(B.FiError) as ei:          # NHD decode needs a power-of-two page size
        ws5.plan(b5.qo_indptr, b5.kv_indptr, b5.kv_indices, b5.last_page_len, 5, False)
    assert ei.value.status == 3
