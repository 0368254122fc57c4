"""GPU parity of decode over FP8 (e4m3) KV pages against the float64 oracle.  Source: page
"FlashInfer：面向 LLM 推理服务的高效可定制注意力引擎", 核心机制 8 (paper App. F: KV-cache stored
as fp8, queries and outputs kept in 16-bit floats), in both page layouts (核心机制 5)."""
import dataclasses

import numpy as np
import pytest

from oracle import attention as A
from serving_attention_plan_gb300 import workloads as W

from .gpu_helpers import alloc_out, assert_close, torch_mod

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from serving_attention_plan_gb300 import build
    build.build()
    assert torch_mod().cuda.is_available()


def run_fp8(b8, k_scale, v_scale, num_sms=0, window=-1, cap=0.0, layout="HND"):
    from serving_attention_plan_gb300 import binding as B
    torch = torch_mod()
    dev = torch.device("cuda", 0)
    q = torch.from_numpy(np.ascontiguousarray(b8.q).view(np.int16)).to(dev).view(torch.bfloat16)
    k = torch.from_numpy(np.ascontiguousarray(b8.k_pages)).to(dev)
    v = torch.from_numpy(np.ascontiguousarray(b8.v_pages)).to(dev)
    o, lse = alloc_out(b8)
    ws = B.Workspace(b8.batch_size, max(b8.total_q, 1), max(int(b8.kv_indptr[-1]), 1), b8.num_qo_heads,
                     b8.num_kv_heads, b8.head_dim, num_sms)
    ws.set_kv_dtype("e4m3", k_scale, v_scale)
    if window >= 0 or cap > 0 or layout != "HND":
        ws.set_variant(window, cap, layout)
    ws.plan(b8.qo_indptr, b8.kv_indptr, b8.kv_indices, b8.last_page_len, b8.page_size, b8.causal)
    ws.run(q, k, v, o, lse)
    torch.cuda.synchronize()
    assert ws.get_error() == 0
    return o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64), ws


CASES = [
    # (hq, hk, page, q range, kv range, causal, SM budget, k_scale, v_scale, window, cap, layout)
    (32, 8, 16, (1, 1), (1, 900), False, 0, 0.5, 2.0, -1, 0.0, "HND"),      # g = 4
    (32, 8, 16, (1, 1), (1, 2000), False, 0, 0.25, 1.0, -1, 0.0, "HND"),    # every SM: split rows merged
    (64, 8, 1, (1, 1), (1, 700), False, 3, 1.0, 0.5, -1, 0.0, "HND"),       # g = 8, page 1
    (8, 8, 16, (1, 2), (2, 500), True, 4, 2.0, 1.0, -1, 0.0, "HND"),        # g = 1, 2 query tokens, causal
    (16, 4, 32, (1, 2), (2, 800), True, 2, 0.5, 0.5, 100, 20.0, "HND"),     # window + soft-cap
    (32, 8, 16, (1, 1), (1, 2000), False, 0, 0.5, 2.0, -1, 0.0, "NHD"),     # NHD, split rows merged
    (8, 2, 64, (1, 2), (2, 900), True, 3, 1.0, 0.25, 150, 30.0, "NHD"),     # NHD, page 64, window + cap
    (8, 1, 4, (1, 1), (1, 300), False, 2, 2.0, 1.0, -1, 0.0, "NHD"),        # NHD, one KV head, page 4
]


def as_nhd(b):
    """The same pages stored [pages, page_size, H_kv, D]."""
    return dataclasses.replace(b, k_pages=np.ascontiguousarray(b.k_pages.transpose(0, 2, 1, 3)),
                               v_pages=np.ascontiguousarray(b.v_pages.transpose(0, 2, 1, 3)))


@pytest.mark.parametrize("case", range(len(CASES)))
def test_fp8_decode_parity(case):
    hq, hk, ps, qr, kr, causal, n_sms, ks, vs, window, cap, layout = CASES[case]
    b = W.random_small_batch(5000 + case, batch=9, num_qo_heads=hq, num_kv_heads=hk, page_size=ps, causal=causal,
                             q_len_range=qr, kv_len_range=kr, extra_pages=3)
    b8 = W.as_e4m3(b, ks, vs)
    if layout == "NHD":
        b8 = as_nhd(b8)
    o, lse, ws = run_fp8(b8, ks, vs, n_sms, window, cap, layout)
    assert ws.info()[1] == 0
    if case in (1, 5):
        assert ws.info()[7] > 0
    ro, rl = A.batch_attention(b8, layout=layout, k_scale=ks, v_scale=vs, window_left=window, soft_cap=cap)
    assert_close(o, lse, ro, rl)


def test_fp8_llama3_8b_decode_full():
    b8 = W.as_e4m3(W.llama3_8b_decode(), 0.5, 0.5)
    o, lse, _ = run_fp8(b8, 0.5, 0.5)
    ro, rl = A.batch_attention(b8, k_scale=0.5, v_scale=0.5)
    assert_close(o, lse, ro, rl)


def test_fp8_reruns_bit_identical():
    b8 = W.as_e4m3(W.random_small_batch(5100, batch=5, num_qo_heads=32, num_kv_heads=8, page_size=16,
                                        causal=False, kv_len_range=(500, 3000)), 1.0, 1.0)
    o1, l1, ws = run_fp8(b8, 1.0, 1.0)
    assert ws.info()[7] > 0
    o2, l2, _ = run_fp8(b8, 1.0, 1.0)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_fp8_unsupported_plans_rejected():
    from serving_attention_plan_gb300 import binding as B
    ws = B.Workspace(4, 64, 64, 8, 2)
    for bad in [dict(kv_dtype="e4m3", k_scale=0.0), dict(kv_dtype="e4m3", v_scale=-1.0)]:
        with pytest.raises(B.FiError) as ei:
            ws.set_kv_dtype(**bad)
        assert ei.value.status == 1
    ws.set_kv_dtype("e4m3", 1.0, 1.0)
    pre = W.random_small_batch(5200, batch=2, num_qo_heads=8, num_kv_heads=2, page_size=16, causal=True,
                               q_len_range=(20, 30), kv_len_range=(30, 60))
    with pytest.raises(B.FiError) as ei:          # tensor-core tiles read bf16 pages only
        ws.plan(pre.qo_indptr, pre.kv_indptr, pre.kv_indices, pre.last_page_len, 16, True)
    assert ei.value.status == 3
    dec = W.random_small_batch(5201, batch=2, num_qo_heads=12, num_kv_heads=3, page_size=16, causal=False,
                               kv_len_range=(30, 60))
    ws3 = B.Workspace(4, 64, 64, 12, 3)
    ws3.set_kv_dtype("e4m3", 1.0, 1.0)
    ws3.set_variant(kv_layout="NHD")
    with pytest.raises(B.FiError) as ei:          # NHD pages need a power-of-two KV head count
        ws3.plan(dec.qo_indptr, dec.kv_indptr, dec.kv_indices, dec.last_page_len, 16, False)
    assert ei.value.status == 3
    odd = W.random_small_batch(5202, batch=2, num_qo_heads=8, num_kv_heads=2, page_size=12, causal=False,
                               kv_len_range=(30, 60))
    ws4 = B.Workspace(4, 64, 64, 8, 2)
    ws4.set_kv_dtype("e4m3", 1.0, 1.0)
    with pytest.raises(B.FiError) as ei:          # the e4m3 loader needs a power-of-two page size
        ws4.plan(odd.qo_indptr, odd.kv_indptr, odd.kv_indices, odd.last_page_len, 12, False)
    assert ei.value.status == 3
