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
    (32, 8, 8, (1, 1), (1, 900), False, 0, 0.5, 1.0, -1, 0.0, "HND"),       # page 8: smallest whole-page box
    (32, 8, 128, (1, 1), (1, 1500), False, 0, 1.0, 0.5, -1, 0.0, "HND"),    # page 128: 64-token boxes in a page
    (16, 4, 128, (1, 2), (2, 1200), True, 3, 0.5, 2.0, -1, 0.0, "NHD"),     # NHD, page 128, causal
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


def test_fp8_decode_ignores_codes_past_the_last_token():
    """Pages of 8 or more tokens are copied whole: NaN codes (0x7f) in the unused slots of each
    request's last page must not reach any output."""
    b = W.random_small_batch(5400, batch=9, num_qo_heads=32, num_kv_heads=8, page_size=16, causal=False,
                             q_len_range=(1, 1), kv_len_range=(1, 900), extra_pages=3)
    b8 = W.as_e4m3(b, 0.5, 1.0)
    k, v = b8.k_pages.copy(), b8.v_pages.copy()  # HND [pages, H_kv, page, D]
    for i in range(b8.batch_size):
        lo, hi = int(b8.kv_indptr[i]), int(b8.kv_indptr[i + 1])
        if hi > lo:
            last, n = int(b8.kv_indices[hi - 1]), int(b8.last_page_len[i])
            k[last, :, n:, :] = 0x7F
            v[last, :, n:, :] = 0x7F
    o, lse, _ = run_fp8(dataclasses.replace(b8, k_pages=k, v_pages=v), 0.5, 1.0)
    ro, rl = A.batch_attention(b8, k_scale=0.5, v_scale=1.0)
    assert np.isfinite(o).all()
    assert_close(o, lse, ro, rl)


def test_fp8_prefill_ignores_codes_past_the_last_token():
    """Tensor-core tiles over e4m3 pages: NaN codes (0x7f) in the unused slots of each request's last page
    must not reach any output."""
    b = W.random_small_batch(5410, batch=5, num_qo_heads=8, num_kv_heads=2, page_size=16, causal=True,
                             q_len_range=(20, 150), kv_len_range=(150, 700), extra_pages=3)
    b8 = W.as_e4m3(b, 0.5, 1.0)
    k, v = b8.k_pages.copy(), b8.v_pages.copy()
    for i in range(b8.batch_size):
        lo, hi = int(b8.kv_indptr[i]), int(b8.kv_indptr[i + 1])
        if hi > lo:
            last, n = int(b8.kv_indices[hi - 1]), int(b8.last_page_len[i])
            k[last, :, n:, :] = 0x7F
            v[last, :, n:, :] = 0x7F
    o, lse, ws = run_fp8(dataclasses.replace(b8, k_pages=k, v_pages=v), 0.5, 1.0, num_sms=3)
    assert ws.info()[1] == 1
    ro, rl = A.batch_attention(b8, k_scale=0.5, v_scale=1.0)
    assert np.isfinite(o).all()
    assert_close(o, lse, ro, rl)


TC_CASES = [
    # (hq, hk, page, q range, kv range, causal, SM budget, k_scale, v_scale, window, cap, layout):
    # requests of more than 8 rows, so the plan takes tensor-core tiles
    (32, 8, 16, (9, 200), (200, 700), True, 0, 0.5, 2.0, -1, 0.0, "HND"),     # g = 4, every SM
    (8, 8, 8, (20, 150), (150, 2000), True, 40, 2.0, 0.5, -1, 0.0, "HND"),    # g = 1, page 8, split rows
    (16, 2, 32, (5, 90), (0, 400), False, 2, 1.0, 1.0, -1, 0.0, "HND"),       # g = 8, page 32, empty KV rows
    (12, 4, 128, (10, 90), (90, 500), True, 2, 0.25, 4.0, -1, 0.0, "HND"),    # g = 3, page 128
    (32, 8, 16, (30, 300), (300, 800), True, 4, 0.5, 0.5, 100, 20.0, "HND"),  # window + soft-cap
    (32, 8, 16, (9, 200), (200, 700), True, 0, 0.5, 2.0, -1, 0.0, "NHD"),     # NHD, split rows
    (8, 2, 64, (20, 100), (100, 600), True, 2, 1.0, 0.25, 150, 30.0, "NHD"),  # NHD, page 64, window + cap
]


@pytest.mark.parametrize("case", range(len(TC_CASES)))
def test_fp8_tensor_core_parity(case):
    """e4m3 pages on 256-row tensor-core tiles: the producer widens each K/V tile to f16 in shared
    memory, and the kernel's result matches the oracle over the decoded codes."""
    hq, hk, ps, qr, kr, causal, n_sms, ks, vs, window, cap, layout = TC_CASES[case]
    b = W.random_small_batch(5200 + case, batch=5, num_qo_heads=hq, num_kv_heads=hk, page_size=ps, causal=causal,
                             q_len_range=qr, kv_len_range=kr, extra_pages=3, scale=0.5)
    b8 = W.as_e4m3(b, ks, vs)
    if layout == "NHD":
        b8 = as_nhd(b8)
    o, lse, ws = run_fp8(b8, ks, vs, n_sms, window, cap, layout)
    assert ws.info()[1] == 1
    if case in (1, 5):
        assert ws.info()[7] > 0  # split rows, merged by the contraction kernel
    ro, rl = A.batch_attention(b8, layout=layout, k_scale=ks, v_scale=vs, window_left=window, soft_cap=cap)
    assert_close(o, lse, ro, rl)


def test_fp8_ragged_causal_prefill_full():
    """The full ragged causal batch over e4m3 pages, in the benchmark's launch configuration, every row."""
    b8 = W.as_e4m3(W.ragged_causal_prefill(), 0.25, 0.25)
    o, lse, ws = run_fp8(b8, 0.25, 0.25)
    assert ws.info()[1] == 1
    ro, rl = A.batch_attention(b8, k_scale=0.25, v_scale=0.25)
    assert_close(o, lse, ro, rl)


def test_fp8_tensor_core_reruns_bit_identical():
    b8 = W.as_e4m3(W.random_small_batch(5300, batch=4, num_qo_heads=32, num_kv_heads=8, page_size=16, causal=True,
                                        q_len_range=(100, 400), kv_len_range=(400, 1500), scale=0.5), 0.5, 0.5)
    o1, l1, ws = run_fp8(b8, 0.5, 0.5)
    assert ws.info()[1] == 1 and ws.info()[7] > 0
    o2, l2, _ = run_fp8(b8, 0.5, 0.5)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


FP8_COMPOSABLE_CASES = [
    # (seed, n_req, hq, hk, page, q_len, own range, groups, prefix range, causal, SM budget, k_scale, v_scale)
    (7400, 12, 32, 8, 16, 1, (1, 600), 2, (200, 1500), False, 0, 0.5, 2.0),
    (7401, 9, 8, 2, 16, 2, (2, 300), 3, (100, 900), True, 12, 1.0, 0.5),   # few CTAs: shared rows split
]


@pytest.mark.parametrize("case", range(len(FP8_COMPOSABLE_CASES)))
def test_fp8_composable_matches_oracle(case):
    """One composable plan over e4m3 pages: the shared sub-matrix on tensor-core tiles (widened in
    shared memory), the per-request rows on FP8 decode tiles merging the shared slots."""
    from serving_attention_plan_gb300 import binding as B
    from .test_gpu_composable import composable_batch
    seed, n_req, hq, hk, ps, ql, own, ng, pre, causal, n_sms, ks, vs = FP8_COMPOSABLE_CASES[case]
    shared, unique = composable_batch(seed, n_req, hq, hk, ps, ql, own, ng, pre, causal)
    s8, u8 = W.as_e4m3(shared, ks, vs), W.as_e4m3(unique, ks, vs)  # one pool: the same codes in both
    torch = torch_mod()
    dev = torch.device("cuda", 0)
    q = torch.from_numpy(np.ascontiguousarray(u8.q).view(np.int16)).to(dev).view(torch.bfloat16)
    k = torch.from_numpy(np.ascontiguousarray(u8.k_pages)).to(dev)
    v = torch.from_numpy(np.ascontiguousarray(u8.v_pages)).to(dev)
    o, lse = alloc_out(u8)
    ws = B.Workspace(max(u8.batch_size, s8.batch_size), u8.total_q, max(int(u8.kv_indptr[-1]), int(s8.kv_indptr[-1])),
                     hq, hk, 128, n_sms)
    ws.set_kv_dtype("e4m3", ks, vs)
    ws.plan_composable((s8.qo_indptr, s8.kv_indptr, s8.kv_indices, s8.last_page_len),
                       (u8.qo_indptr, u8.kv_indptr, u8.kv_indices, u8.last_page_len), ps, causal)
    assert ws.info()[1] == 2
    ws.run(q, k, v, o, lse)
    torch.cuda.synchronize()
    assert ws.get_error() == 0
    so, sl = A.batch_attention(s8, k_scale=ks, v_scale=vs)
    po = np.zeros((u8.total_q,) + so.shape[1:])
    pl = np.full((u8.total_q, so.shape[1]), -np.inf)
    po[: so.shape[0]], pl[: sl.shape[0]] = so, sl
    uo, ul = A.batch_attention(u8, k_scale=ks, v_scale=vs)
    ro, rl = A.merge_states(po, pl, uo, ul)
    assert_close(o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64), ro, rl)


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
    ws.plan(pre.qo_indptr, pre.kv_indptr, pre.kv_indices, pre.last_page_len, 16, True)
    assert ws.info()[1] == 1                      # tensor-core tiles take e4m3 pages (widened in shared memory)
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
