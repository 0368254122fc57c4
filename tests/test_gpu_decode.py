"""GPU parity of the decode path (<= 8-row tiles) against the float64 oracle, through the C ABI."""
import dataclasses

import numpy as np
import pytest

from oracle import attention as A
from serving_attention_plan_gb300 import workloads as W

from .gpu_helpers import alloc_out, assert_close, run_library, to_device, torch_mod

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from serving_attention_plan_gb300 import build
    build.build()
    torch = torch_mod()
    assert torch.cuda.is_available()


def test_tiny_decode_full():
    b = W.tiny_decode()
    o, lse, _ = run_library(b)
    ro, rl = A.batch_attention(b)
    assert_close(o, lse, ro, rl)


CASES = [
    # (hq, hk, page_size, q_len range, kv range, causal, num_ctas)
    (8, 2, 16, (1, 1), (0, 700), False, 0),
    (8, 2, 16, (1, 1), (0, 700), False, 3),      # few CTAs: long rows split and merged in-kernel
    (32, 8, 16, (0, 1), (0, 300), False, 5),
    (64, 8, 1, (1, 1), (0, 900), False, 7),      # page size 1, g = 8
    (4, 4, 3, (1, 1), (1, 200), True, 2),        # g = 1, odd page size
    (8, 4, 64, (1, 4), (4, 500), True, 4),       # g = 2, up to 4 query tokens (8 rows), causal
    (8, 8, 5, (1, 2), (2, 333), True, 9),        # g = 1, 2 query tokens
    (16, 8, 16, (1, 4), (0, 100), False, 1),     # one CTA does everything
    (16, 4, 32, (1, 2), (2, 600), True, 6),      # g = 4, 2 query tokens: 8-row tiles, tensor-core consumer
    (8, 8, 8, (1, 8), (8, 400), True, 3),        # g = 1, up to 8 query tokens: one causal limit per row
    (32, 8, 24, (1, 1), (0, 700), False, 4),     # g = 4, page 24: bulk loader, CUDA-core consumer
    (64, 8, 12, (1, 1), (0, 900), True, 5),      # g = 8, page 12: bulk loader, CUDA-core consumer
    (32, 8, 4, (1, 1), (0, 600), False, 4),      # g = 4, page 4: 16-byte copies, tensor-core consumer
    (32, 8, 128, (1, 1), (0, 2000), False, 0),   # g = 4, page 128: 32-token TMA boxes inside a page
]


@pytest.mark.parametrize("case", range(len(CASES)))
@pytest.mark.parametrize("seed", [0, 1])
def test_random_decode_parity(case, seed):
    hq, hk, ps, qr, kr, causal, n_cta = CASES[case]
    b = W.random_small_batch(1000 * case + seed, batch=17, num_qo_heads=hq, num_kv_heads=hk, page_size=ps,
                             causal=causal, q_len_range=qr, kv_len_range=kr, extra_pages=7)
    o, lse, ws = run_library(b, num_sms=n_cta)
    assert ws.info()[1] == 0  # decode path
    ro, rl = A.batch_attention(b)
    assert_close(o, lse, ro, rl)


def test_llama3_8b_decode_full():
    b = W.llama3_8b_decode()
    o, lse, ws = run_library(b)
    ro, rl = A.batch_attention(b)
    assert_close(o, lse, ro, rl)


def test_skewed_long_decode_full():
    """Full-size skewed batch in the benchmark's launch configuration, every row of every head."""
    b = W.skewed_long_decode()
    o, lse, ws = run_library(b)
    h = ws.info()
    assert h[7] == 8  # the 131072-token request is split on each KV head
    ro, rl = A.batch_attention(b)
    assert_close(o, lse, ro, rl)


def test_bit_identical_reruns():
    torch = torch_mod()
    b = W.random_small_batch(77, batch=33, num_qo_heads=64, num_kv_heads=8, page_size=1, causal=False,
                             kv_len_range=(0, 4000), extra_pages=3)
    dev = to_device(b)
    o1, l1, ws = run_library(b, num_sms=11, dev=dev)
    for _ in range(3):
        o2, l2, _ = run_library(b, ws=ws, dev=dev)
        assert np.array_equal(o1, o2) and np.array_equal(l1, l2, equal_nan=True)
    del torch


def test_cuda_graph_replay_matches():
    """A captured fi_run replays bit-identically and serves a later plan of the same path and tile."""
    torch = torch_mod()
    from serving_attention_plan_gb300 import binding as B
    mk = lambda seed: W.random_small_batch(seed, batch=20, num_qo_heads=32, num_kv_heads=8, page_size=16,
                                           causal=False, kv_len_range=(1, 3000))
    b, b2 = mk(78), mk(79)
    pool = max(b.num_pages, b2.num_pages)
    q1, k1, v1 = to_device(b)
    q2, k2, v2 = to_device(b2)
    q = q1.clone()
    k = torch.zeros((pool,) + tuple(k1.shape[1:]), dtype=k1.dtype, device=k1.device)
    v = torch.zeros_like(k)
    k[: k1.shape[0]].copy_(k1)
    v[: v1.shape[0]].copy_(v1)
    ws = B.Workspace(64, 64, 8192, 32, 8, 128, 13)   # capacity for both plans
    o_ref, l_ref, _ = run_library(b, ws=ws, dev=(q, k, v))
    o, lse = alloc_out(b)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        ws.run(q, k, v, o, lse, stream=s)
    for _ in range(3):
        o.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(o.float().cpu().numpy(), o_ref)
        assert np.array_equal(lse.cpu().numpy().astype(np.float64), l_ref)
    ws.plan(b2.qo_indptr, b2.kv_indptr, b2.kv_indices, b2.last_page_len, 16, False)
    q.copy_(q2)
    k[: k2.shape[0]].copy_(k2)
    v[: v2.shape[0]].copy_(v2)
    torch.cuda.synchronize()
    o.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    ro, rl = A.batch_attention(b2)
    assert_close(o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64), ro, rl)


def test_out_of_range_page_rejected_on_host():
    from serving_attention_plan_gb300 import binding as B
    b = W.random_small_batch(80, batch=4, num_qo_heads=8, num_kv_heads=2, page_size=16, causal=False,
                             kv_len_range=(16, 64), extra_pages=0)
    q, k, v = to_device(b)
    o, lse = alloc_out(b)
    ws = B.Workspace(4, 4, 64, 8, 2)
    ws.plan(b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, 16, False)
    with pytest.raises(B.FiError) as ei:
        ws.run(q, k[:-1], v[:-1], o, lse)  # the pool view no longer holds the largest page id
    assert ei.value.status == 1


def test_unaligned_rows_rejected_on_host():
    """q, K and V rows move in 16-byte copies: a base address off a 16-byte boundary is refused before
    any launch, by fi_run and by fi_decode_noalloc."""
    from serving_attention_plan_gb300 import binding as B
    b = W.random_small_batch(81, batch=4, num_qo_heads=8, num_kv_heads=2, page_size=16, causal=False,
                             kv_len_range=(16, 64))
    q, k, v = to_device(b)
    o, lse = alloc_out(b)
    ws = B.Workspace(4, 4, 64, 8, 2)
    ws.plan(b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, 16, False)
    torch = torch_mod()

    def shifted(t):  # the same values, 8 bytes past a 16-byte boundary
        flat = torch.empty(t.numel() + 8, dtype=t.dtype, device=t.device)
        out = flat[4:4 + t.numel()].view(t.shape)
        out.copy_(t)
        return out

    q_off, k_off = shifted(q), shifted(k)
    for qq, kk in ((q_off, k), (q, k_off)):
        with pytest.raises(B.FiError) as ei:
            ws.run(qq, kk, v, o, lse)
        assert ei.value.status == 1
    with pytest.raises(B.FiError) as ei:
        B.decode_noalloc(b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, 8, 2, 16, False, q_off, k, v, o,
                         lse)
    assert ei.value.status == 1


@pytest.mark.parametrize("prefill", [False, True])
def test_dependent_launch_reads_the_previous_output(prefill):
    """Back-to-back runs on one stream, the second reading the first's output as its q: a run is
    launched as a programmatic dependent of the kernel before it and may start its set-up early, so
    this checks that it reads nothing before that kernel has finished."""
    import dataclasses
    torch = torch_mod()
    from serving_attention_plan_gb300 import binding as B
    if prefill:
        b = W.random_small_batch(91, batch=6, num_qo_heads=32, num_kv_heads=8, page_size=16, causal=True,
                                 q_len_range=(100, 400), kv_len_range=(400, 1200), scale=0.5)
    else:
        b = W.random_small_batch(90, batch=96, num_qo_heads=32, num_kv_heads=8, page_size=16, causal=False,
                                 kv_len_range=(500, 3000))
    q, k, v = to_device(b)
    o1, lse1 = alloc_out(b)
    o2, lse2 = alloc_out(b)
    ws = B.Workspace(b.batch_size, b.total_q, int(b.kv_indptr[-1]), b.num_qo_heads, b.num_kv_heads, 128)
    ws.plan(b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, b.page_size, b.causal)
    assert ws.info()[1] == (1 if prefill else 0)
    for _ in range(3):
        o2.fill_(float("nan"))
        ws.run(q, k, v, o1, lse1)
        ws.run(o1, k, v, o2, lse2)  # q of the second run = output of the first
        torch.cuda.synchronize()
        assert ws.get_error() == 0
        b2 = dataclasses.replace(b, q=o1.view(torch.int16).cpu().numpy().view(np.uint16))
        ro, rl = A.batch_attention(b2)
        assert_close(o2.float().cpu().numpy().astype(np.float64), lse2.cpu().numpy().astype(np.float64), ro, rl)


def test_merge_states_kernel():
    torch = torch_mod()
    from serving_attention_plan_gb300 import binding as B
    rng = np.random.default_rng(5)
    rows, heads = 37, 6
    oa = rng.standard_normal((rows, heads, 128)).astype(np.float32)
    ob = rng.standard_normal((rows, heads, 128)).astype(np.float32)
    la = (rng.standard_normal((rows, heads)) * 20).astype(np.float32)
    lb = (rng.standard_normal((rows, heads)) * 20).astype(np.float32)
    la[0, 0] = -np.inf
    la[1, :] = lb[1, :] = -np.inf
    dev = lambda x: torch.from_numpy(x).cuda()
    ta, tb = dev(oa).bfloat16(), dev(ob).bfloat16()
    o = torch.empty_like(ta)
    lse = torch.empty((rows, heads), dtype=torch.float32, device="cuda")
    B.merge_states(ta, dev(la), tb, dev(lb), o, lse)
    torch.cuda.synchronize()
    ro, rl = A.merge_states(ta.float().cpu().numpy(), la, tb.float().cpu().numpy(), lb)
    assert_close(o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64), ro, rl)


@pytest.mark.parametrize("name", ["llama3_8b_decode", "skewed_long_decode"])
def test_many_back_to_back_launches(name):
    """Hundreds of launches in a row: no pipeline wait may time out and every output stays bit-identical."""
    torch = torch_mod()
    b = W.by_name(name)
    dev = to_device(b)
    o_ref, l_ref, ws = run_library(b, dev=dev)
    q, k, v = dev
    o, lse = alloc_out(b)
    for _ in range(300):
        ws.run(q, k, v, o, lse)
    torch.cuda.synchronize()
    assert ws.get_error() == 0
    assert np.array_equal(o.float().cpu().numpy(), o_ref)
    assert np.array_equal(lse.cpu().numpy().astype(np.float64), l_ref)


def test_decode_ignores_values_past_the_last_token():
    """Pages of 8 or more tokens are copied whole: NaN values in the unused slots of each request's
    last page must not reach any output (rows 4 and 8 of a tile, g = 4 and g = 8)."""
    for hq in (32, 64):
        b = W.random_small_batch(95 + hq, batch=12, num_qo_heads=hq, num_kv_heads=8, page_size=16, causal=False,
                                 q_len_range=(1, 1), kv_len_range=(1, 700), extra_pages=3)
        k, v = b.k_pages.copy(), b.v_pages.copy()  # HND [pages, H_kv, page, D] bf16 bits
        for i in range(b.batch_size):
            lo, hi = int(b.kv_indptr[i]), int(b.kv_indptr[i + 1])
            if hi > lo:
                last, n = int(b.kv_indices[hi - 1]), int(b.last_page_len[i])
                k[last, :, n:, :] = 0x7FC0
                v[last, :, n:, :] = 0x7FC0
        o, lse, ws = run_library(dataclasses.replace(b, k_pages=k, v_pages=v))
        ro, rl = A.batch_attention(b)
        assert np.isfinite(o).all()
        assert_close(o, lse, ro, rl)
