"""GPU parity of the tcgen05 tensor-core path against the float64 oracle, through the C ABI."""
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
    assert torch_mod().cuda.is_available()


def test_single_tile_causal():
    """One request of 32 tokens x g=4 (half of one 256-row item), one KV tile: the smallest tensor-core case."""
    b = W.random_small_batch(1, batch=1, num_qo_heads=8, num_kv_heads=2, page_size=16, causal=True,
                             q_len_range=(32, 32), kv_len_range=(32, 32), extra_pages=0)
    o, lse, ws = run_library(b, num_sms=1)
    assert ws.info()[1] == 1
    ro, rl = A.batch_attention(b)
    assert_close(o, lse, ro, rl)


CASES = [
    # (hq, hk, page_size, q range, kv range, causal, SM budget)
    (8, 2, 16, (9, 40), (40, 300), True, 4),
    (8, 2, 16, (3, 300), (300, 700), True, 0),
    (32, 8, 16, (100, 600), (600, 1200), True, 3),   # few CTAs: long chunks, split rows merged in-kernel
    (4, 4, 8, (20, 150), (1, 500), False, 5),        # g = 1, page 8, non-causal
    (16, 8, 32, (5, 200), (0, 400), False, 2),       # g = 2, page 32, empty KV rows
    (64, 8, 64, (2, 40), (50, 900), True, 7),        # g = 8, page 64
    (8, 8, 128, (17, 130), (10, 600), True, 1),      # g = 1, page 128, causal rows with no visible key
    (12, 4, 16, (10, 90), (90, 400), True, 2),       # g = 3: 42-token tiles of 126 rows
    (64, 4, 16, (3, 60), (60, 500), True, 3),        # g = 16: 16-token items
    (64, 4, 32, (1, 1), (1, 900), False, 0),         # g = 16 decode: 16 rows a request, tensor-core items
    (128, 4, 16, (2, 30), (30, 300), True, 2),       # g = 32: 8-token items
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_random_prefill_parity(case):
    hq, hk, ps, qr, kr, causal, n_sms = CASES[case]
    b = W.random_small_batch(2000 + case, batch=5, num_qo_heads=hq, num_kv_heads=hk, page_size=ps, causal=causal,
                             q_len_range=qr, kv_len_range=kr, extra_pages=4, scale=0.5)
    o, lse, ws = run_library(b, num_sms=n_sms)
    assert ws.info()[1] == 1
    ro, rl = A.batch_attention(b)
    assert_close(o, lse, ro, rl)


def test_ragged_causal_prefill_full():
    """Full-size ragged causal batch in the benchmark's launch configuration (every SM, the benchmark's
    chunking and queues), compared with the oracle on every row of every head."""
    b = W.ragged_causal_prefill()
    o, lse, ws = run_library(b)
    h = ws.info()
    assert h[1] == 1 and h[2] == 64
    ro, rl = A.batch_attention(b)
    assert_close(o, lse, ro, rl)


def test_prefill_bit_identical_reruns():
    # few long rows on 8 CTAs: L_kv ~ 1800 keys, so every row is cut into chunks merged in-kernel
    b = W.random_small_batch(2100, batch=2, num_qo_heads=8, num_kv_heads=2, page_size=16, causal=True,
                             q_len_range=(10, 30), kv_len_range=(3000, 4000), scale=0.5)
    dev = to_device(b)
    o1, l1, ws = run_library(b, num_sms=8, dev=dev)
    assert ws.info()[7] > 0
    for _ in range(2):
        o2, l2, _ = run_library(b, ws=ws, dev=dev)
        assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    ro, rl = A.batch_attention(b)
    assert_close(o1, l1, ro, rl)


def test_shared_prefix_composable():
    """Composable formats: prefix block row (tensor cores, split) + suffix rows (CUDA cores), merged with ⊕."""
    torch = torch_mod()
    from serving_attention_plan_gb300 import binding as B
    sp = W.shared_prefix_decode()
    dev = to_device(sp.flat)
    po, pl, wp = run_library(sp.prefix, dev=dev)
    so, sl, ws_ = run_library(sp.suffix, dev=dev)
    assert wp.info()[1] == 1 and ws_.info()[1] == 0
    t = lambda x, dt: torch.from_numpy(x).to(dt).cuda()
    o = torch.empty((64, 32, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((64, 32), dtype=torch.float32, device="cuda")
    B.merge_states(t(po, torch.bfloat16), t(pl, torch.float32), t(so, torch.bfloat16), t(sl, torch.float32), o, lse)
    torch.cuda.synchronize()
    ro, rl = A.batch_attention(sp.flat)
    assert_close(o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64), ro, rl)


def test_graph_replay_with_split_rows():
    """A captured tensor-core launch replays bit-identically and follows re-plans of the same total_q,
    with and without split rows (the split count is read from the plan, the launch is cooperative)."""
    torch = torch_mod()
    from serving_attention_plan_gb300 import binding as B
    mk = lambda seed, kr: W.random_small_batch(seed, batch=3, num_qo_heads=8, num_kv_heads=2, page_size=16,
                                               causal=True, q_len_range=(40, 40), kv_len_range=kr, scale=0.5)
    plans = [mk(2200, (1500, 3000)), mk(2201, (40, 200)), mk(2202, (2000, 4000))]
    pool = max(b.num_pages for b in plans)
    devs = [to_device(b) for b in plans]
    q = devs[0][0].clone()
    k = torch.zeros((pool,) + tuple(devs[0][1].shape[1:]), dtype=devs[0][1].dtype, device="cuda")
    v = torch.zeros_like(k)
    ws = B.Workspace(4, 120, pool, 8, 2, 128, 16)   # 16 CTAs: long rows split into 2-3 chunks
    o, lse = alloc_out(plans[0])
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = None
    for i, b in enumerate(plans):
        qi, ki, vi = devs[i]
        q.copy_(qi)
        k[: ki.shape[0]].copy_(ki)
        v[: vi.shape[0]].copy_(vi)
        ws.plan(b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, 16, True)
        assert ws.info()[1] == 1 and (ws.info()[7] > 0) == (i != 1)
        torch.cuda.synchronize()
        if g is None:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                ws.run(q, k, v, o, lse, stream=s)
        outs = []
        for _ in range(2):
            o.fill_(float("nan"))
            g.replay()
            torch.cuda.synchronize()
            outs.append((o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)))
        assert ws.get_error() == 0
        assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1])
        ro, rl = A.batch_attention(b)
        assert_close(outs[0][0], outs[0][1], ro, rl)


def test_prefill_ignores_values_past_the_last_token():
    """Tensor-core tiles copy whole pages: NaN values in the unused slots of each request's last page
    must not reach any output (the V rows past the last key are cleared before P.V)."""
    import dataclasses
    for ps in (16, 64):
        b = W.random_small_batch(2600 + ps, batch=5, num_qo_heads=8, num_kv_heads=2, page_size=ps, causal=True,
                                 q_len_range=(20, 150), kv_len_range=(150, 700), extra_pages=3, scale=0.5)
        k, v = b.k_pages.copy(), b.v_pages.copy()  # HND [pages, H_kv, page, D] bf16 bits
        for i in range(b.batch_size):
            lo, hi = int(b.kv_indptr[i]), int(b.kv_indptr[i + 1])
            if hi > lo:
                last, n = int(b.kv_indices[hi - 1]), int(b.last_page_len[i])
                k[last, :, n:, :] = 0x7FC0
                v[last, :, n:, :] = 0x7FC0
        o, lse, ws = run_library(dataclasses.replace(b, k_pages=k, v_pages=v), num_sms=3)
        assert ws.info()[1] == 1
        ro, rl = A.batch_attention(b)
        assert np.isfinite(o).all()
        assert_close(o, lse, ro, rl)

