"""GPU parity of the tcgen05 tensor-core path against the float64 oracle, through the C ABI."""
import numpy as np
import pytest

from oracle import attention as A
from serving_attention_plan_gb300 import workloads as W

from .gpu_helpers import assert_close, run_library, to_device, torch_mod

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from serving_attention_plan_gb300 import build
    build.build()
    assert torch_mod().cuda.is_available()


def test_single_tile_causal():
    """One request, one 128-row tile (32 tokens x g=4), one KV tile: the smallest tensor-core case."""
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


def test_ragged_causal_prefill_sampled():
    """Full-size ragged causal batch in the benchmark's launch configuration; oracle on sampled rows."""
    b = W.ragged_causal_prefill()
    o, lse, ws = run_library(b)
    h = ws.info()
    assert h[1] == 1 and h[2] == 32
    rng = np.random.default_rng(0)
    l_q = np.diff(b.qo_indptr)
    for i in rng.choice(b.batch_size, size=4, replace=False):
        for hq in rng.choice(b.num_qo_heads, size=3, replace=False):
            toks = np.unique(np.concatenate([[0, l_q[i] - 1], rng.integers(0, l_q[i], size=14)]))
            ro, rl = A.attention_rows(b, int(i), int(hq), toks)
            rows = int(b.qo_indptr[i]) + toks
            assert_close(o[rows, hq], lse[rows, hq], ro, rl)


def test_prefill_bit_identical_reruns():
    # few long rows on 16 CTAs: L_kv ~ 900 keys, so every row is cut into chunks merged in-kernel
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
