"""GPU parity of composable formats: attention of one KV sub-matrix merged (⊕) into the state of
another by the kernel that writes the rows (fi_run_merge), against the float64 oracle of the
whole KV.  Source: page "FlashInfer：面向 LLM 推理服务的高效可定制注意力引擎", 核心机制 2
(paper §3.1.2, Fig. 3) and 术语与记号 "Attention State 与 ⊕" (paper §2.2)."""
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
    assert torch_mod().cuda.is_available()


def split_pages(b, frac):
    """Two batches over disjoint page sets of every request: its first pages and the rest."""
    head_i, head_p, head_l, tail_i, tail_p, tail_l = [], [0], [], [], [0], []
    for i in range(b.batch_size):
        pages = b.kv_indices[b.kv_indptr[i]:b.kv_indptr[i + 1]]
        n_head = int(len(pages) * frac)
        if n_head == len(pages) and len(pages) > 0:
            n_head -= 1  # the partial last page stays in the tail
        head_i.append(pages[:n_head])
        tail_i.append(pages[n_head:])
        head_p.append(head_p[-1] + n_head)
        tail_p.append(tail_p[-1] + len(pages) - n_head)
        head_l.append(b.page_size if n_head else 0)
        tail_l.append(int(b.last_page_len[i]) if len(pages) > n_head else 0)
    mk = lambda idx, ptr, last: dataclasses.replace(
        b, kv_indices=np.concatenate(idx).astype(np.int32), kv_indptr=np.array(ptr, np.int32),
        last_page_len=np.array(last, np.int32))
    return mk(head_i, head_p, head_l), mk(tail_i, tail_p, tail_l)


def run_split(b, frac, num_sms):
    from serving_attention_plan_gb300 import binding as B
    torch = torch_mod()
    head, tail = split_pages(b, frac)
    dev = to_device(b)
    o, lse, ws_h = run_library(head, num_sms=num_sms, dev=dev)
    o_t = torch.from_numpy(o).to(torch.bfloat16).cuda()
    l_t = torch.from_numpy(lse).to(torch.float32).cuda()
    ws = B.Workspace(tail.batch_size, tail.total_q, max(int(tail.kv_indptr[-1]), 1), b.num_qo_heads,
                     b.num_kv_heads, 128, num_sms)
    ws.plan(tail.qo_indptr, tail.kv_indptr, tail.kv_indices, tail.last_page_len, b.page_size, b.causal)
    ws.run_merge(dev[0], dev[1], dev[2], o_t, l_t, o_t, l_t)   # in place
    torch.cuda.synchronize()
    assert ws.get_error() == 0
    return (o_t.float().cpu().numpy().astype(np.float64), l_t.cpu().numpy().astype(np.float64), ws_h.info(),
            ws.info())


CASES = [
    # (hq, hk, page, q range, kv range, SM budget, head fraction)
    (8, 1, 16, (1, 1), (0, 4000), 5, 0.5),        # decode path, g = 8, split rows in both parts
    (64, 8, 1, (1, 1), (1, 600), 0, 0.3),         # decode path, g = 8, page 1
    (8, 2, 16, (20, 80), (0, 1500), 32, 0.5),     # tensor-core path, split rows (contraction kernel merges)
    (16, 4, 32, (40, 90), (100, 700), 0, 0.7),    # tensor-core path, direct writes merge in the epilogue
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_run_merge_matches_whole_kv(case):
    hq, hk, ps, qr, kr, n_sms, frac = CASES[case]
    b = W.random_small_batch(3000 + case, batch=7, num_qo_heads=hq, num_kv_heads=hk, page_size=ps, causal=False,
                             q_len_range=qr, kv_len_range=kr, extra_pages=3, scale=0.5)
    o, lse, h_head, h_tail = run_split(b, frac, n_sms)
    assert h_head[1] == h_tail[1] == (0 if qr[1] == 1 else 1)
    if case in (0, 2):
        assert h_head[7] > 0 and h_tail[7] > 0
    ro, rl = A.batch_attention(b)
    assert_close(o, lse, ro, rl)


def test_shared_prefix_fused_merge():
    """Prefix block row on tensor cores, then the suffix decode writes prefix ⊕ suffix in place."""
    torch = torch_mod()
    from serving_attention_plan_gb300 import binding as B
    sp = W.shared_prefix_decode()
    dev = to_device(sp.flat)
    po, pl, _ = run_library(sp.prefix, dev=dev)
    o = torch.from_numpy(po).to(torch.bfloat16).cuda()
    lse = torch.from_numpy(pl).to(torch.float32).cuda()
    ws = B.Workspace(64, 64, int(sp.suffix.kv_indptr[-1]), 32, 8)
    ws.plan(sp.suffix.qo_indptr, sp.suffix.kv_indptr, sp.suffix.kv_indices, sp.suffix.last_page_len, 16, False)
    outs = []
    for _ in range(2):
        o2, l2 = o.clone(), lse.clone()
        ws.run_merge(dev[0], dev[1], dev[2], o, lse, o2, l2)
        torch.cuda.synchronize()
        outs.append((o2.float().cpu().numpy().astype(np.float64), l2.cpu().numpy().astype(np.float64)))
    assert ws.get_error() == 0
    assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1])
    ro, rl = A.batch_attention(sp.flat)
    assert_close(outs[0][0], outs[0][1], ro, rl)


def test_run_merge_rejects_half_state():
    from serving_attention_plan_gb300 import binding as B
    b = W.random_small_batch(3100, batch=2, num_qo_heads=8, num_kv_heads=2, page_size=16, causal=False,
                             kv_len_range=(16, 64))
    q, k, v = to_device(b)
    o, lse = alloc_out(b)
    ws = B.Workspace(2, 2, int(b.kv_indptr[-1]), 8, 2)
    ws.plan(b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, 16, False)
    with pytest.raises(B.FiError) as ei:
        ws.run_merge(q, k, v, o, None, o, lse)
    assert ei.value.status == 1


# ---- one composable plan: shared sub-matrix + per-request rows, one reduction map ----------------

def composable_batch(seed, n_req, hq, hk, ps, q_len, own_range, n_groups, prefix_range, causal):
    """Per-request rows with their own pages, plus groups of consecutive requests that share a prefix
    (the shared sub-matrix), all pages drawn from one pool."""
    rng = np.random.default_rng(seed)
    own = rng.integers(own_range[0], own_range[1] + 1, size=n_req)
    cuts = sorted(set(rng.integers(1, n_req, size=max(0, n_groups - 1)).tolist()) | {0, n_req})
    plens = rng.integers(prefix_range[0], prefix_range[1] + 1, size=len(cuts) - 1)
    n_shared = int(sum((int(x) + ps - 1) // ps for x in plens))
    n_own = int(sum((int(x) + ps - 1) // ps for x in own))
    b = W.make_paged_batch(rng, f"composable_{seed}", np.full(n_req, q_len), own, hq, hk, ps, causal,
                           pool_pages=n_own + n_shared + 2, scale=0.7)
    free = np.setdiff1d(np.arange(b.num_pages), b.kv_indices)
    rng.shuffle(free)
    s_qo, s_kv, s_last = [0], [0], []
    for (lo, hi), plen in zip(zip(cuts[:-1], cuts[1:]), plens):
        s_qo.append(int(b.qo_indptr[hi]))
        n_p = (int(plen) + ps - 1) // ps
        s_kv.append(s_kv[-1] + n_p)
        s_last.append(int(plen) - (n_p - 1) * ps if n_p else 0)
    shared = dataclasses.replace(b, qo_indptr=np.array(s_qo, np.int32), kv_indptr=np.array(s_kv, np.int32),
                                 kv_indices=free[: s_kv[-1]].astype(np.int32),
                                 last_page_len=np.array(s_last, np.int32), causal=False)
    return shared, b


def composable_reference(shared, unique):
    """Oracle: each row's state over its group's shared keys ⊕ its state over its own keys."""
    so, sl = A.batch_attention(shared)
    po = np.zeros((unique.total_q,) + so.shape[1:])
    pl = np.full((unique.total_q, so.shape[1]), -np.inf)
    po[: so.shape[0]], pl[: sl.shape[0]] = so, sl
    uo, ul = A.batch_attention(unique)
    return A.merge_states(po, pl, uo, ul)


def run_composable(shared, unique, num_sms=0, ws=None, dev=None):
    from serving_attention_plan_gb300 import binding as B
    torch = torch_mod()
    if ws is None:
        ws = B.Workspace(max(unique.batch_size, shared.batch_size), unique.total_q,
                         max(int(unique.kv_indptr[-1]), int(shared.kv_indptr[-1]), 1), unique.num_qo_heads,
                         unique.num_kv_heads, 128, num_sms)
    q, k, v = dev if dev is not None else to_device(unique)
    o, lse = alloc_out(unique)
    ws.plan_composable((shared.qo_indptr, shared.kv_indptr, shared.kv_indices, shared.last_page_len),
                       (unique.qo_indptr, unique.kv_indptr, unique.kv_indices, unique.last_page_len),
                       unique.page_size, unique.causal)
    ws.run(q, k, v, o, lse)
    torch.cuda.synchronize()
    assert ws.get_error() == 0
    return o.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64), ws


def test_shared_prefix_one_plan_matches_flat_oracle():
    """The shared-prefix workload as one composable plan (two launches): every row equals attention over
    prefix ++ own suffix, and reruns are bit-identical."""
    sp = W.shared_prefix_decode()
    dev = to_device(sp.flat)
    o, lse, ws = run_composable(sp.prefix, sp.suffix, dev=dev)
    assert ws.info()[1] == 2
    ro, rl = A.batch_attention(sp.flat)
    assert_close(o, lse, ro, rl)
    o2, l2, _ = run_composable(sp.prefix, sp.suffix, ws=ws, dev=dev)
    assert np.array_equal(o, o2) and np.array_equal(lse, l2)


COMPOSABLE_CASES = [
    # (n_req, hq, hk, page, q_len, own range, groups, prefix range, causal, SM budget); the workspace holds
    # 2 x budget partial slots, and every chunk of the shared part takes one
    (9, 8, 2, 16, 1, (0, 300), 2, (0, 700), False, 0),
    (20, 8, 2, 16, 1, (1, 900), 3, (100, 2000), False, 16),     # few CTAs: long shared rows split in chunks
    (7, 8, 4, 8, 2, (2, 200), 2, (1, 400), True, 6),            # 2 query tokens (4 rows), causal own part
    (33, 64, 8, 32, 1, (0, 500), 4, (0, 3000), False, 24),      # g = 8, page 32, empty prefixes possible
    (5, 16, 16, 16, 4, (4, 100), 1, (50, 300), True, 10),       # g = 1, 4 tokens per request
    (8, 8, 2, 16, 1, (1, 50), 1, (20000, 20000), False, 0),     # 74 shared slots a row: lists of more than 32
    (12, 8, 2, 16, 1, (1, 200), 1, (3000, 4000), False, 0),     # 13 shared slots a row
    (80, 2, 1, 16, 1, (1, 60), 1, (100, 300), False, 2),        # 80 deferred units in one CTA: 16 merged at once
]


@pytest.mark.parametrize("case", range(len(COMPOSABLE_CASES)))
def test_composable_matches_oracle(case):
    n_req, hq, hk, ps, ql, own, ng, pre, causal, n_sms = COMPOSABLE_CASES[case]
    shared, unique = composable_batch(7000 + case, n_req, hq, hk, ps, ql, own, ng, pre, causal)
    o, lse, ws = run_composable(shared, unique, num_sms=n_sms)
    assert ws.info()[1] == 2
    ro, rl = composable_reference(shared, unique)
    assert_close(o, lse, ro, rl)


def test_composable_unsupported_combinations():
    from serving_attention_plan_gb300 import binding as B
    shared, unique = composable_batch(7100, 6, 8, 2, 16, 1, (1, 100), 2, (10, 100), False)
    ws = B.Workspace(8, 64, 64, 8, 2)
    ws.set_variant(window_left=-1, logits_soft_cap=5.0)
    with pytest.raises(B.FiError) as ei:
        ws.plan_composable((shared.qo_indptr, shared.kv_indptr, shared.kv_indices, shared.last_page_len),
                           (unique.qo_indptr, unique.kv_indptr, unique.kv_indices, unique.last_page_len), 16, False)
    assert ei.value.status == 3
    # per-request rows beyond a decode tile (here 3 tokens x g = 4 = 12 rows)
    shared, unique = composable_batch(7101, 4, 8, 2, 16, 3, (3, 100), 1, (10, 100), True)
    ws = B.Workspace(8, 64, 64, 8, 2)
    with pytest.raises(B.FiError) as ei:
        ws.plan_composable((shared.qo_indptr, shared.kv_indptr, shared.kv_indices, shared.last_page_len),
                           (unique.qo_indptr, unique.kv_indptr, unique.kv_indices, unique.last_page_len), 16, True)
    assert ei.value.status == 3
