"""C-ABI library on the CPU: it loads, exports what include/fi.h declares, and its
host planner equals the oracle's plain restatement bit for bit (no GPU calls)."""
import os
import re

import numpy as np
import pytest

from oracle import planner as P
from serving_attention_plan_gb300 import binding as B
from serving_attention_plan_gb300 import build as BLD
from serving_attention_plan_gb300 import workloads as W


@pytest.fixture(scope="module")
def lib():
    BLD.build()
    return B.lib()


def test_exports_every_declared_symbol(lib, repo_root):
    header = open(os.path.join(repo_root, "include", "fi.h")).read()
    declared = set(re.findall(r"^\s*(?:int|const char\*)\s+(fi_\w+)\s*\(", header, flags=re.M))
    assert len(declared) >= 12
    for name in sorted(declared):
        assert hasattr(lib, name), name
    assert lib.fi_status_string(0) == b"ok"


def _compare(qo, kv, last, hq, hk, ps, causal, n_cta, **kw):
    got = B.plan_compute(qo, kv, last, hq, hk, ps, causal, n_cta, **kw)
    ref = P.serialize(P.plan(qo, kv, last, hq, hk, ps, causal, n_cta, **kw))
    assert got.shape == ref.shape, (got.shape, ref.shape)
    a, b = P.deserialize(got), P.deserialize(ref)
    for key in ("header", "cta_indptr", "items", "units", "slot_unit"):
        assert np.array_equal(a[key], b[key]), key
    return a


def _case(rng, ps_choices=(1, 8, 16, 32)):
    batch = int(rng.integers(1, 40))
    hk = int(rng.choice([1, 2, 8]))
    g = int(rng.choice([1, 2, 4, 8]))
    ps = int(rng.choice(ps_choices))
    causal = bool(rng.integers(0, 2))
    prefill = bool(rng.integers(0, 2))
    lq = rng.integers(0, 700, size=batch) if prefill else rng.integers(0, 2, size=batch)
    lk = rng.integers(0, 5000, size=batch)
    if causal:
        lk = np.maximum(lk, lq)
    if rng.integers(0, 3) == 0:
        lk[int(rng.integers(0, batch))] = int(rng.integers(30000, 140000))
    n_p = (lk + ps - 1) // ps
    kv = np.concatenate([[0], np.cumsum(n_p)])
    last = np.where(n_p > 0, lk - (n_p - 1) * ps, 0)
    qo = np.concatenate([[0], np.cumsum(lq)])
    return qo, kv, last, hk * g, hk, ps, causal


@pytest.mark.parametrize("seed", range(60))
def test_cpp_planner_matches_oracle(lib, seed):
    rng = np.random.default_rng(500 + seed)
    qo, kv, last, hq, hk, ps, causal = _case(rng)
    n_cta = int(rng.choice([1, 7, 148, 152, 304]))
    g = hq // hk
    if int(np.diff(qo).max(initial=0)) * g > 8 and (ps % 8 or 128 % ps):
        with pytest.raises(B.FiError) as ei:
            B.plan_compute(qo, kv, last, hq, hk, ps, causal, n_cta)
        assert ei.value.status == 3
        return
    _compare(qo, kv, last, hq, hk, ps, causal, n_cta,
             alpha=int(rng.integers(0, 4)), beta=int(rng.integers(1, 4)), l_min=int(rng.choice([1, 64, 256])))


@pytest.mark.parametrize("seed", range(6))
def test_cpp_planner_matches_oracle_with_large_cost_weights(lib, seed):
    """Weights whose costs do not fit the planner's packed 64-bit sort and queue keys take its general
    path; both paths must give the restatement's plan."""
    rng = np.random.default_rng(900 + seed)
    qo, kv, last, hq, hk, ps, causal = _case(rng)
    if int(np.diff(qo).max(initial=0)) * (hq // hk) > 8 and (ps % 8 or 128 % ps):
        return
    _compare(qo, kv, last, hq, hk, ps, causal, int(rng.choice([7, 152])), alpha=1 << 40, beta=1 << 12, l_min=64)


def test_hand_worked_plan_through_abi(lib, repo_root):
    import json
    gd = json.load(open(os.path.join(repo_root, "tests", "golden", "plan_hand_worked.json")))
    a = gd["inputs"]
    got = P.deserialize(B.plan_compute(a["qo_indptr"], a["kv_indptr"], a["last_page_len"], a["num_qo_heads"],
                                       a["num_kv_heads"], a["page_size"], a["causal"], a["num_ctas"],
                                       alpha=a["alpha"], beta=a["beta"], l_min=a["l_min"]))
    assert got["header"].tolist() == gd["expected"]["header"]
    assert got["items"].tolist() == gd["expected"]["items"]
    assert got["cta_indptr"].tolist() == gd["expected"]["cta_indptr"]


@pytest.mark.parametrize("name", ["tiny_decode", "llama3_8b_decode", "skewed_long_decode", "ragged_causal_prefill"])
def test_workload_plans_match(lib, name):
    """The five workloads' plans (lengths only, 152 CTAs) agree between C++ and the restatement."""
    b = {
        "tiny_decode": W.tiny_decode,
        "llama3_8b_decode": W.llama3_8b_decode,
        "skewed_long_decode": W.skewed_long_decode,
        "ragged_causal_prefill": W.ragged_causal_prefill,
    }[name](with_data=False)
    a = _compare(b.qo_indptr, b.kv_indptr, b.last_page_len, b.num_qo_heads, b.num_kv_heads, b.page_size, b.causal, 152)
    if name == "skewed_long_decode":
        assert a["header"][7] == 8          # the long request splits on each of its 8 KV heads
    if name == "ragged_causal_prefill":
        assert a["header"][1] == 1 and a["header"][2] == 64   # 256-row tiles: 64 tokens x g = 4


@pytest.mark.parametrize("name", W.KERNEL_DIST_WORKLOADS)
def test_kernel_distribution_plans_match(lib, name):
    """Kernel-level batches (16 requests; constant / uniform / Zipf lengths): C++ plan == restatement."""
    dist, mode = name.split("_")[1:]
    b = W.kernel_dist(dist, mode, with_data=False)
    a = _compare(b.qo_indptr, b.kv_indptr, b.last_page_len, b.num_qo_heads, b.num_kv_heads, b.page_size, b.causal, 152)
    assert a["header"][1] == (1 if mode == "prefill" else 0)


def test_kernel_distribution_lengths():
    """Lengths follow the stated distributions and are reproducible from the seed."""
    import numpy as np
    for name in W.KERNEL_DIST_WORKLOADS:
        dist, mode = name.split("_")[1:]
        b1 = W.kernel_dist(dist, mode, with_data=False)
        b2 = W.kernel_dist(dist, mode, with_data=False)
        assert np.array_equal(b1.kv_indptr, b2.kv_indptr) and np.array_equal(b1.last_page_len, b2.last_page_len)
        n_p = np.diff(b1.kv_indptr)
        lkv = (n_p - 1) * b1.page_size + b1.last_page_len
        assert b1.batch_size == 16
        if dist == "constant":
            assert np.all(lkv == 1024)
        elif dist == "uniform":
            assert lkv.min() >= 512 and lkv.max() <= 1024
        else:
            assert np.all(lkv % 512 == 0) and lkv.min() >= 512 and lkv.max() <= 16384
        if mode == "prefill":
            assert np.array_equal(np.diff(b1.qo_indptr), lkv) and b1.causal
        else:
            assert np.all(np.diff(b1.qo_indptr) == 1) and not b1.causal


def test_shared_prefix_plans_match(lib):
    sp = W.shared_prefix_decode()
    for part in (sp.prefix, sp.suffix):
        _compare(part.qo_indptr, part.kv_indptr, part.last_page_len, part.num_qo_heads, part.num_kv_heads,
                 part.page_size, part.causal, 152)
    pre = P.deserialize(B.plan_compute(sp.prefix.qo_indptr, sp.prefix.kv_indptr, sp.prefix.last_page_len, 32, 8, 16,
                                       False, 152))
    assert pre["header"][1] == 1 and pre["header"][7] > 0   # tensor-core tiles, split across CTAs


def test_plan_ignores_page_ids_and_is_deterministic(lib):
    rng = np.random.default_rng(3)
    qo, kv, last, hq, hk, ps, causal = _case(rng, ps_choices=(16,))
    a = B.plan_compute(qo, kv, last, hq, hk, ps, causal, 152)
    b = B.plan_compute(qo, kv, last, hq, hk, ps, causal, 152)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("bad", ["qo_not_monotone", "kv_start", "last_zero", "last_big", "head_dim", "heads"])
def test_invalid_inputs_rejected(lib, bad):
    qo = np.array([0, 1, 2]); kv = np.array([0, 2, 3]); last = np.array([5, 16]); hq, hk, d = 8, 2, 128
    expect = 1
    if bad == "qo_not_monotone":
        qo = np.array([0, 2, 1])
    elif bad == "kv_start":
        kv = np.array([1, 2, 3])
    elif bad == "last_zero":
        last = np.array([0, 16])
    elif bad == "last_big":
        last = np.array([17, 16])
    elif bad == "head_dim":
        d, expect = 64, 3
    elif bad == "heads":
        hq, expect = 7, 3
    with pytest.raises(B.FiError) as ei:
        B.plan_compute(qo, kv, last, hq, hk, 16, False, 4, head_dim=d)
    assert ei.value.status == expect


def test_tensor_core_path_page_size_rule(lib):
    qo = np.array([0, 100]); kv = np.array([0, 100]); last = np.array([1])
    with pytest.raises(B.FiError) as ei:
        B.plan_compute(qo, kv, last, 8, 2, 1, True, 4)   # 400 rows, page size 1: not tiled by TMA boxes
    assert ei.value.status == 3


@pytest.mark.parametrize("seed", range(30))
def test_cpp_planner_matches_oracle_with_window(lib, seed):
    """Sliding-window plans (causal): C++ == restatement, bit for bit; non-causal windows rejected."""
    rng = np.random.default_rng(800 + seed)
    qo, kv, last, hq, hk, ps, causal = _case(rng, ps_choices=(1, 8, 16))
    n_cta = int(rng.choice([1, 7, 152]))
    w = int(rng.choice([0, 3, 64, 999, 10 ** 6]))
    g = hq // hk
    if int(np.diff(qo).max(initial=0)) * g > 8 and ps % 8:
        return
    if not causal:
        with pytest.raises(B.FiError) as ei:
            B.plan_compute(qo, kv, last, hq, hk, ps, False, n_cta, window_left=w)
        assert ei.value.status == 3
        return
    _compare(qo, kv, last, hq, hk, ps, True, n_cta, window_left=w)


def test_key_positions_beyond_int32_items_rejected(lib):
    """Item fields are int32: a KV length above 2^30 (page ids may repeat, page sizes are unbounded) is
    UNSUPPORTED rather than wrapped.  Both the workspace planner and the allocation-free entry point run
    this same planner code, so both reject it."""
    ps = 1 << 20
    qo = np.array([0, 1]); kv = np.array([0, 1025]); last = np.array([ps])  # 1025 pages of 2^20 keys
    with pytest.raises(B.FiError) as ei:
        B.plan_compute(qo, kv, last, 8, 2, ps, False, 4)
    assert ei.value.status == 3
    kv = np.array([0, 1024]); last = np.array([1])                          # 2^30 - 2^20 + 1 keys: fine
    assert B.plan_compute(qo, kv, last, 8, 2, ps, False, 4)[0] == 0x46495031


def _composable_case(rng):
    """Random shared-prefix groups (tensor-core tiles) over decode requests with their own pages."""
    g = int(rng.choice([1, 2, 4, 8]))
    hk = int(rng.choice([1, 2, 8]))
    ps = int(rng.choice([8, 16, 32]))
    n_req = int(rng.integers(1, 40))
    q_len = int(rng.integers(1, 8 // g + 1))
    qo = np.arange(n_req + 1) * q_len
    kv_lens = rng.integers(0, 900, size=n_req)
    kv = np.concatenate([[0], np.cumsum((kv_lens + ps - 1) // ps)])
    last = np.where(kv_lens > 0, kv_lens - (np.maximum((kv_lens + ps - 1) // ps, 1) - 1) * ps, 0)
    # shared groups: contiguous runs of requests (some requests in none), each with its own prefix
    cuts = sorted(set(rng.integers(0, n_req + 1, size=int(rng.integers(1, 4))).tolist()) | {0, n_req})
    s_qo, s_kv, s_last = [0], [0], []
    for lo, hi in zip(cuts[:-1], cuts[1:]):
        if hi == lo:
            continue
        s_qo.append(int(qo[hi]) - int(qo[cuts[0]]) + s_qo[0])
        plen = int(rng.integers(0, 3000))
        s_kv.append(s_kv[-1] + (plen + ps - 1) // ps)
        s_last.append(plen - (max((plen + ps - 1) // ps, 1) - 1) * ps if plen > 0 else 0)
    return (np.array(s_qo), np.array(s_kv), np.array(s_last)), (qo, kv, last), g * hk, hk, ps


@pytest.mark.parametrize("seed", range(25))
def test_composable_plan_matches_oracle(lib, seed):
    """Composable plans (shared sub-matrix on tensor-core tiles, per-request rows on decode tiles, one
    reduction map with the shared slots each unit merges): C++ == restatement, bit for bit."""
    rng = np.random.default_rng(900 + seed)
    shared, unique, hq, hk, ps = _composable_case(rng)
    n_cta = int(rng.choice([1, 5, 152]))
    causal = bool(rng.integers(0, 2))
    got = B.plan_composable_compute(shared, unique, hq, hk, ps, causal, n_cta)
    a, b, ext = P.plan_composable(shared, unique, hq, hk, ps, causal, n_cta)
    want = P.serialize_composable(a, b, ext)
    assert np.array_equal(got, want)


def test_shared_prefix_composable_plan(lib):
    """The shared-prefix workload: 64 requests share one 8192-token prefix.  Every suffix unit lists
    the prefix's chunk slots of its KV head, and the plan is the restatement's."""
    sp = W.shared_prefix_decode()
    shared = (sp.prefix.qo_indptr, sp.prefix.kv_indptr, sp.prefix.last_page_len)
    unique = (sp.suffix.qo_indptr, sp.suffix.kv_indptr, sp.suffix.last_page_len)
    got = B.plan_composable_compute(shared, unique, 32, 8, 16, False, 152)
    a, b, ext = P.plan_composable(shared, unique, 32, 8, 16, False, 152)
    assert np.array_equal(got, P.serialize_composable(a, b, ext))
    assert a.path == P.PATH_TENSOR and b.path == P.PATH_DECODE
    n_chunks = a.units[0]["n_chunks"]
    assert all(u["ext_count"] == n_chunks for u in b.units)   # each suffix unit merges every prefix chunk of its head
    assert len(ext) == len(b.units) * n_chunks


@pytest.mark.parametrize("case", [
    # (n_req, hq, hk, page, own range, prefix length, SM budget)
    (8, 8, 2, 16, (1, 50), 20000, 152),   # one long prefix over many CTAs: 74 shared slots a row
    (80, 2, 1, 16, (1, 60), 300, 2),      # one decode CTA holding 80 units with shared states
])
def test_composable_plan_long_slot_lists_and_crowded_ctas(lib, case):
    """Composable plans at the ends the kernels treat specially: rows that merge dozens of shared
    slots, and a decode CTA with more units to merge than its deferred list holds.  C++ ==
    restatement, bit for bit, and the slot lists have the lengths those cases rely on."""
    n_req, hq, hk, ps, own, plen, n_cta = case
    rng = np.random.default_rng(1234 + n_req)
    own_lens = rng.integers(own[0], own[1] + 1, size=n_req)
    qo = np.arange(n_req + 1)
    kv = np.concatenate([[0], np.cumsum((own_lens + ps - 1) // ps)])
    last = own_lens - ((own_lens + ps - 1) // ps - 1) * ps
    n_p = (plen + ps - 1) // ps
    shared = (np.array([0, n_req]), np.array([0, n_p]), np.array([plen - (n_p - 1) * ps]))
    unique = (qo, kv, last)
    got = B.plan_composable_compute(shared, unique, hq, hk, ps, False, n_cta)
    a, b, ext = P.plan_composable(shared, unique, hq, hk, ps, False, n_cta)
    assert np.array_equal(got, P.serialize_composable(a, b, ext))
    counts = [u["ext_count"] for u in b.units]
    if plen > 10000:
        assert max(counts) > 32          # longer than one warp's lanes
    else:
        assert len(b.queues) == 1 and len(b.units) > 64
