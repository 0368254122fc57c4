"""Pins for the plain-Python planner restatement (CPU only).

Checks the planner against a plan worked by hand, against coverage and bound
invariants computed by brute force, and against Graham's bound for
longest-processing-time-first list scheduling (makespan <= (4/3 - 1/(3m)) OPT),
with OPT found by exhaustive search on tiny instances.  Source: page
"FlashInfer：面向 LLM 推理服务的高效可定制注意力引擎", 核心机制 6 (paper §3.3.1,
Alg. 1) and 核心机制 7 (paper App. D.2-D.3).
"""
import itertools
import json
import os

import numpy as np
import pytest

from oracle import planner as P

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_hand_worked_plan():
    gd = json.load(open(os.path.join(GOLDEN, "plan_hand_worked.json")))
    a = gd["inputs"]
    p = P.plan(a["qo_indptr"], a["kv_indptr"], a["last_page_len"], a["num_qo_heads"], a["num_kv_heads"],
               a["page_size"], a["causal"], a["num_ctas"], alpha=a["alpha"], beta=a["beta"], l_min=a["l_min"])
    flat = P.deserialize(P.serialize(p))
    e = gd["expected"]
    assert flat["header"].tolist() == e["header"]
    assert flat["cta_indptr"].tolist() == e["cta_indptr"]
    assert flat["items"].tolist() == e["items"]
    assert flat["units"].tolist() == e["units"]
    assert flat["slot_unit"].tolist() == e["slot_unit"]
    assert p.loads == e["loads"]


def _random_case(rng):
    batch = int(rng.integers(1, 12))
    hk = int(rng.choice([1, 2, 4]))
    g = int(rng.choice([1, 2, 4, 8]))
    ps = int(rng.choice([1, 4, 16]))
    causal = bool(rng.integers(0, 2))
    prefill = bool(rng.integers(0, 2))
    lq = rng.integers(0, 300, size=batch) if prefill else np.ones(batch, np.int64)
    lk = np.maximum(lq, rng.integers(0, 3000, size=batch)) if causal else rng.integers(0, 3000, size=batch)
    if rng.integers(0, 3) == 0:
        lk[0] = int(rng.integers(20000, 60000))          # one long request
    n_p = (lk + ps - 1) // ps
    kv_indptr = np.concatenate([[0], np.cumsum(n_p)])
    last = np.where(n_p > 0, lk - (n_p - 1) * ps, 0)
    qo_indptr = np.concatenate([[0], np.cumsum(lq)])
    n_cta = int(rng.choice([1, 3, 16, 152]))
    return dict(qo_indptr=qo_indptr, kv_indptr=kv_indptr, last=last, hq=hk * g, hk=hk, ps=ps, causal=causal,
                n_cta=n_cta, lq=lq, lk=lk)


@pytest.mark.parametrize("seed", range(40))
def test_coverage_and_bounds(seed):
    rng = np.random.default_rng(seed)
    c = _random_case(rng)
    p = P.plan(c["qo_indptr"], c["kv_indptr"], c["last"], c["hq"], c["hk"], c["ps"], c["causal"], c["n_cta"])
    lq, lk, g = c["lq"], c["lk"], c["hq"] // c["hk"]
    # tile rule
    if int(lq.max(initial=0)) * g <= 8:
        assert p.path == P.PATH_DECODE and p.rows_tile >= int(lq.max(initial=1)) * g
    else:
        assert p.path == P.PATH_TENSOR and p.tile_tokens * g <= P.TC_ROWS and p.rows_tile == P.TC_ROWS
    # chunk bound: a whole number of pages, at least l_min and at least total / #CTA
    total = sum(c["hk"] * -(-int(lq[i]) // p.tile_tokens) * int(lk[i]) for i in range(len(lq)))
    assert p.num_ctas == c["n_cta"] * (P.TC_CTAS_PER_SM if p.path == P.PATH_TENSOR else P.DECODE_CTAS_PER_SM)
    assert p.l_kv_chunk % c["ps"] == 0 and p.l_kv_chunk >= 256 and p.l_kv_chunk * p.num_ctas >= total
    # every (request, kv head, tile) covers its visible keys exactly once with contiguous chunks
    by_unit = {}
    for it in p.items:
        by_unit.setdefault((it["request"], it["kv_head"], it["tile"]), []).append(it)
    n_units = 0
    for i in range(len(lq)):
        n_tiles = -(-int(lq[i]) // p.tile_tokens)
        for h in range(c["hk"]):
            for j in range(n_tiles):
                n_units += 1
                chunks = sorted(by_unit[(i, h, j)], key=lambda x: x["chunk"])
                toks = range(j * p.tile_tokens, min((j + 1) * p.tile_tokens, int(lq[i])))
                # brute force: largest number of keys any token of the tile may see
                keys = np.arange(int(lk[i]))
                e = 0
                for t in toks:
                    e = max(e, int(np.count_nonzero((keys <= lk[i] - lq[i] + t) | (not c["causal"]))))
                pos = 0
                for ch in chunks:
                    assert ch["kv_lo"] == pos and ch["kv_hi"] >= ch["kv_lo"]
                    assert ch["kv_hi"] - ch["kv_lo"] <= p.l_kv_chunk
                    assert ch["kv_lo"] % c["ps"] == 0
                    pos = ch["kv_hi"]
                assert pos == e
                # direct write iff a single chunk
                if len(chunks) == 1:
                    assert chunks[0]["slot"] == -1
                else:
                    slots = [ch["slot"] for ch in chunks]
                    assert slots == list(range(slots[0], slots[0] + len(chunks)))
                # the diagonal offset places token u of the tile at key limit diag + u
                if c["causal"]:
                    for t in toks:
                        assert chunks[0]["diag"] + (t - j * p.tile_tokens) == lk[i] - lq[i] + t
    assert sum(1 for _ in by_unit) == n_units
    # partial-output bound (App. D.3): partial tiles < 2 * #CTA
    assert len(p.slot_unit) < 2 * p.num_ctas or len(p.slot_unit) == 0
    # each item exactly once; queues in non-increasing cost (longest first)
    seen = sorted(k for q in p.queues for k in q)
    assert seen == list(range(len(p.items)))
    for q in p.queues:
        costs = [p.items[k]["cost"] for k in q]
        assert costs == sorted(costs, reverse=True)
    # list-scheduling bound: makespan <= sum/m + (1 - 1/m) * max cost
    costs = [it["cost"] for it in p.items]
    if costs:
        assert max(p.loads) <= sum(costs) / p.num_ctas + (1 - 1 / p.num_ctas) * max(costs) + 1e-9
    assert sum(p.loads) == sum(costs)


def _opt_makespan(costs, m):
    best = None
    for assign in itertools.product(range(m), repeat=len(costs)):
        loads = [0] * m
        for c, a in zip(costs, assign):
            loads[a] += c
        best = max(loads) if best is None else min(best, max(loads))
    return best


@pytest.mark.parametrize("seed", range(60))
def test_graham_lpt_bound_tiny(seed):
    """LPT makespan <= (4/3 - 1/(3m)) * OPT; OPT by exhaustive search over all assignments."""
    rng = np.random.default_rng(1000 + seed)
    m = int(rng.integers(2, 4))
    n = int(rng.integers(m + 1, 9))
    lk = rng.integers(1, 200, size=n)
    kv_indptr = np.concatenate([[0], np.cumsum(lk)])          # page size 1
    p = P.plan(np.arange(n + 1), kv_indptr, np.ones(n, np.int64), 1, 1, 1, False, m, l_min=10 ** 6)
    costs = [it["cost"] for it in p.items]
    assert len(costs) == n
    opt = _opt_makespan(costs, m)
    assert max(p.loads) * 3 * m <= (4 * m - 1) * opt


def test_plan_deterministic():
    rng = np.random.default_rng(77)
    c = _random_case(rng)
    a = P.serialize(P.plan(c["qo_indptr"], c["kv_indptr"], c["last"], c["hq"], c["hk"], c["ps"], c["causal"], c["n_cta"]))
    b = P.serialize(P.plan(c["qo_indptr"], c["kv_indptr"], c["last"], c["hq"], c["hk"], c["ps"], c["causal"], c["n_cta"]))
    assert np.array_equal(a, b)


def test_skewed_long_request_is_split():
    """The 131072-token request of the skewed decode workload is chunked; short ones write directly."""
    lk = np.array([131072] + [640] * 63)
    kv_indptr = np.concatenate([[0], np.cumsum(lk)])
    p = P.plan(np.arange(65), kv_indptr, np.ones(64, np.int64), 64, 8, 1, False, 152)
    long_items = [it for it in p.items if it["request"] == 0]
    assert len(long_items) > 8 and all(it["slot"] >= 0 for it in long_items)
    assert all(it["slot"] == -1 for it in p.items if it["request"] != 0)
    assert len(p.units) == 8


@pytest.mark.parametrize("seed", range(30))
def test_sliding_window_coverage(seed):
    """With a window (causal), a tile's chunks cover exactly [first key any of its tokens can see,
    last key), the start rounded down to a page; brute force over the tokens' windows."""
    rng = np.random.default_rng(900 + seed)
    c = _random_case(rng)
    if not c["causal"]:
        with pytest.raises(ValueError):
            P.plan(c["qo_indptr"], c["kv_indptr"], c["last"], c["hq"], c["hk"], c["ps"], False, c["n_cta"],
                   window_left=5)
        return
    w = int(rng.choice([0, 1, 17, 300, 5000]))
    p = P.plan(c["qo_indptr"], c["kv_indptr"], c["last"], c["hq"], c["hk"], c["ps"], True, c["n_cta"],
               window_left=w)
    lq, lk = c["lq"], c["lk"]
    by_unit = {}
    for it in p.items:
        by_unit.setdefault((it["request"], it["kv_head"], it["tile"]), []).append(it)
    for (i, h, j), chunks in by_unit.items():
        chunks = sorted(chunks, key=lambda x: x["chunk"])
        toks = range(j * p.tile_tokens, min((j + 1) * p.tile_tokens, int(lq[i])))
        vis = [k for t in toks for k in range(int(lk[i])) if lk[i] - lq[i] + t - w <= k <= lk[i] - lq[i] + t]
        lo, hi = chunks[0]["kv_lo"], chunks[-1]["kv_hi"]
        if vis:
            assert lo <= min(vis) and min(vis) - lo < c["ps"] and lo % c["ps"] == 0
            assert hi == max(vis) + 1
        else:
            assert lo == hi
        for a, b in zip(chunks, chunks[1:]):
            assert a["kv_hi"] == b["kv_lo"] and b["kv_lo"] % c["ps"] == 0
        assert all(ch["kv_hi"] - ch["kv_lo"] <= p.l_kv_chunk for ch in chunks)
    costs = [it["cost"] for it in p.items]
    if costs:
        assert max(p.loads) <= sum(costs) / p.num_ctas + (1 - 1 / p.num_ctas) * max(costs) + 1e-9


def test_wide_window_plan_equals_no_window_chunks():
    """A window longer than every KV reads the same keys as no window (only L_kv's sum differs)."""
    lk = np.array([700, 1500, 90])
    lq = np.array([3, 1, 90])
    kv = np.concatenate([[0], np.cumsum((lk + 15) // 16)])
    last = lk - ((lk + 15) // 16 - 1) * 16
    qo = np.concatenate([[0], np.cumsum(lq)])
    a = P.plan(qo, kv, last, 8, 2, 16, True, 4, window_left=10 ** 6)
    b = P.plan(qo, kv, last, 8, 2, 16, True, 4)
    cover = lambda pl: sorted((it["request"], it["kv_head"], it["tile"], it["kv_lo"]) for it in pl.items if it["chunk"] == 0)
    assert cover(a) == cover(b)
