"""Pins for the float64 attention oracle (CPU only).

Each test checks the oracle against something other than itself: explicit
brute force, an independent library routine, closed forms, hand-worked values,
or an algebraic invariant of the attention state (page "FlashInfer：面向 LLM
推理服务的高效可定制注意力引擎", 术语与记号 "Attention State 与 ⊕", paper §2.2;
核心机制 1-2, paper §3.1.1-3.1.2).
"""
import json
import math
import os

import numpy as np
import pytest

from oracle import attention as A
from serving_attention_plan_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
TOL = 1e-12


def _brute_force(b, scale, window_left=-1, soft_cap=0.0):
    """Explicit loops, Python floats, math.exp: the attention definition element by element."""
    d = b.head_dim
    g = b.num_qo_heads // b.num_kv_heads
    out_o = {}
    out_l = {}
    for i in range(b.batch_size):
        n_pages = int(b.kv_indptr[i + 1] - b.kv_indptr[i])
        # walk the page list, collecting key/value rows in order
        for h in range(b.num_qo_heads):
            hk = h // g
            keys, vals = [], []
            for pi in range(n_pages):
                page = int(b.kv_indices[b.kv_indptr[i] + pi])
                rows = b.page_size if pi < n_pages - 1 else int(b.last_page_len[i])
                for r in range(rows):
                    keys.append([float(x) for x in A.bf16_to_f64(b.k_pages[page, hk, r])])
                    vals.append([float(x) for x in A.bf16_to_f64(b.v_pages[page, hk, r])])
            lq = int(b.qo_indptr[i + 1] - b.qo_indptr[i])
            lk = len(keys)
            for t in range(lq):
                row = int(b.qo_indptr[i]) + t
                q = [float(x) for x in A.bf16_to_f64(b.q[row, h])]
                allowed = [j for j in range(lk) if (not b.causal) or j <= lk - lq + t]
                if window_left >= 0:
                    allowed = [j for j in allowed if j >= lk - lq + t - window_left]
                if not allowed:
                    out_o[(row, h)] = [0.0] * d
                    out_l[(row, h)] = -math.inf
                    continue
                s = {j: scale * sum(q[c] * keys[j][c] for c in range(d)) for j in allowed}
                if soft_cap > 0:
                    s = {j: soft_cap * math.tanh(x / soft_cap) for j, x in s.items()}
                m = max(s.values())
                z = sum(math.exp(s[j] - m) for j in allowed)
                out_l[(row, h)] = m + math.log(z)
                out_o[(row, h)] = [sum(math.exp(s[j] - m) / z * vals[j][c] for j in allowed) for c in range(d)]
    return out_o, out_l


@pytest.mark.parametrize("seed", range(6))
def test_brute_force_tiny(seed):
    rng = np.random.default_rng(100 + seed)
    d = int(rng.choice([4, 8]))
    hk = int(rng.choice([1, 2]))
    g = int(rng.choice([1, 2, 3]))
    ps = int(rng.choice([1, 2, 3]))
    causal = bool(seed % 2)
    b = W.random_small_batch(seed, batch=int(rng.integers(1, 4)), num_qo_heads=hk * g, num_kv_heads=hk,
                             page_size=ps, causal=causal, q_len_range=(0, 4), kv_len_range=(0, 9),
                             head_dim=d)
    scale = 1.0 / math.sqrt(d)
    o, lse = A.batch_attention(b)
    bo, bl = _brute_force(b, scale)
    assert len(bo) == b.total_q * b.num_qo_heads
    for (row, h), ref in bo.items():
        np.testing.assert_allclose(o[row, h], ref, rtol=0, atol=TOL)
        if math.isinf(bl[(row, h)]):
            assert np.isneginf(lse[row, h])
        else:
            assert abs(lse[row, h] - bl[(row, h)]) <= TOL


def test_golden_two_keys():
    gd = json.load(open(os.path.join(GOLDEN, "two_key_softmax.json")))
    q = np.array([gd["q"]])
    k = np.array(gd["k"])
    v = np.array(gd["v"])
    o, l = A.attention_state(q, k, v, [2], gd["scale"])
    np.testing.assert_allclose(o[0], gd["o_full"], atol=TOL)
    assert abs(l[0] - gd["lse_full"]) <= TOL
    o, l = A.attention_state(q, k, v, [1], gd["scale"])
    np.testing.assert_allclose(o[0], gd["o_first_key_only"], atol=TOL)
    assert abs(l[0] - gd["lse_first_key_only"]) <= TOL
    m = gd["merge"]
    o, l = A.merge_states(np.array([m["o_a"]]), np.array([m["lse_a"]]), np.array([m["o_b"]]), np.array([m["lse_b"]]))
    np.testing.assert_allclose(o[0], m["o"], atol=TOL)
    assert abs(l[0] - m["lse"]) <= TOL


def test_sdpa_and_logsumexp_special_case():
    """Dense contiguous inputs: torch float64 SDPA (O) and torch.logsumexp of explicit scores (LSE)."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(7)
    for causal in (False, True):
        lq, lk, d = 7, 11, 16
        q = rng.standard_normal((lq, d))
        k = rng.standard_normal((lk, d))
        v = rng.standard_normal((lk, d))
        scale = 1.0 / math.sqrt(d)
        vis = A.visible_counts(lq, lk, causal)
        o, lse = A.attention_state(q, k, v, vis, scale)
        mask = torch.ones(lq, lk, dtype=torch.bool)
        if causal:
            mask = torch.ones(lq, lk, dtype=torch.bool).tril(diagonal=lk - lq)
        tq, tk, tv = (torch.from_numpy(x)[None, None] for x in (q, k, v))
        ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask[None, None], scale=scale)
        np.testing.assert_allclose(o, ref[0, 0].numpy(), atol=TOL)
        s = (torch.from_numpy(q) @ torch.from_numpy(k).T) * scale
        s = s.masked_fill(~mask, -math.inf)
        np.testing.assert_allclose(lse, torch.logsumexp(s, dim=-1).numpy(), atol=TOL)


def test_scipy_logsumexp():
    sp = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(8)
    q = rng.standard_normal((3, 8))
    k = rng.standard_normal((20, 8))
    v = rng.standard_normal((20, 8))
    _, lse = A.attention_state(q, k, v, [20, 5, 1], 0.3)
    for r, n in enumerate([20, 5, 1]):
        assert abs(lse[r] - sp.logsumexp(0.3 * (q[r] @ k[:n].T))) <= TOL


def test_closed_forms():
    rng = np.random.default_rng(9)
    d, n = 16, 13
    scale = 1.0 / math.sqrt(d)
    q = rng.standard_normal((4, d))
    k = rng.standard_normal((n, d))
    # constant V => O = V
    vc = np.tile(rng.standard_normal(d), (n, 1))
    o, _ = A.attention_state(q, k, vc, n, scale)
    np.testing.assert_allclose(o, np.tile(vc[0], (4, 1)), atol=TOL)
    # identical keys => uniform weights, O = mean(V), LSE = log n + scale q.k
    v = rng.standard_normal((n, d))
    kk = np.tile(rng.standard_normal(d), (n, 1))
    o, l = A.attention_state(q, kk, v, n, scale)
    np.testing.assert_allclose(o, np.tile(v.mean(0), (4, 1)), atol=TOL)
    np.testing.assert_allclose(l, math.log(n) + scale * (q @ kk[0]), atol=TOL)
    # single key => O = v, LSE = scale q.k
    o, l = A.attention_state(q, k[:1], v[:1], 1, scale)
    np.testing.assert_allclose(o, np.tile(v[0], (4, 1)), atol=TOL)
    np.testing.assert_allclose(l, scale * (q @ k[0]), atol=TOL)
    # q = 0 => O = mean(V), LSE = log n
    o, l = A.attention_state(np.zeros((1, d)), k, v, n, scale)
    np.testing.assert_allclose(o[0], v.mean(0), atol=TOL)
    assert abs(l[0] - math.log(n)) <= TOL
    # no visible key => identity state
    o, l = A.attention_state(q, k, v, 0, scale)
    assert np.all(o == 0) and np.all(np.isneginf(l))


def _contiguous_state(b, i, h, layout="HND"):
    """Attention of request i / head h computed from a gather-free contiguous copy."""
    g = b.num_qo_heads // b.num_kv_heads
    lq, lk = A.request_lengths(b.qo_indptr, b.kv_indptr, b.last_page_len, b.page_size)
    pages = [int(x) for x in b.kv_indices[b.kv_indptr[i]:b.kv_indptr[i + 1]]]
    if layout == "HND":
        k = np.concatenate([b.k_pages[p, h // g] for p in pages], 0) if pages else np.zeros((0, b.head_dim), np.uint16)
        v = np.concatenate([b.v_pages[p, h // g] for p in pages], 0) if pages else np.zeros((0, b.head_dim), np.uint16)
    k = A.bf16_to_f64(k[:lk[i]])
    v = A.bf16_to_f64(v[:lk[i]])
    q = A.bf16_to_f64(b.q[b.qo_indptr[i]:b.qo_indptr[i + 1], h])
    return A.attention_state(q, k, v, A.visible_counts(int(lq[i]), int(lk[i]), b.causal), 1 / math.sqrt(b.head_dim))


def test_paged_equals_contiguous_and_layouts():
    b = W.random_small_batch(11, batch=5, num_qo_heads=4, num_kv_heads=2, page_size=3, causal=True,
                             q_len_range=(1, 5), kv_len_range=(0, 20), head_dim=8)
    o, l = A.batch_attention(b)
    for i in range(b.batch_size):
        for h in range(b.num_qo_heads):
            oc, lc = _contiguous_state(b, i, h)
            s = slice(b.qo_indptr[i], b.qo_indptr[i + 1])
            assert np.array_equal(o[s, h], oc)
            assert np.array_equal(l[s, h], lc)
    # NHD storage of the same pages gives bit-identical results
    bn = W.PagedBatch(b.name, b.num_qo_heads, b.num_kv_heads, b.head_dim, b.page_size, b.causal, b.qo_indptr,
                      b.kv_indptr, b.kv_indices, b.last_page_len, b.q, np.ascontiguousarray(b.k_pages.transpose(0, 2, 1, 3)),
                      np.ascontiguousarray(b.v_pages.transpose(0, 2, 1, 3)))
    o2, l2 = A.batch_attention(bn, layout="NHD")
    assert np.array_equal(o, o2) and np.array_equal(l, l2)


def test_physical_page_permutation_invariance():
    b = W.random_small_batch(12, batch=4, num_qo_heads=2, num_kv_heads=1, page_size=4, causal=False,
                             kv_len_range=(1, 30), extra_pages=5, head_dim=8)
    o, l = A.batch_attention(b)
    perm = np.random.default_rng(5).permutation(b.num_pages)
    k2 = np.empty_like(b.k_pages)
    v2 = np.empty_like(b.v_pages)
    k2[perm] = b.k_pages
    v2[perm] = b.v_pages
    b2 = W.PagedBatch(b.name, b.num_qo_heads, b.num_kv_heads, b.head_dim, b.page_size, b.causal, b.qo_indptr,
                      b.kv_indptr, perm[b.kv_indices].astype(np.int32), b.last_page_len, b.q, k2, v2)
    o2, l2 = A.batch_attention(b2)
    assert np.array_equal(o, o2) and np.array_equal(l, l2)


def test_merge_split_invariance():
    """State over [0, n) == merge of states over any split into pieces, in any order or tree."""
    rng = np.random.default_rng(13)
    d, n = 8, 40
    q = rng.standard_normal((3, d))
    k = rng.standard_normal((n, d))
    v = rng.standard_normal((n, d))
    full_o, full_l = A.attention_state(q, k, v, n, 0.4)
    for trial in range(20):
        cuts = sorted(rng.integers(0, n + 1, size=int(rng.integers(1, 6))).tolist())
        bounds = [0] + cuts + [n]
        pieces = [A.attention_state(q, k[a:b], v[a:b], b - a, 0.4) for a, b in zip(bounds[:-1], bounds[1:])]
        order = rng.permutation(len(pieces))
        states = [pieces[j] for j in order]
        while len(states) > 1:          # random merge tree
            j = int(rng.integers(0, len(states) - 1))
            m = A.merge_states(*states[j], *states[j + 1])
            states = states[:j] + [m] + states[j + 2:]
        np.testing.assert_allclose(states[0][0], full_o, atol=TOL)
        np.testing.assert_allclose(states[0][1], full_l, atol=TOL)


def test_merge_identity_and_commutativity():
    rng = np.random.default_rng(14)
    o = rng.standard_normal((5, 4))
    l = rng.standard_normal(5)
    empty_o, empty_l = np.zeros((5, 4)), np.full(5, -np.inf)
    mo, ml = A.merge_states(o, l, empty_o, empty_l)
    np.testing.assert_allclose(mo, o, atol=TOL)
    np.testing.assert_allclose(ml, l, atol=TOL)
    mo, ml = A.merge_states(empty_o, empty_l, empty_o, empty_l)
    assert np.all(mo == 0) and np.all(np.isneginf(ml))
    o2 = rng.standard_normal((5, 4))
    l2 = rng.standard_normal(5) * 30
    a = A.merge_states(o, l, o2, l2)
    b = A.merge_states(o2, l2, o, l)
    np.testing.assert_allclose(a[0], b[0], atol=TOL)
    np.testing.assert_allclose(a[1], b[1], atol=TOL)


def test_causal_rules():
    b = W.random_small_batch(15, batch=4, num_qo_heads=2, num_kv_heads=1, page_size=2, causal=True,
                             q_len_range=(1, 6), kv_len_range=(6, 14), head_dim=8)
    o, l = A.batch_attention(b)
    lq, lk = A.request_lengths(b.qo_indptr, b.kv_indptr, b.last_page_len, b.page_size)
    for i in range(b.batch_size):
        for h in range(2):
            for t in range(int(lq[i])):
                # row t of causal == non-causal attention over keys [0, l_kv - l_q + t]
                n_vis = int(lk[i] - lq[i] + t + 1)
                k = A.gather_kv(b.k_pages, b.kv_indptr, b.kv_indices, n_vis, b.page_size, i, 0)
                v = A.gather_kv(b.v_pages, b.kv_indptr, b.kv_indices, n_vis, b.page_size, i, 0)
                q = A.bf16_to_f64(b.q[b.qo_indptr[i] + t, h])[None]
                ro, rl = A.attention_state(q, k, v, n_vis, 1 / math.sqrt(8))
                np.testing.assert_allclose(o[b.qo_indptr[i] + t, h], ro[0], atol=TOL)
                assert abs(l[b.qo_indptr[i] + t, h] - rl[0]) <= TOL
    # one query token: causal == non-causal
    b1 = W.random_small_batch(16, batch=3, num_qo_heads=2, num_kv_heads=1, page_size=4, causal=True,
                              kv_len_range=(1, 20), head_dim=8)
    o1, l1 = A.batch_attention(b1)
    b1.causal = False
    o2, l2 = A.batch_attention(b1)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_gqa_equals_repeated_mha():
    b = W.random_small_batch(17, batch=3, num_qo_heads=6, num_kv_heads=2, page_size=2, causal=True,
                             q_len_range=(1, 3), kv_len_range=(1, 9), head_dim=8)
    o, l = A.batch_attention(b)
    rep = lambda x: np.repeat(x, 3, axis=1)
    bm = W.PagedBatch(b.name, 6, 6, 8, 2, True, b.qo_indptr, b.kv_indptr, b.kv_indices, b.last_page_len, b.q,
                      rep(b.k_pages), rep(b.v_pages))
    o2, l2 = A.batch_attention(bm)
    assert np.array_equal(o, o2) and np.array_equal(l, l2)


def test_composable_prefix_suffix_equals_flat():
    """Composable formats (核心机制 2, paper §3.1.2): prefix state merged with suffix state == flat attention."""
    sp = W.shared_prefix_decode(n_req=5, prefix_len=32, lo=3, hi=21)
    fo, fl = A.batch_attention(sp.flat)
    po, pl = A.batch_attention(sp.prefix)
    so, sl = A.batch_attention(sp.suffix)
    mo, ml = A.merge_states(po, pl, so, sl)
    np.testing.assert_allclose(mo, fo, atol=TOL)
    np.testing.assert_allclose(ml, fl, atol=TOL)


def test_workload_shapes():
    b = W.tiny_decode()
    lq, lk = A.request_lengths(b.qo_indptr, b.kv_indptr, b.last_page_len, b.page_size)
    assert lk.tolist() == [37, 128, 255, 512] and lq.tolist() == [1, 1, 1, 1]
    assert b.k_pages.shape == (128, 2, 16, 128) and len(set(b.kv_indices.tolist())) == 59


# ---- attention variants: sliding window and logit soft-cap (问题背景 挑战二; 核心机制 5, paper §3.2.3)

@pytest.mark.parametrize("seed", range(4))
def test_variants_brute_force_tiny(seed):
    rng = np.random.default_rng(700 + seed)
    b = W.random_small_batch(700 + seed, batch=3, num_qo_heads=4, num_kv_heads=2, page_size=3, causal=True,
                             q_len_range=(1, 6), kv_len_range=(1, 14), head_dim=4)
    w = int(rng.integers(0, 6))
    cap = float(rng.choice([0.0, 0.7, 3.0]))
    scale = 1.0 / math.sqrt(b.head_dim)
    o, l = A.batch_attention(b, window_left=w, soft_cap=cap)
    bo, bl = _brute_force(b, scale, window_left=w, soft_cap=cap)
    for (row, h), val in bo.items():
        np.testing.assert_allclose(o[row, h], val, atol=TOL)
        if math.isinf(bl[(row, h)]):
            assert np.isneginf(l[row, h])
        else:
            assert abs(l[row, h] - bl[(row, h)]) <= TOL


def test_sliding_window_special_cases():
    b = W.random_small_batch(720, batch=5, num_qo_heads=4, num_kv_heads=2, page_size=4, causal=True,
                             q_len_range=(1, 7), kv_len_range=(1, 40), head_dim=8)
    o, l = A.batch_attention(b)
    # a window at least as long as every KV changes nothing
    o2, l2 = A.batch_attention(b, window_left=64)
    assert np.array_equal(o, o2) and np.array_equal(l, l2)
    # window 0: each token sees only the key at its own position: O = v_p, LSE = scale q.k_p
    o0, l0 = A.batch_attention(b, window_left=0)
    scale = 1.0 / math.sqrt(b.head_dim)
    lq, lk = A.request_lengths(b.qo_indptr, b.kv_indptr, b.last_page_len, b.page_size)
    g = b.num_qo_heads // b.num_kv_heads
    for i in range(b.batch_size):
        for h in range(b.num_qo_heads):
            k = A.gather_kv(b.k_pages, b.kv_indptr, b.kv_indices, int(lk[i]), b.page_size, i, h // g)
            v = A.gather_kv(b.v_pages, b.kv_indptr, b.kv_indices, int(lk[i]), b.page_size, i, h // g)
            for t in range(int(lq[i])):
                row, pos = int(b.qo_indptr[i]) + t, int(lk[i] - lq[i] + t)
                if pos < 0:
                    assert np.isneginf(l0[row, h]) and np.all(o0[row, h] == 0)
                    continue
                q = A.bf16_to_f64(b.q[row, h])
                np.testing.assert_allclose(o0[row, h], v[pos], atol=TOL)
                assert abs(l0[row, h] - scale * float(q @ k[pos])) <= TOL


def test_sliding_window_is_attention_over_the_window():
    """Windowed state == plain state over the contiguous slice of keys p - w .. p."""
    b = W.random_small_batch(721, batch=4, num_qo_heads=2, num_kv_heads=1, page_size=5, causal=True,
                             q_len_range=(1, 9), kv_len_range=(5, 60), head_dim=8)
    w = 7
    o, l = A.batch_attention(b, window_left=w)
    scale = 1.0 / math.sqrt(b.head_dim)
    lq, lk = A.request_lengths(b.qo_indptr, b.kv_indptr, b.last_page_len, b.page_size)
    for i in range(b.batch_size):
        for h in range(b.num_qo_heads):
            k = A.gather_kv(b.k_pages, b.kv_indptr, b.kv_indices, int(lk[i]), b.page_size, i, 0)
            v = A.gather_kv(b.v_pages, b.kv_indptr, b.kv_indices, int(lk[i]), b.page_size, i, 0)
            for t in range(int(lq[i])):
                row, pos = int(b.qo_indptr[i]) + t, int(lk[i] - lq[i] + t)
                lo = max(0, pos - w)
                ks, vs = k[lo:pos + 1], v[lo:pos + 1]
                oo, ll = A.attention_state(A.bf16_to_f64(b.q[row:row + 1, h]), ks, vs, ks.shape[0], scale)
                np.testing.assert_allclose(o[row, h], oo[0], atol=TOL)
                assert abs(l[row, h] - ll[0]) <= TOL or (np.isneginf(l[row, h]) and np.isneginf(ll[0]))


def test_soft_cap_closed_forms_and_bounds():
    rng = np.random.default_rng(722)
    d, n = 16, 11
    scale = 1.0 / math.sqrt(d)
    q = 3.0 * rng.standard_normal((5, d))
    k = 3.0 * rng.standard_normal((n, d))
    v = rng.standard_normal((n, d))
    # an enormous cap is the plain softmax
    o, l = A.attention_state(q, k, v, n, scale)
    o1, l1 = A.attention_state(q, k, v, n, scale, soft_cap=1e9)
    np.testing.assert_allclose(o1, o, atol=1e-9)
    np.testing.assert_allclose(l1, l, atol=1e-9)
    for cap in (0.5, 2.0, 30.0):
        # identical keys: weights stay uniform; LSE = log n + cap tanh(scale q.k / cap)
        kk = np.tile(k[0], (n, 1))
        oc, lc = A.attention_state(q, kk, v, n, scale, soft_cap=cap)
        np.testing.assert_allclose(oc, np.tile(v.mean(0), (5, 1)), atol=TOL)
        np.testing.assert_allclose(lc, math.log(n) + cap * np.tanh(scale * (q @ k[0]) / cap), atol=TOL)
        # single key: O = v, LSE = cap tanh(scale q.k / cap)
        o1k, l1k = A.attention_state(q, k[:1], v[:1], 1, scale, soft_cap=cap)
        np.testing.assert_allclose(o1k, np.tile(v[0], (5, 1)), atol=TOL)
        np.testing.assert_allclose(l1k, cap * np.tanh(scale * (q @ k[0]) / cap), atol=TOL)
        # every capped logit lies in (-cap, cap): log n - cap < LSE < log n + cap
        _, lb = A.attention_state(q, k, v, n, scale, soft_cap=cap)
        assert np.all(lb < math.log(n) + cap) and np.all(lb > math.log(n) - cap)


def test_window_needs_causal():
    b = W.random_small_batch(723, batch=2, num_qo_heads=2, num_kv_heads=1, page_size=4, causal=False,
                             kv_len_range=(1, 10), head_dim=8)
    with pytest.raises(ValueError):
        A.batch_attention(b, window_left=3)


# ---- FP8 (e4m3) KV (核心机制 8 / paper App. F; the format's own definition) -----------------------

def test_e4m3_decoder_pins():
    """Values fixed by the format: 1.0, the extremes, subnormal spacing, sign symmetry, NaN, ordering."""
    d = A.e4m3_to_f64(np.arange(256, dtype=np.uint8))
    assert d[0x38] == 1.0 and d[0x40] == 2.0 and d[0x30] == 0.5
    assert d[0x7E] == 448.0                       # largest finite value
    assert d[0x08] == 2.0 ** -6                   # smallest normal
    assert d[0x01] == 2.0 ** -9                   # smallest subnormal
    assert d[0x00] == 0.0 and d[0x80] == 0.0
    assert np.isnan(d[0x7F]) and np.isnan(d[0xFF]) and np.isnan(d).sum() == 2
    np.testing.assert_array_equal(d[0x80:0xFF], -d[0x00:0x7F])
    pos = d[0x00:0x7F]
    assert np.all(np.diff(pos) > 0)               # codes ascend with value
    # every normal binade holds 8 evenly spaced values; the next binade doubles them
    for c in range(0x08, 0x77):
        assert d[c + 8] == 2.0 * d[c]
    # subnormals are the multiples of 2^-9 below the smallest normal
    np.testing.assert_array_equal(d[0x00:0x08], np.arange(8) * 2.0 ** -9)


def test_fp8_attention_equals_dequantized_bf16_free_attention():
    """Attention over e4m3 pages with scales == attention over the same values given as float64 pages."""
    rng = np.random.default_rng(730)
    b = W.random_small_batch(730, batch=3, num_qo_heads=4, num_kv_heads=2, page_size=4, causal=False,
                             kv_len_range=(1, 20), head_dim=8)
    codes_k = rng.integers(0, 0x7E, size=b.k_pages.shape, dtype=np.uint8) | (rng.integers(0, 2, size=b.k_pages.shape, dtype=np.uint8) << 7)
    codes_v = rng.integers(0, 0x7E, size=b.v_pages.shape, dtype=np.uint8)
    b8 = W.PagedBatch(b.name, b.num_qo_heads, b.num_kv_heads, b.head_dim, b.page_size, b.causal, b.qo_indptr,
                      b.kv_indptr, b.kv_indices, b.last_page_len, b.q, codes_k, codes_v)
    o, l = A.batch_attention(b8, k_scale=0.25, v_scale=3.0)
    bf = W.PagedBatch(b.name, b.num_qo_heads, b.num_kv_heads, b.head_dim, b.page_size, b.causal, b.qo_indptr,
                      b.kv_indptr, b.kv_indices, b.last_page_len, b.q, 0.25 * A.e4m3_to_f64(codes_k),
                      3.0 * A.e4m3_to_f64(codes_v))
    o2, l2 = A.batch_attention(bf)
    np.testing.assert_allclose(o, o2, atol=TOL)
    np.testing.assert_allclose(l, l2, atol=TOL)


def test_fp8_pages_layout_invariant():
    """e4m3 pages stored HND [pages, H_kv, page_size, D] or NHD [pages, page_size, H_kv, D] hold the
    same codes at the same (page, head, row): attention over them is identical, bit for bit."""
    b = W.random_small_batch(731, batch=4, num_qo_heads=6, num_kv_heads=3, page_size=4, causal=True,
                             q_len_range=(1, 3), kv_len_range=(1, 23), head_dim=8)
    b8 = W.as_e4m3(b, 0.5, 2.0)
    nhd = W.PagedBatch(b8.name, b8.num_qo_heads, b8.num_kv_heads, b8.head_dim, b8.page_size, b8.causal,
                       b8.qo_indptr, b8.kv_indptr, b8.kv_indices, b8.last_page_len, b8.q,
                       np.ascontiguousarray(b8.k_pages.transpose(0, 2, 1, 3)),
                       np.ascontiguousarray(b8.v_pages.transpose(0, 2, 1, 3)))
    o1, l1 = A.batch_attention(b8, k_scale=0.5, v_scale=2.0)
    o2, l2 = A.batch_attention(nhd, layout="NHD", k_scale=0.5, v_scale=2.0)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


# ---- bfloat16 decoding and rounding (术语与记号 fixes bf16 inputs with fp32 accumulation) ----------

def test_bf16_decoder_pins_all_bit_patterns():
    """bf16_to_f64 against torch's own bfloat16 -> float64 cast on all 65536 bit patterns (NaNs by
    class, everything else bit for bit), plus values the format fixes by definition: bf16 keeps the
    sign, the 8 exponent bits (bias 127) and the top 7 mantissa bits of an IEEE float32."""
    torch = pytest.importorskip("torch")
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore"):  # signalling NaN patterns widen to quiet NaNs
        ours = A.bf16_to_f64(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert nan.sum() == 2 * 127  # exponent all ones, mantissa non-zero, either sign
    assert np.array_equal(ours[~nan].view(np.uint64), ref[~nan].view(np.uint64))  # bit for bit, -0 included
    # values fixed by the format, independent of any library
    assert ours[0x3F80] == 1.0 and ours[0xBF80] == -1.0 and ours[0x4000] == 2.0 and ours[0x3F00] == 0.5
    assert ours[0x3FC0] == 1.5 and ours[0x3F81] == 1.0 + 2.0 ** -7           # last mantissa bit = 2^-7
    assert ours[0x0080] == 2.0 ** -126 and ours[0x0001] == 2.0 ** -133      # smallest normal, subnormal
    assert ours[0x7F7F] == (2.0 - 2.0 ** -7) * 2.0 ** 127                   # largest finite
    assert ours[0x7F80] == np.inf and ours[0xFF80] == -np.inf
    assert ours[0x0000] == 0.0 and np.signbit(ours[0x8000]) and ours[0x8000] == 0.0
    # a byte-order or shift mistake would swap these two
    assert ours[0x4049] == 3.140625 and ours[0x4940] != 3.140625


def test_bf16_rounding_of_the_input_generator():
    """The generator's float32 -> bf16 rounding (nearest, ties to even) equals torch's cast on a large
    random sample, on exact ties, on subnormals and at the overflow edge."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(77)
    x = np.concatenate([
        rng.standard_normal(200_000, dtype=np.float32),
        (rng.standard_normal(50_000, dtype=np.float32) * np.float32(1e-39)),    # float32 subnormals
        rng.uniform(-3e38, 3e38, 50_000).astype(np.float32),                      # rounds to inf near the top
    ])
    hi = rng.integers(0, 1 << 16, 20_000, dtype=np.uint32)
    hi = hi[((hi >> 7) & 0xFF) != 0xFF]                                           # finite upper halves only
    ties = ((hi << 16) | np.uint32(0x8000)).view(np.float32)                      # exactly half way
    near = ((hi << 16) | np.uint32(0x7FFF)).view(np.float32)                      # just below half way
    x = np.concatenate([x, ties, near, np.float32([0.0, -0.0, 1.0, 3.4028235e38, -3.4028235e38])])
    ours = W.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    # ties go to the even upper half: 1 + 2^-8 (half an ulp above 1) rounds down to 1, 1 + 3*2^-8 up
    assert W.f32_to_bf16_bits(np.float32([1.0 + 2.0 ** -8]))[0] == 0x3F80
    assert W.f32_to_bf16_bits(np.float32([1.0 + 3 * 2.0 ** -8]))[0] == 0x3F82
