"""Plain-Python restatement of the load-balancing plan -- test infrastructure only.

Follows page "FlashInfer：面向 LLM 推理服务的高效可定制注意力引擎",
核心机制 6 "负载均衡调度" (paper §3.3.1, Algorithm 1, Figure 6) and
核心机制 7 (paper Appendix D.1-D.3), in that order:

  * tile cost cost(l_q, l_kv) = alpha * l_q + beta * l_kv;
  * the largest KV chunk L_kv = sum_i ceil(l_qo,i / T_q) * l_kv,i / #CTA;
  * work sorted longest-first, then handed out through a priority queue of CTAs;
  * no atomic aggregation: partial outputs of a split request go to fixed
    workspace slots and a reduction map fixes the order they are merged in;
  * only "long" work is split; everything else writes the final output directly;
  * partial outputs are bounded by 2 * #CTA tiles.

Readings (the algorithm listing itself is not on the page; these are listed in
the design notes):
  * Path / tile (核心机制 4, paper §3.2.2): rows of a tile are (query token, query
    head in group) pairs.  If every request has l_q * g <= 8 rows, the whole
    batch takes the decode path with one tile per (request, KV head)
    covering all its query tokens, and rows_tile is the smallest of 1, 2, 4, 8
    that fits; otherwise the tensor-core path with 256-row tiles,
    tile_tokens = 256 // g.
  * #CTA = k * (SM budget), k fixed per path: 1 for both paths (核心机制 7,
    paper App. D.3: #CTA = k x #SM).
  * KV heads count as separate units in the L_kv sum; L_kv is raised to l_min
    (default 256) and rounded up to a whole number of pages.
  * A unit (request, KV head, query tile) sees e keys: l_kv, or under the causal
    mask the keys visible to the tile's last token.  It is cut into
    n = ceil(e / L_kv) chunks, evened out: chunk size cs = ceil(ceil(e / n) / page)
    pages, and the chunks are [c*cs, min(e, (c+1)*cs)).  A unit with e = 0 is one
    empty chunk (it writes the empty state).
  * cost of an item = alpha * rows + beta * chunk length, rows = tokens in tile * g;
    defaults alpha = beta = 1.
  * Sort: cost descending, ties by enumeration order (request, KV head, tile,
    chunk ascending).  Priority queue: smallest accumulated cost first, ties to
    the lowest CTA id.
  * Slots are numbered in enumeration order of the split units, chunk by chunk.

The serialised form (`serialize`) is what the library's host-only plan entry
point must reproduce bit for bit.
"""
from __future__ import annotations

import heapq
from dataclasses import dataclass

import numpy as np

PATH_DECODE = 0
PATH_TENSOR = 1
TC_ROWS = 256
DECODE_MAX_ROWS = 8
DECODE_CTAS_PER_SM = 1
TC_CTAS_PER_SM = 1
NOT_CAUSAL_DIAG = 1 << 30
PLAN_MAGIC = 0x46495031
HEADER_LEN = 16
ITEM_FIELDS = 8
UNIT_FIELDS = 8


def _ceil_div(a: int, b: int) -> int:
    return -(-a // b)


@dataclass
class Plan:
    path: int
    tile_tokens: int
    rows_tile: int
    group: int
    num_ctas: int
    l_kv_chunk: int
    page_size: int
    causal: bool
    num_qo_heads: int
    num_kv_heads: int
    head_dim: int
    batch: int
    items: list            # enumeration order; each a dict
    order: list            # item indices in assignment (sorted) order
    cta_of: list           # CTA of each item (by enumeration index)
    queues: list           # per CTA: item indices in queue order
    units: list            # split units: dict(first_slot, n_chunks, q_start, q_len, kv_head)
    slot_unit: list
    loads: list            # accumulated cost per CTA


def choose_path(l_q, group: int, force_tensor: bool = False):
    """Tile choice (核心机制 4, paper §3.2.2): decode tiles for <= 8 rows, 256-row tensor-core tiles otherwise
    (or always, for the shared part of a composable plan)."""
    max_rows = int(max((int(x) for x in l_q), default=0)) * group
    if max_rows <= DECODE_MAX_ROWS and not force_tensor:
        tile_tokens = max(1, int(max((int(x) for x in l_q), default=1)))
        rows = 1
        while rows < tile_tokens * group:
            rows *= 2
        return PATH_DECODE, tile_tokens, rows
    if group > TC_ROWS:
        raise ValueError("group size above 256 rows")
    return PATH_TENSOR, TC_ROWS // group, TC_ROWS


def plan(qo_indptr, kv_indptr, last_page_len, num_qo_heads: int, num_kv_heads: int, page_size: int,
         causal: bool, num_sms: int, head_dim: int = 128, alpha: int = 1, beta: int = 1,
         l_min: int = 256, window_left: int = -1, force_tensor: bool = False, all_slots: bool = False) -> Plan:
    """window_left >= 0: sliding window (causal plans only); each tile reads only the keys its
    tokens' windows reach, from the first token's window start rounded down to a page.
    force_tensor: tensor-core tiles whatever the rows; all_slots: every unit, split or not, writes its
    chunks' partial states to slots (both used by the shared part of a composable plan)."""
    if window_left >= 0 and not causal:
        raise ValueError("the sliding window is read with causal masks")
    qo = [int(x) for x in qo_indptr]
    kv = [int(x) for x in kv_indptr]
    last = [int(x) for x in last_page_len]
    batch = len(qo) - 1
    g = num_qo_heads // num_kv_heads

    # a1: lengths
    l_q = [qo[i + 1] - qo[i] for i in range(batch)]
    l_kv = []
    for i in range(batch):
        n_p = kv[i + 1] - kv[i]
        l_kv.append((n_p - 1) * page_size + last[i] if n_p > 0 else 0)

    # a2: path and tile
    path, tile_tokens, rows_tile = choose_path(l_q, g, force_tensor)
    num_ctas = (TC_CTAS_PER_SM if path == PATH_TENSOR else DECODE_CTAS_PER_SM) * num_sms

    def extent(i, q0, qn):
        """Keys [lo, e) that tile rows q0 .. q0+qn-1 of request i can see."""
        if not causal:
            return 0, l_kv[i]
        e = min(max(l_kv[i] - l_q[i] + q0 + qn, 0), l_kv[i])
        lo = 0
        if window_left >= 0:
            lo = max(0, l_kv[i] - l_q[i] + q0 - window_left) // page_size * page_size
            lo = min(lo, e)
        return lo, e

    # a3: KV chunk bound (with a window: the keys each tile reads, which is all a window touches)
    total = 0
    for i in range(batch):
        if window_left < 0:
            total += num_kv_heads * _ceil_div(l_q[i], tile_tokens) * l_kv[i]
        else:
            for j in range(_ceil_div(l_q[i], tile_tokens)):
                q0 = j * tile_tokens
                lo, e = extent(i, q0, min(tile_tokens, l_q[i] - q0))
                total += num_kv_heads * (e - lo)
    l_chunk = max(_ceil_div(total, num_ctas), l_min)
    l_chunk = _ceil_div(l_chunk, page_size) * page_size

    # a4: units -> chunks (items); a6: slots of split units
    items, units, slot_unit = [], [], []
    for i in range(batch):
        n_tiles = _ceil_div(l_q[i], tile_tokens)
        for h in range(num_kv_heads):
            for j in range(n_tiles):
                q0 = j * tile_tokens
                qn = min(tile_tokens, l_q[i] - q0)
                lo_e, e = extent(i, q0, qn)
                diag = l_kv[i] - l_q[i] + q0 if causal else NOT_CAUSAL_DIAG
                if e - lo_e == 0:
                    n, cs = 1, 0
                else:
                    n = _ceil_div(e - lo_e, l_chunk)
                    cs = _ceil_div(_ceil_div(e - lo_e, n), page_size) * page_size
                    n = _ceil_div(e - lo_e, cs)
                unit = -1
                if n > 1 or all_slots:
                    unit = len(units)
                    units.append(dict(first_slot=len(slot_unit), n_chunks=n, q_start=qo[i] + q0, q_len=qn,
                                      kv_head=h, ext_first=0, ext_count=0))
                    slot_unit.extend([unit] * n)
                for c in range(n):
                    lo, hi = lo_e + c * cs, min(e, lo_e + (c + 1) * cs)
                    items.append(dict(
                        request=i, kv_head=h, tile=j, chunk=c,
                        page_base=kv[i], q_start=qo[i] + q0, q_len=qn, kv_lo=lo, kv_hi=hi, diag=diag,
                        slot=(units[unit]["first_slot"] + c) if unit >= 0 else -1,
                        cost=alpha * qn * g + beta * (hi - lo),
                    ))

    # a5: longest first, then a min-priority queue of CTAs keyed (load, cta id)
    order = sorted(range(len(items)), key=lambda k: (-items[k]["cost"], k))
    heap = [(0, c) for c in range(num_ctas)]
    heapq.heapify(heap)
    cta_of = [0] * len(items)
    queues = [[] for _ in range(num_ctas)]
    for k in order:
        load, c = heapq.heappop(heap)
        cta_of[k] = c
        queues[c].append(k)
        heapq.heappush(heap, (load + items[k]["cost"], c))
    loads = [0] * num_ctas
    for load, c in heap:
        loads[c] = load

    return Plan(path, tile_tokens, rows_tile, g, num_ctas, l_chunk, page_size, bool(causal), num_qo_heads,
                num_kv_heads, head_dim, batch, items, order, cta_of, queues, units, slot_unit, loads)


def serialize(p: Plan) -> np.ndarray:
    """Flat int32 form: header[16] | cta_indptr | items (queue order) | units | slot_unit."""
    header = [PLAN_MAGIC, p.path, p.tile_tokens, p.rows_tile, p.group, p.num_ctas, len(p.items), len(p.units),
              len(p.slot_unit), p.l_kv_chunk, p.page_size, int(p.causal), p.num_qo_heads, p.num_kv_heads,
              p.head_dim, p.batch]
    indptr = [0]
    for q in p.queues:
        indptr.append(indptr[-1] + len(q))
    flat_items = []
    for q in p.queues:
        for k in q:
            it = p.items[k]
            flat_items += [it["page_base"], it["q_start"], it["q_len"], it["kv_head"], it["kv_lo"], it["kv_hi"],
                           it["diag"], it["slot"]]
    flat_units = []
    for u in p.units:
        flat_units += [u["first_slot"], u["n_chunks"], u["q_start"], u["q_len"], u["kv_head"], u.get("ext_first", 0),
                       u.get("ext_count", 0), 0]
    return np.array(header + indptr + flat_items + flat_units + list(p.slot_unit), dtype=np.int64).astype(np.int32)


def deserialize(buf) -> dict:
    """Split a flat plan back into named int32 arrays (used to compare plans field by field)."""
    buf = np.asarray(buf, dtype=np.int32)
    h = buf[:HEADER_LEN]
    n_cta, n_items, n_units, n_slots = int(h[5]), int(h[6]), int(h[7]), int(h[8])
    o = HEADER_LEN
    indptr = buf[o:o + n_cta + 1]
    o += n_cta + 1
    items = buf[o:o + n_items * ITEM_FIELDS].reshape(n_items, ITEM_FIELDS)
    o += n_items * ITEM_FIELDS
    units = buf[o:o + n_units * UNIT_FIELDS].reshape(n_units, UNIT_FIELDS)
    o += n_units * UNIT_FIELDS
    slot_unit = buf[o:o + n_slots]
    o += n_slots
    return dict(header=h, cta_indptr=indptr, items=items, units=units, slot_unit=slot_unit, length=o)


# ---------------------------------------------------------------------------
# Composable formats (核心机制 2, paper §3.1.2, Figure 3)
# ---------------------------------------------------------------------------
EXT_ROW_BIAS = 512
TC_KEY_COST = (4, 3)   # a 256-row tensor-core key costs about 4/3 of a decode key of SM time


def plan_composable(shared, unique, num_qo_heads: int, num_kv_heads: int, page_size: int, causal: bool,
                    num_sms: int, head_dim: int = 128):
    """One plan over two BSR sub-matrices of the same query rows, with one reduction map.

    `shared` and `unique` are (qo_indptr, kv_indptr, last_page_len).  The shared part (block rows such
    as a prefix shared by a group of requests) sees all of its keys, takes tensor-core tiles and writes
    every chunk to a slot.  The per-request part takes decode tiles; its slots are numbered after the
    shared ones.  Each of its units lists, in order, the shared slots holding states of its rows: one
    entry (slot, packed) per chunk of every shared tile that holds some of its tokens, packed =
    (row offset + 512) | (rows of the shared tile << 16).  Split units get the list first, in unit
    order; then every single-chunk item (queue order) whose rows have shared states gets a unit of its
    own (first slot -1, one chunk) and the slot field -(2 + unit).
    """
    # SM budget split (both parts run at once on disjoint SMs): the shared part gets
    # round(num_sms * c_a / (c_a + c_b)) CTAs, at least 1 and leaving at least 1, where c_a = 4 x its
    # keys and c_b = 3 x the per-request keys (a key of a 256-row tensor-core tile costs about 4/3 of a
    # decode key of SM time)
    def keys(qo, kv, last):
        qo, kv, last = [int(x) for x in qo], [int(x) for x in kv], [int(x) for x in last]
        tot = 0
        for i in range(len(qo) - 1):
            n_p = kv[i + 1] - kv[i]
            if qo[i + 1] > qo[i] and n_p > 0:
                tot += num_kv_heads * ((n_p - 1) * page_size + last[i])
        return tot
    n_a = num_sms
    if num_sms > 1:
        c_a, c_b = TC_KEY_COST[0] * keys(*shared), TC_KEY_COST[1] * keys(*unique)
        n_a = (2 * num_sms * c_a + (c_a + c_b)) // (2 * (c_a + c_b)) if c_a + c_b > 0 else 1
        n_a = min(max(n_a, 1), num_sms - 1)
    a = plan(*shared, num_qo_heads, num_kv_heads, page_size, False, n_a, head_dim, force_tensor=True,
             all_slots=True)
    # one adjustment toward one chunk per CTA: fewer chunks than CTAs -> one CTA per chunk; more but at
    # most twice as many -> as many CTAs as chunks (leaving one SM); then the shared part is planned again
    items = len(a.items)
    if items < n_a:
        n_adj = max(items, 1)
    elif num_sms > 1 and n_a < items <= 2 * n_a:
        n_adj = min(items, num_sms - 1)
    else:
        n_adj = n_a
    if n_adj != n_a:
        n_a = n_adj
        a = plan(*shared, num_qo_heads, num_kv_heads, page_size, False, n_a, head_dim, force_tensor=True,
                 all_slots=True)
    n_b = num_sms - n_a if num_sms > 1 else 1
    b = plan(*unique, num_qo_heads, num_kv_heads, page_size, causal, n_b, head_dim)
    if b.path != PATH_DECODE:
        raise ValueError("the per-request part must take decode tiles")
    g = num_qo_heads // num_kv_heads
    s_a = len(a.slot_unit)
    for it in b.items:
        if it["slot"] >= 0:
            it["slot"] += s_a
    for u in b.units:
        u["first_slot"] += s_a
    b.slot_unit = [-1] * s_a + list(b.slot_unit)
    a_qo = [int(x) for x in shared[0]]
    base = [0]
    for i in range(len(a_qo) - 1):
        base.append(base[-1] + num_kv_heads * _ceil_div(a_qo[i + 1] - a_qo[i], a.tile_tokens))
    ext = []

    def add_ext(q0, qn, h):
        count = 0
        for i in range(len(a_qo) - 1):
            lo, hi = max(q0, a_qo[i]), min(q0 + qn, a_qo[i + 1])
            if lo >= hi:
                continue
            n_tiles = _ceil_div(a_qo[i + 1] - a_qo[i], a.tile_tokens)
            for j in range((lo - a_qo[i]) // a.tile_tokens, (hi - 1 - a_qo[i]) // a.tile_tokens + 1):
                u = a.units[base[i] + h * n_tiles + j]
                packed = ((q0 - u["q_start"]) * g + EXT_ROW_BIAS) | ((u["q_len"] * g) << 16)
                for c in range(u["n_chunks"]):
                    ext.append((u["first_slot"] + c, packed))
                    count += 1
        return count

    for u in b.units:
        u["ext_first"] = len(ext)
        u["ext_count"] = add_ext(u["q_start"], u["q_len"], u["kv_head"])
    for q in b.queues:
        for k in q:
            it = b.items[k]
            if it["slot"] != -1:
                continue
            first = len(ext)
            cnt = add_ext(it["q_start"], it["q_len"], it["kv_head"])
            if cnt == 0:
                continue
            b.units.append(dict(first_slot=-1, n_chunks=1, q_start=it["q_start"], q_len=it["q_len"],
                                kv_head=it["kv_head"], ext_first=first, ext_count=cnt))
            it["slot"] = -(2 + len(b.units) - 1)
    return a, b, ext


def serialize_composable(a: Plan, b: Plan, ext) -> np.ndarray:
    """shared plan | per-request plan (its header's slot count = all slots) | ext pairs."""
    sa = serialize(a)
    sb = serialize(b)
    sb[8] = len(b.slot_unit)
    flat_ext = [v for pair in ext for v in pair]
    return np.concatenate([sa, sb, np.array(flat_ext, dtype=np.int64).astype(np.int32)])
