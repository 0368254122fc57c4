// Host planner: lengths -> tile -> KV chunk bound -> chunks -> longest-first
// assignment through a CTA priority queue -> reduction map.
//
// Page "FlashInfer：面向 LLM 推理服务的高效可定制注意力引擎":
//   核心机制 6 "负载均衡调度" (paper §3.3.1, Alg. 1, Fig. 6): tile cost
//     alpha * l_q + beta * l_kv; largest KV chunk L_kv = sum ceil(l_qo/T_q) * l_kv / #CTA;
//     work sorted longest-first and assigned through a CTA priority queue;
//     no atomic aggregation, so the merge order of partial outputs is fixed.
//   核心机制 7 (paper App. D.2): only work longer than the chunk bound is split;
//     the rest writes the final output directly.  App. D.3: partial outputs
//     stay below 2 * #CTA tiles.
//   核心机制 4 (paper §3.2.2): tiles of at most 8 rows take the decode kernel
//     (the page runs them on CUDA cores, since an MMA needs at least 16 query
//     rows), larger ones 256-row tensor-core tiles (two 128-row MMA tiles per KV tile).
//
// Rules fixed where the page is silent (the same ones the test-side
// restatement uses, so the two must agree bit for bit):
//   * rows of a tile are (query token, query head of the group) pairs; if every
//     request has l_q * g <= 8 the decode path takes one tile per (request, KV
//     head) with rows_tile the smallest of 1, 2, 4, 8 that fits; otherwise
//     128-row tensor-core tiles of 128 / g tokens;
//   * KV heads are separate units of the L_kv sum; L_kv >= l_min and is a whole
//     number of pages;
//   * a unit sees e keys (under the causal mask: those of its last token) and is
//     cut into n = ceil(e / L_kv) chunks of cs = pages(ceil(e / n)) tokens;
//   * #CTA = k * (SM budget) with k fixed per path (kDecodeCtasPerSm = kTcCtasPerSm = 1: one
//     persistent CTA per SM on either path);
//   * item cost = alpha * rows + beta * chunk length;
//   * sort by cost descending, ties by enumeration order; the queue pops the
//     least-loaded CTA, ties to the lowest CTA id.
#include "plan.h"

#include <algorithm>
#include <climits>
#include <cstring>
#include <functional>
#include <utility>

#include "../../include/fi.h"

namespace fi {

namespace {

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// a1: query and KV length of request i
inline int64_t len_q(const PlanInput& in, int i) { return int64_t(in.qo_indptr[i + 1]) - in.qo_indptr[i]; }
inline int64_t len_kv(const PlanInput& in, int i) {
  const int64_t n_pages = int64_t(in.kv_indptr[i + 1]) - in.kv_indptr[i];
  return n_pages > 0 ? (n_pages - 1) * in.page_size + in.last_page_len[i] : 0;
}

// keys [lo, e) that tile rows q0 .. q0+qn-1 of request i can see
void extent(const PlanInput& in, int i, int64_t q0, int64_t qn, int64_t* lo, int64_t* e) {
  const int64_t lq = len_q(in, i), lkv = len_kv(in, i);
  *lo = 0;
  if (!in.causal) {
    *e = lkv;
    return;
  }
  *e = std::min(std::max<int64_t>(lkv - lq + q0 + qn, 0), lkv);
  if (in.window_left >= 0) {
    *lo = std::max<int64_t>(0, lkv - lq + q0 - in.window_left) / in.page_size * in.page_size;
    *lo = std::min(*lo, *e);
  }
}

// a4: every unit (request, KV head, query tile) in enumeration order, cut into n chunks of cs keys
// from lo_e (n = 1, cs = 0 when it sees no key); visit(i, h, q0, qn, lo_e, e, cs, n, diag).
template <class Visit>
void for_each_unit(const PlanInput& in, const PlanShape& s, Visit&& visit) {
  const int ps = in.page_size;
  for (int i = 0; i < in.batch; ++i) {
    const int64_t lq = len_q(in, i), lkv = len_kv(in, i);
    const int64_t n_tiles = ceil_div(lq, s.tile_tokens);
    for (int h = 0; h < in.num_kv_heads; ++h) {
      for (int64_t j = 0; j < n_tiles; ++j) {
        const int64_t q0 = j * s.tile_tokens;
        const int64_t qn = std::min<int64_t>(s.tile_tokens, lq - q0);
        int64_t lo_e, e;
        extent(in, i, q0, qn, &lo_e, &e);
        const int64_t diag = in.causal ? lkv - lq + q0 : kNotCausalDiag;
        int64_t n = 1, cs = 0;
        const int64_t ext = e - lo_e;
        if (ext > 0 && ext <= s.l_chunk) {
          // one chunk (the common case; the general rule below gives the same n and cs)
          cs = (ps & (ps - 1)) == 0 ? (ext + ps - 1) & ~int64_t(ps - 1) : ceil_div(ext, ps) * ps;
        } else if (ext > 0) {
          n = ceil_div(ext, s.l_chunk);
          cs = ceil_div(ceil_div(ext, n), ps) * ps;
          n = ceil_div(ext, cs);
        }
        visit(i, h, q0, qn, lo_e, e, cs, n, diag);
      }
    }
  }
}

}  // namespace

int validate_input(const PlanInput& in) {
  if (in.batch < 0 || in.qo_indptr == nullptr || in.kv_indptr == nullptr) return FI_ERR_INVALID_ARG;
  if (in.batch > 0 && in.last_page_len == nullptr) return FI_ERR_INVALID_ARG;
  if (in.num_qo_heads <= 0 || in.num_kv_heads <= 0 || in.page_size <= 0 || in.num_sms <= 0)
    return FI_ERR_INVALID_ARG;
  if (in.causal != 0 && in.causal != 1) return FI_ERR_INVALID_ARG;
  if (in.window_left >= 0 && !in.causal) return FI_ERR_UNSUPPORTED;  // the window is read with causal masks
  if (in.head_dim != kHeadDim) return FI_ERR_UNSUPPORTED;
  if (in.num_qo_heads % in.num_kv_heads != 0) return FI_ERR_UNSUPPORTED;
  if (in.qo_indptr[0] != 0 || in.kv_indptr[0] != 0) return FI_ERR_INVALID_ARG;
  for (int i = 0; i < in.batch; ++i) {
    if (in.qo_indptr[i + 1] < in.qo_indptr[i]) return FI_ERR_INVALID_ARG;
    if (in.kv_indptr[i + 1] < in.kv_indptr[i]) return FI_ERR_INVALID_ARG;
    const int32_t n_pages = in.kv_indptr[i + 1] - in.kv_indptr[i];
    const int32_t last = in.last_page_len[i];
    if (last < 0 || last > in.page_size) return FI_ERR_INVALID_ARG;
    if (n_pages > 0 && last < 1) return FI_ERR_INVALID_ARG;
  }
  return FI_OK;
}

int plan_shape(const PlanInput& in, const CostModel& cm, PlanShape* s) {
  int st = validate_input(in);
  if (st != FI_OK) return st;
  if (cm.alpha < 0 || cm.beta < 1 || cm.l_min < 1) return FI_ERR_INVALID_ARG;
  const int B = in.batch;
  const int g = in.num_qo_heads / in.num_kv_heads;
  const int ps = in.page_size;

  // a1: lengths (key positions must stay within int32 item fields)
  int64_t max_lq = 0;
  for (int i = 0; i < B; ++i) {
    if (len_kv(in, i) > (int64_t(1) << 30)) return FI_ERR_UNSUPPORTED;
    max_lq = std::max(max_lq, len_q(in, i));
  }

  // a2: path and tile
  if (!in.force_tensor && max_lq * g <= kDecodeMaxRows) {
    s->path = kPathDecode;
    s->tile_tokens = static_cast<int>(std::max<int64_t>(1, max_lq));
    s->rows_tile = 1;
    while (s->rows_tile < s->tile_tokens * g) s->rows_tile *= 2;
  } else {
    if (g > kTcRows) return FI_ERR_UNSUPPORTED;
    // tensor-core tiles read whole 128-key tiles page by page through TMA boxes
    if (ps % 8 != 0 || kTcKeys % ps != 0) return FI_ERR_UNSUPPORTED;
    s->path = kPathTensor;
    s->tile_tokens = kTcRows / g;
    s->rows_tile = kTcRows;
  }
  s->group = g;
  s->num_ctas = (s->path == kPathTensor ? kTcCtasPerSm : kDecodeCtasPerSm) * in.num_sms;

  // a3: KV chunk bound (with a window: the keys each tile reads, which is all a window touches)
  int64_t total = 0;
  for (int i = 0; i < B; ++i) {
    const int64_t lq = len_q(in, i);
    if (in.window_left < 0) {
      total += int64_t(in.num_kv_heads) * ceil_div(lq, s->tile_tokens) * len_kv(in, i);
    } else {
      for (int64_t j = 0; j < ceil_div(lq, s->tile_tokens); ++j) {
        int64_t lo, e;
        extent(in, i, j * s->tile_tokens, std::min<int64_t>(s->tile_tokens, lq - j * s->tile_tokens), &lo, &e);
        total += int64_t(in.num_kv_heads) * (e - lo);
      }
    }
  }
  int64_t l_chunk = std::max<int64_t>(ceil_div(total, s->num_ctas), cm.l_min);
  l_chunk = ceil_div(l_chunk, ps) * ps;
  if (l_chunk > (int64_t(1) << 30)) return FI_ERR_UNSUPPORTED;
  s->l_chunk = l_chunk;

  // exact sizes of the plan (a4, a6)
  int64_t W = 0, U = 0, S = 0;
  for_each_unit(in, *s, [&](int, int, int64_t, int64_t, int64_t, int64_t, int64_t, int64_t n, int64_t) {
    W += n;
    if (n > 1 || in.all_slots) {
      U += 1;
      S += n;
    }
  });
  if (W > INT32_MAX / kItemFields) return FI_ERR_UNSUPPORTED;
  s->n_items = W;
  s->n_units = U;
  s->n_slots = S;
  return FI_OK;
}

void plan_fill(const PlanInput& in, const CostModel& cm, const PlanShape& s, const PlanStorage& st,
               int32_t* header) {
  const int g = s.group;
  // a4: units -> chunks; a6: slots of split units (enumeration order)
  int64_t W = 0, U = 0, S = 0;
  for_each_unit(in, s, [&](int i, int h, int64_t q0, int64_t qn, int64_t lo_e, int64_t e, int64_t cs, int64_t n,
                           int64_t diag) {
    int32_t first_slot = -1;
    if (n > 1 || in.all_slots) {
      first_slot = static_cast<int32_t>(S);
      int32_t* u = st.units + U * kUnitFields;
      u[U_FIRST_SLOT] = first_slot;
      u[U_N_CHUNKS] = static_cast<int32_t>(n);
      u[U_Q_START] = in.qo_indptr[i] + static_cast<int32_t>(q0);
      u[U_Q_LEN] = static_cast<int32_t>(qn);
      u[U_KV_HEAD] = h;
      u[5] = u[6] = u[7] = 0;
      for (int64_t c = 0; c < n; ++c) st.slot_unit[S + c] = static_cast<int32_t>(U);
      U += 1;
      S += n;
    }
    for (int64_t c = 0; c < n; ++c) {
      const int64_t lo = lo_e + c * cs, hi = std::min(e, lo_e + (c + 1) * cs);
      int32_t* w = st.work + W * kItemFields;
      w[I_PAGE_BASE] = in.kv_indptr[i];
      w[I_Q_START] = in.qo_indptr[i] + static_cast<int32_t>(q0);
      w[I_Q_LEN] = static_cast<int32_t>(qn);
      w[I_KV_HEAD] = h;
      w[I_KV_LO] = static_cast<int32_t>(lo);
      w[I_KV_HI] = static_cast<int32_t>(hi);
      w[I_DIAG] = static_cast<int32_t>(diag);
      w[I_SLOT] = first_slot >= 0 ? first_slot + static_cast<int32_t>(c) : -1;
      st.cost[W] = cm.alpha * qn * g + cm.beta * (hi - lo);
      st.order[W] = static_cast<int32_t>(W);
      W += 1;
    }
  });

  // a5: longest first (ties: enumeration order), then a min-queue of (load, CTA id)
  const int64_t* cost = st.cost;
  const int C = s.num_ctas;
  int64_t max_cost = 0, sum_cost = 0;
  for (int64_t k = 0; k < W; ++k) {
    max_cost = std::max(max_cost, cost[k]);
    sum_cost += cost[k];
  }
  // Both orders are total and the same as the tuple comparisons below; packed into one 64-bit key
  // when the values fit (they do for any batch within the workspace limits and cost model weights
  // up to 2^20), which makes the sort and the queue several times faster.
  const bool packed = max_cost < (int64_t(1) << 34) && W < (int64_t(1) << 28) &&
                      sum_cost < (int64_t(1) << 46) && C <= (1 << 16);
  if (packed) {
    // sort key: (max_cost - cost) << 28 | index, ascending = cost descending, then index ascending
    uint64_t* key = st.cost_key;
    for (int64_t k = 0; k < W; ++k) key[k] = (uint64_t(max_cost - cost[k]) << 28) | uint64_t(k);
    std::sort(key, key + W);
    for (int64_t k = 0; k < W; ++k) st.order[k] = static_cast<int32_t>(key[k] & ((uint64_t(1) << 28) - 1));
    // min-queue of (load << 16 | CTA id): the root is replaced and sifted down once per item
    uint64_t* q = key;  // the sort keys are no longer needed
    for (int c = 0; c < C; ++c) {
      q[c] = uint64_t(c);  // load 0: already a heap (ids ascending)
      st.count[c] = 0;
      if (st.loads) st.loads[c] = 0;
    }
    for (int64_t k = 0; k < W; ++k) {
      const int32_t it = st.order[k];
      const uint64_t top = q[0];
      const int32_t cta = static_cast<int32_t>(top & 0xFFFFu);
      st.cta_of[it] = cta;
      st.count[cta] += 1;
      const uint64_t v = top + (uint64_t(cost[it]) << 16);
      if (st.loads) st.loads[cta] = static_cast<int64_t>(v >> 16);
      int i = 0;
      for (;;) {
        const int l = 2 * i + 1;
        if (l >= C) break;
        const int m = (l + 1 < C && q[l + 1] < q[l]) ? l + 1 : l;
        if (q[m] >= v) break;
        q[i] = q[m];
        i = m;
      }
      q[i] = v;
    }
  } else {
    std::sort(st.order, st.order + W,
              [cost](int32_t a, int32_t b) { return cost[a] > cost[b] || (cost[a] == cost[b] && a < b); });
    std::greater<std::pair<int64_t, int32_t>> later;
    for (int c = 0; c < C; ++c) {
      st.heap[c] = {0, c};
      st.count[c] = 0;
      if (st.loads) st.loads[c] = 0;
    }
    std::make_heap(st.heap, st.heap + C, later);
    for (int64_t k = 0; k < W; ++k) {
      const int32_t it = st.order[k];
      std::pop_heap(st.heap, st.heap + C, later);
      std::pair<int64_t, int32_t>& top = st.heap[C - 1];
      st.cta_of[it] = top.second;
      st.count[top.second] += 1;
      top.first += cost[it];
      if (st.loads) st.loads[top.second] = top.first;
      std::push_heap(st.heap, st.heap + C, later);
    }
  }

  // queues in CSR form: each CTA's items in the order they were assigned
  st.cta_indptr[0] = 0;
  for (int c = 0; c < C; ++c) st.cta_indptr[c + 1] = st.cta_indptr[c] + st.count[c];
  for (int c = 0; c < C; ++c) st.count[c] = st.cta_indptr[c];  // fill cursors
  for (int64_t k = 0; k < W; ++k) {
    const int32_t it = st.order[k];
    const int32_t pos = st.count[st.cta_of[it]]++;
    std::memcpy(st.items + size_t(pos) * kItemFields, st.work + size_t(it) * kItemFields,
                sizeof(int32_t) * kItemFields);
  }

  int32_t* hd = header;
  hd[H_MAGIC] = kPlanMagic;
  hd[H_PATH] = s.path;
  hd[H_TILE_TOKENS] = s.tile_tokens;
  hd[H_ROWS_TILE] = s.rows_tile;
  hd[H_GROUP] = g;
  hd[H_NUM_CTAS] = C;
  hd[H_NUM_ITEMS] = static_cast<int32_t>(W);
  hd[H_NUM_UNITS] = static_cast<int32_t>(U);
  hd[H_NUM_SLOTS] = static_cast<int32_t>(S);
  hd[H_LKV] = static_cast<int32_t>(s.l_chunk);
  hd[H_PAGE_SIZE] = in.page_size;
  hd[H_CAUSAL] = in.causal;
  hd[H_HQO] = in.num_qo_heads;
  hd[H_HKV] = in.num_kv_heads;
  hd[H_HEAD_DIM] = in.head_dim;
  hd[H_BATCH] = in.batch;
}

int build_plan(const PlanInput& in, const CostModel& cm, Plan* out) {
  PlanShape s;
  const int st = plan_shape(in, cm, &s);
  if (st != FI_OK) return st;
  const size_t W = size_t(s.n_items), C = size_t(s.num_ctas);
  out->cta_indptr.assign(C + 1, 0);
  out->items.assign(W * kItemFields, 0);
  out->units.assign(size_t(s.n_units) * kUnitFields, 0);
  out->slot_unit.assign(size_t(s.n_slots), 0);
  out->loads.assign(C, 0);
  std::vector<int32_t> work(W * kItemFields), order(W), cta_of(W), count(C);
  std::vector<int64_t> cost(W);
  std::vector<std::pair<int64_t, int32_t>> heap(C);
  std::vector<uint64_t> key(std::max(W, C));
  PlanStorage ps{out->cta_indptr.data(), out->items.data(), out->units.data(), out->slot_unit.data(),
                 out->loads.data(), work.data(), cost.data(), order.data(), cta_of.data(), count.data(),
                 heap.data(), key.data()};
  plan_fill(in, cm, s, ps, out->header);
  return FI_OK;
}

int build_composable_plan(const PlanInput& shared_in, const PlanInput& unique_in, const CostModel& cm,
                          ComposablePlan* out) {
  if (shared_in.num_qo_heads != unique_in.num_qo_heads || shared_in.num_kv_heads != unique_in.num_kv_heads ||
      shared_in.head_dim != unique_in.head_dim || shared_in.page_size != unique_in.page_size ||
      shared_in.num_sms != unique_in.num_sms)
    return FI_ERR_INVALID_ARG;
  if (shared_in.batch < 0 || unique_in.batch < 0 || shared_in.qo_indptr == nullptr || unique_in.qo_indptr == nullptr)
    return FI_ERR_INVALID_ARG;
  // the shared rows are query tokens of the per-request part
  if (shared_in.qo_indptr[shared_in.batch] > unique_in.qo_indptr[unique_in.batch]) return FI_ERR_INVALID_ARG;
  PlanInput a = shared_in, b = unique_in;
  a.causal = 0;  // every shared key precedes the requests' own keys: all of it is visible
  a.window_left = -1;
  a.force_tensor = 1;
  a.all_slots = 1;
  b.force_tensor = 0;
  b.all_slots = 0;
  int st = validate_input(a);
  if (st == FI_OK) st = validate_input(b);
  if (st != FI_OK) return st;
  // split the SM budget: both parts run at once on disjoint SMs
  int64_t keys_a = 0, keys_b = 0;
  for (int i = 0; i < a.batch; ++i)
    if (len_q(a, i) > 0) keys_a += int64_t(a.num_kv_heads) * len_kv(a, i);
  for (int i = 0; i < b.batch; ++i)
    if (len_q(b, i) > 0) keys_b += int64_t(b.num_kv_heads) * len_kv(b, i);
  const int sms = shared_in.num_sms;
  int n_a = sms;
  if (sms > 1) {
    const int64_t c_a = int64_t(kTcKeyCostNum) * keys_a, c_b = int64_t(kTcKeyCostDen) * keys_b;
    n_a = c_a + c_b > 0 ? static_cast<int>((2 * int64_t(sms) * c_a + (c_a + c_b)) / (2 * (c_a + c_b))) : 1;
    n_a = std::min(std::max(n_a, 1), sms - 1);
  }
  a.num_sms = n_a;
  st = build_plan(a, cm, &out->shared);
  if (st != FI_OK) return st;
  // more shared chunks than CTAs would give some CTAs two: take as many CTAs as chunks (leaving at
  // least one SM) and plan the shared part once more
  // one adjustment toward one chunk per CTA: fewer chunks than CTAs leaves SMs idle, so take one
  // CTA per chunk; more (but at most twice as many) would give some CTAs two, so take as many CTAs
  // as chunks, leaving at least one SM
  const int items_a = out->shared.header[H_NUM_ITEMS];
  const int n_adj = items_a < n_a ? std::max(items_a, 1)
                    : (sms > 1 && items_a > n_a && items_a <= 2 * n_a) ? std::min(items_a, sms - 1) : n_a;
  if (n_adj != n_a) {
    n_a = n_adj;
    a.num_sms = n_a;
    st = build_plan(a, cm, &out->shared);
    if (st != FI_OK) return st;
  }
  b.num_sms = sms > 1 ? sms - n_a : 1;
  st = build_plan(b, cm, &out->unique);
  if (st != FI_OK) return st;
  if (out->unique.header[H_PATH] != kPathDecode) return FI_ERR_UNSUPPORTED;  // per-request rows must be decode tiles
  const int g = a.num_qo_heads / a.num_kv_heads;
  const int32_t s_a = out->shared.header[H_NUM_SLOTS];
  const int tok_a = out->shared.header[H_TILE_TOKENS];

  // per-request slots come after the shared ones
  Plan& u = out->unique;
  for (size_t k = 0; k < u.items.size(); k += kItemFields)
    if (u.items[k + I_SLOT] >= 0) u.items[k + I_SLOT] += s_a;
  for (size_t k = 0; k < u.units.size(); k += kUnitFields) u.units[k + U_FIRST_SLOT] += s_a;
  std::vector<int32_t> slot_unit(size_t(s_a), -1);
  slot_unit.insert(slot_unit.end(), u.slot_unit.begin(), u.slot_unit.end());
  u.slot_unit = std::move(slot_unit);

  // shared units in enumeration order: block row i, KV head h, tile j
  std::vector<int64_t> unit_base(size_t(a.batch) + 1, 0);
  for (int i = 0; i < a.batch; ++i) {
    const int64_t lq = int64_t(a.qo_indptr[i + 1]) - a.qo_indptr[i];
    unit_base[i + 1] = unit_base[i] + int64_t(a.num_kv_heads) * ((lq + tok_a - 1) / tok_a);
  }
  const std::vector<int32_t>& ua = out->shared.units;
  // ext entries of per-request rows [q0, q0 + qn) of KV head h: every chunk of every shared tile
  // that holds some of those tokens, block rows and tiles in order
  auto add_ext = [&](int32_t q0, int32_t qn, int32_t h) -> int32_t {
    int32_t count = 0;
    for (int i = 0; i < a.batch; ++i) {
      const int32_t lo = std::max(q0, a.qo_indptr[i]), hi = std::min(q0 + qn, a.qo_indptr[i + 1]);
      if (lo >= hi) continue;
      const int64_t n_tiles = (int64_t(a.qo_indptr[i + 1]) - a.qo_indptr[i] + tok_a - 1) / tok_a;
      const int64_t j0 = (lo - a.qo_indptr[i]) / tok_a, j1 = (hi - 1 - a.qo_indptr[i]) / tok_a;
      for (int64_t j = j0; j <= j1; ++j) {
        const int32_t* rec = &ua[size_t(unit_base[i] + int64_t(h) * n_tiles + j) * kUnitFields];
        const int32_t offset = (q0 - rec[U_Q_START]) * g;
        const int32_t packed = (offset + kExtRowBias) | ((rec[U_Q_LEN] * g) << 16);
        for (int32_t c = 0; c < rec[U_N_CHUNKS]; ++c) {
          out->ext.push_back(rec[U_FIRST_SLOT] + c);
          out->ext.push_back(packed);
          ++count;
        }
      }
    }
    return count;
  };
  // split units first (unit order), then single-chunk items with shared states (queue order)
  for (size_t k = 0; k < u.units.size(); k += kUnitFields) {
    const int32_t first = static_cast<int32_t>(out->ext.size() / 2);
    const int32_t cnt = add_ext(u.units[k + U_Q_START], u.units[k + U_Q_LEN], u.units[k + U_KV_HEAD]);
    u.units[k + 5] = first;
    u.units[k + 6] = cnt;
  }
  for (size_t k = 0; k < u.items.size(); k += kItemFields) {
    if (u.items[k + I_SLOT] != -1) continue;
    const int32_t first = static_cast<int32_t>(out->ext.size() / 2);
    const int32_t cnt = add_ext(u.items[k + I_Q_START], u.items[k + I_Q_LEN], u.items[k + I_KV_HEAD]);
    if (cnt == 0) continue;
    const int32_t unit = static_cast<int32_t>(u.units.size() / kUnitFields);
    const int32_t rec[kUnitFields] = {-1, 1, u.items[k + I_Q_START], u.items[k + I_Q_LEN], u.items[k + I_KV_HEAD],
                                      first, cnt, 0};
    u.units.insert(u.units.end(), rec, rec + kUnitFields);
    u.items[k + I_SLOT] = -(2 + unit);
  }
  u.header[H_NUM_UNITS] = static_cast<int32_t>(u.units.size() / kUnitFields);
  u.header[H_NUM_SLOTS] = s_a + u.header[H_NUM_SLOTS];
  return FI_OK;
}

}  // namespace fi

extern "C" int fi_plan_compute(const int32_t* qo_indptr, const int32_t* kv_indptr, const int32_t* last_page_len,
                               int batch, int num_qo_heads, int num_kv_heads, int head_dim, int page_size, int causal,
                               int num_sms, int64_t alpha, int64_t beta, int32_t l_min, int32_t window_left,
                               int32_t* out, int64_t capacity, int64_t* out_len) {
  if (out_len == nullptr) return FI_ERR_INVALID_ARG;
  fi::PlanInput in{qo_indptr, kv_indptr, last_page_len, batch, num_qo_heads, num_kv_heads, head_dim, page_size,
                   causal, num_sms, window_left};
  fi::CostModel cm;
  cm.alpha = alpha;
  cm.beta = beta;
  cm.l_min = l_min;
  fi::Plan p;
  const int st = fi::build_plan(in, cm, &p);
  if (st != FI_OK) return st;
  const int64_t need = fi::kHeaderLen + static_cast<int64_t>(p.cta_indptr.size() + p.items.size() + p.units.size() +
                                                             p.slot_unit.size());
  *out_len = need;
  if (out == nullptr || capacity < need) return FI_ERR_CAPACITY;
  int32_t* o = out;
  std::memcpy(o, p.header, sizeof(p.header));
  o += fi::kHeaderLen;
  for (const auto* v : {&p.cta_indptr, &p.items, &p.units, &p.slot_unit}) {
    if (!v->empty()) std::memcpy(o, v->data(), v->size() * sizeof(int32_t));
    o += v->size();
  }
  return FI_OK;
}

extern "C" int fi_plan_composable_compute(const int32_t* shared_qo_indptr, const int32_t* shared_kv_indptr,
                                          const int32_t* shared_last_page_len, int shared_batch,
                                          const int32_t* qo_indptr, const int32_t* kv_indptr,
                                          const int32_t* last_page_len, int batch, int num_qo_heads, int num_kv_heads,
                                          int head_dim, int page_size, int causal, int num_sms, int32_t* out,
                                          int64_t capacity, int64_t* out_len) {
  if (out_len == nullptr) return FI_ERR_INVALID_ARG;
  fi::PlanInput a{shared_qo_indptr, shared_kv_indptr, shared_last_page_len, shared_batch, num_qo_heads, num_kv_heads,
                  head_dim, page_size, 0, num_sms};
  fi::PlanInput b{qo_indptr, kv_indptr, last_page_len, batch, num_qo_heads, num_kv_heads, head_dim, page_size, causal,
                  num_sms};
  fi::ComposablePlan cp;
  const int st = fi::build_composable_plan(a, b, fi::CostModel(), &cp);
  if (st != FI_OK) return st;
  const fi::Plan* parts[2] = {&cp.shared, &cp.unique};
  int64_t need = 0;
  for (const fi::Plan* p : parts)
    need += fi::kHeaderLen + static_cast<int64_t>(p->cta_indptr.size() + p->items.size() + p->units.size() +
                                                  p->slot_unit.size());
  need += static_cast<int64_t>(cp.ext.size());
  *out_len = need;
  if (out == nullptr || capacity < need) return FI_ERR_CAPACITY;
  int32_t* o = out;
  for (const fi::Plan* p : parts) {
    std::memcpy(o, p->header, sizeof(p->header));
    o += fi::kHeaderLen;
    for (const auto* v : {&p->cta_indptr, &p->items, &p->units, &p->slot_unit}) {
      if (!v->empty()) std::memcpy(o, v->data(), v->size() * sizeof(int32_t));
      o += v->size();
    }
  }
  if (!cp.ext.empty()) std::memcpy(o, cp.ext.data(), cp.ext.size() * sizeof(int32_t));
  return FI_OK;
}
