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
//     rows), larger ones 128-row tensor-core tiles.
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
//   * #CTA = k * (SM budget) with k fixed per path (kDecodeCtasPerSm = 1,
//     kTcCtasPerSm = 2: two tensor-core CTAs share an SM);
//   * item cost = alpha * rows + beta * chunk length;
//   * sort by cost descending, ties by enumeration order; the queue pops the
//     least-loaded CTA, ties to the lowest CTA id.
#include "plan.h"

#include <algorithm>
#include <cstring>
#include <functional>
#include <numeric>
#include <queue>
#include <utility>

#include "../../include/fi.h"

namespace fi {

namespace {

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

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

int build_plan(const PlanInput& in, const CostModel& cm, Plan* out) {
  int st = validate_input(in);
  if (st != FI_OK) return st;
  if (cm.alpha < 0 || cm.beta < 1 || cm.l_min < 1) return FI_ERR_INVALID_ARG;
  const int B = in.batch;
  const int g = in.num_qo_heads / in.num_kv_heads;
  const int ps = in.page_size;

  // a1: lengths
  std::vector<int64_t> lq(B), lkv(B);
  int64_t max_lq = 0;
  for (int i = 0; i < B; ++i) {
    lq[i] = in.qo_indptr[i + 1] - in.qo_indptr[i];
    const int64_t n_pages = in.kv_indptr[i + 1] - in.kv_indptr[i];
    lkv[i] = n_pages > 0 ? (n_pages - 1) * ps + in.last_page_len[i] : 0;
    if (lkv[i] > (int64_t(1) << 30)) return FI_ERR_UNSUPPORTED;
    max_lq = std::max(max_lq, lq[i]);
  }

  // a2: path and tile
  int path, tile_tokens, rows_tile;
  if (max_lq * g <= kDecodeMaxRows) {
    path = kPathDecode;
    tile_tokens = static_cast<int>(std::max<int64_t>(1, max_lq));
    rows_tile = 1;
    while (rows_tile < tile_tokens * g) rows_tile *= 2;
  } else {
    if (g > kTcRows) return FI_ERR_UNSUPPORTED;
    // tensor-core tiles read whole 128-key tiles page by page through TMA boxes
    if (ps % 8 != 0 || kTcRows % ps != 0) return FI_ERR_UNSUPPORTED;
    path = kPathTensor;
    tile_tokens = kTcRows / g;
    rows_tile = kTcRows;
  }
  const int num_ctas = (path == kPathTensor ? kTcCtasPerSm : kDecodeCtasPerSm) * in.num_sms;

  // keys [lo, e) that tile rows q0 .. q0+qn-1 of request i can see
  auto extent = [&](int i, int64_t q0, int64_t qn, int64_t* lo, int64_t* e) {
    if (!in.causal) {
      *lo = 0;
      *e = lkv[i];
      return;
    }
    *e = std::min(std::max<int64_t>(lkv[i] - lq[i] + q0 + qn, 0), lkv[i]);
    *lo = 0;
    if (in.window_left >= 0) {
      *lo = std::max<int64_t>(0, lkv[i] - lq[i] + q0 - in.window_left) / ps * ps;
      *lo = std::min(*lo, *e);
    }
  };

  // a3: KV chunk bound (with a window: the keys each tile reads, which is all a window touches)
  int64_t total = 0;
  for (int i = 0; i < B; ++i) {
    if (in.window_left < 0) {
      total += int64_t(in.num_kv_heads) * ceil_div(lq[i], tile_tokens) * lkv[i];
    } else {
      for (int64_t j = 0; j < ceil_div(lq[i], tile_tokens); ++j) {
        int64_t lo, e;
        extent(i, j * tile_tokens, std::min<int64_t>(tile_tokens, lq[i] - j * tile_tokens), &lo, &e);
        total += int64_t(in.num_kv_heads) * (e - lo);
      }
    }
  }
  int64_t l_chunk = std::max<int64_t>(ceil_div(total, num_ctas), cm.l_min);
  l_chunk = ceil_div(l_chunk, ps) * ps;
  if (l_chunk > (int64_t(1) << 30)) return FI_ERR_UNSUPPORTED;

  // a4: units -> chunks; a6: slots of split units (enumeration order)
  struct Work {
    int32_t f[kItemFields];
    int64_t cost;
  };
  std::vector<Work> work;
  std::vector<int32_t> units, slot_unit;
  for (int i = 0; i < B; ++i) {
    const int64_t n_tiles = ceil_div(lq[i], tile_tokens);
    for (int h = 0; h < in.num_kv_heads; ++h) {
      for (int64_t j = 0; j < n_tiles; ++j) {
        const int64_t q0 = j * tile_tokens;
        const int64_t qn = std::min<int64_t>(tile_tokens, lq[i] - q0);
        int64_t lo_e, e;
        extent(i, q0, qn, &lo_e, &e);
        const int64_t diag = in.causal ? lkv[i] - lq[i] + q0 : kNotCausalDiag;
        int64_t n, cs;
        if (e - lo_e == 0) {
          n = 1;
          cs = 0;
        } else {
          n = ceil_div(e - lo_e, l_chunk);
          cs = ceil_div(ceil_div(e - lo_e, n), ps) * ps;
          n = ceil_div(e - lo_e, cs);
        }
        int32_t first_slot = -1;
        if (n > 1) {
          const int32_t unit = static_cast<int32_t>(units.size() / kUnitFields);
          first_slot = static_cast<int32_t>(slot_unit.size());
          const int32_t u[kUnitFields] = {first_slot, static_cast<int32_t>(n), in.qo_indptr[i] + static_cast<int32_t>(q0),
                                          static_cast<int32_t>(qn), h, 0, 0, 0};
          units.insert(units.end(), u, u + kUnitFields);
          slot_unit.insert(slot_unit.end(), static_cast<size_t>(n), unit);
        }
        for (int64_t c = 0; c < n; ++c) {
          const int64_t lo = lo_e + c * cs, hi = std::min(e, lo_e + (c + 1) * cs);
          Work w;
          w.f[I_PAGE_BASE] = in.kv_indptr[i];
          w.f[I_Q_START] = in.qo_indptr[i] + static_cast<int32_t>(q0);
          w.f[I_Q_LEN] = static_cast<int32_t>(qn);
          w.f[I_KV_HEAD] = h;
          w.f[I_KV_LO] = static_cast<int32_t>(lo);
          w.f[I_KV_HI] = static_cast<int32_t>(hi);
          w.f[I_DIAG] = static_cast<int32_t>(diag);
          w.f[I_SLOT] = first_slot >= 0 ? first_slot + static_cast<int32_t>(c) : -1;
          w.cost = cm.alpha * qn * g + cm.beta * (hi - lo);
          work.push_back(w);
        }
      }
    }
  }

  // a5: longest first (ties: enumeration order), then a min-queue of (load, cta id)
  const size_t W = work.size();
  std::vector<int32_t> order(W);
  std::iota(order.begin(), order.end(), 0);
  std::stable_sort(order.begin(), order.end(), [&](int32_t a, int32_t b) { return work[a].cost > work[b].cost; });
  using Entry = std::pair<int64_t, int32_t>;
  std::priority_queue<Entry, std::vector<Entry>, std::greater<Entry>> queue;
  for (int32_t c = 0; c < num_ctas; ++c) queue.push({0, c});
  std::vector<int32_t> cta_of(W);
  std::vector<int32_t> count(num_ctas, 0);
  std::vector<int64_t> loads(num_ctas, 0);
  for (int32_t k : order) {
    Entry top = queue.top();
    queue.pop();
    cta_of[k] = top.second;
    count[top.second] += 1;
    top.first += work[k].cost;
    loads[top.second] = top.first;
    queue.push(top);
  }

  out->cta_indptr.assign(num_ctas + 1, 0);
  for (int c = 0; c < num_ctas; ++c) out->cta_indptr[c + 1] = out->cta_indptr[c] + count[c];
  out->items.assign(W * kItemFields, 0);
  std::vector<int32_t> fill(out->cta_indptr.begin(), out->cta_indptr.end() - 1);
  for (int32_t k : order) {
    const int32_t pos = fill[cta_of[k]]++;
    std::memcpy(&out->items[size_t(pos) * kItemFields], work[k].f, sizeof(work[k].f));
  }
  out->units = std::move(units);
  out->slot_unit = std::move(slot_unit);
  out->loads = std::move(loads);

  int32_t* h = out->header;
  h[H_MAGIC] = kPlanMagic;
  h[H_PATH] = path;
  h[H_TILE_TOKENS] = tile_tokens;
  h[H_ROWS_TILE] = rows_tile;
  h[H_GROUP] = g;
  h[H_NUM_CTAS] = num_ctas;
  h[H_NUM_ITEMS] = static_cast<int32_t>(W);
  h[H_NUM_UNITS] = static_cast<int32_t>(out->units.size() / kUnitFields);
  h[H_NUM_SLOTS] = static_cast<int32_t>(out->slot_unit.size());
  h[H_LKV] = static_cast<int32_t>(l_chunk);
  h[H_PAGE_SIZE] = ps;
  h[H_CAUSAL] = in.causal;
  h[H_HQO] = in.num_qo_heads;
  h[H_HKV] = in.num_kv_heads;
  h[H_HEAD_DIM] = in.head_dim;
  h[H_BATCH] = B;
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
