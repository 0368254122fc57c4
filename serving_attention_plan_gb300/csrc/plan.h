// Host planner of the paged serving-attention library (C++17, no CUDA).
//
// Builds the per-step work plan described on page "FlashInfer：面向 LLM 推理服务
// 的高效可定制注意力引擎", 核心机制 6 (paper §3.3.1, Alg. 1) and 核心机制 7
// (paper App. D.2-D.3).  The rules fixed where the page is silent are listed
// beside `build_plan`.
#pragma once

#include <cstdint>
#include <utility>
#include <vector>

namespace fi {

constexpr int kHeadDim = 128;
constexpr int kPathDecode = 0;
constexpr int kPathTensor = 1;
constexpr int kPathComposable = 2;  // header[H_PATH] of a composable plan (both paths, one reduction map)
constexpr int kTcRows = 256;          // rows of a tensor-core tile: two 128-row tcgen05 tiles sharing each KV tile
constexpr int kTcKeys = 128;          // keys of a tensor-core KV tile
constexpr int kDecodeMaxRows = 8;     // largest tile the CUDA-core decode path takes
constexpr int kDecodeCtasPerSm = 1;   // persistent CTAs per SM of each path (#CTA = k * #SM)
constexpr int kTcCtasPerSm = 1;
constexpr int32_t kNotCausalDiag = 1 << 30;
constexpr int32_t kPlanMagic = 0x46495031;
constexpr int kHeaderLen = 16;
constexpr int kItemFields = 8;
constexpr int kUnitFields = 8;

// Header slots.
enum HeaderSlot {
  H_MAGIC = 0, H_PATH, H_TILE_TOKENS, H_ROWS_TILE, H_GROUP, H_NUM_CTAS, H_NUM_ITEMS, H_NUM_UNITS,
  H_NUM_SLOTS, H_LKV, H_PAGE_SIZE, H_CAUSAL, H_HQO, H_HKV, H_HEAD_DIM, H_BATCH
};

// Item fields: one chunk of one (request, KV head, query tile).
enum ItemField { I_PAGE_BASE = 0, I_Q_START, I_Q_LEN, I_KV_HEAD, I_KV_LO, I_KV_HI, I_DIAG, I_SLOT };
// Split-unit fields: the reduction map of one split (request, KV head, query tile).
enum UnitField { U_FIRST_SLOT = 0, U_N_CHUNKS, U_Q_START, U_Q_LEN, U_KV_HEAD };

struct CostModel {
  int64_t alpha = 1;
  int64_t beta = 1;
  int32_t l_min = 256;
};

struct PlanInput {
  const int32_t* qo_indptr;
  const int32_t* kv_indptr;
  const int32_t* last_page_len;
  int batch;
  int num_qo_heads;
  int num_kv_heads;
  int head_dim;
  int page_size;
  int causal;
  int num_sms;  // SM budget; the plan's #CTA is k * num_sms with k fixed per path
  int window_left = -1;  // >= 0: sliding window (causal plans): token at position p sees keys p - w .. p
  int force_tensor = 0;  // 1: tensor-core tiles even when every request fits a decode tile
  int all_slots = 0;     // 1: every unit, split or not, writes its chunks' partial states to slots
};

// Attention variant of a plan (问题背景 挑战二; 核心机制 5, paper §3.2.3): a sliding window on
// causal masks, a logit soft-cap, and the page layout.
struct Variant {
  int window_left = -1;  // < 0: none
  float soft_cap = 0.f;  // <= 0: none
  int kv_layout = 0;     // FI_KV_LAYOUT_HND or FI_KV_LAYOUT_NHD
  int kv_dtype = 0;      // FI_KV_DTYPE_BF16 or FI_KV_DTYPE_E4M3
  float k_scale = 1.f;   // e4m3 pages: K = k_scale * code, V = v_scale * code
  float v_scale = 1.f;
};

struct Plan {
  int32_t header[kHeaderLen];
  std::vector<int32_t> cta_indptr;   // [num_ctas + 1]
  std::vector<int32_t> items;        // [n_items * kItemFields], CTA queue order
  std::vector<int32_t> units;        // [n_units * kUnitFields]
  std::vector<int32_t> slot_unit;    // [n_slots]
  std::vector<int64_t> loads;        // accumulated cost per CTA
};

// Returns an fi_status code (0 = ok).
int build_plan(const PlanInput& in, const CostModel& cost, Plan* out);

// The same planner in two passes over caller-owned storage, for callers that must not allocate:
// plan_shape fixes the path, tile, #CTA, chunk bound and the exact counts of items, split rows and
// slots; plan_fill then writes the plan into the given arrays (it allocates nothing).  build_plan is
// these two passes over vectors, so every caller gets the same plan bit for bit.
struct PlanShape {
  int path, tile_tokens, rows_tile, group, num_ctas;
  int64_t l_chunk;
  int64_t n_items, n_units, n_slots;
};

struct PlanStorage {
  // outputs, in the layout of Plan
  int32_t* cta_indptr;  // [num_ctas + 1]
  int32_t* items;       // [n_items * kItemFields], CTA queue order
  int32_t* units;       // [n_units * kUnitFields]
  int32_t* slot_unit;   // [n_slots]
  int64_t* loads;       // [num_ctas] accumulated cost per CTA (may be null)
  // work arrays of the fill pass
  int32_t* work;        // [n_items * kItemFields], enumeration order
  int64_t* cost;        // [n_items]
  int32_t* order;       // [n_items]
  int32_t* cta_of;      // [n_items]
  int32_t* count;       // [num_ctas]
  std::pair<int64_t, int32_t>* heap;  // [num_ctas] (load, CTA id)
  uint64_t* cost_key;  // [max(n_items, num_ctas)]: packed sort keys, then the packed queue
};

int plan_shape(const PlanInput& in, const CostModel& cost, PlanShape* shape);

// Composable formats (核心机制 2, paper §3.1.2, Fig. 3): a shared sub-matrix (block rows such as a
// prefix shared by a group of requests, Br = the group's query tokens) and a per-request sub-matrix
// (Br = 1) over the same query rows, in one plan with one reduction map.  The shared part takes
// tensor-core tiles and writes every chunk to a partial slot; the per-request part takes decode
// tiles, its slots are numbered after the shared part's, and each of its units lists the shared
// slots that hold states of its rows (ext: pairs {slot, packed}, packed = (row offset + 512) |
// (rows of the shared tile << 16); the unit's row r is row `offset + r` of that slot when it lies in
// [0, rows)).  A single-chunk unit with shared states gets a unit record too (first slot -1) and its
// item's slot field is -(2 + unit).  Unit fields 5 and 6 hold the unit's first ext entry and count.
constexpr int kExtRowBias = 512;
// SM budget split of a composable plan: the shared part gets N_tc = round(num_sms * c_a / (c_a + c_b))
// CTAs (at least 1, and at least 1 left for the other part when num_sms > 1), then set once to its
// number of chunks when that is smaller, or larger but at most twice as large (one chunk per CTA);
// the per-request part gets the rest; both run at once, one CTA per SM.  c_a = kTcKeyCostNum *
// (keys the shared units see) and c_b = kTcKeyCostDen * (keys the per-request units see): a key of a
// 256-row tensor-core tile costs about 4/3 of a decode key in SM time (measured on GB300 with the
// shared-prefix batch: 0.025 us*SM per key on tensor-core tiles, 0.019 on decode tiles).
constexpr int kTcKeyCostNum = 4;
constexpr int kTcKeyCostDen = 3;
struct ComposablePlan {
  Plan shared;
  Plan unique;
  std::vector<int32_t> ext;  // [n_ext * 2]
};
int build_composable_plan(const PlanInput& shared, const PlanInput& unique, const CostModel& cost,
                          ComposablePlan* out);
void plan_fill(const PlanInput& in, const CostModel& cost, const PlanShape& shape, const PlanStorage& st,
               int32_t* header);

// Checks that only depend on the inputs (same rules as build_plan's validation).
int validate_input(const PlanInput& in);

}  // namespace fi
