// C ABI of the library: workspace, plan upload, run, merge, errors.
//
// Page "FlashInfer：面向 LLM 推理服务的高效可定制注意力引擎", 核心机制 7
// "CUDAGraph 兼容的静态化手段" (paper App. D.1-D.3): the workspace is
// allocated once at maximum capacity with constant segment offsets; the plan
// is computed in page-locked host memory and sent to its segments with
// cudaMemcpyAsync; the persistent kernel has a fixed grid.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>
#include <new>
#include <string>

#include "../../include/fi.h"
#include "decode_launch.cuh"
#include "merge_kernel.cuh"
#include "plan.h"
#include "prefill_launch.h"

namespace {

thread_local std::string g_last_error;

int cuda_fail(cudaError_t e, const char* what) {
  g_last_error = std::string(what) + ": " + cudaGetErrorString(e);
  return FI_ERR_CUDA;
}

#define FI_CUDA(call)                                        \
  do {                                                       \
    cudaError_t e_ = (call);                                 \
    if (e_ != cudaSuccess) return cuda_fail(e_, #call);      \
  } while (0)

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace

int fi::record_cuda_error(cudaError_t e, const char* what) { return cuda_fail(e, what); }

struct fi_workspace {
  int device = 0;
  int max_batch = 0, max_total_q = 0, max_kv_pages = 0;
  int hqo = 0, hkv = 0, head_dim = 0, num_sms = 0, max_ctas = 0;
  int64_t max_items = 0, max_units = 0, max_slots = 0;
  fi::CostModel cost;
  fi::Variant variant;       // as set for the next fi_plan
  fi::Variant plan_variant;  // the one the current plan was made with (used by fi_run)

  // segment byte offsets; [0, plan_bytes) is mirrored in pinned host memory.  The a_* segments and
  // the ext list hold the shared part of a composable plan.
  size_t off_header = 0, off_cta = 0, off_items = 0, off_units = 0, off_slot_unit = 0, off_kv = 0, plan_bytes = 0;
  size_t off_a_header = 0, off_a_cta = 0, off_a_items = 0, off_a_kv = 0, off_ext = 0;
  int64_t max_ext = 0;
  size_t off_counters = 0, off_err = 0, off_part_lse = 0, off_part_o = 0, dev_bytes = 0;
  char* dbuf = nullptr;
  char* hbuf = nullptr;
  cudaEvent_t copy_done = nullptr;
  bool copy_pending = false;

  bool has_plan = false;
  bool composable = false;
  int32_t header[fi::kHeaderLen] = {0};
  int32_t a_header[fi::kHeaderLen] = {0};
  int32_t max_page = -1;
  int64_t plan_nnz = 0;
  int32_t plan_total_q = 0;
};

namespace {

// HND pages: power-of-two page sizes of 8 or more tokens take the TMA copier (unless `tma` is
// false), smaller ones the 16-byte-copy loader, others the bulk-copy loader.  The page layout and
// the attention variant are template flags, so the plain HND path compiles without a trace of them.
template <int R>
int launch_decode(int grid, const fi::DecodeParams& p, cudaStream_t stream, bool var, bool pdl = false,
                  bool tma = true) {
  using fi::kDecodeCopiers;
  constexpr int kV = fi::kDecodeVariant;
  if (tma && p.page_shift >= 0 && p.page_size >= 8) {
    CUtensorMap tm_k, tm_v;
    const int hkv = int(p.page_stride / (int64_t(p.page_size) * fi::kHeadDim));
    const int box_rows = p.page_size < fi::kStageTokens ? p.page_size : fi::kStageTokens;  // as the copier's boxes
    if (!fi::make_decode_map_bf16(&tm_k, p.k, hkv, p.page_size, p.num_pages, box_rows) ||
        !fi::make_decode_map_bf16(&tm_v, p.v, hkv, p.page_size, p.num_pages, box_rows))
      return FI_ERR_INVALID_ARG;
    return var ? fi::launch_decode_tma_as<R, kV>(grid, p, tm_k, tm_v, stream, pdl)
               : fi::launch_decode_tma_as<R, 0>(grid, p, tm_k, tm_v, stream, pdl);
  }
  if (p.page_shift >= 0)
    return var ? fi::launch_decode_as<R, kDecodeCopiers, kV>(grid, p, stream, pdl)
               : fi::launch_decode_as<R, kDecodeCopiers, 0>(grid, p, stream, pdl);
  return var ? fi::launch_decode_as<R, 0, kV>(grid, p, stream, pdl)
             : fi::launch_decode_as<R, 0, 0>(grid, p, stream, pdl);
}

bool var_on(const fi::Variant& v) { return v.window_left >= 0 || v.soft_cap > 0.f; }

}  // namespace

extern "C" {

const char* fi_status_string(int status) {
  switch (status) {
    case FI_OK: return "ok";
    case FI_ERR_INVALID_ARG: return "invalid argument";
    case FI_ERR_CAPACITY: return "workspace capacity exceeded";
    case FI_ERR_UNSUPPORTED: return "unsupported shape";
    case FI_ERR_CUDA: return "CUDA error";
    case FI_ERR_DEVICE: return "device-side check failed";
    case FI_ERR_NO_PLAN: return "no plan";
    default: return "unknown status";
  }
}

const char* fi_last_error_message(void) { return g_last_error.c_str(); }

int fi_device_sm_count(int* out) {
  if (out == nullptr) return FI_ERR_INVALID_ARG;
  int dev = 0;
  FI_CUDA(cudaGetDevice(&dev));
  FI_CUDA(cudaDeviceGetAttribute(out, cudaDevAttrMultiProcessorCount, dev));
  return FI_OK;
}

int fi_workspace_create(int max_batch, int max_total_q, int max_kv_pages, int num_qo_heads, int num_kv_heads,
                        int head_dim, int num_sms, fi_workspace** out) {
  if (out == nullptr) return FI_ERR_INVALID_ARG;
  *out = nullptr;
  if (max_batch < 1 || max_total_q < 1 || max_kv_pages < 1 || num_qo_heads < 1 || num_kv_heads < 1 || num_sms < 0)
    return FI_ERR_INVALID_ARG;
  if (head_dim != fi::kHeadDim || num_qo_heads % num_kv_heads != 0) return FI_ERR_UNSUPPORTED;
  int dev = 0;
  FI_CUDA(cudaGetDevice(&dev));
  if (num_sms == 0) FI_CUDA(cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev));

  fi_workspace* ws = new (std::nothrow) fi_workspace();
  if (ws == nullptr) return FI_ERR_CAPACITY;
  ws->device = dev;
  ws->max_batch = max_batch;
  ws->max_total_q = max_total_q;
  ws->max_kv_pages = max_kv_pages;
  ws->hqo = num_qo_heads;
  ws->hkv = num_kv_heads;
  ws->head_dim = head_dim;
  ws->num_sms = num_sms;
  ws->max_ctas = std::max(fi::kTcCtasPerSm, fi::kDecodeCtasPerSm) * num_sms;
  // App. D.3 bound: partial tiles < 2 * #CTA, hence split rows < #CTA; a composable plan's decode
  // part adds a unit record per (request, KV head) whose rows merge shared states
  ws->max_slots = 2 * int64_t(ws->max_ctas);
  ws->max_units = ws->max_ctas + int64_t(num_kv_heads) * max_batch;
  ws->max_items = int64_t(num_kv_heads) * max_total_q + ws->max_slots;
  // each shared slot holds 256 rows, so at most 256 per-request units list it
  ws->max_ext = ws->max_slots * fi::kTcRows;

  size_t off = 0;
  auto seg = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  ws->off_header = seg(sizeof(int32_t) * fi::kHeaderLen);
  ws->off_cta = seg(sizeof(int32_t) * (ws->max_ctas + 1));
  ws->off_items = seg(sizeof(int32_t) * fi::kItemFields * ws->max_items);
  ws->off_units = seg(sizeof(int32_t) * fi::kUnitFields * ws->max_units);
  ws->off_slot_unit = seg(sizeof(int32_t) * ws->max_slots);
  ws->off_kv = seg(sizeof(int32_t) * size_t(max_kv_pages));
  ws->off_a_header = seg(sizeof(int32_t) * fi::kHeaderLen);
  ws->off_a_cta = seg(sizeof(int32_t) * (ws->max_ctas + 1));
  ws->off_a_items = seg(sizeof(int32_t) * fi::kItemFields * ws->max_items);
  ws->off_a_kv = seg(sizeof(int32_t) * size_t(max_kv_pages));
  ws->off_ext = seg(sizeof(int32_t) * 2 * ws->max_ext);
  ws->plan_bytes = off;
  ws->off_counters = seg(sizeof(uint32_t) * ws->max_units);
  ws->off_err = seg(sizeof(int32_t) * 4);
  ws->off_part_lse = seg(sizeof(float) * ws->max_slots * fi::kTcRows);
  ws->off_part_o = seg(sizeof(float) * ws->max_slots * fi::kTcRows * fi::kHeadDim);
  ws->dev_bytes = off;

  cudaError_t e = cudaMalloc(&ws->dbuf, ws->dev_bytes);
  if (e == cudaSuccess) e = cudaMemset(ws->dbuf + ws->off_counters, 0, ws->off_part_lse - ws->off_counters);
  if (e == cudaSuccess) e = cudaHostAlloc(reinterpret_cast<void**>(&ws->hbuf), ws->plan_bytes, cudaHostAllocDefault);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ws->copy_done, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    const int st = cuda_fail(e, "fi_workspace_create");
    fi_workspace_destroy(ws);
    return st;
  }
  *out = ws;
  return FI_OK;
}

int fi_workspace_destroy(fi_workspace* ws) {
  if (ws == nullptr) return FI_OK;
  if (ws->copy_done != nullptr) {
    cudaEventSynchronize(ws->copy_done);
    cudaEventDestroy(ws->copy_done);
  }
  if (ws->hbuf != nullptr) cudaFreeHost(ws->hbuf);
  if (ws->dbuf != nullptr) cudaFree(ws->dbuf);
  delete ws;
  return FI_OK;
}

int fi_workspace_set_cost_model(fi_workspace* ws, int64_t alpha, int64_t beta, int32_t l_min) {
  if (ws == nullptr || alpha < 0 || beta < 1 || l_min < 1) return FI_ERR_INVALID_ARG;
  ws->cost.alpha = alpha;
  ws->cost.beta = beta;
  ws->cost.l_min = l_min;
  return FI_OK;
}

int fi_workspace_set_variant(fi_workspace* ws, int32_t window_left, float logits_soft_cap, int32_t kv_layout) {
  if (ws == nullptr || window_left < -1 || !(logits_soft_cap >= 0.f) || logits_soft_cap > 1e30f ||
      (kv_layout != FI_KV_LAYOUT_HND && kv_layout != FI_KV_LAYOUT_NHD))
    return FI_ERR_INVALID_ARG;
  ws->variant.window_left = window_left;
  ws->variant.soft_cap = logits_soft_cap;
  ws->variant.kv_layout = kv_layout;
  return FI_OK;
}

int fi_workspace_set_kv_dtype(fi_workspace* ws, int32_t kv_dtype, float k_scale, float v_scale) {
  if (ws == nullptr || (kv_dtype != FI_KV_DTYPE_BF16 && kv_dtype != FI_KV_DTYPE_E4M3) || !(k_scale > 0.f) ||
      !(v_scale > 0.f) || k_scale > 1e30f || v_scale > 1e30f)
    return FI_ERR_INVALID_ARG;
  ws->variant.kv_dtype = kv_dtype;
  ws->variant.k_scale = k_scale;
  ws->variant.v_scale = v_scale;
  return FI_OK;
}

int fi_plan(fi_workspace* ws, const int32_t* qo_indptr, const int32_t* kv_indptr, const int32_t* kv_indices,
            const int32_t* last_page_len, int batch, int num_qo_heads, int num_kv_heads, int head_dim, int page_size,
            int causal, void* stream) {
  if (ws == nullptr) return FI_ERR_INVALID_ARG;
  if (num_qo_heads != ws->hqo || num_kv_heads != ws->hkv || head_dim != ws->head_dim) return FI_ERR_INVALID_ARG;
  if (batch > ws->max_batch) return FI_ERR_CAPACITY;
  fi::PlanInput in{qo_indptr, kv_indptr, last_page_len, batch, num_qo_heads, num_kv_heads, head_dim, page_size,
                   causal, ws->num_sms, ws->variant.window_left};
  int st = fi::validate_input(in);
  if (st != FI_OK) return st;
  const int64_t nnz = kv_indptr[batch];
  if (qo_indptr[batch] > ws->max_total_q || nnz > ws->max_kv_pages) return FI_ERR_CAPACITY;
  if (nnz > 0 && kv_indices == nullptr) return FI_ERR_INVALID_ARG;
  int32_t max_page = -1;
  for (int64_t k = 0; k < nnz; ++k) {
    if (kv_indices[k] < 0) return FI_ERR_INVALID_ARG;
    max_page = std::max(max_page, kv_indices[k]);
  }
  fi::Plan plan;
  st = fi::build_plan(in, ws->cost, &plan);
  if (st != FI_OK) return st;
  // NHD decode reads page rows with the 16-byte-copy loader (power-of-two pages); its kernels are
  // instantiated for 1, 2, 4, 8 and 16 KV heads
  // e4m3 pages on decode tiles: power-of-two pages (the FP8 decode kernel's loader); tensor-core
  // tiles widen e4m3 pages in their producer and take the page sizes of bf16 pages
  if (ws->variant.kv_dtype == FI_KV_DTYPE_E4M3 && plan.header[fi::H_PATH] == fi::kPathDecode &&
      (page_size & (page_size - 1)) != 0)
    return FI_ERR_UNSUPPORTED;
  if (ws->variant.kv_layout == FI_KV_LAYOUT_NHD && plan.header[fi::H_PATH] == fi::kPathDecode &&
      ((page_size & (page_size - 1)) != 0 || (num_kv_heads & (num_kv_heads - 1)) != 0 || num_kv_heads > 16))
    return FI_ERR_UNSUPPORTED;
  const int64_t n_items = plan.header[fi::H_NUM_ITEMS], n_units = plan.header[fi::H_NUM_UNITS],
                n_slots = plan.header[fi::H_NUM_SLOTS];
  if (n_items > ws->max_items || n_units > ws->max_units || n_slots > ws->max_slots) return FI_ERR_CAPACITY;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (ws->copy_pending) {
    FI_CUDA(cudaEventSynchronize(ws->copy_done));
    ws->copy_pending = false;
  }
  char* h = ws->hbuf;
  std::memcpy(h + ws->off_header, plan.header, sizeof(plan.header));
  std::memcpy(h + ws->off_cta, plan.cta_indptr.data(), plan.cta_indptr.size() * sizeof(int32_t));
  if (n_items) std::memcpy(h + ws->off_items, plan.items.data(), plan.items.size() * sizeof(int32_t));
  if (n_units) std::memcpy(h + ws->off_units, plan.units.data(), plan.units.size() * sizeof(int32_t));
  if (n_slots) std::memcpy(h + ws->off_slot_unit, plan.slot_unit.data(), plan.slot_unit.size() * sizeof(int32_t));
  if (nnz) std::memcpy(h + ws->off_kv, kv_indices, size_t(nnz) * sizeof(int32_t));

  struct Seg {
    size_t off, bytes;
  } segs[] = {
      {ws->off_header, sizeof(plan.header)},
      {ws->off_cta, plan.cta_indptr.size() * sizeof(int32_t)},
      {ws->off_items, plan.items.size() * sizeof(int32_t)},
      {ws->off_units, plan.units.size() * sizeof(int32_t)},
      {ws->off_slot_unit, plan.slot_unit.size() * sizeof(int32_t)},
      {ws->off_kv, size_t(nnz) * sizeof(int32_t)},
  };
  // adjacent segments go up in one copy when the unused capacity between them is small (it goes up
  // too, and nothing reads it): fewer copy calls on the host path of every step
  constexpr size_t kMergeGap = 16 << 10;
  size_t run_off = 0, run_end = 0;  // the pending copy [run_off, run_end)
  for (const Seg& sg : segs) {
    if (sg.bytes == 0) continue;
    if (run_end > run_off && sg.off - run_end <= kMergeGap) {
      run_end = sg.off + sg.bytes;
      continue;
    }
    if (run_end > run_off)
      FI_CUDA(cudaMemcpyAsync(ws->dbuf + run_off, h + run_off, run_end - run_off, cudaMemcpyHostToDevice, s));
    run_off = sg.off;
    run_end = sg.off + sg.bytes;
  }
  if (run_end > run_off)
    FI_CUDA(cudaMemcpyAsync(ws->dbuf + run_off, h + run_off, run_end - run_off, cudaMemcpyHostToDevice, s));
  FI_CUDA(cudaEventRecord(ws->copy_done, s));
  ws->copy_pending = true;
  std::memcpy(ws->header, plan.header, sizeof(plan.header));
  ws->max_page = max_page;
  ws->plan_nnz = nnz;
  ws->plan_total_q = qo_indptr[batch];
  ws->has_plan = true;
  ws->composable = false;
  ws->plan_variant = ws->variant;
  return FI_OK;
}

int fi_plan_composable(fi_workspace* ws, const int32_t* shared_qo_indptr, const int32_t* shared_kv_indptr,
                       const int32_t* shared_kv_indices, const int32_t* shared_last_page_len, int shared_batch,
                       const int32_t* qo_indptr, const int32_t* kv_indptr, const int32_t* kv_indices,
                       const int32_t* last_page_len, int batch, int num_qo_heads, int num_kv_heads, int head_dim,
                       int page_size, int causal, void* stream) {
  if (ws == nullptr) return FI_ERR_INVALID_ARG;
  if (num_qo_heads != ws->hqo || num_kv_heads != ws->hkv || head_dim != ws->head_dim) return FI_ERR_INVALID_ARG;
  if (batch > ws->max_batch || shared_batch > ws->max_batch) return FI_ERR_CAPACITY;
  const fi::Variant& var = ws->variant;
  if (var.window_left >= 0 || var.soft_cap > 0.f || var.kv_layout != FI_KV_LAYOUT_HND)
    return FI_ERR_UNSUPPORTED;  // composable plans run the plain HND kernels (bf16 or e4m3 pages)
  if (var.kv_dtype == FI_KV_DTYPE_E4M3 && (page_size & (page_size - 1)) != 0)
    return FI_ERR_UNSUPPORTED;  // the per-request rows' FP8 decode loader wants power-of-two pages
  fi::PlanInput a{shared_qo_indptr, shared_kv_indptr, shared_last_page_len, shared_batch, num_qo_heads, num_kv_heads,
                  head_dim, page_size, 0, ws->num_sms};
  fi::PlanInput b{qo_indptr, kv_indptr, last_page_len, batch, num_qo_heads, num_kv_heads, head_dim, page_size, causal,
                  ws->num_sms};
  int st = fi::validate_input(a);
  if (st == FI_OK) st = fi::validate_input(b);
  if (st != FI_OK) return st;
  const int64_t nnz_a = shared_kv_indptr[shared_batch], nnz_b = kv_indptr[batch];
  if (qo_indptr[batch] > ws->max_total_q || nnz_a > ws->max_kv_pages || nnz_b > ws->max_kv_pages)
    return FI_ERR_CAPACITY;
  if ((nnz_a > 0 && shared_kv_indices == nullptr) || (nnz_b > 0 && kv_indices == nullptr)) return FI_ERR_INVALID_ARG;
  int32_t max_page = -1;
  for (int64_t k = 0; k < nnz_a; ++k) {
    if (shared_kv_indices[k] < 0) return FI_ERR_INVALID_ARG;
    max_page = std::max(max_page, shared_kv_indices[k]);
  }
  for (int64_t k = 0; k < nnz_b; ++k) {
    if (kv_indices[k] < 0) return FI_ERR_INVALID_ARG;
    max_page = std::max(max_page, kv_indices[k]);
  }
  fi::ComposablePlan cp;
  st = fi::build_composable_plan(a, b, ws->cost, &cp);
  if (st != FI_OK) return st;
  const fi::Plan& pa = cp.shared;
  const fi::Plan& pb = cp.unique;
  if (pa.header[fi::H_NUM_ITEMS] > ws->max_items || pb.header[fi::H_NUM_ITEMS] > ws->max_items ||
      pb.header[fi::H_NUM_UNITS] > ws->max_units || pb.header[fi::H_NUM_SLOTS] > ws->max_slots ||
      int64_t(cp.ext.size() / 2) > ws->max_ext)
    return FI_ERR_CAPACITY;
  // the per-request units' own states wait for the merge past the used slots of the partial region
  if (int64_t(pb.header[fi::H_NUM_UNITS]) * fi::kDecodeMaxRows >
      (ws->max_slots - pb.header[fi::H_NUM_SLOTS]) * int64_t(fi::kTcRows))
    return FI_ERR_CAPACITY;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (ws->copy_pending) {
    FI_CUDA(cudaEventSynchronize(ws->copy_done));
    ws->copy_pending = false;
  }
  char* h = ws->hbuf;
  struct Seg {
    size_t off;
    const void* src;
    size_t bytes;
  } segs[] = {
      {ws->off_header, pb.header, sizeof(pb.header)},
      {ws->off_cta, pb.cta_indptr.data(), pb.cta_indptr.size() * sizeof(int32_t)},
      {ws->off_items, pb.items.data(), pb.items.size() * sizeof(int32_t)},
      {ws->off_units, pb.units.data(), pb.units.size() * sizeof(int32_t)},
      {ws->off_slot_unit, pb.slot_unit.data(), pb.slot_unit.size() * sizeof(int32_t)},
      {ws->off_kv, kv_indices, size_t(nnz_b) * sizeof(int32_t)},
      {ws->off_a_header, pa.header, sizeof(pa.header)},
      {ws->off_a_cta, pa.cta_indptr.data(), pa.cta_indptr.size() * sizeof(int32_t)},
      {ws->off_a_items, pa.items.data(), pa.items.size() * sizeof(int32_t)},
      {ws->off_a_kv, shared_kv_indices, size_t(nnz_a) * sizeof(int32_t)},
      {ws->off_ext, cp.ext.data(), cp.ext.size() * sizeof(int32_t)},
  };
  for (const Seg& sg : segs) {
    if (sg.bytes == 0) continue;
    std::memcpy(h + sg.off, sg.src, sg.bytes);
    FI_CUDA(cudaMemcpyAsync(ws->dbuf + sg.off, h + sg.off, sg.bytes, cudaMemcpyHostToDevice, s));
  }
  FI_CUDA(cudaEventRecord(ws->copy_done, s));
  ws->copy_pending = true;
  std::memcpy(ws->header, pb.header, sizeof(pb.header));
  ws->header[fi::H_PATH] = fi::kPathComposable;
  std::memcpy(ws->a_header, pa.header, sizeof(pa.header));
  ws->max_page = max_page;
  ws->plan_nnz = nnz_a + nnz_b;
  ws->plan_total_q = qo_indptr[batch];
  ws->has_plan = true;
  ws->composable = true;
  ws->plan_variant = ws->variant;
  return FI_OK;
}

int fi_run(fi_workspace* ws, const void* q, const void* k_pages, const void* v_pages, int num_pages, void* o,
           float* lse, void* stream) {
  return fi_run_merge(ws, q, k_pages, v_pages, num_pages, nullptr, nullptr, o, lse, stream);
}

int fi_run_merge(fi_workspace* ws, const void* q, const void* k_pages, const void* v_pages, int num_pages,
                 const void* o_prev, const float* lse_prev, void* o, float* lse, void* stream) {
  if (ws == nullptr) return FI_ERR_INVALID_ARG;
  if ((o_prev == nullptr) != (lse_prev == nullptr)) return FI_ERR_INVALID_ARG;
  if (!ws->has_plan) return FI_ERR_NO_PLAN;
  if (num_pages < 0 || ws->max_page >= num_pages) return FI_ERR_INVALID_ARG;
  const int32_t* h = ws->header;
  const bool any_rows = h[fi::H_NUM_ITEMS] > 0;
  if (any_rows && (q == nullptr || o == nullptr || lse == nullptr)) return FI_ERR_INVALID_ARG;
  if (ws->plan_nnz > 0 && (k_pages == nullptr || v_pages == nullptr)) return FI_ERR_INVALID_ARG;
  // q, K and V rows move in 16-byte copies (and TMA boxes on the tensor-core path)
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k_pages) | reinterpret_cast<uintptr_t>(v_pages)) & 15)
    return FI_ERR_INVALID_ARG;
  if (!any_rows) return FI_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int ps = h[fi::H_PAGE_SIZE];
  const float scale_log2 = fi::kLog2e / std::sqrt(float(ws->head_dim));
  char* d = ws->dbuf;

  if (ws->composable) {
    if (o_prev != nullptr) return FI_ERR_UNSUPPORTED;
    // 1: the shared sub-matrix on tensor-core tiles, every chunk to a slot (no contraction launch)
    const int32_t* ha = ws->a_header;
    if (ha[fi::H_NUM_ITEMS] > 0) {
      fi::PrefillArgs a{};
      a.cta_indptr = reinterpret_cast<const int32_t*>(d + ws->off_a_cta);
      a.items = reinterpret_cast<const int32_t*>(d + ws->off_a_items);
      a.units = reinterpret_cast<const int32_t*>(d + ws->off_units);
      a.slot_unit = reinterpret_cast<const int32_t*>(d + ws->off_slot_unit);
      a.kv_indices = reinterpret_cast<const int32_t*>(d + ws->off_a_kv);
      a.q = q;
      a.k = k_pages;
      a.v = v_pages;
      a.o = o;
      a.lse = lse;
      a.part_o = reinterpret_cast<float*>(d + ws->off_part_o);
      a.part_lse = reinterpret_cast<float*>(d + ws->off_part_lse);
      a.header = reinterpret_cast<const int32_t*>(d + ws->off_a_header);
      a.err = reinterpret_cast<int32_t*>(d + ws->off_err);
      a.num_pages = num_pages;
      a.page_size = ps;
      a.hqo = ws->hqo;
      a.hkv = ws->hkv;
      a.group = ha[fi::H_GROUP];
      a.tile_tokens = ha[fi::H_TILE_TOKENS];
      a.total_q = ws->plan_total_q;
      a.num_ctas = ha[fi::H_NUM_CTAS];
      a.scale_log2 = scale_log2;
      if (ws->plan_variant.kv_dtype == FI_KV_DTYPE_E4M3) {
        a.fp8 = 1;
        a.scale_log2 *= ws->plan_variant.k_scale;
        a.v_scale = ws->plan_variant.v_scale;
      }
      a.window_left = -1;
      a.cap_log2 = 0.f;
      a.nhd = 0;
      a.contract = 0;
      const int st = fi::launch_prefill(a, s);
      if (st != FI_OK) return st;
    }
    // 2: the per-request rows on decode tiles; each merges its own chunks and the shared slots
    fi::DecodeParams p{};
    p.cta_indptr = reinterpret_cast<const int32_t*>(d + ws->off_cta);
    p.items = reinterpret_cast<const int32_t*>(d + ws->off_items);
    p.units = reinterpret_cast<const int32_t*>(d + ws->off_units);
    p.slot_unit = reinterpret_cast<const int32_t*>(d + ws->off_slot_unit);
    p.kv_indices = reinterpret_cast<const int32_t*>(d + ws->off_kv);
    p.q = static_cast<const __nv_bfloat16*>(q);
    p.k = static_cast<const __nv_bfloat16*>(k_pages);
    p.v = static_cast<const __nv_bfloat16*>(v_pages);
    p.o = static_cast<__nv_bfloat16*>(o);
    p.lse = lse;
    p.part_o = reinterpret_cast<float*>(d + ws->off_part_o);
    p.part_lse = reinterpret_cast<float*>(d + ws->off_part_lse);
    p.ext = reinterpret_cast<const int2*>(d + ws->off_ext);
    // deferred own states: the partial region past the plan's slots (capacity checked at plan time)
    const size_t used_rows = size_t(h[fi::H_NUM_SLOTS]) * fi::kTcRows;
    p.def_o = reinterpret_cast<float*>(d + ws->off_part_o) + used_rows * fi::kHeadDim;
    p.def_lse = reinterpret_cast<float*>(d + ws->off_part_lse) + used_rows;
    p.counters = reinterpret_cast<uint32_t*>(d + ws->off_counters);
    p.err = reinterpret_cast<int32_t*>(d + ws->off_err);
    p.page_stride = (long long)ws->hkv * ps * fi::kHeadDim;
    p.head_stride = (long long)ps * fi::kHeadDim;
    p.window_left = -1;
    p.v_scale = 1.f;
    p.num_pages = num_pages;
    p.page_size = ps;
    p.page_shift = (ps & (ps - 1)) == 0 ? __builtin_ctz(unsigned(ps)) : -1;
    p.hqo = ws->hqo;
    p.group = h[fi::H_GROUP];
    p.slot_rows = fi::kTcRows;
    p.scale_log2 = scale_log2;
    if (ws->plan_variant.kv_dtype == FI_KV_DTYPE_E4M3) {
      // the FP8 decode kernel merges each row's shared slots as it finishes the row (no deferred
      // merges) and starts after the shared part's launch has completed (stream order)
      p.scale_log2 *= ws->plan_variant.k_scale;
      p.v_scale = ws->plan_variant.v_scale;
      return fi::launch_decode_fp8(h[fi::H_ROWS_TILE], false, h[fi::H_NUM_CTAS], p, s);
    }
    const bool pdl = ha[fi::H_NUM_ITEMS] > 0;
    // the per-request rows keep the 16-byte-copy loader: with the TMA copier the shared-prefix step
    // measured slower on GB300 (60.4 against 58.2 us), although plain decode batches were faster
    switch (h[fi::H_ROWS_TILE]) {
      case 1: return launch_decode<1>(h[fi::H_NUM_CTAS], p, s, false, pdl, false);
      case 2: return launch_decode<2>(h[fi::H_NUM_CTAS], p, s, false, pdl, false);
      case 4: return launch_decode<4>(h[fi::H_NUM_CTAS], p, s, false, pdl, false);
      case 8: return launch_decode<8>(h[fi::H_NUM_CTAS], p, s, false, pdl, false);
      default: return FI_ERR_UNSUPPORTED;
    }
  }

  if (h[fi::H_PATH] == fi::kPathDecode) {
    fi::DecodeParams p{};
    p.cta_indptr = reinterpret_cast<const int32_t*>(d + ws->off_cta);
    p.items = reinterpret_cast<const int32_t*>(d + ws->off_items);
    p.units = reinterpret_cast<const int32_t*>(d + ws->off_units);
    p.slot_unit = reinterpret_cast<const int32_t*>(d + ws->off_slot_unit);
    p.kv_indices = reinterpret_cast<const int32_t*>(d + ws->off_kv);
    p.q = static_cast<const __nv_bfloat16*>(q);
    p.k = static_cast<const __nv_bfloat16*>(k_pages);
    p.v = static_cast<const __nv_bfloat16*>(v_pages);
    p.o = static_cast<__nv_bfloat16*>(o);
    p.lse = lse;
    p.o_prev = static_cast<const __nv_bfloat16*>(o_prev);
    p.lse_prev = lse_prev;
    p.part_o = reinterpret_cast<float*>(d + ws->off_part_o);
    p.part_lse = reinterpret_cast<float*>(d + ws->off_part_lse);
    p.counters = reinterpret_cast<uint32_t*>(d + ws->off_counters);
    p.err = reinterpret_cast<int32_t*>(d + ws->off_err);
    const fi::Variant& var = ws->plan_variant;
    const bool nhd = var.kv_layout == FI_KV_LAYOUT_NHD;
    p.page_stride = (long long)ws->hkv * ps * fi::kHeadDim;
    p.head_stride = nhd ? fi::kHeadDim : (long long)ps * fi::kHeadDim;
    p.window_left = var.window_left;
    p.cap_log2 = var.soft_cap > 0.f ? var.soft_cap * fi::kLog2e : 0.f;
    p.inv_cap_log2 = var.soft_cap > 0.f ? 1.f / p.cap_log2 : 0.f;
    p.v_scale = 1.f;
    p.num_pages = num_pages;
    p.page_size = ps;
    p.page_shift = (ps & (ps - 1)) == 0 ? __builtin_ctz(unsigned(ps)) : -1;
    p.hqo = ws->hqo;
    p.group = h[fi::H_GROUP];
    p.slot_rows = fi::kTcRows;
    p.scale_log2 = scale_log2;
    // launched as a programmatic dependent: the CTAs set up their shared memory while the previous
    // kernel on the stream drains, then wait for it before the first global read
    p.wait_prior = 1;
    if (var.kv_dtype == FI_KV_DTYPE_E4M3) {  // every field above is set before this launch
      p.scale_log2 *= var.k_scale;           // logits of the stored codes, scaled back to K
      p.v_scale = var.v_scale;
      return fi::launch_decode_fp8(h[fi::H_ROWS_TILE], nhd, h[fi::H_NUM_CTAS], p, s, true);
    }
    const bool variant = var_on(var);
    if (nhd)
      return fi::launch_decode_nhd(h[fi::H_ROWS_TILE], __builtin_ctz(unsigned(ws->hkv)), h[fi::H_NUM_CTAS], p, s,
                                   true);
    switch (h[fi::H_ROWS_TILE]) {
      case 1: return launch_decode<1>(h[fi::H_NUM_CTAS], p, s, variant, true);
      case 2: return launch_decode<2>(h[fi::H_NUM_CTAS], p, s, variant, true);
      case 4: return launch_decode<4>(h[fi::H_NUM_CTAS], p, s, variant, true);
      case 8: return launch_decode<8>(h[fi::H_NUM_CTAS], p, s, variant, true);
      default: return FI_ERR_UNSUPPORTED;
    }
  }

  fi::PrefillArgs a{};
  a.cta_indptr = reinterpret_cast<const int32_t*>(d + ws->off_cta);
  a.items = reinterpret_cast<const int32_t*>(d + ws->off_items);
  a.units = reinterpret_cast<const int32_t*>(d + ws->off_units);
  a.slot_unit = reinterpret_cast<const int32_t*>(d + ws->off_slot_unit);
  a.kv_indices = reinterpret_cast<const int32_t*>(d + ws->off_kv);
  a.q = q;
  a.k = k_pages;
  a.v = v_pages;
  a.o = o;
  a.lse = lse;
  a.o_prev = o_prev;
  a.lse_prev = lse_prev;
  a.part_o = reinterpret_cast<float*>(d + ws->off_part_o);
  a.part_lse = reinterpret_cast<float*>(d + ws->off_part_lse);
  a.header = reinterpret_cast<const int32_t*>(d + ws->off_header);
  a.err = reinterpret_cast<int32_t*>(d + ws->off_err);
  a.num_pages = num_pages;
  a.page_size = ps;
  a.hqo = ws->hqo;
  a.hkv = ws->hkv;
  a.group = h[fi::H_GROUP];
  a.tile_tokens = h[fi::H_TILE_TOKENS];
  a.total_q = ws->plan_total_q;
  a.num_ctas = h[fi::H_NUM_CTAS];
  a.scale_log2 = scale_log2;
  a.window_left = ws->plan_variant.window_left;
  a.cap_log2 = ws->plan_variant.soft_cap > 0.f ? ws->plan_variant.soft_cap * fi::kLog2e : 0.f;
  a.nhd = ws->plan_variant.kv_layout == FI_KV_LAYOUT_NHD ? 1 : 0;
  if (ws->plan_variant.kv_dtype == FI_KV_DTYPE_E4M3) {
    a.fp8 = 1;
    a.scale_log2 *= ws->plan_variant.k_scale;  // logits of the stored codes, scaled back to K
    a.v_scale = ws->plan_variant.v_scale;
  }
  return fi::launch_prefill(a, s);
}

int fi_merge_states(const void* o_a, const float* lse_a, const void* o_b, const float* lse_b, void* o, float* lse,
                    int rows, int heads, int head_dim, void* stream) {
  if (rows < 0 || heads < 1) return FI_ERR_INVALID_ARG;
  if (head_dim != fi::kHeadDim) return FI_ERR_UNSUPPORTED;
  if (rows == 0) return FI_OK;
  if (!o_a || !lse_a || !o_b || !lse_b || !o || !lse) return FI_ERR_INVALID_ARG;
  const long long n = (long long)rows * heads;
  int blocks = int(std::min<long long>((n + 7) / 8, 4096));
  fi::merge_states_kernel<<<blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const __nv_bfloat16*>(o_a), lse_a, static_cast<const __nv_bfloat16*>(o_b), lse_b,
      static_cast<__nv_bfloat16*>(o), lse, n);
  FI_CUDA(cudaGetLastError());
  return FI_OK;
}

int fi_get_error(fi_workspace* ws, int32_t* err_bits) {
  if (ws == nullptr || err_bits == nullptr) return FI_ERR_INVALID_ARG;
  FI_CUDA(cudaDeviceSynchronize());
  int32_t* d = reinterpret_cast<int32_t*>(ws->dbuf + ws->off_err);
  FI_CUDA(cudaMemcpy(err_bits, d, sizeof(int32_t), cudaMemcpyDeviceToHost));
  FI_CUDA(cudaMemset(d, 0, sizeof(int32_t)));
  FI_CUDA(cudaDeviceSynchronize());
  return FI_OK;
}

int fi_plan_info(const fi_workspace* ws, int32_t* header16) {
  if (ws == nullptr || header16 == nullptr) return FI_ERR_INVALID_ARG;
  if (!ws->has_plan) return FI_ERR_NO_PLAN;
  std::memcpy(header16, ws->header, sizeof(ws->header));
  return FI_OK;
}

}  // extern "C"
