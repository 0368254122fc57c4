// fi_decode_noalloc: the CUDA-core decode path with no allocation at all.
//
// Who needs it: callers that may not allocate device memory themselves or let
// a library do it -- serving runtimes that reserve the whole GPU for their own
// memory pool up front, plugin hosts whose allocator the library must not
// touch, or code paths that run with allocation forbidden.  They still own q,
// the KV pages, o and lse; everything else this call needs (the plan, the copy
// of the page indices, the split-row counters and the partial-output slots)
// lives in one file-scope device array of fixed size, and the host-side plan
// is built in static host storage.  No cudaMalloc / cudaFree / cudaHostAlloc
// and no heap allocation happens on this path.
//
// Contract (also stated in include/fi.h):
//   * the device array is kNoAllocScratchBytes (4 MiB) long and every GPU that
//     loads the library holds it until the process exits;
//   * a batch whose plan, page indices and partial slots do not fit is
//     rejected with FI_ERR_CAPACITY; a batch whose tiles need the tensor-core
//     path is rejected with FI_ERR_UNSUPPORTED;
//   * every call shares the array and the host staging storage: calls that
//     overlap on the GPU (e.g. on two streams) race, and concurrent host calls
//     are serialised by a mutex;
//   * the first call on a device looks up the array's device address
//     (cudaGetSymbolAddress, with that device current) and sets the kernel's
//     shared-memory attribute; make that first call before any stream capture.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <functional>
#include <mutex>
#include <utility>

#include "../../include/fi.h"
#include "decode_kernel.cuh"
#include "plan.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(FI_NOALLOC_SCRATCH_BYTES);
constexpr int kMaxDevices = 64;
constexpr int kMaxCtas = 1024;
constexpr int kNaWarps = 8;
constexpr int kNaStages = 8;
constexpr int kNaSlotRows = fi::kDecodeMaxRows;  // decode tiles have at most 8 rows
// An item takes at least kItemFields int32 in the scratch, which bounds the item count.
constexpr int64_t kMaxItems = int64_t(kNoAllocScratchBytes / (sizeof(int32_t) * fi::kItemFields));

// Scratch of every call: plan segments, page-index copy, split counters, error word, partial slots.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Host-side storage of the plan builder and of the staged plan (static: no heap use).
struct HostWork {
  int32_t f[fi::kItemFields];
  int64_t cost;
};
static HostWork g_work[kMaxItems];
static int32_t g_order[kMaxItems];
static int32_t g_cta_of[kMaxItems];
static int32_t g_count[kMaxCtas];
static std::pair<int64_t, int32_t> g_heap[kMaxCtas];
static unsigned char g_stage[kNoAllocScratchBytes];
static std::mutex g_mutex;

static void* g_dev_scratch[kMaxDevices];
static bool g_dev_ready[kMaxDevices];

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// Same rules as fi::build_plan (decode path only), written into static storage.
// Returns an fi_status; fills header / queues into the staging layout below.
struct Layout {
  size_t header, cta, items, units, slot_unit, kv, counters, err, part_lse, part_o, end;
};

int plan_static(const fi::PlanInput& in, int32_t* header, int64_t* n_items_out, int64_t* n_units_out,
                int64_t* n_slots_out, int32_t** units_out, int32_t* slot_unit_tmp, int64_t slot_cap,
                int32_t* units_tmp, int64_t unit_cap) {
  const int B = in.batch;
  const int g = in.num_qo_heads / in.num_kv_heads;
  const int ps = in.page_size;
  int64_t max_lq = 0;
  for (int i = 0; i < B; ++i) max_lq = std::max<int64_t>(max_lq, in.qo_indptr[i + 1] - in.qo_indptr[i]);
  if (max_lq * g > fi::kDecodeMaxRows) return FI_ERR_UNSUPPORTED;
  const int tile_tokens = static_cast<int>(std::max<int64_t>(1, max_lq));
  int rows_tile = 1;
  while (rows_tile < tile_tokens * g) rows_tile *= 2;

  auto lkv_of = [&](int i) -> int64_t {
    const int64_t n_p = in.kv_indptr[i + 1] - in.kv_indptr[i];
    return n_p > 0 ? (n_p - 1) * ps + in.last_page_len[i] : 0;
  };
  int64_t total = 0;
  for (int i = 0; i < B; ++i) {
    const int64_t lq = in.qo_indptr[i + 1] - in.qo_indptr[i];
    total += int64_t(in.num_kv_heads) * ((lq + tile_tokens - 1) / tile_tokens) * lkv_of(i);
  }
  const fi::CostModel cm;  // default cost model (alpha = beta = 1, l_min = 256)
  int64_t l_chunk = std::max<int64_t>((total + in.num_sms - 1) / in.num_sms, cm.l_min);
  l_chunk = (l_chunk + ps - 1) / ps * ps;

  int64_t W = 0, U = 0, S = 0;
  for (int i = 0; i < B; ++i) {
    const int64_t lq = in.qo_indptr[i + 1] - in.qo_indptr[i];
    const int64_t lkv = lkv_of(i);
    const int64_t n_tiles = (lq + tile_tokens - 1) / tile_tokens;
    for (int h = 0; h < in.num_kv_heads; ++h) {
      for (int64_t j = 0; j < n_tiles; ++j) {
        const int64_t q0 = j * tile_tokens, qn = std::min<int64_t>(tile_tokens, lq - q0);
        int64_t e, diag;
        if (in.causal) {
          e = std::min(std::max<int64_t>(lkv - lq + q0 + qn, 0), lkv);
          diag = lkv - lq + q0;
        } else {
          e = lkv;
          diag = fi::kNotCausalDiag;
        }
        int64_t n = 1, cs = 0;
        if (e > 0) {
          n = (e + l_chunk - 1) / l_chunk;
          cs = ((e + n - 1) / n + ps - 1) / ps * ps;
          n = (e + cs - 1) / cs;
        }
        int32_t first_slot = -1;
        if (n > 1) {
          if (U + 1 > unit_cap || S + n > slot_cap) return FI_ERR_CAPACITY;
          first_slot = static_cast<int32_t>(S);
          int32_t* u = units_tmp + U * fi::kUnitFields;
          u[0] = first_slot;
          u[1] = static_cast<int32_t>(n);
          u[2] = in.qo_indptr[i] + static_cast<int32_t>(q0);
          u[3] = static_cast<int32_t>(qn);
          u[4] = h;
          u[5] = u[6] = u[7] = 0;
          for (int64_t c = 0; c < n; ++c) slot_unit_tmp[S + c] = static_cast<int32_t>(U);
          ++U;
          S += n;
        }
        for (int64_t c = 0; c < n; ++c) {
          if (W >= kMaxItems) return FI_ERR_CAPACITY;
          const int64_t lo = c * cs, hi = std::min(e, (c + 1) * cs);
          HostWork& w = g_work[W];
          w.f[fi::I_PAGE_BASE] = in.kv_indptr[i];
          w.f[fi::I_Q_START] = in.qo_indptr[i] + static_cast<int32_t>(q0);
          w.f[fi::I_Q_LEN] = static_cast<int32_t>(qn);
          w.f[fi::I_KV_HEAD] = h;
          w.f[fi::I_KV_LO] = static_cast<int32_t>(lo);
          w.f[fi::I_KV_HI] = static_cast<int32_t>(hi);
          w.f[fi::I_DIAG] = static_cast<int32_t>(diag);
          w.f[fi::I_SLOT] = first_slot >= 0 ? first_slot + static_cast<int32_t>(c) : -1;
          w.cost = cm.alpha * qn * g + cm.beta * (hi - lo);
          g_order[W] = static_cast<int32_t>(W);
          ++W;
        }
      }
    }
  }
  // longest first, ties by enumeration order; then a min-heap of (load, cta id)
  std::sort(g_order, g_order + W, [](int32_t a, int32_t b) {
    return g_work[a].cost > g_work[b].cost || (g_work[a].cost == g_work[b].cost && a < b);
  });
  const int C = in.num_sms;  // decode path: one CTA per SM
  for (int c = 0; c < C; ++c) {
    g_heap[c] = {0, c};
    g_count[c] = 0;
  }
  std::greater<std::pair<int64_t, int32_t>> cmp;
  std::make_heap(g_heap, g_heap + C, cmp);
  for (int64_t k = 0; k < W; ++k) {
    const int32_t it = g_order[k];
    std::pop_heap(g_heap, g_heap + C, cmp);
    auto& top = g_heap[C - 1];
    g_cta_of[it] = top.second;
    g_count[top.second] += 1;
    top.first += g_work[it].cost;
    std::push_heap(g_heap, g_heap + C, cmp);
  }
  header[fi::H_MAGIC] = fi::kPlanMagic;
  header[fi::H_PATH] = fi::kPathDecode;
  header[fi::H_TILE_TOKENS] = tile_tokens;
  header[fi::H_ROWS_TILE] = rows_tile;
  header[fi::H_GROUP] = g;
  header[fi::H_NUM_CTAS] = C;
  header[fi::H_NUM_ITEMS] = static_cast<int32_t>(W);
  header[fi::H_NUM_UNITS] = static_cast<int32_t>(U);
  header[fi::H_NUM_SLOTS] = static_cast<int32_t>(S);
  header[fi::H_LKV] = static_cast<int32_t>(l_chunk);
  header[fi::H_PAGE_SIZE] = ps;
  header[fi::H_CAUSAL] = in.causal;
  header[fi::H_HQO] = in.num_qo_heads;
  header[fi::H_HKV] = in.num_kv_heads;
  header[fi::H_HEAD_DIM] = in.head_dim;
  header[fi::H_BATCH] = B;
  *n_items_out = W;
  *n_units_out = U;
  *n_slots_out = S;
  *units_out = units_tmp;
  return FI_OK;
}

// Once per device, with that device current: device address of the scratch array
// and the decode kernels' shared-memory attribute.
int device_setup(int dev, void** scratch) {
  if (dev < 0 || dev >= kMaxDevices) return FI_ERR_UNSUPPORTED;
  if (!g_dev_ready[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) return FI_ERR_CUDA;
    const cudaError_t e1 = cudaFuncSetAttribute(fi::decode_kernel<1, kNaWarps, kNaStages>,
                                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                int(sizeof(fi::DecodeSmem<1, kNaWarps, kNaStages>)));
    const cudaError_t e2 = cudaFuncSetAttribute(fi::decode_kernel<2, kNaWarps, kNaStages>,
                                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                int(sizeof(fi::DecodeSmem<2, kNaWarps, kNaStages>)));
    const cudaError_t e4 = cudaFuncSetAttribute(fi::decode_kernel<4, kNaWarps, kNaStages>,
                                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                int(sizeof(fi::DecodeSmem<4, kNaWarps, kNaStages>)));
    const cudaError_t e8 = cudaFuncSetAttribute(fi::decode_kernel<8, kNaWarps, kNaStages>,
                                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                int(sizeof(fi::DecodeSmem<8, kNaWarps, kNaStages>)));
    if (e1 != cudaSuccess || e2 != cudaSuccess || e4 != cudaSuccess || e8 != cudaSuccess) return FI_ERR_CUDA;
    g_dev_scratch[dev] = ptr;
    g_dev_ready[dev] = true;
  }
  *scratch = g_dev_scratch[dev];
  return FI_OK;
}

template <int R>
cudaError_t launch(const fi::DecodeParams& p, int grid, cudaStream_t s) {
  fi::decode_kernel<R, kNaWarps, kNaStages>
      <<<grid, (kNaWarps + 1) * 32, sizeof(fi::DecodeSmem<R, kNaWarps, kNaStages>), s>>>(p);
  return cudaGetLastError();
}

}  // namespace

extern "C" int fi_decode_noalloc(const int32_t* qo_indptr, const int32_t* kv_indptr, const int32_t* kv_indices,
                                 const int32_t* last_page_len, int batch, int num_qo_heads, int num_kv_heads,
                                 int head_dim, int page_size, int causal, const void* q, const void* k_pages,
                                 const void* v_pages, int num_pages, void* o, float* lse, void* stream) {
  std::lock_guard<std::mutex> lock(g_mutex);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FI_ERR_CUDA;
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return FI_ERR_CUDA;
  const int num_ctas = std::min(sms, kMaxCtas);
  fi::PlanInput in{qo_indptr, kv_indptr, last_page_len, batch, num_qo_heads, num_kv_heads, head_dim, page_size,
                   causal, num_ctas};
  int st = fi::validate_input(in);
  if (st != FI_OK) return st;
  const int64_t nnz = kv_indptr[batch];
  if (nnz > 0 && kv_indices == nullptr) return FI_ERR_INVALID_ARG;
  int32_t max_page = -1;
  for (int64_t k = 0; k < nnz; ++k) {
    if (kv_indices[k] < 0) return FI_ERR_INVALID_ARG;
    max_page = std::max(max_page, kv_indices[k]);
  }
  if (num_pages < 0 || max_page >= num_pages) return FI_ERR_INVALID_ARG;

  // Partial slots and split rows are bounded by 2 * #CTA and #CTA (App. D.3 bound).
  const int64_t slot_cap = 2 * int64_t(num_ctas), unit_cap = num_ctas;
  static int32_t units_tmp[kMaxCtas * fi::kUnitFields];
  static int32_t slot_unit_tmp[2 * kMaxCtas];
  int32_t header[fi::kHeaderLen];
  int64_t W = 0, U = 0, S = 0;
  int32_t* units = nullptr;
  st = plan_static(in, header, &W, &U, &S, &units, slot_unit_tmp, slot_cap, units_tmp, unit_cap);
  if (st != FI_OK) return st;

  Layout L;
  size_t off = 0;
  auto seg = [&](size_t bytes) {
    const size_t o = off;
    off = align256(off + bytes);
    return o;
  };
  L.header = seg(sizeof(int32_t) * fi::kHeaderLen);
  L.cta = seg(sizeof(int32_t) * (num_ctas + 1));
  L.items = seg(sizeof(int32_t) * fi::kItemFields * size_t(W));
  L.units = seg(sizeof(int32_t) * fi::kUnitFields * size_t(U));
  L.slot_unit = seg(sizeof(int32_t) * size_t(S));
  L.kv = seg(sizeof(int32_t) * size_t(nnz));
  const size_t staged = off;
  L.counters = seg(sizeof(uint32_t) * size_t(std::max<int64_t>(U, 1)));
  L.err = seg(sizeof(int32_t) * 4);
  L.part_lse = seg(sizeof(float) * size_t(S) * kNaSlotRows);
  L.part_o = seg(sizeof(float) * size_t(S) * kNaSlotRows * fi::kHeadDim);
  L.end = off;
  if (L.end > kNoAllocScratchBytes) return FI_ERR_CAPACITY;
  if (W > 0 && (q == nullptr || o == nullptr || lse == nullptr)) return FI_ERR_INVALID_ARG;
  if (nnz > 0 && (k_pages == nullptr || v_pages == nullptr)) return FI_ERR_INVALID_ARG;

  void* scratch = nullptr;
  st = device_setup(dev, &scratch);
  if (st != FI_OK) return st;
  if (W == 0) return FI_OK;

  // stage the plan: header | per-CTA queues | split rows | slot -> split row | page ids
  unsigned char* h = g_stage;
  std::memcpy(h + L.header, header, sizeof(header));
  int32_t* cta = reinterpret_cast<int32_t*>(h + L.cta);
  cta[0] = 0;
  for (int c = 0; c < num_ctas; ++c) cta[c + 1] = cta[c] + g_count[c];
  int32_t* items = reinterpret_cast<int32_t*>(h + L.items);
  for (int c = 0; c < num_ctas; ++c) g_count[c] = cta[c];  // reuse as fill cursors
  for (int64_t k = 0; k < W; ++k) {
    const int32_t it = g_order[k];
    const int32_t pos = g_count[g_cta_of[it]]++;
    std::memcpy(items + size_t(pos) * fi::kItemFields, g_work[it].f, sizeof(g_work[it].f));
  }
  if (U) std::memcpy(h + L.units, units, sizeof(int32_t) * fi::kUnitFields * size_t(U));
  if (S) std::memcpy(h + L.slot_unit, slot_unit_tmp, sizeof(int32_t) * size_t(S));
  if (nnz) std::memcpy(h + L.kv, kv_indices, sizeof(int32_t) * size_t(nnz));

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned char* d = static_cast<unsigned char*>(scratch);
  // the array keeps the previous call's contents: counters and the error word must start at zero
  if (cudaMemcpyAsync(d, h, staged, cudaMemcpyHostToDevice, s) != cudaSuccess) return FI_ERR_CUDA;
  if (cudaMemsetAsync(d + L.counters, 0, L.part_lse - L.counters, s) != cudaSuccess) return FI_ERR_CUDA;

  fi::DecodeParams p{};  // value-initialised: optional fields (o_prev, lse_prev) stay null
  p.cta_indptr = reinterpret_cast<const int32_t*>(d + L.cta);
  p.items = reinterpret_cast<const int32_t*>(d + L.items);
  p.units = reinterpret_cast<const int32_t*>(d + L.units);
  p.slot_unit = reinterpret_cast<const int32_t*>(d + L.slot_unit);
  p.kv_indices = reinterpret_cast<const int32_t*>(d + L.kv);
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.k = static_cast<const __nv_bfloat16*>(k_pages);
  p.v = static_cast<const __nv_bfloat16*>(v_pages);
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.part_o = reinterpret_cast<float*>(d + L.part_o);
  p.part_lse = reinterpret_cast<float*>(d + L.part_lse);
  p.counters = reinterpret_cast<uint32_t*>(d + L.counters);
  p.err = reinterpret_cast<int32_t*>(d + L.err);
  p.page_stride = (long long)num_kv_heads * page_size * fi::kHeadDim;
  p.head_stride = (long long)page_size * fi::kHeadDim;
  p.window_left = -1;  // no window, no soft-cap (cap_log2 = 0)
  p.num_pages = num_pages;
  p.page_size = page_size;
  p.hqo = num_qo_heads;
  p.group = header[fi::H_GROUP];
  p.slot_rows = kNaSlotRows;
  p.scale_log2 = fi::kLog2e / std::sqrt(float(head_dim));
  cudaError_t e;
  switch (header[fi::H_ROWS_TILE]) {
    case 1: e = launch<1>(p, num_ctas, s); break;
    case 2: e = launch<2>(p, num_ctas, s); break;
    case 4: e = launch<4>(p, num_ctas, s); break;
    case 8: e = launch<8>(p, num_ctas, s); break;
    default: return FI_ERR_UNSUPPORTED;
  }
  return e == cudaSuccess ? FI_OK : FI_ERR_CUDA;
}
