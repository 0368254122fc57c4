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
//     shared-memory attribute.
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
// The first 256 bytes of the array hold the device-side error word (FI_DEVERR_* bits).  Calls only
// add bits to it; fi_decode_noalloc_get_error reads and clears it.  The plan follows at this offset.
constexpr size_t kErrBytes = 256;

// Scratch of every call: error word, plan segments, page-index copy, split counters, partial slots.
// A file-scope __device__ array starts zeroed when the module loads.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Host-side storage of the planner's work arrays and of the staged plan (static: no heap use).
static int32_t g_work[kMaxItems * fi::kItemFields];
static int64_t g_cost[kMaxItems];
static int32_t g_order[kMaxItems];
static int32_t g_cta_of[kMaxItems];
static int32_t g_count[kMaxCtas];
static std::pair<int64_t, int32_t> g_heap[kMaxCtas];
static uint64_t g_key[kMaxItems > kMaxCtas ? kMaxItems : kMaxCtas];
static unsigned char g_stage[kNoAllocScratchBytes];
static std::mutex g_mutex;

static void* g_dev_scratch[kMaxDevices];
static bool g_dev_ready[kMaxDevices];

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// Byte offsets of the segments inside the array.
struct Layout {
  size_t header, cta, items, units, slot_unit, kv, counters, part_lse, part_o, end;
};

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

  // the same planner as fi_plan (default cost model), in two passes over static storage
  const fi::CostModel cm;
  fi::PlanShape shape;
  st = fi::plan_shape(in, cm, &shape);
  if (st != FI_OK) return st;
  if (shape.path != fi::kPathDecode) return FI_ERR_UNSUPPORTED;  // some request has more than 8 rows
  if (shape.n_items > kMaxItems || shape.num_ctas > kMaxCtas) return FI_ERR_CAPACITY;
  const int64_t W = shape.n_items, U = shape.n_units, S = shape.n_slots;

  Layout L;
  size_t off = kErrBytes;
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
  L.part_lse = seg(sizeof(float) * size_t(S) * kNaSlotRows);
  L.part_o = seg(sizeof(float) * size_t(S) * kNaSlotRows * fi::kHeadDim);
  L.end = off;
  if (L.end > kNoAllocScratchBytes) return FI_ERR_CAPACITY;
  if (W > 0 && (q == nullptr || o == nullptr || lse == nullptr)) return FI_ERR_INVALID_ARG;
  if (nnz > 0 && (k_pages == nullptr || v_pages == nullptr)) return FI_ERR_INVALID_ARG;
  // the kernel moves q, K and V rows with 16-byte copies
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k_pages) | reinterpret_cast<uintptr_t>(v_pages)) & 15)
    return FI_ERR_INVALID_ARG;

  void* scratch = nullptr;
  st = device_setup(dev, &scratch);
  if (st != FI_OK) return st;
  if (W == 0) return FI_OK;

  // plan straight into the staging copy of the array: header | per-CTA queues | split rows |
  // slot -> split row | page ids
  unsigned char* h = g_stage;
  int32_t header[fi::kHeaderLen];
  fi::PlanStorage ps{reinterpret_cast<int32_t*>(h + L.cta), reinterpret_cast<int32_t*>(h + L.items),
                     reinterpret_cast<int32_t*>(h + L.units), reinterpret_cast<int32_t*>(h + L.slot_unit),
                     nullptr, g_work, g_cost, g_order, g_cta_of, g_count, g_heap, g_key};
  fi::plan_fill(in, cm, shape, ps, header);
  std::memcpy(h + L.header, header, sizeof(header));
  if (nnz) std::memcpy(h + L.kv, kv_indices, sizeof(int32_t) * size_t(nnz));

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned char* d = static_cast<unsigned char*>(scratch);
  // the array keeps the previous call's contents: the split counters must start at zero (the error
  // word before the plan is left alone: it collects bits until fi_decode_noalloc_get_error)
  if (cudaMemcpyAsync(d + L.header, h + L.header, staged - L.header, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return FI_ERR_CUDA;
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
  p.err = reinterpret_cast<int32_t*>(d);  // the error word at the start of the array
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

// Read and clear the error word of the array on the current device.  Synchronises the device (a
// kernel still running would add bits after the read).  No allocation: symbol copies only.
extern "C" int fi_decode_noalloc_get_error(int32_t* err_bits) {
  if (err_bits == nullptr) return FI_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_mutex);
  const int32_t zero = 0;
  if (cudaDeviceSynchronize() != cudaSuccess) return FI_ERR_CUDA;
  if (cudaMemcpyFromSymbol(err_bits, g_noalloc_scratch, sizeof(int32_t), 0, cudaMemcpyDeviceToHost) != cudaSuccess)
    return FI_ERR_CUDA;
  if (cudaMemcpyToSymbol(g_noalloc_scratch, &zero, sizeof(int32_t), 0, cudaMemcpyHostToDevice) != cudaSuccess)
    return FI_ERR_CUDA;
  return cudaDeviceSynchronize() == cudaSuccess ? FI_OK : FI_ERR_CUDA;
}
