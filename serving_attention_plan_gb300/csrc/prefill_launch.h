// Launch interface of the tensor-core (tcgen05) tile path.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace fi {

struct PrefillArgs {
  const int32_t* cta_indptr;
  const int32_t* items;
  const int32_t* units;
  const int32_t* slot_unit;
  const int32_t* kv_indices;
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  const void* o_prev;      // optional: state of the same rows over a disjoint key set, merged in
  const float* lse_prev;
  float* part_o;
  float* part_lse;
  const int32_t* header;  // the plan's header in device memory
  int32_t* err;
  int num_pages;
  int page_size;
  int hqo;
  int hkv;
  int group;
  int tile_tokens;
  int total_q;   // rows of q / o (capacity of the workspace)
  int num_ctas;
  float scale_log2;  // with e4m3 pages: times k_scale
  float v_scale = 1.f;  // e4m3 pages: V = v_scale * code
  int fp8 = 0;          // K and V pages hold e4m3 codes
  int window_left;  // < 0: none
  float cap_log2;   // <= 0: no soft-cap; else cap * log2(e)
  int nhd;          // page layout NHD instead of HND
  int contract = 1; // 0: no contraction kernel (a composable plan's shared part: its slots are merged
                    // by the per-request decode launch)
};

// Returns an fi_status.
int launch_prefill(const PrefillArgs& a, cudaStream_t stream);

// Records the text of a failed CUDA call for fi_last_error_message; returns FI_ERR_CUDA.
int record_cuda_error(cudaError_t e, const char* what);

// Tensor map of e4m3 K or V pages for the FP8 decode kernel's TMA copier: one box is box_rows
// (the copier's min(page_size, stage tokens)) rows of 128 codes of one page and KV head, 128-byte
// swizzled.  HND pages [pages][H_kv][page_size][128] map as (code, token in page, page * H_kv +
// head), NHD pages [pages][page_size][H_kv][128] as (code, head, token in page, page).  Returns
// false if the driver's encoder is missing or refuses the map.
bool make_decode_map_e4m3(CUtensorMap* m, const void* base, int hkv, int page_size, int num_pages, bool nhd,
                          int box_rows);

// Tensor map of bf16 HND K or V pages [pages][H_kv][page_size][128] for the decode kernel's TMA
// copier: (dim, token in page, page * H_kv + head), one box 64 dims x box_rows tokens (the copier's
// min(page_size, stage tokens)), 128-byte swizzled.  Returns false if the driver's encoder is
// missing or refuses the map.
bool make_decode_map_bf16(CUtensorMap* m, const void* base, int hkv, int page_size, int num_pages, int box_rows);

}  // namespace fi
