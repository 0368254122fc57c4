// Tensor-core tile path: paged-KV attention for 256-row work items on tcgen05, with the merge of
// split-KV partial states.
//
// Page "FlashInfer：面向 LLM 推理服务的高效可定制注意力引擎":
//   核心机制 3-4 (paper §3.2, §3.2.2): query tiles of >= 16 rows run on tensor
//     cores; scattered KV tiles are gathered into contiguous shared memory
//     first.  Here the gather is done by TMA: each page of a 128-key tile is one
//     3-D tensor box (page-head, token in page, dim) landing in a 128-byte
//     swizzled shared-memory tile (the TMA sparse gather the paper leaves as
//     future work, 核心机制 8 / App. B).  GQA heads fold into the rows
//     (术语与记号 "GQA 头组融合", App. A): a tile is 128/g tokens x g heads.
//   实验与指标 (paper §4.2): causal prefill with the mask aligned to the end of
//     each request's KV.
//   核心机制 6-7 (paper §3.3.1, App. D): persistent CTAs walk the plan's queues
//     and write the partial states of split rows to workspace slots; the
//     contraction follows in a second kernel chained by programmatic dependent
//     launch, so its launch overlaps the attention tail and every SM shares it,
//     each row summing its chunks in the plan's slot order.  (A 256-row partial
//     state is 128 KB.  Merged by the last chunk's CTA alone, as the decode kernel
//     does with its <= 8-row states, a 128-row state cut into 19 chunks took
//     ~70 us with the earlier 128-row design; an in-kernel grid barrier would need
//     a cooperative launch, which the driver refused for that two-CTA-per-SM grid.)
//
// One CTA per SM (all 512 TMEM columns, ~200 KB of shared memory), 16 warps = 4 warpgroups.
// A work item is 256 rows (256/g tokens x g heads) as two 128-row MMA tiles, Q0 (rows 0-127)
// and Q1 (rows 128-255), that share every KV tile: each 128-key K and V tile is fetched once for
// 256 query rows, which halves the L2 traffic and the TMA box count per flop.
//   warps 0-3       softmax of Q0: thread t owns row t (TMEM lane t)
//   warps 4-7       softmax of Q1
//   warps 8-11      epilogue: O / l and LSE of both halves of a finished item, to the output or
//                   a partial slot
//   warp 12         TMA producer of K (two stages) and of each item's Q tile
//   warp 13         TMA producer of V (two stages)
//   warp 14         TMEM allocation and issue of S_h = Q_h K^T (one thread)
//   warp 15         issue of O_h += P_h V (one thread)
// The MMAs work on 64-key sub-tiles of each 128-key K/V tile.  TMEM: two score buffers per half,
// S_h,0 and S_h,1 (64 fp32 columns each, columns 0-255), and O0, O1 (256-511).  The softmax of half
// h overwrites the first 32 columns of a sub-tile's S buffer with its P (bf16 pairs), the A operand
// of O_h += P_h V, so P.V reads only V from shared memory.  With two S buffers per half, the QK of
// sub-tile u + 1 waits only for the P.V of u - 1, so it runs while the softmax works on u, and the
// two halves' MMAs fill each other's gaps.  QK and P.V come from two issuing threads, so neither's
// waits stall the other; O is handed to the epilogue as soon as the item's last P.V of that half
// completes.
// Online softmax in base 2 with a lazy rescale: O and l are rescaled only when a row's running
// maximum grows by more than 8 (a factor 256), which keeps exp2 arguments <= 8 and changes the
// result only by rounding.
// FP8 (e4m3) KV pages (核心机制 8, paper App. F: the KV-cache in fp8, queries and outputs in 16-bit
// floats): each page's code rows land by TMA, unswizzled, in the second 64-dim half of the stage;
// the producer warp then widens them in place to f16 in the layout above (one conversion per two
// codes, exact) and releases the stage to the MMA with a second barrier.  The MMAs then run on f16
// operands: the two producer warps convert each item's Q tile from bf16 to f16 in place once it has
// landed, and the softmax writes P as f16.  K = k_scale * code is folded into the logit scale and
// V = v_scale * code into the epilogue's 1 / l.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "../../include/fi.h"
#include "device_common.cuh"
#include "plan.h"
#include "prefill_launch.h"
#include "tcgen05.cuh"

namespace fi {
namespace {

constexpr int kTile = 128;                  // rows of an MMA tile (one half of an item), keys of a KV tile
constexpr int kHalfBytes = kTile * 128;     // one 64-dim half of a 128-row bf16 tile (16 KB)
constexpr int kTileBytes = 2 * kHalfBytes;  // full 128 x 128 bf16 tile
constexpr int kItemRows = 2 * kTile;        // rows of a work item (kTcRows)
constexpr int kQHalfBytes = kItemRows * 128;  // one 64-dim half of the item's Q (32 KB)
constexpr int kThreads = 512;
// Register split after launch (512 threads x 128): the two softmax warpgroups take 176 each (a
// row of 128 scores in registers), the epilogue warpgroup 104 (it streams O out 32 columns at a
// time), the producer/MMA warpgroup 56: 128 * (176 + 176 + 104 + 56) = 65536 = 512 * 128.
constexpr uint32_t kSoftmaxRegs = 176;
constexpr uint32_t kEpilogueRegs = 104;
constexpr uint32_t kControlRegs = 56;
constexpr uint32_t kTmemCols = 512;
constexpr int kSub = 64;           // keys of an MMA sub-tile (two per K/V tile)
constexpr uint32_t kColS = 0;      // S_h,b at columns 128 h + 64 b
constexpr uint32_t kColO = 256;    // O_h at columns 256 + 128 h
constexpr int kKvStages = 2;       // K and V shared-memory stages each
constexpr float kRescaleThreshold = 8.0f;
constexpr unsigned kFull = 0xffffffffu;
static_assert(kItemRows == kTcRows, "a tensor-core work item is two 128-row MMA tiles");

struct PrefillParams {
  const int32_t* cta_indptr;
  const int32_t* items;
  const int32_t* units;
  const int32_t* slot_unit;
  const int32_t* kv_indices;
  __nv_bfloat16* o;
  float* lse;
  const __nv_bfloat16* o_prev;  // optional state of the same rows over other keys, merged into o / lse
  const float* lse_prev;
  float* part_o;
  float* part_lse;
  int32_t* err;
  int num_pages;
  int page_size;
  int hqo;
  int hkv;
  int group;
  int slot_rows;
  uint32_t q_tile_bytes;  // bytes of one Q tile as TMA writes it (2 halves x rows x 128 B)
  float scale_log2;  // includes k_scale with e4m3 pages
  float v_scale;     // 1 for bf16 pages
  int window_left;   // >= 0: a row at key position p sees keys p - window_left .. p
  float cap_log2;    // > 0: logit soft-cap in the log2 domain, s -> cap_log2 * tanh(s / cap_log2)
  // 1: launched as a programmatic dependent of the previous kernel on the stream: the CTA sets up
  // its barriers and tensor memory, then waits for that kernel before any global read
  int wait_prior;
};

struct PrefillSmem {
  uint8_t q[2 * kQHalfBytes];        // item Q: [2 dim halves][256 rows][128 B], 128B-swizzled
  uint8_t k[kKvStages][kTileBytes];  // [stage][2 dim halves][128 keys][128 B]
  uint8_t v[kKvStages][kTileBytes];
  float stat_m[2][kItemRows];        // [item parity][row]: running max at the end of the item
  float stat_l[2][kItemRows];        // [item parity][row]: row sum
  uint64_t q_full, q_empty, k_full[kKvStages], k_empty[kKvStages], v_full[kKvStages], v_empty[kKvStages];
  uint64_t k_ready[kKvStages], v_ready[kKvStages];     // e4m3 pages: the stage widened to f16
  uint64_t q_ready;                                    // e4m3 pages: the item's Q converted to f16
  uint64_t s_full[2][2], p_full[2][2], pv_done[2][2];  // [half][S buffer]
  uint64_t o_free[2];                                   // per half of the item
  uint64_t stat_full[2], stat_empty[2];                  // per item parity
  uint32_t tmem_base;
  int abort;
};

struct Item {
  int page_base, q_start, q_len, kv_head, kv_lo, kv_hi, diag, slot;
  __device__ __forceinline__ void load(const int32_t* items, int pos) {
    const int4 a = __ldg(reinterpret_cast<const int4*>(items + size_t(pos) * kItemFields));
    const int4 b = __ldg(reinterpret_cast<const int4*>(items + size_t(pos) * kItemFields + 4));
    page_base = a.x;
    q_start = a.y;
    q_len = a.z;
    kv_head = a.w;
    kv_lo = b.x;
    kv_hi = b.y;
    diag = b.z;
    slot = b.w;
  }
  __device__ __forceinline__ int tiles() const { return (kv_hi - kv_lo + kTile - 1) / kTile; }
  __device__ __forceinline__ int subs() const { return (kv_hi - kv_lo + kSub - 1) / kSub; }
};

// ---------------------------------------------------------------------------------------------
// warps 12 (K and the item's Q) and 13 (V): TMA producers
// ---------------------------------------------------------------------------------------------
// Two e4m3 codes (bits 0-15) -> f16x2 (code of bits 0-7 in the low half), exactly.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_codes) {
  uint32_t h;
  const uint16_t v = static_cast<uint16_t>(two_codes);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(v));
  return h;
}

// Two floats -> f16x2 (lo in the low half), round to nearest even.
__device__ __forceinline__ uint32_t f2_to_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// e4m3 pages: the stage's 128 keys x 128 codes arrived as 128-byte rows in its second 64-dim half;
// rewrite them as f16 in the MMA layout [2 dim halves][128 keys][128 B] (16-byte chunk c of row r
// at position c ^ (r % 8)).  Eight lanes take one row, one 16-byte chunk of codes each, so each
// shared-memory phase reads one whole row without bank conflicts; a row is read whole before any
// lane writes, and writes go only to that row's place in each half (the second half's row is the
// staged row itself), so rows never overlap.
__device__ __forceinline__ void widen_stage(uint8_t* stage, int lane) {
  const int c = lane & 7;  // staged chunk: dims 16c .. 16c + 15
  const uint32_t base = smem_u32(stage);
  const uint32_t half_off = uint32_t(c >> 2) * kHalfBytes;
  const int m = (2 * c) & 7;  // output chunks m, m + 1 of that half
#pragma unroll 4
  for (int i = 0; i < kTile / 4; ++i) {
    const int r = 4 * i + (lane >> 3);
    uint32_t w0, w1, w2, w3;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(w0), "=r"(w1), "=r"(w2), "=r"(w3)
                 : "r"(base + kHalfBytes + uint32_t(r * 128 + 16 * c))
                 : "memory");
    __syncwarp();
    const uint32_t row = base + half_off + uint32_t(r * 128);
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(row + uint32_t(((m ^ (r & 7)) << 4))),
                 "r"(e4m3x2_to_f16x2(w0)), "r"(e4m3x2_to_f16x2(w0 >> 16)), "r"(e4m3x2_to_f16x2(w1)),
                 "r"(e4m3x2_to_f16x2(w1 >> 16))
                 : "memory");
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(row + uint32_t((((m + 1) ^ (r & 7)) << 4))),
                 "r"(e4m3x2_to_f16x2(w2)), "r"(e4m3x2_to_f16x2(w2 >> 16)), "r"(e4m3x2_to_f16x2(w3)),
                 "r"(e4m3x2_to_f16x2(w3 >> 16))
                 : "memory");
    __syncwarp();
  }
}

// e4m3 pages: rows 128 h .. 128 h + 127 of the item's Q (both 64-dim halves), bf16 -> f16 in place
// (element positions unchanged, so the swizzle is unchanged).  A bf16 value is exactly a float
// whose low 16 bits are zero; f16 keeps it exactly within f16's normal range.
__device__ __forceinline__ void q_to_f16(uint8_t* q, int h, int lane) {
#pragma unroll 1
  for (int kh = 0; kh < 2; ++kh) {
    const uint32_t base = smem_u32(q + kh * kQHalfBytes + h * kHalfBytes);
#pragma unroll 4
    for (int i = lane; i < kHalfBytes / 16; i += 32) {
      uint32_t w[4];
      asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                   : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                   : "r"(base + uint32_t(16 * i))
                   : "memory");
#pragma unroll
      for (int j = 0; j < 4; ++j)
        w[j] = f2_to_f16x2(__uint_as_float(w[j] << 16), __uint_as_float(w[j] & 0xFFFF0000u));
      asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(base + uint32_t(16 * i)), "r"(w[0]), "r"(w[1]),
                   "r"(w[2]), "r"(w[3])
                   : "memory");
    }
  }
}

template <bool kNhd, bool kIsK, bool kFp8>
__device__ void producer(const PrefillParams& p, PrefillSmem& sm, const CUtensorMap* tm_q, const CUtensorMap* tm_kv,
                         int begin, int end) {
  const int lane = threadIdx.x & 31;
  const int ps = p.page_size;
  const int ppt = kTile / ps;  // pages per KV tile (<= 16)
  const int oob_page = p.num_pages * p.hkv;
  uint8_t* ring = kIsK ? &sm.k[0][0] : &sm.v[0][0];
  uint64_t* full = kIsK ? sm.k_full : sm.v_full;
  uint64_t* empty = kIsK ? sm.k_empty : sm.v_empty;
  uint64_t* ready = kIsK ? sm.k_ready : sm.v_ready;
  int tt = 0, nq = 0;  // KV tiles and Q tiles issued
  int nw = 0;          // e4m3: tiles widened (one behind the loads, so a load is in flight while widening)
  int nqc = 0;         // e4m3: Q tiles converted
  bool ok = true;
  // e4m3: once item nqc's Q has landed, convert this warp's half of its rows to f16 (K warp rows
  // 0-127, V warp rows 128-255) for the f16 MMAs
  auto convert_q = [&]() {
    ok = __all_sync(kFull, mbar_wait(&sm.q_full, nqc & 1, p.err, &sm.abort));
    if (!ok) return;
    q_to_f16(sm.q, kIsK ? 0 : 1, lane);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.q_ready);
    ++nqc;
  };
  // e4m3: wait for tile nw's codes, widen them, hand the stage to the MMA issuer
  auto widen_next = [&]() {
    const int st = nw % kKvStages;
    ok = __all_sync(kFull, mbar_wait(&full[st], (nw / kKvStages) & 1, p.err, &sm.abort));
    if (!ok) return;
    widen_stage(ring + st * kTileBytes, lane);
    fence_proxy_async_smem();  // the MMAs read the widened tile through the async proxy
    __syncwarp();
    if (lane == 0) mbar_arrive(&ready[st]);
    ++nw;
  };
  for (int pos = begin; pos < end && ok; ++pos) {
    Item it;
    it.load(p.items, pos);
    const int n_tiles = it.tiles();
    if (n_tiles == 0) continue;
    for (int t = 0; t < n_tiles && ok; ++t) {
      const int base = it.kv_lo + t * kTile;
      // out-of-range page(-head) coordinate: the box reads as zeros
      int z = kNhd ? p.num_pages : oob_page;
      if (lane < ppt) {
        const int pp = base / ps + lane;
        if (pp * ps < it.kv_hi) {
          const int page = __ldg(p.kv_indices + it.page_base + pp);
          if (page >= 0 && page < p.num_pages) {
            z = kNhd ? page : page * p.hkv + it.kv_head;
          } else {
            atomicOr(p.err, FI_DEVERR_PAGE_OOB);
          }
        }
      }
      // e4m3: widen the previous tile before waiting for this one's stage, so the widening
      // overlaps the MMAs of the tile before it (issuing this tile's load first, when its stage is
      // already free, measured slower)
      if constexpr (kFp8) {
        if (nw < tt) widen_next();
        if (!ok) break;
      }
      const int st = tt % kKvStages;
      if (tt >= kKvStages)
        ok = __all_sync(kFull, mbar_wait(&empty[st], ((tt / kKvStages) - 1) & 1, p.err, &sm.abort));
      if (!ok) break;
      if (lane == 0) mbar_arrive_expect_tx(&full[st], kFp8 ? kTileBytes / 2 : kTileBytes);
      __syncwarp();
      if (lane < ppt) {
        uint8_t* dst = ring + st * kTileBytes + lane * ps * 128;
        if constexpr (kFp8) {
          // one page of one KV head, 128 codes a row, into the second half (unswizzled)
          if constexpr (kNhd)
            tc::tma_load_4d(dst + kHalfBytes, tm_kv, 0, it.kv_head, 0, z, &full[st]);
          else
            tc::tma_load_3d(dst + kHalfBytes, tm_kv, 0, 0, z, &full[st]);
        } else if constexpr (kNhd) {
          // one page of one KV head: HND box (64 dims, page_size tokens, 1 page-head), NHD box
          // (64 dims, 1 head, page_size tokens, 1 page)
          tc::tma_load_4d(dst, tm_kv, 0, it.kv_head, 0, z, &full[st]);
          tc::tma_load_4d(dst + kHalfBytes, tm_kv, 64, it.kv_head, 0, z, &full[st]);
        } else {
          tc::tma_load_3d(dst, tm_kv, 0, 0, z, &full[st]);
          tc::tma_load_3d(dst + kHalfBytes, tm_kv, 64, 0, z, &full[st]);
        }
      }
      ++tt;
      if constexpr (kIsK) {
        // the item's Q, after its first K tile (so that load is not held up behind the wait for
        // the previous item's last QK to free the Q buffer)
        if (t == 0) {
          if (nq >= 1) ok = __all_sync(kFull, mbar_wait(&sm.q_empty, (nq - 1) & 1, p.err, &sm.abort));
          if (!ok) break;
          if (lane == 0) {
            mbar_arrive_expect_tx(&sm.q_full, p.q_tile_bytes);
            tc::tma_load_3d(sm.q, tm_q, 0, it.kv_head * p.group, it.q_start, &sm.q_full);
            tc::tma_load_3d(sm.q + kQHalfBytes, tm_q, 64, it.kv_head * p.group, it.q_start, &sm.q_full);
          }
          ++nq;
          if constexpr (kFp8) convert_q();
          if (!ok) break;
        }
      } else if constexpr (kFp8) {
        if (t == 0) convert_q();
        if (!ok) break;
      }
    }
  }
  if constexpr (kFp8) {
    while (ok && nw < tt) widen_next();
  }
  // never leave with tensor copies still landing in this CTA's shared memory
  if constexpr (kIsK) {
    if (nq > 0) mbar_wait_bounded(&sm.q_full, (nq - 1) & 1);
  }
  for (int k = max(0, tt - kKvStages); k < tt; ++k) mbar_wait_bounded(&full[k % kKvStages], (k / kKvStages) & 1);
}

// ---------------------------------------------------------------------------------------------
// MMA issue, two threads: warp 14 issues S_h = Q_h K^T, warp 15 issues O_h += P_h V.  Every
// dependency between them goes through a barrier (S_h free = the half's last P.V done; P_h ready
// = the softmax's arrivals), so each thread's waits overlap the other's issue.
// ---------------------------------------------------------------------------------------------
template <bool kFp8>
__device__ void qk_issuer(const PrefillParams& p, PrefillSmem& sm, uint32_t tmem, int begin, int end) {
  uint64_t* k_in = kFp8 ? sm.k_ready : sm.k_full;  // e4m3: the widened stage
  uint64_t* q_in = kFp8 ? &sm.q_ready : &sm.q_full;  // e4m3: Q converted to f16
  // A = Q_h (K-major), B = K rows (K-major); f16 operands with e4m3 pages
  constexpr uint32_t idesc_qk = kFp8 ? tc::idesc_f16_f32(kTile, kSub, 0, 0) : tc::idesc_bf16_f32(kTile, kSub, 0, 0);
  const uint32_t q_addr = smem_u32(sm.q), k_addr = smem_u32(sm.k[0]);
  int tt = 0, uu = 0, nq = 0;  // K/V tiles, sub-tiles, items
  for (int pos = begin; pos < end; ++pos) {
    Item it;
    it.load(p.items, pos);
    const int n_tiles = it.tiles(), n_sub = it.subs();
    if (n_tiles == 0) continue;
    if (!mbar_wait(q_in, nq & 1, p.err, &sm.abort)) return;
    for (int t = 0; t < n_tiles; ++t, ++tt) {
      const int ks_ = tt % kKvStages;
      if (!mbar_wait(&k_in[ks_], (tt / kKvStages) & 1, p.err, &sm.abort)) return;
      for (int sub = 0; sub < 2 && 2 * t + sub < n_sub; ++sub, ++uu) {
        const int b = uu & 1;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          // S_h,b last held P_h(uu - 2): its P.V must have completed
          if (uu >= 2 && !mbar_wait(&sm.pv_done[h][b], ((uu >> 1) - 1) & 1, p.err, &sm.abort)) return;
          tc::fence_after_sync();
#pragma unroll
          for (int kh = 0; kh < 2; ++kh) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              // K-major, 128B swizzle: a 16-element k step is 32 B inside the 128-B row; 8-row
              // groups 1024 B apart; Q_h is rows 128 h .. of the item's Q, the sub-tile's keys are
              // rows 64 sub .. of the K tile
              const uint64_t a = tc::smem_desc(q_addr + kh * kQHalfBytes + h * kHalfBytes + kk * 32, 16, 1024,
                                               tc::kLayoutSw128);
              const uint64_t bd = tc::smem_desc(k_addr + ks_ * kTileBytes + kh * kHalfBytes + sub * (kSub * 128) + kk * 32,
                                                16, 1024, tc::kLayoutSw128);
              tc::mma_ss(tmem + kColS + uint32_t(h * kTile + b * kSub), a, bd, idesc_qk, (kh | kk) != 0 ? 1u : 0u);
            }
          }
          tc::commit(&sm.s_full[h][b]);
        }
      }
      tc::commit(&sm.k_empty[ks_]);
      if (t == n_tiles - 1) tc::commit(&sm.q_empty);
    }
    ++nq;
  }
}

template <bool kFp8>
__device__ void pv_issuer(const PrefillParams& p, PrefillSmem& sm, uint32_t tmem, int begin, int end) {
  uint64_t* v_in = kFp8 ? sm.v_ready : sm.v_full;
  // A = P_h (TMEM), B = V (MN-major); f16 operands with e4m3 pages
  constexpr uint32_t idesc_pv = kFp8 ? tc::idesc_f16_f32(kTile, kTile, 0, 1) : tc::idesc_bf16_f32(kTile, kTile, 0, 1);
  const uint32_t v_addr = smem_u32(sm.v[0]);
  int tt = 0, uu = 0, nq = 0;
  for (int pos = begin; pos < end; ++pos) {
    Item it;
    it.load(p.items, pos);
    const int n_tiles = it.tiles(), n_sub = it.subs();
    if (n_tiles == 0) continue;
    for (int t = 0; t < n_tiles; ++t, ++tt) {
      const int vs = tt % kKvStages;
      if (!mbar_wait(&v_in[vs], (tt / kKvStages) & 1, p.err, &sm.abort)) return;
      if (t == n_tiles - 1) {
        // The item's last page may hold slots past its last key: the page box brought them in, and
        // a NaN there would survive its zero weight in P.V.  Clear those V rows (the rest of the
        // tile past that page came in as zeros).
        const int base = it.kv_lo + t * kTile;
        const int r0 = it.kv_hi - base;
        const int r1 = min(kTile, (it.kv_hi + p.page_size - 1) / p.page_size * p.page_size - base);
        if (r0 < r1) {
          uint8_t* st = sm.v[vs];
          for (int r = r0; r < r1; ++r) {
#pragma unroll
            for (int c = 0; c < 16; ++c)
              *reinterpret_cast<uint4*>(st + (c >> 3) * kHalfBytes + r * 128 + (c & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();  // the MMAs read the stage through the async proxy
        }
      }
      for (int sub = 0; sub < 2 && 2 * t + sub < n_sub; ++sub, ++uu) {
        const int b = uu & 1;
        const bool first = t == 0 && sub == 0;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (!mbar_wait(&sm.p_full[h][b], (uu >> 1) & 1, p.err, &sm.abort)) return;
          // the item's first P.V overwrites O_h once the epilogue has read the previous item's O_h out
          if (first && nq > 0 && !mbar_wait(&sm.o_free[h], (nq - 1) & 1, p.err, &sm.abort)) return;
          tc::fence_after_sync();
#pragma unroll
          for (int ks = 0; ks < kSub / 16; ++ks) {
            // V as B (K = keys, N = dims), MN-major 128B swizzle: a 16-key step is two 8-row groups
            // (2048 B); the second 64-dim half is the leading-dimension step (16 KB)
            const uint64_t bd = tc::smem_desc(v_addr + vs * kTileBytes + sub * (kSub * 128) + ks * 2048, kHalfBytes,
                                              1024, tc::kLayoutSw128);
            tc::mma_ts(tmem + kColO + uint32_t(h * kTile), tmem + kColS + uint32_t(h * kTile + b * kSub) + ks * 8, bd,
                       idesc_pv, (!first || ks > 0) ? 1u : 0u);
          }
          tc::commit(&sm.pv_done[h][b]);
        }
      }
      tc::commit(&sm.v_empty[vs]);
    }
    ++nq;
  }
}

// ---------------------------------------------------------------------------------------------
// warps 0-7: softmax of the two halves; warps 8-11: epilogue and the output of an item
// ---------------------------------------------------------------------------------------------

// Output row of (token, head) for item row `row`.
__device__ __forceinline__ size_t out_row(const PrefillParams& p, const Item& it, int row) {
  return (size_t)(it.q_start + row / p.group) * p.hqo + it.kv_head * p.group + row % p.group;
}

// 32 output values -> bf16 at dst (32 consecutive dims).
__device__ __forceinline__ void store_bf16_32(__nv_bfloat16* dst_ptr, const float (&v)[32]) {
  uint4* dst = reinterpret_cast<uint4*>(dst_ptr);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 w;
    w.x = f2_to_bf16x2(v[8 * q + 0], v[8 * q + 1]);
    w.y = f2_to_bf16x2(v[8 * q + 2], v[8 * q + 3]);
    w.z = f2_to_bf16x2(v[8 * q + 4], v[8 * q + 5]);
    w.w = f2_to_bf16x2(v[8 * q + 6], v[8 * q + 7]);
    dst[q] = w;
  }
}

__device__ __forceinline__ float lse_out(float lse2) { return (lse2 == -INFINITY) ? -INFINITY : lse2 * kLn2; }

// Hardware tanh (relative error about 2^-11, so a capped logit is within about 7e-4 * cap): one
// instruction per score, where the exp2-based tanh would double the softmax's per-score work.
__device__ __forceinline__ float tanh_fast(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// One 64-key sub-tile of half h: scores -> (soft-cap) -> mask keys outside [lo, lim) -> online
// softmax update -> P into the first 32 columns of the sub-tile's S buffer.
template <bool kMasked, bool kCap, bool kF16>
__device__ __forceinline__ void softmax_sub(const uint32_t t_s, const uint32_t t_o, int lo, int lim, float scale,
                                            float& m, float& l, bool first, PrefillSmem& sm, uint64_t* pv_done,
                                            int pv_parity, const PrefillParams& p, bool& alive) {
  uint32_t s[kSub];
  tc::tmem_ld32(t_s + 0, *reinterpret_cast<uint32_t(*)[32]>(s + 0));
  tc::tmem_ld32(t_s + 32, *reinterpret_cast<uint32_t(*)[32]>(s + 32));
  tc::tmem_wait_ld();
  if (kCap) {
    // capped logits in the log2 domain; the scale is then already applied
    const float in_scale = scale / p.cap_log2;
#pragma unroll
    for (int j = 0; j < kSub; ++j) s[j] = __float_as_uint(p.cap_log2 * tanh_fast(__uint_as_float(s[j]) * in_scale));
    scale = 1.f;
  }
  // row maximum of the (scaled) scores with 8 independent partial maxima
  float mx8[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) mx8[j] = -INFINITY;
#pragma unroll
  for (int j = 0; j < kSub; ++j) {
    if (kMasked) s[j] = (j < lim && j >= lo) ? s[j] : __float_as_uint(-INFINITY);
    mx8[j & 7] = fmaxf(mx8[j & 7], __uint_as_float(s[j]));
  }
  const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                         fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
  const float m_new = fmaxf(m, mx * scale);  // scale > 0: max of scaled = scaled max
  float alpha = 1.f;
  bool need = false;
  if (first) {
    m = m_new;
  } else {
    need = m_new > m + kRescaleThreshold;  // also true when m = -inf and m_new is finite
    if (need) {
      alpha = fast_exp2(m - m_new);
      l *= alpha;
      m = m_new;
    }
  }
  const float m_use = (m == -INFINITY) ? 0.f : m;
  // p = 2^(s * scale - m): one packed FMA per pair, then ex2; 4 packed partial sums
  const float2 sc2 = make_float2(scale, scale), nm2 = make_float2(-m_use, -m_use);
  float2 sum4[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) sum4[j] = make_float2(0.f, 0.f);
#pragma unroll
  for (int j = 0; j < kSub / 2; ++j) {
    const float2 x = __ffma2_rn(make_float2(__uint_as_float(s[2 * j]), __uint_as_float(s[2 * j + 1])), sc2, nm2);
    const float2 pp = make_float2(fast_exp2(x.x), fast_exp2(x.y));
    sum4[j & 3] = __fadd2_rn(sum4[j & 3], pp);
    s[j] = kF16 ? f2_to_f16x2(pp.x, pp.y) : f2_to_bf16x2(pp.x, pp.y);  // P overwrites the front of S in place
  }
  const float2 s01 = __fadd2_rn(sum4[0], sum4[1]), s23 = __fadd2_rn(sum4[2], sum4[3]);
  const float2 s0123 = __fadd2_rn(s01, s23);
  l += s0123.x + s0123.y;
  tc::tmem_st32(t_s + 0, *reinterpret_cast<uint32_t(*)[32]>(s + 0));
  tc::tmem_wait_st();
  if (__any_sync(kFull, need)) {
    // O_h was last written by the previous sub-tile's P.V: wait for it, then rescale in place
    alive = alive && __all_sync(kFull, mbar_wait(pv_done, pv_parity, p.err, &sm.abort));
    tc::fence_after_sync();
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t o[32];
      tc::tmem_ld32(t_o + 32 * c, o);
      tc::tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
      tc::tmem_st32(t_o + 32 * c, o);
    }
    tc::tmem_wait_st();
  }
}

// Softmax warpgroup of half h (rows 128 h .. 128 h + 127 of each item).
template <bool kWin, bool kCap, bool kF16>
__device__ void softmax_group(const PrefillParams& p, PrefillSmem& sm, uint32_t tmem, int begin, int end, int h) {
  const int r = threadIdx.x & (kTile - 1);  // == TMEM lane
  const int row = h * kTile + r;             // row of the item
  const int lane = threadIdx.x & 31;
  const uint32_t lane_base = tmem + (uint32_t((r >> 5) * 32) << 16);
  const uint32_t t_o = lane_base + kColO + uint32_t(h * kTile);
  const float scale = p.scale_log2;
  int uu = 0, nit = 0;
  bool alive = true;
  for (int pos = begin; pos < end; ++pos, ++nit) {
    Item it;
    it.load(p.items, pos);
    const int n_sub = it.subs();
    const int u = row / p.group;
    float m = -INFINITY, l = 0.f;
    for (int t = 0; t < n_sub; ++t, ++uu) {
      const int b = uu & 1;
      const uint32_t t_s = lane_base + kColS + uint32_t(h * kTile + b * kSub);
      const int base = it.kv_lo + t * kSub;
      const int lim = max(0, min(kSub, min(it.kv_hi - base, it.diag + u + 1 - base)));
      // sliding window: keys below diag + u - window_left are masked
      const int lo = kWin ? min(kSub, max(0, it.diag + u - p.window_left - base)) : 0;
      alive = alive && __all_sync(kFull, mbar_wait(&sm.s_full[h][b], (uu >> 1) & 1, p.err, &sm.abort));
      if (alive) {
        tc::fence_after_sync();
        // the P.V that last wrote O_h: sub-tile uu - 1, in the other S buffer
        uint64_t* prev_pv = &sm.pv_done[h][b ^ 1];
        const int prev_parity = ((uu - 1) >> 1) & 1;
        if (__all_sync(kFull, lim >= kSub && lo <= 0))
          softmax_sub<false, kCap, kF16>(t_s, t_o, lo, lim, scale, m, l, t == 0, sm, prev_pv, prev_parity, p, alive);
        else
          softmax_sub<true, kCap, kF16>(t_s, t_o, lo, lim, scale, m, l, t == 0, sm, prev_pv, prev_parity, p, alive);
        tc::fence_before_sync();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.p_full[h][b]);
    }
    // the item's statistics for the epilogue
    const int ib = nit & 1;
    if (nit >= 2)
      alive = alive && __all_sync(kFull, mbar_wait(&sm.stat_empty[ib], ((nit >> 1) - 1) & 1, p.err, &sm.abort));
    sm.stat_m[ib][row] = m;
    sm.stat_l[ib][row] = l;
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.stat_full[ib]);
  }
}

// Epilogue group: for each item and each half, O / l and LSE to the output (merged with a given
// state) or to the item's partial slot.
__device__ void epilogue_group(const PrefillParams& p, PrefillSmem& sm, uint32_t tmem, int begin, int end) {
  const int r = threadIdx.x & (kTile - 1);  // == TMEM lane
  const int lane = threadIdx.x & 31;
  const uint32_t lane_base = tmem + (uint32_t((r >> 5) * 32) << 16);
  int tt = 0, nit = 0;
  bool alive = true;
  for (int pos = begin; pos < end; ++pos, ++nit) {
    Item it;
    it.load(p.items, pos);
    const int n_tiles = it.subs();  // sub-tiles
    const int rows_valid = it.q_len * p.group;
    const int ib = nit & 1;
    alive = alive && __all_sync(kFull, mbar_wait(&sm.stat_full[ib], (nit >> 1) & 1, p.err, &sm.abort));
    float m2[2], l2[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      m2[h] = sm.stat_m[ib][h * kTile + r];
      l2[h] = sm.stat_l[ib][h * kTile + r];
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.stat_empty[ib]);
    const int last = tt + n_tiles - 1;
    tt += n_tiles;
#pragma unroll 1
    for (int h = 0; h < 2; ++h) {
      const int row = h * kTile + r;
      float lse2 = -INFINITY, inv = 0.f;
      if (l2[h] > 0.f) {
        lse2 = m2[h] + fast_log2(l2[h]);
        inv = p.v_scale / l2[h];  // V = v_scale * code with e4m3 pages
      }
      const bool live = n_tiles > 0;
      if (live) alive = alive && __all_sync(kFull, mbar_wait(&sm.pv_done[h][last & 1], (last >> 1) & 1, p.err, &sm.abort));
      tc::fence_after_sync();
      // weights of this state (unnormalised O) and of the given one, and the output's LSE
      float wa = inv, wb = 0.f;
      size_t orow = 0;
      const bool write = row < rows_valid;
      if (write && it.slot < 0) {
        orow = out_row(p, it, row);
        if (p.o_prev) {
          const float p2 = p.lse_prev[orow] * kLog2e;
          const float mm = fmaxf(lse2, p2);
          if (mm == -INFINITY) {
            wa = 0.f;
          } else {
            const float a = fast_exp2(lse2 - mm), b = fast_exp2(p2 - mm);
            wa = a * inv / (a + b);
            wb = b / (a + b);
            lse2 = mm + fast_log2(a + b);
          }
        }
      }
      const uint32_t t_o = lane_base + kColO + uint32_t(h * kTile);
      // O_h streamed out 32 columns at a time
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t o[32];
        if (live && alive) {
          tc::tmem_ld32(t_o + 32 * c, o);
          tc::tmem_wait_ld();
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) o[j] = 0u;
        }
        if (!write) continue;
        if (it.slot < 0) {
          float v[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(o[j]) * wa;
          if (wb != 0.f) {
            const uint4* src = reinterpret_cast<const uint4*>(p.o_prev + orow * kHeadDim + 32 * c);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              const uint4 raw = src[q4];
              const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
              for (int hh = 0; hh < 4; ++hh) {
                const float2 f = bf16x2_to_f2(w4[hh]);
                v[8 * q4 + 2 * hh] += wb * f.x;
                v[8 * q4 + 2 * hh + 1] += wb * f.y;
              }
            }
          }
          store_bf16_32(p.o + orow * kHeadDim + 32 * c, v);
        } else {
          const size_t srow = (size_t)it.slot * p.slot_rows + row;
          float4* dst = reinterpret_cast<float4*>(p.part_o + srow * kHeadDim + 32 * c);
#pragma unroll
          for (int j = 0; j < 8; ++j)
            dst[j] = make_float4(__uint_as_float(o[4 * j]) * inv, __uint_as_float(o[4 * j + 1]) * inv,
                                 __uint_as_float(o[4 * j + 2]) * inv, __uint_as_float(o[4 * j + 3]) * inv);
        }
      }
      if (live) {
        // O_h has been read: the next item's first P.V may overwrite it
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.o_free[h]);
      }
      if (write) {
        if (it.slot < 0)
          p.lse[orow] = lse_out(lse2);
        else
          p.part_lse[(size_t)it.slot * p.slot_rows + row] = lse2;
      }
    }
  }
}

template <bool kWin, bool kCap, bool kNhd, bool kFp8>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ PrefillParams p, const __grid_constant__ CUtensorMap tm_q,
                   const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v) {
  extern __shared__ unsigned char smem_raw[];
  // 128B-swizzled tiles want 1024-byte alignment
  PrefillSmem& sm = *reinterpret_cast<PrefillSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(&sm.q_full, 1);
    mbar_init(&sm.q_empty, 1);
    mbar_init(&sm.q_ready, 2);  // one arrival per producer warp
    for (int b = 0; b < kKvStages; ++b) {
      mbar_init(&sm.k_full[b], 1);
      mbar_init(&sm.k_empty[b], 1);
      mbar_init(&sm.v_full[b], 1);
      mbar_init(&sm.v_empty[b], 1);
      mbar_init(&sm.k_ready[b], 1);
      mbar_init(&sm.v_ready[b], 1);
    }
    for (int h = 0; h < 2; ++h) {
      for (int b = 0; b < 2; ++b) {
        mbar_init(&sm.s_full[h][b], 1);
        mbar_init(&sm.p_full[h][b], 4);  // one arrival per warp of the half's softmax group
        mbar_init(&sm.pv_done[h][b], 1);
      }
      mbar_init(&sm.o_free[h], 4);      // one arrival per epilogue warp
      mbar_init(&sm.stat_full[h], 8);   // one arrival per softmax warp (both groups)
      mbar_init(&sm.stat_empty[h], 4);  // one arrival per epilogue warp
    }
    sm.abort = 0;
    fence_mbar_init();
  }
  if (warp == 12 && (threadIdx.x & 31) == 0) {
    tc::tma_prefetch_desc(&tm_q);
    tc::tma_prefetch_desc(&tm_k);
    tc::tma_prefetch_desc(&tm_v);
  }
  if (warp == 14) {
    tc::tmem_alloc(&sm.tmem_base, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (p.wait_prior) asm volatile("griddepcontrol.wait;" ::: "memory");
  // the launch that follows (the contraction, or the next kernel) may be scheduled from here on; it
  // waits for this grid to complete before it reads anything this grid writes.  Triggered after the
  // wait above, so a follower can never run ahead of the kernel before this one.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const uint32_t tmem = sm.tmem_base;
  const int begin = __ldg(p.cta_indptr + blockIdx.x);
  const int end = __ldg(p.cta_indptr + blockIdx.x + 1);
  if ((tmem & 0xFFFFu) + kTmemCols > 512u) {  // not an address this CTA can use: report, do nothing
    if (threadIdx.x == 0) atomicOr(p.err, FI_DEVERR_TMEM);
  } else if (warp < 8) {
    tc::regs_increase<kSoftmaxRegs>();
    softmax_group<kWin, kCap, kFp8>(p, sm, tmem, begin, end, warp >> 2);
  } else if (warp < 12) {
    static_assert(kEpilogueRegs < 128 && kControlRegs < 128 && kSoftmaxRegs > 128,
                  "setmaxnreg.inc only raises and setmaxnreg.dec only lowers the launch count (128)");
    tc::regs_decrease<kEpilogueRegs>();
    epilogue_group(p, sm, tmem, begin, end);
  } else {
    tc::regs_decrease<kControlRegs>();
    if (warp == 12) {
      producer<kNhd, true, kFp8>(p, sm, &tm_q, &tm_k, begin, end);
    } else if (warp == 13) {
      producer<kNhd, false, kFp8>(p, sm, &tm_q, &tm_v, begin, end);
    } else if (warp == 14 && (threadIdx.x & 31) == 0) {
      qk_issuer<kFp8>(p, sm, tmem, begin, end);
    } else if (warp == 15 && (threadIdx.x & 31) == 0) {
      pv_issuer<kFp8>(p, sm, tmem, begin, end);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 14) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------------------------
// contraction of split rows: a second kernel, chained by programmatic dependent launch
// ---------------------------------------------------------------------------------------------
// One warp per (unit, tile row); lane l owns dims 4l..4l+3, so each load of a partial row is one
// coalesced 512-byte access.  A row's chunks are summed in slot (plan) order with up to
// kContractUnroll loads in flight: the result does not depend on which warp runs the task, so
// reruns are bit-identical.  The number of split units is read from the plan in device memory,
// so a captured launch follows later plans.
struct ContractParams {
  const int32_t* header;
  const int32_t* units;
  const float* part_o;
  const float* part_lse;
  __nv_bfloat16* o;
  float* lse;
  const __nv_bfloat16* o_prev;
  const float* lse_prev;
  int hqo;
  int group;
  int slot_rows;
};

constexpr int kContractThreads = 256;
constexpr int kContractUnroll = 8;

__global__ void __launch_bounds__(kContractThreads) contract_kernel(const __grid_constant__ ContractParams p) {
  // the attention grid has completed and its partial states are visible after this
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // the next launch on the stream may start its set-up (it waits for this grid before reading)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const int n_warps = gridDim.x * (kContractThreads / 32);
  const int tasks = __ldg(p.header + H_NUM_UNITS) * kTcRows;
  for (int t = blockIdx.x * (kContractThreads / 32) + (threadIdx.x >> 5); t < tasks; t += n_warps) {
    const int unit = t / kTcRows, row = t % kTcRows;
    const int4 u = __ldg(reinterpret_cast<const int4*>(p.units + unit * kUnitFields));
    const int first = u.x, n = u.y, q_start = u.z;
    if (row >= u.w * p.group) continue;  // rows of the tile beyond its query tokens
    const int kv_head = __ldg(p.units + unit * kUnitFields + U_KV_HEAD);
    const float* lse_col = p.part_lse + (size_t)first * p.slot_rows + row;
    float mx = -INFINITY;
    for (int c = lane; c < n; c += 32) mx = fmaxf(mx, __ldcg(lse_col + (size_t)c * p.slot_rows));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const float m_use = (mx == -INFINITY) ? 0.f : mx;
    float sum = 0.f;
    for (int c = lane; c < n; c += 32) sum += fast_exp2(__ldcg(lse_col + (size_t)c * p.slot_rows) - m_use);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    const float inv_l = (mx == -INFINITY) ? 0.f : 1.f / sum;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    const float4* src = reinterpret_cast<const float4*>(p.part_o + ((size_t)first * p.slot_rows + row) * kHeadDim) + lane;
    const size_t chunk_stride = (size_t)p.slot_rows * kHeadDim / 4;  // float4s between slots
    for (int cb = 0; cb < n; cb += 32) {
      const int c = cb + lane;
      const float wl = (c < n) ? fast_exp2(__ldcg(lse_col + (size_t)c * p.slot_rows) - m_use) * inv_l : 0.f;
      const int nb = min(32, n - cb);
      for (int j = 0; j < nb; j += kContractUnroll) {
        float4 a[kContractUnroll];
#pragma unroll
        for (int k = 0; k < kContractUnroll; ++k)
          a[k] = (j + k < nb) ? __ldcg(src + (size_t)(cb + j + k) * chunk_stride) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int k = 0; k < kContractUnroll; ++k) {
          const float w = __shfl_sync(0xffffffffu, wl, (j + k) & 31);
          if (j + k < nb) {
            acc.x += w * a[k].x;
            acc.y += w * a[k].y;
            acc.z += w * a[k].z;
            acc.w += w * a[k].w;
          }
        }
      }
    }
    const size_t orow = (size_t)(q_start + row / p.group) * p.hqo + kv_head * p.group + row % p.group;
    float lse2 = (mx == -INFINITY) ? -INFINITY : mx + fast_log2(sum);
    if (p.o_prev)
      merge_prev4(acc, lse2, *reinterpret_cast<const uint2*>(p.o_prev + orow * kHeadDim + 4 * lane), p.lse_prev[orow]);
    uint2 packed;
    packed.x = f2_to_bf16x2(acc.x, acc.y);
    packed.y = f2_to_bf16x2(acc.z, acc.w);
    *reinterpret_cast<uint2*>(p.o + orow * kHeadDim + 4 * lane) = packed;
    if (lane == 0) p.lse[orow] = lse_out(lse2);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

bool make_map(CUtensorMap* m, const void* base, uint64_t d1, uint64_t d2, uint64_t stride1_bytes,
              uint64_t stride2_bytes, uint32_t box1, uint32_t box2) {
  const cuuint64_t dims[3] = {uint64_t(kHeadDim), d1, d2};
  const cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
  const cuuint32_t box[3] = {64u, box1, box2};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// NHD pages [pages, page_size, H_kv, 128]: dims (dim, head, token in page, page); a box is 64 dims
// of one head and one page, i.e. page_size rows of 128 B, as the HND box lands.  e4m3 pages (one
// byte an element): a box is all 128 dims of a row, unswizzled, so it also lands as 128-B rows.
bool make_map_nhd(CUtensorMap* m, const void* base, uint64_t hkv, uint64_t page_size, uint64_t pages, bool e4m3) {
  const uint64_t row = uint64_t(kHeadDim) * (e4m3 ? 1 : 2);
  const cuuint64_t dims[4] = {uint64_t(kHeadDim), hkv, page_size, pages};
  const cuuint64_t strides[3] = {row, row * hkv, row * hkv * page_size};
  const cuuint32_t box[4] = {e4m3 ? 128u : 64u, 1u, uint32_t(page_size), 1u};
  const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  return encode_fn()(m, e4m3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                     const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     e4m3 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// e4m3 HND pages: (dim, token in page, page * H_kv + head) with 1-byte elements; a box is one
// page-head, page_size rows of 128 codes, unswizzled.
bool make_map_e4m3(CUtensorMap* m, const void* base, uint64_t page_size, uint64_t page_heads) {
  const cuuint64_t dims[3] = {uint64_t(kHeadDim), page_size, page_heads};
  const cuuint64_t strides[2] = {uint64_t(kHeadDim), uint64_t(kHeadDim) * page_size};
  const cuuint32_t box[3] = {128u, uint32_t(page_size), 1u};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool make_decode_map_e4m3(CUtensorMap* m, const void* base, int hkv, int page_size, int num_pages, bool nhd,
                          int box_rows) {
  if (encode_fn() == nullptr || box_rows < 1 || box_rows > page_size) return false;
  const cuuint32_t rows = cuuint32_t(box_rows);
  const cuuint64_t row = uint64_t(kHeadDim);  // one byte a code
  if (nhd) {
    const cuuint64_t dims[4] = {row, uint64_t(hkv), uint64_t(page_size), uint64_t(num_pages)};
    const cuuint64_t strides[3] = {row, row * hkv, row * hkv * page_size};
    const cuuint32_t box[4] = {128u, 1u, rows, 1u};
    const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides, box, estr,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  }
  const cuuint64_t dims[3] = {row, uint64_t(page_size), uint64_t(num_pages) * uint64_t(hkv)};
  const cuuint64_t strides[2] = {row, row * page_size};
  const cuuint32_t box[3] = {128u, rows, 1u};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_decode_map_bf16(CUtensorMap* m, const void* base, int hkv, int page_size, int num_pages, int box_rows) {
  if (encode_fn() == nullptr || box_rows < 1 || box_rows > page_size) return false;
  const uint64_t row = uint64_t(kHeadDim) * 2;
  return make_map(m, base, uint64_t(page_size), uint64_t(num_pages) * uint64_t(hkv), row, row * page_size,
                  uint32_t(box_rows), 1u);
}

int launch_prefill(const PrefillArgs& a, cudaStream_t stream) {
  if (encode_fn() == nullptr) return record_cuda_error(cudaErrorNotSupported, "cuTensorMapEncodeTiled entry point");
  if (a.page_size % 8 != 0 || kTile % a.page_size != 0 || a.group > kItemRows || a.group * a.tile_tokens > kItemRows)
    return FI_ERR_UNSUPPORTED;
  if (a.total_q < 1 || a.num_pages < 1) return FI_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(a.q) % 16 || reinterpret_cast<uintptr_t>(a.k) % 16 ||
      reinterpret_cast<uintptr_t>(a.v) % 16)
    return FI_ERR_INVALID_ARG;
  CUtensorMap tq, tk, tv;
  const uint64_t row_bytes = uint64_t(kHeadDim) * 2;
  // q: (dim, head, token); a box is 64 dims x g heads x (256/g) tokens = up to 256 rows of 128 B
  if (!make_map(&tq, a.q, uint64_t(a.hqo), uint64_t(a.total_q), row_bytes, row_bytes * a.hqo, uint32_t(a.group),
                uint32_t(a.tile_tokens)))
    return FI_ERR_INVALID_ARG;
  // k, v: (dim, token in page, page * H_kv + head); a box is one page-head half
  const uint64_t page_heads = uint64_t(a.num_pages) * a.hkv;
  if (a.nhd) {
    if (!make_map_nhd(&tk, a.k, uint64_t(a.hkv), uint64_t(a.page_size), uint64_t(a.num_pages), a.fp8 != 0) ||
        !make_map_nhd(&tv, a.v, uint64_t(a.hkv), uint64_t(a.page_size), uint64_t(a.num_pages), a.fp8 != 0))
      return FI_ERR_INVALID_ARG;
  } else if (a.fp8) {
    if (!make_map_e4m3(&tk, a.k, uint64_t(a.page_size), page_heads) ||
        !make_map_e4m3(&tv, a.v, uint64_t(a.page_size), page_heads))
      return FI_ERR_INVALID_ARG;
  } else if (!make_map(&tk, a.k, uint64_t(a.page_size), page_heads, row_bytes, row_bytes * a.page_size,
                       uint32_t(a.page_size), 1u) ||
             !make_map(&tv, a.v, uint64_t(a.page_size), page_heads, row_bytes, row_bytes * a.page_size,
                       uint32_t(a.page_size), 1u)) {
    return FI_ERR_INVALID_ARG;
  }

  PrefillParams p{};
  p.cta_indptr = a.cta_indptr;
  p.items = a.items;
  p.units = a.units;
  p.slot_unit = a.slot_unit;
  p.kv_indices = a.kv_indices;
  p.o = static_cast<__nv_bfloat16*>(a.o);
  p.lse = a.lse;
  p.o_prev = static_cast<const __nv_bfloat16*>(a.o_prev);
  p.lse_prev = a.lse_prev;
  p.part_o = a.part_o;
  p.part_lse = a.part_lse;
  p.err = a.err;
  p.num_pages = a.num_pages;
  p.page_size = a.page_size;
  p.hqo = a.hqo;
  p.hkv = a.hkv;
  p.group = a.group;
  p.slot_rows = kTcRows;
  p.q_tile_bytes = uint32_t(2 * 128 * a.group * a.tile_tokens);
  p.scale_log2 = a.scale_log2;
  p.v_scale = a.v_scale;
  p.window_left = a.window_left;
  p.cap_log2 = a.cap_log2;
  p.wait_prior = 1;

  const size_t smem = sizeof(PrefillSmem) + 1024;
  // window, soft-cap, page layout and e4m3 pages are template flags: the plain bf16 HND kernel
  // carries none of them
  using Kernel = void (*)(PrefillParams, CUtensorMap, CUtensorMap, CUtensorMap);
  const Kernel kernels[16] = {
      prefill_kernel<false, false, false, false>, prefill_kernel<false, false, true, false>,
      prefill_kernel<false, true, false, false>,  prefill_kernel<false, true, true, false>,
      prefill_kernel<true, false, false, false>,  prefill_kernel<true, false, true, false>,
      prefill_kernel<true, true, false, false>,   prefill_kernel<true, true, true, false>,
      prefill_kernel<false, false, false, true>,  prefill_kernel<false, false, true, true>,
      prefill_kernel<false, true, false, true>,   prefill_kernel<false, true, true, true>,
      prefill_kernel<true, false, false, true>,   prefill_kernel<true, false, true, true>,
      prefill_kernel<true, true, false, true>,    prefill_kernel<true, true, true, true>};
  const Kernel kernel = kernels[(a.fp8 ? 8 : 0) + (a.window_left >= 0 ? 4 : 0) + (a.cap_log2 > 0.f ? 2 : 0) +
                                (a.nhd ? 1 : 0)];
  static std::once_flag once;
  static cudaError_t attr = cudaSuccess;
  std::call_once(once, [&] {
    for (int i = 0; i < 16 && attr == cudaSuccess; ++i)
      attr = cudaFuncSetAttribute(kernels[i], cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  });
  if (attr != cudaSuccess) return record_cuda_error(attr, "cudaFuncSetAttribute(prefill_kernel)");
  // a programmatic dependent of the previous kernel on the stream: set-up overlaps its tail
  cudaError_t e;
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(a.num_ctas));
    cfg.blockDim = dim3(unsigned(kThreads));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kernel, p, tq, tk, tv);
    if (e == cudaSuccess) e = cudaGetLastError();
  }
  if (e == cudaSuccess && !a.contract) return FI_OK;
  if (e == cudaSuccess) {
    // the contraction of split rows; launched for every plan of this path (it reads the number
    // of split units from the plan), so a captured pair stays valid across plans
    ContractParams c{};
    c.header = a.header;
    c.units = a.units;
    c.part_o = a.part_o;
    c.part_lse = a.part_lse;
    c.o = p.o;
    c.lse = a.lse;
    c.o_prev = p.o_prev;
    c.lse_prev = a.lse_prev;
    c.hqo = a.hqo;
    c.group = a.group;
    c.slot_rows = kTcRows;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(a.num_ctas));
    cfg.blockDim = dim3(unsigned(kContractThreads));
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, contract_kernel, c);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e == cudaSuccess) return FI_OK;
    return record_cuda_error(e, "contract_kernel launch");
  }
  cudaFuncAttributes fa;
  char what[256] = "prefill_kernel launch";
  if (cudaFuncGetAttributes(&fa, kernel) == cudaSuccess)
    snprintf(what, sizeof(what), "prefill_kernel launch (regs %d, max threads %d, static smem %zu, dyn smem %zu/%d, local %zu)",
             fa.numRegs, fa.maxThreadsPerBlock, fa.sharedSizeBytes, smem, fa.maxDynamicSharedSizeBytes,
             fa.localSizeBytes);
  return record_cuda_error(e, what);
}

}  // namespace fi
