// Persistent decode kernel: paged-KV attention for tiles of <= 8 rows, fused with the merge of
// split-KV partial states.
//
// Page "FlashInfer：面向 LLM 推理服务的高效可定制注意力引擎":
//   核心机制 3 (paper §3.2): scattered KV tiles are gathered into contiguous
//     shared memory, after which sparse and dense KV share one kernel body.
//     Each 32-token stage of a page-head run lands in a ring of shared-memory
//     stages that keeps many copies in flight.
//   核心机制 4 (paper §3.2.2): the pages run query tile 1 on CUDA cores, since
//     an MMA needs >= 16 rows; GQA heads of one KV head fold into the rows
//     (术语与记号 "GQA 头组融合", paper App. A), so one KV load serves g rows.
//     Here the tensor-core consumer puts the stage's KV tokens on the MMA's
//     16-row side instead (S^T = K Q^T, O^T = V^T P^T), which lifts that limit
//     for 1..8 rows.
//   核心机制 6-7 (paper §3.3.1, App. D): one persistent CTA per queue of the
//     plan; attention and the contraction of partial outputs in one kernel;
//     a split row is merged by whichever of its chunks finishes last, reading
//     the slots in the plan's fixed order (an arrival counter only counts; it
//     never accumulates data), so results are bit-identical run to run.
//
// CTA layout, two loaders selectable per instantiation (kCopiers):
//   bulk (kCopiers = 0): warp 0 = producer (page-index prefetch + one bulk async copy per
//           page-head run); any page size;
//   LDGSTS: warp 0 = page-index warp (4-byte cp.async into an index ring), warps 1..kCopiers =
//           copiers taking stages round-robin (16-byte cp.async of K/V rows, 512 B per warp
//           instruction); power-of-two page sizes.  The bulk engine keeps only a few copies in
//           flight per SM, which caps a page-sized copy stream well below HBM bandwidth; 16-byte
//           copies do not share that limit.
// The remaining NW warps are consumers.  Consumer warps take the CTA's KV stages round-robin
// (stage n -> warp n % NW); each keeps an online-softmax state, and at the end
// of a work item the NW states are merged through shared memory in warp order.
// Two consumer bodies:
//   tensor-core (kMma, with the LDGSTS loader): warp-level m16n8k16 MMA, see decode_consumer_mma;
//   CUDA cores (with the bulk loader): lane = (half tl, dim-lane dl) for q.k, dl owning dims
//     8*dl..8*dl+7 and tl tokens, partial dots of 16 (token, row) pairs transposed through
//     shared memory and summed; for p.v a lane owns dims 4*lane..4*lane+3 of all R rows.
// Scores are kept in the log2 domain.
#pragma once

#include <cuda.h>

#include <climits>

#include "device_common.cuh"
#include "plan.h"
#include "tcgen05.cuh"

namespace fi {

struct DecodeParams {
  const int32_t* cta_indptr;
  const int32_t* items;
  const int32_t* units;
  const int32_t* slot_unit;
  const int32_t* kv_indices;
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  __nv_bfloat16* o;
  float* lse;
  const __nv_bfloat16* o_prev;  // optional state of the same rows over other keys, merged into o / lse
  const float* lse_prev;
  float* part_o;    // [slots][slot_rows][128] fp32, normalised O
  float* part_lse;  // [slots][slot_rows] fp32, log2 domain
  const int2* ext;  // composable plans: shared-part slots each unit merges (see build_composable_plan)
  float* def_o;     // composable plans: a unit's own state before that merge, [unit][8 rows][128]
  float* def_lse;   //   and its log2-domain LSE, [unit][8 rows]
  uint32_t* counters;
  int32_t* err;
  long long page_stride;   // elements per page (H_kv * page_size * 128)
  long long head_stride;   // elements between KV heads of a page (HND: page_size * 128; NHD: 128)
  int num_pages;
  int page_size;
  int page_shift;  // log2(page_size) when it is a power of two (LDGSTS loader), else -1
  int hqo;
  int group;
  int slot_rows;
  float scale_log2;
  int window_left;  // >= 0: a row at key position p sees keys p - window_left .. p
  float cap_log2;   // > 0: logit soft-cap in the log2 domain, s -> cap_log2 * tanh(s / cap_log2)
  float inv_cap_log2;
  float v_scale;  // FP8 pages: V = v_scale * e4m3 code (the K scale is folded into scale_log2)
  // 1: launched as a programmatic dependent of the previous kernel on the stream, which may still be
  // running: the CTA sets up its shared memory, then waits for that kernel before any global read
  int wait_prior;
};


constexpr int kStageTokens = 32;
constexpr int kIdxDepth = 4;  // page-index prefetch distance of the bulk producer (stages)
constexpr int kIdxSlots = 8;  // page-index ring of the LDGSTS loader (stages)
constexpr int kRedHalf = 336; // words between the two halves of the transpose scratch
constexpr int kRedRow = 20;   // words per lane row of the transpose scratch
constexpr int kMaxDeferred = 64;  // deferred composable merges a CTA keeps (more are merged at once)

// kMma: the tensor-core consumer needs neither the transpose scratch nor the probability buffer.
template <int R, int NW, int S, bool kMma = false>
struct DecodeSmem {
  __nv_bfloat16 kv[S][2][kStageTokens][kHeadDim];  // [stage][K|V][token][dim]
  float red[kMma ? 1 : NW][2][2 * kRedHalf];  // per consumer warp: double-buffered transpose scratch
  float pbuf[kMma ? 1 : NW][kStageTokens * R];
  float alpha[NW][8];
  float macc[NW][R][kHeadDim];
  float mm[NW][8];
  float ml[NW][8];
  int32_t idx[kIdxSlots][32];
  uint64_t full[S];
  uint64_t empty[S];
  uint64_t idx_full[kIdxSlots];
  uint64_t idx_empty[kIdxSlots];
  // Stage last consumed from / last issued into each ring slot.  Stages are dealt round-robin to
  // several consumer (and copier) warps, so the next user of a slot may arrive before the slot's
  // previous phase has completed; a parity wait would then pass on the phase before.  Waiting
  // first for the slot's previous stage keeps every parity wait unambiguous.
  int slot_consumed[S];
  int slot_filled[S];
  int deferred[kMaxDeferred];  // composable plans: units whose merge with the shared states waits for the end
  int n_deferred;
  int flag;
  int abort;
};

// Walks the stages of one CTA's queue in order: (item, stage within item).
template <int kT>
struct StageCursorT {
  int pos, end;
  int st, nst;
  int page_base, kv_head, kv_lo, kv_hi;
  // fields of item `pre`, read one item ahead so that crossing into the next item does not wait for
  // a load in the loader's loop
  int pre = -1;
  int4 pa = {0, 0, 0, 0}, pb = {0, 0, 0, 0};

  __device__ __forceinline__ bool load(const int32_t* items) {
    while (pos < end) {
      int4 a, b;
      if (pre == pos) {
        a = pa;
        b = pb;
      } else {
        a = __ldg(reinterpret_cast<const int4*>(items + size_t(pos) * kItemFields));
        b = __ldg(reinterpret_cast<const int4*>(items + size_t(pos) * kItemFields + 4));
      }
      if (pos + 1 < end) {
        pa = __ldg(reinterpret_cast<const int4*>(items + size_t(pos + 1) * kItemFields));
        pb = __ldg(reinterpret_cast<const int4*>(items + size_t(pos + 1) * kItemFields + 4));
        pre = pos + 1;
      }
      page_base = a.x;
      kv_head = a.w;
      kv_lo = b.x;
      kv_hi = b.y;
      nst = (kv_hi - kv_lo + kT - 1) / kT;
      st = 0;
      if (nst > 0) return true;
      ++pos;
    }
    return false;
  }
  __device__ __forceinline__ bool next(const int32_t* items) {
    if (++st < nst) return true;
    ++pos;
    return load(items);
  }
  __device__ __forceinline__ int tok0() const { return kv_lo + st * kT; }
  __device__ __forceinline__ int ntok() const { return min(kT, kv_hi - tok0()); }
};
using StageCursor = StageCursorT<kStageTokens>;

template <int R, int NW, int S, bool kMs>
__device__ __forceinline__ void decode_producer(const DecodeParams& p, DecodeSmem<R, NW, S, kMs>& sm, int begin, int end) {
  const int lane = threadIdx.x & 31;
  const int ps = p.page_size;
  const uint64_t policy = policy_evict_first();
  StageCursor cur{begin, end, 0, 0, 0, 0, 0, 0};
  StageCursor ahead = cur;
  bool cur_ok = cur.load(p.items);
  bool ahead_ok = ahead.load(p.items);

  auto fetch = [&](const StageCursor& c, int32_t* dst) {
    const int t0 = c.tok0();
    const int first = t0 / ps;
    const int nseg = (t0 + c.ntok() - 1) / ps - first + 1;
    if (lane < nseg) cp_async_4(dst + lane, p.kv_indices + c.page_base + first + lane);
  };

#pragma unroll
  for (int d = 0; d < kIdxDepth; ++d) {
    if (ahead_ok) {
      fetch(ahead, sm.idx[d]);
      ahead_ok = ahead.next(p.items);
    }
    cp_async_commit();
  }

  int issued = 0;
  for (int n = 0; cur_ok; ++n) {
    cp_async_wait<kIdxDepth - 1>();
    const int t0 = cur.tok0();
    const int nt = cur.ntok();
    const int first = t0 / ps;
    const int nseg = (t0 + nt - 1) / ps - first + 1;
    int page = (lane < nseg) ? sm.idx[n % kIdxDepth][lane] : 0;
    __syncwarp();
    if (ahead_ok) {
      fetch(ahead, sm.idx[n % kIdxDepth]);
      ahead_ok = ahead.next(p.items);
    }
    cp_async_commit();

    const int slot = n % S;
    const int fill = n / S;
    if (fill > 0) {
      const bool got = mbar_wait(&sm.empty[slot], (fill - 1) & 1, p.err, &sm.abort);
      if (!__all_sync(0xffffffffu, got)) break;
    }

    int seg_lo = 0, seg_n = 0;
    bool ok = false;
    if (lane < nseg) {
      const int pg_tok = (first + lane) * ps;
      seg_lo = max(t0, pg_tok);
      seg_n = min(t0 + nt, pg_tok + ps) - seg_lo;
      ok = page >= 0 && page < p.num_pages;
      if (!ok) atomicOr(p.err, FI_DEVERR_PAGE_OOB);
    }
    const uint32_t bytes = ok ? uint32_t(seg_n) * (2u * kHeadDim * 2u) : 0u;
    const uint32_t total = __reduce_add_sync(0xffffffffu, bytes);
    if (lane == 0) mbar_arrive_expect_tx(&sm.full[slot], total);
    __syncwarp();
    if (ok) {
      const long long src = (long long)page * p.page_stride + (long long)cur.kv_head * p.head_stride +
                            (long long)(seg_lo - (first + lane) * ps) * kHeadDim;
      const uint32_t nb = uint32_t(seg_n) * kHeadDim * 2u;
      bulk_g2s(&sm.kv[slot][0][seg_lo - t0][0], p.k + src, nb, &sm.full[slot], policy);
      bulk_g2s(&sm.kv[slot][1][seg_lo - t0][0], p.v + src, nb, &sm.full[slot], policy);
    }
    cur_ok = cur.next(p.items);
    issued = n + 1;
  }
  cp_async_wait<0>();
  // never leave with bulk copies still landing in this CTA's shared memory
  for (int n = max(0, issued - S); n < issued; ++n) mbar_wait_bounded(&sm.full[n % S], (n / S) & 1);
}

// LDGSTS loader, warp 0: page ids of each stage into a ring of kIdxSlots x kT entries (kT tokens
// per stage: up to kT pages).
template <int R, int NW, int S, class SM, int kT = kStageTokens>
__device__ __forceinline__ void decode_index_warp(const DecodeParams& p, SM& sm, int begin, int end) {
  const int lane = threadIdx.x & 31;
  StageCursorT<kT> c{begin, end, 0, 0, 0, 0, 0, 0};
  bool ok = c.load(p.items);
  for (int n = 0; ok; ++n) {
    const int slot = n % kIdxSlots, fill = n / kIdxSlots;
    if (fill > 0 && !__all_sync(0xffffffffu, mbar_wait(&sm.idx_empty[slot], (fill - 1) & 1, p.err, &sm.abort))) break;
    const int t0 = c.tok0();
    const int first = t0 >> p.page_shift;
    const int nseg = ((t0 + c.ntok() - 1) >> p.page_shift) - first + 1;
    if (lane < nseg) cp_async_4(&sm.idx[slot][lane], p.kv_indices + c.page_base + first + lane);
    if constexpr (kT > 32) {
      if (lane + 32 < nseg) cp_async_4(&sm.idx[slot][lane + 32], p.kv_indices + c.page_base + first + lane + 32);
    }
    cp_async_arrive_noinc(&sm.idx_full[slot]);
    ok = c.next(p.items);
  }
  cp_async_wait_all();
}

// LDGSTS loader, copier warp `cw` of kCopiers: stages cw, cw + kCopiers, ... -- the stage's K and V
// rows, 16 bytes per lane per instruction.
// Copy c (0..1023) of a stage: K/V = c / 512, token = (c % 512) / 16, 16-byte chunk = c % 16,
// so each warp instruction moves two consecutive 256-byte rows.
// kNhdStride: 0 for HND pages, else the elements between tokens of an NHD page-head (H_kv * 128).
template <int R, int NW, int S, int kCopiers, bool kSwizzle, int kNhdStride, bool kMs>
__device__ __forceinline__ void decode_copier_warp(const DecodeParams& p, DecodeSmem<R, NW, S, kMs>& sm, int begin,
                                                   int end, int cw) {
  const int lane = threadIdx.x & 31;
  const int sh = p.page_shift;
  const int row_mask = p.page_size - 1;
  StageCursor c{begin, end, 0, 0, 0, 0, 0, 0};
  bool ok = c.load(p.items);
  for (int k = 0; k < cw && ok; ++k) ok = c.next(p.items);
  for (int n = cw; ok; n += kCopiers) {
    const int islot = n % kIdxSlots;
    if (!__all_sync(0xffffffffu, mbar_wait(&sm.idx_full[islot], (n / kIdxSlots) & 1, p.err, &sm.abort))) break;
    const int t0 = c.tok0();
    const int nt = c.ntok();
    const int first = t0 >> sh;
    const int nseg = ((t0 + nt - 1) >> sh) - first + 1;
    int pg = (lane < nseg) ? sm.idx[islot][lane] : 0;
    if (lane < nseg && (pg < 0 || pg >= p.num_pages)) {
      atomicOr(p.err, FI_DEVERR_PAGE_OOB);
      pg = -1;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.idx_empty[islot]);
    const int slot = n % S, fill = n / S;
    if (!__all_sync(0xffffffffu, spin_until_eq(&sm.slot_filled[slot], n - S, p.err, &sm.abort))) break;
    if (fill > 0 && !__all_sync(0xffffffffu, mbar_wait(&sm.empty[slot], (fill - 1) & 1, p.err, &sm.abort))) break;
    const __nv_bfloat16* kb = p.k + (long long)c.kv_head * p.head_stride;
    const __nv_bfloat16* vb = p.v + (long long)c.kv_head * p.head_stride;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int tok = 2 * j + (lane >> 4);  // same tokens for the K half (j) and the V half (j + 16)
      const int pos = t0 + tok;
      const int seg = min(max((pos >> sh) - first, 0), 31);
      const int page = __shfl_sync(0xffffffffu, pg, seg);
      if (tok < nt && page >= 0) {
        // One 64-bit expression with a compile-time row stride: this loop issues a 16-byte copy per
        // lane per step, and measured on GB300 a run-time stride (multiply or shift) here cost a
        // third of the copy rate, as did forming the row term in 32 bits.
        const long long off = (long long)page * p.page_stride +
                              (long long)(pos & row_mask) * (kNhdStride ? kNhdStride : kHeadDim) + (lane & 15) * 8;
        const int chunk = kSwizzle ? ((lane & 15) ^ (tok & 7)) : (lane & 15);
        cp_async_16(&sm.kv[slot][0][tok][chunk * 8], kb + off);
        cp_async_16(&sm.kv[slot][1][tok][chunk * 8], vb + off);
      }
    }
    cp_async_arrive_noinc(&sm.full[slot]);
    __syncwarp();
    if (lane == 0) *reinterpret_cast<volatile int*>(&sm.slot_filled[slot]) = n;
    for (int k = 0; k < kCopiers && ok; ++k) ok = c.next(p.items);
  }
  cp_async_wait_all();
}

// TMA copier (HND pages of 8 or more tokens, tensor-core consumer): copier warp `cw` issues its
// stages as tensor boxes of min(page_size, 32) tokens of one page and KV head, 64 dims each, so a
// stage's K (and V) lands as two 64-dim halves [2][32 tokens][64] in the 128-byte swizzle: 16-byte
// chunk c of token t's half at chunk position c ^ (t & 7).  A box of 8 or more rows is at least
// 1 KB, so boxes start on 1 KB boundaries.  The copies bypass the load/store pipeline the
// consumers' shared-memory instructions use.  Boxes are whole pages, so a request's last page may
// bring rows past its last token; the consumers clear those rows' V before the P.V MMAs.
// tm_k / tm_v map (dim, token in page, page * H_kv + head).
template <int R, int NW, int S, int kCopiers, bool kMs>
__device__ __forceinline__ void decode_tma_copier(const DecodeParams& p, DecodeSmem<R, NW, S, kMs>& sm,
                                                  const CUtensorMap* tm_k, const CUtensorMap* tm_v, int begin, int end,
                                                  int cw) {
  const int lane = threadIdx.x & 31;
  const int box_tok = min(p.page_size, kStageTokens);
  const int hkv = int(p.page_stride >> (p.page_shift + 7));  // page stride = H_kv * page_size * 128
  StageCursor c{begin, end, 0, 0, 0, 0, 0, 0};
  bool ok = c.load(p.items);
  for (int k = 0; k < cw && ok; ++k) ok = c.next(p.items);
  int issued_last = -1;
  for (int n = cw; ok; n += kCopiers) {
    const int islot = n % kIdxSlots;
    if (!__all_sync(0xffffffffu, mbar_wait(&sm.idx_full[islot], (n / kIdxSlots) & 1, p.err, &sm.abort))) break;
    const int t0 = c.tok0();
    const int nt = c.ntok();
    // stages start on a page boundary, or on a 32-token boundary inside a longer page
    const int nbox = (nt + box_tok - 1) / box_tok;
    int pg = (lane < nbox) ? sm.idx[islot][lane] : -1;
    if (lane < nbox && (pg < 0 || pg >= p.num_pages)) {
      atomicOr(p.err, FI_DEVERR_PAGE_OOB);
      pg = -1;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.idx_empty[islot]);
    const int slot = n % S, fill = n / S;
    if (!__all_sync(0xffffffffu, spin_until_eq(&sm.slot_filled[slot], n - S, p.err, &sm.abort))) break;
    if (fill > 0 && !__all_sync(0xffffffffu, mbar_wait(&sm.empty[slot], (fill - 1) & 1, p.err, &sm.abort))) break;
    const uint32_t bytes = pg >= 0 ? uint32_t(4 * box_tok * 128) : 0u;  // K and V, two 128-byte halves a row
    const uint32_t total = __reduce_add_sync(0xffffffffu, bytes);
    if (lane == 0) mbar_arrive_expect_tx(&sm.full[slot], total);
    __syncwarp();
    if (pg >= 0) {
      const int y = t0 & (p.page_size - 1) & ~(box_tok - 1);
      const int z = pg * hkv + c.kv_head;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        __nv_bfloat16* dk = &sm.kv[slot][0][0][0] + h * (kStageTokens * 64) + lane * box_tok * 64;
        __nv_bfloat16* dv = &sm.kv[slot][1][0][0] + h * (kStageTokens * 64) + lane * box_tok * 64;
        tc::tma_load_3d(dk, tm_k, 64 * h, y, z, &sm.full[slot]);
        tc::tma_load_3d(dv, tm_v, 64 * h, y, z, &sm.full[slot]);
      }
    }
    __syncwarp();
    if (lane == 0) *reinterpret_cast<volatile int*>(&sm.slot_filled[slot]) = n;
    issued_last = n;
    for (int k = 0; k < kCopiers && ok; ++k) ok = c.next(p.items);
  }
  // A normal run needs no drain: the consumers wait for every stage to land before the CTA ends.
  // After an abort, wait (bounded) for this warp's recent stages so that no tensor copy is still
  // landing in shared memory when the CTA exits.
  if (*reinterpret_cast<volatile int*>(&sm.abort)) {
    for (int n = issued_last; n >= 0 && n > issued_last - S; n -= kCopiers) mbar_wait_bounded(&sm.full[n % S], (n / S) & 1);
  }
}

template <int R>
__device__ __forceinline__ void load_q_rows(const DecodeParams& p, int q_start, int q_len, int kv_head, int dl,
                                            float2 (&q2)[R][4]) {
  const int rows_valid = q_len * p.group;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    if (r < rows_valid) {
      const int tok = q_start + r / p.group;
      const int head = kv_head * p.group + r % p.group;
      const uint4 raw = __ldg(reinterpret_cast<const uint4*>(p.q + ((size_t)tok * p.hqo + head) * kHeadDim + 8 * dl));
      const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float2 f = bf16x2_to_f2(w[c]);
        q2[r][c] = make_float2(f.x * p.scale_log2, f.y * p.scale_log2);
      }
    } else {
#pragma unroll
      for (int c = 0; c < 4; ++c) q2[r][c] = make_float2(0.f, 0.f);
    }
  }
}

// Composable plans: the state (O, lse2) of row r of a unit merged (⊕, in list order) with the states
// the shared part's tensor-core launch left for the same row in its slots.  That launch precedes this
// one in the stream (chained by programmatic dependent launch), so its slots are read after
// griddepcontrol.wait, which returns once it has completed.  Called by a whole warp for one row
// (lane = dq): lane e reads entry e's LSE, the weights come from warp reductions, and the lanes'
// partial outputs are loaded kMergeBatch at a time, so the slots' latencies overlap.
constexpr int kMergeBatch = 8;
__device__ __forceinline__ void merge_ext(const DecodeParams& p, int unit, int r, int dq, float4& O, float& lse2) {
  const int ef = __ldg(p.units + unit * kUnitFields + 5), ec = __ldg(p.units + unit * kUnitFields + 6);
  if (ec == 0) return;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // pass 1: the largest LSE (lanes take entries e = lane, lane + 32, ...)
  float M = lse2;
  for (int e = dq; e < ec; e += 32) {
    const int2 x = __ldg(p.ext + ef + e);
    const int row = (x.y & 0xFFFF) - kExtRowBias + r;
    if (row >= 0 && row < (x.y >> 16)) M = fmaxf(M, __ldcg(p.part_lse + (size_t)x.x * p.slot_rows + row));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  if (M == -INFINITY) {
    O = make_float4(0.f, 0.f, 0.f, 0.f);
    lse2 = -INFINITY;
    return;
  }
  const float w0 = (lse2 == -INFINITY) ? 0.f : fast_exp2(lse2 - M);
  float L = 0.f;
  float4 acc = make_float4(w0 * O.x, w0 * O.y, w0 * O.z, w0 * O.w);
  for (int eb = 0; eb < ec; eb += 32) {
    // this lane's entry of the batch of 32: its slot row and weight
    const int e = eb + dq;
    size_t srow = 0;
    float w = 0.f;
    if (e < ec) {
      const int2 x = __ldg(p.ext + ef + e);
      const int row = (x.y & 0xFFFF) - kExtRowBias + r;
      if (row >= 0 && row < (x.y >> 16)) {
        srow = (size_t)x.x * p.slot_rows + row;
        w = fast_exp2(__ldcg(p.part_lse + srow) - M);
      }
    }
    L += w;
    const int nb = min(32, ec - eb);
    for (int j = 0; j < nb; j += kMergeBatch) {
      float4 a[kMergeBatch];
      float wj[kMergeBatch];
#pragma unroll
      for (int k = 0; k < kMergeBatch; ++k) {
        const int src = (j + k) & 31;
        wj[k] = __shfl_sync(0xffffffffu, w, src);
        const unsigned long long sr = __shfl_sync(0xffffffffu, (unsigned long long)srow, src);
        a[k] = (j + k < nb && wj[k] != 0.f)
                   ? __ldcg(reinterpret_cast<const float4*>(p.part_o + sr * kHeadDim + 4 * dq))
                   : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int k = 0; k < kMergeBatch; ++k) {
        acc.x += wj[k] * a[k].x;
        acc.y += wj[k] * a[k].y;
        acc.z += wj[k] * a[k].z;
        acc.w += wj[k] * a[k].w;
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
  L += w0;
  const float inv = 1.f / L;
  O = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  lse2 = M + fast_log2(L);
}

// End of a work item, all NW consumer warps: merge their (O, m, l) states from shared memory in
// warp order, then write the row (single chunk) or its partial state, and if this chunk is the
// last of a split row to finish, contract all of the row's slots in plan order.
// Composable plans (kDefer): a row that also has states of the shared part (written by the
// concurrent tensor-core launch) is kept in the unit's deferred buffer and merged with them at the
// end of the CTA's queue (decode_deferred_merges); with the CTA's list full it is merged at once.
template <int R, int NW, int S, class SM, bool kDefer = true>
__device__ __forceinline__ void decode_finish_item(const DecodeParams& p, SM& sm, int ctid, int q_start, int kv_head,
                                                   int rows_valid, int slot_out) {
  // one decision for all threads: read before this item changes the list
  bool defer_ok = false;
  if constexpr (kDefer) defer_ok = sm.n_deferred < kMaxDeferred;
  auto keep = [&](int unit, int r, int dq, const float4& O, float lse2) {
    *reinterpret_cast<float4*>(p.def_o + ((size_t)unit * kDecodeMaxRows + r) * kHeadDim + 4 * dq) = O;
    if (dq == 0) p.def_lse[(size_t)unit * kDecodeMaxRows + r] = lse2;
  };
  for (int u = ctid; u < R * 32; u += NW * 32) {
    const int r = u >> 5, dq = u & 31;
    float M = -INFINITY;
#pragma unroll
    for (int ww = 0; ww < NW; ++ww) M = fmaxf(M, sm.mm[ww][r]);
    float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
    float L = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int ww = 0; ww < NW; ++ww) {
        const float s = fast_exp2(sm.mm[ww][r] - M);
        const float4 a = *reinterpret_cast<const float4*>(&sm.macc[ww][r][4 * dq]);
        L += s * sm.ml[ww][r];
        O.x += s * a.x;
        O.y += s * a.y;
        O.z += s * a.z;
        O.w += s * a.w;
      }
      const float inv = 1.f / L;
      O.x *= inv;
      O.y *= inv;
      O.z *= inv;
      O.w *= inv;
    }
    const float lse2 = (M == -INFINITY) ? -INFINITY : M + fast_log2(L);
    if (r < rows_valid) {
      if (slot_out < 0) {
        const int tok = q_start + r / p.group;
        const int head = kv_head * p.group + r % p.group;
        const size_t orow = (size_t)tok * p.hqo + head;
        float lse_w = lse2;
        if (slot_out <= -2) {  // composable: the shared part's states of these rows
          if (defer_ok) {
            keep(-slot_out - 2, r, dq, O, lse2);
            continue;
          }
          merge_ext(p, -slot_out - 2, r, dq, O, lse_w);
        }
        if (p.o_prev)
          merge_prev4(O, lse_w, *reinterpret_cast<const uint2*>(p.o_prev + orow * kHeadDim + 4 * dq), p.lse_prev[orow]);
        uint2 packed;
        packed.x = f2_to_bf16x2(O.x, O.y);
        packed.y = f2_to_bf16x2(O.z, O.w);
        *reinterpret_cast<uint2*>(p.o + orow * kHeadDim + 4 * dq) = packed;
        if (dq == 0) p.lse[orow] = lse_w * kLn2;
      } else {
        const size_t srow = (size_t)slot_out * p.slot_rows + r;
        *reinterpret_cast<float4*>(p.part_o + srow * kHeadDim + 4 * dq) = O;
        if (dq == 0) p.part_lse[srow] = lse2;
      }
    }
  }
  if constexpr (kDefer) {
    if (slot_out <= -2 && defer_ok && ctid == 0) sm.deferred[sm.n_deferred++] = -slot_out - 2;
  }

  if (slot_out >= 0) {
    // contraction of a split row: the last chunk to finish merges all slots in order
    named_bar_sync(1, NW * 32);
    const int unit = __ldg(p.slot_unit + slot_out);
    if (ctid == 0) {
      __threadfence();
      const uint32_t prev = atomicAdd(p.counters + unit, 1u);
      const int n_chunks = __ldg(p.units + unit * kUnitFields + U_N_CHUNKS);
      sm.flag = (prev == uint32_t(n_chunks - 1)) ? 1 : 0;
      if (sm.flag) __threadfence();
    }
    named_bar_sync(1, NW * 32);
    if (sm.flag) {
      const int first = __ldg(p.units + unit * kUnitFields + U_FIRST_SLOT);
      const int n_chunks = __ldg(p.units + unit * kUnitFields + U_N_CHUNKS);
      const bool has_ext = p.ext != nullptr && __ldg(p.units + unit * kUnitFields + 6) > 0;
      for (int u = ctid; u < R * 32; u += NW * 32) {
        const int r = u >> 5, dq = u & 31;
        if (r >= rows_valid) continue;
        float M = -INFINITY;
        for (int c = 0; c < n_chunks; ++c) M = fmaxf(M, __ldcg(p.part_lse + (size_t)(first + c) * p.slot_rows + r));
        float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
        float L = 0.f;
        if (M != -INFINITY) {
          for (int c = 0; c < n_chunks; ++c) {
            const size_t srow = (size_t)(first + c) * p.slot_rows + r;
            const float s = fast_exp2(__ldcg(p.part_lse + srow) - M);
            const float4 a = __ldcg(reinterpret_cast<const float4*>(p.part_o + srow * kHeadDim + 4 * dq));
            L += s;
            O.x += s * a.x;
            O.y += s * a.y;
            O.z += s * a.z;
            O.w += s * a.w;
          }
          const float inv = 1.f / L;
          O.x *= inv;
          O.y *= inv;
          O.z *= inv;
          O.w *= inv;
        }
        const int tok = q_start + r / p.group;
        const int head = kv_head * p.group + r % p.group;
        const size_t orow = (size_t)tok * p.hqo + head;
        float lse_w = (M == -INFINITY) ? -INFINITY : M + fast_log2(L);
        if (has_ext) {  // composable: as for single-chunk rows
          if (defer_ok) {
            keep(unit, r, dq, O, lse_w);
            continue;
          }
          merge_ext(p, unit, r, dq, O, lse_w);
        }
        if (p.o_prev)
          merge_prev4(O, lse_w, *reinterpret_cast<const uint2*>(p.o_prev + orow * kHeadDim + 4 * dq), p.lse_prev[orow]);
        uint2 packed;
        packed.x = f2_to_bf16x2(O.x, O.y);
        packed.y = f2_to_bf16x2(O.z, O.w);
        *reinterpret_cast<uint2*>(p.o + orow * kHeadDim + 4 * dq) = packed;
        if (dq == 0) p.lse[orow] = lse_w * kLn2;
      }
      if (ctid == 0) p.counters[unit] = 0u;
      if constexpr (kDefer) {
        if (has_ext && defer_ok && ctid == 0) sm.deferred[sm.n_deferred++] = unit;
      }
    }
  }
  named_bar_sync(1, NW * 32);
}

// Composable plans, after the CTA's last item, all NW consumer warps: wait once for the shared part's
// launch to complete, then merge every deferred unit's rows (kept by decode_finish_item) with the
// shared states of the same rows and write the outputs; a warp per row.
template <int R, int NW, int S, class SM>
__device__ __forceinline__ void decode_deferred_merges(const DecodeParams& p, SM& sm, int w) {
  const int nd = sm.n_deferred;  // final: the last decode_finish_item ended with a barrier
  if (nd == 0) return;
  const int lane = threadIdx.x & 31;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  for (int task = w; task < nd * R; task += NW) {
    const int unit = sm.deferred[task / R], r = task % R;
    const int q_start = __ldg(p.units + unit * kUnitFields + U_Q_START);
    const int q_len = __ldg(p.units + unit * kUnitFields + U_Q_LEN);
    const int kv_head = __ldg(p.units + unit * kUnitFields + U_KV_HEAD);
    if (r >= q_len * p.group) continue;
    float4 O = __ldcg(reinterpret_cast<const float4*>(p.def_o + ((size_t)unit * kDecodeMaxRows + r) * kHeadDim) + lane);
    float lse2 = __ldcg(p.def_lse + (size_t)unit * kDecodeMaxRows + r);
    merge_ext(p, unit, r, lane, O, lse2);
    const size_t orow = (size_t)(q_start + r / p.group) * p.hqo + kv_head * p.group + r % p.group;
    uint2 packed;
    packed.x = f2_to_bf16x2(O.x, O.y);
    packed.y = f2_to_bf16x2(O.z, O.w);
    *reinterpret_cast<uint2*>(p.o + orow * kHeadDim + 4 * lane) = packed;
    if (lane == 0) p.lse[orow] = lse2 * kLn2;
  }
}

// Composable plans, tensor-core consumer kernel, after every warp of the CTA is done with its
// queue (a CTA barrier precedes this): all warps merge the deferred units' rows with the shared
// part's states.  A warp takes kMergeTasks (unit, row) tasks at a time.  Everything that does not
// depend on the shared part's launch -- the unit's fields, its shared-slot list, the row's own
// state -- is loaded before the wait for that launch, so that only the slots' LSEs and states are
// read after it, the tasks' loads in flight together.  Lane e holds shared entry e of a task (entry
// lists longer than kMergeFast go through merge_ext).  Same sums as merge_ext, in the same order.
constexpr int kMergeFast = 8;
constexpr int kMergeTasks = 3;  // (unit, row) tasks a warp merges together
// Not inlined: its register needs then leave the allocation of the decode loop alone (inlined, the
// kernel measured 0.2 % slower on plain decode batches, which never call it).
template <int R, class SM>
__device__ __noinline__ void decode_deferred_merges_cta(const DecodeParams& p, SM& sm, int warp, int nwarps) {
  const int nd = sm.n_deferred;  // final: every warp passed the barrier before this call
  if (nd == 0) return;
  const int lane = threadIdx.x & 31;
  const int ntask = nd * R;
  bool waited = false;
  for (int t0 = warp; t0 < ntask; t0 += kMergeTasks * nwarps) {
    int unit[kMergeTasks], rr[kMergeTasks], ec[kMergeTasks], ef[kMergeTasks];
    size_t orow[kMergeTasks], srow[kMergeTasks];
    bool live[kMergeTasks], ent[kMergeTasks];
    float4 O[kMergeTasks];
    float lse_own[kMergeTasks];
#pragma unroll
    for (int b = 0; b < kMergeTasks; ++b) {
      const int t = t0 + b * nwarps;
      live[b] = false;
      ent[b] = false;
      ec[b] = 0;
      ef[b] = 0;
      srow[b] = 0;
      orow[b] = 0;
      unit[b] = 0;
      rr[b] = 0;
      O[b] = make_float4(0.f, 0.f, 0.f, 0.f);
      lse_own[b] = -INFINITY;
      if (t >= ntask) continue;
      unit[b] = sm.deferred[t / R];
      rr[b] = t % R;
      const int* uf = p.units + unit[b] * kUnitFields;
      const int q_len = __ldg(uf + U_Q_LEN);
      if (rr[b] >= q_len * p.group) continue;
      live[b] = true;
      const int q_start = __ldg(uf + U_Q_START), kv_head = __ldg(uf + U_KV_HEAD);
      orow[b] = (size_t)(q_start + rr[b] / p.group) * p.hqo + kv_head * p.group + rr[b] % p.group;
      ef[b] = __ldg(uf + 5);
      ec[b] = __ldg(uf + 6);
      const size_t drow = (size_t)unit[b] * kDecodeMaxRows + rr[b];
      O[b] = __ldcg(reinterpret_cast<const float4*>(p.def_o + drow * kHeadDim) + lane);
      lse_own[b] = __ldcg(p.def_lse + drow);
      if (ec[b] <= kMergeFast && lane < ec[b]) {
        const int2 x = __ldg(p.ext + ef[b] + lane);
        const int row = (x.y & 0xFFFF) - kExtRowBias + rr[b];
        if (row >= 0 && row < (x.y >> 16)) {
          srow[b] = (size_t)x.x * p.slot_rows + row;
          ent[b] = true;
        }
      }
    }
    if (!waited) {
      asm volatile("griddepcontrol.wait;" ::: "memory");  // the shared part's launch has completed
      waited = true;
    }
    // the slots' LSEs of the tasks, then their weights
    float le[kMergeTasks], wgt[kMergeTasks], M[kMergeTasks], L[kMergeTasks];
#pragma unroll
    for (int b = 0; b < kMergeTasks; ++b) le[b] = ent[b] ? __ldcg(p.part_lse + srow[b]) : -INFINITY;
#pragma unroll
    for (int b = 0; b < kMergeTasks; ++b) {
      float m = le[b];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      M[b] = fmaxf(m, lse_own[b]);
      wgt[b] = (le[b] == -INFINITY || M[b] == -INFINITY) ? 0.f : fast_exp2(le[b] - M[b]);
      float l = wgt[b];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
      const float w0 = (lse_own[b] == -INFINITY || M[b] == -INFINITY) ? 0.f : fast_exp2(lse_own[b] - M[b]);
      L[b] = l + w0;
      O[b] = make_float4(w0 * O[b].x, w0 * O[b].y, w0 * O[b].z, w0 * O[b].w);
    }
    // the slots' states: entry e of task b from lane e's slot row, every task's loads issued first
    float4 a[kMergeTasks][kMergeFast];
    float wj[kMergeTasks][kMergeFast];
#pragma unroll
    for (int b = 0; b < kMergeTasks; ++b) {
#pragma unroll
      for (int e = 0; e < kMergeFast; ++e) {
        wj[b][e] = __shfl_sync(0xffffffffu, wgt[b], e);
        const unsigned long long sr = __shfl_sync(0xffffffffu, (unsigned long long)srow[b], e);
        a[b][e] = (ec[b] <= kMergeFast && e < ec[b] && wj[b][e] != 0.f)
                      ? __ldcg(reinterpret_cast<const float4*>(p.part_o + sr * kHeadDim) + lane)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int b = 0; b < kMergeTasks; ++b) {
      if (!live[b]) continue;
      float4 acc = O[b];
      float lse2;
      if (ec[b] <= kMergeFast) {
#pragma unroll
        for (int e = 0; e < kMergeFast; ++e) {
          acc.x += wj[b][e] * a[b][e].x;
          acc.y += wj[b][e] * a[b][e].y;
          acc.z += wj[b][e] * a[b][e].z;
          acc.w += wj[b][e] * a[b][e].w;
        }
        if (M[b] == -INFINITY) {
          acc = make_float4(0.f, 0.f, 0.f, 0.f);
          lse2 = -INFINITY;
        } else {
          const float inv = 1.f / L[b];
          acc = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
          lse2 = M[b] + fast_log2(L[b]);
        }
      } else {  // a long entry list: the general merge
        const size_t drow = (size_t)unit[b] * kDecodeMaxRows + rr[b];
        acc = __ldcg(reinterpret_cast<const float4*>(p.def_o + drow * kHeadDim) + lane);
        lse2 = lse_own[b];
        merge_ext(p, unit[b], rr[b], lane, acc, lse2);
      }
      uint2 packed;
      packed.x = f2_to_bf16x2(acc.x, acc.y);
      packed.y = f2_to_bf16x2(acc.z, acc.w);
      *reinterpret_cast<uint2*>(p.o + orow[b] * kHeadDim + 4 * lane) = packed;
      if (lane == 0) p.lse[orow[b]] = lse2 * kLn2;
    }
  }
}

template <int R, int NW, int S, bool kVar, bool kMs>
__device__ __forceinline__ void decode_consumer(const DecodeParams& p, DecodeSmem<R, NW, S, kMs>& sm, int begin, int end,
                                                int w) {
  constexpr int NT = 16 / R;  // tokens per half per sub-batch
  const int lane = threadIdx.x & 31;
  const int tl = lane >> 4, dl = lane & 15;
  const int my_row = dl % R;
  const int ctid = w * 32 + lane;

  float* pb = sm.pbuf[w];
  int stage_n = 0;
  bool alive = true;

  for (int pos = begin; pos < end; ++pos) {
    const int4 ia = __ldg(reinterpret_cast<const int4*>(p.items + size_t(pos) * kItemFields));
    const int4 ib = __ldg(reinterpret_cast<const int4*>(p.items + size_t(pos) * kItemFields + 4));
    const int q_start = ia.y, q_len = ia.z, kv_head = ia.w;
    const int kv_lo = ib.x, kv_hi = ib.y, diag = ib.z, slot_out = ib.w;
    const int nst = (kv_hi - kv_lo + kStageTokens - 1) / kStageTokens;

    float2 q2[R][4];
    load_q_rows<R>(p, q_start, q_len, kv_head, dl, q2);
    float2 acc[R][2];
#pragma unroll
    for (int r = 0; r < R; ++r) acc[r][0] = acc[r][1] = make_float2(0.f, 0.f);
    float m_run = -INFINITY, l_run = 0.f;
    // token limits of my score row: key j visible iff row_low <= j <= diag + (row / g)
    const int row_limit = diag + my_row / p.group;
    const int row_low = (kVar && p.window_left >= 0) ? row_limit - p.window_left : INT_MIN;

    for (int st = 0; st < nst; ++st) {
      const int n = stage_n + st;
      if (n % NW != w) continue;
      const int slot = n % S;
      if (!alive) continue;
      const bool got = spin_until_eq(&sm.slot_consumed[slot], n - S, p.err, &sm.abort) &&
                       mbar_wait(&sm.full[slot], (n / S) & 1, p.err, &sm.abort);
      if (!__all_sync(0xffffffffu, got)) {
        alive = false;  // keep joining the named barriers; outputs of an aborted run are undefined
        continue;
      }
      const int t0 = kv_lo + st * kStageTokens;
      const int nt = min(kStageTokens, kv_hi - t0);
      const __nv_bfloat16* Ks = &sm.kv[slot][0][0][0];
      const __nv_bfloat16* Vs = &sm.kv[slot][1][0][0];

      // ---- scores: R sub-batches of 2*NT tokens -------------------------------
      float sc[R];
#pragma unroll
      for (int b = 0; b < R; ++b) {
        float part[16];
#pragma unroll
        for (int u = 0; u < NT; ++u) {
          const int t = b * 2 * NT + tl * NT + u;
          const uint4 raw = *reinterpret_cast<const uint4*>(Ks + t * kHeadDim + 8 * dl);
          const float2 k0 = bf16x2_to_f2(raw.x), k1 = bf16x2_to_f2(raw.y);
          const float2 k2 = bf16x2_to_f2(raw.z), k3 = bf16x2_to_f2(raw.w);
#pragma unroll
          for (int r = 0; r < R; ++r) {
            float2 s2 = __fmul2_rn(q2[r][0], k0);
            s2 = __ffma2_rn(q2[r][1], k1, s2);
            s2 = __ffma2_rn(q2[r][2], k2, s2);
            s2 = __ffma2_rn(q2[r][3], k3, s2);
            part[u * R + r] = s2.x + s2.y;
          }
        }
        // two scratch buffers alternate, so one warp barrier per sub-batch suffices and the sum of
        // this sub-batch can overlap the products of the next
        float* red = sm.red[w][b & 1];
        float4* rw = reinterpret_cast<float4*>(red + tl * kRedHalf + dl * kRedRow);
#pragma unroll
        for (int c = 0; c < 4; ++c) rw[c] = make_float4(part[4 * c], part[4 * c + 1], part[4 * c + 2], part[4 * c + 3]);
        __syncwarp();
        float s4[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) s4[j] = red[tl * kRedHalf + j * kRedRow + dl];
#pragma unroll
        for (int j = 4; j < 16; ++j) s4[j & 3] += red[tl * kRedHalf + j * kRedRow + dl];
        const float s = (s4[0] + s4[1]) + (s4[2] + s4[3]);
        const int t = b * 2 * NT + tl * NT + dl / R;
        bool vis = (t < nt) && (t0 + t <= row_limit);
        float sv = s;
        if constexpr (kVar) {
          vis = vis && (t0 + t >= row_low);
          if (p.cap_log2 > 0.f) sv = p.cap_log2 * tanh_exp2(s * p.inv_cap_log2);
        }
        sc[b] = vis ? sv : -INFINITY;
      }

      // ---- online softmax over the stage --------------------------------------
      float mx = sc[0];
#pragma unroll
      for (int b = 1; b < R; ++b) mx = fmaxf(mx, sc[b]);
#pragma unroll
      for (int msk = R; msk < 32; msk <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, msk));
      const float m_new = fmaxf(m_run, mx);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = fast_exp2(m_run - m_use);
      float psum = 0.f;
#pragma unroll
      for (int b = 0; b < R; ++b) {
        const float pv = fast_exp2(sc[b] - m_use);
        psum += pv;
        pb[b * 32 + lane] = pv;
      }
#pragma unroll
      for (int msk = R; msk < 32; msk <<= 1) psum += __shfl_xor_sync(0xffffffffu, psum, msk);
      l_run = l_run * alpha + psum;
      m_run = m_new;
      if (tl == 0 && dl < R) sm.alpha[w][dl] = alpha;
      __syncwarp();

      // ---- p.v -------------------------------------------------------------------
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const float a = sm.alpha[w][r];
        acc[r][0] = __fmul2_rn(acc[r][0], make_float2(a, a));
        acc[r][1] = __fmul2_rn(acc[r][1], make_float2(a, a));
      }
      // tokens alternate between two accumulator sets (when registers allow) to halve the FMA chain
      constexpr int kSets = R <= 4 ? 2 : 1;
      float2 acc2[R][2];
#pragma unroll
      for (int r = 0; r < R; ++r) acc2[r][0] = acc2[r][1] = make_float2(0.f, 0.f);
#pragma unroll 4
      for (int t = 0; t < nt; ++t) {
        const uint2 raw = *reinterpret_cast<const uint2*>(Vs + t * kHeadDim + 4 * lane);
        const float2 v0 = bf16x2_to_f2(raw.x), v1 = bf16x2_to_f2(raw.y);
        float pr[R];
        if constexpr (R >= 4) {
#pragma unroll
          for (int c = 0; c < R / 4; ++c) {
            const float4 p4 = *reinterpret_cast<const float4*>(pb + t * R + 4 * c);
            pr[4 * c] = p4.x;
            pr[4 * c + 1] = p4.y;
            pr[4 * c + 2] = p4.z;
            pr[4 * c + 3] = p4.w;
          }
        } else {
#pragma unroll
          for (int r = 0; r < R; ++r) pr[r] = pb[t * R + r];
        }
        if (kSets == 2 && (t & 1)) {
#pragma unroll
          for (int r = 0; r < R; ++r) {
            const float2 pp = make_float2(pr[r], pr[r]);
            acc2[r][0] = __ffma2_rn(pp, v0, acc2[r][0]);
            acc2[r][1] = __ffma2_rn(pp, v1, acc2[r][1]);
          }
        } else {
#pragma unroll
          for (int r = 0; r < R; ++r) {
            const float2 pp = make_float2(pr[r], pr[r]);
            acc[r][0] = __ffma2_rn(pp, v0, acc[r][0]);
            acc[r][1] = __ffma2_rn(pp, v1, acc[r][1]);
          }
        }
      }
      if (kSets == 2) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
          acc[r][0] = __fadd2_rn(acc[r][0], acc2[r][0]);
          acc[r][1] = __fadd2_rn(acc[r][1], acc2[r][1]);
        }
      }
      __syncwarp();
      if (lane == 0) {
        *reinterpret_cast<volatile int*>(&sm.slot_consumed[slot]) = n;
        mbar_arrive(&sm.empty[slot]);
      }
    }
    stage_n += nst;

    // ---- merge the NW warp states of this item --------------------------------
#pragma unroll
    for (int r = 0; r < R; ++r)
      *reinterpret_cast<float4*>(&sm.macc[w][r][4 * lane]) =
          make_float4(acc[r][0].x, acc[r][0].y, acc[r][1].x, acc[r][1].y);
    if (tl == 0 && dl < R) {
      sm.mm[w][dl] = m_run;
      sm.ml[w][dl] = l_run;
    }
    named_bar_sync(1, NW * 32);
    decode_finish_item<R, NW, S>(p, sm, ctid, q_start, kv_head, q_len * p.group, slot_out);
  }
  if (p.ext) decode_deferred_merges<R, NW, S>(p, sm, w);
}

// Tensor-core consumer (warp-level m16n8k16 MMA, bf16 in, fp32 accumulate), used with the
// LDGSTS loader.  With R = 8 rows the CUDA-core body needs 8 FMAs per K/V element pair, which
// at HBM rate is most of the SM's FP32 issue; here one stage of 32 tokens is 32 MMAs.
//   S^T[token][row] = K Q^T  : A = K tile (ldmatrix), B = Q^T held in registers for the item;
//   O^T[dim][row]  += V^T P^T : A = V^T (ldmatrix.trans), B = P^T, obtained from the S^T
//                               accumulator fragment by a packed bf16 8x8 transpose (movmatrix).
// Rows R < 8 are padded with zero queries.  The loader stores 16-byte chunk c of token t at
// chunk position c ^ (t & 7), so the eight row addresses of every ldmatrix hit distinct banks.
// Lane l holds query rows 2(l%4), 2(l%4)+1; a row's running max is reduced over the 8 lanes
// that share it; its running sum stays per lane until the end of the item.
// kHalves: the stages hold K and V as two 64-dim halves [2][32 tokens][64], chunk c of a half-row
// at c ^ (t & 7) (the TMA copier's layout), and may hold rows past the stage's last token from a
// request's last page: their V is cleared before the P.V MMAs.  Otherwise [32 tokens][128], chunk
// c (of 16) at c ^ (t & 7), and rows past the last token hold earlier stages' rows.
template <int R, int NW, int S, bool kVar, bool kHalves, bool kMs>
__device__ __forceinline__ void decode_consumer_mma(const DecodeParams& p, DecodeSmem<R, NW, S, kMs>& sm, int begin,
                                                    int end, int w) {
  const int lane = threadIdx.x & 31;
  const int qd = lane & 3;   // row pair 2*qd, 2*qd+1 of the score / output fragments
  const int gq = lane >> 2;  // token (scores) / dim (output) index within an 8-block
  const int ctid = w * 32 + lane;
  // ldmatrix row addresses (element offsets within a stage's K or V tile), swizzled chunks
  const int lk_tok = (lane & 7) + ((lane >> 3) & 1) * 8, lk_chunk = lane >> 4;  // K: m = token, k = dim
  const int lv_tok = (lane & 7) + (lane >> 4) * 8, lv_chunk = (lane >> 3) & 1;  // V^T: m = dim, k = token
  // element offset of 16-byte chunk c16 (of 16) of token t within a stage's K or V tile
  auto chunk_at = [](int t, int c16) {
    if constexpr (kHalves)
      return (c16 >> 3) * (kStageTokens * 64) + t * 64 + (((c16 & 7) ^ (t & 7)) * 8);
    else
      return t * kHeadDim + ((c16 ^ (t & 7)) * 8);
  };

  int stage_n = 0;
  bool alive = true;

  // B fragments of Q^T for an item: row gq, dims 16ks + 2qd (+1) and 16ks + 8 + 2qd (+1); rows past
  // the item's rows are zero
  auto load_q = [&](const int4& a, uint32_t (&dst)[8][2]) {
    const int r = gq;
    if (r < R && r < a.z * p.group) {
      const int tok = a.y + r / p.group;
      const int head = a.w * p.group + r % p.group;
      const uint32_t* qrow = reinterpret_cast<const uint32_t*>(p.q + ((size_t)tok * p.hqo + head) * kHeadDim);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        dst[ks][0] = __ldg(qrow + 8 * ks + qd);
        dst[ks][1] = __ldg(qrow + 8 * ks + 4 + qd);
      }
    } else {
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) dst[ks][0] = dst[ks][1] = 0u;
    }
  };
  // The next item's fields are read when an item starts and its query rows as soon as this warp has
  // issued its last stage of the current item, so both loads overlap the end-of-item merge instead of
  // stalling the next item's first stage (the copier warps stop when the ring is full).
  int4 na = make_int4(0, 0, 0, 0), nb = make_int4(0, 0, 0, 0);
  uint32_t qn[8][2];
  if (begin < end) {
    na = __ldg(reinterpret_cast<const int4*>(p.items + size_t(begin) * kItemFields));
    nb = __ldg(reinterpret_cast<const int4*>(p.items + size_t(begin) * kItemFields + 4));
    load_q(na, qn);
  }

  for (int pos = begin; pos < end; ++pos) {
    const int4 ia = na, ib = nb;
    const int q_start = ia.y, q_len = ia.z, kv_head = ia.w;
    const int kv_lo = ib.x, kv_hi = ib.y, diag = ib.z, slot_out = ib.w;
    const int nst = (kv_hi - kv_lo + kStageTokens - 1) / kStageTokens;
    const int rows_valid = q_len * p.group;
    uint32_t qb[8][2];
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      qb[ks][0] = qn[ks][0];
      qb[ks][1] = qn[ks][1];
    }
    const bool more = pos + 1 < end;
    if (more) {
      na = __ldg(reinterpret_cast<const int4*>(p.items + size_t(pos + 1) * kItemFields));
      nb = __ldg(reinterpret_cast<const int4*>(p.items + size_t(pos + 1) * kItemFields + 4));
    }
    float o[8][4];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
    const int lim0 = diag + (2 * qd) / p.group, lim1 = diag + (2 * qd + 1) / p.group;
    const int low0 = (kVar && p.window_left >= 0) ? lim0 - p.window_left : INT_MIN;
    const int low1 = (kVar && p.window_left >= 0) ? lim1 - p.window_left : INT_MIN;

    for (int st = 0; st < nst; ++st) {
      const int n = stage_n + st;
      if (n % NW != w) continue;
      const int slot = n % S;
      if (!alive) continue;
      const bool got = spin_until_eq(&sm.slot_consumed[slot], n - S, p.err, &sm.abort) &&
                       mbar_wait(&sm.full[slot], (n / S) & 1, p.err, &sm.abort);
      if (!__all_sync(0xffffffffu, got)) {
        alive = false;  // keep joining the named barriers; outputs of an aborted run are undefined
        continue;
      }
      const int t0 = kv_lo + st * kStageTokens;
      const int nt = min(kStageTokens, kv_hi - t0);
      const int n_mt = nt > 16 ? 2 : 1;  // 16-token halves that hold any key of this stage
      const __nv_bfloat16* Ks = &sm.kv[slot][0][0][0];
      const __nv_bfloat16* Vs = &sm.kv[slot][1][0][0];

      // ---- S^T = K Q^T -----------------------------------------------------------
      float s[2][4];
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        s[mt][0] = s[mt][1] = s[mt][2] = s[mt][3] = 0.f;
        if (mt < n_mt) {
          const int tok = 16 * mt + lk_tok;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            uint32_t a[4];
            ldsm_x4(a, Ks + chunk_at(tok, 2 * ks + lk_chunk));
            mma_16816(s[mt], a, qb[ks][0], qb[ks][1]);
          }
        }
      }
      // ---- online softmax (log2 domain) ------------------------------------------
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int t = 16 * mt + 8 * h + gq;
          const bool in = t < nt;
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            bool vis = in && (t0 + t <= (e ? lim1 : lim0));
            float sv = s[mt][2 * h + e] * p.scale_log2;
            if constexpr (kVar) {
              vis = vis && (t0 + t >= (e ? low1 : low0));
              if (p.cap_log2 > 0.f) sv = p.cap_log2 * tanh_exp2(sv * p.inv_cap_log2);
            }
            const float v = vis ? sv : -INFINITY;
            s[mt][2 * h + e] = v;
            mx[e] = fmaxf(mx[e], v);
          }
        }
      }
      float alpha[2], m_use[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        mx[e] = fmaxf(mx[e], __shfl_xor_sync(0xffffffffu, mx[e], 4));
        mx[e] = fmaxf(mx[e], __shfl_xor_sync(0xffffffffu, mx[e], 8));
        mx[e] = fmaxf(mx[e], __shfl_xor_sync(0xffffffffu, mx[e], 16));
        const float m_new = fmaxf(m_run[e], mx[e]);
        m_use[e] = (m_new == -INFINITY) ? 0.f : m_new;
        alpha[e] = fast_exp2(m_run[e] - m_use[e]);
        m_run[e] = m_new;
        l_run[e] *= alpha[e];
      }
      uint32_t pb[2][2];
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const float p0 = fast_exp2(s[mt][2 * h] - m_use[0]);
          const float p1 = fast_exp2(s[mt][2 * h + 1] - m_use[1]);
          l_run[0] += p0;
          l_run[1] += p1;
          pb[mt][h] = movmatrix_trans(f2_to_bf16x2(p0, p1));
        }
      }
      // ---- O^T += V^T P^T -----------------------------------------------------------
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        o[mt][0] *= alpha[0];
        o[mt][1] *= alpha[1];
        o[mt][2] *= alpha[0];
        o[mt][3] *= alpha[1];
      }
#pragma unroll
      for (int kt = 0; kt < 2; ++kt) {
        if (kt < n_mt) {
          const int tok = 16 * kt + lv_tok;
          // kHalves, short stage: this lane's V^T fragments hold tokens 16 kt + 2 qd (+1) in a[0],
          // a[1] and those + 8 in a[2], a[3] (low half: the even token)
          uint32_t m_lo = 0xFFFFFFFFu, m_hi = 0xFFFFFFFFu;
          if (kHalves && nt < kStageTokens) {
            const int tl = 16 * kt + 2 * qd;
            m_lo = (tl < nt ? 0x0000FFFFu : 0u) | (tl + 1 < nt ? 0xFFFF0000u : 0u);
            m_hi = (tl + 8 < nt ? 0x0000FFFFu : 0u) | (tl + 9 < nt ? 0xFFFF0000u : 0u);
          }
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            uint32_t a[4];
            ldsm_x4_trans(a, Vs + chunk_at(tok, 2 * mt + lv_chunk));
            if (kHalves) {
              a[0] &= m_lo;
              a[1] &= m_lo;
              a[2] &= m_hi;
              a[3] &= m_hi;
            }
            mma_16816(o[mt], a, pb[kt][0], pb[kt][1]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) {
        *reinterpret_cast<volatile int*>(&sm.slot_consumed[slot]) = n;
        mbar_arrive(&sm.empty[slot]);
      }
    }
    stage_n += nst;
    if (more) load_q(na, qn);  // lands while the item's states are merged

    // ---- merge the NW warp states of this item --------------------------------
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      l_run[e] += __shfl_xor_sync(0xffffffffu, l_run[e], 4);
      l_run[e] += __shfl_xor_sync(0xffffffffu, l_run[e], 8);
      l_run[e] += __shfl_xor_sync(0xffffffffu, l_run[e], 16);
    }
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int r = 2 * qd + e;
      if (r < R) {
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          sm.macc[w][r][16 * mt + gq] = o[mt][e];
          sm.macc[w][r][16 * mt + 8 + gq] = o[mt][2 + e];
        }
        if (gq == 0) {
          sm.mm[w][r] = m_run[e];
          sm.ml[w][r] = l_run[e];
        }
      }
    }
    named_bar_sync(1, NW * 32);
    decode_finish_item<R, NW, S>(p, sm, ctid, q_start, kv_head, rows_valid, slot_out);
  }
  // composable plans: the deferred merges follow in decode_body, by every warp of the CTA
}

// kMma selects the tensor-core consumer (LDGSTS loader only, whose copies it swizzles).
// kFlags: kDecodeNhd (NHD pages, 16-byte-copy loader only; bits 4-6 hold log2(H_kv)),
// kDecodeVariant (sliding window / soft-cap).
constexpr int kDecodeNhd = 1;
constexpr int kDecodeVariant = 2;
constexpr int kDecodeTma = 8;  // HND pages of 8+ tokens: TMA copier, stages in 64-dim halves
constexpr int kDecodeNhdHeadsShift = 4;
// kFlags & kDecodeTma: the copiers issue TMA boxes (tm_k / tm_v) instead of 16-byte copies; the
// stages then hold 64-dim halves and shared memory is aligned to 1 KB here (the launch adds the
// slack) for the 128-byte swizzle.
template <int R, int NW, int S, int kCopiers, bool kMma, int kFlags>
__device__ __forceinline__ void decode_body(const DecodeParams& p, const CUtensorMap* tm_k, const CUtensorMap* tm_v) {
  static_assert(!kMma || kCopiers > 0, "the tensor-core consumer reads swizzled LDGSTS stages");
  static_assert(!(kFlags & kDecodeNhd) || kCopiers > 0, "NHD pages are read by the 16-byte-copy loader");
  constexpr bool kVar = (kFlags & kDecodeVariant) != 0;
  constexpr bool kTma = (kFlags & kDecodeTma) != 0;
  static_assert(!kTma || (kMma && !(kFlags & kDecodeNhd)), "the TMA copier feeds the tensor-core consumer, HND pages");
  constexpr bool kLdgsts = kCopiers > 0;
  constexpr int kLoaders = kLdgsts ? 1 + kCopiers : 1;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  auto& sm = *reinterpret_cast<DecodeSmem<R, NW, S, kMma>*>(
      kTma ? ((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023)) : reinterpret_cast<uintptr_t>(smem_raw));
  const int warp = threadIdx.x >> 5;
  if constexpr (kTma) {
    if (threadIdx.x == 32) {  // first copier warp: fetch the two maps while the CTA sets up
      tc::tma_prefetch_desc(tm_k);
      tc::tma_prefetch_desc(tm_v);
    }
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      sm.slot_consumed[s] = s - S;
      sm.slot_filled[s] = s - S;
      // LDGSTS: one arrival per lane of the stage's copier; TMA and bulk copies: the expect-tx arrival
      mbar_init(&sm.full[s], kLdgsts && !kTma ? 32 : 1);
      mbar_init(&sm.empty[s], 1);
    }
    for (int s = 0; s < kIdxSlots; ++s) {
      mbar_init(&sm.idx_full[s], 32);
      mbar_init(&sm.idx_empty[s], 1);
    }
    sm.abort = 0;
    sm.flag = 0;
    sm.n_deferred = 0;
    fence_mbar_init();
  }
  if constexpr (kMma) {
    // Rows past the end of a short stage are read by the P.V MMA with weight 0: they must hold
    // finite values, so the V ring starts zeroed (later it holds earlier stages' V rows).
    for (int i = threadIdx.x; i < S * kStageTokens * kHeadDim / 8; i += blockDim.x) {
      const int st = i / (kStageTokens * kHeadDim / 8), rem = i % (kStageTokens * kHeadDim / 8);
      reinterpret_cast<uint4*>(&sm.kv[st][1][0][0])[rem] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  __syncthreads();
  if (p.wait_prior) asm volatile("griddepcontrol.wait;" ::: "memory");
  // a following launch made dependent on this one may start its own set-up as SMs free up; it waits
  // for this grid before it reads memory.  Triggered after the wait above, so a follower can never
  // run ahead of the kernel before this one.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int begin = __ldg(p.cta_indptr + blockIdx.x);
  const int end = __ldg(p.cta_indptr + blockIdx.x + 1);
  if (warp >= kLoaders) {
    if constexpr (kMma)
      decode_consumer_mma<R, NW, S, kVar, kTma>(p, sm, begin, end, warp - kLoaders);
    else
      decode_consumer<R, NW, S, kVar>(p, sm, begin, end, warp - kLoaders);
  } else if (!kLdgsts) {
    decode_producer<R, NW, S>(p, sm, begin, end);
  } else if (warp == 0) {
    decode_index_warp<R, NW, S>(p, sm, begin, end);
  } else if constexpr (kTma) {
    decode_tma_copier<R, NW, S, kCopiers>(p, sm, tm_k, tm_v, begin, end, warp - 1);
  } else {
    constexpr int kNhdStride = (kFlags & kDecodeNhd) ? kHeadDim << ((kFlags >> kDecodeNhdHeadsShift) & 7) : 0;
    decode_copier_warp<R, NW, S, kCopiers, kMma, kNhdStride>(p, sm, begin, end, warp - 1);
  }
  if constexpr (kMma) {
    // composable plans: once every warp is done (the consumers' last item merge ended with their
    // barrier, so the deferred list is final), all warps merge the deferred rows with the shared
    // part's states.  Every role of this kernel returns here, aborted or not.
    if (p.ext != nullptr) {
      __syncthreads();
      decode_deferred_merges_cta<R>(p, sm, warp, int(blockDim.x >> 5));
    }
  }
}

template <int R, int NW, int S, int kCopiers = 0, bool kMma = false, int kFlags = 0>
__global__ void __launch_bounds__((NW + (kCopiers ? 1 + kCopiers : 1)) * 32, 1)
    decode_kernel(const __grid_constant__ DecodeParams p) {
  static_assert(!(kFlags & kDecodeTma), "TMA copies run in decode_kernel_tma");
  decode_body<R, NW, S, kCopiers, kMma, kFlags>(p, nullptr, nullptr);
}

template <int R, int NW, int S, int kCopiers, int kFlags>
__global__ void __launch_bounds__((NW + 1 + kCopiers) * 32, 1)
    decode_kernel_tma(const __grid_constant__ DecodeParams p, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v) {
  decode_body<R, NW, S, kCopiers, true, kFlags | kDecodeTma>(p, &tm_k, &tm_v);
}

}  // namespace fi
