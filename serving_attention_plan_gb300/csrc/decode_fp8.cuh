// Decode tiles over FP8 (e4m3) KV pages.
//
// Page "FlashInfer：面向 LLM 推理服务的高效可定制注意力引擎", 核心机制 8 (paper App. F):
// a mixed-precision kernel keeps queries and outputs in 16-bit floats and the KV-cache in fp8,
// dequantising with a fast numeric converter.  Here: one scale per tensor (K = k_scale * code,
// V = v_scale * code); the 16-byte-copy loader moves 128-byte K/V rows (half the bytes of bf16)
// into a ring of 64-token stages (8 KB of K + 8 KB of V: the bytes of a bf16 stage, so the
// loader's fixed cost per stage is spread over as many bytes), 16-byte chunk c of token t at
// chunk position c ^ (t & 7).
// Consumer warps read MMA fragments straight from the e4m3 stage with ldmatrix (b16 view: each
// lane receives four codes) and widen them in registers to f16 (exact), then run f16 warp MMAs
// (Q converted from bf16 once per item, P rounded to f16).  The K scale is folded into the
// logit scale and the V scale into the output.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>

#include "decode_kernel.cuh"
#include "tcgen05.cuh"

namespace fi {

constexpr int kFp8StageTokens = 64;

template <int R, int NW, int S>
struct DecodeSmemFp8 {
  uint8_t kv8[S][2][kFp8StageTokens][kHeadDim];  // [stage][K|V][token][dim chunks swizzled] e4m3 codes
  float macc[NW][R][kHeadDim];
  float mm[NW][8];
  float ml[NW][8];
  int32_t idx[kIdxSlots][kFp8StageTokens];
  uint64_t full[S];
  uint64_t empty[S];
  uint64_t idx_full[kIdxSlots];
  uint64_t idx_empty[kIdxSlots];
  int slot_consumed[S];  // as in DecodeSmem: keeps every parity wait unambiguous
  int slot_filled[S];
  int flag;
  int abort;
};

// Two e4m3 codes -> f16x2 (code of bits 0-7 in the low half), exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_codes) {
  uint32_t r;
  const uint16_t v = static_cast<uint16_t>(two_codes);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
  return r;
}

// d (16x8 fp32) += a (16x16 f16, row-major) * b (16x8 f16, column-major)
__device__ __forceinline__ void mma_16816_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
               "{%0,%1,%2,%3};"
               : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
               : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t f2_to_f16x2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Copier warp `cw` of kCopiers: stages cw, cw + kCopiers, ...; a warp instruction moves four
// 128-byte rows (lane = token (lane / 8) of the four, 16-byte chunk lane % 8).  HND pages hold a
// head's rows 128 bytes apart; NHD pages (kNhd) H_kv * 128 bytes apart, i.e. the page stride over
// the page size, a power of two (H_kv is one for NHD decode).  Page ids of the
// stage's segments: lane l holds those of segments l and l + 32 (64 segments only with 1-token
// pages; stages start on a page boundary, so segment = token >> page_shift).
template <int R, int NW, int S, int kCopiers, bool kNhd>
__device__ __forceinline__ void decode_copier_fp8(const DecodeParams& p, DecodeSmemFp8<R, NW, S>& sm, int begin,
                                                  int end, int cw) {
  const int lane = threadIdx.x & 31;
  const int sh = p.page_shift;
  const int row_mask = p.page_size - 1;
  const int nhd_row_shift = kNhd ? __ffsll(p.page_stride >> sh) - 1 : 0;  // log2(H_kv * 128)
  StageCursorT<kFp8StageTokens> c{begin, end, 0, 0, 0, 0, 0, 0};
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
    int pg_hi = (lane + 32 < nseg) ? sm.idx[islot][lane + 32] : 0;
    if (lane < nseg && (pg < 0 || pg >= p.num_pages)) {
      atomicOr(p.err, FI_DEVERR_PAGE_OOB);
      pg = -1;
    }
    if (lane + 32 < nseg && (pg_hi < 0 || pg_hi >= p.num_pages)) {
      atomicOr(p.err, FI_DEVERR_PAGE_OOB);
      pg_hi = -1;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.idx_empty[islot]);
    const int slot = n % S, fill = n / S;
    if (!__all_sync(0xffffffffu, spin_until_eq(&sm.slot_filled[slot], n - S, p.err, &sm.abort))) break;
    if (fill > 0 && !__all_sync(0xffffffffu, mbar_wait(&sm.empty[slot], (fill - 1) & 1, p.err, &sm.abort))) break;
    const uint8_t* kb = reinterpret_cast<const uint8_t*>(p.k) + (long long)c.kv_head * p.head_stride;
    const uint8_t* vb = reinterpret_cast<const uint8_t*>(p.v) + (long long)c.kv_head * p.head_stride;
#pragma unroll
    for (int j = 0; j < kFp8StageTokens / 4; ++j) {
      const int tok = 4 * j + (lane >> 3);
      const int pos = t0 + tok;
      const int seg = min(max((pos >> sh) - first, 0), kFp8StageTokens - 1);
      int page = __shfl_sync(0xffffffffu, pg, seg & 31);
      if (j >= 8) {  // tokens 32..63: segment >= 32 only for 1-token pages
        const int hi = __shfl_sync(0xffffffffu, pg_hi, seg & 31);
        page = seg >= 32 ? hi : page;
      }
      if (tok < nt && page >= 0) {
        long long off;
        if constexpr (kNhd) {
          off = (long long)page * p.page_stride + ((long long)(pos & row_mask) << nhd_row_shift) + (lane & 7) * 16;
        } else {
          off = (long long)page * p.page_stride + (long long)(pos & row_mask) * kHeadDim + (lane & 7) * 16;
        }
        const int sw = ((lane & 7) ^ (tok & 7)) * 16;
        cp_async_16(&sm.kv8[slot][0][tok][sw], kb + off);
        cp_async_16(&sm.kv8[slot][1][tok][sw], vb + off);
      }
    }
    cp_async_arrive_noinc(&sm.full[slot]);
    __syncwarp();
    if (lane == 0) *reinterpret_cast<volatile int*>(&sm.slot_filled[slot]) = n;
    for (int k = 0; k < kCopiers && ok; ++k) ok = c.next(p.items);
  }
  cp_async_wait_all();
}

// TMA variant of the copier (pages of at least 8 tokens): copier warp `cw` issues its stages as
// tensor boxes, one per page (or per 64-token run of a longer page) for K and one for V, each box
// page_tokens rows of 128 codes landing in the 128-byte swizzle, which puts 16-byte chunk c of
// token t at chunk position c ^ (t & 7): the layout the consumers read.  A box of 8 or more rows
// is at least 1 KB, so every box starts on a 1 KB boundary of the stage.  The copies bypass the
// load/store pipeline the consumers' shared-memory instructions use.  Boxes are whole pages, so a
// request's last page may bring codes past its last token: those rows are masked by the consumers.
// tm_k / tm_v: HND (codes, token in page, page * H_kv + head) or NHD (codes, head, token, page).
template <int R, int NW, int S, int kCopiers, bool kNhd>
__device__ __forceinline__ void decode_tma_copier_fp8(const DecodeParams& p, DecodeSmemFp8<R, NW, S>& sm,
                                                      const CUtensorMap* tm_k, const CUtensorMap* tm_v, int begin,
                                                      int end, int cw) {
  const int lane = threadIdx.x & 31;
  const int sh = p.page_shift;
  const int box_tok = min(p.page_size, kFp8StageTokens);  // rows of a box
  const int hkv = int(p.page_stride >> (sh + 7));        // page stride = H_kv * page_size * 128 codes
  StageCursorT<kFp8StageTokens> c{begin, end, 0, 0, 0, 0, 0, 0};
  bool ok = c.load(p.items);
  for (int k = 0; k < cw && ok; ++k) ok = c.next(p.items);
  int issued_last = -1;  // this warp's last stage
  for (int n = cw; ok; n += kCopiers) {
    const int islot = n % kIdxSlots;
    if (!__all_sync(0xffffffffu, mbar_wait(&sm.idx_full[islot], (n / kIdxSlots) & 1, p.err, &sm.abort))) break;
    const int t0 = c.tok0();
    const int nt = c.ntok();
    // boxes of this stage: pages from the stage's first token (stages start on a page boundary, or
    // on a 64-token boundary inside a longer page)
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
    const uint32_t bytes = pg >= 0 ? uint32_t(2 * box_tok * kHeadDim) : 0u;
    const uint32_t total = __reduce_add_sync(0xffffffffu, bytes);
    if (lane == 0) mbar_arrive_expect_tx(&sm.full[slot], total);
    __syncwarp();
    if (pg >= 0) {
      const int y = t0 & (p.page_size - 1) & ~(box_tok - 1);  // 0 unless pages are longer than a stage
      uint8_t* dk = &sm.kv8[slot][0][lane * box_tok][0];
      uint8_t* dv = &sm.kv8[slot][1][lane * box_tok][0];
      if constexpr (kNhd) {
        tc::tma_load_4d(dk, tm_k, 0, c.kv_head, y, pg, &sm.full[slot]);
        tc::tma_load_4d(dv, tm_v, 0, c.kv_head, y, pg, &sm.full[slot]);
      } else {
        tc::tma_load_3d(dk, tm_k, 0, y, pg * hkv + c.kv_head, &sm.full[slot]);
        tc::tma_load_3d(dv, tm_v, 0, y, pg * hkv + c.kv_head, &sm.full[slot]);
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

// Consumer warp w: stages w, w + NW, ... of the CTA's queue.  Fragment layouts as in
// decode_consumer_mma, with the reduction dimension permuted where that lets ldmatrix hand each
// lane whole code groups (a permutation of the summed index changes nothing):
//   S^T = K Q^T: an x4 ldmatrix of tokens 16mt..+15 x dim chunks 2kb, 2kb+1 gives lane (gq, qd)
//     codes of dims 16c + 4qd .. +3 of tokens gq and gq + 8; MMA k-slot 2qd, 2qd+1 takes dims
//     16c + 4qd, +1 and k-slot 8 + 2qd, +1 takes dims 16c + 4qd + 2, +3, so the Q^T fragment of
//     query row gq is dims 16c + 4qd .. +3 (one 8-byte load per chunk c).
//   O^T += V^T P^T: an x4 transposing ldmatrix of tokens 16kt..+15 x chunks 2db, 2db+1 gives lane
//     (gq, qd) codes of tokens 2qd, 2qd+1 (and 8 + those) at dims 2gq, 2gq+1 of each chunk; a byte
//     permute splits them into the even-dim and the odd-dim fragment, so output tile mt = 2db + e
//     holds dims 32db + 2gq + e (rows gq) and 32db + 16 + 2gq + e (rows gq + 8).
// kWholePages: stages were filled with whole pages (the TMA copier), so rows past the stage's last
// token may hold codes from past a request's last token (possibly NaN codes): their V codes are
// cleared before the P.V MMAs, where a zero weight would not cancel a NaN.
template <int R, int NW, int S, bool kWholePages = false>
__device__ __forceinline__ void decode_consumer_fp8(const DecodeParams& p, DecodeSmemFp8<R, NW, S>& sm, int begin,
                                                    int end, int w) {
  const int lane = threadIdx.x & 31;
  const int qd = lane & 3;
  const int gq = lane >> 2;
  const int ctid = w * 32 + lane;
  const int lk_tok = (lane & 7) + ((lane >> 3) & 1) * 8, lk_chunk = lane >> 4;  // K x4: tokens, then chunk
  const int lv_tok = (lane & 7) + ((lane >> 3) & 1) * 8, lv_chunk = lane >> 4;  // V x4: same matrices

  int stage_n = 0;
  bool alive = true;
  for (int pos = begin; pos < end; ++pos) {
    const int4 ia = __ldg(reinterpret_cast<const int4*>(p.items + size_t(pos) * kItemFields));
    const int4 ib = __ldg(reinterpret_cast<const int4*>(p.items + size_t(pos) * kItemFields + 4));
    const int q_start = ia.y, q_len = ia.z, kv_head = ia.w;
    const int kv_lo = ib.x, kv_hi = ib.y, diag = ib.z, slot_out = ib.w;
    const int nst = (kv_hi - kv_lo + kFp8StageTokens - 1) / kFp8StageTokens;
    const int rows_valid = q_len * p.group;

    // Q^T fragments in f16: query row gq, dims 16c + 4qd .. +3 for chunk c
    uint32_t qb[8][2];
    if (gq < R && gq < rows_valid) {
      const int tok = q_start + gq / p.group;
      const int head = kv_head * p.group + gq % p.group;
      const uint2* qrow = reinterpret_cast<const uint2*>(p.q + ((size_t)tok * p.hqo + head) * kHeadDim);
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint2 u = __ldg(qrow + 4 * c + qd);
        const float2 a = bf16x2_to_f2(u.x), b = bf16x2_to_f2(u.y);
        qb[c][0] = f2_to_f16x2(a.x, a.y);
        qb[c][1] = f2_to_f16x2(b.x, b.y);
      }
    } else {
#pragma unroll
      for (int c = 0; c < 8; ++c) qb[c][0] = qb[c][1] = 0u;
    }
    float o[8][4];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
    const int lim0 = diag + (2 * qd) / p.group, lim1 = diag + (2 * qd + 1) / p.group;
    const int low0 = p.window_left >= 0 ? lim0 - p.window_left : INT_MIN;
    const int low1 = p.window_left >= 0 ? lim1 - p.window_left : INT_MIN;

    for (int st = 0; st < nst; ++st) {
      const int n = stage_n + st;
      if (n % NW != w) continue;
      const int slot = n % S;
      if (!alive) continue;
      const bool got = spin_until_eq(&sm.slot_consumed[slot], n - S, p.err, &sm.abort) &&
                       mbar_wait(&sm.full[slot], (n / S) & 1, p.err, &sm.abort);
      if (!__all_sync(0xffffffffu, got)) {
        alive = false;
        continue;
      }
      const int t0 = kv_lo + st * kFp8StageTokens;
      const int nt = min(kFp8StageTokens, kv_hi - t0);
      const int n_mt = (nt + 15) >> 4;
      const uint8_t* Ks = &sm.kv8[slot][0][0][0];
      const uint8_t* Vs = &sm.kv8[slot][1][0][0];

      constexpr int kMt = kFp8StageTokens / 16;
      float s[kMt][4];
#pragma unroll
      for (int mt = 0; mt < kMt; ++mt) {
        s[mt][0] = s[mt][1] = s[mt][2] = s[mt][3] = 0.f;
        if (mt < n_mt) {
          const int tok = 16 * mt + lk_tok;
          const uint8_t* row = Ks + tok * kHeadDim;
#pragma unroll
          for (int kb = 0; kb < 4; ++kb) {
            uint32_t r[4];
            ldsm_x4(r, row + (((2 * kb + lk_chunk) ^ (tok & 7)) * 16));
#pragma unroll
            for (int h = 0; h < 2; ++h) {  // chunk 2kb + h: registers r[2h] (token gq), r[2h+1] (gq + 8)
              uint32_t a[4];
              a[0] = e4m3x2_to_f16x2(r[2 * h]);
              a[1] = e4m3x2_to_f16x2(r[2 * h + 1]);
              a[2] = e4m3x2_to_f16x2(r[2 * h] >> 16);
              a[3] = e4m3x2_to_f16x2(r[2 * h + 1] >> 16);
              mma_16816_f16(s[mt], a, qb[2 * kb + h][0], qb[2 * kb + h][1]);
            }
          }
        }
      }
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int mt = 0; mt < kMt; ++mt) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int t = 16 * mt + 8 * h + gq;
          const bool in = t < nt;
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const bool vis = in && (t0 + t <= (e ? lim1 : lim0)) && (t0 + t >= (e ? low1 : low0));
            float sv = s[mt][2 * h + e] * p.scale_log2;
            if (p.cap_log2 > 0.f) sv = p.cap_log2 * tanh_exp2(sv * p.inv_cap_log2);
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
      uint32_t pb[kMt][2];
#pragma unroll
      for (int mt = 0; mt < kMt; ++mt) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const float p0 = fast_exp2(s[mt][2 * h] - m_use[0]);
          const float p1 = fast_exp2(s[mt][2 * h + 1] - m_use[1]);
          l_run[0] += p0;
          l_run[1] += p1;
          pb[mt][h] = movmatrix_trans(f2_to_f16x2(p0, p1));
        }
      }
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        o[mt][0] *= alpha[0];
        o[mt][1] *= alpha[1];
        o[mt][2] *= alpha[0];
        o[mt][3] *= alpha[1];
      }
#pragma unroll
      for (int kt = 0; kt < kMt; ++kt) {
        if (kt < n_mt) {
          const int tok = 16 * kt + lv_tok;
          const uint8_t* row = Vs + tok * kHeadDim;
#pragma unroll
          for (int db = 0; db < 4; ++db) {
            // r[0]: tokens 2qd, 2qd+1 x dims 2gq, 2gq+1 of chunk 2db; r[1]: tokens + 8;
            // r[2], r[3]: the same for chunk 2db + 1.  Bytes of each: [t0 d0, t0 d1, t1 d0, t1 d1].
            uint32_t r[4];
            ldsm_x4_trans(r, row + (((2 * db + lv_chunk) ^ (tok & 7)) * 16));
            if (kWholePages && nt < kFp8StageTokens) {
              // tokens of r[0] / r[2]: 16 kt + 2 qd (bytes 0-1) and + 1 (bytes 2-3); r[1] / r[3]: + 8
              const int tl = 16 * kt + 2 * qd;
              const uint32_t m_lo = (tl < nt ? 0x0000FFFFu : 0u) | (tl + 1 < nt ? 0xFFFF0000u : 0u);
              const uint32_t m_hi = (tl + 8 < nt ? 0x0000FFFFu : 0u) | (tl + 9 < nt ? 0xFFFF0000u : 0u);
              r[0] &= m_lo;
              r[2] &= m_lo;
              r[1] &= m_hi;
              r[3] &= m_hi;
            }
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              uint32_t a[4];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                // fragment order: (chunk 2db, tokens lo), (chunk 2db+1, lo), (2db, hi), (2db+1, hi)
                const uint32_t x = r[(i & 1) * 2 + (i >> 1)];
                const uint32_t y = __byte_perm(x, 0u, 0x3120);  // [t0 d0, t1 d0, t0 d1, t1 d1]
                a[i] = e4m3x2_to_f16x2(e ? (y >> 16) : y);
              }
              mma_16816_f16(o[2 * db + e], a, pb[kt][0], pb[kt][1]);
            }
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
        for (int db = 0; db < 4; ++db) {  // the V scale enters with the unnormalised output
#pragma unroll
          for (int ee = 0; ee < 2; ++ee) {
            sm.macc[w][r][32 * db + 2 * gq + ee] = o[2 * db + ee][e] * p.v_scale;
            sm.macc[w][r][32 * db + 16 + 2 * gq + ee] = o[2 * db + ee][2 + e] * p.v_scale;
          }
        }
        if (gq == 0) {
          sm.mm[w][r] = m_run[e];
          sm.ml[w][r] = l_run[e];
        }
      }
    }
    named_bar_sync(1, NW * 32);
    decode_finish_item<R, NW, S, DecodeSmemFp8<R, NW, S>, false>(p, sm, ctid, q_start, kv_head, rows_valid, slot_out);
  }
}

// kTma: the copiers issue tensor boxes of whole pages (pages of 8 or more tokens) instead of
// 16-byte copies; tm_k / tm_v are then the K and V page maps (unused otherwise).  Shared memory is
// aligned to 1 KB here (the launch adds the slack): the boxes land 128-byte swizzled.
template <int R, int NW, int S, int kCopiers, bool kNhd, bool kTma = false>
__global__ void __launch_bounds__((NW + 1 + kCopiers) * 32, 1)
    decode_kernel_fp8(const __grid_constant__ DecodeParams p, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  auto& sm = *reinterpret_cast<DecodeSmemFp8<R, NW, S>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                          ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  if constexpr (kTma) {
    if (threadIdx.x == 32) {  // first copier warp: fetch the two maps while the CTA sets up
      tc::tma_prefetch_desc(&tm_k);
      tc::tma_prefetch_desc(&tm_v);
    }
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      sm.slot_consumed[s] = s - S;
      sm.slot_filled[s] = s - S;
      // LDGSTS: one arrival per lane of the stage's copier; TMA: the copier's expect-tx arrival
      mbar_init(&sm.full[s], kTma ? 1 : 32);
      mbar_init(&sm.empty[s], 1);
    }
    for (int s = 0; s < kIdxSlots; ++s) {
      mbar_init(&sm.idx_full[s], 32);
      mbar_init(&sm.idx_empty[s], 1);
    }
    sm.abort = 0;
    sm.flag = 0;
    fence_mbar_init();
  }
  // Rows past the end of a short stage are read by the P.V MMA with weight 0: they must hold
  // finite values, so the V ring starts as zero codes (later: earlier stages' codes).
  for (int i = threadIdx.x; i < S * kFp8StageTokens * kHeadDim / 16; i += blockDim.x) {
    const int st = i / (kFp8StageTokens * kHeadDim / 16), rem = i % (kFp8StageTokens * kHeadDim / 16);
    reinterpret_cast<uint4*>(&sm.kv8[st][1][0][0])[rem] = make_uint4(0u, 0u, 0u, 0u);
  }
  __syncthreads();
  if (p.wait_prior) asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");  // as in decode_kernel
  const int begin = __ldg(p.cta_indptr + blockIdx.x);
  const int end = __ldg(p.cta_indptr + blockIdx.x + 1);
  if (warp > kCopiers) {
    decode_consumer_fp8<R, NW, S, kTma>(p, sm, begin, end, warp - 1 - kCopiers);
  } else if (warp == 0) {
    decode_index_warp<R, NW, S, DecodeSmemFp8<R, NW, S>, kFp8StageTokens>(p, sm, begin, end);
  } else if constexpr (kTma) {
    decode_tma_copier_fp8<R, NW, S, kCopiers, kNhd>(p, sm, &tm_k, &tm_v, begin, end, warp - 1);
  } else {
    decode_copier_fp8<R, NW, S, kCopiers, kNhd>(p, sm, begin, end, warp - 1);
  }
}

}  // namespace fi
