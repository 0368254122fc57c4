// Merge of two attention states per (row, head): the composable-format step.
//
// Page "FlashInfer：面向 LLM 推理服务的高效可定制注意力引擎", 术语与记号
// "Attention State 与 ⊕" (paper §2.2) and 核心机制 2 (paper §3.1.2, Fig. 3):
// states over disjoint key sets combine with an associative operator,
//   s = log(e^s_a + e^s_b),  O = e^(s_a - s) O_a + e^(s_b - s) O_b,
// identity (0, -inf).  Evaluated in base 2 with the larger LSE factored out.
#pragma once

#include "device_common.cuh"

namespace fi {

// One warp per (row, head); lane owns 4 of the 128 dims.
__global__ void __launch_bounds__(256) merge_states_kernel(const __nv_bfloat16* __restrict__ o_a,
                                                           const float* __restrict__ lse_a,
                                                           const __nv_bfloat16* __restrict__ o_b,
                                                           const float* __restrict__ lse_b, __nv_bfloat16* o,
                                                           float* lse, long long n_rows) {
  const int lane = threadIdx.x & 31;
  const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long r = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < n_rows; r += warps) {
    const float sa = lse_a[r] * kLog2e;
    const float sb = lse_b[r] * kLog2e;
    const float m = fmaxf(sa, sb);
    const uint2 ra = *reinterpret_cast<const uint2*>(o_a + r * kHeadDim + 4 * lane);
    const uint2 rb = *reinterpret_cast<const uint2*>(o_b + r * kHeadDim + 4 * lane);
    float4 out = make_float4(0.f, 0.f, 0.f, 0.f);
    float s_out = -INFINITY;
    if (m != -INFINITY) {
      const float wa = fast_exp2(sa - m), wb = fast_exp2(sb - m);
      const float z = wa + wb;
      const float ia = wa / z, ib = wb / z;
      const float2 a0 = bf16x2_to_f2(ra.x), a1 = bf16x2_to_f2(ra.y);
      const float2 b0 = bf16x2_to_f2(rb.x), b1 = bf16x2_to_f2(rb.y);
      out = make_float4(ia * a0.x + ib * b0.x, ia * a0.y + ib * b0.y, ia * a1.x + ib * b1.x, ia * a1.y + ib * b1.y);
      s_out = (m + fast_log2(z)) * kLn2;
    }
    __syncwarp();  // every lane has read its inputs before o (which may alias o_a/o_b) is written
    uint2 packed;
    packed.x = f2_to_bf16x2(out.x, out.y);
    packed.y = f2_to_bf16x2(out.z, out.w);
    *reinterpret_cast<uint2*>(o + r * kHeadDim + 4 * lane) = packed;
    if (lane == 0) lse[r] = s_out;
  }
}

}  // namespace fi
