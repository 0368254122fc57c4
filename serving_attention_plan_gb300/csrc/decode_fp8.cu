// Launch of the FP8-KV decode kernel (核心机制 8, paper App. F), one instantiation per rows-per-tile.
#include "decode_fp8.cuh"
#include "decode_launch.cuh"
#include "prefill_launch.h"

namespace fi {

namespace {

// Eight consumer warps and a ring of 16 KB stages: 12, or 11 when R = 8 rows need a larger merge
// buffer.  Measured on GB300 (Llama-3-8B-shaped batch): 4 / 6 / 10 consumer warps were slower, and
// so were two warps per stage (32 tokens each) and widening the codes with integer ops instead of
// the cvt instruction.
constexpr int kFp8Warps = 8;
template <int R>
constexpr int kFp8Stages = R >= 8 ? 11 : 12;

template <int R, bool kNhd, bool kTma>
int launch_fp8_as(int grid, const DecodeParams& p, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                  cudaStream_t stream, bool pdl) {
  using Smem = DecodeSmemFp8<R, kFp8Warps, kFp8Stages<R>>;
  constexpr size_t kSmemBytes = sizeof(Smem) + 1024;  // slack for the kernel's 1 KB alignment
  static_assert(kSmemBytes <= 227 * 1024, "decode shared memory exceeds the per-CTA limit");
  auto kernel = decode_kernel_fp8<R, kFp8Warps, kFp8Stages<R>, kDecodeCopiers, kNhd, kTma>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [&] {
    attr_err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kSmemBytes));
  });
  if (attr_err != cudaSuccess) return record_cuda_error(attr_err, "cudaFuncSetAttribute(decode fp8)");
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(grid));
  cfg.blockDim = dim3((kFp8Warps + 1 + kDecodeCopiers) * 32);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, p, tm_k, tm_v);
  return e == cudaSuccess ? FI_OK : record_cuda_error(e, "decode_kernel_fp8 launch");
}

// Pages of 8 or more tokens take the TMA copier (each box at least 1 KB, so boxes start on the
// 1 KB boundaries the 128-byte swizzle needs); smaller pages the 16-byte copies.
template <int R, bool kNhd>
int launch_fp8_rows(int grid, const DecodeParams& p, cudaStream_t stream, bool pdl) {
  CUtensorMap tm_k{}, tm_v{};
  if (p.page_size < 8) return launch_fp8_as<R, kNhd, false>(grid, p, tm_k, tm_v, stream, pdl);
  const int hkv = int(p.page_stride / (int64_t(p.page_size) * kHeadDim));
  const int box_rows = p.page_size < kFp8StageTokens ? p.page_size : kFp8StageTokens;  // as the copier's boxes
  if (!make_decode_map_e4m3(&tm_k, p.k, hkv, p.page_size, p.num_pages, kNhd, box_rows) ||
      !make_decode_map_e4m3(&tm_v, p.v, hkv, p.page_size, p.num_pages, kNhd, box_rows))
    return FI_ERR_INVALID_ARG;
  return launch_fp8_as<R, kNhd, true>(grid, p, tm_k, tm_v, stream, pdl);
}

}  // namespace

int launch_decode_fp8(int rows_tile, bool nhd, int grid, const DecodeParams& p, cudaStream_t stream, bool pdl) {
  if (p.page_shift < 0) return FI_ERR_UNSUPPORTED;
  switch (rows_tile * 2 + (nhd ? 1 : 0)) {
    case 2: return launch_fp8_rows<1, false>(grid, p, stream, pdl);
    case 3: return launch_fp8_rows<1, true>(grid, p, stream, pdl);
    case 4: return launch_fp8_rows<2, false>(grid, p, stream, pdl);
    case 5: return launch_fp8_rows<2, true>(grid, p, stream, pdl);
    case 8: return launch_fp8_rows<4, false>(grid, p, stream, pdl);
    case 9: return launch_fp8_rows<4, true>(grid, p, stream, pdl);
    case 16: return launch_fp8_rows<8, false>(grid, p, stream, pdl);
    case 17: return launch_fp8_rows<8, true>(grid, p, stream, pdl);
    default: return FI_ERR_UNSUPPORTED;
  }
}

}  // namespace fi
