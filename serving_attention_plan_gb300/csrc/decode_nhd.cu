// Decode kernels for NHD pages ([pages, page_size, H_kv, 128]), one per rows-per-tile and
// log2(H_kv) in 0..4; they carry the attention-variant code too (the page layout and variants of
// 核心机制 5, paper §3.2.3).  Separate from the HND kernels so the two compile in parallel.
#include "decode_launch.cuh"

namespace fi {

namespace {

template <int R>
int launch_nhd_rows(int log2_heads, int grid, const DecodeParams& p, cudaStream_t stream, bool pdl) {
  constexpr int kF = kDecodeNhd | kDecodeVariant;
  switch (log2_heads) {
    case 0: return launch_decode_as<R, kDecodeCopiers, kF | (0 << kDecodeNhdHeadsShift)>(grid, p, stream, pdl);
    case 1: return launch_decode_as<R, kDecodeCopiers, kF | (1 << kDecodeNhdHeadsShift)>(grid, p, stream, pdl);
    case 2: return launch_decode_as<R, kDecodeCopiers, kF | (2 << kDecodeNhdHeadsShift)>(grid, p, stream, pdl);
    case 3: return launch_decode_as<R, kDecodeCopiers, kF | (3 << kDecodeNhdHeadsShift)>(grid, p, stream, pdl);
    case 4: return launch_decode_as<R, kDecodeCopiers, kF | (4 << kDecodeNhdHeadsShift)>(grid, p, stream, pdl);
    default: return FI_ERR_UNSUPPORTED;
  }
}

}  // namespace

int launch_decode_nhd(int rows_tile, int log2_heads, int grid, const DecodeParams& p, cudaStream_t stream,
                      bool pdl) {
  if (p.page_shift < 0) return FI_ERR_UNSUPPORTED;
  switch (rows_tile) {
    case 1: return launch_nhd_rows<1>(log2_heads, grid, p, stream, pdl);
    case 2: return launch_nhd_rows<2>(log2_heads, grid, p, stream, pdl);
    case 4: return launch_nhd_rows<4>(log2_heads, grid, p, stream, pdl);
    case 8: return launch_nhd_rows<8>(log2_heads, grid, p, stream, pdl);
    default: return FI_ERR_UNSUPPORTED;
  }
}

}  // namespace fi
