// Launch of the decode kernel, shared by the translation units that instantiate it.
#pragma once

#include <cuda_runtime.h>

#include <mutex>

#include "../../include/fi.h"
#include "decode_kernel.cuh"
#include "prefill_launch.h"

namespace fi {

// Consumer warps and ring depth (32-token stages) of the decode CTA, per tile height R and
// consumer kind, from sweeps on GB300.  The 16-byte-copy loader (power-of-two page sizes) feeds
// tensor-core consumers, which spend little issue per stage and keep no transpose scratch,
// leaving the shared memory to a 12-stage ring; four of them hide the stage latency (two fall
// behind).  Against the CUDA-core consumers they raised the Llama-3-8B-shaped batch (R = 4) from
// 0.75 to 0.99 of the measured copy bandwidth, the skewed batch (R = 8) from 0.35 to 0.85, and
// g = 1 / g = 2 batches of the same lengths from 0.96 / 0.90 to 1.00 / 0.99.  The bulk loader
// (other page sizes) feeds CUDA-core consumers: eight warps hide the latency of the R <= 4 math;
// R = 8 needs more registers per thread, so four.
constexpr int kDecodeCopiers = 3;  // copier warps of the 16-byte-copy loader: ~0.9 of HBM in flight
template <int R, bool kMma>
struct DecodeConfig {
  static constexpr int kWarps = kMma ? 4 : (R >= 8 ? 4 : 8);
  static constexpr int kStages = kMma ? 12 : (R >= 8 ? 11 : 9);
};

// pdl: launched with programmatic stream serialisation, so it may start while the previous kernel
// on the stream finishes: with p.wait_prior it waits for that kernel before its first global read
// (a plain run: only its shared-memory set-up overlaps); without (a composable plan's per-request
// part, whose only reads of the previous kernel's output are the shared slots) it waits with
// griddepcontrol.wait before it reads those slots.
template <int R, int kCopiers, int kFlags>
int launch_decode_as(int grid, const DecodeParams& p, cudaStream_t stream, bool pdl = false) {
  constexpr bool kMma = kCopiers > 0;
  constexpr int kDecodeWarps = DecodeConfig<R, kMma>::kWarps;
  constexpr int kDecodeStages = DecodeConfig<R, kMma>::kStages;
  using Smem = DecodeSmem<R, kDecodeWarps, kDecodeStages, kMma>;
  static_assert(sizeof(Smem) <= 227 * 1024, "decode shared memory exceeds the per-CTA limit");
  auto kernel = decode_kernel<R, kDecodeWarps, kDecodeStages, kCopiers, kMma, kFlags>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [&] {
    attr_err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(sizeof(Smem)));
  });
  if (attr_err != cudaSuccess) return record_cuda_error(attr_err, "cudaFuncSetAttribute(decode)");
  const unsigned threads = unsigned((kDecodeWarps + (kCopiers ? 1 + kCopiers : 1)) * 32);
  if (pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(grid));
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = sizeof(Smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, p);
    return e == cudaSuccess ? FI_OK : record_cuda_error(e, "decode_kernel launch (programmatic)");
  }
  kernel<<<grid, threads, sizeof(Smem), stream>>>(p);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? FI_OK : record_cuda_error(e, "decode_kernel launch");
}

// Tensor-core decode with the TMA copier (HND pages of 8+ tokens); tm_k / tm_v as built by
// make_decode_map_bf16.  pdl as for launch_decode_as.
template <int R, int kFlags>
int launch_decode_tma_as(int grid, const DecodeParams& p, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                         cudaStream_t stream, bool pdl) {
  constexpr int kDecodeWarps = DecodeConfig<R, true>::kWarps;
  constexpr int kDecodeStages = DecodeConfig<R, true>::kStages;
  using Smem = DecodeSmem<R, kDecodeWarps, kDecodeStages, true>;
  constexpr size_t kSmemBytes = sizeof(Smem) + 1024;  // slack for the kernel's 1 KB alignment
  static_assert(kSmemBytes <= 227 * 1024, "decode shared memory exceeds the per-CTA limit");
  auto kernel = decode_kernel_tma<R, kDecodeWarps, kDecodeStages, kDecodeCopiers, kFlags>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [&] {
    attr_err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kSmemBytes));
  });
  if (attr_err != cudaSuccess) return record_cuda_error(attr_err, "cudaFuncSetAttribute(decode tma)");
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(grid));
  cfg.blockDim = dim3(unsigned((kDecodeWarps + 1 + kDecodeCopiers) * 32));
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, p, tm_k, tm_v);
  return e == cudaSuccess ? FI_OK : record_cuda_error(e, "decode_kernel_tma launch");
}

// NHD decode (16-byte-copy loader): the page-row stride H_kv * 128 is a compile-time constant of
// the kernel (a run-time stride in its copy loop measured a third slower), so the kernel is
// instantiated per rows-per-tile and per log2(H_kv) in 0..4.  pdl as for launch_decode_as.
// Returns an fi_status.
int launch_decode_nhd(int rows_tile, int log2_heads, int grid, const DecodeParams& p, cudaStream_t stream,
                      bool pdl = false);

// FP8 (e4m3) KV pages, HND or NHD layout, 16-byte-copy loader (power-of-two pages).  pdl as for
// launch_decode_as.  Returns an fi_status.
int launch_decode_fp8(int rows_tile, bool nhd, int grid, const DecodeParams& p, cudaStream_t stream,
                      bool pdl = false);

}  // namespace fi
