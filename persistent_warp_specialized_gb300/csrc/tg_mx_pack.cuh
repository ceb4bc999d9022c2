// tg_mx_pack.cuh -- the scale pack of the block-scaled MXFP8 GEMM (tg_mxfp8_pack_scales).
//
// Row-major E8M0 scales sf [rows, 4 * k_blocks] become atoms: out[(k * row_blocks + b) * 512 +
// (r % 32) * 16 + (r / 32) * 4 + j] = sf[b * 128 + r, 4 k + j] (0 for rows >= rows), for every
// k-block k, row block b and r < 128 -- the source layout of tcgen05.cp .32x128b.warpx4 (see
// tg_mx_kernel.cuh; the CTA-pair kernel's epilogue warps read it one 16-byte row per lane and
// write it with tcgen05.st).  A block takes 128 rows x 8 k-blocks at a time: it reads each row's
// 32 bytes (eight 4-byte words, neighbouring threads on neighbouring words), reorders them in
// shared memory, and writes the eight 512-byte atoms with neighbouring threads on neighbouring
// words.  blockIdx.x is the row block; the groups of 8 k-blocks are strided over blockIdx.y,
// whose grid extent is capped at 65535, so every K below 2^31 is covered.
#pragma once

#include <cstdint>

#include "tg_config.h"
#include "tg_ptx.cuh"

namespace tg {

constexpr uint32_t kMxPackKb = 8;          // k-blocks per block of the pack
constexpr uint32_t kMxPackThreads = 256;

__global__ void __launch_bounds__(kMxPackThreads)
    mx_pack_scales_kernel(const uint8_t* __restrict__ sf, uint8_t* __restrict__ out,
                          uint32_t rows, uint32_t k_blocks, uint32_t row_blocks) {
  // words of k-block j of the tile, in atom order: word t = row (t % 4) * 32 + t / 4
  __shared__ uint32_t tile[kMxPackKb][kBM];
  grid_dependency_wait();      // launched like the GEMM kernels (programmatic serialization)
  grid_launch_dependents();
  const uint32_t b = blockIdx.x;                       // row block
  const uint32_t groups = (k_blocks + kMxPackKb - 1) / kMxPackKb;
  const uint64_t row_bytes = static_cast<uint64_t>(k_blocks) * 4u;
  for (uint32_t g = blockIdx.y; g < groups; g += gridDim.y) {
    const uint32_t k0 = g * kMxPackKb;                 // first k-block of the tile
    for (uint32_t i = threadIdx.x; i < kMxPackKb * kBM; i += kMxPackThreads) {
      const uint32_t r = i / kMxPackKb, j = i % kMxPackKb;
      const uint32_t row = b * kBM + r, k = k0 + j;
      const uint32_t v =
          (row < rows && k < k_blocks)
              ? *reinterpret_cast<const uint32_t*>(sf + static_cast<uint64_t>(row) * row_bytes + 4u * k)
              : 0u;
      tile[j][(r % 32u) * 4u + r / 32u] = v;
    }
    __syncthreads();
    for (uint32_t i = threadIdx.x; i < kMxPackKb * kBM; i += kMxPackThreads) {
      const uint32_t j = i / kBM, t = i % kBM;
      const uint32_t k = k0 + j;
      if (k < k_blocks)
        reinterpret_cast<uint32_t*>(out + (static_cast<uint64_t>(k) * row_blocks + b) * kMxSfAtomBytes)[t] =
            tile[j][t];
    }
    __syncthreads();   // the tile is read before the next group overwrites it
  }
}

}  // namespace tg
