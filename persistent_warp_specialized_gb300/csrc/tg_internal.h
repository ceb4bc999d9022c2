// tg_internal.h -- interface between the C-ABI translation unit (tg_api.cu) and the
// translation unit that holds the kernels (tg_gemm.cu).  Not installed, not part of the ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace tg {

struct GemmLaunch {
  CUtensorMap tmA, tmB, tmC;
  void* C;
  uint32_t M, N, K;
  uint32_t m_blocks, n_blocks, k_blocks, group;
  uint32_t split_from, total_units;
  uint32_t column_major;
  uint32_t dynamic;
  uint32_t epi_direct;
  uint32_t grid;
  uint64_t watchdog_ns;
  int32_t* trace;
  int64_t inject_skip_phase;
  uint32_t sk_tiles, sk_epoch, sk_slot_f4;   // stream-K tail (0 tiles: none)
  uint32_t* sk_flags;
  float4* sk_partials;
};

// the block-scaled MXFP8 GEMM (one CTA per 128 x 256 tile, the single variant's schedule)
struct MxLaunch {
  CUtensorMap tmA, tmB, tmC;
  CUtensorMap tmSFA, tmSFB;   // pair variant: the packed scales as rows of 128 words
  const void* SFA;   // packed scale atoms (mx_pack_scales_kernel)
  const void* SFB;
  uint32_t sfa_blocks, sfb_blocks;   // row blocks of 128 per k-block in the packed arrays
  uint32_t M, N, K;
  uint32_t m_blocks, n_blocks, k_blocks, group;
  uint32_t split_from, total_units;
  uint32_t column_major;
  uint32_t grid;
  uint64_t watchdog_ns;
  int32_t* trace;
  int64_t inject_skip_phase;
};

// kernel variants: one CTA per 128 x 256 tile, or a CTA pair (cta_group::2) per 256 x 256 tile
enum Variant { kVariantSingle = 1, kVariantPair = 2, kVariantPairWide = 3 };

// Sets the dynamic shared-memory limit of every GEMM instantiation on the current device and
// returns how many CTA pairs of the pair kernels can be resident at once (*max_pairs: the
// smaller of the dense and the MXFP8 pair kernel).
cudaError_t prepare_gemm_kernels(int* max_pairs);
// dtype 0 = fp16, 1 = bf16.  For the pair variants l.grid counts CTAs (even) and l.m_blocks
// counts 256-row pair tiles (l.n_blocks: 512-column tiles for kVariantPairWide).
cudaError_t launch_gemm(int dtype, bool debug, int variant, const GemmLaunch& l,
                        cudaStream_t stream);
// out_dtype 0 = fp16, 1 = bf16; variant kVariantSingle or kVariantPair (l.grid counts CTAs)
cudaError_t launch_mxfp8(int out_dtype, bool debug, int variant, const MxLaunch& l,
                         cudaStream_t stream);
// row-major scales [rows, 4 * k_blocks] -> atoms [k_blocks][row_blocks][512]
cudaError_t launch_mx_pack(const void* sf, void* out, uint32_t rows, uint32_t k_blocks,
                           uint32_t row_blocks, cudaStream_t stream);
// C[0 .. bytes) = 0 (bytes a multiple of 16, C 16-byte aligned)
cudaError_t launch_zero_fill(void* C, uint64_t bytes, cudaStream_t stream);
// rows of 5 int32 (worker, w, bx, by, part) over the units [0, units); tiles below
// split_from are whole (part -1)
cudaError_t launch_tile_schedule(uint32_t m_blocks, uint32_t n_blocks, uint32_t num_workers,
                                 uint32_t group, uint32_t split_from, uint32_t units,
                                 uint32_t column_major, int32_t* out_dev, cudaStream_t stream);
cudaError_t clear_watchdog_status(cudaStream_t stream);
// synchronises ``stream``, returns the status word in *out and clears it
cudaError_t read_and_clear_watchdog_status(unsigned int* out, cudaStream_t stream);

}  // namespace tg
