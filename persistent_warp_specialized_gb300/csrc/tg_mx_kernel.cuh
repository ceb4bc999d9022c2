// tg_mx_kernel.cuh -- persistent, warp-specialized block-scaled MXFP8 GEMM for sm_103a.
//
//   C[i, j] = sum_k A[i, k] 2^(SFA[i, k / 32] - 127) * B[j, k] 2^(SFB[j, k / 32] - 127)
//
// The second workload of "[Feature] Introduce tile scheduler #2441"
// (examples/blockscaled_gemm_sm100/gemm_mxfp8_blockscaled_1d1d.py): TMA-load, MMA and
// epilogue roles, each walking the tiles with its own PersistentTileScheduler on the single
// iteration clock w, with the page's scale-factor transpose done ahead of the GEMM by
// mx_pack_scales_kernel (scales in the tcgen05.cp source layout).  Here:
//   * warp 0, one lane: producer.  Per tile and k-block (phase p = w * k_blocks + k, slot
//     s = p % S): wait consumed[s], arm loaded[s] with the stage's bytes, TMA-load A (128 rows
//     x 128 bytes) and B (256 rows x 128 bytes as two boxes; one for a half-width unit), and
//     bulk-copy the k-block's packed scale atoms (A rows m0..m0+127: 512 bytes; B rows
//     n0..n0+255: 1 KiB, 512 bytes for a half-width unit) into the stage's atom set;
//   * warp 1, one lane: MMA issuer.  Per k-block: wait loaded[s], copy the atoms into the
//     stage's TMEM scale slot (tcgen05.cp .32x128b.warpx4), issue four tcgen05.mma
//     kind::mxf8f6f4.block_scale 128 x 256 x 32 (byte id kk of each scale word for the kk-th
//     32-element block), commit to consumed[s].  After the k-loop, commit to tmem_full;
//   * warps 4..7: epilogue.  Wait tmem_full, copy the warp's 32 lanes x 256 columns to
//     registers as packed output pairs, release the accumulator (tmem_empty), then stage and
//     TMA-store 32 x 64 chunks (clipped at M and N);
//   * warp 2 owns the TMEM allocation (512 columns: accumulator and scale slots).
// A TMEM scale slot is rewritten only after loaded[s] of a later phase, which the producer
// arms only after consumed[s] of the phase that last used it.  Every wait is bounded by the
// same watchdog as the dense kernels.
//
// Shared memory (1024-byte aligned): S stages of 48 KiB (A then B, both K-major with the
// 128-byte swizzle); S atom sets of 1536 bytes; one 32 x 128-byte epilogue staging buffer per
// epilogue warp.
#pragma once

#include "tg_gemm_kernel.cuh"

namespace tg {

struct MxParams {
  const uint8_t* SFA;          // packed scale atoms of A: [K / 128][row blocks of A][512]
  const uint8_t* SFB;          // packed scale atoms of B: [K / 128][row blocks of B][512]
  uint32_t M, N, K;
  uint32_t sfa_blocks, sfb_blocks;   // row blocks (of 128) per k-block in the packed arrays
  uint32_t m_blocks, n_blocks, k_blocks, group;
  uint32_t split_from, total_units, column_major;
  uint64_t watchdog_ns;
  int32_t* trace;              // debug instantiation only; may be null (5 int32 per unit)
  int64_t inject_skip_phase;   // debug instantiation only; -1 = none
};

struct __align__(8) MxCtl {
  uint64_t loaded[kMxStages];
  uint64_t consumed[kMxStages];
  uint64_t tmem_full;
  uint64_t tmem_empty;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

// Stores one 32 x 64 chunk held as packed output pairs (lane = row; w[c] = columns 2c, 2c + 1)
// through this warp's staging buffer and a TMA store clipped at the tensor's edge.  The one
// buffer is rewritten only after the previous store from it has finished reading it.
__device__ __forceinline__ void mx_store_chunk(const uint32_t (&w)[32], uint32_t lane,
                                               uint32_t sbuf, const CUtensorMap* tmC, uint32_t M,
                                               uint32_t N, int32_t row0, int32_t x) {
  if (lane == 0) bulk_wait_group_read<0>();
  __syncwarp();
  const uint32_t row_addr = sbuf + lane * 128u;
#pragma unroll
  for (uint32_t c = 0; c < 8; ++c)
    st_shared_v4(row_addr + ((c ^ (lane & 7u)) << 4), w[4 * c + 0], w[4 * c + 1], w[4 * c + 2],
                 w[4 * c + 3]);
  fence_proxy_async_shared();
  __syncwarp();
  if (lane == 0) {
    if (row0 < static_cast<int32_t>(M) && x < static_cast<int32_t>(N)) {
      if (kCPolicy != 0)
        tma_store_2d_hint(tmC, sbuf, x, row0, l2_policy<kCPolicy>());
      else
        tma_store_2d(tmC, sbuf, x, row0);
    }
    bulk_commit_group();
  }
  __syncwarp();
}

// OUT: 0 = fp16 output, 1 = bf16 output.  DEBUG adds the unit trace and fault injection.
template <int OUT, bool DEBUG>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_mxfp8_ws_kernel(const __grid_constant__ CUtensorMap tmA,
                         const __grid_constant__ CUtensorMap tmB,
                         const __grid_constant__ CUtensorMap tmC, const MxParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ MxCtl ctl;

  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sA0 = sbase;                                   // + s * kMxStageBytes
  const uint32_t sB0 = sbase + kMxABytes;                       // + s * kMxStageBytes
  const uint32_t sAtom0 = sbase + kMxStages * kMxStageBytes;    // + s * kMxAtomSetBytes
  const uint32_t sEpi = sAtom0 + kMxAtomRegionBytes;

  const uint32_t bar_loaded = smem_u32(&ctl.loaded[0]);
  const uint32_t bar_consumed = smem_u32(&ctl.consumed[0]);
  const uint32_t bar_tmem_full = smem_u32(&ctl.tmem_full);
  const uint32_t bar_tmem_empty = smem_u32(&ctl.tmem_empty);
  const uint32_t bar_drain = smem_u32(&ctl.drain);

  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < kMxStages; ++s) {
      mbar_init(bar_loaded + 8u * s, 1);
      mbar_init(bar_consumed + 8u * s, 1);
    }
    mbar_init(bar_tmem_full, 1);
    mbar_init(bar_tmem_empty, kEpiThreads);
    mbar_init(bar_drain, 1);
    ctl.abort = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB);
    prefetch_tensormap(&tmC);
  }
  __syncwarp();
  if (warp == 2) {
    tmem_alloc(smem_u32(&ctl.tmem_base), kTmemCols);
    tmem_relinquish_alloc_permit();
  }
  tcgen05_fence_before_sync();
  __syncthreads();
  tcgen05_fence_after_sync();
  // Launched with programmatic stream serialization: this CTA may start while the previous
  // kernel in the stream is finishing.  Nothing above touches global memory; nothing below
  // runs before that kernel has completed.  Then the next launch may be scheduled.
  grid_dependency_wait();
  grid_launch_dependents();

  const uint32_t tmem_base = ctl.tmem_base;
  volatile int* abort_flag = &ctl.abort;
  const uint64_t limit = p.watchdog_ns;
  const uint64_t k_blocks = p.k_blocks;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      PersistentTileScheduler sched(p.m_blocks, p.n_blocks, p.group, gridDim.x, p.split_from,
                                    p.total_units, p.column_major);
      sched.init(blockIdx.x);
      uint32_t pending = 0;       // stages whose latest operand fill may still be in flight
      uint32_t pending_par = 0;
      bool ok = true;
      while (ok && sched.valid()) {
        const uint64_t w = sched.current_iter;
        const bool half = sched.half_unit();
        const int32_t m0 = static_cast<int32_t>(sched.m_idx * kBM);
        const int32_t n0 = static_cast<int32_t>(sched.n_idx * kBN) + (half ? sched.part * (kBN / 2) : 0);
        const uint32_t sfb_bytes = half ? kMxSfAtomBytes : 2 * kMxSfAtomBytes;
        const uint32_t tx_bytes = kMxABytes + (half ? kMxBHalfBytes : kMxBBytes) + kMxSfAtomBytes + sfb_bytes;
        const uint32_t ma = static_cast<uint32_t>(m0) / kBM;      // A's row block
        const uint32_t nb = static_cast<uint32_t>(n0) / kBM;      // B's first row block
        for (uint32_t k = 0; k < p.k_blocks; ++k) {
          const uint64_t phase = w * k_blocks + k;
          const uint32_t s = static_cast<uint32_t>(phase % kMxStages);
          const uint32_t par = static_cast<uint32_t>((phase / kMxStages) & 1u);
          if (!wait_or_abort(bar_consumed + 8u * s, par ^ 1u, abort_flag, limit, kRoleProducer)) {
            ok = false;
            break;
          }
          pending &= ~(1u << s);
          if (DEBUG && injected_skip(p.inject_skip_phase, phase))
            continue;  // injected fault: the operands of this phase are never loaded
          const uint32_t full = bar_loaded + 8u * s;
          const int32_t kx = static_cast<int32_t>(k * kMxBK);
          mbar_arrive_expect_tx(full, tx_bytes);
          tma_load_2d(sA0 + s * kMxStageBytes, &tmA, full, kx, m0);
          tma_load_2d(sB0 + s * kMxStageBytes, &tmB, full, kx, n0);
          if (!half) tma_load_2d(sB0 + s * kMxStageBytes + kMxBHalfBytes, &tmB, full, kx, n0 + kBN / 2);
          const uint32_t atom = sAtom0 + s * kMxAtomSetBytes;
          bulk_load(atom, p.SFA + (static_cast<uint64_t>(k) * p.sfa_blocks + ma) * kMxSfAtomBytes,
                    kMxSfAtomBytes, full);
          bulk_load(atom + kMxSfAtomBytes,
                    p.SFB + (static_cast<uint64_t>(k) * p.sfb_blocks + nb) * kMxSfAtomBytes, sfb_bytes, full);
          pending |= 1u << s;
          pending_par = (pending_par & ~(1u << s)) | (par << s);
        }
        sched.next_tile();
      }
      if (!ok) {
        for (uint32_t s = 0; s < kMxStages; ++s)
          if ((pending >> s) & 1u)
            wait_bounded(bar_loaded + 8u * s, (pending_par >> s) & 1u, limit, kRoleDrain);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      PersistentTileScheduler sched(p.m_blocks, p.n_blocks, p.group, gridDim.x, p.split_from,
                                    p.total_units, p.column_major);
      sched.init(blockIdx.x);
      bool ok = true;
      while (ok && sched.valid()) {
        const uint32_t w = sched.current_iter;
        if (!wait_or_abort(bar_tmem_empty, (w & 1u) ^ 1u, abort_flag, limit, kRoleMma)) {
          ok = false;
          break;
        }
        tcgen05_fence_after_sync();
        const bool half = sched.half_unit();
        const uint32_t idesc = half ? idesc_mxf8(kBM, kBN / 2, 0, 0) : idesc_mxf8(kBM, kBN, 0, 0);
        for (uint32_t k = 0; k < p.k_blocks; ++k) {
          const uint64_t phase = static_cast<uint64_t>(w) * k_blocks + k;
          const uint32_t s = static_cast<uint32_t>(phase % kMxStages);
          const uint32_t par = static_cast<uint32_t>((phase / kMxStages) & 1u);
          if (!wait_or_abort(bar_loaded + 8u * s, par, abort_flag, limit, kRoleMma)) {
            ok = false;
            break;
          }
          tcgen05_fence_after_sync();
          const uint32_t atom = sAtom0 + s * kMxAtomSetBytes;
          const uint32_t t_sf = tmem_base + kMxAccCols + s * kMxSfColsPerStage;
          tmem_cp_32x128b_x4(t_sf, smem_desc_plain(atom, 128, 128));
          tmem_cp_32x128b_x4(t_sf + 4, smem_desc_plain(atom + kMxSfAtomBytes, 128, 128));
          if (!half) tmem_cp_32x128b_x4(t_sf + 8, smem_desc_plain(atom + 2 * kMxSfAtomBytes, 128, 128));
          const uint32_t a_addr = sA0 + s * kMxStageBytes;
          const uint32_t b_addr = sB0 + s * kMxStageBytes;
#pragma unroll
          for (uint32_t kk = 0; kk < kMxBK / kMxUmmaK; ++kk) {
            // both operands K-major: advance 32 one-byte elements along the swizzle row
            const uint64_t a_desc = smem_desc_sw128(a_addr + kk * kMxUmmaK, 16, 1024);
            const uint64_t b_desc = smem_desc_sw128(b_addr + kk * kMxUmmaK, 16, 1024);
            umma_mxf8(tmem_base, a_desc, b_desc, idesc | (kk << 29) | (kk << 4), t_sf, t_sf + 4,
                      (k | kk) != 0u ? 1u : 0u);
          }
          umma_commit(bar_consumed + 8u * s);
        }
        if (!ok) break;
        umma_commit(bar_tmem_full);
        sched.next_tile();
      }
      umma_commit(bar_drain);
      wait_bounded(bar_drain, 0, limit, kRoleDrain);
    }
    __syncwarp();
  } else if (warp >= kFirstEpiWarp) {
    // ------------------------------------------------------------ epilogue
    const uint32_t q = warp - kFirstEpiWarp;       // TMEM lanes 32q .. 32q + 31
    PersistentTileScheduler sched(p.m_blocks, p.n_blocks, p.group, gridDim.x, p.split_from,
                                  p.total_units, p.column_major);
    sched.init(blockIdx.x);
    const uint32_t sbuf = sEpi + q * kEpiBufBytes;
    while (sched.valid()) {
      const uint32_t w = sched.current_iter;
      const bool got = wait_or_abort(bar_tmem_full, w & 1u, abort_flag, limit, kRoleEpilogue);
      if (!__all_sync(0xffffffffu, got)) break;
      tcgen05_fence_after_sync();
      const bool half = sched.half_unit();
      const int32_t row0 = static_cast<int32_t>(sched.m_idx * kBM + q * 32u);
      const int32_t col0 = static_cast<int32_t>(sched.n_idx * kBN) + (half ? sched.part * (kBN / 2) : 0);
      const uint32_t t_row = tmem_base + ((q * 32u) << 16);
      uint32_t packed[kBN / kEpiN][kEpiN / 2];
#pragma unroll
      for (uint32_t j = 0; j < kBN / kEpiN; ++j) {
        if (half && j >= kBN / kEpiN / 2) break;
#pragma unroll
        for (uint32_t h = 0; h < 2; ++h) {   // 32 columns at a time keeps the copy small
          uint32_t v[32];
          tmem_ld_32x32b_x32(t_row + j * kEpiN + h * 32u, v);
#pragma unroll
          for (uint32_t c = 0; c < 16; ++c) packed[j][16 * h + c] = pack_out<OUT>(v[2 * c], v[2 * c + 1]);
        }
      }
      tcgen05_fence_before_sync();
      mbar_arrive(bar_tmem_empty);   // accumulator in registers: the next tile may start
#pragma unroll
      for (uint32_t j = 0; j < kBN / kEpiN; ++j) {
        if (half && j >= kBN / kEpiN / 2) break;
        mx_store_chunk(packed[j], lane, sbuf, &tmC, p.M, p.N, row0,
                       col0 + static_cast<int32_t>(j * kEpiN));
      }
      if (DEBUG && p.trace != nullptr && q == 0 && lane == 0) {
        int32_t* tr = p.trace + 5ull * sched.linear_idx;
        tr[0] = static_cast<int32_t>(blockIdx.x);
        tr[1] = static_cast<int32_t>(w);
        tr[2] = static_cast<int32_t>(sched.m_idx);
        tr[3] = static_cast<int32_t>(sched.n_idx);
        tr[4] = sched.part;
      }
      sched.next_tile();
    }
    if (lane == 0) bulk_wait_group<0>();
    __syncwarp();
  }

  tcgen05_fence_before_sync();
  __syncthreads();
  if (warp == 2) {
    tcgen05_fence_after_sync();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace tg
