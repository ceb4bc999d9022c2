// tg_gemm_pair_wide_kernel.cuh -- the CTA-pair GEMM with 256 x 512 output tiles.
//
// The pair kernel of tg_gemm_pair_kernel.cuh ("[Feature] Introduce tile scheduler #2441",
// ``gemm_persistent_2cta``) with twice the tile width: one unit is 256 rows x 512 columns,
// computed as two N-halves of 256 columns, each by tcgen05.mma cta_group::2 M = 256, N = 256,
// K = 16 into its own half of TMEM (columns 0..255 and 256..511).  Per k-block of 64 each CTA
// loads one A box 128 x 64 (16 KiB, its 128 rows) and four B boxes 64 x 64 (8 KiB each: its
// 128 columns of each N-half), 48 KiB per stage, 4 stages.  Against the 256 x 256 pair tile:
//   * A is loaded once for 512 columns instead of 256: 25 % fewer bytes from L2 into shared
//     memory per flop;
//   * a stage holds as much MMA work as the 256 x 256 kernel's 128-deep stage (0.68 us at the
//     bf16 peak), and a refill has three stages instead of two to arrive;
//   * the tail split's half units are 256 x 256 (whole N-halves) rather than 256 x 128;
//   * there is one accumulator (all 512 TMEM columns), so the next unit's MMAs wait for the
//     epilogue to read the previous one out.  To keep that wait short, the epilogue copies a
//     whole N-half into registers (converted to the output type: 128 words per thread) and
//     hands it back on its own barrier (tmem_empty[h]) before storing any of it; the MMA waits
//     for half 0 before its first k-block and for half 1 only after N-half 0 of the first
//     kWideDefer k-blocks, whose ring slots it releases once half 1 has caught up on them.  A
//     half unit hands back its unused half at once, so both barriers complete once per unit
//     and the parity of unit w is (w & 1) ^ 1.
// Everything else -- the scheduler, the single iteration clock with slot phase % S, the odd
// CTA's loads completing on the even CTA's barrier, multicast commits, bounded waits with the
// pair abort, the TMA-store epilogue -- is the pair kernel's.  Included by exactly one
// translation unit, after tg_gemm_pair_kernel.cuh.
#pragma once

#include "tg_gemm_pair_kernel.cuh"
#include "tg_streamk.cuh"
#include "tg_wide_config.h"

namespace tg {

struct __align__(8) WideCtl {
  uint64_t loaded[kWideStages];      // used in the even CTA only
  uint64_t consumed[kWideStages];
  uint64_t tmem_full;
  uint64_t tmem_empty[2];            // per N-half; used in the even CTA only (pair_report_warp)
  uint64_t drain;
  uint64_t odd_done;                 // even CTA: the odd producer has stopped filling
  PairFills<kWideStages> fills;
  uint32_t sink[kEpiWarps];          // even CTA: target of the odd epilogue warps' st.async
  uint64_t sk_bar[kEpiWarps];        // per epilogue warp: stream-K contributions landed
  uint32_t tmem_base;
  int abort;
};

// DT: 0 = fp16, 1 = bf16.  p.m_blocks counts 256-row tiles, p.n_blocks 512-column tiles.
template <int DT, bool DEBUG>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    gemm_pair_wide_ws_kernel(const __grid_constant__ CUtensorMap tmA,
                             const __grid_constant__ CUtensorMap tmB,
                             const __grid_constant__ CUtensorMap tmC, const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ WideCtl ctl;

  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t rank = cluster_ctarank();          // 0: even CTA (issues the MMA), 1: odd
  const uint32_t pair = blockIdx.x >> 1;
  const uint32_t num_pairs = gridDim.x >> 1;
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sA0 = sbase;                 // stage s: A at sA0 + s * kWideStageBytes,
  const uint32_t sB0 = sbase + kWideABytes;   // then B chunks (2 h + c) of 8 KiB
  const uint32_t sEpi = sbase + kWideStages * kWideStageBytes;

  const uint32_t bar_loaded = smem_u32(&ctl.loaded[0]);
  const uint32_t bar_consumed = smem_u32(&ctl.consumed[0]);
  const uint32_t bar_tmem_full = smem_u32(&ctl.tmem_full);
  const uint32_t bar_tmem_empty = smem_u32(&ctl.tmem_empty[0]);
  const uint32_t bar_drain = smem_u32(&ctl.drain);

  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < kWideStages; ++s) {
      mbar_init(bar_loaded + 8u * s, 1);
      mbar_init(bar_consumed + 8u * s, 1);
    }
    mbar_init(bar_tmem_full, 1);
    mbar_init(bar_tmem_empty, kEpiWarps);
#pragma unroll
    for (int q = 0; q < kEpiWarps; ++q) mbar_init(smem_u32(&ctl.sk_bar[q]), 1);
    mbar_init(bar_tmem_empty + 8u, kEpiWarps);
    mbar_init(bar_drain, 1);
    mbar_init(smem_u32(&ctl.odd_done), 1);
#pragma unroll
    for (int st = 0; st < kWideStages; ++st) ctl.fills.par[st] = 0;
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
    tmem_alloc_pair(smem_u32(&ctl.tmem_base), kTmemCols);
    tmem_relinquish_alloc_permit_pair();
  }
  tcgen05_fence_before_sync();
  cluster_sync();   // both CTAs' barriers exist before any remote arrive or complete_tx
  tcgen05_fence_after_sync();
  // Launched with programmatic stream serialization: this CTA may start while the previous
  // kernel in the stream is finishing.  Nothing above touches global memory; nothing below
  // runs before that kernel has completed.  Then the next launch may be scheduled.
  grid_dependency_wait();
  grid_launch_dependents();

  const uint32_t tmem_base = ctl.tmem_base;
  volatile int* abort_flag = &ctl.abort;
  const uint32_t peer_abort = mapa_shared(smem_u32(&ctl.abort), rank ^ 1u);
  const uint64_t limit = p.watchdog_ns;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      PersistentTileScheduler sched(p.m_blocks, p.n_blocks, p.group, num_pairs, p.split_from,
                                    p.total_units, p.column_major, p.k_blocks, p.sk_tiles);
      sched.init(pair);
      bool ok = true;
      uint64_t phase = 0;   // k-blocks filled so far: the ring position of the next one
      while (ok && sched.valid()) {
        const bool half = sched.half_unit();          // half unit: the N-half ``part`` alone
        const uint32_t halves = half ? 1u : 2u;
        const int32_t m0 = static_cast<int32_t>(sched.m_idx * kPairBM + rank * kBM);
        const int32_t n0 = static_cast<int32_t>(sched.n_idx * kWideBN) + (half ? sched.part * kBN : 0);
        const uint32_t tx_bytes = 2u * (kWideABytes + halves * 2u * kWideBChunkBytes);
        for (uint32_t k = sched.k_lo; k < sched.k_hi; ++k, ++phase) {
          const uint32_t s = static_cast<uint32_t>(phase % kWideStages);
          const uint32_t par = static_cast<uint32_t>((phase / kWideStages) & 1u);
          if (!pair_wait_or_abort(bar_consumed + 8u * s, par ^ 1u, abort_flag, peer_abort, limit,
                                  kRoleProducer)) {
            ok = false;
            break;
          }
          if (DEBUG && injected_skip(p.inject_skip_phase, phase))
            continue;  // injected fault: this CTA never arms or fills this phase
          const uint32_t full_even = mapa_shared(bar_loaded + 8u * s, 0);
          if (rank == 0) mbar_arrive_expect_tx(bar_loaded + 8u * s, tx_bytes);
          const int32_t kx = static_cast<int32_t>(k) * kWideBK;
          tma_load_2d_pair(sA0 + s * kWideStageBytes, &tmA, full_even, kx, m0);
#pragma unroll
          for (uint32_t h = 0; h < 2; ++h) {
            if (h >= halves) break;
            // CTA r loads columns [128 r, 128 r + 128) of N-half h as two 64-column chunks
#pragma unroll
            for (uint32_t c = 0; c < 2; ++c) {
              const uint32_t dst = sB0 + s * kWideStageBytes + (2u * h + c) * kWideBChunkBytes;
              const int32_t nx = n0 + static_cast<int32_t>(h * kBN + rank * kPairBNHalf + c * kBChunkCols);
              tma_load_2d_pair(dst, &tmB, full_even, nx, kx);
            }
          }
          record_fill(ctl.fills, s, phase, par, tx_bytes / 2u);
        }
        sched.next_tile();
      }
      // the odd producer has stopped filling: its records are final (see pair_drain_fills)
      if (rank == 1) mbar_arrive_cluster(mapa_shared(smem_u32(&ctl.odd_done), 0));
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    if (lane == 0 && rank == 0) {
      constexpr uint32_t idesc = idesc_f16(DT, kPairBM, kBN, /*A K-major*/ 0, /*B N-major*/ 1);
      PersistentTileScheduler sched(p.m_blocks, p.n_blocks, p.group, num_pairs, p.split_from,
                                    p.total_units, p.column_major, p.k_blocks, p.sk_tiles);
      sched.init(pair);
      bool ok = true;
      uint64_t phase0 = 0;   // ring position of the current unit's first k-block
      // MMAs of N-half h for the k-block in ring slot s (k: its index within the unit)
      auto issue_half = [&](uint32_t s, uint32_t h, uint32_t k) {
        const uint32_t a_addr = sA0 + s * kWideStageBytes;
        const uint32_t b_addr = sB0 + s * kWideStageBytes + 2u * h * kWideBChunkBytes;
#pragma unroll
        for (uint32_t kk = 0; kk < kWideBK / kUmmaK; ++kk) {
          const uint64_t a_desc = smem_desc_sw128(a_addr + kk * kUmmaK * kElemBytes, 16, 1024);
          const uint64_t b_desc =
              smem_desc_sw128(b_addr + kk * kUmmaK * 128u, kWideBChunkBytes, 1024);
          umma_f16_pair(tmem_base + h * kBN, a_desc, b_desc, idesc, (k | kk) != 0u ? 1u : 0u);
        }
      };
      while (ok && sched.valid()) {
        const uint32_t w = sched.current_iter;
        const uint32_t halves = sched.half_unit() ? 1u : 2u;
        const uint32_t nk = sched.k_hi - sched.k_lo;   // k-blocks of this unit (k counts them)
        // N-half 1 of the first ``defer`` k-blocks waits until the epilogue has handed half 1
        // back; those slots are released only once both halves have read them
        const uint32_t defer = halves == 2u ? (kWideDefer < nk ? kWideDefer : nk - 1u) : 0u;
        for (uint32_t k = 0; k < nk; ++k) {
          const uint64_t phase = phase0 + k;
          const uint32_t s = static_cast<uint32_t>(phase % kWideStages);
          const uint32_t par = static_cast<uint32_t>((phase / kWideStages) & 1u);
          if (!pair_wait_or_abort(bar_loaded + 8u * s, par, abort_flag, peer_abort, limit,
                                  kRoleMma)) {
            ok = false;
            break;
          }
          tcgen05_fence_after_sync();
          if (k == 0) {
            // half 0 of the previous unit's accumulator has been read out by both epilogues
            if (!pair_wait_or_abort<true>(bar_tmem_empty, (w & 1u) ^ 1u, abort_flag, peer_abort,
                                    limit, kRoleMma)) {
              ok = false;
              break;
            }
            tcgen05_fence_after_sync();
          }
          issue_half(s, 0, k);
          if (halves == 1u) {
            umma_commit_pair_multicast(bar_consumed + 8u * s, 0x3);
            continue;
          }
          if (k < defer) continue;   // slot s stays held until half 1 has read it
          if (k == defer) {
            if (!pair_wait_or_abort<true>(bar_tmem_empty + 8u, (w & 1u) ^ 1u, abort_flag, peer_abort,
                                    limit, kRoleMma)) {
              ok = false;
              break;
            }
            tcgen05_fence_after_sync();
            for (uint32_t j = 0; j < defer; ++j) {   // catch half 1 up, releasing each slot
              const uint32_t sj = static_cast<uint32_t>((phase0 + j) % kWideStages);
              issue_half(sj, 1, j);
              umma_commit_pair_multicast(bar_consumed + 8u * sj, 0x3);
            }
          }
          issue_half(s, 1, k);
          umma_commit_pair_multicast(bar_consumed + 8u * s, 0x3);
        }
        if (!ok) break;
        umma_commit_pair_multicast(bar_tmem_full, 0x3);
        phase0 += nk;
        sched.next_tile();
      }
      umma_commit_pair_multicast(bar_drain, 0x1);
      wait_bounded(bar_drain, 0, limit, kRoleDrain);
    }
    __syncwarp();
  } else if (warp >= kFirstEpiWarp) {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const uint32_t q = warp - kFirstEpiWarp;
    const uint32_t sink_even = mapa_shared(smem_u32(&ctl.sink[q]), 0);
    PersistentTileScheduler sched(p.m_blocks, p.n_blocks, p.group, num_pairs, p.split_from,
                                  p.total_units, p.column_major, p.k_blocks, p.sk_tiles);
    sched.init(pair);
    uint32_t chunk = 0;
    uint32_t sk_bar_uses = 0;   // phases of ctl.sk_bar[q] used so far
    while (sched.valid()) {
      const uint32_t w = sched.current_iter;
      const bool got = pair_wait_or_abort(bar_tmem_full, w & 1u, abort_flag, peer_abort, limit,
                                          kRoleEpilogue);
      if (!__all_sync(0xffffffffu, got)) break;
      tcgen05_fence_after_sync();
      const bool half = sched.half_unit();
      const uint32_t halves = half ? 1u : 2u;
      const int32_t row0 = static_cast<int32_t>(sched.m_idx * kPairBM + rank * kBM + q * 32u);
      const int32_t col0 = static_cast<int32_t>(sched.n_idx) * kWideBN + (half ? sched.part * kBN : 0);
      const uint32_t t_row = tmem_base + ((q * 32u) << 16);
      // stream-K tail: a contribution goes to this worker's slot (chunk 4h + j for N-half h),
      // half by half, and is not stored; an owned tile first adds the contributions of workers
      // sk_lowest_worker .. pair - 1 into its accumulator, half by half, then is stored below
      const int32_t kind = sched.part;
      bool sk_ok = true;
      if (kind == 2) {
#pragma unroll 1
        for (uint32_t h = 0; h < 2; ++h) {
          sk_write_slot(sk_slot(p.sk_partials, p.sk_slot_f4, pair, rank), t_row + h * kBN,
                        kBN / kEpiN, h * (kBN / kEpiN), q, lane, sEpi + q * 2u * kEpiBufBytes,
                        sEpi + (q * 2u + 1u) * kEpiBufBytes);
          tcgen05_fence_before_sync();
          pair_report_warp(bar_tmem_empty + 8u * h, rank, lane, sink_even);
        }
        sk_publish(p.sk_flags + sk_flag_index(pair, rank, q), p.sk_epoch, lane);
      } else if (kind == 3) {
        const uint32_t c_lo = sk_lowest_worker(pair, num_pairs, p.sk_tiles, p.k_blocks,
                                               sched.sk_tile);
#pragma unroll 1
        for (uint32_t h = 0; h < 2 && sk_ok; ++h)
          sk_ok = sk_gather(p, c_lo, pair, num_pairs, rank, q, lane, t_row + h * kBN, kBN / kEpiN,
                            h * (kBN / kEpiN), sA0 + q * (kWideStages * kWideStageBytes / kEpiWarps),
                            smem_u32(&ctl.sk_bar[q]), &sk_bar_uses, h == 0, abort_flag,
                            peer_abort, limit);
      }
      if (!__all_sync(0xffffffffu, sk_ok)) break;
#pragma unroll 1
      for (uint32_t h = 0; h < 2 && kind != 2; ++h) {
        if (h >= halves) {
          tcgen05_fence_before_sync();
          pair_report_warp(bar_tmem_empty + 8u * h, rank, lane, sink_even);   // unused half
          continue;
        }
        // the whole N-half into registers, converted (4 chunks x 32 words per lane), then
        // hand it back to the MMA before any of it is stored
        uint32_t pk[kBN / kEpiN][kEpiN / 2];
#pragma unroll
        for (uint32_t j = 0; j < kBN / kEpiN; ++j) {
          uint32_t v[64];
          tmem_ld_32x32b_x64(t_row + h * kBN + j * kEpiN, v);
          pack_chunk<DT>(v, pk[j]);
        }
        tcgen05_fence_before_sync();
        pair_report_warp(bar_tmem_empty + 8u * h, rank, lane, sink_even);
#pragma unroll
        for (uint32_t j = 0; j < kBN / kEpiN; ++j, ++chunk) {
          const uint32_t sbuf = sEpi + (q * 2u + (chunk & 1u)) * kEpiBufBytes;
          epilogue_store_packed(pk[j], lane, sbuf, &tmC, p, row0,
                                col0 + static_cast<int32_t>(h * kBN + j * kEpiN));
        }
      }
      if (DEBUG && p.trace != nullptr && rank == 0 && q == 0 && lane == 0) {
        int32_t* tr = p.trace + 5ull * sched.linear_idx;
        tr[0] = static_cast<int32_t>(pair);
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

  __syncthreads();   // every role of this CTA has left its loop
  if (rank == 0 && warp == 0 && lane == 0 && *abort_flag)
    pair_drain_fills(bar_loaded, ctl.fills, mapa_shared(smem_u32(&ctl.fills), 1),
                     smem_u32(&ctl.odd_done), limit);
  tcgen05_fence_before_sync();
  cluster_sync();   // neither CTA leaves while the pair may still touch its smem or TMEM
  if (warp == 2) {
    tcgen05_fence_after_sync();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

}  // namespace tg
