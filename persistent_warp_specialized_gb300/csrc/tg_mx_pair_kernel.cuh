// tg_mx_pair_kernel.cuh -- the CTA-pair (tcgen05 cta_group::2) block-scaled MXFP8 GEMM.
//
// The page's MXFP8 example runs on CTA pairs ("[Feature] Introduce tile scheduler #2441",
// examples/blockscaled_gemm_sm100/gemm_mxfp8_blockscaled_1d1d.py, ``cluster_size = 2``, and
// the review comments on its ``bx = m_idx * cluster_size + cta_id``).  A cluster of two CTAs
// shares one 256 x 256 output tile of the product defined in tg_mx_kernel.cuh; the scheduler
// runs per pair over ceil(M / 256) x ceil(N / 256) tiles (with the tail split into 128-wide
// half units), as in tg_gemm_pair_kernel.cuh.
//
// Per CTA r and stage j of the unit (phase p = w * stages + j; operand slot s = p % S, scale
// slot a = p % A with A = S + D, the scale ring running D stages ahead), for each of the
// stage's k-blocks k:
//   * producer (lane 0 of warp 0, both CTAs): wait its own consumed[s] (phase p - S); load the
//     atoms of phase p + D into scale slot (p + D) % A -- the SFA atom of row block 2m + r and
//     the two SFB atoms of the unit's first row block, by TMA onto this CTA's sf_loaded of that
//     slot (a second scheduler cursor walks the units D stages ahead; phases 0 .. D - 1 are
//     loaded first); then the even CTA arms its loaded[s] with both CTAs' operand bytes and each
//     CTA TMA-loads (.cta_group::2, completing on the even CTA's loaded[s]) A rows 256 m + 128 r
//     (128 x 128 bytes) and B rows n0 + 128 r (n0 + 64 r in a half unit; 128 rows, of which the
//     MMA reads the first 64 then).  Scale slot (p + D) % A last held phase p - S, consumed;
//   * MMA (lane 0 of warp 1, even CTA): wait tmem_empty before the unit (one accumulator); per
//     stage wait loaded[s] and sf_ready[a]; four tcgen05.mma cta_group::2
//     kind::mxf8f6f4.block_scale 256 x N x 32 per k-block into each CTA's 128 rows of the
//     accumulator, scales from TMEM scale slot a; commit with CTA mask 0b11 to consumed[s]
//     (both CTAs); after the k-loop to tmem_full;
//   * epilogue warps (warps 4..7, both CTAs; warp 4 + q reaches TMEM lanes 32q .. 32q + 31)
//     keep the scale slots filled and drain the accumulator.  Scale slot of phase p: once
//     sf_loaded[a] has completed, lane i reads row i of each atom (16 bytes: the words of rows
//     i, i + 32, i + 64, i + 96) and writes them with tcgen05.st to columns 0..3 (SFA), 4..7
//     and 8..11 (SFB) of the k-block's TMEM scale slot, the same words in every quadrant; then
//     waits for the writes, fences, and reports on the even CTA's sf_ready[a]
//     (pair_report_warp: one report per warp, st.async from the odd CTA).  The warp polls: it
//     writes slots in phase order as their atoms land until tmem_full of its next unit
//     completes, then copies its 32 lanes of the accumulator to registers, reports on the even
//     CTA's tmem_empty, and stores the four 32 x 64 chunks as in tg_mx_kernel.cuh, writing one
//     more slot (if ready) before each chunk after the first.
// The scale slots are written by the epilogue's threads, not by tcgen05.cp from the MMA
// thread: a .cta_group::2 copy costs the tensor pipe about 4 % of a k-block each, three per
// k-block, and the epilogue warps are idle for all but one drain per unit.  Bounded waits,
// abort propagation to the peer and the closing cluster barrier are those of
// tg_gemm_pair_kernel.cuh; each producer also waits for its own atom loads still in flight.
//
// Shared memory (1024-byte aligned): S stages of KB k-blocks (KB x 16 KiB of A, then KB x 16
// KiB of B, K-major, 128-byte swizzle), A x KB atom sets of 1536 bytes, one 4 KiB epilogue
// buffer per epilogue warp.  TMEM: the 256-column accumulator, then A x KB scale slots of 16
// columns.
#pragma once

#include "tg_gemm_pair_kernel.cuh"
#include "tg_mx_kernel.cuh"

namespace tg {

struct __align__(8) MxPairCtl {
  uint64_t loaded[kMxPairStages];    // used in the even CTA only
  uint64_t consumed[kMxPairStages];
  uint64_t sf_loaded[kMxPairSfSlots];  // this CTA's atoms of scale slot a have landed
  uint64_t sf_ready[kMxPairSfSlots];   // used in the even CTA only: both CTAs wrote scale slot a
  uint64_t tmem_full;
  uint64_t tmem_empty;               // used in the even CTA only (signalled like sf_ready)
  uint64_t drain;
  uint64_t odd_done;                 // even CTA: the odd producer has stopped filling
  PairFills<kMxPairStages> fills;
  uint32_t sink[kEpiWarps];          // even CTA: target of the odd epilogue warps' st.async
  uint32_t tmem_base;
  int abort;
};

// OUT: 0 = fp16 output, 1 = bf16 output.  p.m_blocks counts 256-row pair tiles.
template <int OUT, bool DEBUG>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    gemm_mxfp8_pair_ws_kernel(const __grid_constant__ CUtensorMap tmA,
                              const __grid_constant__ CUtensorMap tmB,
                              const __grid_constant__ CUtensorMap tmC,
                              const __grid_constant__ CUtensorMap tmSFA,
                              const __grid_constant__ CUtensorMap tmSFB, const MxParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ MxPairCtl ctl;

  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t rank = cluster_ctarank();          // 0: even CTA (issues the MMA), 1: odd
  const uint32_t pair = blockIdx.x >> 1;
  const uint32_t num_pairs = gridDim.x >> 1;
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  // stage s: A k-blocks g at sA0 + s * kMxPairStageBytes + g * kMxABytes, then B k-blocks at
  // sB0 + s * kMxPairStageBytes + g * kMxPairBBytes; atom set (a, g) of scale slot a at
  // sAtom0 + (a * KB + g) * 1536
  const uint32_t sA0 = sbase;
  const uint32_t sB0 = sbase + kMxPairKB * kMxABytes;
  const uint32_t sAtom0 = sbase + kMxPairStages * kMxPairStageBytes;
  const uint32_t sEpi = sAtom0 + kMxPairAtomRegionBytes;

  const uint32_t bar_loaded = smem_u32(&ctl.loaded[0]);
  const uint32_t bar_consumed = smem_u32(&ctl.consumed[0]);
  const uint32_t bar_sf_loaded = smem_u32(&ctl.sf_loaded[0]);
  const uint32_t bar_sf_ready = smem_u32(&ctl.sf_ready[0]);
  const uint32_t bar_tmem_full = smem_u32(&ctl.tmem_full);
  const uint32_t bar_tmem_empty = smem_u32(&ctl.tmem_empty);
  const uint32_t bar_drain = smem_u32(&ctl.drain);

  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < kMxPairStages; ++s) {
      mbar_init(bar_loaded + 8u * s, 1);
      mbar_init(bar_consumed + 8u * s, 1);
    }
#pragma unroll
    for (int a = 0; a < kMxPairSfSlots; ++a) {
      mbar_init(bar_sf_loaded + 8u * a, 1);
      mbar_init(bar_sf_ready + 8u * a, kEpiWarps);   // see pair_report_warp
    }
    mbar_init(bar_tmem_full, 1);
    mbar_init(bar_tmem_empty, kEpiWarps);
    mbar_init(bar_drain, 1);
    mbar_init(smem_u32(&ctl.odd_done), 1);
#pragma unroll
    for (int st = 0; st < kMxPairStages; ++st) ctl.fills.par[st] = 0;
    ctl.abort = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB);
    prefetch_tensormap(&tmC);
    prefetch_tensormap(&tmSFA);
    prefetch_tensormap(&tmSFB);
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
  const uint64_t k_stages = (p.k_blocks + kMxPairKB - 1) / kMxPairKB;   // stages per unit

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      PersistentTileScheduler sched(p.m_blocks, p.n_blocks, p.group, num_pairs, p.split_from,
                                    p.total_units, p.column_major);
      sched.init(pair);
      // the scale stream: its own cursor, kMxPairSfAhead stages ahead of the operands
      PersistentTileScheduler sf_sched(p.m_blocks, p.n_blocks, p.group, num_pairs,
                                       p.split_from, p.total_units, p.column_major);
      sf_sched.init(pair);
      uint32_t sf_j = 0;                       // stage of sf_sched's unit loaded next
      uint64_t sf_phase = 0;                   // phase whose atoms are loaded next
      uint32_t sf_armed = 0, sf_armed_par = 0; // scale slots armed; parity of their last phase
      // Loads the atoms of phase sf_phase, if this pair has it, into scale slot sf_phase % A.
      // The slot last held phase sf_phase - A, whose MMAs have completed once the producer has
      // seen consumed of every phase up to sf_phase - A (true at every call below).
      auto load_atoms = [&]() {
        if (!sf_sched.valid()) return;
        const uint32_t a = static_cast<uint32_t>(sf_phase % kMxPairSfSlots);
        const uint32_t par = static_cast<uint32_t>((sf_phase / kMxPairSfSlots) & 1u);
        const bool half = sf_sched.half_unit();
        const int32_t nu =
            static_cast<int32_t>(sf_sched.n_idx * kBN) + (half ? sf_sched.part * (kBN / 2) : 0);
        const int32_t sfa_row = static_cast<int32_t>(sf_sched.m_idx * 2 + rank);  // A row block
        const int32_t sfb_row = nu / kBM;                                        // first B row block
        const uint32_t sf_full = bar_sf_loaded + 8u * a;
        mbar_arrive_expect_tx(sf_full, kMxPairSfTxBytes);
#pragma unroll
        for (uint32_t g = 0; g < kMxPairKB; ++g) {
          const uint32_t k = sf_j * kMxPairKB + g;   // past K: zero-filled, never read
          const uint32_t atom = sAtom0 + (a * kMxPairKB + g) * kMxAtomSetBytes;
          tma_load_2d(atom, &tmSFA, sf_full, 0, static_cast<int32_t>(k * p.sfa_blocks) + sfa_row);
          tma_load_2d(atom + kMxSfAtomBytes, &tmSFB, sf_full, 0,
                      static_cast<int32_t>(k * p.sfb_blocks) + sfb_row);
        }
        sf_armed |= 1u << a;
        sf_armed_par = (sf_armed_par & ~(1u << a)) | (par << a);
        ++sf_phase;
        if (++sf_j == k_stages) {
          sf_j = 0;
          sf_sched.next_tile();
        }
      };
      for (int i = 0; i < kMxPairSfAhead; ++i) load_atoms();
      bool ok = true;
      while (ok && sched.valid()) {
        const uint64_t w = sched.current_iter;
        const bool half = sched.half_unit();
        const int32_t m0 = static_cast<int32_t>(sched.m_idx * (2 * kBM) + rank * kBM);
        const int32_t nu = static_cast<int32_t>(sched.n_idx * kBN) + (half ? sched.part * (kBN / 2) : 0);
        const int32_t nr = nu + static_cast<int32_t>(rank) * (half ? kBN / 4 : kBN / 2);
        for (uint32_t j = 0; j < k_stages; ++j) {
          const uint64_t phase = w * k_stages + j;
          const uint32_t s = static_cast<uint32_t>(phase % kMxPairStages);
          const uint32_t par = static_cast<uint32_t>((phase / kMxPairStages) & 1u);
          if (!pair_wait_or_abort(bar_consumed + 8u * s, par ^ 1u, abort_flag, peer_abort, limit,
                                  kRoleProducer)) {
            ok = false;
            break;
          }
          load_atoms();   // phase + ahead; its scale slot last held phase - S
          if (DEBUG && injected_skip(p.inject_skip_phase, phase))
            continue;  // injected fault: this CTA never arms or fills this phase's operands
          const uint32_t full_even = mapa_shared(bar_loaded + 8u * s, 0);
          if (rank == 0) mbar_arrive_expect_tx(bar_loaded + 8u * s, kMxPairTxBytes);
#pragma unroll
          for (uint32_t g = 0; g < kMxPairKB; ++g) {
            // k-blocks past K read as zeros (TMA fill past the tensor's edge)
            const int32_t kx = static_cast<int32_t>((j * kMxPairKB + g) * kMxBK);
            tma_load_2d_pair(sA0 + s * kMxPairStageBytes + g * kMxABytes, &tmA, full_even, kx, m0);
            tma_load_2d_pair(sB0 + s * kMxPairStageBytes + g * kMxPairBBytes, &tmB, full_even, kx, nr);
          }
          record_fill(ctl.fills, s, phase, par, kMxPairTxBytes / 2u);
        }
        sched.next_tile();
      }
      if (!ok) {   // atom loads of this CTA still in flight land before it may leave
        for (uint32_t a = 0; a < kMxPairSfSlots; ++a)
          if ((sf_armed >> a) & 1u)
            wait_bounded(bar_sf_loaded + 8u * a, (sf_armed_par >> a) & 1u, limit, kRoleDrain);
      }
      // the odd producer has stopped filling: its records are final (see pair_drain_fills)
      if (rank == 1) mbar_arrive_cluster(mapa_shared(smem_u32(&ctl.odd_done), 0));
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    if (lane == 0 && rank == 0) {
      PersistentTileScheduler sched(p.m_blocks, p.n_blocks, p.group, num_pairs, p.split_from,
                                    p.total_units, p.column_major);
      sched.init(pair);
      bool ok = true;
      while (ok && sched.valid()) {
        const uint32_t w = sched.current_iter;
        if (!pair_wait_or_abort<true>(bar_tmem_empty, (w & 1u) ^ 1u, abort_flag, peer_abort,
                                      limit, kRoleMma)) {
          ok = false;
          break;
        }
        tcgen05_fence_after_sync();
        const uint32_t idesc = sched.half_unit() ? idesc_mxf8(2 * kBM, kBN / 2, 0, 0)
                                               : idesc_mxf8(2 * kBM, kBN, 0, 0);
        for (uint32_t j = 0; j < k_stages; ++j) {
          const uint64_t phase = static_cast<uint64_t>(w) * k_stages + j;
          const uint32_t s = static_cast<uint32_t>(phase % kMxPairStages);
          const uint32_t par = static_cast<uint32_t>((phase / kMxPairStages) & 1u);
          const uint32_t a = static_cast<uint32_t>(phase % kMxPairSfSlots);
          const uint32_t a_par = static_cast<uint32_t>((phase / kMxPairSfSlots) & 1u);
          if (!pair_wait_or_abort(bar_loaded + 8u * s, par, abort_flag, peer_abort, limit,
                                  kRoleMma) ||
              !pair_wait_or_abort<true>(bar_sf_ready + 8u * a, a_par, abort_flag, peer_abort,
                                        limit, kRoleMma)) {
            ok = false;
            break;
          }
          tcgen05_fence_after_sync();
#pragma unroll
          for (uint32_t g = 0; g < kMxPairKB; ++g) {
            const uint32_t k = j * kMxPairKB + g;
            if (k >= p.k_blocks) break;   // the zero-filled tail of the last stage
            const uint32_t t_sf = tmem_base + kMxAccCols + (a * kMxPairKB + g) * kMxSfColsPerStage;
            const uint32_t a_addr = sA0 + s * kMxPairStageBytes + g * kMxABytes;
            const uint32_t b_addr = sB0 + s * kMxPairStageBytes + g * kMxPairBBytes;
#pragma unroll
            for (uint32_t kk = 0; kk < kMxBK / kMxUmmaK; ++kk) {
              const uint64_t a_desc = smem_desc_sw128(a_addr + kk * kMxUmmaK, 16, 1024);
              const uint64_t b_desc = smem_desc_sw128(b_addr + kk * kMxUmmaK, 16, 1024);
              umma_mxf8_pair(tmem_base, a_desc, b_desc, idesc | (kk << 29) | (kk << 4), t_sf,
                             t_sf + 4, (k | kk) != 0u ? 1u : 0u);
            }
          }
          umma_commit_pair_multicast(bar_consumed + 8u * s, 0x3);
        }
        if (!ok) break;
        umma_commit_pair_multicast(bar_tmem_full, 0x3);
        sched.next_tile();
      }
      umma_commit_pair_multicast(bar_drain, 0x1);
      wait_bounded(bar_drain, 0, limit, kRoleDrain);
    }
    __syncwarp();
  } else if (warp >= kFirstEpiWarp) {
    // ------------------------------------------------- scale slots and epilogue (both CTAs)
    const uint32_t q = warp - kFirstEpiWarp;       // TMEM lanes 32q .. 32q + 31
    PersistentTileScheduler sched(p.m_blocks, p.n_blocks, p.group, num_pairs, p.split_from,
                                  p.total_units, p.column_major);
    sched.init(pair);
    const uint32_t sbuf = sEpi + q * kEpiBufBytes;
    const uint32_t t_row = tmem_base + ((q * 32u) << 16);
    const uint32_t sink_even = mapa_shared(smem_u32(&ctl.sink[q]), 0);  // st.async target
    // scale phases of this pair: k_stages per unit it runs
    const uint32_t my_units =
        pair < p.total_units ? (p.total_units - 1u - pair) / num_pairs + 1u : 0u;
    const uint32_t total_ph = my_units * static_cast<uint32_t>(k_stages);
    uint32_t ps = 0;   // next phase whose scale slot this warp writes (phases < 2^32)
    // Writes the scale slot of phase ps into this warp's lane quadrant if its atoms have landed
    // (every lane must see the phase complete, each through its own barrier read); lane i
    // takes row i of each atom: the words of rows i, i + 32, i + 64, i + 96.
    auto write_scales = [&]() -> bool {
      if (ps >= total_ph) return false;
      const uint32_t a = ps % kMxPairSfSlots;
      const uint32_t par = (ps / kMxPairSfSlots) & 1u;
      if (!__all_sync(0xffffffffu, mbar_test_wait(bar_sf_loaded + 8u * a, par))) return false;
#pragma unroll
      for (uint32_t g = 0; g < kMxPairKB; ++g) {
        const uint32_t atom = sAtom0 + (a * kMxPairKB + g) * kMxAtomSetBytes + lane * 16u;
        uint32_t v[16];
        ld_shared_v4(atom, v[0], v[1], v[2], v[3]);
        ld_shared_v4(atom + kMxSfAtomBytes, v[4], v[5], v[6], v[7]);
        ld_shared_v4(atom + 2 * kMxSfAtomBytes, v[8], v[9], v[10], v[11]);
        v[12] = v[13] = v[14] = v[15] = 0u;
        tmem_st_32x32b_x16(t_row + kMxAccCols + (a * kMxPairKB + g) * kMxSfColsPerStage, v);
      }
      tcgen05_wait_st();
      tcgen05_fence_before_sync();
      pair_report_warp(bar_sf_ready + 8u * a, rank, lane, sink_even);
      ++ps;
      return true;
    };
    bool ok = true;
    while (ok && sched.valid()) {
      const uint32_t w = sched.current_iter;
      // keep the MMA supplied with scale slots until this unit's accumulator is complete
      uint64_t t_progress = globaltimer_ns();
      for (;;) {
        if (__all_sync(0xffffffffu, mbar_test_wait(bar_tmem_full, w & 1u))) break;
        if (write_scales()) {
          t_progress = globaltimer_ns();
          continue;
        }
        if (__any_sync(0xffffffffu, *abort_flag != 0)) {
          ok = false;
          break;
        }
        const bool late = globaltimer_ns() - t_progress > limit;
        if (__shfl_sync(0xffffffffu, late ? 1 : 0, 0)) {
          if (lane == 0) {
            *abort_flag = 1;
            st_shared_cluster_u32(peer_abort, 1u);
            atomicOr(&g_watchdog_status, kRoleEpilogue);
          }
          ok = false;
          break;
        }
      }
      if (!ok) break;
      tcgen05_fence_after_sync();
      const bool half = sched.half_unit();
      const int32_t row0 = static_cast<int32_t>(sched.m_idx * (2 * kBM) + rank * kBM + q * 32u);
      const int32_t col0 = static_cast<int32_t>(sched.n_idx * kBN) + (half ? sched.part * (kBN / 2) : 0);
      uint32_t packed[kBN / kEpiN][kEpiN / 2];
#pragma unroll
      for (uint32_t j = 0; j < kBN / kEpiN; ++j) {
        if (half && j >= kBN / kEpiN / 2) break;
#pragma unroll
        for (uint32_t h = 0; h < 2; ++h) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(t_row + j * kEpiN + h * 32u, v);
#pragma unroll
          for (uint32_t c = 0; c < 16; ++c) packed[j][16 * h + c] = pack_out<OUT>(v[2 * c], v[2 * c + 1]);
        }
      }
      tcgen05_fence_before_sync();
      pair_report_warp(bar_tmem_empty, rank, lane, sink_even);   // the next tile may start
#pragma unroll
      for (uint32_t j = 0; j < kBN / kEpiN; ++j) {
        if (half && j >= kBN / kEpiN / 2) break;
        if (j >= 1) write_scales();   // the next unit's MMAs run meanwhile
        mx_store_chunk(packed[j], lane, sbuf, &tmC, p.M, p.N, row0,
                       col0 + static_cast<int32_t>(j * kEpiN));
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
