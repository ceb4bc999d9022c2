// tg_gemm_pair_kernel.cuh -- the CTA-pair (tcgen05 cta_group::2) persistent GEMM.
//
// "[Feature] Introduce tile scheduler #2441", gemm_tcgen5mma_ws_persistent.py,
// ``gemm_persistent_2cta``: a cluster of two CTAs (``cluster_dims=2``) shares one 256 x 256
// output tile.  Each CTA loads its own 128-row slice of A and its own half of B's columns
// (``(by * 2 + cta_id) * block_N // 2``); only the even CTA issues the MMA
// (``use_2cta=True``), arrivals on ``loaded`` and ``tmem_empty`` go to the even CTA's
// barriers (``mbarrier_arrive(..., 0)``), and the MMA completions are signalled to both CTAs
// (``arrive_2cta=True``).  The scheduler runs per cluster (``init(block_id // cluster_size)``)
// over ceil(M / 256) x ceil(N / 256) pair tiles, and CTA r works on rows 256 * m_idx + 128 r
// (the page's ``bx = m_idx * cluster_size + cta_id``).  When M is not a multiple of 256 the
// odd CTA's slice of the last pair row lies partly or wholly past M: its TMA loads read zeros
// there and its stores are clipped or skipped, so nothing outside A or C is touched (the
// out-of-bounds ``bx`` the review of the PR warns about).
//
// Per CTA and k-block of 128: two A boxes 128 x 64 (32 KiB) and two B boxes 64 x 128 (32 KiB)
// into the CTA's own ring slot; both CTAs' bytes complete on the even CTA's ``loaded[s]``,
// which the even CTA arms with 128 KiB.  The MMA (M = 256, N = 256, K = 16, eight per k-block) reads A
// rows 0..127 and B columns 0..127 from the even CTA's slot and the rest from the odd
// CTA's slot at the same offset, and writes 128 rows into each CTA's TMEM.  tcgen05.commit
// with a CTA mask of 0b11 completes ``consumed[s]`` and ``tmem_full[w & 1]`` in both CTAs.
// Both CTAs' epilogue warps report on the even CTA's ``tmem_empty[w & 1]`` (pair_report_warp).
// A unit covers k-blocks sched.k_lo .. k_hi - 1 (all of them except in the stream-K tail), and
// the ring position is the count of k-blocks the role has handled so far.  In the tail a
// contribution's accumulator goes to the workspace instead of C, and an owned tile adds the
// contributions before it is stored (tg_streamk.cuh).
//
// All tcgen05 instructions of this kernel use cta_group::2.  Waits are bounded exactly as in
// the single-CTA kernel; an abort also raises the peer CTA's flag, and the pair meets at a
// cluster barrier before TMEM is freed, so neither CTA leaves while the other may still
// read its shared memory or write its TMEM.  Included by exactly one translation unit, after
// tg_gemm_kernel.cuh.
#pragma once

#include "tg_gemm_kernel.cuh"
#include "tg_streamk.cuh"

namespace tg {

// What a producer of a CTA pair last put on each ring slot, for the abort path: the phase
// (low 32 bits), 2 | the phase's parity on the slot (0: the slot was never filled), and this
// CTA's bytes of that fill.  Each CTA keeps its own in its shared memory.
template <int S>
struct PairFills {
  uint32_t phase[S];
  uint32_t par[S];
  uint32_t bytes[S];
};

struct __align__(8) PairCtl {
  uint64_t loaded[kPairStages];      // used in the even CTA only
  uint64_t consumed[kPairStages];
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];            // used in the even CTA only (see pair_report_warp)
  uint64_t drain;
  uint64_t odd_done;                 // even CTA: the odd producer has stopped filling
  PairFills<kPairStages> fills;
  uint32_t sink[kEpiWarps];          // even CTA: target of the odd epilogue warps' st.async
  uint64_t sk_bar[kEpiWarps];        // per epilogue warp: stream-K contributions landed
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ void st_shared_cluster_u32(uint32_t cluster_addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}

// Like wait_or_abort, but a timeout also raises the peer CTA's abort flag.  CLUSTER: acquire
// at cluster scope, for a phase that the peer CTA's threads complete with release semantics.
template <bool CLUSTER = false>
__device__ __forceinline__ bool pair_wait_or_abort(uint32_t bar, uint32_t parity,
                                                   volatile int* abort_flag,
                                                   uint32_t peer_abort_addr, uint64_t limit_ns,
                                                   uint32_t role) {
  auto ready = [&]() {
    return CLUSTER ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
  };
  if (ready()) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 16; ++i)
      if (ready()) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > limit_ns) {
      *abort_flag = 1;
      st_shared_cluster_u32(peer_abort_addr, 1u);
      atomicOr(&g_watchdog_status, role);
      return false;
    }
  }
}

// One epilogue warp reports to the pair's MMA thread on the even CTA's barrier ``bar`` (its
// shared::cta address; initialised with a count of kEpiWarps): the warp has finished its
// tcgen05 accesses and fenced them (tcgen05.fence::before_thread_sync).  Lane 0 reports for the
// warp: in the even CTA an arrive that expects 4 transaction bytes, in the odd CTA a 4-byte
// st.async to ``sink_even`` (an unused word of the even CTA) that completes them with release
// semantics at cluster scope.  The waiter acquires at cluster scope.  One report per warp,
// and st.async rather than a release-arrive on the peer's barrier, which held the warp for
// about 1250 cycles.
__device__ __forceinline__ void pair_report_warp(uint32_t bar, uint32_t rank, uint32_t lane,
                                                 uint32_t sink_even) {
  __syncwarp();
  if (lane == 0) {
    if (rank == 0)
      mbar_arrive_expect_tx(bar, 4);
    else
      st_async_u32(sink_even, 0u, mapa_shared(bar, 0));
  }
}

// Waits (every lane, acquire at gpu scope) until a stream-K flag holds ``epoch``; bounded like
// pair_wait_or_abort.  The contributor is a lower-numbered worker that started its tail before
// this one, so the wait ends unless a peer stopped.
__device__ __forceinline__ bool sk_wait_flag(const uint32_t* flag, uint32_t epoch,
                                             volatile int* abort_flag, uint32_t peer_abort_addr,
                                             uint64_t limit_ns) {
  if (ld_acquire_gpu(flag) == epoch) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 16; ++i)
      if (ld_acquire_gpu(flag) == epoch) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > limit_ns) {
      *abort_flag = 1;
      st_shared_cluster_u32(peer_abort_addr, 1u);
      atomicOr(&g_watchdog_status, kRoleEpilogue);
      return false;
    }
  }
}

// Contribution of one epilogue warp: its lanes' fp32 accumulator, ``chunks`` chunks of 64
// columns from TMEM address t_col (chunk indices c0 ..), staged through the warp's two 4 KiB
// buffers (half a chunk each) and bulk-stored into ``slot``.  Lane 0 issues the copies; the
// caller publishes (sk_publish), which waits for them.
__device__ __forceinline__ void sk_write_slot(float4* slot, uint32_t t_col, uint32_t chunks,
                                              uint32_t c0, uint32_t q, uint32_t lane,
                                              uint32_t sbuf0, uint32_t sbuf1) {
  if (lane == 0) bulk_wait_group_read<0>();   // earlier stores are done reading the buffers
  __syncwarp();
#pragma unroll 1
  for (uint32_t j = 0; j < chunks; ++j) {
    uint32_t v[64];
    tmem_ld_32x32b_x64(t_col + j * kEpiN, v);
#pragma unroll
    for (uint32_t hh = 0; hh < 2; ++hh) {
      const uint32_t buf = hh ? sbuf1 : sbuf0;
      if (j > 0 || hh > 0) {
        if (lane == 0) bulk_wait_group_read<1>();   // the other buffer's copy may still read
        __syncwarp();
      }
#pragma unroll
      for (uint32_t g = 0; g < 8; ++g)
        st_shared_v4(buf + (g * 32u + lane) * 16u, v[4 * (8 * hh + g)], v[4 * (8 * hh + g) + 1],
                     v[4 * (8 * hh + g) + 2], v[4 * (8 * hh + g) + 3]);
      fence_proxy_async_shared();
      __syncwarp();
      if (lane == 0) {
        bulk_store(slot + sk_chunk_f4(c0 + j, q) + 8u * hh * 32u, buf, 4096u);
        bulk_commit_group();
      }
    }
  }
}

// Owner of a stream-K tile, one epilogue warp: adds the contributions of workers c_lo .. c_hi - 1
// (those with a tail range) to its lanes' fp32 accumulator, ``chunks`` chunks of 64 columns at
// TMEM address t_col (chunk indices c0 ..): per contribution, wait for its flag (``wait_flags``),
// bulk-load the warp's part into ``region`` (chunks x 8 KiB of idle shared memory) on the warp's
// barrier ``bar`` (phase count ``*bar_uses``), then read, add and write back each chunk.  False
// if a wait ran out or the CTA is stopping.
__device__ bool sk_gather(const GemmParams& p, uint32_t c_lo, uint32_t c_hi, uint32_t workers,
                          uint32_t rank, uint32_t q, uint32_t lane, uint32_t t_col,
                          uint32_t chunks, uint32_t c0, uint32_t region, uint32_t bar,
                          uint32_t* bar_uses, bool wait_flags, volatile int* abort_flag,
                          uint32_t peer_abort, uint64_t limit) {
#pragma unroll 1
  for (uint32_t c = c_lo; c < c_hi; ++c) {
    if (!sk_has_range(c, workers, p.sk_tiles, p.k_blocks)) continue;
    const bool seen = !wait_flags || sk_wait_flag(p.sk_flags + sk_flag_index(c, rank, q),
                                                  p.sk_epoch, abort_flag, peer_abort, limit);
    if (!__all_sync(0xffffffffu, seen)) return false;
    const float4* slot = sk_slot(p.sk_partials, p.sk_slot_f4, c, rank);
    if (lane == 0) {
      fence_proxy_async_global();   // the flag was acquired; the copies read after it
      mbar_arrive_expect_tx(bar, chunks * 8192u);
      for (uint32_t j = 0; j < chunks; ++j)
        bulk_load(region + j * 8192u, slot + sk_chunk_f4(c0 + j, q), 8192u, bar);
    }
    const bool landed = pair_wait_or_abort(bar, *bar_uses & 1u, abort_flag, peer_abort, limit,
                                           kRoleEpilogue);
    ++*bar_uses;
    if (!__all_sync(0xffffffffu, landed)) return false;
#pragma unroll 1
    for (uint32_t j = 0; j < chunks; ++j) {
      uint32_t v[64];
      tmem_ld_32x32b_x64(t_col + j * kEpiN, v);
#pragma unroll
      for (uint32_t g = 0; g < 16; ++g) {
        uint32_t x0, x1, x2, x3;
        ld_shared_v4(region + j * 8192u + (g * 32u + lane) * 16u, x0, x1, x2, x3);
        v[4 * g] = __float_as_uint(__uint_as_float(v[4 * g]) + __uint_as_float(x0));
        v[4 * g + 1] = __float_as_uint(__uint_as_float(v[4 * g + 1]) + __uint_as_float(x1));
        v[4 * g + 2] = __float_as_uint(__uint_as_float(v[4 * g + 2]) + __uint_as_float(x2));
        v[4 * g + 3] = __float_as_uint(__uint_as_float(v[4 * g + 3]) + __uint_as_float(x3));
      }
#pragma unroll
      for (uint32_t i = 0; i < 4; ++i) {
        uint32_t (&part)[16] = *reinterpret_cast<uint32_t(*)[16]>(&v[16 * i]);
        tmem_st_32x32b_x16(t_col + j * kEpiN + 16u * i, part);
      }
      tcgen05_wait_st();
    }
    __syncwarp();   // every lane has read the region before the next contribution overwrites it
  }
  return true;
}

template <int S>
__device__ __forceinline__ void record_fill(PairFills<S>& f, uint32_t s, uint64_t phase,
                                            uint32_t par, uint32_t bytes) {
  f.phase[s] = static_cast<uint32_t>(phase);
  f.par[s] = 2u | par;
  f.bytes[s] = bytes;
}

// The abort path of a CTA pair: run by one thread of the even CTA once every role of that CTA
// has left its loop, before the closing cluster barrier (which the odd CTA cannot pass any
// earlier).  Every TMA load of either CTA completes on the even CTA's ``loaded`` barriers; this
// waits until all of them have landed, so neither CTA leaves while a copy may still write its
// shared memory.  Once the odd producer has said on ``bar_odd_done`` that it has stopped, its
// fill records are read over DSMEM and compared slot by slot with this CTA's:
//  * the odd CTA filled a phase this CTA never armed (this producer stopped one ring earlier):
//    arm that phase with the odd CTA's bytes and wait for it;
//  * this CTA armed a phase the odd CTA never filled: count the odd CTA's share as done (both
//    CTAs load the same shapes, so it equals this CTA's bytes) and wait for this CTA's loads;
//  * both filled the same phase: wait for it.
// The two producers' last fills of a slot are the same phase or one ring apart, since each
// waits for the slot to be consumed, and consuming needs both CTAs' bytes.
template <int S>
__device__ void pair_drain_fills(uint32_t bar_loaded, const PairFills<S>& own,
                                 uint32_t odd_fills, uint32_t bar_odd_done, uint64_t limit) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait_cluster(bar_odd_done, 0)) {
    if (globaltimer_ns() - t0 > limit) {
      atomicOr(&g_watchdog_status, kRoleDrain);
      return;
    }
  }
#pragma unroll 1
  for (uint32_t s = 0; s < static_cast<uint32_t>(S); ++s) {
    const uint32_t e_par = own.par[s];
    const uint32_t o_par = ld_shared_cluster_u32(odd_fills + 4u * (S + s));
    if (!(e_par & 2u) && !(o_par & 2u)) continue;
    const uint32_t bar = bar_loaded + 8u * s;
    const uint32_t o_phase = ld_shared_cluster_u32(odd_fills + 4u * s);
    const int32_t ahead = static_cast<int32_t>(o_phase - own.phase[s]);
    if ((o_par & 2u) && (!(e_par & 2u) || ahead > 0)) {
      mbar_arrive_expect_tx(bar, ld_shared_cluster_u32(odd_fills + 4u * (2 * S + s)));
      wait_bounded(bar, o_par & 1u, limit, kRoleDrain);
    } else {
      if (!(o_par & 2u) || ahead != 0) mbar_complete_tx(bar, own.bytes[s]);
      wait_bounded(bar, e_par & 1u, limit, kRoleDrain);
    }
  }
}

// DT: 0 = fp16, 1 = bf16.  p.m_blocks counts 256-row pair tiles, p.n_blocks 256-column tiles.
template <int DT, bool DEBUG>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    gemm_pair_ws_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmC, const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ PairCtl ctl;

  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t rank = cluster_ctarank();          // 0: even CTA (issues the MMA), 1: odd
  const uint32_t pair = blockIdx.x >> 1;
  const uint32_t num_pairs = gridDim.x >> 1;
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sA0 = sbase;                        // A of stage s: sA0 + s * kPairStageBytes
  const uint32_t sB0 = sbase + kPairABytes;              // B of stage s: sB0 + s * kPairStageBytes
  const uint32_t sEpi = sbase + kPairStages * kPairStageBytes;

  const uint32_t bar_loaded = smem_u32(&ctl.loaded[0]);
  const uint32_t bar_consumed = smem_u32(&ctl.consumed[0]);
  const uint32_t bar_tmem_full = smem_u32(&ctl.tmem_full[0]);
  const uint32_t bar_tmem_empty = smem_u32(&ctl.tmem_empty[0]);
  const uint32_t bar_drain = smem_u32(&ctl.drain);

  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < kPairStages; ++s) {
      mbar_init(bar_loaded + 8u * s, 1);
      mbar_init(bar_consumed + 8u * s, 1);
    }
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_tmem_full + 8u * b, 1);
      mbar_init(bar_tmem_empty + 8u * b, kEpiWarps);
    }
    mbar_init(bar_drain, 1);
    mbar_init(smem_u32(&ctl.odd_done), 1);
#pragma unroll
    for (int q = 0; q < kEpiWarps; ++q) mbar_init(smem_u32(&ctl.sk_bar[q]), 1);
#pragma unroll
    for (int st = 0; st < kPairStages; ++st) ctl.fills.par[st] = 0;
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
      const uint64_t pol_a = l2_policy<kAPolicy>();
      const uint64_t pol_b = l2_policy<kBPolicy>();
      bool ok = true;
      uint64_t phase = 0;   // k-blocks filled so far: the ring position of the next one
      while (ok && sched.valid()) {
        const bool half = sched.half_unit();          // half-width unit of the tail split
        const int32_t m0 = static_cast<int32_t>(sched.m_idx * kPairBM + rank * kBM);
        // whole unit: CTA r loads columns [128 r, 128 r + 128) of the 256-wide tile;
        // half unit (128 wide, starting at 128 * part): CTA r loads [64 r, 64 r + 64) of it
        const int32_t n0 = static_cast<int32_t>(sched.n_idx * kBN) +
                           (half ? sched.part * (kBN / 2) + static_cast<int32_t>(rank) * (kPairBNHalf / 2)
                                 : static_cast<int32_t>(rank) * kPairBNHalf);
        const uint32_t b_chunks = half ? kPairBNHalf / kBChunkCols / 2 : kPairBNHalf / kBChunkCols;
        const uint32_t tx_bytes = 2u * (kPairABytes + b_chunks * kPairBChunkBytes);
        for (uint32_t k = sched.k_lo; k < sched.k_hi; ++k, ++phase) {
          const uint32_t s = static_cast<uint32_t>(phase % kPairStages);
          const uint32_t par = static_cast<uint32_t>((phase / kPairStages) & 1u);
          if (!pair_wait_or_abort(bar_consumed + 8u * s, par ^ 1u, abort_flag, peer_abort, limit,
                                  kRoleProducer)) {
            ok = false;
            break;
          }
          if (DEBUG && injected_skip(p.inject_skip_phase, phase))
            continue;  // injected fault: this CTA never arms or fills this phase
          const uint32_t full_even = mapa_shared(bar_loaded + 8u * s, 0);
          if (rank == 0) mbar_arrive_expect_tx(bar_loaded + 8u * s, tx_bytes);
          const int32_t kx = static_cast<int32_t>(k) * kPairBK;
#pragma unroll
          for (uint32_t a = 0; a < kPairKAtoms; ++a) {
            const uint32_t dst = sA0 + s * kPairStageBytes + a * kAAtomBytes;
            const int32_t ax = kx + static_cast<int32_t>(a * kKAtom);
            if (kAPolicy != 0)
              tma_load_2d_pair_hint(dst, &tmA, full_even, ax, m0, pol_a);
            else
              tma_load_2d_pair(dst, &tmA, full_even, ax, m0);
          }
#pragma unroll
          for (uint32_t c = 0; c < kPairBNHalf / kBChunkCols; ++c) {
            if (c >= b_chunks) break;
            const uint32_t dst = sB0 + s * kPairStageBytes + c * kPairBChunkBytes;
            const int32_t nx = n0 + static_cast<int32_t>(c * kBChunkCols);
            if (kBPolicy != 0)
              tma_load_2d_pair_hint(dst, &tmB, full_even, nx, kx, pol_b);
            else
              tma_load_2d_pair(dst, &tmB, full_even, nx, kx);
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
      constexpr uint32_t idesc_full = idesc_f16(DT, kPairBM, kBN, /*A K-major*/ 0, /*B N-major*/ 1);
      constexpr uint32_t idesc_half = idesc_f16(DT, kPairBM, kBN / 2, 0, 1);
      PersistentTileScheduler sched(p.m_blocks, p.n_blocks, p.group, num_pairs, p.split_from,
                                    p.total_units, p.column_major, p.k_blocks, p.sk_tiles);
      sched.init(pair);
      bool ok = true;
      uint64_t phase = 0;
      while (ok && sched.valid()) {
        const uint32_t w = sched.current_iter;
        const uint32_t buf = w & 1u;
        if (!pair_wait_or_abort<true>(bar_tmem_empty + 8u * buf, ((w >> 1) & 1u) ^ 1u, abort_flag,
                                peer_abort, limit, kRoleMma)) {
          ok = false;
          break;
        }
        tcgen05_fence_after_sync();
        const uint32_t d_tmem = tmem_base + buf * kBN;
        const uint32_t idesc = sched.half_unit() ? idesc_half : idesc_full;
        for (uint32_t k = sched.k_lo; k < sched.k_hi; ++k, ++phase) {
          const uint32_t s = static_cast<uint32_t>(phase % kPairStages);
          const uint32_t par = static_cast<uint32_t>((phase / kPairStages) & 1u);
          if (!pair_wait_or_abort(bar_loaded + 8u * s, par, abort_flag, peer_abort, limit,
                                  kRoleMma)) {
            ok = false;
            break;
          }
          tcgen05_fence_after_sync();
          const uint32_t a_addr = sA0 + s * kPairStageBytes;
          const uint32_t b_addr = sB0 + s * kPairStageBytes;
#pragma unroll
          for (uint32_t kk = 0; kk < kPairBK / kUmmaK; ++kk) {
            const uint32_t a_off = (kk / (kKAtom / kUmmaK)) * kAAtomBytes +
                                   (kk % (kKAtom / kUmmaK)) * kUmmaK * kElemBytes;
            const uint64_t a_desc = smem_desc_sw128(a_addr + a_off, 16, 1024);
            const uint64_t b_desc = smem_desc_sw128(b_addr + kk * kUmmaK * 128u, kPairBChunkBytes, 1024);
            umma_f16_pair(d_tmem, a_desc, b_desc, idesc, (k != sched.k_lo || kk != 0u) ? 1u : 0u);
          }
          umma_commit_pair_multicast(bar_consumed + 8u * s, 0x3);
        }
        if (!ok) break;
        umma_commit_pair_multicast(bar_tmem_full + 8u * buf, 0x3);
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
      const uint32_t buf = w & 1u;
      const bool got = pair_wait_or_abort(bar_tmem_full + 8u * buf, (w >> 1) & 1u, abort_flag,
                                          peer_abort, limit, kRoleEpilogue);
      if (!__all_sync(0xffffffffu, got)) break;
      tcgen05_fence_after_sync();
      const bool half = sched.half_unit();
      const int32_t row0 =
          static_cast<int32_t>(sched.m_idx * kPairBM + rank * kBM + q * 32u);
      const int32_t col0 = static_cast<int32_t>(sched.n_idx) * kBN + (half ? sched.part * (kBN / 2) : 0);
      const uint32_t chunks = half ? kBN / kEpiN / 2 : kBN / kEpiN;
      const uint32_t t_row = tmem_base + ((q * 32u) << 16) + buf * kBN;
      // stream-K tail: a contribution goes to this worker's slot (no store); an owned tile first
      // adds the contributions of workers sk_lowest_worker .. pair - 1 into its accumulator
      const int32_t kind = sched.part;
      if (kind == 2) {
        sk_write_slot(sk_slot(p.sk_partials, p.sk_slot_f4, pair, rank), t_row, chunks, 0, q,
                      lane, sEpi + q * 2u * kEpiBufBytes, sEpi + (q * 2u + 1u) * kEpiBufBytes);
        tcgen05_fence_before_sync();
        pair_report_warp(bar_tmem_empty + 8u * buf, rank, lane, sink_even);
        sk_publish(p.sk_flags + sk_flag_index(pair, rank, q), p.sk_epoch, lane);
      } else {
        if (kind == 3 &&
            !sk_gather(p, sk_lowest_worker(pair, num_pairs, p.sk_tiles, p.k_blocks, sched.sk_tile),
                       pair, num_pairs, rank, q, lane, t_row, chunks, 0,
                       sA0 + q * (kPairStages * kPairStageBytes / kEpiWarps),
                       smem_u32(&ctl.sk_bar[q]), &sk_bar_uses, true, abort_flag, peer_abort,
                       limit))
          break;
#pragma unroll 1
        for (uint32_t j = 0; j < chunks; ++j, ++chunk) {
          uint32_t v[64];
          tmem_ld_32x32b_x64(t_row + j * kEpiN, v);
          if (j == chunks - 1) {
            tcgen05_fence_before_sync();
            pair_report_warp(bar_tmem_empty + 8u * buf, rank, lane, sink_even);
          }
          const uint32_t sbuf = sEpi + (q * 2u + (chunk & 1u)) * kEpiBufBytes;
          epilogue_store_chunk<DT>(v, lane, sbuf, &tmC, p, row0,
                                   col0 + static_cast<int32_t>(j * kEpiN));
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
