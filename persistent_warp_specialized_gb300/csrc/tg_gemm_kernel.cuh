// tg_gemm_kernel.cuh -- persistent, warp-specialized GEMM for sm_103a (tcgen05 + TMA).
//
// Structure ("[Feature] Introduce tile scheduler #2441", gemm_tcgen5mma_ws_persistent.py,
// ``gemm_persistent``, and the sequence diagram of the PR conversation):
//   * one CTA per SM (grid = min(#SMs, #tiles)) loops over output tiles of 128 x 256;
//   * warp 0 (one lane): TMA producer.  For each tile and k-block, phase = w * k_blocks + k,
//     slot s = phase % S: wait consumed[s] (parity ((phase / S) & 1) ^ 1), arm loaded[s]
//     with the stage's byte count, load the A box (128 x 64) and four B boxes (64 x 64);
//   * warp 1 (one lane): MMA issuer.  For tile w: wait tmem_empty[w & 1] (parity
//     ((w / 2) & 1) ^ 1); for each k-block wait loaded[s] (parity (phase / S) & 1) and issue
//     four tcgen05.mma 128 x 256 x 16 into accumulator w & 1, the first with accumulate off
//     (clear_accum = k == 0); tcgen05.commit -> consumed[s] frees the slot when those MMAs
//     are done.  After the k-loop, tcgen05.commit -> tmem_full[w & 1];
//   * warps 4..7: epilogue.  Wait tmem_full[w & 1] (parity (w / 2) & 1), copy the 32 TMEM
//     lanes of the warp to registers 64 columns at a time, release the accumulator
//     (arrive tmem_empty[w & 1]) as soon as the last columns are in registers -- before
//     the global stores, as on the page -- then convert to the output type, stage each
//     32 x 64 chunk in shared memory (128-byte swizzle) and TMA-store it (store_block_N
//     chunks through C_shared, the page's use_tma_store path).  The TMA store clips rows
//     >= M and columns >= N, which is the boundary masking of partial edge tiles;
//   * warp 2 allocates the 512 TMEM columns at start and frees them at exit.
// Every role builds its own PersistentTileScheduler and follows ``while valid(): ...
// next_tile()``; the scheduler's ``current_iter`` is the single clock w.
//
// Every wait is bounded (watchdog): a wait that has not completed after ``watchdog_ns``
// sets the per-device status word and a CTA-wide abort flag, every role then leaves its
// loop at its next wait, the producer waits (bounded) for the loads it still has in
// flight, the MMA thread waits (bounded) for its MMAs, the epilogue waits for its stores,
// and the CTA frees TMEM and exits.  The host reads the status word (tg_device_status).
//
// Shared memory layout (dynamic, 1024-byte aligned): stage s at s * 48 KiB holds A
// (128 rows x 128 bytes, K-major, 128-byte swizzle: row r's 16-byte chunk c sits at chunk
// c ^ (r % 8)) followed by B as four 8 KiB column chunks (64 K-rows x 64 N-columns each,
// N-major, same swizzle); then 8 epilogue staging buffers (2 per epilogue warp) of
// 32 rows x 128 bytes.  This header is included by exactly one translation unit.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "tg_config.h"
#include "tg_ptx.cuh"
#include "tg_tile_scheduler.cuh"

namespace tg {

struct GemmParams {
  void* C;                     // output base (used by the direct-store epilogue)
  uint32_t M, N, K;
  uint32_t m_blocks, n_blocks, k_blocks, group;
  uint32_t split_from, total_units;   // tail split of the scheduler (see tg_tile_scheduler.cuh)
  uint32_t column_major;              // scheduler order option
  uint32_t dynamic;                   // 1: units handed out by cluster launch control
  uint32_t epi_direct;                // 1: the epilogue stores from registers (no TMA store)
  uint64_t watchdog_ns;
  int32_t* trace;              // debug instantiation only; may be null (5 int32 per unit)
  int64_t inject_skip_phase;   // debug instantiation only; -1 = none
  // stream-K tail of the CTA-pair kernels (tg_streamk.cuh); sk_tiles = 0: none
  uint32_t sk_tiles;
  uint32_t sk_epoch;           // this launch's flag value
  uint32_t sk_slot_f4;         // float4s per (worker, CTA) partial slot
  uint32_t* sk_flags;
  float4* sk_partials;
};

// Debug fault injection: ``inject`` = cta * 2^32 + phase names a pipeline phase that the producer
// of CTA ``cta`` skips (-1: none).
__device__ __forceinline__ bool injected_skip(int64_t inject, uint64_t phase) {
  return inject >= 0 && (static_cast<uint64_t>(inject) & 0xFFFFFFFFull) == phase &&
         (static_cast<uint64_t>(inject) >> 32) == blockIdx.x;
}

// Per-device status word of the watchdog (bits: kRole*).  Read and cleared by the host.
__device__ unsigned int g_watchdog_status = 0;

struct __align__(16) GemmCtl {
  uint4 sched_resp[kSchedSlots];      // cluster-launch-control responses (dynamic mode)
  uint64_t sched_full[kSchedSlots];
  uint64_t sched_empty[kSchedSlots];
  uint64_t loaded[kStages];
  uint64_t consumed[kStages];
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

// Wait for the phase of parity ``parity`` of ``bar``; false if the CTA is aborting or the
// wait ran past ``limit_ns`` (then this thread raises the abort and records ``role``).
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity,
                                              volatile int* abort_flag, uint64_t limit_ns,
                                              uint32_t role) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 16; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > limit_ns) {
      *abort_flag = 1;
      atomicOr(&g_watchdog_status, role);
      return false;
    }
  }
}

// Bounded wait used while shutting down (ignores the abort flag).
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                             uint32_t role) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 16; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > limit_ns) {
      atomicOr(&g_watchdog_status, role);
      return false;
    }
  }
}

template <int DT>
__device__ __forceinline__ uint32_t pack_out(uint32_t lo_bits, uint32_t hi_bits) {
  const float lo = __uint_as_float(lo_bits);
  const float hi = __uint_as_float(hi_bits);
  if constexpr (DT == 1) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
  } else {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
}

// Converts one 64-column chunk of a warp's accumulator rows (v: lane = row, fp32 bits) to the
// output type: pk[i] holds columns 2i and 2i + 1 (round to nearest even).
template <int DT>
__device__ __forceinline__ void pack_chunk(const uint32_t (&v)[64], uint32_t (&pk)[32]) {
#pragma unroll
  for (uint32_t i = 0; i < 32; ++i) pk[i] = pack_out<DT>(v[2 * i], v[2 * i + 1]);
}

// Stores this warp's 32 rows x 64 columns, already converted (pk: lane = row, 32 words of two
// output values), at rows row0 .. row0 + 31 and columns x .. x + 63 of C.  Rows >= M and
// columns >= N are not written.
//  * staged (default): each lane writes its row as eight 16-byte chunks into a 128-byte
//    swizzled staging buffer (chunk c of row r at chunk c ^ (r % 8): conflict-free), the
//    warp fences the writes into the async proxy, and lane 0 issues one TMA store, which
//    clips at the tensor's edge.  Two buffers per warp alternate; before one is rewritten,
//    lane 0 waits until the store that read it is done.  One bulk group per chunk.
//  * direct (p.epi_direct): each lane stores its row's 128 bytes with 16-byte stores.
__device__ __forceinline__ void epilogue_store_packed(const uint32_t (&pk)[32], uint32_t lane,
                                                      uint32_t sbuf, const CUtensorMap* tmC,
                                                      const GemmParams& p, int32_t row0,
                                                      int32_t x) {
  if (p.epi_direct) {
    const int32_t row = row0 + static_cast<int32_t>(lane);
    if (row < static_cast<int32_t>(p.M)) {
      char* base = static_cast<char*>(p.C) +
                   (static_cast<uint64_t>(row) * p.N + static_cast<uint64_t>(x)) * kElemBytes;
#pragma unroll
      for (uint32_t c = 0; c < 8; ++c) {
        if (x + static_cast<int32_t>(8 * c) < static_cast<int32_t>(p.N))
          st_global_v4(base + 16 * c, pk[4 * c + 0], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      }
    }
  } else {
    if (lane == 0) bulk_wait_group_read<1>();   // the store that last read sbuf is done
    __syncwarp();
    const uint32_t row_addr = sbuf + lane * 128u;
#pragma unroll
    for (uint32_t c = 0; c < 8; ++c)
      st_shared_v4(row_addr + ((c ^ (lane & 7u)) << 4), pk[4 * c + 0], pk[4 * c + 1],
                   pk[4 * c + 2], pk[4 * c + 3]);
    fence_proxy_async_shared();
    __syncwarp();
    if (lane == 0) {
      if (row0 < static_cast<int32_t>(p.M) && x < static_cast<int32_t>(p.N)) {
        if (kCPolicy != 0)
          tma_store_2d_hint(tmC, sbuf, x, row0, l2_policy<kCPolicy>());
        else
          tma_store_2d(tmC, sbuf, x, row0);
      }
      bulk_commit_group();   // one group per chunk, empty when the chunk is outside C
    }
  }
  __syncwarp();   // converged for the next warp-collective tcgen05.ld
}

// Converts and stores one 64-column chunk of the accumulator (v: lane = row, fp32 bits); see
// epilogue_store_packed.
template <int DT>
__device__ __forceinline__ void epilogue_store_chunk(const uint32_t (&v)[64], uint32_t lane,
                                                     uint32_t sbuf, const CUtensorMap* tmC,
                                                     const GemmParams& p, int32_t row0,
                                                     int32_t x) {
  uint32_t pk[32];
  pack_chunk<DT>(v, pk);
  epilogue_store_packed(pk, lane, sbuf, tmC, p, row0, x);
}

// Dynamic persistence (cluster launch control).  The grid holds one CTA per work unit; a CTA
// first runs the unit of its own index, then takes over the units of CTAs that have not been
// launched yet: warp 3 asks the hardware to cancel one pending CTA at a time
// (clusterlaunchcontrol.try_cancel) into a ring of kSchedSlots responses.  Fetch j (0-based:
// the unit that follows the CTA's iteration j) sits in slot j % kSchedSlots, the (j /
// kSchedSlots)-th use of that slot, completed on sched_full; each of the kSchedConsumers
// readers arrives on sched_empty once it has read it.  A response that cancelled nothing ends
// the CTA's traversal.
enum ClcNext : int { kClcUnit = 0, kClcDone = 1, kClcAbort = 2 };

// ``j``: the iteration just finished (the fetch index); the next unit becomes iteration j + 1.
__device__ __forceinline__ int clc_next_unit(PersistentTileScheduler& sched, uint32_t j,
                                             uint32_t resp0, uint32_t full0, uint32_t empty0,
                                             volatile int* abort_flag, uint64_t limit,
                                             uint32_t role, bool warp_wide, bool arrive) {
  const uint32_t slot = j % kSchedSlots;
  const uint32_t par = (j / kSchedSlots) & 1u;
  bool got = wait_or_abort(full0 + 8u * slot, par, abort_flag, limit, role);
  if (warp_wide) got = __all_sync(0xffffffffu, got);
  if (!got) {
    sched.finish();
    return kClcAbort;
  }
  uint32_t unit = 0;
  const bool cancelled = clc_response(resp0 + 16u * slot, &unit);
  if (warp_wide) __syncwarp();
  if (arrive) mbar_arrive(empty0 + 8u * slot);
  if (!cancelled) {
    sched.finish();
    return kClcDone;
  }
  sched.jump(unit, j + 1);
  return kClcUnit;
}

// A and B loads of one k-block slot, with the configured L2 policies.
__device__ __forceinline__ void load_operand(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                             int32_t x, int32_t y, uint64_t policy, int kind) {
  if (kind != 0)
    tma_load_2d_hint(dst, map, bar, x, y, policy);
  else
    tma_load_2d(dst, map, bar, x, y);
}

// DT: 0 = fp16, 1 = bf16 (input and output).  DEBUG adds the tile trace and fault injection.
template <int DT, bool DEBUG>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_persistent_ws_kernel(const __grid_constant__ CUtensorMap tmA,
                              const __grid_constant__ CUtensorMap tmB,
                              const __grid_constant__ CUtensorMap tmC, const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ GemmCtl ctl;

  const uint32_t warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sA0 = sbase;                     // A of stage s: sA0 + s * kStageBytes
  const uint32_t sB0 = sbase + kABytes;           // B of stage s: sB0 + s * kStageBytes
  const uint32_t sEpi = sbase + kStages * kStageBytes;

  const uint32_t bar_loaded = smem_u32(&ctl.loaded[0]);
  const uint32_t bar_consumed = smem_u32(&ctl.consumed[0]);
  const uint32_t bar_tmem_full = smem_u32(&ctl.tmem_full[0]);
  const uint32_t bar_tmem_empty = smem_u32(&ctl.tmem_empty[0]);
  const uint32_t bar_drain = smem_u32(&ctl.drain);
  const uint32_t sched_resp0 = smem_u32(&ctl.sched_resp[0]);
  const uint32_t sched_full0 = smem_u32(&ctl.sched_full[0]);
  const uint32_t sched_empty0 = smem_u32(&ctl.sched_empty[0]);

  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar_loaded + 8u * s, 1);
      mbar_init(bar_consumed + 8u * s, 1);
    }
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_tmem_full + 8u * b, 1);
      mbar_init(bar_tmem_empty + 8u * b, kEpiThreads);
    }
    mbar_init(bar_drain, 1);
#pragma unroll
    for (int i = 0; i < kSchedSlots; ++i) {
      mbar_init(sched_full0 + 8u * i, 1);
      mbar_init(sched_empty0 + 8u * i, kSchedConsumers);
    }
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
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      PersistentTileScheduler sched(p.m_blocks, p.n_blocks, p.group, gridDim.x, p.split_from,
                                    p.total_units, p.column_major);
      sched.init(blockIdx.x);
      const uint64_t pol_a = l2_policy<kAPolicy>();
      const uint64_t pol_b = l2_policy<kBPolicy>();
      uint32_t pending = 0;       // stages whose latest fill may still be in flight
      uint32_t pending_par = 0;   // parity of that fill, one bit per stage
      bool ok = true;
      while (ok && sched.valid()) {
        const uint64_t w = sched.current_iter;
        const bool half = sched.half_unit();              // half-width unit of the tail split
        const int32_t m0 = static_cast<int32_t>(sched.m_idx) * kBM;
        const int32_t n0 = static_cast<int32_t>(sched.n_idx) * kBN + (half ? sched.part * (kBN / 2) : 0);
        const uint32_t b_chunks = half ? kBN / kBChunkCols / 2 : kBN / kBChunkCols;
        const uint32_t tx_bytes = kABytes + b_chunks * kBChunkBytes;
        for (uint32_t k = 0; k < p.k_blocks; ++k) {
          const uint64_t phase = w * k_blocks + k;
          const uint32_t s = static_cast<uint32_t>(phase % kStages);
          const uint32_t par = static_cast<uint32_t>((phase / kStages) & 1u);
          if (!wait_or_abort(bar_consumed + 8u * s, par ^ 1u, abort_flag, limit, kRoleProducer)) {
            ok = false;
            break;
          }
          pending &= ~(1u << s);
          if (DEBUG && injected_skip(p.inject_skip_phase, phase))
            continue;  // injected fault: this CTA never fills this phase
          const uint32_t full = bar_loaded + 8u * s;
          mbar_arrive_expect_tx(full, tx_bytes);
          const int32_t kx = static_cast<int32_t>(k) * kBK;
#pragma unroll
          for (uint32_t a = 0; a < kKAtoms; ++a)
            load_operand(sA0 + s * kStageBytes + a * kAAtomBytes, &tmA, full,
                         kx + static_cast<int32_t>(a * kKAtom), m0, pol_a, kAPolicy);
#pragma unroll
          for (uint32_t c = 0; c < kBN / kBChunkCols; ++c)
            if (c < b_chunks)
              load_operand(sB0 + s * kStageBytes + c * kBChunkBytes, &tmB, full,
                           n0 + static_cast<int32_t>(c * kBChunkCols), kx, pol_b, kBPolicy);
          pending |= 1u << s;
          pending_par = (pending_par & ~(1u << s)) | (par << s);
        }
        if (p.dynamic) {
          if (clc_next_unit(sched, static_cast<uint32_t>(w), sched_resp0, sched_full0, sched_empty0,
                            abort_flag, limit, kRoleProducer, false, true) == kClcAbort)
            ok = false;
        } else {
          sched.next_tile();
        }
      }
      if (!ok) {
        for (uint32_t s = 0; s < kStages; ++s)
          if ((pending >> s) & 1u)
            wait_bounded(bar_loaded + 8u * s, (pending_par >> s) & 1u, limit, kRoleDrain);
      }
    }
    __syncwarp();   // reconverge before the CTA-wide barrier below
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_full = idesc_f16(DT, kBM, kBN, /*A K-major*/ 0, /*B N-major*/ 1);
      constexpr uint32_t idesc_half = idesc_f16(DT, kBM, kBN / 2, 0, 1);
      PersistentTileScheduler sched(p.m_blocks, p.n_blocks, p.group, gridDim.x, p.split_from,
                                    p.total_units, p.column_major);
      sched.init(blockIdx.x);
      bool ok = true;
      while (ok && sched.valid()) {
        const uint32_t w = sched.current_iter;
        const uint32_t buf = w & 1u;
        if (!wait_or_abort(bar_tmem_empty + 8u * buf, ((w >> 1) & 1u) ^ 1u, abort_flag, limit,
                           kRoleMma)) {
          ok = false;
          break;
        }
        tcgen05_fence_after_sync();
        const uint32_t d_tmem = tmem_base + buf * kBN;
        const uint32_t idesc = sched.half_unit() ? idesc_half : idesc_full;
        for (uint32_t k = 0; k < p.k_blocks; ++k) {
          const uint64_t phase = static_cast<uint64_t>(w) * k_blocks + k;
          const uint32_t s = static_cast<uint32_t>(phase % kStages);
          const uint32_t par = static_cast<uint32_t>((phase / kStages) & 1u);
          if (!wait_or_abort(bar_loaded + 8u * s, par, abort_flag, limit, kRoleMma)) {
            ok = false;
            break;
          }
          tcgen05_fence_after_sync();
          const uint32_t a_addr = sA0 + s * kStageBytes;
          const uint32_t b_addr = sB0 + s * kStageBytes;
#pragma unroll
          for (uint32_t kk = 0; kk < kBK / kUmmaK; ++kk) {
            // A: K-major, one 16 KiB atom per 64 K; inside an atom advance 16 elements =
            //    32 bytes along the swizzle row; SBO = 1024 bytes between 8-row groups.
            // B: N-major, advance 16 K-rows = 2048 bytes; LBO = one 64-column chunk
            //    (block_K rows x 128 bytes) between chunks, SBO = 1024 bytes between 8-row groups.
            const uint32_t a_off = (kk / (kKAtom / kUmmaK)) * kAAtomBytes +
                                   (kk % (kKAtom / kUmmaK)) * kUmmaK * kElemBytes;
            const uint64_t a_desc = smem_desc_sw128(a_addr + a_off, 16, 1024);
            const uint64_t b_desc = smem_desc_sw128(b_addr + kk * kUmmaK * 128u, kBChunkBytes, 1024);
            umma_f16(d_tmem, a_desc, b_desc, idesc, (k | kk) != 0u ? 1u : 0u);
          }
          umma_commit(bar_consumed + 8u * s);
        }
        if (!ok) break;
        umma_commit(bar_tmem_full + 8u * buf);
        if (p.dynamic) {
          if (clc_next_unit(sched, w, sched_resp0, sched_full0, sched_empty0, abort_flag, limit,
                            kRoleMma, false, true) == kClcAbort)
            ok = false;
        } else {
          sched.next_tile();
        }
      }
      // every MMA this thread issued has finished before TMEM can be released
      umma_commit(bar_drain);
      wait_bounded(bar_drain, 0, limit, kRoleDrain);
    }
    __syncwarp();
  } else if (warp == 3) {
    // ------------------------------------------------------------ unit fetcher (dynamic mode)
    if (lane == 0 && p.dynamic) {
      for (uint32_t j = 0;; ++j) {   // fetch j: the unit of this CTA's iteration j + 1
        const uint32_t slot = j % kSchedSlots;
        const uint32_t par = (j / kSchedSlots) & 1u;
        if (!wait_or_abort(sched_empty0 + 8u * slot, par ^ 1u, abort_flag, limit, kRoleSched))
          break;
        mbar_arrive_expect_tx(sched_full0 + 8u * slot, 16);
        clc_try_cancel(sched_resp0 + 16u * slot, sched_full0 + 8u * slot);
        if (!wait_or_abort(sched_full0 + 8u * slot, par, abort_flag, limit, kRoleSched)) {
          wait_bounded(sched_full0 + 8u * slot, par, limit, kRoleDrain);  // let it land
          break;
        }
        uint32_t unit;
        if (!clc_response(sched_resp0 + 16u * slot, &unit)) break;   // nothing left to take
      }
    }
    __syncwarp();
  } else if (warp >= kFirstEpiWarp) {
    // ------------------------------------------------------------ epilogue
    const uint32_t q = warp - kFirstEpiWarp;       // TMEM lanes 32q .. 32q + 31
    PersistentTileScheduler sched(p.m_blocks, p.n_blocks, p.group, gridDim.x, p.split_from,
                                    p.total_units, p.column_major);
    sched.init(blockIdx.x);
    uint32_t chunk = 0;
    while (sched.valid()) {
      const uint32_t w = sched.current_iter;
      const uint32_t buf = w & 1u;
      const bool got = wait_or_abort(bar_tmem_full + 8u * buf, (w >> 1) & 1u, abort_flag, limit,
                                     kRoleEpilogue);
      if (!__all_sync(0xffffffffu, got)) break;
      tcgen05_fence_after_sync();
      const bool half = sched.half_unit();
      const int32_t row0 = static_cast<int32_t>(sched.m_idx) * kBM + static_cast<int32_t>(q) * 32;
      const int32_t col0 = static_cast<int32_t>(sched.n_idx) * kBN + (half ? sched.part * (kBN / 2) : 0);
      const uint32_t chunks = half ? kBN / kEpiN / 2 : kBN / kEpiN;
      const uint32_t t_row = tmem_base + ((q * 32u) << 16) + buf * kBN;
#pragma unroll 1
      for (uint32_t j = 0; j < chunks; ++j, ++chunk) {
        uint32_t v[64];
        tmem_ld_32x32b_x64(t_row + j * kEpiN, v);
        if (j == chunks - 1) {
          // accumulator fully in registers: hand it back to the MMA warp before storing
          tcgen05_fence_before_sync();
          mbar_arrive(bar_tmem_empty + 8u * buf);
        }
        const uint32_t sbuf = sEpi + (q * 2u + (chunk & 1u)) * kEpiBufBytes;
        epilogue_store_chunk<DT>(v, lane, sbuf, &tmC, p, row0,
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
      if (p.dynamic) {
        if (clc_next_unit(sched, w, sched_resp0, sched_full0, sched_empty0, abort_flag, limit,
                          kRoleEpilogue, true, lane == 0) == kClcAbort)
          break;
      } else {
        sched.next_tile();
      }
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
