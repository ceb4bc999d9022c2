// tg_wide_config.h -- compile-time constants of the wide CTA-pair GEMM (tg_gemm_pair_wide_kernel.cuh),
// shared by that kernel and the host code that sizes its launch and tensor maps.
#pragma once

#include "tg_config.h"

namespace tg {

// Wide CTA-pair variant: 256 x 512 output tiles as two N-halves of 256 (two MMAs of
// 256 x 256 x 16 per k-step into the two halves of TMEM, one accumulator).  Per CTA and
// k-block of 64: A 128 x 64 (16 KiB) and its 128 columns of each N-half (4 chunks of 8 KiB),
// 48 KiB per stage, 4 stages: each stage holds the MMA work of a 128-deep stage of the
// 256 x 256 pair, and A is loaded once for 512 columns.
constexpr int kWideBN = 2 * kBN;                                   // 512 columns per unit
constexpr int kWideBK = 64;
constexpr int kWideStages = 4;
constexpr uint32_t kWideABytes = kBM * kWideBK * kElemBytes;                 // 16 KiB
constexpr uint32_t kWideBChunkBytes = kWideBK * kBChunkCols * kElemBytes;    // 8 KiB
constexpr uint32_t kWideStageBytes = kWideABytes + 4 * kWideBChunkBytes;    // 48 KiB per CTA
constexpr uint32_t kWideSmemBytes = kSmemAlignSlack + kWideStages * kWideStageBytes + kEpiSmemBytes;
// At the start of a unit the MMA may run N-half 0 of the first kWideDefer k-blocks before the
// epilogue has handed N-half 1 of the previous unit back (those ring slots are released once
// half 1 has read them too).  One k-block measured best on GB300 (8192^3: 2004-2007 TFLOP/s
// against 1995-1997 with none; two or three gained nothing more, since held slots delay refills).
#ifndef TG_WIDE_DEFER
#define TG_WIDE_DEFER 1
#endif
constexpr uint32_t kWideDefer = TG_WIDE_DEFER;
static_assert(kWideDefer < kWideStages, "deferred k-blocks hold ring slots");
static_assert(kWideSmemBytes + 256 <= 232448, "shared memory per CTA (wide pair variant)");
static_assert(kWideStages * kWideStageBytes / kEpiWarps >= (kBN / kEpiN) * 8192,
              "a stream-K owner stages one N-half of a contribution per warp in the ring");
static_assert(kWideBK == kKAtom, "a wide stage holds one 128-byte swizzle atom of A");
static_assert(2 * kBN <= (int)kTmemCols, "the wide accumulator spans both TMEM halves");

}  // namespace tg
