// tg_config.h -- compile-time tiling of the persistent warp-specialized GEMM.
//
// The pages leave block_M / block_N / block_K / num_stages / store_block_N open (they are
// parameters of ``gemm_persistent`` in "[Feature] Introduce tile scheduler #2441",
// gemm_tcgen5mma_ws_persistent.py, ``main``).  Values chosen for sm_103a:
//   block_M = 128   the M of one cta_group::1 tcgen05.mma; TMEM lane i holds row i
//   block_N = 256   the largest N of one tcgen05.mma; two fp32 accumulators of 256 columns
//                   fill all 512 TMEM columns (the page's C_tmem_0 / C_tmem_1)
//   block_K = 64    64 x 2 bytes = 128 bytes: exactly one row of the 128-byte swizzle atom
//   num_stages = 4  4 x 48 KiB of operand ring; with 32 KiB of epilogue staging it fits in
//                   the 227 KiB a CTA may use
//   store_block_N = 64   the epilogue drains and stores 64 columns (128 bytes) at a time
//   group = 8       the page's group_size of the grouped tile order
// Warp roles (256 threads, as the page's ``threads=256``): warp 0 issues TMA loads, warp 1
// issues tcgen05.mma, warp 2 owns the TMEM allocation, warps 4..7 are the epilogue (warp
// 4 + q may only touch TMEM lanes 32q..32q+31).
#pragma once

#include <cstdint>

namespace tg {

constexpr int kBM = 128;
#ifndef TG_BN
#define TG_BN 256
#endif
constexpr int kBN = TG_BN;
#ifndef TG_BK
#define TG_BK 64
#endif
constexpr int kBK = TG_BK;               // a multiple of 64: kKAtoms 128-byte swizzle atoms
constexpr int kKAtom = 64;               // K elements of one 128-byte swizzle row
constexpr int kKAtoms = kBK / kKAtom;
// Ring depths can be overridden at compile time (-DTG_STAGES=, -DTG_PAIR_STAGES=) to tune.
#ifndef TG_STAGES
#define TG_STAGES 4
#endif
#ifndef TG_PAIR_STAGES
#define TG_PAIR_STAGES 3
#endif
#ifndef TG_PAIR_BK
#define TG_PAIR_BK 128
#endif
// L2 policy of the A and B loads (0 none, 1 evict_first, 2 evict_last, 3 evict_normal)
#ifndef TG_A_POLICY
#define TG_A_POLICY 0
#endif
#ifndef TG_B_POLICY
#define TG_B_POLICY 0
#endif
// L2 policy of the epilogue's TMA stores of C (0 none, 1 evict_first): C is written once and
// never read back by the kernel.  Measured on GB300 (same box, 3 alternating rounds, TFLOP/s,
// none / evict_first): 4096^3 1775 / 1782, 4000 x 7000 x 2048 1658 / 1668, 8192^3 and 6144^3
// unchanged; DRAM bytes at 8192^3 unchanged.
#ifndef TG_C_POLICY
#define TG_C_POLICY 1
#endif
constexpr int kStages = TG_STAGES;
constexpr int kAPolicy = TG_A_POLICY;
constexpr int kBPolicy = TG_B_POLICY;
constexpr int kCPolicy = TG_C_POLICY;
constexpr int kEpiN = 64;
#ifndef TG_GROUP
#define TG_GROUP 8
#endif
constexpr int kGroup = TG_GROUP;         // the page's group_size
constexpr int kThreads = 256;
constexpr int kUmmaK = 16;                 // K of one tcgen05.mma kind::f16
constexpr int kEpiWarps = 4;
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kFirstEpiWarp = 4;

constexpr uint32_t kElemBytes = 2;
constexpr uint32_t kAAtomBytes = kBM * kKAtom * kElemBytes;      // 16 KiB: one K atom of A
constexpr uint32_t kABytes = kBM * kBK * kElemBytes;             // 16 KiB at block_K 64
constexpr uint32_t kBBytes = kBK * kBN * kElemBytes;             // 32 KiB
constexpr uint32_t kStageBytes = kABytes + kBBytes;              // 48 KiB: expect_tx per stage
constexpr uint32_t kBChunkCols = 64;                             // one 128-byte swizzle row of B
constexpr uint32_t kBChunkBytes = kBK * kBChunkCols * kElemBytes;  // 8 KiB
constexpr uint32_t kEpiBufBytes = 32 * kEpiN * kElemBytes;       // 4 KiB: 32 rows x 128 bytes
constexpr uint32_t kSmemAlignSlack = 1024;
constexpr uint32_t kEpiSmemBytes = kEpiWarps * 2 * kEpiBufBytes;
constexpr uint32_t kSmemBytes = kSmemAlignSlack + kStages * kStageBytes + kEpiSmemBytes;
constexpr uint32_t kTmemCols = 512;

static_assert(kKAtom * kElemBytes == 128, "a K atom spans one 128-byte swizzle row");
static_assert(kBK % kKAtom == 0 && kBK <= 256, "block_K: a multiple of 64, at most 256");
static_assert(kEpiN * kElemBytes == 128, "store_block_N must span one 128-byte swizzle row");
static_assert(kBN % kBChunkCols == 0 && kBN % kEpiN == 0, "block_N tiling");
static_assert(kBM == 128 && kBN % 16 == 0 && kBN <= 256, "tcgen05.mma cta_group::1 shape");
static_assert(2 * kBN <= (int)kTmemCols, "two accumulators must fit in TMEM");
static_assert(kSmemBytes + 256 <= 232448, "shared memory per CTA");

// CTA-pair variant (tcgen05 cta_group::2, the page's gemm_persistent_2cta): a cluster of two
// CTAs computes a 256 x 256 output tile.  CTA r of the pair loads A rows [128r, 128r + 128)
// and B columns [128r, 128r + 128) of the tile; one 256 x 256 x 16 MMA issued by the even CTA
// reads both halves, and each CTA's TMEM holds its 128 rows x 256 columns.  The pair takes
// block_K = 128 per stage (64 KiB per CTA, three stages): measured on GB300, the fixed cost
// of each stage hand-over (barrier waits, commit, refill) weighs less with eight MMAs per
// stage than with four, more than the shallower ring costs (8192^3: +9 %, 4096^3: +15 %
// over block_K 64 with six stages).
constexpr int kPairBM = 2 * kBM;                                  // 256 rows per pair tile
constexpr int kPairBNHalf = kBN / 2;                              // B columns one CTA loads
constexpr int kPairStages = TG_PAIR_STAGES;
constexpr int kPairBK = TG_PAIR_BK;
constexpr int kPairKAtoms = kPairBK / kKAtom;
constexpr uint32_t kPairABytes = kBM * kPairBK * kElemBytes;          // 32 KiB
constexpr uint32_t kPairBChunkBytes = kPairBK * kBChunkCols * kElemBytes;  // 16 KiB
constexpr uint32_t kPairBBytes = kPairBK * kPairBNHalf * kElemBytes;  // 32 KiB
constexpr uint32_t kPairStageBytes = kPairABytes + kPairBBytes;       // 64 KiB per CTA
constexpr uint32_t kPairTxBytes = 2 * kPairStageBytes;            // both CTAs' bytes, one barrier
constexpr uint32_t kPairSmemBytes = kSmemAlignSlack + kPairStages * kPairStageBytes + kEpiSmemBytes;
static_assert(kPairSmemBytes + 256 <= 232448, "shared memory per CTA (pair variant)");
static_assert(kPairBNHalf % kBChunkCols == 0, "pair B half must be whole 64-column chunks");
static_assert(kPairBK % kKAtom == 0 && kPairBK <= 256, "pair block_K: a multiple of 64, <= 256");
static_assert(kPairStages * kPairStageBytes / kEpiWarps >= (kBN / kEpiN) * 8192,
              "a stream-K owner stages one contribution per epilogue warp in the operand ring");

// Block-scaled MXFP8 kernel (the PR's gemm_mxfp8_blockscaled_1d1d): E4M3 A [M, K] and B [N, K],
// both K-major, one E8M0 scale per 32 K-elements of each A row and each B column, fp32
// accumulation, bf16/fp16 out; one CTA per 128 x 256 output tile on the same scheduler.
//   block_K = 128 one-byte elements: one 128-byte swizzle row, four MMAs of K = 32, and the
//   4 scales of each row that one 32-bit TMEM word holds.
//   Scales reach the kernel packed (tg_mxfp8_pack_scales): for each 128-element k-block and
//   each block of 128 rows, one 512-byte atom with row r's 4 scales at byte (r % 32) * 16 +
//   (r / 32) * 4 -- the source layout of tcgen05.cp .32x128b.warpx4, which replicates an atom
//   into all four 32-lane TMEM quadrants (measured on GB300: the MMA reads the scale of A row r
//   at lane r, column r / 32, and that of B column n at column n / 32 in the quadrant of the
//   output row it serves).  The producer bulk-copies a stage's atoms (512 bytes of A, 1 KiB
//   of B) with its operands, on the same barrier.  (Reordering row-major scales inside the
//   kernel -- a per-lane gather, or a transpose warp -- put the scale loads' latency on the
//   MMA's path: 41 % of the fp8 rate, measured.)
//   TMEM: one 256-column accumulator plus 16 scale columns per stage (SFA 4, SFB 8): two
//   accumulators would take all 512 columns.  The epilogue copies the whole accumulator to
//   registers before releasing it, so the MMA role waits only for that copy.
#ifndef TG_MX_STAGES
#define TG_MX_STAGES 4
#endif
constexpr int kMxStages = TG_MX_STAGES;
constexpr int kMxBK = 128;                                     // K elements (bytes) per stage
constexpr int kMxBlock = 32;                                   // elements per scale
constexpr int kMxUmmaK = 32;                                   // K of one kind::mxf8f6f4 MMA
constexpr uint32_t kMxABytes = kBM * kMxBK;                    // 16 KiB
constexpr uint32_t kMxBHalfBytes = (kBN / 2) * kMxBK;          // 16 KiB: 128 columns of B
constexpr uint32_t kMxBBytes = kBN * kMxBK;                    // 32 KiB
constexpr uint32_t kMxStageBytes = kMxABytes + kMxBBytes;      // 48 KiB
constexpr uint32_t kMxSfAtomBytes = 512;                       // 128 rows x 4 scales
constexpr uint32_t kMxAtomSetBytes = 3 * kMxSfAtomBytes;       // SFA atom + two SFB atoms
constexpr uint32_t kMxAtomRegionBytes = (kMxStages * kMxAtomSetBytes + 1023u) & ~1023u;
constexpr uint32_t kMxEpiSmemBytes = kEpiWarps * kEpiBufBytes; // one staging buffer per warp
constexpr uint32_t kMxSmemBytes =
    kSmemAlignSlack + kMxStages * kMxStageBytes + kMxAtomRegionBytes + kMxEpiSmemBytes;
constexpr uint32_t kMxAccCols = kBN;                           // TMEM columns [0, 256)
constexpr uint32_t kMxSfColsPerStage = 16;
constexpr uint32_t kMxPackRows = 2 * kBM;                      // packed rows pad to 256
static_assert(kMxSmemBytes + 512 <= 232448, "shared memory per CTA (MXFP8)");
static_assert(kMxAccCols + kMxStages * kMxSfColsPerStage <= kTmemCols, "MXFP8 TMEM budget");
static_assert(kMxBK == 4 * kMxBlock, "one 4-byte scale word per row and k-block");

// CTA-pair MXFP8 kernel (tcgen05 cta_group::2; the page's example is 2-CTA): a cluster of two
// CTAs computes a 256 x 256 output tile.  CTA r loads A rows [128r, 128r + 128) and B rows
// (N) [128r, 128r + 128) of the tile (for a 128-wide half unit: [64r, 64r + 128), of which the
// MMA reads 64), its own SFA atom and both SFB atoms, by TMA completing on the even CTA's
// barrier; the even CTA copies the atoms into both CTAs' TMEM (tcgen05.cp .cta_group::2 copies
// each CTA's shared memory into its own TMEM, measured) and issues 256 x 256 x 32 MMAs.  Half
// of B per CTA makes a k-block 32 KiB; stages of two k-blocks (eight MMAs per hand-over, three
// stages) ran faster than six stages of one.
// A stage holds TG_MX_PAIR_KB k-blocks of 128 (each: 16 KiB of A, 16 KiB of B, 1.5 KiB of
// atoms per CTA); a K tail leaves the last stage partly zero-filled by TMA.
#ifndef TG_MX_PAIR_KB
#define TG_MX_PAIR_KB 2
#endif
#ifndef TG_MX_PAIR_STAGES
#define TG_MX_PAIR_STAGES (6 / TG_MX_PAIR_KB)
#endif
constexpr int kMxPairKB = TG_MX_PAIR_KB;
constexpr int kMxPairStages = TG_MX_PAIR_STAGES;
constexpr uint32_t kMxPairBBytes = (kBN / 2) * kMxBK;              // 16 KiB: 128 rows of B
constexpr uint32_t kMxPairKbBytes = kMxABytes + kMxPairBBytes;     // 32 KiB per k-block
constexpr uint32_t kMxPairStageBytes = kMxPairKB * kMxPairKbBytes;  // A blocks, then B blocks
constexpr uint32_t kMxPairTxBytes = 2 * kMxPairKB * kMxPairKbBytes;   // A, B of both CTAs
constexpr uint32_t kMxPairSfTxBytes = kMxPairKB * kMxAtomSetBytes;     // one CTA's atoms
// The scale atoms run TG_MX_PAIR_SF_AHEAD stages ahead of the operands through a ring of their
// own (shared-memory atom sets and TMEM scale slots): stage p's atoms are loaded together with
// the operands of stage p - ahead, so the epilogue warps that write them into TMEM have
// ahead + S - 1 stages of MMA time to do it.  Measured on GB300 (MXFP8 GEMM TFLOP/s, two
// alternating rounds; 8192^3 / 6144^3 / 4096^3): ahead 1: 3423 / 3294 / 2897, ahead 2: 3408 /
// 3281 / 2870; one k-block per stage (6 stages), ahead 2: 2937 / 2805 / 2346, ahead 4: 2820.
#ifndef TG_MX_PAIR_SF_AHEAD
#define TG_MX_PAIR_SF_AHEAD 1
#endif
constexpr int kMxPairSfAhead = TG_MX_PAIR_SF_AHEAD;
constexpr int kMxPairSfSlots = kMxPairStages + kMxPairSfAhead;      // stages in the scale ring
constexpr uint32_t kMxPairAtomRegionBytes =
    (kMxPairSfSlots * kMxPairKB * kMxAtomSetBytes + 1023u) & ~1023u;
constexpr uint32_t kMxPairSmemBytes = kSmemAlignSlack + kMxPairStages * kMxPairStageBytes +
                                      kMxPairAtomRegionBytes + kMxEpiSmemBytes;
static_assert(kMxPairSmemBytes + 512 <= 232448, "shared memory per CTA (MXFP8 pair)");
static_assert(kMxAccCols + kMxPairSfSlots * kMxPairKB * kMxSfColsPerStage <= kTmemCols,
              "MXFP8 pair TMEM budget");
static_assert(kMxPairSfSlots <= 32, "atom slots tracked in one 32-bit mask");

// watchdog: bits of the per-device status word naming the role that gave up a wait
constexpr uint32_t kRoleProducer = 1u;
constexpr uint32_t kRoleMma = 2u;
constexpr uint32_t kRoleEpilogue = 4u;
constexpr uint32_t kRoleDrain = 8u;
constexpr uint32_t kRoleSched = 16u;
// dynamic persistence: try_cancel responses kept in flight, and the threads that read each
// (producer thread, MMA thread, one lane per epilogue warp)
constexpr int kSchedSlots = 2;
constexpr uint32_t kSchedConsumers = 2 + kEpiWarps;
constexpr uint64_t kDefaultWatchdogNs = 1ull << 32;  // about 4.3 s

}  // namespace tg
