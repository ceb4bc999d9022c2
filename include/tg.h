/*
 * tg.h -- C ABI of the persistent, warp-specialized GEMM for GB300 (sm_103a).
 *
 *   C[M, N] = A[M, K] . B[K, N]      fp16 or bf16 in, fp32 accumulation, same type out
 *
 * The operation is the one ``gemm_persistent`` computes in "[Feature] Introduce tile
 * scheduler #2441" (examples/gemm_sm100/gemm_tcgen5mma_ws_persistent.py): row-major
 * A [M, K] and B [K, N] (``T.tcgen05_gemm(A_shared, B_shared, ...)`` with neither operand
 * transposed), fp32 accumulation in tensor memory, and a cast of the accumulator to the
 * output type in the epilogue.  The call convention -- plain pointers, an int status,
 * a readable last-error string -- follows the host wrapper that TileLang generates
 * ("tilelang", Generated Kernel Source: ``init()``, ``call(A, B, C, stream)`` returning
 * 0 or -1, ``get_last_error()``), and the argument checks follow the host checks of its
 * lowered host module ("tilelang", 1.2 Pass Pipeline, Host IRModule: null data pointers,
 * rank-2 row-major with unit inner stride and no byte offset, "vectorize dimension
 * divisible by 8").
 *
 * Conventions for every entry point:
 *   - Pointers named *_dev are device pointers of the current CUDA device, allocated by the
 *     caller (cudaMalloc or any allocator built on it); the library never frees them and
 *     keeps no pointer after the call returns.  Matrices are dense row-major with no
 *     padding: the row stride of A is K elements, of B and C it is N elements.
 *   - ``stream`` is a cudaStream_t (NULL = the legacy default stream).  GEMM entry points
 *     are asynchronous: TG_OK means the work was enqueued; faults during execution surface
 *     at the caller's next synchronisation, as with any CUDA launch.  The GEMM and scale-pack
 *     kernels are launched with programmatic dependent launch: their CTAs may start while the
 *     previous kernel in the stream is finishing, but wait for it to complete before their
 *     first access to global memory, so the stream's order of memory effects is kept.
 *   - A negative return is an error; tg_last_error() then holds a message (thread-local;
 *     valid until the next call on the same thread).  On error nothing was enqueued.
 */
#ifndef TG_H
#define TG_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* element types: input, output and (internally) fp32 accumulation */
enum { TG_F16 = 0, TG_BF16 = 1 };

/* kernel variants (tg_gemm_persistent_ex, tg_gemm_persistent_debug, tg_gemm_launch_shape) */
enum {
  TG_VARIANT_AUTO = 0,    /* the library's choice for the problem (what tg_gemm_persistent runs) */
  TG_VARIANT_SINGLE = 1,  /* one CTA per 128 x 256 output tile, tcgen05 cta_group::1 */
  TG_VARIANT_PAIR = 2,    /* a CTA pair per 256 x 256 output tile, tcgen05 cta_group::2
                             ("[Feature] Introduce tile scheduler #2441", gemm_persistent_2cta) */
  TG_VARIANT_PAIR_WIDE = 3, /* dense GEMM only: a CTA pair per 256 x 512 output tile, as two
                               N-halves of 256 into the two halves of TMEM (one accumulator),
                               block_K 64 x 4 stages; A is loaded once per 512 columns */
  /* OR'ed into a variant: walk tiles exactly as the page's scheduler does.  By default, when
     the last partial wave of tiles would keep at most half of the workers busy, each of its
     tiles is cut into two half-width (N) units so that wave takes half a tile's time; see
     tg_tile_schedule_ex. */
  TG_SCHEDULE_PLAIN = 0x100,
  /* OR'ed into a variant (or into tg_tile_schedule_ex's flags): the scheduler's column_major
     order -- panels of ``group`` M-tiles with ids running along M first, the grouped decode
     with the roles of M and N exchanged.  Default: panels of N-tiles, N first, as the page. */
  TG_SCHEDULE_COLUMN_MAJOR = 0x200,
  /* OR'ed into TG_VARIANT_SINGLE: dynamic persistence.  One CTA is launched per work unit; the
     ~#SMs that run first keep going and take over the units of CTAs not yet launched by
     cancelling those launches (cluster launch control, clusterlaunchcontrol.try_cancel), so
     units go to whichever SM frees up first.  The unit-to-CTA assignment is then decided at run
     time (the debug trace records it); the set of units and their decode are unchanged. */
  TG_SCHEDULE_DYNAMIC = 0x400,
  /* OR'ed into a variant of the dense GEMM: the epilogue stores each thread's row of the tile
     with 16-byte stores straight from registers (the page's direct C_local_cast store) instead
     of staging it in shared memory for a TMA store (the page's use_tma_store, the default). */
  TG_EPILOGUE_DIRECT = 0x800,
  /* tg_gemm_launch_shape flag: describe the block-scaled MXFP8 GEMM's launch (tg_gemm_mxfp8*),
     whose variants are SINGLE and PAIR, instead of the dense GEMM's. */
  TG_SHAPE_MXFP8 = 0x1000,
  /* OR'ed into a PAIR, PAIR_WIDE or AUTO variant of tg_gemm_persistent_ws or
     tg_gemm_persistent_debug (with a workspace): split the last partial wave of tiles along K
     (the stream-K tail described at tg_gemm_persistent_ws) whenever there is one. */
  TG_SCHEDULE_STREAMK = 0x2000,
  /* tg_gemm_launch_shape flag: describe the launch of tg_gemm_persistent_ws (with a workspace). */
  TG_SHAPE_WORKSPACE = 0x4000,
  /* tg_tile_schedule_ex flag: apply the tail split (the GEMM does unless TG_SCHEDULE_PLAIN) */
  TG_SCHEDULE_SPLIT_TAIL = 0x1
};

/* OR'ed into a variant: the group width of the grouped tile order (the scheduler's
   swizzle_size), 1..255; 0 (not given) = 8, the page's group_size. */
#define TG_SCHEDULE_GROUP(g) (((int)(g) & 0xFF) << 16)

/* status codes */
enum {
  TG_OK = 0,
  TG_ERR_ARG = -1,     /* null/non-device pointer, negative size, unknown dtype, C overlapping A or B */
  TG_ERR_ALIGN = -2,   /* pointer not 16-byte aligned, or N or K not a multiple of 8 (TMA row strides
                          must be multiples of 16 bytes) */
  TG_ERR_CUDA = -3,    /* a CUDA runtime/driver call failed, or the device is not sm_103 */
  TG_ERR_TIMEOUT = -4  /* a bounded wait inside the kernel gave up (watchdog); see tg_device_status */
};

/*
 * tg_gemm_persistent -- C = A . B on ``stream``.
 *   A_dev [M, K], B_dev [K, N], C_dev [M, N]; all of type ``dtype`` (TG_F16 or TG_BF16).
 *   M, N, K >= 0 and < 2^31.  N % 8 == 0 and K % 8 == 0.  All three pointers 16-byte aligned.
 *   C must not overlap A or B.  M == 0 or N == 0: nothing is done.  K == 0: C is zero-filled.
 * Persistent kernels walk the output tiles in grouped order (see tg_tile_schedule): one CTA
 * per SM on 128 x 256 tiles, or one CTA pair per two SMs on 256 x 256 or 256 x 512 tiles, with
 * the kernel and the traversal chosen as TG_VARIANT_AUTO describes at tg_gemm_persistent_ex.  Partial edge tiles in
 * M and N and a partial last k-block are handled inside the kernel (zero-filled loads,
 * clipped stores).
 */
int tg_gemm_persistent(const void* A_dev, const void* B_dev, void* C_dev,
                       int64_t M, int64_t N, int64_t K, int dtype, void* stream);

/*
 * tg_gemm_persistent_ex -- tg_gemm_persistent with an explicit kernel variant (TG_VARIANT_*).
 * Same arguments, rules and results; TG_ERR_ARG for an unknown variant.  The pair variant
 * walks ceil(M/256) x ceil(N/256) tiles with one scheduler worker per CTA pair, the wide pair
 * variant ceil(M/256) x ceil(N/512) tiles (its tail-split half units are 256 x 256).
 * TG_VARIANT_AUTO takes the wide pair variant when its tiles fill at least one wave of resident
 * pairs and K >= 6144, or four waves and K >= 4096; else the pair variant when its tiles fill at
 * least one wave, or when K >= 4096 and M >= 256; else the single one.  Unless the variant carries TG_SCHEDULE_PLAIN,
 * TG_SCHEDULE_COLUMN_MAJOR or TG_SCHEDULE_GROUP, AUTO also picks the traversal: whole rows of
 * tiles when all of B fits in 64 MiB (half of the L2), whole columns when only A does, else
 * groups of 8 in row order, or for the wide pair variant groups of round(sqrt(2 x workers))
 * M-tiles in column order (tg_gemm_launch_shape reports the choice).
 */
int tg_gemm_persistent_ex(const void* A_dev, const void* B_dev, void* C_dev,
                          int64_t M, int64_t N, int64_t K, int dtype, void* stream, int variant);

/*
 * tg_gemm_persistent_ws -- tg_gemm_persistent_ex with a workspace.  With TG_SCHEDULE_STREAMK
 * in ``variant`` the CTA-pair variants split the last partial wave of tiles along K (a stream-K
 * tail) instead of cutting its tiles into half-width units.  With T tiles over P CTA pairs, the
 * R = T mod P tiles that come last in the traversal have their k-blocks, numbered tile-major,
 * cut into P contiguous ranges, one per pair.  The pair holding a tail tile's last k-block owns
 * the tile: the other pairs that meet it write their fp32 partial sums to the workspace, and the
 * owner adds them to its own before converting and storing the tile.  Each pair works its
 * contribution before the tile it owns, so an owner waits only on lower-numbered pairs.  The
 * library never takes this tail unasked (AUTO included): measured on GB300 it was slower than
 * the half-width units at every size tried, the partial sums' round trip costing about what the
 * idle part of the last wave does.  Without TG_SCHEDULE_STREAMK the workspace is unused.
 * Results are those of tg_gemm_persistent_ex up to the order of fp32 additions (bit-identical
 * where the sums are exact).
 *   workspace_dev: NULL, or a device buffer of workspace_bytes, 256-byte aligned, of at least
 *     tg_gemm_workspace_bytes(M, N, K, variant) bytes; its contents need no initialisation and
 *     are scratch.  It must not be used by another call that may run at the same time (another
 *     stream).  TG_SCHEDULE_STREAMK with NULL or a smaller buffer: TG_ERR_ARG.
 *     TG_SCHEDULE_PLAIN and the single-CTA variant never take the stream-K tail.
 * Every wait on another pair is bounded by the watchdog (TG_ERR_TIMEOUT through
 * tg_device_status).  Same argument rules and errors as tg_gemm_persistent_ex otherwise.
 */
int tg_gemm_persistent_ws(const void* A_dev, const void* B_dev, void* C_dev, int64_t M,
                          int64_t N, int64_t K, int dtype, void* stream, int variant,
                          void* workspace_dev, int64_t workspace_bytes);

/*
 * tg_gemm_workspace_bytes -- the workspace tg_gemm_persistent_ws needs for this problem and
 * variant (TG_SCHEDULE_STREAMK included) on the current device: 0 when it takes no stream-K tail;
 * otherwise (pairs x 8) flags of 4 bytes padded to 256, then one fp32 slice of 128 x tile_n per
 * pair and CTA.
 * Returns the byte count or a negative error code.
 */
int64_t tg_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, int variant);

/*
 * tg_tile_schedule -- the tile order the GEMM kernel follows, for inspection.
 * The persistent scheduler of "[Feature] Introduce tile scheduler #2441"
 * (``PersistentTileScheduler(..., swizzle_size=group_size)``, ``init(block_id)``,
 * ``valid()``, ``next_tile()``) runs on the device, one thread per worker, with the same
 * scheduler code the GEMM kernel's three roles use.
 *   m_blocks, n_blocks >= 1 with m_blocks * n_blocks < 2^31; num_sms >= 1 (workers); group >= 1.
 *   out_host: HOST buffer of 4 * m_blocks * n_blocks int32, filled with rows
 *   (worker, w, bx, by) ordered by worker, then by the worker's iteration clock w;
 *   bx is the M-tile, by the N-tile.
 * Synchronous (uses and synchronises the legacy default stream; allocates and frees a
 * temporary device buffer).  Returns the row count (= m_blocks * n_blocks) or an error.
 */
int tg_tile_schedule(int m_blocks, int n_blocks, int num_sms, int group, int32_t* out_host);

/*
 * tg_tile_schedule_ex -- the unit order of the GEMM kernel, with or without the tail split.
 *   flags: TG_SCHEDULE_SPLIT_TAIL and/or TG_SCHEDULE_COLUMN_MAJOR (others: TG_ERR_ARG).
 *   Without TG_SCHEDULE_SPLIT_TAIL: the rows of tg_tile_schedule, each with part = -1.
 *   With it: with T = m_blocks * n_blocks tiles and R = T mod num_sms, if
 *     0 < 2R <= num_sms the last R tiles of the grouped order become 2R half-width units:
 *     unit ids 0 .. T-R-1 are whole tiles (part -1), unit T-R+2i+h is half h (0 = left,
 *     1 = right, in N) of tile T-R+i; workers step through unit ids with the grid stride.
 *   out_host: HOST buffer of 5 int32 per unit (there are at most 2 * m_blocks * n_blocks units),
 *     rows (worker, w, bx, by, part) ordered by worker, then w.
 * Synchronous.  Returns the number of units (rows) or an error.
 */
int tg_tile_schedule_ex(int m_blocks, int n_blocks, int num_sms, int group, int flags,
                        int32_t* out_host);

/*
 * tg_tile_schedule_noalloc -- tg_tile_schedule_ex without any device allocation.  The pages
 * have no counterpart of this call; it is an addition of this library.
 *   tg_tile_schedule and tg_tile_schedule_ex stage their rows in a device buffer that they
 *   allocate and free inside the call.  Not every caller can let a library do that: a process
 *   whose device memory is all handed out by its own pool allocator (a fresh cudaMalloc can fail
 *   there, or take memory the pool counts on), or a host thread that must not stall, since
 *   cudaFree waits for all work on the device.  This call stages the rows in a fixed array that
 *   is part of the library's device image instead, TG_SCHEDULE_NOALLOC_MAX_UNITS rows of 5
 *   int32 (1.25 MiB), which every GPU that loads the library holds until the process exits;
 *   it calls no allocation routine.
 *   Arguments, flags, rows and return value: as tg_tile_schedule_ex.  A call with more than
 *   TG_SCHEDULE_NOALLOC_MAX_UNITS units returns TG_ERR_ARG before it touches the device.
 *   Every call looks up the array's address in the current device's context (the first call
 *   on a device also loads the library's device image there): make that first call before
 *   any stream capture.  All calls on a device share the one array,
 *   so calls that overlapped on the GPU would race; each call therefore holds a process-wide
 *   lock from its launch until its rows are on the host, and returns only then (legacy default
 *   stream).  Nothing needs clearing between calls: every row copied back is written by the
 *   call that copies it.
 */
#define TG_SCHEDULE_NOALLOC_MAX_UNITS 65536
int tg_tile_schedule_noalloc(int m_blocks, int n_blocks, int num_sms, int group, int flags,
                             int32_t* out_host);

/* Message of the last failed call on this thread ("" if none). */
const char* tg_last_error(void);

/*
 * tg_gemm_config -- the compile-time tiling, for callers that size schedules or buffers.
 * Any pointer may be NULL.  Returns TG_OK.
 */
int tg_gemm_config(int* block_m, int* block_n, int* block_k, int* stages, int* group);

/*
 * tg_gemm_launch_shape -- the persistent launch the library would use for an M x N x K
 * dense GEMM on the current device with ``variant`` (TG_VARIANT_* with any TG_SCHEDULE_* flags;
 * AUTO is resolved as tg_gemm_persistent resolves it), or, with TG_SHAPE_MXFP8, for the
 * block-scaled MXFP8 GEMM (AUTO resolved as tg_gemm_mxfp8 resolves it; no traversal choice).
 *   *variant_out: the concrete variant; *tile_m, *tile_n: the output tile of one scheduler
 *   worker (256 x 512 for PAIR_WIDE); *m_tiles, *n_tiles: the tile grid; *workers: scheduler
 *   workers (CTAs for SINGLE, CTA pairs for PAIR and PAIR_WIDE); *ctas: CTAs launched;
 *   *split_from, *units: the tail split (units below split_from are whole tiles;
 *   split_from == units: no split); *group, *column_major: the traversal (the grouped order's
 *   width and whether it runs along M first).  With TG_VARIANT_AUTO and no TG_SCHEDULE_PLAIN,
 *   TG_SCHEDULE_COLUMN_MAJOR or TG_SCHEDULE_GROUP flag, the library also picks the traversal,
 *   as tg_gemm_persistent_ex describes.  With TG_SHAPE_WORKSPACE: the launch of
 *   tg_gemm_persistent_ws; *sk_tiles: the stream-K tail's tiles (0: none), which then follow the
 *   split_from whole tiles, and unit ids run to *units = split_from + 2 x workers (pair c's
 *   contribution is unit split_from + 2c, its owned tile split_from + 2c + 1);
 *   *workspace_bytes: the workspace that launch needs.  Any pointer may be NULL.
 * Queries the device once (first call); launches nothing.  Returns TG_OK or an error.
 */
int tg_gemm_launch_shape(int64_t M, int64_t N, int64_t K, int variant, int* variant_out,
                         int* tile_m, int* tile_n, int* m_tiles, int* n_tiles, int* workers,
                         int* ctas, int* split_from, int* units, int* group, int* column_major,
                         int* sk_tiles, int64_t* workspace_bytes);

/*
 * tg_gemm_persistent_debug -- the same GEMM, synchronously, with two inspection aids.
 *   variant: TG_VARIANT_* as in tg_gemm_persistent_ex.
 *   trace_dev: NULL or a device buffer of 5 int32 per work unit (tg_gemm_launch_shape's
 *     *units); row u (the unit id) receives (worker, w, bx, by, part) as the epilogue that
 *     stored unit u saw them (worker = CTA, or CTA pair) -- evidence that the kernel followed
 *     the schedule of tg_tile_schedule_ex.
 *   watchdog_ns: limit for every wait inside the kernel (0 = the default, which every other
 *     entry point uses: 2^32 ns, about 4.3 s, plus 2 us per k-block of K, so that a wait that
 *     spans one tile's whole K is not cut short).
 *   inject_skip_phase: -1 for none; otherwise cta * 2^32 + phase: the producer of CTA ``cta``
 *     (0 when inject_skip_phase < 2^32) never arms or fills that pipeline phase, so the MMA
 *     role's wait on it cannot complete: the watchdog must fire, every role must stop, and the
 *     call must return TG_ERR_TIMEOUT with the context intact.  In the CTA-pair kernels CTA 0 is
 *     the even CTA of pair 0 (the other CTA of the pair still fills the phase) and CTA 1 the odd
 *     one (the even CTA has armed the phase for both).
 *   workspace_dev, workspace_bytes: as in tg_gemm_persistent_ws (NULL, 0: none); a stream-K
 *     tail segment's trace row has part 2 (a contribution) or 3 (an owned tile).
 * Synchronises ``stream``.  Returns TG_OK, TG_ERR_TIMEOUT or another error.
 */
int tg_gemm_persistent_debug(const void* A_dev, const void* B_dev, void* C_dev,
                             int64_t M, int64_t N, int64_t K, int dtype, void* stream, int variant,
                             int32_t* trace_dev, uint64_t watchdog_ns, int64_t inject_skip_phase,
                             void* workspace_dev, int64_t workspace_bytes);

/*
 * tg_device_status -- synchronises ``stream``, then reads and clears the current device's
 * watchdog word.  TG_OK if no kernel launched by this library on the device gave up a wait
 * since the last call; TG_ERR_TIMEOUT otherwise (its output must not be trusted).
 */
int tg_device_status(void* stream);

/*
 * tg_gemm_persistent_host -- end-to-end form for data that lives in host memory.
 *   A_host [M, K], B_host [K, N] are copied to the caller's device buffers A_dev, B_dev, the
 *   GEMM runs into C_dev, and C_dev is copied back to C_host, all enqueued on ``stream`` in
 *   that order.  Host buffers should be page-locked (cudaHostAlloc) for the copies to be
 *   asynchronous.  Same size, type and alignment rules as tg_gemm_persistent.
 */
int tg_gemm_persistent_host(const void* A_host, const void* B_host, void* C_host,
                            void* A_dev, void* B_dev, void* C_dev,
                            int64_t M, int64_t N, int64_t K, int dtype, void* stream);

/*
 * Block-scaled MXFP8 GEMM: the second workload of "[Feature] Introduce tile scheduler #2441"
 * (examples/blockscaled_gemm_sm100/gemm_mxfp8_blockscaled_1d1d.py), on the same persistent
 * scheduler and warp roles, in the OCP Microscaling formats ("1d1d": A scaled per row and B
 * per column, along K only, one scale per 32 elements):
 *
 *   C[i, j] = sum_k A[i, k] * 2^(SA[i, k / 32] - 127) * B[j, k] * 2^(SB[j, k / 32] - 127)
 *
 * A [M, K] and B [N, K] hold E4M3 bytes (1 sign, 4 exponent bits with bias 7, 3 fraction
 * bits), row-major: both K-contiguous, so B is passed as N rows of K.  SA [M, K / 32] and
 * SB [N, K / 32] hold E8M0 bytes (2^(e - 127)), row-major.  The GEMM reads the scales
 * packed by tg_mxfp8_pack_scales, the page's scale-factor transpose done ahead of the GEMM
 * (weights' scales can be packed once).
 *
 * Packed layout of the scales of a [rows, K] operand: for each 128-element k-block k and each
 * block b of 128 rows (rows padded to a multiple of 256), 512 bytes at offset
 * (k * row_blocks + b) * 512 holding, for r < 128 and j < 4, scale [128 b + r, 4 k + j] at
 * byte (r % 32) * 16 + (r / 32) * 4 + j (0 for padding rows); row_blocks = 2 * ceil(rows / 256).
 */

/* Bytes of the packed scales of a [rows, K] operand (K % 128 == 0), or a negative error. */
int64_t tg_mxfp8_scale_bytes(int64_t rows, int64_t K);

/*
 * tg_mxfp8_pack_scales -- row-major scales sf_dev [rows, K / 32] (4-byte aligned) into
 * packed_dev (tg_mxfp8_scale_bytes(rows, K) bytes, 16-byte aligned, not overlapping sf_dev),
 * on ``stream``.  rows >= 0, K % 128 == 0.  Asynchronous.
 */
int tg_mxfp8_pack_scales(const void* sf_dev, void* packed_dev, int64_t rows, int64_t K,
                         void* stream);

/*
 * tg_gemm_mxfp8 -- C = the block-scaled product above, on ``stream``.
 *   A_dev [M, K], B_dev [N, K]: E4M3; SFA_dev, SFB_dev: packed scales of A and of B.
 *   C_dev [M, N]: out_dtype (TG_BF16 or TG_F16), row-major; products are accumulated in fp32
 *     and rounded once to nearest even.
 *   M, N, K >= 0 and < 2^31; K % 128 == 0; N % 8 == 0.  All five pointers 16-byte aligned.
 *   C must not overlap any input.  M == 0 or N == 0: nothing is done.  K == 0: C is
 *   zero-filled.
 * Kernels: one CTA per 128 x 256 output tile (TG_VARIANT_SINGLE), or a CTA pair per 256 x 256
 * tile (TG_VARIANT_PAIR, tcgen05 cta_group::2); tg_gemm_mxfp8 (TG_VARIANT_AUTO) takes the pair
 * kernel when its tiles fill at least one wave of resident pairs, or when K >= 4096 and
 * M >= 256, else the single one, and tg_gemm_launch_shape gives the launch of either.  Persistent,
 * grouped order with the tail split.  Asynchronous; errors as for tg_gemm_persistent.
 * Inputs that hold NaN patterns give unspecified outputs.
 */
int tg_gemm_mxfp8(const void* A_dev, const void* SFA_dev, const void* B_dev, const void* SFB_dev,
                  void* C_dev, int64_t M, int64_t N, int64_t K, int out_dtype, void* stream);

/* tg_gemm_mxfp8 with an explicit kernel: variant TG_VARIANT_AUTO, _SINGLE or _PAIR, optionally
   OR'ed with TG_SCHEDULE_PLAIN and/or TG_SCHEDULE_COLUMN_MAJOR (others: TG_ERR_ARG). */
int tg_gemm_mxfp8_ex(const void* A_dev, const void* SFA_dev, const void* B_dev,
                     const void* SFB_dev, void* C_dev, int64_t M, int64_t N, int64_t K,
                     int out_dtype, void* stream, int variant);

/*
 * tg_gemm_mxfp8_debug -- tg_gemm_mxfp8_ex, synchronously, with the inspection aids of
 * tg_gemm_persistent_debug (trace of 5 int32 per unit, watchdog limit, injected missing fill).
 *   flags: as tg_gemm_mxfp8_ex's variant.  (TG_EPILOGUE_DIRECT is a dense-GEMM option:
 *   TG_ERR_ARG here.)
 */
int tg_gemm_mxfp8_debug(const void* A_dev, const void* SFA_dev, const void* B_dev,
                        const void* SFB_dev, void* C_dev, int64_t M, int64_t N, int64_t K,
                        int out_dtype, void* stream, int flags, int32_t* trace_dev,
                        uint64_t watchdog_ns, int64_t inject_skip_phase);

#ifdef __cplusplus
}
#endif

#endif /* TG_H */
