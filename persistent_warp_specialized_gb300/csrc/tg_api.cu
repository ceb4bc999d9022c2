// tg_api.cu -- the C ABI declared in include/tg.h: argument checks, TMA descriptor
// encoding, persistent grid sizing and launch.
//
// The checks follow the host-side asserts TileLang emits before a launch ("tilelang",
// 1.2 Pass Pipeline, Host IRModule: non-null data, rank-2 row-major with unit inner
// stride and zero byte offset, inner dimension divisible by 8), and the descriptor set-up
// follows its generated ``call()`` ("tilelang", Generated Kernel Source:
// cuTensorMapEncodeTiled per operand, error text kept for get_last_error()).
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <mutex>

#include "../../include/tg.h"
#include "tg_config.h"
#include "tg_wide_config.h"
#include "tg_internal.h"
#include "tg_tile_scheduler.cuh"

namespace {

thread_local char g_err[1024] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return code;
}

int fail_cuda(const char* what, cudaError_t e) {
  return fail(TG_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// Per-device facts, established once per device: SM count, arch, kernel attributes.
struct DeviceInfo {
  int state = 0;  // 0 unknown, 1 ready, -1 unsupported
  int sms = 0;
  int max_pairs = 0;  // CTA pairs of the pair kernel resident at once
  char why[256] = "";
};
constexpr int kMaxDevices = 64;
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

int device_ready(int* sms_out, int* max_pairs_out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda("cudaGetDevice", e);
  if (dev < 0 || dev >= kMaxDevices) return fail(TG_ERR_CUDA, "device ordinal %d unsupported", dev);
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (d.state == 0) {
    int major = 0, minor = 0, sms = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return fail_cuda("cudaDeviceGetAttribute", e);
    if (major != 10 || minor != 3) {
      d.state = -1;
      snprintf(d.why, sizeof(d.why), "device %d is sm_%d%d; this library is built for sm_103a",
               dev, major, minor);
    } else if ((e = tg::prepare_gemm_kernels(&d.max_pairs)) != cudaSuccess) {
      return fail_cuda("preparing the GEMM kernels (shared memory limit, cluster occupancy)", e);
    } else {
      d.state = 1;
      d.sms = sms;
    }
  }
  if (d.state < 0) return fail(TG_ERR_CUDA, "%s", d.why);
  if (sms_out) *sms_out = d.sms;
  if (max_pairs_out) *max_pairs_out = d.max_pairs;
  return TG_OK;
}

// The pointer must be device memory of the current device (TMA reads it directly).
int check_device_ptr(const void* p, const char* name) {
  cudaPointerAttributes a;
  cudaError_t e = cudaPointerGetAttributes(&a, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(TG_ERR_ARG, "%s: not a CUDA pointer (%s)", name, cudaGetErrorString(e));
  }
  int dev = 0;
  cudaGetDevice(&dev);
  if (a.type != cudaMemoryTypeDevice || a.device != dev)
    return fail(TG_ERR_ARG, "%s: must be device memory of the current device %d", name, dev);
  return TG_OK;
}

bool overlaps(const void* a, uint64_t abytes, const void* b, uint64_t bbytes) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + bbytes && b0 < a0 + abytes;
}

// A row-major [outer, inner] matrix of ``elem_bytes``-byte elements, boxes of
// box_outer rows x box_inner elements landing with the 128-byte swizzle (or none).
int encode_tiled(CUtensorMap* map, CUtensorMapDataType dt, uint32_t elem_bytes, const void* base,
                 uint64_t inner, uint64_t outer, uint32_t box_inner, uint32_t box_outer,
                 const char* name, bool swizzle = true) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(TG_ERR_CUDA, "cuTensorMapEncodeTiled unavailable from the driver");
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * elem_bytes};  // bytes between rows
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(TG_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with CUresult %d", name, (int)r);
  return TG_OK;
}

int encode_2d(CUtensorMap* map, int dtype, const void* base, uint64_t inner, uint64_t outer,
              uint32_t box_inner, uint32_t box_outer, const char* name) {
  return encode_tiled(map,
                      dtype == TG_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                       : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                      tg::kElemBytes, base, inner, outer, box_inner, box_outer, name);
}

constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1;

// Shared validation of the GEMM entry points.  *nothing_to_do is set for M == 0 or N == 0.
int validate(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K, int dtype,
             bool* nothing_to_do) {
  *nothing_to_do = false;
  if (dtype != TG_F16 && dtype != TG_BF16) return fail(TG_ERR_ARG, "unknown dtype %d", dtype);
  if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
    return fail(TG_ERR_ARG, "sizes must be in [0, 2^31): M=%lld N=%lld K=%lld", (long long)M,
                (long long)N, (long long)K);
  if (M == 0 || N == 0) {
    *nothing_to_do = true;
    return TG_OK;
  }
  if (!C || (K > 0 && (!A || !B))) return fail(TG_ERR_ARG, "null matrix pointer");
  if (N % 8 != 0 || K % 8 != 0)
    return fail(TG_ERR_ALIGN, "N=%lld and K=%lld must be multiples of 8 (16-byte row strides)",
                (long long)N, (long long)K);
  if ((reinterpret_cast<uintptr_t>(C) & 15u) ||
      (K > 0 && ((reinterpret_cast<uintptr_t>(A) & 15u) || (reinterpret_cast<uintptr_t>(B) & 15u))))
    return fail(TG_ERR_ALIGN, "A, B and C must be 16-byte aligned");
  const uint64_t m_blocks = (M + tg::kBM - 1) / tg::kBM, n_blocks = (N + tg::kBN - 1) / tg::kBN;
  if (m_blocks * n_blocks > static_cast<uint64_t>(kMaxDim))
    return fail(TG_ERR_ARG, "too many output tiles");
  int rc;
  if ((rc = check_device_ptr(C, "C")) != TG_OK) return rc;
  if (K > 0) {
    if ((rc = check_device_ptr(A, "A")) != TG_OK) return rc;
    if ((rc = check_device_ptr(B, "B")) != TG_OK) return rc;
    const uint64_t cb = uint64_t(M) * N * tg::kElemBytes;
    if (overlaps(C, cb, A, uint64_t(M) * K * tg::kElemBytes) ||
        overlaps(C, cb, B, uint64_t(K) * N * tg::kElemBytes))
      return fail(TG_ERR_ARG, "C overlaps A or B");
  }
  return TG_OK;
}

// The default limit of every bounded wait in the kernels when the caller gives none: the
// fixed kDefaultWatchdogNs plus 2 us per k-block of K.  The longest legitimate wait spans one
// unit's whole K (the epilogue waiting for its accumulator), and a k-block takes at most about
// 0.5 us on GB300 even on a CTA pair's half-width unit, so with K near 2^31 (2^25 k-blocks of
// 64, ~12 s per unit, measured) a fixed limit of ~4 s stopped a correct GEMM.
uint64_t default_watchdog_ns(uint32_t k_blocks) {
  return tg::kDefaultWatchdogNs + uint64_t(k_blocks) * 2000u;
}

// The variant TG_VARIANT_AUTO resolves to (both GEMMs): the CTA-pair kernel once its 256 x 256
// tiles fill at least one wave of resident pairs (measured faster there at every workload
// size), or below a wave once K >= 4096 and M fills the pair's 256 rows; else the single-CTA
// kernel, whose smaller tiles spread a short-K problem over more SMs.  Below a wave, a 256 x 256
// pair MMA reads fewer shared-memory bytes per flop than the single CTA's 128 x 256 one, which
// pays once K is long enough to amortise the pair's pipeline fill.  Same box, L2 flushed before
// each of 50 launches, medians (single / pair TFLOP/s): dense bf16 1024 x 1024 x 4096 323 / 350,
// x 8192 365 / 419, 512 x 512 x 8192 94 / 110, 1536 x 1536 x 4096 675 / 755, 2048 x 2048 x 4096
// 1119 / 1117; MXFP8 1024 x 1024 x 8192 524 / 599, 512 x 512 x 8192 131 / 150, 2048 x 2048 x
// 4096 1523 / 1525 (back to back, 1890 / 2007).  With K <= 2048 the single kernel is as fast or
// faster (dense 1024^3 175 / 150, 2048^3 839 / 838; MXFP8 1024 x 1024 x 2048 back to back 435 /
// 404).
int auto_variant(int64_t M, int64_t N, int64_t K, int max_pairs) {
  const int64_t pair_tiles = ((M + tg::kPairBM - 1) / tg::kPairBM) * ((N + tg::kBN - 1) / tg::kBN);
  if (max_pairs < 1) return TG_VARIANT_SINGLE;
  return (pair_tiles >= max_pairs || (K >= 4096 && M >= tg::kPairBM)) ? TG_VARIANT_PAIR
                                                                      : TG_VARIANT_SINGLE;
}

// The dense GEMM's choice: the wide pair kernel (256 x 512 tiles) when its tiles fill at least
// one wave of resident pairs and K is long enough for the once-per-tile drain of its single
// accumulator to stay small, else as auto_variant.  Measured on GB300 (same box, medians of 5
// alternating bursts, pair / wide TFLOP/s): K >= 6144 favours wide at every size tried (6144^3
// 1835 / 1894, 4096 x 4096 x 8192 1711 / 1763 at 1.7 waves, 4096 x 8192 x 8192 1838 / 1874,
// 8192^3 +2.6 %); K = 4096 ties (8192 x 8192 1904 / 1894, 12288 x 12288 1937 / 1939, 6144 x 6144
// 1858 / 1862), so wide is kept there only for four waves or more; K = 2048 favours the pair
// kernel (8192 x 8192 1858 / 1773).
int auto_variant_dense(int64_t M, int64_t N, int64_t K, int max_pairs) {
  const int64_t wide_tiles =
      ((M + tg::kPairBM - 1) / tg::kPairBM) * ((N + tg::kWideBN - 1) / tg::kWideBN);
  if (max_pairs > 0 && ((K >= 6144 && wide_tiles >= max_pairs) ||
                        (K >= 4096 && wide_tiles >= 4 * int64_t(max_pairs))))
    return TG_VARIANT_PAIR_WIDE;
  return auto_variant(M, N, K, max_pairs);
}

bool pair_variant(int v) { return v == TG_VARIANT_PAIR || v == TG_VARIANT_PAIR_WIDE; }

// The traversal TG_VARIANT_AUTO gives the dense kernel it picks when the caller names neither
// an order nor a group width (the page's scheduler options ``column_major`` and
// ``swizzle_size``).  When all of B fits in half of the L2, whole rows of tiles (group = the
// number of N-tiles) read each row slab of A from DRAM once while B stays resident; when only A
// fits, whole columns do the same with the roles exchanged.  Otherwise a wave of P tiles covers
// a block of them, and the operand bytes it touches (its A rows plus its B columns) are least
// when both extents match: about sqrt(P tile_n / tile_m) M-tiles by sqrt(P tile_m / tile_n)
// N-tiles.  For the square 256 x 256 pair tiles (P = 76) that is the page's group of 8 (row
// order); for the wide pair kernel's 256 x 512 tiles it is groups of 12 M-tiles in column order.
// Measured on GB300 (medians of alternating rounds, TFLOP/s): pair kernel 4096^3 rows 1797 vs
// groups of 8 1745, 4000 x 7000 x 2048 rows of 16 1637 vs 1612, 8192^3 groups of 8 best; wide
// kernel, column order groups of 12 vs row order groups of 8: 8192^3 1959 vs 1944 (3000
// back-to-back launches: 1741 vs 1716), 6144^3 1924 vs 1908, 8192 x 8192 x 16384 2009 vs 1986.
struct Raster {
  uint32_t group, column_major;
};
constexpr uint64_t kHalfL2Bytes = 64ull << 20;

Raster auto_raster(int64_t M, int64_t N, int64_t K, uint32_t m_tiles, uint32_t n_tiles,
                   uint32_t tile_m, uint32_t tile_n, uint32_t workers) {
  const uint64_t a_bytes = uint64_t(M) * K * tg::kElemBytes;
  const uint64_t b_bytes = uint64_t(K) * N * tg::kElemBytes;
  if (b_bytes <= kHalfL2Bytes) return {n_tiles < 255u ? n_tiles : 255u, 0u};
  if (a_bytes <= kHalfL2Bytes) return {m_tiles < 255u ? m_tiles : 255u, 1u};
  if (tile_n > tile_m) {   // wide tiles: panels of M-tiles, as many as balance the wave
    const double g = std::sqrt(double(workers) * tile_n / tile_m);
    const uint32_t gi = static_cast<uint32_t>(g + 0.5);
    return {gi < 1u ? 1u : (gi > 255u ? 255u : gi), 1u};
  }
  return {static_cast<uint32_t>(tg::kGroup), 0u};
}

// Workspace of the stream-K tail: one flag per (worker, CTA, epilogue warp), padded to 256
// bytes, then one fp32 slice of 128 rows x tile_n per (worker, CTA).
uint64_t sk_flag_bytes(uint32_t workers) {
  return (uint64_t(workers) * 2 * tg::kEpiWarps * 4 + 255) / 256 * 256;
}
uint64_t sk_partial_bytes(uint32_t workers, uint32_t tile_n) {
  return uint64_t(workers) * 2 * tg::kBM * tile_n * 4;
}

struct Shape {
  uint32_t tile_m, tile_n, m_tiles, n_tiles, workers, ctas, split_from, units;
  uint32_t sk_tiles;       // stream-K tail tiles (0: none); then units = split_from = whole tiles
  uint64_t sk_bytes;       // workspace the stream-K tail needs
};

int block_k_of(int variant) {
  return variant == TG_VARIANT_PAIR        ? tg::kPairBK
         : variant == TG_VARIANT_PAIR_WIDE ? tg::kWideBK
                                           : tg::kBK;
}

// Persistent launch of a concrete variant: one worker per SM (SINGLE) or per resident CTA
// pair (PAIR), never more workers than work units; the last partial wave is split into
// half-width units unless ``plain`` (the page's traversal) is asked for, or, for the CTA-pair
// variants when ``streamk`` is asked for (with a workspace), along K (the stream-K tail of
// tg_tile_scheduler.cuh).  The library never takes the stream-K tail by itself: measured on
// GB300 it lost to the half-width units at every size tried (the partial sums' round trip
// through memory costs about what the idle part of the last wave does).
Shape launch_shape(int64_t M, int64_t N, int64_t K, int variant, bool plain, bool dynamic,
                   int sms, int max_pairs, bool streamk = false) {
  Shape sh;
  sh.tile_m = pair_variant(variant) ? tg::kPairBM : tg::kBM;
  sh.tile_n = variant == TG_VARIANT_PAIR_WIDE ? tg::kWideBN : tg::kBN;
  sh.m_tiles = static_cast<uint32_t>((M + sh.tile_m - 1) / sh.tile_m);
  sh.n_tiles = static_cast<uint32_t>((N + sh.tile_n - 1) / sh.tile_n);
  const uint32_t tiles = sh.m_tiles * sh.n_tiles;
  const uint32_t slots = pair_variant(variant) ? uint32_t(max_pairs) : uint32_t(sms);
  const uint32_t bk = static_cast<uint32_t>(block_k_of(variant));
  const uint32_t k_blocks = static_cast<uint32_t>((uint64_t(K) + bk - 1) / bk);
  sh.sk_tiles = 0;
  sh.sk_bytes = 0;
  const uint32_t rem = tiles % slots;
  if (streamk && !plain && !dynamic && pair_variant(variant) && k_blocks > 0 && rem > 0) {
    sh.sk_tiles = rem;
    sh.split_from = sh.units = tiles - rem;
    sh.workers = slots;   // every worker takes a range of the tail
    sh.ctas = 2 * sh.workers;
    sh.sk_bytes = sk_flag_bytes(sh.workers) + sk_partial_bytes(sh.workers, sh.tile_n);
    return sh;
  }
  if (plain) {
    sh.split_from = sh.units = tiles;
  } else {
    tg::PersistentTileScheduler::tail_split(tiles, slots, sh.split_from, sh.units);
  }
  // dynamic persistence launches one CTA per unit; only ~#SMs run at once and they take over
  // the rest through cluster launch control
  sh.workers = dynamic ? sh.units : (sh.units < slots ? sh.units : slots);
  sh.ctas = pair_variant(variant) ? 2 * sh.workers : sh.workers;
  return sh;
}

constexpr int kGroupBits = TG_SCHEDULE_GROUP(0xFF);
constexpr int kScheduleFlags = TG_SCHEDULE_PLAIN | TG_SCHEDULE_COLUMN_MAJOR |
                               TG_SCHEDULE_DYNAMIC | TG_EPILOGUE_DIRECT | TG_SCHEDULE_STREAMK |
                               kGroupBits;

bool known_variant(int v) {
  const int kernel = v & ~kScheduleFlags;
  return kernel == TG_VARIANT_AUTO || kernel == TG_VARIANT_SINGLE || kernel == TG_VARIANT_PAIR ||
         kernel == TG_VARIANT_PAIR_WIDE;
}

// The group width a variant asks for (TG_SCHEDULE_GROUP), or the default.
uint32_t group_of(int v) {
  const uint32_t g = (static_cast<uint32_t>(v) & static_cast<uint32_t>(kGroupBits)) >> 16;
  return g ? g : static_cast<uint32_t>(tg::kGroup);
}

// True when TG_VARIANT_AUTO also chooses the traversal: the caller named no order, no group
// width and not the page's plain traversal.
bool auto_traversal(int variant) {
  return (variant & ~kScheduleFlags) == TG_VARIANT_AUTO &&
         (variant & (TG_SCHEDULE_PLAIN | TG_SCHEDULE_COLUMN_MAJOR | kGroupBits)) == 0;
}

// Epoch of a launch with a stream-K tail: never 0, distinct for 2^32 - 1 launches.
std::atomic<uint32_t> g_sk_epoch{0};

uint32_t next_sk_epoch() {
  uint32_t e = ++g_sk_epoch;
  while (e == 0) e = ++g_sk_epoch;
  return e;
}

int gemm_impl(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K, int dtype,
              void* stream, int variant, bool debug, int32_t* trace, uint64_t watchdog_ns,
              int64_t inject, void* workspace = nullptr, int64_t workspace_bytes = 0) {
  if (!known_variant(variant)) return fail(TG_ERR_ARG, "unknown variant %d", variant);
  const bool force_sk = (variant & TG_SCHEDULE_STREAMK) != 0;
  if (force_sk && !workspace) return fail(TG_ERR_ARG, "TG_SCHEDULE_STREAMK needs a workspace");
  if (workspace_bytes < 0) return fail(TG_ERR_ARG, "negative workspace size");
  if (workspace) {
    int rc = check_device_ptr(workspace, "workspace");
    if (rc != TG_OK) return rc;
    if (reinterpret_cast<uintptr_t>(workspace) & 255u)
      return fail(TG_ERR_ALIGN, "the workspace must be 256-byte aligned");
  }
  const bool plain = (variant & TG_SCHEDULE_PLAIN) != 0;
  uint32_t column_major = (variant & TG_SCHEDULE_COLUMN_MAJOR) ? 1u : 0u;
  const bool dynamic = (variant & TG_SCHEDULE_DYNAMIC) != 0;
  uint32_t group = group_of(variant);
  const uint32_t epi_direct = (variant & TG_EPILOGUE_DIRECT) ? 1u : 0u;
  const bool choose_traversal = auto_traversal(variant);
  variant &= ~kScheduleFlags;
  bool nothing = false;
  int rc = validate(A, B, C, M, N, K, dtype, &nothing);
  if (rc != TG_OK || nothing) return rc;
  int sms = 0, max_pairs = 0;
  if ((rc = device_ready(&sms, &max_pairs)) != TG_OK) return rc;
  if (variant == TG_VARIANT_AUTO) variant = auto_variant_dense(M, N, K, max_pairs);
  if (pair_variant(variant) && max_pairs < 1)
    return fail(TG_ERR_CUDA, "no CTA pair of the pair kernel fits on this device");
  if (dynamic && variant != TG_VARIANT_SINGLE)
    return fail(TG_ERR_ARG, "TG_SCHEDULE_DYNAMIC needs the single-CTA variant");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (K == 0) {
    cudaError_t e = tg::launch_zero_fill(C, uint64_t(M) * N * tg::kElemBytes, s);
    return e == cudaSuccess ? TG_OK : fail_cuda("zero fill launch", e);
  }
  tg::GemmLaunch l;
  if ((rc = encode_2d(&l.tmA, dtype, A, K, M, tg::kKAtom, tg::kBM, "A")) != TG_OK) return rc;
  const int block_k = block_k_of(variant);
  if ((rc = encode_2d(&l.tmB, dtype, B, N, K, tg::kBChunkCols, block_k, "B")) != TG_OK) return rc;
  if ((rc = encode_2d(&l.tmC, dtype, C, N, M, tg::kEpiN, 32, "C")) != TG_OK) return rc;
  l.C = C;
  l.M = static_cast<uint32_t>(M);
  l.N = static_cast<uint32_t>(N);
  l.K = static_cast<uint32_t>(K);
  const Shape sh = launch_shape(M, N, K, variant, plain, dynamic, sms, max_pairs, force_sk);
  if (sh.sk_tiles && uint64_t(workspace_bytes) < sh.sk_bytes)
    return fail(TG_ERR_ARG, "workspace of %lld bytes; the stream-K tail needs %llu",
                static_cast<long long>(workspace_bytes),
                static_cast<unsigned long long>(sh.sk_bytes));
  if (choose_traversal) {
    const Raster r = auto_raster(M, N, K, sh.m_tiles, sh.n_tiles, sh.tile_m, sh.tile_n,
                                 sh.workers);
    group = r.group;
    column_major = r.column_major;
  }
  l.m_blocks = sh.m_tiles;
  l.n_blocks = sh.n_tiles;
  l.split_from = sh.split_from;
  l.total_units = sh.units;
  l.column_major = column_major;
  l.dynamic = dynamic ? 1u : 0u;
  l.epi_direct = epi_direct;
  l.k_blocks = static_cast<uint32_t>((K + block_k - 1) / block_k);
  l.group = group;
  l.grid = sh.ctas;
  l.watchdog_ns = watchdog_ns ? watchdog_ns : default_watchdog_ns(l.k_blocks);
  l.trace = trace;
  l.inject_skip_phase = inject;
  l.sk_tiles = sh.sk_tiles;
  l.sk_epoch = sh.sk_tiles ? next_sk_epoch() : 0u;
  l.sk_slot_f4 = tg::kBM * sh.tile_n / 4;
  l.sk_flags = sh.sk_tiles ? static_cast<uint32_t*>(workspace) : nullptr;
  l.sk_partials = sh.sk_tiles ? reinterpret_cast<float4*>(static_cast<char*>(workspace) +
                                                          sk_flag_bytes(sh.workers))
                              : nullptr;
  cudaError_t e;
  if (debug && (e = tg::clear_watchdog_status(s)) != cudaSuccess)
    return fail_cuda("clearing the watchdog word", e);
  if ((e = tg::launch_gemm(dtype, debug, variant, l, s)) != cudaSuccess)
    return fail_cuda("GEMM launch", e);
  if (debug) {
    unsigned int st = 0;
    if ((e = tg::read_and_clear_watchdog_status(&st, s)) != cudaSuccess)
      return fail_cuda("GEMM execution", e);
    if (st)
      return fail(TG_ERR_TIMEOUT, "watchdog: a wait gave up (roles 0x%x: 1 producer, 2 MMA, "
                  "4 epilogue, 8 shutdown)", st);
  }
  return TG_OK;
}

// ---------------------------------------------------------------- block-scaled MXFP8
// Row blocks (of 128) of a packed scale array: the rows rounded up to a multiple of 256, so
// that the two atoms of a 256-row B tile always exist.
uint64_t mx_row_blocks(int64_t rows) {
  return (uint64_t(rows) + tg::kMxPackRows - 1) / tg::kMxPackRows * (tg::kMxPackRows / tg::kBM);
}

uint64_t mx_packed_bytes(int64_t rows, int64_t K) {
  return uint64_t(K) / tg::kMxBK * mx_row_blocks(rows) * tg::kMxSfAtomBytes;
}

int validate_mx(const void* A, const void* SFA, const void* B, const void* SFB, void* C,
                int64_t M, int64_t N, int64_t K, int out_dtype, bool* nothing_to_do) {
  *nothing_to_do = false;
  if (out_dtype != TG_F16 && out_dtype != TG_BF16)
    return fail(TG_ERR_ARG, "unknown output dtype %d", out_dtype);
  if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
    return fail(TG_ERR_ARG, "sizes must be in [0, 2^31): M=%lld N=%lld K=%lld", (long long)M,
                (long long)N, (long long)K);
  if (M == 0 || N == 0) {
    *nothing_to_do = true;
    return TG_OK;
  }
  if (!C || (K > 0 && (!A || !B || !SFA || !SFB))) return fail(TG_ERR_ARG, "null matrix pointer");
  if (K % tg::kMxBK != 0)
    return fail(TG_ERR_ALIGN, "K=%lld must be a multiple of %d (whole scale words per row)",
                (long long)K, tg::kMxBK);
  if (N % 8 != 0) return fail(TG_ERR_ALIGN, "N=%lld must be a multiple of 8", (long long)N);
  if ((reinterpret_cast<uintptr_t>(C) & 15u) ||
      (K > 0 && ((reinterpret_cast<uintptr_t>(A) & 15u) || (reinterpret_cast<uintptr_t>(B) & 15u))))
    return fail(TG_ERR_ALIGN, "A, B and C must be 16-byte aligned");
  if (K > 0 && ((reinterpret_cast<uintptr_t>(SFA) & 15u) || (reinterpret_cast<uintptr_t>(SFB) & 15u)))
    return fail(TG_ERR_ALIGN, "SFA and SFB must be 16-byte aligned");
  const uint64_t m_blocks = (M + tg::kBM - 1) / tg::kBM, n_blocks = (N + tg::kBN - 1) / tg::kBN;
  if (m_blocks * n_blocks > static_cast<uint64_t>(kMaxDim))
    return fail(TG_ERR_ARG, "too many output tiles");
  int rc;
  if ((rc = check_device_ptr(C, "C")) != TG_OK) return rc;
  if (K > 0) {
    if ((rc = check_device_ptr(A, "A")) != TG_OK) return rc;
    if ((rc = check_device_ptr(B, "B")) != TG_OK) return rc;
    if ((rc = check_device_ptr(SFA, "SFA")) != TG_OK) return rc;
    if ((rc = check_device_ptr(SFB, "SFB")) != TG_OK) return rc;
    const uint64_t cb = uint64_t(M) * N * tg::kElemBytes;
    if (overlaps(C, cb, A, uint64_t(M) * K) || overlaps(C, cb, B, uint64_t(N) * K) ||
        overlaps(C, cb, SFA, mx_packed_bytes(M, K)) || overlaps(C, cb, SFB, mx_packed_bytes(N, K)))
      return fail(TG_ERR_ARG, "C overlaps an input");
  }
  return TG_OK;
}

int mx_impl(const void* A, const void* SFA, const void* B, const void* SFB, void* C, int64_t M,
            int64_t N, int64_t K, int out_dtype, void* stream, int flags, bool debug,
            int32_t* trace, uint64_t watchdog_ns, int64_t inject) {
  int variant = flags & ~(TG_SCHEDULE_PLAIN | TG_SCHEDULE_COLUMN_MAJOR | kGroupBits);
  if (variant != TG_VARIANT_AUTO && variant != TG_VARIANT_SINGLE && variant != TG_VARIANT_PAIR)
    return fail(TG_ERR_ARG, "unknown MXFP8 variant or schedule flags 0x%x", flags);
  const uint32_t group = group_of(flags);
  bool nothing = false;
  int rc = validate_mx(A, SFA, B, SFB, C, M, N, K, out_dtype, &nothing);
  if (rc != TG_OK || nothing) return rc;
  int sms = 0, max_pairs = 0;
  if ((rc = device_ready(&sms, &max_pairs)) != TG_OK) return rc;
  if (variant == TG_VARIANT_AUTO) variant = auto_variant(M, N, K, max_pairs);
  if (variant == TG_VARIANT_PAIR && max_pairs < 1)
    return fail(TG_ERR_CUDA, "no CTA pair of the MXFP8 pair kernel fits on this device");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (K == 0) {
    cudaError_t e = tg::launch_zero_fill(C, uint64_t(M) * N * tg::kElemBytes, s);
    return e == cudaSuccess ? TG_OK : fail_cuda("zero fill launch", e);
  }
  tg::MxLaunch l;
  if ((rc = encode_tiled(&l.tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, A, K, M, tg::kMxBK, tg::kBM,
                         "A")) != TG_OK)
    return rc;
  if ((rc = encode_tiled(&l.tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, B, K, N, tg::kMxBK,
                         tg::kBN / 2, "B")) != TG_OK)
    return rc;
  if ((rc = encode_2d(&l.tmC, out_dtype, C, N, M, tg::kEpiN, 32, "C")) != TG_OK) return rc;
  l.sfa_blocks = static_cast<uint32_t>(mx_row_blocks(M));
  l.sfb_blocks = static_cast<uint32_t>(mx_row_blocks(N));
  if (variant == TG_VARIANT_PAIR) {
    // the packed scales as rows of 128 32-bit words, one row per atom: one atom of A and two
    // adjacent atoms of B per box
    const uint64_t k_blocks = uint64_t(K) / tg::kMxBK;
    if ((rc = encode_tiled(&l.tmSFA, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, SFA, 128,
                           k_blocks * l.sfa_blocks, 128, 1, "SFA", false)) != TG_OK)
      return rc;
    if ((rc = encode_tiled(&l.tmSFB, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, SFB, 128,
                           k_blocks * l.sfb_blocks, 128, 2, "SFB", false)) != TG_OK)
      return rc;
  } else {
    l.tmSFA = l.tmA;   // unused by the single-CTA kernel
    l.tmSFB = l.tmA;
  }
  const Shape sh = launch_shape(M, N, K, variant, (flags & TG_SCHEDULE_PLAIN) != 0, false, sms,
                                max_pairs);
  l.SFA = SFA;
  l.SFB = SFB;
  l.M = static_cast<uint32_t>(M);
  l.N = static_cast<uint32_t>(N);
  l.K = static_cast<uint32_t>(K);
  l.m_blocks = sh.m_tiles;
  l.n_blocks = sh.n_tiles;
  l.k_blocks = static_cast<uint32_t>(K / tg::kMxBK);
  l.group = group;
  l.split_from = sh.split_from;
  l.total_units = sh.units;
  l.column_major = (flags & TG_SCHEDULE_COLUMN_MAJOR) ? 1u : 0u;
  l.grid = sh.ctas;
  l.watchdog_ns = watchdog_ns ? watchdog_ns : default_watchdog_ns(l.k_blocks);
  l.trace = trace;
  l.inject_skip_phase = inject;
  cudaError_t e;
  if (debug && (e = tg::clear_watchdog_status(s)) != cudaSuccess)
    return fail_cuda("clearing the watchdog word", e);
  if ((e = tg::launch_mxfp8(out_dtype, debug, variant, l, s)) != cudaSuccess)
    return fail_cuda("MXFP8 GEMM launch", e);
  if (debug) {
    unsigned int st = 0;
    if ((e = tg::read_and_clear_watchdog_status(&st, s)) != cudaSuccess)
      return fail_cuda("MXFP8 GEMM execution", e);
    if (st)
      return fail(TG_ERR_TIMEOUT, "watchdog: a wait gave up (roles 0x%x: 1 producer, 2 MMA, "
                  "4 epilogue, 8 shutdown)", st);
  }
  return TG_OK;
}

}  // namespace

// Scratch of tg_tile_schedule_noalloc: TG_SCHEDULE_NOALLOC_MAX_UNITS rows of 5 int32 in the
// library's device image, so that call needs no allocation.  In host code the name stands for a
// host-side shadow, not a device address: every call looks the device address up with
// cudaGetSymbolAddress on the current device and passes it to the scheduler kernel.  The
// address is not cached, because a context torn down and created again (cudaDeviceReset) loads
// the image anew, possibly elsewhere.
static __device__ __align__(256) int32_t g_schedule_scratch[5 * TG_SCHEDULE_NOALLOC_MAX_UNITS];

namespace {

std::mutex g_schedule_scratch_mu;   // one call at a time uses the array

}  // namespace

extern "C" {

int64_t tg_mxfp8_scale_bytes(int64_t rows, int64_t K) {
  if (rows < 0 || K < 0 || rows > kMaxDim || K > kMaxDim)
    return fail(TG_ERR_ARG, "sizes must be in [0, 2^31): rows=%lld K=%lld", (long long)rows,
                (long long)K);
  if (K % tg::kMxBK != 0)
    return fail(TG_ERR_ALIGN, "K=%lld must be a multiple of %d", (long long)K, tg::kMxBK);
  return static_cast<int64_t>(mx_packed_bytes(rows, K));
}

int tg_mxfp8_pack_scales(const void* sf_dev, void* packed_dev, int64_t rows, int64_t K,
                         void* stream) {
  const int64_t bytes = tg_mxfp8_scale_bytes(rows, K);
  if (bytes < 0) return static_cast<int>(bytes);
  if (bytes == 0) return TG_OK;
  if (!packed_dev || (rows > 0 && !sf_dev)) return fail(TG_ERR_ARG, "null scale pointer");
  if ((reinterpret_cast<uintptr_t>(packed_dev) & 15u) ||
      (rows > 0 && (reinterpret_cast<uintptr_t>(sf_dev) & 3u)))
    return fail(TG_ERR_ALIGN, "packed scales must be 16-byte aligned, row-major scales 4-byte");
  int rc;
  if ((rc = check_device_ptr(packed_dev, "packed scales")) != TG_OK) return rc;
  if (rows > 0) {
    if ((rc = check_device_ptr(sf_dev, "scales")) != TG_OK) return rc;
    if (overlaps(sf_dev, uint64_t(rows) * K / tg::kMxBlock, packed_dev, uint64_t(bytes)))
      return fail(TG_ERR_ARG, "packed scales overlap the row-major scales");
  }
  cudaError_t e = tg::launch_mx_pack(sf_dev, packed_dev, static_cast<uint32_t>(rows),
                                     static_cast<uint32_t>(K / tg::kMxBK),
                                     static_cast<uint32_t>(mx_row_blocks(rows)),
                                     static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? TG_OK : fail_cuda("scale pack launch", e);
}

int tg_gemm_mxfp8(const void* A_dev, const void* SFA_dev, const void* B_dev, const void* SFB_dev,
                  void* C_dev, int64_t M, int64_t N, int64_t K, int out_dtype, void* stream) {
  return mx_impl(A_dev, SFA_dev, B_dev, SFB_dev, C_dev, M, N, K, out_dtype, stream, 0, false,
                 nullptr, 0, -1);
}

int tg_gemm_mxfp8_ex(const void* A_dev, const void* SFA_dev, const void* B_dev,
                     const void* SFB_dev, void* C_dev, int64_t M, int64_t N, int64_t K,
                     int out_dtype, void* stream, int variant) {
  return mx_impl(A_dev, SFA_dev, B_dev, SFB_dev, C_dev, M, N, K, out_dtype, stream, variant, false,
                 nullptr, 0, -1);
}

int tg_gemm_mxfp8_debug(const void* A_dev, const void* SFA_dev, const void* B_dev,
                        const void* SFB_dev, void* C_dev, int64_t M, int64_t N, int64_t K,
                        int out_dtype, void* stream, int flags, int32_t* trace_dev,
                        uint64_t watchdog_ns, int64_t inject_skip_phase) {
  if (trace_dev) {
    int rc = check_device_ptr(trace_dev, "trace");
    if (rc != TG_OK) return rc;
  }
  return mx_impl(A_dev, SFA_dev, B_dev, SFB_dev, C_dev, M, N, K, out_dtype, stream, flags, true,
                 trace_dev, watchdog_ns, inject_skip_phase);
}

int tg_gemm_persistent(const void* A_dev, const void* B_dev, void* C_dev, int64_t M, int64_t N,
                       int64_t K, int dtype, void* stream) {
  return gemm_impl(A_dev, B_dev, C_dev, M, N, K, dtype, stream, TG_VARIANT_AUTO, false, nullptr,
                   0, -1);
}

int tg_gemm_persistent_ex(const void* A_dev, const void* B_dev, void* C_dev, int64_t M,
                          int64_t N, int64_t K, int dtype, void* stream, int variant) {
  if (variant & TG_SCHEDULE_STREAMK)
    return fail(TG_ERR_ARG, "TG_SCHEDULE_STREAMK needs a workspace (tg_gemm_persistent_ws)");
  return gemm_impl(A_dev, B_dev, C_dev, M, N, K, dtype, stream, variant, false, nullptr, 0, -1);
}

int tg_gemm_persistent_ws(const void* A_dev, const void* B_dev, void* C_dev, int64_t M,
                          int64_t N, int64_t K, int dtype, void* stream, int variant,
                          void* workspace_dev, int64_t workspace_bytes) {
  return gemm_impl(A_dev, B_dev, C_dev, M, N, K, dtype, stream, variant, false, nullptr, 0, -1,
                   workspace_dev, workspace_bytes);
}

int64_t tg_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, int variant) {
  int sk_tiles = 0;
  int64_t bytes = 0;
  int rc = tg_gemm_launch_shape(M, N, K, variant | TG_SHAPE_WORKSPACE, nullptr, nullptr, nullptr,
                                nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                                nullptr, &sk_tiles, &bytes);
  return rc != TG_OK ? rc : bytes;
}

int tg_gemm_launch_shape(int64_t M, int64_t N, int64_t K, int variant, int* variant_out,
                         int* tile_m, int* tile_n, int* m_tiles, int* n_tiles, int* workers,
                         int* ctas, int* split_from, int* units, int* group,
                         int* column_major, int* sk_tiles, int64_t* workspace_bytes) {
  const bool mxfp8 = (variant & TG_SHAPE_MXFP8) != 0;
  const bool with_ws = (variant & TG_SHAPE_WORKSPACE) != 0;
  variant &= ~(TG_SHAPE_MXFP8 | TG_SHAPE_WORKSPACE);
  if (!known_variant(variant)) return fail(TG_ERR_ARG, "unknown variant %d", variant);
  const bool force_sk = (variant & TG_SCHEDULE_STREAMK) != 0;
  if (force_sk && (mxfp8 || !with_ws))
    return fail(TG_ERR_ARG, "TG_SCHEDULE_STREAMK: dense GEMM with a workspace only");
  const bool plain = (variant & TG_SCHEDULE_PLAIN) != 0;
  const bool dynamic = (variant & TG_SCHEDULE_DYNAMIC) != 0;
  const bool choose_traversal = auto_traversal(variant) && !mxfp8;
  Raster r = {group_of(variant), (variant & TG_SCHEDULE_COLUMN_MAJOR) ? 1u : 0u};
  variant &= ~kScheduleFlags;
  if (mxfp8 && (dynamic || variant == TG_VARIANT_PAIR_WIDE))
    return fail(TG_ERR_ARG, "the MXFP8 GEMM has the single and pair variants only");
  if (M < 1 || N < 1 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
    return fail(TG_ERR_ARG, "sizes must be M, N in [1, 2^31), K in [0, 2^31)");
  int sms = 0, max_pairs = 0;
  int rc = device_ready(&sms, &max_pairs);
  if (rc != TG_OK) return rc;
  if (variant == TG_VARIANT_AUTO)
    variant = mxfp8 ? auto_variant(M, N, K, max_pairs) : auto_variant_dense(M, N, K, max_pairs);
  if (dynamic && variant != TG_VARIANT_SINGLE)
    return fail(TG_ERR_ARG, "TG_SCHEDULE_DYNAMIC needs the single-CTA variant");
  const Shape sh = launch_shape(M, N, K, variant, plain, dynamic, sms, max_pairs,
                                with_ws && !mxfp8 && force_sk);
  if (choose_traversal)
    r = auto_raster(M, N, K, sh.m_tiles, sh.n_tiles, sh.tile_m, sh.tile_n, sh.workers);
  if (variant_out) *variant_out = variant;
  if (group) *group = static_cast<int>(r.group);
  if (column_major) *column_major = static_cast<int>(r.column_major);
  if (tile_m) *tile_m = static_cast<int>(sh.tile_m);
  if (tile_n) *tile_n = static_cast<int>(sh.tile_n);
  if (m_tiles) *m_tiles = static_cast<int>(sh.m_tiles);
  if (n_tiles) *n_tiles = static_cast<int>(sh.n_tiles);
  if (workers) *workers = static_cast<int>(sh.workers);
  if (ctas) *ctas = static_cast<int>(sh.ctas);
  if (split_from) *split_from = static_cast<int>(sh.split_from);
  // with a stream-K tail, unit ids (the debug trace's rows) run up to split_from + 2 workers
  if (units) *units = static_cast<int>(sh.sk_tiles ? sh.units + 2 * sh.workers : sh.units);
  if (sk_tiles) *sk_tiles = static_cast<int>(sh.sk_tiles);
  if (workspace_bytes) *workspace_bytes = static_cast<int64_t>(sh.sk_bytes);
  return TG_OK;
}

int tg_gemm_persistent_debug(const void* A_dev, const void* B_dev, void* C_dev, int64_t M,
                             int64_t N, int64_t K, int dtype, void* stream, int variant,
                             int32_t* trace_dev, uint64_t watchdog_ns, int64_t inject_skip_phase,
                             void* workspace_dev, int64_t workspace_bytes) {
  if (trace_dev) {
    int rc = check_device_ptr(trace_dev, "trace");
    if (rc != TG_OK) return rc;
  }
  return gemm_impl(A_dev, B_dev, C_dev, M, N, K, dtype, stream, variant, true, trace_dev,
                   watchdog_ns, inject_skip_phase, workspace_dev, workspace_bytes);
}

// Runs the device scheduler over [0, units) and copies rows of ``width`` int32 (4: without
// the part column, 5: with it) to the host.
int schedule_rows(int m_blocks, int n_blocks, int num_sms, int group, uint32_t split_from,
                  uint32_t units, uint32_t column_major, int width, int32_t* out_host) {
  const uint64_t rows = units;
  int32_t* d = nullptr;
  cudaError_t e = cudaMalloc(&d, rows * 5 * sizeof(int32_t));
  if (e != cudaSuccess) return fail_cuda("cudaMalloc", e);
  e = tg::launch_tile_schedule(m_blocks, n_blocks, num_sms, group, split_from, units,
                               column_major, d, nullptr);
  if (e == cudaSuccess) {
    if (width == 5) {
      e = cudaMemcpy(out_host, d, rows * 5 * sizeof(int32_t), cudaMemcpyDeviceToHost);
    } else {  // drop the part column: a strided 2-D copy of 4 of every 5 int32
      e = cudaMemcpy2D(out_host, 4 * sizeof(int32_t), d, 5 * sizeof(int32_t), 4 * sizeof(int32_t),
                       rows, cudaMemcpyDeviceToHost);
    }
  }
  cudaError_t e2 = cudaFree(d);
  if (e != cudaSuccess) return fail_cuda("tile schedule", e);
  if (e2 != cudaSuccess) return fail_cuda("cudaFree", e2);
  return static_cast<int>(rows);
}

int check_schedule_args(int m_blocks, int n_blocks, int num_sms, int group, const void* out) {
  if (m_blocks < 1 || n_blocks < 1 || num_sms < 1 || group < 1)
    return fail(TG_ERR_ARG, "m_blocks, n_blocks, num_sms and group must be >= 1");
  if (int64_t(m_blocks) * n_blocks > (int64_t(1) << 30)) return fail(TG_ERR_ARG, "too many tiles");
  if (!out) return fail(TG_ERR_ARG, "null output buffer");
  return TG_OK;
}

int tg_tile_schedule(int m_blocks, int n_blocks, int num_sms, int group, int32_t* out_host) {
  int rc = check_schedule_args(m_blocks, n_blocks, num_sms, group, out_host);
  if (rc != TG_OK) return rc;
  const uint32_t tiles = uint32_t(m_blocks) * uint32_t(n_blocks);
  return schedule_rows(m_blocks, n_blocks, num_sms, group, tiles, tiles, 0, 4, out_host);
}

int tg_tile_schedule_ex(int m_blocks, int n_blocks, int num_sms, int group, int flags,
                        int32_t* out_host) {
  int rc = check_schedule_args(m_blocks, n_blocks, num_sms, group, out_host);
  if (rc != TG_OK) return rc;
  if (flags & ~(TG_SCHEDULE_SPLIT_TAIL | TG_SCHEDULE_COLUMN_MAJOR))
    return fail(TG_ERR_ARG, "unknown schedule flags 0x%x", flags);
  const uint32_t tiles = uint32_t(m_blocks) * uint32_t(n_blocks);
  uint32_t first = tiles, units = tiles;
  if (flags & TG_SCHEDULE_SPLIT_TAIL)
    tg::PersistentTileScheduler::tail_split(tiles, uint32_t(num_sms), first, units);
  return schedule_rows(m_blocks, n_blocks, num_sms, group, first, units,
                       (flags & TG_SCHEDULE_COLUMN_MAJOR) ? 1u : 0u, 5, out_host);
}

int tg_tile_schedule_noalloc(int m_blocks, int n_blocks, int num_sms, int group, int flags,
                             int32_t* out_host) {
  int rc = check_schedule_args(m_blocks, n_blocks, num_sms, group, out_host);
  if (rc != TG_OK) return rc;
  if (flags & ~(TG_SCHEDULE_SPLIT_TAIL | TG_SCHEDULE_COLUMN_MAJOR))
    return fail(TG_ERR_ARG, "unknown schedule flags 0x%x", flags);
  const uint32_t tiles = uint32_t(m_blocks) * uint32_t(n_blocks);
  uint32_t first = tiles, units = tiles;
  if (flags & TG_SCHEDULE_SPLIT_TAIL)
    tg::PersistentTileScheduler::tail_split(tiles, uint32_t(num_sms), first, units);
  if (units > TG_SCHEDULE_NOALLOC_MAX_UNITS)
    return fail(TG_ERR_ARG,
                "tg_tile_schedule_noalloc: %u units exceed its fixed scratch of %d units "
                "(use tg_tile_schedule_ex)",
                units, TG_SCHEDULE_NOALLOC_MAX_UNITS);
  std::lock_guard<std::mutex> lock(g_schedule_scratch_mu);
  int32_t* scratch = nullptr;   // the array's address in the current device's context
  cudaError_t e = cudaGetSymbolAddress((void**)&scratch, g_schedule_scratch);
  if (e != cudaSuccess) return fail_cuda("address of the schedule scratch", e);
  e = tg::launch_tile_schedule(uint32_t(m_blocks), uint32_t(n_blocks), uint32_t(num_sms),
                               uint32_t(group), first, units,
                               (flags & TG_SCHEDULE_COLUMN_MAJOR) ? 1u : 0u, scratch, nullptr);
  if (e != cudaSuccess) return fail_cuda("tile schedule", e);
  e = cudaMemcpy(out_host, scratch, uint64_t(units) * 5 * sizeof(int32_t), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail_cuda("copy of the schedule to the host", e);
  return static_cast<int>(units);
}

const char* tg_last_error(void) { return g_err; }

int tg_gemm_config(int* block_m, int* block_n, int* block_k, int* stages, int* group) {
  if (block_m) *block_m = tg::kBM;
  if (block_n) *block_n = tg::kBN;
  if (block_k) *block_k = tg::kBK;
  if (stages) *stages = tg::kStages;
  if (group) *group = tg::kGroup;
  return TG_OK;
}

int tg_device_status(void* stream) {
  unsigned int st = 0;
  cudaError_t e = tg::read_and_clear_watchdog_status(&st, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda("tg_device_status", e);
  if (st) return fail(TG_ERR_TIMEOUT, "watchdog fired (roles 0x%x)", st);
  return TG_OK;
}

int tg_gemm_persistent_host(const void* A_host, const void* B_host, void* C_host, void* A_dev,
                            void* B_dev, void* C_dev, int64_t M, int64_t N, int64_t K, int dtype,
                            void* stream) {
  bool nothing = false;
  int rc = validate(A_dev, B_dev, C_dev, M, N, K, dtype, &nothing);
  if (rc != TG_OK || nothing) return rc;
  if (!C_host || (K > 0 && (!A_host || !B_host))) return fail(TG_ERR_ARG, "null host pointer");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (K > 0) {
    if ((e = cudaMemcpyAsync(A_dev, A_host, uint64_t(M) * K * tg::kElemBytes,
                             cudaMemcpyHostToDevice, s)) != cudaSuccess)
      return fail_cuda("copy of A to the device", e);
    if ((e = cudaMemcpyAsync(B_dev, B_host, uint64_t(K) * N * tg::kElemBytes,
                             cudaMemcpyHostToDevice, s)) != cudaSuccess)
      return fail_cuda("copy of B to the device", e);
  }
  if ((rc = tg_gemm_persistent(A_dev, B_dev, C_dev, M, N, K, dtype, stream)) != TG_OK) return rc;
  if ((e = cudaMemcpyAsync(C_host, C_dev, uint64_t(M) * N * tg::kElemBytes,
                           cudaMemcpyDeviceToHost, s)) != cudaSuccess)
    return fail_cuda("copy of C to the host", e);
  return TG_OK;
}

}  // extern "C"
