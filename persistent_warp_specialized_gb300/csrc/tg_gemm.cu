// tg_gemm.cu -- instantiations and launchers of the sm_103a kernels behind the C ABI:
// the persistent warp-specialized GEMM (fp16 and bf16, product and debug builds; single CTA,
// CTA pair and wide CTA pair), the
// block-scaled MXFP8 GEMM (single CTA and CTA pair), the tile-schedule inspection kernel, and the zero fill used when
// K == 0.  All kernels share this translation unit's watchdog status word.
#include <utility>

#include "tg_gemm_kernel.cuh"
#include "tg_gemm_pair_kernel.cuh"
#include "tg_gemm_pair_wide_kernel.cuh"
#include "tg_internal.h"
#include "tg_mx_kernel.cuh"
#include "tg_mx_pack.cuh"
#include "tg_mx_pair_kernel.cuh"

namespace tg {

namespace {

// One thread per worker runs the scheduler the GEMM roles run and writes its rows
// (worker, w, bx, by); rows are ordered by worker, then w.  Worker c owns
// q + (c < r) tiles where total = q * P + r, so its first row is c * q + min(c, r).
__global__ void tile_schedule_kernel(uint32_t m_blocks, uint32_t n_blocks, uint32_t num_workers,
                                     uint32_t group, uint32_t split_from, uint32_t units,
                                     uint32_t column_major, int32_t* __restrict__ out) {
  const uint32_t c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= num_workers) return;
  const uint32_t q = units / num_workers;
  const uint32_t r = units % num_workers;
  uint64_t row = static_cast<uint64_t>(c) * q + (c < r ? c : r);
  PersistentTileScheduler sched(m_blocks, n_blocks, group, num_workers, split_from, units,
                                column_major);
  sched.init(c);
  while (sched.valid()) {
    int32_t* o = out + 5 * row;
    o[0] = static_cast<int32_t>(c);
    o[1] = static_cast<int32_t>(sched.current_iter);
    o[2] = static_cast<int32_t>(sched.m_idx);
    o[3] = static_cast<int32_t>(sched.n_idx);
    o[4] = sched.part;
    ++row;
    sched.next_tile();
  }
}

__global__ void zero_fill_kernel(uint4* __restrict__ dst, uint64_t n16) {
  const uint64_t stride = static_cast<uint64_t>(gridDim.x) * blockDim.x;
  for (uint64_t i = static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16;
       i += stride)
    dst[i] = make_uint4(0u, 0u, 0u, 0u);
}

GemmParams params_of(const GemmLaunch& l) {
  GemmParams p;
  p.C = l.C;
  p.M = l.M;
  p.N = l.N;
  p.K = l.K;
  p.m_blocks = l.m_blocks;
  p.n_blocks = l.n_blocks;
  p.k_blocks = l.k_blocks;
  p.group = l.group;
  p.split_from = l.split_from;
  p.column_major = l.column_major;
  p.dynamic = l.dynamic;
  p.epi_direct = l.epi_direct;
  p.total_units = l.total_units;
  p.watchdog_ns = l.watchdog_ns;
  p.trace = l.trace;
  p.inject_skip_phase = l.inject_skip_phase;
  p.sk_tiles = l.sk_tiles;
  p.sk_epoch = l.sk_epoch;
  p.sk_slot_f4 = l.sk_slot_f4;
  p.sk_flags = l.sk_flags;
  p.sk_partials = l.sk_partials;
  return p;
}

// Launches ``kernel`` with programmatic stream serialization: it may be scheduled while the
// previous kernel in the stream is still finishing (as that kernel's CTAs exit).  Every kernel
// launched this way issues griddepcontrol.wait before its first global memory access, so the
// stream's ordering of memory effects is unchanged; what overlaps is the launch itself and each
// CTA's set-up (barriers, TMEM allocation, descriptor prefetch).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, uint32_t threads, size_t smem,
                       cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

template <int DT, bool DEBUG>
cudaError_t launch_one(const GemmLaunch& l, cudaStream_t stream) {
  return launch_pdl(gemm_persistent_ws_kernel<DT, DEBUG>, l.grid, kThreads, kSmemBytes, stream,
                    l.tmA, l.tmB, l.tmC, params_of(l));
}

template <int DT, bool DEBUG>
cudaError_t launch_pair(const GemmLaunch& l, cudaStream_t stream) {
  return launch_pdl(gemm_pair_ws_kernel<DT, DEBUG>, l.grid, kThreads, kPairSmemBytes, stream,
                    l.tmA, l.tmB, l.tmC, params_of(l));
}

template <int DT, bool DEBUG>
cudaError_t launch_pair_wide(const GemmLaunch& l, cudaStream_t stream) {
  return launch_pdl(gemm_pair_wide_ws_kernel<DT, DEBUG>, l.grid, kThreads, kWideSmemBytes, stream,
                    l.tmA, l.tmB, l.tmC, params_of(l));
}

template <int DT, bool DEBUG>
cudaError_t set_smem_attr() {
  cudaError_t e = cudaFuncSetAttribute(gemm_persistent_ws_kernel<DT, DEBUG>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(gemm_pair_ws_kernel<DT, DEBUG>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kPairSmemBytes));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(gemm_pair_wide_ws_kernel<DT, DEBUG>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(kWideSmemBytes));
}

MxParams mx_params_of(const MxLaunch& l) {
  MxParams p;
  p.SFA = static_cast<const uint8_t*>(l.SFA);
  p.SFB = static_cast<const uint8_t*>(l.SFB);
  p.M = l.M;
  p.N = l.N;
  p.K = l.K;
  p.sfa_blocks = l.sfa_blocks;
  p.sfb_blocks = l.sfb_blocks;
  p.m_blocks = l.m_blocks;
  p.n_blocks = l.n_blocks;
  p.k_blocks = l.k_blocks;
  p.group = l.group;
  p.split_from = l.split_from;
  p.total_units = l.total_units;
  p.column_major = l.column_major;
  p.watchdog_ns = l.watchdog_ns;
  p.trace = l.trace;
  p.inject_skip_phase = l.inject_skip_phase;
  return p;
}

template <int OUT, bool DEBUG>
cudaError_t launch_mx(const MxLaunch& l, cudaStream_t stream) {
  return launch_pdl(gemm_mxfp8_ws_kernel<OUT, DEBUG>, l.grid, kThreads, kMxSmemBytes, stream,
                    l.tmA, l.tmB, l.tmC, mx_params_of(l));
}

template <int OUT, bool DEBUG>
cudaError_t launch_mx_pair(const MxLaunch& l, cudaStream_t stream) {
  return launch_pdl(gemm_mxfp8_pair_ws_kernel<OUT, DEBUG>, l.grid, kThreads, kMxPairSmemBytes,
                    stream, l.tmA, l.tmB, l.tmC, l.tmSFA, l.tmSFB, mx_params_of(l));
}

template <int OUT, bool DEBUG>
cudaError_t set_mx_smem_attr() {
  cudaError_t e = cudaFuncSetAttribute(gemm_mxfp8_ws_kernel<OUT, DEBUG>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kMxSmemBytes));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(gemm_mxfp8_pair_ws_kernel<OUT, DEBUG>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(kMxPairSmemBytes));
}

}  // namespace

cudaError_t prepare_gemm_kernels(int* max_pairs) {
  cudaError_t e;
  if ((e = set_smem_attr<0, false>()) != cudaSuccess) return e;
  if ((e = set_smem_attr<1, false>()) != cudaSuccess) return e;
  if ((e = set_smem_attr<0, true>()) != cudaSuccess) return e;
  if ((e = set_smem_attr<1, true>()) != cudaSuccess) return e;
  if ((e = set_mx_smem_attr<0, false>()) != cudaSuccess) return e;
  if ((e = set_mx_smem_attr<1, false>()) != cudaSuccess) return e;
  if ((e = set_mx_smem_attr<0, true>()) != cudaSuccess) return e;
  if ((e = set_mx_smem_attr<1, true>()) != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kPairSmemBytes;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int clusters = 0, mx_clusters = 0, wide_clusters = 0;
  e = cudaOccupancyMaxActiveClusters(&clusters, gemm_pair_ws_kernel<1, false>, &cfg);
  if (e != cudaSuccess) return e;
  cfg.dynamicSmemBytes = kWideSmemBytes;
  e = cudaOccupancyMaxActiveClusters(&wide_clusters, gemm_pair_wide_ws_kernel<1, false>, &cfg);
  if (e != cudaSuccess) return e;
  if (wide_clusters < clusters) clusters = wide_clusters;
  cfg.dynamicSmemBytes = kMxPairSmemBytes;
  e = cudaOccupancyMaxActiveClusters(&mx_clusters, gemm_mxfp8_pair_ws_kernel<1, false>, &cfg);
  if (e != cudaSuccess) return e;
  *max_pairs = clusters < mx_clusters ? clusters : mx_clusters;
  return cudaSuccess;
}

cudaError_t launch_gemm(int dtype, bool debug, int variant, const GemmLaunch& l,
                        cudaStream_t stream) {
  if (variant == kVariantPair) {
    if (dtype == 0)
      return debug ? launch_pair<0, true>(l, stream) : launch_pair<0, false>(l, stream);
    return debug ? launch_pair<1, true>(l, stream) : launch_pair<1, false>(l, stream);
  }
  if (variant == kVariantPairWide) {
    if (dtype == 0)
      return debug ? launch_pair_wide<0, true>(l, stream) : launch_pair_wide<0, false>(l, stream);
    return debug ? launch_pair_wide<1, true>(l, stream) : launch_pair_wide<1, false>(l, stream);
  }
  if (dtype == 0) return debug ? launch_one<0, true>(l, stream) : launch_one<0, false>(l, stream);
  return debug ? launch_one<1, true>(l, stream) : launch_one<1, false>(l, stream);
}

cudaError_t launch_mxfp8(int out_dtype, bool debug, int variant, const MxLaunch& l,
                         cudaStream_t stream) {
  if (variant == kVariantPair) {
    if (out_dtype == 0)
      return debug ? launch_mx_pair<0, true>(l, stream) : launch_mx_pair<0, false>(l, stream);
    return debug ? launch_mx_pair<1, true>(l, stream) : launch_mx_pair<1, false>(l, stream);
  }
  if (out_dtype == 0) return debug ? launch_mx<0, true>(l, stream) : launch_mx<0, false>(l, stream);
  return debug ? launch_mx<1, true>(l, stream) : launch_mx<1, false>(l, stream);
}

cudaError_t launch_mx_pack(const void* sf, void* out, uint32_t rows, uint32_t k_blocks,
                           uint32_t row_blocks, cudaStream_t stream) {
  if (k_blocks == 0 || row_blocks == 0) return cudaSuccess;
  const uint32_t groups = (k_blocks + kMxPackKb - 1) / kMxPackKb;
  const dim3 grid(row_blocks, groups < 65535u ? groups : 65535u);   // the kernel strides over y
  return launch_pdl(mx_pack_scales_kernel, grid, kMxPackThreads, 0, stream,
                    static_cast<const uint8_t*>(sf), static_cast<uint8_t*>(out), rows, k_blocks,
                    row_blocks);
}

cudaError_t launch_zero_fill(void* C, uint64_t bytes, cudaStream_t stream) {
  const uint64_t n16 = bytes / 16;
  if (n16 == 0) return cudaSuccess;
  uint64_t blocks = (n16 + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  zero_fill_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(static_cast<uint4*>(C), n16);
  return cudaGetLastError();
}

cudaError_t launch_tile_schedule(uint32_t m_blocks, uint32_t n_blocks, uint32_t num_workers,
                                 uint32_t group, uint32_t split_from, uint32_t units,
                                 uint32_t column_major, int32_t* out_dev, cudaStream_t stream) {
  const uint32_t threads = 128;
  const uint32_t blocks = (num_workers + threads - 1) / threads;
  tile_schedule_kernel<<<blocks, threads, 0, stream>>>(m_blocks, n_blocks, num_workers, group,
                                                       split_from, units, column_major, out_dev);
  return cudaGetLastError();
}

cudaError_t clear_watchdog_status(cudaStream_t stream) {
  const unsigned int zero = 0;
  return cudaMemcpyToSymbolAsync(g_watchdog_status, &zero, sizeof(zero), 0,
                                 cudaMemcpyHostToDevice, stream);
}

cudaError_t read_and_clear_watchdog_status(unsigned int* out, cudaStream_t stream) {
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return e;
  e = cudaMemcpyFromSymbol(out, g_watchdog_status, sizeof(*out));
  if (e != cudaSuccess) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_watchdog_status, &zero, sizeof(zero));
}

}  // namespace tg
