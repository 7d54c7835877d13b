// mma_peak.cu -- the rate of the block-scaled tensor-core instruction the grouped GEMMs are built
// on, measured on the device at hand: the roofline against which their TFLOP/s are reported.
//
// Every cluster of two CTAs (one per SM) keeps one A tile (its 128 rows x 128 K bytes), its half
// of a 256-row B tile and the scale atoms of one K step resident in shared memory, copies the
// scales into TMEM once, and then issues `iters` K steps of four pair MMAs (M = 256, N = 256)
// back to back into one TMEM accumulator: no data movement, no barrier waits between MMAs, one
// commit at the end.  MXFP8: kind::mxf8f6f4 with E4M3 operands, K = 32 per MMA, one UE8M0 atom
// per 128 rows; NVFP4: kind::mxf4nvf4 with packed E2M1 operands, K = 64 per MMA, one UE4M3 atom per
// 128 rows per MMA.  Operands are a fixed non-zero byte pattern with unit scales (the arithmetic
// is not checked; only the time is used).
#include <cuda_runtime.h>

#include <algorithm>

#include "mx_device.cuh"
#include "mx_internal.h"
#include "mxfp8moe.h"

namespace mx {
namespace {

constexpr int PK_THREADS = 128;
constexpr int PK_A = 0, PK_B = 16384, PK_SF = 32768, PK_BAR = PK_SF + 12 * 512;
// Far more shared memory than the kernel uses, so that no two CTAs share an SM (each allocates
// all 512 TMEM columns).
constexpr int PK_SMEM = 200 * 1024;
constexpr uint64_t kPeakWaitNs = 10000000000ull;   // 10 s: the host caps a launch well below

template <bool NV>
__global__ void __launch_bounds__(PK_THREADS, 1) k_mma_peak(int64_t iters, uint32_t* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* done = reinterpret_cast<uint64_t*>(smem + PK_BAR);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(done + 1);
  const int warp = threadIdx.x >> 5;
  const bool leader = cluster_cta_rank() == 0;

  // operands: bytes 0x00..0x76 (finite E4M3 codes, no NaN; as E2M1 pairs any byte is finite),
  // scale bytes 0x7F (UE8M0 2^0) or 0x38 (UE4M3 1.0)
  for (int i = threadIdx.x; i < PK_SF / 16; i += PK_THREADS) {
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t b = static_cast<uint32_t>(16 * i + 4 * j);
      w[j] = ((b * 29u + 7u) & 0x76u) | ((((b + 1) * 29u + 7u) & 0x76u) << 8) |
             ((((b + 2) * 29u + 7u) & 0x76u) << 16) | ((((b + 3) * 29u + 7u) & 0x76u) << 24);
    }
    *reinterpret_cast<uint4*>(smem + 16 * i) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  const uint32_t one4 = NV ? 0x38383838u : 0x7F7F7F7Fu;
  for (int i = threadIdx.x; i < 12 * 512 / 16; i += PK_THREADS)
    *reinterpret_cast<uint4*>(smem + PK_SF + 16 * i) = make_uint4(one4, one4, one4, one4);
  fence_proxy_async_smem();   // the tensor core reads these through the async proxy
  if (threadIdx.x == 0) {
    mbar_init(done, 1);
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc_pair(tmem_holder, 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();   // both CTAs' operands and barriers are in place
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (leader && threadIdx.x == 0) {
    const uint32_t a0 = smem_u32(smem + PK_A), b0 = smem_u32(smem + PK_B), sf0 = smem_u32(smem + PK_SF);
    if constexpr (NV) {   // MMA k: A atom at column 256 + 4k, B atoms at 272 + 8k (+4)
      for (int a = 0; a < 4; ++a) {
        tc_copy_sf_pair(tmem + 256 + 4 * a, sdesc_sf_atom(sf0 + 512 * a));
        tc_copy_sf_pair(tmem + 272 + 8 * a, sdesc_sf_atom(sf0 + 512 * (4 + a)));
        tc_copy_sf_pair(tmem + 276 + 8 * a, sdesc_sf_atom(sf0 + 512 * (8 + a)));
      }
      const uint32_t idesc = idesc_nvf4(256, 256);
      for (int64_t i = 0; i < iters; ++i) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
          tc_mma_nvf4_pair(tmem, sdesc_kmajor_sw128(a0 + 32 * k), sdesc_kmajor_sw128(b0 + 32 * k), idesc,
                           tmem + 256 + 4 * k, tmem + 272 + 8 * k, (i | k) != 0 ? 1u : 0u);
      }
    } else {
      tc_copy_sf_pair(tmem + 256, sdesc_sf_atom(sf0));
      tc_copy_sf_pair(tmem + 260, sdesc_sf_atom(sf0 + 512));
      tc_copy_sf_pair(tmem + 264, sdesc_sf_atom(sf0 + 1024));
      const uint32_t idesc = idesc_mxf8_e4m3(256, 256);
      for (int64_t i = 0; i < iters; ++i) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
          tc_mma_mxf8_pair(tmem, sdesc_kmajor_sw128(a0 + 32 * k), sdesc_kmajor_sw128(b0 + 32 * k),
                           idesc_with_sf_id(idesc, k), tmem + 256, tmem + 260, (i | k) != 0 ? 1u : 0u);
      }
    }
    tc_commit_pair_both(done);
  }
  // every MMA writes both CTAs' TMEM: each CTA waits for the commit before it frees TMEM
  if (threadIdx.x == 0 && iters > 0 && !mbar_wait_bounded(done, 0, nullptr, kPeakWaitNs))
    atomicOr(err, ERR_TIMEOUT_DRAIN);
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
}

}  // namespace
}  // namespace mx

using namespace mx;

extern "C" int mxfp8_mma_peak(int64_t iters, int format, void* workspace, int* clusters, void* stream) {
  if (iters < 0 || iters > (int64_t(1) << 24) || workspace == nullptr || clusters == nullptr ||
      (reinterpret_cast<uintptr_t>(workspace) & 3u) != 0 || (format != 0 && format != 1))
    return MXFP8_ERR_INVALID_ARG;
  const auto kernel = format == 1 ? k_mma_peak<true> : k_mma_peak<false>;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, PK_SMEM) != cudaSuccess)
    return MXFP8_ERR_CUDA;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(PK_THREADS, 1, 1);
  cfg.dynamicSmemBytes = PK_SMEM;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(2, 1, 1);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess || n <= 0) return MXFP8_ERR_CUDA;
  cfg.gridDim = dim3(2 * n, 1, 1);
  if (cudaMemsetAsync(workspace, 0, sizeof(uint32_t), cfg.stream) != cudaSuccess) return MXFP8_ERR_CUDA;
  if (cudaLaunchKernelEx(&cfg, kernel, iters, static_cast<uint32_t*>(workspace)) != cudaSuccess)
    return MXFP8_ERR_CUDA;
  *clusters = n;
  return MXFP8_OK;
}
