// moe_routing.cu -- the steps on either side of the grouped expert MLP: dispatch (sort the
// router's (token, slot) choices by expert) and combine (sum each token's expert outputs).
//
// Page "Efficient MoE training for biological foundation models", Key technical approaches,
// item 1: GroupedLinear works on tokens gathered per expert with per-expert counts
// (split_sizes); section "Dense vs. MoE scaling": each token activates a small subset of the
// experts.  The router itself (a small GEMM + top-k) is outside this library: its choices come
// in as expert ids [T, k].
//
// Dispatch is a stable counting sort on the device, so split_sizes never visit the host:
//   k_permute_count    per chunk of 1024 (token, slot) pairs: per-expert counts (shared atomics)
//   k_permute_scan     one block: per expert, running offsets over chunks; split_sizes; expert
//                      offsets (exclusive scan)
//   k_permute_scatter  per chunk, one warp walks the chunk in order 32 pairs at a time; pairs
//                      with the same expert in a group are ranked with __match_any_sync, so the
//                      rows of every expert keep (token, slot) order.
// Combine is HBM-bound: each thread sums 8 consecutive columns of a token's k rows in fp32 and
// writes them back as bf16 with one 16-byte store.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "mx_device.cuh"
#include "mx_internal.h"
#include "mxfp8moe.h"

namespace mx {
namespace {

constexpr int PERMUTE_CHUNK = 1024;
constexpr int MAX_E = 1024;

__global__ void __launch_bounds__(256) k_permute_count(const int32_t* experts, int64_t n, int E, int32_t* counts,
                                                       uint32_t* err) {
  __shared__ int hist[MAX_E];
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int64_t base = static_cast<int64_t>(blockIdx.x) * PERMUTE_CHUNK;
  for (int i = threadIdx.x; i < PERMUTE_CHUNK; i += blockDim.x) {
    const int64_t idx = base + i;
    if (idx < n) {
      const int e = experts[idx];
      if (e >= 0 && e < E) atomicAdd(&hist[e], 1);
      else atomicOr(err, ERR_EXPERT_RANGE);
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) counts[static_cast<int64_t>(blockIdx.x) * E + e] = hist[e];
}

// counts[c][e] -> first sorted row of chunk c's pairs of expert e.
__global__ void __launch_bounds__(1024) k_permute_scan(int32_t* counts, int nchunks, int E, int32_t* split_sizes) {
  __shared__ int s_tot[MAX_E];
  const int e = threadIdx.x;
  int total = 0;
  if (e < E) {
    for (int c = 0; c < nchunks; ++c) {
      const int v = counts[static_cast<int64_t>(c) * E + e];
      counts[static_cast<int64_t>(c) * E + e] = total;
      total += v;
    }
    split_sizes[e] = total;
  }
  s_tot[e] = e < E ? total : 0;
  __syncthreads();
  for (int d = 1; d < MAX_E; d <<= 1) {   // inclusive scan of expert totals
    const int a = e >= d ? s_tot[e - d] : 0;
    __syncthreads();
    s_tot[e] += a;
    __syncthreads();
  }
  if (e < E) {
    const int start = s_tot[e] - total;   // exclusive
    for (int c = 0; c < nchunks; ++c) counts[static_cast<int64_t>(c) * E + e] += start;
  }
}

__global__ void __launch_bounds__(32) k_permute_scatter(const int32_t* experts, const float* gates, int64_t n, int k,
                                                        int E, const int32_t* chunk_base, int32_t* row_of_slot,
                                                        int32_t* token_of_row, float* gates_sorted) {
  __shared__ int next_row[MAX_E];
  const int lane = threadIdx.x;
  for (int e = lane; e < E; e += 32) next_row[e] = chunk_base[static_cast<int64_t>(blockIdx.x) * E + e];
  __syncwarp();
  const int64_t base = static_cast<int64_t>(blockIdx.x) * PERMUTE_CHUNK;
  for (int g = 0; g < PERMUTE_CHUNK; g += 32) {
    const int64_t idx = base + g + lane;
    const bool in = idx < n;
    const int e = in ? experts[idx] : -1;
    const bool ok = in && e >= 0 && e < E;
    const uint32_t same = __match_any_sync(0xFFFFFFFFu, ok ? e : -1);
    const uint32_t lower = same & ((1u << lane) - 1u);
    if (ok) {
      const int row = next_row[e] + __popc(lower);
      row_of_slot[idx] = row;
      token_of_row[row] = static_cast<int32_t>(idx / k);
      if (gates) gates_sorted[row] = gates[idx];
    }
    __syncwarp();
    // the highest lane of each expert group advances that expert's counter
    if (ok && (same >> lane) == 1u) next_row[e] += __popc(same);
    __syncwarp();
  }
}

__device__ __forceinline__ void add8(float* acc, const uint4 w) {
  acc[0] += bf16_lo(w.x); acc[1] += bf16_hi(w.x);
  acc[2] += bf16_lo(w.y); acc[3] += bf16_hi(w.y);
  acc[4] += bf16_lo(w.z); acc[5] += bf16_hi(w.z);
  acc[6] += bf16_lo(w.w); acc[7] += bf16_hi(w.w);
}

// out[t, :] = sum_j y[row_of_slot[t, j], :]; one CTA per (token, 2048 columns).
constexpr int COMBINE_THREADS = 256;
// Row ids outside [0, T*k) contribute nothing.
__global__ void __launch_bounds__(COMBINE_THREADS) k_combine(const uint16_t* y, const int32_t* row_of_slot, int k,
                                                             int64_t H, int64_t nrows, uint16_t* out) {
  const int64_t t = blockIdx.x;
  const int64_t col = (static_cast<int64_t>(blockIdx.y) * COMBINE_THREADS + threadIdx.x) * 8;
  if (col >= H) return;
  float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  for (int j = 0; j < k; ++j) {
    const int64_t r = __ldg(row_of_slot + t * k + j);
    if (r < 0 || r >= nrows) continue;
    add8(acc, __ldcs(reinterpret_cast<const uint4*>(y + r * H + col)));
  }
  uint4 o;
  o.x = pack_bf16x2(acc[0], acc[1]);
  o.y = pack_bf16x2(acc[2], acc[3]);
  o.z = pack_bf16x2(acc[4], acc[5]);
  o.w = pack_bf16x2(acc[6], acc[7]);
  __stcs(reinterpret_cast<uint4*>(out + t * H + col), o);
}

// dst[i, :] = src[index[i], :] for rows of `words` 32-bit words (zeros where index[i] is outside
// [0, nsrc)); a pure copy, so any element type travels bit for bit.  One thread per 16 bytes
// when rows are whole 16-byte chunks, else per word.
template <bool VEC>
__global__ void __launch_bounds__(256) k_gather_rows(const uint32_t* src, int64_t nsrc, int64_t words,
                                                     const int32_t* index, int64_t n, uint32_t* dst) {
  const int64_t per_row = VEC ? words / 4 : words;
  const int64_t total = n * per_row;
  for (int64_t q = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; q < total;
       q += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t i = q / per_row, c = q - i * per_row;
    const int64_t r = __ldg(index + i);
    const bool in = r >= 0 && r < nsrc;
    if (VEC) {
      const uint4 v = in ? __ldg(reinterpret_cast<const uint4*>(src + r * words) + c) : make_uint4(0u, 0u, 0u, 0u);
      reinterpret_cast<uint4*>(dst + i * words)[c] = v;
    } else {
      dst[i * words + c] = in ? __ldg(src + r * words + c) : 0u;
    }
  }
}

}  // namespace

cudaError_t launch_gather_rows(const void* src, int64_t nsrc, int64_t row_bytes, const int32_t* index, int64_t n,
                               void* dst, int sms, cudaStream_t stream) {
  const int64_t words = row_bytes / 4;
  const bool vec = row_bytes % 16 == 0 && (reinterpret_cast<uintptr_t>(src) & 15u) == 0 &&
                   (reinterpret_cast<uintptr_t>(dst) & 15u) == 0;
  const int64_t items = n * (vec ? words / 4 : words);
  const int64_t blocks = std::min<int64_t>((items + 255) / 256, static_cast<int64_t>(sms) * 8);
  if (blocks <= 0) return cudaSuccess;
  if (vec)
    k_gather_rows<true><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(static_cast<const uint32_t*>(src), nsrc,
                                                                           words, index, n, static_cast<uint32_t*>(dst));
  else
    k_gather_rows<false><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(static_cast<const uint32_t*>(src), nsrc,
                                                                            words, index, n, static_cast<uint32_t*>(dst));
  return cudaGetLastError();
}

size_t permute_workspace_bytes(int64_t n, int E) {
  const int64_t nchunks = (n + PERMUTE_CHUNK - 1) / PERMUTE_CHUNK;
  return 256 + static_cast<size_t>(nchunks) * E * sizeof(int32_t);
}

cudaError_t launch_permute(const int32_t* experts, const float* gates, int64_t T, int k, int E,
                           int32_t* split_sizes, int32_t* row_of_slot, int32_t* token_of_row, float* gates_sorted,
                           void* workspace, cudaStream_t stream) {
  const int64_t n = T * k;
  uint32_t* err = static_cast<uint32_t*>(workspace);
  int32_t* counts = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) + 256);
  const int nchunks = static_cast<int>((n + PERMUTE_CHUNK - 1) / PERMUTE_CHUNK);
  cudaError_t e = cudaMemsetAsync(err, 0, sizeof(uint32_t), stream);
  if (e != cudaSuccess) return e;
  if (nchunks == 0) {
    e = cudaMemsetAsync(split_sizes, 0, sizeof(int32_t) * E, stream);
    return e;
  }
  k_permute_count<<<nchunks, 256, 0, stream>>>(experts, n, E, counts, err);
  k_permute_scan<<<1, 1024, 0, stream>>>(counts, nchunks, E, split_sizes);
  k_permute_scatter<<<nchunks, 32, 0, stream>>>(experts, gates, n, k, E, counts, row_of_slot, token_of_row,
                                                gates_sorted);
  return cudaGetLastError();
}

cudaError_t launch_combine(const void* y, const int32_t* row_of_slot, int64_t T, int k, int64_t H, void* out,
                           cudaStream_t stream) {
  const dim3 grid(static_cast<unsigned>(T), static_cast<unsigned>((H / 8 + COMBINE_THREADS - 1) / COMBINE_THREADS));
  k_combine<<<grid, COMBINE_THREADS, 0, stream>>>(static_cast<const uint16_t*>(y), row_of_slot, k, H, T * k,
                                                  static_cast<uint16_t*>(out));
  return cudaGetLastError();
}

}  // namespace mx
