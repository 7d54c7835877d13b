// nvfp4.cu -- the NVFP4 variant of the expert-MLP chain: tensor amax, NVFP4 quantization, and the
// extern "C" entry points of the NVFP4 forward.
//
// The Llama 3 recipe page ("TransformerEngine-accelerated Llama 3 training with native PyTorch
// training loop") names NVFP4 beside MXFP8 as a quantized-training recipe (feature table; section
// "Quantized Training (FP8 / MXFP8 / NVFP4)") without defining it; this library takes NVIDIA's
// published NVFP4: E2M1 elements, one E4M3 scale per 16 consecutive values, and a per-tensor
// binary32 encode scale s_enc = 448 * 6 / amax (1 for an all-zero tensor).  A block is quantized
// as S = E4M3(fl32(fl32(amax_block / 6) * s_enc)), r = fl32(s_enc / S) (0 if S = 0), code_i =
// E2M1(fl32(v_i * r)): every rounding explicit, in binary32, round to nearest even, saturating.
//
// Quantization is two kernels: k_nv_amax reduces max|x| over the whole tensor (one read of x),
// k_nv_quantize reads it back and quantizes one 16-value block per thread (32 bytes of bf16 in,
// 8 bytes of codes and 1 scale byte out; a warp moves 1 KB contiguous).
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "mx_device.cuh"
#include "mx_internal.h"
#include "mxfp8moe.h"

namespace mx {
namespace {

constexpr int NV_AMAX_THREADS = 256;
constexpr int NV_Q_THREADS = 128;

// max |x| of a bf16 tensor of n8 * 8 values, as float bits, atomically max-ed into *out (which
// holds 0 or a previous maximum).  Cleared sign bits make every bf16 a non-negative number whose
// bit pattern orders like its value, so the maximum is taken on 16-bit integers.
__global__ void __launch_bounds__(NV_AMAX_THREADS) k_nv_amax(const uint4* x, int64_t n8, uint32_t* out) {
  uint32_t m = 0;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * NV_AMAX_THREADS + threadIdx.x; i < n8;
       i += static_cast<int64_t>(gridDim.x) * NV_AMAX_THREADS) {
    const uint4 w = __ldcs(x + i);
    m = __vmaxu2(m, __vmaxu2(__vmaxu2(w.x & 0x7FFF7FFFu, w.y & 0x7FFF7FFFu), __vmaxu2(w.z & 0x7FFF7FFFu,
                                                                                       w.w & 0x7FFF7FFFu)));
  }
  m = max(m & 0xFFFFu, m >> 16) << 16;   // the larger half, as float bits
  m = __reduce_max_sync(0xFFFFFFFFu, m);
  __shared__ uint32_t s_max[NV_AMAX_THREADS / 32];
  if ((threadIdx.x & 31) == 0) s_max[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < NV_AMAX_THREADS / 32; ++w) m = max(m, s_max[w]);
    atomicMax(out, m);
  }
}

struct NvQuantArgs {
  const uint16_t* x;
  int64_t M, K;           // source rows and columns
  uint8_t* q;             // [rows_out, K/2] packed codes
  uint8_t* sf;            // scale codes
  int64_t kt;             // tensor-core layout: atoms per 128-row tile (= 4 * ceil(K/256))
  int64_t nb_out;         // 16-value blocks written per row (tensor-core layout: 16 * ceil(K/256))
  const float* amax;      // the tensor's largest magnitude (device)
  const SchedHeader* meta;  // gather mode only
  int E;
};

// MMA: scale codes in the tensor-core layout (blocks past K, up to the next multiple of 256
// values, get scale 0: the GEMMs read whole 256-value K steps); otherwise compact [M, K/16].
// GATHER: output row p is the expert-padded row space of a grouped MLP (a zero row past the
// expert's count), as in the MXFP8 activation quantize.
// Grid: x = output row, y = chunk of NV_Q_THREADS blocks of that row.
template <bool MMA, bool GATHER>
__global__ void __launch_bounds__(NV_Q_THREADS) k_nv_quantize(const NvQuantArgs a) {
  const int64_t p = blockIdx.x;
  const int64_t kb = static_cast<int64_t>(blockIdx.y) * NV_Q_THREADS + threadIdx.x;
  if (kb >= a.nb_out) return;
  int64_t src = p;
  bool zero = false;
  if constexpr (GATHER) {
    if (p >= a.meta->pad_rows) return;
    const int32_t* row_off = reinterpret_cast<const int32_t*>(a.meta + 1);
    const int32_t* pad_off = row_off + (a.E + 1);
    int lo = 0, hi = a.E;   // largest e with pad_off[e] <= p: the (non-empty) owner of the row
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(pad_off + mid) <= p) lo = mid; else hi = mid;
    }
    const int64_t local = p - __ldg(pad_off + lo);
    zero = local >= __ldg(row_off + lo + 1) - __ldg(row_off + lo);
    src = __ldg(row_off + lo) + local;
  }
  uint32_t sfc = 0;
  if (kb < a.K / 16) {
    const float s_enc = nv_encode_scale(*a.amax);
    uint4 w0 = make_uint4(0u, 0u, 0u, 0u), w1 = w0;
    if (!zero) {
      const uint4* px = reinterpret_cast<const uint4*>(a.x + src * a.K + kb * 16);
      w0 = __ldcs(px);
      w1 = __ldcs(px + 1);
    }
    uint32_t m = __vmaxu2(__vmaxu2(__vmaxu2(w0.x & 0x7FFF7FFFu, w0.y & 0x7FFF7FFFu),
                                   __vmaxu2(w0.z & 0x7FFF7FFFu, w0.w & 0x7FFF7FFFu)),
                          __vmaxu2(__vmaxu2(w1.x & 0x7FFF7FFFu, w1.y & 0x7FFF7FFFu),
                                   __vmaxu2(w1.z & 0x7FFF7FFFu, w1.w & 0x7FFF7FFFu)));
    const float amax = __uint_as_float(max(m & 0xFFFFu, m >> 16) << 16);
    float r;
    sfc = nv_block_scale(amax, s_enc, &r);
    auto c8 = [&](const uint4 w) {
      return e2m1x8(__fmul_rn(bf16_lo(w.x), r), __fmul_rn(bf16_hi(w.x), r), __fmul_rn(bf16_lo(w.y), r),
                    __fmul_rn(bf16_hi(w.y), r), __fmul_rn(bf16_lo(w.z), r), __fmul_rn(bf16_hi(w.z), r),
                    __fmul_rn(bf16_lo(w.w), r), __fmul_rn(bf16_hi(w.w), r));
    };
    __stcs(reinterpret_cast<uint2*>(a.q + p * (a.K / 2) + kb * 8), make_uint2(c8(w0), c8(w1)));
  }
  if constexpr (MMA)
    a.sf[sf_mma_offset(p, kb, a.kt)] = static_cast<uint8_t>(sfc);
  else
    a.sf[p * (a.K / 16) + kb] = static_cast<uint8_t>(sfc);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

cudaError_t launch_amax(const void* x, int64_t n, uint32_t* out, cudaStream_t stream) {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t n8 = n / 8;
  const int64_t want = (n8 + NV_AMAX_THREADS - 1) / NV_AMAX_THREADS;
  const int grid = static_cast<int>(want < 8LL * sms ? (want > 0 ? want : 1) : 8LL * sms);
  k_nv_amax<<<grid, NV_AMAX_THREADS, 0, stream>>>(static_cast<const uint4*>(x), n8, out);
  return cudaGetLastError();
}

}  // namespace

int64_t nv_sf_atoms_per_tile(int64_t K) { return (K + 255) / 256 * 4; }

bool nv_ws_layout(int64_t R, int64_t H, int64_t F, int E, NvWsLayout* out) {
  WsLayout f;
  if (!ws_layout(R, H, F, E, &f)) return false;
  auto al = [](size_t v) { return (v + 255) & ~static_cast<size_t>(255); };
  NvWsLayout L{};
  L.r_pad = f.r_pad;
  L.x_kt = nv_sf_atoms_per_tile(H);
  L.h_kt = nv_sf_atoms_per_tile(F);
  const size_t tiles = static_cast<size_t>(L.r_pad / 128);
  L.meta = 0;
  L.amax = al(sizeof(SchedHeader) + 3 * static_cast<size_t>(E + 1) * sizeof(int32_t));
  L.xq = al(L.amax + 2 * sizeof(uint32_t));
  L.xsf = al(L.xq + static_cast<size_t>(L.r_pad) * (H / 2));
  L.hq = al(L.xsf + tiles * L.x_kt * 512);
  L.hsf = al(L.hq + static_cast<size_t>(L.r_pad) * (F / 2));
  L.total = al(L.hsf + tiles * L.h_kt * 512);
  *out = L;
  return true;
}

cudaError_t launch_nv_amax_quantize_gather(const void* x, int64_t R, int64_t H, const SchedHeader* meta, int E,
                                           int64_t r_pad, uint32_t* amax_word, uint8_t* xq, uint8_t* xsf,
                                           cudaStream_t stream) {
  if (cudaMemsetAsync(amax_word, 0, sizeof(uint32_t), stream) != cudaSuccess) return cudaErrorUnknown;
  if (R > 0 && launch_amax(x, R * H, amax_word, stream) != cudaSuccess) return cudaErrorUnknown;
  NvQuantArgs a{};
  a.x = static_cast<const uint16_t*>(x);
  a.M = R;
  a.K = H;
  a.q = xq;
  a.sf = xsf;
  a.kt = nv_sf_atoms_per_tile(H);
  a.nb_out = 4 * a.kt;
  a.amax = reinterpret_cast<const float*>(amax_word);
  a.meta = meta;
  a.E = E;
  if (r_pad == 0) return cudaSuccess;
  const dim3 grid(static_cast<unsigned>(r_pad), static_cast<unsigned>((a.nb_out + NV_Q_THREADS - 1) / NV_Q_THREADS));
  k_nv_quantize<true, true><<<grid, NV_Q_THREADS, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace mx

using namespace mx;

extern "C" {

size_t nvfp4_sf_bytes(int64_t M, int64_t K, int sf_layout) {
  if (M < 0 || K < 0 || K % 16 != 0) return 0;
  if (sf_layout == MXFP8_SF_COMPACT) return static_cast<size_t>(M) * (K / 16);
  if (sf_layout == MXFP8_SF_MMA) return static_cast<size_t>((M + 127) / 128) * nv_sf_atoms_per_tile(K) * 512;
  return 0;
}

int nvfp4_quantize(const void* x, int64_t M, int64_t K, int sf_layout, uint8_t* q, uint8_t* sf, float* amax,
                   void* stream) {
  if (M < 0 || K < 0 || K % 16 != 0) return MXFP8_ERR_INVALID_ARG;
  if (sf_layout != MXFP8_SF_COMPACT && sf_layout != MXFP8_SF_MMA) return MXFP8_ERR_INVALID_ARG;
  if (sf_layout == MXFP8_SF_MMA && (M % 128 != 0 || K % 128 != 0)) return MXFP8_ERR_UNSUPPORTED;
  if (amax == nullptr || (reinterpret_cast<uintptr_t>(amax) & 3u) != 0) return MXFP8_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (M == 0 || K == 0) {
    return cudaMemsetAsync(amax, 0, sizeof(float), s) == cudaSuccess ? MXFP8_OK : MXFP8_ERR_CUDA;
  }
  if (x == nullptr || q == nullptr || sf == nullptr || !aligned16(x) || !aligned16(q)) return MXFP8_ERR_INVALID_ARG;
  if (M > INT32_MAX) return MXFP8_ERR_UNSUPPORTED;
  if (cudaMemsetAsync(amax, 0, sizeof(float), s) != cudaSuccess) return MXFP8_ERR_CUDA;
  if (launch_amax(x, M * K, reinterpret_cast<uint32_t*>(amax), s) != cudaSuccess) return MXFP8_ERR_CUDA;
  NvQuantArgs a{};
  a.x = static_cast<const uint16_t*>(x);
  a.M = M;
  a.K = K;
  a.q = q;
  a.sf = sf;
  a.kt = nv_sf_atoms_per_tile(K);
  a.nb_out = sf_layout == MXFP8_SF_MMA ? 4 * a.kt : K / 16;
  a.amax = amax;
  const dim3 grid(static_cast<unsigned>(M), static_cast<unsigned>((a.nb_out + NV_Q_THREADS - 1) / NV_Q_THREADS));
  if (sf_layout == MXFP8_SF_MMA)
    k_nv_quantize<true, false><<<grid, NV_Q_THREADS, 0, s>>>(a);
  else
    k_nv_quantize<false, false><<<grid, NV_Q_THREADS, 0, s>>>(a);
  return cudaGetLastError() == cudaSuccess ? MXFP8_OK : MXFP8_ERR_CUDA;
}

size_t nvfp4_grouped_mlp_workspace_size(int64_t R, int64_t H, int64_t F, int E) {
  NvWsLayout L;
  if (!nv_ws_layout(R, H, F, E, &L)) return 0;
  return L.total;
}

int nvfp4_grouped_mlp_workspace_layout(int64_t R, int64_t H, int64_t F, int E, uint64_t* out) {
  NvWsLayout L;
  if (out == nullptr || !nv_ws_layout(R, H, F, E, &L)) return MXFP8_ERR_INVALID_ARG;
  out[0] = L.meta;
  out[1] = L.amax;
  out[2] = L.xq;
  out[3] = L.xsf;
  out[4] = L.hq;
  out[5] = L.hsf;
  out[6] = static_cast<uint64_t>(L.r_pad);
  return MXFP8_OK;
}

int nvfp4_grouped_mlp_fwd(const void* x_sorted, int64_t R, int64_t H, int64_t F, int E, const int32_t* split_sizes,
                          const float* gates, const uint8_t* w1_q, const uint8_t* w1_sf, const float* w1_amax,
                          const uint8_t* w2_q, const uint8_t* w2_sf, const float* w2_amax, float h_amax, void* y,
                          void* workspace, size_t workspace_bytes, void* stream, void* const* stage_events) {
  if (R < 0 || E < 1 || E > 1024 || H <= 0 || F <= 0) return MXFP8_ERR_INVALID_ARG;
  if (H % 256 != 0 || F % 128 != 0) return MXFP8_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(E) * 2 * F > INT32_MAX || static_cast<int64_t>(E) * H > INT32_MAX)
    return MXFP8_ERR_UNSUPPORTED;
  if (!(h_amax > 0.0f) || !(h_amax <= 3.402823466e38f)) return MXFP8_ERR_INVALID_ARG;
  const void* ptrs[] = {x_sorted, split_sizes, w1_q, w1_sf, w2_q, w2_sf, y, workspace};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned16(p)) return MXFP8_ERR_INVALID_ARG;
  if (w1_amax == nullptr || w2_amax == nullptr) return MXFP8_ERR_INVALID_ARG;
  if (gates != nullptr && !aligned16(gates)) return MXFP8_ERR_INVALID_ARG;
  NvWsLayout L;
  if (!nv_ws_layout(R, H, F, E, &L)) return MXFP8_ERR_UNSUPPORTED;
  if (workspace_bytes < L.total || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MXFP8_ERR_WORKSPACE;
  return launch_nvfp4_grouped_mlp(x_sorted, R, H, F, E, split_sizes, gates, w1_q, w1_sf, w1_amax, w2_q, w2_sf,
                                  w2_amax, h_amax, y, workspace, L, static_cast<cudaStream_t>(stream), stage_events);
}

}  // extern "C"
