// quantize.cu -- MXFP8 quantization of bf16 matrices (row-wise and/or column-wise blocks of 32).
//
// Operation: page "Efficient MoE training for biological foundation models", Key technical
// approaches, item 2 (8-bit values, one scale per 32 consecutive values); the scale rule is the
// OCP MX v1.0 one (see mx_device.cuh).
//
// HBM-bound design: one CTA of 256 threads owns a 32-row x 256-column tile.  Each thread loads
// 8 consecutive bf16 of 4 rows with 128-bit loads (a warp reads 512 contiguous bytes of a row),
// so the tile is read exactly once for both directions:
//   - row-wise: a 32-block is 4 neighbouring lanes; its amax takes two xor-shuffles, then each
//     lane writes its 8 codes as one 8-byte store (a warp writes 256 contiguous bytes);
//   - column-wise: each thread reduces its 8 columns over its 4 rows, warps exchange the partial
//     maxima through 8 KB of shared memory, and each thread quantizes its own 4 x 8 values with
//     the column scales (stores again 256 contiguous bytes per warp and row).
// No values are staged in shared memory; only the column maxima are.
#include <cuda_runtime.h>

#include "mx_device.cuh"
#include "mx_internal.h"
#include "mxfp8moe.h"

namespace mx {
namespace {

constexpr int QT_ROWS = 32;
constexpr int QT_COLS = 256;
constexpr int QT_THREADS = 256;

struct QuantArgs {
  const uint16_t* x;
  int64_t M, K;        // rows / columns of the source matrix
  uint8_t* q_row;
  uint8_t* sf_row;
  uint8_t* q_col;
  uint8_t* sf_col;
  int64_t kt_row;      // tensor-core layout: atoms per 128-row tile for row-wise bytes
  int64_t kt_col;      // tensor-core layout: atoms per 128-column tile for column-wise bytes
  const SchedHeader* meta;  // gather mode only
  int E;
};

__device__ __forceinline__ void unpack8(const uint4 w, float* v) {
  v[0] = bf16_lo(w.x); v[1] = bf16_hi(w.x);
  v[2] = bf16_lo(w.y); v[3] = bf16_hi(w.y);
  v[4] = bf16_lo(w.z); v[5] = bf16_hi(w.z);
  v[6] = bf16_lo(w.w); v[7] = bf16_hi(w.w);
}

// ROW / COL: directions produced.  MMA: scale bytes in the tensor-core layout instead of the
// compact one.  GATHER: rows are the expert-padded row space of a grouped MLP; padded row p of
// expert e reads source row row_off[e] + (p - pad_off[e]) or is a zero row past the expert's
// count.
template <bool ROW, bool COL, bool MMA, bool GATHER>
__global__ void __launch_bounds__(QT_THREADS) k_quantize(const QuantArgs a) {
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t K = a.K;
  const int64_t row0 = static_cast<int64_t>(blockIdx.x) * QT_ROWS;
  const int64_t col = static_cast<int64_t>(blockIdx.y) * QT_COLS + lane * 8;
  const bool col_ok = col < K;   // K % 32 == 0, so a 4-lane block group is all in or all out

  int64_t src[4];
  if constexpr (GATHER) {
    const int32_t pad_rows = a.meta->pad_rows;
    if (row0 >= pad_rows) return;  // whole tile past the last expert (pad_rows % 128 == 0)
    const int32_t* row_off = reinterpret_cast<const int32_t*>(a.meta + 1);
    const int32_t* pad_off = row_off + (a.E + 1);
    int lo = 0, hi = a.E;  // largest e with pad_off[e] <= row0: the (non-empty) owner of the tile
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (pad_off[mid] <= row0) lo = mid; else hi = mid;
    }
    const int64_t local0 = row0 - pad_off[lo] + warp * 4;
    const int64_t cnt = row_off[lo + 1] - row_off[lo];
#pragma unroll
    for (int i = 0; i < 4; ++i) src[i] = (local0 + i < cnt) ? row_off[lo] + local0 + i : -1;
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t r = row0 + warp * 4 + i;
      src[i] = r < a.M ? r : -1;
    }
  }

  float v[4][8];
  uint4 w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (src[i] >= 0 && col_ok)
      w[i] = __ldcs(reinterpret_cast<const uint4*>(a.x + src[i] * K + col));
    else
      w[i] = make_uint4(0u, 0u, 0u, 0u);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) unpack8(w[i], v[i]);

  if constexpr (ROW) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float m = 0.0f;
#pragma unroll
      for (int k = 0; k < 8; ++k) m = fmaxf(m, fabsf(v[i][k]));
      m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
      m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
      const uint32_t sfb = e8m0_from_amax(m);
      const uint2 q = quant8(v[i], e8m0_inverse_scale(sfb));
      const int64_t r_out = row0 + warp * 4 + i;
      const bool row_out_ok = GATHER ? true : (src[i] >= 0);
      if (row_out_ok && col_ok) {
        __stcs(reinterpret_cast<uint2*>(a.q_row + r_out * K + col), q);
        if ((lane & 3) == 0) {
          const int64_t blk = col >> 5;
          if constexpr (MMA)
            a.sf_row[sf_mma_offset(r_out, blk, a.kt_row)] = static_cast<uint8_t>(sfb);
          else
            a.sf_row[r_out * (K >> 5) + blk] = static_cast<uint8_t>(sfb);
        }
      }
    }
  }

  if constexpr (COL) {
    __shared__ __align__(16) float red[QT_THREADS / 32][QT_COLS];
    float cm[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      cm[k] = fmaxf(fmaxf(fabsf(v[0][k]), fabsf(v[1][k])), fmaxf(fabsf(v[2][k]), fabsf(v[3][k])));
    }
    reinterpret_cast<float4*>(&red[warp][lane * 8])[0] = make_float4(cm[0], cm[1], cm[2], cm[3]);
    reinterpret_cast<float4*>(&red[warp][lane * 8])[1] = make_float4(cm[4], cm[5], cm[6], cm[7]);
    __syncthreads();
#pragma unroll
    for (int ww = 0; ww < QT_THREADS / 32; ++ww) {
      const float4 lo = reinterpret_cast<const float4*>(&red[ww][lane * 8])[0];
      const float4 hi = reinterpret_cast<const float4*>(&red[ww][lane * 8])[1];
      cm[0] = fmaxf(cm[0], lo.x); cm[1] = fmaxf(cm[1], lo.y); cm[2] = fmaxf(cm[2], lo.z); cm[3] = fmaxf(cm[3], lo.w);
      cm[4] = fmaxf(cm[4], hi.x); cm[5] = fmaxf(cm[5], hi.y); cm[6] = fmaxf(cm[6], hi.z); cm[7] = fmaxf(cm[7], hi.w);
    }
    uint32_t sfb[8];
    float inv[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      sfb[k] = e8m0_from_amax(cm[k]);
      inv[k] = e8m0_inverse_scale(sfb[k]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (src[i] >= 0 && col_ok) {
        uint2 q;
        q.x = e4m3x2(v[i][0] * inv[0], v[i][1] * inv[1]) | (e4m3x2(v[i][2] * inv[2], v[i][3] * inv[3]) << 16);
        q.y = e4m3x2(v[i][4] * inv[4], v[i][5] * inv[5]) | (e4m3x2(v[i][6] * inv[6], v[i][7] * inv[7]) << 16);
        __stcs(reinterpret_cast<uint2*>(a.q_col + (row0 + warp * 4 + i) * K + col), q);
      }
    }
    if (warp == 0 && col_ok) {
      const int64_t rb = row0 >> 5;
      if constexpr (MMA) {
#pragma unroll
        for (int k = 0; k < 8; ++k) a.sf_col[sf_mma_offset(col + k, rb, a.kt_col)] = static_cast<uint8_t>(sfb[k]);
      } else {
        uint2 s;
        s.x = sfb[0] | (sfb[1] << 8) | (sfb[2] << 16) | (sfb[3] << 24);
        s.y = sfb[4] | (sfb[5] << 8) | (sfb[6] << 16) | (sfb[7] << 24);
        *reinterpret_cast<uint2*>(a.sf_col + rb * K + col) = s;
      }
    }
  }
}

template <bool ROW, bool COL, bool MMA>
cudaError_t launch_dirs(const QuantArgs& a, cudaStream_t stream) {
  const dim3 grid(static_cast<unsigned>((a.M + QT_ROWS - 1) / QT_ROWS),
                  static_cast<unsigned>((a.K + QT_COLS - 1) / QT_COLS));
  k_quantize<ROW, COL, MMA, false><<<grid, QT_THREADS, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quantize(const void* x, int64_t M, int64_t K, int dirs, int sf_layout, uint8_t* q_row,
                            uint8_t* sf_row, uint8_t* q_col, uint8_t* sf_col, cudaStream_t stream) {
  QuantArgs a{};
  a.x = static_cast<const uint16_t*>(x);
  a.M = M;
  a.K = K;
  a.q_row = q_row;
  a.sf_row = sf_row;
  a.q_col = q_col;
  a.sf_col = sf_col;
  a.kt_row = (K / 32 + 3) / 4;
  a.kt_col = ((M + 31) / 32 + 3) / 4;
  const bool row = dirs & MXFP8_ROWWISE, col = dirs & MXFP8_COLWISE, mma = sf_layout == MXFP8_SF_MMA;
  if (row && col) return mma ? launch_dirs<true, true, true>(a, stream) : launch_dirs<true, true, false>(a, stream);
  if (row) return mma ? launch_dirs<true, false, true>(a, stream) : launch_dirs<true, false, false>(a, stream);
  return mma ? launch_dirs<false, true, true>(a, stream) : launch_dirs<false, true, false>(a, stream);
}

cudaError_t launch_quantize_gather(const void* x, int64_t R, int64_t H, const SchedHeader* meta, int E,
                                   int64_t r_pad, uint8_t* xq, uint8_t* xsf, cudaStream_t stream) {
  QuantArgs a{};
  a.x = static_cast<const uint16_t*>(x);
  a.M = R;
  a.K = H;
  a.q_row = xq;
  a.sf_row = xsf;
  a.kt_row = H / 128;
  a.meta = meta;
  a.E = E;
  const dim3 grid(static_cast<unsigned>(r_pad / QT_ROWS), static_cast<unsigned>((H + QT_COLS - 1) / QT_COLS));
  k_quantize<true, false, true, true><<<grid, QT_THREADS, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace mx
