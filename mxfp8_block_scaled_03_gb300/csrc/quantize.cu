// quantize.cu -- MXFP8 quantization of bf16 matrices (row-wise and/or column-wise blocks of 32).
//
// Operation: page "Efficient MoE training for biological foundation models", Key technical
// approaches, item 2 (8-bit values, one scale per 32 consecutive values); the scale rule is the
// OCP MX v1.0 one (see mx_device.cuh).
//
// HBM-bound design: one CTA of 256 threads owns a 64-row x 256-column tile.  Each thread loads
// 8 consecutive bf16 of 8 rows with 128-bit loads (a warp reads 512 contiguous bytes of a row;
// 128 bytes in flight per thread, 32 KB per CTA, up to 4 CTAs per SM) and keeps them packed, so
// the tile is read exactly once for both directions:
//   - row-wise: a 32-block is 4 neighbouring lanes; its amax is a packed bf16x2 max then two
//     xor-shuffles, and each lane writes its 8 codes as one 8-byte store (a warp writes 256
//     contiguous bytes);
//   - column-wise: each thread reduces its 8 columns over its 8 rows (packed), the four warps of
//     a 32-row block exchange the partial maxima through 4 KB of shared memory, and each thread
//     quantizes its own 8 x 8 values with the column scales.
// No values are staged in shared memory; only the column maxima are.  Max of magnitudes is exact
// in bf16, so the block amax equals the one computed in higher precision.
#include <cuda_runtime.h>

#include "mx_device.cuh"
#include "mx_internal.h"
#include "mxfp8moe.h"

namespace mx {
namespace {

constexpr int QT_THREADS = 256;
constexpr int QT_RPT = 8;                              // rows per thread
constexpr int QT_ROWS = QT_RPT * (QT_THREADS / 32);    // 64 rows per tile
constexpr int QT_COLS = 256;                           // 8 bf16 per lane

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
  const int32_t* tok;       // gather mode: source row of every sorted row (NULL: the sorted row itself)
};

__device__ __forceinline__ float max_halves(uint32_t m) { return fmaxf(bf16_lo(m), bf16_hi(m)); }

// 8 bf16 (one uint4) times a common inverse scale -> 8 codes.
__device__ __forceinline__ uint2 quant8_bf16(const uint4 w, float inv) {
  uint2 o;
  o.x = e4m3x2(bf16_lo(w.x) * inv, bf16_hi(w.x) * inv) | (e4m3x2(bf16_lo(w.y) * inv, bf16_hi(w.y) * inv) << 16);
  o.y = e4m3x2(bf16_lo(w.z) * inv, bf16_hi(w.z) * inv) | (e4m3x2(bf16_lo(w.w) * inv, bf16_hi(w.w) * inv) << 16);
  return o;
}

// 8 bf16 times 8 per-column inverse scales -> 8 codes.
__device__ __forceinline__ uint2 quant8_bf16(const uint4 w, const float* inv) {
  uint2 o;
  o.x = e4m3x2(bf16_lo(w.x) * inv[0], bf16_hi(w.x) * inv[1]) |
        (e4m3x2(bf16_lo(w.y) * inv[2], bf16_hi(w.y) * inv[3]) << 16);
  o.y = e4m3x2(bf16_lo(w.z) * inv[4], bf16_hi(w.z) * inv[5]) |
        (e4m3x2(bf16_lo(w.w) * inv[6], bf16_hi(w.w) * inv[7]) << 16);
  return o;
}

// ROW / COL: directions produced.  MMA: scale bytes in the tensor-core layout instead of the
// compact one.  GATHER: rows are the expert-padded row space of a grouped MLP; padded row p of
// expert e is sorted row r = row_off[e] + (p - pad_off[e]), read from source row tok[r] (or r
// when tok is NULL), or a zero row past the expert's count.
//
// Thread (warp w, lane l) owns rows 8w..8w+7 of the 64-row tile and columns 8l..8l+7 of the
// 256-column tile, kept as packed bf16 (8 x 16 bytes in flight per thread).  A column-wise block
// of 32 rows is warps 4b..4b+3.
template <bool ROW, bool COL, bool MMA, bool GATHER>
__global__ void __launch_bounds__(QT_THREADS, (ROW && COL) || GATHER ? 3 : 4) k_quantize(const QuantArgs a) {
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t K = a.K;
  const int64_t row0 = static_cast<int64_t>(blockIdx.x) * QT_ROWS;
  const int64_t rw0 = row0 + warp * QT_RPT;             // first row of this thread
  const int64_t col = static_cast<int64_t>(blockIdx.y) * QT_COLS + lane * 8;
  const bool col_ok = col < K;   // K % 32 == 0, so a 4-lane block group is all in or all out

  int64_t src0;      // (sorted) row of this thread's first row (rows are consecutive)
  int nsrc;          // how many of its QT_RPT rows exist in the source
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
    const int64_t local = rw0 - pad_off[lo];
    const int64_t cnt = row_off[lo + 1] - row_off[lo];
    src0 = row_off[lo] + local;
    const int64_t left = cnt - local;
    nsrc = left <= 0 ? 0 : (left >= QT_RPT ? QT_RPT : static_cast<int>(left));
  } else {
    src0 = rw0;
    const int64_t left = a.M - rw0;
    nsrc = left <= 0 ? 0 : (left >= QT_RPT ? QT_RPT : static_cast<int>(left));
  }

  int64_t src[QT_RPT];
#pragma unroll
  for (int i = 0; i < QT_RPT; ++i) {
    src[i] = src0 + i;
    if (GATHER && a.tok != nullptr && i < nsrc) {
      src[i] = __ldg(a.tok + src0 + i);
      if (src[i] < 0 || src[i] >= a.M) {   // out-of-range token id: report it, quantize a zero row
        atomicOr(const_cast<uint32_t*>(&a.meta->error), ERR_TOKEN_RANGE);
        src[i] = -1;
      }
    }
  }
  uint4 w[QT_RPT];
#pragma unroll
  for (int i = 0; i < QT_RPT; ++i) {
    if (i < nsrc && col_ok && src[i] >= 0)
      w[i] = __ldcs(reinterpret_cast<const uint4*>(a.x + src[i] * K + col));
    else
      w[i] = make_uint4(0u, 0u, 0u, 0u);
  }

  if constexpr (ROW) {
    // rows written: all QT_RPT in gather mode (padding rows become zeros), else the real ones
    const int nout = GATHER ? QT_RPT : nsrc;
#pragma unroll
    for (int i = 0; i < QT_RPT; ++i) {
      const uint32_t m2 = absmax_bf16x2(absmax_bf16x2(w[i].x, w[i].y), absmax_bf16x2(w[i].z, w[i].w));
      float m = max_halves(m2);
      m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
      m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
      const uint32_t sfb = e8m0_from_amax(m);
      if (i < nout && col_ok) {
        const int64_t r = rw0 + i;
        __stcs(reinterpret_cast<uint2*>(a.q_row + r * K + col), quant8_bf16(w[i], e8m0_inverse_scale(sfb)));
        if ((lane & 3) == 0) {
          const int64_t blk = col >> 5;
          if constexpr (MMA)
            a.sf_row[sf_mma_offset(r, blk, a.kt_row)] = static_cast<uint8_t>(sfb);
          else
            a.sf_row[r * (K >> 5) + blk] = static_cast<uint8_t>(sfb);
        }
      }
    }
  }

  if constexpr (COL) {
    __shared__ __align__(16) uint4 red[QT_THREADS / 32][32];
    uint4 cm = make_uint4(absmax_bf16x2(w[0].x), absmax_bf16x2(w[0].y), absmax_bf16x2(w[0].z),
                          absmax_bf16x2(w[0].w));
#pragma unroll
    for (int i = 1; i < QT_RPT; ++i) {
      cm.x = absmax_bf16x2(cm.x, w[i].x);
      cm.y = absmax_bf16x2(cm.y, w[i].y);
      cm.z = absmax_bf16x2(cm.z, w[i].z);
      cm.w = absmax_bf16x2(cm.w, w[i].w);
    }
    red[warp][lane] = cm;
    __syncthreads();
    const int b = warp >> 2;   // column block (32 rows) this warp belongs to
#pragma unroll
    for (int ww = 0; ww < 4; ++ww) {
      const uint4 o = red[4 * b + ww][lane];
      cm.x = absmax_bf16x2(cm.x, o.x);
      cm.y = absmax_bf16x2(cm.y, o.y);
      cm.z = absmax_bf16x2(cm.z, o.z);
      cm.w = absmax_bf16x2(cm.w, o.w);
    }
    const float cmax[8] = {bf16_lo(cm.x), bf16_hi(cm.x), bf16_lo(cm.y), bf16_hi(cm.y),
                           bf16_lo(cm.z), bf16_hi(cm.z), bf16_lo(cm.w), bf16_hi(cm.w)};
    uint32_t sfb[8];
    float inv[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      sfb[k] = e8m0_from_amax(cmax[k]);
      inv[k] = e8m0_inverse_scale(sfb[k]);
    }
#pragma unroll
    for (int i = 0; i < QT_RPT; ++i)
      if (i < nsrc && col_ok)
        __stcs(reinterpret_cast<uint2*>(a.q_col + (rw0 + i) * K + col), quant8_bf16(w[i], inv));
    const int64_t rb = (row0 >> 5) + b;
    if ((warp & 3) == 0 && col_ok && rb * 32 < a.M) {
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

// Column-wise MXFP8 with the codes written transposed, for GEMMs that contract over the rows of
// a matrix (the weight gradients, and the backward GEMMs that contract weights over their other
// axis).  Source [M, K] bf16 -> qT [K, m_out]: row c of qT holds column c of the source, each run
// of 32 consecutive source rows is one block.  Scale bytes go to sfT: the tensor-core layout of
// the [K, m_out] code matrix, or compact [K, m_out / 32].  GATHER: source rows are the
// expert-padded row space (as in k_quantize), padding rows are zeros.
//
// One CTA of 256 threads owns 128 source rows x 128 source columns, read with 128-bit loads into
// shared memory (34 KB with padding).  Word w (a bf16 pair) of tile row r sits at word
// w ^ 8 (r / 32): rows 32 apart fall on different banks, so the column pass, whose warps read
// four 32-row blocks at once, is free of bank conflicts.  Column pass: thread t takes the column
// pair 2 (t / 4), 2 (t / 4) + 1 and the 32-row block t % 4; it reads 32 packed bf16 pairs down the
// columns, takes both columns' amax on the packed pairs and writes each column's 32 codes (two
// 16-byte stores), so the four threads of a column write its 128 codes as one line.  ROW: the same
// tile also yields the row-wise MXFP8 of those rows (thread t: 32-column block t % 4 of rows t / 4
// and t / 4 + 64; tensor-core scale layout), four threads writing a row's 128 codes as one line,
// so a tensor needed in both directions is read from memory once.  (Storing 16 bytes per thread
// to 32 different rows per warp instruction kept the L1 pipe 80% busy at 62% of HBM bandwidth.)
constexpr int QTT_ROWS = 128;
constexpr int QTT_COLS = 128;
constexpr int QTT_W = QTT_COLS / 2 + 4;   // words per tile row (4 words of padding)
// word swizzle of tile row r: 8 (r / 32) (multiples of 4 words keep 16-byte chunks whole)
__device__ __forceinline__ int qtt_swz(int r) { return (r >> 5) << 3; }

struct QuantTArgs {
  const uint16_t* x;
  int64_t M, K;        // source rows (rows past M read as zeros) / columns
  int64_t m_out;       // columns of qT (rows of the source space, a multiple of 128 in MMA layout)
  uint8_t* qT;
  uint8_t* sfT;
  bool mma;
  uint8_t* q_row;           // ROW: codes [m_out, K] (row-major, rows of the tile's row space)
  uint8_t* sf_row;          // ROW: scale bytes, tensor-core layout of [m_out, K]
  const SchedHeader* meta;  // gather mode only
  int E;
  const int32_t* tok;
};

template <bool GATHER, bool ROW>
__global__ void __launch_bounds__(256, 5) k_quantize_t(const QuantTArgs a) {   // 5 blocks per SM: 48 registers
  __shared__ __align__(16) uint16_t tile[QTT_ROWS][2 * QTT_W];
  const int tid = threadIdx.x;
  const int64_t row0 = static_cast<int64_t>(blockIdx.x) * QTT_ROWS;
  const int64_t col0 = static_cast<int64_t>(blockIdx.y) * QTT_COLS;
  // source rows of the tile: first_src .. first_src + nsrc - 1 (the rest read as zeros)
  int64_t first_src = row0;
  int64_t nsrc = a.M - row0;
  if constexpr (GATHER) {
    const int32_t pad_rows = a.meta->pad_rows;
    if (row0 >= pad_rows) {
      nsrc = 0;
    } else {
      const int32_t* row_off = reinterpret_cast<const int32_t*>(a.meta + 1);
      const int32_t* pad_off = row_off + (a.E + 1);
      int lo = 0, hi = a.E;   // largest e with pad_off[e] <= row0 (experts span whole 256-row pairs)
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (pad_off[mid] <= row0) lo = mid; else hi = mid;
      }
      first_src = row_off[lo] + (row0 - pad_off[lo]);
      nsrc = (row_off[lo + 1] - row_off[lo]) - (row0 - pad_off[lo]);
    }
  }
  nsrc = nsrc < 0 ? 0 : (nsrc > QTT_ROWS ? QTT_ROWS : nsrc);
  uint32_t* tw = reinterpret_cast<uint32_t*>(&tile[0][0]);   // words, row pitch QTT_W
  // load: 128 rows x 16 chunks of 16 bytes; thread t takes chunk t % 16 of rows t / 16 + 16 j
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int rr = tid / 16 + 16 * j;
    const int ch = tid % 16;
    uint4 w = make_uint4(0u, 0u, 0u, 0u);
    if (rr < nsrc) {
      int64_t src = first_src + rr;
      if (GATHER && a.tok != nullptr) {
        src = __ldg(a.tok + src);
        if (src < 0 || src >= a.M) {
          atomicOr(const_cast<uint32_t*>(&a.meta->error), ERR_TOKEN_RANGE);
          src = -1;
        }
      }
      if (src >= 0 && col0 + ch * 8 < a.K) w = __ldcs(reinterpret_cast<const uint4*>(a.x + src * a.K + col0 + ch * 8));
    }
    *reinterpret_cast<uint4*>(tw + rr * QTT_W + ((4 * ch) ^ qtt_swz(rr))) = w;
  }
  __syncthreads();
  if constexpr (ROW) {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int rr = tid / 4 + 64 * k;
      const int cb = tid % 4;   // 32-column block inside the tile
      const int64_t rcol = col0 + cb * 32;
      uint4 w[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        w[j] = *reinterpret_cast<const uint4*>(tw + rr * QTT_W + ((16 * cb + 4 * j) ^ qtt_swz(rr)));
      uint32_t m2 = absmax_bf16x2(absmax_bf16x2(w[0].x, w[0].y), absmax_bf16x2(w[0].z, w[0].w));
#pragma unroll
      for (int j = 1; j < 4; ++j)
        m2 = absmax_bf16x2(m2, absmax_bf16x2(absmax_bf16x2(w[j].x, w[j].y), absmax_bf16x2(w[j].z, w[j].w)));
      if (rcol < a.K) {
        const uint32_t sfb = e8m0_from_amax(max_halves(m2));
        const float inv = e8m0_inverse_scale(sfb);
        const uint2 q0 = quant8_bf16(w[0], inv), q1 = quant8_bf16(w[1], inv), q2 = quant8_bf16(w[2], inv),
                    q3 = quant8_bf16(w[3], inv);
        uint4* dst = reinterpret_cast<uint4*>(a.q_row + (row0 + rr) * a.K + rcol);   // 16-byte aligned
        dst[0] = make_uint4(q0.x, q0.y, q1.x, q1.y);
        dst[1] = make_uint4(q2.x, q2.y, q3.x, q3.y);
        a.sf_row[sf_mma_offset(row0 + rr, rcol >> 5, a.K / 128)] = static_cast<uint8_t>(sfb);
      }
    }
  }
  const int cp = tid / 4;   // column pair
  const int rb = tid % 4;   // 32-row block inside the tile
  const int64_t col = col0 + 2 * cp;
  if (col >= a.K) return;
  uint32_t pk[32];          // packed bf16 pairs (column col in the low half)
  uint32_t m2 = 0;
  const int wsw = cp ^ (8 * rb);   // the swizzled word of this column pair in rows of block rb
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    pk[i] = tw[(rb * 32 + i) * QTT_W + wsw];
    m2 = absmax_bf16x2(m2, pk[i]);
  }
  const int64_t blk = (row0 >> 5) + rb;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint32_t sfb = e8m0_from_amax(h == 0 ? bf16_lo(m2) : bf16_hi(m2));
    const float inv = e8m0_inverse_scale(sfb);
    uint32_t q[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint32_t a0 = pk[4 * k], a1 = pk[4 * k + 1], a2 = pk[4 * k + 2], a3 = pk[4 * k + 3];
      const float v0 = h ? bf16_hi(a0) : bf16_lo(a0), v1 = h ? bf16_hi(a1) : bf16_lo(a1);
      const float v2 = h ? bf16_hi(a2) : bf16_lo(a2), v3 = h ? bf16_hi(a3) : bf16_lo(a3);
      q[k] = e4m3x2(v0 * inv, v1 * inv) | (e4m3x2(v2 * inv, v3 * inv) << 16);
    }
    uint4* dst = reinterpret_cast<uint4*>(a.qT + (col + h) * a.m_out + row0 + rb * 32);   // 16-byte aligned
    dst[0] = make_uint4(q[0], q[1], q[2], q[3]);
    dst[1] = make_uint4(q[4], q[5], q[6], q[7]);
    if (a.mma)
      a.sfT[sf_mma_offset(col + h, blk, a.m_out / 128)] = static_cast<uint8_t>(sfb);
    else
      a.sfT[(col + h) * (a.m_out >> 5) + blk] = static_cast<uint8_t>(sfb);
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
                                   int64_t r_pad, const int32_t* token_of_row, int64_t x_rows, uint8_t* xq,
                                   uint8_t* xsf, cudaStream_t stream) {
  QuantArgs a{};
  a.tok = token_of_row;
  a.x = static_cast<const uint16_t*>(x);
  a.M = token_of_row ? x_rows : R;   // rows of x (token rows when gathering through token_of_row)
  a.K = H;
  a.q_row = xq;
  a.sf_row = xsf;
  a.kt_row = H / 128;
  a.meta = meta;
  a.E = E;
  const dim3 grid(static_cast<unsigned>((r_pad + QT_ROWS - 1) / QT_ROWS),
                  static_cast<unsigned>((H + QT_COLS - 1) / QT_COLS));
  k_quantize<true, false, true, true><<<grid, QT_THREADS, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_quantize_t(const void* x, int64_t M, int64_t K, int64_t m_out, bool mma, uint8_t* qT,
                              uint8_t* sfT, const SchedHeader* meta, int E, const int32_t* token_of_row,
                              int64_t x_rows, cudaStream_t stream, uint8_t* q_row, uint8_t* sf_row) {
  QuantTArgs a{};
  a.x = static_cast<const uint16_t*>(x);
  a.M = meta ? (token_of_row ? x_rows : M) : M;
  a.K = K;
  a.m_out = m_out;
  a.qT = qT;
  a.sfT = sfT;
  a.mma = mma;
  a.meta = meta;
  a.E = E;
  a.tok = token_of_row;
  const dim3 grid(static_cast<unsigned>((m_out + QTT_ROWS - 1) / QTT_ROWS),
                  static_cast<unsigned>((K + QTT_COLS - 1) / QTT_COLS));
  a.q_row = q_row;
  a.sf_row = sf_row;
  const bool row = q_row != nullptr;
  if (meta) {
    if (row)
      k_quantize_t<true, true><<<grid, 256, 0, stream>>>(a);
    else
      k_quantize_t<true, false><<<grid, 256, 0, stream>>>(a);
  } else {
    if (row)
      k_quantize_t<false, true><<<grid, 256, 0, stream>>>(a);
    else
      k_quantize_t<false, false><<<grid, 256, 0, stream>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace mx
