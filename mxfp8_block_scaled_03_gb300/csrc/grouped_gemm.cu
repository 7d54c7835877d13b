// grouped_gemm.cu -- the fused MXFP8 grouped expert MLP on sm_103a: forward and backward GEMMs.
//
// Operation (page "Efficient MoE training for biological foundation models", Key technical
// approaches): GroupedLinear over per-expert row counts split_sizes (item 1), MXFP8 operands
// with one E8M0 scale per 32 values along K (item 2), and the fused
// GroupedLinear -> ScaledSwiGLU -> GroupedLinear forward in which the SwiGLU activation and the
// routing-weight multiply run inside the first GEMM and the intermediate is requantized to MXFP8
// there, so it never exists in 16-bit memory (item 3), with its corresponding backward.
//
// Forward pipeline of one call (one stream, no host synchronization):
//   1. k_schedule    split_sizes -> prefix sums, expert-padded row offsets (every expert padded to
//                    a multiple of 256 rows), tile counts, sum check (error word on mismatch).
//   2. k_quantize    x_sorted -> x_q (E4M3) + scale bytes in the tensor-core layout, rows moved
//                    into the expert-padded row space so every 256-row tile pair is one expert's.
//   3. k_grouped_gemm_pair<GEMM_SWIGLU>  per pair tile (expert e, 256 rows, 128 columns of F):
//                    [G | U] = x_q W1[e, {gate, up} rows]^T accumulated in TMEM, then
//                    h = gate * silu(G) * U, requantized to h_q + scale bytes (and, in a training
//                    forward, [G | U] saved as bf16).
//   4. k_grouped_gemm_pair<GEMM_OUT>     per pair tile (expert e, 256 rows, 256 columns of H):
//                    y = h_q W2[e]^T -> bf16, stored only for the expert's real rows.
// Backward (launch_grouped_mlp_bwd): GEMM_DGRAD (dh = dy W2 with the ScaledSwiGLU backward in the
// epilogue, which writes dGU and h already quantized: dGU row-wise for dx, dGU and h column-wise
// with transposed codes for the weight gradients), GEMM_OUT (dx = dGU W1), GEMM_WGRAD (dW2, dW1
// over each expert's rows).  NVFP4 forward (launch_nvfp4_grouped_mlp): the FMT_NV instances of the
// two forward GEMMs.
//
// Main kernel (k_grouped_gemm_pair, persistent clusters of two CTAs on two SMs, 512 threads each):
// one tcgen05.mma.cta_group::2 computes a 256 x 256 tile, each CTA loading its own 128 rows of A
// and half of B (32 KB per K step) plus the step's scale atoms, 3 stages of two K steps, the
// scales moved into TMEM by the MMA thread itself (tcgen05.cp); roles and synchronization are
// described above the kernel.  k_grouped_gemm is the single-CTA
// kernel (M=128, 4 stages of 48 KB): GroupedLinear 2 uses it when H % 256 != 0, and both forward
// GEMMs use it where no CTA pair can be co-scheduled.  Its structure:
//   TMA producer  A tile (128 rows x 128 K bytes), B tile (BN rows x 128) and the 512-byte scale
//                 atoms of both, all completing on one mbarrier per stage.
//   scale warps   four warps copy the stage's scale atoms into TMEM with tcgen05.st (one TMEM lane
//                 quarter each) and signal the MMA issuer (in this kernel, with one barrier wait
//                 per 4 MMAs, tcgen05.cp from the MMA thread was slower; the pair kernel, with 8
//                 MMAs per wait, issues its copies itself).
//   MMA issuer    allocates TMEM; one thread issues 4 block-scaled MMAs (M=128, N=BN, K=32 each)
//                 per stage into one fp32 accumulator of BN columns and commits the stage back.
//   epilogue      eight warps read their 32 TMEM lanes (rows) and half of the columns into
//                 registers, release the accumulator at once (so the next tile's MMAs overlap
//                 the epilogue math), then compute and store.
// Every mbarrier wait is bounded; a timeout sets a bit in the workspace error word and all roles
// drain and exit.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdlib>
#include <mutex>

#include "mx_device.cuh"
#include "mx_internal.h"
#include "mxfp8moe.h"

namespace mx {
namespace {

constexpr int BM = 128;                    // rows per tile (MMA M)
constexpr int BK = 128;                    // K per stage: 128 E4M3 bytes = one 128B swizzle row
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK;           // 16 KB
constexpr int B_BYTES_MAX = 256 * BK;      // 32 KB (N = 256)
constexpr int SF_ATOM = 512;               // 128 rows x 4 scale blocks
constexpr int STAGE_BYTES = 51200;         // A + B + 3 scale atoms, rounded up to 1 KB
// Warp roles (4 warpgroups):
//   warpgroup 0 (warps 0-3)   scale staging: warp w copies the stage's scale atoms from shared
//                             memory into TMEM lanes 32w..32w+31 (tcgen05.st)
//   warpgroup 1 (warps 4-7)   warp 4: TMA producer (lane 0 issues); warp 5: TMEM allocation and
//                             MMA issue (lane 0); warps 6-7 idle
//   warpgroups 2-3 (8-15)     epilogue: warp w reads TMEM lanes 32*(w%4).. and half (w-8)/4 of
//                             the accumulator columns
// Registers: launched with 128 per thread; warpgroups 0-1 give theirs down to 56 so that the
// epilogue warpgroups can hold 200 (4*32*56*2 + 8*32*200 = 512*128).
constexpr int NUM_THREADS = 512;
constexpr int WARP_PRODUCER = 4;
constexpr int WARP_MMA = 5;
constexpr int FIRST_EPI_WARP = 8;
constexpr int NUM_EPI_WARPS = 8;
constexpr int NUM_SF_WARPS = 4;
constexpr uint32_t BAR_EPI = 1;            // hardware barrier of the epilogue warps
constexpr uint32_t BAR_SF = 2;             // hardware barrier of the scale-staging warps
constexpr uint32_t BAR_STAGGER = 3;        // 3..6: pair kernel, the two epilogue warps of a lane quarter
constexpr uint32_t REGS_LOW = 56;
constexpr uint32_t REGS_HIGH = 200;
static_assert(2 * 128 * REGS_LOW + 256 * REGS_HIGH == NUM_THREADS * 128, "register split must equal the launch pool");
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t ACC_COL = 0;            // accumulator: up to 256 fp32 columns
constexpr uint32_t SFA_COL = 256;          // 4 columns per stage
constexpr uint32_t SFB_COL = 272;          // 8 columns per stage
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 256 + 1024;
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;  // 2 s per individual wait
static_assert(A_BYTES + B_BYTES_MAX + 3 * SF_ATOM <= STAGE_BYTES, "stage layout");
static_assert(STAGE_BYTES % 1024 == 0, "stages keep 1024-byte alignment for the 128B swizzle");
static_assert(SFB_COL + 8 * STAGES <= TMEM_COLS, "TMEM budget");

// GEMM_SWIGLU  forward GroupedLinear 1 + ScaledSwiGLU + requant (optionally saving [G | U])
// GEMM_OUT     A B^T -> bf16 rows (forward GroupedLinear 2; backward dx = dGU W1)
// GEMM_DGRAD   backward dh = dy W2 with the ScaledSwiGLU backward in the epilogue
// GEMM_WGRAD   weight gradient of every expert: A^T B over the expert's rows (K varies by expert)
enum GemmMode { GEMM_SWIGLU = 0, GEMM_OUT = 1, GEMM_DGRAD = 2, GEMM_WGRAD = 3 };

// Operand formats of the pair kernel.
//   FMT_MX  MXFP8: E4M3 bytes, one UE8M0 scale per 32 values of K.  A K step (BK = 128 bytes of a
//           row) is four MMAs of K = 32 sharing one 512-byte scale atom per 128 rows (the MMA
//           selects the byte of each 32-bit scale word).
//   FMT_NV  NVFP4: packed E2M1 (two values per byte), one UE4M3 scale per 16 values.  A K step
//           (128 bytes = 256 values of a row) is four MMAs of K = 64, each with its own atom of
//           four scales per row: four atoms per 128 rows per step.  Only the forward GEMMs
//           (GEMM_SWIGLU, GEMM_OUT) run on it.
enum PairFmt { FMT_MX = 0, FMT_NV = 1 };

struct GemmParams {
  const SchedHeader* meta;
  const uint8_t* a_sf;     // scale bytes of A (tensor-core layout, padded rows)
  const uint8_t* b_sf;     // scale bytes of B (tensor-core layout, weight rows)
  int E;
  int KT;                  // K / 128
  int NT;                  // column tiles per expert
  int BN;                  // MMA N (256, or 128 for GEMM_OUT when H % 256 != 0)
  int b_rows_per_expert;   // 2F (GEMM_SWIGLU) or H (GEMM_OUT)
  int F;                   // GEMM_SWIGLU: row offset of the up projection inside an expert
  int n_fastest;           // tile order inside an expert: 1 = column tiles fastest, 0 = row tiles
  int group_m;             // pair kernel with n_fastest: row-tile pairs per group (0: no groups).
                           // Inside an expert, groups of group_m row pairs run one after the other
                           // and, in a group, its row pairs fastest: the tiles in flight cover
                           // group_m row bands x (clusters / group_m) weight column tiles, so each
                           // band stays in L2 across all column tiles and each weight column tile is
                           // read once per group instead of once per wave of tiles
  int64_t y_rows;          // GEMM_OUT: rows of y (the TMA store map's extent)
  // GEMM_SWIGLU epilogue
  const float* gates;
  uint8_t* hq;
  uint8_t* hsf;
  int64_t ldh;             // F
  // GEMM_OUT epilogue
  uint16_t* y;
  int64_t ldy;             // H
  uint32_t* err;
  uint64_t timeout_ns;     // limit of each pipeline wait (producer, MMA, epilogue, scale staging)
  uint64_t drain_ns;       // limit of each teardown wait for copies or MMAs still in flight
  // operand addressing of the pair kernel
  int a_kt;                // scale atoms per 128-row tile of A (K extent of A / 128)
  int b_kt;                // same for B
  int a_sf_tiles;          // 128-row tiles of A's scale array (pair kernel: extent of its scale map)
  int b_sf_tiles;          // same for B
  int b_kofs;              // expert e's block of B starts at K column e * b_kofs (weights stored
                           // transposed as one [N, E*K] matrix); 0 for the forward
  // GEMM_SWIGLU in a training forward: [G | U] saved as bf16 [R_pad, 2F] (NULL: not saved)
  uint16_t* gu_out;
  // GEMM_DGRAD epilogue
  const uint16_t* gu;      // saved [G | U]
  uint8_t* dguq;           // [dG | dU] row-wise MXFP8 codes [R_pad, 2F]
  uint8_t* dgusf;          //   their scale bytes (tensor-core layout of [R_pad, 2F])
  uint8_t* dguT;           // [dG | dU] and then h column-wise MXFP8, codes transposed: one
                           // [3F, R_pad] matrix (the target of the epilogue's bulk tensor stores)
  uint8_t* dguTsf;         //   scale bytes of [dG | dU] (tensor-core layout of [2F, R_pad])
  uint8_t* hTsf;           //   scale bytes of h (tensor-core layout of [F, R_pad])
  int64_t r_pad;           // rows of the padded row space (columns of the transposed codes)
  int64_t t_kt;            // r_pad / 128: scale atoms per 128-row tile of the transposed matrices
  float* dgate_part;       // [R_pad, F / 128] partial sums of the routing-weight gradient
  // GEMM_WGRAD
  int wg_mt, wg_nt;        // 256-row tiles of A's rows (M / 256) and of B's rows (N / 256)
  int wg_m_fastest;        // 1: A tiles run fastest inside an expert (keeps the smaller A block in L2)
  int b_rows;              // rows of B when its last 256-row tile may be half past the end (GEMM_DGRAD,
                           // GEMM_WGRAD with N % 256 == 128): that half reads zeros and is not stored;
                           // 0 when every tile is whole
  int64_t wg_m, wg_n;      // rows and columns of each expert's gradient block
  float* dw;               // [E, M, N] fp32
  // NVFP4 operands (FMT_NV): the per-tensor magnitudes the encode scales 2688 / amax come from
  const float* nv_amax_a;  // device (A = x: written by the amax kernel); NULL: nv_amax_a_val
  float nv_amax_a_val;     // A = h in GroupedLinear 2: the caller's magnitude for the intermediate
  const float* nv_amax_b;  // device: the weight's magnitude (written by its quantization)
  float nv_out_amax;       // GEMM_SWIGLU: magnitude the intermediate's encode scale derives from
  uint32_t* nv_out_seen;   // GEMM_SWIGLU: largest |h| of the call (float bits, atomicMax) or NULL
  int64_t h_kt;            // GEMM_SWIGLU: scale atoms per 128-row tile of h
};

struct TileInfo {
  int e, n, pad_row0, src_row0, valid;
  // pair kernel: rows of this CTA's A tile and of the pair's two B halves, K offsets, K steps
  int a_row, b_row0, b_row1, a_k0, b_k0, steps;
};

// Work unit u -> (expert, column tile, 128-row tile).  Units are ordered expert by expert; inside
// an expert either the row tiles or the column tiles run fastest, so the tiles in flight at once
// share one operand in L2 (GEMM 1: the expert's activations and a few weight column tiles;
// GEMM 2: one row tile of the intermediate and the expert's whole W2).
__device__ __forceinline__ void decode_unit(int u, const GemmParams& p, TileInfo& t) {
  const int32_t* row_off = reinterpret_cast<const int32_t*>(p.meta + 1);
  const int32_t* pad_off = row_off + (p.E + 1);
  const int32_t* mt_off = pad_off + (p.E + 1);
  int lo = 0, hi = p.E;  // largest e with mt_off[e] * NT <= u (skips empty experts)
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(mt_off + mid) * p.NT <= u) lo = mid; else hi = mid;
  }
  const int e = lo;
  const int m0 = __ldg(mt_off + e);
  const int mt_e = __ldg(mt_off + e + 1) - m0;
  const int local = u - m0 * p.NT;
  int n, tt;
  if (p.n_fastest) {
    tt = local / p.NT;
    n = local - tt * p.NT;
  } else {
    n = local / mt_e;
    tt = local - n * mt_e;
  }
  const int r0 = __ldg(row_off + e);
  t.e = e;
  t.n = n;
  t.pad_row0 = __ldg(pad_off + e) + BM * tt;
  t.src_row0 = r0 + BM * tt;
  t.valid = min(BM, __ldg(row_off + e + 1) - r0 - BM * tt);
}

// First row of B box i (128 rows) of a tile: GEMM 1 boxes are the gate rows and the up rows of
// column tile n; GEMM 2 boxes are consecutive W2 rows.
template <int MODE>
__device__ __forceinline__ int b_box_row(const GemmParams& p, const TileInfo& t, int i) {
  const int brow0 = t.e * p.b_rows_per_expert;
  return MODE == GEMM_SWIGLU ? brow0 + i * p.F + t.n * 128 : brow0 + t.n * p.BN + i * 128;
}

// Lane 0 waits, the whole warp learns the outcome (keeps .sync.aligned instructions convergent).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const volatile int* abort, uint64_t timeout,
                                          uint32_t* err, uint32_t err_bit, int lane) {
  int ok = 1;
  if (lane == 0) {
    ok = mbar_wait_bounded(bar, parity, abort, timeout) ? 1 : 0;
    if (!ok) {
      atomicOr(err, err_bit);
      *const_cast<volatile int*>(abort) = 1;
    }
  }
  return __shfl_sync(0xFFFFFFFFu, ok, 0) != 0;
}

// Single-thread form for loops that run in one lane only (the MMA issuer).
__device__ __forceinline__ bool lane_wait(uint64_t* bar, uint32_t parity, const volatile int* abort, uint64_t timeout,
                                          uint32_t* err, uint32_t err_bit) {
  if (mbar_wait_bounded(bar, parity, abort, timeout)) return true;
  atomicOr(err, err_bit);
  *const_cast<volatile int*>(abort) = 1;
  return false;
}

__device__ __forceinline__ void tmem_st_32x32b_x4(uint32_t taddr, const uint4 v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// 16 registers per thread -> 16 consecutive TMEM columns of this warp's 32 lanes.
__device__ __forceinline__ void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}

template <uint32_t N>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

// Saved pre-activations [G | U] ([r_pad, 2F] bf16) are stored in blocks of 32 rows x 8 columns
// (512 contiguous bytes, row-major inside): the epilogue thread of padded row p reads and writes
// 8 columns with one 16-byte access, and the 32 lanes of a warp (32 consecutive rows) cover one
// block, so every such warp access is one contiguous 512-byte transfer.
__device__ __forceinline__ int64_t gu_offset(int64_t prow, int64_t j, int64_t two_f) {
  return ((prow >> 5) * (two_f >> 3) + (j >> 3)) * 256 + (prow & 31) * 8 + (j & 7);
}

// Epilogue math of one tile for the thread holding tile row r and column half `half`, from the
// accumulator values v already read out of TMEM.
//   GEMM_SWIGLU: v[0..63] gate columns 64*half.., v[64..127] the matching up columns;
//                h = gate_r * silu(G) * U, two 32-blocks requantized to E4M3 codes + E8M0 bytes
//                (written straight into the tensor-core scale layout GroupedLinear 2 reads).
//   GEMM_OUT:    v[0..BN/2) columns BN/2*half.. -> bf16, stored for the expert's real rows only.
//   NVFP4 (FMT_NV): accumulators are first multiplied by alpha = 1 / (s_a s_b), the product of the
//                operands' per-tensor decode scales; GEMM_SWIGLU requantizes h to NVFP4 under the
//                encode scale s_out (four 16-value blocks per thread, E4M3 block scales).
// One MXFP8 block of 32 bf16 values (pairs x2[i] = values 2i, 2i + 1) -> 32 E4M3 codes (q[k]: values
// 4k .. 4k + 3, lowest byte first); returns the block's UE8M0 scale byte.
__device__ __forceinline__ uint32_t quantize_block32(const uint32_t (&x2)[16], uint32_t (&q)[8]) {
  // block amax on packed magnitudes: max.xorsign.abs keeps the larger magnitude of each half
  // (its sign, the XOR of the operands' signs, is cleared at the end)
  uint32_t m2 = x2[0];
#pragma unroll
  for (int i = 1; i < 16; ++i) asm("max.xorsign.abs.bf16x2 %0, %0, %1;" : "+r"(m2) : "r"(x2[i]));
  m2 &= 0x7FFF7FFFu;
  const uint32_t sfb = e8m0_from_amax(fmaxf(bf16_lo(m2), bf16_hi(m2)));
  const float inv = e8m0_inverse_scale(sfb);
  const uint64_t inv2 = f2_pack(inv, inv);
#pragma unroll
  for (int k = 0; k < 8; ++k)   // the exact power-of-two scaling, two values per instruction
    q[k] = e4m3x2_f2(f2_mul(f2_pack(bf16_lo(x2[2 * k]), bf16_hi(x2[2 * k])), inv2)) |
           (e4m3x2_f2(f2_mul(f2_pack(bf16_lo(x2[2 * k + 1]), bf16_hi(x2[2 * k + 1])), inv2)) << 16);
  return sfb;
}

// The same, codes stored at dst (32-byte aligned).
__device__ __forceinline__ uint32_t quantize_block32_to(const uint32_t (&x2)[16], uint8_t* dst) {
  uint32_t q[8];
  const uint32_t sfb = quantize_block32(x2, q);
  st_global_32B(dst, make_uint4(q[0], q[1], q[2], q[3]), make_uint4(q[4], q[5], q[6], q[7]));
  return sfb;
}

// Column-wise MXFP8 blocks of a warp: lane l holds 32 bf16 values of its row, the warp's 32
// lanes being 32 consecutive rows.  The 32 x 32 block passes through the warp's 2 KB of shared
// memory (rows of 64 bytes; 16-byte chunk j of row i stored at chunk j ^ ((i >> 1) & 3), so that
// both the row writes and the column reads are free of bank conflicts):
//   colblock_acquire  waits until the buffer's previous bulk store has read it (before the first
//                     colblock_put of a block);
//   colblock_put      writes chunk j (columns 8j .. 8j + 7, as four bf16 pairs) of the lane's row;
//   colblock_quantize (after all four chunks) has lane l read column l, take its block scale
//                     (returned, the UE8M0 byte of column l) and put its 32 E4M3 codes (rows in
//                     order) as row l of a 32 x 32-byte tile in the same buffer (32B swizzle:
//                     16-byte chunk j of row l at j ^ ((l >> 2) & 1)), which one lane then writes
//                     with a bulk tensor store to (x, y) of the transposed code matrix `tm`.
__device__ __forceinline__ void colblock_acquire(int lane) {
  if (lane == 0) bulk_wait_read_all();
  __syncwarp();
}

__device__ __forceinline__ void colblock_put(uint8_t* buf, int lane, int j, uint4 w) {
  *reinterpret_cast<uint4*>(buf + lane * 64 + 16 * (j ^ ((lane >> 1) & 3))) = w;
}

__device__ __forceinline__ uint32_t colblock_quantize(uint8_t* buf, int lane, const CUtensorMap* tm, int x, int y) {
  __syncwarp();   // every lane's row is in place
  const int cj = lane >> 3, cw = 4 * ((lane & 7) >> 1);   // chunk and word of column `lane` in a row
  const uint32_t sel = (lane & 1) ? 0x7632u : 0x5410u;      // its half of the word, from both rows
  uint32_t c2[16];                                 // column `lane`, rows (2i, 2i + 1) as bf16 pairs
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int o = 16 * (cj ^ (i & 3)) + cw;        // rows 2i and 2i + 1 share the swizzle
    c2[i] = __byte_perm(*reinterpret_cast<const uint32_t*>(buf + (2 * i) * 64 + o),
                        *reinterpret_cast<const uint32_t*>(buf + (2 * i + 1) * 64 + o), sel);
  }
  uint32_t q[8];
  const uint32_t sfb = quantize_block32(c2, q);
  __syncwarp();   // all columns are read: the buffer takes the codes
  const int sw = (lane >> 2) & 1;
  *reinterpret_cast<uint4*>(buf + lane * 32 + 16 * sw) = make_uint4(q[0], q[1], q[2], q[3]);
  *reinterpret_cast<uint4*>(buf + lane * 32 + 16 * (sw ^ 1)) = make_uint4(q[4], q[5], q[6], q[7]);
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(tm, buf, x, y);
    bulk_commit_group();
  }
  return sfb;
}

template <int MODE, int FMT = FMT_MX>
__device__ __forceinline__ void epilogue_tile(const GemmParams& p, const TileInfo& t, uint32_t* v, int r,
                                              int half, int BN, float alpha = 1.0f, float s_out = 1.0f,
                                              uint8_t* wbuf = nullptr, uint32_t t_park = 0,
                                              const CUtensorMap* tmT = nullptr) {
  if (MODE == GEMM_SWIGLU && FMT == FMT_NV) {
    const bool real = r < t.valid;
    const float gate = real ? (p.gates ? __ldg(p.gates + t.src_row0 + r) : 1.0f) : 0.0f;
    const int64_t prow = t.pad_row0 + r;
    const int c0 = t.n * 128 + 64 * half;                     // first column of F this thread holds
    const uint64_t one2 = f2_pack(1.0f, 1.0f), al2 = f2_pack(alpha, alpha), gate2 = f2_pack(gate, gate);
    uint32_t q[8];
    uint32_t sfw = 0;
    float hmax = 0.0f;
#pragma unroll
    for (int b = 0; b < 4; ++b) {   // 16-value blocks
      float h[16];
      float amax = 0.0f;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int c = 16 * b + 2 * i;
        const uint64_t g = f2_mul(f2_pack(__uint_as_float(v[c]), __uint_as_float(v[c + 1])), al2);
        const uint64_t up = f2_mul(f2_pack(__uint_as_float(v[64 + c]), __uint_as_float(v[64 + c + 1])), al2);
        const uint64_t d = f2_add(f2_pack(__expf(-f2_lo(g)), __expf(-f2_hi(g))), one2);   // 1 + e^-g
        const uint64_t sig = f2_pack(__fdividef(1.0f, f2_lo(d)), __fdividef(1.0f, f2_hi(d)));
        const uint64_t hv = f2_mul(f2_mul(f2_mul(g, sig), up), gate2);
        h[2 * i] = f2_lo(hv);
        h[2 * i + 1] = f2_hi(hv);
        amax = fmaxf(amax, fmaxf(fabsf(h[2 * i]), fabsf(h[2 * i + 1])));
      }
      float rm;
      const uint32_t sfc = nv_block_scale(amax, s_out, &rm);
      q[2 * b] = e2m1x8(__fmul_rn(h[0], rm), __fmul_rn(h[1], rm), __fmul_rn(h[2], rm), __fmul_rn(h[3], rm),
                        __fmul_rn(h[4], rm), __fmul_rn(h[5], rm), __fmul_rn(h[6], rm), __fmul_rn(h[7], rm));
      q[2 * b + 1] = e2m1x8(__fmul_rn(h[8], rm), __fmul_rn(h[9], rm), __fmul_rn(h[10], rm), __fmul_rn(h[11], rm),
                            __fmul_rn(h[12], rm), __fmul_rn(h[13], rm), __fmul_rn(h[14], rm), __fmul_rn(h[15], rm));
      sfw |= sfc << (8 * b);
      hmax = fmaxf(hmax, amax);
    }
    // 64 codes = 32 bytes of row prow; the 4 block scales are one 32-bit word of one atom
    st_global_32B(p.hq + prow * (p.ldh / 2) + c0 / 2, make_uint4(q[0], q[1], q[2], q[3]),
                  make_uint4(q[4], q[5], q[6], q[7]));
    const int64_t atom = (prow / BM) * p.h_kt + c0 / 64;
    uint8_t* sfp = p.hsf + atom * SF_ATOM + (r & 31) * 16 + ((r >> 5) & 3) * 4;
    *reinterpret_cast<uint32_t*>(sfp) = sfw;
    // F % 256 == 128: GroupedLinear 2's last K step runs half past F, over two atoms of zero codes
    // (the TMA fills its codes with zeros); the last column tile gives them zero scales
    if (p.ldh % 256 != 0 && t.n == p.ldh / 128 - 1) *reinterpret_cast<uint32_t*>(sfp + 2 * SF_ATOM) = 0u;
    if (p.nv_out_seen != nullptr) {
      const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(hmax));   // non-negative floats
      if ((threadIdx.x & 31) == 0) atomicMax(p.nv_out_seen, m);
    }
  } else if (MODE == GEMM_SWIGLU) {
    const bool real = r < t.valid;
    const float gate = real ? (p.gates ? __ldg(p.gates + t.src_row0 + r) : 1.0f) : 0.0f;
    uint8_t* hrow = p.hq + static_cast<int64_t>(t.pad_row0 + r) * p.ldh + t.n * 128 + 64 * half;
    uint32_t sf_pair = 0;
    const uint64_t one2 = f2_pack(1.0f, 1.0f);
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      // column pairs in f32x2 arithmetic: hs = silu(G) * U; h = gate * hs.  The gate is one
      // factor per row, so it moves out of the block maximum and into the quantization
      // multiplier: max|fl(gate hs)| = fl(|gate| max|hs|) (rounding is monotonic) and
      // fl(hs fl(gate 2^-s)) = fl(gate hs) 2^-s (power-of-two scaling is exact): the same codes and
      // scale byte as rounding h itself.
      uint64_t hs[16];
      float amax = 0.0f;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const uint64_t g = f2_pack(__uint_as_float(v[32 * b + 2 * i]), __uint_as_float(v[32 * b + 2 * i + 1]));
        const uint64_t up =
            f2_pack(__uint_as_float(v[64 + 32 * b + 2 * i]), __uint_as_float(v[64 + 32 * b + 2 * i + 1]));
        const uint64_t d = f2_add(f2_pack(__expf(-f2_lo(g)), __expf(-f2_hi(g))), one2);   // 1 + e^-g
        const uint64_t sig = f2_pack(__fdividef(1.0f, f2_lo(d)), __fdividef(1.0f, f2_hi(d)));
        hs[i] = f2_mul(f2_mul(g, sig), up);
        amax = fmaxf(amax, fmaxf(fabsf(f2_lo(hs[i])), fabsf(f2_hi(hs[i]))));
      }
      const uint32_t sfb = e8m0_from_amax(fabsf(gate) * amax);
      const float gi = gate * e8m0_inverse_scale(sfb);
      const uint64_t gi2 = f2_pack(gi, gi);
      uint32_t q[8];
#pragma unroll
      for (int k = 0; k < 8; ++k)
        q[k] = e4m3x2_f2(f2_mul(hs[2 * k], gi2)) | (e4m3x2_f2(f2_mul(hs[2 * k + 1], gi2)) << 16);
      // one full 32-byte sector per store (two 16-byte stores cost GroupedLinear 1 about 3%)
      st_global_32B(hrow + 32 * b, make_uint4(q[0], q[1], q[2], q[3]), make_uint4(q[4], q[5], q[6], q[7]));
      sf_pair |= sfb << (8 * b);
    }
    // scale bytes of blocks (2*half, 2*half+1) of column tile n for padded row pad_row0 + r
    const int64_t atom = static_cast<int64_t>(t.pad_row0 / BM) * (p.ldh / 128) + t.n;
    *reinterpret_cast<uint16_t*>(p.hsf + atom * SF_ATOM + (r & 31) * 16 + (r >> 5) * 4 + 2 * half) =
        static_cast<uint16_t>(sf_pair);
    if (p.gu_out != nullptr) {   // training forward: keep the pre-activations for the backward
      const int64_t prow = t.pad_row0 + r, j0 = t.n * 128 + 64 * half;
#pragma unroll
      for (int c = 0; c < 64; c += 8) {
        uint4 og, ou;
        og.x = pack_bf16x2(__uint_as_float(v[c + 0]), __uint_as_float(v[c + 1]));
        og.y = pack_bf16x2(__uint_as_float(v[c + 2]), __uint_as_float(v[c + 3]));
        og.z = pack_bf16x2(__uint_as_float(v[c + 4]), __uint_as_float(v[c + 5]));
        og.w = pack_bf16x2(__uint_as_float(v[c + 6]), __uint_as_float(v[c + 7]));
        ou.x = pack_bf16x2(__uint_as_float(v[64 + c + 0]), __uint_as_float(v[64 + c + 1]));
        ou.y = pack_bf16x2(__uint_as_float(v[64 + c + 2]), __uint_as_float(v[64 + c + 3]));
        ou.z = pack_bf16x2(__uint_as_float(v[64 + c + 4]), __uint_as_float(v[64 + c + 5]));
        ou.w = pack_bf16x2(__uint_as_float(v[64 + c + 6]), __uint_as_float(v[64 + c + 7]));
        *reinterpret_cast<uint4*>(p.gu_out + gu_offset(prow, j0 + c, 2 * p.ldh)) = og;
        *reinterpret_cast<uint4*>(p.gu_out + gu_offset(prow, p.ldh + j0 + c, 2 * p.ldh)) = ou;
      }
    }
  } else if (MODE == GEMM_DGRAD) {
    // v = dh for 128 columns f of F.  From the saved bf16 pre-activations g, u and the gate:
    //   s = silu(g) = g * sig(g),  s' = sig(g) * (1 + g * (1 - sig(g))) = sig(g) + s * (1 - sig(g))
    //   dG = dh * gate * u * s',  dU = dh * gate * s,  h = gate * s * u,  dgate += dh * s * u
    // dG, dU and h are rounded to bf16 (the tensors the backward hands between its GEMMs) and leave
    // this epilogue quantized the way the next GEMMs read them:
    //   [dG | dU] row-wise (blocks of 32 along 2F of this thread's row) -> codes [r_pad, 2F] and
    //     scale bytes, the dx GEMM's A operand;
    //   [dG | dU] and h column-wise (blocks of 32 rows: this warp's 32 lanes, one 32-row block of
    //     the expert because experts start at multiples of 256 padded rows) -> transposed codes
    //     [2F, r_pad] / [F, r_pad] and scale bytes, the weight-gradient GEMMs' operands.  Each
    //     32 x 32 block goes through the warp's 2 KB of shared memory: lanes write their rows, then
    //     lane l reads column l, takes its block scale and writes its 32 codes as one contiguous
    //     32-byte piece of a transposed row.
    // Padding rows carry zeros (gate 0, dh 0), so column blocks see zero rows there and their
    // row-wise codes are zero.
    const int64_t F = p.ldh;
    const int64_t prow = t.pad_row0 + r;
    const int f0 = t.n * 256 + 128 * half;
    if (f0 >= F) return;   // the half of the last column tile that lies past F (whole warps)
    const bool real = r < t.valid;
    const float gate = real ? (p.gates ? __ldg(p.gates + t.src_row0 + r) : 1.0f) : 0.0f;
    const uint64_t gate2 = f2_pack(gate, gate), one2 = f2_pack(1.0f, 1.0f), mone2 = f2_pack(-1.0f, -1.0f);
    uint64_t part2 = f2_pack(0.0f, 0.0f);
    uint32_t rsf_g = 0, rsf_u = 0;                 // row-wise scale bytes of this row's dG / dU blocks
    const int lane = static_cast<int>(threadIdx.x & 31);
    const int64_t prow0 = prow - lane;             // first row of the warp's 32-row block
#pragma unroll 1
    for (int b = 0; b < 4; ++b) {                  // 32 columns f0 + 32b .. (in v[0 .. 31])
      uint32_t dg[16], du[16];                     // bf16 pairs of columns (2i, 2i + 1) of the block
      if (b == 1) {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = v[32 + i];
      } else if (b >= 2) {                         // the upper 64 columns back from TMEM
        tmem_ld_32x32b_x32(t_park + 32 * (b - 2), v);
        tmem_ld_wait();
      }
      colblock_acquire(lane);
#pragma unroll
      for (int c16 = 0; c16 < 2; ++c16) {
        uint4 gw2[2] = {make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u)};
        uint4 uw2[2] = {gw2[0], gw2[0]};
        const int fc = f0 + 32 * b + 16 * c16;
        if (real) {   // blocked layout (gu_offset), prefetched into L2 at the tile's start
          gw2[0] = __ldcs(reinterpret_cast<const uint4*>(p.gu + gu_offset(prow, fc, 2 * F)));
          gw2[1] = __ldcs(reinterpret_cast<const uint4*>(p.gu + gu_offset(prow, fc + 8, 2 * F)));
          uw2[0] = __ldcs(reinterpret_cast<const uint4*>(p.gu + gu_offset(prow, F + fc, 2 * F)));
          uw2[1] = __ldcs(reinterpret_cast<const uint4*>(p.gu + gu_offset(prow, F + fc + 8, 2 * F)));
        }
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const uint32_t gw[4] = {gw2[hh].x, gw2[hh].y, gw2[hh].z, gw2[hh].w};
          const uint32_t uw[4] = {uw2[hh].x, uw2[hh].y, uw2[hh].z, uw2[hh].w};
          uint32_t hp[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {   // column pairs in f32x2 arithmetic
            const int k = 8 * c16 + 4 * hh + i;   // pair index inside the 32-column block
            const int c = 2 * k;                  // accumulator column (in v)
            const uint64_t g = f2_pack(bf16_lo(gw[i]), bf16_hi(gw[i]));
            const uint64_t u = f2_pack(bf16_lo(uw[i]), bf16_hi(uw[i]));
            const uint64_t dh = f2_pack(__uint_as_float(v[c]), __uint_as_float(v[c + 1]));
            const uint64_t d = f2_add(f2_pack(__expf(-f2_lo(g)), __expf(-f2_hi(g))), one2);   // 1 + e^-g
            const uint64_t sig = f2_pack(__fdividef(1.0f, f2_lo(d)), __fdividef(1.0f, f2_hi(d)));
            const uint64_t sl = f2_mul(g, sig);                                    // silu(g)
            const uint64_t su = f2_mul(sl, u);                                     // silu(g) u
            const uint64_t dsl = f2_fma(sl, f2_fma(sig, mone2, one2), sig);   // silu'(g) = sig + silu(g)(1 - sig)
            const uint64_t dhg = f2_mul(dh, gate2);
            part2 = f2_fma(dh, su, part2);
            const uint64_t dgv = f2_mul(f2_mul(dhg, u), dsl);
            const uint64_t duv = f2_mul(dhg, sl);
            const uint64_t hv = f2_mul(gate2, su);
            dg[k] = pack_bf16x2(f2_lo(dgv), f2_hi(dgv));
            du[k] = pack_bf16x2(f2_lo(duv), f2_hi(duv));
            hp[i] = pack_bf16x2(f2_lo(hv), f2_hi(hv));
          }
          colblock_put(wbuf, lane, 2 * c16 + hh, make_uint4(hp[0], hp[1], hp[2], hp[3]));   // h goes first
        }
      }
      const int fb = f0 + 32 * b;
      const int64_t cblk = prow0 >> 5;
      const int x = static_cast<int>(prow0);
      // h column-wise; [dG | dU] row-wise (this row's block of each) and column-wise.  Transposed
      // codes: rows [0, F) dG, [F, 2F) dU, [2F, 3F) h of one [3F, r_pad] matrix.
      p.hTsf[sf_mma_offset(fb + lane, cblk, p.t_kt)] =
          static_cast<uint8_t>(colblock_quantize(wbuf, lane, tmT, x, static_cast<int>(2 * F) + fb));
      rsf_g |= quantize_block32_to(dg, p.dguq + prow * 2 * F + fb) << (8 * b);
      colblock_acquire(lane);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        colblock_put(wbuf, lane, j, make_uint4(dg[4 * j], dg[4 * j + 1], dg[4 * j + 2], dg[4 * j + 3]));
      p.dguTsf[sf_mma_offset(fb + lane, cblk, p.t_kt)] =
          static_cast<uint8_t>(colblock_quantize(wbuf, lane, tmT, x, fb));
      rsf_u |= quantize_block32_to(du, p.dguq + prow * 2 * F + F + fb) << (8 * b);
      colblock_acquire(lane);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        colblock_put(wbuf, lane, j, make_uint4(du[4 * j], du[4 * j + 1], du[4 * j + 2], du[4 * j + 3]));
      p.dguTsf[sf_mma_offset(F + fb + lane, cblk, p.t_kt)] =
          static_cast<uint8_t>(colblock_quantize(wbuf, lane, tmT, x, static_cast<int>(F) + fb));
    }
    // row-wise scale bytes: blocks f0/32 .. +3 of dG and (F + f0)/32 .. +3 of dU, one word each
    *reinterpret_cast<uint32_t*>(p.dgusf + sf_mma_offset(prow, f0 / 32, 2 * F / 128)) = rsf_g;
    *reinterpret_cast<uint32_t*>(p.dgusf + sf_mma_offset(prow, (F + f0) / 32, 2 * F / 128)) = rsf_u;
    p.dgate_part[prow * (F / 128) + f0 / 128] = f2_lo(part2) + f2_hi(part2);
  } else {
    if (r < t.valid) {
      const int ncols = BN / 2;
      uint16_t* yrow = p.y + static_cast<int64_t>(t.src_row0 + r) * p.ldy + t.n * BN + ncols * half;
      auto val = [&](int i) {
        if constexpr (FMT == FMT_NV) return __fmul_rn(__uint_as_float(v[i]), alpha);
        return __uint_as_float(v[i]);
      };
#pragma unroll
      for (int c = 0; c < 128; c += 16) {
        if (c < ncols) {   // 16 columns = one 32-byte store
          uint4 o[2];
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const int cc = c + 8 * k;
            o[k].x = pack_bf16x2(val(cc + 0), val(cc + 1));
            o[k].y = pack_bf16x2(val(cc + 2), val(cc + 3));
            o[k].z = pack_bf16x2(val(cc + 4), val(cc + 5));
            o[k].w = pack_bf16x2(val(cc + 6), val(cc + 7));
          }
          st_global_32B(yrow + c, o[0], o[1]);
        }
      }
    }
  }
}

template <int MODE>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    k_grouped_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);  // tiles and scale atoms landed
  uint64_t* sf_full = full + STAGES;                                            // scales written to TMEM
  uint64_t* empty = sf_full + STAGES;                                           // MMAs done with the stage
  uint64_t* acc_full = empty + STAGES;
  uint64_t* acc_empty = acc_full + 1;
  uint64_t* drained = acc_empty + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drained + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&sf_full[s], NUM_SF_WARPS);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, NUM_EPI_WARPS);
    mbar_init(drained, 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == WARP_MMA) {
    tmem_alloc(tmem_holder, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  const int total_units = p.meta->num_mtiles * p.NT;
  const int BN = p.BN;

  if (warp < NUM_SF_WARPS) {
    regs_dec<REGS_LOW>();
    // ---------------- scale staging: shared memory -> TMEM (lanes of quarter `warp`) ----------------
    // Doing this with tcgen05.cp from the MMA thread stalled the tensor pipe (about a third of the
    // kernel's time); reading the atoms from global memory here instead of from the stage was
    // slower still (load latency under the TMA traffic).
    const uint32_t t_lanes = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const int nsfb = BN / 128;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < total_units; u += gridDim.x) {
      for (int kb = 0; kb < p.KT; ++kb) {
        bool got = true;
        if (threadIdx.x == 0) got = lane_wait(&full[stage], phase, abort_flag, p.timeout_ns, p.err, ERR_TIMEOUT_SF);
        if (!group_and(BAR_SF, NUM_SF_WARPS * 32, got)) {
          ok = false;
          break;
        }
        // row `lane` of each atom -> TMEM lane 32*warp + lane, 4 columns: every lane quarter holds
        // the whole atom, the layout the block-scaled MMA reads
        const uint8_t* sSFA = smem + stage * STAGE_BYTES + A_BYTES + B_BYTES_MAX;
        const uint8_t* sSFB = sSFA + SF_ATOM;
        tmem_st_32x32b_x4(t_lanes + SFA_COL + 4 * stage, *reinterpret_cast<const uint4*>(sSFA + lane * 16));
        tmem_st_32x32b_x4(t_lanes + SFB_COL + 8 * stage, *reinterpret_cast<const uint4*>(sSFB + lane * 16));
        if (nsfb == 2)
          tmem_st_32x32b_x4(t_lanes + SFB_COL + 8 * stage + 4,
                            *reinterpret_cast<const uint4*>(sSFB + SF_ATOM + lane * 16));
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sf_full[stage]);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else if (warp < FIRST_EPI_WARP) {
    regs_dec<REGS_LOW>();
    if (warp == WARP_PRODUCER) {
      // ---------------- TMA producer (lane 0 issues) ----------------
      uint32_t issued_mask = 0, issued_parity = 0;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      const uint32_t stage_tx = A_BYTES + BN * BK + SF_ATOM + (BN / 128) * SF_ATOM;
      for (int u = blockIdx.x; ok && u < total_units; u += gridDim.x) {
        TileInfo t;
        decode_unit(u, p, t);
        const int a_tile = t.pad_row0 / BM;
        for (int kb = 0; kb < p.KT; ++kb) {
          if (!warp_wait(&empty[stage], phase ^ 1u, abort_flag, p.timeout_ns, p.err, ERR_TIMEOUT_PRODUCER, lane)) {
            ok = false;
            break;
          }
          if (lane == 0) {
            uint8_t* sA = smem + stage * STAGE_BYTES;
            uint8_t* sB = sA + A_BYTES;
            uint8_t* sSFA = sB + B_BYTES_MAX;
            uint8_t* sSFB = sSFA + SF_ATOM;
            mbar_arrive_expect_tx(&full[stage], stage_tx);
            tma_load_2d(sA, &tmA, &full[stage], kb * BK, t.pad_row0);
            bulk_load(sSFA, p.a_sf + (static_cast<int64_t>(a_tile) * p.KT + kb) * SF_ATOM, SF_ATOM, &full[stage]);
            if (MODE == GEMM_SWIGLU) {
              const int g0 = b_box_row<MODE>(p, t, 0);   // gate rows
              const int u0 = b_box_row<MODE>(p, t, 1);   // up rows
              tma_load_2d(sB, &tmB, &full[stage], kb * BK, g0);
              tma_load_2d(sB + 128 * BK, &tmB, &full[stage], kb * BK, u0);
              bulk_load(sSFB, p.b_sf + (static_cast<int64_t>(g0 / 128) * p.KT + kb) * SF_ATOM, SF_ATOM, &full[stage]);
              bulk_load(sSFB + SF_ATOM, p.b_sf + (static_cast<int64_t>(u0 / 128) * p.KT + kb) * SF_ATOM, SF_ATOM,
                        &full[stage]);
            } else {
              // written out rather than looped: a runtime-count loop around these copies measured
              // 25% slower (GroupedLinear 1, same copies in the same order)
              const int b0 = b_box_row<MODE>(p, t, 0);
              tma_load_2d(sB, &tmB, &full[stage], kb * BK, b0);
              if (BN == 256) tma_load_2d(sB + 128 * BK, &tmB, &full[stage], kb * BK, b0 + 128);
              bulk_load(sSFB, p.b_sf + (static_cast<int64_t>(b0 / 128) * p.KT + kb) * SF_ATOM, SF_ATOM, &full[stage]);
              if (BN == 256)
                bulk_load(sSFB + SF_ATOM, p.b_sf + (static_cast<int64_t>(b0 / 128 + 1) * p.KT + kb) * SF_ATOM, SF_ATOM,
                          &full[stage]);
            }
          }
          __syncwarp();
          issued_mask |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Every copy this warp started must land before the CTA may exit.
      if (lane == 0)
        for (int s = 0; s < STAGES; ++s)
          if ((issued_mask >> s) & 1u)
            if (!mbar_wait_bounded(&full[s], (issued_parity >> s) & 1u, nullptr, p.drain_ns))
              atomicOr(p.err, ERR_TIMEOUT_DRAIN);
      __syncwarp();
    } else if (warp == WARP_MMA) {
      // ---------------- MMA issuer (the loop runs in lane 0 alone) ----------------
      if (lane == 0) {
        const uint32_t idesc = idesc_mxf8_e4m3(BM, BN);
        int stage = 0;
        uint32_t phase = 0, acc_phase = 0;
        bool issued = false, ok = true;
        for (int u = blockIdx.x; ok && u < total_units; u += gridDim.x) {
          if (!lane_wait(acc_empty, acc_phase ^ 1u, abort_flag, p.timeout_ns, p.err, ERR_TIMEOUT_MMA)) break;
          tc_fence_after();
          for (int kb = 0; kb < p.KT; ++kb) {
            // sf_full implies full: the scale warps waited for the stage's data before signalling
            if (!lane_wait(&sf_full[stage], phase, abort_flag, p.timeout_ns, p.err, ERR_TIMEOUT_MMA)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a0 = smem_u32(smem + stage * STAGE_BYTES), b0 = a0 + A_BYTES;
            const uint32_t t_sfa = tmem + SFA_COL + 4 * stage;
            const uint32_t t_sfb = tmem + SFB_COL + 8 * stage;
#pragma unroll
            for (int k = 0; k < BK / 32; ++k) {
              tc_mma_mxf8(tmem + ACC_COL, sdesc_kmajor_sw128(a0 + 32 * k), sdesc_kmajor_sw128(b0 + 32 * k),
                          idesc_with_sf_id(idesc, k), t_sfa, t_sfb, (kb | k) != 0 ? 1u : 0u);
            }
            tc_commit(&empty[stage]);
            issued = true;
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          tc_commit(acc_full);
          acc_phase ^= 1u;
        }
        if (issued) {
          tc_commit(drained);
          if (!mbar_wait_bounded(drained, 0, nullptr, p.drain_ns)) atomicOr(p.err, ERR_TIMEOUT_DRAIN);
        }
      }
      __syncwarp();
    }
  } else {
    regs_inc<REGS_HIGH>();
    // ---------------- epilogue ----------------
    const int quarter = warp & 3;                        // TMEM lanes this warp may read
    const int half = (warp - FIRST_EPI_WARP) >> 2;       // which half of the accumulator columns
    const int r = quarter * 32 + lane;                   // tile row held by this thread
    const uint32_t t_row = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    uint32_t acc_phase = 0;
    for (int u = blockIdx.x; u < total_units; u += gridDim.x) {
      TileInfo t;
      decode_unit(u, p, t);
      bool got = true;
      if (warp == FIRST_EPI_WARP && lane == 0)
        got = lane_wait(acc_full, acc_phase, abort_flag, p.timeout_ns, p.err, ERR_TIMEOUT_EPILOGUE);
      if (!group_and(BAR_EPI, NUM_EPI_WARPS * 32, got)) break;
      tc_fence_after();
      uint32_t v[128];
      if (MODE == GEMM_SWIGLU) {
        // gate columns [64*half, 64*half + 64) and the matching up columns 128 further on
        tmem_ld_32x32b_x32(t_row + ACC_COL + 64 * half, v);
        tmem_ld_32x32b_x32(t_row + ACC_COL + 64 * half + 32, v + 32);
        tmem_ld_32x32b_x32(t_row + ACC_COL + 128 + 64 * half, v + 64);
        tmem_ld_32x32b_x32(t_row + ACC_COL + 128 + 64 * half + 32, v + 96);
      } else {
        if (BN == 256) {
          tmem_ld_32x32b_x32(t_row + ACC_COL + 128 * half, v);
          tmem_ld_32x32b_x32(t_row + ACC_COL + 128 * half + 32, v + 32);
          tmem_ld_32x32b_x32(t_row + ACC_COL + 128 * half + 64, v + 64);
          tmem_ld_32x32b_x32(t_row + ACC_COL + 128 * half + 96, v + 96);
        } else {
          tmem_ld_32x32b_x32(t_row + ACC_COL + 64 * half, v);
          tmem_ld_32x32b_x32(t_row + ACC_COL + 64 * half + 32, v + 32);
        }
      }
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty);   // accumulator may be overwritten from here on
      acc_phase ^= 1u;

      epilogue_tile<MODE>(p, t, v, r, half, BN);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == WARP_MMA) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------------------------
// CTA-pair kernel: one tcgen05.mma.cta_group::2 computes a 256 x 256 tile on two SMs.
// CTA rank r of the pair holds row tile 2q + r of the expert (its 128 rows of A) and half of the
// 256-row B tile (GroupedLinear 1: r = 0 the gate rows, r = 1 the up rows; GroupedLinear 2: W2 rows
// 256n + 128r ..), so each SM loads 32 KB per K step for the same MMA work that costs the
// single-CTA kernel 48 KB.  Each CTA's TMEM receives its own 128 rows x 256 columns of the
// accumulator.
//
// A stage of the data ring holds two K steps (K = 256: 8 MMAs per barrier wait; a tile with an odd
// number of steps ends on a half stage).  The MMA thread shares its warp scheduler with two
// epilogue warps; while those run their math, every instruction of the issuing loop waits longer,
// and with one wait per 4 MMAs the tensor pipe ran dry in those stretches (K = 128 stages: about
// 10% slower GroupedLinear 1).
//
// Synchronization is arranged so that the data ring has one hop per direction:
//   full[s]      (leader)  both CTAs' tile copies complete on the leader's barrier (.cta_group::2
//                          copies); the leader's producer posts the byte count of both halves
//   empty[s]     (both)    the leader's MMA commit, multicast to both CTAs
// and the accumulator hand-off:
//   acc_full     (both)    the tile's MMAs completed (leader's commit, multicast)
//   acc_empty    (leader)  both CTAs' epilogues read their accumulator out (16 warp arrivals)
// The block scales of a K step (this CTA's A atom and both B atoms, 3 x 512 bytes) travel in the
// same stage as its tiles, by TMA onto the same barrier.  The MMA thread copies them into TMEM with
// tcgen05.cp just before the step's MMAs: copies and MMAs issued by one thread run in order, so no
// other warp and no other barrier takes part.  A TMEM scale slot belongs to one sub-buffer of the
// ring and is rewritten only after the stage's empty barrier, i.e. after the MMAs that read it.
// (A separate 16-slot scale ring, filled by four tcgen05.st warps and a second producer and
// synchronized by three more barrier kinds, was about 3% slower on GroupedLinear 1.)
// Warp roles: warp 4 producer (both CTAs), warp 5 MMA issuer (leader CTA; the MMA warp of the
// second CTA only takes part in the TMEM allocation), warps 8-15 epilogue, warps 0-3 NVFP4 scale
// staging (FMT_NV); the other role warps idle.
// ---------------------------------------------------------------------------------------------
constexpr int P_STEP_BYTES = 2 * 128 * BK;                    // own A tile + own half of the B tile
// Epilogue staging: each epilogue warp owns 2 KB of shared memory, used as two 1 KB buffers of
// 32 rows x 32 bytes (32B swizzle) for TMA stores of 16 bf16 columns of y (GEMM_OUT), as one 2 KB
// buffer of 32 rows x 16 fp32 columns for the weight gradients' TMA stores (GEMM_WGRAD), or as one
// 32 x 32 bf16 block that GEMM_DGRAD transposes through
constexpr int P_WG_BUF_BYTES = 1024;                           // per warp: two of these
constexpr int P_WG_CHUNK = 16;                                 // GEMM_WGRAD: fp32 columns per TMA store
constexpr int P_EPI_BYTES = NUM_EPI_WARPS * 2 * P_WG_BUF_BYTES;
// GEMM_DGRAD (MXFP8): TMEM columns past the scale slots where each epilogue warp parks the upper
// 64 of its 128 accumulator columns (64 * half + 0 .. 63).
constexpr uint32_t P_PARK_COL = 384;
constexpr uint32_t P_REGS_LOW = 64;
constexpr uint32_t P_REGS_HIGH = 192;
static_assert(2 * 128 * P_REGS_LOW + 256 * P_REGS_HIGH == NUM_THREADS * 128, "register split must equal the launch pool");

// Shared-memory and TMEM layout of the pair kernel per format.  A stage holds SUB K steps; a
// step's sub-buffer holds the CTA's own A tile, its half of the B tile and the step's scale atoms
// (own A atoms, then the atoms of both B halves).  One TMEM scale slot per sub-buffer.
//   MXFP8: the MMA thread copies the step's 3 atoms into the slot (tcgen05.cp); A: 4 columns
//          (row 32j+i of the atom at lane i of every quarter, column j), B: 8 (two atoms).
//   NVFP4: each CTA's four otherwise idle role warps write the slot with tcgen05.st, each into its
//          own TMEM lane quarter (twelve tcgen05.cp per step in the MMA thread's stream cost a
//          quarter of the GEMM time).  The image is the one the copies would leave: MMA k's A atom
//          at SFA + 4k (row 32j+i at lane i of every quarter, column j), its two B atoms at
//          SFB + 8k (+4); every scale address stays a multiple of 4 columns.  With 48 columns per
//          slot, TMEM holds 4 slots beside the 256-column accumulator, hence 2 stages of 2 steps.
template <int FMT>
struct PairLayout {
  static constexpr int SF_ATOMS = FMT == FMT_NV ? 4 : 1;      // scale atoms per 128 rows per K step
  static constexpr int STAGES = FMT == FMT_NV ? 5 : 3;
  static constexpr int SUB = FMT == FMT_NV ? 1 : 2;          // K steps per stage
  static constexpr int SF_BYTES = 3 * SF_ATOMS * SF_ATOM;
  static constexpr int SUBBUF_BYTES = P_STEP_BYTES + (SF_BYTES + 1023) / 1024 * 1024;
  static constexpr int STAGE_BYTES = SUB * SUBBUF_BYTES;
  static constexpr int SF_SLOTS = STAGES * SUB;
  static constexpr int DATA_BYTES = STAGES * STAGE_BYTES;
  static constexpr int BAR_OFFSET = DATA_BYTES + P_EPI_BYTES;
  // full, empty per stage; NVFP4 also sf_full (this CTA's scale atoms landed) and sf_ready (both
  // CTAs' scales are in TMEM) per stage; acc_full, acc_empty, drained
  static constexpr int NUM_BARS = (FMT == FMT_NV ? 4 : 2) * STAGES + 3;
  static constexpr int SMEM_BYTES = BAR_OFFSET + NUM_BARS * 8 + 8 + 1024;
  static constexpr uint32_t SFA_SLOT_COLS = FMT == FMT_NV ? 16 : 4;
  static constexpr uint32_t SFB_SLOT_COLS = FMT == FMT_NV ? 32 : 8;
  static constexpr uint32_t SFA_COL = 256;
  static constexpr uint32_t SFB_COL = SFA_COL + SFA_SLOT_COLS * SF_SLOTS;
  static_assert(P_STEP_BYTES % 1024 == 0 && SUBBUF_BYTES % 1024 == 0, "pair stages keep 1024-byte alignment");
  static_assert(SFB_COL + SFB_SLOT_COLS * SF_SLOTS <= TMEM_COLS, "pair TMEM budget");
  static_assert(FMT != FMT_MX || (SFB_COL + SFB_SLOT_COLS * SF_SLOTS <= P_PARK_COL && P_PARK_COL + 128 <= TMEM_COLS),
                "GEMM_DGRAD parking columns");
  static_assert(SMEM_BYTES <= 232448, "pair shared memory budget");
};

// Pair unit u -> (expert, column tile, pair of row tiles); this CTA takes row tile 2q + rank.
// Experts own an even number of 128-row tiles (their rows are padded to a multiple of 256).
__device__ __forceinline__ void decode_pair_unit(int u, int rank, const GemmParams& p, TileInfo& t) {
  const int32_t* row_off = reinterpret_cast<const int32_t*>(p.meta + 1);
  const int32_t* pad_off = row_off + (p.E + 1);
  const int32_t* mt_off = pad_off + (p.E + 1);
  int lo = 0, hi = p.E;  // largest e with (mt_off[e] / 2) * NT <= u (skips empty experts)
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if ((__ldg(mt_off + mid) >> 1) * p.NT <= u) lo = mid; else hi = mid;
  }
  const int e = lo;
  const int q0 = __ldg(mt_off + e) >> 1;
  const int pairs = (__ldg(mt_off + e + 1) >> 1) - q0;
  const int local = u - q0 * p.NT;
  int n, q;
  if (p.n_fastest && p.group_m > 0) {
    const int g = local / (p.group_m * p.NT);          // group of group_m row pairs
    const int in_g = min(p.group_m, pairs - g * p.group_m);
    const int w = local - g * p.group_m * p.NT;
    n = w / in_g;
    q = g * p.group_m + (w - n * in_g);
  } else if (p.n_fastest) {
    q = local / p.NT;
    n = local - q * p.NT;
  } else {
    n = local / pairs;
    q = local - n * pairs;
  }
  const int tt = 2 * q + rank;
  const int r0 = __ldg(row_off + e);
  t.e = e;
  t.n = n;
  t.pad_row0 = __ldg(pad_off + e) + BM * tt;
  t.src_row0 = r0 + BM * tt;
  t.valid = min(BM, __ldg(row_off + e + 1) - r0 - BM * tt);
}

// Pair unit u -> this CTA's tile: rows of its A tile, the pair's two B halves, K offsets and K
// steps.  Forward and dgrad modes: A rows are expert-padded activation rows (row-tile pairs of an
// expert, decode_pair_unit), B rows are weight rows.  GEMM_WGRAD: units run expert by expert over
// (256-row tile of A's rows, 256-row tile of B's rows) with B tiles fastest, and the K range is the
// expert's padded rows (no steps for an empty expert).
template <int MODE>
__device__ __forceinline__ void decode_pair_tile(int u, int rank, const GemmParams& p, TileInfo& t) {
  if constexpr (MODE == GEMM_WGRAD) {
    const int32_t* pad_off = reinterpret_cast<const int32_t*>(p.meta + 1) + (p.E + 1);
    const int per = p.wg_mt * p.wg_nt;
    const int e = u / per;
    const int rem = u - e * per;
    int mt;
    if (p.wg_m_fastest) {
      t.n = rem / p.wg_mt;
      mt = rem - t.n * p.wg_mt;
    } else {
      mt = rem / p.wg_nt;
      t.n = rem - mt * p.wg_nt;
    }
    t.e = e;
    t.a_row = mt * 256 + 128 * rank;
    t.b_row0 = t.n * 256;
    t.b_row1 = t.n * 256 + 128;
    t.a_k0 = __ldg(pad_off + e);
    t.b_k0 = t.a_k0;
    t.steps = (__ldg(pad_off + e + 1) - t.a_k0) / BK;
    t.pad_row0 = t.a_row;
    t.src_row0 = 0;
    t.valid = BM;
  } else {
    decode_pair_unit(u, rank, p, t);
    t.a_row = t.pad_row0;
    t.b_row0 = b_box_row<MODE>(p, t, 0);
    t.b_row1 = b_box_row<MODE>(p, t, 1);
    t.a_k0 = 0;
    t.b_k0 = t.e * p.b_kofs;
    t.steps = p.KT;
  }
}

template <int MODE>
__device__ __forceinline__ int pair_total_units(const GemmParams& p) {
  if constexpr (MODE == GEMM_WGRAD) return p.E * p.wg_mt * p.wg_nt;
  return (p.meta->num_mtiles >> 1) * p.NT;
}

// Bounded wait shared by the warp (lane 0 polls).  On timeout it records `err_bit`, and raises the
// abort flag of this CTA and of the other CTA of the pair so that every role of both drains.
__device__ __forceinline__ bool pair_wait(uint64_t* bar, uint32_t parity, const volatile int* abort,
                                          uint32_t peer_abort, const GemmParams& p, uint32_t err_bit, int lane) {
  int ok = 1;
  if (lane == 0) {
    ok = mbar_wait_bounded(bar, parity, abort, p.timeout_ns) ? 1 : 0;
    if (!ok) {
      atomicOr(p.err, err_bit);
      *const_cast<volatile int*>(abort) = 1;
      st_remote_u32(peer_abort, 1u);
    }
  }
  return __shfl_sync(0xFFFFFFFFu, ok, 0) != 0;
}

// Barriers completed by hardware (tile copies, MMA commits) are waited on with CTA-scope acquire
// even where the other CTA's copies or the leader's commits complete them: their data is visible
// once the phase completes.  Barriers that threads of the other CTA arrive on (scale warps after
// tcgen05.wait::st, epilogue warps after tcgen05.wait::ld) are waited on with cluster-scope acquire.
__device__ __forceinline__ bool pair_lane_wait(uint64_t* bar, uint32_t parity, bool cluster_scope, const volatile int* abort,
                                               uint32_t peer_abort, const GemmParams& p, uint32_t err_bit) {
  if (cluster_scope ? mbar_wait_cluster_bounded(bar, parity, abort, p.timeout_ns)
                    : mbar_wait_bounded(bar, parity, abort, p.timeout_ns))
    return true;
  atomicOr(p.err, err_bit);
  *const_cast<volatile int*>(abort) = 1;
  st_remote_u32(peer_abort, 1u);
  return false;
}

template <int MODE, int FMT>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    k_grouped_gemm_pair(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmSB,
                        const __grid_constant__ CUtensorMap tmD, const GemmParams p) {
  using L = PairLayout<FMT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::BAR_OFFSET);
  uint64_t* empty = full + L::STAGES;
  uint64_t* acc_full = empty + L::STAGES;
  uint64_t* acc_empty = acc_full + 1;
  uint64_t* drained = acc_empty + 1;
  uint64_t* sf_full = drained + 1;            // NVFP4 only
  uint64_t* sf_ready = sf_full + L::STAGES;   // NVFP4 only (waited on in the leader)
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drained + 1 + (FMT == FMT_NV ? 2 * L::STAGES : 0));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_cta_rank();
  const bool leader = rank == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < L::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      if constexpr (FMT == FMT_NV) {
        mbar_init(&sf_full[s], 1);
        mbar_init(&sf_ready[s], 2 * NUM_SF_WARPS);
      }
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 2 * NUM_EPI_WARPS);
    mbar_init(drained, 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == WARP_MMA) {   // one warp of each CTA of the pair allocates collectively
    tmem_alloc_pair(tmem_holder, TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();   // the peer's barriers exist before any remote arrive, copy or commit
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  const int total_units = pair_total_units<MODE>(p);
  const int first_unit = static_cast<int>(cluster_index());
  const int unit_stride = static_cast<int>(cluster_count());
  const uint32_t peer_abort = map_to_cta(const_cast<int*>(abort_flag), rank ^ 1u);
  uint32_t prod_issued = 0;   // producer warp: stages it issued copies for
  if (warp < FIRST_EPI_WARP) {
    regs_dec<P_REGS_LOW>();
    if (warp == WARP_PRODUCER) {
      // ---------------- tile producer (both CTAs; lane 0 issues) ----------------
      const uint32_t leader_full = map_to_cta(full, 0);
      const uint64_t keep_policy = l2_policy_evict_last();
      uint32_t issued_mask = 0, issued_parity = 0;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int u = first_unit; ok && u < total_units; u += unit_stride) {
        TileInfo t;
        decode_pair_tile<MODE>(u, static_cast<int>(rank), p, t);
        const int b_own = rank == 0 ? t.b_row0 : t.b_row1;
        // scale atoms (512 bytes: 128 rows x 4 blocks) of the tile's first K step; step kb adds kb.
        // Past the end of B (half of a last tile) any valid atom will do: those B rows are zeros.
        const int a_atom0 = (t.a_row / 128) * p.a_kt + L::SF_ATOMS * (t.a_k0 / BK);
        const int b_atom0 = (t.b_row0 / 128) * p.b_kt + L::SF_ATOMS * (t.b_k0 / BK);
        const int b_row1 = (p.b_rows > 0 && t.b_row1 >= p.b_rows) ? t.b_row0 : t.b_row1;
        const int b_atom1 = (b_row1 / 128) * p.b_kt + L::SF_ATOMS * (t.b_k0 / BK);
        if constexpr (MODE == GEMM_DGRAD) {
          // the epilogue of this tile reads the saved g and u of its 128 rows x 256 columns of F:
          // have L2 fetch them while the tile's MMAs run (in the blocked layout each 32-row block's
          // 256 columns of G, and of U, are 16 KB in one piece)
          if (lane < 8) {
            const int64_t prow = t.pad_row0 + 32 * (lane & 3);
            const int64_t j = (lane < 4 ? 0 : p.ldh) + t.n * 256;
            prefetch_l2(p.gu + gu_offset(prow, j, 2 * p.ldh), t.n * 256 + 256 <= p.ldh ? 16384 : 8192);
          }
        }
        for (int kb = 0, nsub = 0; kb < t.steps; kb += nsub) {
          nsub = min(L::SUB, t.steps - kb);
          if (!pair_wait(&empty[stage], phase ^ 1u, abort_flag, peer_abort, p, ERR_TIMEOUT_PRODUCER, lane)) {
            ok = false;
            break;
          }
          if (lane == 0) {
            const uint32_t bar = leader_full + stage * 8;
            for (int j = 0; j < nsub; ++j) {
              uint8_t* sA = smem + stage * L::STAGE_BYTES + j * L::SUBBUF_BYTES;
              const int k0 = (kb + j) * BK;
              if constexpr (MODE == GEMM_DGRAD)   // dy tiles are reused by every column tile: keep them in L2
                tma_load_2d_pair_hint(sA, &tmA, bar, t.a_k0 + k0, t.a_row, keep_policy);
              else
                tma_load_2d_pair(sA, &tmA, bar, t.a_k0 + k0, t.a_row);
              tma_load_2d_pair(sA + A_BYTES, &tmB, bar, t.b_k0 + k0, b_own);
              // scale atoms: 2 rows of 256 bytes each in the maps; a box holds the step's SF_ATOMS atoms
              // (NVFP4: onto this CTA's own sf_full, which its scale warps wait on)
              uint8_t* sS = sA + P_STEP_BYTES;
              const int ka = L::SF_ATOMS * (kb + j);
              if constexpr (FMT == FMT_NV) {
                tma_load_2d(sS, &tmSA, &sf_full[stage], 0, 2 * (a_atom0 + ka));
                tma_load_2d(sS + L::SF_ATOMS * SF_ATOM, &tmSB, &sf_full[stage], 0, 2 * (b_atom0 + ka));
                tma_load_2d(sS + 2 * L::SF_ATOMS * SF_ATOM, &tmSB, &sf_full[stage], 0, 2 * (b_atom1 + ka));
              } else {
                tma_load_2d_pair(sS, &tmSA, bar, 0, 2 * (a_atom0 + ka));
                tma_load_2d_pair(sS + SF_ATOM, &tmSB, bar, 0, 2 * (b_atom0 + ka));
                tma_load_2d_pair(sS + 2 * SF_ATOM, &tmSB, bar, 0, 2 * (b_atom1 + ka));
              }
            }
            if constexpr (FMT == FMT_NV) {
              if (leader) mbar_arrive_expect_tx(&full[stage], 2 * nsub * P_STEP_BYTES);
              mbar_arrive_expect_tx(&sf_full[stage], nsub * L::SF_BYTES);
            } else if (leader) {
              mbar_arrive_expect_tx(&full[stage], 2 * nsub * (P_STEP_BYTES + L::SF_BYTES));
            }
          }
          __syncwarp();
          ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
          issued_mask |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == L::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Copies must land before the CTA exits.  The leader's barriers count both CTAs' copies and
      // the MMA warp waits for every stage it consumes; after an abort, the leader waits here
      // (bounded) for the stages it issued.  The second CTA's copies complete on the leader's
      // barriers, so it cannot wait for them itself: after the pair's closing cluster barrier,
      // where every abort raised in either CTA is visible, it gives them a fixed 200 us to land
      // (they depend on nothing but memory) before a second cluster barrier lets either CTA exit.
      if (lane == 0 && leader)
        for (int s = 0; s < L::STAGES; ++s)
          if ((issued_mask >> s) & 1u)
            if (!mbar_wait_bounded(&full[s], (issued_parity >> s) & 1u, nullptr, p.drain_ns))
              atomicOr(p.err, ERR_TIMEOUT_DRAIN);
      if (FMT == FMT_NV && lane == 0)   // this CTA's own scale copies
        for (int s = 0; s < L::STAGES; ++s)
          if ((issued_mask >> s) & 1u)
            if (!mbar_wait_bounded(&sf_full[s], (issued_parity >> s) & 1u, nullptr, p.drain_ns))
              atomicOr(p.err, ERR_TIMEOUT_DRAIN);
      prod_issued = issued_mask;
      __syncwarp();
    } else if (warp == WARP_MMA && leader) {
      // ---------------- pair MMA issuer (leader CTA; the loop runs in lane 0 alone) ----------------
      if (lane == 0) {
        const uint32_t idesc = FMT == FMT_NV ? idesc_nvf4(2 * BM, 256) : idesc_mxf8_e4m3(2 * BM, 256);
        int stage = 0;
        uint32_t phase = 0, acc_phase = 0;
        bool issued = false, ok = true;
        for (int u = first_unit; ok && u < total_units; u += unit_stride) {
          int steps = p.KT;
          if constexpr (MODE == GEMM_WGRAD) {
            TileInfo t;
            decode_pair_tile<MODE>(u, 0, p, t);
            steps = t.steps;
            if (steps == 0) continue;   // empty expert: the epilogue writes zeros without the accumulator
          }
          if (!pair_lane_wait(acc_empty, acc_phase ^ 1u, true, abort_flag, peer_abort, p, ERR_TIMEOUT_MMA)) break;
          tc_fence_after();
          for (int kb = 0; kb < steps; kb += L::SUB) {
            // full: the stage's tiles and scale atoms are in both CTAs' shared memory (NVFP4: the
            // tiles; sf_ready: both CTAs' scale warps have written the stage's scales into TMEM)
            if (!pair_lane_wait(&full[stage], phase, false, abort_flag, peer_abort, p, ERR_TIMEOUT_MMA)) {
              ok = false;
              break;
            }
            if (FMT == FMT_NV && !pair_lane_wait(&sf_ready[stage], phase, true, abort_flag, peer_abort, p,
                                                 ERR_TIMEOUT_MMA)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t st0 = smem_u32(smem + stage * L::STAGE_BYTES);
#pragma unroll
            for (int j = 0; j < L::SUB; ++j) {
              if (j > 0 && kb + j >= steps) break;   // half stage at the end of an odd tile
              const uint32_t a0 = st0 + j * L::SUBBUF_BYTES, b0 = a0 + A_BYTES, sf0 = a0 + P_STEP_BYTES;
              const int slot = stage * L::SUB + j;
              const uint32_t t_sfa = tmem + L::SFA_COL + L::SFA_SLOT_COLS * slot;
              const uint32_t t_sfb = tmem + L::SFB_COL + L::SFB_SLOT_COLS * slot;
              if constexpr (FMT == FMT_NV) {
                // scales already in TMEM (scale warps): MMA k's A atom at t_sfa + 4k, B's at t_sfb + 8k
                (void)sf0;
#pragma unroll
                for (int k = 0; k < 4; ++k)
                  tc_mma_nvf4_pair(tmem + ACC_COL, sdesc_kmajor_sw128(a0 + 32 * k), sdesc_kmajor_sw128(b0 + 32 * k),
                                   idesc, t_sfa + 4 * k, t_sfb + 8 * k, ((kb + j) | k) != 0 ? 1u : 0u);
              } else {
                // scales of the step into TMEM (both CTAs, each from its own shared memory); the MMAs
                // below are issued after them by this thread and see them in order
                tc_copy_sf_pair(t_sfa, sdesc_sf_atom(sf0));
                tc_copy_sf_pair(t_sfb, sdesc_sf_atom(sf0 + SF_ATOM));
                tc_copy_sf_pair(t_sfb + 4, sdesc_sf_atom(sf0 + 2 * SF_ATOM));
#pragma unroll
                for (int k = 0; k < BK / 32; ++k) {
                  tc_mma_mxf8_pair(tmem + ACC_COL, sdesc_kmajor_sw128(a0 + 32 * k), sdesc_kmajor_sw128(b0 + 32 * k),
                                   idesc_with_sf_id(idesc, k), t_sfa, t_sfb, ((kb + j) | k) != 0 ? 1u : 0u);
                }
              }
            }
            tc_commit_pair_both(&empty[stage]);
            issued = true;
            if (++stage == L::STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          tc_commit_pair_both(acc_full);
          acc_phase ^= 1u;
        }
        if (issued) {
          tc_commit_pair_local(drained);
          if (!mbar_wait_bounded(drained, 0, nullptr, p.drain_ns)) atomicOr(p.err, ERR_TIMEOUT_DRAIN);
        }
      }
      __syncwarp();
    } else if (FMT == FMT_NV && warp < NUM_SF_WARPS) {
      // ---------------- NVFP4 scale staging (both CTAs; warp q writes TMEM lane quarter q) ----------------
      // Per step, lane i of every warp: the 16 bytes of row i of each A atom k (rows i, 32+i, 64+i,
      // 96+i) -> columns SFA + 4k .. +3, and of each B atom (half h, MMA k) -> SFB + 8k + 4h .. +3,
      // in the warp's own lane quarter: every quarter gets the same image.  The stage's scales land
      // on this CTA's sf_full; when both of its steps are written, each warp arrives on the leader's
      // sf_ready.
      const uint32_t q = static_cast<uint32_t>(warp & 3);
      const uint32_t t_lanes = tmem + ((32u * q) << 16);
      const uint32_t leader_sf_ready = map_to_cta(sf_ready, 0);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int u = first_unit; ok && u < total_units; u += unit_stride) {
        const int steps = p.KT;
        for (int kb = 0; kb < steps; kb += L::SUB) {
          if (!pair_wait(&sf_full[stage], phase, abort_flag, peer_abort, p, ERR_TIMEOUT_SF, lane)) {
            ok = false;
            break;
          }
#pragma unroll 1
          for (int j = 0; j < L::SUB; ++j) {
            if (j > 0 && kb + j >= steps) break;   // half stage at the end of an odd tile
            const uint8_t* sS = smem + stage * L::STAGE_BYTES + j * L::SUBBUF_BYTES + P_STEP_BYTES;
            const int slot = stage * L::SUB + j;
            uint32_t a[16];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint4 w = *reinterpret_cast<const uint4*>(sS + k * SF_ATOM + 16 * lane);
              a[4 * k + 0] = w.x;
              a[4 * k + 1] = w.y;
              a[4 * k + 2] = w.z;
              a[4 * k + 3] = w.w;
            }
            tmem_st_32x32b_x16(t_lanes + L::SFA_COL + L::SFA_SLOT_COLS * slot, a);
#pragma unroll
            for (int k0 = 0; k0 < 4; k0 += 2) {   // B atoms of MMAs k0, k0 + 1: 16 columns per store
              uint32_t b[16];
#pragma unroll
              for (int k = 0; k < 2; ++k)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                  const uint4 w = *reinterpret_cast<const uint4*>(sS + (4 + 4 * h + k0 + k) * SF_ATOM + 16 * lane);
                  b[8 * k + 4 * h + 0] = w.x;
                  b[8 * k + 4 * h + 1] = w.y;
                  b[8 * k + 4 * h + 2] = w.z;
                  b[8 * k + 4 * h + 3] = w.w;
                }
              tmem_st_32x32b_x16(t_lanes + L::SFB_COL + L::SFB_SLOT_COLS * slot + 8 * k0, b);
            }
          }
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            if (leader)
              mbar_arrive(&sf_ready[stage]);
            else
              mbar_arrive_remote(leader_sf_ready + 8u * static_cast<uint32_t>(stage));
          }
          if (++stage == L::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
  } else {
    regs_inc<P_REGS_HIGH>();
    // ---------------- epilogue (both CTAs, own 128 rows) ----------------
    const int quarter = warp & 3;
    const int half = (warp - FIRST_EPI_WARP) >> 2;
    const int r = quarter * 32 + lane;
    const uint32_t t_row = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t leader_acc_empty = map_to_cta(acc_empty, 0);
    float alpha = 1.0f, s_out = 1.0f;
    if constexpr (FMT == FMT_NV) {   // dequantization of the product: 1 / (s_a s_b)
      const float s_a = nv_encode_scale(p.nv_amax_a != nullptr ? *p.nv_amax_a : p.nv_amax_a_val);
      const float s_b = nv_encode_scale(*p.nv_amax_b);
      alpha = __frcp_rn(__fmul_rn(s_a, s_b));
      s_out = nv_encode_scale(p.nv_out_amax);
    }
    uint32_t acc_phase = 0;
    for (int u = first_unit; u < total_units; u += unit_stride) {
      TileInfo t;
      decode_pair_tile<MODE>(u, static_cast<int>(rank), p, t);
      if (MODE == GEMM_WGRAD && t.steps == 0) {   // expert without rows: its gradient block is zero
        if (t.n * 256 + 128 * half >= p.wg_n) continue;
        float* drow = p.dw + (static_cast<int64_t>(t.e) * p.wg_m + t.a_row + r) * p.wg_n + t.n * 256 + 128 * half;
        for (int c = 0; c < 128; c += 8) st_global_32B_cs(drow + c, make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u));
        continue;
      }
      bool got = true;
      if (warp == FIRST_EPI_WARP && lane == 0)
        got = pair_lane_wait(acc_full, acc_phase, false, abort_flag, peer_abort, p, ERR_TIMEOUT_EPILOGUE);
      if (!group_and(BAR_EPI, NUM_EPI_WARPS * 32, got)) break;
      tc_fence_after();
      uint32_t v[128];
      if (MODE == GEMM_SWIGLU) {
        tmem_ld_32x32b_x32(t_row + ACC_COL + 64 * half, v);
        tmem_ld_32x32b_x32(t_row + ACC_COL + 64 * half + 32, v + 32);
        tmem_ld_32x32b_x32(t_row + ACC_COL + 128 + 64 * half, v + 64);
        tmem_ld_32x32b_x32(t_row + ACC_COL + 128 + 64 * half + 32, v + 96);
      } else {
        tmem_ld_32x32b_x32(t_row + ACC_COL + 128 * half, v);
        tmem_ld_32x32b_x32(t_row + ACC_COL + 128 * half + 32, v + 32);
        tmem_ld_32x32b_x32(t_row + ACC_COL + 128 * half + 64, v + 64);
        tmem_ld_32x32b_x32(t_row + ACC_COL + 128 * half + 96, v + 96);
      }
      tmem_ld_wait();
      if constexpr (MODE == GEMM_DGRAD) {
        // the upper 64 of the 128 columns wait in TMEM columns no MMA writes (registers hold 64
        // fewer values through the first half of the epilogue)
        tmem_st_32x32b_x16(t_row + P_PARK_COL + 64 * half, v + 64);
        tmem_st_32x32b_x16(t_row + P_PARK_COL + 64 * half + 16, v + 80);
        tmem_st_32x32b_x16(t_row + P_PARK_COL + 64 * half + 32, v + 96);
        tmem_st_32x32b_x16(t_row + P_PARK_COL + 64 * half + 48, v + 112);
        tmem_st_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(leader_acc_empty);   // the leader may overwrite TMEM
      acc_phase ^= 1u;
      if constexpr (MODE == GEMM_WGRAD) {
        // 128 fp32 columns of this warp's 32 rows, 16 columns per TMA store from the warp's 2 KB
        // staging buffer (row-per-lane global stores touched 32 rows per instruction and held the
        // epilogue up; eight 2 KB stores per tile half beat sixteen 1 KB ones double-buffered, and
        // thirty-two 512-byte ones four-buffered were slower still: the stores' count matters).
        if (t.n * 256 + 128 * half < p.wg_n) {
          const int col0 = t.n * 256 + 128 * half;
          const int grow = t.e * p.wg_m + t.a_row + quarter * 32;   // row in the [E * wg_m, wg_n] view
          uint8_t* wbuf = smem + L::DATA_BYTES + (warp - FIRST_EPI_WARP) * 2 * P_WG_BUF_BYTES;
#pragma unroll
          for (int c = 0; c < 128; c += P_WG_CHUNK) {
            uint8_t* buf = wbuf;
            if (lane == 0) bulk_wait_read_all();   // the previous store has read the buffer
            __syncwarp();
            // row `lane`: four 16-byte chunks (64 bytes), 64B swizzle (chunk j of row i at
            // j ^ ((i >> 1) & 3)), so that the eight rows of each shared-memory wavefront fall in
            // distinct banks (unswizzled 64-byte rows put four of them in one bank group)
#pragma unroll
            for (int j = 0; j < 4; ++j)
              *reinterpret_cast<uint4*>(buf + lane * 64 + 16 * (j ^ ((lane >> 1) & 3))) =
                  make_uint4(v[c + 4 * j], v[c + 4 * j + 1], v[c + 4 * j + 2], v[c + 4 * j + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmD, buf, col0 + c, grow);
              bulk_commit_group();
            }
          }
        }
      } else if (MODE == GEMM_OUT) {
        // y: 16 bf16 columns at a time.  A warp whose 32 rows are all real rows of the expert writes
        // them by TMA stores from a double-buffered 1 KB staging area: a warp instruction writes 512
        // contiguous bytes of shared memory and the rows leave as whole lines (row-per-lane 32-byte
        // global stores touch 32 lines per instruction and throttled the epilogue of short-K
        // tiles).  A warp whose rows run past the expert's last row stores its real rows directly:
        // y is not padded, the next rows belong to the next expert.
        const bool via_tma = p.y_rows > 0 && quarter * 32 + 31 < t.valid;
        const int col0 = t.n * 256 + 128 * half;
        const int grow = t.src_row0 + quarter * 32;
        uint8_t* wbuf = smem + L::DATA_BYTES + (warp - FIRST_EPI_WARP) * 2 * P_WG_BUF_BYTES;
        uint16_t* yrow = p.y + static_cast<int64_t>(t.src_row0 + r) * p.ldy + col0;
        auto val = [&](int i) {
          if constexpr (FMT == FMT_NV) return __fmul_rn(__uint_as_float(v[i]), alpha);
          return __uint_as_float(v[i]);
        };
#pragma unroll
        for (int c = 0; c < 128; c += 16) {
          uint4 o[2];
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const int cc = c + 8 * k;
            o[k].x = pack_bf16x2(val(cc + 0), val(cc + 1));
            o[k].y = pack_bf16x2(val(cc + 2), val(cc + 3));
            o[k].z = pack_bf16x2(val(cc + 4), val(cc + 5));
            o[k].w = pack_bf16x2(val(cc + 6), val(cc + 7));
          }
          if (via_tma) {
            uint8_t* buf = wbuf + ((c / 16) & 1) * P_WG_BUF_BYTES;
            if (lane == 0) bulk_wait_read_le1();   // the store that last used this buffer has read it
            __syncwarp();
            // row `lane`: two 16-byte chunks, 32B swizzle (chunk j of row i at j ^ ((i >> 2) & 1))
            const int sw = (lane >> 2) & 1;
            *reinterpret_cast<uint4*>(buf + lane * 32 + 16 * sw) = o[0];
            *reinterpret_cast<uint4*>(buf + lane * 32 + 16 * (sw ^ 1)) = o[1];
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmD, buf, col0 + c, grow);
              bulk_commit_group();
            }
          } else if (r < t.valid) {
            st_global_32B(yrow + c, o[0], o[1]);
          }
        }
      } else {
        // GroupedLinear 1: the two warps of a lane quarter share a scheduler with each other and
        // (for one quarter) with the MMA thread; they run their SwiGLU/quantize math one after the
        // other, so at most one of them competes for issue slots at a time (1.5% faster).  Half 0
        // is never a tile ahead of half 1: both pass the epilogue barrier of every tile.
        if (MODE == GEMM_SWIGLU && half == 1) asm volatile("bar.sync %0, 64;" ::"r"(BAR_STAGGER + quarter) : "memory");
        epilogue_tile<MODE, FMT>(p, t, v, r, half, 256, alpha, s_out,
                                 smem + L::DATA_BYTES + (warp - FIRST_EPI_WARP) * 2 * P_WG_BUF_BYTES,
                                 t_row + P_PARK_COL + 64 * half, &tmD);
        if (MODE == GEMM_SWIGLU && half == 0) asm volatile("bar.arrive %0, 64;" ::"r"(BAR_STAGGER + quarter) : "memory");
      }
    }
    if ((MODE == GEMM_WGRAD || MODE == GEMM_OUT || MODE == GEMM_DGRAD) && lane == 0)
      bulk_wait_all();   // stores complete before exit
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();   // all pair MMAs are done and no remote arrive targets an exited CTA
  if (!leader && warp == WARP_PRODUCER && lane == 0 && prod_issued != 0 && *abort_flag) {
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 200000ull) {
    }
  }
  cluster_sync_all();   // the second CTA's copies have landed on the leader's barriers
  if (warp == WARP_MMA) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem, TMEM_COLS);
  }
}

// One block of 1024 threads: inclusive scans of split sizes and of 128-row tile counts.  Every
// expert gets an even number of tiles (its rows padded to a multiple of 256), so the pair kernel's
// two row tiles always belong to one expert.
__global__ void __launch_bounds__(1024) k_schedule(const int32_t* split, int E, int64_t R, SchedHeader* meta) {
  __shared__ long long s_rows[1024];
  __shared__ int s_tiles[1024];

  __shared__ int s_neg;
  const int t = threadIdx.x;
  if (t == 0) s_neg = 0;
  __syncthreads();
  int v = t < E ? split[t] : 0;
  if (v < 0) {
    atomicOr(&s_neg, 1);
    v = 0;
  }
  s_rows[t] = v;
  s_tiles[t] = 2 * ((v + 2 * BM - 1) / (2 * BM));
  __syncthreads();
  for (int d = 1; d < 1024; d <<= 1) {
    const long long a = t >= d ? s_rows[t - d] : 0;
    const int b = t >= d ? s_tiles[t - d] : 0;
    __syncthreads();
    s_rows[t] += a;
    s_tiles[t] += b;
    __syncthreads();
  }
  int32_t* row_off = reinterpret_cast<int32_t*>(meta + 1);
  int32_t* pad_off = row_off + (E + 1);
  int32_t* mt_off = pad_off + (E + 1);
  const long long total = s_rows[E - 1];
  const bool bad = s_neg || total != R;
  if (t < E) {
    const long long rows_before = t == 0 ? 0 : s_rows[t - 1];
    const int tiles_before = t == 0 ? 0 : s_tiles[t - 1];
    row_off[t] = static_cast<int32_t>(rows_before);
    pad_off[t] = bad ? 0 : tiles_before * BM;
    mt_off[t] = bad ? 0 : tiles_before;
  }
  if (t == 0) {
    row_off[E] = static_cast<int32_t>(total);
    pad_off[E] = bad ? 0 : s_tiles[E - 1] * BM;
    mt_off[E] = bad ? 0 : s_tiles[E - 1];
    meta->error = (s_neg ? ERR_SPLIT_NEGATIVE : 0u) | (total != R ? ERR_SPLIT_SUM : 0u);
    meta->num_mtiles = bad ? 0 : s_tiles[E - 1];
    meta->pad_rows = bad ? 0 : s_tiles[E - 1] * BM;
    meta->E = E;
  }
}

// ---- host side -------------------------------------------------------------------------------

// Limit of every pipeline wait: 2 s, or the value in ns of the environment variable
// MXFP8MOE_WAIT_LIMIT_NS when it holds a positive integer (read at each call; failure-path tests
// use it to make waits run out without any change to the kernels).  Teardown waits for copies and
// MMAs in flight always keep the full 2 s.
uint64_t pipeline_wait_ns() {
  const char* v = getenv("MXFP8MOE_WAIT_LIMIT_NS");
  if (v == nullptr || *v == 0) return kWaitTimeoutNs;
  char* end = nullptr;
  const unsigned long long n = strtoull(v, &end, 10);
  return (end != nullptr && *end == 0 && n > 0) ? static_cast<uint64_t>(n) : kWaitTimeoutNs;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D byte matrix [rows, cols] (row pitch = cols), 128 x 128 boxes, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), static_cast<cuuint32_t>(BM)};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A tensor-core scale array (512-byte atoms) as a 2-D byte matrix of 256-byte rows, boxes of
// 2 * `box_atoms` rows: box (0, 2a) is atoms a .. a + box_atoms - 1.
bool make_sf_map(CUtensorMap* m, const void* base, uint64_t atoms, uint32_t box_atoms = 1) {
  auto enc = tensor_map_encoder();
  if (!enc || atoms == 0) return false;
  cuuint64_t dims[2] = {256, 2 * atoms};
  cuuint64_t strides[1] = {256};
  cuuint32_t box[2] = {256, 2 * box_atoms};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// y [rows, cols] bf16 as the target of TMA stores: boxes of 32 rows x 16 columns (32-byte rows, 32B
// swizzle), matching the GEMM_OUT epilogue's staging buffers.
bool make_y_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols) {
  auto enc = tensor_map_encoder();
  if (!enc || rows == 0 || cols == 0) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {16, 32};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The backward's transposed column-wise codes [rows, cols] bytes as the target of TMA stores:
// boxes of 32 rows x 32 bytes (32B swizzle), matching the dh epilogue's staging tiles.
bool make_t_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols) {
  auto enc = tensor_map_encoder();
  if (!enc || rows == 0 || cols == 0) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The fp32 weight gradient [E * wg_m, wg_n] as the target of TMA stores: boxes of 32 rows x 16
// columns (64-byte rows, 64B swizzle), matching the GEMM_WGRAD epilogue's staging buffer.
bool make_dw_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols) {
  auto enc = tensor_map_encoder();
  if (!enc || rows == 0 || cols == 0) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 4};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(P_WG_CHUNK), 32};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct DeviceInfo {
  int sms = 0;
  int pair_clusters[4] = {0, 0, 0, 0};   // co-resident CTA pairs of each pair-kernel mode (0: none)
  int nv_pair_clusters[2] = {0, 0};      // same for the NVFP4 forward GEMMs
  bool attr_set = false;
};

template <int MODE, int FMT = FMT_MX>
cudaLaunchConfig_t pair_config(int clusters, cudaLaunchAttribute* attr, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2 * clusters, 1, 1);
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = PairLayout<FMT>::SMEM_BYTES;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

template <int MODE, int FMT = FMT_MX>
int max_pair_clusters() {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pair_config<MODE, FMT>(64, attr, nullptr);
  int n = 0;
  if (cudaFuncSetAttribute(k_grouped_gemm_pair<MODE, FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           PairLayout<FMT>::SMEM_BYTES) != cudaSuccess ||
      cudaOccupancyMaxActiveClusters(&n, k_grouped_gemm_pair<MODE, FMT>, &cfg) != cudaSuccess) {
    cudaGetLastError();   // clear: the single-CTA kernels are used instead
    return 0;
  }
  return n;
}

template <int MODE, int FMT = FMT_MX>
cudaError_t launch_pair(int clusters, const CUtensorMap& a, const CUtensorMap& b, const GemmParams& p,
                        cudaStream_t stream) {
  constexpr uint32_t box_atoms = PairLayout<FMT>::SF_ATOMS;
  CUtensorMap sa, sb, d = a;   // d: the store target of GEMM_WGRAD (dW), GEMM_OUT (y), GEMM_DGRAD
                               // (transposed codes of dGU and h)
  if (!make_sf_map(&sa, p.a_sf, static_cast<uint64_t>(p.a_sf_tiles) * p.a_kt, box_atoms) ||
      !make_sf_map(&sb, p.b_sf, static_cast<uint64_t>(p.b_sf_tiles) * p.b_kt, box_atoms))
    return cudaErrorInvalidValue;
  if (MODE == GEMM_WGRAD && !make_dw_map(&d, p.dw, static_cast<uint64_t>(p.E) * p.wg_m, p.wg_n))
    return cudaErrorInvalidValue;
  if (MODE == GEMM_OUT && p.y_rows > 0 && !make_y_map(&d, p.y, static_cast<uint64_t>(p.y_rows), p.ldy))
    return cudaErrorInvalidValue;
  if (MODE == GEMM_DGRAD && !make_t_map(&d, p.dguT, static_cast<uint64_t>(3 * p.ldh), static_cast<uint64_t>(p.r_pad)))
    return cudaErrorInvalidValue;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pair_config<MODE, FMT>(clusters, attr, stream);
  return cudaLaunchKernelEx(&cfg, k_grouped_gemm_pair<MODE, FMT>, a, b, sa, sb, d, p);
}

bool device_setup(DeviceInfo** out) {
  static DeviceInfo info[64];
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  std::lock_guard<std::mutex> lock(mu);
  DeviceInfo& d = info[dev];
  if (!d.attr_set) {
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
    if (cudaFuncSetAttribute(k_grouped_gemm<GEMM_SWIGLU>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) !=
        cudaSuccess)
      return false;
    if (cudaFuncSetAttribute(k_grouped_gemm<GEMM_OUT>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) !=
        cudaSuccess)
      return false;
    // MXFP8MOE_SINGLE_CTA=1 selects the single-CTA kernels (also used where no CTA pair fits)
    const char* single = getenv("MXFP8MOE_SINGLE_CTA");
    if (single == nullptr || single[0] != '1') {
      d.pair_clusters[GEMM_SWIGLU] = max_pair_clusters<GEMM_SWIGLU>();
      d.pair_clusters[GEMM_OUT] = max_pair_clusters<GEMM_OUT>();
    }
    // the backward runs on CTA pairs only
    d.pair_clusters[GEMM_DGRAD] = max_pair_clusters<GEMM_DGRAD>();
    d.pair_clusters[GEMM_WGRAD] = max_pair_clusters<GEMM_WGRAD>();
    // the NVFP4 forward runs on CTA pairs only
    d.nv_pair_clusters[GEMM_SWIGLU] = max_pair_clusters<GEMM_SWIGLU, FMT_NV>();
    d.nv_pair_clusters[GEMM_OUT] = max_pair_clusters<GEMM_OUT, FMT_NV>();
    d.attr_set = true;
  }
  *out = &d;
  return true;
}

}  // namespace

cudaError_t launch_schedule(const int32_t* split, int E, int64_t R, SchedHeader* meta, cudaStream_t stream) {
  k_schedule<<<1, 1024, 0, stream>>>(split, E, R, meta);
  return cudaGetLastError();
}

int launch_grouped_mlp(const void* x_sorted, int64_t R, int64_t H, int64_t F, int E, const int32_t* split,
                       const float* gates, const uint8_t* w1_q, const uint8_t* w1_sf, const uint8_t* w2_q,
                       const uint8_t* w2_sf, void* y, void* workspace, const WsLayout& L, cudaStream_t stream,
                       void* const* events, const int32_t* token_of_row, int64_t x_rows, uint16_t* gu_out) {
  DeviceInfo* dev = nullptr;
  if (!device_setup(&dev)) return MXFP8_ERR_CUDA;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  SchedHeader* meta = reinterpret_cast<SchedHeader*>(ws + L.meta);
  uint8_t* xq = ws + L.xq;
  uint8_t* xsf = ws + L.xsf;
  uint8_t* hq = ws + L.hq;
  uint8_t* hsf = ws + L.hsf;

  CUtensorMap mA1, mB1, mA2, mB2;
  if (!make_map(&mA1, xq, L.r_pad, H) || !make_map(&mB1, w1_q, static_cast<uint64_t>(E) * 2 * F, H) ||
      !make_map(&mA2, hq, L.r_pad, F) || !make_map(&mB2, w2_q, static_cast<uint64_t>(E) * H, F))
    return MXFP8_ERR_CUDA;

  auto mark = [&](int i) {
    return events == nullptr || events[i] == nullptr ||
           cudaEventRecord(static_cast<cudaEvent_t>(events[i]), stream) == cudaSuccess;
  };
  if (!mark(0)) return MXFP8_ERR_CUDA;
  if (launch_schedule(split, E, R, meta, stream) != cudaSuccess) return MXFP8_ERR_CUDA;
  if (!mark(1)) return MXFP8_ERR_CUDA;
  if (launch_quantize_gather(x_sorted, R, H, meta, E, L.r_pad, token_of_row, x_rows, xq, xsf, stream) !=
      cudaSuccess)
    return MXFP8_ERR_CUDA;
  if (!mark(2)) return MXFP8_ERR_CUDA;

  const int max_mtiles = static_cast<int>(L.r_pad / BM);
  GemmParams p1{};
  p1.meta = meta;
  p1.a_sf = xsf;
  p1.b_sf = w1_sf;
  p1.E = E;
  p1.KT = static_cast<int>(H / BK);
  p1.NT = static_cast<int>(F / 128);
  p1.BN = 256;
  p1.b_rows_per_expert = static_cast<int>(2 * F);
  p1.F = static_cast<int>(F);
  p1.n_fastest = 0;
  p1.gates = gates;
  p1.hq = hq;
  p1.hsf = hsf;
  p1.ldh = F;
  p1.err = &meta->error;
  p1.timeout_ns = pipeline_wait_ns();
  p1.drain_ns = kWaitTimeoutNs;
  p1.a_kt = p1.KT;
  p1.b_kt = p1.KT;
  p1.a_sf_tiles = static_cast<int>(L.r_pad / BM);
  p1.b_sf_tiles = static_cast<int>(static_cast<int64_t>(E) * 2 * F / BM);
  p1.gu_out = gu_out;
  // persistent: one CTA per SM (shared memory, registers and TMEM each allow only one)
  if (dev->pair_clusters[0] > 0) {
    const int c1 = static_cast<int>(
        std::min<int64_t>(dev->pair_clusters[0], std::max<int64_t>(1, static_cast<int64_t>(max_mtiles / 2) * p1.NT)));
    if (launch_pair<GEMM_SWIGLU>(c1, mA1, mB1, p1, stream) != cudaSuccess) return MXFP8_ERR_CUDA;
  } else {
    const int grid1 = static_cast<int>(std::min<int64_t>(dev->sms, static_cast<int64_t>(max_mtiles) * p1.NT));
    k_grouped_gemm<GEMM_SWIGLU><<<grid1, NUM_THREADS, SMEM_BYTES, stream>>>(mA1, mB1, p1);
    if (cudaGetLastError() != cudaSuccess) return MXFP8_ERR_CUDA;
  }
  if (!mark(3)) return MXFP8_ERR_CUDA;

  GemmParams p2{};
  p2.meta = meta;
  p2.a_sf = hsf;
  p2.b_sf = w2_sf;
  p2.E = E;
  p2.KT = static_cast<int>(F / BK);
  p2.BN = (H % 256 == 0) ? 256 : 128;
  p2.NT = static_cast<int>(H / p2.BN);
  p2.b_rows_per_expert = static_cast<int>(H);
  p2.F = static_cast<int>(F);
  p2.n_fastest = 1;
  p2.group_m = 8;
  p2.y_rows = R;
  p2.y = static_cast<uint16_t*>(y);
  p2.ldy = H;
  p2.err = &meta->error;
  p2.timeout_ns = p1.timeout_ns;
  p2.drain_ns = kWaitTimeoutNs;
  p2.a_kt = p2.KT;
  p2.b_kt = p2.KT;
  p2.a_sf_tiles = static_cast<int>(L.r_pad / BM);
  p2.b_sf_tiles = static_cast<int>(static_cast<int64_t>(E) * H / BM);
  if (p2.BN == 256 && dev->pair_clusters[1] > 0) {
    const int c2 = static_cast<int>(
        std::min<int64_t>(dev->pair_clusters[1], std::max<int64_t>(1, static_cast<int64_t>(max_mtiles / 2) * p2.NT)));
    if (launch_pair<GEMM_OUT>(c2, mA2, mB2, p2, stream) != cudaSuccess) return MXFP8_ERR_CUDA;
  } else {   // 128-column output tiles (H % 256 != 0), or no CTA pair fits: single-CTA kernel
    const int grid2 = static_cast<int>(std::min<int64_t>(dev->sms, static_cast<int64_t>(max_mtiles) * p2.NT));
    k_grouped_gemm<GEMM_OUT><<<grid2, NUM_THREADS, SMEM_BYTES, stream>>>(mA2, mB2, p2);
    if (cudaGetLastError() != cudaSuccess) return MXFP8_ERR_CUDA;
  }
  if (!mark(4)) return MXFP8_ERR_CUDA;
  return MXFP8_OK;
}

int launch_nvfp4_grouped_mlp(const void* x_sorted, int64_t R, int64_t H, int64_t F, int E, const int32_t* split,
                             const float* gates, const uint8_t* w1_q, const uint8_t* w1_sf, const float* w1_amax,
                             const uint8_t* w2_q, const uint8_t* w2_sf, const float* w2_amax, float h_amax, void* y,
                             void* workspace, const NvWsLayout& L, cudaStream_t stream, void* const* events) {
  DeviceInfo* dev = nullptr;
  if (!device_setup(&dev)) return MXFP8_ERR_CUDA;
  if (dev->nv_pair_clusters[GEMM_SWIGLU] <= 0 || dev->nv_pair_clusters[GEMM_OUT] <= 0) return MXFP8_ERR_UNSUPPORTED;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  SchedHeader* meta = reinterpret_cast<SchedHeader*>(ws + L.meta);
  uint32_t* amax = reinterpret_cast<uint32_t*>(ws + L.amax);   // [0] max|x|, [1] max|h| seen
  uint8_t* xq = ws + L.xq;
  uint8_t* xsf = ws + L.xsf;
  uint8_t* hq = ws + L.hq;
  uint8_t* hsf = ws + L.hsf;
  // packed E2M1: a row of K values is K / 2 bytes; the GEMMs' K step is 128 bytes = 256 values
  CUtensorMap mA1, mB1, mA2, mB2;
  if (!make_map(&mA1, xq, L.r_pad, H / 2) || !make_map(&mB1, w1_q, static_cast<uint64_t>(E) * 2 * F, H / 2) ||
      !make_map(&mA2, hq, L.r_pad, F / 2) || !make_map(&mB2, w2_q, static_cast<uint64_t>(E) * H, F / 2))
    return MXFP8_ERR_CUDA;
  auto mark = [&](int i) {
    return events == nullptr || events[i] == nullptr ||
           cudaEventRecord(static_cast<cudaEvent_t>(events[i]), stream) == cudaSuccess;
  };
  if (!mark(0)) return MXFP8_ERR_CUDA;
  if (launch_schedule(split, E, R, meta, stream) != cudaSuccess) return MXFP8_ERR_CUDA;
  if (cudaMemsetAsync(amax + 1, 0, sizeof(uint32_t), stream) != cudaSuccess) return MXFP8_ERR_CUDA;
  if (!mark(1)) return MXFP8_ERR_CUDA;
  if (launch_nv_amax_quantize_gather(x_sorted, R, H, meta, E, L.r_pad, amax, xq, xsf, stream) != cudaSuccess)
    return MXFP8_ERR_CUDA;
  if (!mark(2)) return MXFP8_ERR_CUDA;

  const int max_mtiles = static_cast<int>(L.r_pad / BM);
  GemmParams p1{};
  p1.meta = meta;
  p1.a_sf = xsf;
  p1.b_sf = w1_sf;
  p1.E = E;
  p1.KT = static_cast<int>((H + 255) / 256);
  p1.NT = static_cast<int>(F / 128);
  p1.BN = 256;
  p1.b_rows_per_expert = static_cast<int>(2 * F);
  p1.F = static_cast<int>(F);
  p1.n_fastest = 0;
  p1.gates = gates;
  p1.hq = hq;
  p1.hsf = hsf;
  p1.ldh = F;
  p1.err = &meta->error;
  p1.timeout_ns = pipeline_wait_ns();
  p1.drain_ns = kWaitTimeoutNs;
  p1.a_kt = static_cast<int>(L.x_kt);
  p1.b_kt = static_cast<int>(L.x_kt);
  p1.a_sf_tiles = max_mtiles;
  p1.b_sf_tiles = static_cast<int>(static_cast<int64_t>(E) * 2 * F / BM);
  p1.nv_amax_a = reinterpret_cast<const float*>(amax);
  p1.nv_amax_b = w1_amax;
  p1.nv_out_amax = h_amax;
  p1.nv_out_seen = amax + 1;
  p1.h_kt = L.h_kt;
  const int c1 = static_cast<int>(std::min<int64_t>(dev->nv_pair_clusters[GEMM_SWIGLU],
                                                    std::max<int64_t>(1, static_cast<int64_t>(max_mtiles / 2) * p1.NT)));
  if (launch_pair<GEMM_SWIGLU, FMT_NV>(c1, mA1, mB1, p1, stream) != cudaSuccess) return MXFP8_ERR_CUDA;
  if (!mark(3)) return MXFP8_ERR_CUDA;

  GemmParams p2{};
  p2.meta = meta;
  p2.a_sf = hsf;
  p2.b_sf = w2_sf;
  p2.E = E;
  p2.KT = static_cast<int>((F + 255) / 256);
  p2.BN = 256;
  p2.NT = static_cast<int>(H / 256);
  p2.b_rows_per_expert = static_cast<int>(H);
  p2.F = static_cast<int>(F);
  p2.n_fastest = 1;
  p2.group_m = 8;
  p2.y_rows = R;
  p2.y = static_cast<uint16_t*>(y);
  p2.ldy = H;
  p2.err = &meta->error;
  p2.timeout_ns = p1.timeout_ns;
  p2.drain_ns = kWaitTimeoutNs;
  p2.a_kt = static_cast<int>(L.h_kt);
  p2.b_kt = static_cast<int>(L.h_kt);
  p2.a_sf_tiles = max_mtiles;
  p2.b_sf_tiles = static_cast<int>(static_cast<int64_t>(E) * H / BM);
  p2.nv_amax_a = nullptr;
  p2.nv_amax_a_val = h_amax;
  p2.nv_amax_b = w2_amax;
  const int c2 = static_cast<int>(std::min<int64_t>(dev->nv_pair_clusters[GEMM_OUT],
                                                    std::max<int64_t>(1, static_cast<int64_t>(max_mtiles / 2) * p2.NT)));
  if (launch_pair<GEMM_OUT, FMT_NV>(c2, mA2, mB2, p2, stream) != cudaSuccess) return MXFP8_ERR_CUDA;
  if (!mark(4)) return MXFP8_ERR_CUDA;
  return MXFP8_OK;
}

namespace {

// dgates[r] = sum of the partial sums of sorted row r (over the 128-column slices of F), read
// from the row's place in the expert-padded row space.
__global__ void __launch_bounds__(256) k_dgate_reduce(const SchedHeader* meta, int E, int64_t R, int nparts,
                                                     const float* part, float* dgates) {
  const int64_t r = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (r >= R || meta->num_mtiles == 0) return;
  const int32_t* row_off = reinterpret_cast<const int32_t*>(meta + 1);
  const int32_t* pad_off = row_off + (E + 1);
  int lo = 0, hi = E;   // largest e with row_off[e] <= r, skipping empty experts
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (row_off[mid] <= r) lo = mid; else hi = mid;
  }
  const int64_t prow = pad_off[lo] + (r - row_off[lo]);
  float acc = 0.0f;
  for (int i = 0; i < nparts; ++i) acc += part[prow * nparts + i];
  dgates[r] = acc;
}

template <int MODE>
int run_pair(const DeviceInfo* dev, int units, const CUtensorMap& a, const CUtensorMap& b, const GemmParams& p,
             cudaStream_t stream) {
  if (dev->pair_clusters[MODE] <= 0) return MXFP8_ERR_UNSUPPORTED;
  const int c = std::min(dev->pair_clusters[MODE], std::max(1, units));
  return launch_pair<MODE>(c, a, b, p, stream) == cudaSuccess ? MXFP8_OK : MXFP8_ERR_CUDA;
}

}  // namespace

bool bwd_ws_layout(int64_t R, int64_t H, int64_t F, int E, BwdWsLayout* out) {
  WsLayout f;
  if (!ws_layout(R, H, F, E, &f)) return false;
  const size_t rp = static_cast<size_t>(f.r_pad);
  auto al = [](size_t v) { return (v + 255) & ~static_cast<size_t>(255); };
  BwdWsLayout L{};
  L.r_pad = f.r_pad;
  L.meta = 0;
  L.dyq = f.xq;                                   // after the schedule, as in the forward workspace
  L.dysf = al(L.dyq + rp * H);
  L.dyT = al(L.dysf + rp * H / 32);
  L.dyTsf = al(L.dyT + rp * H);
  L.xT = al(L.dyTsf + rp * H / 32);
  L.xTsf = al(L.xT + rp * H);
  L.dguq = al(L.xTsf + rp * H / 32);
  L.dgusf = al(L.dguq + rp * 2 * F);
  L.dguT = al(L.dgusf + rp * 2 * F / 32);
  L.hT = L.dguT + rp * 2 * F;                     // right after dGU's codes: one [3F, r_pad] matrix
  L.dguTsf = al(L.hT + rp * F);
  L.hTsf = al(L.dguTsf + rp * 2 * F / 32);
  L.part = al(L.hTsf + rp * F / 32);
  L.total = al(L.part + rp * (F / 128) * sizeof(float));
  *out = L;
  return true;
}

int launch_grouped_mlp_bwd(const void* x_sorted, int64_t R, int64_t H, int64_t F, int E, const int32_t* split,
                           const float* gates, const uint16_t* saved_gu, const uint8_t* w1t_q, const uint8_t* w1t_sf,
                           const uint8_t* w2t_q, const uint8_t* w2t_sf, const void* dy, void* dx, float* dgates,
                           float* dw1, float* dw2, void* workspace, const BwdWsLayout& L, cudaStream_t stream,
                           void* const* events, const int32_t* token_of_row, int64_t x_rows) {
  DeviceInfo* dev = nullptr;
  if (!device_setup(&dev)) return MXFP8_ERR_CUDA;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  SchedHeader* meta = reinterpret_cast<SchedHeader*>(ws + L.meta);
  const int64_t rp = L.r_pad;
  auto mark = [&](int i) {
    return events == nullptr || events[i] == nullptr ||
           cudaEventRecord(static_cast<cudaEvent_t>(events[i]), stream) == cudaSuccess;
  };
  CUtensorMap mDy, mW2t, mDgu, mW1t, mDyT, mHT, mDguT, mXT;
  if (!make_map(&mDy, ws + L.dyq, rp, H) || !make_map(&mW2t, w2t_q, F, static_cast<uint64_t>(E) * H) ||
      !make_map(&mDgu, ws + L.dguq, rp, 2 * F) || !make_map(&mW1t, w1t_q, H, static_cast<uint64_t>(E) * 2 * F) ||
      !make_map(&mDyT, ws + L.dyT, H, rp) || !make_map(&mHT, ws + L.hT, F, rp) ||
      !make_map(&mDguT, ws + L.dguT, 2 * F, rp) || !make_map(&mXT, ws + L.xT, H, rp))
    return MXFP8_ERR_CUDA;

  // 0: schedule and the quantizations of dy (row-wise and column-wise in one pass) and x
  if (!mark(0)) return MXFP8_ERR_CUDA;
  if (launch_schedule(split, E, R, meta, stream) != cudaSuccess) return MXFP8_ERR_CUDA;
  // with token_of_row, x and dy are token rows ([x_rows, H]): sorted row r reads token
  // token_of_row[r] (the gradient of the combine is this same gather of the output gradient)
  if (launch_quantize_t(dy, R, H, rp, true, ws + L.dyT, ws + L.dyTsf, meta, E, token_of_row, x_rows, stream,
                        ws + L.dyq, ws + L.dysf) != cudaSuccess ||
      launch_quantize_t(x_sorted, R, H, rp, true, ws + L.xT, ws + L.xTsf, meta, E, token_of_row, x_rows, stream) !=
          cudaSuccess)
    return MXFP8_ERR_CUDA;
  if (!mark(1)) return MXFP8_ERR_CUDA;

  const int pairs = static_cast<int>(rp / 256);
  GemmParams base{};
  base.meta = meta;
  base.E = E;
  base.F = static_cast<int>(F);
  base.err = &meta->error;
  base.timeout_ns = pipeline_wait_ns();
  base.drain_ns = kWaitTimeoutNs;
  int st;

  // 1: dh = dy W2 (W2 quantized along H) with the ScaledSwiGLU backward -> dGU row-wise and
  //    column-wise, h column-wise (MXFP8), dgate parts
  GemmParams pd = base;
  pd.a_sf = ws + L.dysf;
  pd.b_sf = w2t_sf;
  pd.KT = static_cast<int>(H / BK);
  pd.NT = static_cast<int>((F + 255) / 256);
  pd.b_rows = static_cast<int>(F);
  pd.BN = 256;
  pd.b_rows_per_expert = 0;
  pd.b_kofs = static_cast<int>(H);
  pd.a_kt = static_cast<int>(H / BK);
  pd.b_kt = static_cast<int>(static_cast<int64_t>(E) * H / BK);
  pd.a_sf_tiles = static_cast<int>(rp / BM);
  pd.b_sf_tiles = static_cast<int>(F / BM);
  pd.n_fastest = 0;
  pd.gates = gates;
  pd.ldh = F;
  pd.gu = saved_gu;
  pd.dguq = ws + L.dguq;
  pd.dgusf = ws + L.dgusf;
  pd.dguT = ws + L.dguT;
  pd.dguTsf = ws + L.dguTsf;
  pd.hTsf = ws + L.hTsf;
  pd.r_pad = rp;
  pd.t_kt = rp / BM;
  pd.dgate_part = reinterpret_cast<float*>(ws + L.part);
  if ((st = run_pair<GEMM_DGRAD>(dev, pairs * pd.NT, mDy, mW2t, pd, stream)) != MXFP8_OK) return st;
  if (!mark(2)) return MXFP8_ERR_CUDA;

  // 2: the routing-weight gradient from the dh epilogue's partial sums (dGU and h left that epilogue
  //    already quantized, row-wise and column-wise)
  if (dgates != nullptr) {
    k_dgate_reduce<<<static_cast<unsigned>((R + 255) / 256 > 0 ? (R + 255) / 256 : 1), 256, 0, stream>>>(
        meta, E, R, static_cast<int>(F / 128), reinterpret_cast<const float*>(ws + L.part), dgates);
    if (cudaGetLastError() != cudaSuccess) return MXFP8_ERR_CUDA;
  }
  if (!mark(3)) return MXFP8_ERR_CUDA;

  // 3: dx = dGU W1 (W1 quantized along 2F)
  GemmParams px = base;
  px.a_sf = ws + L.dgusf;
  px.b_sf = w1t_sf;
  px.KT = static_cast<int>(2 * F / BK);
  px.NT = static_cast<int>(H / 256);
  px.BN = 256;
  px.b_rows_per_expert = 0;
  px.b_kofs = static_cast<int>(2 * F);
  px.a_kt = px.KT;
  px.b_kt = static_cast<int>(static_cast<int64_t>(E) * 2 * F / BK);
  px.a_sf_tiles = static_cast<int>(rp / BM);
  px.b_sf_tiles = static_cast<int>(H / BM);
  px.n_fastest = 1;
  px.y = static_cast<uint16_t*>(dx);
  px.ldy = H;
  px.y_rows = R;
  if ((st = run_pair<GEMM_OUT>(dev, pairs * px.NT, mDgu, mW1t, px, stream)) != MXFP8_OK) return st;
  if (!mark(4)) return MXFP8_ERR_CUDA;

  // 4: weight gradients over each expert's rows
  GemmParams pw = base;
  pw.a_kt = static_cast<int>(rp / BK);
  pw.b_kt = pw.a_kt;
  pw.KT = 0;
  pw.a_sf = ws + L.dyTsf;
  pw.b_sf = ws + L.hTsf;
  pw.wg_mt = static_cast<int>(H / 256);
  pw.wg_nt = static_cast<int>((F + 255) / 256);
  pw.b_rows = static_cast<int>(F);
  pw.wg_m = H;
  pw.wg_n = F;
  pw.wg_m_fastest = 1;   // dy^T (H rows) is the smaller operand: keep it in L2, stream h^T once
  pw.a_sf_tiles = static_cast<int>(H / BM);
  pw.b_sf_tiles = static_cast<int>(F / BM);
  pw.dw = dw2;
  if ((st = run_pair<GEMM_WGRAD>(dev, E * pw.wg_mt * pw.wg_nt, mDyT, mHT, pw, stream)) != MXFP8_OK) return st;
  if (!mark(5)) return MXFP8_ERR_CUDA;
  pw.a_sf = ws + L.dguTsf;
  pw.b_sf = ws + L.xTsf;
  pw.wg_mt = static_cast<int>(2 * F / 256);
  pw.wg_nt = static_cast<int>(H / 256);
  pw.b_rows = 0;
  pw.wg_m = 2 * F;
  pw.wg_n = H;
  pw.wg_m_fastest = 0;   // x^T (H rows) is the smaller operand: keep it in L2, stream dGU^T once
  pw.a_sf_tiles = static_cast<int>(2 * F / BM);
  pw.b_sf_tiles = static_cast<int>(H / BM);
  pw.dw = dw1;
  if ((st = run_pair<GEMM_WGRAD>(dev, E * pw.wg_mt * pw.wg_nt, mDguT, mXT, pw, stream)) != MXFP8_OK) return st;
  if (!mark(6)) return MXFP8_ERR_CUDA;
  return MXFP8_OK;
}

}  // namespace mx
