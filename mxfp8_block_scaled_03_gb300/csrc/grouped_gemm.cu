// grouped_gemm.cu -- the fused MXFP8 grouped expert MLP forward on sm_103a.
//
// Operation (page "Efficient MoE training for biological foundation models", Key technical
// approaches): GroupedLinear over per-expert row counts split_sizes (item 1), MXFP8 operands
// with one E8M0 scale per 32 values along K (item 2), and the fused
// GroupedLinear -> ScaledSwiGLU -> GroupedLinear forward in which the SwiGLU activation and the
// routing-weight multiply run inside the first GEMM and the intermediate is requantized to MXFP8
// there, so it never exists in 16-bit memory (item 3).
//
// Device pipeline of one call (one stream, no host synchronization):
//   1. k_schedule    split_sizes -> prefix sums, expert-padded row offsets, 128-row tile counts,
//                    sum check (error word on mismatch).
//   2. k_quantize    x_sorted -> x_q (E4M3) + scale bytes in the tensor-core layout, rows moved
//                    into an expert-padded row space so every 128-row tile belongs to one expert.
//   3. k_grouped_gemm<GEMM_SWIGLU>  per tile (expert e, 128 rows, 128 columns of F):
//                    [G | U] = x_q W1[e, {gate, up} rows]^T accumulated in TMEM, then
//                    h = gate * silu(G) * U, requantized to h_q + scale bytes.
//   4. k_grouped_gemm<GEMM_OUT>     per tile (expert e, 128 rows, BN columns of H):
//                    y = h_q W2[e]^T -> bf16, stored only for the expert's real rows.
//
// GEMM kernel structure (persistent, one 512-thread CTA per SM, 4-stage shared-memory ring):
//   TMA producer  A tile (128 rows x 128 K bytes), B tile (BN rows x 128) and the 512-byte scale
//                 atoms of both, all completing on one mbarrier per stage.
//   scale warps   four warps copy the stage's scale atoms into TMEM with tcgen05.st (one TMEM lane
//                 quarter each) and signal the MMA issuer; doing this with tcgen05.cp from the
//                 MMA thread stalled the tensor pipe (about a third of the kernel's time).
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

enum GemmMode { GEMM_SWIGLU = 0, GEMM_OUT = 1 };

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
  // GEMM_SWIGLU epilogue
  const float* gates;
  uint8_t* hq;
  uint8_t* hsf;
  int64_t ldh;             // F
  // GEMM_OUT epilogue
  uint16_t* y;
  int64_t ldy;             // H
  uint32_t* err;
  uint64_t timeout_ns;
};

struct TileInfo {
  int e, n, pad_row0, src_row0, valid;
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

__device__ __forceinline__ void tmem_st_32x32b_x4(uint32_t taddr, const uint4 v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

template <uint32_t N>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
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
        if (!warp_wait(&full[stage], phase, abort_flag, p.timeout_ns, p.err, ERR_TIMEOUT_SF, lane)) {
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
            if (!mbar_wait_bounded(&full[s], (issued_parity >> s) & 1u, nullptr, p.timeout_ns))
              atomicOr(p.err, ERR_TIMEOUT_DRAIN);
      __syncwarp();
    } else if (warp == WARP_MMA) {
      // ---------------- MMA issuer (lane 0 issues) ----------------
      const uint32_t idesc = idesc_mxf8_e4m3(BM, BN);
      int stage = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool issued = false, ok = true;
      for (int u = blockIdx.x; ok && u < total_units; u += gridDim.x) {
        if (!warp_wait(acc_empty, acc_phase ^ 1u, abort_flag, p.timeout_ns, p.err, ERR_TIMEOUT_MMA, lane)) break;
        tc_fence_after();
        for (int kb = 0; kb < p.KT; ++kb) {
          // sf_full implies full: the scale warps waited for the stage's data before signalling
          if (!warp_wait(&sf_full[stage], phase, abort_flag, p.timeout_ns, p.err, ERR_TIMEOUT_MMA, lane)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (lane == 0) {
            const uint8_t* sA = smem + stage * STAGE_BYTES;
            const uint8_t* sB = sA + A_BYTES;
            const uint32_t t_sfa = tmem + SFA_COL + 4 * stage;
            const uint32_t t_sfb = tmem + SFB_COL + 8 * stage;
            const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
#pragma unroll
            for (int k = 0; k < BK / 32; ++k) {
              tc_mma_mxf8(tmem + ACC_COL, sdesc_kmajor_sw128(a0 + 32 * k), sdesc_kmajor_sw128(b0 + 32 * k),
                          idesc_with_sf_id(idesc, k), t_sfa, t_sfb, (kb | k) != 0 ? 1u : 0u);
            }
            tc_commit(&empty[stage]);
          }
          __syncwarp();
          issued = true;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if (lane == 0) tc_commit(acc_full);
        __syncwarp();
        acc_phase ^= 1u;
      }
      if (issued && lane == 0) {
        tc_commit(drained);
        if (!mbar_wait_bounded(drained, 0, nullptr, p.timeout_ns)) atomicOr(p.err, ERR_TIMEOUT_DRAIN);
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
      if (!warp_wait(acc_full, acc_phase, abort_flag, p.timeout_ns, p.err, ERR_TIMEOUT_EPILOGUE, lane)) break;
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

      if (MODE == GEMM_SWIGLU) {
        const bool real = r < t.valid;
        const float gate = real ? (p.gates ? __ldg(p.gates + t.src_row0 + r) : 1.0f) : 0.0f;
        uint8_t* hrow = p.hq + static_cast<int64_t>(t.pad_row0 + r) * p.ldh + t.n * 128 + 64 * half;
        uint32_t sf_pair = 0;
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          float h[32];
          float amax = 0.0f;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float g = __uint_as_float(v[32 * b + i]);
            const float up = __uint_as_float(v[64 + 32 * b + i]);
            const float s = __fdividef(g, 1.0f + __expf(-g));
            h[i] = gate * s * up;
            amax = fmaxf(amax, fabsf(h[i]));
          }
          const uint32_t sfb = e8m0_from_amax(amax);
          const float inv = e8m0_inverse_scale(sfb);
          const uint2 t0 = quant8(h + 0, inv), t1 = quant8(h + 8, inv), t2 = quant8(h + 16, inv),
                      t3 = quant8(h + 24, inv);
          reinterpret_cast<uint4*>(hrow + 32 * b)[0] = make_uint4(t0.x, t0.y, t1.x, t1.y);
          reinterpret_cast<uint4*>(hrow + 32 * b)[1] = make_uint4(t2.x, t2.y, t3.x, t3.y);
          sf_pair |= sfb << (8 * b);
        }
        // scale bytes of blocks (2*half, 2*half+1) of column tile n for padded row pad_row0 + r
        const int64_t atom = static_cast<int64_t>(t.pad_row0 / BM) * (p.ldh / 128) + t.n;
        *reinterpret_cast<uint16_t*>(p.hsf + atom * SF_ATOM + (r & 31) * 16 + (r >> 5) * 4 + 2 * half) =
            static_cast<uint16_t>(sf_pair);
      } else {
        if (r < t.valid) {
          const int ncols = BN / 2;
          uint16_t* yrow = p.y + static_cast<int64_t>(t.src_row0 + r) * p.ldy + t.n * BN + ncols * half;
#pragma unroll
          for (int c = 0; c < 128; c += 8) {
            if (c < ncols) {
              uint4 o;
              o.x = pack_bf16x2(__uint_as_float(v[c + 0]), __uint_as_float(v[c + 1]));
              o.y = pack_bf16x2(__uint_as_float(v[c + 2]), __uint_as_float(v[c + 3]));
              o.z = pack_bf16x2(__uint_as_float(v[c + 4]), __uint_as_float(v[c + 5]));
              o.w = pack_bf16x2(__uint_as_float(v[c + 6]), __uint_as_float(v[c + 7]));
              *reinterpret_cast<uint4*>(yrow + c) = o;
            }
          }
        }
      }
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

// One block of 1024 threads: inclusive scans of split sizes and of 128-row tile counts.
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
  s_tiles[t] = (v + BM - 1) / BM;
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

struct DeviceInfo {
  int sms = 0;
  bool attr_set = false;
};

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
                       void* const* events, const int32_t* token_of_row, int64_t x_rows) {
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
  p1.timeout_ns = kWaitTimeoutNs;
  // persistent: one CTA per SM (shared memory, registers and TMEM each allow only one)
  const int grid1 = static_cast<int>(std::min<int64_t>(dev->sms, static_cast<int64_t>(max_mtiles) * p1.NT));
  k_grouped_gemm<GEMM_SWIGLU><<<grid1, NUM_THREADS, SMEM_BYTES, stream>>>(mA1, mB1, p1);
  if (cudaGetLastError() != cudaSuccess) return MXFP8_ERR_CUDA;
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
  p2.y = static_cast<uint16_t*>(y);
  p2.ldy = H;
  p2.err = &meta->error;
  p2.timeout_ns = kWaitTimeoutNs;
  const int grid2 = static_cast<int>(std::min<int64_t>(dev->sms, static_cast<int64_t>(max_mtiles) * p2.NT));
  k_grouped_gemm<GEMM_OUT><<<grid2, NUM_THREADS, SMEM_BYTES, stream>>>(mA2, mB2, p2);
  if (cudaGetLastError() != cudaSuccess) return MXFP8_ERR_CUDA;
  if (!mark(4)) return MXFP8_ERR_CUDA;
  return MXFP8_OK;
}

}  // namespace mx
