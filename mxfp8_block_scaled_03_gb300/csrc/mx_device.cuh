// mx_device.cuh -- device-side building blocks for sm_103a: MXFP8 element/scale arithmetic and
// thin inline-PTX wrappers for mbarrier, TMA (cp.async.bulk*) and the 5th-generation tensor core
// (tcgen05: TMEM allocation, block-scaled MMA, shared->TMEM copies, TMEM loads).
//
// The MXFP8 rule implemented here (blocks of 32 consecutive values sharing one scale: page
// "Efficient MoE training for biological foundation models", Key technical approaches, item 2;
// scale rule read as OCP MX v1.0): E8M0 byte = clamp(floor(log2 amax) - 8 + 127, 0, 254),
// element = RNE_E4M3(v * 2^-(byte-127)) saturated to +-448.
#pragma once
#include <cstdint>
#include <cuda.h>   // CUtensorMap (type only; the driver entry point is fetched at run time)
#include <cuda_bf16.h>

namespace mx {

// ------------------------------------------------------------------------------------------
// MXFP8 arithmetic
// ------------------------------------------------------------------------------------------

// E8M0 byte of a block from its largest magnitude (amax >= 0, finite).  For a normal float the
// biased exponent field is floor(log2 amax) + 127, so the byte is field - 8; subnormal or zero
// amax (field 0) and anything below 2^-119 clamp to byte 0 (s = -127).  The top clamp (254) is
// never reached from finite floats (field <= 254 gives byte <= 246).
__device__ __forceinline__ uint32_t e8m0_from_amax(float amax) {
  const int field = static_cast<int>(__float_as_uint(amax) >> 23);
  return static_cast<uint32_t>(field > 8 ? field - 8 : 0);
}

// 2^-(byte-127) as a float: exponent field 127 - (byte - 127) = 254 - byte, always normal for
// bytes in [0, 246].
__device__ __forceinline__ float e8m0_inverse_scale(uint32_t byte) {
  return __uint_as_float((254u - byte) << 23);
}

// Two floats -> two E4M3 codes, round to nearest even, saturating to +-448 (lo -> low byte).
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Eight values times a common inverse scale -> eight codes (element 0 in the lowest byte).
__device__ __forceinline__ uint2 quant8(const float* v, float inv) {
  uint2 o;
  o.x = e4m3x2(v[0] * inv, v[1] * inv) | (e4m3x2(v[2] * inv, v[3] * inv) << 16);
  o.y = e4m3x2(v[4] * inv, v[5] * inv) | (e4m3x2(v[6] * inv, v[7] * inv) << 16);
  return o;
}

// Packed pairs of floats for the f32x2 arithmetic of sm_100-family SMs (one instruction per pair,
// each lane rounded to nearest like its scalar counterpart; lo in the low 32 bits).
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float f2_lo(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v)); }
__device__ __forceinline__ float f2_hi(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v >> 32)); }
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
// A packed pair -> two E4M3 codes (see e4m3x2).
__device__ __forceinline__ uint32_t e4m3x2_f2(uint64_t v) { return e4m3x2(f2_lo(v), f2_hi(v)); }

// bf16 halves of a 32-bit word -> floats (exact).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two floats -> packed bf16x2, round to nearest even (lo -> low half).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&p);
}

// max of |a| and |b| per bf16 half (sign bits cleared, so the maximum is exact).
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a & 0x7FFF7FFFu), "r"(b & 0x7FFF7FFFu));
  return r;
}

__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t a) { return a & 0x7FFF7FFFu; }

// Byte offset of (row, block) in the tensor-core scale-factor layout: 512-byte atoms of
// 128 rows x 4 blocks, atoms ordered row-tile-major with `kt` atoms per row tile; inside an atom
// row 32*j + i, block b sits at 16*i + 4*j + b.
__device__ __forceinline__ int64_t sf_mma_offset(int64_t row, int64_t blk, int64_t kt) {
  return ((row >> 7) * kt + (blk >> 2)) * 512 + (row & 31) * 16 + ((row >> 5) & 3) * 4 + (blk & 3);
}

// ------------------------------------------------------------------------------------------
// NVFP4 arithmetic (E2M1 elements, one E4M3 scale per 16 values, a per-tensor binary32 encode
// scale 448 * 6 / amax): NVIDIA's published format, named as a recipe on the Llama 3 recipe page.
// Every decision is taken in binary32 with explicitly rounded operations.
// ------------------------------------------------------------------------------------------

// Per-tensor encode scale from the tensor's largest magnitude: 2688 / amax (1 for an all-zero
// tensor, at most FLT_MAX).
__device__ __forceinline__ float nv_encode_scale(float amax) {
  return amax == 0.0f ? 1.0f : fminf(__fdiv_rn(2688.0f, amax), 3.402823466e38f);
}

// E4M3 code of a non-negative binary32 value, round to nearest even, saturating at 448.
__device__ __forceinline__ uint32_t e4m3_code(float t) { return e4m3x2(t, 0.0f) & 0xFFu; }

// Value of an E4M3 code (non-negative codes 0x00..0x7E), exact: 2^(E-7) (1 + M/8), or M 2^-9.
__device__ __forceinline__ float e4m3_value(uint32_t c) {
  const uint32_t e = (c >> 3) & 15u, m = c & 7u;
  return e == 0 ? __uint_as_float(0x3B000000u) * static_cast<float>(m)        // 2^-9 * M
                : __uint_as_float(((e + 120u) << 23) | (m << 20));
}

// Block scale and element multiplier of one 16-value block of NVFP4 from its largest magnitude:
// S = E4M3(fl32(fl32(amax / 6) * s_enc)); r = fl32(s_enc / S) (0 when S = 0, at most FLT_MAX).
__device__ __forceinline__ uint32_t nv_block_scale(float amax, float s_enc, float* r) {
  const uint32_t code = e4m3_code(__fmul_rn(__fdiv_rn(amax, 6.0f), s_enc));
  const float S = e4m3_value(code);
  *r = S == 0.0f ? 0.0f : fminf(__fdiv_rn(s_enc, S), 3.402823466e38f);
  return code;
}

// Eight binary32 values -> eight E2M1 codes in one word (value 2i in the low nibble of byte i,
// value 2i+1 in its high nibble), round to nearest even, saturating at 6.
__device__ __forceinline__ uint32_t e2m1x8(float v0, float v1, float v2, float v3, float v4, float v5, float v6,
                                           float v7) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(r)
      : "f"(v0), "f"(v1), "f"(v2), "f"(v3), "f"(v4), "f"(v5), "f"(v6), "f"(v7));
  return r;
}

// ------------------------------------------------------------------------------------------
// Generic helpers
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------------------------------------
// mbarrier
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// try_wait with a suspend-time hint: a thread whose phase is not complete yet is suspended until
// the phase completes or about kSuspendNs pass.  Suspended waiters cost the tensor pipe far less
// than waiters that return at once and poll again (measured: 12 polling warps slowed a CTA-pair
// MMA stream by 15%, suspended ones by 7%).
constexpr uint32_t kSuspendNs = 8192;
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendNs)
      : "memory");
  return ok != 0;
}

// Wait for the phase of `bar` with the given parity to complete.  Gives up (returns false) after
// `timeout_ns` of wall time, or early when *abort becomes non-zero (abort may be null).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, const volatile int* abort,
                                                  uint64_t timeout_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (abort != nullptr && *abort) return false;
    if (globaltimer_ns() - t0 > timeout_ns) return false;
  }
}

// Barrier over `nthreads` threads (whole warps) on hardware barrier `id` that also returns the AND
// of every thread's `v`: one thread of a group waits on an mbarrier, the others learn the outcome
// here without polling.
__device__ __forceinline__ bool group_and(uint32_t id, uint32_t nthreads, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

// ------------------------------------------------------------------------------------------
// TMA / bulk copies (global -> shared, completion counted on an mbarrier)
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// ------------------------------------------------------------------------------------------
// tcgen05 (tensor memory + MMA)
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* holder, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(holder)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Arrive on `bar` once every tcgen05 operation this thread issued so far has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// Shared memory matrix descriptor, K-major operand staged by TMA with 128-byte swizzle: rows of
// 128 bytes, 8-row groups 1024 bytes apart (stride byte offset), leading byte offset unused,
// descriptor version 1 (bits 46-47), swizzle mode 2 = 128B (bits 61-63).
__device__ __forceinline__ uint64_t sdesc_kmajor_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1) << 16;
  d |= static_cast<uint64_t>(1024 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Shared memory descriptor of one 512-byte scale-factor atom (32 rows x 16 bytes, no swizzle,
// 8-row groups 128 bytes apart) as the source of tcgen05.cp.
__device__ __forceinline__ uint64_t sdesc_sf_atom(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(128 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  return d;
}

// Instruction descriptor of kind::mxf8f6f4 with block scaling: A and B E4M3 (format 0),
// both K-major, UE8M0 scales (bit 23), N >> 3 in bits 17-22, M >> 4 in bits 24-28, and the byte
// of each 32-bit TMEM scale word to use (A: bits 29-30, B: bits 4-5).
__host__ __device__ constexpr uint32_t idesc_mxf8_e4m3(uint32_t M, uint32_t N) {
  return ((N >> 3) << 17) | (1u << 23) | ((M >> 4) << 24);
}
__device__ __forceinline__ uint32_t idesc_with_sf_id(uint32_t idesc, uint32_t id) {
  return idesc | (id << 4) | (id << 29);
}

// tcgen05.cp of one 512-byte scale-factor atom from shared memory to TMEM columns [taddr, taddr+4),
// replicated into all four 32-lane quarters (lane i, column j holds the 4 bytes of atom row i,
// word j).
// Pair form: issued by the leader CTA, each CTA of the pair copies the atom at this shared-memory
// address of its own into the same TMEM columns of its own.
__device__ __forceinline__ void tc_copy_sf_pair(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T with per-32-K block scales taken from TMEM.
__device__ __forceinline__ void tc_mma_mxf8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// 32-byte global stores (one full sector per lane); the address must be 32-byte aligned.
__device__ __forceinline__ void st_global_32B(void* p, uint4 a, uint4 b) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(a.x), "r"(a.y), "r"(a.z),
               "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w)
               : "memory");
}
// Same, marked streaming (evict first): for outputs no later kernel of the call reads soon.
__device__ __forceinline__ void st_global_32B_cs(void* p, uint4 a, uint4 b) {
  asm volatile("st.global.cs.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(a.x), "r"(a.y), "r"(a.z),
               "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w)
               : "memory");
}

// ------------------------------------------------------------------------------------------
// Thread-block clusters and the CTA pair (cta_group::2)
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_cta_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_index() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_count() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Shared::cluster address of the same shared-memory object in CTA `cta` of the cluster.
__device__ __forceinline__ uint32_t map_to_cta(const void* p, uint32_t cta) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(cta));
  return r;
}
// Arrive on a barrier of another CTA of the cluster (default .release.cta semantics).  Every use
// follows tcgen05.wait::st or tcgen05.wait::ld, which block until this thread's TMEM accesses have
// completed, so the arrive has no pending writes to publish; a .release.cluster arrive here cost
// about a third of the pair kernel's time.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ void st_remote_u32(uint32_t cluster_addr, uint32_t v) {
  asm volatile("st.relaxed.cluster.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}
// try_wait with cluster-scope acquire, for barriers that threads of the other CTA of the pair
// arrive on, so that what they wrote before arriving is visible after the wait.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendNs)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_cluster_bounded(uint64_t* bar, uint32_t parity, const volatile int* abort,
                                                          uint64_t timeout_ns) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if (abort != nullptr && *abort) return false;
    if (globaltimer_ns() - t0 > timeout_ns) return false;
  }
}
// Ask L2 to fetch [p, p + bytes) ahead of its use (16-byte aligned, bytes % 16 == 0).
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(p)), "r"(bytes)
               : "memory");
}
// Tile copy into this CTA's shared memory whose completion is counted on an mbarrier that may sit
// in either CTA of the pair (`bar_cluster` is a shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* map, uint32_t bar_cluster, int32_t x,
                                                 int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.cta_group::2 [%0], [%1, {%3, %4}], "
      "[%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y)
      : "memory");
}
// TMA store of a 2-D box from this CTA's shared memory, tracked by the thread's bulk groups.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(src)), "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until at most one committed bulk group of this thread still reads shared memory.
__device__ __forceinline__ void bulk_wait_read_le1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
// Wait until every committed bulk group of this thread has completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// every committed bulk store has finished reading its shared-memory source
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// Same copy with an L2 cache-policy hint (from l2_policy_evict_last).
__device__ __forceinline__ void tma_load_2d_pair_hint(void* dst, const CUtensorMap* map, uint32_t bar_cluster,
                                                      int32_t x, int32_t y, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.cta_group::2.L2::cache_hint "
      "[%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y), "l"(policy)
      : "memory");
}
// L2 policy that keeps lines resident ahead of streaming traffic (operands reused by many tiles).
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* holder, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(holder)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// Arrive once on the mbarrier at this offset in both CTAs of the pair when every tcgen05 operation
// this thread issued so far has completed.
__device__ __forceinline__ void tc_commit_pair_both(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(static_cast<uint16_t>(3))
      : "memory");
}
// Same, arriving only on this CTA's barrier.
__device__ __forceinline__ void tc_commit_pair_local(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
// Pair MMA: D (128 lanes of each CTA) (+)= A (128 rows from each CTA) * B^T (N rows, half from each
// CTA's shared memory at the same offsets), block scales from TMEM of each CTA.
__device__ __forceinline__ void tc_mma_mxf8_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                 uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Instruction descriptor of kind::mxf4nvf4 with block scaling (NVFP4): A and B E2M1 (format 1 of
// this kind, bits 7-9 and 10-12), both K-major, UE4M3 scales (bit 23 clear), N >> 3 in bits
// 17-22, M >> 4 in bits 24-28, dense K = 64 (bit 31 clear); the scale-factor ids stay 0 (with
// four scales per row and MMA every byte of the 32-bit TMEM word is used).
__host__ __device__ constexpr uint32_t idesc_nvf4(uint32_t M, uint32_t N) {
  return (1u << 7) | (1u << 10) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// Pair MMA on NVFP4 operands: D (+)= A * B^T with K = 64 (32 bytes of packed E2M1 per row), a
// UE4M3 scale per 16 values of K (four per row: one 512-byte atom of A and two of B in TMEM).
__device__ __forceinline__ void tc_mma_nvf4_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                 uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// 32 consecutive TMEM columns of this warp's 32 lanes -> 32 registers per thread.
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

}  // namespace mx
