// mx_internal.h -- host-side declarations shared by the library's translation units.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace mx {

// Bits of the device error word (first 4 bytes of a grouped_mlp_fwd workspace).
enum : uint32_t {
  ERR_SPLIT_SUM = 1u << 0,        // split_sizes do not add up to R
  ERR_SPLIT_NEGATIVE = 1u << 1,   // a negative split size
  ERR_EXPERT_RANGE = 1u << 2,     // an expert id outside [0, E) given to the permute
  ERR_TOKEN_RANGE = 1u << 3,      // a token id outside [0, T) in token_of_row
  ERR_TIMEOUT_PRODUCER = 1u << 8, // TMA producer gave up waiting for a free stage
  ERR_TIMEOUT_MMA = 1u << 9,      // MMA issuer gave up waiting for data or a free accumulator
  ERR_TIMEOUT_EPILOGUE = 1u << 10,// epilogue gave up waiting for an accumulator
  ERR_TIMEOUT_DRAIN = 1u << 11,   // teardown gave up waiting for copies / MMAs in flight
  ERR_TIMEOUT_SF = 1u << 12,      // scale-staging warps gave up waiting for a free TMEM slot
};
constexpr uint32_t ERR_TIMEOUT_MASK = 0x1F00u;

// Device schedule written by the schedule kernel at the start of the workspace.  Arrays of E+1
// int32 follow the header: row_off (prefix sums of split_sizes), pad_off (prefix sums of
// 256 * ceil(split/256): each expert's first row in the padded row space), mt_off (prefix sums
// of 2 * ceil(split/256): each expert's first 128-row tile).
struct SchedHeader {
  uint32_t error;
  int32_t num_mtiles;   // total 128-row tiles over all experts (0 on a split error)
  int32_t pad_rows;     // 128 * num_mtiles
  int32_t E;
  int32_t reserved[12];
};
static_assert(sizeof(SchedHeader) == 64, "schedule header is 64 bytes");

struct WsLayout {
  size_t meta, xq, xsf, hq, hsf, total;
  int64_t r_pad;   // row capacity of the padded row space
};
bool ws_layout(int64_t R, int64_t H, int64_t F, int E, WsLayout* out);

// Backward workspace: schedule, then (all in the expert-padded row space of r_pad rows)
//   dyq/dysf    dy row-wise (blocks along H), tensor-core scale layout        [r_pad, H]
//   dyT/dyTsf   dy column-wise, codes transposed (blocks along rows)          [H, r_pad]
//   xT/xTsf     x column-wise, transposed                                    [H, r_pad]
//   dguq/dgusf  dGU row-wise                                                 [r_pad, 2F]
//   dguT/dguTsf dGU column-wise, transposed                                  [2F, r_pad]
//   hT/hTsf     h column-wise, transposed                                    [F, r_pad]
// (dGU and h are written quantized by the dh GEMM's epilogue; no bf16 copy is kept.)
//   part        partial sums of the routing-weight gradient (float)          [r_pad, F/128]
struct BwdWsLayout {
  size_t meta, dyq, dysf, dyT, dyTsf, xT, xTsf, dguq, dgusf, dguT, dguTsf, hT, hTsf, part, total;
  int64_t r_pad;
};
bool bwd_ws_layout(int64_t R, int64_t H, int64_t F, int E, BwdWsLayout* out);

// Quantize launchers (quantize.cu).  Return a cudaError_t from the launch.
cudaError_t launch_quantize(const void* x, int64_t M, int64_t K, int dirs, int sf_layout, uint8_t* q_row,
                            uint8_t* sf_row, uint8_t* q_col, uint8_t* sf_col, cudaStream_t stream);
// Row-wise MXFP8 of the sorted rows into the expert-padded row space (rows beyond an expert's
// count are written as zeros), scale bytes in the tensor-core layout.  Sorted row r is x row
// token_of_row[r], or x row r when token_of_row is NULL.
cudaError_t launch_quantize_gather(const void* x, int64_t R, int64_t H, const SchedHeader* meta, int E,
                                   int64_t r_pad, const int32_t* token_of_row, int64_t x_rows, uint8_t* xq,
                                   uint8_t* xsf, cudaStream_t stream);
// Column-wise MXFP8 with transposed codes: x [M, K] -> qT [K, m_out] (m_out % 128 == 0), scale
// bytes in the tensor-core layout of [K, m_out] (mma) or compact [K, m_out/32].  With meta, the
// m_out rows are the expert-padded row space gathered from the sorted rows of x (through
// token_of_row when given; then x has x_rows rows).
// q_row / sf_row (optional, K % 128 == 0): also the row-wise MXFP8 of the same rows, scale bytes
// in the tensor-core layout, from the same read of x.
cudaError_t launch_quantize_t(const void* x, int64_t M, int64_t K, int64_t m_out, bool mma, uint8_t* qT,
                              uint8_t* sfT, const SchedHeader* meta, int E, const int32_t* token_of_row,
                              int64_t x_rows, cudaStream_t stream, uint8_t* q_row = nullptr,
                              uint8_t* sf_row = nullptr);

// Dispatch and combine around the grouped MLP (moe_routing.cu).
size_t permute_workspace_bytes(int64_t n, int E);
cudaError_t launch_permute(const int32_t* experts, const float* gates, int64_t T, int k, int E, int32_t* split_sizes,
                           int32_t* row_of_slot, int32_t* token_of_row, float* gates_sorted, void* workspace,
                           cudaStream_t stream);
cudaError_t launch_gather_rows(const void* src, int64_t nsrc, int64_t row_bytes, const int32_t* index, int64_t n,
                               void* dst, int sms, cudaStream_t stream);
cudaError_t launch_combine(const void* y, const int32_t* row_of_slot, int64_t T, int k, int64_t H, void* out,
                           cudaStream_t stream);

// Grouped MLP launchers (grouped_gemm.cu).
cudaError_t launch_schedule(const int32_t* split, int E, int64_t R, SchedHeader* meta, cudaStream_t stream);
// Enqueues schedule, activation quantize and both grouped GEMMs; returns an mxfp8_status.
// `events` (may be null): 5 cudaEvent_t recorded on `stream` before each of the 4 kernels and
// after the last one.
// token_of_row (may be NULL): sorted row r reads x row token_of_row[r] (fused gather).
int launch_grouped_mlp(const void* x_sorted, int64_t R, int64_t H, int64_t F, int E, const int32_t* split,
                       const float* gates, const uint8_t* w1_q, const uint8_t* w1_sf, const uint8_t* w2_q,
                       const uint8_t* w2_sf, void* y, void* workspace, const WsLayout& L, cudaStream_t stream,
                       void* const* events, const int32_t* token_of_row = nullptr, int64_t x_rows = 0,
                       uint16_t* gu_out = nullptr);
// gu_out (may be NULL): training forward, [G | U] saved as bf16 [r_pad, 2F] for the backward.

// Backward of the grouped MLP (all GEMMs on CTA pairs; needs H % 256 == 0 and F % 128 == 0).
// `events` (may be null): 7 events recorded on `stream` around its stages.
int launch_grouped_mlp_bwd(const void* x_sorted, int64_t R, int64_t H, int64_t F, int E, const int32_t* split,
                           const float* gates, const uint16_t* saved_gu, const uint8_t* w1t_q, const uint8_t* w1t_sf,
                           const uint8_t* w2t_q, const uint8_t* w2t_sf, const void* dy, void* dx, float* dgates,
                           float* dw1, float* dw2, void* workspace, const BwdWsLayout& L, cudaStream_t stream,
                           void* const* events, const int32_t* token_of_row = nullptr, int64_t x_rows = 0);

// ---- NVFP4 forward (nvfp4.cu, grouped_gemm.cu) ----
// Scale atoms per 128-row tile of an NVFP4 tensor-core scale array for K values per row: K is
// padded to a multiple of 256 (one K step of the GEMMs), four 512-byte atoms per step.
int64_t nv_sf_atoms_per_tile(int64_t K);
// Workspace of nvfp4_grouped_mlp_fwd: schedule, two words (largest |x| and largest |h| of the
// call, float bits), then in the expert-padded row space x codes [r_pad, H/2] and their scale
// atoms, h codes [r_pad, F/2] and their scale atoms.
struct NvWsLayout {
  size_t meta, amax, xq, xsf, hq, hsf, total;
  int64_t r_pad, x_kt, h_kt;
};
bool nv_ws_layout(int64_t R, int64_t H, int64_t F, int E, NvWsLayout* out);
// Clears *amax_word, reduces max|x| into it, then quantizes the sorted rows into the padded row
// space (zero rows past each expert's count), scale codes in the tensor-core layout.
cudaError_t launch_nv_amax_quantize_gather(const void* x, int64_t R, int64_t H, const SchedHeader* meta, int E,
                                           int64_t r_pad, uint32_t* amax_word, uint8_t* xq, uint8_t* xsf,
                                           cudaStream_t stream);
// Schedule, activation amax + quantize, GroupedLinear 1 + ScaledSwiGLU + NVFP4 requant, GroupedLinear 2;
// returns an mxfp8_status.  events: NULL or 5 events recorded around the stages.
int launch_nvfp4_grouped_mlp(const void* x_sorted, int64_t R, int64_t H, int64_t F, int E, const int32_t* split,
                             const float* gates, const uint8_t* w1_q, const uint8_t* w1_sf, const float* w1_amax,
                             const uint8_t* w2_q, const uint8_t* w2_sf, const float* w2_amax, float h_amax, void* y,
                             void* workspace, const NvWsLayout& L, cudaStream_t stream, void* const* events);

}  // namespace mx
