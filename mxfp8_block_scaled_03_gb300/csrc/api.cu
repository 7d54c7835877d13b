// api.cu -- the extern "C" boundary declared in include/mxfp8moe.h: argument checks, workspace
// layout, and dispatch to the kernels' launchers.  No call allocates device memory or
// synchronizes the host, except mxfp8_check_device_error (which reads the error word).
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "mx_internal.h"
#include "mxfp8moe.h"

namespace mx {

namespace {
constexpr size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
// A buffer of `rows` rows: 16-byte aligned, and non-NULL unless it holds no rows.
bool rows_ok(const void* p, int64_t rows) { return p == nullptr ? rows == 0 : aligned16(p); }
}  // namespace

bool ws_layout(int64_t R, int64_t H, int64_t F, int E, WsLayout* out) {
  if (R < 0 || H <= 0 || F <= 0 || E < 1 || E > 1024) return false;
  if (R > static_cast<int64_t>(INT32_MAX) - 128 * static_cast<int64_t>(E)) return false;
  WsLayout L{};
  L.r_pad = ((R + 255 * static_cast<int64_t>(E)) + 255) / 256 * 256;   // experts padded to 256 rows
  L.meta = 0;
  L.xq = align256(sizeof(SchedHeader) + 3 * static_cast<size_t>(E + 1) * sizeof(int32_t));
  L.xsf = align256(L.xq + static_cast<size_t>(L.r_pad) * H);
  L.hq = align256(L.xsf + static_cast<size_t>(L.r_pad) * H / 32);
  L.hsf = align256(L.hq + static_cast<size_t>(L.r_pad) * F);
  L.total = align256(L.hsf + static_cast<size_t>(L.r_pad) * F / 32);
  *out = L;
  return true;
}

}  // namespace mx

using namespace mx;

extern "C" {

int mxfp8_abi_version(void) { return 1; }

const char* mxfp8_status_string(int status) {
  switch (status) {
    case MXFP8_OK: return "ok";
    case MXFP8_ERR_INVALID_ARG: return "invalid argument";
    case MXFP8_ERR_UNSUPPORTED: return "unsupported shape";
    case MXFP8_ERR_WORKSPACE: return "workspace too small or misaligned";
    case MXFP8_ERR_CUDA: return "CUDA call failed";
    case MXFP8_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    case MXFP8_ERR_SPLIT_MISMATCH: return "split_sizes do not sum to R (or are negative)";
    default: return "unknown status";
  }
}

size_t mxfp8_sf_bytes(int64_t M, int64_t K, int direction, int sf_layout) {
  if (M < 0 || K < 0 || K % 32 != 0) return 0;
  if (sf_layout == MXFP8_SF_COMPACT) {
    if (direction == MXFP8_ROWWISE) return static_cast<size_t>(M) * (K / 32);
    if (direction == MXFP8_COLWISE) return static_cast<size_t>((M + 31) / 32) * K;
    return 0;
  }
  if (sf_layout == MXFP8_SF_MMA) {
    if (direction == MXFP8_ROWWISE) return static_cast<size_t>((M + 127) / 128) * ((K / 32 + 3) / 4) * 512;
    if (direction == MXFP8_COLWISE) return static_cast<size_t>((K + 127) / 128) * (((M + 31) / 32 + 3) / 4) * 512;
  }
  return 0;
}

int mxfp8_quantize(const void* x, int64_t M, int64_t K, int dirs, int sf_layout, uint8_t* q_row, uint8_t* sf_row,
                   uint8_t* q_col, uint8_t* sf_col, void* stream) {
  if (M < 0 || K < 0 || K % 32 != 0) return MXFP8_ERR_INVALID_ARG;
  if (dirs < 1 || dirs > 3) return MXFP8_ERR_INVALID_ARG;
  if (sf_layout != MXFP8_SF_COMPACT && sf_layout != MXFP8_SF_MMA) return MXFP8_ERR_INVALID_ARG;
  const bool row = dirs & MXFP8_ROWWISE, col = dirs & MXFP8_COLWISE;
  if (sf_layout == MXFP8_SF_MMA && (M % 128 != 0 || K % 128 != 0)) return MXFP8_ERR_UNSUPPORTED;
  if (M == 0 || K == 0) return MXFP8_OK;
  if (x == nullptr || !aligned16(x)) return MXFP8_ERR_INVALID_ARG;
  if (row && (q_row == nullptr || sf_row == nullptr || !aligned16(q_row) || !aligned16(sf_row)))
    return MXFP8_ERR_INVALID_ARG;
  if (col && (q_col == nullptr || sf_col == nullptr || !aligned16(q_col) || !aligned16(sf_col)))
    return MXFP8_ERR_INVALID_ARG;
  if ((M + 31) / 32 > INT32_MAX || (K + 255) / 256 > 65535) return MXFP8_ERR_UNSUPPORTED;
  const cudaError_t e =
      launch_quantize(x, M, K, dirs, sf_layout, q_row, sf_row, q_col, sf_col, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MXFP8_OK : MXFP8_ERR_CUDA;
}

size_t grouped_mlp_workspace_size(int64_t R, int64_t H, int64_t F, int E) {
  WsLayout L;
  if (!ws_layout(R, H, F, E, &L)) return 0;
  return L.total;
}

int grouped_mlp_workspace_layout(int64_t R, int64_t H, int64_t F, int E, uint64_t* out) {
  WsLayout L;
  if (out == nullptr || !ws_layout(R, H, F, E, &L)) return MXFP8_ERR_INVALID_ARG;
  out[0] = L.meta;  // the error word is the first field of the schedule header
  out[1] = L.meta;
  out[2] = L.xq;
  out[3] = L.xsf;
  out[4] = L.hq;
  out[5] = L.hsf;
  out[6] = static_cast<uint64_t>(L.r_pad);
  return MXFP8_OK;
}

static int grouped_mlp_fwd_impl(const void* x_sorted, int64_t R, int64_t H, int64_t F, int E,
                                const int32_t* split_sizes, const float* gates, const uint8_t* w1_q,
                                const uint8_t* w1_sf, const uint8_t* w2_q, const uint8_t* w2_sf, void* y,
                                void* workspace, size_t workspace_bytes, void* stream, void* const* events,
                                const int32_t* token_of_row = nullptr, int64_t x_rows = 0,
                                void* saved = nullptr, size_t saved_bytes = 0) {
  if (R < 0 || E < 1 || E > 1024 || H <= 0 || F <= 0) return MXFP8_ERR_INVALID_ARG;
  if (H % 128 != 0 || F % 128 != 0) return MXFP8_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(E) * 2 * F > INT32_MAX || static_cast<int64_t>(E) * H > INT32_MAX)
    return MXFP8_ERR_UNSUPPORTED;
  const void* ptrs[] = {split_sizes, w1_q, w1_sf, w2_q, w2_sf, workspace};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned16(p)) return MXFP8_ERR_INVALID_ARG;
  // row buffers: required when they hold rows (a call without routed rows may pass NULL)
  if (!rows_ok(x_sorted, token_of_row != nullptr ? x_rows : R) || !rows_ok(y, R) || !rows_ok(gates, 0))
    return MXFP8_ERR_INVALID_ARG;
  WsLayout L;
  if (!ws_layout(R, H, F, E, &L)) return MXFP8_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < L.total) return MXFP8_ERR_WORKSPACE;
  if (saved != nullptr && (!aligned16(saved) || saved_bytes < static_cast<size_t>(L.r_pad) * 2 * F * 2))
    return MXFP8_ERR_WORKSPACE;
  return launch_grouped_mlp(x_sorted, R, H, F, E, split_sizes, gates, w1_q, w1_sf, w2_q, w2_sf, y, workspace, L,
                            static_cast<cudaStream_t>(stream), events, token_of_row, x_rows,
                            static_cast<uint16_t*>(saved));
}

int grouped_mlp_fwd(const void* x_sorted, int64_t R, int64_t H, int64_t F, int E, const int32_t* split_sizes,
                    const float* gates, const uint8_t* w1_q, const uint8_t* w1_sf, const uint8_t* w2_q,
                    const uint8_t* w2_sf, void* y, void* workspace, size_t workspace_bytes, void* stream) {
  return grouped_mlp_fwd_impl(x_sorted, R, H, F, E, split_sizes, gates, w1_q, w1_sf, w2_q, w2_sf, y, workspace,
                              workspace_bytes, stream, nullptr);
}

int grouped_mlp_fwd_timed(const void* x_sorted, int64_t R, int64_t H, int64_t F, int E, const int32_t* split_sizes,
                          const float* gates, const uint8_t* w1_q, const uint8_t* w1_sf, const uint8_t* w2_q,
                          const uint8_t* w2_sf, void* y, void* workspace, size_t workspace_bytes, void* stream,
                          void* const* stage_events) {
  if (stage_events == nullptr) return MXFP8_ERR_INVALID_ARG;
  return grouped_mlp_fwd_impl(x_sorted, R, H, F, E, split_sizes, gates, w1_q, w1_sf, w2_q, w2_sf, y, workspace,
                              workspace_bytes, stream, stage_events);
}

int grouped_mlp_fwd_tokens(const void* x_tokens, int64_t T, const int32_t* token_of_row, int64_t R, int64_t H,
                           int64_t F, int E, const int32_t* split_sizes, const float* gates_sorted,
                           const uint8_t* w1_q, const uint8_t* w1_sf, const uint8_t* w2_q, const uint8_t* w2_sf,
                           void* y_rows, void* workspace, size_t workspace_bytes, void* stream) {
  if (T < 0 || !rows_ok(token_of_row, R)) return MXFP8_ERR_INVALID_ARG;
  return grouped_mlp_fwd_impl(x_tokens, R, H, F, E, split_sizes, gates_sorted, w1_q, w1_sf, w2_q, w2_sf, y_rows,
                              workspace, workspace_bytes, stream, nullptr, token_of_row, T);
}

size_t moe_permute_workspace_size(int64_t T, int k, int E) {
  if (T < 0 || k < 1 || E < 1 || E > 1024 || T * k > INT32_MAX) return 0;
  return permute_workspace_bytes(T * k, E);
}

int moe_permute(const int32_t* experts, const float* gates, int64_t T, int k, int E, int32_t* split_sizes,
                int32_t* row_of_slot, int32_t* token_of_row, float* gates_sorted, void* workspace,
                size_t workspace_bytes, void* stream) {
  if (T < 0 || k < 1 || E < 1 || E > 1024 || T * k > INT32_MAX) return MXFP8_ERR_INVALID_ARG;
  if (split_sizes == nullptr || workspace == nullptr || !aligned16(workspace)) return MXFP8_ERR_INVALID_ARG;
  if (T > 0 && (experts == nullptr || row_of_slot == nullptr || token_of_row == nullptr)) return MXFP8_ERR_INVALID_ARG;
  if ((gates == nullptr) != (gates_sorted == nullptr)) return MXFP8_ERR_INVALID_ARG;
  if (workspace_bytes < permute_workspace_bytes(T * k, E)) return MXFP8_ERR_WORKSPACE;
  const cudaError_t e = launch_permute(experts, gates, T, k, E, split_sizes, row_of_slot, token_of_row, gates_sorted,
                                       workspace, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MXFP8_OK : MXFP8_ERR_CUDA;
}

int moe_combine(const void* y_rows, const int32_t* row_of_slot, int64_t T, int k, int64_t H, void* out,
                void* stream) {
  if (T < 0 || k < 1 || H <= 0 || H % 8 != 0 || T * k > INT32_MAX) return MXFP8_ERR_INVALID_ARG;
  if (T == 0) return MXFP8_OK;
  if (y_rows == nullptr || row_of_slot == nullptr || out == nullptr || !aligned16(y_rows) || !aligned16(out))
    return MXFP8_ERR_INVALID_ARG;
  const cudaError_t e = launch_combine(y_rows, row_of_slot, T, k, H, out, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MXFP8_OK : MXFP8_ERR_CUDA;
}

int moe_gather_rows(const void* src, int64_t nsrc, int64_t row_bytes, const int32_t* index, int64_t n, void* dst,
                    void* stream) {
  if (nsrc < 0 || n < 0 || row_bytes <= 0 || row_bytes % 4 != 0) return MXFP8_ERR_INVALID_ARG;
  if (n == 0) return MXFP8_OK;
  if (index == nullptr || dst == nullptr || (nsrc > 0 && src == nullptr)) return MXFP8_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(src) & 3u) != 0 || (reinterpret_cast<uintptr_t>(dst) & 3u) != 0)
    return MXFP8_ERR_INVALID_ARG;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return MXFP8_ERR_CUDA;
  const cudaError_t e = launch_gather_rows(src, nsrc, row_bytes, index, n, dst, sms, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MXFP8_OK : MXFP8_ERR_CUDA;
}

size_t grouped_mlp_saved_bytes(int64_t R, int64_t H, int64_t F, int E) {
  WsLayout L;
  if (!ws_layout(R, H, F, E, &L)) return 0;
  return static_cast<size_t>(L.r_pad) * 2 * F * 2;
}

int grouped_mlp_fwd_train(const void* x_sorted, int64_t R, int64_t H, int64_t F, int E, const int32_t* split_sizes,
                          const float* gates, const uint8_t* w1_q, const uint8_t* w1_sf, const uint8_t* w2_q,
                          const uint8_t* w2_sf, void* y, void* saved, size_t saved_bytes, void* workspace,
                          size_t workspace_bytes, void* stream) {
  if (saved == nullptr) return MXFP8_ERR_INVALID_ARG;
  return grouped_mlp_fwd_impl(x_sorted, R, H, F, E, split_sizes, gates, w1_q, w1_sf, w2_q, w2_sf, y, workspace,
                              workspace_bytes, stream, nullptr, nullptr, 0, saved, saved_bytes);
}

size_t grouped_mlp_bwd_workspace_size(int64_t R, int64_t H, int64_t F, int E) {
  BwdWsLayout L;
  if (!bwd_ws_layout(R, H, F, E, &L)) return 0;
  return L.total;
}

int grouped_mlp_bwd_workspace_layout(int64_t R, int64_t H, int64_t F, int E, uint64_t* out) {
  BwdWsLayout L;
  if (out == nullptr || !bwd_ws_layout(R, H, F, E, &L)) return MXFP8_ERR_INVALID_ARG;
  out[0] = L.meta;
  out[1] = L.dguq;
  out[2] = L.dgusf;
  out[3] = L.dguT;
  out[4] = L.dguTsf;
  out[5] = L.hT;
  out[6] = L.hTsf;
  out[7] = static_cast<uint64_t>(L.r_pad);
  return MXFP8_OK;
}

static int grouped_mlp_bwd_impl(const void* x_sorted, int64_t R, int64_t H, int64_t F, int E,
                                const int32_t* split_sizes, const float* gates, const void* saved,
                                size_t saved_bytes, const uint8_t* w1t_q, const uint8_t* w1t_sf,
                                const uint8_t* w2t_q, const uint8_t* w2t_sf, const void* dy, void* dx, float* dgates,
                                float* dw1, float* dw2, void* workspace, size_t workspace_bytes, void* stream,
                                void* const* events, const int32_t* token_of_row = nullptr, int64_t x_rows = 0) {
  if (R < 0 || E < 1 || E > 1024 || H <= 0 || F <= 0 || x_rows < 0) return MXFP8_ERR_INVALID_ARG;
  if (token_of_row != nullptr && !aligned16(token_of_row)) return MXFP8_ERR_INVALID_ARG;
  if (H % 256 != 0 || F % 128 != 0) return MXFP8_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(E) * 2 * F > INT32_MAX || static_cast<int64_t>(E) * H > INT32_MAX)
    return MXFP8_ERR_UNSUPPORTED;
  const void* ptrs[] = {split_sizes, saved, w1t_q, w1t_sf, w2t_q, w2t_sf, dw1, dw2, workspace};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned16(p)) return MXFP8_ERR_INVALID_ARG;
  // row buffers: required when they hold rows (a call without routed rows may pass NULL)
  const int64_t src_rows = token_of_row != nullptr ? x_rows : R;
  if (!rows_ok(x_sorted, src_rows) || !rows_ok(dy, src_rows) || !rows_ok(dx, R) || !rows_ok(gates, 0) ||
      !rows_ok(dgates, 0))
    return MXFP8_ERR_INVALID_ARG;
  BwdWsLayout L;
  if (!bwd_ws_layout(R, H, F, E, &L)) return MXFP8_ERR_UNSUPPORTED;
  if (saved_bytes < static_cast<size_t>(L.r_pad) * 2 * F * 2) return MXFP8_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < L.total) return MXFP8_ERR_WORKSPACE;
  return launch_grouped_mlp_bwd(x_sorted, R, H, F, E, split_sizes, gates, static_cast<const uint16_t*>(saved),
                                w1t_q, w1t_sf, w2t_q, w2t_sf, dy, dx, dgates, dw1, dw2, workspace, L,
                                static_cast<cudaStream_t>(stream), events, token_of_row, x_rows);
}

int grouped_mlp_bwd(const void* x_sorted, int64_t R, int64_t H, int64_t F, int E, const int32_t* split_sizes,
                    const float* gates, const void* saved, size_t saved_bytes, const uint8_t* w1t_q,
                    const uint8_t* w1t_sf, const uint8_t* w2t_q, const uint8_t* w2t_sf, const void* dy, void* dx,
                    float* dgates, float* dw1, float* dw2, void* workspace, size_t workspace_bytes, void* stream) {
  return grouped_mlp_bwd_impl(x_sorted, R, H, F, E, split_sizes, gates, saved, saved_bytes, w1t_q, w1t_sf, w2t_q,
                              w2t_sf, dy, dx, dgates, dw1, dw2, workspace, workspace_bytes, stream, nullptr);
}

int grouped_mlp_bwd_timed(const void* x_sorted, int64_t R, int64_t H, int64_t F, int E, const int32_t* split_sizes,
                          const float* gates, const void* saved, size_t saved_bytes, const uint8_t* w1t_q,
                          const uint8_t* w1t_sf, const uint8_t* w2t_q, const uint8_t* w2t_sf, const void* dy,
                          void* dx, float* dgates, float* dw1, float* dw2, void* workspace, size_t workspace_bytes,
                          void* stream, void* const* stage_events) {
  if (stage_events == nullptr) return MXFP8_ERR_INVALID_ARG;
  return grouped_mlp_bwd_impl(x_sorted, R, H, F, E, split_sizes, gates, saved, saved_bytes, w1t_q, w1t_sf, w2t_q,
                              w2t_sf, dy, dx, dgates, dw1, dw2, workspace, workspace_bytes, stream, stage_events);
}

int grouped_mlp_fwd_tokens_train(const void* x_tokens, int64_t T, const int32_t* token_of_row, int64_t R,
                                 int64_t H, int64_t F, int E, const int32_t* split_sizes, const float* gates_sorted,
                                 const uint8_t* w1_q, const uint8_t* w1_sf, const uint8_t* w2_q, const uint8_t* w2_sf,
                                 void* y_rows, void* saved, size_t saved_bytes, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  if (T < 0 || !rows_ok(token_of_row, R) || saved == nullptr) return MXFP8_ERR_INVALID_ARG;
  return grouped_mlp_fwd_impl(x_tokens, R, H, F, E, split_sizes, gates_sorted, w1_q, w1_sf, w2_q, w2_sf, y_rows,
                              workspace, workspace_bytes, stream, nullptr, token_of_row, T, saved, saved_bytes);
}

int grouped_mlp_bwd_tokens(const void* x_tokens, int64_t T, const int32_t* token_of_row, int64_t R, int64_t H,
                           int64_t F, int E, const int32_t* split_sizes, const float* gates_sorted, const void* saved,
                           size_t saved_bytes, const uint8_t* w1t_q, const uint8_t* w1t_sf, const uint8_t* w2t_q,
                           const uint8_t* w2t_sf, const void* d_out_tokens, void* dx_rows, float* dgates_sorted,
                           float* dw1, float* dw2, void* workspace, size_t workspace_bytes, void* stream) {
  if (T < 0 || !rows_ok(token_of_row, R)) return MXFP8_ERR_INVALID_ARG;
  return grouped_mlp_bwd_impl(x_tokens, R, H, F, E, split_sizes, gates_sorted, saved, saved_bytes, w1t_q, w1t_sf,
                              w2t_q, w2t_sf, d_out_tokens, dx_rows, dgates_sorted, dw1, dw2, workspace,
                              workspace_bytes, stream, nullptr, token_of_row, T);
}

int mxfp8_quantize_colwise_t(const void* x, int64_t M, int64_t K, int sf_layout, uint8_t* q_t, uint8_t* sf_t,
                             void* stream) {
  if (M < 0 || K < 0 || K % 32 != 0) return MXFP8_ERR_INVALID_ARG;
  if (sf_layout != MXFP8_SF_COMPACT && sf_layout != MXFP8_SF_MMA) return MXFP8_ERR_INVALID_ARG;
  if (M % 128 != 0 || (sf_layout == MXFP8_SF_MMA && K % 128 != 0)) return MXFP8_ERR_UNSUPPORTED;
  if (M == 0 || K == 0) return MXFP8_OK;
  if (x == nullptr || q_t == nullptr || sf_t == nullptr || !aligned16(x) || !aligned16(q_t))
    return MXFP8_ERR_INVALID_ARG;
  const cudaError_t e = launch_quantize_t(x, M, K, M, sf_layout == MXFP8_SF_MMA, q_t, sf_t, nullptr, 0, nullptr, 0,
                                          static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MXFP8_OK : MXFP8_ERR_CUDA;
}

int mxfp8_check_device_error(const void* workspace, void* stream, uint32_t* flags) {
  if (workspace == nullptr) return MXFP8_ERR_INVALID_ARG;
  uint32_t w = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&w, workspace, sizeof(w), cudaMemcpyDeviceToHost, s) != cudaSuccess) return MXFP8_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MXFP8_ERR_CUDA;
  if (flags) *flags = w;
  if (w & ERR_TIMEOUT_MASK) return MXFP8_ERR_DEVICE_TIMEOUT;
  if (w & (ERR_SPLIT_SUM | ERR_SPLIT_NEGATIVE)) return MXFP8_ERR_SPLIT_MISMATCH;
  if (w & (ERR_EXPERT_RANGE | ERR_TOKEN_RANGE)) return MXFP8_ERR_INVALID_ARG;
  return MXFP8_OK;
}

}  // extern "C"
