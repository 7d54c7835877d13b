/*
 * mxfp8moe.h -- C ABI of the GB300 (sm_103a) MXFP8 expert-MLP library.
 *
 * The operations are those of the page "Efficient MoE training for biological foundation
 * models" (news summary of NVIDIA's Transformer Engine MoE post), section "Key technical
 * approaches in the recipe":
 *   item 1  GroupedLinear: many per-expert linears in one call over tokens grouped by expert,
 *           with per-expert token counts split_sizes;
 *   item 2  MXFP8: 8-bit E4M3 values, one scale per block of 32 consecutive values;
 *   item 3  the fused forward GroupedLinear -> ScaledSwiGLU -> GroupedLinear, which applies the
 *           routing weight together with the SwiGLU activation and does not keep the
 *           intermediate in 16-bit memory.
 * The block scale rule is not printed on the pages; this library uses the OCP MX v1.0 rule:
 * shared exponent s = floor(log2(block amax)) - 8 clamped to [-127, 127], stored as the E8M0
 * byte s + 127 (an all-zero block gets byte 0); each element is x * 2^-s rounded to the nearest
 * E4M3 value, ties to even, saturated to +-448.
 *
 * Conventions for every call
 *   - Pointers marked (device) are CUDA device (or managed) addresses owned by the caller; the
 *     library never allocates, frees or keeps them after the call returns.  Pointers marked
 *     (host) are ordinary host memory read during the call.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).  All work
 *     is enqueued on it; no call synchronizes the host except mxfp8_check_device_error.
 *   - Every device pointer must be 16-byte aligned unless its call says otherwise.  bf16
 *     tensors are row-major IEEE bfloat16.
 *   - Return value: an mxfp8_status.  Argument errors are detected on the host before anything
 *     is enqueued and leave all buffers untouched.  Conditions only visible on the device
 *     (split_sizes that do not add up to R, a pipeline wait that timed out) set bits in the
 *     error word inside the caller's workspace; read them with mxfp8_check_device_error.
 *     No call aborts, throws or traps.
 */
#ifndef MXFP8MOE_H
#define MXFP8MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MXFP8_OK = 0,
    MXFP8_ERR_INVALID_ARG = 1,     /* null/unaligned pointer, negative or inconsistent size   */
    MXFP8_ERR_UNSUPPORTED = 2,     /* shape outside what the kernels support (see each call)  */
    MXFP8_ERR_WORKSPACE = 3,       /* workspace smaller than grouped_mlp_workspace_size()     */
    MXFP8_ERR_CUDA = 4,            /* a CUDA runtime/driver call failed (launch, attribute)   */
    MXFP8_ERR_DEVICE_TIMEOUT = 5,  /* a bounded device-side wait gave up (from check only)    */
    MXFP8_ERR_SPLIT_MISMATCH = 6   /* sum(split_sizes) != R or a negative count (check only)  */
} mxfp8_status;

/* Direction flags for mxfp8_quantize (may be OR-ed). */
enum { MXFP8_ROWWISE = 1, MXFP8_COLWISE = 2 };

/* Scale-factor layouts.
 *   MXFP8_SF_COMPACT: row-wise bytes [M, K/32] row-major; column-wise bytes [ceil(M/32), K].
 *   MXFP8_SF_MMA: the layout the block-scaled tensor-core MMA consumes.  For a matrix of `rows`
 *     rows and `kb` = K/32 blocks per row, bytes are grouped in 512-byte atoms of 128 rows x 4
 *     blocks; atom (rt, kt) starts at byte 512 * (rt * ceil(kb/4) + kt) and holds the byte of
 *     row r = 128*rt + 32*j + i and block 4*kt + b at offset 16*i + 4*j + b.  Column-wise scales
 *     use it with rows = K (columns of x) and kb = ceil(M/32).                                  */
enum { MXFP8_SF_COMPACT = 0, MXFP8_SF_MMA = 1 };

/* Bytes of the scale-factor buffer for one direction and layout (0 on bad arguments). */
size_t mxfp8_sf_bytes(int64_t M, int64_t K, int direction, int sf_layout);

/*
 * mxfp8_quantize -- MXFP8 quantization of a bf16 matrix (item 2 above).
 *   x       (device) bf16 [M, K], row-major.
 *   dirs    MXFP8_ROWWISE and/or MXFP8_COLWISE.  Row-wise blocks are 32 consecutive elements of
 *           a row; column-wise blocks are 32 consecutive rows of one column (a last block of
 *           fewer rows uses the rows present).  Both directions are produced from one read of x.
 *   q_row   (device) E4M3 codes [M, K] (row-wise), or NULL when not requested.
 *   sf_row  (device) row-wise E8M0 bytes, mxfp8_sf_bytes(M, K, MXFP8_ROWWISE, sf_layout) bytes.
 *   q_col   (device) E4M3 codes [M, K] in x's layout (column-wise), or NULL.
 *   sf_col  (device) column-wise E8M0 bytes, mxfp8_sf_bytes(M, K, MXFP8_COLWISE, sf_layout).
 * Requirements: M >= 0, K % 32 == 0; with MXFP8_SF_MMA also M % 128 == 0 and K % 128 == 0.
 * M == 0 or K == 0 is a no-op.  Outputs are fully overwritten.  Results are bit-exact with the
 * rule above.
 */
int mxfp8_quantize(const void* x, int64_t M, int64_t K, int dirs, int sf_layout,
                   uint8_t* q_row, uint8_t* sf_row, uint8_t* q_col, uint8_t* sf_col, void* stream);

/* Workspace bytes grouped_mlp_fwd needs for these sizes (0 on bad arguments).  It holds the
 * device tile schedule, the error word, the quantized activations and the quantized
 * intermediate, each in an expert-padded row space (every expert's rows rounded up to a multiple
 * of 256) of at most R + 255*E rows. */
size_t grouped_mlp_workspace_size(int64_t R, int64_t H, int64_t F, int E);

/*
 * grouped_mlp_fwd -- fused MXFP8 grouped expert MLP forward (items 1-3 above):
 *   for each expert e and each of its rows r (rows are grouped by expert in x_sorted):
 *     g = xq_r W1[e, 0:F]^T,  u = xq_r W1[e, F:2F]^T            (GroupedLinear 1, fp32 accum.)
 *     h = gate_r * silu(g) * u,  silu(g) = g / (1 + exp(-g))    (ScaledSwiGLU)
 *     hq = MXFP8(h) row-wise along F                            (never stored in bf16)
 *     y_r = bf16( hq W2[e]^T )                                  (GroupedLinear 2)
 *   where xq_r is the row-wise MXFP8 quantization of x_sorted[r] (done inside the call).
 * Arguments:
 *   x_sorted    (device) bf16 [R, H], rows grouped by expert in expert order.
 *   split_sizes (device) int32 [E], rows per expert; may contain zeros; must sum to R.
 *   gates       (device) float [R] per-row routing weight, or NULL for 1.
 *   w1_q,w1_sf  (device) W1 [E, 2F, H] E4M3 codes + row-wise E8M0 bytes in MXFP8_SF_MMA layout
 *               for the [E*2F, H] matrix (as mxfp8_quantize(W1, E*2F, H, ROWWISE, SF_MMA)
 *               writes them).  Rows [0, F) of each expert are the gate projection, [F, 2F) up.
 *   w2_q,w2_sf  (device) W2 [E, H, F] codes + bytes in MXFP8_SF_MMA layout for [E*H, F].
 *   y           (device) bf16 [R, H] output, rows in x_sorted's order; fully overwritten.
 *   workspace   (device) at least grouped_mlp_workspace_size(R, H, F, E) bytes, 256-byte
 *               aligned.  It must not be shared by two calls in flight at the same time.
 * Requirements: R >= 0, 1 <= E <= 1024, H % 128 == 0, F % 128 == 0, H, F >= 128.  With R == 0
 * (no routed rows, e.g. an expert-parallel rank that received no tokens) x_sorted and y may be
 * NULL; the call still checks split_sizes on the device.  The same holds for the row buffers of
 * the other grouped-MLP calls below (x, the output gradient, dx, token_of_row).
 * The call never reads split_sizes on the host.  If they do not sum to R (or one is negative),
 * the kernels do no work, y is left unspecified and the workspace's error word reports
 * MXFP8_ERR_SPLIT_MISMATCH.
 */
int grouped_mlp_fwd(const void* x_sorted, int64_t R, int64_t H, int64_t F, int E,
                    const int32_t* split_sizes, const float* gates,
                    const uint8_t* w1_q, const uint8_t* w1_sf,
                    const uint8_t* w2_q, const uint8_t* w2_sf,
                    void* y, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Dispatch and combine around the grouped MLP (page section "Dense vs. MoE scaling": each token
 * uses a few of the experts; item 1: GroupedLinear runs on tokens gathered per expert).  The
 * router (a small GEMM + top-k) is not part of this library: its choices arrive as expert ids.
 *
 * moe_permute -- stable sort of the router's (token, slot) choices by expert, on the device.
 *   experts      (device) int32 [T, k]: expert of slot j of token t, in [0, E).
 *   gates        (device) float [T, k] routing weights, or NULL (then gates_sorted must be NULL).
 *   split_sizes  (device, out) int32 [E]: rows per expert.
 *   row_of_slot  (device, out) int32 [T, k]: sorted row of each (token, slot).
 *   token_of_row (device, out) int32 [T*k]: token of each sorted row.
 *   gates_sorted (device, out) float [T*k] or NULL.
 *   workspace    (device) moe_permute_workspace_size(T, k, E) bytes, 16-byte aligned; its first
 *                4 bytes are an error word (mxfp8_check_device_error: MXFP8_ERR_INVALID_ARG when
 *                an expert id is out of range; such slots are skipped and the outputs are then
 *                incomplete).
 * Rows of one expert keep (token, slot) order; experts follow each other in id order, so
 * sorted row r of expert e is split_sizes[0] + ... + split_sizes[e-1] + (rank of the slot).
 * Requirements: T >= 0, k >= 1, 1 <= E <= 1024, T*k < 2^31.
 */
size_t moe_permute_workspace_size(int64_t T, int k, int E);
int moe_permute(const int32_t* experts, const float* gates, int64_t T, int k, int E,
                int32_t* split_sizes, int32_t* row_of_slot, int32_t* token_of_row, float* gates_sorted,
                void* workspace, size_t workspace_bytes, void* stream);

/*
 * grouped_mlp_fwd_tokens -- grouped_mlp_fwd reading token rows directly: sorted row r is row
 * token_of_row[r] of x_tokens [T, H] (the gather is fused into the activation quantize, so the
 * [R, H] sorted copy of x is never written).  Other arguments as grouped_mlp_fwd (gates are in
 * sorted order).  token_of_row (device) int32 [R], values in [0, T); out-of-range ids read as
 * zero rows and set MXFP8_ERR_INVALID_ARG in the workspace error word.
 */
int grouped_mlp_fwd_tokens(const void* x_tokens, int64_t T, const int32_t* token_of_row, int64_t R, int64_t H,
                           int64_t F, int E, const int32_t* split_sizes, const float* gates_sorted,
                           const uint8_t* w1_q, const uint8_t* w1_sf, const uint8_t* w2_q, const uint8_t* w2_sf,
                           void* y_rows, void* workspace, size_t workspace_bytes, void* stream);

/*
 * moe_combine -- out[t] = sum_j y_rows[row_of_slot[t, j]] (fp32 sum, bf16 round to nearest even).
 * The routing weight is already inside y (grouped_mlp_fwd applies it with the SwiGLU), so the
 * combine is a plain sum.  y_rows (device) bf16 [T*k, H]; row_of_slot (device) int32 [T, k];
 * out (device) bf16 [T, H], fully overwritten.  Requirements: H % 8 == 0, 16-byte aligned
 * pointers.  Row ids outside [0, T*k) contribute nothing.
 */
int moe_combine(const void* y_rows, const int32_t* row_of_slot, int64_t T, int k, int64_t H, void* out,
                void* stream);

/*
 * moe_gather_rows -- dst[i] = src[index[i]] for i < n: rows of row_bytes bytes, copied bit for
 * bit whatever their element type (token rows to the ranks that own their experts and back,
 * routing-weight gradients to (token, slot) order).  src (device) [nsrc rows], index (device)
 * int32 [n], dst (device, out) [n rows], fully overwritten; a row whose index lies outside
 * [0, nsrc) is written as zeros.  Requirements: row_bytes % 4 == 0, 4-byte aligned pointers
 * (16-byte rows on 16-byte aligned pointers move as 16-byte words).  n == 0 is a no-op.
 */
int moe_gather_rows(const void* src, int64_t nsrc, int64_t row_bytes, const int32_t* index, int64_t n, void* dst,
                    void* stream);

/* grouped_mlp_fwd with per-kernel timing: identical work and results, and additionally records
 * the 5 caller-created CUDA events stage_events[0..4] (cudaEvent_t as void*, host array) on
 * `stream` before the schedule, activation-quantize, GroupedLinear-1 (+ScaledSwiGLU, requant)
 * and GroupedLinear-2 kernels and after the last one, so cudaEventElapsedTime between
 * consecutive events gives each kernel's device time.  stage_events must not be NULL (use
 * grouped_mlp_fwd instead); an individual NULL entry skips that record. */
int grouped_mlp_fwd_timed(const void* x_sorted, int64_t R, int64_t H, int64_t F, int E,
                          const int32_t* split_sizes, const float* gates,
                          const uint8_t* w1_q, const uint8_t* w1_sf,
                          const uint8_t* w2_q, const uint8_t* w2_sf,
                          void* y, void* workspace, size_t workspace_bytes, void* stream,
                          void* const* stage_events);

/* grouped_mlp_fwd_noalloc -- grouped_mlp_fwd for callers that cannot allocate device memory.
 * The pages have no counterpart: this is a library convenience, not a step of the method.
 * Some callers cannot call cudaMalloc where they run the forward (allocator hooks, out-of-memory
 * handlers, hosts whose memory pool is owned elsewhere).  This variant takes the same inputs and
 * output as grouped_mlp_fwd but no workspace: its scratch is one 64 MiB file-scope device array.
 *   - Problems whose grouped_mlp_workspace_size() exceeds 64 MiB return MXFP8_ERR_WORKSPACE
 *     before anything is enqueued.
 *   - The first call on a device is a set-up call: with that device current it looks up the
 *     array's device address (cudaGetSymbolAddress) and sets the kernels' launch attributes.
 *     Under CUDA's lazy module loading (the default) this is when the array and the library's
 *     kernels are loaded onto that device, which takes device memory inside the driver; the
 *     device then holds the array until the process exits.  So make the first call on each
 *     device while allocation is still allowed, and before any stream capture.  Later calls on
 *     that device allocate nothing.
 *   - All calls on a device share the array and leave the last call's contents in it; nothing
 *     in it needs to start at zero.  Calls that overlap on the GPU race on it.
 *   - Device-side conditions (split_sizes not summing to R, a timed-out wait) are not reported;
 *     use grouped_mlp_fwd with a workspace and mxfp8_check_device_error to see them.
 *   - No call makes cudaMalloc, cudaFree or any allocating library call. */
int grouped_mlp_fwd_noalloc(const void* x_sorted, int64_t R, int64_t H, int64_t F, int E,
                            const int32_t* split_sizes, const float* gates,
                            const uint8_t* w1_q, const uint8_t* w1_sf,
                            const uint8_t* w2_q, const uint8_t* w2_sf,
                            void* y, void* stream);

/*
 * Backward of the grouped MLP (page item 3: the fused forward op has a corresponding fused
 * backward op; the pages give no further detail).  Reading implemented, as in MXFP8 training:
 * gradients pass straight through every quantization; each backward GEMM takes MXFP8 operands
 * with blocks of 32 along its own contraction axis; the tensors handed from one backward GEMM to
 * the next ([dG | dU] and h) are bf16; the forward's pre-activations [G | U] are saved as bf16.
 * For sorted row r of expert e, with s = silu(g), s' = sig(g) (1 + g (1 - sig(g))):
 *   dh     = dy_r W2[e]                 (MXFP8: dy along H, W2 along H)
 *   dG     = dh * gate_r * u * s',  dU = dh * gate_r * s,  dgate_r = sum_j dh_j s_j u_j
 *   dx_r   = [dG | dU] W1[e]            (MXFP8 along 2F)
 *   dW2[e] = dy_e^T h_e,  dW1[e] = [dG | dU]_e^T x_e    (MXFP8 along the expert's rows)
 *
 * grouped_mlp_saved_bytes -- bytes of the saved pre-activations of one training forward
 *   (bf16 [G | U] in the expert-padded row space); 0 on bad arguments.
 * grouped_mlp_fwd_train -- grouped_mlp_fwd that also writes those pre-activations to `saved`
 *   (device, saved_bytes >= grouped_mlp_saved_bytes, 16-byte aligned, caller-owned; keep it
 *   until the backward has run).  Same results and errors as grouped_mlp_fwd.
 * grouped_mlp_bwd -- all arguments on the device unless noted:
 *   x_sorted, split_sizes, gates   as given to the forward (gates may be NULL for 1).
 *   saved        the forward's pre-activations (grouped_mlp_fwd_train).
 *   w1t_q,w1t_sf W1 quantized along 2F: mxfp8_quantize_colwise_t(W1 [E*2F, H], SF_MMA), i.e.
 *                codes [H, E*2F] (row k holds column k of the stacked W1) + bytes.
 *   w2t_q,w2t_sf W2 quantized along H: mxfp8_quantize_colwise_t(W2 [E*H, F], SF_MMA): codes
 *                [F, E*H] + bytes.
 *   dy           bf16 [R, H] gradient of y, rows in x_sorted's order.
 *   dx           bf16 [R, H] out.   dgates  float [R] out, or NULL to skip.
 *   dw1          float [E, 2F, H] out (gradient of W1).   dw2  float [E, H, F] out.
 *   workspace    grouped_mlp_bwd_workspace_size(R, H, F, E) bytes, 256-byte aligned.
 * Requirements: H % 256 == 0, F % 128 == 0 (all backward GEMMs run on CTA pairs with 256-wide
 * tiles; MXFP8_ERR_UNSUPPORTED otherwise), 1 <= E <= 1024.  Outputs are fully overwritten (an
 * expert without rows gets zero weight gradients).  Split errors and timeouts are reported in
 * the workspace error word as for the forward.
 * grouped_mlp_bwd_timed additionally records 7 caller-created events (stage_events[0..6]) around
 * its stages: quantizations of dy and x | dh + ScaledSwiGLU backward with dGU and h quantized in
 * its epilogue | dgate reduction | dx | dW2 | dW1.
 */
size_t grouped_mlp_saved_bytes(int64_t R, int64_t H, int64_t F, int E);
int grouped_mlp_fwd_train(const void* x_sorted, int64_t R, int64_t H, int64_t F, int E, const int32_t* split_sizes,
                          const float* gates, const uint8_t* w1_q, const uint8_t* w1_sf, const uint8_t* w2_q,
                          const uint8_t* w2_sf, void* y, void* saved, size_t saved_bytes, void* workspace,
                          size_t workspace_bytes, void* stream);
size_t grouped_mlp_bwd_workspace_size(int64_t R, int64_t H, int64_t F, int E);
/* Byte offsets of the pieces of a grouped_mlp_bwd workspace that hold the quantized [dG | dU]
 * and h the dh GEMM's epilogue writes, for inspection by tests.  All live in the expert-padded
 * row space of R_pad rows (padding rows are zero values); codes are E4M3, scale bytes UE8M0 in
 * the tensor-core layout (mxfp8_quantize, MXFP8_SF_MMA) of the matrix named:
 *   [0] error word
 *   [1] [dG | dU] row-wise codes [R_pad, 2F]        [2] their scale bytes ([R_pad, 2F])
 *   [3] [dG | dU] column-wise codes, transposed [2F, R_pad]   [4] their scale bytes ([2F, R_pad])
 *   [5] h column-wise codes, transposed [F, R_pad]  [6] their scale bytes ([F, R_pad])
 *   [7] R_pad (not an offset)
 * out: 8 entries (host).  Returns MXFP8_OK or MXFP8_ERR_INVALID_ARG. */
int grouped_mlp_bwd_workspace_layout(int64_t R, int64_t H, int64_t F, int E, uint64_t* out);
int grouped_mlp_bwd(const void* x_sorted, int64_t R, int64_t H, int64_t F, int E, const int32_t* split_sizes,
                    const float* gates, const void* saved, size_t saved_bytes, const uint8_t* w1t_q,
                    const uint8_t* w1t_sf, const uint8_t* w2t_q, const uint8_t* w2t_sf, const void* dy, void* dx,
                    float* dgates, float* dw1, float* dw2, void* workspace, size_t workspace_bytes, void* stream);
int grouped_mlp_bwd_timed(const void* x_sorted, int64_t R, int64_t H, int64_t F, int E, const int32_t* split_sizes,
                          const float* gates, const void* saved, size_t saved_bytes, const uint8_t* w1t_q,
                          const uint8_t* w1t_sf, const uint8_t* w2t_q, const uint8_t* w2t_sf, const void* dy,
                          void* dx, float* dgates, float* dw1, float* dw2, void* workspace, size_t workspace_bytes,
                          void* stream, void* const* stage_events);

/* The MoE layer in training (f1 around the backward): grouped_mlp_fwd_tokens_train is
 * grouped_mlp_fwd_tokens that also saves the pre-activations (as grouped_mlp_fwd_train);
 * grouped_mlp_bwd_tokens is grouped_mlp_bwd reading x and the output gradient as token rows:
 * sorted row r reads row token_of_row[r] of x_tokens [T, H] and of d_out_tokens [T, H].  That
 * gather is the gradient of moe_combine; the caller finishes the layer's backward with
 * moe_combine(dx_rows, row_of_slot) (the gradient of the token gather) and picks
 * dgates_sorted[row_of_slot[t, j]] for the routing weight of (t, j) (moe_gather_rows).  Other arguments, outputs
 * and errors as grouped_mlp_fwd_train / grouped_mlp_bwd (dx_rows and dgates_sorted in sorted-row
 * order); token ids outside [0, T) read zero rows and set MXFP8_ERR_INVALID_ARG in the workspace
 * error word. */
int grouped_mlp_fwd_tokens_train(const void* x_tokens, int64_t T, const int32_t* token_of_row, int64_t R,
                                 int64_t H, int64_t F, int E, const int32_t* split_sizes, const float* gates_sorted,
                                 const uint8_t* w1_q, const uint8_t* w1_sf, const uint8_t* w2_q, const uint8_t* w2_sf,
                                 void* y_rows, void* saved, size_t saved_bytes, void* workspace,
                                 size_t workspace_bytes, void* stream);
int grouped_mlp_bwd_tokens(const void* x_tokens, int64_t T, const int32_t* token_of_row, int64_t R, int64_t H,
                           int64_t F, int E, const int32_t* split_sizes, const float* gates_sorted, const void* saved,
                           size_t saved_bytes, const uint8_t* w1t_q, const uint8_t* w1t_sf, const uint8_t* w2t_q,
                           const uint8_t* w2t_sf, const void* d_out_tokens, void* dx_rows, float* dgates_sorted,
                           float* dw1, float* dw2, void* workspace, size_t workspace_bytes, void* stream);

/* mxfp8_quantize_colwise_t -- column-wise MXFP8 (blocks of 32 consecutive rows, item 2) with the
 * codes written transposed, the operand form of GEMMs that contract over x's rows.
 *   x    (device) bf16 [M, K], row-major.
 *   q_t  (device, out) E4M3 codes [K, M]: row k holds column k of x.
 *   sf_t (device, out) E8M0 bytes of the [K, M] code matrix with blocks along its rows:
 *        compact [K, M/32], or MXFP8_SF_MMA layout (mxfp8_sf_bytes(K, M, ROWWISE, SF_MMA)).
 * Requirements: M % 128 == 0, K % 32 == 0 (K % 128 == 0 for MXFP8_SF_MMA), 16-byte aligned
 * pointers.  Same rule and rounding as mxfp8_quantize; M == 0 or K == 0 is a no-op. */
int mxfp8_quantize_colwise_t(const void* x, int64_t M, int64_t K, int sf_layout, uint8_t* q_t, uint8_t* sf_t,
                             void* stream);

/* Byte offsets of the pieces of a grouped_mlp_fwd workspace, for inspection by tests:
 *   [0] error word (uint32)   [1] schedule          [2] quantized activations [R_pad, H]
 *   [3] their E8M0 bytes (MXFP8_SF_MMA layout)      [4] quantized intermediate [R_pad, F]
 *   [5] its E8M0 bytes (MXFP8_SF_MMA layout)        [6] R_pad (row capacity, not an offset)
 * Expert e's rows start at padded row sum_{e'<e} 256*ceil(split[e']/256); padding rows are 0.
 * Returns MXFP8_OK, or MXFP8_ERR_INVALID_ARG for bad sizes.  out must hold 7 entries (host). */
int grouped_mlp_workspace_layout(int64_t R, int64_t H, int64_t F, int E, uint64_t* out);

/* Copies the workspace's error word to the host (synchronizes `stream`) and maps it to a
 * status: MXFP8_OK, MXFP8_ERR_SPLIT_MISMATCH, MXFP8_ERR_INVALID_ARG (bad expert or token id) or
 * MXFP8_ERR_DEVICE_TIMEOUT.  Works on grouped_mlp_fwd and moe_permute workspaces.  The raw bits go to
 * *flags when flags is not NULL (host). */
int mxfp8_check_device_error(const void* workspace, void* stream, uint32_t* flags);

/*
 * NVFP4 variant of the chain.  The page "TransformerEngine-accelerated Llama 3 training with
 * native PyTorch training loop" lists NVFP4 beside MXFP8 among its quantized-training recipes
 * (feature table; section "Quantized Training (FP8 / MXFP8 / NVFP4)") and defines nothing of
 * it; this library takes NVIDIA's published NVFP4:
 *   - elements E2M1 (values 0, 0.5, 1, 1.5, 2, 3, 4, 6 with a sign), stored two per byte: value
 *     2i of a row in the low nibble of byte i, value 2i+1 in its high nibble, sign in bit 3;
 *   - one E4M3 scale code per 16 consecutive values of a row;
 *   - one binary32 encode scale per tensor, s_enc = 448 * 6 / amax(tensor) (1 if amax = 0, at
 *     most FLT_MAX), kept as the tensor's amax (a device float);
 *   - block quantization in binary32, round to nearest even, saturating:
 *       S = E4M3(fl32(fl32(amax_block / 6) * s_enc)),  r = fl32(s_enc / S) (0 if S = 0),
 *       code_i = E2M1(fl32(v_i * r));  the pair stands for code_i * S / s_enc.
 * Scale layouts: MXFP8_SF_COMPACT is [M, K/16] row-major.  MXFP8_SF_MMA is the tensor-core
 * layout of MXFP8_SF_MMA with 16-value blocks in place of 32-value ones and each row's blocks
 * padded to a multiple of 16 (K to a multiple of 256) with zero codes: atom (rt, kt) of 128
 * rows x 4 blocks at byte 512 * (rt * 4*ceil(K/256) + kt), row 32j+i, block 4kt+b at 16i+4j+b.
 *
 * nvfp4_sf_bytes -- bytes of the scale-code buffer (0 on bad arguments).
 * nvfp4_quantize -- NVFP4 of a bf16 matrix.
 *   x    (device) bf16 [M, K] row-major, finite.   q (device, out) codes [M, K/2].
 *   sf   (device, out) nvfp4_sf_bytes(M, K, sf_layout) bytes.
 *   amax (device, out) float: max |x| over the whole matrix (it defines s_enc; pass it to
 *        nvfp4_grouped_mlp_fwd with the codes).  Two kernels: a reduction for amax, then the
 *        quantization.
 *   Requirements: K % 16 == 0; with MXFP8_SF_MMA also M % 128 == 0, K % 128 == 0; 16-byte aligned
 *   x and q, 4-byte aligned amax.  Results are bit-exact with the rule above.
 */
size_t nvfp4_sf_bytes(int64_t M, int64_t K, int sf_layout);
int nvfp4_quantize(const void* x, int64_t M, int64_t K, int sf_layout, uint8_t* q, uint8_t* sf, float* amax,
                   void* stream);

/*
 * nvfp4_grouped_mlp_fwd -- grouped_mlp_fwd with NVFP4 operands (tcgen05 kind::mxf4nvf4 block-scaled
 * MMA, CTA pairs):
 *     xq_r = NVFP4 of x_sorted row r under the encode scale of max|x_sorted| (computed inside);
 *     g, u = xq_r W1[e, gate/up]^T, h = gate_r * silu(g) * u  (fp32 accumulation, dequantized by
 *            1 / (s_x s_w1));
 *     hq = NVFP4 of h along F under the encode scale of h_amax (values beyond it saturate: the
 *          intermediate's largest value is not known before GroupedLinear 1 has run, so the
 *          caller supplies the magnitude, e.g. the one the previous call observed);
 *     y_r = bf16( hq W2[e]^T / (s_h s_w2) ).
 *   w1_q/w1_sf/w1_amax: nvfp4_quantize(W1 [E*2F, H], MXFP8_SF_MMA) outputs (rows [0, F) of each
 *   expert gate, [F, 2F) up); w2_q/w2_sf/w2_amax: the same for W2 [E*H, F].
 *   h_amax (host) > 0.  stage_events: NULL, or 5 caller-created events recorded around the
 *   schedule, activation amax + quantize, GroupedLinear 1 (+ScaledSwiGLU, requant) and
 *   GroupedLinear 2 stages.  Other arguments as grouped_mlp_fwd; the workspace
 *   (nvfp4_grouped_mlp_workspace_size bytes, 256-byte aligned) also receives, as float bits, the
 *   largest |x| and the largest |h| the call saw (nvfp4_grouped_mlp_workspace_layout entry 1:
 *   two words).  Requirements: H % 256 == 0, F % 128 == 0, 1 <= E <= 1024, a GPU where two-CTA
 *   clusters fit (MXFP8_ERR_UNSUPPORTED otherwise).  Device-side errors as for grouped_mlp_fwd.
 * nvfp4_grouped_mlp_workspace_layout -- byte offsets: [0] error word, [1] the two amax words,
 *   [2] x codes [R_pad, H/2], [3] their scale codes (MXFP8_SF_MMA), [4] h codes [R_pad, F/2],
 *   [5] their scale codes (MXFP8_SF_MMA), [6] R_pad (not an offset).  out: 7 entries (host).
 */
size_t nvfp4_grouped_mlp_workspace_size(int64_t R, int64_t H, int64_t F, int E);
int nvfp4_grouped_mlp_workspace_layout(int64_t R, int64_t H, int64_t F, int E, uint64_t* out);
int nvfp4_grouped_mlp_fwd(const void* x_sorted, int64_t R, int64_t H, int64_t F, int E, const int32_t* split_sizes,
                          const float* gates, const uint8_t* w1_q, const uint8_t* w1_sf, const float* w1_amax,
                          const uint8_t* w2_q, const uint8_t* w2_sf, const float* w2_amax, float h_amax, void* y,
                          void* workspace, size_t workspace_bytes, void* stream, void* const* stage_events);

/* mxfp8_mma_peak -- measurement aid, with no counterpart on the pages: the rate of the
 * block-scaled tensor-core instruction this library's GEMMs are built on, on the device at hand
 * (the roofline their TFLOP/s are reported against).  Launches one cluster of two CTAs per pair
 * of SMs (as many as fit; their number goes to *clusters, host); each cluster issues `iters`
 * K steps of four tcgen05.mma.cta_group::2 block-scaled MMAs (M = 256, N = 256) back to back on
 * operands resident in shared memory: format 0 = kind::mxf8f6f4 (E4M3, UE8M0 scales, K = 32), so
 * one launch performs clusters * iters * 4 * 2*256*256*32 floating-point operations; format 1 =
 * kind::mxf4nvf4 (E2M1, UE4M3 scales, K = 64): clusters * iters * 4 * 2*256*256*64.  Time it
 * with events on `stream`.  workspace (device, 4-byte aligned, >= 4 bytes) receives an error
 * word (mxfp8_check_device_error reports MXFP8_ERR_DEVICE_TIMEOUT if the final wait ran out).
 * Requirements: 0 <= iters <= 2^24, format 0 or 1. */
int mxfp8_mma_peak(int64_t iters, int format, void* workspace, int* clusters, void* stream);

/* Static description of a status code. */
const char* mxfp8_status_string(int status);

/* ABI version of this header (bumped on any incompatible change). */
int mxfp8_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MXFP8MOE_H */
