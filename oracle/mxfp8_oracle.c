/*
 * mxfp8_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, single-purpose CPU restatement of the MXFP8 expert-MLP forward described on
 * "Efficient MoE training for biology foundation models with Transformer Engine" (NVIDIA news
 * summary), sections "1) Fragmented expert kernels", "2) Model size and activation memory" and
 * "3) Quantization overhead in low-precision training".  Only tests/, the package's smoke check
 * and the bench's CPU-baseline leg may load it.  It shares no code, header, table or constant
 * generator with the CUDA library; neither includes the other.
 *
 * What it computes (all arithmetic in IEEE binary64 unless stated):
 *   - E4M3 decode / encode.  E4M3 is the 8-bit float with 1 sign bit, 4 exponent bits (bias 7)
 *     and 3 mantissa bits, no infinities, S.1111.111 = NaN, largest finite value 448
 *     (the 8-bit element type of MXFP8, section 2).
 *   - MXFP8 block quantization: one power-of-two scale shared by every run of 32 consecutive
 *     values (section 2).  The pages do not give the scale rule; the reading taken is the OCP Microscaling (MX) v1.0 one: shared
 *     exponent s = floor(log2(amax)) - 8 (8 = exponent of E4M3's largest binade), clamped to
 *     the E8M0 range [-127, 127], stored as the biased byte s + 127; each element is
 *     v * 2^-s rounded to the nearest E4M3 value, ties to even mantissa, saturated to +-448.
 *   - GroupedLinear over split_sizes (section 1) -> SwiGLU with the per-token routing weight
 *     applied (section 3 names this ScaledSwiGLU) -> MXFP8 requantization of the intermediate
 *     (section 3: the fused op keeps intermediates out of 16-bit memory) -> GroupedLinear.
 *
 * Every step follows its definition directly: no blocking, fusion or reordering.  Rows are
 * independent, so threads split rows; each row's arithmetic is the same loop nest a reader
 * would write by hand.
 *
 * Build: gcc -O2 -std=c11 -fPIC -shared -pthread -ffp-contract=off mxfp8_oracle.c -lm
 * (-ffp-contract=off keeps aarch64 and x86-64 results identical: no fused multiply-add).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <pthread.h>

#define ORA_OK 0
#define ORA_BAD_ARG 1
#define ORA_SPLIT_MISMATCH 6

/* ------------------------------------------------------------------------------------------ */
/* bf16 and E4M3 codecs                                                                         */
/* ------------------------------------------------------------------------------------------ */

/* bf16 is the upper half of an IEEE binary32; widening to double is exact. */
double ora_bf16_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* E4M3 value of a code: (-1)^S * 2^(E-7) * (1 + M/8) for E >= 1, (-1)^S * 2^-6 * (M/8) for E = 0. */
double ora_e4m3_decode(uint8_t c) {
    int sign = (c >> 7) & 1;
    int e = (c >> 3) & 15;
    int m = c & 7;
    double mag;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        mag = ldexp((double)m / 8.0, -6);
    else
        mag = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -mag : mag;
}

/* Nearest E4M3 code to an exactly known finite value t; ties go to the even mantissa;
 * |t| >= 448 saturates to +-448 (0x7E / 0xFE).  The sign of zero is kept.
 * The grid spacing in the binade [2^e, 2^(e+1)) is 2^(e-3); below 2^-6 the spacing stays 2^-9
 * (subnormals).  t / spacing is exact (power-of-two scaling) and rint() rounds it to nearest,
 * ties to even, under the default rounding mode.  The even integer is the even mantissa. */
uint8_t ora_e4m3_encode(double t) {
    uint8_t sign = signbit(t) ? 0x80 : 0x00;
    double a = fabs(t);
    int ex, e, code_e, code_m;
    double r, v;
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);
    if (a == 0.0) return sign;
    (void)frexp(a, &ex);          /* a = f * 2^ex with f in [0.5, 1): floor(log2 a) = ex - 1 */
    e = ex - 1;
    if (e < -6) e = -6;           /* subnormal range shares the spacing of the lowest binade */
    r = rint(ldexp(a, 3 - e));    /* a in units of 2^(e-3), rounded */
    v = ldexp(r, e - 3);          /* rounded magnitude; can carry into the next binade */
    if (v == 0.0) return sign;
    (void)frexp(v, &ex);
    e = ex - 1;
    if (e < -6) {                 /* subnormal: v = M * 2^-9 */
        code_e = 0;
        code_m = (int)ldexp(v, 9);
    } else {
        code_e = e + 7;
        code_m = (int)(ldexp(v, -e) * 8.0 - 8.0);
    }
    return (uint8_t)(sign | (code_e << 3) | code_m);
}

/* ------------------------------------------------------------------------------------------ */
/* MXFP8 block quantization                                                                     */
/* ------------------------------------------------------------------------------------------ */

/* Shared exponent of a block from its largest magnitude: floor(log2(amax)) - 8, clamped to
 * [-127, 127]; an all-zero block takes the smallest scale (log2(0) = -inf clamps to -127).
 * floor(log2) comes from frexp, which is exact, never from log2(). */
int ora_block_exponent(double amax) {
    int ex, s;
    if (amax == 0.0) return -127;
    (void)frexp(amax, &ex);
    s = (ex - 1) - 8;
    if (s < -127) s = -127;
    if (s > 127) s = 127;
    return s;
}

/* Quantize n (<= 32) values that form one block.  Writes n codes and returns the E8M0 byte. */
uint8_t ora_quantize_block(const double* v, int n, uint8_t* codes) {
    double amax = 0.0;
    int i, s;
    for (i = 0; i < n; ++i)
        if (fabs(v[i]) > amax) amax = fabs(v[i]);
    s = ora_block_exponent(amax);
    for (i = 0; i < n; ++i) codes[i] = ora_e4m3_encode(ldexp(v[i], -s));
    return (uint8_t)(s + 127);
}

/* Value of a code under its block's E8M0 byte. */
double ora_dequant(uint8_t code, uint8_t sf) { return ldexp(ora_e4m3_decode(code), (int)sf - 127); }

/* Encode an array of exact values (test hook for the codec). */
void ora_e4m3_encode_array(const double* t, int64_t n, uint8_t* out) {
    int64_t i;
    for (i = 0; i < n; ++i) out[i] = ora_e4m3_encode(t[i]);
}

void ora_e4m3_decode_array(const uint8_t* c, int64_t n, double* out) {
    int64_t i;
    for (i = 0; i < n; ++i) out[i] = ora_e4m3_decode(c[i]);
}

/* ---- threading helper: split [0, n) into contiguous chunks --------------------------------- */
typedef void (*ora_range_fn)(void* ctx, int64_t begin, int64_t end);
typedef struct { ora_range_fn fn; void* ctx; int64_t begin, end; } ora_job;

static void* ora_job_main(void* p) {
    ora_job* j = (ora_job*)p;
    j->fn(j->ctx, j->begin, j->end);
    return NULL;
}

void ora_parallel(ora_range_fn fn, void* ctx, int64_t n, int nthreads) {
    pthread_t th[256];
    ora_job jobs[256];
    int t;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((int64_t)nthreads > n) nthreads = (int)(n > 0 ? n : 1);
    for (t = 0; t < nthreads; ++t) {
        jobs[t].fn = fn;
        jobs[t].ctx = ctx;
        jobs[t].begin = n * t / nthreads;
        jobs[t].end = n * (t + 1) / nthreads;
    }
    for (t = 1; t < nthreads; ++t)
        if (pthread_create(&th[t], NULL, ora_job_main, &jobs[t]) != 0) jobs[t].fn = NULL;
    fn(ctx, jobs[0].begin, jobs[0].end);
    for (t = 1; t < nthreads; ++t) {
        if (jobs[t].fn) pthread_join(th[t], NULL);
        else fn(ctx, jobs[t].begin, jobs[t].end);   /* thread creation failed: do it here */
    }
}

/* ---- row-wise: blocks of 32 along K of each row of a row-major [M, K] bf16 matrix ---------- */
typedef struct { const uint16_t* x; int64_t M, K; uint8_t *q, *sf; } ora_rowq_ctx;

static void ora_rowq_range(void* p, int64_t r0, int64_t r1) {
    ora_rowq_ctx* c = (ora_rowq_ctx*)p;
    double v[32];
    int64_t r, b, i;
    for (r = r0; r < r1; ++r)
        for (b = 0; b < c->K / 32; ++b) {
            for (i = 0; i < 32; ++i) v[i] = ora_bf16_to_double(c->x[r * c->K + b * 32 + i]);
            c->sf[r * (c->K / 32) + b] = ora_quantize_block(v, 32, c->q + r * c->K + b * 32);
        }
}

/* q: [M, K] codes; sf: [M, K/32] E8M0 bytes, row-major ("compact"). K must be a multiple of 32. */
int ora_quantize_rowwise(const uint16_t* x, int64_t M, int64_t K, uint8_t* q, uint8_t* sf, int nthreads) {
    ora_rowq_ctx c;
    if (!x || !q || !sf || M < 0 || K < 0 || K % 32) return ORA_BAD_ARG;
    c.x = x; c.M = M; c.K = K; c.q = q; c.sf = sf;
    ora_parallel(ora_rowq_range, &c, M, nthreads);
    return ORA_OK;
}

/* ---- column-wise: blocks of 32 consecutive rows down each column ----------------------------
 * Codes keep the input's [M, K] layout; sf is [ceil(M/32), K] row-major.  A last block with
 * fewer than 32 rows takes its amax over the rows present. */
typedef struct { const uint16_t* x; int64_t M, K; uint8_t *q, *sf; } ora_colq_ctx;

static void ora_colq_range(void* p, int64_t c0, int64_t c1) {
    ora_colq_ctx* c = (ora_colq_ctx*)p;
    double v[32];
    uint8_t codes[32];
    int64_t col, rb, i, n;
    for (col = c0; col < c1; ++col)
        for (rb = 0; rb < (c->M + 31) / 32; ++rb) {
            n = c->M - rb * 32;
            if (n > 32) n = 32;
            for (i = 0; i < n; ++i) v[i] = ora_bf16_to_double(c->x[(rb * 32 + i) * c->K + col]);
            c->sf[rb * c->K + col] = ora_quantize_block(v, (int)n, codes);
            for (i = 0; i < n; ++i) c->q[(rb * 32 + i) * c->K + col] = codes[i];
        }
}

int ora_quantize_colwise(const uint16_t* x, int64_t M, int64_t K, uint8_t* q, uint8_t* sf, int nthreads) {
    ora_colq_ctx c;
    if (!x || !q || !sf || M < 0 || K < 0) return ORA_BAD_ARG;
    c.x = x; c.M = M; c.K = K; c.q = q; c.sf = sf;
    ora_parallel(ora_colq_range, &c, K, nthreads);
    return ORA_OK;
}

/* ------------------------------------------------------------------------------------------ */
/* Grouped expert MLP forward                                                                   */
/* ------------------------------------------------------------------------------------------ */
/*
 * Inputs:
 *   x      [R, H] bf16, rows grouped by expert: expert e owns rows [off_e, off_e + split[e])
 *          with off_e = split[0] + ... + split[e-1] (GroupedLinear's split_sizes, section 1).
 *   gates  [R] float routing weights, or NULL for all ones.
 *   w1q/w1sf: expert weights W1 = [E, 2F, H] as codes + compact row-wise E8M0 bytes
 *          ([E*2F, H/32]); rows [0, F) of each expert are the SwiGLU gate projection, rows
 *          [F, 2F) the up projection (reading: the pages do not order the halves).
 *   w2q/w2sf: W2 = [E, H, F] codes + compact row-wise E8M0 bytes ([E*H, F/32]).
 * For each requested row r (expert e):
 *   a   = dequant(rowwise MXFP8 of x_r)                                 (length H)
 *   g_j = sum_k a_k * W1[e, j, k],   u_j = sum_k a_k * W1[e, F+j, k]      (GroupedLinear 1)
 *   h_j = gate_r * (g_j / (1 + exp(-g_j))) * u_j                         (ScaledSwiGLU)
 *   hq  = rowwise MXFP8 of h (blocks of 32 along F)                      (requantization)
 *   y_i = sum_j dequant(hq)_j * W2[e, i, j]                              (GroupedLinear 2)
 * Outputs (for the nrows rows listed in `rows`): y [nrows, H] in double, and optionally the
 * intermediate codes hq [nrows, F] and their E8M0 bytes hsf [nrows, F/32].
 */
typedef struct {
    const uint16_t* x; int64_t R, H, F; int E;
    const int64_t* off; const float* gates;
    double code_val[256];   /* ora_e4m3_decode(c) for every code c */
    double scale_val[256];  /* 2^(b-127) for every E8M0 byte b (255 is never produced) */
    const uint8_t *w1q, *w1sf, *w2q, *w2sf;
    const int64_t* rows; double* y; uint8_t *hq, *hsf;
} ora_mlp_ctx;

static void ora_mlp_range(void* p, int64_t i0, int64_t i1) {
    ora_mlp_ctx* c = (ora_mlp_ctx*)p;
    const int64_t H = c->H, F = c->F;
    double* xv = (double*)malloc(sizeof(double) * (size_t)H);
    double* a = (double*)malloc(sizeof(double) * (size_t)H);
    double* h = (double*)malloc(sizeof(double) * (size_t)F);
    double* hd = (double*)malloc(sizeof(double) * (size_t)F);
    uint8_t* xq = (uint8_t*)malloc((size_t)H);
    uint8_t* hq = (uint8_t*)malloc((size_t)F);
    uint8_t* xsf = (uint8_t*)malloc((size_t)(H / 32));
    uint8_t* hsf = (uint8_t*)malloc((size_t)(F / 32));
    int64_t i, k, j, b;
    for (i = i0; i < i1; ++i) {
        int64_t r = c->rows[i];
        int e = 0;
        double gate;
        while (!(r >= c->off[e] && r < c->off[e + 1])) ++e;  /* expert that owns row r */
        gate = c->gates ? (double)c->gates[r] : 1.0;
        /* quantize the activation row, blocks of 32 along H */
        for (k = 0; k < H; ++k) xv[k] = ora_bf16_to_double(c->x[r * H + k]);
        for (b = 0; b < H / 32; ++b) xsf[b] = ora_quantize_block(xv + b * 32, 32, xq + b * 32);
        for (k = 0; k < H; ++k) a[k] = ora_dequant(xq[k], xsf[k / 32]);
        /* GroupedLinear 1 and ScaledSwiGLU */
        for (j = 0; j < F; ++j) {
            const int64_t rg = ((int64_t)e * 2 * F + j), ru = ((int64_t)e * 2 * F + F + j);
            double g = 0.0, u = 0.0;
            for (k = 0; k < H; ++k) {
                g += a[k] * (c->code_val[c->w1q[rg * H + k]] * c->scale_val[c->w1sf[rg * (H / 32) + k / 32]]);
                u += a[k] * (c->code_val[c->w1q[ru * H + k]] * c->scale_val[c->w1sf[ru * (H / 32) + k / 32]]);
            }
            h[j] = gate * (g / (1.0 + exp(-g))) * u;
        }
        /* requantize the intermediate, blocks of 32 along F */
        for (b = 0; b < F / 32; ++b) hsf[b] = ora_quantize_block(h + b * 32, 32, hq + b * 32);
        for (j = 0; j < F; ++j) hd[j] = ora_dequant(hq[j], hsf[j / 32]);
        /* GroupedLinear 2 */
        for (k = 0; k < H; ++k) {
            const int64_t rw = (int64_t)e * H + k;
            double acc = 0.0;
            for (j = 0; j < F; ++j)
                acc += hd[j] * (c->code_val[c->w2q[rw * F + j]] * c->scale_val[c->w2sf[rw * (F / 32) + j / 32]]);
            c->y[i * H + k] = acc;
        }
        if (c->hq) memcpy(c->hq + i * F, hq, (size_t)F);
        if (c->hsf) memcpy(c->hsf + i * (F / 32), hsf, (size_t)(F / 32));
    }
    free(xv); free(a); free(h); free(hd); free(xq); free(hq); free(xsf); free(hsf);
}

int ora_grouped_mlp_rows(const uint16_t* x, int64_t R, int64_t H, int64_t F, int E,
                         const int32_t* split, const float* gates,
                         const uint8_t* w1q, const uint8_t* w1sf, const uint8_t* w2q, const uint8_t* w2sf,
                         const int64_t* rows, int64_t nrows, double* y, uint8_t* hq, uint8_t* hsf,
                         int nthreads) {
    ora_mlp_ctx c;
    int64_t* off;
    int64_t total = 0, i;
    int e;
    if (!x || !split || !w1q || !w1sf || !w2q || !w2sf || !y || (nrows > 0 && !rows)) return ORA_BAD_ARG;
    if (R < 0 || H <= 0 || F <= 0 || E <= 0 || H % 32 || F % 32 || nrows < 0) return ORA_BAD_ARG;
    off = (int64_t*)malloc(sizeof(int64_t) * (size_t)(E + 1));
    off[0] = 0;
    for (e = 0; e < E; ++e) {
        if (split[e] < 0) { free(off); return ORA_BAD_ARG; }
        total += split[e];
        off[e + 1] = total;
    }
    if (total != R) { free(off); return ORA_SPLIT_MISMATCH; }
    for (i = 0; i < nrows; ++i)
        if (rows[i] < 0 || rows[i] >= R) { free(off); return ORA_BAD_ARG; }
    c.x = x; c.R = R; c.H = H; c.F = F; c.E = E; c.off = off; c.gates = gates;
    c.w1q = w1q; c.w1sf = w1sf; c.w2q = w2q; c.w2sf = w2sf;
    c.rows = rows; c.y = y; c.hq = hq; c.hsf = hsf;
    for (i = 0; i < 256; ++i) {
        c.code_val[i] = ora_e4m3_decode((uint8_t)i);
        c.scale_val[i] = ldexp(1.0, (int)i - 127);   /* exact: a power of two, no product rounds */
    }
    ora_parallel(ora_mlp_range, &c, nrows, nthreads);
    free(off);
    return ORA_OK;
}

/* ------------------------------------------------------------------------------------------ */
/* Dispatch and combine around the grouped MLP                                                  */
/* ------------------------------------------------------------------------------------------ */
/* Page section "Dense vs. MoE scaling": each token uses k of the E experts; item 1: GroupedLinear
 * runs on the tokens gathered per expert.  Dispatch = stable sort of the (token, slot) pairs by
 * expert id (ties keep token-then-slot order), written out as a counting sort:
 *   split[e]          number of pairs choosing expert e
 *   row_of_slot[t,j]  position of pair (t, j) in the sorted order
 *   token_of_row[r]   token of sorted row r;  gates_sorted[r] its routing weight. */
int ora_moe_permute(const int32_t* experts, const float* gates, int64_t T, int k, int E, int32_t* split,
                    int32_t* row_of_slot, int32_t* token_of_row, float* gates_sorted) {
    int64_t i, n = T * (int64_t)k;
    int64_t* next;
    int e;
    if (T < 0 || k < 1 || E < 1 || !split || (n > 0 && (!experts || !row_of_slot || !token_of_row)))
        return ORA_BAD_ARG;
    for (i = 0; i < n; ++i)
        if (experts[i] < 0 || experts[i] >= E) return ORA_BAD_ARG;
    for (e = 0; e < E; ++e) split[e] = 0;
    for (i = 0; i < n; ++i) split[experts[i]] += 1;
    next = (int64_t*)malloc(sizeof(int64_t) * (size_t)E);
    next[0] = 0;
    for (e = 1; e < E; ++e) next[e] = next[e - 1] + split[e - 1];
    for (i = 0; i < n; ++i) {                 /* pairs visited in (token, slot) order */
        const int64_t r = next[experts[i]]++;
        row_of_slot[i] = (int32_t)r;
        token_of_row[r] = (int32_t)(i / k);
        if (gates && gates_sorted) gates_sorted[r] = gates[i];
    }
    free(next);
    return ORA_OK;
}

/* out[t, :] = sum over j of y[row_of_slot[t, j], :]   (binary64) */
int ora_moe_combine(const double* y, const int32_t* row_of_slot, int64_t T, int k, int64_t H, double* out) {
    int64_t t, c;
    int j;
    if (T < 0 || k < 1 || H < 1 || (T > 0 && (!y || !row_of_slot || !out))) return ORA_BAD_ARG;
    for (t = 0; t < T; ++t)
        for (c = 0; c < H; ++c) {
            double acc = 0.0;
            for (j = 0; j < k; ++j) acc += y[(int64_t)row_of_slot[t * k + j] * H + c];
            out[t * H + c] = acc;
        }
    return ORA_OK;
}

/* ------------------------------------------------------------------------------------------ */
/* Backward of the grouped MLP                                                                  */
/* ------------------------------------------------------------------------------------------ */
/* Section 3 names a fused backward op for the same GroupedLinear -> ScaledSwiGLU ->
 * GroupedLinear chain without spelling it out.  The reading taken is the usual one for MXFP8
 * training:
 *   - gradients pass straight through every quantization (the quantized tensor's gradient is
 *     used as the gradient of the tensor it came from);
 *   - every backward GEMM takes MXFP8 operands with blocks of 32 along that GEMM's contraction
 *     axis: along H for dh = dy W2, along 2F for dx = dGU W1, along the expert's rows for the
 *     weight gradients (32-row blocks counted from the expert's first row, the last one padded
 *     with zeros);
 *   - the two tensors the backward hands from one GEMM to the next, dGU = [dG | dU] and the
 *     activation h for dW2, are bf16 tensors, so they are rounded to bf16 before they are
 *     quantized (x and dy are bf16 inputs already);
 *   - the forward saves its pre-activations g, u for the backward as bf16, so the backward's
 *     SwiGLU derivative starts from bf16(g), bf16(u).
 * With a = dequant(Q_row(x_r)), g_j, u_j, h_j as in the forward, and
 *   s_j = g_j / (1 + exp(-g_j))                       (silu)
 *   s'_j = sigma_j * (1 + g_j * (1 - sigma_j)),  sigma_j = 1 / (1 + exp(-g_j))
 * the backward of row r (expert e) is
 *   dh_j    = sum_k dequant(Q_row(dy_r))_k * W2t[e, j, k]       (W2 quantized along H)
 *   dG_j    = dh_j * gate_r * u_j * s'_j,   dU_j = dh_j * gate_r * s_j
 *   dgate_r = sum_j dh_j * s_j * u_j
 *   dx_r,k  = sum_j dequant(Q_row(bf16(dGU_r)))_j * W1t[e, k, j] (W1 quantized along 2F)
 * and the weight gradients of expert e are
 *   dW2[e, i, j] = sum_r dequant(Q_col(dy))_{r,i} * dequant(Q_col(bf16(h)))_{r,j}
 *   dW1[e, j, k] = sum_r dequant(Q_col(bf16(dGU)))_{r,j} * dequant(Q_col(x))_{r,k}
 * W2t holds, for each expert, W2[e]^T = [F, H] quantized row-wise (i.e. W2 quantized along H);
 * W1t holds W1[e]^T = [H, 2F] quantized row-wise (W1 quantized along 2F). */

/* Nearest bf16 value of a finite double, ties to even (binary32 exponent range; bf16 subnormals
 * keep the fixed spacing 2^-133; overflow is not reached by the values this file produces). */
double ora_round_bf16(double v) {
    int ex, e;
    double a = fabs(v), q;
    if (a == 0.0) return v;
    (void)frexp(a, &ex);
    e = ex - 1;                     /* a in [2^e, 2^(e+1)) */
    if (e < -126) e = -126;         /* subnormal range: spacing 2^-133 */
    q = ldexp(rint(ldexp(a, 7 - e)), e - 7);
    return v < 0 ? -q : q;
}

uint16_t ora_double_to_bf16_bits(double v) {
    float f = (float)ora_round_bf16(v);   /* exact: the value has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

typedef struct {
    const uint16_t *x, *dy; int64_t R, H, F; int E;
    const int64_t* off; const float* gates;
    double code_val[256], scale_val[256];
    const uint8_t *w1q, *w1sf, *w2tq, *w2tsf, *w1tq, *w1tsf;
    const int64_t* rows; double *dx, *dgate; uint16_t *dgu_out, *h_out, *gu_out;
    /* entries of the weight gradients */
    int which; const int64_t* ent; double* dw;
    /* 1: quantize and round as documented; 0: every quantization and bf16 rounding of x, dy and
     * the intermediates is the identity (a test hook that exposes the calculus alone) */
    int quant;
} ora_bwd_ctx;

static int ora_expert_of(const ora_bwd_ctx* c, int64_t r) {
    int e = 0;
    while (!(r >= c->off[e] && r < c->off[e + 1])) ++e;
    return e;
}

static double ora_wval(const ora_bwd_ctx* c, const uint8_t* q, const uint8_t* sf, int64_t row, int64_t K, int64_t k) {
    return c->code_val[q[row * K + k]] * c->scale_val[sf[row * (K / 32) + k / 32]];
}

/* dequant(Q_row(v)) for a length-n vector (n % 32 == 0), in place. */
static void ora_qdq_row(double* v, int64_t n) {
    uint8_t codes[32];
    int64_t b;
    int i;
    for (b = 0; b < n / 32; ++b) {
        uint8_t sf = ora_quantize_block(v + b * 32, 32, codes);
        for (i = 0; i < 32; ++i) v[b * 32 + i] = ora_dequant(codes[i], sf);
    }
}

/* dequant(Q_col(v)) for the values of one column over an expert's n rows: blocks of 32 from the
 * first row, the last block shorter (its zero padding does not change the block's amax). */
static void ora_qdq_col(double* v, int64_t n) {
    uint8_t codes[32];
    int64_t b;
    int i;
    for (b = 0; b < n; b += 32) {
        int len = (int)((n - b) < 32 ? (n - b) : 32);
        uint8_t sf = ora_quantize_block(v + b, len, codes);
        for (i = 0; i < len; ++i) v[b + i] = ora_dequant(codes[i], sf);
    }
}

static double ora_bwd_round(const ora_bwd_ctx* c, double v) { return c->quant ? ora_round_bf16(v) : v; }

/* Saved forward pre-activations g_j, u_j of a row of expert e from its dequantized activation a
 * (bf16-rounded as the forward saves them). */
static void ora_row_gu(const ora_bwd_ctx* c, int e, const double* a, int64_t j, double* g, double* u) {
    const int64_t H = c->H, F = c->F;
    const int64_t rg = (int64_t)e * 2 * F + j, ru = (int64_t)e * 2 * F + F + j;
    double gg = 0.0, uu = 0.0;
    int64_t k;
    for (k = 0; k < H; ++k) {
        gg += a[k] * ora_wval(c, c->w1q, c->w1sf, rg, H, k);
        uu += a[k] * ora_wval(c, c->w1q, c->w1sf, ru, H, k);
    }
    *g = ora_bwd_round(c, gg);
    *u = ora_bwd_round(c, uu);
}

static void ora_row_a(const ora_bwd_ctx* c, int64_t r, double* a) {
    int64_t k;
    for (k = 0; k < c->H; ++k) a[k] = ora_bf16_to_double(c->x[r * c->H + k]);
    if (c->quant) ora_qdq_row(a, c->H);
}

static void ora_row_dyq(const ora_bwd_ctx* c, int64_t r, double* d) {
    int64_t k;
    for (k = 0; k < c->H; ++k) d[k] = ora_bf16_to_double(c->dy[r * c->H + k]);
    if (c->quant) ora_qdq_row(d, c->H);
}

static double ora_row_dh(const ora_bwd_ctx* c, int e, const double* dyq, int64_t j) {
    double acc = 0.0;
    int64_t k;
    for (k = 0; k < c->H; ++k) acc += dyq[k] * ora_wval(c, c->w2tq, c->w2tsf, (int64_t)e * c->F + j, c->H, k);
    return acc;
}

static void ora_bwd_rows_range(void* p, int64_t i0, int64_t i1) {
    ora_bwd_ctx* c = (ora_bwd_ctx*)p;
    const int64_t H = c->H, F = c->F;
    double* a = (double*)malloc(sizeof(double) * (size_t)H);
    double* dyq = (double*)malloc(sizeof(double) * (size_t)H);
    double* dgu = (double*)malloc(sizeof(double) * (size_t)(2 * F));
    int64_t i, j, k;
    for (i = i0; i < i1; ++i) {
        const int64_t r = c->rows[i];
        const int e = ora_expert_of(c, r);
        const double gate = c->gates ? (double)c->gates[r] : 1.0;
        double dgate = 0.0;
        ora_row_a(c, r, a);
        ora_row_dyq(c, r, dyq);
        for (j = 0; j < F; ++j) {
            double g, u, dh, sig, sl, dsl;
            ora_row_gu(c, e, a, j, &g, &u);
            if (c->gu_out) {
                c->gu_out[i * 2 * F + j] = ora_double_to_bf16_bits(g);
                c->gu_out[i * 2 * F + F + j] = ora_double_to_bf16_bits(u);
            }
            dh = ora_row_dh(c, e, dyq, j);
            sig = 1.0 / (1.0 + exp(-g));
            sl = g * sig;
            dsl = sig * (1.0 + g * (1.0 - sig));
            dgu[j] = dh * gate * u * dsl;
            dgu[F + j] = dh * gate * sl;
            dgate += dh * sl * u;
            if (c->h_out) c->h_out[i * F + j] = ora_double_to_bf16_bits(gate * sl * u);
        }
        for (j = 0; j < 2 * F; ++j) {
            dgu[j] = ora_bwd_round(c, dgu[j]);
            if (c->dgu_out) c->dgu_out[i * 2 * F + j] = ora_double_to_bf16_bits(dgu[j]);
        }
        if (c->quant) ora_qdq_row(dgu, 2 * F);
        for (k = 0; k < H; ++k) {
            double acc = 0.0;
            for (j = 0; j < 2 * F; ++j) acc += dgu[j] * ora_wval(c, c->w1tq, c->w1tsf, (int64_t)e * H + k, 2 * F, j);
            c->dx[i * H + k] = acc;
        }
        c->dgate[i] = dgate;
    }
    free(a); free(dyq); free(dgu);
}

/* One weight-gradient entry per index: ent[3i..3i+2] = (e, row, col) of dW2 [E, H, F]
 * (which == 2) or of dW1 [E, 2F, H] (which == 1). */
static void ora_bwd_dw_range(void* p, int64_t i0, int64_t i1) {
    ora_bwd_ctx* c = (ora_bwd_ctx*)p;
    const int64_t H = c->H, F = c->F;
    double* a = (double*)malloc(sizeof(double) * (size_t)H);
    double* dyq = (double*)malloc(sizeof(double) * (size_t)H);
    int64_t i, r;
    for (i = i0; i < i1; ++i) {
        const int e = (int)c->ent[3 * i];
        const int64_t ri = c->ent[3 * i + 1], ci = c->ent[3 * i + 2];
        const int64_t r0 = c->off[e], n = c->off[e + 1] - c->off[e];
        double* va = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
        double* vb = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
        double acc = 0.0;
        for (r = 0; r < n; ++r) {
            const int64_t row = r0 + r;
            const double gate = c->gates ? (double)c->gates[row] : 1.0;
            double g, u, sig, sl;
            ora_row_a(c, row, a);
            if (c->which == 2) {   /* dW2[e, ri, ci]: dy column ri, h column ci */
                va[r] = ora_bf16_to_double(c->dy[row * H + ri]);
                ora_row_gu(c, e, a, ci, &g, &u);
                sig = 1.0 / (1.0 + exp(-g));
                vb[r] = ora_bwd_round(c, gate * (g * sig) * u);
            } else {               /* dW1[e, ri, ci]: dGU column ri, x column ci */
                const int64_t jj = ri < F ? ri : ri - F;
                double dh, dsl;
                ora_row_dyq(c, row, dyq);
                ora_row_gu(c, e, a, jj, &g, &u);
                dh = ora_row_dh(c, e, dyq, jj);
                sig = 1.0 / (1.0 + exp(-g));
                sl = g * sig;
                dsl = sig * (1.0 + g * (1.0 - sig));
                va[r] = ora_bwd_round(c, ri < F ? dh * gate * u * dsl : dh * gate * sl);
                vb[r] = ora_bf16_to_double(c->x[row * H + ci]);
            }
        }
        if (c->quant) {
            ora_qdq_col(va, n);
            ora_qdq_col(vb, n);
        }
        for (r = 0; r < n; ++r) acc += va[r] * vb[r];
        c->dw[i] = acc;
        free(va); free(vb);
    }
    free(a); free(dyq);
}

static int ora_bwd_setup(ora_bwd_ctx* c, const uint16_t* x, int64_t R, int64_t H, int64_t F, int E,
                         const int32_t* split, const float* gates, const uint8_t* w1q, const uint8_t* w1sf,
                         const uint8_t* w2tq, const uint8_t* w2tsf, const uint16_t* dy) {
    int64_t total = 0, i;
    int e;
    if (!x || !split || !w1q || !w1sf || !w2tq || !w2tsf || !dy) return ORA_BAD_ARG;
    if (R < 0 || H <= 0 || F <= 0 || E <= 0 || H % 32 || F % 32) return ORA_BAD_ARG;
    memset(c, 0, sizeof *c);
    c->off = (int64_t*)malloc(sizeof(int64_t) * (size_t)(E + 1));
    ((int64_t*)c->off)[0] = 0;
    for (e = 0; e < E; ++e) {
        if (split[e] < 0) { free((void*)c->off); return ORA_BAD_ARG; }
        total += split[e];
        ((int64_t*)c->off)[e + 1] = total;
    }
    if (total != R) { free((void*)c->off); return ORA_SPLIT_MISMATCH; }
    c->x = x; c->dy = dy; c->R = R; c->H = H; c->F = F; c->E = E; c->gates = gates;
    c->w1q = w1q; c->w1sf = w1sf; c->w2tq = w2tq; c->w2tsf = w2tsf;
    for (i = 0; i < 256; ++i) {
        c->code_val[i] = ora_e4m3_decode((uint8_t)i);
        c->scale_val[i] = ldexp(1.0, (int)i - 127);
    }
    return ORA_OK;
}

int ora_grouped_mlp_bwd_rows(const uint16_t* x, int64_t R, int64_t H, int64_t F, int E, const int32_t* split,
                             const float* gates, const uint8_t* w1q, const uint8_t* w1sf, const uint8_t* w2tq,
                             const uint8_t* w2tsf, const uint8_t* w1tq, const uint8_t* w1tsf, const uint16_t* dy,
                             const int64_t* rows, int64_t nrows, double* dx, double* dgate, uint16_t* dgu,
                             uint16_t* h, uint16_t* gu, int quant, int nthreads) {
    ora_bwd_ctx c;
    int64_t i;
    int rc = ora_bwd_setup(&c, x, R, H, F, E, split, gates, w1q, w1sf, w2tq, w2tsf, dy);
    if (rc != ORA_OK) return rc;
    if (!w1tq || !w1tsf || !dx || !dgate || nrows < 0 || (nrows > 0 && !rows)) {
        free((void*)c.off);
        return ORA_BAD_ARG;
    }
    for (i = 0; i < nrows; ++i)
        if (rows[i] < 0 || rows[i] >= R) { free((void*)c.off); return ORA_BAD_ARG; }
    c.w1tq = w1tq; c.w1tsf = w1tsf; c.rows = rows; c.dx = dx; c.dgate = dgate; c.dgu_out = dgu; c.h_out = h;
    c.gu_out = gu;
    c.quant = quant != 0;
    ora_parallel(ora_bwd_rows_range, &c, nrows, nthreads);
    free((void*)c.off);
    return ORA_OK;
}

int ora_grouped_mlp_bwd_dw(const uint16_t* x, int64_t R, int64_t H, int64_t F, int E, const int32_t* split,
                           const float* gates, const uint8_t* w1q, const uint8_t* w1sf, const uint8_t* w2tq,
                           const uint8_t* w2tsf, const uint16_t* dy, int which, const int64_t* ent, int64_t n,
                           double* dw, int quant, int nthreads) {
    ora_bwd_ctx c;
    int64_t i;
    int rc = ora_bwd_setup(&c, x, R, H, F, E, split, gates, w1q, w1sf, w2tq, w2tsf, dy);
    if (rc != ORA_OK) return rc;
    if ((which != 1 && which != 2) || !dw || n < 0 || (n > 0 && !ent)) { free((void*)c.off); return ORA_BAD_ARG; }
    for (i = 0; i < n; ++i) {
        const int64_t e = ent[3 * i], ri = ent[3 * i + 1], ci = ent[3 * i + 2];
        const int64_t nr = which == 2 ? H : 2 * F, nc = which == 2 ? F : H;
        if (e < 0 || e >= E || ri < 0 || ri >= nr || ci < 0 || ci >= nc) { free((void*)c.off); return ORA_BAD_ARG; }
    }
    c.which = which; c.ent = ent; c.dw = dw; c.quant = quant != 0;
    ora_parallel(ora_bwd_dw_range, &c, n, nthreads);
    free((void*)c.off);
    return ORA_OK;
}

int ora_abi_version(void) { return 1; }
