/*
 * nvfp4_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * CPU restatement of the NVFP4 variant of the expert-MLP forward.  The Llama 3 recipe page
 * ("TransformerEngine-accelerated Llama 3 training with native PyTorch training loop") lists
 * NVFP4 beside MXFP8 as a quantized-training recipe (feature table; section "Quantized Training
 * (FP8 / MXFP8 / NVFP4)") but defines nothing of the format.  The reading taken is NVIDIA's
 * published NVFP4 definition:
 *   - elements are E2M1 (FP4): 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit, no
 *     infinity or NaN; magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6;
 *   - every run of 16 consecutive values shares one scale stored as an E4M3 value;
 *   - a second, per-tensor fp32 scale maps the tensor's largest magnitude A onto the largest
 *     value the two levels together reach (E4M3 max 448 times E2M1 max 6):
 *       s_enc = 448 * 6 / A   (1 when A = 0, at most FLT_MAX).
 * Quantizing a block v[0..15] under s_enc, every step in IEEE binary32 with round to nearest
 * even (the precision the GPU kernels decide in; the pages fix none):
 *       amax = max |v_i|
 *       S    = E4M3(fl32(fl32(amax / 6) * s_enc))      RNE, saturated to 448 (the block scale)
 *       r    = 0 if S = 0, else min(fl32(s_enc / S), FLT_MAX)
 *       q_i  = E2M1(fl32(v_i * r))                      RNE (ties to even mantissa), saturated to 6
 * and the value the pair (q_i, S) stands for is q_i * S / s_enc.
 * The NVFP4 expert MLP is the MXFP8 one (mxfp8_oracle.c) with NVFP4 operands: x quantized
 * row-wise along H under its own s_enc; W1 [E*2F, H] and W2 [E*H, F] each quantized row-wise as
 * one tensor with one s_enc; the intermediate h, computed in binary64, enters the encoder as
 * binary32 and is quantized row-wise along F under the encode scale derived the same way from
 * a caller-supplied magnitude h_amax (its largest value cannot be known before the first GEMM
 * has run; values beyond h_amax saturate).  Sums are binary64.
 *
 * Codes are kept one per byte here (4-bit value in the low nibble, sign in bit 3); the packing
 * of two codes per byte is a layout matter left to the callers.
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORA_OK 0
#define ORA_BAD_ARG 1
#define ORA_SPLIT_MISMATCH 6

/* from mxfp8_oracle.c (same library) */
double ora_bf16_to_double(uint16_t b);
double ora_e4m3_decode(uint8_t c);
uint8_t ora_e4m3_encode(double t);
typedef void (*ora_range_fn)(void* ctx, int64_t begin, int64_t end);
void ora_parallel(ora_range_fn fn, void* ctx, int64_t n, int nthreads);

/* E2M1 value of a 4-bit code: (-1)^S * 2^(E-1) * (1 + M/2) for E >= 1, (-1)^S * M/2 for E = 0. */
double ora_e2m1_decode(uint8_t c) {
    int sign = (c >> 3) & 1, e = (c >> 1) & 3, m = c & 1;
    double mag = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return sign ? -mag : mag;
}

/* Nearest E2M1 code to an exact finite value; ties go to the even mantissa; |t| >= 6 saturates
 * to 6.  Grid spacing: 0.5 below 2 (the subnormal step and the binade [1, 2)), 1 in [2, 4),
 * 2 in [4, 8).  t / spacing is exact and rint() rounds it to nearest, ties to even; with these
 * spacings an even multiple is an even mantissa. */
uint8_t ora_e2m1_encode(double t) {
    uint8_t sign = signbit(t) ? 0x8 : 0x0;
    double a = fabs(t), step, v;
    int e, m;
    if (a >= 6.0) return (uint8_t)(sign | 0x7);
    step = a < 2.0 ? 0.5 : (a < 4.0 ? 1.0 : 2.0);
    v = rint(a / step) * step;            /* may carry into the next binade (1.75 -> 2) */
    if (v == 0.0) return sign;
    if (v < 1.0) return (uint8_t)(sign | 0x1);   /* 0.5: subnormal */
    e = v < 2.0 ? 1 : (v < 4.0 ? 2 : 3);
    m = (int)(2.0 * (v / ldexp(1.0, e - 1) - 1.0));   /* v = 2^(e-1) * (1 + m/2) */
    return (uint8_t)(sign | (e << 1) | m);
}

/* Per-tensor encode scale from the tensor's largest magnitude (binary32). */
float ora_nvfp4_encode_scale(float amax) {
    volatile float q;
    if (amax == 0.0f) return 1.0f;
    q = 2688.0f / amax;
    return q > FLT_MAX ? FLT_MAX : q;
}

/* Quantize n (<= 16) binary32 values forming one block under s_enc: n codes, returns the E4M3
 * code of the block scale.  Every product and quotient is rounded to binary32 on its own
 * (volatile stores keep the compiler from widening or fusing them). */
uint8_t ora_nvfp4_quantize_block(const float* v, int n, float s_enc, uint8_t* codes) {
    float amax = 0.0f;
    volatile float sfv, t, r;
    double S;
    uint8_t sf;
    int i;
    for (i = 0; i < n; ++i)
        if (fabsf(v[i]) > amax) amax = fabsf(v[i]);
    sfv = amax / 6.0f;
    t = sfv * s_enc;
    sf = ora_e4m3_encode((double)t);
    S = ora_e4m3_decode(sf);
    if (S == 0.0) {
        r = 0.0f;
    } else {
        r = s_enc / (float)S;
        if (r > FLT_MAX) r = FLT_MAX;
    }
    for (i = 0; i < n; ++i) {
        volatile float x = v[i] * r;
        codes[i] = ora_e2m1_encode((double)x);
    }
    return sf;
}

double ora_nvfp4_dequant(uint8_t code, uint8_t sf, float s_enc) {
    return ora_e2m1_decode(code) * ora_e4m3_decode(sf) / (double)s_enc;
}

void ora_e2m1_encode_array(const double* t, int64_t n, uint8_t* out) {
    int64_t i;
    for (i = 0; i < n; ++i) out[i] = ora_e2m1_encode(t[i]);
}

/* Largest magnitude of a bf16 tensor (as binary32: exact). */
float ora_bf16_amax(const uint16_t* x, int64_t n) {
    float a = 0.0f;
    int64_t i;
    for (i = 0; i < n; ++i) {
        float v = (float)fabs(ora_bf16_to_double(x[i]));
        if (v > a) a = v;
    }
    return a;
}

/* ---- row-wise NVFP4 of a bf16 [M, K] matrix (K % 16 == 0) under the encode scale of its own
 * largest magnitude: codes [M, K] (one per byte), E4M3 scale codes [M, K/16], *s_enc_out. */
typedef struct { const uint16_t* x; int64_t M, K; float s_enc; uint8_t *q, *sf; } ora_nv_rowq_ctx;

static void ora_nv_rowq_range(void* p, int64_t r0, int64_t r1) {
    ora_nv_rowq_ctx* c = (ora_nv_rowq_ctx*)p;
    float v[16];
    int64_t r, b;
    int i;
    for (r = r0; r < r1; ++r)
        for (b = 0; b < c->K / 16; ++b) {
            for (i = 0; i < 16; ++i) v[i] = (float)ora_bf16_to_double(c->x[r * c->K + b * 16 + i]);
            c->sf[r * (c->K / 16) + b] = ora_nvfp4_quantize_block(v, 16, c->s_enc, c->q + r * c->K + b * 16);
        }
}

int ora_nvfp4_quantize_rowwise(const uint16_t* x, int64_t M, int64_t K, uint8_t* q, uint8_t* sf, float* s_enc_out,
                               int nthreads) {
    ora_nv_rowq_ctx c;
    if (!x || !q || !sf || !s_enc_out || M < 0 || K < 0 || K % 16) return ORA_BAD_ARG;
    c.x = x; c.M = M; c.K = K; c.q = q; c.sf = sf;
    c.s_enc = ora_nvfp4_encode_scale(ora_bf16_amax(x, M * K));
    *s_enc_out = c.s_enc;
    ora_parallel(ora_nv_rowq_range, &c, M, nthreads);
    return ORA_OK;
}

/* Row-wise NVFP4 of binary32 values under a given encode scale (test hook for the encoder). */
int ora_nvfp4_quantize_f32(const float* v, int64_t M, int64_t K, float s_enc, uint8_t* q, uint8_t* sf) {
    int64_t r, b;
    if (!v || !q || !sf || M < 0 || K < 0 || K % 16) return ORA_BAD_ARG;
    for (r = 0; r < M; ++r)
        for (b = 0; b < K / 16; ++b)
            sf[r * (K / 16) + b] = ora_nvfp4_quantize_block(v + r * K + b * 16, 16, s_enc, q + r * K + b * 16);
    return ORA_OK;
}

/* ---- the NVFP4 grouped expert MLP, rows listed in `rows` ----------------------------------------
 * x [R, H] bf16 grouped by expert (split), gates [R] or NULL (ones); w1q/w1sf/s_w1: W1 [E*2F, H]
 * from ora_nvfp4_quantize_rowwise (rows [0, F) of each expert gate, [F, 2F) up); w2q/w2sf/s_w2:
 * W2 [E*H, F]; h_amax: the magnitude the intermediate's encode scale is derived from.
 * For row r of expert e:  a = dq(NVFP4_row(x_r; s_x)) with s_x from the largest |x| over all R
 * rows;  g, u = a W1[e, gate/up]^T;  h = gate_r * silu(g) * u;  hq = NVFP4_row(fl32(h); s_h);
 * y = dq(hq) W2[e]^T.  Outputs y [n, H] (binary64), optionally hq [n, F], hsf [n, F/16]. */
typedef struct {
    const uint16_t* x; int64_t R, H, F; int E;
    const int64_t* off; const float* gates;
    const uint8_t *w1q, *w1sf, *w2q, *w2sf;
    float s_x, s_w1, s_w2, s_h;
    const int64_t* rows; double* y; uint8_t *hq, *hsf;
} ora_nv_mlp_ctx;

static void ora_nv_mlp_range(void* p, int64_t i0, int64_t i1) {
    ora_nv_mlp_ctx* c = (ora_nv_mlp_ctx*)p;
    const int64_t H = c->H, F = c->F;
    float* xv = (float*)malloc(sizeof(float) * (size_t)H);
    float* hf = (float*)malloc(sizeof(float) * (size_t)F);
    double* a = (double*)malloc(sizeof(double) * (size_t)H);
    double* hd = (double*)malloc(sizeof(double) * (size_t)F);
    uint8_t* xq = (uint8_t*)malloc((size_t)H);
    uint8_t* xsf = (uint8_t*)malloc((size_t)(H / 16));
    uint8_t* hq = (uint8_t*)malloc((size_t)F);
    uint8_t* hsf = (uint8_t*)malloc((size_t)(F / 16));
    int64_t i, j, k, b;
    for (i = i0; i < i1; ++i) {
        const int64_t r = c->rows[i];
        int e = 0;
        double gate;
        while (!(r >= c->off[e] && r < c->off[e + 1])) ++e;
        gate = c->gates ? (double)c->gates[r] : 1.0;
        for (k = 0; k < H; ++k) xv[k] = (float)ora_bf16_to_double(c->x[r * H + k]);
        for (b = 0; b < H / 16; ++b) xsf[b] = ora_nvfp4_quantize_block(xv + b * 16, 16, c->s_x, xq + b * 16);
        for (k = 0; k < H; ++k) a[k] = ora_nvfp4_dequant(xq[k], xsf[k / 16], c->s_x);
        for (j = 0; j < F; ++j) {
            const int64_t rg = (int64_t)e * 2 * F + j, ru = (int64_t)e * 2 * F + F + j;
            double g = 0.0, u = 0.0, h;
            for (k = 0; k < H; ++k) {
                g += a[k] * ora_nvfp4_dequant(c->w1q[rg * H + k], c->w1sf[rg * (H / 16) + k / 16], c->s_w1);
                u += a[k] * ora_nvfp4_dequant(c->w1q[ru * H + k], c->w1sf[ru * (H / 16) + k / 16], c->s_w1);
            }
            h = gate * (g / (1.0 + exp(-g))) * u;
            hf[j] = (float)h;
        }
        for (b = 0; b < F / 16; ++b) hsf[b] = ora_nvfp4_quantize_block(hf + b * 16, 16, c->s_h, hq + b * 16);
        for (j = 0; j < F; ++j) hd[j] = ora_nvfp4_dequant(hq[j], hsf[j / 16], c->s_h);
        for (k = 0; k < H; ++k) {
            const int64_t rw = (int64_t)e * H + k;
            double acc = 0.0;
            for (j = 0; j < F; ++j)
                acc += hd[j] * ora_nvfp4_dequant(c->w2q[rw * F + j], c->w2sf[rw * (F / 16) + j / 16], c->s_w2);
            c->y[i * H + k] = acc;
        }
        if (c->hq) memcpy(c->hq + i * F, hq, (size_t)F);
        if (c->hsf) memcpy(c->hsf + i * (F / 16), hsf, (size_t)(F / 16));
    }
    free(xv); free(hf); free(a); free(hd); free(xq); free(xsf); free(hq); free(hsf);
}

int ora_nvfp4_grouped_mlp_rows(const uint16_t* x, int64_t R, int64_t H, int64_t F, int E, const int32_t* split,
                               const float* gates, const uint8_t* w1q, const uint8_t* w1sf, float s_w1,
                               const uint8_t* w2q, const uint8_t* w2sf, float s_w2, float h_amax,
                               const int64_t* rows, int64_t nrows, double* y, uint8_t* hq, uint8_t* hsf,
                               float* s_x_out, int nthreads) {
    ora_nv_mlp_ctx c;
    int64_t* off;
    int64_t total = 0, i;
    int e;
    if (!x || !split || !w1q || !w1sf || !w2q || !w2sf || !y || (nrows > 0 && !rows)) return ORA_BAD_ARG;
    if (R < 0 || H <= 0 || F <= 0 || E <= 0 || H % 16 || F % 16 || nrows < 0 || !(h_amax >= 0.0f))
        return ORA_BAD_ARG;
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
    c.s_x = ora_nvfp4_encode_scale(ora_bf16_amax(x, R * H));
    c.s_w1 = s_w1; c.s_w2 = s_w2; c.s_h = ora_nvfp4_encode_scale(h_amax);
    c.rows = rows; c.y = y; c.hq = hq; c.hsf = hsf;
    if (s_x_out) *s_x_out = c.s_x;
    ora_parallel(ora_nv_mlp_range, &c, nrows, nthreads);
    free(off);
    return ORA_OK;
}
