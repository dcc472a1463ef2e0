/*
 * CPU oracle for ROCmFP2 and HFP4G32 block-quantized GEMV / GEMM.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link
 * or call this file: it exists so the tests, the smoke check and the CPU
 * baseline of the benchmark can check the CUDA kernels against a plain,
 * slow, obviously correct restatement of the method.  It shares no code,
 * headers, tables or constants with the CUDA library.
 *
 * Style: single-threaded loops in the order the pages describe, fp64 for the
 * outputs, no blocking or reordering.  Compile with -ffp-contract=off so no
 * multiply-add is fused (the scale search compares fp64 sums bit for bit).
 *
 * Sources (page title, section):
 *  [R]  "ROCmFP2 codebook research report" (llm.ciru.ai), sections
 *       "01 Storage" (10-byte block layout), "02 Quantization" (codebook,
 *       worked example, UE4M3 scale byte, scale search) and "03 Runtime"
 *       (int8 expansion, dot4, rescale dA*(d0*S0 + d1*S1)).
 *  [H]  "HFP4" (hipfire.dev quant-formats), sections "Element format (OCP
 *       E2M1)", "Block scale - UE8M0", "Per-row second-level scale (FP16)",
 *       "Byte layout - HFP4G32", "Nibble packing", "Quantization recipe" and
 *       "v1 correctness-anchor inner loop"; its mention of NVIDIA NVFP4
 *       (16-element blocks with an E4M3 scale) for the block-scaled FP4
 *       form at the end of this file.
 *
 * Readings where the pages are silent (each is also listed in the design notes):
 *  - Scale search: every legal byte 0x00..0x7E is tried in ascending order and
 *    the first strict minimum of the squared error wins (ties go to the
 *    smaller byte).  The "start near max|x|/4" hint only changes the order of
 *    an exhaustive search, so it is not needed.
 *  - x = +0 or -0 takes the positive side (code 10); both sides tie in error.
 *  - Byte 0x00 (s = 0): codes are inner by sign and reconstruct to 0.
 *  - Code choice divides in fp32: fabsf(x / s) <= 2.5f.
 *  - Tensor layout: blocks row-major, K/32 blocks per row, no row header.
 *  - Q8_1-style activation blocks: d = amax/127 (fp32 division), q =
 *    roundf(a/d) (fp32 division, half away from zero), clamped to +-127,
 *    d == 0 gives q = 0.  No sum field.
 *  - E2M1 magnitudes {0, .5, 1, 1.5, 2, 3, 4, 6} (the OCP MX lattice the HFP4
 *    page names; the only 8-level lattice with maximum 6 and gaps .5/1/2).
 *    Ties round to the even mantissa; negative values keep the sign bit.
 *  - HFP4 row scale: rs = fp16(max|W|/6) rounded to nearest even; every later
 *    step uses the stored fp16 value.  rs == 0 gives an all-zero row (e = 0).
 *    Block exponent: the smallest e in [0, 254] with bmax <= 6 * 2^(e-127).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_EINVAL (-1)

/* ------------------------------------------------------------------------ */
/* [R] 02 Quantization: "four signed integer reconstruction levels", code
 * 00 -> -4, 01 -> -1, 10 -> +1, 11 -> +4. */
static const int orc_codebook[4] = {-4, -1, +1, +4};

int orc_codebook_value(int code) { return orc_codebook[code & 3]; }

/* [R] 02 Quantization, "One scale byte, 127 legal values": E = b >> 3,
 * M = b & 7; E = 0 -> M * 2^-10, else (8 + M) * 2^(E - 11).  0x7F and above
 * are rejected. */
int orc_ue4m3(int b, double *s)
{
    if (b < 0 || b > 0x7E) return ORC_EINVAL;
    int E = b >> 3, M = b & 7;
    *s = (E == 0) ? ldexp((double)M, -10) : ldexp((double)(8 + M), E - 11);
    return ORC_OK;
}

/* [R] 02 Quantization: sign chooses the side, |x / scale| <= 2.5 is inner,
 * otherwise outer.  s == 0 (byte 0x00): inner by sign (reading above). */
int orc_rfp2_code(float x, float s)
{
    int neg = x < 0.0f;
    int inner;
    if (s == 0.0f) {
        inner = 1;
    } else {
        float m = fabsf(x / s);
        inner = m <= 2.5f;
    }
    if (neg) return inner ? 1 : 0;
    return inner ? 2 : 3;
}

/* Squared reconstruction error of one 16-value half at scale byte b, summed
 * in index order in fp64 ([R] 02: "keep the scale with the lowest squared
 * reconstruction error"). */
double orc_rfp2_half_sse(const float *x, int b)
{
    double sd;
    if (orc_ue4m3(b, &sd) != ORC_OK) return INFINITY;
    float s = (float)sd; /* exact: at most 4 significant bits */
    double sse = 0.0;
    for (int i = 0; i < 16; i++) {
        int code = orc_rfp2_code(x[i], s);
        float r = (float)orc_codebook[code] * s; /* exact */
        double e = (double)x[i] - (double)r;
        sse = sse + e * e;
    }
    return sse;
}

/* Exhaustive scale search for one half: returns the chosen byte and writes the
 * 16 codes.  Ascending bytes, strict < keeps the first minimum. */
int orc_rfp2_quantize_half(const float *x, uint8_t *codes)
{
    int best = 0;
    double best_sse = orc_rfp2_half_sse(x, 0);
    for (int b = 1; b <= 0x7E; b++) {
        double sse = orc_rfp2_half_sse(x, b);
        if (sse < best_sse) {
            best_sse = sse;
            best = b;
        }
    }
    double sd;
    orc_ue4m3(best, &sd);
    for (int i = 0; i < 16; i++) codes[i] = (uint8_t)orc_rfp2_code(x[i], (float)sd);
    return best;
}

/* [R] 01 Storage: a block of 32 weights is 8 code bytes (q0 = weights 0-3,
 * ..., q7 = weights 28-31; four 2-bit selectors little-endian, weight 4j+i in
 * bits 2i..2i+1 of byte j) then e0 (scale of weights 0-15) and e1 (16-31).
 * W is fp32 [M, K] row-major, K % 32 == 0; out is uint8 [M, K/32, 10]. */
int orc_rfp2_pack(const float *W, int64_t M, int64_t K, uint8_t *out)
{
    if (M < 0 || K < 0 || K % 32 != 0) return ORC_EINVAL;
    for (int64_t i = 0; i < M * K; i++)
        if (!isfinite(W[i])) return ORC_EINVAL;
    int64_t nb = K / 32;
    for (int64_t m = 0; m < M; m++) {
        for (int64_t j = 0; j < nb; j++) {
            const float *x = W + m * K + 32 * j;
            uint8_t *blk = out + (m * nb + j) * 10;
            uint8_t codes[32];
            int e0 = orc_rfp2_quantize_half(x, codes);
            int e1 = orc_rfp2_quantize_half(x + 16, codes + 16);
            memset(blk, 0, 8);
            for (int i = 0; i < 32; i++)
                blk[i / 4] |= (uint8_t)(codes[i] << (2 * (i % 4)));
            blk[8] = (uint8_t)e0;
            blk[9] = (uint8_t)e1;
        }
    }
    return ORC_OK;
}

/* Importance-weighted scale search ([R] "05 Completed experiment": the same
 * squared reconstruction error with each term weighted by
 * importance_i * sqrt(sigma^2 + x_i^2); only the chosen scale changes, not
 * the block, the codebook or the code rule).  The page does not define
 * sigma^2; it is read as twice the mean of x^2 over the 32-weight block.
 * Terms are summed in index order in fp64: w_i * (e_i * e_i). */
double orc_rfp2_block_sigma2(const float *x32)
{
    double s2 = 0.0;
    for (int i = 0; i < 32; i++) s2 = s2 + (double)x32[i] * (double)x32[i];
    return 2.0 * s2 / 32.0;
}

double orc_rfp2_half_wsse(const float *x, const float *imp, double sigma2, int b)
{
    double sd;
    if (orc_ue4m3(b, &sd) != ORC_OK) return INFINITY;
    float s = (float)sd;
    double sse = 0.0;
    for (int i = 0; i < 16; i++) {
        int code = orc_rfp2_code(x[i], s);
        float r = (float)orc_codebook[code] * s;
        double e = (double)x[i] - (double)r;
        double w = (double)imp[i] * sqrt(sigma2 + (double)x[i] * (double)x[i]);
        sse = sse + w * (e * e);
    }
    return sse;
}

/* Weighted search of one half: ascending bytes, first strict minimum. */
int orc_rfp2_quantize_half_weighted(const float *x, const float *imp, double sigma2,
                                    uint8_t *codes)
{
    int best = 0;
    double best_sse = orc_rfp2_half_wsse(x, imp, sigma2, 0);
    for (int b = 1; b <= 0x7E; b++) {
        double sse = orc_rfp2_half_wsse(x, imp, sigma2, b);
        if (sse < best_sse) {
            best_sse = sse;
            best = b;
        }
    }
    double sd;
    orc_ue4m3(best, &sd);
    for (int i = 0; i < 16; i++) codes[i] = (uint8_t)orc_rfp2_code(x[i], (float)sd);
    return best;
}

/* orc_rfp2_pack with the weighted search; importance fp32 [K] (one value per
 * input column, finite and >= 0). */
int orc_rfp2_pack_weighted(const float *W, int64_t M, int64_t K, const float *imp, uint8_t *out)
{
    if (M < 0 || K < 0 || K % 32 != 0) return ORC_EINVAL;
    for (int64_t i = 0; i < M * K; i++)
        if (!isfinite(W[i])) return ORC_EINVAL;
    for (int64_t k = 0; k < K; k++)
        if (!isfinite(imp[k]) || imp[k] < 0.0f) return ORC_EINVAL;
    int64_t nb = K / 32;
    for (int64_t m = 0; m < M; m++) {
        for (int64_t j = 0; j < nb; j++) {
            const float *x = W + m * K + 32 * j;
            uint8_t *blk = out + (m * nb + j) * 10;
            uint8_t codes[32];
            double sigma2 = orc_rfp2_block_sigma2(x);
            int e0 = orc_rfp2_quantize_half_weighted(x, imp + 32 * j, sigma2, codes);
            int e1 = orc_rfp2_quantize_half_weighted(x + 16, imp + 32 * j + 16, sigma2, codes + 16);
            memset(blk, 0, 8);
            for (int i = 0; i < 32; i++)
                blk[i / 4] |= (uint8_t)(codes[i] << (2 * (i % 4)));
            blk[8] = (uint8_t)e0;
            blk[9] = (uint8_t)e1;
        }
    }
    return ORC_OK;
}

/* Code of weight i (0..31) of a block and the scale byte of its half. */
static int blk_code(const uint8_t *blk, int i) { return (blk[i / 4] >> (2 * (i % 4))) & 3; }
static int blk_scale_byte(const uint8_t *blk, int i) { return blk[8 + i / 16]; }

/* Reconstructed weights: w = codebook[code] * scale ([R] 02), fp32 (exact).
 * Returns ORC_EINVAL on a scale byte >= 0x7F. */
int orc_rfp2_decode(const uint8_t *P, int64_t M, int64_t K, float *What)
{
    if (K % 32 != 0) return ORC_EINVAL;
    int64_t nb = K / 32;
    for (int64_t m = 0; m < M; m++)
        for (int64_t j = 0; j < nb; j++) {
            const uint8_t *blk = P + (m * nb + j) * 10;
            for (int i = 0; i < 32; i++) {
                double s;
                if (orc_ue4m3(blk_scale_byte(blk, i), &s) != ORC_OK) return ORC_EINVAL;
                What[m * K + 32 * j + i] = (float)(orc_codebook[blk_code(blk, i)] * s);
            }
        }
    return ORC_OK;
}

/* Count of scale bytes >= 0x7F (the page rejects 0x7F). */
int64_t orc_rfp2_count_bad_scales(const uint8_t *P, int64_t nblocks)
{
    int64_t bad = 0;
    for (int64_t j = 0; j < nblocks; j++) {
        if (P[j * 10 + 8] > 0x7E) bad++;
        if (P[j * 10 + 9] > 0x7E) bad++;
    }
    return bad;
}

/* Q8_1-style activation blocks ([R] 03 Runtime names Q8_1 activations; the
 * per-32 layout and d = max|a|/127 are the statement of the problem):
 * x fp32 [N, K] -> q int8 [N, K], d fp32 [N, K/32]. */
int orc_quantize_act(const float *x, int64_t N, int64_t K, int8_t *q, float *d)
{
    if (K % 32 != 0) return ORC_EINVAL;
    int64_t nb = K / 32;
    for (int64_t n = 0; n < N; n++)
        for (int64_t j = 0; j < nb; j++) {
            const float *a = x + n * K + 32 * j;
            float amax = 0.0f;
            for (int i = 0; i < 32; i++)
                if (fabsf(a[i]) > amax) amax = fabsf(a[i]);
            float dd = amax / 127.0f;
            d[n * nb + j] = dd;
            for (int i = 0; i < 32; i++) {
                int v = 0;
                if (dd != 0.0f) {
                    float r = roundf(a[i] / dd); /* half away from zero */
                    if (r > 127.0f) r = 127.0f;
                    if (r < -127.0f) r = -127.0f;
                    v = (int)r;
                }
                q[n * K + 32 * j + i] = (int8_t)v;
            }
        }
    return ORC_OK;
}

/* [R] 03 Runtime, DOT4: integer sum of one 16-weight half against int8
 * activations, codebook values as signed int8. */
static int32_t half_sum(const uint8_t *blk, int h, const int8_t *qa)
{
    int32_t s = 0;
    for (int i = 16 * h; i < 16 * h + 16; i++) s += orc_codebook[blk_code(blk, i)] * (int32_t)qa[i];
    return s;
}

/* Every int32 half sum: partials[n, m, K/16] for q int8 [N, K]. */
int orc_rfp2_half_partials(const uint8_t *P, int64_t M, int64_t K, const int8_t *q, int64_t N,
                           int32_t *partials)
{
    if (K % 32 != 0) return ORC_EINVAL;
    int64_t nb = K / 32;
    for (int64_t n = 0; n < N; n++)
        for (int64_t m = 0; m < M; m++)
            for (int64_t j = 0; j < nb; j++) {
                const uint8_t *blk = P + (m * nb + j) * 10;
                const int8_t *qa = q + n * K + 32 * j;
                int32_t *out = partials + (n * M + m) * (K / 16) + 2 * j;
                out[0] = half_sum(blk, 0, qa);
                out[1] = half_sum(blk, 1, qa);
            }
    return ORC_OK;
}

/* [R] 03 Runtime, RESCALE: y = sum over blocks of dA * (d0 * S0 + d1 * S1),
 * accumulated in fp64.  y is fp64 [N, nrows]; rows[] selects which weight
 * rows to compute (all rows: rows = 0..M-1). */
int orc_rfp2_gemv_rows(const uint8_t *P, int64_t M, int64_t K, const int64_t *rows, int64_t nrows,
                       const int8_t *q, const float *d, int64_t N, double *y)
{
    if (K % 32 != 0) return ORC_EINVAL;
    int64_t nb = K / 32;
    for (int64_t n = 0; n < N; n++)
        for (int64_t r = 0; r < nrows; r++) {
            int64_t m = rows[r];
            if (m < 0 || m >= M) return ORC_EINVAL;
            double acc = 0.0;
            for (int64_t j = 0; j < nb; j++) {
                const uint8_t *blk = P + (m * nb + j) * 10;
                double d0, d1;
                if (orc_ue4m3(blk[8], &d0) != ORC_OK || orc_ue4m3(blk[9], &d1) != ORC_OK)
                    return ORC_EINVAL;
                const int8_t *qa = q + n * K + 32 * j;
                double s0 = (double)half_sum(blk, 0, qa), s1 = (double)half_sum(blk, 1, qa);
                acc = acc + (double)d[n * nb + j] * (d0 * s0 + d1 * s1);
            }
            y[n * nrows + r] = acc;
        }
    return ORC_OK;
}

/* Second, independent formulation: y = sum_k w_k * (q_k * dA) with the
 * decoded weight w_k, fp64, one weight at a time. */
int orc_rfp2_gemv_brute(const uint8_t *P, int64_t M, int64_t K, const int8_t *q, const float *d,
                        int64_t N, double *y)
{
    if (K % 32 != 0) return ORC_EINVAL;
    int64_t nb = K / 32;
    for (int64_t n = 0; n < N; n++)
        for (int64_t m = 0; m < M; m++) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; k++) {
                const uint8_t *blk = P + (m * nb + k / 32) * 10;
                int i = (int)(k % 32);
                double s;
                if (orc_ue4m3(blk_scale_byte(blk, i), &s) != ORC_OK) return ORC_EINVAL;
                double w = (double)orc_codebook[blk_code(blk, i)] * s;
                double a = (double)q[n * K + k] * (double)d[n * nb + k / 32];
                acc = acc + w * a;
            }
            y[n * M + m] = acc;
        }
    return ORC_OK;
}

/* MoE expert-indexed GEMV (MUL_MAT_ID as a GEMV over the routed experts'
 * rows, "HRX on the Radeon iGPU", section "MoE decode and the kernel cache"):
 * W uint8 [E, M, K/32, 10]; ids int32 [T, top_k]; q/d the quantized
 * activations of the T tokens; y fp64 [T, top_k, nrows] for the selected rows.
 * An id outside [0, E) returns ORC_EINVAL. */
int orc_rfp2_moe_rows(const uint8_t *P, int64_t E, int64_t M, int64_t K, const int32_t *ids,
                      int64_t T, int64_t top_k, const int64_t *rows, int64_t nrows,
                      const int8_t *q, const float *d, double *y)
{
    if (K % 32 != 0) return ORC_EINVAL;
    int64_t expert_bytes = M * (K / 32) * 10;
    for (int64_t t = 0; t < T; t++)
        for (int64_t j = 0; j < top_k; j++) {
            int64_t e = ids[t * top_k + j];
            if (e < 0 || e >= E) return ORC_EINVAL;
            int rc = orc_rfp2_gemv_rows(P + e * expert_bytes, M, K, rows, nrows,
                                        q + t * K, d + t * (K / 32), 1,
                                        y + (t * top_k + j) * nrows);
            if (rc != ORC_OK) return rc;
        }
    return ORC_OK;
}

/* Prefill: Y[n, m] = sum_k w[m, k] * X[n, k] in fp64, X given as bf16 bits,
 * the weights decoded exactly; no activation quantization on this path.
 * Computes the selected weight rows only: y fp64 [N, nrows]. */
int orc_rfp2_gemm_rows(const uint8_t *P, int64_t M, int64_t K, const uint16_t *X, int64_t N,
                       const int64_t *rows, int64_t nrows, double *y)
{
    if (K % 32 != 0) return ORC_EINVAL;
    float *w = (float *)malloc(sizeof(float) * (size_t)K);
    if (!w) return ORC_EINVAL;
    int64_t nb = K / 32;
    for (int64_t r = 0; r < nrows; r++) {
        int64_t m = rows[r];
        if (m < 0 || m >= M || orc_rfp2_decode(P + m * nb * 10, 1, K, w) != ORC_OK) {
            free(w);
            return ORC_EINVAL;
        }
        for (int64_t n = 0; n < N; n++) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; k++) {
                uint32_t bits = (uint32_t)X[n * K + k] << 16;
                float xf;
                memcpy(&xf, &bits, 4);
                acc = acc + (double)w[k] * (double)xf;
            }
            y[n * nrows + r] = acc;
        }
    }
    free(w);
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* HFP4G32.  [H] "Element format (OCP E2M1)": sixteen codes, eight magnitudes;
 * code bit 3 is the sign, bits 0-2 index the magnitudes in increasing order. */
static const double orc_e2m1_mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double orc_e2m1_value(int code)
{
    double v = orc_e2m1_mag[code & 7];
    return (code & 8) ? -v : v;
}

/* Nearest E2M1 code to v (ties to the even mantissa, i.e. the even index);
 * the sign bit follows signbit(v). */
int orc_e2m1_encode(double v)
{
    double a = fabs(v);
    int best = 0;
    double best_err = fabs(a - orc_e2m1_mag[0]);
    for (int i = 1; i < 8; i++) {
        double err = fabs(a - orc_e2m1_mag[i]);
        if (err < best_err || (err == best_err && (i % 2 == 0) && (best % 2 == 1))) {
            best = i;
            best_err = err;
        }
    }
    return best | (signbit(v) ? 8 : 0);
}

/* [H] "Block scale - UE8M0": e in [0, 254] means 2^(e - 127); 0xFF is NaN. */
double orc_ue8m0(int e)
{
    if (e == 0xFF) return NAN;
    return ldexp(1.0, e - 127);
}

int64_t orc_hfp4_row_bytes(int64_t K) { return 16 + 17 * (K / 32); }

/* [H] "Quantization recipe (HFP4G32)" and "Byte layout": per row a 16-byte
 * header (f16 row_scale_a, f16 row_scale_b = 0, u16 block count K/32, u8
 * flags = 0, reserved zeros) then K/32 blocks of (UE8M0 byte, 16 nibble
 * bytes, element 2b in the low nibble of byte b).  Returns ORC_EINVAL when K
 * is not a multiple of 32 or max|W|/6 rounds to an infinite fp16. */
int orc_hfp4_pack(const float *W, int64_t M, int64_t K, uint8_t *out)
{
    if (K % 32 != 0 || K / 32 > 0xFFFF) return ORC_EINVAL;
    int64_t rb = orc_hfp4_row_bytes(K), nb = K / 32;
    for (int64_t m = 0; m < M; m++) {
        const float *w = W + m * K;
        uint8_t *row = out + m * rb;
        float amax = 0.0f;
        for (int64_t k = 0; k < K; k++) {
            if (!isfinite(w[k])) return ORC_EINVAL;
            if (fabsf(w[k]) > amax) amax = fabsf(w[k]);
        }
        _Float16 rs16 = (_Float16)(amax / 6.0f); /* IEEE round to nearest even */
        float rs = (float)rs16;
        if (!isfinite(rs)) return ORC_EINVAL;
        uint16_t rs_bits;
        memcpy(&rs_bits, &rs16, 2);
        memset(row, 0, 16);
        row[0] = (uint8_t)(rs_bits & 0xFF);
        row[1] = (uint8_t)(rs_bits >> 8);
        row[4] = (uint8_t)(nb & 0xFF);
        row[5] = (uint8_t)(nb >> 8);
        for (int64_t j = 0; j < nb; j++) {
            uint8_t *blk = row + 16 + 17 * j;
            float wn[32];
            float bmax = 0.0f;
            for (int i = 0; i < 32; i++) {
                wn[i] = (rs == 0.0f) ? 0.0f : w[32 * j + i] / rs;
                if (fabsf(wn[i]) > bmax) bmax = fabsf(wn[i]);
            }
            int e = 0;
            while (e < 254 && !((double)bmax <= 6.0 * ldexp(1.0, e - 127))) e++;
            blk[0] = (uint8_t)e;
            memset(blk + 1, 0, 16);
            for (int i = 0; i < 32; i++) {
                double v = ldexp((double)wn[i], 127 - e);
                int c = orc_e2m1_encode(v);
                blk[1 + i / 2] |= (uint8_t)(c << (4 * (i % 2)));
            }
        }
    }
    return ORC_OK;
}

static float f16_bits_to_float(uint16_t b)
{
    _Float16 h;
    memcpy(&h, &b, 2);
    return (float)h;
}

/* [H] "Per-row second-level scale": value = row_scale_a * 2^(e - 127) *
 * E2M1[nibble], computed in fp64 and stored as fp32 (exact unless it leaves
 * the fp32 range).  A block byte 0xFF decodes to NaN. */
int orc_hfp4_decode(const uint8_t *P, int64_t M, int64_t K, double *What)
{
    if (K % 32 != 0) return ORC_EINVAL;
    int64_t rb = orc_hfp4_row_bytes(K), nb = K / 32;
    for (int64_t m = 0; m < M; m++) {
        const uint8_t *row = P + m * rb;
        double rs = (double)f16_bits_to_float((uint16_t)(row[0] | (row[1] << 8)));
        for (int64_t j = 0; j < nb; j++) {
            const uint8_t *blk = row + 16 + 17 * j;
            double sc = rs * orc_ue8m0(blk[0]);
            for (int i = 0; i < 32; i++) {
                int c = (blk[1 + i / 2] >> (4 * (i % 2))) & 15;
                What[m * K + 32 * j + i] = sc * orc_e2m1_value(c);
            }
        }
    }
    return ORC_OK;
}

/* HFP4 GEMV in the shape of the page's correctness-anchor loop ([H] "v1
 * correctness-anchor inner loop"): per block sc = row_scale_a * 2^(e-127),
 * per element sc * lut[nibble] * x, accumulated in fp64.  x fp32 [N, K]; y
 * fp64 [N, nrows] over the selected rows. */
int orc_hfp4_gemv_rows(const uint8_t *P, int64_t M, int64_t K, const int64_t *rows, int64_t nrows,
                       const float *x, int64_t N, double *y)
{
    if (K % 32 != 0) return ORC_EINVAL;
    int64_t rb = orc_hfp4_row_bytes(K), nb = K / 32;
    for (int64_t n = 0; n < N; n++)
        for (int64_t r = 0; r < nrows; r++) {
            int64_t m = rows[r];
            if (m < 0 || m >= M) return ORC_EINVAL;
            const uint8_t *row = P + m * rb;
            double rs = (double)f16_bits_to_float((uint16_t)(row[0] | (row[1] << 8)));
            double acc = 0.0;
            for (int64_t j = 0; j < nb; j++) {
                const uint8_t *blk = row + 16 + 17 * j;
                double sc = rs * orc_ue8m0(blk[0]);
                for (int i = 0; i < 32; i++) {
                    int c = (blk[1 + i / 2] >> (4 * (i % 2))) & 15;
                    acc = acc + sc * orc_e2m1_value(c) * (double)x[n * K + 32 * j + i];
                }
            }
            y[n * nrows + r] = acc;
        }
    return ORC_OK;
}

/* fp32 -> fp16 round to nearest even, and back (for the tests' pins). */
uint16_t orc_f32_to_f16_bits(float v)
{
    _Float16 h = (_Float16)v;
    uint16_t b;
    memcpy(&b, &h, 2);
    return b;
}

float orc_f16_bits_to_f32(uint16_t b) { return f16_bits_to_float(b); }

/* ------------------------------------------------------------------------ */
/* Block-scaled FP4 (NVFP4) form of ROCmFP2.  The pages name NVFP4 only as a
 * reference format ([H] "HFP4 ... NVIDIA NVFP4": 16-element blocks with an
 * E4M3 scale).  Readings (no page defines them):
 *  - An NVFP4 block is 16 E2M1 elements (the lattice above) times one
 *    E4M3FN scale byte (sign 0; E = bits 3-6, bias 7; E = 0 is subnormal
 *    M * 2^-9; 0x7F is NaN), times a per-tensor fp32 factor.
 *  - ROCmFP2 weights need no rounding: [R] 02's closed form makes s(b) half
 *    the E4M3FN value of the same byte, so codebook * s(b) = (codebook / 2) *
 *    E4M3FN(b) with codebook / 2 in {-2, -0.5, 0.5, 2}, all E2M1 values.
 *    The weight factor is 1.
 *  - Activations (one token row x of K values) follow NVIDIA's published
 *    recipe, in fp32 as written: g = 2688 / amax(x) (448 * 6; g = 1 for an
 *    all-zero row); per 16 values t = (bmax / 6) * g, scale byte = E4M3FN of
 *    t rounded to nearest (ties to even), saturating at 448; element code =
 *    nearest E2M1 of (x * g) / s (ties to the even mantissa, saturating at
 *    6; the sign bit follows signbit); a block whose scale byte is 0 stores
 *    +0 codes.  The value is E2M1 * E4M3FN(byte) / g. */

double orc_e4m3fn_value(int b)
{
    int E = (b >> 3) & 15, M = b & 7;
    double v;
    if (E == 15 && M == 7) return NAN;
    v = E == 0 ? M * ldexp(1.0, -9) : (8 + M) * ldexp(1.0, E - 10);
    return (b & 0x80) ? -v : v;
}

/* Nearest non-negative E4M3FN byte to v >= 0 (ties to the even byte, which
 * is the even mantissa), saturating at 0x7E = 448: a search over all bytes. */
int orc_e4m3fn_encode(double v)
{
    int best = 0;
    double best_err = fabs(v - orc_e4m3fn_value(0));
    for (int b = 1; b <= 0x7E; b++) {
        double err = fabs(v - orc_e4m3fn_value(b));
        if (err < best_err || (err == best_err && (b % 2 == 0) && (best % 2 == 1))) {
            best = b;
            best_err = err;
        }
    }
    return best;
}

/* Weights: codes [M, K] (one E2M1 code per byte) and scale bytes [M, K/16]. */
int orc_rfp2_to_nvfp4(const uint8_t *P, int64_t M, int64_t K, uint8_t *codes, uint8_t *sbytes)
{
    if (!P || !codes || !sbytes || M < 0 || K < 0 || K % 32) return ORC_EINVAL;
    int64_t KB = K / 32;
    for (int64_t m = 0; m < M; m++)
        for (int64_t kb = 0; kb < KB; kb++) {
            const uint8_t *blk = P + (m * KB + kb) * 10;
            for (int i = 0; i < 32; i++)
                codes[m * K + kb * 32 + i] =
                    (uint8_t)orc_e2m1_encode(orc_codebook_value(blk_code(blk, i)) / 2.0);
            sbytes[m * (K / 16) + kb * 2] = blk[8];
            sbytes[m * (K / 16) + kb * 2 + 1] = blk[9];
        }
    return ORC_OK;
}

/* Activations: codes [N, K], scale bytes [N, K/16], g [N] (K % 16 == 0). */
int orc_nvfp4_quant_act(const float *x, int64_t N, int64_t K, uint8_t *codes, uint8_t *sbytes,
                        float *g)
{
    if (!x || !codes || !sbytes || !g || N < 0 || K < 0 || K % 16) return ORC_EINVAL;
    for (int64_t n = 0; n < N; n++) {
        const float *xr = x + n * K;
        float amax = 0.0f;
        for (int64_t k = 0; k < K; k++)
            if (fabsf(xr[k]) > amax) amax = fabsf(xr[k]);
        float gn = amax > 0.0f ? 2688.0f / amax : 1.0f;
        g[n] = gn;
        for (int64_t j = 0; j < K / 16; j++) {
            float bmax = 0.0f;
            for (int i = 0; i < 16; i++)
                if (fabsf(xr[j * 16 + i]) > bmax) bmax = fabsf(xr[j * 16 + i]);
            float t = (bmax / 6.0f) * gn;
            int b = orc_e4m3fn_encode((double)t);
            float s = (float)orc_e4m3fn_value(b);
            sbytes[n * (K / 16) + j] = (uint8_t)b;
            for (int i = 0; i < 16; i++) {
                uint8_t c = 0;
                if (s != 0.0f) {
                    float u = xr[j * 16 + i] * gn;
                    float e = u / s;
                    c = (uint8_t)orc_e2m1_encode((double)e);
                }
                codes[n * K + j * 16 + i] = c;
            }
        }
    }
    return ORC_OK;
}

/* y[n, r] = (1 / g[n]) * sum_k E2M1(w[m, k]) E4M3FN(ws[m, k/16]) E2M1(x[n, k])
 * E4M3FN(xs[n, k/16]) for m = rows[r], in fp64. */
int orc_nvfp4_gemm_rows(const uint8_t *wc, const uint8_t *ws, int64_t M, int64_t K,
                        const uint8_t *xc, const uint8_t *xs, const float *g, int64_t N,
                        const int64_t *rows, int64_t nrows, double *y)
{
    if (!wc || !ws || !xc || !xs || !g || !rows || !y || K % 16) return ORC_EINVAL;
    for (int64_t r = 0; r < nrows; r++) {
        int64_t m = rows[r];
        if (m < 0 || m >= M) return ORC_EINVAL;
        for (int64_t n = 0; n < N; n++) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; k++) {
                double w = orc_e2m1_value(wc[m * K + k]) * orc_e4m3fn_value(ws[m * (K / 16) + k / 16]);
                double a = orc_e2m1_value(xc[n * K + k]) * orc_e4m3fn_value(xs[n * (K / 16) + k / 16]);
                acc += w * a;
            }
            y[n * nrows + r] = acc / (double)g[n];
        }
    }
    return ORC_OK;
}
