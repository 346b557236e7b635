/*
 * oracle.c -- plain, slow CPU reference of the Q4_K mixture-of-experts FFN.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * CPU-baseline leg of bench.py load this library.  It shares no code,
 * header, table or constant with the CUDA path in
 * quantized_moe_expert_gemv_gb300/csrc/, and neither side includes the other.
 *
 * What it computes (the method, as the sparkinfer pages describe it):
 *   sparkinfer README (luciferlive112116), "Layout" table: the kernels
 *   directory holds a "fused quantized MoE expert FFN", a "decode GEMV" and
 *   "GGUF dequant"; the moe directory holds a "sync-free MoE router + expert
 *   dispatch (on-device counts)".  Its opening section keeps experts
 *   "quantized-resident, dequantized on-read" for greedy bs=1 decode of a
 *   Q4_K_M GGUF Qwen3-30B-A3B.  The SP-RKINFER README (gittensor-ai-lab),
 *   "Benchmark - Qwen3.8-27B" prefill note, has the grouped/prefill variant
 *   dequantize "Q4_K into the GEMM operand on every pass".
 *
 * Per token the MoE FFN is
 *   z      = W_r x (+ bias)                       router logits, E values
 *   ids    = the k largest z (descending; equal z -> lower expert index)
 *   w_i    = softmax(z)[ids_i] / sum_j softmax(z)[ids_j]   (renormalised)
 *   g, u   = W_gate[e] x, W_up[e] x               (I values each)
 *   h      = silu(g) * u,  silu(g) = g / (1 + exp(-g))
 *   y      = W_down[e] h                          (H values)
 *   out    = sum_i w_i y_i
 * and, optionally, the block around it: x replaced by rmsnorm(x) = x * gamma /
 * sqrt(mean(x^2) + eps) on the way in and out = x + sum_i w_i y_i on the way
 * out (a pre-normed block with its residual);
 * with every expert matrix stored as GGUF Q4_K super-blocks (or NVFP4
 * super-blocks, defined below) and read as the fp32 weights the format's
 * decode defines.
 *
 * Precision: all products and sums are fp64 over the exact fp32 weights and
 * the exact fp32 value of each bf16 activation; results are rounded to
 * fp32 once at the end.  The top-k choice is taken on the logits rounded
 * to fp32 (the precision the GPU path decides in).
 *
 * Q4_K (GGUF) super-block, 144 bytes per 256 weights, byte order:
 *   bytes 0-1   d     (IEEE binary16, little-endian)
 *   bytes 2-3   dmin  (IEEE binary16, little-endian)
 *   bytes 4-15  scales[12]: eight 6-bit scales sc_j and eight 6-bit mins m_j
 *   bytes 16-143 qs[128]: 4-bit codes q
 *   sub-block j (j = 0..7) covers weights 32j .. 32j+31 of the block;
 *   qs[32i + l] holds weight l of sub-block 2i in its low nibble and
 *   weight l of sub-block 2i+1 in its high nibble;
 *   j < 4 : sc_j = scales[j] & 63,  m_j = scales[j+4] & 63
 *   j >= 4: sc_j = (scales[j+4] & 15) | ((scales[j-4] >> 6) << 4)
 *           m_j  = (scales[j+4] >> 4) | ((scales[j]   >> 6) << 4)
 *   weight = d * sc_j * q - dmin * m_j
 *
 * No function here is tuned: loops follow the definitions one term at a time.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_QK 256
#define OR_BLOCK_BYTES 144

int or_version(void) { return 1; }

/* IEEE 754 binary16 -> exact double.  1 sign bit, 5 exponent bits (bias 15),
 * 10 fraction bits; exponent 0 is subnormal (fraction * 2^-24), exponent 31
 * is inf/nan. */
double or_half_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int f = h & 1023;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24);
    } else if (e == 31) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + f), e - 25);
    }
    return sign ? -v : v;
}

/* bf16 bit pattern -> exact double (bf16 is the top half of an fp32). */
double or_bf16_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* The 6-bit scale and min of sub-block j, as the Q4_K format packs them. */
void or_q4k_scale_min(const uint8_t *scales, int j, int *sc, int *m) {
    if (j < 4) {
        *sc = scales[j] & 63;
        *m = scales[j + 4] & 63;
    } else {
        *sc = (scales[j + 4] & 15) | ((scales[j - 4] >> 6) << 4);
        *m = (scales[j + 4] >> 4) | ((scales[j] >> 6) << 4);
    }
}

/* Decode one super-block into 256 fp32 weights.  The value d*sc*q - dmin*m
 * is formed exactly in fp64 (each product has at most 21 significant bits)
 * and rounded to fp32 once. */
static void or_q4k_block(const uint8_t *blk, float *out) {
    double d = or_half_to_double((uint16_t)(blk[0] | (blk[1] << 8)));
    double dmin = or_half_to_double((uint16_t)(blk[2] | (blk[3] << 8)));
    const uint8_t *scales = blk + 4;
    const uint8_t *qs = blk + 16;
    for (int j = 0; j < 8; ++j) {
        int sc, m;
        or_q4k_scale_min(scales, j, &sc, &m);
        int i = j / 2;
        for (int l = 0; l < 32; ++l) {
            int byte = qs[32 * i + l];
            int q = (j % 2 == 0) ? (byte & 15) : (byte >> 4);
            double w = d * (double)sc * (double)q - dmin * (double)m;
            out[32 * j + l] = (float)w;
        }
    }
}

void or_q4k_dequant(const uint8_t *blocks, int64_t n_blocks, float *out) {
    for (int64_t b = 0; b < n_blocks; ++b)
        or_q4k_block(blocks + b * OR_BLOCK_BYTES, out + b * OR_QK);
}

/* ------------------------------------------------------------------ Q5_K
 * Another GGUF K-quant block type (a Q4_K_M / Q5_K_M file mixes K-quant
 * types; the pages name Q4_K_M files but give no mix).  The layout is GGUF's
 * Q5_K, taken from the format's public definition (a reading: the pages do not
 * define it): 176 bytes per 256 weights,
 *   bytes 0-1    d (binary16),  bytes 2-3  dmin (binary16)
 *   bytes 4-15   scales[12]: the same eight 6-bit scales and mins as Q4_K
 *   bytes 16-47  qh[32]: bit j of qh[l] is the fifth (value-16) bit of
 *                weight l of sub-block j
 *   bytes 48-175 qs[128]: the low four bits, arranged as Q4_K's qs
 *   q = low4 + 16 * high bit (0..31),  weight = d * sc_j * q - dmin * m_j */
#define OR_Q5K_BLOCK_BYTES 176

static void or_q5k_block(const uint8_t *blk, float *out) {
    double d = or_half_to_double((uint16_t)(blk[0] | (blk[1] << 8)));
    double dmin = or_half_to_double((uint16_t)(blk[2] | (blk[3] << 8)));
    const uint8_t *scales = blk + 4;
    const uint8_t *qh = blk + 16;
    const uint8_t *qs = blk + 48;
    for (int j = 0; j < 8; ++j) {
        int sc, m;
        or_q4k_scale_min(scales, j, &sc, &m);
        int i = j / 2;
        for (int l = 0; l < 32; ++l) {
            int byte = qs[32 * i + l];
            int low4 = (j % 2 == 0) ? (byte & 15) : (byte >> 4);
            int q = low4 + 16 * ((qh[l] >> j) & 1);
            double w = d * (double)sc * (double)q - dmin * (double)m;  /* exact in fp64 */
            out[32 * j + l] = (float)w;
        }
    }
}

void or_q5k_dequant(const uint8_t *blocks, int64_t n_blocks, float *out) {
    for (int64_t b = 0; b < n_blocks; ++b)
        or_q5k_block(blocks + b * OR_Q5K_BLOCK_BYTES, out + b * OR_QK);
}

/* One row of a Q4_K matrix with `cols` input columns, as fp32 weights. */
static void or_q4k_row(const uint8_t *row_blocks, int cols, float *out) {
    or_q4k_dequant(row_blocks, cols / OR_QK, out);
}

/* ------------------------------------------------------------------ NVFP4
 * NVFP4 experts (the sparkinfer README's "Milestone 2" names NVFP4 experts as
 * the next bytes-per-token step; the SP-RKINFER README, "Native NVFP4 - two
 * supported checkpoints", runs NVFP4 weights directly; the CuTe-DSL README's
 * moe row lists a W4A16 mode: BF16 activations, inline FP4 weight dequant).
 * The pages give no bit layout; the format is taken as NVIDIA defines NVFP4:
 *   element  E2M1: bit 3 sign, bits 2-1 exponent e (bias 1), bit 0 mantissa m;
 *            e = 0: value m * 0.5 (subnormal); e > 0: 2^(e-1) * (1 + m/2)
 *   block    16 consecutive elements of a row share one scale in FP8 E4M3:
 *            bit 7 sign, bits 6-3 exponent E (bias 7), bits 2-0 mantissa M;
 *            E = 0: M/8 * 2^-6 (subnormal); E = 15 and M = 7: NaN (no inf);
 *            otherwise 2^(E-7) * (1 + M/8)
 *   tensor   one fp32 scale g per expert matrix
 *   weight = e2m1 * e4m3 * g
 * Storage (this library's reading; a lossless repack of a checkpoint's
 * separate code and scale tensors): super-blocks of 256 weights, 144 bytes,
 *   bytes 0-15    the E4M3 scales of weights 16j .. 16j+15 (j = 0..15)
 *   bytes 16-143  codes: byte 16 + l holds weight 2l in its low nibble and
 *                 weight 2l+1 in its high nibble. */
double or_e2m1_to_double(int code) {
    int sign = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
    double v = e == 0 ? 0.5 * (double)m : ldexp(1.0 + 0.5 * (double)m, e - 1);
    return sign ? -v : v;
}

double or_e4m3_to_double(uint8_t b) {
    int sign = (b >> 7) & 1, E = (b >> 3) & 15, M = b & 7;
    double v;
    if (E == 15 && M == 7) v = NAN;
    else if (E == 0) v = ldexp((double)M / 8.0, -6);
    else v = ldexp(1.0 + (double)M / 8.0, E - 7);
    return sign ? -v : v;
}

/* Decode NVFP4 super-blocks into fp32 weights: e2m1 * e4m3 * g formed in
 * fp64 (exact: at most 2 + 4 + 24 significant bits) and rounded once. */
void or_nvfp4_dequant(const uint8_t *blocks, int64_t n_blocks, float g, float *out) {
    for (int64_t b = 0; b < n_blocks; ++b) {
        const uint8_t *blk = blocks + b * OR_BLOCK_BYTES;
        for (int i = 0; i < OR_QK; ++i) {
            int byte = blk[16 + i / 2];
            int code = (i % 2 == 0) ? (byte & 15) : (byte >> 4);
            double w = or_e2m1_to_double(code) * or_e4m3_to_double(blk[i / 16]) * (double)g;
            out[b * OR_QK + i] = (float)w;
        }
    }
}

/* Router logits in fp64: z_e = sum_c W_r[e][c] * x_c (+ bias_e). */
void or_router_logits(const float *router_w, const float *bias, const uint16_t *x_bf16,
                      int E, int H, double *z) {
    for (int e = 0; e < E; ++e) {
        double s = 0.0;
        for (int c = 0; c < H; ++c)
            s += (double)router_w[(int64_t)e * H + c] * or_bf16_to_double(x_bf16[c]);
        if (bias) s += (double)bias[e];
        z[e] = s;
    }
}

/* The k largest of z32, in descending order; equal values -> lower index
 * first.  Selection by repeated scan: pick the best not yet taken. */
void or_topk(const float *z32, int E, int k, int32_t *ids) {
    unsigned char *taken = (unsigned char *)calloc((size_t)E, 1);
    for (int i = 0; i < k; ++i) {
        int best = -1;
        for (int e = 0; e < E; ++e) {
            if (taken[e]) continue;
            if (best < 0 || z32[e] > z32[best]) best = e;
        }
        taken[best] = 1;
        ids[i] = best;
    }
    free(taken);
}

/* Renormalised softmax weights of the selected experts: the softmax over
 * all E logits, divided by its sum over the selected ones. */
void or_renorm_weights(const double *z, int E, const int32_t *ids, int k, double *w) {
    double zmax = z[0];
    for (int e = 1; e < E; ++e)
        if (z[e] > zmax) zmax = z[e];
    double total = 0.0;
    for (int e = 0; e < E; ++e) total += exp(z[e] - zmax);
    double sel = 0.0;
    for (int i = 0; i < k; ++i) sel += exp(z[ids[i]] - zmax) / total;
    for (int i = 0; i < k; ++i) w[i] = (exp(z[ids[i]] - zmax) / total) / sel;
}

/* z_(k) - z_(k+1) of the fp64 logits (the k-th and (k+1)-th largest, found
 * by repeated scan); +inf when k == E. */
static double or_margin(const double *z, int E, int k) {
    if (k >= E) return INFINITY;
    unsigned char *taken = (unsigned char *)calloc((size_t)E, 1);
    double kth = 0.0, next = 0.0;
    for (int i = 0; i <= k; ++i) {
        int best = -1;
        for (int e = 0; e < E; ++e)
            if (!taken[e] && (best < 0 || z[e] > z[best])) best = e;
        taken[best] = 1;
        if (i == k - 1) kth = z[best];
        if (i == k) next = z[best];
    }
    free(taken);
    return kth - next;
}

/* Route T tokens: ids [T][k], weights [T][k]; optionally the fp64 logits
 * [T][E] and each token's margin z_(k) - z_(k+1) (sorted fp64 logits;
 * +inf when k == E). */
void or_route_tokens(const float *router_w, const float *bias, const uint16_t *x_bf16,
                     int T, int E, int H, int k, int32_t *ids, double *w,
                     double *z_out, double *margin) {
    double *z = (double *)malloc(sizeof(double) * (size_t)E);
    float *z32 = (float *)malloc(sizeof(float) * (size_t)E);
    for (int t = 0; t < T; ++t) {
        or_router_logits(router_w, bias, x_bf16 + (int64_t)t * H, E, H, z);
        for (int e = 0; e < E; ++e) z32[e] = (float)z[e];
        or_topk(z32, E, k, ids + (int64_t)t * k);
        or_renorm_weights(z, E, ids + (int64_t)t * k, k, w + (int64_t)t * k);
        if (z_out)
            for (int e = 0; e < E; ++e) z_out[(int64_t)t * E + e] = z[e];
        if (margin) margin[t] = or_margin(z, E, k);
    }
    free(z);
    free(z32);
}

static double or_silu(double g) { return g / (1.0 + exp(-g)); }

#define OR_WTYPE_Q4_K 12
#define OR_WTYPE_Q5_K 13
#define OR_WTYPE_NVFP4 100

/* Bytes of one 256-weight block of the format. */
static int64_t or_block_bytes(int wtype) { return wtype == OR_WTYPE_Q5_K ? OR_Q5K_BLOCK_BYTES : OR_BLOCK_BYTES; }

/* One row of `cols` weights of any format as fp32 (g: the matrix's NVFP4
 * tensor scale, unused otherwise). */
static void or_row(int wtype, const uint8_t *row_blocks, int cols, float g, float *out) {
    if (wtype == OR_WTYPE_NVFP4) or_nvfp4_dequant(row_blocks, cols / OR_QK, g, out);
    else if (wtype == OR_WTYPE_Q5_K) or_q5k_dequant(row_blocks, cols / OR_QK, out);
    else or_q4k_row(row_blocks, cols, out);
}

/* One expert's SwiGLU FFN in fp64, weights of type wtype:
 *   g_r = sum_c Wg[r][c] x_c,  u_r = sum_c Wu[r][c] x_c,  h_r = silu(g_r) u_r,
 *   y_c = sum_r Wd[c][r] h_r.
 * wg, wu: this expert's [I][H/256] blocks; wd: its [H][I/256] blocks; gg,
 * gu, gd: the three matrices' NVFP4 tensor scales (ignored for Q4_K). */
void or_expert_ffn_wt(int wtype, const uint8_t *wg, const uint8_t *wu, const uint8_t *wd, float gg,
                      float gu, float gd, int H, int I, const double *x, double *h_out, double *y) {
    float *row = (float *)malloc(sizeof(float) * (size_t)(H > I ? H : I));
    double *h = (double *)malloc(sizeof(double) * (size_t)I);
    int64_t gate_row_bytes = (int64_t)(H / OR_QK) * or_block_bytes(wtype);
    int64_t down_row_bytes = (int64_t)(I / OR_QK) * or_block_bytes(wtype);
    for (int r = 0; r < I; ++r) {
        double g = 0.0, u = 0.0;
        or_row(wtype, wg + r * gate_row_bytes, H, gg, row);
        for (int c = 0; c < H; ++c) g += (double)row[c] * x[c];
        or_row(wtype, wu + r * gate_row_bytes, H, gu, row);
        for (int c = 0; c < H; ++c) u += (double)row[c] * x[c];
        h[r] = or_silu(g) * u;
        if (h_out) h_out[r] = h[r];
    }
    for (int c = 0; c < H; ++c) {
        double s = 0.0;
        or_row(wtype, wd + c * down_row_bytes, I, gd, row);
        for (int r = 0; r < I; ++r) s += (double)row[r] * h[r];
        y[c] = s;
    }
    free(row);
    free(h);
}

/* The Q4_K expert FFN (as or_expert_ffn_wt with Q4_K weights). */
void or_expert_ffn(const uint8_t *wg, const uint8_t *wu, const uint8_t *wd,
                   int H, int I, const double *x, double *h_out, double *y) {
    or_expert_ffn_wt(OR_WTYPE_Q4_K, wg, wu, wd, 0.f, 0.f, 0.f, H, I, x, h_out, y);
}

/* The whole MoE FFN for one token, experts of type wtype (gsc: the NVFP4
 * tensor scales [E][3] of each expert's gate, up and down matrices, or NULL
 * for Q4_K).  Outputs: ids [k], w [k], out32 [H] (fp32-rounded), and
 * optionally out64 [H] and h [k][I] (fp64). */
void or_moe_token_wt(int wtype, const uint8_t *w_gate, const uint8_t *w_up, const uint8_t *w_down,
                     const float *gsc, const float *router_w, const float *bias, int H, int I, int E,
                     int k, const uint16_t *x_bf16, int32_t *ids, double *w, float *out32,
                     double *out64, double *h_out) {
    double *x = (double *)malloc(sizeof(double) * (size_t)H);
    double *y = (double *)malloc(sizeof(double) * (size_t)H);
    double *acc = (double *)calloc((size_t)H, sizeof(double));
    for (int c = 0; c < H; ++c) x[c] = or_bf16_to_double(x_bf16[c]);
    or_route_tokens(router_w, bias, x_bf16, 1, E, H, k, ids, w, NULL, NULL);
    int64_t gate_expert_bytes = (int64_t)I * (H / OR_QK) * or_block_bytes(wtype);
    int64_t down_expert_bytes = (int64_t)H * (I / OR_QK) * or_block_bytes(wtype);
    for (int i = 0; i < k; ++i) {
        int e = ids[i];
        or_expert_ffn_wt(wtype, w_gate + e * gate_expert_bytes, w_up + e * gate_expert_bytes,
                         w_down + e * down_expert_bytes, gsc ? gsc[3 * e] : 0.f, gsc ? gsc[3 * e + 1] : 0.f,
                         gsc ? gsc[3 * e + 2] : 0.f, H, I, x, h_out ? h_out + (int64_t)i * I : NULL, y);
        for (int c = 0; c < H; ++c) acc[c] += w[i] * y[c];
    }
    for (int c = 0; c < H; ++c) {
        out32[c] = (float)acc[c];
        if (out64) out64[c] = acc[c];
    }
    free(x);
    free(y);
    free(acc);
}

void or_moe_token(const uint8_t *w_gate, const uint8_t *w_up, const uint8_t *w_down,
                  const float *router_w, const float *bias, int H, int I, int E, int k,
                  const uint16_t *x_bf16, int32_t *ids, double *w, float *out32,
                  double *out64, double *h_out) {
    or_moe_token_wt(OR_WTYPE_Q4_K, w_gate, w_up, w_down, NULL, router_w, bias, H, I, E, k, x_bf16, ids, w,
                    out32, out64, h_out);
}

/* Pre-MoE RMSNorm (the "rmsnorm" kernel of the sparkinfer README's "Layout"
 * table runs before the MoE block of each layer):
 *   xn_c = x_c * gamma_c / sqrt(mean_c(x_c^2) + eps)     (fp64) */
void or_rmsnorm(const uint16_t *x_bf16, const float *gamma, float eps, int H, double *xn) {
    double ss = 0.0;
    for (int c = 0; c < H; ++c) {
        double v = or_bf16_to_double(x_bf16[c]);
        ss += v * v;
    }
    double inv = 1.0 / sqrt(ss / (double)H + (double)eps);
    for (int c = 0; c < H; ++c) xn[c] = or_bf16_to_double(x_bf16[c]) * inv * (double)gamma[c];
}

/* Routing of T tokens of a pre-normed block: as or_route_tokens on
 * rmsnorm(x) (fp64), with the same outputs. */
void or_route_tokens_prenorm(const float *router_w, const float *bias, const float *gamma, float eps,
                             const uint16_t *x_bf16, int T, int E, int H, int k, int32_t *ids,
                             double *w, double *z_out, double *margin) {
    double *xn = (double *)malloc(sizeof(double) * (size_t)H);
    double *z = (double *)malloc(sizeof(double) * (size_t)E);
    float *z32 = (float *)malloc(sizeof(float) * (size_t)E);
    for (int t = 0; t < T; ++t) {
        or_rmsnorm(x_bf16 + (int64_t)t * H, gamma, eps, H, xn);
        for (int e = 0; e < E; ++e) {
            double s = 0.0;
            for (int c = 0; c < H; ++c) s += (double)router_w[(int64_t)e * H + c] * xn[c];
            if (bias) s += (double)bias[e];
            z[e] = s;
            z32[e] = (float)s;
        }
        or_topk(z32, E, k, ids + (int64_t)t * k);
        or_renorm_weights(z, E, ids + (int64_t)t * k, k, w + (int64_t)t * k);
        if (z_out)
            for (int e = 0; e < E; ++e) z_out[(int64_t)t * E + e] = z[e];
        if (margin) margin[t] = or_margin(z, E, k);
    }
    free(xn);
    free(z);
    free(z32);
}

/* One token through the pre-normed MoE block with its residual:
 *   xn  = rmsnorm(x; gamma, eps)
 *   z   = W_r xn (+ bias);  ids, w as in or_moe_token (top-k decided on
 *         the logits rounded to fp32)
 *   out = x + sum_i w_i W_down[e_i] (silu(W_gate[e_i] xn) * W_up[e_i] xn)
 * Outputs: ids [k], w [k], out32 [H] (rounded once), optionally out64 [H]
 * and the fp64 logits z [E]. */
void or_moe_token_prenorm(const uint8_t *w_gate, const uint8_t *w_up, const uint8_t *w_down,
                          const float *router_w, const float *bias, const float *gamma, float eps,
                          int H, int I, int E, int k, const uint16_t *x_bf16, int32_t *ids,
                          double *w, float *out32, double *out64, double *z_out) {
    double *xn = (double *)malloc(sizeof(double) * (size_t)H);
    double *y = (double *)malloc(sizeof(double) * (size_t)H);
    double *acc = (double *)malloc(sizeof(double) * (size_t)H);
    double *z = (double *)malloc(sizeof(double) * (size_t)E);
    float *z32 = (float *)malloc(sizeof(float) * (size_t)E);
    or_rmsnorm(x_bf16, gamma, eps, H, xn);
    for (int e = 0; e < E; ++e) {
        double s = 0.0;
        for (int c = 0; c < H; ++c) s += (double)router_w[(int64_t)e * H + c] * xn[c];
        if (bias) s += (double)bias[e];
        z[e] = s;
        z32[e] = (float)s;
        if (z_out) z_out[e] = s;
    }
    or_topk(z32, E, k, ids);
    or_renorm_weights(z, E, ids, k, w);
    for (int c = 0; c < H; ++c) acc[c] = or_bf16_to_double(x_bf16[c]);  /* the residual */
    int64_t gate_expert_bytes = (int64_t)I * (H / OR_QK) * OR_BLOCK_BYTES;
    int64_t down_expert_bytes = (int64_t)H * (I / OR_QK) * OR_BLOCK_BYTES;
    for (int i = 0; i < k; ++i) {
        int e = ids[i];
        or_expert_ffn(w_gate + e * gate_expert_bytes, w_up + e * gate_expert_bytes,
                      w_down + e * down_expert_bytes, H, I, xn, NULL, y);
        for (int c = 0; c < H; ++c) acc[c] += w[i] * y[c];
    }
    for (int c = 0; c < H; ++c) {
        out32[c] = (float)acc[c];
        if (out64) out64[c] = acc[c];
    }
    free(xn);
    free(y);
    free(acc);
    free(z);
    free(z32);
}

/* Grouped-prefill bookkeeping for T tokens routed top-k (ids [T][k]):
 *   counts[e]   = number of (token, slot) pairs routed to e
 *   offsets[e]  = sum of counts[0..e-1]  (exclusive scan; offsets[E] = T*k)
 *   perm[j]     = pair id p = t*k + slot at position j, ordered by expert
 *                 and, within one expert, by increasing pair id. */
void or_counts_offsets_perm(const int32_t *ids, int T, int k, int E,
                            int32_t *counts, int32_t *offsets, int32_t *perm) {
    int64_t P = (int64_t)T * k;
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (int64_t p = 0; p < P; ++p) counts[ids[p]] += 1;
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    int64_t pos = 0;
    for (int e = 0; e < E; ++e)
        for (int64_t p = 0; p < P; ++p)
            if (ids[p] == e) perm[pos++] = (int32_t)p;
}

/* ---------------------------------------------------------------------
 * int8-activation mode (the "on-read dp4a MMVQ" of the sparkinfer README,
 * "Milestone 1", with the activation quantised once per vector -- "one
 * quantise per activation"): an approximation of the FFN above, defined
 * here step by step so that a kernel taking the same steps can be checked
 * closely, and the approximation itself measured against the exact FFN.
 * The pages give no activation format; this reading takes 32-column blocks
 * (one Q4_K sub-block each):
 *   mx = max_l |v_l| over the block (v the activation as fp32),
 *   inv = fp32(127 / mx) (0 when mx = 0),  q_l = round-half-even(v_l * inv)
 *   (the product taken exactly), so |q_l| <= 127,
 *   d = fp32(mx * fp32(1/127)),  s = sum_l v_l (the exact block sum).
 * A Q4_K row dot over one sub-block j of a block (dsc = d*sc_j, dm = dmin*m_j
 * as fp32 products, c_l the 4-bit codes) is then
 *   dsc * d * sum_l c_l q_l  -  dm * s
 * -- the scale term on the quantised activation, the min term on the exact
 * one.  x is quantised this way; h = silu(g) u is rounded to fp32 and then
 * quantised the same way for the down projection.
 * ------------------------------------------------------------------- */

/* Quantise n (a multiple of 32) fp32 values per 32-value block. */
void or_act8_quant(const float *v, int n, int8_t *q, float *d, double *s) {
    for (int b = 0; b < n / 32; ++b) {
        float mx = 0.f;
        double sum = 0.0;
        for (int l = 0; l < 32; ++l) {
            float a = fabsf(v[32 * b + l]);
            if (a > mx) mx = a;
            sum += (double)v[32 * b + l];
        }
        float inv = mx > 0.f ? 127.0f / mx : 0.f;
        for (int l = 0; l < 32; ++l) q[32 * b + l] = (int8_t)nearbyint((double)v[32 * b + l] * (double)inv);
        d[b] = mx * (1.0f / 127.0f);
        s[b] = sum;
    }
}

/* One Q4_K row of `cols` weights dotted with a quantised activation. */
static double or_q4k_row_dot_act8(const uint8_t *row_blocks, int cols, const int8_t *q, const float *d,
                                  const double *s) {
    double acc = 0.0;
    for (int b = 0; b < cols / OR_QK; ++b) {
        const uint8_t *blk = row_blocks + (int64_t)b * OR_BLOCK_BYTES;
        float dd = (float)or_half_to_double((uint16_t)(blk[0] | (blk[1] << 8)));
        float dmin = (float)or_half_to_double((uint16_t)(blk[2] | (blk[3] << 8)));
        for (int j = 0; j < 8; ++j) {
            int sc, m;
            or_q4k_scale_min(blk + 4, j, &sc, &m);
            float dsc = dd * (float)sc, dm = dmin * (float)m;
            int64_t isum = 0;
            for (int l = 0; l < 32; ++l) {
                uint8_t byte = blk[16 + 32 * (j / 2) + l];
                int c = (j & 1) ? (byte >> 4) : (byte & 15);
                isum += (int64_t)c * q[b * OR_QK + 32 * j + l];
            }
            int sb = b * 8 + j;
            acc += (double)dsc * (double)d[sb] * (double)isum - (double)dm * s[sb];
        }
    }
    return acc;
}

/* One Q4_K expert's FFN in the int8-activation mode (x: the exact activation
 * as fp64, converted to fp32 for the quantisation -- bf16 inputs are exact). */
void or_expert_ffn_act8(const uint8_t *wg, const uint8_t *wu, const uint8_t *wd, int H, int I,
                        const double *x, double *h_out, double *y) {
    float *xf = (float *)malloc(sizeof(float) * (size_t)H);
    int8_t *xq = (int8_t *)malloc((size_t)H);
    float *xd = (float *)malloc(sizeof(float) * (size_t)(H / 32));
    double *xs = (double *)malloc(sizeof(double) * (size_t)(H / 32));
    float *hf = (float *)malloc(sizeof(float) * (size_t)I);
    int8_t *hq = (int8_t *)malloc((size_t)I);
    float *hd = (float *)malloc(sizeof(float) * (size_t)(I / 32));
    double *hs = (double *)malloc(sizeof(double) * (size_t)(I / 32));
    int64_t gate_row_bytes = (int64_t)(H / OR_QK) * OR_BLOCK_BYTES;
    int64_t down_row_bytes = (int64_t)(I / OR_QK) * OR_BLOCK_BYTES;
    for (int c = 0; c < H; ++c) xf[c] = (float)x[c];
    or_act8_quant(xf, H, xq, xd, xs);
    for (int r = 0; r < I; ++r) {
        double g = or_q4k_row_dot_act8(wg + r * gate_row_bytes, H, xq, xd, xs);
        double u = or_q4k_row_dot_act8(wu + r * gate_row_bytes, H, xq, xd, xs);
        double h = or_silu(g) * u;
        if (h_out) h_out[r] = h;
        hf[r] = (float)h;
    }
    or_act8_quant(hf, I, hq, hd, hs);
    for (int c = 0; c < H; ++c) y[c] = or_q4k_row_dot_act8(wd + c * down_row_bytes, I, hq, hd, hs);
    free(xf);
    free(xq);
    free(xd);
    free(xs);
    free(hf);
    free(hq);
    free(hd);
    free(hs);
}

/* The MoE FFN for one token in the int8-activation mode: the routing of
 * or_moe_token (exact logits), the experts by or_expert_ffn_act8. */
void or_moe_token_act8(const uint8_t *w_gate, const uint8_t *w_up, const uint8_t *w_down, const float *router_w,
                       const float *bias, int H, int I, int E, int k, const uint16_t *x_bf16, int32_t *ids,
                       double *w, double *out64) {
    double *x = (double *)malloc(sizeof(double) * (size_t)H);
    double *y = (double *)malloc(sizeof(double) * (size_t)H);
    for (int c = 0; c < H; ++c) {
        x[c] = or_bf16_to_double(x_bf16[c]);
        out64[c] = 0.0;
    }
    or_route_tokens(router_w, bias, x_bf16, 1, E, H, k, ids, w, NULL, NULL);
    int64_t gate_expert_bytes = (int64_t)I * (H / OR_QK) * OR_BLOCK_BYTES;
    int64_t down_expert_bytes = (int64_t)H * (I / OR_QK) * OR_BLOCK_BYTES;
    for (int i = 0; i < k; ++i) {
        int e = ids[i];
        or_expert_ffn_act8(w_gate + e * gate_expert_bytes, w_up + e * gate_expert_bytes,
                           w_down + e * down_expert_bytes, H, I, x, NULL, y);
        for (int c = 0; c < H; ++c) out64[c] += w[i] * y[c];
    }
    free(x);
    free(y);
}
