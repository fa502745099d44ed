/*
 * oracle.c -- plain, slow CPU statement of the FP8 (e4m3) block-scaled linear
 * layer.  TEST INFRASTRUCTURE ONLY: tests/, __graft_entry__.smoke() and the
 * bench's CPU-baseline / reference legs may load it; the product library never
 * does, and this file shares no code, header or table with the CUDA path.
 *
 * Sources (pages on DeepSeek-V3):
 *   [hub/FP8]   "DeepSeek-V3" repository overview (pomoai hub), section
 *               "FP8 混合精度训练：首次在 671B 模型上验证": 128x128 weight blocks
 *               with one fp32 scale each (weight_scale_inv), activations
 *               quantized per token per 128 channels, float8 e4m3, and the
 *               linear() excerpt: act_quant -> fp8_gemm -> (+bias), with
 *               weight_dequant as the bf16 branch.
 *   [blog/FP8]  88811315.cn post on DeepSeek v3, Float8 paragraph: E4M3 only,
 *               fp32 accumulation at a fixed interval of FP8 multiply-adds.
 *   [qd/FP8]    qdgithub overview, section "FP8 量化：存储与计算的平衡":
 *               blockwise FP8 compute, dequantisation on CUDA cores.
 *   E4M3 itself is the OCP 8-bit floating point format "E4M3" (bias 7, no
 *   infinities, S.1111.111 = NaN, largest finite 448); the pages only say
 *   "float8 e4m3".
 *
 * Readings where the pages are silent (the later functions state their own
 * readings beside their code):
 *   R1 e4m3 = OCP E4M3 ("fn"): saturating encode, max 448.
 *   R2 scale s = amax / 448 in fp32 with IEEE round-to-nearest division, and
 *      the stored scale is the dequantisation multiplier (w ~= dec(q) * s).
 *   R3 the value encoded is the fp32 quotient RN32(x / s) (not x * (1/s)).
 *   R4 an all-zero group/block has s = 0 and codes +-0 (sign of the input).
 *   R5 encode = round to nearest, ties to even mantissa, any |v| > 448
 *      (including +-Inf) saturates to +-448, NaN -> 0x7F, sign kept on zero.
 *   R6 the ragged last weight row-block takes its amax over valid rows only.
 *   R7 gemm: per 128-wide K chunk kb the exact partial sum
 *      B_kb = sum_k dec(xq) dec(wq) is scaled by sx[m,kb] * sw[n/128,kb]
 *      and promoted into the running sum; output rounded to bf16 only for
 *      reporting (the GPU result is compared against the fp64 value).
 *
 * Compiled with: gcc -O2 -std=c11 -fPIC -shared -ffp-contract=off
 *                -fno-fast-math  (see oracle/build.py)
 * so that every float operation below is one IEEE binary32 operation.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_BLOCK 128          /* [hub/FP8]: 128x128 weight blocks, 1x128 activation groups */
#define ORC_E4M3_MAX 448.0f    /* OCP E4M3 largest finite magnitude (S.1111.110) */

#ifndef ORC_MUTANT
#define ORC_MUTANT 0           /* >0 plants a deliberate mistake (tests/test_oracle_mutants.py) */
#endif

/* ------------------------------------------------------------------ */
/* bf16 <-> fp32                                                       */
/* ------------------------------------------------------------------ */

/* bf16 is the top half of an fp32 bit pattern, so widening is exact. */
float orc_bf16_to_f32(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* fp32 -> bf16, round to nearest, ties to even (on the dropped 16 bits). */
uint16_t orc_f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) /* NaN: keep sign, quiet */
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lower = u & 0xFFFFu;
    uint32_t upper = u >> 16;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u)))
        upper += 1u; /* carries into the exponent correctly, Inf on overflow */
    return (uint16_t)upper;
}

/* ------------------------------------------------------------------ */
/* E4M3 codec                                                          */
/* ------------------------------------------------------------------ */

/* Decode one code: sign bit 7, exponent bits 6..3 (bias 7), mantissa 2..0.
 * e = 0 is subnormal: m/8 * 2^-6.  S.1111.111 is NaN; there is no Inf. */
double orc_e4m3_decode(uint8_t c) {
    int s = (c >> 7) & 1;
    int e = (c >> 3) & 0xF;
    int m = c & 7;
    double mag;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        mag = ldexp((double)m / 8.0, -6);
    else
        mag = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -mag : mag;
}

/* Encode fp32 -> E4M3 by integer arithmetic on the fp32 bit pattern (R5).
 * The step (quantum) of E4M3 at |v| is 2^(E-3) for a normal E4M3 result with
 * unbiased exponent E >= -6, and 2^-9 below 2^-6 (subnormals). */
uint8_t orc_e4m3_encode(float v) {
    uint32_t u;
    memcpy(&u, &v, 4);
    uint8_t sign = (uint8_t)((u >> 24) & 0x80u);
    uint32_t a = u & 0x7FFFFFFFu;
    if (a > 0x7F800000u)
        return 0x7F;                 /* NaN */
    if (a >= 0x7F800000u)
        return sign | 0x7E;          /* +-Inf saturates */
    if (a < 0x00800000u)
        return sign;                 /* fp32 zero / subnormal: far below 2^-10 */

    int E = (int)(a >> 23) - 127;                /* |v| = sig * 2^(E-23) */
    uint32_t sig = (a & 0x7FFFFFu) | 0x800000u;  /* 24-bit significand */
    int qexp = (E < -6 ? -6 : E) - 3;            /* exponent of the E4M3 step */
    int shift = qexp - (E - 23);                 /* >= 20 */
    uint32_t n;
    if (shift >= 32) {
        n = 0;                                   /* |v| < 2^-33: rounds to 0 */
    } else {
        n = sig >> shift;
        uint32_t rem = sig & ((1u << shift) - 1u);
        uint32_t half = 1u << (shift - 1);
#if ORC_MUTANT == 3
        if (rem >= half) /* mutant: ties away from zero */
            n += 1;
#else
        if (rem > half || (rem == half && (n & 1u)))
            n += 1;                              /* ties to even */
#endif
    }
    if (n == 0)
        return sign;
    if (n == 16) {                               /* rounded up into the next binade */
        n = 8;
        qexp += 1;
    }
    if (qexp == -9 && n < 8)                     /* subnormal: m/8 * 2^-6 */
        return sign | (uint8_t)n;
    int ebits = qexp + 10;                       /* value = (n/8) * 2^(qexp+3), n in [8,16) */
    int mbits = (int)n - 8;
    if (ebits > 15 || (ebits == 15 && mbits == 7))
        return sign | 0x7E;                      /* beyond 448: saturate */
    return sign | (uint8_t)((ebits << 3) | mbits);
}

/* Second, independent encoder: exhaustive nearest search over the 127
 * non-negative finite codes, ties to the even code.  Used only to cross-check
 * orc_e4m3_encode in the tests. */
uint8_t orc_e4m3_encode_search(float v) {
    if (isnan(v))
        return 0x7F;
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs((double)v);
    if (a >= 448.0)
        return sign | 0x7E;
    int best = 0;
    double bestd = a; /* distance to code 0 */
    for (int c = 1; c <= 0x7E; c++) {
        double d = fabs(orc_e4m3_decode((uint8_t)c) - a);
        if (d < bestd || (d == bestd && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            bestd = d;
        }
    }
    return sign | (uint8_t)best;
}

void orc_e4m3_encode_array(const float* v, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; i++)
        out[i] = orc_e4m3_encode(v[i]);
}

void orc_e4m3_encode_search_array(const float* v, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; i++)
        out[i] = orc_e4m3_encode_search(v[i]);
}

/* ------------------------------------------------------------------ */
/* Quantisers                                                          */
/* ------------------------------------------------------------------ */

/* The scale of a group / block from its amax (R2). */
static float orc_scale_from_amax(float amax) {
#if ORC_MUTANT == 1
    return amax / 447.0f; /* mutant: wrong e4m3 maximum */
#else
    return amax / ORC_E4M3_MAX;
#endif
}

/* One element: R3 + R4. */
static uint8_t orc_quantize_one(float x, float amax, float s) {
    if (amax == 0.0f)
        return signbit(x) ? 0x80 : 0x00;
#if ORC_MUTANT == 2
    return orc_e4m3_encode(x * (ORC_E4M3_MAX / amax)); /* mutant: reciprocal multiply */
#else
    return orc_e4m3_encode(x / s);
#endif
}

/* act_quant [hub/FP8]: per row m and per group g of 128 channels,
 * amax = max |x|, s = amax/448, q = e4m3(x/s).
 * x: bf16 bits [M, K] with row stride ldx; xq: [M, K] with row stride ldq;
 * sx: fp32 [M, lds] (group g of row m at sx[m*lds + g]).  K % 128 == 0. */
void orc_act_quant(const uint16_t* x, int64_t M, int64_t K, int64_t ldx,
                   uint8_t* xq, int64_t ldq, float* sx, int64_t lds) {
    int64_t G = K / ORC_BLOCK;
    for (int64_t m = 0; m < M; m++) {
        for (int64_t g = 0; g < G; g++) {
            const uint16_t* xg = x + m * ldx + g * ORC_BLOCK;
            float amax = 0.0f;
            for (int k = 0; k < ORC_BLOCK; k++)
                amax = fmaxf(amax, fabsf(orc_bf16_to_f32(xg[k])));
            float s = orc_scale_from_amax(amax);
            for (int k = 0; k < ORC_BLOCK; k++)
                xq[m * ldq + g * ORC_BLOCK + k] = orc_quantize_one(orc_bf16_to_f32(xg[k]), amax, s);
            sx[m * lds + g] = s;
        }
    }
}

/* weight_quant [hub/FP8]: per 128x128 block (nb, kb) of w [N, K] (row-major,
 * row stride K), amax over the block's valid rows (R6), s = amax/448,
 * q = e4m3(w/s).  sw: fp32 [ceil(N/128), K/128] row-major. */
void orc_weight_quant(const uint16_t* w, int64_t N, int64_t K, uint8_t* wq, float* sw) {
    int64_t NB = (N + ORC_BLOCK - 1) / ORC_BLOCK, KB = K / ORC_BLOCK;
    for (int64_t nb = 0; nb < NB; nb++) {
        int64_t n_end = (nb + 1) * ORC_BLOCK < N ? (nb + 1) * ORC_BLOCK : N;
        for (int64_t kb = 0; kb < KB; kb++) {
            float amax = 0.0f;
            for (int64_t n = nb * ORC_BLOCK; n < n_end; n++)
                for (int64_t k = kb * ORC_BLOCK; k < (kb + 1) * ORC_BLOCK; k++)
                    amax = fmaxf(amax, fabsf(orc_bf16_to_f32(w[n * K + k])));
            float s = orc_scale_from_amax(amax);
            for (int64_t n = nb * ORC_BLOCK; n < n_end; n++)
                for (int64_t k = kb * ORC_BLOCK; k < (kb + 1) * ORC_BLOCK; k++)
                    wq[n * K + k] = orc_quantize_one(orc_bf16_to_f32(w[n * K + k]), amax, s);
            sw[nb * KB + kb] = s;
        }
    }
}

/* weight_dequant [hub/FP8] (the bf16 branch of linear(), and the FP8->BF16
 * checkpoint cast): w = bf16_rne(fp32(dec(q)) * s_block), one fp32 multiply. */
void orc_weight_dequant(const uint8_t* wq, const float* sw, int64_t N, int64_t K, uint16_t* w) {
    int64_t KB = K / ORC_BLOCK;
    for (int64_t n = 0; n < N; n++)
        for (int64_t k = 0; k < K; k++) {
            float q = (float)orc_e4m3_decode(wq[n * K + k]); /* exact in fp32 */
            float s = sw[(n / ORC_BLOCK) * KB + k / ORC_BLOCK];
            w[n * K + k] = orc_f32_to_bf16_rne(q * s);
        }
}

/* ------------------------------------------------------------------ */
/* GEMM                                                                */
/* ------------------------------------------------------------------ */

/* fp8_gemm [hub/FP8] with per-chunk promotion [blog/FP8], R7:
 *   y[m,n] = sum_kb (sx[m,kb] * sw[n/128,kb]) * B_kb[m,n]
 *   B_kb[m,n] = sum_{k in chunk kb} dec(xq[m,k]) * dec(wq[n,k])
 * All in fp64.  Each product of two e4m3 values has <= 8 significant bits and
 * lies in [2^-18, 2^18); 128 of them sum exactly in fp64, and the scale
 * product of two fp32 numbers is exact in fp64.  Also returns
 *   L[m,n] = sum_k |dec(xq[m,k]) sx[m,k/128]| * |dec(wq[n,k]) sw[n/128,k/128]|
 * used by the error bound.  Only the rows listed in `rows` (nrows of them)
 * are computed; y and L are [nrows, N] row-major.
 * Codes are decoded through a table of the 256 decoded values (dec is exact,
 * so the table changes no value).  Built with -fopenmp (liboracle_omp.so, for full-size
 * parity checks) the listed rows are shared out between threads; each output
 * element is still computed by one thread in the order written here. */
void orc_gemm_rows(const uint8_t* xq, int64_t ldq, const float* sx, int64_t lds,
                   const uint8_t* wq, const float* sw,
                   int64_t N, int64_t K, const int64_t* rows, int64_t nrows,
                   double* y, double* L) {
    int64_t KB = K / ORC_BLOCK;
    double dec[256];
    for (int c = 0; c < 256; c++)
        dec[c] = orc_e4m3_decode((uint8_t)c);
#ifdef _OPENMP
#pragma omp parallel
#endif
    {
        double* xd = (double*)malloc(sizeof(double) * (size_t)K);
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int64_t r = 0; r < nrows; r++) {
            int64_t m = rows[r];
            for (int64_t k = 0; k < K; k++)
                xd[k] = dec[xq[m * ldq + k]];
            for (int64_t n = 0; n < N; n++) {
                const uint8_t* wrow = wq + n * K;
                double acc = 0.0, lsum = 0.0;
#if ORC_MUTANT == 5
                int64_t kb_end = KB - 1; /* mutant: last K chunk dropped */
#else
                int64_t kb_end = KB;
#endif
                for (int64_t kb = 0; kb < kb_end; kb++) {
                    double b = 0.0, babs = 0.0;
                    /* b and babs are exact whatever the order of the terms
                     * (see above), so the threaded build may split these two
                     * sums across vector lanes without changing them. */
#ifdef _OPENMP
#pragma omp simd reduction(+ : b, babs)
#endif
                    for (int64_t k = kb * ORC_BLOCK; k < (kb + 1) * ORC_BLOCK; k++) {
                        double p = xd[k] * dec[wrow[k]];
                        b += p;
                        babs += fabs(p);
                    }
#if ORC_MUTANT == 4
                    double scale = (double)sx[m * lds + kb] * (double)sw[kb * ((N + 127) / 128) + n / ORC_BLOCK]; /* mutant: scale grid transposed */
#else
                    double scale = (double)sx[m * lds + kb] * (double)sw[(n / ORC_BLOCK) * KB + kb];
#endif
                    acc += scale * b;
                    lsum += fabs(scale) * babs;
                }
                y[r * N + n] = acc;
                L[r * N + n] = lsum;
            }
        }
        free(xd);
    }
}

/* bias: the pages' linear() adds the bias after fp8_gemm ("DeepSeek-V3"
 * repository overview, section "FP8 混合精度训练", the linear() excerpt:
 * y += bias).  y[r][n] += bf16 value of bias[n], in fp64. */
void orc_add_bias_rows(double* y, int64_t nrows, int64_t N, const uint16_t* bias) {
    for (int64_t r = 0; r < nrows; r++)
        for (int64_t n = 0; n < N; n++)
#if ORC_MUTANT == 6
            y[r * N + n] -= (double)orc_bf16_to_f32(bias[n]); /* mutant: bias subtracted */
#else
            y[r * N + n] += (double)orc_bf16_to_f32(bias[n]);
#endif
}

/* The expert activation between w1/w3 and w2 (the pages' Expert forward,
 * "DeepSeek-V3" repository overview, MoE section: w2(silu(w1(x)) * w3(x))):
 * h = silu(a) * b with silu(v) = v / (1 + exp(-v)), in fp64. */
void orc_swiglu(const double* a, const double* b, int64_t n, double* h) {
    for (int64_t i = 0; i < n; i++) {
#if ORC_MUTANT == 7
        double s = a[i] / (1.0 + exp(a[i])); /* mutant: sign of the exponent flipped */
#else
        double s = a[i] / (1.0 + exp(-a[i]));
#endif
        h[i] = s * b[i];
    }
}

/* grouped_gemm: the same product per expert g over token rows
 * offsets[g] .. offsets[g+1]-1 of xq/sx, with expert weights
 * wq + g*N*K (row-major [N, K]) and scales sw + g*ceil(N/128)*(K/128).
 * Computes the listed global rows (each must lie in some expert's range);
 * rows outside every range are left untouched.  The listed rows of one
 * expert go to orc_gemm_rows together, so each expert's weight is decoded
 * once. */
void orc_grouped_gemm_rows(const uint8_t* xq, int64_t ldq, const float* sx, int64_t lds,
                           const uint8_t* wq, const float* sw, const int32_t* offsets, int32_t G,
                           int64_t N, int64_t K, const int64_t* rows, int64_t nrows,
                           double* y, double* L) {
    int64_t NB = (N + ORC_BLOCK - 1) / ORC_BLOCK, KB = K / ORC_BLOCK;
    int64_t* sel = (int64_t*)malloc(sizeof(int64_t) * (size_t)(nrows > 0 ? nrows : 1));
    int64_t* pos = (int64_t*)malloc(sizeof(int64_t) * (size_t)(nrows > 0 ? nrows : 1));
    for (int32_t g = 0; g < G; g++) {
        int64_t n_sel = 0;
        for (int64_t r = 0; r < nrows; r++)
            if (rows[r] >= offsets[g] && rows[r] < offsets[g + 1]) {
                sel[n_sel] = rows[r];
                pos[n_sel] = r;
                n_sel++;
            }
        if (n_sel == 0)
            continue;
        double* yg = (double*)malloc(sizeof(double) * (size_t)n_sel * (size_t)N);
        double* lg = (double*)malloc(sizeof(double) * (size_t)n_sel * (size_t)N);
        orc_gemm_rows(xq, ldq, sx, lds, wq + (int64_t)g * N * K, sw + (int64_t)g * NB * KB,
                      N, K, sel, n_sel, yg, lg);
        for (int64_t i = 0; i < n_sel; i++) {
            memcpy(y + pos[i] * N, yg + i * N, sizeof(double) * (size_t)N);
            memcpy(L + pos[i] * N, lg + i * N, sizeof(double) * (size_t)N);
        }
        free(yg);
        free(lg);
    }
    free(sel);
    free(pos);
}

/* MoE dispatch: the routed expert computation runs on the token rows
 * gathered expert by expert (page 2 section 2-2: every token keeps its
 * selected experts, none is dropped, so each of a token's top-k selections
 * contributes one row).  Row r of the output is the quantised token
 * token_of_row[r]: its e4m3 codes and its per-128-channel scales, copied
 * unchanged.  A token id outside [0, tokens) yields an all-zero row.
 *   xq [tokens, ldq] e4m3, sx [tokens, lds] fp32 -> xr [R, K], sr [R, K/128]. */
void orc_moe_dispatch(const uint8_t* xq, int64_t ldq, const float* sx, int64_t lds, int64_t tokens,
                      int64_t K, const int32_t* token_of_row, int64_t R, uint8_t* xr, float* sr) {
    int64_t KB = K / ORC_BLOCK;
    for (int64_t r = 0; r < R; r++) {
        int64_t t = token_of_row[r];
        int ok = t >= 0 && t < tokens;
        for (int64_t k = 0; k < K; k++) xr[r * K + k] = ok ? xq[t * ldq + k] : 0;
        for (int64_t kb = 0; kb < KB; kb++)
#if ORC_MUTANT == 9
            sr[r * KB + kb] = ok ? sx[(r % tokens) * lds + kb] : 0.0f; /* mutant: scale of the wrong row */
#else
            sr[r * KB + kb] = ok ? sx[t * lds + kb] : 0.0f;
#endif
    }
}

/* MoE combine: the layer's output for token t is the sum, over its top-k
 * selected experts, of each expert's output weighted by the token's gate
 * value for that expert -- the sigmoid affinity s, not the bias-adjusted
 * score, which only steers the selection (page 2 section 2-2; sigmoid scoring
 * and the route_scale factor 2.5 are in the config block of
 * "671B 参数如何「激活」37B？") -- plus the shared experts' output, which every
 * token receives (page 3, the shared-expert paragraph on DeepSeekMoE):
 *   y[t,d] = z[t,d] + sum_{k<topk} w[r_k] * yk[r_k, d],  r_k = rows_of_token[t,k],
 * in fp64.  L[t,d] = |z[t,d]| + sum_k |w[r_k] yk[r_k,d]| (for error bounds).
 * yk [R, ldyk] fp64 (the expert outputs, one row per routed pair); w [R] the
 * gate value of each row; z [tokens, ldz] fp64 or NULL (= 0).  A row id
 * outside [0, R) contributes nothing. */
void orc_moe_combine(const double* yk, int64_t ldyk, int64_t R, const float* w, const int32_t* rows_of_token,
                     int64_t tokens, int32_t topk, int64_t dim, const double* z, int64_t ldz,
                     double* y, double* L) {
    for (int64_t t = 0; t < tokens; t++) {
        for (int64_t d = 0; d < dim; d++) {
            double acc = z ? z[t * ldz + d] : 0.0;
            double mag = fabs(acc);
#if ORC_MUTANT == 8
            for (int32_t k = 0; k + 1 < topk; k++) { /* mutant: last routed expert dropped */
#else
            for (int32_t k = 0; k < topk; k++) {
#endif
                int64_t r = rows_of_token[t * topk + k];
                if (r < 0 || r >= R) continue;
                double term = (double)w[r] * yk[r * ldyk + d];
                acc += term;
                mag += fabs(term);
            }
            y[t * dim + d] = acc;
            L[t * dim + d] = mag;
        }
    }
}

/* MoE gate (router): sigmoid affinities s = sigmoid(x . wg_e) for the E
 * routed experts (config block of "671B 参数如何「激活」37B？": sigmoid scoring,
 * 8 expert groups of which 4 are kept, top-8 of 256, route_scale 2.5); the
 * per-expert bias steers the selection only (page 2 section 2-2: selection
 * looks at affinity + bias, the FFN output keeps the original gating
 * values).  Readings where the pages are silent: a group's score is the
 * largest biased score in it; ties go to the lower index; the gate values
 * are the selected (unbiased) affinities normalised to sum 1, times
 * route_scale.  All in fp64 from the bf16 inputs.  ids [T, top_k] are the
 * selected experts in descending biased score; w [T, top_k] their gate
 * values; s_out [T, E] (may be NULL) the affinities. */
void orc_moe_gate(const uint16_t* x, const uint16_t* wg, const float* bias, int64_t T, int64_t dim, int32_t E,
                  int32_t n_groups, int32_t topk_groups, int32_t top_k, double route_scale, int32_t* ids,
                  double* w, double* s_out) {
    double* s = (double*)malloc(sizeof(double) * (size_t)E);
    double* b = (double*)malloc(sizeof(double) * (size_t)E);
    int* keep = (int*)malloc(sizeof(int) * (size_t)E);
    double* gscore = (double*)malloc(sizeof(double) * (size_t)n_groups);
    int* gsel = (int*)malloc(sizeof(int) * (size_t)n_groups);
    int32_t per = E / n_groups;
    for (int64_t t = 0; t < T; t++) {
        for (int32_t e = 0; e < E; e++) {
            double acc = 0.0;
            for (int64_t k = 0; k < dim; k++)
                acc += (double)orc_bf16_to_f32(x[t * dim + k]) * (double)orc_bf16_to_f32(wg[(int64_t)e * dim + k]);
            s[e] = 1.0 / (1.0 + exp(-acc));
#if ORC_MUTANT == 10
            b[e] = s[e];                                  /* mutant: the bias ignored in the selection */
#else
            b[e] = s[e] + (double)bias[e];
#endif
            if (s_out) s_out[t * E + e] = s[e];
        }
        for (int32_t g = 0; g < n_groups; g++) {
            double m = -INFINITY;
            for (int32_t i = 0; i < per; i++) if (b[g * per + i] > m) m = b[g * per + i];
            gscore[g] = m;
            gsel[g] = 0;
        }
        for (int32_t r = 0; r < topk_groups; r++) {          /* the best remaining group, lower index on ties */
            int32_t best = -1;
            for (int32_t g = 0; g < n_groups; g++)
                if (!gsel[g] && (best < 0 || gscore[g] > gscore[best])) best = g;
            gsel[best] = 1;
        }
        for (int32_t e = 0; e < E; e++) keep[e] = gsel[e / per];
        double ssum = 0.0;
        for (int32_t r = 0; r < top_k; r++) {                /* the best remaining kept expert */
            int32_t best = -1;
            for (int32_t e = 0; e < E; e++)
                if (keep[e] && (best < 0 || b[e] > b[best])) best = e;
            ids[t * top_k + r] = best;
            keep[best] = 0;
            ssum += s[best];
        }
        for (int32_t r = 0; r < top_k; r++)
#if ORC_MUTANT == 11
            w[t * top_k + r] = s[ids[t * top_k + r]] * route_scale; /* mutant: not normalised */
#else
            w[t * top_k + r] = s[ids[t * top_k + r]] / ssum * route_scale;
#endif
    }
    free(s); free(b); free(keep); free(gscore); free(gsel);
}

/* MoE routing tables: the (token, k) selections grouped by expert, tokens
 * in order within an expert (a stable counting sort), so that each expert's
 * rows are contiguous for the grouped GEMM:
 *   offsets [E+1]: rows of expert e are offsets[e] .. offsets[e+1]-1
 *   token_of_row [T*top_k], weight_of_row [T*top_k] (the pair's gate value),
 *   rows_of_token [T, top_k]: the routed row of selection (t, k). */
void orc_moe_route(const int32_t* ids, const float* w, int64_t T, int32_t top_k, int32_t E, int32_t* offsets,
                   int32_t* token_of_row, int32_t* rows_of_token, float* weight_of_row) {
    int32_t* next = (int32_t*)calloc((size_t)E + 1, sizeof(int32_t));
    for (int32_t e = 0; e <= E; e++) offsets[e] = 0;
    for (int64_t i = 0; i < T * top_k; i++) offsets[ids[i] + 1]++;
    for (int32_t e = 0; e < E; e++) offsets[e + 1] += offsets[e];
    for (int32_t e = 0; e < E; e++) next[e] = offsets[e];
#if ORC_MUTANT == 12
    for (int64_t t = T - 1; t >= 0; t--) {                  /* mutant: tokens in reverse within an expert */
#else
    for (int64_t t = 0; t < T; t++) {
#endif
        for (int32_t k = 0; k < top_k; k++) {
            int32_t e = ids[t * top_k + k];
            int32_t r = next[e]++;
            token_of_row[r] = (int32_t)t;
            rows_of_token[t * top_k + k] = r;
            weight_of_row[r] = w[t * top_k + k];
        }
    }
    free(next);
}

/* Power-of-two scales: the pages pass a scale format (scale_fmt) to
 * act_quant without defining it ("DeepSeek-V3" repository overview, the
 * linear() excerpt).  Reading: a UE8M0-style scale, an unsigned power of two
 * with no mantissa, rounded up so that nothing saturates -- s = 2^e with e
 * the smallest integer such that amax <= 448 * 2^e; then x / s is exact and
 * q = e4m3(x / s) only rounds.  An all-zero group or block has s = 0 (R4). */
static float orc_pow2_scale(float amax) {
    if (amax == 0.0f)
        return 0.0f;
    int e;
    frexp((double)amax / 448.0, &e);        /* 2^(e-1) <= amax/448 < 2^e, up to rounding */
    e -= 2;                                 /* step up from below with exact comparisons */
    while (ldexp(448.0, e) < (double)amax) e++;
#if ORC_MUTANT == 16
    e -= 1;                                 /* mutant: rounded down (the top codes saturate) */
#endif
    return (float)ldexp(1.0, e);
}

/* act_quant with power-of-two scales; layout as orc_act_quant. */
void orc_act_quant_pow2(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, uint8_t* xq, int64_t ldq, float* sx,
                        int64_t lds) {
    int64_t G = K / ORC_BLOCK;
    for (int64_t m = 0; m < M; m++) {
        for (int64_t g = 0; g < G; g++) {
            const uint16_t* xg = x + m * ldx + g * ORC_BLOCK;
            float amax = 0.0f;
            for (int k = 0; k < ORC_BLOCK; k++) amax = fmaxf(amax, fabsf(orc_bf16_to_f32(xg[k])));
            float s = orc_pow2_scale(amax);
            for (int k = 0; k < ORC_BLOCK; k++) {
                float v = orc_bf16_to_f32(xg[k]);
                xq[m * ldq + g * ORC_BLOCK + k] = amax == 0.0f ? (signbit(v) ? 0x80 : 0x00) : orc_e4m3_encode(v / s);
            }
            sx[m * lds + g] = s;
        }
    }
}

/* weight_quant with power-of-two scales: per 128x128 block (the ragged last
 * row block over its valid rows, R6) s = 2^e as above, q = e4m3(w / s).
 * Layout as orc_weight_quant. */
void orc_weight_quant_pow2(const uint16_t* w, int64_t N, int64_t K, uint8_t* wq, float* sw) {
    int64_t NB = (N + ORC_BLOCK - 1) / ORC_BLOCK, KB = K / ORC_BLOCK;
    for (int64_t nb = 0; nb < NB; nb++) {
        int64_t n_end = (nb + 1) * ORC_BLOCK < N ? (nb + 1) * ORC_BLOCK : N;
        for (int64_t kb = 0; kb < KB; kb++) {
            float amax = 0.0f;
            for (int64_t n = nb * ORC_BLOCK; n < n_end; n++)
                for (int64_t k = kb * ORC_BLOCK; k < (kb + 1) * ORC_BLOCK; k++)
                    amax = fmaxf(amax, fabsf(orc_bf16_to_f32(w[n * K + k])));
            float s = orc_pow2_scale(amax);
            for (int64_t n = nb * ORC_BLOCK; n < n_end; n++)
                for (int64_t k = kb * ORC_BLOCK; k < (kb + 1) * ORC_BLOCK; k++) {
                    float v = orc_bf16_to_f32(w[n * K + k]);
                    wq[n * K + k] = amax == 0.0f ? (signbit(v) ? 0x80 : 0x00) : orc_e4m3_encode(v / s);
                }
            sw[nb * KB + kb] = s;
        }
    }
}

/* ------------------------------------------------------------------ */
/* Backward GEMMs (training)                                           */
/* ------------------------------------------------------------------ */
/* The pages run training in E4M3 in both directions, with block-wise
 * scaling (88811315.cn post, the Float8 paragraph: E4M3 for forward and
 * backward alike, instead of E5M2 for gradients), but give no granularity
 * for the backward GEMMs.  Reading taken: every operand is grouped in 128s
 * along the contraction dimension of the GEMM it feeds, so each 128-wide
 * chunk of a dot product carries one scale per row and one per column -- the
 * forward's structure -- and the weight keeps its 128x128 blocks.
 *   dgrad  dX = dY W      (contraction over N): dY in 1x128 groups along N
 *                         (act_quant applied to dY), W's blocks reused.
 *   wgrad  dW = dY^T X    (contraction over the tokens M): dY and X in 128x1
 *                         groups along M (act_quant_cols).               */

/* act_quant_cols: per column k and per block mb of 128 rows (the last block
 * may be ragged: amax over its valid rows, as R6), amax = max |x|,
 * s = amax/448, q = e4m3(x/s).  x: bf16 bits [M, K] row stride ldx; xq [M, K]
 * row stride ldq; sx fp32 [ceil(M/128), K] row-major (block mb, column k at
 * sx[mb*K + k]). */
void orc_act_quant_cols(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, uint8_t* xq, int64_t ldq, float* sx) {
    int64_t MB = (M + ORC_BLOCK - 1) / ORC_BLOCK;
    for (int64_t mb = 0; mb < MB; mb++) {
        int64_t m0 = mb * ORC_BLOCK, m1 = m0 + ORC_BLOCK < M ? m0 + ORC_BLOCK : M;
#if ORC_MUTANT == 13
        int64_t m_amax = m1 - 1 > m0 ? m1 - 1 : m1;   /* mutant: the block's last row left out of the amax */
#else
        int64_t m_amax = m1;
#endif
        for (int64_t k = 0; k < K; k++) {
            float amax = 0.0f;
            for (int64_t m = m0; m < m_amax; m++) amax = fmaxf(amax, fabsf(orc_bf16_to_f32(x[m * ldx + k])));
            float s = orc_scale_from_amax(amax);
            for (int64_t m = m0; m < m1; m++) xq[m * ldq + k] = orc_quantize_one(orc_bf16_to_f32(x[m * ldx + k]), amax, s);
            sx[mb * K + k] = s;
        }
    }
}

/* dgrad: dX[m,k] = sum_nb sdy[m,nb] * sw[nb, k/128] * B_nb[m,k],
 *   B_nb[m,k] = sum_{n in chunk nb} dec(dyq[m,n]) * dec(wq[n,k]),
 * exact fp64 per chunk as in orc_gemm_rows.  dyq [M, N] row stride ldq,
 * sdy [M, lds] (1x128 groups along N), wq [N, K], sw [ceil(N/128), K/128];
 * N % 128 == 0.  Only the listed rows; dx and L are [nrows, K]. */
void orc_gemm_dgrad_rows(const uint8_t* dyq, int64_t ldq, const float* sdy, int64_t lds, const uint8_t* wq,
                         const float* sw, int64_t N, int64_t K, const int64_t* rows, int64_t nrows, double* dx,
                         double* L) {
    int64_t NB = N / ORC_BLOCK, KB = K / ORC_BLOCK;
    double* dyd = (double*)malloc(sizeof(double) * (size_t)N);
    for (int64_t r = 0; r < nrows; r++) {
        int64_t m = rows[r];
        for (int64_t n = 0; n < N; n++) dyd[n] = orc_e4m3_decode(dyq[m * ldq + n]);
        for (int64_t k = 0; k < K; k++) {
            double acc = 0.0, lsum = 0.0;
            for (int64_t nb = 0; nb < NB; nb++) {
                double b = 0.0, babs = 0.0;
                for (int64_t n = nb * ORC_BLOCK; n < (nb + 1) * ORC_BLOCK; n++) {
                    double p = dyd[n] * orc_e4m3_decode(wq[n * K + k]);
                    b += p;
                    babs += fabs(p);
                }
#if ORC_MUTANT == 14
                double scale = (double)sdy[m * lds + nb] * (double)sw[(k / ORC_BLOCK) * NB + nb]; /* mutant: the weight's block grid read as if stored transposed */
#else
                double scale = (double)sdy[m * lds + nb] * (double)sw[nb * KB + k / ORC_BLOCK];
#endif
                acc += scale * b;
                lsum += fabs(scale) * babs;
            }
            dx[r * K + k] = acc;
            L[r * K + k] = lsum;
        }
    }
    free(dyd);
}

/* wgrad: dW[n,k] = sum_mb sdy[mb,n] * sx[mb,k] * B_mb[n,k],
 *   B_mb[n,k] = sum_{m in block mb} dec(dyq[m,n]) * dec(xq[m,k]),
 * exact fp64 per block (a block holds at most 128 products).  dyq [M, N]
 * row stride ldd, sdy [ceil(M/128), N]; xq [M, K] row stride ldx,
 * sx [ceil(M/128), K] (both from orc_act_quant_cols); the last block of
 * tokens may be ragged.  Only the listed rows n of dW are computed; dw and
 * L are [nrows, K].  Each element's sums run over m in ascending order as
 * written; the loop over k is innermost only so that xq is read along its
 * rows (the order of the terms of any one element is unchanged).  Built
 * with -fopenmp the listed rows are shared out between threads. */
void orc_gemm_wgrad_rows(const uint8_t* dyq, int64_t ldd, const float* sdy, const uint8_t* xq, int64_t ldx,
                         const float* sx, int64_t M, int64_t N, int64_t K, const int64_t* rows, int64_t nrows,
                         double* dw, double* L) {
    int64_t MB = (M + ORC_BLOCK - 1) / ORC_BLOCK;
#if ORC_MUTANT == 15
    if (M % ORC_BLOCK) MB -= 1; /* mutant: a ragged last block of tokens dropped */
#endif
    double dec[256];
    for (int c = 0; c < 256; c++)
        dec[c] = orc_e4m3_decode((uint8_t)c);
#ifdef _OPENMP
#pragma omp parallel
#endif
    {
        double* b = (double*)malloc(sizeof(double) * (size_t)K * 2);
        double* babs = b + K;
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int64_t r = 0; r < nrows; r++) {
            int64_t n = rows[r];
            double* acc = dw + r * K;
            double* lsum = L + r * K;
            for (int64_t k = 0; k < K; k++) {
                acc[k] = 0.0;
                lsum[k] = 0.0;
            }
            for (int64_t mb = 0; mb < MB; mb++) {
                int64_t m0 = mb * ORC_BLOCK, m1 = m0 + ORC_BLOCK < M ? m0 + ORC_BLOCK : M;
                for (int64_t k = 0; k < K; k++) {
                    b[k] = 0.0;
                    babs[k] = 0.0;
                }
                for (int64_t m = m0; m < m1; m++) {
                    double dy = dec[dyq[m * ldd + n]];
                    const uint8_t* xr = xq + m * ldx;
                    for (int64_t k = 0; k < K; k++) {
                        double p = dy * dec[xr[k]];
                        b[k] += p;
                        babs[k] += fabs(p);
                    }
                }
                for (int64_t k = 0; k < K; k++) {
                    double scale = (double)sdy[mb * N + n] * (double)sx[mb * K + k];
                    acc[k] += scale * b[k];
                    lsum[k] += fabs(scale) * babs[k];
                }
            }
        }
        free(b);
    }
}

/* wgrad over every row n: dw and L are [N, K]. */
void orc_gemm_wgrad(const uint8_t* dyq, int64_t ldd, const float* sdy, const uint8_t* xq, int64_t ldx,
                    const float* sx, int64_t M, int64_t N, int64_t K, double* dw, double* L) {
    int64_t* rows = (int64_t*)malloc(sizeof(int64_t) * (size_t)(N > 0 ? N : 1));
    for (int64_t n = 0; n < N; n++)
        rows[n] = n;
    orc_gemm_wgrad_rows(dyq, ldd, sdy, xq, ldx, sx, M, N, K, rows, N, dw, L);
    free(rows);
}

int orc_mutant_id(void) { return ORC_MUTANT; }
