/*
 * CPU oracle for the W4A4 + LoRA quantized linear layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Tests, the smoke check and the CPU-baseline leg
 * of the benchmark call this file; the product path never does.  It shares no
 * code, header, table or constant with the CUDA library.
 *
 * Plain, single-threaded, loop-by-loop code: every function is the definition
 * of one step written out, accumulating in int64 (integer products) or fp64
 * (everything scaled).  Build with -ffp-contract=off and without fast-math so
 * that every float operation is one IEEE binary32 operation with
 * round-to-nearest-even.
 *
 * What it computes (page citations by page title and section):
 *   Y[m,n] = colscale[n] * ( sum_g sA[m,g] sW[n,g] P[m,n,g]
 *                            + sum_j D[m,j] L_up[j,n] ) + bias[n]
 *   P[m,n,g] = sum_{k in group g} qA[m,k] qW[n,k]          (exact integers)
 *   D[m,j]   = sum_k X[m,k] L_down[k,j]                    (unquantised X)
 * - activation quantiser: "W4A4 CUDA Kernel for Voice Clone", 3.6
 *   (fused_quantize_repack_act_kernel): absmax per 64-column group,
 *   scale = max(absmax/7, 1e-10), q = clamp(round-half-even(x/scale), -8, 7);
 * - weight quantiser: same post, 2.1 and 2.3 (round(W/scale), fp16
 *   per-group-64 scales);
 * - per-group integer products, scaled per group and summed: same post, 3.7;
 * - LoRA down from the unquantised X, LoRA up added to the same output
 *   accumulator: same post, 3.6 and 3.7;
 * - column-wise affine after the low-rank residual: "High-Performance Kernel
 *   Design for W4A4 ... on Blackwell Architecture", section 1.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define OR_GROUP 64

/* ---- fp16 <-> fp32, written from the IEEE 754 binary16 definition ------ */

/* binary16 bits -> value (exact). */
float oracle_f16_to_f32(uint16_t h) {
    int s = h >> 15, e = (h >> 10) & 31, m = h & 1023;
    double v;
    if (e == 0) v = ldexp((double)m, -24);                 /* subnormal / zero */
    else if (e == 31) v = m ? NAN : INFINITY;
    else v = ldexp((double)(m + 1024), e - 25);             /* (1.m) 2^(e-15) */
    return (float)(s ? -v : v);
}

/* value -> nearest binary16, ties to even (overflow to infinity). */
uint16_t oracle_f32_to_f16(float f) {
    uint32_t x;
    memcpy(&x, &f, 4);
    uint16_t sign = (uint16_t)((x >> 16) & 0x8000u);
    uint32_t ax = x & 0x7fffffffu;
    if (ax > 0x7f800000u) return (uint16_t)(sign | 0x7e00u);   /* NaN */
    if (ax == 0x7f800000u) return (uint16_t)(sign | 0x7c00u);  /* inf */
    double v = fabs((double)f);
    if (v >= 65520.0) return (uint16_t)(sign | 0x7c00u);      /* past 65504 + half a step */
    int e2;
    frexp(v, &e2);                        /* v in [2^(e2-1), 2^e2) */
    int be = e2 - 1;
    if (v == 0.0 || be < -14) be = -14;   /* subnormals share the smallest binade's step */
    double quantum = ldexp(1.0, be - 10); /* spacing of binary16 numbers there */
    double n = rint(v / quantum);         /* exact scaling; rint ties to even */
    uint32_t bits;
    if (be == -14 && n < 1024.0) {
        bits = (uint32_t)n;               /* subnormal or zero */
    } else {
        if (n == 2048.0) { be += 1; n = 1024.0; }
        bits = ((uint32_t)(be + 15) << 10) | ((uint32_t)n - 1024u);
    }
    return (uint16_t)(sign | bits);
}

/* double value -> nearest binary16, ties to even, in one rounding (no detour
 * through binary32, which could round twice). */
uint16_t oracle_f64_to_f16(double d) {
    if (isnan(d)) return (uint16_t)0x7e00u;
    uint16_t sign = signbit(d) ? 0x8000u : 0u;
    double v = fabs(d);
    if (v >= 65520.0) return (uint16_t)(sign | 0x7c00u);      /* past 65504 + half a step */
    int e2;
    frexp(v, &e2);
    int be = e2 - 1;
    if (v == 0.0 || be < -14) be = -14;
    double quantum = ldexp(1.0, be - 10);
    double n = rint(v / quantum);         /* v / quantum is exact (power-of-two scaling) */
    uint32_t bits;
    if (be == -14 && n < 1024.0) {
        bits = (uint32_t)n;
    } else {
        if (n == 2048.0) { be += 1; n = 1024.0; }
        bits = ((uint32_t)(be + 15) << 10) | ((uint32_t)n - 1024u);
    }
    return (uint16_t)(sign | bits);
}

void oracle_f64_to_f16_array(const double* d, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f64_to_f16(d[i]);
}

/* ---- RMSNorm glue of a stack of linears (Voice Clone post, 3.9), unit gain.
 * For each row m of Y (fp16 bits, row stride ld) over its first K columns:
 *   X[m, k] = fp16( Y[m, k] / sqrt( (sum_k Y[m, k]^2) / K + eps ) ),
 * the sum of squares in double (each square of a binary16 value is exact),
 * 1/sqrt(.) in double, one rounding to binary16 at the end.                  */
void oracle_rmsnorm_f16(const uint16_t* Y, int64_t M, int64_t ld, int64_t K, double eps, uint16_t* X) {
    for (int64_t m = 0; m < M; ++m) {
        const uint16_t* y = Y + m * ld;
        double ss = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double v = (double)oracle_f16_to_f32(y[k]);
            ss += v * v;
        }
        double inv = 1.0 / sqrt(ss / (double)K + eps);
        for (int64_t k = 0; k < K; ++k) X[m * K + k] = oracle_f64_to_f16((double)oracle_f16_to_f32(y[k]) * inv);
    }
}

static int8_t clamp_code(float q) {
    if (q < -8.0f) q = -8.0f;
    if (q > 7.0f) q = 7.0f;
    return (int8_t)q;
}

/* ---- activation quantiser (Voice Clone post, 3.6) ------------------------
 * X: fp16 bits [M, K]; qA: int8 codes [M, K]; sA: fp32 [M, K/64].          */
void oracle_quantize_act(const uint16_t* X, int64_t M, int64_t K, int8_t* qA, float* sA) {
    int64_t G = K / OR_GROUP;
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t g = 0; g < G; ++g) {
            const uint16_t* x = X + m * K + g * OR_GROUP;
            float amax = 0.0f;
            for (int k = 0; k < OR_GROUP; ++k) {
                float v = fabsf(oracle_f16_to_f32(x[k]));
                if (v > amax) amax = v;
            }
            float s = amax / 7.0f;
            if (s < 1e-10f) s = 1e-10f;
            sA[m * G + g] = s;
            for (int k = 0; k < OR_GROUP; ++k)
                qA[m * K + g * OR_GROUP + k] = clamp_code(rintf(oracle_f16_to_f32(x[k]) / s));
        }
    }
}

/* ---- weight quantiser (Voice Clone post, 2.1 / 2.3) ----------------------
 * W: fp32 [N, K]; qW: int8 codes [N, K]; sW: fp16 bits [N, K/64].
 * The scale is absmax/7 rounded to fp16 and floored at 2^-14 (the smallest
 * normal fp16); codes are taken against the stored fp16 scale.             */
void oracle_quantize_weights(const float* W, int64_t N, int64_t K, int8_t* qW, uint16_t* sW) {
    int64_t G = K / OR_GROUP;
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t g = 0; g < G; ++g) {
            const float* w = W + n * K + g * OR_GROUP;
            float amax = 0.0f;
            for (int k = 0; k < OR_GROUP; ++k) {
                float v = fabsf(w[k]);
                if (v > amax) amax = v;
            }
            float s32 = amax / 7.0f;
            if (s32 < 0x1p-14f) s32 = 0x1p-14f;
            uint16_t h = oracle_f32_to_f16(s32);
            sW[n * G + g] = h;
            float s = oracle_f16_to_f32(h);
            for (int k = 0; k < OR_GROUP; ++k)
                qW[n * K + g * OR_GROUP + k] = clamp_code(rintf(w[k] / s));
        }
    }
}

/* ---- per-group integer dot products (Voice Clone post, 3.7 phase 1) -----
 * P[m, n, g] = sum over the 64 k of group g of qA[m,k] qW[n,k].  Returns the
 * number of partials that do not fit int32 (always 0 for 4-bit codes).     */
int64_t oracle_group_partials(const int8_t* qA, const int8_t* qW, int64_t M, int64_t N, int64_t K,
                              int32_t* P) {
    int64_t G = K / OR_GROUP, bad = 0;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n)
            for (int64_t g = 0; g < G; ++g) {
                int64_t acc = 0;
                for (int k = 0; k < OR_GROUP; ++k)
                    acc += (int64_t)qA[m * K + g * OR_GROUP + k] * (int64_t)qW[n * K + g * OR_GROUP + k];
                if (acc > INT32_MAX || acc < INT32_MIN) ++bad;
                P[(m * N + n) * G + g] = (int32_t)acc;
            }
    return bad;
}

/* ---- LoRA down-projection from the unquantised X (3.6, LoRA branch) -----
 * D[m, j] = sum_k X[m,k] L_down[k,j] in fp64.                              */
void oracle_lora_down(const uint16_t* X, const uint16_t* Ld, int64_t M, int64_t K, int64_t r, double* D) {
    for (int64_t m = 0; m < M; ++m)
        for (int64_t j = 0; j < r; ++j) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += (double)oracle_f16_to_f32(X[m * K + k]) * (double)oracle_f16_to_f32(Ld[k * r + j]);
            D[m * r + j] = acc;
        }
}

/* ---- output of one element from quantised operands ----------------------
 * main = sum_g sA sW P ; lora = sum_j D L_up ; y = cs (main + lora) + bias. */
static double output_element(const int8_t* qa_row, const float* sa_row, const int8_t* qw_row,
                             const uint16_t* sw_row, const double* d_row, const uint16_t* Lup,
                             int64_t n, int64_t N, int64_t K, int64_t r, uint16_t cs, uint16_t bias) {
    int64_t G = K / OR_GROUP;
    double main_sum = 0.0;
    for (int64_t g = 0; g < G; ++g) {
        int64_t p = 0;
        for (int k = 0; k < OR_GROUP; ++k)
            p += (int64_t)qa_row[g * OR_GROUP + k] * (int64_t)qw_row[g * OR_GROUP + k];
        main_sum += (double)sa_row[g] * (double)oracle_f16_to_f32(sw_row[g]) * (double)p;
    }
    double lora = 0.0;
    for (int64_t j = 0; j < r; ++j) lora += d_row[j] * (double)oracle_f16_to_f32(Lup[j * N + n]);
    return (double)oracle_f16_to_f32(cs) * (main_sum + lora) + (double)oracle_f16_to_f32(bias);
}

/* Y (fp64) from already-quantised operands and D (all [row-major]). */
void oracle_linear_from_codes(const int8_t* qA, const float* sA, const int8_t* qW, const uint16_t* sW,
                              const double* D, const uint16_t* Lup, const uint16_t* cs,
                              const uint16_t* bias, int64_t M, int64_t N, int64_t K, int64_t r,
                              double* Y) {
    int64_t G = K / OR_GROUP;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n)
            Y[m * N + n] = output_element(qA + m * K, sA + m * G, qW + n * K, sW + n * G, D + m * r, Lup,
                                          n, N, K, r, cs[n], bias[n]);
}

/* Selected outputs (rows[i], cols[i]) of the full layer, from the raw inputs.
 * Quantises only the rows and columns it needs: used at sizes where the whole
 * product is too slow for a single CPU thread.                              */
void oracle_linear_sampled(const uint16_t* X, const float* W, const uint16_t* Ld, const uint16_t* Lup,
                           const uint16_t* cs, const uint16_t* bias, int64_t M, int64_t N, int64_t K,
                           int64_t r, const int64_t* rows, const int64_t* cols, int64_t ns,
                           int8_t* qa_buf /*K*/, float* sa_buf /*K/64*/, int8_t* qw_buf /*K*/,
                           uint16_t* sw_buf /*K/64*/, double* d_buf /*r*/, double* out) {
    (void)M;
    int64_t last_row = -1, last_col = -1;
    for (int64_t i = 0; i < ns; ++i) {
        int64_t m = rows[i], n = cols[i];
        if (m != last_row) {
            oracle_quantize_act(X + m * K, 1, K, qa_buf, sa_buf);
            if (r > 0) oracle_lora_down(X + m * K, Ld, 1, K, r, d_buf);
            last_row = m;
        }
        if (n != last_col) {
            oracle_quantize_weights(W + n * K, 1, K, qw_buf, sw_buf);
            last_col = n;
        }
        out[i] = output_element(qa_buf, sa_buf, qw_buf, sw_buf, d_buf, Lup, n, N, K, r, cs[n], bias[n]);
    }
}

/* ---- W4A16: fp16 activations against the same INT4 weights -------------
 * "INT4 Kernel Architecture, in depth", "W4A16 versus W4A4": the activations
 * stay in fp16 and only the weights are 4-bit, dequantised per group:
 *   Y[m,n] = colscale[n] * ( sum_k X[m,k] * qW[n,k] * sW[n,g(k)]
 *                            + sum_j D[m,j] L_up[j,n] ) + bias[n]
 * with the same weight quantiser, LoRA and column affine as the W4A4 layer.
 * Every product X * q * s is exact in fp64 (11 + 4 + 11 significant bits). */
void oracle_w4a16_from_codes(const uint16_t* X, const int8_t* qW, const uint16_t* sW, const double* D,
                             const uint16_t* Lup, const uint16_t* cs, const uint16_t* bias, int64_t M,
                             int64_t N, int64_t K, int64_t r, double* Y) {
    int64_t G = K / OR_GROUP;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double main_sum = 0.0;
            for (int64_t g = 0; g < G; ++g) {
                double s = (double)oracle_f16_to_f32(sW[n * G + g]);
                for (int k = 0; k < OR_GROUP; ++k) {
                    int64_t kk = g * OR_GROUP + k;
                    main_sum += (double)oracle_f16_to_f32(X[m * K + kk]) * (double)qW[n * K + kk] * s;
                }
            }
            double lora = 0.0;
            for (int64_t j = 0; j < r; ++j) lora += D[m * r + j] * (double)oracle_f16_to_f32(Lup[j * N + n]);
            Y[m * N + n] = (double)oracle_f16_to_f32(cs[n]) * (main_sum + lora) + (double)oracle_f16_to_f32(bias[n]);
        }
}

/* ---- asymmetric 4-bit weights with a zero point, groups of 128 ---------
 * "INT4 Kernel Architecture, in depth", "How the weights are stored": one fp16
 * scale and one zero point per group of 128 input channels of an output row,
 * codes 0..15, value = (q - zero) * scale.  Per row n and group g, in IEEE
 * binary32 with round-to-nearest-even:
 *   lo = min w, hi = max w;  scale = max(hi - lo, 1e-8) / 15;
 *   zero = rint(-lo / scale);  q = clamp(rint(w / scale + zero), 0, 15);
 * then scale is stored rounded to fp16 and zero as fp16 (exact: an integer;
 * a zero point of 0 is stored as +0, whichever sign the rounding gave).
 * W fp32 [N, K]; q uint8 [N, K]; scale, zero fp16 bits [N, K/128].          */
#define OR_GROUP_ASYM 128
void oracle_quantize_weights_asym(const float* W, int64_t N, int64_t K, uint8_t* q, uint16_t* scale,
                                  uint16_t* zero) {
    int64_t G = K / OR_GROUP_ASYM;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t g = 0; g < G; ++g) {
            const float* w = W + n * K + g * OR_GROUP_ASYM;
            float lo = w[0], hi = w[0];
            for (int k = 1; k < OR_GROUP_ASYM; ++k) {
                if (w[k] < lo) lo = w[k];
                if (w[k] > hi) hi = w[k];
            }
            float range = hi - lo;
            if (range < 1e-8f) range = 1e-8f;
            const float s = range / 15.0f;
            const float z = rintf(-lo / s) + 0.0f; /* an integer; +0 rather than -0 when it is zero */
            for (int k = 0; k < OR_GROUP_ASYM; ++k) {
                float v = rintf(w[k] / s + z);
                if (v < 0.0f) v = 0.0f;
                if (v > 15.0f) v = 15.0f;
                q[n * K + g * OR_GROUP_ASYM + k] = (uint8_t)v;
            }
            scale[n * G + g] = oracle_f32_to_f16(s);
            zero[n * G + g] = oracle_f32_to_f16(z);
        }
}

/* W4A16 layer with those weights: fp16 X against (q - zero) * scale,
 *   Y[m,n] = colscale[n] * ( sum_k X[m,k] (q[n,k] - zero[n,g(k)]) scale[n,g(k)]
 *                            + sum_j D[m,j] L_up[j,n] ) + bias[n]
 * in fp64 (each product exact: 11 + 12 + 11 significant bits).              */
void oracle_w4a16_asym_from_codes(const uint16_t* X, const uint8_t* q, const uint16_t* scale, const uint16_t* zero,
                                  const double* D, const uint16_t* Lup, const uint16_t* cs, const uint16_t* bias,
                                  int64_t M, int64_t N, int64_t K, int64_t r, double* Y) {
    int64_t G = K / OR_GROUP_ASYM;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double main_sum = 0.0;
            for (int64_t g = 0; g < G; ++g) {
                double s = (double)oracle_f16_to_f32(scale[n * G + g]);
                double z = (double)oracle_f16_to_f32(zero[n * G + g]);
                for (int k = 0; k < OR_GROUP_ASYM; ++k) {
                    int64_t kk = g * OR_GROUP_ASYM + k;
                    main_sum += (double)oracle_f16_to_f32(X[m * K + kk]) * ((double)q[n * K + kk] - z) * s;
                }
            }
            double lora = 0.0;
            for (int64_t j = 0; j < r; ++j) lora += D[m * r + j] * (double)oracle_f16_to_f32(Lup[j * N + n]);
            Y[m * N + n] = (double)oracle_f16_to_f32(cs[n]) * (main_sum + lora) + (double)oracle_f16_to_f32(bias[n]);
        }
}

/* ---- SiLU(gate) * up on a fused gate|up output ----------------------------
 * "W4A4 CUDA Kernel for Voice Clone", 1 (the decoder layer's MLP: gate_proj
 * and up_proj, then SiLU(gate) x up into down_proj).  Y fp64 [M, 2I] holds the
 * gate outputs in columns 0..I-1 and the up outputs in I..2I-1;
 *   H[m, j] = silu(Y[m, j]) * Y[m, I + j],   silu(v) = v / (1 + exp(-v)),
 * in fp64.                                                                  */
void oracle_silu_mul(const double* Y, int64_t M, int64_t I, double* H) {
    for (int64_t m = 0; m < M; ++m)
        for (int64_t j = 0; j < I; ++j) {
            double g = Y[m * 2 * I + j], u = Y[m * 2 * I + I + j];
            H[m * I + j] = g / (1.0 + exp(-g)) * u;
        }
}

/* ---- whole output rows of the layer from the raw inputs -------------------
 * Y[rows[i], n] for every n, fp64, [nrows, N]: the weights are quantised once
 * (qW_buf [N, K], sW_buf [N, K/64]) and each listed row of X is quantised and
 * projected on its own, then every output element is the definition above.
 * For parity at sizes where the whole product is too slow on one CPU thread
 * but every output column (every output tile) must be reached.             */
void oracle_linear_rows(const uint16_t* X, const float* W, const uint16_t* Ld, const uint16_t* Lup,
                        const uint16_t* cs, const uint16_t* bias, int64_t N, int64_t K, int64_t r,
                        const int64_t* rows, int64_t nrows, int8_t* qW_buf, uint16_t* sW_buf,
                        int8_t* qa_buf, float* sa_buf, double* d_buf, double* Y) {
    int64_t G = K / OR_GROUP;
    oracle_quantize_weights(W, N, K, qW_buf, sW_buf);
    for (int64_t i = 0; i < nrows; ++i) {
        const uint16_t* x = X + rows[i] * K;
        oracle_quantize_act(x, 1, K, qa_buf, sa_buf);
        if (r > 0) oracle_lora_down(x, Ld, 1, K, r, d_buf);
        for (int64_t n = 0; n < N; ++n)
            Y[i * N + n] = output_element(qa_buf, sa_buf, qW_buf + n * K, sW_buf + n * G, d_buf, Lup, n, N, K,
                                          r, cs[n], bias[n]);
    }
}

/* ---- the library's buffer layouts, version 1, written from their statement
 * These functions turn the oracle's codes and scales into the bytes that the
 * C ABI's layout description (include/w4a4.h, layout version 1) gives for the
 * packed weights and for the activation workspace, so that the CUDA packer
 * and the CUDA activation kernel can be compared with them byte for byte.
 * The layout itself is the library's choice (the pages ask for nibble and
 * tile order suited to the kernel: "INT4 Kernel Architecture, in depth",
 * "How the weights are stored"; the weights are repacked once at load: "W4A4
 * CUDA Kernel for Voice Clone", 3.10).  Every byte that the layout defines is
 * written and flagged 1 in `defined`; padding between sections stays 0 / 0.  */

static size_t or_align256(size_t x) { return (x + 255) / 256 * 256; }

/* Section offsets of the packed weight buffer: Ld, qW, sW, Lu, total. */
void oracle_packed_offsets(int64_t N, int64_t K, int64_t r, int64_t* off) {
    size_t G = (size_t)(K / OR_GROUP);
    size_t ld = 0;
    size_t qw = or_align256((size_t)K * (size_t)r * 2);
    size_t sw = or_align256(qw + G * (size_t)N * 32);
    size_t lu = or_align256(sw + G * (size_t)N * 2);
    size_t total = or_align256(lu + (size_t)r * (size_t)N * 2);
    off[0] = (int64_t)ld; off[1] = (int64_t)qw; off[2] = (int64_t)sw; off[3] = (int64_t)lu; off[4] = (int64_t)total;
}

/* Section offsets of the activation workspace: qA, sS, La, flags, total (the
 * minimum size; 160 x 16 uint32 stream-K flags end it). */
void oracle_act_offsets(int64_t M, int64_t K, int64_t r, int64_t* off) {
    size_t MT = (size_t)((M + 127) / 128), G = (size_t)(K / OR_GROUP);
    size_t qa = 0;
    size_t ss = or_align256(MT * G * 2 * 128 * 32);
    size_t la = or_align256(ss + MT * G * 128 * 8);
    size_t fl = or_align256(la + MT * (size_t)(r / 16) * 128 * 32);
    size_t total = or_align256(fl + 160 * 16 * 4);
    off[0] = (int64_t)qa; off[1] = (int64_t)ss; off[2] = (int64_t)la; off[3] = (int64_t)fl; off[4] = (int64_t)total;
}

static void put_byte(uint8_t* out, uint8_t* def, size_t at, uint8_t v) {
    out[at] = v;
    def[at] = 1;
}
static void put_u16(uint8_t* out, uint8_t* def, size_t at, uint16_t v) {
    put_byte(out, def, at, (uint8_t)(v & 0xff));
    put_byte(out, def, at + 1, (uint8_t)(v >> 8));
}

/* Position of code k (0..63) of a group inside its 32-byte weight record:
 * the 32-bit little-endian word at byte 8 q + 4 h holds in nibble j the code
 * of k = 32 h + (j < 4 ? 4 q + j : 16 + 4 q + (j - 4)).  Returns the byte
 * offset and sets *hi when the code is the byte's upper nibble.            */
static int record_position(int k, int* hi) {
    int h = k / 32, kk = k % 32;
    int second = kk >= 16;            /* nibbles 4..7 of the word */
    int rest = second ? kk - 16 : kk; /* 4 q + (j mod 4) */
    int q = rest / 4, j = (rest % 4) + (second ? 4 : 0);
    *hi = j % 2;
    return 8 * q + 4 * h + j / 2;
}

/* Swizzled position of 16-byte chunk c (0/1) in 32-byte row `row` of a plane:
 * the two halves are exchanged when bit 2 of the row index is set.         */
static int swizzled_chunk(int64_t row, int c) { return ((row >> 2) & 1) ? 1 - c : c; }

/* FP8 E4M3 byte of an integer c in [-8, 8], from the format's definition:
 * sign bit, 4-bit exponent with bias 7, 3-bit mantissa (normal numbers
 * 1.mmm x 2^(e-7)); 0 is 0x00.                                               */
static uint8_t e4m3_byte(int c) {
    if (c == 0) return 0;
    int a = c < 0 ? -c : c, e = 0;
    while ((a >> (e + 1)) != 0) ++e;               /* a in [2^e, 2^(e+1)) */
    int mant = ((a << 3) >> e) - 8;                /* a / 2^e = 1 + mant / 8, exact for a <= 8 */
    return (uint8_t)((c < 0 ? 0x80 : 0) | ((e + 7) << 3) | mant);
}

uint8_t oracle_e4m3_of_int(int c) { return e4m3_byte(c); }

/* Packed weights, version 1.  qW int8 [N, K] (codes -8..7), sW fp16 bits
 * [N, K/64], Ld fp16 bits [K, r], Lup fp16 bits [r, N]; out / def of
 * oracle_packed_offsets()[4] bytes, zeroed by the caller.                   */
void oracle_pack_weights_v1(const int8_t* qW, const uint16_t* sW, const uint16_t* Ld, const uint16_t* Lup,
                            int64_t N, int64_t K, int64_t r, uint8_t* out, uint8_t* def) {
    int64_t off[5];
    oracle_packed_offsets(N, K, r, off);
    int64_t G = K / OR_GROUP;
    /* L_down in MMA fragment order: [K/16][r/8][32 lanes][2 words]; lane L,
     * word w of (k-step s, tile t) holds the pair
     * L_down[16 s + 2 (L % 4) + 8 w + {0, 1}][8 t + L / 4].                 */
    for (int64_t s = 0; s < K / 16; ++s)
        for (int64_t t = 0; t < r / 8; ++t)
            for (int L = 0; L < 32; ++L)
                for (int w = 0; w < 2; ++w)
                    for (int e = 0; e < 2; ++e) {
                        int64_t k = 16 * s + 2 * (L % 4) + 8 * w + e, j = 8 * t + L / 4;
                        size_t at = (size_t)off[0] + ((((size_t)s * (size_t)(r / 8) + (size_t)t) * 32 + (size_t)L) * 2 +
                                                      (size_t)w) * 4 + (size_t)e * 2;
                        put_u16(out, def, at, Ld[k * r + j]);
                    }
    /* codes: [G][N][32-byte record], nibble = code + 8 */
    for (int64_t g = 0; g < G; ++g)
        for (int64_t n = 0; n < N; ++n) {
            size_t rec = (size_t)off[1] + ((size_t)g * (size_t)N + (size_t)n) * 32;
            for (int k = 0; k < OR_GROUP; ++k) {
                int hi;
                size_t at = rec + (size_t)record_position(k, &hi);
                uint8_t nib = (uint8_t)(qW[n * K + g * OR_GROUP + k] + 8);
                out[at] = hi ? (uint8_t)((out[at] & 0x0f) | (nib << 4)) : (uint8_t)((out[at] & 0xf0) | nib);
                def[at] = 1;
            }
        }
    /* scales: fp16 [G][N] */
    for (int64_t g = 0; g < G; ++g)
        for (int64_t n = 0; n < N; ++n)
            put_u16(out, def, (size_t)off[2] + ((size_t)g * (size_t)N + (size_t)n) * 2, sW[n * G + g]);
    /* L_up: [r/16][N][32 bytes], row n of plane p = L_up[16 p .. 16 p + 15][n],
     * halves swapped by the 32-byte swizzle of row n                         */
    for (int64_t p = 0; p < r / 16; ++p)
        for (int64_t n = 0; n < N; ++n)
            for (int i = 0; i < 16; ++i) {
                size_t at = (size_t)off[3] + ((size_t)p * (size_t)N + (size_t)n) * 32 +
                            (size_t)swizzled_chunk(n, i / 8) * 16 + (size_t)(i % 8) * 2;
                put_u16(out, def, at, Lup[(16 * p + i) * N + n]);
            }
}

/* Activation workspace, version 1, for rows m < M.  qA int8 [M, K], sA fp32
 * [M, K/64], La fp16 bits [M, r] (lora_act rounded to fp16; may be NULL when
 * r == 0); out / def of oracle_act_offsets()[4] bytes, zeroed by the caller.
 * The stream-K flags (160 x 16 uint32) are zero after the activation step.  */
void oracle_pack_act_v1(const int8_t* qA, const float* sA, const uint16_t* La, int64_t M, int64_t K, int64_t r,
                        uint8_t* out, uint8_t* def) {
    int64_t off[5];
    oracle_act_offsets(M, K, r, off);
    int64_t G = K / OR_GROUP;
    for (int64_t m = 0; m < M; ++m) {
        int64_t mt = m / 128, rr = m % 128;
        for (int64_t g = 0; g < G; ++g) {
            /* codes: plane (k % 64) / 32, row m % 128, byte k % 32 (swizzled) */
            int64_t sum = 0;
            for (int k = 0; k < OR_GROUP; ++k) {
                int8_t c = qA[m * K + g * OR_GROUP + k];
                sum += c;
                size_t plane = (size_t)off[0] + (((size_t)mt * (size_t)G + (size_t)g) * 2 + (size_t)(k / 32)) * 128 * 32;
                int b = k % 32;
                size_t at = plane + (size_t)rr * 32 + (size_t)swizzled_chunk(rr, b / 16) * 16 + (size_t)(b % 16);
                put_byte(out, def, at, e4m3_byte(c));
            }
            /* (sA, SA) fp32 pair per row and group */
            float pair[2] = {sA[m * G + g], (float)sum};
            size_t at = (size_t)off[1] + (((size_t)mt * (size_t)G + (size_t)g) * 128 + (size_t)rr) * 8;
            for (int i = 0; i < 8; ++i) put_byte(out, def, at + (size_t)i, ((const uint8_t*)pair)[i]);
        }
        /* lora_act: [MT][r/16][128][32 bytes], column j in plane j / 16 */
        for (int64_t j = 0; j < r; ++j) {
            int64_t p = j / 16, jj = j % 16;
            size_t at = (size_t)off[2] + (((size_t)mt * (size_t)(r / 16) + (size_t)p) * 128 + (size_t)rr) * 32 +
                        (size_t)swizzled_chunk(rr, (int)(jj / 8)) * 16 + (size_t)(jj % 8) * 2;
            put_u16(out, def, at, La[m * r + j]);
        }
    }
    for (size_t i = 0; i < 160 * 16 * 4; ++i) put_byte(out, def, (size_t)off[3] + i, 0);
}
