/*
 * moe_oracle.c -- the oracle: a plain, slow, FP64 CPU statement of the forward
 * Mixture-of-Experts layer (router, top-k, sort-free layout, MXFP8 quantisation,
 * SwiGLU, weighted combine).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may load, call or link
 * this file: only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline and
 * reference legs use it.  It shares no code, header, table or constant with the
 * CUDA library (token_dispatch_expert_top_gb300/csrc), and the CUDA library shares
 * none with it.
 *
 * Sources.  The method is the one described on
 *   [MoK-2.37x] "Cursor's MoK achieves 2.37x performance boost on NVIDIA GB300
 *               NVL72" (KuCoin news flash; es/vi/hi/zh-hant editions, sections 01-03)
 *   [Kittens]   "Смесь котят: как Cursor создал открытое ядро, ускоряющее обучение
 *               ИИ до 2.4 раз" (qubstore.ru)
 * The pages give no formula for the gate or the number format; those steps follow
 * the layer's stated configuration (softmax over router logits, top-k, gates
 * renormalised to sum 1, SwiGLU experts) and the OCP Microscaling Formats (MX)
 * v1.0 specification for MXFP8 (E4M3 elements, one UE8M0 scale per 32 elements).
 *
 * Everything here is FP64 arithmetic over the stored input values, written as
 * plain loops in the order the definitions state them.  The only parallelism is an
 * OpenMP split over independent rows; no sum is blocked or reordered.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_API __attribute__((visibility("default")))

/* ------------------------------------------------------------------------- */
/* Number formats                                                             */
/* ------------------------------------------------------------------------- */

/* Round a finite v to the binary format with `mant_bits` stored mantissa bits and
 * smallest normal exponent `emin` (values below 2^emin use the fixed subnormal
 * spacing 2^(emin - mant_bits)).  Round to nearest, ties to the even mantissa:
 * the quotient a/spacing is an exact power-of-two scaling, and nearbyint() in the
 * default rounding mode rounds it half-to-even.  No overflow handling here. */
static double round_to_format(double v, int mant_bits, int emin) {
    if (v == 0.0 || !isfinite(v)) return v;
    double a = fabs(v);
    int E;
    frexp(a, &E);          /* a = f * 2^E with f in [0.5, 1) */
    int e = E - 1;         /* e = floor(log2(a)) */
    if (e < emin) e = emin;
    double spacing = ldexp(1.0, e - mant_bits);
    double r = nearbyint(a / spacing) * spacing;
    return copysign(r, v);
}

/* bfloat16: 8 exponent bits (bias 127), 7 mantissa bits; overflow to infinity. */
ORC_API double orc_round_bf16(double v) {
    double r = round_to_format(v, 7, -126);
    const double bf16_max = ldexp(255.0, 120);   /* (2 - 2^-7) * 2^127 */
    if (fabs(r) > bf16_max) r = copysign(INFINITY, v);
    return r;
}

/* IEEE binary32: 23 mantissa bits; overflow to infinity. */
ORC_API double orc_round_f32(double v) {
    double r = round_to_format(v, 23, -126);
    const double f32_max = ldexp((double)((1 << 24) - 1), 104);
    if (fabs(r) > f32_max) r = copysign(INFINITY, v);
    return r;
}

/* OCP E4M3 ("E4M3FN"): sign, 4 exponent bits (bias 7), 3 mantissa bits; no
 * infinities; S.1111.111 is NaN; the largest finite magnitude is 1.75 * 2^8 = 448;
 * subnormals m/8 * 2^-6.  The value of a code: */
ORC_API double orc_e4m3_decode(uint8_t code) {
    int s = code >> 7, ex = (code >> 3) & 15, m = code & 7;
    if (ex == 15 && m == 7) return NAN;
    double mag = (ex == 0) ? ldexp((double)m, -9) : ldexp((double)(8 + m), ex - 10);
    return s ? -mag : mag;
}

/* Encode a finite v: round to nearest-even E4M3, saturating magnitudes above 448
 * to 448 (the MX conversion's saturating mode).  The sign of zero is kept. */
ORC_API uint8_t orc_e4m3_encode(double v) {
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = round_to_format(fabs(v), 3, -6);
    if (a > 448.0) a = 448.0;
    if (a == 0.0) return sign;
    int E;
    frexp(a, &E);
    int e = E - 1;
    uint8_t code;
    if (e < -6) {
        code = (uint8_t)(a / ldexp(1.0, -9));                    /* subnormal: m * 2^-9 */
    } else {
        int m = (int)(a / ldexp(1.0, e) * 8.0) - 8;              /* a = (1 + m/8) 2^e */
        code = (uint8_t)(((e + 7) << 3) | m);
    }
    return sign | code;
}

/* NVFP4 (a reading of NVIDIA's published format: the pages only name it): E2M1
 * elements -- sign, 2 exponent bits (bias 1), 1 mantissa bit, magnitudes
 * {0, 0.5, 1, 1.5, 2, 3, 4, 6}, no infinities or NaN -- with one E4M3 scale per 16
 * consecutive elements along K and one FP32 scale per tensor. */
ORC_API double orc_e2m1_decode(uint8_t code) {
    int s = (code >> 3) & 1, ex = (code >> 1) & 3, m = code & 1;
    double mag = (ex == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, ex - 1);
    return s ? -mag : mag;
}

/* Round to nearest-even E2M1, saturating magnitudes above 6 to 6; the sign of
 * zero is kept.  Returns the 4-bit code. */
ORC_API uint8_t orc_e2m1_encode(double v) {
    uint8_t sign = signbit(v) ? 0x8 : 0x0;
    double a = round_to_format(fabs(v), 1, 0);
    if (a > 6.0) a = 6.0;
    if (a == 0.0) return sign;
    if (a < 1.0) return sign | 1;                                /* subnormal 0.5 */
    int E;
    frexp(a, &E);
    int e = E - 1;                                               /* a = (1 + m/2) 2^e */
    int m = (int)(a / ldexp(1.0, e) * 2.0) - 2;
    return sign | (uint8_t)(((e + 1) << 1) | m);
}

/* Per-tensor scale: amax / (6 * 448) in FP32 (1 for an all-zero tensor), so the
 * largest block scale lands at the top of E4M3's range. */
ORC_API double orc_nvfp4_tensor_scale(const double* in, int64_t n) {
    double amax = 0.0;
    for (int64_t i = 0; i < n; ++i) amax = fmax(amax, fabs(in[i]));
    return amax > 0.0 ? orc_round_f32(amax / 2688.0) : 1.0;
}

/* NVFP4 quantisation along K of a [rows][K] matrix of FP32 values with tensor
 * scale st.  Per block of 16: t = fp32(fp32(amax / 6) / st), its E4M3 code is the
 * block scale sb; d = fp32(sb * st); every element is the E2M1 code of
 * fp32(x / d) (code 0 when d is 0).  Codes are packed two per byte, the lower
 * element in the low nibble: codes [rows][K/2], scales [rows][K/16].  Every FP32
 * step is one correctly rounded operation (an FP64 result rounded once is the
 * FP32 result for these operations). */
ORC_API void orc_quantize_nvfp4(const double* in, int64_t rows, int64_t K, double st,
                                uint8_t* codes, uint8_t* scales) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t b = 0; b < K / 16; ++b) {
            const double* v = in + r * K + b * 16;
            double amax = 0.0;
            for (int t = 0; t < 16; ++t) amax = fmax(amax, fabs(v[t]));
            double t6 = orc_round_f32(orc_round_f32(amax / 6.0) / st);
            uint8_t sb = orc_e4m3_encode(t6);
            double d = orc_round_f32(orc_e4m3_decode(sb) * st);
            scales[r * (K / 16) + b] = sb;
            for (int t = 0; t < 16; t += 2) {
                uint8_t lo = d == 0.0 ? 0 : orc_e2m1_encode(orc_round_f32(v[t] / d));
                uint8_t hi = d == 0.0 ? 0 : orc_e2m1_encode(orc_round_f32(v[t + 1] / d));
                codes[r * (K / 2) + b * 8 + t / 2] = (uint8_t)(lo | (hi << 4));
            }
        }
    }
}

ORC_API void orc_dequantize_nvfp4(const uint8_t* codes, const uint8_t* scales, int64_t rows,
                                  int64_t K, double st, double* out) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < K; ++c) {
            uint8_t byte = codes[r * (K / 2) + c / 2];
            uint8_t q = (c & 1) ? (byte >> 4) : (byte & 15);
            out[r * K + c] = orc_e2m1_decode(q) * orc_e4m3_decode(scales[r * (K / 16) + c / 16]) * st;
        }
}

ORC_API void orc_round_bf16_array(const double* in, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_round_bf16(in[i]);
}

ORC_API void orc_round_f32_array(const double* in, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_round_f32(in[i]);
}

ORC_API void orc_e4m3_encode_array(const double* in, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_encode(in[i]);
}

/* MXFP8 quantisation of a row-major [rows][K] matrix along K (OCP MX v1.0,
 * conversion from a higher-precision vector): each block of 32 consecutive
 * elements of a row gets one shared scale X = 2^s stored as UE8M0 code s + 127,
 * with s = floor(log2(max|v|)) - emax(E4M3) = floor(log2(amax)) - 8, clamped to
 * the UE8M0 range [-127, 127]; an all-zero block takes s = -127.  Each element
 * is stored as E4M3(v / X) (nearest-even, saturating).  K must be a multiple of 32.
 * The pages place this quantisation of activations inside the dispatch, grouped
 * GEMM and SwiGLU data paths ([MoK-2.37x] section 02, last paragraphs). */
ORC_API void orc_quantize_mxfp8(const double* in, int64_t rows, int64_t K,
                                uint8_t* codes, uint8_t* scales) {
    int64_t nb = K / 32;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t b = 0; b < nb; ++b) {
            const double* v = in + r * K + b * 32;
            double amax = 0.0;
            for (int t = 0; t < 32; ++t)
                if (fabs(v[t]) > amax) amax = fabs(v[t]);
            int s;
            if (amax == 0.0) {
                s = -127;
            } else {
                int E;
                frexp(amax, &E);
                s = (E - 1) - 8;
                if (s < -127) s = -127;
                if (s > 127) s = 127;
            }
            scales[r * nb + b] = (uint8_t)(s + 127);
            for (int t = 0; t < 32; ++t)
                codes[r * K + b * 32 + t] = orc_e4m3_encode(ldexp(v[t], -s));
        }
    }
}

/* Value of an MXFP8 matrix: E4M3(code) * 2^(scale - 127). */
ORC_API void orc_dequantize_mxfp8(const uint8_t* codes, const uint8_t* scales,
                                  int64_t rows, int64_t K, double* out) {
    int64_t nb = K / 32;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < K; ++c)
            out[r * K + c] = ldexp(orc_e4m3_decode(codes[r * K + c]),
                                   (int)scales[r * nb + c / 32] - 127);
}

/* ------------------------------------------------------------------------- */
/* Router: softmax, top-k, renormalised gates                                 */
/* ------------------------------------------------------------------------- */

/* For each of n tokens with router logits l[0..E): p = softmax(l); the k experts
 * with the largest logits (softmax is monotone, so these carry the largest p),
 * listed by descending logit with the lower expert index first on equal logits;
 * gates g_j = p[e_j] / sum_j' p[e_j'] ("renormalised to sum 1").  Every token
 * picks a few experts out of many each step ([MoK-2.37x] section 01).
 * probs (nullable) receives the full softmax [n][E]. */
ORC_API void orc_route_topk(const double* logits, int64_t n, int E, int k,
                            int32_t* idx, double* gate, double* probs) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < n; ++t) {
        const double* l = logits + t * E;
        double* p = (double*)malloc(sizeof(double) * (size_t)E);
        char* chosen = (char*)calloc((size_t)E, 1);
        double mx = l[0];
        for (int e = 1; e < E; ++e)
            if (l[e] > mx) mx = l[e];
        double Z = 0.0;
        for (int e = 0; e < E; ++e) {
            p[e] = exp(l[e] - mx);
            Z += p[e];
        }
        for (int e = 0; e < E; ++e) p[e] /= Z;
        if (probs)
            for (int e = 0; e < E; ++e) probs[t * E + e] = p[e];
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e)
                if (!chosen[e] && (best < 0 || l[e] > l[best])) best = e;
            chosen[best] = 1;
            idx[t * k + j] = best;
        }
        double sp = 0.0;
        for (int j = 0; j < k; ++j) sp += p[idx[t * k + j]];
        for (int j = 0; j < k; ++j) gate[t * k + j] = p[idx[t * k + j]] / sp;
        free(p);
        free(chosen);
    }
}

/* ------------------------------------------------------------------------- */
/* Layout ("schedule"): counts, offsets, two-column pull schedule, inverse     */
/* ------------------------------------------------------------------------- */

/* Count the tokens of each expert, place them so that each expert's tokens are
 * contiguous ([MoK-2.37x] section 01: count per expert, decide placement, keep
 * same-expert data together for the grouped GEMM), without sorting ([Kittens],
 * pull paragraph: a two-column schedule built with no sort).
 *   counts[e]  = number of (n, j) with idx[n][j] == e
 *   offsets    = exclusive scan of counts, offsets[E] = N*k (no padding)
 *   slot order inside expert e: ascending token index n (each token picks an
 *              expert at most once), i.e. a stable counting placement
 *   sched[slot] = (source shard, row in shard) = (n / (N/S), n % (N/S)), the only
 *              two things a pulling reader needs ([MoK-2.37x] section 02)
 *   inv[n][j]  = slot of (n, j)
 * N must be a multiple of S. */
ORC_API void orc_layout(const int32_t* idx, int64_t N, int k, int E, int S,
                        int32_t* counts, int32_t* offsets, int32_t* sched, int32_t* inv) {
    int64_t rows_per_shard = N / S;
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (int64_t t = 0; t < N * k; ++t) counts[idx[t]] += 1;
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    int32_t* fill = (int32_t*)malloc(sizeof(int32_t) * (size_t)(E > 0 ? E : 1));
    for (int e = 0; e < E; ++e) fill[e] = offsets[e];
    for (int64_t n = 0; n < N; ++n) {
        for (int j = 0; j < k; ++j) {
            int e = idx[n * k + j];
            int32_t slot = fill[e]++;
            sched[2 * (int64_t)slot + 0] = (int32_t)(n / rows_per_shard);
            sched[2 * (int64_t)slot + 1] = (int32_t)(n % rows_per_shard);
            inv[n * k + j] = slot;
        }
    }
    free(fill);
}

/* ------------------------------------------------------------------------- */
/* Expert nonlinearity and combine                                            */
/* ------------------------------------------------------------------------- */

/* SwiGLU: h = silu(u) * v with silu(u) = u * sigma(u), sigma(u) = 1/(1+e^-u). */
ORC_API void orc_swiglu(const double* u, const double* v, int64_t n, double* h) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) h[i] = u[i] / (1.0 + exp(-u[i])) * v[i];
}

/* Combine + final weighted merge ([MoK-2.37x] sections 02-03): every expert
 * result returns to its token, and out[n] = sum_j g[n][j] * y[inv[n][j]], summed
 * in j order (descending gate logit).  y is [rows_y][H], indexed by inv. */
ORC_API void orc_combine(const double* y, const int32_t* inv, const double* gate,
                         int64_t n, int k, int64_t H, double* out) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < n; ++t) {
        for (int64_t h = 0; h < H; ++h) {
            double acc = 0.0;
            for (int j = 0; j < k; ++j)
                acc += gate[t * k + j] * y[(int64_t)inv[t * k + j] * H + h];
            out[t * H + h] = acc;
        }
    }
}

/* ------------------------------------------------------------------------- */
/* Backward element-wise steps                                                */
/* ------------------------------------------------------------------------- */

/* SwiGLU backward.  With h = silu(u) * v and s = sigma(u):
 *   dh/dv = silu(u) = u * s
 *   dh/du = v * silu'(u),  silu'(u) = s + u * s * (1 - s)
 * so du = dh * v * silu'(u) and dv = dh * silu(u). */
ORC_API void orc_swiglu_backward(const double* u, const double* v, const double* dh, int64_t n,
                                 double* du, double* dv) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        double s = 1.0 / (1.0 + exp(-u[i]));
        du[i] = dh[i] * v[i] * (s + u[i] * s * (1.0 - s));
        dv[i] = dh[i] * u[i] * s;
    }
}

/* Gradient of the renormalised gates with respect to the selected logits.  The
 * renormalised top-k gates are a softmax over the k selected logits,
 * g_j = e^{l_j} / sum_i e^{l_i}, so dg_j/dl_m = g_j (delta_jm - g_m) and
 *   dlogit_m = sum_j dg_j g_j (delta_jm - g_m) = g_m (dg_m - sum_j g_j dg_j).
 * The unselected logits get no gradient: the selection is piecewise constant. */
ORC_API void orc_gate_backward(const double* gate, const double* dgate, int64_t n, int k,
                               double* dlogit_sel) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < n; ++t) {
        double dot = 0.0;
        for (int j = 0; j < k; ++j) dot += gate[t * k + j] * dgate[t * k + j];
        for (int j = 0; j < k; ++j)
            dlogit_sel[t * k + j] = gate[t * k + j] * (dgate[t * k + j] - dot);
    }
}
