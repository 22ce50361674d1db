/*
 * moe_oracle.c -- plain, slow CPU oracle of the routed NVFP4 MoE expert layer.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the package's
 * smoke check and the CPU-baseline leg of the benchmark may load this library.
 * It shares no source, header, table or constant generator with the CUDA path.
 *
 * What it follows (sources are three web pages; cited by title and section):
 *   [MLM]  Megatron-LM PR #8262 "per-token NVFP4 squared-ReLU and SwiGLU MoE via
 *          FlashInfer CuTe DSL": Background (recipe), What is added (weight prep,
 *          per-token input quantization, two-stage finalize), How to extend (the
 *          alpha / fc2_input_scale table), What is tested (parity gaps list).
 *   [FI]   FlashInfer PR #5019 "CuTe DSL NVFP4 W4A16 MegaMoE": Tensor and
 *          numerical contract (canonical layouts, scale-plane size, compute order).
 *
 * Readings taken where the pages are silent (each one is also listed in the
 * design notes of the repository):
 *   R1  E2M1 magnitudes {0,0.5,1,1.5,2,3,4,6}; round to nearest, ties to the even
 *       code; magnitudes above 6 saturate to 6; the sign bit is kept even when the
 *       magnitude rounds to zero.
 *   R2  E4M3 (bias 7, max 448, subnormal step 2^-9) round to nearest even with
 *       saturation to 448.
 *   R3  Row quantizer order: sf = E4M3(fl(fl(amax_b/6)*enc)); r = fl(enc/dec(sf));
 *       code_j = E2M1(fl(v_j*r)); a block whose decoded scale is 0 gets +0 codes.
 *   R4  Per-token scale s = fl(amax*c), enc = fl(2688/amax), c = fl(1/2688);
 *       per-expert w_scale = fl(2688/amax), alpha = fl(1/w_scale).  A zero amax
 *       gives s = 0 (alpha = 0) and all-zero codes and block scales.
 *   R5  Routing order: stable by expert, then token, then slot; ids of -1 are
 *       empty slots; ids outside [-1, E) are treated as empty.
 *   R6  W4A4 forward: FC1 in fp64 over decoded values, times alpha1 and s_t;
 *       activation in fp64 rounded to fp32; row requant (R3/R4) of the activated
 *       row; FC2 in fp64 times alpha2 and s2, rounded to bf16 per route; finalize
 *       sums w[t,k]*route in fp64 for k ascending and rounds once to bf16.
 *   R7  W4A16 forward: FC1 in fp64 over the bf16 input, times alpha1; activation
 *       rounded to bf16; FC2 over that bf16 row times alpha2, bf16 route rows;
 *       the same finalize.
 *   R8  SwiGLU: canonical FC1 rows [0,I) are the gate, [I,2I) the up projection;
 *       a = silu(g)*u with silu(g) = g/(1+exp(-g)); no clamp.
 *   R15 Clamped SwiGLU (Tensor and numerical contract: the clamp caps the gate
 *       above the limit and clips up symmetrically): gate = min(gate, L),
 *       up = min(max(up, -L), L), before silu(gate) * up.
 *   R14 Router: top-K logits per token (ties to the lower expert id, descending),
 *       scores = softmax over the selected K, fp64, rounded to fp32.
 *   R12 Per-tensor recipe (How to extend, "Per-tensor NVFP4 x NVFP4"): the static
 *       FC1 / FC2 input scales a1, a2 are encode scales like w_scale: token rows
 *       and FC2-input rows are quantized with enc = a1 (resp. a2) and carry no
 *       per-row scale; the alphas become fl(1/fl(w_scale*a1)) and
 *       fl(1/fl(w_scale*a2)); codes and block scales of the weights are those of
 *       the per-token recipe.
 *
 * Everything here is scalar C compiled with -ffp-contract=off so every float
 * expression is one IEEE binary32 operation.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* Formats                                                                    */
/* ------------------------------------------------------------------------ */

/* E2M1 value of a 4-bit code: bit 3 is the sign, bits 0..2 index the printed
 * grid {0, 0.5, 1, 1.5, 2, 3, 4, 6} (Background: "NVFP4", E2M1 elements). */
double orc_e2m1_decode(uint8_t code) {
    static const double mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
    double m = mag[code & 7];
    return (code & 8) ? -m : m;
}

/* E2M1 encode (R1).  The decision points are the midpoints of neighbouring grid
 * values; at a midpoint the even code (the one whose mantissa bit is 0) wins. */
uint8_t orc_e2m1_encode(float v) {
    float a = fabsf(v);
    uint8_t m;
    if (a <= 0.25f) m = 0;        /* midpoint 0|0.5 -> 0 (even)   */
    else if (a < 0.75f) m = 1;    /* midpoint 0.5|1 -> 1.0 (even) */
    else if (a <= 1.25f) m = 2;   /* midpoint 1|1.5 -> 1.0        */
    else if (a < 1.75f) m = 3;    /* midpoint 1.5|2 -> 2.0        */
    else if (a <= 2.5f) m = 4;    /* midpoint 2|3 -> 2.0          */
    else if (a < 3.5f) m = 5;     /* midpoint 3|4 -> 4.0          */
    else if (a <= 5.0f) m = 6;    /* midpoint 4|6 -> 4.0          */
    else m = 7;                   /* saturate at 6                */
    return (uint8_t)(m | (signbit(v) ? 8 : 0));
}

/* E4M3 (fn variant) decode: bias 7, subnormals, no infinities (R2). */
double orc_e4m3_decode(uint8_t b) {
    int s = (b >> 7) & 1, e = (b >> 3) & 15, m = b & 7;
    double v;
    if (e == 0) v = ldexp((double)m, -9);
    else v = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

/* E4M3 encode, round to nearest even, saturating at 448 (R2).  The value is
 * divided by the quantum of its binade (a power of two, so exactly), rounded
 * with the default round-to-nearest-even mode and re-assembled. */
uint8_t orc_e4m3_encode(float vf) {
    double v = fabs((double)vf);
    uint8_t sign = signbit(vf) ? 0x80 : 0;
    uint8_t code;
    if (v >= 448.0) {
        code = 0x7E;
    } else if (v < ldexp(1.0, -6)) {
        double q = nearbyint(v / ldexp(1.0, -9)); /* 0..8 */
        code = (uint8_t)q;                        /* 8 is the first normal */
    } else {
        int ex;
        frexp(v, &ex);                /* v = f*2^ex, f in [0.5,1) */
        int e = ex - 1;               /* v in [2^e, 2^(e+1))      */
        double q = nearbyint(v / ldexp(1.0, e - 3)); /* 8..16 */
        if (q >= 16.0) { q = 8.0; e += 1; }
        int biased = e + 7;
        int c = (biased << 3) | ((int)q - 8);
        if (c > 0x7E) c = 0x7E;
        code = (uint8_t)c;
    }
    return (uint8_t)(code | sign);
}

/* bf16 bits -> float, exact. */
static float bf16_to_f32(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* double -> bf16 bits, one rounding, to nearest even.  The value is divided by
 * the bf16 quantum of its binade (2^(e-7); 2^-133 below the normal range),
 * rounded to an integer and scaled back, all exact in double. */
uint16_t orc_f64_to_bf16(double d) {
    if (isnan(d)) return 0x7FC0;
    double a = fabs(d);
    uint16_t sign = signbit(d) ? 0x8000 : 0;
    if (a == 0.0) return sign;
    int ex;
    frexp(a, &ex);
    int e = ex - 1;
    if (e < -126) e = -126;
    double quantum = ldexp(1.0, e - 7);
    double r = nearbyint(a / quantum) * quantum;
    if (r > 3.3895313892515355e38) return (uint16_t)(sign | 0x7F80); /* inf */
    float f = (float)r; /* exact: r has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(sign | ((u >> 16) & 0x7FFF));
}

/* The recipe constant 1/(448*6) as binary32 (How to extend: fc2_input_scale). */
float orc_recipe_c(void) { return 1.0f / 2688.0f; }

/* ------------------------------------------------------------------------ */
/* Quantizers                                                                 */
/* ------------------------------------------------------------------------ */

/* Row quantizer Q (R3): D values (D % 16 == 0), encode scale enc, 1x16 blocks
 * (Background: 1x16 E4M3 block scales, round to nearest, no 2D blocks, no RHT,
 * no stochastic rounding).  codes: D/2 bytes, element 2j in the low nibble.
 * sf: D/16 bytes, linear. */
void orc_quantize_row(const float* v, int64_t D, float enc, uint8_t* codes, uint8_t* sf) {
    for (int64_t b = 0; b < D / 16; ++b) {
        const float* blk = v + 16 * b;
        float amax = 0.0f;
        for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(blk[j]));
        float t = amax / 6.0f;
        float sf_f = t * enc;
        uint8_t s8 = orc_e4m3_encode(sf_f);
        float sfd = (float)orc_e4m3_decode(s8);
        sf[b] = s8;
        uint8_t q[16];
        if (sfd == 0.0f) {
            for (int j = 0; j < 16; ++j) q[j] = 0;
        } else {
            float r = enc / sfd;
            for (int j = 0; j < 16; ++j) {
                float x = blk[j] * r;
                q[j] = orc_e2m1_encode(x);
            }
        }
        for (int j = 0; j < 8; ++j) codes[8 * b + j] = (uint8_t)(q[2 * j] | (q[2 * j + 1] << 4));
    }
}

/* Per-row NVFP4 with one fp32 scale for the row (R4; Background: "one FP32
 * scale per token"; What is added: global scale is the recipe constant).
 * Returns the fp32 decode scale s of the row. */
static float quantize_row_per_token(const float* v, int64_t D, uint8_t* codes, uint8_t* sf) {
    float amax = 0.0f;
    for (int64_t j = 0; j < D; ++j) amax = fmaxf(amax, fabsf(v[j]));
    if (amax == 0.0f) {
        memset(codes, 0, (size_t)(D / 2));
        memset(sf, 0, (size_t)(D / 16));
        return 0.0f;
    }
    float c = orc_recipe_c();
    float s = amax * c;
    float enc = 2688.0f / amax;
    orc_quantize_row(v, D, enc, codes, sf);
    return s;
}

/* Token quantization (stage 2): x bf16 [T][H] -> codes [T][H/2], linear block
 * scales [T][H/16], per-token fp32 scales [T]. */
void orc_quantize_tokens(int64_t T, int64_t H, const uint16_t* x, uint8_t* codes, uint8_t* sf,
                         float* s) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        float* row = (float*)malloc(sizeof(float) * (size_t)H);
        for (int64_t h = 0; h < H; ++h) row[h] = bf16_to_f32(x[t * H + h]);
        s[t] = quantize_row_per_token(row, H, codes + t * (H / 2), sf + t * (H / 16));
        free(row);
    }
}

/* Per-tensor token quantization (R12): every row with the static encode scale
 * a1 (How to extend: "nvfp4_quantize(x, a1_scale) with a fixed scale tensor",
 * no per-token scale). */
void orc_quantize_tokens_static(int64_t T, int64_t H, const uint16_t* x, float a1, uint8_t* codes,
                                uint8_t* sf) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        float* row = (float*)malloc(sizeof(float) * (size_t)H);
        for (int64_t h = 0; h < H; ++h) row[h] = bf16_to_f32(x[t * H + h]);
        orc_quantize_row(row, H, a1, codes + t * (H / 2), sf + t * (H / 16));
        free(row);
    }
}

/* Per-tensor alphas (R12; How to extend: fc1_alpha = 1 / (w_scale * a1_scale),
 * fc2_alpha = 1 / (w_scale * a2_scale)) of one FC stack w bf16 [E][N][D]:
 * w_scale = fl(2688/amax) per expert as in weight prep; 0 for a zero expert. */
void orc_alpha_per_tensor(int64_t E, int64_t N, int64_t D, const uint16_t* w, float a,
                          float* alpha) {
    for (int64_t e = 0; e < E; ++e) {
        const uint16_t* we = w + e * N * D;
        float amax = 0.0f;
        for (int64_t i = 0; i < N * D; ++i) amax = fmaxf(amax, fabsf(bf16_to_f32(we[i])));
        if (amax == 0.0f) {
            alpha[e] = 0.0f;
            continue;
        }
        float w_scale = 2688.0f / amax;
        float prod = w_scale * a;
        alpha[e] = 1.0f / prod;
    }
}

/* Float-input variant used for the requantized FC2 input (R6). */
float orc_quantize_row_per_token_f32(const float* v, int64_t D, uint8_t* codes, uint8_t* sf) {
    return quantize_row_per_token(v, D, codes, sf);
}

/* Weight prep of one FC stack (stage 1): w bf16 [E][N][D] in canonical row
 * order -> codes [E][N][D/2], linear scales [E][N][D/16], alpha [E] (R4; What
 * is added: per-expert FP32 alphas; How to extend: alpha = 1 / w_scale). */
void orc_prepare_fc(int64_t E, int64_t N, int64_t D, const uint16_t* w, uint8_t* codes,
                    uint8_t* sf, float* alpha) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t e = 0; e < E; ++e) {
        float* row = (float*)malloc(sizeof(float) * (size_t)D);
        const uint16_t* we = w + e * N * D;
        float amax = 0.0f;
        for (int64_t i = 0; i < N * D; ++i) amax = fmaxf(amax, fabsf(bf16_to_f32(we[i])));
        uint8_t* ce = codes + e * N * (D / 2);
        uint8_t* se = sf + e * N * (D / 16);
        if (amax == 0.0f) {
            memset(ce, 0, (size_t)(N * D / 2));
            memset(se, 0, (size_t)(N * D / 16));
            alpha[e] = 0.0f;
            free(row);
            continue;
        }
        float w_scale = 2688.0f / amax;
        alpha[e] = 1.0f / w_scale;
        for (int64_t n = 0; n < N; ++n) {
            for (int64_t d = 0; d < D; ++d) row[d] = bf16_to_f32(we[n * D + d]);
            orc_quantize_row(row, D, w_scale, ce + n * (D / 2), se + n * (D / 16));
        }
        free(row);
    }
}

/* Byte offset of block scale (row r, scale column j) in the 128x4-swizzled
 * plane of a matrix with ncols16 = D/16 scale columns (What is added:
 * "128x4-swizzled E4M3 block scales"; Tensor and numerical contract: plane size
 * P = round_up(N,128)*round_up(D/16,4)).  The in-atom order is the 512-byte
 * 128-row x 4-column atom of the public block-scaling layout: 32 groups of 16
 * bytes, group (r mod 32) holding rows r, r+32, r+64, r+96, four scales each. */
int64_t orc_sf_swizzle_offset(int64_t r, int64_t j, int64_t ncols16) {
    int64_t cpad = (ncols16 + 3) / 4 * 4;
    return ((r / 128) * (cpad / 4) + j / 4) * 512 + (r % 32) * 16 + ((r / 32) % 4) * 4 + (j % 4);
}

/* ------------------------------------------------------------------------ */
/* Router: top-k selection and scores (upstream of the expert layer)          */
/* ------------------------------------------------------------------------ */

/* Plain top-K router ([MLM] Performance: "plain top-8", no group-limited
 * routing; R14): per token the K largest logits, ties to the lower expert id,
 * in descending order; scores = softmax over the K selected logits, computed in
 * fp64 (shift by the largest, exp, sum for k ascending) and rounded to fp32.
 * This equals softmax over all experts renormalised over the selected K. */
void orc_route_topk(int64_t T, int64_t E, int64_t K, const float* logits, int32_t* ids,
                    float* w) {
    if (K < 1 || K > E) return; /* no K distinct experts to select */
    for (int64_t t = 0; t < T; ++t) {
        const float* l = logits + t * E;
        unsigned char* taken = (unsigned char*)calloc((size_t)E, 1);
        for (int64_t k = 0; k < K; ++k) {
            int64_t best = -1;
            for (int64_t e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || l[e] > l[best]) best = e; /* strict: lower id wins ties */
            }
            taken[best] = 1;
            ids[t * K + k] = (int32_t)best;
        }
        double* ex = (double*)malloc(sizeof(double) * (size_t)K);
        double m = (double)l[ids[t * K]];
        double sum = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            ex[k] = exp((double)l[ids[t * K + k]] - m);
            sum += ex[k];
        }
        for (int64_t k = 0; k < K; ++k) w[t * K + k] = (float)(ex[k] / sum);
        free(ex);
        free(taken);
    }
}

/* ------------------------------------------------------------------------ */
/* Routing permutation (stage 3)                                              */
/* ------------------------------------------------------------------------ */

/* Stable counting sort of the valid (t,k) routes by expert (R5).
 * counts[E]; perm[R_valid] holds the flat route id t*K+k of each position in
 * expert-major order; inv[T*K] holds the position of each route or -1.
 * Returns R_valid. */
int64_t orc_route(int64_t T, int64_t K, int64_t E, const int32_t* ids, int32_t* counts,
                  int32_t* perm, int32_t* inv) {
    int64_t TK = T * K;
    for (int64_t e = 0; e < E; ++e) counts[e] = 0;
    for (int64_t i = 0; i < TK; ++i)
        if (ids[i] >= 0 && ids[i] < E) counts[ids[i]]++;
    int64_t* start = (int64_t*)malloc(sizeof(int64_t) * (size_t)(E + 1));
    start[0] = 0;
    for (int64_t e = 0; e < E; ++e) start[e + 1] = start[e] + counts[e];
    int64_t R = start[E];
    for (int64_t i = 0; i < TK; ++i) {
        int32_t e = ids[i];
        if (e >= 0 && e < E) {
            int64_t p = start[e]++;
            perm[p] = (int32_t)i;
            inv[i] = (int32_t)p;
        } else {
            inv[i] = -1;
        }
    }
    free(start);
    return R;
}

/* ------------------------------------------------------------------------ */
/* Expert computation                                                         */
/* ------------------------------------------------------------------------ */

/* Decoded NVFP4 element: E2M1 value times decoded E4M3 block scale (exact). */
static inline double dq(const uint8_t* codes, const uint8_t* sf, int64_t i) {
    uint8_t byte = codes[i >> 1];
    uint8_t code = (i & 1) ? (byte >> 4) : (byte & 15);
    return orc_e2m1_decode(code) * orc_e4m3_decode(sf[i >> 4]);
}

/* A whole decoded row (D elements); the dot products below read decoded values
 * from such rows, so each element is decoded once per row instead of once per
 * product (the same values, multiplied and summed in the same order). */
static void dq_row(const uint8_t* codes, const uint8_t* sf, int64_t D, double* out) {
    for (int64_t b = 0; b < D / 16; ++b) {
        const double scale = orc_e4m3_decode(sf[b]); /* one block scale per 16 elements */
        for (int64_t i = 16 * b; i < 16 * b + 16; ++i) {
            uint8_t byte = codes[i >> 1];
            out[i] = orc_e2m1_decode((i & 1) ? (byte >> 4) : (byte & 15)) * scale;
        }
    }
}

static double silu(double g) { return g / (1.0 + exp(-g)); }

/* Activation of one FC1 output row in fp64 (R8).  y has N1 entries (I for
 * squared-ReLU, 2I for SwiGLU in canonical [gate; up] order); a gets I.  With
 * limit > 0 the SwiGLU inputs are clamped first (R15: the gate capped at the
 * limit, the up value clipped to [-limit, limit]). */
static void activation(int act, double limit, int64_t I, const double* y, double* a) {
    for (int64_t n = 0; n < I; ++n) {
        if (act == 0) {
            double r = y[n] > 0.0 ? y[n] : 0.0;
            a[n] = r * r;
        } else {
            double g = y[n], u = y[I + n];
            if (limit > 0.0) {
                if (g > limit) g = limit;
                if (u > limit) u = limit;
                if (u < -limit) u = -limit;
            }
            a[n] = silu(g) * u;
        }
    }
}

typedef struct {
    int64_t E, H, I;
    int32_t act;   /* 0 = squared ReLU, 1 = SwiGLU */
    double limit;  /* > 0: clamped SwiGLU (R15) */
} orc_dims;

/* One route of the W4A4 expert (R6), for token row (xc, xsf, xs) and expert e.
 * a2_static > 0 selects the per-tensor FC2-input quantization (R12).
 * Writes the fp32 activated row (act_out, I values), the requantized FC2 input
 * (fc2c I/2 bytes, fc2sf I/16 bytes, returns s2 through *s2_out) and the bf16
 * route row (route_out, H values). */
static void expert_w4a4(const orc_dims* d, int64_t e, const uint8_t* w1c, const uint8_t* w1sf,
                        const float* a1, const uint8_t* w2c, const uint8_t* w2sf, const float* a2,
                        const uint8_t* xc, const uint8_t* xsf, float xs, float a2_static,
                        float* act_out, uint8_t* fc2c, uint8_t* fc2sf, float* s2_out,
                        uint16_t* route_out) {
    int64_t H = d->H, I = d->I, N1 = d->act ? 2 * I : I;
    double* y = (double*)malloc(sizeof(double) * (size_t)N1);
    double* a = (double*)malloc(sizeof(double) * (size_t)I);
    double* xd = (double*)malloc(sizeof(double) * (size_t)(H > I ? H : I));
    double* wd = (double*)malloc(sizeof(double) * (size_t)(H > I ? H : I));
    const uint8_t* c1 = w1c + e * N1 * (H / 2);
    const uint8_t* s1 = w1sf + e * N1 * (H / 16);
    dq_row(xc, xsf, H, xd);
    for (int64_t n = 0; n < N1; ++n) {
        dq_row(c1 + n * (H / 2), s1 + n * (H / 16), H, wd);
        double acc = 0.0;
        for (int64_t h = 0; h < H; ++h) acc += wd[h] * xd[h];
        y[n] = acc * (double)a1[e] * (double)xs;
    }
    activation(d->act, d->limit, I, y, a);
    for (int64_t n = 0; n < I; ++n) act_out[n] = (float)a[n];
    float s2;
    if (a2_static > 0.0f) { /* per-tensor (R12): static encode scale, no row scale */
        orc_quantize_row(act_out, I, a2_static, fc2c, fc2sf);
        s2 = 1.0f;
    } else {
        s2 = orc_quantize_row_per_token_f32(act_out, I, fc2c, fc2sf);
    }
    *s2_out = s2;
    const uint8_t* c2 = w2c + e * H * (I / 2);
    const uint8_t* sc2 = w2sf + e * H * (I / 16);
    dq_row(fc2c, fc2sf, I, xd);
    for (int64_t h = 0; h < H; ++h) {
        dq_row(c2 + h * (I / 2), sc2 + h * (I / 16), I, wd);
        double acc = 0.0;
        for (int64_t n = 0; n < I; ++n) acc += wd[n] * xd[n];
        route_out[h] = orc_f64_to_bf16(acc * (double)a2[e] * (double)s2);
    }
    free(y);
    free(a);
    free(xd);
    free(wd);
}

/* One route of the W4A16 expert (R7; Tensor and numerical contract: compute
 * order).  x is the bf16 token row.  act_out receives the bf16 handoff row. */
static void expert_w4a16(const orc_dims* d, int64_t e, const uint8_t* w1c, const uint8_t* w1sf,
                         const float* a1, const uint8_t* w2c, const uint8_t* w2sf, const float* a2,
                         const uint16_t* x, uint16_t* act_out, uint16_t* route_out) {
    int64_t H = d->H, I = d->I, N1 = d->act ? 2 * I : I;
    double* y = (double*)malloc(sizeof(double) * (size_t)N1);
    double* a = (double*)malloc(sizeof(double) * (size_t)I);
    double* wd = (double*)malloc(sizeof(double) * (size_t)(H > I ? H : I));
    const uint8_t* c1 = w1c + e * N1 * (H / 2);
    const uint8_t* s1 = w1sf + e * N1 * (H / 16);
    for (int64_t n = 0; n < N1; ++n) {
        dq_row(c1 + n * (H / 2), s1 + n * (H / 16), H, wd);
        double acc = 0.0;
        for (int64_t h = 0; h < H; ++h) acc += wd[h] * (double)bf16_to_f32(x[h]);
        y[n] = acc * (double)a1[e];
    }
    activation(d->act, d->limit, I, y, a);
    for (int64_t n = 0; n < I; ++n) act_out[n] = orc_f64_to_bf16(a[n]);
    const uint8_t* c2 = w2c + e * H * (I / 2);
    const uint8_t* sc2 = w2sf + e * H * (I / 16);
    for (int64_t h = 0; h < H; ++h) {
        dq_row(c2 + h * (I / 2), sc2 + h * (I / 16), I, wd);
        double acc = 0.0;
        for (int64_t n = 0; n < I; ++n) acc += wd[n] * (double)bf16_to_f32(act_out[n]);
        route_out[h] = orc_f64_to_bf16(acc * (double)a2[e]);
    }
    free(y);
    free(a);
    free(wd);
}

/* Deterministic two-stage finalize (stage 6; What is added: "reduces each
 * token's top-k routes in a fixed order"; Tensor and numerical contract: bf16
 * per-route terms times fp32 scores, one final bf16 conversion).  route rows are
 * indexed by inv[t*K+k]; -1 slots contribute nothing. */
void orc_finalize(int64_t T, int64_t K, int64_t H, const uint16_t* route, const int32_t* inv,
                  const float* w, uint16_t* out) {
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t h = 0; h < H; ++h) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                int32_t p = inv[t * K + k];
                if (p < 0) continue;
                acc += (double)w[t * K + k] * (double)bf16_to_f32(route[(int64_t)p * H + h]);
            }
            out[t * H + h] = orc_f64_to_bf16(acc);
        }
    }
}

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Full W4A4 forward (stages 3-6) over already quantized tokens.
 * Weights are canonical and linear (orc_prepare_fc output).  Outputs in the
 * compact permuted order q in [0, R): perm[R], act[R][I] fp32, fc2 codes
 * [R][I/2], scales [R][I/16], s2[R], route rows [R][H]; counts[E]; inv[T*K];
 * out[T][H].  Returns R. */
static int64_t forward_w4a4(const orc_dims* d, int64_t T, int64_t K, const uint8_t* w1c,
                            const uint8_t* w1sf, const float* a1, const uint8_t* w2c,
                            const uint8_t* w2sf, const float* a2, const uint8_t* xc,
                            const uint8_t* xsf, const float* xs, float a2_static,
                            const int32_t* ids, const float* w, int32_t* counts, int32_t* perm,
                            int32_t* inv, float* act, uint8_t* fc2c, uint8_t* fc2sf, float* s2,
                            uint16_t* route, uint16_t* out) {
    int64_t H = d->H, I = d->I;
    int64_t R = orc_route(T, K, d->E, ids, counts, perm, inv);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t q = 0; q < R; ++q) {
        int64_t t = perm[q] / K;
        int64_t e = ids[perm[q]];
        expert_w4a4(d, e, w1c, w1sf, a1, w2c, w2sf, a2, xc + t * (H / 2), xsf + t * (H / 16),
                    xs ? xs[t] : 1.0f, a2_static, act + q * I, fc2c + q * (I / 2),
                    fc2sf + q * (I / 16), s2 + q, route + q * H);
    }
    orc_finalize(T, K, H, route, inv, w, out);
    return R;
}

int64_t orc_forward_w4a4(const orc_dims* d, int64_t T, int64_t K, const uint8_t* w1c,
                         const uint8_t* w1sf, const float* a1, const uint8_t* w2c,
                         const uint8_t* w2sf, const float* a2, const uint8_t* xc,
                         const uint8_t* xsf, const float* xs, const int32_t* ids, const float* w,
                         int32_t* counts, int32_t* perm, int32_t* inv, float* act, uint8_t* fc2c,
                         uint8_t* fc2sf, float* s2, uint16_t* route, uint16_t* out) {
    return forward_w4a4(d, T, K, w1c, w1sf, a1, w2c, w2sf, a2, xc, xsf, xs, 0.0f, ids, w, counts,
                        perm, inv, act, fc2c, fc2sf, s2, route, out);
}

/* Per-tensor W4A4 forward (R12): tokens quantized with the static scale a1
 * (orc_quantize_tokens_static), alphas from orc_alpha_per_tensor, FC2 input
 * quantized with the static scale a2; no per-row scales. */
int64_t orc_forward_w4a4_per_tensor(const orc_dims* d, int64_t T, int64_t K, const uint8_t* w1c,
                                    const uint8_t* w1sf, const float* a1, const uint8_t* w2c,
                                    const uint8_t* w2sf, const float* a2, const uint8_t* xc,
                                    const uint8_t* xsf, float a2_static, const int32_t* ids,
                                    const float* w, int32_t* counts, int32_t* perm, int32_t* inv,
                                    float* act, uint8_t* fc2c, uint8_t* fc2sf, uint16_t* route,
                                    uint16_t* out) {
    float* s2 = (float*)malloc(sizeof(float) * (size_t)(T * K > 0 ? T * K : 1));
    int64_t R = forward_w4a4(d, T, K, w1c, w1sf, a1, w2c, w2sf, a2, xc, xsf, NULL, a2_static, ids,
                             w, counts, perm, inv, act, fc2c, fc2sf, s2, route, out);
    free(s2);
    return R;
}

/* Full W4A16 forward (stages 3, 7, 6) over bf16 tokens x [T][H]. */
int64_t orc_forward_w4a16(const orc_dims* d, int64_t T, int64_t K, const uint8_t* w1c,
                          const uint8_t* w1sf, const float* a1, const uint8_t* w2c,
                          const uint8_t* w2sf, const float* a2, const uint16_t* x,
                          const int32_t* ids, const float* w, int32_t* counts, int32_t* perm,
                          int32_t* inv, uint16_t* act, uint16_t* route, uint16_t* out) {
    int64_t H = d->H, I = d->I;
    int64_t R = orc_route(T, K, d->E, ids, counts, perm, inv);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t q = 0; q < R; ++q) {
        int64_t t = perm[q] / K;
        int64_t e = ids[perm[q]];
        expert_w4a16(d, e, w1c, w1sf, a1, w2c, w2sf, a2, x + t * H, act + q * I, route + q * H);
    }
    orc_finalize(T, K, H, route, inv, w, out);
    return R;
}

/* Dense brute force: every token through every expert it selects, computed
 * straight from the token index without any permutation, then summed for k
 * ascending.  Used only to pin the routed forward. */
void orc_dense_w4a4(const orc_dims* d, int64_t T, int64_t K, const uint8_t* w1c,
                    const uint8_t* w1sf, const float* a1, const uint8_t* w2c, const uint8_t* w2sf,
                    const float* a2, const uint8_t* xc, const uint8_t* xsf, const float* xs,
                    const int32_t* ids, const float* w, uint16_t* out) {
    int64_t H = d->H, I = d->I;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t t = 0; t < T; ++t) {
        float* act = (float*)malloc(sizeof(float) * (size_t)I);
        uint8_t* c = (uint8_t*)malloc((size_t)(I / 2));
        uint8_t* s = (uint8_t*)malloc((size_t)(I / 16));
        uint16_t* r = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(H * d->E));
        int* have = (int*)calloc((size_t)d->E, sizeof(int));
        double* acc = (double*)calloc((size_t)H, sizeof(double));
        for (int64_t e = 0; e < d->E; ++e) {
            int used = 0;
            for (int64_t k = 0; k < K; ++k) used |= (ids[t * K + k] == e);
            if (!used) continue;
            float s2;
            expert_w4a4(d, e, w1c, w1sf, a1, w2c, w2sf, a2, xc + t * (H / 2), xsf + t * (H / 16),
                        xs[t], 0.0f, act, c, s, &s2, r + e * H);
            have[e] = 1;
        }
        for (int64_t k = 0; k < K; ++k) {
            int32_t e = ids[t * K + k];
            if (e < 0 || e >= d->E || !have[e]) continue;
            for (int64_t h = 0; h < H; ++h)
                acc[h] += (double)w[t * K + k] * (double)bf16_to_f32(r[e * H + h]);
        }
        for (int64_t h = 0; h < H; ++h) out[t * H + h] = orc_f64_to_bf16(acc[h]);
        free(act);
        free(c);
        free(s);
        free(r);
        free(have);
        free(acc);
    }
}

/* ------------------------------------------------------------------------ */
/* Array helpers for the tests                                                */
/* ------------------------------------------------------------------------ */

void orc_e2m1_encode_n(const float* v, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_e2m1_encode(v[i]);
}

void orc_e4m3_encode_n(const float* v, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_encode(v[i]);
}

void orc_e4m3_decode_n(const uint8_t* b, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_decode(b[i]);
}

void orc_f64_to_bf16_n(const double* v, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f64_to_bf16(v[i]);
}

/* Scatter a linear [N][D/16] scale plane into the 128x4-swizzled plane of
 * P = round_up(N,128)*round_up(D/16,4) bytes (padding stays 0). */
void orc_sf_to_swizzled(int64_t N, int64_t ncols16, const uint8_t* lin, uint8_t* out) {
    int64_t cpad = (ncols16 + 3) / 4 * 4;
    int64_t npad = (N + 127) / 128 * 128;
    memset(out, 0, (size_t)(npad * cpad));
    for (int64_t r = 0; r < N; ++r)
        for (int64_t j = 0; j < ncols16; ++j)
            out[orc_sf_swizzle_offset(r, j, ncols16)] = lin[r * ncols16 + j];
}
