/*
 * dg_oracle.c -- plain, slow, double-precision CPU oracle for one pass of a uniform-state
 * block text-diffusion sampler's canvas update, and for the pieces of its denoising loop.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the checker, not the product: only the test suite,
 * the smoke check and the benchmark's CPU-baseline leg load it. It shares no source, header,
 * table or constant generator with the CUDA library; every number format, the hash and the
 * softmax statistics are written out here again from their definitions.
 *
 * What it computes, and where that is stated:
 *   - Every pass predicts every slot of the 256-slot canvas through the vocabulary head, keeps
 *     the slots it is most confident about and re-draws the rest uniformly from the vocabulary
 *     ("When to use a diffusion LLM" (devengoratela.com), "How block diffusion works").
 *   - The canvas starts from random vocabulary tokens (uniform-state diffusion; same section).
 *   - The loop stops when the average entropy over the canvas falls below a threshold, when the
 *     tokens are stable across two consecutive steps, or after 48 steps ("DiffusionGemma 26B:
 *     How Google's Text Diffusion Model Generates Tokens in Parallel" (dev.to), "How Diffusion
 *     Changes the Equation"). The loop control itself lives in oracle/oracle.py.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - confidence = max_n p_n of the softmax over the full vocabulary (untempered);
 *   - entropy in nats, H = -sum_n p_n ln p_n;
 *   - argmax ties go to the lowest vocabulary index; top-K ties go to the lower slot index;
 *   - the re-randomiser is the SplitMix64 output function (Steele, Lea & Flood, "Fast
 *     splittable pseudorandom number generators", OOPSLA 2014; Vigna's public-domain
 *     splitmix64.c), keyed as key(seed, pass, row) = sm64(sm64(sm64(seed) ^ pass) ^ row),
 *     and the new token is key mod V.
 *
 * Parallelism: OpenMP over vocabulary rows (logits) and over slot rows (softmax). It is not
 * tuned; it is the definition computed in double.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define OR_F32 0
#define OR_BF16 1
#define OR_E4M3 2
#define OR_NVFP4 3

/* ------------------------------------------------------------------------------------------
 * Number formats.
 * ---------------------------------------------------------------------------------------- */

/* bfloat16: the upper 16 bits of an IEEE binary32. */
double or_bf16_value(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* FP8 E4M3 (OCP 8-bit floating point specification, "E4M3" column): 1 sign bit, 4 exponent
 * bits with bias 7, 3 mantissa bits; no infinities; S.1111.111 is NaN; exponent field 0 holds
 * subnormals m/8 * 2^-6. Largest finite magnitude 1.75 * 2^8 = 448. */
double or_e4m3_value(uint8_t q) {
    int sign = (q >> 7) & 1;
    int e = (q >> 3) & 0xF;
    int m = q & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);              /* (m/8) * 2^(1-7) */
    else
        v = ldexp(1.0 + m / 8.0, e - 7);
    return sign ? -v : v;
}

/* Round x to a number with `sig` significant bits whose last place is at least 2^min_ulp_exp,
 * ties to even (the host's default rounding mode is round-to-nearest-even). */
static double round_sig(double x, int sig, int min_ulp_exp) {
    if (x == 0.0 || !isfinite(x)) return x;
    int e;
    frexp(x, &e);                               /* |x| = f * 2^e, 0.5 <= f < 1 */
    int ulp_exp = e - sig;
    if (ulp_exp < min_ulp_exp) ulp_exp = min_ulp_exp;
    return ldexp(nearbyint(ldexp(x, -ulp_exp)), ulp_exp);
}

/* Round a double to bfloat16, nearest-even (8 significant bits; subnormal spacing 2^-133). */
uint16_t or_bf16_round(double x) {
    if (isnan(x)) return 0x7FC0;
    double r = round_sig(x, 8, -133);
    float f = (float)r;                         /* exact: r has <= 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

/* Round a binary32 to E4M3, nearest-even, saturating to +-448 ("satfinite"): values whose
 * rounded magnitude would exceed 448 (including infinities) become +-448; NaN stays NaN. */
uint8_t or_e4m3_round_satfinite(float xf) {
    double x = (double)xf;
    if (isnan(x)) return 0x7F;
    uint8_t s = signbit(x) ? 0x80 : 0x00;
    double a = fabs(x);
    if (isinf(a)) return s | 0x7E;
    double r = round_sig(a, 4, -9);
    if (r > 448.0) r = 448.0;
    if (r == 0.0) return s;
    if (r < ldexp(1.0, -6)) {                   /* subnormal: r = m * 2^-9 */
        int m = (int)ldexp(r, 9);
        return s | (uint8_t)m;
    }
    int e;
    double f = frexp(r, &e);                    /* r = f * 2^e, leading bit 2^(e-1) */
    int E = e - 1 + 7;
    int m = (int)((2.0 * f - 1.0) * 8.0);       /* exact: 3 fraction bits */
    return s | (uint8_t)(E << 3) | (uint8_t)m;
}

/* Per-row absmax quantisation of bf16 rows to E4M3 with an fp32 scale, in IEEE binary32 as the
 * definition states it: amax = max_k |h_k|; if amax == 0 then scale = 1 and every code is 0;
 * otherwise inv = fp32(448 / amax), q_k = e4m3_satfinite(fp32(h_k * inv)),
 * scale = fp32(amax / 448). */
void or_quant_rows_e4m3(const uint16_t* h, int64_t rows, int64_t d, uint8_t* q, float* scale) {
    for (int64_t r = 0; r < rows; r++) {
        float amax = 0.0f;
        for (int64_t k = 0; k < d; k++) {
            float v = (float)or_bf16_value(h[r * d + k]);
            float a = fabsf(v);
            if (a > amax) amax = a;
        }
        if (amax == 0.0f) {
            scale[r] = 1.0f;
            for (int64_t k = 0; k < d; k++) q[r * d + k] = 0;
            continue;
        }
        volatile float inv = 448.0f / amax;     /* binary32 division, correctly rounded */
        for (int64_t k = 0; k < d; k++) {
            volatile float prod = (float)or_bf16_value(h[r * d + k]) * inv;
            q[r * d + k] = or_e4m3_round_satfinite(prod);
        }
        scale[r] = amax / 448.0f;
    }
}

/* FP4 E2M1 (OCP Microscaling Formats specification, "FP4 (E2M1)"): 1 sign bit, 2 exponent bits
 * with bias 1, 1 mantissa bit; exponent field 0 holds the subnormal 0.5 * m; no infinities or
 * NaN. Magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6. */
double or_e2m1_value(uint8_t q) {
    int sign = (q >> 3) & 1;
    int e = (q >> 1) & 3;
    int m = q & 1;
    double v = (e == 0) ? 0.5 * m : ldexp(1.0 + m / 2.0, e - 1);
    return sign ? -v : v;
}

/* Round a binary32 to E2M1, nearest-even, saturating to +-6; NaN is not representable and maps
 * to +6 here (the quantiser never produces it from finite input). */
uint8_t or_e2m1_round_satfinite(float xf) {
    double x = (double)xf;
    uint8_t s = (!isnan(x) && signbit(x)) ? 0x8 : 0x0;
    double a = fabs(x);
    if (isnan(a) || isinf(a)) return s | 0x7;
    double r = round_sig(a, 2, -1);             /* 2 significant bits, spacing >= 0.5 */
    if (r > 6.0) r = 6.0;
    if (r == 0.0) return s;
    if (r < 1.0) return s | 0x1;                /* the subnormal 0.5 */
    int e;
    double f = frexp(r, &e);                    /* r = f * 2^e, leading bit 2^(e-1) */
    int E = e - 1 + 1;
    int m = (int)((2.0 * f - 1.0) * 2.0);       /* exact: 1 fraction bit */
    return s | (uint8_t)(E << 1) | (uint8_t)m;
}

/* NVFP4 quantisation of bf16 rows (two-level scaling), in IEEE binary32 as stated:
 *   amax = max_k |h_k|; if amax == 0: row scale g = 1, every block scale and code 0.
 *   g = fp32(amax / 2688)                                   (2688 = 448 * 6)
 *   per block of 16 consecutive elements: bmax = max |h_k| over the block,
 *     sb = e4m3_rn_satfinite(fp32(bmax / fp32(6 * g)))      (the block scale, E4M3 >= 0)
 *     if sb == 0 every code of the block is 0, else with db = fp32(value(sb) * g):
 *     q_k = e2m1_rn_satfinite(fp32(h_k / db)).
 * The element value is e2m1(q_k) * value(sb) * g. Codes are packed two per byte, element 2j in the
 * low nibble of byte j and element 2j+1 in the high nibble. d must be a multiple of 16. */
void or_quant_rows_nvfp4(const uint16_t* h, int64_t rows, int64_t d, uint8_t* q, uint8_t* bscale,
                         float* scale) {
    const int64_t nb = d / 16;
    for (int64_t r = 0; r < rows; r++) {
        float amax = 0.0f;
        for (int64_t k = 0; k < d; k++) {
            float a = fabsf((float)or_bf16_value(h[r * d + k]));
            if (a > amax) amax = a;
        }
        uint8_t* qr = q + r * (d / 2);
        memset(qr, 0, (size_t)(d / 2));
        if (amax == 0.0f) {
            scale[r] = 1.0f;
            memset(bscale + r * nb, 0, (size_t)nb);
            continue;
        }
        volatile float g = amax / 2688.0f;
        volatile float g6 = 6.0f * g;
        scale[r] = g;
        for (int64_t b = 0; b < nb; b++) {
            float bmax = 0.0f;
            for (int64_t k = b * 16; k < b * 16 + 16; k++) {
                float a = fabsf((float)or_bf16_value(h[r * d + k]));
                if (a > bmax) bmax = a;
            }
            volatile float t = bmax / g6;
            uint8_t sb = or_e4m3_round_satfinite(t);
            bscale[r * nb + b] = sb;
            double sv = or_e4m3_value(sb);
            if (sv == 0.0) continue;
            volatile float db = (float)sv * g;
            for (int64_t k = b * 16; k < b * 16 + 16; k++) {
                volatile float x = (float)or_bf16_value(h[r * d + k]) / db;
                uint8_t c = or_e2m1_round_satfinite(x);
                qr[k / 2] |= (uint8_t)(c << (4 * (k & 1)));
            }
        }
    }
}

/* Widen one stored operand element to double. */
static inline double operand(int dtype, const void* base, int64_t i) {
    switch (dtype) {
    case OR_F32: return (double)((const float*)base)[i];
    case OR_BF16: return or_bf16_value(((const uint16_t*)base)[i]);
    case OR_NVFP4: return or_e2m1_value((((const uint8_t*)base)[i / 2] >> (4 * (i & 1))) & 0xF);
    default: return or_e4m3_value(((const uint8_t*)base)[i]);
    }
}

/* Block scale of element k of a row (NVFP4 operands): value of the E4M3 scale of its block of
 * 16; 1 for the other formats. */
static inline double block_scale(int dtype, const uint8_t* bscale, int64_t row, int64_t d,
                                 int64_t k) {
    return dtype == OR_NVFP4 ? or_e4m3_value(bscale[row * (d / 16) + k / 16]) : 1.0;
}

/* ------------------------------------------------------------------------------------------
 * Head contraction and softmax statistics for a set of slot rows.
 *
 * logits l[r,n] = sum_k h[r,k] * W[n,k] in double, times h_scale[r] * w_scale[n] for E4M3
 * operands, times inv_temp. Then, per row, a two-pass softmax over the whole vocabulary:
 *   pass 1: m = max_n l_n and a = the smallest n with l_n = m (the argmax);
 *           gap2 = m - max_{n != a} l_n (the top-2 logit gap; +inf when V = 1);
 *   pass 2: with t_n = l_n - m and e_n = exp(t_n), Z = sum_n e_n,
 *           p_n = e_n / Z, conf = max_n p_n = 1 / Z (e_a = 1),
 *           H = -sum_n p_n ln p_n = ln Z - (1/Z) sum_n e_n t_n.
 * ln Z is evaluated as log1p(Z - 1) with Z - 1 summed without the e_a = 1 term, so that the
 * entropy of a near-one-hot row keeps its relative precision.
 * ---------------------------------------------------------------------------------------- */
int or_head_stats(int64_t R, int64_t d, int64_t V, int dtype,
                  const void* h, const float* h_scale,
                  const void* w, const float* w_scale, double inv_temp,
                  const int64_t* rows, int64_t n_rows,
                  int32_t* argmax, double* conf, double* entropy, double* gap2,
                  const uint8_t* h_bscale, const uint8_t* w_bscale) {
    if (R < 0 || d <= 0 || V <= 0 || n_rows < 0) return -1;
    if ((dtype == OR_E4M3 || dtype == OR_NVFP4) && (!h_scale || !w_scale)) return -1;
    if (dtype == OR_NVFP4 && (d % 16 != 0 || !h_bscale || !w_bscale)) return -1;
    const int scaled = dtype == OR_E4M3 || dtype == OR_NVFP4;
    const int64_t RB = 256;                     /* rows per block: bounds the logit buffer */
    double* L = (double*)malloc(sizeof(double) * (size_t)(RB * V));
    double* hd = (double*)malloc(sizeof(double) * (size_t)(RB * d));
    double* hs = (double*)malloc(sizeof(double) * (size_t)RB);
    if (!L || !hd || !hs) { free(L); free(hd); free(hs); return -2; }

    for (int64_t b0 = 0; b0 < n_rows; b0 += RB) {
        int64_t nb = n_rows - b0 < RB ? n_rows - b0 : RB;
        for (int64_t i = 0; i < nb; i++) {
            int64_t r = rows ? rows[b0 + i] : b0 + i;
            for (int64_t k = 0; k < d; k++)
                hd[i * d + k] = operand(dtype, h, r * d + k) * block_scale(dtype, h_bscale, r, d, k);
            hs[i] = scaled ? (double)h_scale[r] : 1.0;
        }
        #pragma omp parallel
        {
            double* wd = (double*)malloc(sizeof(double) * (size_t)d);
            #pragma omp for schedule(static)
            for (int64_t n = 0; n < V; n++) {
                for (int64_t k = 0; k < d; k++)
                    wd[k] = operand(dtype, w, n * d + k) * block_scale(dtype, w_bscale, n, d, k);
                double ws = scaled ? (double)w_scale[n] : 1.0;
                for (int64_t i = 0; i < nb; i++) {
                    double acc = 0.0;
                    const double* hr = hd + i * d;
                    for (int64_t k = 0; k < d; k++) acc += hr[k] * wd[k];
                    L[i * V + n] = acc * hs[i] * ws * inv_temp;
                }
            }
            free(wd);
        }
        #pragma omp parallel for schedule(static)
        for (int64_t i = 0; i < nb; i++) {
            const double* l = L + i * V;
            double m = l[0];
            int64_t a = 0;
            for (int64_t n = 1; n < V; n++)
                if (l[n] > m) { m = l[n]; a = n; }
            double second = -INFINITY;
            for (int64_t n = 0; n < V; n++)
                if (n != a && l[n] > second) second = l[n];
            double zm1 = 0.0, et = 0.0;         /* Z - 1 and sum_n e_n t_n */
            for (int64_t n = 0; n < V; n++) {
                if (n == a) continue;
                double t = l[n] - m;
                double e = exp(t);
                zm1 += e;
                et += e * t;
            }
            double Z = 1.0 + zm1;
            int64_t o = b0 + i;
            argmax[o] = (int32_t)a;
            conf[o] = 1.0 / Z;
            entropy[o] = log1p(zm1) - et / Z;
            if (gap2) gap2[o] = (V > 1) ? m - second : INFINITY;
        }
    }
    free(L); free(hd); free(hs);
    return 0;
}

/* ------------------------------------------------------------------------------------------
 * Counter hash: one SplitMix64 output from state x (Steele, Lea & Flood, OOPSLA 2014; Vigna's
 * splitmix64.c): advance the state by the golden-ratio increment 0x9E3779B97F4A7C15, then apply
 * the variant-13 finaliser (xor-shift 30, multiply, xor-shift 27, multiply, xor-shift 31).
 * ---------------------------------------------------------------------------------------- */
uint64_t or_sm64(uint64_t x) {
    uint64_t z = x + 0x9E3779B97F4A7C15ULL;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

uint64_t or_key(uint64_t seed, uint32_t pass, uint64_t row) {
    return or_sm64(or_sm64(or_sm64(seed) ^ (uint64_t)pass) ^ row);
}

/* Uniform draw over the vocabulary for canvas row `row` at pass `pass` (no exclusions). */
int32_t or_draw(uint64_t seed, uint32_t pass, uint64_t row, int64_t V) {
    return (int32_t)(or_key(seed, pass, row) % (uint64_t)V);
}

/* ------------------------------------------------------------------------------------------
 * Keep / re-randomise for B canvases of S slots (rows r = b*S + slot):
 *   mean_entropy[b] = (1/S) sum_slots H;
 *   rank the slots of canvas b by their keep key, best first, ties to the lower slot, and keep
 *   the first K = min(keep_k, S). The key is the confidence, larger first (keep_rule 0: keep the
 *   slots the model is most confident about, "When to use a diffusion LLM", "How block
 *   diffusion works"), or the entropy, smaller first (keep_rule 1: lock the lowest-entropy tokens
 *   first, "DiffusionGemma 26B: How Google's Text Diffusion Model Generates Tokens in Parallel",
 *   "Architecture Details").
 *   Kept slots take their argmax. The others are re-drawn as key(seed, pass, row_offset + r) mod V
 *   (uniform-state diffusion), or set to mask_id when mask_id >= 0 (the masked-diffusion
 *   variant: re-mask instead of re-randomise, "DiffusionGemma: When Text Generation Stops Being
 *   Sequential", introduction).
 *   kgap[b] = |key(rank K-1) - key(rank K)| when 0 < K < S, else +inf.
 * ---------------------------------------------------------------------------------------- */
static const double* g_key_for_sort;   /* larger is better */
static int64_t g_base_for_sort;

static int by_key_then_slot(const void* pa, const void* pb) {
    int32_t a = *(const int32_t*)pa, b = *(const int32_t*)pb;
    double ka = g_key_for_sort[g_base_for_sort + a], kb = g_key_for_sort[g_base_for_sort + b];
    if (ka > kb) return -1;
    if (ka < kb) return 1;
    return (a < b) ? -1 : (a > b);
}

int or_select(int64_t B, int64_t S, int64_t V, const int32_t* argmax, const double* conf,
              const double* entropy, int64_t keep_k, uint64_t seed, uint32_t pass,
              int keep_rule, int64_t mask_id, uint64_t row_offset,
              int32_t* canvas_out, uint8_t* kept, double* mean_entropy, double* kgap) {
    if (B < 0 || S <= 0 || V <= 0 || keep_k < 0 || (keep_rule != 0 && keep_rule != 1) ||
        mask_id >= V)
        return -1;
    int32_t* order = (int32_t*)malloc(sizeof(int32_t) * (size_t)S);
    double* key = (double*)malloc(sizeof(double) * (size_t)(B * S));
    if (!order || !key) { free(order); free(key); return -2; }
    for (int64_t r = 0; r < B * S; r++) key[r] = keep_rule == 0 ? conf[r] : -entropy[r];
    int64_t K = keep_k < S ? keep_k : S;
    for (int64_t b = 0; b < B; b++) {
        int64_t base = b * S;
        double sum = 0.0;
        for (int64_t j = 0; j < S; j++) sum += entropy[base + j];
        mean_entropy[b] = sum / (double)S;
        for (int64_t j = 0; j < S; j++) order[j] = (int32_t)j;
        g_key_for_sort = key;
        g_base_for_sort = base;
        qsort(order, (size_t)S, sizeof(int32_t), by_key_then_slot);
        for (int64_t j = 0; j < S; j++) kept[base + j] = 0;
        for (int64_t j = 0; j < K; j++) kept[base + order[j]] = 1;
        if (kgap)
            kgap[b] = (K > 0 && K < S) ? key[base + order[K - 1]] - key[base + order[K]] : INFINITY;
        for (int64_t j = 0; j < S; j++) {
            int64_t r = base + j;
            canvas_out[r] = kept[r] ? argmax[r]
                          : mask_id >= 0 ? (int32_t)mask_id
                                         : or_draw(seed, pass, row_offset + (uint64_t)r, V);
        }
    }
    free(order);
    free(key);
    return 0;
}

/* ------------------------------------------------------------------------------------------
 * Synthetic denoiser (a stand-in for the model body; it is test harness, not the method):
 *   x = a * W[y_r] + (1 - a) * W[c_r],  a = min(1, fp32((2 + t) / 10)),  t = pass + 1,
 *   h_r = s_r * x / ||x||_2   (h_r = 0 when x = 0),  s_r = s_content for the first n_content
 *   slots of each canvas and s_pad for the rest; computed in double from the stored head
 *   values (E4M3 codes times their row scale), then rounded to bf16 nearest-even.
 * ---------------------------------------------------------------------------------------- */
int or_synth_denoise(int64_t B, int64_t S, int64_t d, int64_t V, int w_dtype, const void* w,
                     const float* w_scale, const int32_t* y, const int32_t* canvas, uint32_t pass,
                     int64_t n_content, double s_content, double s_pad, uint16_t* h_out) {
    float af = (float)(2 + (int64_t)pass + 1) / 10.0f;   /* binary32 division */
    double a = af < 1.0f ? (double)af : 1.0;
    double* x = (double*)malloc(sizeof(double) * (size_t)d);
    if (!x) return -2;
    for (int64_t r = 0; r < B * S; r++) {
        int64_t ty = y[r], tc = canvas[r];
        if (ty < 0 || ty >= V || tc < 0 || tc >= V) { free(x); return -3; }
        double sy = (w_dtype == OR_E4M3) ? (double)w_scale[ty] : 1.0;
        double sc = (w_dtype == OR_E4M3) ? (double)w_scale[tc] : 1.0;
        double nrm2 = 0.0;
        for (int64_t k = 0; k < d; k++) {
            x[k] = a * operand(w_dtype, w, ty * d + k) * sy
                 + (1.0 - a) * operand(w_dtype, w, tc * d + k) * sc;
            nrm2 += x[k] * x[k];
        }
        double s = ((r % S) < n_content) ? s_content : s_pad;
        double nrm = sqrt(nrm2);
        for (int64_t k = 0; k < d; k++)
            h_out[r * d + k] = or_bf16_round(nrm > 0.0 ? s * x[k] / nrm : 0.0);
    }
    free(x);
    return 0;
}

int or_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Vectorised helpers for the Python wrapper (loops over the scalar definitions above). */
void or_keys(uint64_t seed, uint32_t pass, const uint64_t* rows, int64_t n, uint64_t* out) {
    for (int64_t i = 0; i < n; i++) out[i] = or_key(seed, pass, rows[i]);
}

void or_sm64_many(const uint64_t* x, int64_t n, uint64_t* out) {
    for (int64_t i = 0; i < n; i++) out[i] = or_sm64(x[i]);
}

void or_bf16_round_many(const double* x, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; i++) out[i] = or_bf16_round(x[i]);
}

void or_e4m3_round_many(const float* x, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; i++) out[i] = or_e4m3_round_satfinite(x[i]);
}

void or_e4m3_value_many(const uint8_t* q, int64_t n, double* out) {
    for (int64_t i = 0; i < n; i++) out[i] = or_e4m3_value(q[i]);
}

void or_e2m1_round_many(const float* x, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; i++) out[i] = or_e2m1_round_satfinite(x[i]);
}
void or_e2m1_value_many(const uint8_t* q, int64_t n, double* out) {
    for (int64_t i = 0; i < n; i++) out[i] = or_e2m1_value(q[i]);
}
