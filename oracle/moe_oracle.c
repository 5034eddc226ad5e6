/*
 * moe_oracle.c -- plain, slow CPU oracle of the routed-expert VQ2 MoE layer.
 *
 * TEST INFRASTRUCTURE.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / --impl reference legs of bench.py may load or run this
 * code.  It shares nothing with the CUDA library (no headers, helpers,
 * tables or constants) and neither side includes or imports the other.
 *
 * What it computes, and from which passage of the pages:
 *   - routed experts stored as 2-bit vector codes, about 2.1 bits per weight
 *     (Tandem-vLLM page, "How it works"); the code layout (sign bit + 7-bit
 *     index into a 128-entry fp16 codebook of 4-vectors, fp16 scale per row
 *     per 128 inputs) is the workload definition of the tiny MoE layer;
 *   - the codebook is sign-symmetric: the sign bit negates the 4-vector
 *     (vLLM-Moet page, "2-bit experts on vLLM v0.24.0");
 *   - FP4 experts in MXFP4 form: e2m1 elements with one ue8m0 exponent per
 *     32 (Tandem-vLLM page, "Quality": FP4_TOP keeps the most routed experts
 *     in FP4; vLLM-Moet page, "DeepSeek-V4.1-Flash on 4x RTX PRO 6000":
 *     MXFP4 experts);
 *   - router -> top-k -> expert FC1 (gate, up) -> silu(gate)*up -> FC2 ->
 *     weighted combine (vLLM-Moet page, "What we changed", the MoE-at-decode
 *     row, and "Qwen3.8": silu*up fused into the MoE GEMV);
 *   - nothing is skipped or substituted: the resident part plus the
 *     remainder is the whole layer (Tandem-vLLM page, "How it works").
 *
 * Floating point: everything is fp64 except the router logits, which are
 * also produced in the one fixed fp32 summation order that the GPU kernel
 * uses (so that the integer top-k decision is taken on identical values).
 * The pages do not fix that order; the reading is: lane l (0..31) sums, in
 * increasing h, the exact fp32 products of the inputs h with (h/8) mod 32
 * == l; then the 32 lane sums are combined by a butterfly (xor 16, 8, 4, 2,
 * 1); then the bias is added.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_BAD_ARG -1
#define ORACLE_NO_MEM -4

#define FMT_VQ2 0
#define FMT_FP4 1

/* ------------------------------------------------------------------ */
/* scalar formats                                                      */
/* ------------------------------------------------------------------ */

/* bfloat16: the upper 16 bits of an IEEE binary32. */
static float bf16_value(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* IEEE binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
static double fp16_value(uint16_t h) {
    int sign = (h >> 15) & 1;
    int ex = (h >> 10) & 0x1f;
    int fr = h & 0x3ff;
    double v;
    if (ex == 0)
        v = ldexp((double)fr, -24);               /* subnormal: fr * 2^-24 */
    else if (ex == 31)
        v = fr ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + fr), ex - 25);  /* (1 + fr/1024) * 2^(ex-15) */
    return sign ? -v : v;
}

/* OCP MX e2m1: 1 sign, 2 exponent (bias 1), 1 mantissa bit; no inf/nan. */
static double e2m1_value(unsigned nib) {
    int sign = (nib >> 3) & 1;
    int ex = (nib >> 1) & 3;
    int m = nib & 1;
    double v = (ex == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, ex - 1);
    return sign ? -v : v;
}

/* OCP MX ue8m0 scale: 2^(E-127); E = 255 is NaN (rejected by callers). */
static double e8m0_value(uint8_t e) { return ldexp(1.0, (int)e - 127); }

double oracle_fp16_value(uint16_t h) { return fp16_value(h); }
double oracle_e2m1_value(unsigned nib) { return e2m1_value(nib & 15); }

/* ------------------------------------------------------------------ */
/* router                                                              */
/* ------------------------------------------------------------------ */

/* logits[t,e] = sum_h x[t,h] * w[e,h] + bias[e], in the fixed fp32 order
 * described at the top of this file.  Requires H % 256 == 0. */
int oracle_router_logits_f32(const uint16_t* x, const uint16_t* w, const float* bias,
                             int T, int H, int E, float* logits) {
    if (T < 0 || E <= 0 || H <= 0 || H % 256) return ORACLE_BAD_ARG;
#pragma omp parallel for schedule(static)
    for (long te = 0; te < (long)T * E; ++te) {
        int t = (int)(te / E), e = (int)(te % E);
        float lane[32], next[32];
        for (int l = 0; l < 32; ++l) lane[l] = 0.0f;
        for (int h = 0; h < H; ++h) {
            int l = (h / 8) % 32;
            float p = bf16_value(x[(size_t)t * H + h]) * bf16_value(w[(size_t)e * H + h]);
            lane[l] = lane[l] + p;  /* p is exact: 8-bit x 8-bit significands */
        }
        for (int off = 16; off >= 1; off /= 2) {
            for (int l = 0; l < 32; ++l) next[l] = lane[l] + lane[l ^ off];
            for (int l = 0; l < 32; ++l) lane[l] = next[l];
        }
        float s = lane[0];
        if (bias) s = s + bias[e];
        logits[(size_t)t * E + e] = s;
    }
    return ORACLE_OK;
}

/* The same logits in fp64 (a diagnostic: the margin between the k-th and
 * (k+1)-th logit tells how close a routing decision is to a tie). */
int oracle_router_logits_f64(const uint16_t* x, const uint16_t* w, const float* bias,
                             int T, int H, int E, double* logits) {
    if (T < 0 || E <= 0 || H <= 0) return ORACLE_BAD_ARG;
#pragma omp parallel for schedule(static)
    for (long te = 0; te < (long)T * E; ++te) {
        int t = (int)(te / E), e = (int)(te % E);
        double s = 0.0;
        for (int h = 0; h < H; ++h)
            s += (double)bf16_value(x[(size_t)t * H + h]) * (double)bf16_value(w[(size_t)e * H + h]);
        if (bias) s += (double)bias[e];
        logits[(size_t)t * E + e] = s;
    }
    return ORACLE_OK;
}

/* Top-k of each token's logits: the k largest, ordered by (logit descending,
 * expert id ascending), so that equal logits go to the lower expert id.
 * Weights: renormalize = 1 -> softmax over the k selected logits;
 * renormalize = 0 -> the softmax over all E logits, read at the selected k. */
int oracle_route_topk(const float* logits, int T, int E, int k, int renormalize,
                      int32_t* ids, double* weights) {
    if (T < 0 || E <= 0 || k < 1 || k > E) return ORACLE_BAD_ARG;
    char* taken = (char*)malloc((size_t)E);
    if (!taken) return ORACLE_NO_MEM;
    for (int t = 0; t < T; ++t) {
        const float* l = logits + (size_t)t * E;
        memset(taken, 0, (size_t)E);
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || l[e] > l[best]) best = e;  /* strict: keeps the lower id on ties */
            }
            taken[best] = 1;
            ids[(size_t)t * k + j] = best;
        }
        double top = (double)l[ids[(size_t)t * k]];
        double den = 0.0;
        if (renormalize) {
            for (int j = 0; j < k; ++j) den += exp((double)l[ids[(size_t)t * k + j]] - top);
        } else {
            for (int e = 0; e < E; ++e) den += exp((double)l[e] - top);
        }
        for (int j = 0; j < k; ++j)
            weights[(size_t)t * k + j] = exp((double)l[ids[(size_t)t * k + j]] - top) / den;
    }
    free(taken);
    return ORACLE_OK;
}

/* Token -> expert permutation: a stable counting sort of the pairs
 * p = t*k + j by expert id.  expert_offsets[e] = number of pairs routed to
 * experts below e (so expert_offsets[E] = P); sorted_pair[s] = the pair at
 * sorted position s; pair_to_sorted is its inverse. */
int oracle_permute(const int32_t* ids, int P, int E, int32_t* expert_offsets,
                   int32_t* sorted_pair, int32_t* pair_to_sorted) {
    if (P < 0 || E <= 0) return ORACLE_BAD_ARG;
    int32_t* cursor = (int32_t*)calloc((size_t)E + 1, sizeof(int32_t));
    if (!cursor) return ORACLE_NO_MEM;
    for (int p = 0; p < P; ++p) {
        if (ids[p] < 0 || ids[p] >= E) { free(cursor); return ORACLE_BAD_ARG; }
        cursor[ids[p] + 1] += 1;
    }
    for (int e = 0; e < E; ++e) cursor[e + 1] += cursor[e];
    for (int e = 0; e <= E; ++e) expert_offsets[e] = cursor[e];
    for (int p = 0; p < P; ++p) {
        int s = cursor[ids[p]]++;
        sorted_pair[s] = p;
        pair_to_sorted[p] = s;
    }
    free(cursor);
    return ORACLE_OK;
}

/* ------------------------------------------------------------------ */
/* expert weights                                                      */
/* ------------------------------------------------------------------ */

/* VQ2 matrix [rows, K] -> dense fp64.  Code byte c of row r covers inputs
 * 4q..4q+3: W[r][4q+i] = (c >> 7 ? -1 : +1) * cb[c & 127][i] * scale[r][4q/128]. */
int oracle_decode_vq2(const uint8_t* codes, const uint16_t* scales, const uint16_t* cb,
                      int rows, int K, double* W) {
    if (rows <= 0 || K <= 0 || K % 128) return ORACLE_BAD_ARG;
    int G = K / 4, KB = K / 128;
#pragma omp parallel for schedule(static)
    for (int r = 0; r < rows; ++r) {
        for (int q = 0; q < G; ++q) {
            uint8_t c = codes[(size_t)r * G + q];
            double sgn = (c >> 7) ? -1.0 : 1.0;
            int idx = c & 127;
            double s = fp16_value(scales[(size_t)r * KB + (4 * q) / 128]);
            for (int i = 0; i < 4; ++i)
                W[(size_t)r * K + 4 * q + i] = sgn * fp16_value(cb[idx * 4 + i]) * s;
        }
    }
    return ORACLE_OK;
}

/* FP4 (MXFP4) matrix [rows, K] -> dense fp64.  Byte b of row r holds
 * elements 2b (low nibble) and 2b+1 (high nibble); each element is
 * e2m1(nibble) * 2^(E-127) with E the ue8m0 byte of its 32-element block. */
int oracle_decode_fp4(const uint8_t* codes, const uint8_t* scales, int rows, int K, double* W) {
    if (rows <= 0 || K <= 0 || K % 32) return ORACLE_BAD_ARG;
    int nb = K / 2, KB = K / 32;
    for (long i = 0; i < (long)rows * KB; ++i)
        if (scales[i] == 255) return ORACLE_BAD_ARG;
#pragma omp parallel for schedule(static)
    for (int r = 0; r < rows; ++r) {
        for (int b = 0; b < nb; ++b) {
            uint8_t v = codes[(size_t)r * nb + b];
            for (int h = 0; h < 2; ++h) {
                int col = 2 * b + h;
                unsigned nib = h ? (v >> 4) : (v & 15);
                W[(size_t)r * K + col] = e2m1_value(nib) * e8m0_value(scales[(size_t)r * KB + col / 32]);
            }
        }
    }
    return ORACLE_OK;
}

static int decode_matrix(int fmt, const uint8_t* codes, const void* scales, const uint16_t* cb,
                         int rows, int K, double* W) {
    if (fmt == FMT_VQ2) return oracle_decode_vq2(codes, (const uint16_t*)scales, cb, rows, K, W);
    if (fmt == FMT_FP4) return oracle_decode_fp4(codes, (const uint8_t*)scales, rows, K, W);
    return ORACLE_BAD_ARG;
}

/* y = W x for a dense row-major W [rows, K]. */
static void matvec(const double* W, const double* x, int rows, int K, double* y) {
#pragma omp parallel for schedule(static)
    for (int r = 0; r < rows; ++r) {
        double s = 0.0;
        const double* w = W + (size_t)r * K;
        for (int c = 0; c < K; ++c) s += w[c] * x[c];
        y[r] = s;
    }
}

/* One expert's SwiGLU FFN applied to n token vectors X [n, H] -> Y [n, H]:
 * g = Wg x, u = Wu x, a = silu(g) * u = g / (1 + e^-g) * u, y = Wd a.
 * The weights are decoded to dense fp64 first, then naive matvecs. */
int oracle_expert_ffn(int fmt, const uint8_t* c_gate, const void* s_gate,
                      const uint8_t* c_up, const void* s_up,
                      const uint8_t* c_down, const void* s_down,
                      const uint16_t* cb, int H, int I, int n, const double* X, double* Y) {
    if (H <= 0 || I <= 0 || n < 0) return ORACLE_BAD_ARG;
    double* Wg = (double*)malloc(sizeof(double) * (size_t)I * H);
    double* Wu = (double*)malloc(sizeof(double) * (size_t)I * H);
    double* Wd = (double*)malloc(sizeof(double) * (size_t)H * I);
    double* g = (double*)malloc(sizeof(double) * (size_t)I);
    double* u = (double*)malloc(sizeof(double) * (size_t)I);
    int rc = ORACLE_OK;
    if (!Wg || !Wu || !Wd || !g || !u) { rc = ORACLE_NO_MEM; goto done; }
    if ((rc = decode_matrix(fmt, c_gate, s_gate, cb, I, H, Wg))) goto done;
    if ((rc = decode_matrix(fmt, c_up, s_up, cb, I, H, Wu))) goto done;
    if ((rc = decode_matrix(fmt, c_down, s_down, cb, H, I, Wd))) goto done;
    for (int i = 0; i < n; ++i) {
        matvec(Wg, X + (size_t)i * H, I, H, g);
        matvec(Wu, X + (size_t)i * H, I, H, u);
        for (int r = 0; r < I; ++r) g[r] = g[r] / (1.0 + exp(-g[r])) * u[r];
        matvec(Wd, g, H, I, Y + (size_t)i * H);
    }
done:
    free(Wg); free(Wu); free(Wd); free(g); free(u);
    return rc;
}

/* Weighted combine: out[t] = sum_j include[t*k+j] * w[t,j] * y[t*k+j], in
 * increasing j.  ypair is in pair order (p = t*k + j); include may be NULL
 * (every pair counts). */
int oracle_combine(int T, int k, int H, const double* weights, const double* ypair,
                   const uint8_t* include, double* out) {
    if (T < 0 || k < 1 || H <= 0) return ORACLE_BAD_ARG;
    for (int t = 0; t < T; ++t) {
        double* o = out + (size_t)t * H;
        for (int h = 0; h < H; ++h) o[h] = 0.0;
        for (int j = 0; j < k; ++j) {
            size_t p = (size_t)t * k + j;
            if (include && !include[p]) continue;
            const double* y = ypair + p * H;
            for (int h = 0; h < H; ++h) o[h] += weights[p] * y[h];
        }
    }
    return ORACLE_OK;
}

int oracle_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}
