// Work description shared by the expert-FFN kernels: the workspace layout
// and the schedule records.
#pragma once

#include <cstddef>

#include "common.cuh"

namespace moe {

constexpr int MMA_NT_VQ2 = 32; // tokens per mma.sync chunk of a VQ2 expert (four n8 MMA tiles)
constexpr int MMA_NT_FP4 = 16; // tokens per mma.sync chunk of an FP4 expert (two n8 MMA tiles)
// From this many tokens per call, VQ2 experts with at most MMA_NT_FP4 tokens
// take the 16-token mma.sync configuration (two CTAs per SM) in a launch of
// their own: with many such experts the extra launch pays (measured: prefill
// of 4096 tokens 2.55 -> 2.34 ms per call), with few it does not (batch 32:
// 256 -> 276 us).
constexpr int MMA_SPLIT_T = 128;
constexpr int LUT_KB = 8;      // packed tiles per activation-table K-range (of 128 inputs for VQ2, 64 for FP4)
constexpr int UMMA_MIN = 32;   // tokens from which an expert takes the tcgen05 path (calls of more than UMMA_MIN tokens)
constexpr int UMMA_NT = 256;   // tokens per tcgen05 chunk
constexpr int MAX_LUT_CTAS = 1024;  // grid of the activation-table kernels (one CTA per SM) at most
constexpr int LUT_MAX_M = 3;   // VQ2 experts with up to this many tokens take the activation-table path
// The same in calls of at least MMA_SPLIT_T tokens, where the mma.sync
// kernels run anyway (measured, prefill of 4096 tokens, ms per call: up to 3
// tokens 2.319, 2 tokens 2.312, 1 token 2.291-2.300, none 2.379).
constexpr int LUT_MAX_M_LARGE = 1;
static_assert(LUT_MAX_M_LARGE <= LUT_MAX_M, "the schedule's table-pair arrays are sized by LUT_MAX_M");
// In calls of at most LUT4_MAX_T tokens the FP4 experts take the e2m1
// activation-table path, one table pair per token.  Measured with 52 of 256
// experts FP4 (expert-FFN call, us, e2m1 path / mma.sync path): 1 token
// 50.0 / 100.0, 2 tokens 87.7 / 112.9, 3 tokens 124.0 / 116.0.  Then no
// mma.sync, gather or conversion kernel is launched (every expert takes a
// table); from three tokens on, the FP4 experts with several tokens cost
// less on mma.sync than streamed once per token.
constexpr int LUT4_MAX_T = 2;

// A run of sorted positions of one expert (tensor-core paths).
struct Chunk {
    int32_t expert, start, count, fmt;
};

// One activation-table pair: its expert's code and scale buffers, its sorted
// position and token, and its token group (first table pair, pair count).
struct __align__(16) LutRec {
    const void* codes[3];
    const void* scales[3];
    int32_t sorted, token, gs, gc;
};
static_assert(sizeof(LutRec) == 64 && offsetof(LutRec, codes) == 0 && offsetof(LutRec, scales) == 24,
              "table pair record layout");

// Header words at the start of the workspace.
// HDR_NVQ2: the chunks list holds the 32-token chunks first (HDR_NVQ2 of
// them), then the 16-token ones (FP4, and small VQ2 experts in large calls).
// HDR_NLUT4, HDR_NGROUPS4: the e2m1 table pairs (rec4) and their token groups.
enum : int {
    HDR_NCHUNKS = 0, HDR_NLUT = 1, HDR_ERR = 2, HDR_NGROUPS = 3, HDR_NUMMA = 4, HDR_NVQ2 = 5, HDR_NLUT4 = 6,
    HDR_NGROUPS4 = 7
};

// Activation-table pairs (VQ2 experts with at most LUT_MAX_M tokens, one pair
// per token) are listed sorted by (token, expert) in lut_rec, grouped by
// token: grp_start holds the first pair of each token group, then n_lut.
// p1 / p2 hold their FC1 / FC2 K-range partial sums, lut_cnt one arrival
// counter per (table pair, FC2 row tile of 16 outputs); range holds each FC1
// CTA's unit range, computed by the schedule.
// Experts with at least UMMA_MIN pairs (possible once T >= UMMA_MIN) take
// the tcgen05 path (uchunks: chunks of <= UMMA_NT sorted positions); the
// tensor-core paths read x16s (fp16 activations gathered by sorted position)
// and a16 (fp16 silu(g)*u by sorted position).
// Range: x16s[s] holds x / xsc[s] and a16[s] holds a / asc[s], with xsc and
// asc powers of two that bring the row's largest magnitude to at most 2^14,
// so neither overflows fp16 whatever the range of the activations; the FC1
// epilogues write a in fp32 (a32) and flag the sorted positions they wrote
// (amax), from which the conversion kernel makes a16.
// The e2m1 table pairs (FP4 experts in calls of at most LUT4_MAX_T tokens,
// one pair per token) have their own records (rec4, grouped by token),
// partial sums (p1_4, p2_4) and FC2 arrival counters (cnt4).
struct WsLayout {
    size_t chunks_off, rec_off, grp_start_off, p1_off, p2_off, cnt_off, cnt2_off, range_off;
    size_t rec4_off, p1_4_off, p2_4_off, cnt4_off;
    size_t uchunks_off, x16s_off, a16_off, xsc_off, asc_off, amax_off, a32_off, total;
    int max_chunks, max_lut, max_uchunks, max_lut4;
};

__host__ __device__ inline size_t ws_align(size_t v) { return (v + 255) / 256 * 256; }
__host__ __device__ inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

// K-ranges of the activation-table path for an input length K.
__host__ __device__ inline int lut_jobs(int K) { return ceil_div(K / 128, LUT_KB); }
// K-ranges of the e2m1 table path (LUT_KB tiles of 64 inputs each).
__host__ __device__ inline int lut4_jobs(int K) { return ceil_div(K / 64, LUT_KB); }

// Units [u0, u1) of CTA i of C for jobs j = 0..J-1 covering the units
// [start(j), start(j+1)), start(J) = U, where a0(j) = floor(C start(j) / U).
// With J <= C and every a0(j+1) > a0(j), job j takes the CTAs a0(j) ..
// a0(j+1) - 1, each a contiguous share of it (no CTA builds two tables);
// otherwise CTA i takes [U i / C, U (i+1) / C).
__host__ __device__ inline int lut_cta_of(long long start, int C, int U) { return (int)((long long)C * start / U); }

__host__ __device__ inline WsLayout ws_layout(int T, int k, int E, int H, int I) {
    WsLayout L;
    long long P = (long long)T * k;
    L.max_chunks = (int)(P / MMA_NT_FP4 + E);
    L.max_lut = (int)(P < (long long)LUT_MAX_M * E ? P : (long long)LUT_MAX_M * E);  // table pairs
    size_t o = 256;
    L.chunks_off = o;
    o = ws_align(o + sizeof(Chunk) * (size_t)L.max_chunks);
    L.rec_off = o;
    o = ws_align(o + sizeof(LutRec) * (size_t)L.max_lut);
    L.grp_start_off = o;
    o = ws_align(o + sizeof(int32_t) * ((size_t)L.max_lut + 1));
    L.p1_off = o;
    o = ws_align(o + sizeof(float) * (size_t)L.max_lut * lut_jobs(H) * 2 * I);
    L.p2_off = o;
    o = ws_align(o + sizeof(float) * (size_t)L.max_lut * lut_jobs(I) * H);
    L.cnt_off = o;
    o = ws_align(o + sizeof(int32_t) * (size_t)L.max_lut * (H / 16));
    L.cnt2_off = o;  // single-token calls that combine in the table kernel: one counter per 16 outputs
    o = ws_align(o + sizeof(int32_t) * (size_t)(H / 16));
    L.range_off = o;
    o = ws_align(o + sizeof(int4) * (size_t)MAX_LUT_CTAS);
    L.max_lut4 = T <= LUT4_MAX_T ? (int)P : 0;  // (one pair per (token, expert) at most)
    L.rec4_off = o;
    o = ws_align(o + sizeof(LutRec) * (size_t)L.max_lut4);
    L.p1_4_off = o;
    o = ws_align(o + sizeof(float) * (size_t)L.max_lut4 * lut4_jobs(H) * 2 * I);
    L.p2_4_off = o;
    o = ws_align(o + sizeof(float) * (size_t)L.max_lut4 * lut4_jobs(I) * H);
    L.cnt4_off = o;
    o = ws_align(o + sizeof(int32_t) * (size_t)L.max_lut4 * (H / 16));
    const bool umma = T >= UMMA_MIN;
    L.max_uchunks = umma ? (int)(P / UMMA_NT + E) : 0;
    L.uchunks_off = o;
    o = ws_align(o + sizeof(Chunk) * (size_t)L.max_uchunks);
    L.x16s_off = o;
    o = ws_align(o + sizeof(uint16_t) * (size_t)P * H);
    L.a16_off = o;
    o = ws_align(o + sizeof(uint16_t) * (size_t)P * I);
    L.xsc_off = o;
    o = ws_align(o + sizeof(float) * (size_t)P);
    L.asc_off = o;
    o = ws_align(o + sizeof(float) * (size_t)P);
    L.amax_off = o;
    o = ws_align(o + sizeof(uint32_t) * (size_t)P);
    L.a32_off = o;
    o = ws_align(o + sizeof(float) * (size_t)P * I);
    L.total = o;
    return L;
}

// comb32 / comb16 (single-token FC2 only, either may be null): also write the
// combine of the pairs (moe_combine's arithmetic) using pair_to_sorted.
moe_status launch_lut_fc(bool fc1, bool self, const SlotTableHost* t, const uint16_t* x, const int32_t* offsets,
                         const int32_t* sorted_pair, const float* weights, int k, int P, int mode, float* out,
                         uint8_t* status, char* ws, const WsLayout& L, cudaStream_t s,
                         const int32_t* pair_to_sorted = nullptr, float* comb32 = nullptr,
                         uint16_t* comb16 = nullptr, bool f4 = false);
// x16s, xsc (and amax zeroed) for every sorted position.
moe_status launch_gather_f16(const uint16_t* x, const int32_t* sorted_pair, int k, int H, int P, char* ws,
                             const WsLayout& L, cudaStream_t s);
// a16, asc from a32, amax (the sorted positions the tensor-core FC1 wrote).
moe_status launch_a_to_f16(int P, int I, char* ws, const WsLayout& L, cudaStream_t s);
// 2^e as fp32 for |e| <= 126, and the exponent e (clamped to [-120, 120])
// of the power of two that brings a magnitude m to at most 2^top.
__host__ __device__ inline float exp2_i(int e) {
    union { uint32_t u; float f; } v;
    v.u = (uint32_t)(e + 127) << 23;
    return v.f;
}
__device__ __forceinline__ int range_exponent(float m, int top) {
    int ex = 0;
    frexpf(m, &ex);  // m < 2^ex
    return min(max(ex - top, -120), 120);
}
// silu(g) * u = g * u / (1 + e^-g) with the fast exponential and divide
// intrinsics: no special-value slow paths (the exactly rounded forms cost
// ~100 cycles per value in the tensor-core epilogues), relative error a few
// 1e-6, far below the fp16 rounding of the FC2 operand that follows.  For
// g < -88, e^-g is +inf and the quotient is 0, the limit of silu(g).
__device__ __forceinline__ float silu_mul(float g, float u) { return __fdividef(g, 1.0f + __expf(-g)) * u; }
moe_status launch_umma(bool fc1, const SlotTableHost* t, const int32_t* sorted_pair, const float* weights, int k,
                       int P, int mode, float* out, char* ws, const WsLayout& L, cudaStream_t s);
moe_status launch_mma_fc(bool fc1, const SlotTableHost* t, const int32_t* sorted_pair, const float* weights, int k,
                         int mode, float* out, char* ws, const WsLayout& L, cudaStream_t s, bool split16, bool vq2);
}  // namespace moe
