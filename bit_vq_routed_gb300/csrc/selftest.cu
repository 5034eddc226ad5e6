// Boot self-check (Tandem-vLLM page, "New in 0.2.0": each kernel is checked
// against a reference at boot).
//
// The check runs the tiny routed-expert layer (hidden 256, intermediate 128,
// 8 experts, top-2) through the public entry points and compares what they
// produce with expected values that the CPU oracle computed from the same
// inputs (selftest_expected.h, written by oracle/make_selftest_golden.py).
// The inputs are drawn here, on the GPU, from SplitMix64 (Steele, Lea and
// Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014):
// draw i of stream `tag` is the first output of the generator whose state is
// tag * 2^32 + i.  The values made from a draw v are exact in their formats:
//   g(v) = sum of the 6-bit fields at bits 0, 8, 16 and 24 of v, minus 126;
//   tokens bf16 g/32, router bf16 g/2048, codebook fp16 g/32,
//   VQ2 codes v & 255, VQ2 scales fp16 (40 + v mod 124)/8192,
//   FP4 codes v & 255, FP4 scales ue8m0 118 + v mod 3;
// arrays in row-major order of their logical layouts; token row t uses the
// draws of row t mod 4.  Streams: tokens 1, router 2, codebook 3, VQ2 codes
// 16 + 4e + m, VQ2 scales 48 + 4e + m, FP4 codes 80 + 4e + m, FP4 scales
// 112 + 4e + m (expert e, matrix m = gate, up, down).
//
// Cases, each with the path it reaches:
//   route4     moe_router_logits + moe_route_topk + moe_permute, 4 tokens;
//   route4f    moe_route (one fused kernel), 4 tokens;
//   vq2_t4     per-pair FFN (table kernels: every expert has at most three
//              tokens) + moe_combine;
//   vq2_scat   the same in fused-scatter mode;
//   vq2_t1     moe_route + moe_vq2_expert_ffn_combine on token 0 alone (the
//              self-scheduling single-token kernels with the combine inside);
//   vq2_t16    16 tokens (the four repeated): 4 or 8 tokens per routed
//              expert, the small-batch mma.sync kernels;
//   vq2_t128   128 tokens (the four repeated): every routed expert has at
//              least 32 tokens, so the tcgen05 kernels run;
//   mix_t4 / mix_t128   the mixed-format layer (FP4 experts 1, 3, 5, 7);
//   partial    experts 2 and 7 not resident: pair_status and the partial
//              output of the resident experts.
// Routing must match bit for bit; outputs within max |err| <= 2e-2 * rms and
// sum |err| <= 2e-3 * sum |ref| of the oracle's fp64 values.
#include <math.h>
#include <stdio.h>
#include <string.h>

#include <cuda_bf16.h>
#include <vector>

#include "common.cuh"
#include "selftest_expected.h"

namespace moe {
namespace {

namespace X = selftest_expected;

constexpr int ST_TMAX = 128;
constexpr double ST_MAX_REL_RMS = 2e-2;
constexpr double ST_MEAN_REL = 2e-3;
constexpr double ST_WEIGHT_ATOL = 1e-6;

enum : uint32_t {
    TAG_TOKENS = 1, TAG_ROUTER = 2, TAG_CODEBOOK = 3,
    TAG_VQ2_CODES = 16, TAG_VQ2_SCALES = 48, TAG_FP4_CODES = 80, TAG_FP4_SCALES = 112,
};
enum : int { V_BF16_32, V_BF16_2048, V_FP16_32, V_BYTE, V_VQ2_SCALE, V_UE8M0 };

__device__ __forceinline__ uint64_t splitmix64(uint64_t s) {
    uint64_t z = s + 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

__global__ void st_fill(void* dst, int kind, uint32_t tag, int n, int period) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const uint64_t v = splitmix64(((uint64_t)tag << 32) | (uint64_t)(i % period));
    const int g = (int)(v & 63) + (int)((v >> 8) & 63) + (int)((v >> 16) & 63) + (int)((v >> 24) & 63) - 126;
    switch (kind) {
        case V_BF16_32:
            static_cast<uint16_t*>(dst)[i] = __bfloat16_as_ushort(__float2bfloat16_rn((float)g * 0.03125f));
            break;
        case V_BF16_2048:
            static_cast<uint16_t*>(dst)[i] = __bfloat16_as_ushort(__float2bfloat16_rn((float)g * (1.0f / 2048)));
            break;
        case V_FP16_32:
            static_cast<uint16_t*>(dst)[i] = __half_as_ushort(__float2half_rn((float)g * 0.03125f));
            break;
        case V_BYTE:
            static_cast<uint8_t*>(dst)[i] = (uint8_t)(v & 255);
            break;
        case V_VQ2_SCALE:
            static_cast<uint16_t*>(dst)[i] = __half_as_ushort(__float2half_rn((float)(40 + v % 124) * (1.0f / 8192)));
            break;
        default:  // V_UE8M0
            static_cast<uint8_t*>(dst)[i] = (uint8_t)(118 + v % 3);
            break;
    }
}

// Bump allocator over one device allocation (256-byte aligned pieces).
struct Arena {
    char* base = nullptr;
    size_t off = 0;
    template <class T>
    T* take(size_t count) {
        T* p = reinterpret_cast<T*>(base + off);
        off += (count * sizeof(T) + 255) & ~size_t(255);
        return p;
    }
};

struct Buffers {
    uint16_t *cb, *wr, *x;
    uint8_t* stage_codes;
    void* stage_scales;
    uint8_t *vq2_codes[X::E][3], *fp4_codes[X::E][3];
    uint16_t* vq2_scales[X::E][3];
    uint8_t* fp4_scales[X::E][3];
    float *logits, *weights, *ypair, *out;
    int32_t *ids, *offsets, *sorted_pair, *pair_to_sorted;
    uint8_t* status;
    void *route_ws, *perm_ws, *ffn_ws;
    size_t route_ws_bytes, perm_ws_bytes, ffn_ws_bytes;
};

// Lays out (base == nullptr: only measures) every buffer; returns the size.
size_t layout(char* base, Buffers& b) {
    const int H = X::H, I = X::I, E = X::E, k = X::K, P = ST_TMAX * X::K;
    Arena a;
    a.base = base;
    b.cb = a.take<uint16_t>(512);
    b.wr = a.take<uint16_t>((size_t)E * H);
    b.x = a.take<uint16_t>((size_t)ST_TMAX * H);
    b.stage_codes = a.take<uint8_t>((size_t)H * I / 2);
    b.stage_scales = a.take<uint16_t>((size_t)H * I / 32);
    const int rows[3] = {I, I, H}, K[3] = {H, H, I};
    for (int e = 0; e < E; ++e)
        for (int m = 0; m < 3; ++m) {
            b.vq2_codes[e][m] = a.take<uint8_t>((size_t)rows[m] * K[m] / 4);
            b.vq2_scales[e][m] = a.take<uint16_t>((size_t)rows[m] * K[m] / 128);
            b.fp4_codes[e][m] = a.take<uint8_t>((size_t)rows[m] * K[m] / 2);
            b.fp4_scales[e][m] = a.take<uint8_t>((size_t)rows[m] * K[m] / 32);
        }
    b.logits = a.take<float>((size_t)ST_TMAX * E);
    b.weights = a.take<float>(P);
    b.ypair = a.take<float>((size_t)P * H);
    b.out = a.take<float>((size_t)ST_TMAX * H);
    b.ids = a.take<int32_t>(P);
    b.offsets = a.take<int32_t>(E + 1);
    b.sorted_pair = a.take<int32_t>(P);
    b.pair_to_sorted = a.take<int32_t>(P);
    b.status = a.take<uint8_t>(P);
    b.route_ws_bytes = moe_route_workspace_size(ST_TMAX, k, E);
    b.perm_ws_bytes = moe_permute_workspace_size(ST_TMAX, k, E);
    b.ffn_ws_bytes = moe_vq2_expert_ffn_workspace_size(ST_TMAX, k, E, H, I);
    b.route_ws = a.take<char>(b.route_ws_bytes);
    b.perm_ws = a.take<char>(b.perm_ws_bytes + 16);
    b.ffn_ws = a.take<char>(b.ffn_ws_bytes);
    return a.off;
}

#define ST_TRY(expr)                             \
    do {                                         \
        moe_status st_ = (expr);                 \
        if (st_ != MOE_OK) return st_;           \
    } while (0)
#define ST_CUDA(expr, what)                                       \
    do {                                                          \
        cudaError_t e_ = (expr);                                  \
        if (e_ != cudaSuccess) return cuda_status(e_, what);      \
    } while (0)

moe_status fill(void* dst, int kind, uint32_t tag, int n, int period, cudaStream_t s) {
    st_fill<<<(n + 255) / 256, 256, 0, s>>>(dst, kind, tag, n, period);
    count_launch();
    MOE_LAUNCH_CHECK("moe_selftest: fill");
    return MOE_OK;
}

// Draws and packs the weights of both formats for every expert.
moe_status draw_weights(Buffers& b, cudaStream_t s) {
    const int H = X::H, I = X::I, E = X::E;
    ST_TRY(fill(b.cb, V_FP16_32, TAG_CODEBOOK, 512, 512, s));
    ST_TRY(fill(b.wr, V_BF16_2048, TAG_ROUTER, E * H, E * H, s));
    const int rows[3] = {I, I, H}, K[3] = {H, H, I};
    for (int e = 0; e < E; ++e)
        for (int m = 0; m < 3; ++m) {
            const uint32_t t = 4u * e + m;
            int nc = rows[m] * K[m] / 4, ns = rows[m] * K[m] / 128;
            ST_TRY(fill(b.stage_codes, V_BYTE, TAG_VQ2_CODES + t, nc, nc, s));
            ST_TRY(fill(b.stage_scales, V_VQ2_SCALE, TAG_VQ2_SCALES + t, ns, ns, s));
            ST_TRY(moe_vq2_pack(b.stage_codes, static_cast<uint16_t*>(b.stage_scales), rows[m], K[m],
                                b.vq2_codes[e][m], b.vq2_scales[e][m], s));
            nc = rows[m] * K[m] / 2;
            ns = rows[m] * K[m] / 32;
            ST_TRY(fill(b.stage_codes, V_BYTE, TAG_FP4_CODES + t, nc, nc, s));
            ST_TRY(fill(b.stage_scales, V_UE8M0, TAG_FP4_SCALES + t, ns, ns, s));
            ST_TRY(moe_fp4_pack(b.stage_codes, static_cast<uint8_t*>(b.stage_scales), rows[m], K[m],
                                b.fp4_codes[e][m], b.fp4_scales[e][m], s));
        }
    return MOE_OK;
}

moe_status set_experts(moe_slot_table* t, const Buffers& b, bool mixed, cudaStream_t s) {
    for (int e = 0; e < X::E; ++e) {
        const bool fp4 = mixed && (e & 1);
        moe_expert_desc d;
        d.format = fp4 ? MOE_FMT_FP4 : MOE_FMT_VQ2;
        for (int m = 0; m < 3; ++m) {
            d.codes[m] = fp4 ? (const void*)b.fp4_codes[e][m] : (const void*)b.vq2_codes[e][m];
            d.scales[m] = fp4 ? (const void*)b.fp4_scales[e][m] : (const void*)b.vq2_scales[e][m];
        }
        ST_TRY(moe_slot_table_set(t, e, &d, s));
    }
    return MOE_OK;
}

template <class T>
moe_status fetch(std::vector<T>& h, const T* d, size_t n, cudaStream_t s) {
    h.resize(n);
    ST_CUDA(cudaMemcpyAsync(h.data(), d, n * sizeof(T), cudaMemcpyDeviceToHost, s), "moe_selftest: copy");
    ST_CUDA(cudaStreamSynchronize(s), "moe_selftest: synchronize");
    return MOE_OK;
}

moe_status mismatch(const char* what) {
    set_error("moe_selftest: %s", what);
    return MOE_ERR_MISMATCH;
}

// Routing of T tokens (rows repeating the four) against the expected one.
moe_status check_routing(const Buffers& b, int T, bool with_logits, const char* name, cudaStream_t s) {
    const int k = X::K, E = X::E, P = T * k;
    std::vector<int32_t> ids, off, sp, p2s;
    std::vector<float> w;
    ST_TRY(fetch(ids, b.ids, P, s));
    ST_TRY(fetch(off, b.offsets, E + 1, s));
    ST_TRY(fetch(sp, b.sorted_pair, P, s));
    ST_TRY(fetch(p2s, b.pair_to_sorted, P, s));
    ST_TRY(fetch(w, b.weights, P, s));
    char msg[256];
    if (with_logits) {
        std::vector<float> lg;
        ST_TRY(fetch(lg, b.logits, (size_t)T * E, s));
        for (int i = 0; i < T * E; ++i) {
            uint32_t bits;
            memcpy(&bits, &lg[i], 4);
            if (bits != X::logits_bits[i % (X::T * E)]) {
                snprintf(msg, sizeof msg, "%s: logits[%d] bits 0x%08x, expected 0x%08x", name, i, bits,
                         X::logits_bits[i % (X::T * E)]);
                return mismatch(msg);
            }
        }
    }
    // expected ids / offsets / permutation of T = 4r tokens (r repeats, or one token)
    std::vector<int> cnt(E + 1, 0);
    for (int p = 0; p < P; ++p) {
        const int want = X::ids[p % (X::T * k)];
        if (ids[p] != want) {
            snprintf(msg, sizeof msg, "%s: ids[%d] = %d, expected %d", name, p, ids[p], want);
            return mismatch(msg);
        }
        const double dw = fabs((double)w[p] - X::weights[p % (X::T * k)]);
        if (!(dw <= ST_WEIGHT_ATOL)) {
            snprintf(msg, sizeof msg, "%s: weights[%d] off by %.3g", name, p, dw);
            return mismatch(msg);
        }
        cnt[want + 1]++;
    }
    for (int e = 0; e < E; ++e) cnt[e + 1] += cnt[e];
    for (int e = 0; e <= E; ++e)
        if (off[e] != cnt[e]) {
            snprintf(msg, sizeof msg, "%s: expert_offsets[%d] = %d, expected %d", name, e, off[e], cnt[e]);
            return mismatch(msg);
        }
    // stable counting sort: within an expert, pairs in increasing index
    std::vector<int> cur(cnt.begin(), cnt.end() - 1);
    for (int p = 0; p < P; ++p) {
        const int pos = cur[ids[p]]++;
        if (sp[pos] != p || p2s[p] != pos) {
            snprintf(msg, sizeof msg, "%s: permutation differs at pair %d", name, p);
            return mismatch(msg);
        }
    }
    if (T == X::T) {  // the stored permutation of the four tokens, as the oracle wrote it
        for (int e = 0; e <= E; ++e)
            if (off[e] != X::expert_offsets[e]) return mismatch("route4: offsets differ from the stored ones");
        for (int p = 0; p < P; ++p)
            if (sp[p] != X::sorted_pair[p] || p2s[p] != X::pair_to_sorted[p])
                return mismatch("route4: permutation differs from the stored one");
    }
    return MOE_OK;
}

// out of T tokens against ref rows (row t compares with ref row first + t mod 4).
moe_status check_out(const Buffers& b, int T, int first, const double* ref, const char* name, cudaStream_t s) {
    const int H = X::H;
    std::vector<float> out;
    ST_TRY(fetch(out, b.out, (size_t)T * H, s));
    double ss = 0, sref = 0, serr = 0, emax = 0;
    bool finite = true;
    for (int t = 0; t < T; ++t)
        for (int h = 0; h < H; ++h) {
            const double r = ref[(size_t)((first + t) % X::T) * H + h];
            const double e = fabs((double)out[(size_t)t * H + h] - r);
            finite = finite && isfinite(out[(size_t)t * H + h]);
            ss += r * r;
            sref += fabs(r);
            serr += e;
            emax = e > emax ? e : emax;
        }
    const double rms = sqrt(ss / ((double)T * H));
    if (!finite || !(emax <= ST_MAX_REL_RMS * rms) || !(serr <= ST_MEAN_REL * sref)) {
        char msg[256];
        snprintf(msg, sizeof msg, "%s: max |err| %.3g (rms %.3g), mean relative error %.3g%s", name, emax, rms,
                 sref > 0 ? serr / sref : 0.0, finite ? "" : ", non-finite output");
        return mismatch(msg);
    }
    return MOE_OK;
}

moe_status check_status(const Buffers& b, int P, bool partial, const char* name, cudaStream_t s) {
    std::vector<uint8_t> st;
    ST_TRY(fetch(st, b.status, P, s));
    for (int p = 0; p < P; ++p) {
        const uint8_t want = partial ? X::resident[X::ids[p % (X::T * X::K)]] : 1;
        if (st[p] != want) {
            char msg[160];
            snprintf(msg, sizeof msg, "%s: pair_status[%d] = %d, expected %d", name, p, st[p], want);
            return mismatch(msg);
        }
    }
    return MOE_OK;
}

moe_status route(const Buffers& b, int T, cudaStream_t s) {
    return moe_route(b.x, b.wr, nullptr, T, X::H, X::E, X::K, 1, b.logits, b.ids, b.weights, b.offsets,
                     b.sorted_pair, b.pair_to_sorted, b.route_ws, b.route_ws_bytes, s);
}

// Per-pair FFN of the routed batch, then the combine into b.out.
moe_status ffn_combine(const moe_slot_table* t, const Buffers& b, int T, cudaStream_t s) {
    ST_TRY(moe_vq2_expert_ffn(t, b.x, b.offsets, b.sorted_pair, b.weights, T, X::K, MOE_PER_PAIR, b.ypair,
                              b.status, b.ffn_ws, b.ffn_ws_bytes, s));
    return moe_combine(b.ypair, b.pair_to_sorted, b.weights, b.status, T, X::K, X::H, b.out, nullptr, s);
}

moe_status run_cases(moe_slot_table* vq2, moe_slot_table* mixed, const Buffers& b, cudaStream_t s) {
    const int H = X::H, E = X::E, k = X::K;
    ST_TRY(fill(b.x, V_BF16_32, TAG_TOKENS, ST_TMAX * H, X::T * H, s));
    ST_CUDA(cudaMemsetAsync(b.route_ws, 0, b.route_ws_bytes, s), "moe_selftest: memset");

    // routing, step by step and fused
    ST_TRY(moe_router_logits(b.x, b.wr, nullptr, b.logits, X::T, H, E, s));
    ST_TRY(moe_route_topk(b.logits, X::T, E, k, 1, b.ids, b.weights, s));
    ST_TRY(moe_permute(b.ids, X::T, k, E, b.offsets, b.sorted_pair, b.pair_to_sorted, b.perm_ws,
                       b.perm_ws_bytes, s));
    ST_TRY(check_routing(b, X::T, true, "route4", s));
    ST_CUDA(cudaMemsetAsync(b.ids, 0xFF, sizeof(int32_t) * X::T * k, s), "moe_selftest: memset");
    ST_TRY(route(b, X::T, s));
    ST_TRY(check_routing(b, X::T, true, "route4f", s));

    // all-VQ2 layer, 4 tokens: per pair + combine, then fused scatter
    ST_TRY(ffn_combine(vq2, b, X::T, s));
    ST_TRY(check_status(b, X::T * k, false, "vq2_t4", s));
    ST_TRY(check_out(b, X::T, 0, X::out_vq2, "vq2_t4", s));
    ST_CUDA(cudaMemsetAsync(b.out, 0, sizeof(float) * X::T * H, s), "moe_selftest: memset");
    ST_TRY(moe_vq2_expert_ffn(vq2, b.x, b.offsets, b.sorted_pair, b.weights, X::T, k, MOE_FUSED_SCATTER, b.out,
                              b.status, b.ffn_ws, b.ffn_ws_bytes, s));
    ST_TRY(check_out(b, X::T, 0, X::out_vq2, "vq2_scat", s));

    // mixed-format layer, 4 tokens
    ST_TRY(ffn_combine(mixed, b, X::T, s));
    ST_TRY(check_out(b, X::T, 0, X::out_mixed, "mix_t4", s));

    // token 0 alone: fused routing, expert FFN with the combine inside
    ST_TRY(route(b, 1, s));
    ST_TRY(check_routing(b, 1, true, "route1", s));
    ST_TRY(moe_vq2_expert_ffn_combine(vq2, b.x, b.offsets, b.sorted_pair, b.pair_to_sorted, b.weights, 1, k,
                                      b.ypair, b.status, b.out, nullptr, b.ffn_ws, b.ffn_ws_bytes, s));
    ST_TRY(check_out(b, 1, 0, X::out_vq2, "vq2_t1", s));

    // 16 tokens: 4 or 8 per routed expert (mma.sync)
    ST_TRY(route(b, 16, s));
    ST_TRY(check_routing(b, 16, true, "route16", s));
    ST_TRY(ffn_combine(vq2, b, 16, s));
    ST_TRY(check_out(b, 16, 0, X::out_vq2, "vq2_t16", s));

    // 128 tokens: every routed expert takes at least 32 of them
    ST_TRY(route(b, ST_TMAX, s));
    ST_TRY(check_routing(b, ST_TMAX, true, "route128", s));
    ST_TRY(ffn_combine(vq2, b, ST_TMAX, s));
    ST_TRY(check_out(b, ST_TMAX, 0, X::out_vq2, "vq2_t128", s));
    ST_TRY(ffn_combine(mixed, b, ST_TMAX, s));
    ST_TRY(check_out(b, ST_TMAX, 0, X::out_mixed, "mix_t128", s));

    // the resident subset: experts with resident[e] == 0 evicted
    ST_TRY(route(b, X::T, s));
    for (int e = 0; e < E; ++e)
        if (!X::resident[e]) ST_TRY(moe_slot_table_evict(vq2, e, s));
    ST_TRY(ffn_combine(vq2, b, X::T, s));
    ST_TRY(check_status(b, X::T * k, true, "partial", s));
    ST_TRY(check_out(b, X::T, 0, X::partial_vq2, "partial", s));
    return MOE_OK;
}

// The bounded-wait pattern of the kernels (a limited loop over
// mbarrier.try_wait, then an error code and a return), on mbarriers that
// nothing completes, with both wait primitives the kernels use: plain
// try_wait and try_wait with a 1 us suspend hint.  Short limits (64 and 256
// tries), so the check ends in well under a second whatever the hardware's
// suspend time; the time each wait took (globaltimer, ns) is reported.
__device__ __forceinline__ uint64_t gtimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__global__ void wait_timeout_kernel(int* codes, unsigned long long* ns) {
    __shared__ uint64_t bars[2];
    if (threadIdx.x != 0) return;
    mbar_init(smem_u32(&bars[0]), 1);
    mbar_init(smem_u32(&bars[1]), 1);
    mbar_fence_init();
    codes[0] = 0;
    codes[1] = 0;
    uint64_t t0 = gtimer_ns();
    bool ok = false;
#pragma unroll 1
    for (int it = 0; it < 64 && !ok; ++it) ok = mbar_try_wait(smem_u32(&bars[0]), 0);
    if (!ok) atomicExch(codes + 0, MOE_DEVERR_WAIT_FULL);
    codes[2] = ok ? 1 : 0;
    uint64_t t1 = gtimer_ns();
    ns[0] = t1 - t0;
    ok = false;
#pragma unroll 1
    for (int it = 0; it < 256 && !ok; ++it) ok = mbar_try_wait_sleep(smem_u32(&bars[1]), 0, 1000u);
    if (!ok) atomicExch(codes + 1, MOE_DEVERR_WAIT_EMPTY);
    codes[3] = ok ? 1 : 0;
    ns[1] = gtimer_ns() - t1;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status moe_selftest_wait_timeout(int* codes, cudaStream_t stream) {
    MOE_CHECK_ARG(codes, "moe_selftest_wait_timeout: null codes");
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    cudaError_t ce = cudaStreamIsCapturing(stream, &cap);
    if (ce != cudaSuccess) return cuda_status(ce, "moe_selftest_wait_timeout: stream");
    MOE_CHECK_ARG(cap == cudaStreamCaptureStatusNone, "moe_selftest_wait_timeout: the stream is being captured");
    int* d = nullptr;
    ce = cudaMalloc(&d, 4 * sizeof(int) + 2 * sizeof(unsigned long long));
    if (ce != cudaSuccess) {
        cudaGetLastError();
        set_error("moe_selftest_wait_timeout: cudaMalloc: %s", cudaGetErrorString(ce));
        return MOE_ERR_NO_MEM;
    }
    unsigned long long* dns = reinterpret_cast<unsigned long long*>(d + 4);
    unsigned long long hns[2] = {0, 0};
    wait_timeout_kernel<<<1, 32, 0, stream>>>(d, dns);
    ce = cudaGetLastError();
    if (ce == cudaSuccess) ce = cudaMemcpyAsync(codes, d, 4 * sizeof(int), cudaMemcpyDeviceToHost, stream);
    if (ce == cudaSuccess) ce = cudaMemcpyAsync(hns, dns, sizeof(hns), cudaMemcpyDeviceToHost, stream);
    if (ce == cudaSuccess) ce = cudaStreamSynchronize(stream);
    cudaFree(d);
    if (ce != cudaSuccess) return cuda_status(ce, "moe_selftest_wait_timeout");
    codes[4] = (int)(hns[0] / 1000 > 0x7fffffff ? 0x7fffffff : hns[0] / 1000);  // us
    codes[5] = (int)(hns[1] / 1000 > 0x7fffffff ? 0x7fffffff : hns[1] / 1000);
    if (codes[0] != MOE_DEVERR_WAIT_FULL || codes[1] != MOE_DEVERR_WAIT_EMPTY || codes[2] != 0 || codes[3] != 0) {
        set_error("moe_selftest_wait_timeout: codes %d %d, waits returned %d %d", codes[0], codes[1], codes[2],
                  codes[3]);
        return MOE_ERR_MISMATCH;
    }
    return MOE_OK;
}

extern "C" moe_status moe_selftest(cudaStream_t stream) {
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    cudaError_t ce = cudaStreamIsCapturing(stream, &cap);
    if (ce != cudaSuccess) return cuda_status(ce, "moe_selftest: stream");
    MOE_CHECK_ARG(cap == cudaStreamCaptureStatusNone, "moe_selftest: the stream is being captured");
    Buffers b;
    const size_t bytes = layout(nullptr, b);
    char* base = nullptr;
    ce = cudaMalloc(&base, bytes);
    if (ce != cudaSuccess) {
        cudaGetLastError();
        set_error("moe_selftest: cudaMalloc of %zu bytes: %s", bytes, cudaGetErrorString(ce));
        return MOE_ERR_NO_MEM;
    }
    layout(base, b);
    moe_slot_table *vq2 = nullptr, *mixed = nullptr;
    moe_status st = moe_slot_table_create(X::E, X::H, X::I, b.cb, &vq2);
    if (st == MOE_OK) st = moe_slot_table_create(X::E, X::H, X::I, b.cb, &mixed);
    if (st == MOE_OK) st = draw_weights(b, stream);
    if (st == MOE_OK) st = set_experts(vq2, b, false, stream);
    if (st == MOE_OK) st = set_experts(mixed, b, true, stream);
    if (st == MOE_OK) st = run_cases(vq2, mixed, b, stream);
    // whatever happened, let the enqueued work finish before freeing its memory
    const cudaError_t se = cudaStreamSynchronize(stream);
    if (st == MOE_OK && se != cudaSuccess) st = cuda_status(se, "moe_selftest: synchronize");
    if (vq2) moe_slot_table_destroy(vq2);
    if (mixed) moe_slot_table_destroy(mixed);
    cudaFree(base);
    return st;
}
