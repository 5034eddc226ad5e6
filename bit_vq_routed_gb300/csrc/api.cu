// C ABI entry points: host-side argument checks, the error message, the
// slot table; each hot-path call enqueues kernels only (no host sync).
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>

#include <atomic>

#include "common.cuh"
#include "permute.cuh"

namespace moe {

static std::atomic<uint64_t> g_launches{0};

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

static thread_local char g_err[512] = "";

void set_error(const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
}

moe_status cuda_status(cudaError_t e, const char* what) {
    set_error("%s: %s", what, cudaGetErrorString(e));
    return MOE_ERR_CUDA;
}

int num_sms() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 1;
    return n > 0 ? n : 1;
}

}  // namespace moe

using namespace moe;

extern "C" {

int moe_version(void) { return 1; }

uint64_t moe_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

const char* moe_last_error(void) { return g_err; }

moe_status moe_vq2_pack(const uint8_t* codes, const uint16_t* scales, int rows, int K,
                        uint8_t* packed_codes, uint16_t* packed_scales, cudaStream_t stream) {
    MOE_CHECK_ARG(codes && scales && packed_codes && packed_scales, "moe_vq2_pack: null pointer");
    MOE_CHECK_ARG(rows > 0 && K > 0, "moe_vq2_pack: rows=%d K=%d must be positive", rows, K);
    MOE_CHECK_SUPPORTED(rows % 16 == 0 && K % 128 == 0,
                        "moe_vq2_pack: need rows %% 16 == 0 and K %% 128 == 0 (rows=%d K=%d)", rows, K);
    MOE_CHECK_SUPPORTED(aligned16(codes) && aligned16(packed_codes) && aligned16(scales) &&
                            aligned16(packed_scales),
                        "moe_vq2_pack: pointers must be 16-byte aligned");
    return launch_vq2_pack(codes, scales, rows, K, packed_codes, packed_scales, stream);
}

moe_status moe_fp4_pack(const uint8_t* codes, const uint8_t* scales, int rows, int K,
                        uint8_t* packed_codes, uint8_t* packed_scales, cudaStream_t stream) {
    MOE_CHECK_ARG(codes && scales && packed_codes && packed_scales, "moe_fp4_pack: null pointer");
    MOE_CHECK_ARG(rows > 0 && K > 0, "moe_fp4_pack: rows=%d K=%d must be positive", rows, K);
    MOE_CHECK_SUPPORTED(rows % 16 == 0 && K % 64 == 0,
                        "moe_fp4_pack: need rows %% 16 == 0 and K %% 64 == 0 (rows=%d K=%d)", rows, K);
    MOE_CHECK_SUPPORTED(aligned16(codes) && aligned16(packed_codes) && aligned16(scales) &&
                            aligned16(packed_scales),
                        "moe_fp4_pack: pointers must be 16-byte aligned");
    return launch_fp4_pack(codes, scales, rows, K, packed_codes, packed_scales, stream);
}

moe_status moe_slot_table_create(int num_experts, int H, int I, const uint16_t* codebook,
                                 moe_slot_table** out) {
    MOE_CHECK_ARG(out, "moe_slot_table_create: out is null");
    *out = nullptr;
    MOE_CHECK_ARG(codebook, "moe_slot_table_create: codebook is null");
    MOE_CHECK_ARG(num_experts > 0 && num_experts <= 1024,
                  "moe_slot_table_create: num_experts=%d must be in [1, 1024]", num_experts);
    MOE_CHECK_ARG(H > 0 && I > 0, "moe_slot_table_create: H=%d I=%d must be positive", H, I);
    MOE_CHECK_SUPPORTED(H % 256 == 0 && I % 128 == 0,
                        "moe_slot_table_create: need H %% 256 == 0 and I %% 128 == 0 (H=%d I=%d)", H, I);
    MOE_CHECK_SUPPORTED(aligned16(codebook), "moe_slot_table_create: codebook must be 16-byte aligned");
    moe_slot_table* t = (moe_slot_table*)calloc(1, sizeof(moe_slot_table));
    if (!t) {
        set_error("moe_slot_table_create: out of host memory");
        return MOE_ERR_NO_MEM;
    }
    t->h.E = num_experts;
    t->h.H = H;
    t->h.I = I;
    t->h.codebook = codebook;
    t->h.h_fmt = (uint8_t*)calloc((size_t)num_experts, 1);
    if (!t->h.h_fmt) {
        free(t);
        set_error("moe_slot_table_create: out of host memory");
        return MOE_ERR_NO_MEM;
    }
    cudaError_t e = cudaMalloc(&t->h.d_desc, sizeof(SlotDesc) * (size_t)num_experts);
    if (e != cudaSuccess) {
        free(t->h.h_fmt);
        free(t);
        set_error("moe_slot_table_create: cudaMalloc: %s", cudaGetErrorString(e));
        return MOE_ERR_NO_MEM;
    }
    e = cudaMemset(t->h.d_desc, 0, sizeof(SlotDesc) * (size_t)num_experts);
    if (e != cudaSuccess) {
        cudaFree(t->h.d_desc);
        free(t->h.h_fmt);
        free(t);
        return cuda_status(e, "moe_slot_table_create: cudaMemset");
    }
    *out = t;
    return MOE_OK;
}

moe_status moe_slot_table_set(moe_slot_table* t, int expert_id, const moe_expert_desc* d,
                              cudaStream_t stream) {
    MOE_CHECK_ARG(t && d, "moe_slot_table_set: null table or descriptor");
    MOE_CHECK_ARG(expert_id >= 0 && expert_id < t->h.E, "moe_slot_table_set: expert_id=%d out of [0, %d)",
                  expert_id, t->h.E);
    MOE_CHECK_ARG(d->format == MOE_FMT_VQ2 || d->format == MOE_FMT_FP4,
                  "moe_slot_table_set: unknown format %d", d->format);
    SlotDesc s;
    s.format = d->format;
    s.resident = 1;
    for (int m = 0; m < 3; ++m) {
        MOE_CHECK_ARG(d->codes[m] && d->scales[m], "moe_slot_table_set: null buffer for matrix %d", m);
        MOE_CHECK_SUPPORTED(aligned16(d->codes[m]) && aligned16(d->scales[m]),
                            "moe_slot_table_set: buffers must be 16-byte aligned (matrix %d)", m);
        s.codes[m] = d->codes[m];
        s.scales[m] = d->scales[m];
    }
    moe_status st = launch_slot_set(t->h.d_desc, expert_id, s, stream);
    if (st == MOE_OK) {
        t->h.n_fp4 += (d->format == MOE_FMT_FP4) - (t->h.h_fmt[expert_id] == 1 + MOE_FMT_FP4);
        t->h.h_fmt[expert_id] = (uint8_t)(1 + d->format);
    }
    return st;
}

moe_status moe_slot_table_evict(moe_slot_table* t, int expert_id, cudaStream_t stream) {
    MOE_CHECK_ARG(t, "moe_slot_table_evict: null table");
    MOE_CHECK_ARG(expert_id >= 0 && expert_id < t->h.E,
                  "moe_slot_table_evict: expert_id=%d out of [0, %d)", expert_id, t->h.E);
    SlotDesc s = {};
    moe_status st = launch_slot_set(t->h.d_desc, expert_id, s, stream);
    if (st == MOE_OK) {
        t->h.n_fp4 -= (t->h.h_fmt[expert_id] == 1 + MOE_FMT_FP4);
        t->h.h_fmt[expert_id] = 0;
    }
    return st;
}

int moe_slot_table_resident(const moe_slot_table* t, int expert_id) {
    if (!t || expert_id < 0 || expert_id >= t->h.E) {
        set_error("moe_slot_table_resident: null table or expert_id=%d out of range", expert_id);
        return MOE_ERR_INVALID_ARG;
    }
    return t->h.h_fmt[expert_id] != 0 ? 1 : 0;
}

moe_status moe_confidence_gate(const moe_slot_table* table, const int32_t* ids, const float* weights, int T, int k,
                               int E, float tau, int32_t* gated_ids, cudaStream_t stream) {
    MOE_CHECK_ARG(table, "moe_confidence_gate: null table");
    MOE_CHECK_ARG(T >= 0 && k >= 1 && E >= 1, "moe_confidence_gate: T=%d k=%d E=%d", T, k, E);
    MOE_CHECK_ARG(table->h.E >= 2 * E, "moe_confidence_gate: the table has %d entries, 2E = %d needed", table->h.E,
                  2 * E);
    MOE_CHECK_ARG(!(tau != tau), "moe_confidence_gate: tau is NaN");
    if (T == 0) return MOE_OK;
    MOE_CHECK_ARG(ids && weights && gated_ids, "moe_confidence_gate: null pointer");
    long long P = (long long)T * k;
    MOE_CHECK_SUPPORTED(P <= (1 << 24), "moe_confidence_gate: T*k=%lld above 2^24", P);
    return launch_gate(table->h.d_desc, ids, weights, (int)P, E, tau, gated_ids, stream);
}

moe_status moe_accumulate(float* dst, const float* src, size_t n, cudaStream_t stream) {
    if (n == 0) return MOE_OK;
    MOE_CHECK_ARG(dst && src, "moe_accumulate: null pointer");
    return launch_accumulate(dst, src, n, stream);
}

moe_status moe_slot_table_destroy(moe_slot_table* t) {
    if (!t) return MOE_OK;
    cudaError_t e = cudaFree(t->h.d_desc);
    free(t->h.h_fmt);
    free(t);
    if (e != cudaSuccess) return cuda_status(e, "moe_slot_table_destroy: cudaFree");
    return MOE_OK;
}

moe_status moe_router_logits(const uint16_t* x, const uint16_t* w_router, const float* bias,
                             float* logits, int T, int H, int E, cudaStream_t stream) {
    MOE_CHECK_ARG(T >= 0 && H > 0 && E > 0, "moe_router_logits: T=%d H=%d E=%d", T, H, E);
    if (T == 0) return MOE_OK;
    MOE_CHECK_ARG(x && w_router && logits, "moe_router_logits: null pointer");
    MOE_CHECK_SUPPORTED(H % 256 == 0, "moe_router_logits: H=%d must be a multiple of 256", H);
    MOE_CHECK_SUPPORTED(aligned16(x) && aligned16(w_router) && aligned16(logits) && aligned16(bias),
                        "moe_router_logits: pointers must be 16-byte aligned");
    return launch_router_logits(x, w_router, bias, logits, T, H, E, stream);
}

moe_status moe_route_topk(const float* logits, int T, int E, int k, int renormalize, int32_t* ids,
                          float* weights, cudaStream_t stream) {
    MOE_CHECK_ARG(T >= 0 && E > 0, "moe_route_topk: T=%d E=%d", T, E);
    MOE_CHECK_ARG(k >= 1 && k <= E && k <= 32, "moe_route_topk: k=%d must be in [1, min(E, 32)]", k);
    MOE_CHECK_SUPPORTED(E <= 1024, "moe_route_topk: E=%d above 1024", E);
    MOE_CHECK_ARG(renormalize == 0 || renormalize == 1, "moe_route_topk: renormalize must be 0 or 1");
    if (T == 0) return MOE_OK;
    MOE_CHECK_ARG(logits && ids && weights, "moe_route_topk: null pointer");
    return launch_route_topk(logits, T, E, k, renormalize, ids, weights, stream);
}

// The fused routing's counter, then the permutation's chunk arrays.
size_t moe_route_workspace_size(int T, int k, int E) {
    const long long P = (long long)T * k;
    return 256 + (P > 0 && P <= (1 << 24) && E > 0 ? permute_ws_bytes((int)P, E) : 0);
}

moe_status moe_route(const uint16_t* x, const uint16_t* w_router, const float* bias, int T, int H, int E, int k,
                     int renormalize, float* logits, int32_t* ids, float* weights, int32_t* expert_offsets,
                     int32_t* sorted_pair, int32_t* pair_to_sorted, void* ws, size_t ws_bytes,
                     cudaStream_t stream) {
    MOE_CHECK_ARG(T >= 0 && H > 0 && E > 0, "moe_route: T=%d H=%d E=%d", T, H, E);
    MOE_CHECK_ARG(k >= 1 && k <= E && k <= 32, "moe_route: k=%d must be in [1, min(E, 32)]", k);
    MOE_CHECK_SUPPORTED(E <= 1024, "moe_route: E=%d above 1024", E);
    MOE_CHECK_ARG(renormalize == 0 || renormalize == 1, "moe_route: renormalize must be 0 or 1");
    MOE_CHECK_SUPPORTED((long long)T * k <= (1 << 24), "moe_route: T*k above 2^24");
    MOE_CHECK_ARG(expert_offsets, "moe_route: expert_offsets is null");
    if (T == 0) return launch_permute(ids, 0, E, expert_offsets, sorted_pair, pair_to_sorted, stream);
    MOE_CHECK_ARG(x && w_router && logits && ids && weights && sorted_pair && pair_to_sorted,
                  "moe_route: null pointer");
    MOE_CHECK_SUPPORTED(H % 256 == 0, "moe_route: H=%d must be a multiple of 256", H);
    MOE_CHECK_SUPPORTED(aligned16(x) && aligned16(w_router) && aligned16(logits) && aligned16(bias),
                        "moe_route: pointers must be 16-byte aligned");
    if (route_cluster_ok(T, H, E))
        return launch_route_cluster(x, w_router, bias, H, E, k, renormalize, logits, ids, weights, expert_offsets,
                                    sorted_pair, pair_to_sorted, stream);
    if (route_fused_ok(T, k, H, E)) {
        if (!ws || ws_bytes < moe_route_workspace_size(T, k, E)) {
            set_error("moe_route: workspace of %zu bytes, %zu required", ws_bytes, moe_route_workspace_size(T, k, E));
            return MOE_ERR_WORKSPACE;
        }
        return launch_route_fused(x, w_router, bias, T, H, E, k, renormalize, logits, ids, weights, expert_offsets,
                                  sorted_pair, pair_to_sorted, static_cast<int*>(ws), stream);
    }
    moe_status st = launch_router_logits(x, w_router, bias, logits, T, H, E, stream);
    if (st != MOE_OK) return st;
    if ((st = launch_route_topk(logits, T, E, k, renormalize, ids, weights, stream)) != MOE_OK) return st;
    // (the permutation's chunk arrays follow the fused routing's counter)
    const bool pws = ws && ws_bytes >= 256 + permute_ws_bytes(T * k, E);
    return launch_permute_ws(ids, T * k, E, expert_offsets, sorted_pair, pair_to_sorted, stream,
                             pws ? static_cast<char*>(ws) + 256 : nullptr, pws ? ws_bytes - 256 : 0);
}

size_t moe_permute_workspace_size(int T, int k, int E) {
    const long long P = (long long)T * k;
    return P > 0 && P <= (1 << 24) && E > 0 ? permute_ws_bytes((int)P, E) : 0;
}

moe_status moe_permute(const int32_t* ids, int T, int k, int E, int32_t* expert_offsets,
                       int32_t* sorted_pair, int32_t* pair_to_sorted, void* ws, size_t ws_bytes,
                       cudaStream_t stream) {
    MOE_CHECK_ARG(T >= 0 && k >= 1 && E >= 1, "moe_permute: T=%d k=%d E=%d", T, k, E);
    MOE_CHECK_SUPPORTED(E <= 1024, "moe_permute: E=%d above 1024", E);
    long long P = (long long)T * k;
    MOE_CHECK_SUPPORTED(P <= (1 << 24), "moe_permute: T*k=%lld above 2^24", P);
    MOE_CHECK_ARG(expert_offsets, "moe_permute: expert_offsets is null");
    if (P > 0) MOE_CHECK_ARG(ids && sorted_pair && pair_to_sorted, "moe_permute: null pointer");
    return launch_permute_ws(ids, (int)P, E, expert_offsets, sorted_pair, pair_to_sorted, stream, ws, ws_bytes);
}

size_t moe_vq2_expert_ffn_workspace_size(int T, int k, int E, int H, int I) {
    if (T < 0 || k < 1 || E < 1 || H < 1 || I < 1) return 0;
    return ffn_workspace_size(T, k, E, H, I);
}

moe_status moe_vq2_expert_ffn(const moe_slot_table* table, const uint16_t* x,
                              const int32_t* expert_offsets, const int32_t* sorted_pair,
                              const float* weights, int T, int k, int mode, float* out_or_ypair,
                              uint8_t* pair_status, void* ws, size_t ws_bytes, cudaStream_t stream) {
    MOE_CHECK_ARG(table, "moe_vq2_expert_ffn: null table");
    MOE_CHECK_ARG(T >= 0 && k >= 1, "moe_vq2_expert_ffn: T=%d k=%d", T, k);
    MOE_CHECK_ARG(mode == MOE_FUSED_SCATTER || mode == MOE_PER_PAIR, "moe_vq2_expert_ffn: bad mode %d", mode);
    long long P = (long long)T * k;
    MOE_CHECK_SUPPORTED(P <= (1 << 24), "moe_vq2_expert_ffn: T*k=%lld above 2^24", P);
    if (P == 0) return MOE_OK;
    MOE_CHECK_ARG(x && expert_offsets && sorted_pair && weights && out_or_ypair && pair_status,
                  "moe_vq2_expert_ffn: null pointer");
    MOE_CHECK_SUPPORTED(aligned16(x) && aligned16(out_or_ypair) && aligned16(ws),
                        "moe_vq2_expert_ffn: x, out and ws must be 16-byte aligned");
    size_t need = ffn_workspace_size(T, k, table->h.E, table->h.H, table->h.I);
    if (!ws || ws_bytes < need) {
        set_error("moe_vq2_expert_ffn: workspace %zu bytes, need %zu", ws_bytes, need);
        return MOE_ERR_WORKSPACE;
    }
    return launch_expert_ffn(&table->h, x, expert_offsets, sorted_pair, weights, T, k, mode,
                             out_or_ypair, pair_status, ws, ws_bytes, stream);
}

moe_status moe_vq2_expert_ffn_combine(const moe_slot_table* table, const uint16_t* x,
                                      const int32_t* expert_offsets, const int32_t* sorted_pair,
                                      const int32_t* pair_to_sorted, const float* weights, int T, int k,
                                      float* ypair, uint8_t* pair_status, float* out_f32, uint16_t* out_bf16,
                                      void* ws, size_t ws_bytes, cudaStream_t stream) {
    MOE_CHECK_ARG(table, "moe_vq2_expert_ffn_combine: null table");
    MOE_CHECK_ARG(T >= 0 && k >= 1, "moe_vq2_expert_ffn_combine: T=%d k=%d", T, k);
    long long P = (long long)T * k;
    MOE_CHECK_SUPPORTED(P <= (1 << 24), "moe_vq2_expert_ffn_combine: T*k=%lld above 2^24", P);
    MOE_CHECK_SUPPORTED(T <= 65535, "moe_vq2_expert_ffn_combine: T=%d above 65535", T);
    if (P == 0) return MOE_OK;
    MOE_CHECK_ARG(x && expert_offsets && sorted_pair && pair_to_sorted && weights && ypair && pair_status,
                  "moe_vq2_expert_ffn_combine: null pointer");
    MOE_CHECK_ARG(out_f32 || out_bf16, "moe_vq2_expert_ffn_combine: both outputs are null");
    MOE_CHECK_SUPPORTED(aligned16(x) && aligned16(ypair) && aligned16(ws) && aligned16(out_f32) &&
                            aligned16(out_bf16),
                        "moe_vq2_expert_ffn_combine: x, ypair, outputs and ws must be 16-byte aligned");
    size_t need = ffn_workspace_size(T, k, table->h.E, table->h.H, table->h.I);
    if (!ws || ws_bytes < need) {
        set_error("moe_vq2_expert_ffn_combine: workspace %zu bytes, need %zu", ws_bytes, need);
        return MOE_ERR_WORKSPACE;
    }
    return launch_expert_ffn(&table->h, x, expert_offsets, sorted_pair, weights, T, k, MOE_PER_PAIR, ypair,
                             pair_status, ws, ws_bytes, stream, pair_to_sorted, out_f32, out_bf16);
}

moe_status moe_combine(const float* ypair, const int32_t* pair_to_sorted, const float* weights,
                       const uint8_t* pair_status, int T, int k, int H, float* out_f32,
                       uint16_t* out_bf16, cudaStream_t stream) {
    MOE_CHECK_ARG(T >= 0 && k >= 1 && H >= 1, "moe_combine: T=%d k=%d H=%d", T, k, H);
    if (T == 0) return MOE_OK;
    MOE_CHECK_ARG(out_f32 || out_bf16, "moe_combine: both outputs are null");
    MOE_CHECK_ARG(ypair && pair_to_sorted && weights && pair_status, "moe_combine: null pointer");
    MOE_CHECK_SUPPORTED(H % 4 == 0, "moe_combine: H=%d must be a multiple of 4", H);
    MOE_CHECK_SUPPORTED(aligned16(ypair) && aligned16(out_f32) && aligned16(out_bf16),
                        "moe_combine: pointers must be 16-byte aligned");
    return launch_combine(ypair, pair_to_sorted, weights, pair_status, T, k, H, out_f32, out_bf16, stream);
}

}  // extern "C"
