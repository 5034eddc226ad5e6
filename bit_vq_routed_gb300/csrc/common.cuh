// Shared definitions of the CUDA library: status plumbing, the device-side
// slot descriptor, the packed weight layouts and small PTX wrappers.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <stdint.h>
#include <stddef.h>

#include "moe_vq2.h"

namespace moe {

// ---------------------------------------------------------------- errors
void set_error(const char* fmt, ...);
moe_status cuda_status(cudaError_t e, const char* what);

#define MOE_CHECK_ARG(cond, ...)                         \
    do {                                                 \
        if (!(cond)) {                                   \
            ::moe::set_error(__VA_ARGS__);               \
            return MOE_ERR_INVALID_ARG;                  \
        }                                                \
    } while (0)

#define MOE_CHECK_SUPPORTED(cond, ...)                   \
    do {                                                 \
        if (!(cond)) {                                   \
            ::moe::set_error(__VA_ARGS__);               \
            return MOE_ERR_UNSUPPORTED;                  \
        }                                                \
    } while (0)

#define MOE_LAUNCH_CHECK(what)                                       \
    do {                                                             \
        cudaError_t e_ = cudaGetLastError();                         \
        if (e_ != cudaSuccess) return ::moe::cuda_status(e_, what);  \
    } while (0)

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// ---------------------------------------------------------------- slot table
// One entry of the device descriptor array (64 bytes).
struct SlotDesc {
    int32_t format;    // MOE_FMT_VQ2 / MOE_FMT_FP4
    int32_t resident;  // 0 = not resident
    const void* codes[3];
    const void* scales[3];
};
static_assert(sizeof(SlotDesc) == 56, "slot descriptor layout");

struct SlotTableHost {
    int E, H, I;
    const uint16_t* codebook;  // device fp16 [128*4]
    SlotDesc* d_desc;          // device [E]
};

// ---------------------------------------------------------------- layouts
// Packed VQ2: tile (rt, kb) = 16 rows x 32 groups = 512 bytes.
__host__ __device__ inline size_t vq2_tile_offset(int rt, int kb, int KB) {
    return ((size_t)rt * KB + kb) * 512;
}
// byte inside a tile of (row-in-tile r16, group-in-block g)
__host__ __device__ inline int vq2_in_tile(int r16, int g) {
    return 16 * g + 2 * (r16 & 7) + (r16 >> 3);
}
// Packed FP4: tile (rt, kt) = 16 rows x 64 elements = 512 bytes.
// byte inside a tile holding logical byte lb (0..31 within the 64-element
// block) of row-in-tile r16
__host__ __device__ inline int fp4_in_tile(int r16, int lb) {
    int i = r16 & 7, hi = r16 >> 3;
    int s = lb >> 3, w = lb & 7, j = w & 3, up = w >> 2;
    return 16 * (4 * i + j) + 4 * s + 2 * hi + up;
}

// ---------------------------------------------------------------- PTX
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Four e2m1 pairs (one per byte of w) -> four f16x2 (low nibble -> low half).
__device__ __forceinline__ void e2m1x8_to_f16x8(uint32_t w, uint32_t& r0, uint32_t& r1,
                                                uint32_t& r2, uint32_t& r3) {
    asm("{\n"
        " .reg .b8 b0, b1, b2, b3;\n"
        " mov.b32 {b0, b1, b2, b3}, %4;\n"
        " cvt.rn.f16x2.e2m1x2 %0, b0;\n"
        " cvt.rn.f16x2.e2m1x2 %1, b1;\n"
        " cvt.rn.f16x2.e2m1x2 %2, b2;\n"
        " cvt.rn.f16x2.e2m1x2 %3, b3;\n"
        "}\n"
        : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
        : "r"(w));
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b) { return __uint_as_float(b << 16); }

// ue8m0 exponent byte -> 2^(E-127) as fp32 (E = 0 gives the subnormal 2^-127)
__device__ __forceinline__ float e8m0_to_float(uint32_t e) {
    return e ? __uint_as_float(e << 23) : __uint_as_float(0x00400000u);
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- launchers
int num_sms();

moe_status launch_router_logits(const uint16_t* x, const uint16_t* w, const float* bias, float* logits,
                                int T, int H, int E, cudaStream_t s);
moe_status launch_route_topk(const float* logits, int T, int E, int k, int renorm, int32_t* ids,
                             float* weights, cudaStream_t s);
moe_status launch_permute(const int32_t* ids, int P, int E, int32_t* offsets, int32_t* sorted_pair,
                          int32_t* pair_to_sorted, cudaStream_t s);
moe_status launch_vq2_pack(const uint8_t* codes, const uint16_t* scales, int rows, int K,
                           uint8_t* pc, uint16_t* ps, cudaStream_t s);
moe_status launch_fp4_pack(const uint8_t* codes, const uint8_t* scales, int rows, int K, uint8_t* pc,
                           uint8_t* ps, cudaStream_t s);
moe_status launch_slot_set(SlotDesc* table, int expert_id, SlotDesc d, cudaStream_t s);
size_t ffn_workspace_size(int T, int k, int E, int I);
moe_status launch_expert_ffn(const SlotTableHost* t, const uint16_t* x, const int32_t* offsets,
                             const int32_t* sorted_pair, const float* weights, int T, int k, int mode,
                             float* out, uint8_t* status, void* ws, size_t ws_bytes, cudaStream_t s);
moe_status launch_combine(const float* ypair, const int32_t* p2s, const float* w, const uint8_t* st,
                          int T, int k, int H, float* out32, uint16_t* out16, cudaStream_t s);

}  // namespace moe

// The opaque handle of include/moe_vq2.h.
struct moe_slot_table {
    moe::SlotTableHost h;
};
