// Deterministic weighted combine of per-pair expert outputs.
#include <cuda_bf16.h>

#include "common.cuh"

namespace moe {
namespace {

// out[t, h..h+3] = sum_j status * w * ypair[pair_to_sorted[t*k+j], h..h+3] in
// increasing j.  Lanes j < k fetch pair j's (row, weight) once and broadcast
// them, so each thread issues its k row loads back to back.
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ ypair,
                                                      const int32_t* __restrict__ p2s,
                                                      const float* __restrict__ w,
                                                      const uint8_t* __restrict__ st, int T, int k, int H,
                                                      float* __restrict__ out32,
                                                      uint16_t* __restrict__ out16) {
    pdl_wait();
    // dependents may start their prologues now, unless they may read out16
    // as their activations (then they start when this kernel has finished)
    if (out16 == nullptr) pdl_launch_dependents();
    const int t = blockIdx.y, lane = threadIdx.x & 31;
    const int h = 4 * (blockIdx.x * blockDim.x + threadIdx.x);
    int row = -1;
    float wj = 0.0f;
    if (lane < k) {  // (the three loads in one round trip)
        const int p = t * k + lane;
        const uint8_t sv = st[p];
        const int rv = p2s[p];
        const float wv = w[p];
        if (sv) {
            row = rv;
            wj = wv;
        }
    }
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < k; ++j) {
        const int r = __shfl_sync(0xffffffffu, row, j);
        const float wv = __shfl_sync(0xffffffffu, wj, j);
        if (r >= 0 && h < H) {
            const float4 y = *reinterpret_cast<const float4*>(ypair + (size_t)r * H + h);
            acc.x = __fadd_rn(acc.x, __fmul_rn(wv, y.x));
            acc.y = __fadd_rn(acc.y, __fmul_rn(wv, y.y));
            acc.z = __fadd_rn(acc.z, __fmul_rn(wv, y.z));
            acc.w = __fadd_rn(acc.w, __fmul_rn(wv, y.w));
        }
    }
    if (h < H) {
        if (out32) *reinterpret_cast<float4*>(out32 + (size_t)t * H + h) = acc;
        if (out16) {
            const uint32_t lo = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(acc.x)) |
                                ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(acc.y)) << 16);
            const uint32_t hi = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(acc.z)) |
                                ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(acc.w)) << 16);
            *reinterpret_cast<uint2*>(out16 + (size_t)t * H + h) = make_uint2(lo, hi);
        }
    }
}

// dst[i] += src[i] (the GPU's partial output plus a remainder computed elsewhere)
__global__ void __launch_bounds__(256) accumulate_kernel(float* __restrict__ dst, const float* __restrict__ src,
                                                         size_t n) {
    pdl_wait();
    pdl_launch_dependents();
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
        dst[i] += src[i];
}

// gated[p] = ids[p] + E when weights[p] >= tau and entry E + ids[p] is resident
__global__ void __launch_bounds__(256) gate_kernel(const SlotDesc* __restrict__ desc, const int32_t* __restrict__ ids,
                                                   const float* __restrict__ weights, int P, int E, float tau,
                                                   int32_t* __restrict__ gated) {
    pdl_wait();
    pdl_launch_dependents();
    for (int p = blockIdx.x * blockDim.x + threadIdx.x; p < P; p += gridDim.x * blockDim.x) {
        const int e = ids[p];
        const bool g = e >= 0 && e < E && weights[p] >= tau && desc[E + e].resident != 0;
        gated[p] = g ? e + E : e;
    }
}

}  // namespace

moe_status launch_gate(const SlotDesc* desc, const int32_t* ids, const float* weights, int P, int E, float tau,
                       int32_t* gated, cudaStream_t s) {
    const int blocks = (P + 255) / 256, cap = num_sms() * 4;
    cudaError_t e = launch_pdl(gate_kernel, dim3((unsigned)(blocks < cap ? blocks : cap)), dim3(256), 0, s, desc, ids,
                               weights, P, E, tau, gated);
    if (e != cudaSuccess) return cuda_status(e, "moe_confidence_gate: launch");
    return MOE_OK;
}

moe_status launch_accumulate(float* dst, const float* src, size_t n, cudaStream_t s) {
    const size_t blocks = (n + 255) / 256, cap = (size_t)num_sms() * 8;
    cudaError_t e = launch_pdl(accumulate_kernel, dim3((unsigned)(blocks < cap ? blocks : cap)), dim3(256), 0, s, dst,
                               src, n);
    if (e != cudaSuccess) return cuda_status(e, "moe_accumulate: launch");
    return MOE_OK;
}

moe_status launch_combine(const float* ypair, const int32_t* p2s, const float* w, const uint8_t* st, int T,
                          int k, int H, float* out32, uint16_t* out16, cudaStream_t s) {
    if (T > 65535) {
        set_error("moe_combine: T=%d above 65535", T);
        return MOE_ERR_UNSUPPORTED;
    }
    dim3 grid((unsigned)((H / 4 + 255) / 256), (unsigned)T);
    cudaError_t e = launch_pdl(combine_kernel, grid, dim3(256), 0, s, ypair, p2s, w, st, T, k, H, out32, out16);
    if (e != cudaSuccess) return cuda_status(e, "moe_combine: launch");
    MOE_LAUNCH_CHECK("moe_combine: launch");
    return MOE_OK;
}

}  // namespace moe
