// Deterministic weighted combine of per-pair expert outputs.
#include <cuda_bf16.h>

#include "common.cuh"

namespace moe {
namespace {

__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ ypair,
                                                      const int32_t* __restrict__ p2s,
                                                      const float* __restrict__ w,
                                                      const uint8_t* __restrict__ st, int T, int k, int H,
                                                      float* __restrict__ out32,
                                                      uint16_t* __restrict__ out16) {
    pdl_wait();
    const int t = blockIdx.y;
    const int h = 4 * (blockIdx.x * blockDim.x + threadIdx.x);
    if (h >= H) return;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < k; ++j) {
        const int p = t * k + j;
        if (!st[p]) continue;
        const float wj = w[p];
        const float4 y = *reinterpret_cast<const float4*>(ypair + (size_t)p2s[p] * H + h);
        acc.x = __fadd_rn(acc.x, __fmul_rn(wj, y.x));
        acc.y = __fadd_rn(acc.y, __fmul_rn(wj, y.y));
        acc.z = __fadd_rn(acc.z, __fmul_rn(wj, y.z));
        acc.w = __fadd_rn(acc.w, __fmul_rn(wj, y.w));
    }
    if (out32) *reinterpret_cast<float4*>(out32 + (size_t)t * H + h) = acc;
    if (out16) {
        uint16_t* o = out16 + (size_t)t * H + h;
        o[0] = __bfloat16_as_ushort(__float2bfloat16_rn(acc.x));
        o[1] = __bfloat16_as_ushort(__float2bfloat16_rn(acc.y));
        o[2] = __bfloat16_as_ushort(__float2bfloat16_rn(acc.z));
        o[3] = __bfloat16_as_ushort(__float2bfloat16_rn(acc.w));
    }
    pdl_launch_dependents();
}

}  // namespace

moe_status launch_combine(const float* ypair, const int32_t* p2s, const float* w, const uint8_t* st, int T,
                          int k, int H, float* out32, uint16_t* out16, cudaStream_t s) {
    if (T > 65535) {
        set_error("moe_combine: T=%d above 65535", T);
        return MOE_ERR_UNSUPPORTED;
    }
    dim3 grid((unsigned)((H / 4 + 255) / 256), (unsigned)T);
    combine_kernel<<<grid, 256, 0, s>>>(ypair, p2s, w, st, T, k, H, out32, out16);
    MOE_LAUNCH_CHECK("moe_combine: launch");
    return MOE_OK;
}

}  // namespace moe
