// Operand staging for the tensor-core paths of the expert FFN: the fp16 B
// operands, each row scaled by a power of two so that fp16 holds it whatever
// the range of the activations.
//
//   gather:  x16s[s, :] = fp16(x[t, :] / xsc[s]) for the token t of sorted
//            position s (FC1's B operand), xsc[s] = 2^e with max |x[t, :]|
//            / 2^e <= 2^14; amax[s] is cleared for the FC1 epilogues.
//   convert: a16[s, :] = fp16(a32[s, :] / asc[s]) (FC2's B operand) for the
//            sorted positions the tensor-core FC1 wrote (flag amax[s] set),
//            asc[s] = 2^e with max |a32[s, :]| / 2^e <= 2^14.
//
// Dividing by a power of two is exact, so for activations in fp16's normal
// range the operands, and the results once the epilogues multiply the scale
// back in fp32, are those of an unscaled fp16 conversion, bit for bit.
#include "ffn_common.cuh"

namespace moe {
namespace {

constexpr int THREADS = 256;  // one row per block

__device__ __forceinline__ uint32_t f2_to_h2(float a, float b) {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// Largest value of v over the block (non-negative floats as their bits).
__device__ __forceinline__ uint32_t block_max_u32(uint32_t v, uint32_t* red) {
    v = __reduce_max_sync(0xffffffffu, v);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    uint32_t m = 0;
#pragma unroll
    for (int w = 0; w < THREADS / 32; ++w) m = max(m, red[w]);
    __syncthreads();  // red is reused by the next row
    return m;
}

__global__ void __launch_bounds__(THREADS) gather_f16_kernel(const uint16_t* __restrict__ x,
                                                             const int32_t* __restrict__ sorted_pair, int k, int H,
                                                             int P, uint16_t* __restrict__ x16s,
                                                             float* __restrict__ xsc, uint32_t* __restrict__ amax) {
    __shared__ uint32_t red[THREADS / 32];
    pdl_wait();
    pdl_launch_dependents();  // dependents may start their prologues now
    for (int s = blockIdx.x; s < P; s += gridDim.x) {
        const uint4* row = reinterpret_cast<const uint4*>(x + (size_t)(sorted_pair[s] / k) * H);
        // largest |x| of the row: bf16 magnitudes order as their bits
        uint32_t m2 = 0;
        for (int c = threadIdx.x; c < H / 8; c += THREADS) {
            const uint4 v = row[c];
            m2 = __vmaxu2(m2, __vmaxu2(__vmaxu2(v.x & 0x7fff7fffu, v.y & 0x7fff7fffu),
                                       __vmaxu2(v.z & 0x7fff7fffu, v.w & 0x7fff7fffu)));
        }
        const uint32_t mb = block_max_u32(max(m2 & 0xffffu, m2 >> 16), red);
        const int e = range_exponent(__uint_as_float(mb << 16), 14);
        const float inv = exp2_i(-e);
        uint4* dst = reinterpret_cast<uint4*>(x16s + (size_t)s * H);
        for (int c = threadIdx.x; c < H / 8; c += THREADS) {
            const uint4 v = row[c];
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            uint32_t o[4];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                o[q] = f2_to_h2(__uint_as_float(w[q] << 16) * inv, __uint_as_float(w[q] & 0xffff0000u) * inv);
            dst[c] = make_uint4(o[0], o[1], o[2], o[3]);
        }
        if (threadIdx.x == 0) {
            xsc[s] = exp2_i(e);
            amax[s] = 0;
        }
    }
}

__global__ void __launch_bounds__(THREADS) a_to_f16_kernel(const float* __restrict__ a32,
                                                           const uint32_t* __restrict__ amax, int P, int I,
                                                           uint16_t* __restrict__ a16, float* __restrict__ asc) {
    pdl_wait();
    pdl_launch_dependents();
    __shared__ uint32_t red[THREADS / 32];
    for (int s = blockIdx.x; s < P; s += gridDim.x) {
        if (amax[s] == 0) continue;  // not a tensor-core position
        const float4* src = reinterpret_cast<const float4*>(a32 + (size_t)s * I);
        uint4* dst = reinterpret_cast<uint4*>(a16 + (size_t)s * I);
        // largest |a| of the row (non-negative floats order as their bits)
        uint32_t m = 0;
        for (int c = threadIdx.x; c < I / 4; c += THREADS) {
            const float4 v = src[c];
            m = max(m, __float_as_uint(fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)))));
        }
        const int e = range_exponent(__uint_as_float(block_max_u32(m, red)), 14);
        const float inv = exp2_i(-e);
        for (int c = threadIdx.x; c < I / 8; c += THREADS) {
            const float4 lo = src[2 * c], hi = src[2 * c + 1];
            dst[c] = make_uint4(f2_to_h2(lo.x * inv, lo.y * inv), f2_to_h2(lo.z * inv, lo.w * inv),
                                f2_to_h2(hi.x * inv, hi.y * inv), f2_to_h2(hi.z * inv, hi.w * inv));
        }
        if (threadIdx.x == 0) asc[s] = exp2_i(e);
    }
}

unsigned row_blocks(int P) {
    const long long cap = (long long)num_sms() * 16;
    return (unsigned)(P < cap ? P : cap);
}

}  // namespace

moe_status launch_gather_f16(const uint16_t* x, const int32_t* sorted_pair, int k, int H, int P, char* ws,
                             const WsLayout& L, cudaStream_t s) {
    cudaError_t e = launch_pdl(gather_f16_kernel, dim3(row_blocks(P)), dim3(THREADS), 0, s, x, sorted_pair, k, H, P,
                               reinterpret_cast<uint16_t*>(ws + L.x16s_off), reinterpret_cast<float*>(ws + L.xsc_off),
                               reinterpret_cast<uint32_t*>(ws + L.amax_off));
    if (e != cudaSuccess) return cuda_status(e, "moe_vq2_expert_ffn: gather launch");
    return MOE_OK;
}

moe_status launch_a_to_f16(int P, int I, char* ws, const WsLayout& L, cudaStream_t s) {
    cudaError_t e = launch_pdl(a_to_f16_kernel, dim3(row_blocks(P)), dim3(THREADS), 0, s,
                               reinterpret_cast<const float*>(ws + L.a32_off),
                               reinterpret_cast<const uint32_t*>(ws + L.amax_off), P, I,
                               reinterpret_cast<uint16_t*>(ws + L.a16_off), reinterpret_cast<float*>(ws + L.asc_off));
    if (e != cudaSuccess) return cuda_status(e, "moe_vq2_expert_ffn: conversion launch");
    return MOE_OK;
}

}  // namespace moe
