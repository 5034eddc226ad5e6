// Router logits (fixed fp32 summation order) and top-k + softmax routing.
#include <float.h>
#include <limits.h>

#include "common.cuh"

namespace moe {
namespace {

constexpr unsigned FULL = 0xffffffffu;

__device__ __forceinline__ void unpack_bf16x8(const uint4& v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

// One warp computes NE experts' logits for one token.  Lane l owns the
// 16-byte chunks c = l + 32m (inputs 8c..8c+7) and adds their products in
// increasing input order; bf16 x bf16 products are exact in fp32, so the
// explicit mul + add below equals an FMA.  Then a butterfly over the lanes.
template <int NE>
__global__ void __launch_bounds__(256) router_logits_kernel(const uint16_t* __restrict__ x,
                                                            const uint16_t* __restrict__ w,
                                                            const float* __restrict__ bias,
                                                            float* __restrict__ logits, int T, int H,
                                                            int E) {
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const long warp = ((long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int egroups = (E + NE - 1) / NE;
    const long t = warp / egroups;
    if (t >= T) return;
    const int e0 = (int)(warp % egroups) * NE;
    const int nch = H / 256;
    const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)t * H);
    const uint4* wr[NE];
#pragma unroll
    for (int q = 0; q < NE; ++q) {
        int e = min(e0 + q, E - 1);
        wr[q] = reinterpret_cast<const uint4*>(w + (size_t)e * H);
    }
    float acc[NE];
#pragma unroll
    for (int q = 0; q < NE; ++q) acc[q] = 0.0f;
    constexpr int U = 4;  // chunks fetched per round trip
    for (int m0 = 0; m0 < nch; m0 += U) {
        uint4 xv[U], wv[U][NE];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (m0 + u < nch) {
                xv[u] = __ldg(xr + lane + 32 * (m0 + u));
#pragma unroll
                for (int q = 0; q < NE; ++q) wv[u][q] = __ldg(wr[q] + lane + 32 * (m0 + u));
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (m0 + u < nch) {
                float xf[8];
                unpack_bf16x8(xv[u], xf);
#pragma unroll
                for (int q = 0; q < NE; ++q) {
                    float wf[8];
                    unpack_bf16x8(wv[u][q], wf);
#pragma unroll
                    for (int i = 0; i < 8; ++i) acc[q] = __fadd_rn(acc[q], __fmul_rn(xf[i], wf[i]));
                }
            }
        }
    }
#pragma unroll
    for (int q = 0; q < NE; ++q) {
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) acc[q] = __fadd_rn(acc[q], __shfl_xor_sync(FULL, acc[q], off));
    }
    if (lane < NE) {
        float v = acc[0];
#pragma unroll
        for (int q = 1; q < NE; ++q)
            if (lane == q) v = acc[q];
        int e = e0 + lane;
        if (e < E) logits[(size_t)t * E + e] = bias ? __fadd_rn(v, bias[e]) : v;
    }
    pdl_launch_dependents();
}

__device__ __forceinline__ bool better(float v, int e, float bv, int be) {
    return v > bv || (v == bv && e < be);
}

// Small-batch router: one CTA of 8 warps per (token, 8 experts); the token's
// activations sit in shared memory and each lane first loads all of its
// router-weight chunks, so a warp needs one memory round trip.  Same fixed
// summation order as router_logits_kernel.
__global__ void __launch_bounds__(256) router_logits_small_kernel(const uint16_t* __restrict__ x,
                                                                  const uint16_t* __restrict__ w,
                                                                  const float* __restrict__ bias,
                                                                  float* __restrict__ logits, int T, int H,
                                                                  int E) {
    extern __shared__ __align__(16) uint4 xs[];
    const int t = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = blockIdx.x * 8 + warp;
    const int nch = H / 8;
    pdl_wait();
    for (int i = threadIdx.x; i < nch; i += blockDim.x) xs[i] = reinterpret_cast<const uint4*>(x + (size_t)t * H)[i];
    __syncthreads();
    if (e >= E) return;
    const uint4* wr = reinterpret_cast<const uint4*>(w + (size_t)e * H);
    const int per = H / 256;  // chunks per lane
    float acc = 0.0f;
    constexpr int U = 16;
    for (int m0 = 0; m0 < per; m0 += U) {
        uint4 wv[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (m0 + u < per) wv[u] = __ldg(wr + lane + 32 * (m0 + u));
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (m0 + u < per) {
                float xf[8], wf[8];
                unpack_bf16x8(xs[lane + 32 * (m0 + u)], xf);
                unpack_bf16x8(wv[u], wf);
#pragma unroll
                for (int i = 0; i < 8; ++i) acc = __fadd_rn(acc, __fmul_rn(xf[i], wf[i]));
            }
        }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(FULL, acc, off));
    if (lane == 0) logits[(size_t)t * E + e] = bias ? __fadd_rn(acc, bias[e]) : acc;
    pdl_launch_dependents();
}

// One warp per token: lane l holds logits l, l+32, ...; each lane keeps its
// best not-yet-taken (logit desc, id asc); k rounds of a warp-wide arg-max,
// after which only the lane that owned the winner rescans its values.
template <int NPER>
__global__ void __launch_bounds__(256) route_topk_kernel(const float* __restrict__ logits, int T, int E,
                                                         int k, int renorm, int32_t* __restrict__ ids,
                                                         float* __restrict__ weights) {
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const long t = ((long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (t >= T) return;
    const float* l = logits + (size_t)t * E;
    float v[NPER];
    uint32_t taken = 0;
#pragma unroll
    for (int i = 0; i < NPER; ++i) {
        const int e = lane + 32 * i;
        if (e < E)
            v[i] = l[e];
        else {
            v[i] = -INFINITY;
            taken |= 1u << i;
        }
    }
    float bv = -INFINITY;
    int be = INT_MAX;
    auto rescan = [&]() {
        bv = -INFINITY;
        be = INT_MAX;
#pragma unroll
        for (int i = 0; i < NPER; ++i) {
            const int e = lane + 32 * i;
            if (!((taken >> i) & 1) && better(v[i], e, bv, be)) {
                bv = v[i];
                be = e;
            }
        }
    };
    rescan();
    float sel_v = 0.0f;  // lane j keeps the j-th selected logit
    int sel_e = 0;
    for (int j = 0; j < k; ++j) {
        float wv = bv;
        int we = be;
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) {
            const float ov = __shfl_xor_sync(FULL, wv, off);
            const int oe = __shfl_xor_sync(FULL, we, off);
            if (better(ov, oe, wv, we)) {
                wv = ov;
                we = oe;
            }
        }
        if (lane == j) {
            sel_v = wv;
            sel_e = we;
        }
        if ((we & 31) == lane) {
            taken |= 1u << (we >> 5);
            rescan();
        }
    }
    const float top = __shfl_sync(FULL, sel_v, 0);
    const float num = lane < k ? expf(sel_v - top) : 0.0f;
    float den = 0.0f;
    if (renorm) {
        den = num;
    } else {
#pragma unroll
        for (int i = 0; i < NPER; ++i)
            if (lane + 32 * i < E) den += expf(v[i] - top);
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) den += __shfl_xor_sync(FULL, den, off);
    if (lane < k) {
        ids[(size_t)t * k + lane] = sel_e;
        weights[(size_t)t * k + lane] = num / den;
    }
    pdl_launch_dependents();
}

}  // namespace

moe_status launch_router_logits(const uint16_t* x, const uint16_t* w, const float* bias, float* logits,
                                int T, int H, int E, cudaStream_t s) {
    const int threads = 256;
    const size_t xs_bytes = (size_t)H * 2;
    if (T <= 64 && xs_bytes <= 48 * 1024) {
        dim3 grid((unsigned)((E + 7) / 8), (unsigned)T);
        cudaError_t e = launch_pdl(router_logits_small_kernel, grid, dim3(threads), xs_bytes, s, x, w, bias, logits, T,
                                   H, E);
        if (e != cudaSuccess) return cuda_status(e, "moe_router_logits: launch");
    } else {
        long warps = (long)T * ((E + 3) / 4);
        long blocks = (warps * 32 + threads - 1) / threads;
        cudaError_t e = launch_pdl(router_logits_kernel<4>, dim3((unsigned)blocks), dim3(threads), 0, s, x, w, bias,
                                   logits, T, H, E);
        if (e != cudaSuccess) return cuda_status(e, "moe_router_logits: launch");
    }
    MOE_LAUNCH_CHECK("moe_router_logits: launch");
    return MOE_OK;
}

moe_status launch_route_topk(const float* logits, int T, int E, int k, int renorm, int32_t* ids,
                             float* weights, cudaStream_t s) {
    const int threads = 256;
    const unsigned blocks = (unsigned)(((long)T * 32 + threads - 1) / threads);
    auto kern = E <= 32    ? route_topk_kernel<1>
                : E <= 64  ? route_topk_kernel<2>
                : E <= 128 ? route_topk_kernel<4>
                : E <= 256 ? route_topk_kernel<8>
                : E <= 512 ? route_topk_kernel<16>
                           : route_topk_kernel<32>;
    cudaError_t e = launch_pdl(kern, dim3(blocks), dim3(threads), 0, s, logits, T, E, k, renorm, ids, weights);
    if (e != cudaSuccess) return cuda_status(e, "moe_route_topk: launch");
    MOE_LAUNCH_CHECK("moe_route_topk: launch");
    return MOE_OK;
}

}  // namespace moe
