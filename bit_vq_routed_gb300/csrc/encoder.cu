// VQ2 encoder: dense fp32 weights -> a sign-symmetric codebook of 128
// 4-vectors, 8-bit codes and fp16 scales per row per 128 inputs (the code
// format of the experts; the vLLM-Moet page, "2-bit experts on vLLM
// v0.24.0", fixes the sign-symmetric codebook, and the vLLM-Moet repository
// quantises weights when it starts).  The steps:
//
//   1. block scale sigma = sqrt(mean of the squares of the 128 inputs of a
//      row's block); normalised group vectors u = w / sigma (0 if sigma = 0);
//   2. codebook: k-means with the codebook read as pairs {+c, -c}: u goes to
//      the pair i maximising 2 |u . c_i| - |c_i|^2 with sign s = sign(u . c_i),
//      c_i becomes the mean of s u over its members (kept when it has none);
//      started from the normalised vectors at 128 given indices; the result
//      rounded to fp16 is the codebook;
//   3. encoding: the scale starts at sigma; each iteration assigns the block's
//      32 groups (u = w / scale) and sets the scale to the least-squares fit
//      sum w.q / sum q.q of the chosen codewords q = s c_i; the scale is then
//      rounded to fp16 and the groups assigned against it (code = i, bit 7
//      set for s = -1).
//
// Every decision is made in fp32 in one fixed operation order, each product
// and sum rounded on its own (the round-to-nearest intrinsics are never
// fused): a dot product is ((a0 b0 + a1 b1) + a2 b2) + a3 b3, sums over
// inputs or groups run in increasing order.  The k-means sums are exact
// integers (each component of s u rounded to a multiple of 2^-20, summed in
// int64, first per CTA in shared memory), so the codebook does not depend
// on the order in which members are added; the mean is (sum 2^-20) / count
// in fp64, rounded to fp32.  The results are therefore the same on every run
// and equal, bit for bit, to a sequential computation in that order.
#include "common.cuh"

namespace moe {
namespace {

constexpr int NC = 128;          // codebook pairs
constexpr float FIX = 1048576.f; // 2^20

struct InitIdx {
    long long v[NC];
};

__device__ __forceinline__ float dot4(const float* a, const float* b) {
    float t = __fadd_rn(__fmul_rn(a[0], b[0]), __fmul_rn(a[1], b[1]));
    t = __fadd_rn(t, __fmul_rn(a[2], b[2]));
    return __fadd_rn(t, __fmul_rn(a[3], b[3]));
}

// Best pair (first maximum of 2|u.c_i| - |c_i|^2) and the sign of u.c_i.
__device__ __forceinline__ int best_pair(const float* u, const float* C, const float* norms, bool& neg) {
    int bi = 0;
    float bs = 0.f, bd = 0.f;
#pragma unroll 4
    for (int i = 0; i < NC; ++i) {
        const float d = dot4(u, C + 4 * i);
        const float sc = __fsub_rn(__fmul_rn(2.f, fabsf(d)), norms[i]);
        if (i == 0 || sc > bs) {
            bs = sc;
            bi = i;
            bd = d;
        }
    }
    neg = bd < 0.f;
    return bi;
}

__device__ __forceinline__ void load_u(const float* W, int K, const float* sigma, long long v, float* u) {
    const int G4 = K / 4;
    const long long r = v / G4;
    const int G = (int)(v - r * G4);
    const float s = sigma[r * (K / 128) + G / 32];
    const float* w = W + r * K + 4 * G;
#pragma unroll
    for (int k = 0; k < 4; ++k) u[k] = s != 0.f ? __fdiv_rn(w[k], s) : 0.f;
}

// Step 1: sigma[r, b], the squares summed in increasing input order.
__global__ void __launch_bounds__(256) rms_kernel(const float* __restrict__ W, int rows, int K,
                                                  float* __restrict__ sigma) {
    const int KB = K / 128;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < (long long)rows * KB;
         i += (long long)gridDim.x * blockDim.x) {
        const float* w = W + (i / KB) * K + (i % KB) * 128;
        float s = 0.f;
        for (int q = 0; q < 128; ++q) s = __fadd_rn(s, __fmul_rn(w[q], w[q]));
        sigma[i] = __fsqrt_rn(__fdiv_rn(s, 128.f));
    }
}

// k-means start: the normalised vectors at the given indices; the sums cleared.
__global__ void km_init_kernel(const float* __restrict__ W, int K, const float* __restrict__ sigma, InitIdx init,
                               float* __restrict__ C, unsigned long long* __restrict__ sums,
                               unsigned long long* __restrict__ cnt) {
    const int t = threadIdx.x;
    if (t < NC) load_u(W, K, sigma, init.v[t], C + 4 * t);
    for (int i = t; i < 4 * NC; i += blockDim.x) sums[i] = 0;
    if (t < NC) cnt[t] = 0;
}

// k-means assignment of every normalised group vector, with the signed
// vector's fixed-point components added to its pair's sums.
__global__ void __launch_bounds__(256) km_assign_kernel(const float* __restrict__ W, int rows, int K,
                                                        const float* __restrict__ sigma, const float* __restrict__ C,
                                                        unsigned long long* __restrict__ sums,
                                                        unsigned long long* __restrict__ cnt) {
    __shared__ float sc[4 * NC], sn[NC];
    __shared__ unsigned long long ssum[4 * NC], scnt[NC];
    for (int i = threadIdx.x; i < 4 * NC; i += blockDim.x) {
        sc[i] = C[i];
        ssum[i] = 0;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < NC; i += blockDim.x) {
        sn[i] = dot4(sc + 4 * i, sc + 4 * i);
        scnt[i] = 0;
    }
    __syncthreads();
    const long long n = (long long)rows * (K / 4);
    for (long long v = (long long)blockIdx.x * blockDim.x + threadIdx.x; v < n; v += (long long)gridDim.x * blockDim.x) {
        float u[4];
        load_u(W, K, sigma, v, u);
        bool neg;
        const int bi = best_pair(u, sc, sn, neg);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const long long fx = __float2ll_rn(__fmul_rn(neg ? -u[k] : u[k], FIX));
            atomicAdd(&ssum[4 * bi + k], (unsigned long long)fx);
        }
        atomicAdd(&scnt[bi], 1ull);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < 4 * NC; i += blockDim.x)
        if (ssum[i]) atomicAdd(&sums[i], ssum[i]);
    for (int i = threadIdx.x; i < NC; i += blockDim.x)
        if (scnt[i]) atomicAdd(&cnt[i], scnt[i]);
}

// c_i = (sum 2^-20) / count in fp64, rounded to fp32 (kept without members);
// the sums cleared for the next iteration.  One block of 4 * NC threads.
__global__ void km_update_kernel(float* __restrict__ C, unsigned long long* __restrict__ sums,
                                 unsigned long long* __restrict__ cnt, uint16_t* __restrict__ cb16) {
    const int t = threadIdx.x;
    const long long n = (long long)cnt[t / 4];
    if (n > 0)
        C[t] = __double2float_rn(__ddiv_rn(__dmul_rn(__ll2double_rn((long long)sums[t]), 1.0 / FIX),
                                           __ll2double_rn(n)));
    if (cb16) cb16[t] = __half_as_ushort(__float2half_rn(C[t]));
    __syncthreads();  // every count read before it is cleared
    sums[t] = 0;
    if (t % 4 == 0) cnt[t / 4] = 0;
}

// Step 3, one thread per (row, block).
__global__ void __launch_bounds__(256) encode_kernel(const float* __restrict__ W, int rows, int K,
                                                     const float* __restrict__ sigma, const uint16_t* __restrict__ cb,
                                                     int iters, uint8_t* __restrict__ codes,
                                                     uint16_t* __restrict__ scales) {
    __shared__ float sc[4 * NC], sn[NC];
    for (int i = threadIdx.x; i < 4 * NC; i += blockDim.x) sc[i] = __half2float(__ushort_as_half(cb[i]));
    __syncthreads();
    for (int i = threadIdx.x; i < NC; i += blockDim.x) sn[i] = dot4(sc + 4 * i, sc + 4 * i);
    __syncthreads();
    const int KB = K / 128;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < (long long)rows * KB;
         i += (long long)gridDim.x * blockDim.x) {
        const float* w0 = W + (i / KB) * K + (i % KB) * 128;
        float s = sigma[i];
        for (int it = 0; it < iters; ++it) {
            float num = 0.f, den = 0.f;
            for (int g = 0; g < 32; ++g) {
                const float* w = w0 + 4 * g;
                float u[4], q[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) u[k] = s != 0.f ? __fdiv_rn(w[k], s) : 0.f;
                bool neg;
                const int bi = best_pair(u, sc, sn, neg);
#pragma unroll
                for (int k = 0; k < 4; ++k) q[k] = neg ? -sc[4 * bi + k] : sc[4 * bi + k];
                num = __fadd_rn(num, dot4(w, q));
                den = __fadd_rn(den, dot4(q, q));
            }
            if (den > 0.f) s = __fdiv_rn(num, den);
        }
        const __half s16 = __float2half_rn(s);
        s = __half2float(s16);
        uint8_t* c = codes + (i / KB) * (K / 4) + (i % KB) * 32;
        for (int g = 0; g < 32; ++g) {
            const float* w = w0 + 4 * g;
            float u[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) u[k] = s != 0.f ? __fdiv_rn(w[k], s) : 0.f;
            bool neg;
            const int bi = best_pair(u, sc, sn, neg);
            c[g] = (uint8_t)(bi | (neg ? 0x80 : 0));
        }
        scales[i] = __half_as_ushort(s16);
    }
}

unsigned grid_for_n(long long n) {
    const long long b = (n + 255) / 256, cap = (long long)num_sms() * 8;
    return (unsigned)(b < 1 ? 1 : (b > cap ? cap : b));
}

struct EncWs {
    float* sigma;
    float* C;
    unsigned long long *sums, *cnt;
};
size_t enc_ws_layout(int rows, int K, char* base, EncWs* L) {
    size_t o = 0;
    auto take = [&](size_t bytes) {
        char* p = base ? base + o : nullptr;
        o = (o + bytes + 255) / 256 * 256;
        return p;
    };
    char* a = take(sizeof(float) * (size_t)rows * (K / 128));
    char* b = take(sizeof(float) * 4 * NC);
    char* c = take(sizeof(unsigned long long) * 4 * NC);
    char* d = take(sizeof(unsigned long long) * NC);
    if (L) {
        L->sigma = reinterpret_cast<float*>(a);
        L->C = reinterpret_cast<float*>(b);
        L->sums = reinterpret_cast<unsigned long long*>(c);
        L->cnt = reinterpret_cast<unsigned long long*>(d);
    }
    return o;
}

moe_status check_shape(const char* what, const float* W, int rows, int K) {
    if (!W) {
        set_error("%s: null weights", what);
        return MOE_ERR_INVALID_ARG;
    }
    if (rows <= 0 || K <= 0 || K % 128 != 0) {
        set_error("%s: rows=%d K=%d (K %% 128 == 0 required)", what, rows, K);
        return K % 128 != 0 && rows > 0 && K > 0 ? MOE_ERR_UNSUPPORTED : MOE_ERR_INVALID_ARG;
    }
    return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

size_t moe_vq2_encoder_workspace_size(int rows, int K) {
    if (rows <= 0 || K <= 0) return 0;
    return enc_ws_layout(rows, K, nullptr, nullptr);
}

moe_status moe_vq2_train_codebook(const float* W, int rows, int K, const int64_t* init_idx, int iters,
                                  uint16_t* codebook, float* centroids, void* ws, size_t ws_bytes,
                                  cudaStream_t stream) {
    moe_status st = check_shape("moe_vq2_train_codebook", W, rows, K);
    if (st != MOE_OK) return st;
    MOE_CHECK_ARG(init_idx && codebook && ws, "moe_vq2_train_codebook: null pointer");
    MOE_CHECK_ARG(iters >= 0 && iters <= 10000, "moe_vq2_train_codebook: iters=%d", iters);
    MOE_CHECK_ARG(ws_bytes >= moe_vq2_encoder_workspace_size(rows, K),
                  "moe_vq2_train_codebook: workspace of %zu bytes, %zu needed", ws_bytes,
                  moe_vq2_encoder_workspace_size(rows, K));
    const long long n = (long long)rows * (K / 4);
    InitIdx init;
    for (int i = 0; i < NC; ++i) {
        MOE_CHECK_ARG(init_idx[i] >= 0 && init_idx[i] < n, "moe_vq2_train_codebook: init_idx[%d]=%lld outside [0, %lld)",
                      i, (long long)init_idx[i], n);
        init.v[i] = init_idx[i];
    }
    EncWs L;
    enc_ws_layout(rows, K, static_cast<char*>(ws), &L);
    count_launch();
    rms_kernel<<<grid_for_n((long long)rows * (K / 128)), 256, 0, stream>>>(W, rows, K, L.sigma);
    count_launch();
    km_init_kernel<<<1, 4 * NC, 0, stream>>>(W, K, L.sigma, init, L.C, L.sums, L.cnt);
    for (int it = 0; it < iters; ++it) {
        count_launch();
        km_assign_kernel<<<grid_for_n(n), 256, 0, stream>>>(W, rows, K, L.sigma, L.C, L.sums, L.cnt);
        count_launch();
        km_update_kernel<<<1, 4 * NC, 0, stream>>>(L.C, L.sums, L.cnt, it + 1 == iters ? codebook : nullptr);
    }
    if (iters == 0) {  // the codebook is the starting vectors
        count_launch();
        km_update_kernel<<<1, 4 * NC, 0, stream>>>(L.C, L.sums, L.cnt, codebook);
    }
    MOE_LAUNCH_CHECK("moe_vq2_train_codebook: launch");
    if (centroids) {
        cudaError_t e = cudaMemcpyAsync(centroids, L.C, sizeof(float) * 4 * NC, cudaMemcpyDeviceToDevice, stream);
        if (e != cudaSuccess) return cuda_status(e, "moe_vq2_train_codebook: copy");
    }
    return MOE_OK;
}

moe_status moe_vq2_encode(const float* W, int rows, int K, const uint16_t* codebook, int iters, uint8_t* codes,
                          uint16_t* scales, void* ws, size_t ws_bytes, cudaStream_t stream) {
    moe_status st = check_shape("moe_vq2_encode", W, rows, K);
    if (st != MOE_OK) return st;
    MOE_CHECK_ARG(codebook && codes && scales && ws, "moe_vq2_encode: null pointer");
    MOE_CHECK_ARG(iters >= 0 && iters <= 1000, "moe_vq2_encode: iters=%d", iters);
    MOE_CHECK_ARG(ws_bytes >= moe_vq2_encoder_workspace_size(rows, K),
                  "moe_vq2_encode: workspace of %zu bytes, %zu needed", ws_bytes, moe_vq2_encoder_workspace_size(rows, K));
    EncWs L;
    enc_ws_layout(rows, K, static_cast<char*>(ws), &L);
    const long long nb = (long long)rows * (K / 128);
    count_launch();
    rms_kernel<<<grid_for_n(nb), 256, 0, stream>>>(W, rows, K, L.sigma);
    count_launch();
    encode_kernel<<<grid_for_n(nb), 256, 0, stream>>>(W, rows, K, L.sigma, codebook, iters, codes, scales);
    MOE_LAUNCH_CHECK("moe_vq2_encode: launch");
    return MOE_OK;
}

}  // extern "C"
