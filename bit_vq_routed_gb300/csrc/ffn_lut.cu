// Activation-table path of the expert FFN, for VQ2 experts that receive a
// single token in this call (every expert at decode batch 1, most of them at
// small batches).
//
// For one token, every code byte c of group G contributes
//     scale[r, G/32] * dot(sign(c) * codebook[c & 127], x[4G .. 4G+3])
// and the dot product depends only on (c, G), not on the row.  So a CTA first
// builds, in shared memory, the table L[c][G] of those 256 x 128 values for a
// K-range of 512 inputs (128 KB of fp32, the negated half included so the sign
// costs nothing), then streams the code tiles of many rows through it: one
// 4-byte table read per code byte instead of an 8-byte codebook read plus four
// multiply-adds.  Lanes own groups (8 lanes per 128-input scale block, 4 groups
// each), so at every table read the 32 lanes hit 32 distinct banks.  A lane's
// 4 values of one row share a scale and are summed before one FMA; the 16 row
// sums of a tile are reduced across the warp by a reduce-scatter.  K-range
// partial sums go to the workspace (deterministic, no atomics) and are added
// in a fixed order by the consumer: FC2's table build (which also applies
// silu(g) * u) and the finishing kernel.
//
// Each warp streams its units' code and scale tiles straight into registers
// with 16-byte loads, fetching two units ahead of the one it computes (12
// warps per SM keep about 80 KB in flight).
#include "ffn_common.cuh"

namespace moe {
namespace {

constexpr int CW = 12;                    // warps
constexpr int THREADS = 32 * CW;
constexpr uint32_t LUT_ADDR = 0x10000;    // table: [0x10000, 0x30000) of the shared window
constexpr uint32_t LUT_HALF = 0x10000;    // scale blocks 0-1 | 2-3
constexpr uint32_t DYN_SMEM = 0x30000;    // dynamic shared memory requested
constexpr int MAX_GROUP = 32;             // table pairs of one token (<= k <= 32)

struct __align__(16) Smem {
    float xs[128 * LUT_KB];
    float cb[128 * 4];
    const void* pa[MAX_GROUP];  // per pair of the current group: FC1 gate / FC2 down codes
    const void* pb[MAX_GROUP];  // FC1 up codes
    const void* sa[MAX_GROUP];  // matching scales
    const void* sb[MAX_GROUP];
};

// shared-window byte address of table entry (code c, group g of the K-range)
__device__ __forceinline__ uint32_t lut_addr(int c, int g) {
    const int b = g >> 5, gg = g & 31;
    const int pos = 32 * (b & 1) + ((gg + 8 * b) & 31);
    return LUT_ADDR + (uint32_t)(b >> 1) * LUT_HALF + (uint32_t)c * 256u + 4u * pos;
}

struct UnitRegs {
    uint4 cw[4];  // this lane's 4 chunks: 16 rows x 4 groups
    uint4 sc[2];  // the 16 row scales of this lane's scale block
};

template <bool FC1>
__global__ void __launch_bounds__(THREADS, 1)
    ffn_lut_kernel(const SlotDesc* __restrict__ desc, const uint16_t* __restrict__ codebook,
                   const uint16_t* __restrict__ x, const int32_t* __restrict__ sorted_pair, int k, int H, int I,
                   int* __restrict__ header, const int32_t* __restrict__ lut_s, const int32_t* __restrict__ lut_e,
                   const int32_t* __restrict__ lut_grp, const int32_t* __restrict__ grp_start,
                   const float* __restrict__ p1, float* __restrict__ pout) {
    extern __shared__ __align__(1024) uint8_t dyn[];
    Smem& S = *reinterpret_cast<Smem*>(dyn);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int* err = header + HDR_ERR;

    const int K = FC1 ? H : I;             // inputs of this matrix
    const int R = FC1 ? 2 * I : H;         // rows per pair (FC1: gate rows, then up rows)
    const int KB = K / 128;
    const int KR = lut_jobs(K);
    const int RT = R / 16;
    const int KR1 = lut_jobs(H);

    // the fixed table address needs the low part of dynamic shared memory
    // below it and the allocation to reach past its end
    const uint32_t base = smem_u32(dyn);
    if (base + (uint32_t)sizeof(Smem) > LUT_ADDR || base + DYN_SMEM < LUT_ADDR + 2 * LUT_HALF) {
        if (tid == 0) atomicExch(err, MOE_DEVERR_SMEM_LAYOUT);
        return;
    }
    for (int i = tid; i < 128 * 4; i += THREADS) S.cb[i] = __half2float(__ushort_as_half(codebook[i]));
    pdl_wait();

    const int n_lut = header[HDR_NLUT];
    // Units are (job, row tile) with job = (group, K-range).  FC1 groups are
    // the table pairs of one token (they share the activation table); FC2
    // groups are single pairs (the table depends on the pair's silu(g)*u).
    // A group of gc pairs starting at sorted pair gs owns the units
    // [KR*RT*gs, KR*RT*(gs+gc)), ordered (K-range, pair, row tile).
    // CTA blockIdx.x owns the contiguous range [u0, u1).
    const int per_pair = KR * RT;
    const int U = n_lut * per_pair;
    const int u0 = (int)((long long)U * blockIdx.x / gridDim.x);
    const int u1 = (int)((long long)U * (blockIdx.x + 1) / gridDim.x);

    const int b = lane >> 3;  // scale block of this lane inside the K-range
    uint32_t lbase[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int gg = (lane & 7) + 8 * q;
        const int pos = 32 * (b & 1) + ((gg + 8 * b) & 31);
        lbase[q] = ((uint32_t)(LUT_ADDR + (b >> 1) * LUT_HALF) & 0xffff0000u) | (uint32_t)(4 * pos);
    }

    int u = u0;
    while (u < u1) {
        int gs, gc;
        {
            const int p0 = u / per_pair;
            if (FC1) {
                const int g = lut_grp[p0];
                gs = grp_start[g];
                gc = grp_start[g + 1] - gs;
            } else {
                gs = p0;
                gc = 1;
            }
        }
        const int kr = (u - per_pair * gs) / (RT * gc);
        const int job_start = per_pair * gs + kr * RT * gc;
        const int seg_end = min(u1, job_start + RT * gc);
        const int nkb = min(LUT_KB, KB - LUT_KB * kr);
        const int nin = 128 * nkb;
        const bool active = b < nkb;

        __syncthreads();  // every warp is done with the previous table and pointers
        if (tid < gc) {
            const SlotDesc& d = desc[lut_e[gs + tid]];
            S.pa[tid] = d.codes[FC1 ? 0 : 2];
            S.sa[tid] = d.scales[FC1 ? 0 : 2];
            S.pb[tid] = d.codes[1];
            S.sb[tid] = d.scales[1];
        }
        // inputs of this K-range: FC1 the token's activations, FC2 silu(g)*u
        // of the pair, from FC1's K-range partial sums added in a fixed order
        if (FC1) {
            const int t = sorted_pair[lut_s[gs]] / k;
            for (int i = tid; i < nin; i += THREADS)
                S.xs[i] = __uint_as_float((uint32_t)x[(size_t)t * H + LUT_KB * 128 * kr + i] << 16);
        } else {
            const float* pp = p1 + (size_t)gs * KR1 * 2 * I;
            for (int i = tid; i < nin; i += THREADS) {
                const int gi = LUT_KB * 128 * kr + i;
                float g = 0.0f, up = 0.0f;
                for (int j0 = 0; j0 < KR1; j0 += 8) {  // 8 partials in flight, added in order
                    float pg[8], pu[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        pg[j] = j0 + j < KR1 ? pp[(size_t)(j0 + j) * 2 * I + gi] : 0.0f;
                        pu[j] = j0 + j < KR1 ? pp[(size_t)(j0 + j) * 2 * I + I + gi] : 0.0f;
                    }
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        if (j0 + j < KR1) {
                            g += pg[j];
                            up += pu[j];
                        }
                    }
                }
                S.xs[i] = g / (1.0f + expf(-g)) * up;
            }
        }
        __syncthreads();
        // table entries: +dot for code c, -dot for c + 128; a thread takes one
        // group and the four codes c, c+32, c+64, c+96
        const int G = 32 * nkb;
        for (int idx = tid; idx < 32 * G; idx += THREADS) {
            const int c0 = idx / G, g = idx - c0 * G;
            const float4 xv = *reinterpret_cast<const float4*>(&S.xs[4 * g]);
            const uint32_t a0 = lut_addr(c0, g);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float4 e4 = *reinterpret_cast<const float4*>(&S.cb[4 * (c0 + 32 * q)]);
                float v = e4.x * xv.x;
                v = fmaf(e4.y, xv.y, v);
                v = fmaf(e4.z, xv.z, v);
                v = fmaf(e4.w, xv.w, v);
                const uint32_t a = a0 + 32u * 256u * q;
                sts_f32(a, v);
                sts_f32(a + 128u * 256u, -v);
            }
        }
        __syncthreads();

        // this warp's units of the job: v = u + warp, u + warp + CW, ...; the
        // (pair, row tile) of a unit advances by CW row tiles per step
        auto load_unit = [&](int pi, int rt, UnitRegs& r) {
            const bool second = FC1 && rt >= I / 16;  // an up-matrix row tile
            const int rtm = second ? rt - I / 16 : rt;
            const size_t tile = (size_t)rtm * KB + LUT_KB * kr + b;
            if (active) {
                const uint8_t* c = static_cast<const uint8_t*>(second ? S.pb[pi] : S.pa[pi]) + tile * 512;
                const uint16_t* sp = static_cast<const uint16_t*>(second ? S.sb[pi] : S.sa[pi]) + tile * 16;
#pragma unroll
                for (int q = 0; q < 4; ++q) r.cw[q] = ldg_stream(c + 16 * ((lane & 7) + 8 * q));
                r.sc[0] = ldg_stream(sp);
                r.sc[1] = ldg_stream(sp + 8);
            }
        };
        auto advance = [&](int& pi, int& rt) {
            rt += CW;
            while (rt >= RT) {
                rt -= RT;
                ++pi;
            }
        };
        UnitRegs cur, n1, n2;
        int v = u + warp;
        int pi = (v - job_start) / RT, rt = (v - job_start) - ((v - job_start) / RT) * RT;
        int pi1 = pi, rt1 = rt, pi2, rt2;
        advance(pi1, rt1);
        pi2 = pi1;
        rt2 = rt1;
        advance(pi2, rt2);
        if (v < seg_end) load_unit(pi, rt, cur);
        if (v + CW < seg_end) load_unit(pi1, rt1, n1);
        for (; v < seg_end; v += CW) {
            if (v + 2 * CW < seg_end) load_unit(pi2, rt2, n2);
            float acc[16];
            if (active) {
                float s[16];
                const uint32_t sw[8] = {cur.sc[0].x, cur.sc[0].y, cur.sc[0].z, cur.sc[0].w,
                                        cur.sc[1].x, cur.sc[1].y, cur.sc[1].z, cur.sc[1].w};
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&sw[i]));
                    s[2 * i] = f.x;
                    s[2 * i + 1] = f.y;
                }
#pragma unroll
                for (int r = 0; r < 16; ++r) {  // byte position r of each chunk
                    const uint32_t sel = 0x7604u | ((uint32_t)(r & 3) << 4);
                    float t = 0.0f;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint32_t w = (&cur.cw[q].x)[r >> 2];
                        t += lds_f32(prmt(w, lbase[q], sel));
                    }
                    const int row = (r >> 1) + 8 * (r & 1);  // byte 2i+h holds row i + 8h
                    acc[r] = t * s[row];
                }
            } else {
#pragma unroll
                for (int r = 0; r < 16; ++r) acc[r] = 0.0f;
            }
            // reduce-scatter over the warp: lanes 2p and 2p+1 end with position p
#pragma unroll
            for (int o = 16, n8 = 8; o >= 2; o >>= 1, n8 >>= 1) {
                const bool up = lane & o;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if (i < n8) {
                        const float send = up ? acc[i] : acc[i + n8];
                        const float keep = up ? acc[i + n8] : acc[i];
                        acc[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                    }
                }
            }
            acc[0] += __shfl_xor_sync(0xffffffffu, acc[0], 1);
            if ((lane & 1) == 0) {
                const int p = lane >> 1;
                const int row = (p >> 1) + 8 * (p & 1);
                pout[((size_t)(gs + pi) * KR + kr) * R + (size_t)rt * 16 + row] = acc[0];
            }
            cur = n1;
            n1 = n2;
            pi = pi1;
            rt = rt1;
            pi1 = pi2;
            rt1 = rt2;
            advance(pi2, rt2);
        }
        u = seg_end;
    }
    pdl_launch_dependents();
}

// y = sum of the FC2 K-range partials (fixed order); per-pair store or
// weighted scatter-add.
__global__ void __launch_bounds__(256) lut_finish_kernel(const int* __restrict__ header,
                                                         const int32_t* __restrict__ lut_s,
                                                         const int32_t* __restrict__ sorted_pair,
                                                         const float* __restrict__ weights, int k, int H, int I,
                                                         const float* __restrict__ p2, int mode,
                                                         float* __restrict__ out) {
    pdl_wait();
    const int n_lut = header[HDR_NLUT];
    const int KR2 = lut_jobs(I);
    const int n = n_lut * (H / 4);
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        const int li = i / (H / 4), h = 4 * (i - li * (H / 4));
        float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j = 0; j < KR2; ++j) {
            const float4 v = *reinterpret_cast<const float4*>(p2 + ((size_t)li * KR2 + j) * H + h);
            y.x += v.x;
            y.y += v.y;
            y.z += v.z;
            y.w += v.w;
        }
        const int s = lut_s[li];
        if (mode == MOE_PER_PAIR) {
            *reinterpret_cast<float4*>(out + (size_t)s * H + h) = y;
        } else {
            const int p = sorted_pair[s];
            const float w = weights[p];
            float* o = out + (size_t)(p / k) * H + h;
            atomicAdd(o + 0, w * y.x);
            atomicAdd(o + 1, w * y.y);
            atomicAdd(o + 2, w * y.z);
            atomicAdd(o + 3, w * y.w);
        }
    }
    pdl_launch_dependents();
}

}  // namespace

moe_status launch_lut_fc(bool fc1, const SlotTableHost* t, const uint16_t* x, const int32_t* sorted_pair, int k,
                         char* ws, const WsLayout& L, cudaStream_t s) {
    static_assert(sizeof(Smem) + 1024 <= LUT_ADDR, "shared layout");
    int* header = reinterpret_cast<int*>(ws);
    const int32_t* lut_s = reinterpret_cast<const int32_t*>(ws + L.lut_s_off);
    const int32_t* lut_e = reinterpret_cast<const int32_t*>(ws + L.lut_e_off);
    const int32_t* lut_grp = reinterpret_cast<const int32_t*>(ws + L.lut_grp_off);
    const int32_t* grp_start = reinterpret_cast<const int32_t*>(ws + L.grp_start_off);
    const float* p1 = reinterpret_cast<const float*>(ws + L.p1_off);
    float* pout = reinterpret_cast<float*>(ws + (fc1 ? L.p1_off : L.p2_off));
    auto kern = fc1 ? ffn_lut_kernel<true> : ffn_lut_kernel<false>;
    cudaError_t e = ensure_smem_attr(kern, (int)DYN_SMEM);
    if (e != cudaSuccess) return cuda_status(e, "moe_vq2_expert_ffn: table kernel shared memory");
    e = launch_pdl(kern, dim3((unsigned)num_sms()), dim3(THREADS), DYN_SMEM, s, (const SlotDesc*)t->d_desc,
                   t->codebook, x, sorted_pair, k, t->H, t->I, header, lut_s, lut_e, lut_grp, grp_start, p1, pout);
    if (e != cudaSuccess) return cuda_status(e, "moe_vq2_expert_ffn: table kernel launch");
    MOE_LAUNCH_CHECK("moe_vq2_expert_ffn: table kernel launch");
    return MOE_OK;
}

moe_status launch_lut_finish(const SlotTableHost* t, const int32_t* sorted_pair, const float* weights, int k,
                             int mode, float* out, char* ws, const WsLayout& L, int max_lut, cudaStream_t s) {
    const int* header = reinterpret_cast<const int*>(ws);
    const int32_t* lut_s = reinterpret_cast<const int32_t*>(ws + L.lut_s_off);
    const float* p2 = reinterpret_cast<const float*>(ws + L.p2_off);
    long long n = (long long)max_lut * (t->H / 4);
    long long blocks = (n + 255) / 256;
    long long cap = (long long)num_sms() * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    cudaError_t e = launch_pdl(lut_finish_kernel, dim3((unsigned)blocks), dim3(256), 0, s, header, lut_s, sorted_pair,
                               weights, k, t->H, t->I, p2, mode, out);
    if (e != cudaSuccess) return cuda_status(e, "moe_vq2_expert_ffn: table finish launch");
    MOE_LAUNCH_CHECK("moe_vq2_expert_ffn: table finish launch");
    return MOE_OK;
}

}  // namespace moe
