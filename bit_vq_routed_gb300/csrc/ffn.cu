// Expert FFN over the slot table: schedule, FC1 (gate, up) + silu(gate)*up,
// FC2 with the per-pair store or the weighted scatter-add.
//
// Decode path (this file): tensor-core mma.sync m16n8k16 (fp16 in, fp32
// accumulate) on weights decoded in registers.  A VQ2 code byte is looked up
// in a sign-folded codebook (256 entries: index and negated copies) held in
// shared memory, replicated 16 times so that the 16 lanes of a half-warp hit
// 16 distinct bank pairs; the 4 fp16 values of the entry are exactly one
// thread's A-fragment for one row (the K order inside each 16-wide MMA step
// is permuted so that each thread's 4 k-slots are one code's 4 inputs, and
// the activations use the same permutation).  The row scale is applied per
// 128-input block in fp32 after the block's 8 MMAs.  FP4 (e2m1) bytes are
// converted to f16x2 with cvt and scaled per 32-input block.
// Code tiles stream into shared memory through a per-warp cp.async ring.
#include "ffn_common.cuh"

namespace moe {
namespace {

constexpr int WARPS = 4;         // warps per CTA, one 16-row tile each
constexpr int ROWS = 16 * WARPS;  // rows per work unit
constexpr int STAGES = 8;        // cp.async ring depth per warp
constexpr int STAGE_BYTES = 1024;  // two 512-byte tiles (gate + up) per step
constexpr int CB_COPIES = 16;

// ---------------------------------------------------------------- schedule
// Exclusive scan over the 1024 threads of the block; returns the block total
// through *total.
__device__ int block_exclusive_scan(int v, int* warp_tot, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
    }
    __syncthreads();
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int wv = warp_tot[lane], wi = wv;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            int o = __shfl_up_sync(0xffffffffu, wi, off);
            if (lane >= off) wi += o;
        }
        warp_tot[lane] = wi - wv;
        if (lane == 31) warp_tot[32] = wi;
    }
    __syncthreads();
    *total = warp_tot[32];
    return incl - v + warp_tot[warp];
}

// One CTA of 1024 threads.  Expert e with m_e pairs, if resident:
//   VQ2 with m_e == 1 (and use_lut) -> one activation-table pair;
//   otherwise -> ceil(m_e / NT) tensor-core chunks.
// Table pairs are listed sorted by (token, expert) and grouped by token, so
// the experts of one token share each activation table.  pair_status of every
// pair from the residency of its expert; the header's error word is cleared.
__global__ void __launch_bounds__(1024) schedule_kernel(const SlotDesc* __restrict__ desc, int E,
                                                        const int32_t* __restrict__ offsets,
                                                        const int32_t* __restrict__ sorted_pair, int P, int k,
                                                        uint8_t* __restrict__ status, int* __restrict__ header,
                                                        Chunk* __restrict__ chunks, int32_t* __restrict__ lut_s,
                                                        int32_t* __restrict__ lut_e, int32_t* __restrict__ lut_grp,
                                                        int32_t* __restrict__ grp_start, int use_lut) {
    __shared__ int warp_tot[33];
    __shared__ int s_off[1025];
    __shared__ int s_tok[1024];  // token of each table pair, by expert (INT_MAX otherwise)
    __shared__ int s_sorted_tok[1024];
    __shared__ uint8_t s_res[1024];
    __shared__ uint8_t s_fmt[1024];
    pdl_wait();
    const int tid = threadIdx.x;
    for (int i = tid; i <= E; i += 1024) s_off[i] = offsets[i];
    if (tid < E) {
        s_res[tid] = (uint8_t)(desc[tid].resident != 0);
        s_fmt[tid] = (uint8_t)desc[tid].format;
    }
    __syncthreads();
    const int m = tid < E ? s_off[tid + 1] - s_off[tid] : 0;
    const bool res = tid < E && s_res[tid] && m > 0;
    const bool lut = res && use_lut && m == 1 && s_fmt[tid] == MOE_FMT_VQ2;
    const int n = (res && !lut) ? (m + NT - 1) / NT : 0;
    const int tok = lut ? sorted_pair[s_off[tid]] / k : 0x7fffffff;
    s_tok[tid] = tok;
    int n_chunks, n_lut;
    const int cbase = block_exclusive_scan(n, warp_tot, &n_chunks);
    for (int c = 0; c < n; ++c) {
        Chunk ch;
        ch.expert = tid;
        ch.start = s_off[tid] + c * NT;
        ch.count = min(NT, m - c * NT);
        ch.fmt = s_fmt[tid];
        chunks[cbase + c] = ch;
    }
    block_exclusive_scan(lut ? 1 : 0, warp_tot, &n_lut);  // (its barriers also publish s_tok)
    if (lut) {
        // rank by (token, expert id): a stable sort of the table pairs by token
        int rank = 0;
        for (int e2 = 0; e2 < E; ++e2) {
            const int t2 = s_tok[e2];
            rank += (t2 < tok) || (t2 == tok && e2 < tid);
        }
        lut_s[rank] = s_off[tid];
        lut_e[rank] = tid;
        s_sorted_tok[rank] = tok;
    }
    __syncthreads();
    const bool first = tid < n_lut && (tid == 0 || s_sorted_tok[tid] != s_sorted_tok[tid - 1]);
    int n_groups;
    const int gid = block_exclusive_scan(first ? 1 : 0, warp_tot, &n_groups) + (first ? 1 : 0) - 1;
    if (tid < n_lut) {
        lut_grp[tid] = gid;
        if (first) grp_start[gid] = tid;
    }
    if (tid == 0) {
        grp_start[n_groups] = n_lut;
        header[HDR_NCHUNKS] = n_chunks;
        header[HDR_NLUT] = n_lut;
        header[HDR_ERR] = 0;
        header[HDR_NGROUPS] = n_groups;
    }
    for (int s = tid; s < P; s += 1024) {
        int lo = 0, hi = E;  // find e with off[e] <= s < off[e+1]
        while (hi - lo > 1) {
            int mid = (lo + hi) >> 1;
            if (s_off[mid] <= s) lo = mid; else hi = mid;
        }
        status[sorted_pair[s]] = s_res[lo];
    }
    pdl_launch_dependents();
}

// ---------------------------------------------------------------- helpers
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    unsigned sa = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(sa), "l"(gmem));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }

// x tile row stride in bytes: K fp16 + padding so the B-fragment loads of a
// warp hit distinct banks (VQ2 reads 8 bytes per lane, FP4 4 bytes).
__host__ __device__ inline int xstride_bytes(int K, int fmt) { return 2 * K + (fmt == MOE_FMT_FP4 ? 16 : 32); }

// ---------------------------------------------------------------- main kernel
// FC1 (NMAT = 2: gate and up of the same rows) or FC2 (NMAT = 1: down).
// Work item = (chunk of <= NT tokens of one expert, group of ROWS rows);
// one CTA loops over items.  Shared memory: sign-folded codebook copies
// [256][16] x 8 B, the chunk's activations as fp16 [NT][K], then each warp's
// cp.async ring of STAGES x 1 KB.
template <int NMAT>
__global__ void __launch_bounds__(32 * WARPS, 1) ffn_mma_kernel(
    const SlotDesc* __restrict__ desc, const uint16_t* __restrict__ codebook,
    const uint16_t* __restrict__ x_bf16,   // FC1 input [T, K]
    const float* __restrict__ a_in,        // FC2 input [P(sorted), K]
    const int32_t* __restrict__ sorted_pair, const float* __restrict__ weights, int k, int K, int R,
    const int* __restrict__ header, const Chunk* __restrict__ chunks,
    float* __restrict__ a_out,             // FC1 output [P(sorted), R]
    float* __restrict__ out, int mode) {   // FC2 output
    extern __shared__ __align__(16) uint8_t smem[];
    uint2* cbt = reinterpret_cast<uint2*>(smem);
    uint8_t* xt = smem + 256 * CB_COPIES * 8;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int i = lane >> 2, j = lane & 3;
    uint8_t* ring = xt + NT * (2 * K + 32) + warp * STAGES * STAGE_BYTES;

    pdl_wait();
    const int n_chunks = header[HDR_NCHUNKS];
    const int row_groups = R / ROWS;
    const long n_items = (long)n_chunks * row_groups;
    if (blockIdx.x >= n_items) return;  // no tensor-core work for this CTA
    for (int idx = threadIdx.x; idx < 256 * CB_COPIES; idx += blockDim.x) {
        int c = idx / CB_COPIES;
        const uint2 e = reinterpret_cast<const uint2*>(codebook)[c & 127];
        uint32_t flip = (c & 0x80) ? 0x80008000u : 0u;
        cbt[idx] = make_uint2(e.x ^ flip, e.y ^ flip);
    }

    for (long item = blockIdx.x; item < n_items; item += gridDim.x) {
        const Chunk ch = chunks[item / row_groups];
        const int rg = (int)(item % row_groups);
        const SlotDesc d = desc[ch.expert];
        const int fmt = ch.fmt;
        const int xs = xstride_bytes(K, fmt);
        __syncthreads();  // previous item's readers of xt are done
        // activations of the chunk -> fp16 [NT][K] (zero rows past count)
        for (int idx = threadIdx.x; idx < NT * (K / 8); idx += blockDim.x) {
            const int n = idx / (K / 8), c8 = idx % (K / 8);
            uint4 v = make_uint4(0, 0, 0, 0);
            if (n < ch.count) {
                float f[8];
                if (NMAT == 2) {
                    const int t = sorted_pair[ch.start + n] / k;
                    const uint4 b = *reinterpret_cast<const uint4*>(x_bf16 + (size_t)t * K + 8 * c8);
                    const uint32_t w4[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        f[2 * q] = __uint_as_float(w4[q] << 16);
                        f[2 * q + 1] = __uint_as_float(w4[q] & 0xffff0000u);
                    }
                } else {
                    const float4* src = reinterpret_cast<const float4*>(a_in + (size_t)(ch.start + n) * K + 8 * c8);
                    const float4 p0 = src[0], p1 = src[1];
                    f[0] = p0.x; f[1] = p0.y; f[2] = p0.z; f[3] = p0.w;
                    f[4] = p1.x; f[5] = p1.y; f[6] = p1.z; f[7] = p1.w;
                }
                __half2 h0 = __floats2half2_rn(f[0], f[1]), h1 = __floats2half2_rn(f[2], f[3]);
                __half2 h2 = __floats2half2_rn(f[4], f[5]), h3 = __floats2half2_rn(f[6], f[7]);
                v = make_uint4(*reinterpret_cast<uint32_t*>(&h0), *reinterpret_cast<uint32_t*>(&h1),
                               *reinterpret_cast<uint32_t*>(&h2), *reinterpret_cast<uint32_t*>(&h3));
            }
            *reinterpret_cast<uint4*>(xt + (size_t)n * xs + 16 * c8) = v;
        }
        __syncthreads();

        const int rt = rg * WARPS + warp;  // 16-row tile of this warp
        float acc[NMAT][4];
#pragma unroll
        for (int m = 0; m < NMAT; ++m)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[m][q] = 0.0f;

        // Each step covers 128 inputs (VQ2: one scale block) or 64 (FP4).
        const int step_in = fmt == MOE_FMT_VQ2 ? 128 : 64;
        const int nsteps = K / step_in;
        const uint8_t* cbase[NMAT];
#pragma unroll
        for (int m = 0; m < NMAT; ++m)
            cbase[m] = reinterpret_cast<const uint8_t*>(d.codes[NMAT == 2 ? m : 2]) + (size_t)rt * nsteps * 512;

        auto issue = [&](int st) {
            if (st < nsteps) {
                uint8_t* dst = ring + (st % STAGES) * STAGE_BYTES;
#pragma unroll
                for (int m = 0; m < NMAT; ++m) cp_async16(dst + m * 512 + 16 * lane, cbase[m] + (size_t)st * 512 + 16 * lane);
            }
            cp_async_commit();
        };
#pragma unroll
        for (int st = 0; st < STAGES - 1; ++st) issue(st);

        for (int st = 0; st < nsteps; ++st) {
            issue(st + STAGES - 1);
            cp_async_wait<STAGES - 1>();
            __syncwarp();
            const uint8_t* stg = ring + (st % STAGES) * STAGE_BYTES;
            if (fmt == MOE_FMT_VQ2) {
                const int kb = st;
                float tmp[NMAT][4];
#pragma unroll
                for (int m = 0; m < NMAT; ++m)
#pragma unroll
                    for (int q = 0; q < 4; ++q) tmp[m][q] = 0.0f;
#pragma unroll
                for (int s = 0; s < 8; ++s) {
                    const int G = kb * 32 + 4 * s + j;  // this thread's group
                    const uint2 b = *reinterpret_cast<const uint2*>(xt + (size_t)i * xs + 8 * G);
#pragma unroll
                    for (int m = 0; m < NMAT; ++m) {
                        const uint32_t pr = *reinterpret_cast<const uint16_t*>(stg + m * 512 + 16 * (4 * s + j) + 2 * i);
                        const uint2 lo = cbt[(pr & 0xff) * CB_COPIES + (lane & 15)];
                        const uint2 hi = cbt[(pr >> 8) * CB_COPIES + (lane & 15)];
                        mma_16816(tmp[m], lo.x, hi.x, lo.y, hi.y, b.x, b.y);
                    }
                }
#pragma unroll
                for (int m = 0; m < NMAT; ++m) {
                    const __half* sc = reinterpret_cast<const __half*>(d.scales[NMAT == 2 ? m : 2]) +
                                       ((size_t)rt * nsteps + kb) * 16;
                    const float s_lo = __half2float(sc[i]), s_hi = __half2float(sc[i + 8]);
                    acc[m][0] += s_lo * tmp[m][0];
                    acc[m][1] += s_lo * tmp[m][1];
                    acc[m][2] += s_hi * tmp[m][2];
                    acc[m][3] += s_hi * tmp[m][3];
                }
            } else {
                const int kt = st;
                const int KB32 = K / 32;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    float tmp[NMAT][4];
#pragma unroll
                    for (int m = 0; m < NMAT; ++m)
#pragma unroll
                        for (int q = 0; q < 4; ++q) tmp[m][q] = 0.0f;
#pragma unroll
                    for (int s2 = 0; s2 < 2; ++s2) {
                        const int s = 2 * half + s2;
                        const int e0 = kt * 64 + 16 * s + 2 * j;  // element of k-slot 2j
                        const uint32_t b0 = *reinterpret_cast<const uint32_t*>(xt + (size_t)i * xs + 2 * e0);
                        const uint32_t b1 = *reinterpret_cast<const uint32_t*>(xt + (size_t)i * xs + 2 * (e0 + 8));
#pragma unroll
                        for (int m = 0; m < NMAT; ++m) {
                            const uint32_t w = *reinterpret_cast<const uint32_t*>(stg + m * 512 + 16 * lane + 4 * s);
                            uint32_t r0, r1, r2, r3;  // row i lo, row i hi-k, row i+8 lo, row i+8 hi-k
                            e2m1x8_to_f16x8(w, r0, r1, r2, r3);
                            mma_16816(tmp[m], r0, r2, r1, r3, b0, b1);
                        }
                    }
#pragma unroll
                    for (int m = 0; m < NMAT; ++m) {
                        const uint8_t* sc = reinterpret_cast<const uint8_t*>(d.scales[NMAT == 2 ? m : 2]) +
                                            ((size_t)rt * KB32 + 2 * kt + half) * 16;
                        const float s_lo = e8m0_to_float(sc[i]), s_hi = e8m0_to_float(sc[i + 8]);
                        acc[m][0] += s_lo * tmp[m][0];
                        acc[m][1] += s_lo * tmp[m][1];
                        acc[m][2] += s_hi * tmp[m][2];
                        acc[m][3] += s_hi * tmp[m][3];
                    }
                }
            }
            __syncwarp();
        }
        cp_async_wait<0>();

        // epilogue: accumulator (row i | i+8, token 2j | 2j+1)
        const int r_lo = rt * 16 + i, r_hi = r_lo + 8;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int tok = 2 * j + (q & 1);
            const int row = (q & 2) ? r_hi : r_lo;
            if (tok >= ch.count) continue;
            const int spos = ch.start + tok;
            if (NMAT == 2) {
                a_out[(size_t)spos * R + row] = silu_mul(acc[0][q], acc[NMAT - 1][q]);
            } else if (mode == MOE_PER_PAIR) {
                out[(size_t)spos * R + row] = acc[0][q];
            } else {
                const int p = sorted_pair[spos];
                atomicAdd(out + (size_t)(p / k) * R + row, weights[p] * acc[0][q]);
            }
        }
    }
    pdl_launch_dependents();
}

size_t mma_smem_bytes(int K) { return 256 * CB_COPIES * 8 + (size_t)NT * (2 * K + 32) + WARPS * STAGES * STAGE_BYTES; }

}  // namespace

size_t ffn_workspace_size(int T, int k, int E, int H, int I) { return ws_layout(T, k, E, H, I).total; }

moe_status launch_expert_ffn(const SlotTableHost* t, const uint16_t* x, const int32_t* offsets,
                             const int32_t* sorted_pair, const float* weights, int T, int k, int mode,
                             float* out, uint8_t* status, void* ws, size_t ws_bytes, cudaStream_t s) {
    (void)ws_bytes;
    const int E = t->E, H = t->H, I = t->I;
    const int P = T * k;
    if (k > 32) {  // the experts of one token are handled as one group of at most 32
        set_error("moe_vq2_expert_ffn: k=%d above 32", k);
        return MOE_ERR_UNSUPPORTED;
    }
    const WsLayout L = ws_layout(T, k, E, H, I);
    char* w = static_cast<char*>(ws);
    int* header = reinterpret_cast<int*>(w);
    Chunk* chunks = reinterpret_cast<Chunk*>(w + L.chunks_off);
    int32_t* lut_s = reinterpret_cast<int32_t*>(w + L.lut_s_off);
    int32_t* lut_e = reinterpret_cast<int32_t*>(w + L.lut_e_off);
    int32_t* lut_grp = reinterpret_cast<int32_t*>(w + L.lut_grp_off);
    int32_t* grp_start = reinterpret_cast<int32_t*>(w + L.grp_start_off);
    float* abuf = reinterpret_cast<float*>(w + L.a_off);
    const int use_lut = 1;
    cudaError_t e;

    e = launch_pdl(schedule_kernel, dim3(1), dim3(1024), 0, s, (const SlotDesc*)t->d_desc, E, offsets, sorted_pair, P,
                   k, status, header, chunks, lut_s, lut_e, lut_grp, grp_start, use_lut);
    if (e != cudaSuccess) return cuda_status(e, "moe_vq2_expert_ffn: schedule launch");
    MOE_LAUNCH_CHECK("moe_vq2_expert_ffn: schedule launch");

    const size_t smem1 = mma_smem_bytes(H), smem2 = mma_smem_bytes(I);
    if (smem1 > 227 * 1024 || smem2 > 227 * 1024) {
        set_error("moe_vq2_expert_ffn: H=%d / I=%d too large for the decode kernel's shared memory", H, I);
        return MOE_ERR_UNSUPPORTED;
    }
    e = ensure_smem_attr(ffn_mma_kernel<2>, (int)smem1);
    if (e != cudaSuccess) return cuda_status(e, "moe_vq2_expert_ffn: smem attribute");
    e = ensure_smem_attr(ffn_mma_kernel<1>, (int)smem2);
    if (e != cudaSuccess) return cuda_status(e, "moe_vq2_expert_ffn: smem attribute");

    const unsigned grid = (unsigned)num_sms();
    moe_status st;
    if (use_lut && (st = launch_lut_fc(true, t, x, sorted_pair, k, w, L, s)) != MOE_OK) return st;
    e = launch_pdl(ffn_mma_kernel<2>, dim3(grid), dim3(32 * WARPS), smem1, s, t->d_desc, t->codebook, x,
                   (const float*)nullptr, sorted_pair, weights, k, H, I, (const int*)header, (const Chunk*)chunks,
                   abuf, (float*)nullptr, mode);
    if (e != cudaSuccess) return cuda_status(e, "moe_vq2_expert_ffn: FC1 launch");
    MOE_LAUNCH_CHECK("moe_vq2_expert_ffn: FC1 launch");
    if (use_lut && (st = launch_lut_fc(false, t, x, sorted_pair, k, w, L, s)) != MOE_OK) return st;
    e = launch_pdl(ffn_mma_kernel<1>, dim3(grid), dim3(32 * WARPS), smem2, s, t->d_desc, t->codebook,
                   (const uint16_t*)nullptr, (const float*)abuf, sorted_pair, weights, k, I, H, (const int*)header,
                   (const Chunk*)chunks, (float*)nullptr, out, mode);
    if (e != cudaSuccess) return cuda_status(e, "moe_vq2_expert_ffn: FC2 launch");
    MOE_LAUNCH_CHECK("moe_vq2_expert_ffn: FC2 launch");
    if (use_lut && (st = launch_lut_finish(t, sorted_pair, weights, k, mode, out, w, L, L.max_lut, s)) != MOE_OK)
        return st;
    return MOE_OK;
}

}  // namespace moe
