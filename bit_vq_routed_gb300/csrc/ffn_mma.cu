// Tensor-core mma.sync path of the expert FFN for VQ2 experts with more tokens
// than the activation-table path takes and fewer than the tcgen05 threshold,
// and for FP4 experts with any count.
//
// mma.sync m16n8k16 (fp16 in, fp32 accumulate) on weights decoded in
// registers.  A VQ2 code byte indexes a sign-folded codebook (256 entries:
// each index and its negation) held in shared memory 16 times over, so the two
// half-warps of an 8-byte lookup hit distinct banks; the entry's 4 fp16
// values are exactly one thread's A-fragment for one row: the K order inside
// each 16-wide MMA step is permuted so a thread's 4 k-slots are one code's 4
// inputs, and the activations use the same permutation.  The entry is
// multiplied by its row scale in fp16 (the weight rounded once, as the
// tcgen05 decoders do), which keeps one set of fp32 accumulators (two CTAs
// fit per SM).  FP4 (e2m1) bytes become f16x2 with cvt and are scaled per 32
// inputs.
//
// A CTA of 8 warps takes items (chunk of tokens of one expert, 8 x 32 weight
// rows); each warp owns two 16-row tiles (FC1: the gate and the up tile of the
// same rows; FC2: two down tiles), so every activation fragment feeds two
// tiles.  K is walked in slabs: the chunk's fp16 activations (gathered by
// sorted position) and each warp's code and scale tiles for the next slab
// stream into shared memory with cp.async while the current slab is computed.
// Chunk size, slab length and CTAs per SM come in three configurations (MmaCfg).
#include "ffn_common.cuh"

namespace moe {
namespace {

template <int N>
struct IntTag {
    static constexpr int value = N;
};

constexpr int WARPS = 8;
constexpr int THREADS = 32 * WARPS;
constexpr int CB_COPIES = 16;

// Configurations.  32-token chunks (VQ2; an expert's codes are read once per
// 32 tokens): in calls of at least MMA_SPLIT_T tokens ("wide") 512-input
// slabs and one CTA per SM, below that 256-input slabs and two CTAs per SM
// (measured: batch 32 255 -> 239 us per call with two; prefill of 4096
// tokens 2.33 -> 2.56 ms).  16-token chunks (FP4 experts, the most routed ones
// at small batches with few tokens each, and in large calls the VQ2 experts
// with at most 16 tokens): 256-input slabs, two CTAs per SM, whose independent
// slab barriers hide more latency.
template <int NTOK_, bool WIDE_>
struct MmaCfg {
    static constexpr int NTOK = NTOK_;                   // tokens per chunk
    static constexpr int NNT = NTOK / 8;                 // n8 MMA tiles per chunk
    static constexpr int SLAB = WIDE_ ? 512 : 256;       // inputs per slab (VQ2; FP4 slabs are half as many)
    static constexpr int XSTRIDE = 2 * SLAB + 32;        // bytes per token row of a slab (padding: B-fragment banks)
    // FP4 slabs (SLAB / 2 inputs): rows 4 banks apart, so that the 8 rows x 4
    // k-pairs of a warp's 32-bit B loads hit 32 distinct banks
    static constexpr int XSTRIDE_F4 = SLAB + 16;
    static constexpr int TILE_CODES = 4 * SLAB;          // one 16-row tile x one slab
    static constexpr int TILE_SCALES = SLAB / 4;         // 16 rows x SLAB/128 fp16 (VQ2) or x SLAB/64 ue8m0 (FP4)
    static constexpr int WARP_BYTES = 2 * (TILE_CODES + TILE_SCALES);  // per warp per slab (two tiles)
    static constexpr int MIN_BLOCKS = WIDE_ ? 1 : 2;
    struct __align__(16) Smem {
        uint2 cbt[256 * CB_COPIES];
        uint8_t xs[2][NTOK * XSTRIDE];
        uint8_t w[2][WARPS][WARP_BYTES];
    };
};
static_assert(MMA_NT_VQ2 == 32 && MMA_NT_FP4 == 16, "mma.sync configurations");

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait1() { asm volatile("cp.async.wait_group 1;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait0() { asm volatile("cp.async.wait_group 0;\n" ::: "memory"); }
// shared-memory reads as plain C++ accesses (the compiler may overlap them)
__device__ __forceinline__ uint32_t sh_u16(const uint8_t* p) { return *reinterpret_cast<const uint16_t*>(p); }
__device__ __forceinline__ uint2 sh_u64(const uint8_t* p) { return *reinterpret_cast<const uint2*>(p); }
__device__ __forceinline__ uint32_t sh_u32(const uint8_t* p) { return *reinterpret_cast<const uint32_t*>(p); }
__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
    const __half2 r = __hmul2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
    return *reinterpret_cast<const uint32_t*>(&r);
}

// FC1 = true: A tiles are the gate and up tiles of 16 I-rows, B = x16s (K = H);
// FC1 = false: A tiles are two down tiles (32 H-rows), B = a16 (K = I).
// The B rows are scaled by powers of two (x16s = x / xsc, a16 = a / asc, per
// sorted position); the epilogues multiply the scale back in fp32.  FC1
// writes a in fp32 (a32) and flags each sorted position it wrote (amax).
template <bool FC1, int NTOK_, bool WIDE_>
__global__ void __launch_bounds__(THREADS, MmaCfg<NTOK_, WIDE_>::MIN_BLOCKS)
    ffn_mma_kernel(const SlotDesc* __restrict__ desc, const uint16_t* __restrict__ codebook,
                   const uint16_t* __restrict__ bsrc, const int32_t* __restrict__ sorted_pair,
                   const float* __restrict__ weights, int k, int H, int I, const int* __restrict__ header,
                   const Chunk* __restrict__ chunks, const float* __restrict__ xsc, const float* __restrict__ asc,
                   float* __restrict__ a32, uint32_t* __restrict__ amax, float* __restrict__ out, int mode,
                   int part16) {
    using Cfg = MmaCfg<NTOK_, WIDE_>;
    using Smem = typename Cfg::Smem;
    constexpr int NTOK = Cfg::NTOK, NNT = Cfg::NNT, SLAB = Cfg::SLAB, XSTRIDE = Cfg::XSTRIDE;
    constexpr int XSTRIDE_F4 = Cfg::XSTRIDE_F4;
    static_assert(XSTRIDE_F4 % 16 == 0 && (XSTRIDE_F4 / 4) % 8 == 4, "FP4 row stride: 16-byte rows, 4 banks apart");
    constexpr int TILE_CODES = Cfg::TILE_CODES, TILE_SCALES = Cfg::TILE_SCALES;
    extern __shared__ __align__(16) uint8_t dyn[];
    Smem& S = *reinterpret_cast<Smem*>(dyn);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int i = lane >> 2, j = lane & 3;
    const int K = FC1 ? H : I;
    const int R = FC1 ? I : H;                      // rows per matrix
    const int ROWS = FC1 ? 16 * WARPS : 32 * WARPS;  // rows per item
    const int n_rg = R / ROWS;

    pdl_wait();
    pdl_launch_dependents();  // dependents may start their prologues now
    // the chunks list holds the 32-token chunks, then the 16-token ones: this launch's part
    const int c0 = part16 ? header[HDR_NVQ2] : 0;
    const int n_chunks = (part16 ? header[HDR_NCHUNKS] : header[HDR_NVQ2]) - c0;
    const int n_items = n_chunks * n_rg;
    if ((int)blockIdx.x >= n_items) return;
    for (int idx = tid; idx < 256 * CB_COPIES; idx += THREADS) {
        const int c = idx / CB_COPIES;
        const uint2 e = reinterpret_cast<const uint2*>(codebook)[c & 127];
        const uint32_t flip = (c & 0x80) ? 0x80008000u : 0u;
        S.cbt[idx] = make_uint2(e.x ^ flip, e.y ^ flip);
    }
    const uint8_t* cbt = reinterpret_cast<const uint8_t*>(&S.cbt[0]) + 8 * (lane & 15);

    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
        const Chunk ch = chunks[c0 + item / n_rg];
        const int rg = item % n_rg;
        const SlotDesc& d = desc[ch.expert];
        const bool vq2 = ch.fmt == MOE_FMT_VQ2;
        const int n_nt = (ch.count + 7) >> 3;
        // this warp's two 16-row tiles: (matrix, row tile)
        int mt[2], rtt[2];
        if (FC1) {
            mt[0] = 0, mt[1] = 1;
            rtt[0] = rtt[1] = rg * WARPS + warp;
        } else {
            mt[0] = mt[1] = 2;
            rtt[0] = (rg * WARPS + warp) * 2;
            rtt[1] = rtt[0] + 1;
        }
        const int KB = vq2 ? K / 128 : K / 32;  // scale blocks per row
        const int KT = vq2 ? K / 128 : K / 64;  // 512-byte code tiles per row tile
        const int slab_in = vq2 ? SLAB : SLAB / 2;
        const int nslab = (K + slab_in - 1) / slab_in;
        const int xstride = vq2 ? XSTRIDE : XSTRIDE_F4;

        // issue the cp.async copies of slab sl into buffer sl & 1
        auto issue = [&](int sl) {
            const int buf = sl & 1;
            const int k0 = sl * slab_in, kn = min(slab_in, K - k0);
            // activations: NTOK rows x kn fp16, zero rows past the chunk
            const int chunks_per_row = kn / 8;
            for (int idx = tid; idx < NTOK * chunks_per_row; idx += THREADS) {
                const int n = idx / chunks_per_row, c = idx - n * chunks_per_row;
                const bool valid = n < ch.count;
                const uint16_t* src = bsrc + (size_t)(ch.start + (valid ? n : 0)) * K + k0 + 8 * c;
                cp_async16(smem_u32(&S.xs[buf][n * xstride + 16 * c]), src, valid);
            }
            // this warp's code tiles and scales
            uint8_t* wb = &S.w[buf][warp][0];
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                const uint8_t* cbase = static_cast<const uint8_t*>(d.codes[mt[t]]);
                const int ntile = vq2 ? kn / 128 : kn / 64;  // 512-byte tiles in this slab
                const int tile0 = vq2 ? k0 / 128 : k0 / 64;
                const uint8_t* src = cbase + ((size_t)rtt[t] * KT + tile0) * 512;
                for (int c = lane; c < ntile * 32; c += 32)
                    cp_async16(smem_u32(wb + t * TILE_CODES + 16 * c), src + 16 * c, true);
                const int sblk = vq2 ? kn / 128 : kn / 32;  // scale blocks in this slab
                const int sb0 = vq2 ? k0 / 128 : k0 / 32;
                const int sbytes = vq2 ? 32 * sblk : 16 * sblk;  // 16 rows x (fp16 | ue8m0)
                const uint8_t* ssrc = static_cast<const uint8_t*>(d.scales[mt[t]]) +
                                      ((size_t)rtt[t] * KB + sb0) * (vq2 ? 32 : 16);
                for (int c = lane; c < sbytes / 16; c += 32)
                    cp_async16(smem_u32(wb + 2 * TILE_CODES + t * TILE_SCALES + 16 * c), ssrc + 16 * c, true);
            }
            cp_async_commit();
        };

        float acc[2][NNT][4];
#pragma unroll
        for (int t = 0; t < 2; ++t)
#pragma unroll
            for (int nt = 0; nt < NNT; ++nt)
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[t][nt][q] = 0.0f;

        __syncthreads();  // the previous item is done with both buffers
        issue(0);
        for (int sl = 0; sl < nslab; ++sl) {
            if (sl + 1 < nslab) {
                issue(sl + 1);
                cp_async_wait1();
            } else {
                cp_async_wait0();
            }
            __syncthreads();  // everyone's copies of slab sl have landed
            const int buf = sl & 1;
            const int kn = min(slab_in, K - sl * slab_in);
            const uint8_t* xs = &S.xs[buf][0];
            const uint8_t* wb = &S.w[buf][warp][0];
            if (vq2) {
                for (int kb = 0; kb < kn / 128; ++kb) {
                    // the rows' fp16 scales (rows i and i + 8 of each tile) in both halves
                    uint32_t sl2[2], sh2[2];
#pragma unroll
                    for (int t = 0; t < 2; ++t) {
                        const uint8_t* sa = wb + 2 * TILE_CODES + t * TILE_SCALES + kb * 32;
                        sl2[t] = sh_u16(sa + 2 * i) * 0x10001u;
                        sh2[t] = sh_u16(sa + 2 * (i + 8)) * 0x10001u;
                    }
#pragma unroll
                    for (int s = 0; s < 8; ++s) {
                        const int g = 4 * s + j;  // this thread's group in the scale block
                        uint2 b[NNT];
#pragma unroll
                        for (int nt = 0; nt < NNT; ++nt)
                            if (nt < n_nt) b[nt] = sh_u64(xs + (8 * nt + i) * XSTRIDE + 2 * (kb * 128 + 4 * g));
#pragma unroll
                        for (int t = 0; t < 2; ++t) {
                            const uint32_t pr = sh_u16(wb + t * TILE_CODES + kb * 512 + 16 * g + 2 * i);
                            const uint2 lo = sh_u64(cbt + 128u * (pr & 0xffu));
                            const uint2 hi = sh_u64(cbt + 128u * (pr >> 8));
                            const uint32_t a0 = hmul2_u32(lo.x, sl2[t]), a1 = hmul2_u32(hi.x, sh2[t]);
                            const uint32_t a2 = hmul2_u32(lo.y, sl2[t]), a3 = hmul2_u32(hi.y, sh2[t]);
#pragma unroll
                            for (int nt = 0; nt < NNT; ++nt)
                                if (nt < n_nt) mma_16816(acc[t][nt], a0, a1, a2, a3, b[nt].x, b[nt].y);
                        }
                    }
                }
            } else if constexpr (NTOK == MMA_NT_FP4) {
                // NA: the n8 tiles that hold tokens of this chunk (a compile-time
                // count, so that the block-scale products and the zeroed partial
                // sums of the empty tiles are not computed); the 64-element tiles
                // of a slab two per pass, so that one's loads and conversions
                // overlap the other's MMAs
                auto fp4_slab = [&](auto na_tag) {
                    constexpr int NA = decltype(na_tag)::value;
#pragma unroll 2
                    for (int kt = 0; kt < kn / 64; ++kt) {
                        // this lane's 16 code bytes of each tile (4 words: s = 0..3)
                        uint4 wv[2];
#pragma unroll
                        for (int t = 0; t < 2; ++t)
                            wv[t] = *reinterpret_cast<const uint4*>(wb + t * TILE_CODES + kt * 512 + 16 * lane);
#pragma unroll
                        for (int half = 0; half < 2; ++half) {  // 32-element scale blocks
                            float tmp[2][NA][4];
#pragma unroll
                            for (int t = 0; t < 2; ++t)
#pragma unroll
                                for (int nt = 0; nt < NA; ++nt)
#pragma unroll
                                    for (int q = 0; q < 4; ++q) tmp[t][nt][q] = 0.0f;
#pragma unroll
                            for (int s2 = 0; s2 < 2; ++s2) {
                                const int s = 2 * half + s2;
                                const int e0 = kt * 64 + 16 * s + 2 * j;  // element of k-slot 2j
                                uint32_t b0[NA], b1[NA];
#pragma unroll
                                for (int nt = 0; nt < NA; ++nt) {
                                    b0[nt] = sh_u32(xs + (8 * nt + i) * XSTRIDE_F4 + 2 * e0);
                                    b1[nt] = sh_u32(xs + (8 * nt + i) * XSTRIDE_F4 + 2 * (e0 + 8));
                                }
#pragma unroll
                                for (int t = 0; t < 2; ++t) {
                                    const uint32_t w = (&wv[t].x)[s];
                                    uint32_t r0, r1, r2, r3;  // row i lo-k, row i hi-k, row i+8 lo-k, row i+8 hi-k
                                    e2m1x8_to_f16x8(w, r0, r1, r2, r3);
#pragma unroll
                                    for (int nt = 0; nt < NA; ++nt) mma_16816(tmp[t][nt], r0, r2, r1, r3, b0[nt], b1[nt]);
                                }
                            }
#pragma unroll
                            for (int t = 0; t < 2; ++t) {
                                const uint8_t* sa = wb + 2 * TILE_CODES + t * TILE_SCALES + (2 * kt + half) * 16;
                                const uint32_t e_lo = sa[i], e_hi = sa[i + 8];
                                const float s_lo = e8m0_to_float(e_lo), s_hi = e8m0_to_float(e_hi);
#pragma unroll
                                for (int nt = 0; nt < NA; ++nt) {
                                    acc[t][nt][0] = fmaf(s_lo, tmp[t][nt][0], acc[t][nt][0]);
                                    acc[t][nt][1] = fmaf(s_lo, tmp[t][nt][1], acc[t][nt][1]);
                                    acc[t][nt][2] = fmaf(s_hi, tmp[t][nt][2], acc[t][nt][2]);
                                    acc[t][nt][3] = fmaf(s_hi, tmp[t][nt][3], acc[t][nt][3]);
                                }
                            }
                        }
                    }
                };
                static_assert(NNT == 2, "FP4 chunks: one or two n8 tiles");
                if (n_nt == 1)
                    fp4_slab(IntTag<1>{});
                else
                    fp4_slab(IntTag<2>{});
            }
            __syncthreads();  // buffer buf is free for the copies of slab sl + 2
        }

        // epilogue: acc[t][nt] holds (row i | i+8 of tile t, tokens 8nt + 2j | +1):
        // acc[t][nt][b + 2 hi] is token 8 nt + 2 j + b, row i + 8 hi
#pragma unroll
        for (int nt = 0; nt < NNT; ++nt) {
            if (nt >= n_nt) continue;
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                const int tok = 8 * nt + 2 * j + b;
                const bool valid = tok < ch.count;
                const int spos = ch.start + (valid ? tok : 0);
                const float sc = valid ? (FC1 ? xsc[spos] : asc[spos]) : 0.0f;
                if (FC1) {
                    if (valid) {
#pragma unroll
                        for (int hi = 0; hi < 2; ++hi) {
                            const float g = acc[0][nt][b + 2 * hi] * sc, u = acc[1][nt][b + 2 * hi] * sc;
                            a32[(size_t)spos * I + rtt[0] * 16 + i + 8 * hi] = silu_mul(g, u);
                        }
                        if (i == 0) amax[spos] = 1;  // written: the conversion takes this position
                    }
                } else if (valid) {
#pragma unroll
                    for (int t = 0; t < 2; ++t)
#pragma unroll
                        for (int hi = 0; hi < 2; ++hi) {
                            const int row = rtt[t] * 16 + i + 8 * hi;
                            const float y = acc[t][nt][b + 2 * hi] * sc;
                            if (mode == MOE_PER_PAIR) {
                                out[(size_t)spos * H + row] = y;
                            } else {
                                const int p = sorted_pair[spos];
                                atomicAdd(out + (size_t)(p / k) * H + row, weights[p] * y);
                            }
                        }
                }
            }
        }
    }
}

}  // namespace


template <int NTOK_, bool WIDE_>
static moe_status launch_mma_cfg(bool fc1, const SlotTableHost* t, const int32_t* sorted_pair, const float* weights,
                                 int k, int mode, float* out, char* ws, const WsLayout& L, cudaStream_t s) {
    using Smem = typename MmaCfg<NTOK_, WIDE_>::Smem;
    const int* header = reinterpret_cast<const int*>(ws);
    const Chunk* chunks = reinterpret_cast<const Chunk*>(ws + L.chunks_off);
    const uint16_t* x16s = reinterpret_cast<const uint16_t*>(ws + L.x16s_off);
    const uint16_t* a16 = reinterpret_cast<const uint16_t*>(ws + L.a16_off);
    auto kern = fc1 ? ffn_mma_kernel<true, NTOK_, WIDE_> : ffn_mma_kernel<false, NTOK_, WIDE_>;
    cudaError_t e = ensure_smem_attr(kern, (int)sizeof(Smem));
    if (e != cudaSuccess) return cuda_status(e, "moe_vq2_expert_ffn: mma kernel shared memory");
    e = launch_pdl(kern, dim3((unsigned)(MmaCfg<NTOK_, WIDE_>::MIN_BLOCKS * num_sms())), dim3(THREADS), sizeof(Smem), s,
                   (const SlotDesc*)t->d_desc, t->codebook, fc1 ? x16s : a16, sorted_pair, weights, k, t->H, t->I,
                   header, chunks, reinterpret_cast<const float*>(ws + L.xsc_off),
                   reinterpret_cast<const float*>(ws + L.asc_off), reinterpret_cast<float*>(ws + L.a32_off),
                   reinterpret_cast<uint32_t*>(ws + L.amax_off), out, mode, NTOK_ == MMA_NT_FP4 ? 1 : 0);
    if (e != cudaSuccess) return cuda_status(e, fc1 ? "moe_vq2_expert_ffn: FC1 launch" : "moe_vq2_expert_ffn: FC2 launch");
    return MOE_OK;
}

moe_status launch_mma_fc(bool fc1, const SlotTableHost* t, const int32_t* sorted_pair, const float* weights, int k,
                         int mode, float* out, char* ws, const WsLayout& L, cudaStream_t s, bool split16, bool vq2) {
    // (split16 is set exactly for the calls of at least MMA_SPLIT_T tokens;
    // vq2: the call can have VQ2 experts in 32-token chunks)
    moe_status st = MOE_OK;
    if (vq2)
        st = split16 ? launch_mma_cfg<MMA_NT_VQ2, true>(fc1, t, sorted_pair, weights, k, mode, out, ws, L, s)
                     : launch_mma_cfg<MMA_NT_VQ2, false>(fc1, t, sorted_pair, weights, k, mode, out, ws, L, s);
    if (st == MOE_OK && (t->n_fp4 > 0 || split16))
        st = launch_mma_cfg<MMA_NT_FP4, false>(fc1, t, sorted_pair, weights, k, mode, out, ws, L, s);
    return st;
}

}  // namespace moe
