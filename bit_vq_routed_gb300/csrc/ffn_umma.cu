// Tensor-core (tcgen05) path of the expert FFN for experts that receive a
// prefill-sized batch of tokens (m_e >= UMMA_MIN).  Here the expert FFN is a
// dense contraction: FC1 is [m_e x H] x [H x 2I], FC2 [m_e x I] x [I x H].
//
// One CTA per SM loops over work items (chunk of <= 256 tokens of one
// expert, two 128-row weight tiles: FC1 the gate and the up tile of the same
// 128 rows, FC2 two consecutive down tiles): each decoded weight tile serves
// up to 256 tokens.  Warp roles:
//   - 8 decoder warps turn the item's VQ2 codes into fp16 weights
//     (sign-folded codebook entry x row scale, rounded once to fp16) and store
//     them into shared memory in the 128-byte-swizzled K-major layout the
//     tensor core reads (A operand, 128 rows x 64 per K-block); each thread
//     fetches its codes and row scales (through L1) four K-blocks ahead;
//   - a TMA warp loads the chunk's activations (B operand, 256 tokens x 64,
//     fp16, same swizzle) with cp.async.bulk.tensor from a token-gathered
//     copy in the workspace;
//   - one thread issues tcgen05.mma (M128, N = the chunk's tokens rounded up
//     to 16, at most 256, K16; fp16 in, fp32 in TMEM) and tcgen05.commit
//     frees each stage when the tensor core is done;
//   - 4 epilogue warps read the accumulators back with tcgen05.ld (each warp
//     owns one quarter of the TMEM lanes = weight rows) and store FC1's
//     a = silu(g) * u in fp32 (a conversion kernel then makes the fp16 FC2 B
//     operand), or FC2's y per pair / w*y into the token's output; per 32
//     tokens the values are computed for all columns first (independent
//     chains), then only the chunk's tokens are stored.
// The two accumulators (2 x 256 columns) fill TMEM's 512 columns, so the
// next item's MMAs start when the epilogue has read them (the decoders and
// the TMA warp run ahead meanwhile).  Every wait is bounded: a wait that
// gives up records an error word and the CTA runs on to its end without
// issuing more work.
#include <cudaTypedefs.h>

#include "ffn_common.cuh"

namespace moe {
namespace {

constexpr int UM_M = 128, UM_N = UMMA_NT, UM_K = 64;
constexpr int STAGES = 3;
constexpr int DEC_WARPS = 8, EPI_WARPS = 4;
constexpr int EPI_SLOTS = 1 + DEC_WARPS / 4;  // warps sharing one TMEM lane quarter's epilogue
// registers per thread: each of the SM's four schedulers holds 16384
// registers for its share of the CTA's warps (the busiest holds
// ceil(warps / 4) of them)
constexpr int MAX_REG = 16384 / (32 * ((DEC_WARPS + 2 + EPI_WARPS + 3) / 4)) / 8 * 8;
constexpr int TMA_WARP = DEC_WARPS, MMA_WARP = DEC_WARPS + 1;  // then the epilogue warps
constexpr int THREADS = 32 * (DEC_WARPS + 2 + EPI_WARPS);
constexpr int A_BYTES = UM_M * UM_K * 2;      // 16 KB per A tile
constexpr int B_BYTES = UM_N * UM_K * 2;      // 32 KB
constexpr int CB_COPIES = 16;
// instruction descriptor: D f32, A/B f16, both K-major, M = 128, N = n
// (a multiple of 16, 16..256)
__host__ __device__ constexpr uint32_t idesc_n(int n) {
    return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(UM_M >> 4) << 24);
}

struct __align__(1024) Smem {
    uint8_t a[STAGES][2][A_BYTES];  // FC1: gate tile, up tile; FC2: two down tiles
    uint8_t b[STAGES][B_BYTES];
    uint2 cbt[256 * CB_COPIES];     // sign-folded codebook, 16 copies
    uint64_t full[STAGES], empty[STAGES], acc_full, acc_empty;
    uint32_t tmem_base;
    int failed;
};

// K-major, 128-byte-swizzled shared-memory matrix descriptor (rows of 128 B,
// groups of 8 rows 1024 B apart).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
            "r"(dst),
        "l"(map), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// A decoder thread's share of one K-block: one chunk (16 rows x 1 group =
// 16 code bytes) and the 16 row scales of its tile.
struct DecRegs {
    uint4 c, s0, s1;
};

// FC1 (FC1 = true): items = (chunk, 128-row tile of I), A = gate and up tiles.
// FC2: items = (chunk, 256-row tile of H), A = two 128-row down tiles.
// The B rows are scaled by powers of two (x16s = x / xsc, a16 = a / asc, per
// sorted position); the epilogue multiplies the scale back in fp32.  FC1
// writes a in fp32 (a32) and flags each sorted position it wrote (amax).
template <bool FC1>
__global__ void __maxnreg__(MAX_REG)
    ffn_umma_kernel(const __grid_constant__ CUtensorMap bmap, const SlotDesc* __restrict__ desc,
                    const uint16_t* __restrict__ codebook, const int32_t* __restrict__ sorted_pair,
                    const float* __restrict__ weights, int k, int H, int I, int* __restrict__ header,
                    const Chunk* __restrict__ uchunks, const float* __restrict__ xsc, const float* __restrict__ asc,
                    float* __restrict__ a32, uint32_t* __restrict__ amax, float* __restrict__ out, int mode) {
    extern __shared__ __align__(1024) uint8_t dyn[];
    // the swizzled operand tiles need 1024-byte alignment in the shared window
    Smem& S = *reinterpret_cast<Smem*>(dyn + ((1024u - (smem_u32(dyn) & 1023u)) & 1023u));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int* err = header + HDR_ERR;
    constexpr int NA = 2;                        // A tiles (and accumulators) per item
    constexpr uint32_t TMEM_COLS = NA * UM_N;    // the two accumulators: all 512 columns
    const int K = FC1 ? H : I;
    const int R = FC1 ? I : H;
    const int n_rt = R / (FC1 ? UM_M : 2 * UM_M);
    const int KB = K / 128;  // scale blocks per row
    const int n_kblk = K / UM_K;

    for (int idx = tid; idx < 256 * CB_COPIES; idx += THREADS) {
        const int c = idx / CB_COPIES;
        const uint2 e = reinterpret_cast<const uint2*>(codebook)[c & 127];
        const uint32_t flip = (c & 0x80) ? 0x80008000u : 0u;
        S.cbt[idx] = make_uint2(e.x ^ flip, e.y ^ flip);
    }
    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&S.full[s]), 32 * DEC_WARPS + 1);
            mbar_init(smem_u32(&S.empty[s]), 1);
        }
        mbar_init(smem_u32(&S.acc_full), 1);
        mbar_init(smem_u32(&S.acc_empty), 32 * (EPI_WARPS + DEC_WARPS));
        S.failed = 0;
    }
    if (warp == MMA_WARP) {  // allocate the accumulator columns (whole warp)
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&S.tmem_base)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    mbar_fence_init();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = S.tmem_base;
    pdl_wait();
    pdl_launch_dependents();  // dependents may start their prologues now

    const int n_chunks = header[HDR_NUMMA];
    const int n_items = n_chunks * n_rt;
    auto failed = [&]() { return *reinterpret_cast<volatile int*>(&S.failed) != 0; };
    auto wait = [&](uint64_t* bar, uint32_t parity, int code) {
        if (failed()) return false;
        if (!mbar_wait_sleep_bounded(smem_u32(bar), parity, err, code)) {
            *reinterpret_cast<volatile int*>(&S.failed) = 1;
            return false;
        }
        return true;
    };

    // The epilogue of one item, shared by the three warps of each TMEM lane
    // quarter (its epilogue warp, slot 0, and two decoder warps, slots 1 and
    // 2, which are idle then: their next stages are filled and the MMA waits
    // for the accumulators): 16-column chunks slot, slot + 3, ...  Per chunk
    // the row scales (and FC2's pair weights) are loaded once, one per lane,
    // and the values of all 16 columns computed before the guarded stores.
    auto epi_share = [&](int item, int slot) {
        const Chunk ch = uchunks[item / n_rt];
        const int rt = item % n_rt;
        const int quarter = warp & 3;  // TMEM lanes 32*quarter.. are this warp's
        const int row = quarter * 32 + lane;
        const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16);
        const int n16 = (ch.count + 15) >> 4;
#pragma unroll 1
        for (int c16 = slot; c16 < n16; c16 += EPI_SLOTS) {
            const int c0 = 16 * c16;
            const int nt = min(16, ch.count - c0);  // (the same for every lane)
            const int spos0 = ch.start + c0;
            float v[16];
            tmem_ld16(taddr + c0, v);
            if (FC1) {
                float u[16];
                tmem_ld16(taddr + UM_N + c0, u);
                const float sc_l = lane < nt ? xsc[spos0 + lane] : 0.0f;
                // written: the conversion takes these positions
                if (quarter == 0 && lane < nt) amax[spos0 + lane] = 1;
                float* dst = a32 + (size_t)spos0 * I + rt * UM_M + row;
#pragma unroll
                for (int q = 0; q < 16; ++q) {
                    const float sc = __shfl_sync(0xffffffffu, sc_l, q);
                    v[q] = silu_mul(v[q] * sc, u[q] * sc);
                }
#pragma unroll
                for (int q = 0; q < 16; ++q)
                    if (q < nt) dst[(size_t)q * I] = v[q];
            } else {
                const float sc_l = lane < nt ? asc[spos0 + lane] : 0.0f;
                int tok_l = 0;
                float w_l = 0.0f;
                if (mode != MOE_PER_PAIR && lane < nt) {
                    const int p = sorted_pair[spos0 + lane];
                    tok_l = p / k;
                    w_l = weights[p];
                }
#pragma unroll 1
                for (int t = 0; t < 2; ++t) {
                    if (t == 1) tmem_ld16(taddr + UM_N + c0, v);
                    const int h = rt * 2 * UM_M + t * UM_M + row;
#pragma unroll
                    for (int q = 0; q < 16; ++q) v[q] *= __shfl_sync(0xffffffffu, sc_l, q);
                    if (mode == MOE_PER_PAIR) {
                        float* dst = out + (size_t)spos0 * H + h;
#pragma unroll
                        for (int q = 0; q < 16; ++q)
                            if (q < nt) dst[(size_t)q * H] = v[q];
                    } else {
#pragma unroll
                        for (int q = 0; q < 16; ++q) {
                            const int tok = __shfl_sync(0xffffffffu, tok_l, q);
                            const float w = __shfl_sync(0xffffffffu, w_l, q);
                            if (q < nt) atomicAdd(out + (size_t)tok * H + h, w * v[q]);
                        }
                    }
                }
            }
        }
    };

    if (warp < DEC_WARPS) {
        // ------------------------------------------------ decoders
        // 256 threads = (A tile) x 8 row tiles x 16 groups, one chunk each.
        // A tile byte offset of (row R, 8-byte block g) = 128 R + swizzled
        // block; R & 7 is the chunk row's & 7 (row tiles start at multiples
        // of 16), so the 8 possible block offsets are precomputed.
        const int mat = tid >> 7;
        const int rtile = (tid >> 4) & 7;
        const int g = tid & 15;
        uint32_t boff[8];
#pragma unroll
        for (int r7 = 0; r7 < 8; ++r7)
            boff[r7] = 128u * (uint32_t)(rtile * 16) + ((((uint32_t)(g >> 1)) ^ (uint32_t)r7) << 4) + ((uint32_t)(g & 1) << 3);
        // warp-collective bounded wait: lane 0 polls, the warp follows
        auto warp_wait = [&](uint64_t* bar, uint32_t parity, int code) {
            int ok = 0;
            if (lane == 0) ok = wait(bar, parity, code) ? 1 : 0;
            __syncwarp();
            return __shfl_sync(0xffffffffu, ok, 0) != 0;
        };
        // this warp's share of the previous item's epilogue: when the first
        // STAGES K-blocks of the next item are submitted (or after the last
        // item)
        const int slot = 1 + warp / 4;
        int prev = -1, nprev = 0;
        auto dec_epi = [&]() {
            if (prev < 0) return;
            const int pi = prev;
            prev = -1;
            if (!warp_wait(&S.acc_full, nprev & 1, MOE_DEVERR_WAIT_FULL)) return;
            tc_fence_after();
            epi_share(pi, slot);
            tc_fence_before();
            mbar_arrive(smem_u32(&S.acc_empty));
        };
        int it = 0, nitem = 0;
        for (int item = blockIdx.x; item < n_items; item += gridDim.x, ++nitem) {
            const Chunk ch = uchunks[item / n_rt];
            const int rt = item % n_rt;
            const SlotDesc& d = desc[ch.expert];
            const int m = FC1 ? mat : 2;
            const int rtm = FC1 ? rt * 8 + rtile : rt * 16 + mat * 8 + rtile;
            const uint8_t* codes = static_cast<const uint8_t*>(d.codes[m]) + (size_t)rtm * KB * 512;
            const uint16_t* scales = static_cast<const uint16_t*>(d.scales[m]) + (size_t)rtm * KB * 16;
            auto fetch = [&](int kb64, DecRegs& r) {
                if (kb64 >= n_kblk) return;
                const int kb = kb64 >> 1, half = kb64 & 1;
                // through L1: a scale row serves both K-block halves
                r.c = __ldg(reinterpret_cast<const uint4*>(codes + (size_t)kb * 512 + 16 * (16 * half + g)));
                r.s0 = __ldg(reinterpret_cast<const uint4*>(scales + (size_t)kb * 16));
                r.s1 = __ldg(reinterpret_cast<const uint4*>(scales + (size_t)kb * 16 + 8));
            };
            auto step = [&](int kb64, const DecRegs& r) {
                if (kb64 == STAGES) dec_epi();
                const int stage = it % STAGES, use = it / STAGES;
                ++it;
                if (use > 0 && !warp_wait(&S.empty[stage], (use - 1) & 1, MOE_DEVERR_WAIT_EMPTY)) return;
                uint8_t* abase = &S.a[stage][mat][0];
                const uint32_t cw[4] = {r.c.x, r.c.y, r.c.z, r.c.w};
                const uint32_t sw[8] = {r.s0.x, r.s0.y, r.s0.z, r.s0.w, r.s1.x, r.s1.y, r.s1.z, r.s1.w};
                // the 16 codebook entries are loaded before any store into the
                // tile (the compiler cannot tell the tile from the codebook,
                // so loads placed after a store would wait for it), then
                // scaled and stored: 16 independent chains in flight
                uint2 e[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const uint32_t c = (cw[j >> 2] >> (8 * (j & 3))) & 0xffu;
                    e[j] = S.cbt[c * CB_COPIES + (lane & 15)];
                }
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int row = (j >> 1) + 8 * (j & 1);  // byte 2i+h holds row i + 8h
                    // the row's fp16 scale in both halves
                    const uint32_t s2 = prmt(sw[row >> 1], 0u, (row & 1) ? 0x3232u : 0x1010u);
                    __half2 w0 = __hmul2(*reinterpret_cast<const __half2*>(&e[j].x), *reinterpret_cast<const __half2*>(&s2));
                    __half2 w1 = __hmul2(*reinterpret_cast<const __half2*>(&e[j].y), *reinterpret_cast<const __half2*>(&s2));
                    *reinterpret_cast<uint2*>(abase + boff[row & 7] + 128u * (uint32_t)row) =
                        make_uint2(*reinterpret_cast<uint32_t*>(&w0), *reinterpret_cast<uint32_t*>(&w1));
                }
                fence_async_smem();
                mbar_arrive(smem_u32(&S.full[stage]));
            };
            // codes are fetched four K-blocks ahead of their decode
            DecRegs r0, r1, r2, r3;
            fetch(0, r0);
            fetch(1, r1);
            fetch(2, r2);
            fetch(3, r3);
            for (int kb64 = 0; kb64 < n_kblk; kb64 += 4) {
                step(kb64, r0);
                fetch(kb64 + 4, r0);
                if (kb64 + 1 < n_kblk) {
                    step(kb64 + 1, r1);
                    fetch(kb64 + 5, r1);
                }
                if (kb64 + 2 < n_kblk) {
                    step(kb64 + 2, r2);
                    fetch(kb64 + 6, r2);
                }
                if (kb64 + 3 < n_kblk) {
                    step(kb64 + 3, r3);
                    fetch(kb64 + 7, r3);
                }
            }
            dec_epi();  // (items of at most STAGES K-blocks)
            prev = item;
            nprev = nitem;
        }
        dec_epi();
    } else if (warp == TMA_WARP) {
        // ------------------------------------------------ activations (B)
        if (lane == 0) {
            int it = 0;
            for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
                const Chunk ch = uchunks[item / n_rt];
                for (int kb64 = 0; kb64 < n_kblk; ++kb64, ++it) {
                    const int stage = it % STAGES, use = it / STAGES;
                    if (use > 0 && !wait(&S.empty[stage], (use - 1) & 1, MOE_DEVERR_WAIT_EMPTY)) continue;
                    const uint32_t full = smem_u32(&S.full[stage]);
                    mbar_arrive_expect_tx(full, B_BYTES);
                    tma_load_2d(smem_u32(&S.b[stage][0]), &bmap, kb64 * UM_K, ch.start, full);
                }
            }
        }
    } else if (warp == MMA_WARP) {
        // ------------------------------------------------ MMA issue
        if (lane == 0) {
            int it = 0, nitem = 0;
            for (int item = blockIdx.x; item < n_items; item += gridDim.x, ++nitem) {
                const Chunk ch = uchunks[item / n_rt];
                const uint32_t idesc = idesc_n(min(UM_N, (ch.count + 15) & ~15));
                // the epilogue of the previous item must have read the accumulators
                if (nitem >= 1 && !wait(&S.acc_empty, (nitem - 1) & 1, MOE_DEVERR_WAIT_EMPTY)) break;
                tc_fence_after();
                const uint32_t d0 = tmem;
                for (int kb64 = 0; kb64 < n_kblk; ++kb64, ++it) {
                    const int stage = it % STAGES, use = it / STAGES;
                    if (!wait(&S.full[stage], use & 1, MOE_DEVERR_WAIT_FULL)) break;
                    tc_fence_after();
                    const uint64_t bd = sw128_desc(smem_u32(&S.b[stage][0]));
#pragma unroll
                    for (int t = 0; t < NA; ++t) {
                        const uint64_t ad = sw128_desc(smem_u32(&S.a[stage][t][0]));
#pragma unroll
                        for (int j = 0; j < UM_K / 16; ++j)  // 32 bytes of K per step inside the swizzle row
                            umma_f16(d0 + t * UM_N, ad + 2 * j, bd + 2 * j, idesc, (kb64 > 0 || j > 0) ? 1u : 0u);
                    }
                    umma_commit(smem_u32(&S.empty[stage]));
                }
                umma_commit(smem_u32(&S.acc_full));
            }
        }
    } else {
        // ------------------------------------------------ epilogue
        int nitem = 0;
        for (int item = blockIdx.x; item < n_items; item += gridDim.x, ++nitem) {
            int ok = 0;
            if (lane == 0) ok = wait(&S.acc_full, nitem & 1, MOE_DEVERR_WAIT_FULL) ? 1 : 0;
            __syncwarp();
            if (!__shfl_sync(0xffffffffu, ok, 0)) break;
            tc_fence_after();
            epi_share(item, 0);
            tc_fence_before();
            mbar_arrive(smem_u32(&S.acc_empty));
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == MMA_WARP) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void* p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// 2-D fp16 [rows, cols] row-major, box of 64 columns x 256 rows, 128B swizzle
bool make_map(CUtensorMap* map, const void* base, int rows, int cols) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {(cuuint32_t)UM_K, (cuuint32_t)UM_N};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

static_assert(sizeof(Smem) + 1024 <= 227 * 1024, "tcgen05 kernel shared memory");
size_t umma_smem_bytes() { return sizeof(Smem) + 1024; }

moe_status launch_umma(bool fc1, const SlotTableHost* t, const int32_t* sorted_pair, const float* weights, int k,
                       int P, int mode, float* out, char* ws, const WsLayout& L, cudaStream_t s) {
    int* header = reinterpret_cast<int*>(ws);
    const Chunk* uchunks = reinterpret_cast<const Chunk*>(ws + L.uchunks_off);
    uint16_t* x16s = reinterpret_cast<uint16_t*>(ws + L.x16s_off);
    uint16_t* a16 = reinterpret_cast<uint16_t*>(ws + L.a16_off);
    const int H = t->H, I = t->I;
    CUtensorMap map;
    if (!(fc1 ? make_map(&map, x16s, P, H) : make_map(&map, a16, P, I))) {
        set_error("moe_vq2_expert_ffn: tensor map encoding failed");
        return MOE_ERR_CUDA;
    }
    const int smem = (int)umma_smem_bytes();
    auto kern = fc1 ? ffn_umma_kernel<true> : ffn_umma_kernel<false>;
    cudaError_t e = ensure_smem_attr(kern, smem);
    if (e != cudaSuccess) return cuda_status(e, "moe_vq2_expert_ffn: tensor-core kernel shared memory");
    e = launch_pdl(kern, dim3((unsigned)num_sms()), dim3(THREADS), (size_t)smem, s, map, (const SlotDesc*)t->d_desc,
                   t->codebook, sorted_pair, weights, k, H, I, header, uchunks,
                   reinterpret_cast<const float*>(ws + L.xsc_off), reinterpret_cast<const float*>(ws + L.asc_off),
                   reinterpret_cast<float*>(ws + L.a32_off), reinterpret_cast<uint32_t*>(ws + L.amax_off), out, mode);
    if (e != cudaSuccess) return cuda_status(e, "moe_vq2_expert_ffn: tensor-core launch");
    return MOE_OK;
}

}  // namespace moe
