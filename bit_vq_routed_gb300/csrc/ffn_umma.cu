// Tensor-core (tcgen05) path of the expert FFN for experts that receive a
// prefill-sized batch of tokens (m_e >= UMMA_MIN).  Here the expert FFN is a
// dense contraction: FC1 is [m_e x H] x [H x 2I], FC2 [m_e x I] x [I x H].
//
// One CTA per SM loops over work items (chunk of <= 128 tokens of one expert,
// tile of 128 weight rows).  Per 64-input K-block:
//   - 4 decoder warps turn the tile's VQ2 codes into fp16 weights
//     (sign-folded codebook entry x row scale, rounded once to fp16) and store
//     them into shared memory in the 128-byte-swizzled K-major layout the
//     tensor core reads (A operand, 128 rows x 64);
//   - a TMA warp loads the chunk's activations (B operand, 128 tokens x 64,
//     fp16, same swizzle) with cp.async.bulk.tensor from a token-gathered
//     copy in the workspace;
//   - one thread issues tcgen05.mma (M128 N128 K16, fp16 in, fp32 in TMEM)
//     and tcgen05.commit frees the stage when the tensor core is done.
// After the last K-block the decoder warps read the accumulator back with
// tcgen05.ld (warp w owns TMEM lanes 32w..32w+31 = weight rows) and run the
// epilogue: FC1 rows 0-63 are gate rows and 64-127 the matching up rows, so
// the up half goes through shared memory and a = silu(g) * u is stored as
// fp16 (the FC2 B operand, gathered by sorted position); FC2 stores y per
// pair or adds w * y into the token's output.
// Every wait is bounded: a wait that gives up records an error word and the
// CTA runs on to its end without issuing more work.
#include <cudaTypedefs.h>

#include "ffn_common.cuh"

namespace moe {
namespace {

constexpr int UM_M = 128, UM_N = 128, UM_K = 64;
constexpr int STAGES = 4;
constexpr int DEC_WARPS = 4;                  // decoder + epilogue warps
constexpr int TMA_WARP = 4, MMA_WARP = 5;
constexpr int THREADS = 32 * 6;
constexpr int A_BYTES = UM_M * UM_K * 2;      // 16 KB
constexpr int B_BYTES = UM_N * UM_K * 2;      // 16 KB
constexpr int CB_COPIES = 16;
constexpr uint32_t TMEM_COLS = 128;
// instruction descriptor: D f32, A/B f16, both K-major, N = 128, M = 128
constexpr uint32_t IDESC = (1u << 4) | ((uint32_t)(UM_N >> 3) << 17) | ((uint32_t)(UM_M >> 4) << 24);

struct __align__(1024) Smem {
    uint8_t a[STAGES][A_BYTES];
    uint8_t b[STAGES][B_BYTES];
    float xch[64][UM_N + 1];      // FC1 epilogue: up half of the accumulator
    uint2 cbt[256 * CB_COPIES];   // sign-folded codebook, 16 copies
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
// byte offset of (row r, 8-byte column block j of the 64-element row) in a
// 128B-swizzled K-major tile
__device__ __forceinline__ uint32_t sw128_off(int r, int j) {
    return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((((j >> 1) ^ (r & 7))) << 4) + ((j & 1) << 3));
}

__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(IDESC), "r"(accumulate));
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
            "r"(dst),
        "l"(map), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// FC1 (FC1 = true): items = (chunk, 64-row tile of I); A rows 0-63 gate,
// 64-127 up.  FC2: items = (chunk, 128-row tile of H).
template <bool FC1>
__global__ void __launch_bounds__(THREADS, 1)
    ffn_umma_kernel(const __grid_constant__ CUtensorMap bmap, const SlotDesc* __restrict__ desc,
                    const uint16_t* __restrict__ codebook, const int32_t* __restrict__ sorted_pair,
                    const float* __restrict__ weights, int k, int H, int I, int* __restrict__ header,
                    const Chunk* __restrict__ uchunks, uint16_t* __restrict__ a16, float* __restrict__ out,
                    int mode) {
    extern __shared__ __align__(1024) uint8_t dyn[];
    // the swizzled operand tiles need 1024-byte alignment in the shared window
    Smem& S = *reinterpret_cast<Smem*>(dyn + ((1024u - (smem_u32(dyn) & 1023u)) & 1023u));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int* err = header + HDR_ERR;
    const int K = FC1 ? H : I;
    const int R = FC1 ? I : H;          // weight rows covered by the items of one chunk
    const int ROWS = FC1 ? 64 : 128;    // weight rows per item (FC1: 64 gate + 64 up)
    const int n_rt = R / ROWS;
    const int KB = K / 128;             // scale blocks per row
    const int n_kblk = K / UM_K;

    if ((smem_u32(&S.a[0][0]) & 1023) != 0) {
        if (tid == 0) atomicExch(err, MOE_DEVERR_SMEM_LAYOUT);
        return;
    }
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
        mbar_init(smem_u32(&S.acc_empty), 32 * DEC_WARPS);
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

    const int n_chunks = header[HDR_NUMMA];
    const int n_items = n_chunks * n_rt;
    auto failed = [&]() { return *reinterpret_cast<volatile int*>(&S.failed) != 0; };
    auto wait = [&](uint64_t* bar, uint32_t parity, int code) {
        if (failed()) return false;
        if (!mbar_wait_bounded(smem_u32(bar), parity, err, code)) {
            *reinterpret_cast<volatile int*>(&S.failed) = 1;
            return false;
        }
        return true;
    };

    if (warp < DEC_WARPS) {
        // ------------------------------------------------ decoder + epilogue
        const int rtile = tid >> 4, g = tid & 15;  // 16-row tile of the item, group of the K-block
        int it = 0, nitem = 0;
        for (int item = blockIdx.x; item < n_items; item += gridDim.x, ++nitem) {
            const Chunk ch = uchunks[item / n_rt];
            const int rt = item % n_rt;
            const SlotDesc& d = desc[ch.expert];
            int m, rtm;
            if (FC1) {
                m = rtile >> 2;                 // 0 gate, 1 up
                rtm = rt * 4 + (rtile & 3);
            } else {
                m = 2;
                rtm = rt * 8 + rtile;
            }
            const uint8_t* codes = static_cast<const uint8_t*>(d.codes[m]) + (size_t)rtm * KB * 512;
            const uint16_t* scales = static_cast<const uint16_t*>(d.scales[m]) + (size_t)rtm * KB * 16;
            const int rbase = FC1 ? (rtile >> 2) * 64 + (rtile & 3) * 16 : rtile * 16;
            for (int kb64 = 0; kb64 < n_kblk; ++kb64, ++it) {
                const int stage = it % STAGES, use = it / STAGES;
                const int kb = kb64 >> 1, half = kb64 & 1;
                // fetch this thread's chunk (16 rows x 1 group) and its 16 row scales
                const uint4 cw = ldg_stream(codes + (size_t)kb * 512 + 16 * (16 * half + g));
                const uint4 s0 = ldg_stream(scales + (size_t)kb * 16);
                const uint4 s1 = ldg_stream(scales + (size_t)kb * 16 + 8);
                if (use > 0 && !wait(&S.empty[stage], (use - 1) & 1, MOE_DEVERR_WAIT_EMPTY)) continue;
                const uint32_t sw[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
                const uint32_t cws[4] = {cw.x, cw.y, cw.z, cw.w};
                const uint32_t abase = smem_u32(&S.a[stage][0]);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int c = (cws[j >> 2] >> (8 * (j & 3))) & 0xff;
                    const int row = (j >> 1) + 8 * (j & 1);  // byte 2i+h holds row i + 8h
                    const uint32_t sh = (sw[row >> 1] >> (16 * (row & 1))) & 0xffffu;
                    const __half2 s2 = __halves2half2(__ushort_as_half((unsigned short)sh),
                                                      __ushort_as_half((unsigned short)sh));
                    const uint2 e = S.cbt[c * CB_COPIES + (lane & 15)];
                    __half2 w0 = __hmul2(*reinterpret_cast<const __half2*>(&e.x), s2);
                    __half2 w1 = __hmul2(*reinterpret_cast<const __half2*>(&e.y), s2);
                    const uint32_t off = sw128_off(rbase + row, g);
                    asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(abase + off),
                                 "r"(*reinterpret_cast<uint32_t*>(&w0)), "r"(*reinterpret_cast<uint32_t*>(&w1)));
                }
                fence_async_smem();
                mbar_arrive(smem_u32(&S.full[stage]));
            }
            // epilogue: accumulator rows 32*warp + lane, token columns 0..127
            if (!wait(&S.acc_full, nitem & 1, MOE_DEVERR_WAIT_FULL)) {
                mbar_arrive(smem_u32(&S.acc_empty));
                continue;
            }
            tc_fence_after();
            const int row = warp * 32 + lane;
            const uint32_t taddr = tmem + ((uint32_t)(warp * 32) << 16);
            if (FC1) {
                if (warp >= 2) {  // up rows: hand them to the gate-row threads
#pragma unroll 1
                    for (int c0 = 0; c0 < UM_N; c0 += 32) {
                        float v[32];
                        tmem_ld32(taddr + c0, v);
#pragma unroll
                        for (int i = 0; i < 32; ++i) S.xch[row - 64][c0 + i] = v[i];
                    }
                }
                named_barrier(1, 32 * DEC_WARPS);
                if (warp < 2) {
                    const int irow = rt * 64 + row;
#pragma unroll 1
                    for (int c0 = 0; c0 < UM_N; c0 += 32) {
                        float v[32];
                        tmem_ld32(taddr + c0, v);
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const int tok = c0 + i;
                            if (tok < ch.count) {
                                const float gv = v[i], uv = S.xch[row][tok];
                                const float a = gv / (1.0f + expf(-gv)) * uv;
                                a16[(size_t)(ch.start + tok) * I + irow] = __half_as_ushort(__float2half_rn(a));
                            }
                        }
                    }
                }
                named_barrier(1, 32 * DEC_WARPS);
            } else {
                const int h = rt * 128 + row;
#pragma unroll 1
                for (int c0 = 0; c0 < UM_N; c0 += 32) {
                    float v[32];
                    tmem_ld32(taddr + c0, v);
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int tok = c0 + i;
                        if (tok < ch.count) {
                            const int spos = ch.start + tok;
                            if (mode == MOE_PER_PAIR) {
                                out[(size_t)spos * H + h] = v[i];
                            } else {
                                const int p = sorted_pair[spos];
                                atomicAdd(out + (size_t)(p / k) * H + h, weights[p] * v[i]);
                            }
                        }
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(smem_u32(&S.acc_empty));
        }
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
    } else {
        // ------------------------------------------------ MMA issue
        if (lane == 0) {
            int it = 0, nitem = 0;
            for (int item = blockIdx.x; item < n_items; item += gridDim.x, ++nitem) {
                // the epilogue of the previous item must have read the accumulator
                if (nitem > 0 && !wait(&S.acc_empty, (nitem - 1) & 1, MOE_DEVERR_WAIT_EMPTY)) break;
                tc_fence_after();
                for (int kb64 = 0; kb64 < n_kblk; ++kb64, ++it) {
                    const int stage = it % STAGES, use = it / STAGES;
                    if (!wait(&S.full[stage], use & 1, MOE_DEVERR_WAIT_FULL)) break;
                    tc_fence_after();
                    const uint64_t ad = sw128_desc(smem_u32(&S.a[stage][0]));
                    const uint64_t bd = sw128_desc(smem_u32(&S.b[stage][0]));
#pragma unroll
                    for (int j = 0; j < UM_K / 16; ++j)  // 32 bytes of K per step inside the swizzle row
                        umma_f16(tmem, ad + 2 * j, bd + 2 * j, (kb64 > 0 || j > 0) ? 1u : 0u);
                    umma_commit(smem_u32(&S.empty[stage]));
                }
                umma_commit(smem_u32(&S.acc_full));
            }
            // the last epilogue must finish reading before the columns are freed
            if (nitem > 0) wait(&S.acc_empty, (nitem - 1) & 1, MOE_DEVERR_WAIT_EMPTY);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == MMA_WARP) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
    }
    pdl_launch_dependents();
}

// x16s[s, :] = fp16(x[token of sorted position s, :]) for the tensor-core B operand
__global__ void __launch_bounds__(256) gather_f16_kernel(const uint16_t* __restrict__ x,
                                                         const int32_t* __restrict__ sorted_pair, int k, int H,
                                                         int P, uint16_t* __restrict__ x16s) {
    pdl_wait();
    const long long n = (long long)P * (H / 8);
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
        const int s = (int)(i / (H / 8)), c = (int)(i % (H / 8));
        const int t = sorted_pair[s] / k;
        const uint4 v = *reinterpret_cast<const uint4*>(x + (size_t)t * H + 8 * c);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const __half2 h = __floats2half2_rn(__uint_as_float(w[q] << 16), __uint_as_float(w[q] & 0xffff0000u));
            o[q] = *reinterpret_cast<const uint32_t*>(&h);
        }
        *reinterpret_cast<uint4*>(x16s + (size_t)s * H + 8 * c) = make_uint4(o[0], o[1], o[2], o[3]);
    }
    pdl_launch_dependents();
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

// 2-D fp16 [rows, cols] row-major, box of 64 columns x 128 rows, 128B swizzle
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

size_t umma_smem_bytes() { return sizeof(Smem) + 1024; }

moe_status launch_gather_f16(const uint16_t* x, const int32_t* sorted_pair, int k, int H, int P, uint16_t* x16s,
                             cudaStream_t s) {
    long long n = (long long)P * (H / 8);
    long long blocks = (n + 255) / 256, cap = (long long)num_sms() * 8;
    cudaError_t e = launch_pdl(gather_f16_kernel, dim3((unsigned)(blocks < cap ? blocks : cap)), dim3(256), 0, s, x,
                               sorted_pair, k, H, P, x16s);
    if (e != cudaSuccess) return cuda_status(e, "moe_vq2_expert_ffn: gather launch");
    return MOE_OK;
}

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
                   t->codebook, sorted_pair, weights, k, H, I, header, uchunks, a16, out, mode);
    if (e != cudaSuccess) return cuda_status(e, "moe_vq2_expert_ffn: tensor-core launch");
    return MOE_OK;
}

}  // namespace moe
