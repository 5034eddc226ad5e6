// Shared definitions of the CUDA library: status plumbing, the device-side
// slot descriptor, the packed weight layouts and small PTX wrappers.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <mutex>
#include <stdint.h>
#include <stddef.h>

#include "moe_vq2.h"

namespace moe {

// ---------------------------------------------------------------- errors
void set_error(const char* fmt, ...);
moe_status cuda_status(cudaError_t e, const char* what);

#define MOE_CHECK_ARG(cond, ...)                         \
    do {                                                 \
        if (!(cond)) {                                   \
            ::moe::set_error(__VA_ARGS__);               \
            return MOE_ERR_INVALID_ARG;                  \
        }                                                \
    } while (0)

#define MOE_CHECK_SUPPORTED(cond, ...)                   \
    do {                                                 \
        if (!(cond)) {                                   \
            ::moe::set_error(__VA_ARGS__);               \
            return MOE_ERR_UNSUPPORTED;                  \
        }                                                \
    } while (0)

#define MOE_LAUNCH_CHECK(what)                                       \
    do {                                                             \
        cudaError_t e_ = cudaGetLastError();                         \
        if (e_ != cudaSuccess) return ::moe::cuda_status(e_, what);  \
    } while (0)

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// ---------------------------------------------------------------- slot table
// One entry of the device descriptor array (64 bytes).
struct SlotDesc {
    int32_t format;    // MOE_FMT_VQ2 / MOE_FMT_FP4
    int32_t resident;  // 0 = not resident
    const void* codes[3];
    const void* scales[3];
};
static_assert(sizeof(SlotDesc) == 56, "slot descriptor layout");

struct SlotTableHost {
    int E, H, I;
    const uint16_t* codebook;  // device fp16 [128*4]
    SlotDesc* d_desc;          // device [E]
    uint8_t* h_fmt;            // host mirror: 0 = empty, 1 + format of each entry
    int n_fp4;                 // FP4 entries currently set
};

// ---------------------------------------------------------------- layouts
// Packed VQ2: tile (rt, kb) = 16 rows x 32 groups = 512 bytes.
__host__ __device__ inline size_t vq2_tile_offset(int rt, int kb, int KB) {
    return ((size_t)rt * KB + kb) * 512;
}
// byte inside a tile of (row-in-tile r16, group-in-block g)
__host__ __device__ inline int vq2_in_tile(int r16, int g) {
    return 16 * g + 2 * (r16 & 7) + (r16 >> 3);
}
// Packed FP4: tile (rt, kt) = 16 rows x 64 elements = 512 bytes.
// byte inside a tile holding logical byte lb (0..31 within the 64-element
// block) of row-in-tile r16
__host__ __device__ inline int fp4_in_tile(int r16, int lb) {
    int i = r16 & 7, hi = r16 >> 3;
    int s = lb >> 3, w = lb & 7, j = w & 3, up = w >> 2;
    return 16 * (4 * i + j) + 4 * s + 2 * hi + up;
}

// ---------------------------------------------------------------- PTX
// (not volatile: a pure function of its registers, free to be scheduled
// around the loads that feed it)
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Four e2m1 pairs (one per byte of w) -> four f16x2 (low nibble -> low half).
__device__ __forceinline__ void e2m1x8_to_f16x8(uint32_t w, uint32_t& r0, uint32_t& r1,
                                                uint32_t& r2, uint32_t& r3) {
    asm("{\n"
        " .reg .b8 b0, b1, b2, b3;\n"
        " mov.b32 {b0, b1, b2, b3}, %4;\n"
        " cvt.rn.f16x2.e2m1x2 %0, b0;\n"
        " cvt.rn.f16x2.e2m1x2 %1, b1;\n"
        " cvt.rn.f16x2.e2m1x2 %2, b2;\n"
        " cvt.rn.f16x2.e2m1x2 %3, b3;\n"
        "}\n"
        : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
        : "r"(w));
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b) { return __uint_as_float(b << 16); }

// ue8m0 exponent byte -> 2^(E-127) as fp32 (E = 0 gives the subnormal 2^-127,
// whose bit pattern 0x400000 lies below every E << 23 with E >= 1)
__device__ __forceinline__ float e8m0_to_float(uint32_t e) { return __uint_as_float(max(e << 23, 0x00400000u)); }

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- mbarrier / bulk copy
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait: gives up after max_iter polls, records code in *err and
// returns false (callers then skip their work so every loop still ends).
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, int* err, int code) {
#pragma unroll 1
    for (uint32_t it = 0; it < (1u << 20); ++it)
        if (mbar_try_wait(bar, parity)) return true;
    if (err) atomicExch(err, code);
    return false;
}
// try_wait that may suspend the thread for up to hint_ns nanoseconds while
// the phase is incomplete (it returns as soon as the phase completes), so a
// waiting warp issues a few instructions instead of a spin.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}
// Bounded suspending wait: at most 2^18 tries of up to 1 us each; on
// timeout records code in *err and returns false.
__device__ __forceinline__ bool mbar_wait_sleep_bounded(uint32_t bar, uint32_t parity, int* err, int code) {
#pragma unroll 1
    for (uint32_t it = 0; it < (1u << 18); ++it)
        if (mbar_try_wait_sleep(bar, parity, 1000u)) return true;
    if (err) atomicExch(err, code);
    return false;
}
// 1-D bulk copy global -> shared, completing on an mbarrier (16-byte
// aligned addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}
__device__ __forceinline__ float lds_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ uint4 lds_u128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}
__device__ __forceinline__ void sts_f32(uint32_t addr, float v) {
    asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(v));
}
// 16-byte global load that bypasses L1 allocation (streamed once)
__device__ __forceinline__ uint4 ldg_stream(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
__device__ __forceinline__ void named_barrier(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Error codes recorded in the workspace header's error word.
#define MOE_DEVERR_WAIT_FULL 1
#define MOE_DEVERR_WAIT_EMPTY 2
#define MOE_DEVERR_SMEM_LAYOUT 3

// Launch with programmatic dependent launch allowed: the kernel may start
// while its predecessor on the stream still runs.  Every kernel of the library
// calls pdl_wait() before it touches memory an earlier kernel may write or
// read, and pdl_launch_dependents() right after it -- except a kernel that
// writes a bf16 activation output (the combine's out_bf16), which lets its
// dependents start only when it has finished, and the e2m1 table kernels,
// which touch only what is complete two launches back (or their own
// results) and call pdl_wait() just before they exit.  So when a kernel starts, its
// predecessor has at least passed its own wait, i.e. everything two launches
// back is complete, and so are the bf16 activations the caller passes in (x):
// no library kernel that may still be running writes them.  The slot-table
// writer is launched without programmatic dependent launch, so no later
// kernel starts before it has finished.  The code before the wait
// (shared-memory set-up, constant weights, the slot descriptors, x, and reads
// of results two launches back) overlaps the predecessor's run.
//
// Host-side count of kernel launches the library has issued (a launch made
// inside a stream capture counts once: it becomes one graph node).
void count_launch();

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    count_launch();
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// Sets a kernel's dynamic shared-memory limit once per (kernel, device), so
// later calls (for instance inside a CUDA-graph capture) make no attribute
// call at all.
template <typename F>
inline cudaError_t ensure_smem_attr(F* kern, int bytes) {
    constexpr int kMaxDev = 64;
    struct Entry {
        const void* fn;
        int bytes[kMaxDev];
    };
    static Entry table[16];
    static int n_entries = 0;
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDev) return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    Entry* ent = nullptr;
    for (int i = 0; i < n_entries; ++i)
        if (table[i].fn == (const void*)kern) ent = &table[i];
    if (!ent && n_entries < 16) {
        ent = &table[n_entries++];
        ent->fn = (const void*)kern;
        for (int d = 0; d < kMaxDev; ++d) ent->bytes[d] = 0;
    }
    if (ent && ent->bytes[dev] >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && ent) ent->bytes[dev] = bytes;
    return e;
}

// ---------------------------------------------------------------- launchers
int num_sms();

moe_status launch_router_logits(const uint16_t* x, const uint16_t* w, const float* bias, float* logits,
                                int T, int H, int E, cudaStream_t s);
moe_status launch_route_topk(const float* logits, int T, int E, int k, int renorm, int32_t* ids,
                             float* weights, cudaStream_t s);
// One token: the routing over a thread-block cluster (router.cu).
bool route_cluster_ok(int T, int H, int E);
moe_status launch_route_cluster(const uint16_t* x, const uint16_t* w, const float* bias, int H, int E, int k,
                                int renorm, float* logits, int32_t* ids, float* weights, int32_t* offsets,
                                int32_t* sorted_pair, int32_t* pair_to_sorted, cudaStream_t s);
bool route_fused_ok(int T, int k, int H, int E);
moe_status launch_route_fused(const uint16_t* x, const uint16_t* w, const float* bias, int T, int H, int E, int k,
                              int renorm, float* logits, int32_t* ids, float* weights, int32_t* offsets,
                              int32_t* sorted_pair, int32_t* pair_to_sorted, int* counter, cudaStream_t s);
moe_status launch_permute(const int32_t* ids, int P, int E, int32_t* offsets, int32_t* sorted_pair,
                          int32_t* pair_to_sorted, cudaStream_t s);
moe_status launch_vq2_pack(const uint8_t* codes, const uint16_t* scales, int rows, int K,
                           uint8_t* pc, uint16_t* ps, cudaStream_t s);
moe_status launch_fp4_pack(const uint8_t* codes, const uint8_t* scales, int rows, int K, uint8_t* pc,
                           uint8_t* ps, cudaStream_t s);
moe_status launch_slot_set(SlotDesc* table, int expert_id, SlotDesc d, cudaStream_t s);
size_t ffn_workspace_size(int T, int k, int E, int H, int I);
// With comb32 / comb16 (mode MOE_PER_PAIR): then the combine of the pairs into
// them, as moe_combine does (inside the table kernels for single-token calls).
moe_status launch_expert_ffn(const SlotTableHost* t, const uint16_t* x, const int32_t* offsets,
                             const int32_t* sorted_pair, const float* weights, int T, int k, int mode,
                             float* out, uint8_t* status, void* ws, size_t ws_bytes, cudaStream_t s,
                             const int32_t* pair_to_sorted = nullptr, float* comb32 = nullptr,
                             uint16_t* comb16 = nullptr);
moe_status launch_accumulate(float* dst, const float* src, size_t n, cudaStream_t s);
moe_status launch_gate(const SlotDesc* desc, const int32_t* ids, const float* weights, int P, int E, float tau,
                       int32_t* gated, cudaStream_t s);
moe_status launch_combine(const float* ypair, const int32_t* p2s, const float* w, const uint8_t* st,
                          int T, int k, int H, float* out32, uint16_t* out16, cudaStream_t s);

}  // namespace moe

// The opaque handle of include/moe_vq2.h.
struct moe_slot_table {
    moe::SlotTableHost h;
};
