// moe_vq2_expert_ffn_noalloc: the expert FFN for callers that must not
// allocate device memory (see the declaration in moe_vq2.h).  Its scratch is
// one file-scope device array, reserved when the library's device code is
// loaded on a device (under lazy loading: at the first call here) and held
// until the process exits; no call here allocates or frees device memory.
#include <mutex>

#include "common.cuh"

namespace {

constexpr size_t kScratchBytes = MOE_NOALLOC_SCRATCH_BYTES;

// The scratch every call of moe_vq2_expert_ffn_noalloc uses.  In host code
// this name is only a stand-in for the device symbol: its device address is
// taken with cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_ffn_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_ffn_scratch on the current device, looked up once per
// device (the first call on a device does it, with that device current).
moe_status scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return moe::cuda_status(e, "moe_vq2_expert_ffn_noalloc: cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) {
        moe::set_error("moe_vq2_expert_ffn_noalloc: device %d above the supported %d", dev, kMaxDevices);
        return MOE_ERR_UNSUPPORTED;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_ffn_scratch);
        if (e != cudaSuccess)
            return moe::cuda_status(e, "moe_vq2_expert_ffn_noalloc: cudaGetSymbolAddress (loading the library's "
                                       "device code reserves its 64 MiB scratch; an out-of-memory here means the "
                                       "device had no room left for it)");
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return MOE_OK;
}

}  // namespace

using namespace moe;

extern "C" {

moe_status moe_vq2_expert_ffn_noalloc(const moe_slot_table* table, const uint16_t* x,
                                      const int32_t* expert_offsets, const int32_t* sorted_pair,
                                      const float* weights, int T, int k, int mode, float* out_or_ypair,
                                      uint8_t* pair_status, cudaStream_t stream) {
    MOE_CHECK_ARG(table, "moe_vq2_expert_ffn_noalloc: null table");
    MOE_CHECK_ARG(T >= 0 && k >= 1, "moe_vq2_expert_ffn_noalloc: T=%d k=%d", T, k);
    MOE_CHECK_ARG(mode == MOE_FUSED_SCATTER || mode == MOE_PER_PAIR,
                  "moe_vq2_expert_ffn_noalloc: bad mode %d", mode);
    long long P = (long long)T * k;
    MOE_CHECK_SUPPORTED(P <= (1 << 24), "moe_vq2_expert_ffn_noalloc: T*k=%lld above 2^24", P);
    if (P == 0) return MOE_OK;
    MOE_CHECK_ARG(x && expert_offsets && sorted_pair && weights && out_or_ypair && pair_status,
                  "moe_vq2_expert_ffn_noalloc: null pointer");
    MOE_CHECK_SUPPORTED(aligned16(x) && aligned16(out_or_ypair),
                        "moe_vq2_expert_ffn_noalloc: x and out must be 16-byte aligned");
    const size_t need = ffn_workspace_size(T, k, table->h.E, table->h.H, table->h.I);
    if (need > kScratchBytes) {
        set_error("moe_vq2_expert_ffn_noalloc: T=%d k=%d E=%d H=%d I=%d needs %zu bytes of scratch, above "
                  "the fixed %zu (use moe_vq2_expert_ffn with a caller workspace)",
                  T, k, table->h.E, table->h.H, table->h.I, need, kScratchBytes);
        return MOE_ERR_UNSUPPORTED;
    }
    void* scratch = nullptr;
    moe_status st = scratch_address(&scratch);
    if (st != MOE_OK) return st;
    return launch_expert_ffn(&table->h, x, expert_offsets, sorted_pair, weights, T, k, mode, out_or_ypair,
                             pair_status, scratch, kScratchBytes, stream);
}

}  // extern "C"
