// Token -> expert permutation: histogram, exclusive scan, stable scatter.
#include "permute.cuh"

namespace moe {
namespace {

constexpr int PT = 1024;  // threads of the single CTA

// One CTA.  Shared memory: cursor[E] then wcnt[32][E] (per-warp counts of a
// 1024-pair chunk).  Pairs are scattered chunk by chunk in increasing p;
// inside a chunk a pair's rank among the pairs of its expert is the count
// in lower warps plus the count in lower lanes of its own warp, so equal
// ids keep their pair order (a stable counting sort).
__global__ void __launch_bounds__(PT) permute_kernel(const int32_t* __restrict__ ids, int P, int E,
                                                     int32_t* __restrict__ offsets,
                                                     int32_t* __restrict__ sorted_pair,
                                                     int32_t* __restrict__ pair_to_sorted) {
    extern __shared__ int32_t sm[];
    int32_t* cursor = sm;
    int32_t* wcnt = sm + E;
    __shared__ int32_t warp_tot[32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_wait();
    pdl_launch_dependents();  // dependents may start their prologues now
    for (int i = tid; i < E * 33; i += PT) sm[i] = 0;
    __syncthreads();
    for (int p = tid; p < P; p += PT) atomicAdd(&cursor[ids[p]], 1);
    __syncthreads();
    // exclusive scan of cursor[0..E): thread e owns one entry (E <= 1024)
    int v = tid < E ? cursor[tid] : 0;
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int wv = warp_tot[lane];
        int wi = wv;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            int o = __shfl_up_sync(0xffffffffu, wi, off);
            if (lane >= off) wi += o;
        }
        warp_tot[lane] = wi - wv;
    }
    __syncthreads();
    int excl = incl - v + warp_tot[warp];
    if (tid < E) {
        offsets[tid] = excl;
        cursor[tid] = excl;
    }
    if (tid == 0) offsets[E] = P;
    __syncthreads();
    const unsigned lt = (1u << lane) - 1u;
    for (int base = 0; base < P; base += PT) {
        const int p = base + tid;
        const bool valid = p < P;
        const int e = valid ? ids[p] : -1;
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        const int rank = __popc(peers & lt);
        const bool leader = (__ffs(peers) - 1) == lane;
        if (valid && leader) wcnt[warp * E + e] = __popc(peers);
        __syncthreads();
        if (valid) {
            int pre = 0;
            for (int w2 = 0; w2 < warp; ++w2) pre += wcnt[w2 * E + e];
            const int pos = cursor[e] + pre + rank;
            sorted_pair[pos] = p;
            pair_to_sorted[p] = pos;
        }
        __syncthreads();
        if (valid && leader) {
            atomicAdd(&cursor[e], __popc(peers));
            wcnt[warp * E + e] = 0;
        }
        __syncthreads();
    }
}

// Large calls (P >= PERMUTE_MULTI_P, with a workspace): the same stable
// counting sort over chunks of PT pairs, one CTA each, in three launches:
// each chunk's histogram; per expert the totals, their exclusive scan over
// the experts (the offsets) and each chunk's base position; each chunk's
// scatter, a pair's rank inside its chunk counted as in permute_kernel.  The
// sorted order (expert, then pair index) and so every output is the same.
__global__ void __launch_bounds__(PT) permute_count_kernel(const int32_t* __restrict__ ids, int P, int E,
                                                           int32_t* __restrict__ chunk_cnt) {
    extern __shared__ int32_t sm[];
    const int tid = threadIdx.x;
    pdl_wait();
    pdl_launch_dependents();
    for (int i = tid; i < E; i += PT) sm[i] = 0;
    __syncthreads();
    const int p = blockIdx.x * PT + tid;
    if (p < P) atomicAdd(&sm[ids[p]], 1);
    __syncthreads();
    for (int i = tid; i < E; i += PT) chunk_cnt[(size_t)blockIdx.x * E + i] = sm[i];
}

__global__ void __launch_bounds__(PT) permute_scan_kernel(const int32_t* __restrict__ chunk_cnt, int nch, int P,
                                                          int E, int32_t* __restrict__ offsets,
                                                          int32_t* __restrict__ chunk_base) {
    __shared__ int32_t warp_tot[32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_wait();
    pdl_launch_dependents();
    int v = 0;
    if (tid < E)
        for (int c = 0; c < nch; ++c) v += chunk_cnt[(size_t)c * E + tid];
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int wv = warp_tot[lane];
        int wi = wv;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            int o = __shfl_up_sync(0xffffffffu, wi, off);
            if (lane >= off) wi += o;
        }
        warp_tot[lane] = wi - wv;
    }
    __syncthreads();
    if (tid < E) {
        int run = incl - v + warp_tot[warp];
        offsets[tid] = run;
        for (int c = 0; c < nch; ++c) {
            chunk_base[(size_t)c * E + tid] = run;
            run += chunk_cnt[(size_t)c * E + tid];
        }
    }
    if (tid == 0) offsets[E] = P;
}

__global__ void __launch_bounds__(PT) permute_scatter_kernel(const int32_t* __restrict__ ids, int P, int E,
                                                             const int32_t* __restrict__ chunk_base,
                                                             int32_t* __restrict__ sorted_pair,
                                                             int32_t* __restrict__ pair_to_sorted) {
    extern __shared__ int32_t wcnt[];  // [32][E]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_wait();
    pdl_launch_dependents();
    for (int i = tid; i < 32 * E; i += PT) wcnt[i] = 0;
    __syncthreads();
    const int p = blockIdx.x * PT + tid;
    const bool valid = p < P;
    const int e = valid ? ids[p] : -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    const bool leader = (__ffs(peers) - 1) == lane;
    if (valid && leader) wcnt[warp * E + e] = __popc(peers);
    __syncthreads();
    if (valid) {
        int pre = 0;
        for (int w2 = 0; w2 < warp; ++w2) pre += wcnt[w2 * E + e];
        const int pos = chunk_base[(size_t)blockIdx.x * E + e] + pre + rank;
        sorted_pair[pos] = p;
        pair_to_sorted[p] = pos;
    }
}

}  // namespace

size_t permute_ws_bytes(int P, int E) {
    if (P < PERMUTE_MULTI_P) return 0;
    const size_t nch = ((size_t)P + PT - 1) / PT;
    return 2 * sizeof(int32_t) * nch * (size_t)E;
}

moe_status launch_permute(const int32_t* ids, int P, int E, int32_t* offsets, int32_t* sorted_pair,
                          int32_t* pair_to_sorted, cudaStream_t s) {
    return launch_permute_ws(ids, P, E, offsets, sorted_pair, pair_to_sorted, s, nullptr, 0);
}

moe_status launch_permute_ws(const int32_t* ids, int P, int E, int32_t* offsets, int32_t* sorted_pair,
                             int32_t* pair_to_sorted, cudaStream_t s, void* ws, size_t ws_bytes) {
    if (P >= PERMUTE_MULTI_P && ws && ws_bytes >= permute_ws_bytes(P, E)) {
        const int nch = (P + PT - 1) / PT;
        int32_t* chunk_cnt = static_cast<int32_t*>(ws);
        int32_t* chunk_base = chunk_cnt + (size_t)nch * E;
        const size_t ssm = sizeof(int32_t) * (size_t)E * 32;
        if (ssm > 48 * 1024) {
            cudaError_t ea = ensure_smem_attr(permute_scatter_kernel, (int)ssm);
            if (ea != cudaSuccess) return cuda_status(ea, "moe_permute: shared memory attribute");
        }
        cudaError_t e = launch_pdl(permute_count_kernel, dim3((unsigned)nch), dim3(PT), sizeof(int32_t) * (size_t)E,
                                   s, ids, P, E, chunk_cnt);
        if (e == cudaSuccess)
            e = launch_pdl(permute_scan_kernel, dim3(1), dim3(PT), 0, s, (const int32_t*)chunk_cnt, nch, P, E, offsets,
                           chunk_base);
        if (e == cudaSuccess)
            e = launch_pdl(permute_scatter_kernel, dim3((unsigned)nch), dim3(PT), ssm, s, ids, P, E,
                           (const int32_t*)chunk_base, sorted_pair, pair_to_sorted);
        if (e != cudaSuccess) return cuda_status(e, "moe_permute: launch");
        MOE_LAUNCH_CHECK("moe_permute: launch");
        return MOE_OK;
    }
    size_t smem = sizeof(int32_t) * (size_t)E * 33;
    if (smem > 48 * 1024) {
        cudaError_t ea = ensure_smem_attr(permute_kernel, (int)smem);
        if (ea != cudaSuccess) return cuda_status(ea, "moe_permute: shared memory attribute");
    }
    cudaError_t e = launch_pdl(permute_kernel, dim3(1), dim3(PT), smem, s, ids, P, E, offsets, sorted_pair,
                               pair_to_sorted);
    if (e != cudaSuccess) return cuda_status(e, "moe_permute: launch");
    MOE_LAUNCH_CHECK("moe_permute: launch");
    return MOE_OK;
}

}  // namespace moe
