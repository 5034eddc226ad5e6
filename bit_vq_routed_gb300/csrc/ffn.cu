// Expert FFN over the slot table: the schedule and the launch sequence.
//
// The schedule kernel sorts each resident expert of the call to one path by
// its token count m_e:
//   - VQ2, m_e == 1: the activation-table kernels (ffn_lut.cu);
//   - VQ2, m_e >= 32: the tcgen05 kernels (ffn_umma.cu);
//   - otherwise: the mma.sync kernels (ffn_mma.cu), chunks of <= 32 tokens.
#include "ffn_common.cuh"

namespace moe {
namespace {

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
                                                        int32_t* __restrict__ grp_start, int use_lut,
                                                        Chunk* __restrict__ uchunks, int use_umma) {
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
    const bool um = res && use_umma && m >= UMMA_MIN && s_fmt[tid] == MOE_FMT_VQ2;
    const int n = (res && !lut && !um) ? (m + MMA_NT - 1) / MMA_NT : 0;
    const int nu = um ? (m + UMMA_NT - 1) / UMMA_NT : 0;
    const int tok = lut ? sorted_pair[s_off[tid]] / k : 0x7fffffff;
    s_tok[tid] = tok;
    int n_chunks, n_lut;
    const int cbase = block_exclusive_scan(n, warp_tot, &n_chunks);
    for (int c = 0; c < n; ++c) {
        Chunk ch;
        ch.expert = tid;
        ch.start = s_off[tid] + c * MMA_NT;
        ch.count = min(MMA_NT, m - c * MMA_NT);
        ch.fmt = s_fmt[tid];
        chunks[cbase + c] = ch;
    }
    int n_umma;
    const int ubase = block_exclusive_scan(nu, warp_tot, &n_umma);
    for (int c = 0; c < nu; ++c) {
        Chunk ch;
        ch.expert = tid;
        ch.start = s_off[tid] + c * UMMA_NT;
        ch.count = min(UMMA_NT, m - c * UMMA_NT);
        ch.fmt = s_fmt[tid];
        uchunks[ubase + c] = ch;
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
        header[HDR_NUMMA] = n_umma;
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
    Chunk* uchunks = reinterpret_cast<Chunk*>(w + L.uchunks_off);
    uint16_t* x16s = reinterpret_cast<uint16_t*>(w + L.x16s_off);
    const int use_lut = 1;
    const int use_umma = T >= UMMA_MIN ? 1 : 0;  // an expert gets at most T of the pairs
    // With one token no expert gets two pairs, so the mma.sync kernels only
    // have work if the table holds FP4 experts.
    const bool mma = T > 1 || t->n_fp4 > 0 || !use_lut;

    cudaError_t e = launch_pdl(schedule_kernel, dim3(1), dim3(1024), 0, s, (const SlotDesc*)t->d_desc, E, offsets,
                               sorted_pair, P, k, status, header, chunks, lut_s, lut_e, lut_grp, grp_start, use_lut,
                               uchunks, use_umma);
    if (e != cudaSuccess) return cuda_status(e, "moe_vq2_expert_ffn: schedule launch");
    moe_status st;
    if ((mma || use_umma) && (st = launch_gather_f16(x, sorted_pair, k, H, P, x16s, s)) != MOE_OK) return st;
    if (use_lut && (st = launch_lut_fc(true, t, x, sorted_pair, k, w, L, s)) != MOE_OK) return st;
    if (mma && (st = launch_mma_fc(true, t, sorted_pair, weights, k, mode, out, w, L, s)) != MOE_OK) return st;
    if (use_umma && (st = launch_umma(true, t, sorted_pair, weights, k, P, mode, out, w, L, s)) != MOE_OK) return st;
    if (use_lut && (st = launch_lut_fc(false, t, x, sorted_pair, k, w, L, s)) != MOE_OK) return st;
    if (mma && (st = launch_mma_fc(false, t, sorted_pair, weights, k, mode, out, w, L, s)) != MOE_OK) return st;
    if (use_umma && (st = launch_umma(false, t, sorted_pair, weights, k, P, mode, out, w, L, s)) != MOE_OK) return st;
    if (use_lut && (st = launch_lut_finish(t, sorted_pair, weights, k, mode, out, w, L, L.max_lut, s)) != MOE_OK)
        return st;
    return MOE_OK;
}

}  // namespace moe
