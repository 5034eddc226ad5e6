// Expert FFN over the slot table: the schedule and the launch sequence.
//
// The schedule kernel sorts each resident expert of the call to one path by
// its token count m_e:
//   - VQ2, m_e <= LUT_MAX_M: the activation-table kernels (ffn_lut.cu), one
//     table pair per token;
//   - FP4 in calls of at most LUT4_MAX_T tokens: the e2m1 activation-table
//     kernels (ffn_lut.cu), one table pair per token;
//   - VQ2, m_e >= 32: the tcgen05 kernels (ffn_umma.cu);
//   - otherwise: the mma.sync kernels (ffn_mma.cu), chunks of <= 32 (VQ2) or
//     <= 16 (FP4) tokens.
#include "ffn_common.cuh"

namespace moe {
namespace {

// ---------------------------------------------------------------- schedule
// Scan of a 64-bit value over the 1024 threads of the block (up to three
// counts packed in 21-bit fields); returns this thread's exclusive prefix and
// the block total through *total.
__device__ unsigned long long block_scan64(unsigned long long v, unsigned long long* warp_tot,
                                           unsigned long long* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned long long incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const unsigned long long o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
    }
    __syncthreads();  // an earlier scan's readers are done with warp_tot
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const unsigned long long wv = warp_tot[lane];
        unsigned long long wi = wv;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const unsigned long long o = __shfl_up_sync(0xffffffffu, wi, off);
            if (lane >= off) wi += o;
        }
        warp_tot[lane] = wi - wv;
        if (lane == 31) warp_tot[32] = wi;
    }
    __syncthreads();
    *total = warp_tot[32];
    return incl - v + warp_tot[warp];
}

constexpr int SP_SMEM = 4096;  // sorted_pair entries staged in shared memory
constexpr int MAX_TP = LUT_MAX_M * 1024;  // table pairs at most (E <= 1024)
constexpr size_t SCHED_SMEM = sizeof(int) * (1025 + (MAX_TP + 1) + 4 * MAX_TP + SP_SMEM) + 1024;

// One CTA of 1024 threads.  Expert e with m_e pairs, if resident:
//   VQ2 with m_e <= lut_max_m (LUT_MAX_M, or LUT_MAX_M_LARGE in large calls)
//     -> m_e activation-table pairs
//     (one per token: the expert's codes are streamed once per token, which
//     costs less than the mma.sync decode at such counts);
//   FP4 (and use_lut4: calls of at most LUT4_MAX_T tokens) -> m_e e2m1 table
//     pairs, one per token (grouped by token, in expert order in a group);
//   VQ2 with m_e >= UMMA_MIN (and use_umma) -> ceil(m_e / UMMA_NT) tcgen05 chunks;
//   otherwise -> mma.sync chunks of MMA_NT_VQ2 (VQ2) or MMA_NT_FP4 (FP4,
//     and with split16 VQ2 experts of at most MMA_NT_FP4 tokens) tokens; the
//     chunks of the 32-token configuration are listed first (header
//     HDR_NVQ2 of them), then those of the 16-token one.
// Table pairs are listed sorted by (token, expert) and grouped by token, so
// the experts of one token share each activation table.  pair_status of every
// pair from the residency of its expert; the header's error word is cleared.
// All global inputs are read in one round trip at the start.
__global__ void __launch_bounds__(1024) schedule_kernel(const SlotDesc* __restrict__ desc, int E,
                                                        const int32_t* __restrict__ offsets,
                                                        const int32_t* __restrict__ sorted_pair, int P, int k,
                                                        uint8_t* __restrict__ status, int* __restrict__ header,
                                                        Chunk* __restrict__ chunks, LutRec* __restrict__ recs,
                                                        int32_t* __restrict__ grp_start, int lut_max_m,
                                                        Chunk* __restrict__ uchunks, int use_umma, int H, int I,
                                                        int C, int4* __restrict__ fc1_range, int split16,
                                                        LutRec* __restrict__ recs4, int use_lut4) {
    __shared__ unsigned long long warp_tot[33];
    extern __shared__ __align__(16) int sched_smem[];
    int* s_off = sched_smem;                       // [1025]
    int* s_gs = s_off + 1025;                      // [MAX_TP + 1] first table pair of each token group
    int* s_ptok = s_gs + MAX_TP + 1;               // [MAX_TP] token of each table pair (expert order)
    int* s_pe = s_ptok + MAX_TP;                   // [MAX_TP] expert of each table pair
    int* s_sorted_tok = s_pe + MAX_TP;             // [MAX_TP] token of each table pair, (token, expert) order
    int* s_rank = s_sorted_tok + MAX_TP;           // [MAX_TP] (token, expert) rank of each table pair
    int* s_sp = s_rank + MAX_TP;                   // [SP_SMEM]
    uint8_t* s_res = reinterpret_cast<uint8_t*>(s_sp + SP_SMEM);  // [1024]
    pdl_wait();
    pdl_launch_dependents();  // dependents may start their prologues now
    const int tid = threadIdx.x;
    // the one round trip: offsets, this thread's slot descriptor, sorted_pair
    for (int i = tid; i <= E; i += 1024) s_off[i] = offsets[i];
    SlotDesc d;
    d.format = 0;
    d.resident = 0;
    if (tid < E) d = desc[tid];
    const int nsp = min(P, SP_SMEM);
    for (int i = tid; i < nsp; i += 1024) s_sp[i] = sorted_pair[i];
    if (tid < E) s_res[tid] = (uint8_t)(d.resident != 0);
    __syncthreads();
    auto sp_at = [&](int i) { return i < SP_SMEM ? s_sp[i] : sorted_pair[i]; };

    const int m = tid < E ? s_off[tid + 1] - s_off[tid] : 0;
    const bool res = tid < E && d.resident != 0 && m > 0;
    const bool lut = res && m <= lut_max_m && d.format == MOE_FMT_VQ2;
    const int nl = lut ? m : 0;  // this expert's table pairs
    const bool um = res && use_umma && m >= UMMA_MIN && d.format == MOE_FMT_VQ2;
    const bool fp4 = d.format == MOE_FMT_FP4;
    const bool lut4 = res && use_lut4 && m <= LUT4_MAX_T && fp4;  // (m <= T <= LUT4_MAX_T)
    const bool part2 = fp4 || (split16 && m <= MMA_NT_FP4);  // the 16-token configuration
    const int nt_e = part2 ? MMA_NT_FP4 : MMA_NT_VQ2;  // tokens per mma.sync chunk of this expert
    const int n = (res && !lut && !um && !lut4) ? (m + nt_e - 1) / nt_e : 0;
    const int nu = um ? (m + UMMA_NT - 1) / UMMA_NT : 0;
    // one scan for the three counts (fields of 21 bits: n, nu, table pairs)
    unsigned long long tot;
    const unsigned long long ex =
        block_scan64((unsigned long long)(part2 ? 0 : n) | ((unsigned long long)nu << 21) | ((unsigned long long)nl << 42),
                     warp_tot, &tot);
    // the 16-token chunks, listed after the others
    unsigned long long tot4;
    const unsigned long long ex4 = block_scan64(part2 ? (unsigned long long)n : 0ull, warp_tot, &tot4);
    // the e2m1 table pairs, grouped by token (tokens 0..T-1, T <= 3): field t
    // (21 bits) counts the experts with a pair of token t
    static_assert(LUT4_MAX_T <= 3, "three 21-bit token fields");
    unsigned long long has4 = 0;
    if (lut4)
        for (int q = 0; q < m; ++q) has4 |= 1ull << (21 * (sp_at(s_off[tid] + q) / k));
    unsigned long long tot_t;
    const unsigned long long ex_t = block_scan64(has4, warp_tot, &tot_t);
    const int n_vq2 = (int)(tot & 0x1fffff);
    const int cbase = part2 ? n_vq2 + (int)(ex4 & 0x1fffff) : (int)(ex & 0x1fffff), ubase = (int)((ex >> 21) & 0x1fffff);
    const int n_chunks = n_vq2 + (int)tot4, n_umma = (int)((tot >> 21) & 0x1fffff), n_lut = (int)(tot >> 42);
    const int g40 = (int)(tot_t & 0x1fffff), g41 = (int)((tot_t >> 21) & 0x1fffff), g42 = (int)(tot_t >> 42);
    const int n_lut4 = g40 + g41 + g42;
    const int n_groups4 = (g40 > 0) + (g41 > 0) + (g42 > 0);
    if (lut4) {
        // the pair of token t: after the groups of tokens below t, in expert
        // order; a token's pairs form one group (they share each FC1 table)
        for (int q = 0; q < m; ++q) {
            const int sp = s_off[tid] + q, t = sp_at(sp) / k;
            const int gs = (t > 0 ? g40 : 0) + (t > 1 ? g41 : 0);
            LutRec r;
            for (int mtx = 0; mtx < 3; ++mtx) {
                r.codes[mtx] = d.codes[mtx];
                r.scales[mtx] = d.scales[mtx];
            }
            r.sorted = sp;
            r.token = t;
            r.gs = gs;
            r.gc = t == 0 ? g40 : t == 1 ? g41 : g42;
            recs4[gs + (int)((ex_t >> (21 * t)) & 0x1fffff)] = r;
        }
    }
    for (int c = 0; c < n; ++c) {
        Chunk ch;
        ch.expert = tid;
        ch.start = s_off[tid] + c * nt_e;
        ch.count = min(nt_e, m - c * nt_e);
        ch.fmt = d.format;
        chunks[cbase + c] = ch;
    }
    for (int c = 0; c < nu; ++c) {
        Chunk ch;
        ch.expert = tid;
        ch.start = s_off[tid] + c * UMMA_NT;
        ch.count = min(UMMA_NT, m - c * UMMA_NT);
        ch.fmt = d.format;
        uchunks[ubase + c] = ch;
    }
    // the table pairs of this expert (its tokens, in sorted order)
    const int lbase = (int)(ex >> 42);
    for (int q = 0; q < nl; ++q) {
        s_ptok[lbase + q] = sp_at(s_off[tid] + q) / k;
        s_pe[lbase + q] = tid;
    }
    __syncthreads();
    // rank of each table pair in (token, expert) order, one warp per pair:
    // the pairs with a smaller token, or the same token and a smaller expert
    // (an expert has at most one pair per token)
    {
        const int warp = tid >> 5, lane = tid & 31;
        for (int i = warp; i < n_lut; i += 32) {
            const int te = s_ptok[i], e = s_pe[i];
            int c = 0;
            for (int j2 = lane; j2 < n_lut; j2 += 32) c += (s_ptok[j2] < te) || (s_ptok[j2] == te && s_pe[j2] < e);
            c = __reduce_add_sync(0xffffffffu, c);
            if (lane == 0) {
                s_rank[i] = c;
                s_sorted_tok[c] = te;
            }
        }
    }
    __syncthreads();
    // token groups over the sorted table pairs, LUT_MAX_M per thread
    int fl[LUT_MAX_M], nf = 0;
#pragma unroll
    for (int r = 0; r < LUT_MAX_M; ++r) {
        const int q = LUT_MAX_M * tid + r;
        fl[r] = (q < n_lut && (q == 0 || s_sorted_tok[q] != s_sorted_tok[q - 1])) ? 1 : 0;
        nf += fl[r];
    }
    unsigned long long n_groups64;
    int gid = (int)block_scan64((unsigned long long)nf, warp_tot, &n_groups64);
    const int n_groups = (int)n_groups64;
#pragma unroll
    for (int r = 0; r < LUT_MAX_M; ++r)
        if (fl[r]) {
            grp_start[gid] = LUT_MAX_M * tid + r;
            s_gs[gid] = LUT_MAX_M * tid + r;
            ++gid;
        }
    if (tid == 0) s_gs[n_groups] = n_lut;
    __syncthreads();
    // the expert's own thread writes the records of its table pairs at their ranks
    for (int q = 0; q < nl; ++q) {
        const int rank = s_rank[lbase + q];
        LutRec r;
        for (int mtx = 0; mtx < 3; ++mtx) {
            r.codes[mtx] = d.codes[mtx];
            r.scales[mtx] = d.scales[mtx];
        }
        r.sorted = s_off[tid] + q;
        r.token = s_ptok[lbase + q];
        // the token group of sorted table pair 'rank': the last group start <= rank
        int lo = 0, hi = n_groups;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (s_gs[mid] <= rank) lo = mid; else hi = mid;
        }
        r.gs = s_gs[lo];
        r.gc = s_gs[lo + 1] - r.gs;
        recs[rank] = r;
    }
    // FC1 unit ranges of the C table-kernel CTAs (jobs = (token group, K-range))
    {
        const int KR1 = lut_jobs(H), RT1 = 2 * I / 16;
        const int J = n_groups * KR1, U = n_lut * KR1 * RT1;
        auto start = [&](int j) {
            const int g = j / KR1, kr = j - g * KR1;
            const int gs = s_gs[g], gc = g < n_groups ? s_gs[g + 1] - gs : 0;
            return (gs * KR1 + kr * gc) * RT1;
        };
        int* s_a = s_pe;  // (free after the ranking; C + 1 <= MAX_TP entries)
        __syncthreads();
        bool ok = J > 0 && J <= C;
        if (ok && tid <= J) s_a[tid] = tid == J ? C : lut_cta_of(start(tid), C, U);
        __syncthreads();
        ok = __syncthreads_and(!ok || tid >= J || s_a[tid + 1] > s_a[tid]) && ok;
        if (tid < C) {
            int4 rg;  // (u0, u1, first offset, stride): one job, its CTAs interleaved
            if (ok) {
                int lo = 0, hi = J;  // the job j with s_a[j] <= tid < s_a[j+1]
                while (hi - lo > 1) {
                    const int mid = (lo + hi) >> 1;
                    if (s_a[mid] <= tid) lo = mid; else hi = mid;
                }
                rg = make_int4(start(lo), lo + 1 < J ? start(lo + 1) : U, tid - s_a[lo], s_a[lo + 1] - s_a[lo]);
            } else {  // a contiguous range of units (over jobs)
                rg = make_int4((int)((long long)U * tid / C), (int)((long long)U * (tid + 1) / C), 0, 0);
            }
            fc1_range[tid] = rg;
        }
    }
    if (tid == 0) {
        grp_start[n_groups] = n_lut;
        header[HDR_NCHUNKS] = n_chunks;
        header[HDR_NLUT] = n_lut;
        header[HDR_ERR] = 0;
        header[HDR_NGROUPS] = n_groups;
        header[HDR_NUMMA] = n_umma;
        header[HDR_NVQ2] = n_vq2;
        header[HDR_NLUT4] = n_lut4;
        header[HDR_NGROUPS4] = n_groups4;
    }
    // eight positions per thread at a time: their sorted_pair loads (beyond
    // the staged part) are in flight together
    for (int s0 = tid; s0 < P; s0 += 8 * 1024) {
        int spv[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) spv[u] = s0 + 1024 * u < P ? sp_at(s0 + 1024 * u) : 0;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int s2 = s0 + 1024 * u;
            if (s2 >= P) break;
            int lo = 0, hi = E;  // find e with off[e] <= s2 < off[e+1]
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (s_off[mid] <= s2) lo = mid; else hi = mid;
            }
            status[spv[u]] = s_res[lo];
        }
    }
}

}  // namespace

size_t ffn_workspace_size(int T, int k, int E, int H, int I) { return ws_layout(T, k, E, H, I).total; }

moe_status launch_expert_ffn(const SlotTableHost* t, const uint16_t* x, const int32_t* offsets,
                             const int32_t* sorted_pair, const float* weights, int T, int k, int mode,
                             float* out, uint8_t* status, void* ws, size_t ws_bytes, cudaStream_t s,
                             const int32_t* pair_to_sorted, float* comb32, uint16_t* comb16) {
    (void)ws_bytes;
    const bool comb = comb32 != nullptr || comb16 != nullptr;
    const int E = t->E, H = t->H, I = t->I;
    const int P = T * k;
    if (num_sms() >= MAX_LUT_CTAS) {
        set_error("moe_vq2_expert_ffn: %d SMs above the supported %d", num_sms(), MAX_LUT_CTAS - 1);
        return MOE_ERR_UNSUPPORTED;
    }
    if (k > 32) {  // the experts of one token are handled as one group of at most 32
        set_error("moe_vq2_expert_ffn: k=%d above 32", k);
        return MOE_ERR_UNSUPPORTED;
    }
    const WsLayout L = ws_layout(T, k, E, H, I);
    char* w = static_cast<char*>(ws);
    int* header = reinterpret_cast<int*>(w);
    Chunk* chunks = reinterpret_cast<Chunk*>(w + L.chunks_off);
    LutRec* recs = reinterpret_cast<LutRec*>(w + L.rec_off);
    int32_t* grp_start = reinterpret_cast<int32_t*>(w + L.grp_start_off);
    Chunk* uchunks = reinterpret_cast<Chunk*>(w + L.uchunks_off);
    // VQ2 experts with at most lut_max_m tokens take the table kernels
    const int lut_max_m = T >= MMA_SPLIT_T ? LUT_MAX_M_LARGE : LUT_MAX_M;
    const bool use_lut = lut_max_m > 0;
    // An expert gets at most T of the pairs: at T == UMMA_MIN only an expert
    // routed by every token would qualify, and the 32-token mma.sync chunk
    // serves it as well, so the tcgen05 launches start above that (at
    // batch 32 they found work in one batch of eight and cost two launches).
    const int use_umma = T > UMMA_MIN ? 1 : 0;
    // FP4 experts take the e2m1 table kernels in calls of at most LUT4_MAX_T
    // tokens.
    const bool use_lut4 = T <= LUT4_MAX_T && t->n_fp4 > 0;
    // In calls of at most lut_max_m tokens no expert gets more pairs than the
    // table path takes, so the mma.sync kernels only have work if FP4
    // experts do not take the e2m1 tables.
    const bool mma = T > lut_max_m || (t->n_fp4 > 0 && !use_lut4);
    // (and VQ2 experts only reach them, in 32-token chunks, above lut_max_m)
    const bool mma_vq2 = T > lut_max_m;
    const int split16 = T >= MMA_SPLIT_T ? 1 : 0;

    moe_status st;
    if (T == 1 && t->n_fp4 == 0) {
        // one token, VQ2 experts only: every pair takes the table path and the
        // two table kernels list the pairs themselves (no schedule kernel)
        // (FC1 gets the combine outputs too: it zeroes FC2's counters only
        // where FC2 will use them)
        if ((st = launch_lut_fc(true, true, t, x, offsets, sorted_pair, weights, k, P, mode, out, status, w, L, s,
                                pair_to_sorted, comb32, comb16)) != MOE_OK)
            return st;
        return launch_lut_fc(false, true, t, x, offsets, sorted_pair, weights, k, P, mode, out, status, w, L, s,
                             pair_to_sorted, comb32, comb16);
    }
    cudaError_t e = ensure_smem_attr(schedule_kernel, (int)SCHED_SMEM);
    if (e != cudaSuccess) return cuda_status(e, "moe_vq2_expert_ffn: schedule shared memory");
    e = launch_pdl(schedule_kernel, dim3(1), dim3(1024), SCHED_SMEM, s, (const SlotDesc*)t->d_desc, E, offsets,
                               sorted_pair, P, k, status, header, chunks, recs, grp_start, lut_max_m,
                               uchunks, use_umma, H, I, num_sms(), reinterpret_cast<int4*>(w + L.range_off), split16,
                               reinterpret_cast<LutRec*>(w + L.rec4_off), use_lut4 ? 1 : 0);
    if (e != cudaSuccess) return cuda_status(e, "moe_vq2_expert_ffn: schedule launch");
    if ((mma || use_umma) && (st = launch_gather_f16(x, sorted_pair, k, H, P, w, L, s)) != MOE_OK) return st;
    if (use_lut &&
        (st = launch_lut_fc(true, false, t, x, offsets, sorted_pair, weights, k, P, mode, out, status, w, L, s)) !=
            MOE_OK)
        return st;
    if (use_lut4 && (st = launch_lut_fc(true, false, t, x, offsets, sorted_pair, weights, k, P, mode, out, status, w,
                                        L, s, nullptr, nullptr, nullptr, true)) != MOE_OK)
        return st;
    if (mma && (st = launch_mma_fc(true, t, sorted_pair, weights, k, mode, out, w, L, s, split16, mma_vq2)) != MOE_OK) return st;
    if (use_umma && (st = launch_umma(true, t, sorted_pair, weights, k, P, mode, out, w, L, s)) != MOE_OK) return st;
    if ((mma || use_umma) && (st = launch_a_to_f16(P, I, w, L, s)) != MOE_OK) return st;
    if (use_lut &&
        (st = launch_lut_fc(false, false, t, x, offsets, sorted_pair, weights, k, P, mode, out, status, w, L, s)) !=
            MOE_OK)
        return st;
    if (use_lut4 && (st = launch_lut_fc(false, false, t, x, offsets, sorted_pair, weights, k, P, mode, out, status, w,
                                        L, s, nullptr, nullptr, nullptr, true)) != MOE_OK)
        return st;
    if (mma && (st = launch_mma_fc(false, t, sorted_pair, weights, k, mode, out, w, L, s, split16, mma_vq2)) != MOE_OK) return st;
    if (use_umma && (st = launch_umma(false, t, sorted_pair, weights, k, P, mode, out, w, L, s)) != MOE_OK) return st;
    if (comb) return launch_combine(out, pair_to_sorted, weights, status, T, k, H, comb32, comb16, s);
    return MOE_OK;
}

}  // namespace moe
