// Activation-table path of the expert FFN, for VQ2 experts that receive at
// most LUT_MAX_M tokens in this call (every expert at decode batch 1, most of
// them at small batches): one table pair per (token, expert), the expert's
// codes streamed once per token.  In calls of one or two tokens the FP4 experts
// take the same kernels with e2m1 tables (the F4 instances).
//
// The table, the lane layout and the per-unit lookups are the shared core in
// lut_core.cuh.
//
// K-range partial sums go to the workspace: FC2's table build adds FC1's
// partials in a fixed order and applies silu(g) * u; of FC2's partials, the
// warp that completes a row tile last (one counter per row tile) adds them in
// K-range order and writes y, so every result is independent of timing.
//
// Code tiles are streamed by the copy engine into one shared-memory slot per
// warp (a unit = 16 rows x 1024 inputs: three bulk copies, codes and scales),
// so the code stream never sits in the load/store queue in front of the table
// reads; a warp copies its slot to registers, hands the slot to the copy of
// its next unit, asks L2 for the unit after that, and computes from
// registers.  Waits on the slots are bounded: a wait that runs out records an
// error in the workspace header and the CTA stops.
#include <cuda_bf16.h>

#include "ffn_common.cuh"
#include "lut_core.cuh"

namespace moe {
namespace {

using namespace lut;

constexpr int MAX_GROUP = 32;            // table pairs of one token (<= k <= 32)
constexpr int NSLOT = LW;                // one code slot per warp
constexpr int LOW_SLOTS = 12;            // slots below the table; the rest above it
static_assert(LOW_SLOTS * SLOT_BYTES >= 4 * (1024 + 1), "the expert offsets (E <= 1024) fit in the low slots");
constexpr uint32_t HIGH_BASE = TAB_END;

struct __align__(16) Smem {
    unsigned long long full[NSLOT];        // slot mbarriers (one arrival + the copied bytes)
    alignas(16) float xs[XS_FLOATS];       // (read as float4)
    alignas(16) float cb[128 * 4];         // (read as float4)
    const void* pa[MAX_GROUP];  // per pair of the current group: FC1 gate / FC2 down codes
    const void* pb[MAX_GROUP];  // FC1 up codes
    const void* sa[MAX_GROUP];  // matching scales
    const void* sb[MAX_GROUP];
    // single-token calls (no schedule kernel): every pair's buffers
    const void* all_c[3][MAX_GROUP];
    const void* all_s[3][MAX_GROUP];
    int ys[MAX_GROUP];          // FC2: sorted position of the pair
    int all_ys[MAX_GROUP];
    int e_of_s[MAX_GROUP];
    uint8_t lastf[256];         // FC2: the row tiles whose partials this CTA adds up
    unsigned red[2 * LW];       // table-scale reduction
    int n_self;
    int failed;
};
static_assert(offsetof(Smem, xs) % 16 == 0 && offsetof(Smem, cb) % 16 == 0, "float4 reads of xs and cb");
static_assert(0x400 + ((sizeof(Smem) + 127) / 128 * 128) + LOW_SLOTS * SLOT_BYTES <= TAB &&
                  HIGH_BASE + (NSLOT - LOW_SLOTS) * SLOT_BYTES <= 0x400 + DYN_SMEM && NSLOT >= LOW_SLOTS,
              "shared layout");

// SELF: a single-token call whose experts are all VQ2 (no schedule kernel):
// the kernel lists the call's pairs itself from the expert offsets and the
// slot table (one token group; pairs in sorted order, non-resident ones
// reported and skipped).  comb32 / comb16 (SELF): FC2 also writes the combine
// of the pairs; FC1 gets them only to know which of FC2's counters to zero.
// F4: the FP4 experts of calls of at most LUT4_MAX_T tokens (e2m1 tables
// over K-ranges of 512 inputs; the schedule's second record list, grouped by
// token; never SELF).  These kernels read only what the schedule and the kernels before
// their predecessor wrote (FC2: the e2m1 FC1's partial sums), which is
// complete when they start, because the predecessor lets its dependents
// start only after its own wait.  So they run beside their predecessor's
// last CTAs and wait for it only before they exit, which keeps the chain of
// completions that the kernels after them rely on.
template <bool FC1, bool SELF, bool F4>
__global__ void __maxnreg__(MAX_REG)
    ffn_lut_kernel(const SlotDesc* __restrict__ desc, const int32_t* __restrict__ offsets, int E, int P,
                   uint8_t* __restrict__ status, const uint16_t* __restrict__ codebook, const uint16_t* __restrict__ x,
                   const int32_t* __restrict__ sorted_pair, const float* __restrict__ weights, int k, int H, int I,
                   int* __restrict__ header, const LutRec* __restrict__ recs,
                   const int4* __restrict__ fc1_range, const float* __restrict__ p1, float* __restrict__ pout,
                   int* __restrict__ cnt, int mode, float* __restrict__ out, const int32_t* __restrict__ p2s,
                   float* __restrict__ comb32, uint16_t* __restrict__ comb16, int* __restrict__ cnt2) {
    extern __shared__ __align__(1024) uint8_t dyn[];
    Smem& S = *reinterpret_cast<Smem*>(dyn);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int* err = header + HDR_ERR;

    static_assert(!(F4 && SELF), "FP4 pairs come from the schedule");
    constexpr int TILE_IN = F4 ? 64 : 128;     // inputs per packed tile
    constexpr int KRI = LUT_KB * TILE_IN;      // inputs per K-range
    const int K = FC1 ? H : I;             // inputs of this matrix
    const int R = FC1 ? 2 * I : H;         // rows per pair (FC1: gate rows, then up rows)
    const int KB = K / TILE_IN;
    const int KR = F4 ? lut4_jobs(K) : lut_jobs(K);
    const int RT = R / 16;
    const int KR1 = F4 ? lut4_jobs(H) : lut_jobs(H);
    const int per_pair = KR * RT;          // units of one pair
    const int C = gridDim.x;

    // The fixed table address needs the low part of dynamic shared memory
    // below it and the allocation to reach past its end; the code slots sit
    // around it.
    const uint32_t base = smem_u32(dyn);
    const uint32_t low_base = (base + (uint32_t)sizeof(Smem) + 127u) & ~127u;
    if (low_base + LOW_SLOTS * SLOT_BYTES > TAB || base + DYN_SMEM < HIGH_BASE + (NSLOT - LOW_SLOTS) * SLOT_BYTES) {
        if (tid == 0) atomicExch(err, MOE_DEVERR_SMEM_LAYOUT);
        return;
    }
    const uint32_t slot = warp < LOW_SLOTS ? low_base + warp * SLOT_BYTES : HIGH_BASE + (warp - LOW_SLOTS) * SLOT_BYTES;
    const uint32_t bar = smem_u32(&S.full[warp]);
    if (!F4)
        for (int i = tid; i < 128 * 4; i += THREADS) S.cb[i] = __half2float(__ushort_as_half(codebook[i]));
    if (tid < NSLOT) mbar_init(smem_u32(&S.full[tid]), 1);
    if (tid == 0) S.failed = 0;
    mbar_fence_init();

    // Units are (job, row tile) with job = (group, K-range).  FC1 groups are
    // the table pairs of one token (they share the activation table); FC2
    // groups are single pairs (the table depends on the pair's silu(g)*u).
    // A group of gc pairs starting at table pair gs owns the units
    // [per_pair*gs, per_pair*(gs+gc)), ordered (K-range, pair, row tile).
    // A CTA's work: units [u0, u1) in job order; with s_step > 0 (no more jobs
    // than CTAs) a single job of which it takes the units s_off0 + s_step * i,
    // the job's CTAs interleaved, so that every CTA meets the same mix of
    // pairs and rows.
    int n_lut, u0, u1, s_off0 = 0, s_step = 0;
    bool waited = FC1 || F4;  // FC2 waits for FC1 once its first job's code copies are issued
    // every job is RT units (SELF FC1: one token group of n_lut pairs, KR jobs
    // of n_lut * RT units) -> the proportional split is direct
    auto uniform_range = [&](int J, int job_units) {
        const int U = J * job_units;
        if (U == 0) {
            u0 = u1 = 0;
        } else if (J <= C) {
            // equal jobs: a0(j) = floor(C start(j) / U) = floor(C j / J), all
            // in 32-bit arithmetic (J <= C <= 1024)
            const int jb = ((int)(blockIdx.x + 1) * J - 1) / C;  // a0(jb) <= i < a0(jb + 1)
            const int a0 = C * jb / J;
            const int a1 = C * (jb + 1) / J;
            u0 = jb * job_units;
            u1 = u0 + job_units;
            s_off0 = blockIdx.x - a0;
            s_step = a1 - a0;
        } else {
            u0 = (int)((long long)U * blockIdx.x / C);
            u1 = (int)((long long)U * (blockIdx.x + 1) / C);
        }
    };
    // The table of the K-range whose inputs are in S.xs, with its scale
    // exponent (block-wide); tab_s = 2^e multiplies each unit's sums back.
    float tab_s = 1.0f;
    auto build_table = [&](int nkb) {
        const int e = table_exponent(S.xs, TILE_IN * nkb, F4 ? nullptr : S.cb, S.red, tid);
        tab_s = exp2_int(e);
        if (F4)
            lut::build_table_f4(S.xs, nkb, e, tid);
        else
            lut::build_table(S.xs, S.cb, nkb, e, tid);
    };
    // The token's activations of a K-range into S.xs (as fp32).
    auto load_x = [&](int t, int kr, int nin) {
        for (int i = tid; i < nin; i += THREADS)
            S.xs[xs_at(i)] = __uint_as_float((uint32_t)x[(size_t)t * H + KRI * kr + i] << 16);
    };
    // SELF FC1: the CTA's K-range follows from the grid alone (KR jobs of
    // equal size, see uniform_range), so the activations and the table are
    // built before the wait, while the routing kernel before this one still
    // runs (x is complete at launch: no library kernel still running writes
    // bf16 activations).
    // With two FC2 K-ranges and per-pair output, FC2 adds its two partial
    // sums straight into the zeroed output row (fp32 addition is commutative,
    // so 0 + p0 + p1 does not depend on the order) instead of a finishing
    // step; FC1 zeroes the rows of the table pairs.
    const int KR2 = lut_jobs(I);  // FC2's K-ranges (VQ2)
    const bool fc2_adds = !F4 && mode == MOE_PER_PAIR && KR2 == 2;
    auto zero_rows = [&](auto row_of) {
        const int n4 = H / 4;  // (n_lut <= E <= 1024 table pairs)
        for (int i = blockIdx.x * THREADS + tid; i < n_lut * n4; i += C * THREADS) {
            const int p = i / n4;
            reinterpret_cast<float4*>(out + (size_t)row_of(p) * H)[i - p * n4] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    };
    int pre_kr = -1;
    // SELF: the slot descriptors do not depend on the kernel before this one
    // (only the slot-table writer changes them, and it lets no dependent start
    // before it has finished), so they are staged in the code slots, after the
    // expert offsets, before the wait: the pair listing then needs one round
    // trip to global memory instead of two.
    // (The descriptor words are loaded into registers first, so that their
    // round trip overlaps the activations' (FC1) or the expert offsets' (FC2,
    // whose offsets are two kernels back, so complete).)
    constexpr int DW = 4;  // descriptor words per thread at most
    const int n_dw = E * (int)(sizeof(SlotDesc) / 8);
    const size_t off_bytes = ((size_t)4 * (E + 1) + 15) & ~(size_t)15;
    const bool desc_staged = SELF && n_dw <= DW * THREADS &&
                             off_bytes + sizeof(SlotDesc) * E <= (size_t)LOW_SLOTS * SLOT_BYTES;
    SlotDesc* s_desc = reinterpret_cast<SlotDesc*>(dyn + (low_base - base) + off_bytes);
    unsigned long long dv[DW];
    if (desc_staged) {
        const unsigned long long* src = reinterpret_cast<const unsigned long long*>(desc);
#pragma unroll
        for (int r = 0; r < DW; ++r)
            if (tid + r * THREADS < n_dw) dv[r] = src[tid + r * THREADS];
    }
    constexpr int OW = 3;  // offsets per thread at most (E + 1 <= 1025)
    int ov[OW];
    if (SELF && !FC1) {
#pragma unroll
        for (int r = 0; r < OW; ++r)
            if (tid + r * THREADS <= E) ov[r] = __ldcg(offsets + tid + r * THREADS);
    }
    if (SELF && FC1 && KR <= C) {
        pre_kr = (int)(((long long)(blockIdx.x + 1) * KR - 1) / C);
        const int nkb = min(LUT_KB, KB - LUT_KB * pre_kr);
        load_x(0, pre_kr, 128 * nkb);
    }
    if (desc_staged) {
        unsigned long long* dst = reinterpret_cast<unsigned long long*>(s_desc);
#pragma unroll
        for (int r = 0; r < DW; ++r)
            if (tid + r * THREADS < n_dw) dst[tid + r * THREADS] = dv[r];
    }
    if (SELF && FC1 && KR <= C) {
        __syncthreads();
        build_table(min(LUT_KB, KB - LUT_KB * pre_kr));
    }
    if (SELF) {
        // FC1: the offsets come from the kernel just before (wait first); FC2:
        // they are two kernels back (complete), so FC2 lists its pairs first.
        if (FC1) {
            pdl_wait();
            pdl_launch_dependents();  // (FC1 writes no bf16 activations)
            if (blockIdx.x == 0 && tid == 0) *err = 0;  // this call's error word
        }
        // the offsets are staged in the (still unused) code slots below the table
        int* s_off = reinterpret_cast<int*>(dyn + (low_base - base));
        if (FC1) {
            for (int i = tid; i <= E; i += THREADS) s_off[i] = offsets[i];
        } else {
#pragma unroll
            for (int r = 0; r < OW; ++r)
                if (tid + r * THREADS <= E) s_off[tid + r * THREADS] = ov[r];
        }
        if (tid < MAX_GROUP) S.e_of_s[tid] = -1;
        __syncthreads();
        for (int e = tid; e < E; e += THREADS)  // the expert of each sorted position < P
            for (int sp = max(s_off[e], 0); sp < min(s_off[e + 1], P); ++sp) S.e_of_s[sp] = e;
        __syncthreads();
        if (warp == 0) {
            SlotDesc d;
            d.resident = 0;
            d.format = MOE_FMT_VQ2;
            if (lane < P && S.e_of_s[lane] >= 0) d = desc_staged ? s_desc[S.e_of_s[lane]] : desc[S.e_of_s[lane]];
            const bool res = lane < P && d.resident != 0 && d.format == MOE_FMT_VQ2;
            const unsigned mask = __ballot_sync(0xffffffffu, res);
            const int idx = __popc(mask & ((1u << lane) - 1u));
            if (res) {
#pragma unroll
                for (int mtx = 0; mtx < 3; ++mtx) {
                    S.all_c[mtx][idx] = d.codes[mtx];
                    S.all_s[mtx][idx] = d.scales[mtx];
                }
                S.all_ys[idx] = lane;
            }
            if (FC1 && blockIdx.x == 0 && lane < P) status[sorted_pair[lane]] = res ? 1 : 0;
            if (lane == 0) S.n_self = __popc(mask);
        }
        // the slots were written through the generic proxy; the copies that
        // fill them later are async-proxy writes
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncthreads();
        n_lut = S.n_self;
        uniform_range(FC1 ? KR : n_lut * KR, FC1 ? n_lut * RT : RT);
        if (FC1) {
            // FC2's arrival counters start at zero where FC2 uses them (it
            // leaves them at zero): per row tile when it adds K-range
            // partials through them, per output tile when it combines.  FC1
            // gets FC2's combine outputs only to know that.
            const bool fc2_combines = comb32 != nullptr || comb16 != nullptr;
            if (fc2_combines || (KR2 > 1 && !fc2_adds)) {
                const int nc = n_lut * (H / 16);
                for (int i = blockIdx.x * THREADS + tid; i < nc; i += C * THREADS) cnt[i] = 0;
            }
            if (fc2_combines)
                for (int i = blockIdx.x * THREADS + tid; i < H / 16; i += C * THREADS) cnt2[i] = 0;
            if (fc2_adds) zero_rows([&](int p) { return S.all_ys[p]; });
        }
    } else if (FC1) {
        if (!F4) pdl_wait();
        // everything a dependent kernel may touch before its own wait is complete
        pdl_launch_dependents();
        if (F4) {
            n_lut = __ldcg(header + HDR_NLUT4);
            if (__ldcg(header + HDR_NGROUPS4) <= 1) {
                uniform_range(KR, n_lut * RT);  // one token group
            } else {  // groups of unequal size: a contiguous share of the units
                const int U = n_lut * KR * RT;
                u0 = (int)((long long)U * blockIdx.x / C);
                u1 = (int)((long long)U * (blockIdx.x + 1) / C);
            }
        } else {
            n_lut = header[HDR_NLUT];
            const int4 rg = fc1_range[blockIdx.x];  // computed by the schedule
            u0 = rg.x;
            u1 = rg.y;
            s_off0 = rg.z;
            s_step = rg.w;
        }
        // FC2's arrival counters start at zero
        const int nc = n_lut * (H / 16);
        for (int i = blockIdx.x * THREADS + tid; i < nc; i += C * THREADS) cnt[i] = 0;
        if (fc2_adds) zero_rows([&](int p) { return recs[p].sorted; });
    } else {
        // The schedule is two kernels back, so complete: this CTA's units and
        // their code bytes are known before FC1 completes.
        n_lut = __ldcg(header + (F4 ? HDR_NLUT4 : HDR_NLUT));
        uniform_range(n_lut * KR, RT);
        if (F4) pdl_launch_dependents();
    }

    const bool comb = !FC1 && SELF && (comb32 != nullptr || comb16 != nullptr);
    const bool adds = !FC1 && fc2_adds && !comb;  // (then KR == 2)
    const int b = lane_block(lane);  // scale block of this lane
    const uint32_t lb = TAB | (uint32_t)(4 * lane);
    uint32_t phase = 0;                     // parity of the slot's next completion
    bool pend = false;                      // the slot has a copy in flight
    bool ok = true;                         // this warp's slot waits all completed

    int u = u0;
    while (u < u1) {
        __syncthreads();  // every warp is done with the previous table and pointers
        if (S.failed) break;
        const LutRec& r0 = recs[SELF ? 0 : u / per_pair];
        const int gs = FC1 ? (SELF ? 0 : r0.gs) : u / per_pair;
        const int gc = FC1 ? (SELF ? n_lut : r0.gc) : 1;
        const int kr = (u - per_pair * gs) / (RT * gc);
        const int job_start = per_pair * gs + kr * RT * gc;
        const int seg_end = min(u1, job_start + RT * gc);
        const int nkb = min(LUT_KB, KB - LUT_KB * kr);
        const int nin = TILE_IN * nkb;
        const bool active = b < nkb;
        if (tid < gc) {
            if (SELF) {
                S.pa[tid] = S.all_c[FC1 ? 0 : 2][gs + tid];
                S.sa[tid] = S.all_s[FC1 ? 0 : 2][gs + tid];
                S.pb[tid] = S.all_c[1][gs + tid];
                S.sb[tid] = S.all_s[1][gs + tid];
                S.ys[tid] = S.all_ys[gs + tid];
            } else {
                const LutRec& r = recs[gs + tid];
                S.pa[tid] = r.codes[FC1 ? 0 : 2];
                S.sa[tid] = r.scales[FC1 ? 0 : 2];
                S.pb[tid] = r.codes[1];
                S.sb[tid] = r.scales[1];
                S.ys[tid] = r.sorted;
            }
        }
        const bool prebuilt = SELF && FC1 && kr == pre_kr;  // table built before the wait
        if (FC1 && !prebuilt) load_x(SELF ? 0 : r0.token, kr, nin);  // the token's activations
        __syncthreads();

        // unit v of the job <-> (pair pi of the group, row tile rt); cursors
        // move by LW units without divisions
        struct Cur {
            int pi, rt;
        };
        auto cur_at = [&](int off) {
            Cur c;
            c.pi = off / RT;
            c.rt = off - c.pi * RT;
            return c;
        };
        // this CTA's units of the job: offsets v_first + v_inc * i < v_end;
        // warp w takes i = w, w + LW, ...
        const int v_first = s_step ? s_off0 : u - job_start, v_inc = s_step ? s_step : 1;
        const int v_end = s_step ? RT * gc : seg_end - job_start;
        const int vstep = v_inc * LW;
        int v0 = v_first + v_inc * warp;
        auto advance = [&](Cur c) {
            c.rt += vstep;
            while (c.rt >= RT) {
                c.rt -= RT;
                ++c.pi;
            }
            return c;
        };
        Cur c0 = cur_at(v0);              // the unit computed next
        Cur c1 = advance(c0);             // the one after it
        Cur c2 = advance(c1);
        auto unit_ptrs = [&](Cur cu, const uint8_t*& c, const uint16_t*& sp) {
            const bool second = FC1 && cu.rt >= I / 16;  // an up-matrix row tile
            const int rtm = second ? cu.rt - I / 16 : cu.rt;
            const size_t tile = (size_t)rtm * KB + LUT_KB * kr;
            c = static_cast<const uint8_t*>(second ? S.pb[cu.pi] : S.pa[cu.pi]) + tile * 512;
            sp = static_cast<const uint16_t*>(second ? S.sb[cu.pi] : S.sa[cu.pi]) + tile * 16;
        };
        // Unit at cursor cu into the warp's slot.
        auto issue = [&](Cur cu) {
            pend = true;
            const uint8_t* c;
            const uint16_t* sp;
            unit_ptrs(cu, c, sp);
            issue_unit(slot, bar, c, sp, nkb, lane);
        };
        auto prefetch = [&](Cur cu) {  // ask L2 for the unit at cu
            if (lane == 0) {
                const uint8_t* c;
                const uint16_t* sp;
                unit_ptrs(cu, c, sp);
                (void)sp;
                asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(c), "r"(512u * nkb) : "memory");
            }
        };
        if (v0 < v_end) issue(c0);
        if (v0 + vstep < v_end) prefetch(c1);

        if (!waited) {
            pdl_wait();
            // everything a dependent kernel may touch before its own wait is
            // complete; with a bf16 combine output the dependents start only
            // when this kernel has finished (they may read it as activations)
            if (comb16 == nullptr) pdl_launch_dependents();
            waited = true;
        }
        if (!FC1 && F4) {
            // (FP4: one input per thread, 8 partials of g and of u in flight)
            static_assert(!F4 || KRI <= THREADS, "one input per thread");
            const float* pp = p1 + (size_t)gs * KR1 * 2 * I;
            const int i = tid, gi = KRI * kr + i;
            float g = 0.0f, up = 0.0f;
            for (int j0 = 0; j0 < KR1; j0 += 8) {
                float pg[8], pu[8];
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) {
                    const bool in = i < nin && j0 + jj < KR1;
                    pg[jj] = in ? pp[(size_t)(j0 + jj) * 2 * I + gi] : 0.0f;
                    pu[jj] = in ? pp[(size_t)(j0 + jj) * 2 * I + I + gi] : 0.0f;
                }
#pragma unroll
                for (int jj = 0; jj < 8; ++jj)
                    if (j0 + jj < KR1) {
                        g += pg[jj];
                        up += pu[jj];
                    }
            }
            if (i < nin) S.xs[xs_at(i)] = silu_mul(g, up);
            __syncthreads();
        } else if (!FC1) {
            // silu(g) * u of the pair from FC1's K-range partial sums, added in
            // order: a thread's (up to 4) inputs with 4 partials each in flight
            const float* pp = p1 + (size_t)gs * KR1 * 2 * I;
            for (int i0 = tid; i0 < nin; i0 += 4 * THREADS) {
                float g[4] = {0.0f, 0.0f, 0.0f, 0.0f}, up[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                for (int j0 = 0; j0 < KR1; j0 += 4) {
                    float pg[4][4], pu[4][4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int i = i0 + q * THREADS, gi = KRI * kr + i;
#pragma unroll
                        for (int jj = 0; jj < 4; ++jj) {
                            const bool in = i < nin && j0 + jj < KR1;
                            pg[q][jj] = in ? pp[(size_t)(j0 + jj) * 2 * I + gi] : 0.0f;
                            pu[q][jj] = in ? pp[(size_t)(j0 + jj) * 2 * I + I + gi] : 0.0f;
                        }
                    }
#pragma unroll
                    for (int q = 0; q < 4; ++q)
#pragma unroll
                        for (int jj = 0; jj < 4; ++jj)
                            if (j0 + jj < KR1) {
                                g[q] += pg[q][jj];
                                up[q] += pu[q][jj];
                            }
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int i = i0 + q * THREADS;
                    if (i < nin) S.xs[xs_at(i)] = silu_mul(g[q], up[q]);
                }
            }
            __syncthreads();
        }

        if (!prebuilt) build_table(nkb);
        __syncthreads();

        auto compute_store = [&](const UnitRegs& r, Cur cu) {
            const int pi = cu.pi, rt = cu.rt;
            float acc[1];
            acc[0] = unit_rows<F4>(r, lb, active, lane) * tab_s;
            const int h = rt * 16 + unit_row(lane);  // output row of this lane pair
            auto emit = [&](float y) {  // FC2: the finished y of row h
                const int s = S.ys[pi];
                if (mode == MOE_PER_PAIR) {
                    out[(size_t)s * H + h] = y;
                } else {
                    const int pr = sorted_pair[s];
                    atomicAdd(out + (size_t)(pr / k) * H + h, weights[pr] * y);
                }
            };
            if (adds) {
                if ((lane & 1) == 0) atomicAdd(out + (size_t)S.ys[pi] * H + h, acc[0]);
            } else if (FC1 || KR > 1 || comb) {
                if ((lane & 1) == 0) pout[((size_t)(gs + pi) * KR + kr) * R + h] = acc[0];
            } else if ((lane & 1) == 0) {
                emit(acc[0]);
            }
        };

        // This warp's units of the job: v, v + LW, ...  The slot is copied to
        // registers and handed to the copy of the next unit (the one after
        // that is asked of L2), then the unit is computed from registers.
        for (; v0 < v_end; v0 += vstep) {
            if (!mbar_wait_bounded(bar, phase, err, MOE_DEVERR_WAIT_FULL)) {
                ok = false;
                break;
            }
            phase ^= 1u;
            pend = false;
            UnitRegs r;
            load_unit(r, slot, lane, active);
            __syncwarp();
            // the generic-proxy reads of the slot come before the next copy's writes
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            if (v0 + vstep < v_end) issue(c1);
            if (v0 + 2 * vstep < v_end) prefetch(c2);
            compute_store(r, c0);
            c0 = c1;
            c1 = c2;
            c2 = advance(c2);
        }
        if (!ok) {
            // stop the CTA; a copy this warp still has in flight lands before
            // it leaves (bounded wait again)
            S.failed = 1;
            if (pend) mbar_wait_bounded(bar, phase, nullptr, 0);
            pend = false;
        }
        if (!FC1 && (KR > 1 || comb) && !adds) {
            // FC2 partials of this job's row tiles are all stored: one fence per
            // thread, then per row tile one arrival; the last of the KR units of
            // a row tile adds the partials in K-range order and writes y.  With
            // the combine, the last of the pairs to finish a row tile then
            // writes its 16 outputs.
            __threadfence();
            __syncthreads();
            const int pr = gs;  // FC2 groups are single pairs
            const int s = S.ys[0];
            const int n_my = (v_end - v_first + v_inc - 1) / v_inc;  // this CTA's row tiles
            for (int tb = 0; tb < n_my; tb += 256) {
                const int nt = min(256, n_my - tb);
                for (int t = tid; t < nt; t += THREADS) {
                    int* c = cnt + (size_t)pr * RT + v_first + v_inc * (tb + t);
                    const bool last = atomicAdd(c, 1) == KR - 1;
                    S.lastf[t] = last;
                    if (last) *c = 0;
                }
                __threadfence();
                __syncthreads();
                // the row tiles this CTA finishes: one output row per thread
                for (int idx = tid; idx < 16 * nt; idx += THREADS) {
                    const int t = idx >> 4;
                    if (!S.lastf[t]) continue;
                    const int h = (v_first + v_inc * (tb + t)) * 16 + (idx & 15);
                    const float* src = pout + (size_t)pr * KR * R + h;
                    float y = __ldcg(src);
                    for (int jj = 1; jj < KR; ++jj) y += __ldcg(src + (size_t)jj * R);
                    if (mode == MOE_PER_PAIR) {
                        out[(size_t)s * H + h] = y;
                    } else {
                        const int p = sorted_pair[s];
                        atomicAdd(out + (size_t)(p / k) * H + h, weights[p] * y);
                    }
                }
                if (comb) {
                    // one token: out[h] = sum over pairs j (in order) of w_j y_j,
                    // as moe_combine computes it
                    __threadfence();
                    __syncthreads();
                    for (int t = tid; t < nt; t += THREADS) {
                        if (S.lastf[t]) {
                            int* c = cnt2 + v_first + v_inc * (tb + t);
                            if (atomicAdd(c, 1) == n_lut - 1) {
                                S.lastf[t] = 2;
                                *c = 0;
                            }
                        }
                    }
                    __threadfence();
                    __syncthreads();
                    for (int idx = tid; idx < 16 * nt; idx += THREADS) {
                        const int t = idx >> 4;
                        if (S.lastf[t] != 2) continue;
                        const int h = (v_first + v_inc * (tb + t)) * 16 + (idx & 15);
                        float a = 0.0f;
                        for (int j = 0; j < k; ++j)
                            if (__ldcg(status + j))
                                a = __fadd_rn(a, __fmul_rn(weights[j], __ldcg(out + (size_t)p2s[j] * H + h)));
                        if (comb32) comb32[h] = a;
                        if (comb16) comb16[h] = __bfloat16_as_ushort(__float2bfloat16_rn(a));
                    }
                }
                __syncthreads();  // flags are reused by the next chunk
            }
        }
        u = seg_end;
    }
    if (!waited) {  // a CTA without units still waits for FC1 before it leaves
        pdl_wait();
        if (comb16 == nullptr) pdl_launch_dependents();
    }
    if (F4) pdl_wait();  // (see the kernel's description)
    if (comb && n_lut == 0) {  // no pair computed: the combine is zero
        for (int h = blockIdx.x * THREADS + tid; h < H; h += C * THREADS) {
            if (comb32) comb32[h] = 0.0f;
            if (comb16) comb16[h] = 0;
        }
    }
}

}  // namespace

moe_status launch_lut_fc(bool fc1, bool self, const SlotTableHost* t, const uint16_t* x, const int32_t* offsets,
                         const int32_t* sorted_pair, const float* weights, int k, int P, int mode, float* out,
                         uint8_t* status, char* ws, const WsLayout& L, cudaStream_t s,
                         const int32_t* pair_to_sorted, float* comb32, uint16_t* comb16, bool f4) {
    if (f4 && (self || comb32 || comb16)) {
        set_error("moe_vq2_expert_ffn: FP4 table pairs come from the schedule");
        return MOE_ERR_UNSUPPORTED;
    }
    int* header = reinterpret_cast<int*>(ws);
    const LutRec* recs = reinterpret_cast<const LutRec*>(ws + (f4 ? L.rec4_off : L.rec_off));
    const int4* fc1_range = reinterpret_cast<const int4*>(ws + L.range_off);
    const float* p1 = reinterpret_cast<const float*>(ws + (f4 ? L.p1_4_off : L.p1_off));
    float* pout = reinterpret_cast<float*>(ws + (f4 ? (fc1 ? L.p1_4_off : L.p2_4_off) : (fc1 ? L.p1_off : L.p2_off)));
    int* cnt = reinterpret_cast<int*>(ws + (f4 ? L.cnt4_off : L.cnt_off));
    auto kern = f4 ? (fc1 ? ffn_lut_kernel<true, false, true> : ffn_lut_kernel<false, false, true>)
                   : self ? (fc1 ? ffn_lut_kernel<true, true, false> : ffn_lut_kernel<false, true, false>)
                          : (fc1 ? ffn_lut_kernel<true, false, false> : ffn_lut_kernel<false, false, false>);
    cudaError_t e = ensure_smem_attr(kern, (int)DYN_SMEM);
    if (e != cudaSuccess) return cuda_status(e, "moe_vq2_expert_ffn: table kernel shared memory");
    // One CTA per SM; the single-token FC1 leaves one SM free, so that all of
    // its CTAs are resident (building their tables) while the routing
    // kernel's last CTA still runs.
    const int grid = (self && fc1 && num_sms() > 1) ? num_sms() - 1 : num_sms();
    e = launch_pdl(kern, dim3((unsigned)grid), dim3(THREADS), DYN_SMEM, s, (const SlotDesc*)t->d_desc, offsets,
                   t->E, P, status, t->codebook, x, sorted_pair, weights, k, t->H, t->I, header, recs, fc1_range, p1,
                   pout, cnt, mode, out, pair_to_sorted, comb32, comb16, reinterpret_cast<int*>(ws + L.cnt2_off));
    if (e != cudaSuccess) return cuda_status(e, "moe_vq2_expert_ffn: table kernel launch");
    MOE_LAUNCH_CHECK("moe_vq2_expert_ffn: table kernel launch");
    return MOE_OK;
}

}  // namespace moe
