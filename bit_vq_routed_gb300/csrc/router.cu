// Router logits (fixed fp32 summation order) and top-k + softmax routing.
#include <float.h>
#include <limits.h>

#include <mutex>

#include "common.cuh"

namespace moe {
namespace {

constexpr unsigned FULL = 0xffffffffu;

__device__ __forceinline__ void unpack_bf16x8(const uint4& v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

// Large-batch router: a CTA computes a tile of 16 tokens x 32 experts; warp
// (tg, eg) owns 4 tokens x 16 experts and lane l is the lane-slot l of every
// one of those 64 dot products, so each lane adds exactly the products of the
// inputs h with (h/8) mod 32 == l, in increasing h (the fixed order), then the
// butterfly.  The 256-input slabs of activations and router weights both
// sides of the tile need are staged in shared memory (cp.async, two buffers).
constexpr int RT_T = 16, RT_E = 32, RT_SLAB = 256;

__global__ void __launch_bounds__(256) router_logits_tiled_kernel(const uint16_t* __restrict__ x,
                                                                  const uint16_t* __restrict__ w,
                                                                  const float* __restrict__ bias,
                                                                  float* __restrict__ logits, int T, int H,
                                                                  int E) {
    __shared__ __align__(16) uint16_t xs[2][RT_T][RT_SLAB];
    __shared__ __align__(16) uint16_t ws[2][RT_E][RT_SLAB];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int t0 = blockIdx.x * RT_T, e0 = blockIdx.y * RT_E;
    const int tg = warp >> 1, eg = warp & 1;  // 4 token groups x 2 expert groups
    const int nslab = H / RT_SLAB;
    auto issue = [&](int sl) {
        const int buf = sl & 1;
        // (RT_T + RT_E) rows x 32 16-byte chunks = 1536 chunks, 6 per thread
        for (int c = tid; c < (RT_T + RT_E) * 32; c += 256) {
            const int row = c >> 5, col = (c & 31) * 8;
            const uint16_t* src;
            uint32_t dst;
            bool valid;
            if (row < RT_T) {
                valid = t0 + row < T;
                src = x + (size_t)(valid ? t0 + row : 0) * H + sl * RT_SLAB + col;
                dst = smem_u32(&xs[buf][row][col]);
            } else {
                valid = e0 + row - RT_T < E;
                src = w + (size_t)(valid ? e0 + row - RT_T : 0) * H + sl * RT_SLAB + col;
                dst = smem_u32(&ws[buf][row - RT_T][col]);
            }
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
                         : "memory");
        }
        asm volatile("cp.async.commit_group;\n" ::: "memory");
    };
    pdl_wait();
    pdl_launch_dependents();  // dependents may start their prologues now
    // acc2[a][bp] = (dot (a, 2 bp), dot (a, 2 bp + 1)): the packed fp32 pairs
    // round each product and each sum exactly as the scalar operations do,
    // two experts per instruction
    float2 acc2[4][8];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int bp = 0; bp < 8; ++bp) acc2[a][bp] = make_float2(0.0f, 0.0f);
    issue(0);
    for (int sl = 0; sl < nslab; ++sl) {
        if (sl + 1 < nslab) {
            issue(sl + 1);
            asm volatile("cp.async.wait_group 1;\n" ::: "memory");
        } else {
            asm volatile("cp.async.wait_group 0;\n" ::: "memory");
        }
        __syncthreads();
        const int buf = sl & 1;
        float2 xd[4][8];  // each input twice
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            float xf[8];
            unpack_bf16x8(*reinterpret_cast<const uint4*>(&xs[buf][tg * 4 + a][8 * lane]), xf);
#pragma unroll
            for (int i = 0; i < 8; ++i) xd[a][i] = make_float2(xf[i], xf[i]);
        }
#pragma unroll
        for (int bp = 0; bp < 8; ++bp) {
            float w0[8], w1[8];
            unpack_bf16x8(*reinterpret_cast<const uint4*>(&ws[buf][eg * 16 + 2 * bp][8 * lane]), w0);
            unpack_bf16x8(*reinterpret_cast<const uint4*>(&ws[buf][eg * 16 + 2 * bp + 1][8 * lane]), w1);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float2 w2 = make_float2(w0[i], w1[i]);
#pragma unroll
                for (int a = 0; a < 4; ++a) acc2[a][bp] = __fadd2_rn(acc2[a][bp], __fmul2_rn(xd[a][i], w2));
            }
        }
        __syncthreads();
    }
    float acc[4][16];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int bp = 0; bp < 8; ++bp) {
            acc[a][2 * bp] = acc2[a][bp].x;
            acc[a][2 * bp + 1] = acc2[a][bp].y;
        }
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 16; ++b)
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) acc[a][b] = __fadd_rn(acc[a][b], __shfl_xor_sync(FULL, acc[a][b], off));
    // lane l writes entry (a, b) = (l >> 4 .. , l & 15): 2 passes of 32
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 16; ++b) {
            if (lane == ((a & 1) * 16 + b)) {
                const int t = t0 + tg * 4 + a, e = e0 + eg * 16 + b;
                if (t < T && e < E) logits[(size_t)t * E + e] = bias ? __fadd_rn(acc[a][b], bias[e]) : acc[a][b];
            }
        }
}

// Order-preserving 32-bit key of a logit: a larger logit has a larger key,
// and equal logits have equal keys (-0 is keyed as +0); NaN and absent or
// taken entries get key 0, below every other (-inf: 0x007fffff).
__device__ __forceinline__ unsigned logit_key(float v) {
    unsigned u = __float_as_uint(v);
    if (u == 0x80000000u) u = 0u;
    if ((u & 0x7fffffffu) > 0x7f800000u) return 0u;  // NaN
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_logit(unsigned key) {
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

// The k best of a warp's logits in (logit descending, id ascending) order
// -- equal logits go to the lower id: value i of lane l is expert l + 32 i
// (absent ones marked in taken).  Each round takes the warp-wide largest key
// (__reduce_max_sync) and, among the lanes that hold it, the lowest id
// (__reduce_min_sync); only the lane that owned the winner rescans its
// values.  Lane j < k ends with the j-th selected logit and id.
template <int NPER>
__device__ __forceinline__ void warp_select_topk(const float (&v)[NPER], uint32_t taken, int k, float& sel_v,
                                                 int& sel_e) {
    const int lane = threadIdx.x & 31;
    unsigned key[NPER];
#pragma unroll
    for (int i = 0; i < NPER; ++i) key[i] = logit_key(v[i]);
    unsigned bk = 0;
    int be = INT_MAX;
    auto rescan = [&]() {
        bk = 0;
        be = INT_MAX;
#pragma unroll
        for (int i = 0; i < NPER; ++i)
            if (!((taken >> i) & 1) && key[i] > bk) {  // (i increasing: the first of equal keys has the lowest id)
                bk = key[i];
                be = lane + 32 * i;
            }
    };
    rescan();
    unsigned sel_k = 0;
    sel_e = 0;
    for (int j = 0; j < k; ++j) {
        const unsigned mk = __reduce_max_sync(FULL, bk);
        const int we = __reduce_min_sync(FULL, bk == mk ? be : INT_MAX);
        if (lane == j) {
            sel_k = mk;
            sel_e = we;
        }
        if ((we & 31) == lane) {
            taken |= 1u << (we >> 5);
            rescan();
        }
    }
    sel_v = key_logit(sel_k);
}

// Small-batch router: one CTA of 8 warps per (RS_TG tokens, 8 experts); the
// tokens' activations sit in shared memory and each lane first loads all of
// its router-weight chunks, so a warp needs one memory round trip and uses
// each weight for RS_TG tokens.  Every (token, expert) sum keeps the fixed
// order of router_logits_tiled_kernel (the order moe_vq2.h states).
constexpr int RS_TG = 4;

__global__ void __launch_bounds__(256) router_logits_small_kernel(const uint16_t* __restrict__ x,
                                                                  const uint16_t* __restrict__ w,
                                                                  const float* __restrict__ bias,
                                                                  float* __restrict__ logits, int T, int H,
                                                                  int E) {
    extern __shared__ __align__(16) uint4 xs[];
    const int t0 = blockIdx.y * RS_TG, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ntok = min(RS_TG, T - t0);
    const int e = blockIdx.x * 8 + warp;
    const int nch = H / 8;
    const int per = H / 256;  // chunks per lane
    constexpr int U = 16;
    // the router weights do not depend on earlier kernels, and the activations
    // are complete at launch (no library kernel still running writes them):
    // both are fetched before waiting on the predecessor
    const uint4* wr = reinterpret_cast<const uint4*>(w + (size_t)min(e, E - 1) * H);
    uint4 wv[U];
#pragma unroll
    for (int u = 0; u < U; ++u)
        if (u < per) wv[u] = __ldg(wr + lane + 32 * u);
    for (int i = threadIdx.x; i < ntok * nch; i += blockDim.x)
        xs[i] = reinterpret_cast<const uint4*>(x + (size_t)t0 * H)[i];
    pdl_wait();
    pdl_launch_dependents();  // dependents may start their prologues now
    __syncthreads();
    if (e >= E) return;
    float acc[RS_TG];
#pragma unroll
    for (int tt = 0; tt < RS_TG; ++tt) acc[tt] = 0.0f;
    for (int m0 = 0; m0 < per; m0 += U) {
        if (m0 > 0) {
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (m0 + u < per) wv[u] = __ldg(wr + lane + 32 * (m0 + u));
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (m0 + u < per) {
                float wf[8];
                unpack_bf16x8(wv[u], wf);
#pragma unroll
                for (int tt = 0; tt < RS_TG; ++tt) {
                    if (tt < ntok) {
                        float xf[8];
                        unpack_bf16x8(xs[tt * nch + lane + 32 * (m0 + u)], xf);
#pragma unroll
                        for (int i = 0; i < 8; ++i) acc[tt] = __fadd_rn(acc[tt], __fmul_rn(xf[i], wf[i]));
                    }
                }
            }
        }
    }
#pragma unroll
    for (int tt = 0; tt < RS_TG; ++tt) {
        if (tt < ntok) {
            float a = acc[tt];
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) a = __fadd_rn(a, __shfl_xor_sync(FULL, a, off));
            if (lane == 0) logits[(size_t)(t0 + tt) * E + e] = bias ? __fadd_rn(a, bias[e]) : a;
        }
    }
}

// One warp per token: lane l holds logits l, l+32, ...; each lane keeps its
// best not-yet-taken (logit desc, id asc); k rounds of a warp-wide arg-max,
// after which only the lane that owned the winner rescans its values.
template <int NPER>
__global__ void __launch_bounds__(256) route_topk_kernel(const float* __restrict__ logits, int T, int E,
                                                         int k, int renorm, int32_t* __restrict__ ids,
                                                         float* __restrict__ weights) {
    pdl_wait();
    pdl_launch_dependents();  // dependents may start their prologues now
    const int lane = threadIdx.x & 31;
    const long t = ((long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (t >= T) return;
    const float* l = logits + (size_t)t * E;
    float v[NPER];
    uint32_t taken = 0;
#pragma unroll
    for (int i = 0; i < NPER; ++i) {
        const int e = lane + 32 * i;
        if (e < E)
            v[i] = l[e];
        else {
            v[i] = -INFINITY;
            taken |= 1u << i;
        }
    }
    float sel_v;  // lane j keeps the j-th selected logit and its id
    int sel_e;
    warp_select_topk<NPER>(v, taken, k, sel_v, sel_e);
    const float top = __shfl_sync(FULL, sel_v, 0);
    const float num = lane < k ? expf(sel_v - top) : 0.0f;
    float den = 0.0f;
    if (renorm) {
        den = num;
    } else {
#pragma unroll
        for (int i = 0; i < NPER; ++i)
            if (lane + 32 * i < E) den += expf(v[i] - top);
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) den += __shfl_xor_sync(FULL, den, off);
    if (lane < k) {
        ids[(size_t)t * k + lane] = sel_e;
        weights[(size_t)t * k + lane] = num / den;
    }
}


// Routing of one token by warp 0 of a CTA: top-k of the E logits (read
// through logit_of), softmax weights, and -- the k ids being distinct -- the
// sorted order of the k pairs from the ranks of the ids (offsets[e] = number
// of ids below e).  Bit for bit what route_topk_kernel and permute_kernel give.
template <int NPER, typename LogitOf>
__device__ __forceinline__ void route_one_token(LogitOf logit_of, int E, int k, int renorm, int32_t* __restrict__ ids,
                                                float* __restrict__ weights, int32_t* __restrict__ offsets,
                                                int32_t* __restrict__ sorted_pair,
                                                int32_t* __restrict__ pair_to_sorted) {
    const int lane = threadIdx.x & 31;
    float v[NPER];
    uint32_t taken = 0;
#pragma unroll
    for (int i = 0; i < NPER; ++i) {
        const int ee = lane + 32 * i;
        if (ee < E) {
            v[i] = logit_of(ee);
        } else {
            v[i] = -INFINITY;
            taken |= 1u << i;
        }
    }
    float sel_v;  // lane j keeps the j-th selected logit and its id
    int sel_e;
    warp_select_topk<NPER>(v, taken, k, sel_v, sel_e);
    const float top = __shfl_sync(FULL, sel_v, 0);
    const float num = lane < k ? expf(sel_v - top) : 0.0f;
    float den = 0.0f;
    if (renorm) {
        den = num;
    } else {
#pragma unroll
        for (int i = 0; i < NPER; ++i)
            if (lane + 32 * i < E) den += expf(v[i] - top);
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) den += __shfl_xor_sync(FULL, den, off);
    // the k ids are distinct: rank of pair j = #ids below id_j; per e,
    // offsets[e] = #ids below e
    int rank = 0;
    int cnt[NPER];
#pragma unroll
    for (int i = 0; i < NPER; ++i) cnt[i] = 0;
    for (int j = 0; j < k; ++j) {
        const int idj = __shfl_sync(FULL, sel_e, j);
        rank += idj < sel_e;
#pragma unroll
        for (int i = 0; i < NPER; ++i) cnt[i] += idj < lane + 32 * i;
    }
    if (lane < k) {
        ids[lane] = sel_e;
        weights[lane] = num / den;
        sorted_pair[rank] = lane;
        pair_to_sorted[lane] = rank;
    }
#pragma unroll
    for (int i = 0; i < NPER; ++i)
        if (lane + 32 * i < E) offsets[lane + 32 * i] = cnt[i];
    if (lane == 0) offsets[E] = k;
}

// Whole routing of a small batch in one launch (the three steps above,
// bit for bit): CTA (e8, t) computes the logits of token t for 8 experts as
// router_logits_small_kernel does; the CTA that finishes last (a counter in
// the caller's workspace, back at zero afterwards) then runs the top-k +
// softmax of every token (route_topk_kernel's rounds, one warp per token) and
// the stable counting sort of the pairs by expert (moe_permute's order) on
// its 256 threads.  Shared memory: the token's activations, then ids[P],
// cursor[E] and per-warp counts wcnt[8][E].
template <int NPER>
__global__ void __launch_bounds__(256) route_fused_kernel(const uint16_t* __restrict__ x,
                                                          const uint16_t* __restrict__ w,
                                                          const float* __restrict__ bias, int T, int H, int E,
                                                          int k, int renorm, float* __restrict__ logits,
                                                          int32_t* __restrict__ ids, float* __restrict__ weights,
                                                          int32_t* __restrict__ offsets,
                                                          int32_t* __restrict__ sorted_pair,
                                                          int32_t* __restrict__ pair_to_sorted,
                                                          int* __restrict__ counter) {
    extern __shared__ __align__(16) uint4 xs[];
    __shared__ int s_last;
    const int t = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int e = blockIdx.x * 8 + warp;
    const int nch = H / 8;
    const int per = H / 256;
    constexpr int U = 16;
    const uint4* wr = reinterpret_cast<const uint4*>(w + (size_t)min(e, E - 1) * H);
    uint4 wv[U];
#pragma unroll
    for (int u = 0; u < U; ++u)
        if (u < per) wv[u] = __ldg(wr + lane + 32 * u);
    // The activations are complete at launch (no library kernel still running
    // writes them), so the logits are computed before the wait too: only the
    // global writes wait for the kernels before this one.
    for (int i = tid; i < nch; i += blockDim.x) xs[i] = reinterpret_cast<const uint4*>(x + (size_t)t * H)[i];
    pdl_launch_dependents();  // dependents may start their prologues now
    __syncthreads();
    float acc = 0.0f;
    if (e < E) {
        for (int m0 = 0; m0 < per; m0 += U) {
            if (m0 > 0) {
#pragma unroll
                for (int u = 0; u < U; ++u)
                    if (m0 + u < per) wv[u] = __ldg(wr + lane + 32 * (m0 + u));
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (m0 + u < per) {
                    float xf[8], wf[8];
                    unpack_bf16x8(xs[lane + 32 * (m0 + u)], xf);
                    unpack_bf16x8(wv[u], wf);
#pragma unroll
                    for (int i = 0; i < 8; ++i) acc = __fadd_rn(acc, __fmul_rn(xf[i], wf[i]));
                }
            }
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(FULL, acc, off));
    }
    pdl_wait();
    if (e < E && lane == 0) logits[(size_t)t * E + e] = bias ? __fadd_rn(acc, bias[e]) : acc;
    // the last CTA to finish goes on (thread 0's fence, after the barrier,
    // orders the whole CTA's logits before its arrival)
    __syncthreads();
    if (tid == 0) {
        const int n = gridDim.x * gridDim.y;
        __threadfence();
        const bool last = atomicAdd(counter, 1) == n - 1;
        if (last) {
            *counter = 0;
            __threadfence();
        }
        s_last = last;
    }
    __syncthreads();
    if (!s_last) return;

    if (T == 1) {
        // one token: warp 0 alone (no block barriers)
        if (warp != 0) return;
        route_one_token<NPER>([&](int ee) { return __ldcg(logits + ee); }, E, k, renorm, ids, weights, offsets,
                              sorted_pair, pair_to_sorted);
        return;
    }

    const int P = T * k;
    int32_t* s_ids = reinterpret_cast<int32_t*>(xs);  // (the activations are done with)
    int32_t* cursor = s_ids + P;
    int32_t* wcnt = cursor + E;
    // top-k + softmax, one warp per token
    for (int tt = warp; tt < T; tt += 8) {
        const float* l = logits + (size_t)tt * E;
        float v[NPER];
        uint32_t taken = 0;
#pragma unroll
        for (int i = 0; i < NPER; ++i) {
            const int ee = lane + 32 * i;
            if (ee < E) {
                v[i] = __ldcg(l + ee);
            } else {
                v[i] = -INFINITY;
                taken |= 1u << i;
            }
        }
        float sel_v;  // lane j keeps the j-th selected logit and its id
        int sel_e;
        warp_select_topk<NPER>(v, taken, k, sel_v, sel_e);
        const float top = __shfl_sync(FULL, sel_v, 0);
        const float num = lane < k ? expf(sel_v - top) : 0.0f;
        float den = 0.0f;
        if (renorm) {
            den = num;
        } else {
#pragma unroll
            for (int i = 0; i < NPER; ++i)
                if (lane + 32 * i < E) den += expf(v[i] - top);
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) den += __shfl_xor_sync(FULL, den, off);
        if (lane < k) {
            ids[(size_t)tt * k + lane] = sel_e;
            weights[(size_t)tt * k + lane] = num / den;
            s_ids[tt * k + lane] = sel_e;
        }
    }
    for (int i = tid; i < E * 9; i += blockDim.x) cursor[i] = 0;  // cursor and wcnt
    __syncthreads();
    // histogram, exclusive scan (4 entries per thread), stable scatter
    for (int p = tid; p < P; p += blockDim.x) atomicAdd(&cursor[s_ids[p]], 1);
    __syncthreads();
    __shared__ int warp_tot[8];
    int c4[4], run = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int ee = 4 * tid + q;
        c4[q] = ee < E ? cursor[ee] : 0;
        run += c4[q];
    }
    int incl = run;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(FULL, incl, off);
        if (lane >= off) incl += o;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    int before = 0;
    for (int w2 = 0; w2 < warp; ++w2) before += warp_tot[w2];
    int ex = incl - run + before;
    __syncthreads();
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int ee = 4 * tid + q;
        if (ee < E) {
            offsets[ee] = ex;
            cursor[ee] = ex;
        }
        ex += c4[q];
    }
    if (tid == 0) offsets[E] = P;
    __syncthreads();
    const unsigned lt = (1u << lane) - 1u;
    for (int base0 = 0; base0 < P; base0 += 256) {
        const int p = base0 + tid;
        const bool valid = p < P;
        const int ee = valid ? s_ids[p] : -1;
        const unsigned peers = __match_any_sync(FULL, ee);
        const int rank = __popc(peers & lt);
        const bool leader = (__ffs(peers) - 1) == lane;
        if (valid && leader) wcnt[warp * E + ee] = __popc(peers);
        __syncthreads();
        if (valid) {
            int pre = 0;
            for (int w2 = 0; w2 < warp; ++w2) pre += wcnt[w2 * E + ee];
            const int pos = cursor[ee] + pre + rank;
            sorted_pair[pos] = p;
            pair_to_sorted[p] = pos;
        }
        __syncthreads();
        if (valid && leader) {  // (leaders of several warps may share an expert)
            atomicAdd(&cursor[ee], __popc(peers));
            wcnt[warp * E + ee] = 0;
        }
        __syncthreads();
    }
}

// One token over a thread-block cluster: CTA r of the cluster computes the
// logits of experts e = 16 r + warp + 16 C i (C CTAs; one expert per warp at
// a time, as router_logits_small_kernel does), writes them to logits (the
// call's output) and into the shared memory of CTA 0; the cluster barrier
// publishes them, and warp 0 of CTA 0 routes the token from shared memory (no
// global counter, fence or read-back of the logits).
constexpr int RC_WARPS = 16;

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void st_cta0_f32(uint32_t local_addr, float v) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, 0;" : "=r"(remote) : "r"(local_addr));
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(v) : "memory");
}
__device__ __forceinline__ void cluster_barrier() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

template <int NPER>
__global__ void __launch_bounds__(32 * RC_WARPS) route_cluster_kernel(const uint16_t* __restrict__ x,
                                                                      const uint16_t* __restrict__ w,
                                                                      const float* __restrict__ bias, int H, int E,
                                                                      int k, int renorm, float* __restrict__ logits,
                                                                      int32_t* __restrict__ ids,
                                                                      float* __restrict__ weights,
                                                                      int32_t* __restrict__ offsets,
                                                                      int32_t* __restrict__ sorted_pair,
                                                                      int32_t* __restrict__ pair_to_sorted) {
    extern __shared__ __align__(16) uint4 xs[];
    __shared__ float lg[1024];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nch = H / 8;
    const int per = H / 256;
    const int stride = gridDim.x * RC_WARPS;
    constexpr int U = 16;
    int e = blockIdx.x * RC_WARPS + warp;
    uint4 wv[U];
    auto load_w = [&](int ee, int m0) {
        const uint4* wr = reinterpret_cast<const uint4*>(w + (size_t)min(ee, E - 1) * H);
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (m0 + u < per) wv[u] = __ldg(wr + lane + 32 * (m0 + u));
    };
    load_w(e, 0);
    // The activations are complete at launch (no library kernel still running
    // writes them), so the logits are computed and gathered in CTA 0's shared
    // memory before the wait: only the global writes (CTA 0's, after the
    // cluster barrier) wait for the kernels before this one.
    for (int i = tid; i < nch; i += blockDim.x) xs[i] = reinterpret_cast<const uint4*>(x)[i];
    pdl_launch_dependents();  // dependents may start their prologues now
    __syncthreads();
    for (; e < E; e += stride) {
        float acc = 0.0f;
        for (int m0 = 0; m0 < per; m0 += U) {
            if (m0 > 0) load_w(e, m0);
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (m0 + u < per) {
                    float xf[8], wf[8];
                    unpack_bf16x8(xs[lane + 32 * (m0 + u)], xf);
                    unpack_bf16x8(wv[u], wf);
#pragma unroll
                    for (int i = 0; i < 8; ++i) acc = __fadd_rn(acc, __fmul_rn(xf[i], wf[i]));
                }
            }
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(FULL, acc, off));
        if (lane == 0) st_cta0_f32((uint32_t)__cvta_generic_to_shared(&lg[e]), bias ? __fadd_rn(acc, bias[e]) : acc);
        if (e + stride < E) load_w(e + stride, 0);
    }
    cluster_barrier();  // every CTA's logits are in CTA 0's shared memory
    if (cluster_rank() != 0 || warp != 0) return;
    pdl_wait();
    for (int i = lane; i < E; i += 32) logits[i] = lg[i];
    route_one_token<NPER>([&](int ee) { return lg[ee]; }, E, k, renorm, ids, weights, offsets, sorted_pair,
                          pair_to_sorted);
}

}  // namespace

moe_status launch_router_logits(const uint16_t* x, const uint16_t* w, const float* bias, float* logits,
                                int T, int H, int E, cudaStream_t s) {
    const int threads = 256;
    const size_t xs_bytes = (size_t)H * 2 * RS_TG;
    if (T <= 64 && xs_bytes <= 48 * 1024) {
        dim3 grid((unsigned)((E + 7) / 8), (unsigned)((T + RS_TG - 1) / RS_TG));
        cudaError_t e = launch_pdl(router_logits_small_kernel, grid, dim3(threads), xs_bytes, s, x, w, bias, logits, T,
                                   H, E);
        if (e != cudaSuccess) return cuda_status(e, "moe_router_logits: launch");
    } else {
        dim3 grid((unsigned)((T + RT_T - 1) / RT_T), (unsigned)((E + RT_E - 1) / RT_E));
        cudaError_t e = launch_pdl(router_logits_tiled_kernel, grid, dim3(threads), 0, s, x, w, bias, logits, T, H, E);
        if (e != cudaSuccess) return cuda_status(e, "moe_router_logits: launch");
    }
    MOE_LAUNCH_CHECK("moe_router_logits: launch");
    return MOE_OK;
}

moe_status launch_route_topk(const float* logits, int T, int E, int k, int renorm, int32_t* ids,
                             float* weights, cudaStream_t s) {
    const int threads = 256;
    const unsigned blocks = (unsigned)(((long)T * 32 + threads - 1) / threads);
    auto kern = E <= 32    ? route_topk_kernel<1>
                : E <= 64  ? route_topk_kernel<2>
                : E <= 128 ? route_topk_kernel<4>
                : E <= 256 ? route_topk_kernel<8>
                : E <= 512 ? route_topk_kernel<16>
                           : route_topk_kernel<32>;
    cudaError_t e = launch_pdl(kern, dim3(blocks), dim3(threads), 0, s, logits, T, E, k, renorm, ids, weights);
    if (e != cudaSuccess) return cuda_status(e, "moe_route_topk: launch");
    MOE_LAUNCH_CHECK("moe_route_topk: launch");
    return MOE_OK;
}

size_t route_fused_smem(int T, int k, int H, int E) {
    const size_t act = (size_t)H * 2;
    const size_t tail = sizeof(int32_t) * ((size_t)T * k + (size_t)E * 9);
    return act > tail ? act : tail;
}

bool route_fused_ok(int T, int k, int H, int E) {
    // (one fused kernel is faster than the three steps up to about 8 tokens; the
    // logits of larger batches spread over more CTAs than the counter handshake
    // pays for)
    return T >= 1 && T <= 8 && (long long)T * k <= 1024 && E <= 1024 && route_fused_smem(T, k, H, E) <= 48 * 1024;
}

moe_status launch_route_fused(const uint16_t* x, const uint16_t* w, const float* bias, int T, int H, int E, int k,
                              int renorm, float* logits, int32_t* ids, float* weights, int32_t* offsets,
                              int32_t* sorted_pair, int32_t* pair_to_sorted, int* counter, cudaStream_t s) {
    auto kern = E <= 32    ? route_fused_kernel<1>
                : E <= 64  ? route_fused_kernel<2>
                : E <= 128 ? route_fused_kernel<4>
                : E <= 256 ? route_fused_kernel<8>
                : E <= 512 ? route_fused_kernel<16>
                           : route_fused_kernel<32>;
    dim3 grid((unsigned)((E + 7) / 8), (unsigned)T);
    cudaError_t e = launch_pdl(kern, grid, dim3(256), route_fused_smem(T, k, H, E), s, x, w, bias, T, H, E, k, renorm,
                               logits, ids, weights, offsets, sorted_pair, pair_to_sorted, counter);
    if (e != cudaSuccess) return cuda_status(e, "moe_route: launch");
    MOE_LAUNCH_CHECK("moe_route: launch");
    return MOE_OK;
}


// Allows a kernel's clusters above the portable size once per (kernel,
// device), so that calls inside a stream capture make no attribute call.
template <typename F>
static cudaError_t ensure_cluster_attr(F* kern) {
    constexpr int kMaxDev = 64;
    static const void* done[8][kMaxDev];
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDev) return cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    int slot = -1;
    for (int i = 0; i < 8; ++i) {
        if (done[i][dev] == (const void*)kern) return cudaSuccess;
        if (slot < 0 && done[i][dev] == nullptr) slot = i;
    }
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e == cudaSuccess && slot >= 0) done[slot][dev] = (const void*)kern;
    return e;
}

// CTAs of the one-token cluster: 16 where the device can run clusters of that
// size, else 8, else 0 (no cluster routing).  Checked once per device; the
// first call of a process is expected outside stream capture.
static int route_cluster_size() {
    constexpr int kMaxDev = 64;
    static int cached[kMaxDev];
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 0;
    if (cached[dev] != 0) return cached[dev] > 0 ? cached[dev] : 0;
    int found = -1;
    auto kern = route_cluster_kernel<8>;
    for (int cl : {16, 8}) {
        if (cl > 8 && ensure_cluster_attr(kern) != cudaSuccess) {
            cudaGetLastError();
            continue;
        }
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)cl);
        cfg.blockDim = dim3(32 * RC_WARPS);
        cfg.dynamicSmemBytes = 8192;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)cl;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) == cudaSuccess && n >= 1) {
            found = cl;
            break;
        }
        cudaGetLastError();
    }
    cached[dev] = found;
    return found > 0 ? found : 0;
}

bool route_cluster_ok(int T, int H, int E) {
    return T == 1 && E <= 1024 && (size_t)H * 2 <= 48 * 1024 && route_cluster_size() > 0;
}

moe_status launch_route_cluster(const uint16_t* x, const uint16_t* w, const float* bias, int H, int E, int k,
                                int renorm, float* logits, int32_t* ids, float* weights, int32_t* offsets,
                                int32_t* sorted_pair, int32_t* pair_to_sorted, cudaStream_t s) {
    auto kern = E <= 32    ? route_cluster_kernel<1>
                : E <= 64  ? route_cluster_kernel<2>
                : E <= 128 ? route_cluster_kernel<4>
                : E <= 256 ? route_cluster_kernel<8>
                : E <= 512 ? route_cluster_kernel<16>
                           : route_cluster_kernel<32>;
    const int cl = route_cluster_size();
    if (cl > 8) {
        cudaError_t e = ensure_cluster_attr(kern);
        if (e != cudaSuccess) return cuda_status(e, "moe_route: cluster attribute");
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)cl);
    cfg.blockDim = dim3(32 * RC_WARPS);
    cfg.dynamicSmemBytes = (size_t)H * 2;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cl;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    count_launch();
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, x, w, bias, H, E, k, renorm, logits, ids, weights, offsets,
                                       sorted_pair, pair_to_sorted);
    if (e != cudaSuccess) return cuda_status(e, "moe_route: cluster launch");
    MOE_LAUNCH_CHECK("moe_route: cluster launch");
    return MOE_OK;
}

}  // namespace moe
