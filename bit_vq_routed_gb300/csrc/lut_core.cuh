// The activation-table core shared by the table kernels: the table layout
// in shared memory, the table build, the unit copy into a warp's code slot
// and the per-unit lookups with their warp reduction.
//
// For one token, every code byte c of group G (inputs 4G .. 4G+3) adds
//     scale[r, G/32] * sign(c) * dot(codebook[c & 127], x[4G .. 4G+3])
// to output row r, and the signed dot product depends on (c, G) only.  A CTA
// builds the table L[c][G] of those values for a K-range of 1024 inputs
// (256 codes x 256 groups in fp16, 128 KB; the negated half is stored too, so
// the sign costs nothing), then streams code tiles of many rows through it:
// per code byte one byte permute (the table address), one 2-byte shared load
// and one mixed-precision add of the fp16 entry into an fp32 sum.
//
// Lanes own groups: lane l takes, in scale block b = lane_block(l) of the
// K-range, the 8 groups m, m+4, ..., m+28 with m = l & 3 (one 16-byte load
// each, so each load instruction of the warp reads whole 64-byte runs), and
// its 8 values of a row share one scale.  The table puts every entry a lane
// reads in bank l, whatever the code, so the 32 table reads of a warp never
// conflict, and the group slot becomes the load's immediate offset.  The 16
// row sums of a tile are reduced across the warp by a reduce-scatter.
//
// A unit is 16 rows x 1024 inputs (8 packed tiles: 4 KB of codes, 256 B of
// scales), copied into a warp's slot by three bulk copies.
//
// FP4 (MXFP4) experts use the same table shape with the code byte's two e2m1
// values in place of the codebook row: a byte of group G holds elements 2G
// and 2G + 1, so a table covers 512 inputs, a packed e2m1 tile (16 rows x 64)
// is 512 bytes with the lane ownership of a VQ2 tile, and each row sums its
// two 32-element blocks separately for their ue8m0 scales.
#pragma once

#include "ffn_common.cuh"

namespace moe {
namespace lut {

constexpr int LW = 16;                     // warps of a table-kernel CTA
constexpr int THREADS = 32 * LW;
constexpr int KR_IN = 128 * LUT_KB;        // inputs per K-range: 32 lanes x 8 groups x 4
constexpr uint32_t TAB = 0x10000;          // table: [0x10000, 0x30000) of the shared window
constexpr uint32_t PLANE = 0x10000;        // group slots 0-3 | 4-7
constexpr uint32_t TAB_END = TAB + 2 * PLANE;
constexpr uint32_t DYN_SMEM = 227 * 1024;  // dynamic shared memory requested (the maximum)
// One code slot: tiles 0-3 of the unit (2 KB), tiles 4-7 after 64 bytes of
// skew, then the 8 tiles' row scales (32 bytes each).  The lanes of a
// quarter-warp take scale blocks b and b + 4, so their 16-byte reads of one
// group slot hit 8 distinct bank groups.
constexpr uint32_t HALF_OFF = 4 * 512 + 64;
constexpr uint32_t SCALE_OFF = HALF_OFF + 4 * 512;
constexpr uint32_t SLOT_BYTES = SCALE_OFF + 8 * 32;

// scale block of lane l (the 4 lanes 4q .. 4q+3 share one): blocks b and b + 4
// for the two lane quads of each quarter-warp
__host__ __device__ constexpr int lane_block(int l) { return (((l >> 2) & 1) << 2) | (l >> 3); }

// Inputs of the K-range in shared memory: float i at xs_at(i), a float4 of
// padding after every 32 groups (one scale block), so the table build's
// 16-byte reads of one group in each of the 8 blocks spread over all banks.
__device__ __forceinline__ int xs_at(int i) { return i + 4 * (i >> 7); }
constexpr int XS_FLOATS = KR_IN + KR_IN / 32;

// Register cap: each of the SM's four schedulers holds 16384 registers for
// its share of the CTA's warps (ceil(LW / 4) warps).
constexpr int MAX_REG = 16384 / (32 * ((LW + 3) / 4)) > 255 ? 255 : 16384 / (32 * ((LW + 3) / 4)) / 8 * 8;

// Table entry of lane l, group slot j, code c sits at shared-window byte
//     TAB + (j/4)*PLANE + c*256 + 128*((j/2)&1) + 4*l + 2*(j&1):
// the code fills bits 8-15 (one byte permute), the slot is an immediate.
template <int J>
__device__ __forceinline__ float tab_add(uint32_t addr, float t) {
    constexpr int IMM = (J >> 2) * (int)PLANE + 128 * ((J >> 1) & 1) + 2 * (J & 1);
    uint16_t v;
    asm volatile("ld.shared.b16 %0, [%1+%2];" : "=h"(v) : "r"(addr), "n"(IMM));
    float d;
    asm("add.rn.f32.f16 %0, %1, %2;" : "=f"(d) : "h"(v), "f"(t));
    return d;
}

template <uint32_t SEL>
__device__ __forceinline__ uint32_t prmt_i(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "n"(SEL));
    return d;
}

struct UnitRegs {
    uint4 cw[8];  // group slot j: the 16 code bytes (rows) of group 4j + m
    uint4 sc[2];  // the 16 row scales of this lane's scale block
};

// Sum over the lane's 8 groups of row byte RB (row (RB >> 1) + 8 (RB & 1)).
template <int RB>
__device__ __forceinline__ float row_sum(const UnitRegs& u, uint32_t lb) {
    constexpr uint32_t SEL = 0x7604u | ((uint32_t)(RB & 3) << 4);
    float t = 0.0f;
    t = tab_add<0>(prmt_i<SEL>((&u.cw[0].x)[RB >> 2], lb), t);
    t = tab_add<1>(prmt_i<SEL>((&u.cw[1].x)[RB >> 2], lb), t);
    t = tab_add<2>(prmt_i<SEL>((&u.cw[2].x)[RB >> 2], lb), t);
    t = tab_add<3>(prmt_i<SEL>((&u.cw[3].x)[RB >> 2], lb), t);
    t = tab_add<4>(prmt_i<SEL>((&u.cw[4].x)[RB >> 2], lb), t);
    t = tab_add<5>(prmt_i<SEL>((&u.cw[5].x)[RB >> 2], lb), t);
    t = tab_add<6>(prmt_i<SEL>((&u.cw[6].x)[RB >> 2], lb), t);
    t = tab_add<7>(prmt_i<SEL>((&u.cw[7].x)[RB >> 2], lb), t);
    constexpr int ROW = (RB >> 1) + 8 * (RB & 1);
    const uint32_t s2 = (&u.sc[ROW >> 3].x)[(ROW & 7) >> 1];
    const __half2 h = *reinterpret_cast<const __half2*>(&s2);
    return t * ((ROW & 1) ? __high2float(h) : __low2float(h));
}

// The same sum for packed e2m1 tiles (FP4 experts): a tile is 16 rows x 64
// elements, and the lane's chunk i (16 bytes) holds rows i and i + 8 for its
// 8 groups of 2 elements: byte 4s + 2h + u is row i + 8h, group slot 2s + u.
// Slots 0-3 and 4-7 lie in the tile's two 32-element scale blocks: each part
// is multiplied by its ue8m0 scale (sc[0], sc[1]: one byte per row).
template <int RB>
__device__ __forceinline__ float row_sum_f4(const UnitRegs& u, uint32_t lb) {
    constexpr int ROW = (RB >> 1) + 8 * (RB & 1);
    constexpr int I = ROW & 7, H = ROW >> 3;
    const uint32_t* w = &u.cw[I].x;
    float t0 = 0.0f, t1 = 0.0f;
    t0 = tab_add<0>(prmt_i<0x7604u | ((2 * H) << 4)>(w[0], lb), t0);
    t0 = tab_add<1>(prmt_i<0x7604u | ((2 * H + 1) << 4)>(w[0], lb), t0);
    t0 = tab_add<2>(prmt_i<0x7604u | ((2 * H) << 4)>(w[1], lb), t0);
    t0 = tab_add<3>(prmt_i<0x7604u | ((2 * H + 1) << 4)>(w[1], lb), t0);
    t1 = tab_add<4>(prmt_i<0x7604u | ((2 * H) << 4)>(w[2], lb), t1);
    t1 = tab_add<5>(prmt_i<0x7604u | ((2 * H + 1) << 4)>(w[2], lb), t1);
    t1 = tab_add<6>(prmt_i<0x7604u | ((2 * H) << 4)>(w[3], lb), t1);
    t1 = tab_add<7>(prmt_i<0x7604u | ((2 * H + 1) << 4)>(w[3], lb), t1);
    // ue8m0 byte e -> 2^(e - 127): the byte moved to bits 16-23 (one byte
    // permute), shifted to the exponent field; e = 0 gives 0x400000, the
    // subnormal 2^-127
    constexpr uint32_t SSEL = 0x4044u | (uint32_t)((ROW & 3) << 8);
    const uint32_t b0 = prmt_i<SSEL>((&u.sc[0].x)[ROW >> 2], 0u) << 7;
    const uint32_t b1 = prmt_i<SSEL>((&u.sc[1].x)[ROW >> 2], 0u) << 7;
    const float s0 = __uint_as_float(max(b0, 0x400000u)), s1 = __uint_as_float(max(b1, 0x400000u));
    return fmaf(t1, s1, t0 * s0);
}

// The 16 row sums of a unit, reduced over the warp by a reduce-scatter: lanes
// 2p and 2p+1 end with the sum of row unit_row(lane).  Its first step (lanes
// 16 apart) runs as each pair of row sums (i, i + 8) is ready, so only 8 sums
// stay live.  Inactive lanes (scale block beyond the K-range) add zeros.
template <bool F4 = false>
__device__ __forceinline__ float unit_rows(const UnitRegs& r, uint32_t lb, bool active, int lane) {
    float acc[8];
    const bool up16 = lane & 16;
#define MOE_LUT_PAIR(I)                                                                  \
    {                                                                                    \
        const float lo = active ? (F4 ? row_sum_f4<I>(r, lb) : row_sum<I>(r, lb)) : 0.0f;              \
        const float hi = active ? (F4 ? row_sum_f4<I + 8>(r, lb) : row_sum<I + 8>(r, lb)) : 0.0f;      \
        acc[I] = (up16 ? hi : lo) + __shfl_xor_sync(0xffffffffu, up16 ? lo : hi, 16);   \
    }
    MOE_LUT_PAIR(0)
    MOE_LUT_PAIR(1)
    MOE_LUT_PAIR(2)
    MOE_LUT_PAIR(3)
    MOE_LUT_PAIR(4)
    MOE_LUT_PAIR(5)
    MOE_LUT_PAIR(6)
    MOE_LUT_PAIR(7)
#undef MOE_LUT_PAIR
#pragma unroll
    for (int o = 8, n8 = 4; o >= 2; o >>= 1, n8 >>= 1) {
        const bool upo = lane & o;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (i < n8) {
                const float send = upo ? acc[i] : acc[i + n8];
                const float keep = upo ? acc[i + n8] : acc[i];
                acc[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
            }
        }
    }
    return acc[0] + __shfl_xor_sync(0xffffffffu, acc[0], 1);
}
// The row of the unit whose sum unit_rows leaves in this lane.
__device__ __forceinline__ int unit_row(int lane) {
    const int pp = lane >> 1;
    return (pp >> 1) + 8 * (pp & 1);
}

// The table's power-of-two scale.  Every entry |dot(cb[c], x_G)| is at most
// m = max |x| over the K-range times the largest L1 norm of a codebook row;
// the table holds fp16(entry / s) with s = 2^e, m / s <= 2^15 (e clamped to
// [-120, 120]), and each unit's sums are multiplied back by s.  Both scalings
// are exact, so the fp16 entries cannot overflow whatever the range of the
// inputs, and for inputs in the normal range the results equal those of
// unscaled entries bit for bit.  Block-wide (every thread calls it, after the
// inputs are in xs); red: 2 * LW words of shared scratch, which the caller
// must not pass to another call before a CTA barrier.  Returns e.
// cb == nullptr: e2m1 byte tables, whose entries are at most 6 + 6 = 12 times
// max |x|.
__device__ __forceinline__ int table_exponent(const float* xs, int nin, const float* cb, unsigned* red, int tid) {
    float xm = 0.0f, c1 = 0.0f;
    for (int i = tid; i < nin; i += THREADS) xm = fmaxf(xm, fabsf(xs[xs_at(i)]));
    if (tid < 128)
        c1 = cb ? fabsf(cb[4 * tid]) + fabsf(cb[4 * tid + 1]) + fabsf(cb[4 * tid + 2]) + fabsf(cb[4 * tid + 3]) : 12.0f;
    // non-negative floats order as their bit patterns
    const unsigned ux = __reduce_max_sync(0xffffffffu, __float_as_uint(xm));
    const unsigned uc = __reduce_max_sync(0xffffffffu, __float_as_uint(c1));
    if ((tid & 31) == 0) {
        red[tid >> 5] = ux;
        red[LW + (tid >> 5)] = uc;
    }
    __syncthreads();
    unsigned mx = 0, mc = 0;
    for (int w = 0; w < LW; ++w) {
        mx = max(mx, red[w]);
        mc = max(mc, red[LW + w]);
    }
    int ex = 0, ec = 0;
    frexpf(__uint_as_float(mx), &ex);  // max |x| < 2^ex
    frexpf(__uint_as_float(mc), &ec);
    return min(max(ex + ec - 15, -120), 120);
}
__device__ __forceinline__ float exp2_int(int e) { return __int_as_float((e + 127) << 23); }  // 2^e, |e| <= 126

// Table of one K-range from xs (inputs at xs_at, fp32) and cb (the fp32
// codebook, [128][4]), its entries divided by 2^e (table_exponent): a thread
// takes a quad of words (the 4 lanes 4 lq .. 4 lq + 3 of scale block bq, in
// group-slot pair (j0, j0 + 1), j0 = 4p + 2jj: the 8 consecutive groups
// 32 bq + 4 j0 + 0..7) and every LW-th code.  nkb: scale blocks (x 128
// inputs) in the K-range.
__device__ __forceinline__ void build_table(const float* xs, const float* cb, int nkb, int e, int tid) {
    const int warp = tid >> 5;
    const int q = tid & 31, lq = q & 7, jj = (q >> 3) & 1, p = q >> 4, bq = lane_block(4 * lq);
    if (bq >= nkb) return;
    const int g0 = 32 * bq + 4 * (4 * p + 2 * jj);
    // xp[m][i] = (x[4(g0+m)+i], x[4(g0+4+m)+i]): the low / high half of word m
    float2 xp[4][4];
    const float inv = exp2_int(-e);
#pragma unroll
    for (int mm = 0; mm < 4; ++mm) {
        const float4 lo = *reinterpret_cast<const float4*>(&xs[xs_at(4 * (g0 + mm))]);
        const float4 hi = *reinterpret_cast<const float4*>(&xs[xs_at(4 * (g0 + 4 + mm))]);
        xp[mm][0] = make_float2(lo.x * inv, hi.x * inv);
        xp[mm][1] = make_float2(lo.y * inv, hi.y * inv);
        xp[mm][2] = make_float2(lo.z * inv, hi.z * inv);
        xp[mm][3] = make_float2(lo.w * inv, hi.w * inv);
    }
    const uint32_t a0 = TAB + (uint32_t)p * PLANE + 128u * jj + 16u * lq;
    // (run once per table: kept rolled, two codes per pass, so that its
    // instructions stay few)
#pragma unroll 2
    for (int it = 0; it < 128 / LW; ++it) {
        const int c0 = warp + it * LW;
        const float4 e = *reinterpret_cast<const float4*>(&cb[4 * c0]);
        const float2 ex = make_float2(e.x, e.x), ey = make_float2(e.y, e.y);
        const float2 ez = make_float2(e.z, e.z), ew = make_float2(e.w, e.w);
        uint32_t wv[4];
#pragma unroll
        for (int mm = 0; mm < 4; ++mm) {
            float2 v2 = __fmul2_rn(ex, xp[mm][0]);
            v2 = __ffma2_rn(ey, xp[mm][1], v2);
            v2 = __ffma2_rn(ez, xp[mm][2], v2);
            v2 = __ffma2_rn(ew, xp[mm][3], v2);
            const __half2 hv = __floats2half2_rn(v2.x, v2.y);
            wv[mm] = *reinterpret_cast<const uint32_t*>(&hv);
        }
        const uint32_t a = a0 + 256u * (uint32_t)c0;
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(wv[0]), "r"(wv[1]), "r"(wv[2]),
                     "r"(wv[3]));
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a + 128u * 256u), "r"(wv[0] ^ 0x80008000u),
                     "r"(wv[1] ^ 0x80008000u), "r"(wv[2] ^ 0x80008000u), "r"(wv[3] ^ 0x80008000u));
    }
}

// e2m1 value of a 4-bit code: sign bit 3, exponent bits 1-2 (bias 1), one
// mantissa bit; exponent 0 is the subnormal 0 / 0.5.  (Plain arithmetic, so
// that a constant code folds to a constant.)
__host__ __device__ constexpr float e2m1_value(int n) {
    return ((n & 8) ? -1.0f : 1.0f) *
           (((n & 7) >> 1) ? (float)(2 + (n & 1)) * (float)(1 << ((n & 7) >> 1)) * 0.25f : 0.5f * (float)(n & 1));
}

// The e2m1 table of one K-range (FP4 experts): a code byte holds the two
// elements 2G (low nibble) and 2G + 1 (high nibble) of group G, so entry
// L[v][G] = e2m1(v & 15) x[2G] + e2m1(v >> 4) x[2G + 1], divided by 2^e
// (table_exponent with cb == nullptr); no sign fold (all 256 bytes are
// built).  The K-range holds 512 inputs, nkb tiles of 64; the quads, slots
// and addresses are those of build_table, with 2-input groups.  Warp w
// builds the bytes v = w + 16 i (LW == 16): its low nibble is w, its high
// nibble the step i.
__device__ __forceinline__ void build_table_f4(const float* xs, int nkb, int e, int tid) {
    static_assert(LW == 16, "one low nibble per warp");
    const int warp = tid >> 5;
    const int q = tid & 31, lq = q & 7, jj = (q >> 3) & 1, p = q >> 4, bq = lane_block(4 * lq);
    if (bq >= nkb) return;
    const int i0 = 64 * bq + 32 * p + 16 * jj;  // inputs 2 g0 .. 2 g0 + 15, g0 = 32 bq + 4 (4p + 2jj)
    const float inv = exp2_int(-e);
    const float4 f0 = *reinterpret_cast<const float4*>(&xs[xs_at(i0)]);
    const float4 f1 = *reinterpret_cast<const float4*>(&xs[xs_at(i0 + 4)]);
    const float4 f2 = *reinterpret_cast<const float4*>(&xs[xs_at(i0 + 8)]);
    const float4 f3 = *reinterpret_cast<const float4*>(&xs[xs_at(i0 + 12)]);
    // word mm holds groups g0 + mm (low half) and g0 + 4 + mm (high half):
    // x0[mm] / x1[mm] their first / second elements
    const float2 x0[4] = {make_float2(f0.x * inv, f2.x * inv), make_float2(f0.z * inv, f2.z * inv),
                          make_float2(f1.x * inv, f3.x * inv), make_float2(f1.z * inv, f3.z * inv)};
    const float2 x1[4] = {make_float2(f0.y * inv, f2.y * inv), make_float2(f0.w * inv, f2.w * inv),
                          make_float2(f1.y * inv, f3.y * inv), make_float2(f1.w * inv, f3.w * inv)};
    const float lo = e2m1_value(warp);
    float2 lx[4];  // the low nibble's part, the same for every byte of this warp
#pragma unroll
    for (int mm = 0; mm < 4; ++mm) lx[mm] = __fmul2_rn(make_float2(lo, lo), x0[mm]);
    const uint32_t a0 = TAB + (uint32_t)p * PLANE + 128u * jj + 16u * lq + 256u * (uint32_t)warp;
    // (unrolled by 8: the step's value is a constant up to its sign; a full
    // unroll spills in FC2)
#pragma unroll 8
    for (int it = 0; it < 16; ++it) {
        const float hi = e2m1_value(it);
        uint32_t wv[4];
#pragma unroll
        for (int mm = 0; mm < 4; ++mm) {
            const float2 v2 = __ffma2_rn(make_float2(hi, hi), x1[mm], lx[mm]);
            const __half2 hv = __floats2half2_rn(v2.x, v2.y);
            wv[mm] = *reinterpret_cast<const uint32_t*>(&hv);
        }
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a0 + 256u * 16u * (uint32_t)it), "r"(wv[0]),
                     "r"(wv[1]), "r"(wv[2]), "r"(wv[3]));
    }
}

// One unit (codes c: nkb consecutive packed tiles; scales sp: their nkb x 16
// row scales) into the warp's slot: lane 0 arms the slot's barrier with the
// byte count, lanes 0-2 issue the three bulk copies.
__device__ __forceinline__ void issue_unit(uint32_t slot, uint32_t bar, const uint8_t* c, const uint16_t* sp, int nkb,
                                           int lane) {
    if (lane == 0) mbar_arrive_expect_tx(bar, 544u * nkb);
    __syncwarp();
    if (lane == 0) bulk_g2s(slot, c, 512u * min(nkb, 4), bar);
    if (lane == 1 && nkb > 4) bulk_g2s(slot + HALF_OFF, c + 2048, 512u * (nkb - 4), bar);
    if (lane == 2) bulk_g2s(slot + SCALE_OFF, sp, 32u * nkb, bar);
}

// Asks L2 for one unit's codes and scales (this lane only).
__device__ __forceinline__ void prefetch_unit_l2(const uint8_t* c, const uint16_t* sp, int nkb) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(c), "r"(512u * nkb) : "memory");
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(sp), "r"(32u * nkb) : "memory");
}

// The lane's part of a unit from the slot into registers (lanes of scale
// blocks beyond the K-range load nothing).
__device__ __forceinline__ void load_unit(UnitRegs& r, uint32_t slot, int lane, bool active) {
    if (!active) return;
    const int b = lane_block(lane), m = lane & 3;
    const uint32_t tb = slot + (b < 4 ? 512u * b : HALF_OFF + 512u * (b - 4)) + 16u * m;
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) r.cw[jj] = lds_u128(tb + 64 * jj);
    r.sc[0] = lds_u128(slot + SCALE_OFF + 32 * b);
    r.sc[1] = lds_u128(slot + SCALE_OFF + 32 * b + 16);
}

}  // namespace lut
}  // namespace moe
