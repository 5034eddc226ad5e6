// Host CPU computation of the experts a GPU slot table does not hold (the
// Tandem-vLLM page, "How it works": experts that miss the GPU cache are
// computed by the CPU in parallel with the GPU, nothing skipped or
// substituted; "Speed": the CPU matters as much as the GPU).  Host code only.
//
// The CPU reads the same packed bytes a slot holds (moe_vq2_pack /
// moe_fp4_pack layouts), so the host base of an expert cache serves both the
// slot fills and this path without a second copy.  Per 16-row tile of a
// matrix, the 16-byte chunk of group g holds the codes of the tile's 16 rows,
// so each code selects a 4-vector of the sign-folded codebook that multiplies
// the 4 inputs of the group (one 4-wide multiply-add per code, in portable
// vector C++ that the compiler maps to NEON on aarch64 and SSE on x86-64);
// each row's sum over a 128-input block is scaled by the row's fp16 scale.
// FC1 (gate, up) with silu(g) * u, then FC2 with the remainder of the
// combine, run in fp32 as two parallel steps over a pool of host threads
// (items: 16 rows of gate and up of one expert for all its tokens; 16 rows
// of every listed expert's down matrix for all tokens, then those rows of
// each token's remainder summed in pair order).  The pool's threads poll for
// work for a while before they sleep, so that a call's steps do not pay a
// wake-up each.
#include <cmath>
#include <cstring>
#include <algorithm>
#include <atomic>
#include <chrono>
#include <condition_variable>
#include <functional>
#include <mutex>
#include <thread>
#include <vector>

#include "common.cuh"

namespace moe {
namespace {

typedef float f4 __attribute__((vector_size(16)));

inline float bf16_to_f32(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    std::memcpy(&f, &u, 4);
    return f;
}
inline float fp16_to_f32(uint16_t h) {
    const uint32_t s = (uint32_t)(h >> 15) << 31, e = (h >> 10) & 31, m = h & 1023;
    uint32_t u;
    if (e == 0) {
        if (m == 0) {
            u = s;
        } else {  // subnormal: m * 2^-24
            float f = (float)m * 5.9604644775390625e-8f;
            std::memcpy(&u, &f, 4);
            u |= s;
        }
    } else if (e == 31) {
        u = s | 0x7f800000u | (m << 13);
    } else {
        u = s | ((e + 112) << 23) | (m << 13);
    }
    float f;
    std::memcpy(&f, &u, 4);
    return f;
}
inline float hsum(f4 v) { return (v[0] + v[1]) + (v[2] + v[3]); }

// y[r] (r < 16 rows of tile row rt) = sum over K of W[r][.] v[.] for one
// VQ2 matrix (packed) and one fp32 vector v (K entries, as K/4 4-vectors).
void vq2_tile_rows(const uint8_t* codes, const uint16_t* scales, int K, int rt, const f4* cbs, const f4* v4,
                   float* y16) {
    const int KB = K / 128;
    float tot[16] = {0};
    for (int kb = 0; kb < KB; ++kb) {
        const uint8_t* tile = codes + ((size_t)rt * KB + kb) * 512;
        const uint16_t* sc = scales + ((size_t)rt * KB + kb) * 16;
        const f4* xv = v4 + 32 * kb;
        f4 acc[16];
        for (int b = 0; b < 16; ++b) acc[b] = f4{0.f, 0.f, 0.f, 0.f};
        for (int g = 0; g < 32; ++g) {
            // byte 2i + h of the chunk: row i + 8h (two 8-byte loads; the
            // bytes taken out with shifts, little-endian on both hosts)
            uint64_t w0, w1;
            std::memcpy(&w0, tile + 16 * g, 8);
            std::memcpy(&w1, tile + 16 * g + 8, 8);
            const f4 x = xv[g];
            for (int b = 0; b < 8; ++b) acc[b] += cbs[(w0 >> (8 * b)) & 0xffu] * x;
            for (int b = 0; b < 8; ++b) acc[8 + b] += cbs[(w1 >> (8 * b)) & 0xffu] * x;
        }
        for (int b = 0; b < 16; ++b) {
            const int row = (b >> 1) + 8 * (b & 1);
            tot[row] += hsum(acc[b]) * fp16_to_f32(sc[row]);
        }
    }
    for (int r = 0; r < 16; ++r) y16[r] = tot[r];
}

// ue8m0 byte e -> 2^(e - 127), exactly (e = 0: the subnormal 2^-127, bits
// 0x400000; e = 255: infinity).
inline float e8m0_value(uint8_t e) {
    const uint32_t u = e ? (uint32_t)e << 23 : 0x00400000u;
    float f;
    std::memcpy(&f, &u, 4);
    return f;
}

// The same for one FP4 matrix (packed: 64-element tiles, ue8m0 scale per 32).
void fp4_tile_rows(const uint8_t* codes, const uint8_t* scales, int K, int rt, const float* v, float* y16) {
    static const float E2M1[16] = {0.f, 0.5f, 1.f, 1.5f, 2.f, 3.f, 4.f, 6.f,
                                   -0.f, -0.5f, -1.f, -1.5f, -2.f, -3.f, -4.f, -6.f};
    const int KT = K / 64, KB = K / 32;
    float tot[16] = {0};
    for (int kt = 0; kt < KT; ++kt) {
        const uint8_t* tile = codes + ((size_t)rt * KT + kt) * 512;
        for (int r16 = 0; r16 < 16; ++r16) {
            float part[2] = {0.f, 0.f};  // the tile's two 32-element scale blocks
            for (int lb = 0; lb < 32; ++lb) {  // logical byte of the row within the tile
                const uint8_t byte = tile[fp4_in_tile(r16, lb)];
                const float* xv = v + 64 * kt + 2 * lb;
                part[lb >> 4] += E2M1[byte & 15] * xv[0] + E2M1[byte >> 4] * xv[1];
            }
            for (int h = 0; h < 2; ++h) {
                const uint8_t e = scales[((size_t)rt * KB + 2 * kt + h) * 16 + r16];
                tot[r16] += part[h] * e8m0_value(e);
            }
        }
    }
    for (int r = 0; r < 16; ++r) y16[r] = tot[r];
}

}  // namespace
}  // namespace moe

// ------------------------------------------------------------------ pool
struct moe_cpu_pool {
    std::vector<std::thread> workers;
    std::mutex mu;
    std::condition_variable go, done;
    const std::function<void(int)>* fn = nullptr;
    int n_items = 0;
    std::atomic<int> next{0};
    std::atomic<int> remaining{0};      // workers still on the current job
    std::atomic<unsigned long> gen{0};  // job generation
    std::atomic<bool> stop{false};
    int sleepers = 0;              // workers blocked on `go` (under mu)
    bool caller_sleeping = false;  // the caller blocked on `done` (under mu)
    // how long a worker polls for the next job (and the caller for the end
    // of one) before it blocks: longer than the steps of a call and the GPU
    // work between two calls of a decode loop, so that a call pays no wake-up
    static constexpr long long SPIN_NS = 2000000;
    template <class Pred>
    static bool poll(Pred ready) {
        const auto end = std::chrono::steady_clock::now() + std::chrono::nanoseconds(SPIN_NS);
        for (unsigned i = 1;; ++i) {
            if (ready()) return true;
            if ((i & 255u) == 0 && std::chrono::steady_clock::now() > end) return ready();
        }
    }

    void work() {
        unsigned long seen = 0;
        for (;;) {
            poll([&] { return gen.load(std::memory_order_acquire) != seen || stop.load(std::memory_order_relaxed); });
            unsigned long g = gen.load(std::memory_order_acquire);
            if (g == seen && !stop.load()) {
                std::unique_lock<std::mutex> lk(mu);
                ++sleepers;
                go.wait(lk, [&] { return stop.load() || gen.load(std::memory_order_acquire) != seen; });
                --sleepers;
                g = gen.load(std::memory_order_acquire);
            }
            if (stop.load()) return;
            seen = g;
            // (fn and n_items were written before the generation was published)
            const std::function<void(int)>& f = *fn;
            const int n = n_items;
            for (int i = next.fetch_add(1); i < n; i = next.fetch_add(1)) f(i);
            if (remaining.fetch_sub(1, std::memory_order_acq_rel) == 1) {
                std::lock_guard<std::mutex> lk(mu);
                if (caller_sleeping) done.notify_all();
            }
        }
    }
    // Runs f(0..n-1) over the workers and the calling thread; returns when all are done.
    void parallel_for(int n, const std::function<void(int)>& f) {
        if (n <= 0) return;
        if (workers.empty() || n == 1) {
            for (int i = 0; i < n; ++i) f(i);
            return;
        }
        // every worker has left the previous job (remaining reached 0 after
        // its last claim of an item)
        fn = &f;
        n_items = n;
        next.store(0, std::memory_order_relaxed);
        remaining.store((int)workers.size(), std::memory_order_relaxed);
        gen.fetch_add(1, std::memory_order_release);
        {
            std::lock_guard<std::mutex> lk(mu);
            if (sleepers) go.notify_all();
        }
        for (int i = next.fetch_add(1); i < n; i = next.fetch_add(1)) f(i);
        if (!poll([&] { return remaining.load(std::memory_order_acquire) == 0; })) {
            std::unique_lock<std::mutex> lk(mu);
            caller_sleeping = true;
            done.wait(lk, [&] { return remaining.load(std::memory_order_acquire) == 0; });
            caller_sleeping = false;
        }
    }
};

using namespace moe;

extern "C" {

moe_status moe_cpu_pool_create(int threads, moe_cpu_pool** out) {
    MOE_CHECK_ARG(out, "moe_cpu_pool_create: out is null");
    *out = nullptr;
    int n = threads > 0 ? threads : (int)std::thread::hardware_concurrency();
    if (n < 1) n = 1;
    MOE_CHECK_ARG(n <= 4096, "moe_cpu_pool_create: %d threads", n);
    moe_cpu_pool* p = new (std::nothrow) moe_cpu_pool;
    if (!p) {
        set_error("moe_cpu_pool_create: out of host memory");
        return MOE_ERR_NO_MEM;
    }
    try {
        for (int i = 0; i < n - 1; ++i) p->workers.emplace_back([p] { p->work(); });
    } catch (...) {
        {
            std::lock_guard<std::mutex> lk(p->mu);
            p->stop.store(true);
        }
        p->go.notify_all();
        for (auto& w : p->workers) w.join();
        delete p;
        set_error("moe_cpu_pool_create: could not start %d threads", n - 1);
        return MOE_ERR_NO_MEM;
    }
    *out = p;
    return MOE_OK;
}

int moe_cpu_pool_threads(const moe_cpu_pool* pool) { return pool ? (int)pool->workers.size() + 1 : 0; }

moe_status moe_cpu_pool_destroy(moe_cpu_pool* pool) {
    if (!pool) return MOE_OK;
    {
        std::lock_guard<std::mutex> lk(pool->mu);
        pool->stop.store(true);
    }
    pool->go.notify_all();
    for (auto& w : pool->workers) w.join();
    delete pool;
    return MOE_OK;
}

moe_status moe_cpu_expert_ffn(moe_cpu_pool* pool, int H, int I, const uint16_t* codebook,
                              const moe_expert_desc* experts, int E, const uint16_t* x, const int32_t* ids,
                              const float* weights, const uint8_t* gpu_status, int T, int k, float* out) {
    MOE_CHECK_ARG(pool, "moe_cpu_expert_ffn: null pool");
    MOE_CHECK_ARG(T >= 0 && k >= 1 && E >= 1, "moe_cpu_expert_ffn: T=%d k=%d E=%d", T, k, E);
    MOE_CHECK_SUPPORTED(H > 0 && I > 0 && H % 256 == 0 && I % 128 == 0,
                        "moe_cpu_expert_ffn: need H %% 256 == 0 and I %% 128 == 0 (H=%d I=%d)", H, I);
    if (T == 0) return MOE_OK;
    MOE_CHECK_ARG(codebook && experts && x && ids && weights && gpu_status && out, "moe_cpu_expert_ffn: null pointer");
    const int P = T * k;
    // the pairs to compute, grouped by expert (pairs of one expert share its weights)
    std::vector<int> cnt(E + 1, 0);
    for (int p = 0; p < P; ++p) {
        if (gpu_status[p]) continue;
        const int e = ids[p];
        MOE_CHECK_ARG(e >= 0 && e < E, "moe_cpu_expert_ffn: ids[%d]=%d outside [0, %d)", p, e, E);
        const moe_expert_desc& d = experts[e];
        MOE_CHECK_ARG(d.format == MOE_FMT_VQ2 || d.format == MOE_FMT_FP4, "moe_cpu_expert_ffn: expert %d format %d",
                      e, d.format);
        for (int m = 0; m < 3; ++m)
            MOE_CHECK_ARG(d.codes[m] && d.scales[m], "moe_cpu_expert_ffn: expert %d has a null buffer", e);
        ++cnt[e + 1];
    }
    for (int e = 0; e < E; ++e) cnt[e + 1] += cnt[e];
    const int n_pairs = cnt[E];
    std::vector<int> order(n_pairs), pos(cnt.begin(), cnt.end() - 1);
    for (int p = 0; p < P; ++p)
        if (!gpu_status[p]) order[pos[ids[p]]++] = p;
    std::vector<int> experts_used;
    for (int e = 0; e < E; ++e)
        if (cnt[e + 1] > cnt[e]) experts_used.push_back(e);

    try {
        // (buffers of floats, read as 4-vectors: the allocations are 16-byte
        // aligned and every 4-vector starts at a multiple of 4 floats)
        // sign-folded fp32 codebook
        std::vector<float> cbsv(256 * 4);
        for (int c = 0; c < 256; ++c) {
            const float sg = (c & 0x80) ? -1.0f : 1.0f;
            for (int q = 0; q < 4; ++q) cbsv[4 * c + q] = sg * fp16_to_f32(codebook[4 * (c & 127) + q]);
        }
        const f4* cbs = reinterpret_cast<const f4*>(cbsv.data());
        // inputs of the listed pairs in fp32 (pair order of `order`); a few
        // pairs on this thread
        std::vector<float> xin((size_t)n_pairs * H), a((size_t)n_pairs * I), y((size_t)n_pairs * H);
        auto to_f32 = [&](int q) {
            const uint16_t* xr = x + (size_t)(order[q] / k) * H;
            float* dst = &xin[(size_t)q * H];
            for (int i = 0; i < H; ++i) dst[i] = bf16_to_f32(xr[i]);
        };
        if ((size_t)n_pairs * H <= ((size_t)1 << 16)) {
            for (int q = 0; q < n_pairs; ++q) to_f32(q);
        } else {
            pool->parallel_for(n_pairs, to_f32);
        }
        auto tile_rows = [&](const moe_expert_desc& d, int mtx, int K, int rt, const float* v, float* y16) {
            if (d.format == MOE_FMT_VQ2)
                vq2_tile_rows(static_cast<const uint8_t*>(d.codes[mtx]), static_cast<const uint16_t*>(d.scales[mtx]), K,
                              rt, cbs, reinterpret_cast<const f4*>(v), y16);
            else
                fp4_tile_rows(static_cast<const uint8_t*>(d.codes[mtx]), static_cast<const uint8_t*>(d.scales[mtx]), K,
                              rt, v, y16);
        };
        // FC1 and a = silu(g) * u: items (expert, 16 rows of gate and up)
        const int rt1 = I / 16;
        pool->parallel_for((int)experts_used.size() * rt1, [&](int it) {
            const int e = experts_used[it / rt1], rt = it % rt1;
            const moe_expert_desc& d = experts[e];
            float g16[16], u16[16];
            for (int q = cnt[e]; q < cnt[e + 1]; ++q) {
                const float* xq = &xin[(size_t)q * H];
                tile_rows(d, 0, H, rt, xq, g16);
                tile_rows(d, 1, H, rt, xq, u16);
                float* aq = &a[(size_t)q * I + 16 * rt];
                for (int r = 0; r < 16; ++r) aq[r] = g16[r] / (1.0f + std::exp(-g16[r])) * u16[r];
            }
        });
        // FC2 and the remainder of the combine: items (16 rows of H) over
        // every listed expert and pair, then those rows of each token's
        // remainder, summed in pair order
        std::vector<int> q_of(P, -1);
        for (int q = 0; q < n_pairs; ++q) q_of[order[q]] = q;
        pool->parallel_for(H / 16, [&](int rt) {
            for (int e : experts_used) {
                const moe_expert_desc& d = experts[e];
                for (int q = cnt[e]; q < cnt[e + 1]; ++q)
                    tile_rows(d, 2, I, rt, &a[(size_t)q * I], &y[(size_t)q * H + 16 * rt]);
            }
            for (int t = 0; t < T; ++t) {
                float* o = out + (size_t)t * H + 16 * rt;
                for (int r = 0; r < 16; ++r) o[r] = 0.0f;
                for (int j = 0; j < k; ++j) {
                    const int q = q_of[t * k + j];
                    if (q < 0) continue;
                    const float w = weights[t * k + j];
                    const float* yq = &y[(size_t)q * H + 16 * rt];
                    for (int r = 0; r < 16; ++r) o[r] += w * yq[r];
                }
            }
        });
    } catch (const std::bad_alloc&) {
        set_error("moe_cpu_expert_ffn: out of host memory");
        return MOE_ERR_NO_MEM;
    }
    return MOE_OK;
}

// Host packers: the layouts of moe_vq2_pack / moe_fp4_pack.
moe_status moe_vq2_pack_host(const uint8_t* codes, const uint16_t* scales, int rows, int K, uint8_t* packed_codes,
                             uint16_t* packed_scales) {
    MOE_CHECK_ARG(codes && scales && packed_codes && packed_scales, "moe_vq2_pack_host: null pointer");
    MOE_CHECK_ARG(rows > 0 && K > 0, "moe_vq2_pack_host: rows=%d K=%d must be positive", rows, K);
    MOE_CHECK_SUPPORTED(rows % 16 == 0 && K % 128 == 0,
                        "moe_vq2_pack_host: need rows %% 16 == 0 and K %% 128 == 0 (rows=%d K=%d)", rows, K);
    const int G = K / 4, KB = K / 128;
    for (int r = 0; r < rows; ++r) {
        for (int q = 0; q < G; ++q)
            packed_codes[vq2_tile_offset(r / 16, q / 32, KB) + vq2_in_tile(r % 16, q % 32)] = codes[(size_t)r * G + q];
        for (int kb = 0; kb < KB; ++kb)
            packed_scales[((size_t)(r / 16) * KB + kb) * 16 + r % 16] = scales[(size_t)r * KB + kb];
    }
    return MOE_OK;
}

moe_status moe_fp4_pack_host(const uint8_t* codes, const uint8_t* scales, int rows, int K, uint8_t* packed_codes,
                             uint8_t* packed_scales) {
    MOE_CHECK_ARG(codes && scales && packed_codes && packed_scales, "moe_fp4_pack_host: null pointer");
    MOE_CHECK_ARG(rows > 0 && K > 0, "moe_fp4_pack_host: rows=%d K=%d must be positive", rows, K);
    MOE_CHECK_SUPPORTED(rows % 16 == 0 && K % 64 == 0,
                        "moe_fp4_pack_host: need rows %% 16 == 0 and K %% 64 == 0 (rows=%d K=%d)", rows, K);
    const int NB = K / 2, KT = K / 64, KB = K / 32;
    for (int r = 0; r < rows; ++r) {
        for (int b = 0; b < NB; ++b)
            packed_codes[((size_t)(r / 16) * KT + b / 32) * 512 + fp4_in_tile(r % 16, b % 32)] = codes[(size_t)r * NB + b];
        for (int kb = 0; kb < KB; ++kb)
            packed_scales[((size_t)(r / 16) * KB + kb) * 16 + r % 16] = scales[(size_t)r * KB + kb];
    }
    return MOE_OK;
}

}  // extern "C"
