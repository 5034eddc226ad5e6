// Expert cache: fills slot-table entries from page-locked host copies of the
// experts' packed buffers, on a miss (vLLM-Moet page, "2-bit experts on vLLM
// v0.24.0", "Experts beyond VRAM"; Tandem-vLLM page, "How it works").  Host
// code only: the planning step decides which slot each missing expert takes
// (eviction by routing counts); the fetch enqueues on one stream the
// host-to-device copies of every miss (one cudaMemcpyAsync per buffer, or one
// per expert for a host image in the slot's layout), then one kernel that
// writes the table: the replaced experts' entries cleared, the new ones set.
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <vector>

#include "common.cuh"
#include "slot_batch.cuh"

namespace moe {
namespace {

constexpr size_t SLOT_ALIGN = 256;

size_t round_up(size_t v) { return (v + SLOT_ALIGN - 1) / SLOT_ALIGN * SLOT_ALIGN; }

// Bytes of buffer b of an expert: b = 0..2 codes of gate, up, down; 3..5
// their scales.  Gate and up are [I, H], down is [H, I].
size_t buffer_bytes(int H, int I, int format, int b) {
    const size_t rows = (b % 3 == 2) ? (size_t)H : (size_t)I;
    const size_t K = (b % 3 == 2) ? (size_t)I : (size_t)H;
    if (format == MOE_FMT_VQ2) return b < 3 ? rows * (K / 4) : rows * (K / 128) * 2;
    return b < 3 ? rows * (K / 2) : rows * (K / 32);
}

// Offset of buffer b inside a slot.
size_t buffer_offset(int H, int I, int format, int b) {
    size_t off = 0;
    for (int j = 0; j < b; ++j) off += round_up(buffer_bytes(H, I, format, j));
    return off;
}

struct HostCopy {
    int set = 0;
    int format = 0;
    int image = 0;            // 1: one block in the slot's layout (one copy)
    const void* buf[6] = {};  // codes gate, up, down; scales gate, up, down
};

bool pinned(const void* p, size_t bytes) {
    cudaPointerAttributes a;
    for (const char* q : {static_cast<const char*>(p), static_cast<const char*>(p) + (bytes ? bytes - 1 : 0)}) {
        if (cudaPointerGetAttributes(&a, q) != cudaSuccess) {
            cudaGetLastError();
            return false;
        }
        if (a.type != cudaMemoryTypeHost) return false;
    }
    return true;
}

}  // namespace
}  // namespace moe

// The opaque handle of include/moe_vq2.h.
struct moe_expert_cache {
    moe_slot_table* table;
    char* pool;
    size_t slot_bytes;
    int num_slots;
    std::vector<moe::HostCopy> host;     // [E]
    std::vector<int32_t> slot_expert;    // [num_slots]: expert held, -1 = free
    std::vector<uint64_t> counts;        // [E] routing counts
    std::vector<uint64_t> last_step;     // [E] last step named (0 = never)
    uint64_t step;
    uint64_t hits, misses, unplaced, bytes;
};

using namespace moe;

extern "C" {

size_t moe_expert_cache_slot_bytes(int H, int I, int format) {
    if (H <= 0 || I <= 0 || (format != MOE_FMT_VQ2 && format != MOE_FMT_FP4)) return 0;
    return buffer_offset(H, I, format, 6);
}

moe_status moe_expert_cache_plan(int num_experts, int num_slots, int32_t* slot_expert, uint64_t* counts,
                                 uint64_t* last_step, uint64_t step, const int32_t* request, int n,
                                 int32_t* fill_slot, int32_t* evicted, int* n_unplaced) {
    MOE_CHECK_ARG(num_experts > 0 && num_slots >= 0 && n >= 0,
                  "moe_expert_cache_plan: num_experts=%d num_slots=%d n=%d", num_experts, num_slots, n);
    MOE_CHECK_ARG(counts && last_step && (num_slots == 0 || slot_expert) &&
                      (n == 0 || (request && fill_slot && evicted)),
                  "moe_expert_cache_plan: null pointer");
    // holder[e] = slot of expert e or -1; every check before any update
    std::vector<int32_t> holder((size_t)num_experts, -1);
    for (int s = 0; s < num_slots; ++s) {
        const int32_t e = slot_expert[s];
        MOE_CHECK_ARG(e >= -1 && e < num_experts, "moe_expert_cache_plan: slot %d holds expert %d", s, (int)e);
        if (e < 0) continue;
        MOE_CHECK_ARG(holder[e] < 0, "moe_expert_cache_plan: expert %d held by slots %d and %d", (int)e,
                      (int)holder[e], s);
        holder[e] = s;
    }
    for (int i = 0; i < n; ++i)
        MOE_CHECK_ARG(request[i] >= 0 && request[i] < num_experts, "moe_expert_cache_plan: request[%d]=%d", i,
                      (int)request[i]);
    for (int e = 0; e < num_experts; ++e)
        MOE_CHECK_ARG(step > last_step[e], "moe_expert_cache_plan: step %llu not above expert %d's last step %llu",
                      (unsigned long long)step, e, (unsigned long long)last_step[e]);

    // The step's routing counts; last_step == step then marks "named now".
    std::vector<uint8_t> first((size_t)n, 0);
    for (int i = 0; i < n; ++i) {
        const int32_t e = request[i];
        if (last_step[e] != step) {
            last_step[e] = step;
            ++counts[e];
            first[i] = 1;
        }
    }
    int left = 0;
    for (int i = 0; i < n; ++i) {
        fill_slot[i] = -1;
        evicted[i] = -1;
        const int32_t e = request[i];
        if (!first[i] || holder[e] >= 0) continue;  // a repeat or a hit
        int s = -1;
        for (int j = 0; j < num_slots && s < 0; ++j)
            if (slot_expert[j] < 0) s = j;
        if (s < 0) {
            // the least routed expert not named by this step; ties: the one
            // named longest ago, then the lower id
            for (int j = 0; j < num_slots; ++j) {
                const int32_t v = slot_expert[j];
                if (last_step[v] == step) continue;
                if (s < 0) {
                    s = j;
                    continue;
                }
                const int32_t b = slot_expert[s];
                if (counts[v] < counts[b] || (counts[v] == counts[b] && (last_step[v] < last_step[b] ||
                                                                         (last_step[v] == last_step[b] && v < b))))
                    s = j;
            }
        }
        if (s < 0) {
            ++left;
            continue;
        }
        if (slot_expert[s] >= 0) {
            evicted[i] = slot_expert[s];
            holder[slot_expert[s]] = -1;
        }
        slot_expert[s] = e;
        holder[e] = s;
        fill_slot[i] = s;
    }
    if (n_unplaced) *n_unplaced = left;
    return MOE_OK;
}

moe_status moe_expert_cache_create(moe_slot_table* table, void* pool, size_t pool_bytes, size_t slot_bytes,
                                   moe_expert_cache** out) {
    MOE_CHECK_ARG(out, "moe_expert_cache_create: out is null");
    *out = nullptr;
    MOE_CHECK_ARG(table && pool, "moe_expert_cache_create: null table or pool");
    const int H = table->h.H, I = table->h.I;
    MOE_CHECK_SUPPORTED((reinterpret_cast<uintptr_t>(pool) & (SLOT_ALIGN - 1)) == 0,
                        "moe_expert_cache_create: the pool must be 256-byte aligned");
    MOE_CHECK_ARG(slot_bytes % SLOT_ALIGN == 0 && slot_bytes >= moe_expert_cache_slot_bytes(H, I, MOE_FMT_VQ2),
                  "moe_expert_cache_create: slot_bytes=%zu must be a multiple of 256 and at least %zu", slot_bytes,
                  moe_expert_cache_slot_bytes(H, I, MOE_FMT_VQ2));
    MOE_CHECK_ARG(pool_bytes / slot_bytes >= 1 && pool_bytes / slot_bytes <= (1u << 20),
                  "moe_expert_cache_create: pool_bytes=%zu holds %zu slots of %zu bytes", pool_bytes,
                  pool_bytes / slot_bytes, slot_bytes);
    moe_expert_cache* c = new (std::nothrow) moe_expert_cache();
    if (!c) {
        set_error("moe_expert_cache_create: out of host memory");
        return MOE_ERR_NO_MEM;
    }
    try {
        c->table = table;
        c->pool = static_cast<char*>(pool);
        c->slot_bytes = slot_bytes;
        c->num_slots = (int)(pool_bytes / slot_bytes);
        const size_t E = (size_t)table->h.E;
        c->host.assign(E, HostCopy());
        c->slot_expert.assign((size_t)c->num_slots, -1);
        c->counts.assign(E, 0);
        c->last_step.assign(E, 0);
    } catch (...) {
        delete c;
        set_error("moe_expert_cache_create: out of host memory");
        return MOE_ERR_NO_MEM;
    }
    c->step = 0;
    c->hits = c->misses = c->unplaced = c->bytes = 0;
    *out = c;
    return MOE_OK;
}

moe_status moe_expert_cache_set_host(moe_expert_cache* c, int expert_id, const moe_host_expert* h) {
    MOE_CHECK_ARG(c && h, "moe_expert_cache_set_host: null cache or host expert");
    const int E = c->table->h.E, H = c->table->h.H, I = c->table->h.I;
    MOE_CHECK_ARG(expert_id >= 0 && expert_id < E, "moe_expert_cache_set_host: expert_id=%d out of [0, %d)",
                  expert_id, E);
    MOE_CHECK_ARG(h->format == MOE_FMT_VQ2 || h->format == MOE_FMT_FP4,
                  "moe_expert_cache_set_host: unknown format %d", h->format);
    MOE_CHECK_SUPPORTED(moe_expert_cache_slot_bytes(H, I, h->format) <= c->slot_bytes,
                        "moe_expert_cache_set_host: a format-%d expert needs %zu bytes, slots hold %zu", h->format,
                        moe_expert_cache_slot_bytes(H, I, h->format), c->slot_bytes);
    HostCopy hc;
    hc.set = 1;
    hc.format = h->format;
    for (int b = 0; b < 6; ++b) {
        const void* p = b < 3 ? h->codes[b] : h->scales[b - 3];
        MOE_CHECK_ARG(p, "moe_expert_cache_set_host: null buffer %d", b);
        MOE_CHECK_SUPPORTED(pinned(p, buffer_bytes(H, I, h->format, b)),
                            "moe_expert_cache_set_host: buffer %d of expert %d is not page-locked host memory", b,
                            expert_id);
        hc.buf[b] = p;
    }
    c->host[expert_id] = hc;
    return MOE_OK;
}

moe_status moe_expert_cache_set_host_image(moe_expert_cache* c, int expert_id, int format, const void* image) {
    MOE_CHECK_ARG(c && image, "moe_expert_cache_set_host_image: null cache or image");
    const int E = c->table->h.E, H = c->table->h.H, I = c->table->h.I;
    MOE_CHECK_ARG(expert_id >= 0 && expert_id < E, "moe_expert_cache_set_host_image: expert_id=%d out of [0, %d)",
                  expert_id, E);
    MOE_CHECK_ARG(format == MOE_FMT_VQ2 || format == MOE_FMT_FP4,
                  "moe_expert_cache_set_host_image: unknown format %d", format);
    const size_t bytes = moe_expert_cache_slot_bytes(H, I, format);
    MOE_CHECK_SUPPORTED(bytes <= c->slot_bytes, "moe_expert_cache_set_host_image: a format-%d expert needs %zu "
                        "bytes, slots hold %zu", format, bytes, c->slot_bytes);
    MOE_CHECK_SUPPORTED(pinned(image, bytes),
                        "moe_expert_cache_set_host_image: the image of expert %d is not page-locked host memory",
                        expert_id);
    HostCopy hc;
    hc.set = 1;
    hc.format = format;
    hc.image = 1;
    for (int b = 0; b < 6; ++b) hc.buf[b] = static_cast<const char*>(image) + buffer_offset(H, I, format, b);
    c->host[expert_id] = hc;
    return MOE_OK;
}

moe_status moe_expert_cache_fetch(moe_expert_cache* c, const int32_t* experts, int n, cudaStream_t stream,
                                  int* n_fetched, int* n_unplaced, int* recapture) {
    MOE_CHECK_ARG(c && n >= 0 && (n == 0 || experts), "moe_expert_cache_fetch: null cache or ids, or n=%d", n);
    SlotTableHost& t = c->table->h;
    const int E = t.E, H = t.H, I = t.I;
    for (int i = 0; i < n; ++i) {
        MOE_CHECK_ARG(experts[i] >= 0 && experts[i] < E, "moe_expert_cache_fetch: expert %d out of [0, %d)",
                      (int)experts[i], E);
        MOE_CHECK_ARG(c->host[experts[i]].set, "moe_expert_cache_fetch: expert %d has no host copy",
                      (int)experts[i]);
    }
    // A slot whose table entry the caller evicted is free again.
    for (int s = 0; s < c->num_slots; ++s)
        if (c->slot_expert[s] >= 0 && t.h_fmt[c->slot_expert[s]] == 0) c->slot_expert[s] = -1;
    // Experts that the caller made resident itself are left out of the plan.
    std::vector<uint8_t> held((size_t)E, 0);
    for (int s = 0; s < c->num_slots; ++s)
        if (c->slot_expert[s] >= 0) held[c->slot_expert[s]] = 1;
    std::vector<int32_t> req, fill, ev;
    req.reserve((size_t)n);
    for (int i = 0; i < n; ++i)
        if (held[experts[i]] || t.h_fmt[experts[i]] == 0) req.push_back(experts[i]);
    fill.assign(req.size(), -1);
    ev.assign(req.size(), -1);
    int left = 0;
    const bool had_fp4 = t.n_fp4 > 0;
    moe_status st = moe_expert_cache_plan(E, c->num_slots, c->slot_expert.data(), c->counts.data(),
                                          c->last_step.data(), c->step + 1, req.data(), (int)req.size(),
                                          fill.data(), ev.data(), &left);
    if (st != MOE_OK) return st;
    ++c->step;
    // The copies of every miss are enqueued first, then one launch (per 32
    // entries) writes the table: the replaced experts' entries cleared, the
    // new ones set.  Nothing else runs on the stream in between, so no
    // kernel sees a replaced expert's entry while its slot is refilled.
    struct Upd {
        int32_t id;
        SlotDesc d;
    };
    std::vector<Upd> upd;
    upd.reserve(2 * req.size());
    size_t failed_at = req.size();
    cudaError_t copy_err = cudaSuccess;
    int fetched = 0;
    uint64_t nbytes = 0;
    std::vector<uint8_t> seen((size_t)E, 0);
    for (size_t i = 0; i < req.size(); ++i) {
        const int32_t e = req[i];
        if (fill[i] < 0) {
            if (!seen[e] && held[e]) ++c->hits;
            seen[e] = 1;
            continue;
        }
        seen[e] = 1;
        const int s = fill[i];
        if (ev[i] >= 0) upd.push_back(Upd{ev[i], SlotDesc{}});
        const HostCopy& hc = c->host[e];
        char* base = c->pool + (size_t)s * c->slot_bytes;
        SlotDesc d = {};
        d.format = hc.format;
        d.resident = 1;
        uint64_t eb = 0;
        for (int b = 0; b < 6 && copy_err == cudaSuccess; ++b) {
            char* dst = base + buffer_offset(H, I, hc.format, b);
            if (b < 3) d.codes[b] = dst; else d.scales[b - 3] = dst;
            eb += buffer_bytes(H, I, hc.format, b);
            if (hc.image && b > 0) continue;  // one copy of the whole image
            const size_t bytes = hc.image ? moe_expert_cache_slot_bytes(H, I, hc.format)
                                          : buffer_bytes(H, I, hc.format, b);
            copy_err = cudaMemcpyAsync(dst, hc.buf[b], bytes, cudaMemcpyHostToDevice, stream);
        }
        if (copy_err != cudaSuccess) {
            failed_at = i;
            break;
        }
        upd.push_back(Upd{e, d});
        ++fetched;
        nbytes += eb;
    }
    if (failed_at < req.size()) {
        // the failed request's slot is free (its old expert's entry is
        // cleared below); the later requests' slots keep what they held
        c->slot_expert[fill[failed_at]] = -1;
        for (size_t j = failed_at + 1; j < req.size(); ++j)
            if (fill[j] >= 0) c->slot_expert[fill[j]] = ev[j];
    }
    // the outputs as far as the call got, on the error returns too
    auto outputs = [&]() {
        if (n_fetched) *n_fetched = fetched;
        if (n_unplaced) *n_unplaced = left;
        if (recapture) *recapture = had_fp4 != (t.n_fp4 > 0);
    };
    for (size_t u0 = 0; u0 < upd.size(); u0 += SLOT_BATCH) {
        SlotBatch b;
        b.n = (int)std::min(upd.size() - u0, (size_t)SLOT_BATCH);
        for (int j = 0; j < b.n; ++j) {
            b.ids[j] = upd[u0 + j].id;
            b.d[j] = upd[u0 + j].d;
        }
        if ((st = launch_slot_set_many(t.d_desc, b, stream)) != MOE_OK) {
            outputs();
            return st;
        }
        for (int j = 0; j < b.n; ++j) {  // the host mirror of the table, as set / evict keep it
            const int id = b.ids[j];
            const int f = b.d[j].resident ? 1 + b.d[j].format : 0;
            t.n_fp4 += (f == 1 + MOE_FMT_FP4) - (t.h_fmt[id] == 1 + MOE_FMT_FP4);
            t.h_fmt[id] = (uint8_t)f;
        }
    }
    c->misses += (uint64_t)fetched;
    c->bytes += nbytes;
    if (failed_at < req.size()) {
        outputs();
        return cuda_status(copy_err, "moe_expert_cache_fetch: cudaMemcpyAsync");
    }
    c->unplaced += (uint64_t)left;
    outputs();
    return MOE_OK;
}

int moe_expert_cache_slot_of(const moe_expert_cache* c, int expert_id) {
    if (!c || expert_id < 0 || expert_id >= c->table->h.E) return -1;
    for (int s = 0; s < c->num_slots; ++s)
        if (c->slot_expert[s] == expert_id) return c->table->h.h_fmt[expert_id] ? s : -1;
    return -1;
}

moe_status moe_expert_cache_stats(const moe_expert_cache* c, uint64_t* hits, uint64_t* misses,
                                  uint64_t* unplaced, uint64_t* bytes_fetched) {
    MOE_CHECK_ARG(c, "moe_expert_cache_stats: null cache");
    if (hits) *hits = c->hits;
    if (misses) *misses = c->misses;
    if (unplaced) *unplaced = c->unplaced;
    if (bytes_fetched) *bytes_fetched = c->bytes;
    return MOE_OK;
}

moe_status moe_expert_cache_destroy(moe_expert_cache* c, cudaStream_t stream) {
    if (!c) return MOE_OK;
    moe_status st = MOE_OK;
    for (int s = 0; s < c->num_slots; ++s) {
        const int32_t e = c->slot_expert[s];
        if (e >= 0 && c->table->h.h_fmt[e] != 0 && st == MOE_OK) st = moe_slot_table_evict(c->table, e, stream);
    }
    delete c;
    return st;
}

}  // extern "C"
