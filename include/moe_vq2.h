/*
 * moe_vq2.h -- C ABI of the routed-expert VQ2 MoE layer on one GB300 (sm_103a).
 *
 * The layer, as the pages state the problem:
 *   - each token's router picks its top-k experts (vLLM-Moet page, "What we
 *     changed": "7 launches from router to FC1" at decode; the router's
 *     top-k, "2-bit experts on vLLM v0.24.0");
 *   - each chosen expert's FC1 (gate, up), silu(gate)*up and FC2 run from
 *     weights stored as 2-bit vector codes, about 2.1 bits per weight
 *     (Tandem-vLLM page, "How it works"), with a sign-symmetric codebook
 *     (vLLM-Moet page, "2-bit experts on vLLM v0.24.0"); the most routed
 *     experts may stay in FP4 (Tandem-vLLM page, "Quality": FP4_TOP);
 *   - a GPU cache holds the resident experts; the others are computed
 *     elsewhere and nothing is skipped or substituted (Tandem-vLLM page,
 *     "How it works"; vLLM-Moet page: "the GPU as an expert cache ... a miss
 *     is fetched and the step's graph replayed, bit-identical");
 *   - the experts' outputs are combined by router weight.
 *
 * Conventions (every entry point):
 *   - Returns a moe_status.  MOE_OK is 0; negative values are errors, and
 *     moe_last_error() then returns a message (thread-local, valid until the
 *     next call on the same thread).
 *   - All array arguments are DEVICE pointers owned by the caller unless a
 *     comment says otherwise; the library never frees them.  Pointers must
 *     be 16-byte aligned.
 *   - Arguments are checked on the host before anything is enqueued; a
 *     failed check enqueues nothing.  Calls only enqueue work on the given
 *     stream: they never synchronise the host with the device.
 *   - Activations: bf16 (uint16_t bit patterns).  Codebook and VQ2 scales:
 *     fp16 (uint16_t bit patterns).  FP4 scales: ue8m0 bytes.
 *   - Shapes: T tokens, H hidden, I expert intermediate, E experts, k top-k,
 *     P = T*k (token, slot) pairs, pair p = t*k + j.
 */
#ifndef MOE_VQ2_H
#define MOE_VQ2_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int moe_status;
#define MOE_OK 0
#define MOE_ERR_INVALID_ARG -1 /* null / negative / out-of-range argument        */
#define MOE_ERR_UNSUPPORTED -2 /* shape or alignment this build does not handle  */
#define MOE_ERR_CUDA -3        /* a CUDA runtime call or launch failed          */
#define MOE_ERR_NO_MEM -4      /* a library allocation failed                   */
#define MOE_ERR_WORKSPACE -5   /* workspace missing or smaller than required    */
#define MOE_ERR_TIMEOUT -6     /* reserved: a bounded device wait gave up        */
#define MOE_ERR_MISMATCH -7    /* moe_selftest: a result differs from its check  */

#define MOE_FMT_VQ2 0 /* 2-bit vector codes + fp16 row scales per 128 inputs */
#define MOE_FMT_FP4 1 /* MXFP4: e2m1 elements + ue8m0 scale per 32 inputs     */

#define MOE_FUSED_SCATTER 0 /* out[t] += w[t,j] * y  (fp32 atomics, caller zeroes out) */
#define MOE_PER_PAIR 1      /* ypair[sorted position] = y (deterministic)               */

int moe_version(void);
const char* moe_last_error(void);

/* ---------------------------------------------------------------------- */
/* Weight formats and packing                                              */
/* ---------------------------------------------------------------------- */
/*
 * Logical VQ2 matrix W [rows, K] (the expert code of the Tandem-vLLM page,
 * "How it works", with the sign-symmetric codebook of the vLLM-Moet page):
 *   codes  uint8 [rows, K/4]: code c of row r, group q covers inputs 4q..4q+3;
 *          bit 7 = sign (1 = negative), bits 0-6 = codebook index;
 *   scales fp16  [rows, K/128]: one scale per row per 128 inputs;
 *   codebook fp16 [128, 4], one per layer;
 *   W[r][4q+i] = (c >> 7 ? -1 : 1) * codebook[c & 127][i] * scales[r][4q/128].
 *
 * Packed VQ2 (what the slot table points at), same byte counts:
 *   codes: tiles of 16 rows x 32 groups (128 inputs), 512 bytes each, tile
 *          (rt, kb) at byte (rt*(K/128) + kb)*512; inside a tile byte
 *          16*g + 2*i + h holds the code of row 16*rt + i + 8*h, group
 *          32*kb + g (g < 32, i < 8, h < 2);
 *   scales: 16 fp16 per tile, at element (rt*(K/128) + kb)*16 + (r - 16*rt).
 *
 * Logical FP4 matrix [rows, K] (MXFP4, OCP MX v1.0):
 *   codes  uint8 [rows, K/2]: byte b of row r holds elements 2b (low nibble)
 *          and 2b+1 (high nibble), each e2m1;
 *   scales uint8 [rows, K/32]: ue8m0 exponent E, scale 2^(E-127); E = 255
 *          (NaN) is not allowed.
 * Packed FP4: tiles of 16 rows x 64 elements, 512 bytes each, tile (rt, kt)
 *   at byte (rt*(K/64) + kt)*512; inside a tile the 16 bytes at 16*(4*i + j)
 *   hold, for s = 0..3, the four bytes [row i: b, row i: b+4, row i+8: b,
 *   row i+8: b+4] with b = 32*kt + 8*s + j (rows relative to 16*rt);
 *   scales: 16 bytes per (rt, 32-element block kb), at (rt*(K/32) + kb)*16
 *   + (r - 16*rt).
 *
 * Requirements: rows % 16 == 0; K % 128 == 0 (VQ2) or K % 64 == 0 (FP4).
 * The pack calls read the logical arrays and write the packed ones; source
 * and destination must not overlap.  Sizes are unchanged by packing.
 */
moe_status moe_vq2_pack(const uint8_t* codes, const uint16_t* scales, int rows, int K,
                        uint8_t* packed_codes, uint16_t* packed_scales, cudaStream_t stream);
moe_status moe_fp4_pack(const uint8_t* codes, const uint8_t* scales, int rows, int K,
                        uint8_t* packed_codes, uint8_t* packed_scales, cudaStream_t stream);

/* ---------------------------------------------------------------------- */
/* Expert-slot table (the GPU expert cache of the Tandem-vLLM page, "How it */
/* works": "a GPU cache holds the most-used ones")                           */
/* ---------------------------------------------------------------------- */
typedef struct moe_slot_table moe_slot_table;

typedef struct moe_expert_desc {
    int format;                /* MOE_FMT_VQ2 or MOE_FMT_FP4                       */
    const void* codes[3];      /* packed codes of gate [I,H], up [I,H], down [H,I] */
    const void* scales[3];     /* packed scales of the same three matrices         */
} moe_expert_desc;

/* Creates a table of num_experts entries, all non-resident, for one layer
 * with hidden H and intermediate I.  codebook: device fp16 [128*4], the
 * layer's codebook; it must outlive the table.  Allocates a small device
 * descriptor array (the only memory the table owns).  H % 256 == 0 and
 * I % 128 == 0. */
moe_status moe_slot_table_create(int num_experts, int H, int I, const uint16_t* codebook,
                                 moe_slot_table** out);
/* Makes expert_id resident with the given packed buffers (not copied: they
 * must stay valid while the entry is set).  Setting an id again replaces it.
 * Enqueued on stream: work launched later on the same stream sees it. */
moe_status moe_slot_table_set(moe_slot_table* t, int expert_id, const moe_expert_desc* d,
                              cudaStream_t stream);
/* Marks expert_id non-resident (enqueued on stream). */
moe_status moe_slot_table_evict(moe_slot_table* t, int expert_id, cudaStream_t stream);
/* Frees the descriptor array; the caller must have synchronised the streams
 * that used the table. */
moe_status moe_slot_table_destroy(moe_slot_table* t);

/* ---------------------------------------------------------------------- */
/* Expert cache: misses fetched from host memory (vLLM-Moet page, "2-bit    */
/* experts on vLLM v0.24.0", "Experts beyond VRAM": the base lives in host  */
/* RAM, the GPU is an expert cache, a miss is fetched and the step's graph  */
/* replayed, bit-identical to a resident forward; Tandem-vLLM page, "How it */
/* works": the GPU cache holds the most-used experts)                       */
/* ---------------------------------------------------------------------- */
/*
 * The cache fills the entries of one slot table from page-locked host copies
 * of the experts' packed buffers, into fixed-size slots carved from a device
 * pool that the caller owns.  The expert kernels read the table's
 * descriptors on the device, so a CUDA graph of a forward pass captured once
 * stays valid while the cache changes which experts are resident: after a
 * fetch, replaying the same graph computes the newly resident experts.  The
 * result of a pair does not depend on the slot (the address) its expert's
 * buffers sit at, nor on which other experts are resident, so a forward
 * replayed after the fetch of its misses is bit-identical to a forward with
 * every expert resident.
 *
 * Eviction by routing counts: every fetch call is one step; each distinct
 * expert it names gains one count and is stamped with the step number.  A
 * named expert that is not resident takes the free slot with the lowest
 * index, else the slot of the resident expert that this step does not name
 * with the smallest (count, last step named, expert id).  Experts named in
 * the step are never evicted by it; when the step names more experts than
 * there are slots, the ones that find no slot stay non-resident (their pairs
 * are reported in pair_status, as for any non-resident expert).
 *
 * A cache is used by one host thread at a time (its calls are not
 * synchronised with each other).  The caller must not set or evict, through
 * moe_slot_table_set / _evict, the entries of experts the cache holds; an
 * entry the caller evicts anyway frees its slot at the next fetch.
 */
typedef struct moe_expert_cache moe_expert_cache;

typedef struct moe_host_expert {
    int format;                /* MOE_FMT_VQ2 or MOE_FMT_FP4                        */
    const void* codes[3];      /* page-locked HOST copies of the packed codes       */
    const void* scales[3];     /* and scales of gate [I,H], up [I,H], down [H,I]    */
} moe_host_expert;

/* Bytes one slot needs for an expert of the given format at hidden H and
 * intermediate I: the six packed buffers, each starting on a 256-byte
 * boundary.  Returns 0 for an unknown format or a non-positive shape. */
size_t moe_expert_cache_slot_bytes(int H, int I, int format);

/* Creates a cache for `table` over the caller's device memory `pool`
 * (pool_bytes, 256-byte aligned), cut into floor(pool_bytes / slot_bytes)
 * slots of slot_bytes each (a multiple of 256, at least
 * moe_expert_cache_slot_bytes(H, I, MOE_FMT_VQ2)).  The pool and the table
 * must outlive the cache.  Host memory only: allocates and enqueues nothing
 * on the device. */
moe_status moe_expert_cache_create(moe_slot_table* table, void* pool, size_t pool_bytes, size_t slot_bytes,
                                   moe_expert_cache** out);

/* Registers the host copy of expert_id (replacing an earlier one; a resident
 * copy of the expert is not refreshed).  The buffers are not copied now and
 * must stay valid and unchanged while the cache may fetch them; they must be
 * page-locked (cudaHostAlloc / cudaHostRegister), so that the fetch copies
 * are asynchronous.  The format's buffers must fit in one slot. */
moe_status moe_expert_cache_set_host(moe_expert_cache* c, int expert_id, const moe_host_expert* h);

/* Registers the host copy of expert_id as one block: `image` holds, in
 * page-locked host memory of moe_expert_cache_slot_bytes(H, I, format)
 * bytes, the six packed buffers at their slot offsets (codes of gate, up,
 * down, then scales of gate, up, down; each at the sum of the sizes before
 * it, every size rounded up to 256 bytes).  A fetch of such an expert is one
 * host-to-device copy instead of six. */
moe_status moe_expert_cache_set_host_image(moe_expert_cache* c, int expert_id, int format, const void* image);

/* One step: makes the experts in `experts` (HOST array of n ids, repeats
 * allowed) resident, in the order named, by the rule above.  It enqueues on
 * `stream` the host-to-device copies of every miss into its slot, then one
 * kernel (per 32 entries) that writes the table: the entries of the experts
 * replaced cleared, those of the new ones set.  The work that read a
 * replaced expert must be ordered before `stream`, and nothing may read the
 * table on another stream while the fetch runs (both hold when the forward
 * passes run on the same stream).  An expert already set in the table by
 * the caller is left as it is.  Every named expert must have a host copy,
 * else nothing is enqueued (MOE_ERR_INVALID_ARG).  After MOE_ERR_CUDA the
 * cache and the table may disagree (a slot may already hold the copy of an
 * expert whose entry was not written): destroy both.  The outputs are
 * written on that error too, counting what the call had done.
 * Outputs (each may be NULL): n_fetched = experts copied in, n_unplaced =
 * named experts left non-resident for lack of a slot, recapture = 1 if the
 * call changed whether the table holds any FP4 expert (the expert-FFN call
 * chooses its kernels by that on the host, so a graph captured before must
 * then be captured again), else 0. */
moe_status moe_expert_cache_fetch(moe_expert_cache* c, const int32_t* experts, int n, cudaStream_t stream,
                                  int* n_fetched, int* n_unplaced, int* recapture);

/* Slot index holding expert_id, or -1 (not resident through this cache, or
 * an out-of-range id).  Host bookkeeping: valid in stream order. */
int moe_expert_cache_slot_of(const moe_expert_cache* c, int expert_id);

/* Counters since creation: experts named and resident already (hits), named
 * and fetched (misses), named and left without a slot (unplaced), and the
 * bytes copied from host to device. */
moe_status moe_expert_cache_stats(const moe_expert_cache* c, uint64_t* hits, uint64_t* misses,
                                  uint64_t* unplaced, uint64_t* bytes_fetched);

/* Host-only planning step of moe_expert_cache_fetch, for callers that manage
 * slots and copies themselves (and testable without a GPU).  Every array
 * here is a HOST array.  State arrays (read and updated):
 *   slot_expert [num_slots]: the expert held by each slot, or -1;
 *   counts [num_experts], last_step [num_experts]: the routing counts and the
 *     last step each expert was named (0 = never).
 * `step` numbers this call and must be above every last_step.  request: n
 * expert ids.  Outputs, one entry per request: fill_slot[i] = the slot that
 * request i is copied into, or -1 (a hit, a repeat of an earlier request of
 * the call, or no slot left: those are counted in n_unplaced); evicted[i] =
 * the expert that slot held before, or -1.
 * Returns MOE_ERR_INVALID_ARG for a bad id, a slot_expert entry out of range
 * or held twice, or a step not above every last_step (nothing is updated). */
moe_status moe_expert_cache_plan(int num_experts, int num_slots, int32_t* slot_expert, uint64_t* counts,
                                 uint64_t* last_step, uint64_t step, const int32_t* request, int n,
                                 int32_t* fill_slot, int32_t* evicted, int* n_unplaced);

/* Enqueues on `stream` the eviction from the table of every expert that the
 * cache made resident, then frees the host bookkeeping.  The pool may be
 * reused once that work has run. */
moe_status moe_expert_cache_destroy(moe_expert_cache* c, cudaStream_t stream);

/* ---------------------------------------------------------------------- */
/* Hot path                                                                */
/* ---------------------------------------------------------------------- */

/* Router logits (the router of the vLLM-Moet page, "What we changed", MoE
 * at decode): logits[t,e] = sum_h x[t,h]*w_router[e,h] + bias[e], fp32.
 * x bf16 [T,H], w_router bf16 [E,H] row-major, bias fp32 [E] or NULL,
 * logits fp32 [T,E].  The sum runs in one fixed order so that repeated
 * runs and the CPU reference give identical bits: lane l = (h/8) mod 32
 * adds its exact products in increasing h, then the 32 lane sums combine
 * by a butterfly (xor 16, 8, 4, 2, 1), then the bias is added.
 * Requires H % 256 == 0, T >= 0, E >= 1. */
moe_status moe_router_logits(const uint16_t* x, const uint16_t* w_router, const float* bias,
                             float* logits, int T, int H, int E, cudaStream_t stream);

/* Top-k routing + softmax weights: for each token the k largest logits,
 * ordered by (logit descending, expert id ascending) -- equal logits go to
 * the lower id.  renormalize = 1: weights = softmax over the k selected
 * logits; 0: the softmax over all E logits read at the k selected.
 * logits fp32 [T,E] -> ids int32 [T,k], weights fp32 [T,k].
 * Requires 1 <= k <= min(E, 32), E <= 1024. */
moe_status moe_route_topk(const float* logits, int T, int E, int k, int renormalize,
                          int32_t* ids, float* weights, cudaStream_t stream);

/* Token -> expert permutation (no padding rows; the vLLM-Moet page, "What
 * we changed", names padding every expert to 128 rows as the cost to
 * avoid): a stable counting sort of the pairs p by ids[p].
 * expert_offsets int32 [E+1] (offsets[e] = pairs routed to experts below e),
 * sorted_pair int32 [P] (pair at each sorted position), pair_to_sorted
 * int32 [P] (inverse).  Requires every id in [0, E), E <= 1024, P <= 2^24.
 * ws: device workspace of moe_permute_workspace_size() bytes (may be NULL
 * when that size is 0): from 8192 pairs the sort runs over chunks of 1024
 * pairs on many CTAs and keeps per-chunk counts there (no initialisation
 * needed); with a smaller or NULL workspace it runs on one CTA, with the
 * same outputs. */
size_t moe_permute_workspace_size(int T, int k, int E);
moe_status moe_permute(const int32_t* ids, int T, int k, int E, int32_t* expert_offsets,
                       int32_t* sorted_pair, int32_t* pair_to_sorted, void* ws, size_t ws_bytes,
                       cudaStream_t stream);

/* The whole routing in one call: moe_router_logits, moe_route_topk and
 * moe_permute of the same arguments, with the same outputs bit for bit
 * (logits, ids, weights, expert_offsets, sorted_pair, pair_to_sorted).  For
 * small batches (T <= 8, E <= 1024) it is one kernel launch (fewer kernel
 * boundaries per layer at decode): for one token a thread-block cluster
 * computes the logits, gathers them in one CTA's shared memory and that CTA
 * routes the token; for 2..8 tokens the CTA that finishes its share of the
 * logits last does the top-k and the permutation.  Otherwise it enqueues the
 * three steps.
 * ws: moe_route_workspace_size() bytes of device memory holding a counter
 * (and, for large calls, the permutation's per-chunk counts); zero-fill it
 * once before the first call (each call leaves the counter at zero).
 * Calls that share a workspace must not overlap on the GPU. */
size_t moe_route_workspace_size(int T, int k, int E);
moe_status moe_route(const uint16_t* x, const uint16_t* w_router, const float* bias, int T, int H, int E,
                     int k, int renormalize, float* logits, int32_t* ids, float* weights,
                     int32_t* expert_offsets, int32_t* sorted_pair, int32_t* pair_to_sorted, void* ws,
                     size_t ws_bytes, cudaStream_t stream);

/* Expert FFN over the resident experts (Tandem-vLLM page, "How it works";
 * vLLM-Moet page, "Qwen3.8": silu*up fused into the MoE GEMV): for every
 * pair p routed to a resident expert e,
 *     g = Wg_e x_t,  u = Wu_e x_t,  a = silu(g) * u,  y = Wd_e a,
 * with the weights decoded from the slot table's packed codes.
 * mode MOE_FUSED_SCATTER: out_or_ypair is fp32 [T,H] and receives
 *     w[p] * y by fp32 atomic adds (the caller zeroes it first; the order of
 *     the adds, and so the low bits, may differ between runs);
 * mode MOE_PER_PAIR: out_or_ypair is fp32 [P,H]; row s receives y of the
 *     pair at sorted position s (run-to-run deterministic).
 * pair_status uint8 [P]: 1 if pair p was computed, 0 if its expert is not
 * resident (such pairs are skipped, never substituted; their rows of ypair
 * are left untouched).  expert_offsets/sorted_pair come from moe_permute
 * over the same ids; weights fp32 [T,k] from moe_route_topk.
 * ws: moe_vq2_expert_ffn_workspace_size(T, k, E, H, I) bytes of device
 * memory (scratch: the schedule, the fp32 intermediate a [P, I] and the
 * K-range partial sums of the activation-table pairs).  Its contents need
 * no initialisation.  A bounded device-side wait that ran out is recorded in
 * the int32 word at byte 8 of ws (0 = none); such a wait gives up after about
 * 1 to 4 seconds (measured by moe_selftest_wait_timeout's per-try times).  Calls that share a workspace
 * must not overlap on the GPU.
 * Requires H % 256 == 0, I % 128 == 0, k <= 32, x 16-byte aligned. */
size_t moe_vq2_expert_ffn_workspace_size(int T, int k, int E, int H, int I);
moe_status moe_vq2_expert_ffn(const moe_slot_table* table, const uint16_t* x,
                              const int32_t* expert_offsets, const int32_t* sorted_pair,
                              const float* weights, int T, int k, int mode, float* out_or_ypair,
                              uint8_t* pair_status, void* ws, size_t ws_bytes,
                              cudaStream_t stream);

/* Scratch-free variant of moe_vq2_expert_ffn (the pages have no counterpart:
 * this entry point exists for library users, not for the method).
 *
 * Some callers cannot call cudaMalloc (or any allocator) at the point where
 * they run the layer: a host that owns every byte of device memory through
 * its own fixed arena or pool and forbids library allocations, a real-time
 * or serving loop that must not pay allocation latency or risk an
 * out-of-memory in the middle of a step, or code running where allocation is
 * not allowed.  This call takes no workspace: it computes exactly what
 * moe_vq2_expert_ffn computes (same arguments and outputs) using a scratch
 * area of MOE_NOALLOC_SCRATCH_BYTES that is a static device array of the
 * library, held until the process exits.  Under CUDA's lazy module loading
 * (the default) the array is reserved on a device only when the library's
 * device code is first loaded there, which the first call of this entry
 * point forces; a caller that sizes its own arena from the free device
 * memory should make one call first, so that the 64 MiB are already taken.
 * It never calls cudaMalloc, cudaFree or an allocating library routine.
 *
 * Limits and rules:
 *   - the call fails with MOE_ERR_UNSUPPORTED, and enqueues nothing, when
 *     moe_vq2_expert_ffn_workspace_size(T, k, E, H, I) exceeds
 *     MOE_NOALLOC_SCRATCH_BYTES (64 MiB: at H = 4096, I = 2048 this covers
 *     decode batches of up to 32 tokens at top-8, and more);
 *   - the first call on each device looks up the device address of the
 *     static array (cudaGetSymbolAddress, with that device current) and
 *     keeps it for the life of the process; make that first call before any
 *     stream capture on the device.  The address belongs to the device's
 *     context: after cudaDeviceReset on a device, do not call this entry
 *     point on it again in the same process;
 *   - every call on a device shares the one array, which keeps the contents
 *     of the last call (no part of it needs to start at zero: each call
 *     writes what it reads).  Calls whose work overlaps on the GPU (on
 *     different streams, or from different host threads without ordering)
 *     race on it: order them on one stream or with events. */
#define MOE_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
moe_status moe_vq2_expert_ffn_noalloc(const moe_slot_table* table, const uint16_t* x,
                                      const int32_t* expert_offsets, const int32_t* sorted_pair,
                                      const float* weights, int T, int k, int mode, float* out_or_ypair,
                                      uint8_t* pair_status, cudaStream_t stream);

/* moe_vq2_expert_ffn in per-pair mode followed by moe_combine, in one call:
 * ypair and pair_status as moe_vq2_expert_ffn writes them, out_f32 /
 * out_bf16 as moe_combine(ypair, pair_to_sorted, weights, pair_status)
 * writes them, bit for bit.  For single-token calls whose slot table holds
 * VQ2 experts only, the combine runs inside the expert kernels (the last of
 * the pairs to finish 16 outputs writes them: no separate kernel).  Same
 * workspace as moe_vq2_expert_ffn. */
moe_status moe_vq2_expert_ffn_combine(const moe_slot_table* table, const uint16_t* x,
                                      const int32_t* expert_offsets, const int32_t* sorted_pair,
                                      const int32_t* pair_to_sorted, const float* weights, int T, int k,
                                      float* ypair, uint8_t* pair_status, float* out_f32, uint16_t* out_bf16,
                                      void* ws, size_t ws_bytes, cudaStream_t stream);

/* Deterministic combine: out[t] = sum over j = 0..k-1 (in that order) of
 * pair_status[t*k+j] * weights[t,j] * ypair[pair_to_sorted[t*k+j]].
 * ypair fp32 [P,H] (per-pair mode of moe_vq2_expert_ffn); out_f32 fp32
 * [T,H] and/or out_bf16 bf16 [T,H] (round to nearest even of the fp32
 * result); either may be NULL but not both (T = 0 is a no-op that reads
 * no pointer). */
moe_status moe_combine(const float* ypair, const int32_t* pair_to_sorted, const float* weights,
                       const uint8_t* pair_status, int T, int k, int H, float* out_f32,
                       uint16_t* out_bf16, cudaStream_t stream);

/* ---------------------------------------------------------------------- */
/* Experts the GPU does not hold, computed on the host's cores              */
/* ---------------------------------------------------------------------- */
/*
 * Tandem-vLLM page, "How it works": experts that miss the GPU cache are
 * computed by the CPU in parallel with the GPU; nothing is skipped or
 * substituted.  The GPU computes the pairs of its resident experts
 * (moe_vq2_expert_ffn reports the others with pair_status 0) and their
 * combine (moe_combine: the partial output); meanwhile the host computes
 * the pairs with status 0 (moe_cpu_expert_ffn: the remainder); the layer's
 * output is partial + remainder (moe_accumulate on the device).
 */
typedef struct moe_cpu_pool moe_cpu_pool;

/* A pool of host threads for moe_cpu_expert_ffn: threads - 1 workers (the
 * calling thread is the last one); threads <= 0 takes every hardware thread.
 * One pool serves one caller at a time.  Errors: MOE_ERR_INVALID_ARG,
 * MOE_ERR_NO_MEM (threads could not be started). */
moe_status moe_cpu_pool_create(int threads, moe_cpu_pool** out);
/* Threads of the pool, the calling one included (0 for NULL). */
int moe_cpu_pool_threads(const moe_cpu_pool* pool);
moe_status moe_cpu_pool_destroy(moe_cpu_pool* pool);

/* The remainder of the combine over the pairs the GPU did not compute:
 *     out[t] = sum over j = 0..k-1 (in that order) with gpu_status[t*k+j]
 *              == 0 of weights[t,j] * y_{t,j},
 *     y_{t,j} = Wd_e (silu(Wg_e x_t) * (Wu_e x_t)),  e = ids[t,j],
 * in fp32 on the pool's threads, from HOST copies of the experts' packed
 * codes and scales (the layouts of moe_vq2_pack / moe_fp4_pack: the bytes a
 * slot holds, e.g. an expert cache's page-locked base).
 * experts: host array [E] of descriptors with host pointers; the entries of
 * the experts that gpu_status names need all six buffers, the others are not
 * read.  codebook: host fp16 [128*4]; x: host bf16 [T, H]; ids int32 and
 * weights fp32 [T, k] (host copies of moe_route's outputs); gpu_status:
 * host uint8 [T*k] (pair_status of moe_vq2_expert_ffn, or computed from
 * moe_slot_table_resident before the GPU call); out: host fp32 [T, H],
 * written (rows of tokens without such a pair are zero).  Synchronous: it
 * returns when out is written; it touches no device memory and makes no
 * CUDA call, so it overlaps GPU work the caller enqueued before.
 * Requires H % 256 == 0, I % 128 == 0.  Errors: MOE_ERR_INVALID_ARG (a null
 * pointer, an id outside [0, E), a needed expert without buffers),
 * MOE_ERR_UNSUPPORTED (shape), MOE_ERR_NO_MEM (host scratch). */
moe_status moe_cpu_expert_ffn(moe_cpu_pool* pool, int H, int I, const uint16_t* codebook,
                              const moe_expert_desc* experts, int E, const uint16_t* x, const int32_t* ids,
                              const float* weights, const uint8_t* gpu_status, int T, int k, float* out);

/* dst[i] += src[i] for i < n, fp32, on the device (the GPU's partial output
 * plus the host's remainder, copied to the device).  Enqueue only. */
moe_status moe_accumulate(float* dst, const float* src, size_t n, cudaStream_t stream);

/* 1 if the table holds an entry for expert_id, 0 if not (from the table's
 * host mirror: no device access, no synchronisation); MOE_ERR_INVALID_ARG
 * for a null table or an id out of range. */
int moe_slot_table_resident(const moe_slot_table* t, int expert_id);

/* moe_vq2_pack / moe_fp4_pack on the host (the same packed layouts, for a
 * host-resident base or where no GPU is at hand): host pointers, no CUDA
 * call.  Same requirements and errors as the device calls. */
moe_status moe_vq2_pack_host(const uint8_t* codes, const uint16_t* scales, int rows, int K,
                             uint8_t* packed_codes, uint16_t* packed_scales);
moe_status moe_fp4_pack_host(const uint8_t* codes, const uint8_t* scales, int rows, int K,
                             uint8_t* packed_codes, uint8_t* packed_scales);

/* ---------------------------------------------------------------------- */
/* Confidence gate over an FP4 delta cache                                  */
/* ---------------------------------------------------------------------- */
/*
 * vLLM-Moet page, "2-bit experts on vLLM v0.24.0": a delta cache and a
 * confidence gate bring FP4 back where it matters; its bench table runs
 * "FP4 delta (auto) + confidence gate tau=0.60".  The pages say no more; this
 * library's reading:
 *   - a slot table of (at least) 2E entries holds expert e's 2-bit base at
 *     entry e and, while the delta cache holds them, e's FP4 weights at entry
 *     E + e (any number of them, set like any entry or by an expert cache);
 *   - the confidence of a pair is its router weight; a pair whose weight is
 *     at least tau and whose expert's FP4 entry is set uses the FP4 weights,
 *     every other pair the 2-bit base.
 * moe_confidence_gate writes gated_ids [T, k] (device int32): ids + E for
 * such pairs, ids otherwise (entry residency read on the device, so a
 * captured graph follows the cache).  moe_permute over the gated ids with
 * 2E experts, moe_vq2_expert_ffn over the 2E-entry table and moe_combine
 * then compute the layer; nothing else changes.  tau = 0.60 is the pages'
 * value; a tau above 1 turns the gate off.  ids, weights: device, from
 * moe_route_topk (E = the router's expert count).  Errors:
 * MOE_ERR_INVALID_ARG (null pointers, a table of fewer than 2E entries, NaN
 * tau). */
moe_status moe_confidence_gate(const moe_slot_table* table, const int32_t* ids, const float* weights, int T, int k,
                               int E, float tau, int32_t* gated_ids, cudaStream_t stream);

/* ---------------------------------------------------------------------- */
/* VQ2 encoder: dense weights -> codebook, codes and scales                 */
/* ---------------------------------------------------------------------- */
/*
 * The vLLM-Moet page ("2-bit experts on vLLM v0.24.0") puts the routed
 * experts on a sign-symmetric 2-bit codebook (naive 2-bit fails through sign
 * asymmetry); the German vLLM-Moet page quantises the weights at start-up.
 * The pages give no algorithm; this library's (every decision in fp32 in one
 * fixed operation order, the k-means sums exact integers, so results are the
 * same on every run):
 *   1. block scale sigma[r, b] = sqrt(mean of W[r, i]^2 over the 128 inputs
 *      of block b); normalised group vectors u = W[r, 4g..4g+3] / sigma;
 *   2. codebook (moe_vq2_train_codebook): k-means over the normalised
 *      vectors with the codebook read as 128 pairs {+c, -c}: u goes to the
 *      pair i maximising 2 |u . c_i| - |c_i|^2, sign s = sign(u . c_i); c_i
 *      becomes the mean of s u over its members; started from the vectors at
 *      init_idx (host int64 [128], indices into the rows*K/4 groups,
 *      row-major); the codebook is the result rounded to fp16;
 *   3. encoding (moe_vq2_encode): the block's scale starts at sigma; each
 *      iteration assigns its 32 groups (u = W / scale) and refits the scale by
 *      least squares (sum W.q / sum q.q, q = s c_i); the scale is rounded to
 *      fp16 and the groups assigned once more: codes uint8 [rows, K/4] (bit 7
 *      = 1 for s = -1), scales fp16 [rows, K/128], the logical layout of
 *      moe_vq2_pack.
 * W: device fp32 [rows, K] row-major, K % 128 == 0.  ws: device scratch of
 * moe_vq2_encoder_workspace_size(rows, K) bytes.  centroids (optional):
 * device fp32 [128*4], the codebook before rounding.  Enqueue only.
 * Errors: MOE_ERR_INVALID_ARG (null pointers, an index out of range, a
 * workspace too small), MOE_ERR_UNSUPPORTED (K % 128 != 0), MOE_ERR_CUDA.
 */
size_t moe_vq2_encoder_workspace_size(int rows, int K);
moe_status moe_vq2_train_codebook(const float* W, int rows, int K, const int64_t* init_idx, int iters,
                                  uint16_t* codebook, float* centroids, void* ws, size_t ws_bytes,
                                  cudaStream_t stream);
moe_status moe_vq2_encode(const float* W, int rows, int K, const uint16_t* codebook, int iters, uint8_t* codes,
                          uint16_t* scales, void* ws, size_t ws_bytes, cudaStream_t stream);

/* Boot self-check (Tandem-vLLM page, "New in 0.2.0": each kernel is checked
 * against a reference at boot).  Runs a tiny layer (hidden 256, intermediate
 * 128, 8 experts, top-2) through the entry points above on the current
 * device: the router and top-k step by step and fused, the permutation, the
 * expert FFN on 1, 4, 16 and 128 tokens (the table kernels, the
 * small-batch mma.sync kernels and the tcgen05 kernels), an all-VQ2 and a
 * mixed VQ2/FP4 layer, both output modes, the fused expert-FFN + combine and
 * a layer with two experts not resident.  The inputs are drawn on the GPU
 * from a counter-based generator (SplitMix64); the results are compared with
 * values computed from the same draws by the CPU reference and compiled into
 * the library: routing (logits bits, ids, offsets, permutation) exactly,
 * router weights within 1e-6, layer outputs within max |err| <= 2e-2 *
 * rms(ref) and sum |err| <= 2e-3 * sum |ref|.
 * Unlike the hot-path calls it allocates and frees device memory (a few MB),
 * synchronises `stream` and must not be called while the stream is being
 * captured.  Returns MOE_OK, MOE_ERR_MISMATCH (moe_last_error() names the
 * first failing case and value), MOE_ERR_NO_MEM, MOE_ERR_CUDA, or the error
 * of a failing entry point. */
moe_status moe_selftest(cudaStream_t stream);

/* Self-check of the bounded-wait pattern the kernels use (a limited loop of
 * mbarrier.try_wait, then an error code in the workspace and a return): one
 * thread waits on two mbarriers that nothing completes, with plain try_wait
 * (64 tries) and with try_wait and a 1 us suspend hint (256 tries).  Both give
 * up, record their codes and return, so the context stays usable.  codes:
 * HOST int[6]: the two recorded codes (MOE_DEVERR_WAIT_FULL = 1,
 * MOE_DEVERR_WAIT_EMPTY = 2), the two waits' results (0 = gave up) and the
 * microseconds each wait took.  Allocates and frees 32 bytes, synchronises
 * `stream`; not while the stream is being captured.  Returns MOE_OK when both
 * waits gave up as designed, else MOE_ERR_MISMATCH, MOE_ERR_NO_MEM or
 * MOE_ERR_CUDA. */
moe_status moe_selftest_wait_timeout(int* codes, cudaStream_t stream);

/* Number of kernel launches the library has issued on the host since it was
 * loaded, over all devices and threads (atomic).  A launch made while a
 * stream is being captured counts once, as the one kernel node it adds to
 * the graph; replays of the graph are not counted.  Never fails. */
uint64_t moe_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_VQ2_H */
