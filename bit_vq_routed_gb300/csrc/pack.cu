// Logical -> packed weight layouts (see moe_vq2.h), and the slot writer.
#include "common.cuh"
#include "slot_batch.cuh"

namespace moe {
namespace {

__global__ void vq2_pack_codes(const uint8_t* __restrict__ src, int rows, int K, uint8_t* __restrict__ dst) {
    const int G = K / 4, KB = K / 128;
    const long n = (long)rows * G;
    for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x) {
        int r = (int)(i / G), q = (int)(i % G);
        dst[vq2_tile_offset(r / 16, q / 32, KB) + vq2_in_tile(r % 16, q % 32)] = src[i];
    }
}

__global__ void vq2_pack_scales(const uint16_t* __restrict__ src, int rows, int K, uint16_t* __restrict__ dst) {
    const int KB = K / 128;
    const long n = (long)rows * KB;
    for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x) {
        int r = (int)(i / KB), kb = (int)(i % KB);
        dst[((size_t)(r / 16) * KB + kb) * 16 + r % 16] = src[i];
    }
}

__global__ void fp4_pack_codes(const uint8_t* __restrict__ src, int rows, int K, uint8_t* __restrict__ dst) {
    const int NB = K / 2, KT = K / 64;
    const long n = (long)rows * NB;
    for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x) {
        int r = (int)(i / NB), b = (int)(i % NB);
        dst[((size_t)(r / 16) * KT + b / 32) * 512 + fp4_in_tile(r % 16, b % 32)] = src[i];
    }
}

__global__ void fp4_pack_scales(const uint8_t* __restrict__ src, int rows, int K, uint8_t* __restrict__ dst) {
    const int KB = K / 32;
    const long n = (long)rows * KB;
    for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long)gridDim.x * blockDim.x) {
        int r = (int)(i / KB), kb = (int)(i % KB);
        dst[((size_t)(r / 16) * KB + kb) * 16 + r % 16] = src[i];
    }
}

__global__ void slot_set_kernel(SlotDesc* table, int expert_id, SlotDesc d) { table[expert_id] = d; }

// (distinct ids: the writes of one batch do not depend on their order)
__global__ void slot_set_many_kernel(SlotDesc* table, SlotBatch b) {
    if ((int)threadIdx.x < b.n) table[b.ids[threadIdx.x]] = b.d[threadIdx.x];
}

unsigned grid_for(long n) {
    long b = (n + 255) / 256;
    long cap = (long)num_sms() * 16;
    return (unsigned)(b < 1 ? 1 : (b > cap ? cap : b));
}

}  // namespace

moe_status launch_vq2_pack(const uint8_t* codes, const uint16_t* scales, int rows, int K, uint8_t* pc,
                           uint16_t* ps, cudaStream_t s) {
    count_launch();
    vq2_pack_codes<<<grid_for((long)rows * K / 4), 256, 0, s>>>(codes, rows, K, pc);
    count_launch();
    vq2_pack_scales<<<grid_for((long)rows * K / 128), 256, 0, s>>>(scales, rows, K, ps);
    MOE_LAUNCH_CHECK("moe_vq2_pack: launch");
    return MOE_OK;
}

moe_status launch_fp4_pack(const uint8_t* codes, const uint8_t* scales, int rows, int K, uint8_t* pc,
                           uint8_t* ps, cudaStream_t s) {
    count_launch();
    fp4_pack_codes<<<grid_for((long)rows * K / 2), 256, 0, s>>>(codes, rows, K, pc);
    count_launch();
    fp4_pack_scales<<<grid_for((long)rows * K / 32), 256, 0, s>>>(scales, rows, K, ps);
    MOE_LAUNCH_CHECK("moe_fp4_pack: launch");
    return MOE_OK;
}

moe_status launch_slot_set_many(SlotDesc* table, const SlotBatch& b, cudaStream_t s) {
    if (b.n <= 0) return MOE_OK;
    count_launch();
    slot_set_many_kernel<<<1, SLOT_BATCH, 0, s>>>(table, b);
    MOE_LAUNCH_CHECK("moe_expert_cache_fetch: slot-table launch");
    return MOE_OK;
}

moe_status launch_slot_set(SlotDesc* table, int expert_id, SlotDesc d, cudaStream_t s) {
    count_launch();
    slot_set_kernel<<<1, 1, 0, s>>>(table, expert_id, d);
    MOE_LAUNCH_CHECK("moe_slot_table_set: launch");
    return MOE_OK;
}

}  // namespace moe
