// Batched slot-table writes: up to SLOT_BATCH descriptor writes to distinct
// entries in one launch (a kernel parameter of about 2 KB), used by the
// expert cache to publish one fetch's evictions and new entries at once.
#pragma once

#include "common.cuh"

namespace moe {

constexpr int SLOT_BATCH = 32;
struct SlotBatch {
    int n;
    int ids[SLOT_BATCH];
    SlotDesc d[SLOT_BATCH];
};
static_assert(sizeof(SlotBatch) <= 4000, "kernel parameter size");
moe_status launch_slot_set_many(SlotDesc* table, const SlotBatch& b, cudaStream_t s);

}  // namespace moe
