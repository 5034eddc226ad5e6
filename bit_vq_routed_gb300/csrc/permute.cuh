// The token -> expert permutation's launcher with its workspace (permute.cu).
#pragma once

#include "common.cuh"

namespace moe {

// From this many pairs the permutation runs over chunks of 1024 pairs on
// many CTAs (three launches), when the caller's workspace holds
// permute_ws_bytes(P, E); below, or without that workspace, one CTA.
constexpr int PERMUTE_MULTI_P = 8192;
size_t permute_ws_bytes(int P, int E);
moe_status launch_permute_ws(const int32_t* ids, int P, int E, int32_t* offsets, int32_t* sorted_pair,
                             int32_t* pair_to_sorted, cudaStream_t s, void* ws, size_t ws_bytes);

}  // namespace moe
