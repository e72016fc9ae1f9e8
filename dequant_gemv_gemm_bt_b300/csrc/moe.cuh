// Mixture-of-experts harness-step launchers.
#pragma once
#include <algorithm>
#include "bt_common.cuh"

namespace bt {
cudaError_t launch_moe_route(const int32_t* ids, int tokens, int top_k, int E, int32_t* offsets,
                             int32_t* pair_index, int32_t* pair_row, int32_t* pair_token, cudaStream_t st);
cudaError_t launch_swiglu(const void* in, bt_dtype id, int rows, int inter, void* out, bt_dtype od,
                          cudaStream_t st);
cudaError_t launch_combine(const void* yg, bt_dtype yd, const float* gates, const int32_t* pair_row, int tokens,
                           int top_k, int hidden, void* out, bt_dtype od, cudaStream_t st);
}  // namespace bt
