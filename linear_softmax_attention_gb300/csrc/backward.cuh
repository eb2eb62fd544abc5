// Backward passes (simt.cu): gradients of the bidirectional and causal
// forward passes with respect to Q, K and V.
#pragma once

#include "common.cuh"

namespace favor {

// dQ, dK, dV of the causal pass for dO (workspace: bwd_plan(s).bytes);
// fm: favor_feature_map.
cudaError_t simt_bwd_causal(const void* Q, const void* K, const void* V, const void* dO, void* dQ, void* dK,
                            void* dV, const float* omega, float scale, const Shape& s, bool bf16, void* ws, int32_t* st,
                            cudaStream_t stream, int fm);

}  // namespace favor
