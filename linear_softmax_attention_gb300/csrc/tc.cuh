// Tensor-core (tcgen05) FAVOR+ path: bf16 operands, fp32 accumulation.
#pragma once

#include "common.cuh"

namespace favor {

bool tc_supported(bool causal, int d, int m, bool bf16);
size_t tc_workspace_bytes(bool causal, const Shape& s);
// fm: favor_feature_map (FAVOR_FM_PRF or FAVOR_FM_RELU; 1 + elu runs on the CUDA-core kernels)
cudaError_t tc_state(bool causal, const void* K, const void* V, const float* omega, float scale, const Shape& s,
                     void* ws, int32_t* status, cudaStream_t stream, int fm = FAVOR_FM_PRF);
cudaError_t tc_output(bool causal, const void* Q, const void* K, const void* V, void* O, const float* omega,
                      float scale, const Shape& s, void* ws, int32_t* status, cudaStream_t stream,
                      int fm = FAVOR_FM_PRF);

// d = 128, one feature block per CTA (tc_fs.cu); reached through the calls above
bool fs_supported(bool causal, int d, int m, bool bf16);
size_t fs_workspace_bytes(bool causal, const Shape& s);
cudaError_t fs_state(bool causal, const void* K, const void* V, const float* omega, float scale, const Shape& s,
                     void* ws, int32_t* status, cudaStream_t stream, int fm);
cudaError_t fs_output(bool causal, const void* Q, const void* K, const void* V, void* O, float scale, const Shape& s,
                      void* ws, int32_t* status, cudaStream_t stream, int fm);

}  // namespace favor
