// Tensor-core (tcgen05) FAVOR+ path: bf16 operands, fp32 accumulation.
#pragma once

#include "common.cuh"

namespace favor {

bool tc_supported(bool causal, int d, int m, bool bf16);
size_t tc_workspace_bytes(bool causal, const Shape& s);
// fm: favor_feature_map (FAVOR_FM_PRF, FAVOR_FM_RELU or FAVOR_FM_ELU1).  zvec
// (bidirectional, d = 64, optional): the merged state's normaliser row per
// head, [BH][m] fp32, besides the bf16 image.
cudaError_t tc_state(bool causal, const void* K, const void* V, const float* omega, float scale, const Shape& s,
                     void* ws, int32_t* status, cudaStream_t stream, int fm = FAVOR_FM_PRF, float* zvec = nullptr);
cudaError_t tc_output(bool causal, const void* Q, const void* K, const void* V, void* O, const float* omega,
                      float scale, const Shape& s, void* ws, int32_t* status, cudaStream_t stream,
                      int fm = FAVOR_FM_PRF);

// Workspace of the d = 64 bidirectional tensor-core forward (tc.cu).  The
// tensor-core backward (tc_bwd.cu) runs that forward's state stage, keeps its
// layout and puts the gradient's state image after it.
struct TcLayout {
  size_t off_omega_img, off_counters, off_partS, off_state_img, bytes;
};
TcLayout tc_bidir_layout(const Shape& s);

// Gradients of the bidirectional pass on the tensor cores (tc_bwd.cu): bf16,
// d = 64, m in {128, 256}
bool tc_bwd_supported(bool causal, int d, int m, bool bf16);
size_t tc_bwd_workspace_bytes(const Shape& s);
cudaError_t tc_bwd_bidir(const void* Q, const void* K, const void* V, const void* dO, void* dQ, void* dK, void* dV,
                         const float* omega, float scale, const Shape& s, void* ws, int32_t* status,
                         cudaStream_t stream, int fm);

// d = 128, one feature block per CTA (tc_fs.cu); reached through the calls above
bool fs_supported(bool causal, int d, int m, bool bf16);
size_t fs_workspace_bytes(bool causal, const Shape& s);
cudaError_t fs_state(bool causal, const void* K, const void* V, const float* omega, float scale, const Shape& s,
                     void* ws, int32_t* status, cudaStream_t stream, int fm);
cudaError_t fs_output(bool causal, const void* Q, const void* K, const void* V, void* O, float scale, const Shape& s,
                      void* ws, int32_t* status, cudaStream_t stream, int fm);

}  // namespace favor
