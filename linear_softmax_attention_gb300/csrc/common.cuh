// Shared device/host helpers of the FAVOR+ library (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "favor.h"

namespace favor {

constexpr int kMaxD = 128;
constexpr int kMaxM = 512;
constexpr float kLog2e = 1.4426950408889634f;

// ---- element loads / stores -------------------------------------------------
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// ---- key reference ------------------------------------------------------------
// The workspace header holds, for each block of 8 rows of Omega, the largest
// squared row norm (written by the prep kernel).  R = max_i |w_i|^2 / 2 - 40
// bounds every key-feature exponent from above by 40 (prep.cu explains why);
// W = max_i |w_i|.
constexpr float kKeyHeadroom = 40.0f;
constexpr int kPrepRows = 8;
__device__ __forceinline__ void key_reference(const float* hdr, int m, float* R, float* W) {
  const int n = (m + kPrepRows - 1) / kPrepRows;
  float w2 = hdr[0];
  for (int i = 1; i < n; ++i) w2 = fmaxf(w2, hdr[i]);
  *R = 0.5f * w2 - kKeyHeadroom;
  *W = sqrtf(w2);
}

// ---- device-side status -----------------------------------------------------
// First non-zero code wins; later errors do not overwrite it.
__device__ __forceinline__ void report_status(int32_t* status, int code) {
  if (status != nullptr) atomicCAS(reinterpret_cast<int*>(status), 0, code);
}

// ---- reductions -------------------------------------------------------------
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
// Block-wide max; `scratch` holds >= 32 floats; every thread gets the result.
__device__ __forceinline__ float block_max(float v, float* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = (blockDim.x + 31) >> 5;
  v = warp_max(v);
  __syncthreads();
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  float r = (lane < nwarps) ? scratch[lane] : -INFINITY;
  r = warp_max(r);
  return r;
}

}  // namespace favor

// ---- host-side launchers (defined in the .cu files) -------------------------
namespace favor {

struct Shape {
  int B, H, L, d, m;
  int BH() const { return B * H; }
};

// Every workspace starts with a 256-byte header written by launch_prep at the
// start of each state stage: per block of 8 rows of Omega, the largest
// squared row norm (read back through key_reference).
constexpr size_t kWsHeader = 256;

// Workspace plan of the CUDA-core path.
struct SimtPlan {
  int n_fb;          // feature blocks of kSimtFB features
  int n_split;       // bidirectional: L splits per head; causal: superchunks
  int chunk;         // tokens per split / superchunk (multiple of the tile)
  size_t off_partS, off_state, bytes;
};

SimtPlan simt_plan(bool causal, const Shape& s);
// Backward (simt.cu): workspace = the forward state's plus dN^ [BH][L][d+1],
// then for the bidirectional pass dS~ partials and dS~, for the causal pass
// one [m][d+1] state per (head, chunk of c_chunk tokens) in the same place.
struct BwdPlan {
  SimtPlan fwd;
  int c_chunk, c_n;  // causal: tokens per chunk, chunks per head
  size_t off_dn, off_dpart, off_dstate, off_cstate, bytes;
};
BwdPlan bwd_plan(const Shape& s);
cudaError_t simt_bwd_bidir(const void* Q, const void* K, const void* V, const void* dO, void* dQ, void* dK, void* dV,
                           const float* omega, float scale, const Shape& s, bool bf16, void* ws, int32_t* st,
                           cudaStream_t stream, int fm);
cudaError_t simt_state_export(const void* K, const void* V, const float* omega, float scale, const Shape& s,
                              bool bf16, void* ws, float* state, cudaStream_t stream);
// One decode step for every (b, h): decode.cu.
cudaError_t launch_decode_step(const void* q, const void* k, const void* v, void* o, int BH, int d,
                               const float* omega, int m, bool bf16, float scale, float* state, int32_t* status,
                               cudaStream_t stream);
// fm: favor_feature_map (FAVOR_FM_PRF, FAVOR_FM_RELU or FAVOR_FM_ELU1)
cudaError_t simt_bidir_state(const void* K, const void* V, const float* omega, float scale,
                             const Shape& s, bool bf16, void* ws, int32_t* st, cudaStream_t stream,
                             int fm = FAVOR_FM_PRF);
cudaError_t simt_bidir_output(const void* Q, void* O, const float* omega, float scale,
                              const Shape& s, bool bf16, void* ws, int32_t* st, cudaStream_t stream,
                              int fm = FAVOR_FM_PRF);
cudaError_t simt_causal_state(const void* K, const void* V, const float* omega, float scale,
                              const Shape& s, bool bf16, void* ws, int32_t* st, cudaStream_t stream,
                              int fm = FAVOR_FM_PRF);
cudaError_t simt_causal_output(const void* Q, const void* K, const void* V, void* O,
                               const float* omega, float scale, const Shape& s, bool bf16, void* ws,
                               int32_t* st, cudaStream_t stream, int fm = FAVOR_FM_PRF);

// The checked, dispatched body of every forward entry point (stage: 1 state,
// 2 output, 3 both).
favor_status run_call(bool causal, int stage, const void* Q, const void* K, const void* V, void* O, int B, int H,
                      int L, int d, const float* omega, int m, favor_dtype dt, float qk_scale, void* workspace,
                      size_t ws_bytes, int32_t* dev_status, void* stream);

// Raises a kernel's dynamic shared-memory limit once per device and size, so
// that calls made later (including under CUDA graph capture) issue no
// attribute call.
cudaError_t ensure_dynamic_smem(const void* kernel, size_t bytes);
// SM count of the current device (cached).
int sm_count();

// Row-norm maxima (and optionally the fp16 Omega image) into the workspace;
// also zeroes `n_counters` words at `counters` (the split-merge counters).
cudaError_t launch_prep(const float* omega, int m, int d, float* header, uint8_t* image, uint32_t* counters,
                        int n_counters, cudaStream_t stream);

cudaError_t launch_build_orf(uint64_t seed, int m, int d, int orthogonal, float* omega,
                             cudaStream_t stream);

}  // namespace favor
