// Incremental causal FAVOR+: one new token per (b, h), the prefix state
// carried between calls.
//
// "From Performer to Linear Attention" (Su), §Concentrating Attention: a
// causal linear attention is a unidirectional RNN.  "Performer — Rethinking
// Attention with Performers" (digest), §Methods, causal bullet: the state is
// the prefix sum G_t = sum_{s<=t} phi(k_s) v_s^T (with z_t = sum phi(k_s)
// beside it).  Per call and head:
//   state += phi(s k) [v ; 1]^T,  o = phi(s q)^T state[:, :d] / phi(s q)^T state[:, d]
// The state is fp32 [m][d+1] per head, row i = feature i; its key features
// use the reference R = max_i |w_i|^2 / 2 - 40 of the sequence kernels, so a
// state from favor_decode_prefill continues here.  The query features use
// s |q| max_i |w_i| - 20 (the largest possible exponent less 20): a per-query
// constant, it cancels in the ratio ("From Performer to Linear Attention",
// §Simple Derivation).
//
// One CTA per head.  Bound by the state's HBM traffic: m (d+1) fp32 read and
// written per head and token (133 KB at m = 256, d = 64); Omega (m x d fp32)
// is read by every CTA and stays in L2.
#include "common.cuh"

namespace favor {
namespace {

constexpr int kDecThreads = 256;
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kDecFeat = kMaxM / kDecThreads;      // features per thread (m <= 512)
constexpr int kDecCols = (kMaxD + 1 + 31) / 32;    // state columns per lane (d + 1 <= 129)
constexpr float kDecQueryHeadroom = 20.0f;

template <typename T>
__global__ void __launch_bounds__(kDecThreads) decode_step_kernel(const T* __restrict__ q, const T* __restrict__ k,
                                                                  const T* __restrict__ v, T* __restrict__ o,
                                                                  const float* __restrict__ omega, int d, int m,
                                                                  float scale, float* __restrict__ state,
                                                                  int32_t* __restrict__ status) {
  __shared__ float qs[kMaxD], ks[kMaxD], vs[kMaxD + 1];
  __shared__ float phq[kMaxM], phk[kMaxM];
  __shared__ float part[kDecWarps][kMaxD + 1];
  __shared__ float num[kMaxD + 1];
  __shared__ float wred[kDecWarps];
  __shared__ float sqn[2];
  const int bh = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ld = d + 1;

  for (int j = tid; j < d; j += kDecThreads) {
    const size_t e = (size_t)bh * d + j;
    qs[j] = to_f32(q[e]);
    ks[j] = to_f32(k[e]);
    vs[j] = to_f32(v[e]);
  }
  if (tid == 0) vs[d] = 1.f;
  __syncthreads();
  if (warp < 2) {
    const float* x = warp == 0 ? qs : ks;
    float a = 0.f;
    for (int j = lane; j < d; j += 32) a = fmaf(x[j], x[j], a);
    a = warp_sum(a);
    if (lane == 0) sqn[warp] = a;
  }

  // w_f.q, w_f.k and |w_f|^2 for the features f = tid + 256 i of this thread
  float pq[kDecFeat], pk[kDecFeat];
  float w2max = 0.f;
#pragma unroll
  for (int i = 0; i < kDecFeat; ++i) {
    const int f = tid + i * kDecThreads;
    float dq = 0.f, dk = 0.f, w2 = 0.f;
    if (f < m) {
      const float* w = omega + (size_t)f * d;
      for (int j = 0; j < d; ++j) {
        const float wj = __ldg(w + j);
        dq = fmaf(wj, qs[j], dq);
        dk = fmaf(wj, ks[j], dk);
        w2 = fmaf(wj, wj, w2);
      }
      w2max = fmaxf(w2max, w2);
    }
    pq[i] = dq;
    pk[i] = dk;
  }
  w2max = warp_max(w2max);
  if (lane == 0) wred[warp] = w2max;
  __syncthreads();
  float w2 = wred[0];
  for (int i = 1; i < kDecWarps; ++i) w2 = fmaxf(w2, wred[i]);
  const float R = 0.5f * w2 - kKeyHeadroom;
  const float bq = scale * sqrtf(w2) * sqrtf(sqn[0]) - kDecQueryHeadroom;
  const float hk = 0.5f * scale * scale * sqn[1];
#pragma unroll
  for (int i = 0; i < kDecFeat; ++i) {
    const int f = tid + i * kDecThreads;
    if (f < m) {
      phk[f] = expf(scale * pk[i] - hk - R);
      phq[f] = expf(scale * pq[i] - bq);
    }
  }
  __syncthreads();

  // state rows: warp w takes features w, w + 8, ...; lane l columns l + 32c,
  // so every row is read and written with whole-warp coalesced accesses
  float* st = state + (size_t)bh * m * ld;
  float vr[kDecCols], acc[kDecCols];
#pragma unroll
  for (int c = 0; c < kDecCols; ++c) {
    const int j = lane + 32 * c;
    vr[c] = j < ld ? vs[j] : 0.f;
    acc[c] = 0.f;
  }
#pragma unroll 4
  for (int f = warp; f < m; f += kDecWarps) {
    float* row = st + (size_t)f * ld;
    const float a = phk[f], b = phq[f];
#pragma unroll
    for (int c = 0; c < kDecCols; ++c) {
      const int j = lane + 32 * c;
      if (j < ld) {
        const float g = fmaf(a, vr[c], row[j]);
        row[j] = g;
        acc[c] = fmaf(b, g, acc[c]);
      }
    }
  }
#pragma unroll
  for (int c = 0; c < kDecCols; ++c) {
    const int j = lane + 32 * c;
    if (j < ld) part[warp][j] = acc[c];
  }
  __syncthreads();
  // numerators and normaliser, warps summed in a fixed order
  for (int j = tid; j < ld; j += kDecThreads) {
    float s_ = 0.f;
    for (int w = 0; w < kDecWarps; ++w) s_ += part[w][j];
    num[j] = s_;
  }
  __syncthreads();
  const float den = num[d];
  if (tid == 0 && (!(den > 0.f) || !isfinite(den))) report_status(status, FAVOR_ERR_NONFINITE);
  const float inv = 1.0f / den;
  for (int j = tid; j < d; j += kDecThreads) o[(size_t)bh * d + j] = from_f32<T>(num[j] * inv);
}

}  // namespace

cudaError_t launch_decode_step(const void* q, const void* k, const void* v, void* o, int BH, int d,
                               const float* omega, int m, bool bf16, float scale, float* state, int32_t* status,
                               cudaStream_t stream) {
  if (bf16) {
    decode_step_kernel<__nv_bfloat16><<<BH, kDecThreads, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
        static_cast<const __nv_bfloat16*>(v), static_cast<__nv_bfloat16*>(o), omega, d, m, scale, state, status);
  } else {
    decode_step_kernel<float><<<BH, kDecThreads, 0, stream>>>(static_cast<const float*>(q),
                                                              static_cast<const float*>(k),
                                                              static_cast<const float*>(v), static_cast<float*>(o),
                                                              omega, d, m, scale, state, status);
  }
  return cudaGetLastError();
}

}  // namespace favor
