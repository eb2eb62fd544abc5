// Projection matrix Omega for FAVOR+: orthogonal random features (ORF) or iid.
//
// "Performer — Rethinking Attention with Performers" (digest), §Methods, ORF
// bullet: the rows of the random projection are orthogonalised by
// Gram–Schmidt; the Zettelkasten note on orthogonality: block by block when
// m > d.  arXiv:2009.14794v4 summary, §A.2 FAVOR+: orthogonality is imposed
// while each sample keeps its marginal.  Here each orthonormal row is given
// the length of an independent N(0, I_d) vector so that its marginal stays
// N(0, I_d).
#include "common.cuh"

namespace favor {
namespace {

// SplitMix64 (Steele, Lea & Flood 2014): word i of the stream seeded `seed`.
__device__ __forceinline__ uint64_t splitmix_word(uint64_t seed, uint64_t i) {
  uint64_t z = seed + (i + 1ull) * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// Box–Muller (cosine branch) from two 23-bit fields; u = (k + 1/2) / 2^23 is
// exact in fp32.
__device__ __forceinline__ float normal_from_word(uint64_t w) {
  const float u1 = (static_cast<float>(static_cast<uint32_t>(w >> 41)) + 0.5f) * (1.0f / 8388608.0f);
  const float u2 =
      (static_cast<float>(static_cast<uint32_t>((w >> 18) & 0x7FFFFFull)) + 0.5f) * (1.0f / 8388608.0f);
  return sqrtf(-2.0f * logf(u1)) * cospif(2.0f * u2);
}

constexpr int kTPR = 4;                 // threads per row of a block
constexpr int kCW = kMaxD / kTPR;       // max columns per thread

__device__ __forceinline__ float group4_sum(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 1);
  v += __shfl_xor_sync(0xffffffffu, v, 2);
  return v;
}

// One CTA per d x d block; thread (row r = tid/4, part p = tid%4) keeps
// columns p*cw .. p*cw+cw-1 of row r in registers.  Two Gram–Schmidt sweeps
// (the second re-orthogonalises, which fp32 needs), then row r is scaled by
// the length of its own Gaussian vector.
__global__ void __launch_bounds__(kMaxD * kTPR) orf_block_kernel(uint64_t seed, int m, int d,
                                                                 float* __restrict__ omega) {
  __shared__ float qbuf[2][kMaxD];
  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  const int r = tid / kTPR;
  const int p = tid % kTPR;
  const int cw = (d + kTPR - 1) / kTPR;
  const bool row_ok = r < d;

  float g[kCW];
  float len2 = 0.f;
#pragma unroll
  for (int k = 0; k < kCW; ++k) {
    const int c = p * cw + k;
    g[k] = 0.f;
    if (k < cw && c < d && row_ok) {
      const uint64_t idx = (((uint64_t)b * d + r) * d + c) * 2ull;
      g[k] = normal_from_word(splitmix_word(seed, idx));
      const float x = normal_from_word(splitmix_word(seed, idx + 1ull));
      len2 = fmaf(x, x, len2);
    }
  }
  const float len = sqrtf(group4_sum(len2));

  for (int sweep = 0; sweep < 2; ++sweep) {
    for (int i = 0; i < d; ++i) {
      float* q = qbuf[i & 1];
      float n2 = 0.f;
#pragma unroll
      for (int k = 0; k < kCW; ++k) n2 = fmaf(g[k], g[k], n2);
      n2 = group4_sum(n2);
      if (r == i) {
        const float inv = 1.0f / sqrtf(n2);
#pragma unroll
        for (int k = 0; k < kCW; ++k) {
          g[k] *= inv;
          const int c = p * cw + k;
          if (k < cw && c < d) q[c] = g[k];
        }
      }
      __syncthreads();
      float dot = 0.f;
#pragma unroll
      for (int k = 0; k < kCW; ++k) {
        const int c = p * cw + k;
        if (k < cw && c < d) dot = fmaf(q[c], g[k], dot);
      }
      dot = group4_sum(dot);
      if (row_ok && r > i) {
#pragma unroll
        for (int k = 0; k < kCW; ++k) {
          const int c = p * cw + k;
          if (k < cw && c < d) g[k] = fmaf(-dot, q[c], g[k]);
        }
      }
    }
  }
  const int row = b * d + r;
  if (row_ok && row < m) {
#pragma unroll
    for (int k = 0; k < kCW; ++k) {
      const int c = p * cw + k;
      if (k < cw && c < d) omega[(size_t)row * d + c] = g[k] * len;
    }
  }
}

__global__ void iid_kernel(uint64_t seed, int m, int d, float* __restrict__ omega) {
  const int n = m * d;
  for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < n; e += gridDim.x * blockDim.x) {
    omega[e] = normal_from_word(splitmix_word(seed, (uint64_t)e * 2ull));
  }
}

}  // namespace

cudaError_t launch_build_orf(uint64_t seed, int m, int d, int orthogonal, float* omega,
                             cudaStream_t stream) {
  if (orthogonal) {
    const int nb = (m + d - 1) / d;
    const int threads = ((d * kTPR + 31) / 32) * 32;
    orf_block_kernel<<<nb, threads, 0, stream>>>(seed, m, d, omega);
  } else {
    const int n = m * d;
    iid_kernel<<<(n + 255) / 256, 256, 0, stream>>>(seed, m, d, omega);
  }
  return cudaGetLastError();
}

}  // namespace favor
