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

__device__ __forceinline__ float group4_sum(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 1);
  v += __shfl_xor_sync(0xffffffffu, v, 2);
  return v;
}

// One CTA per d x d block; thread (row r = tid/4, part p = tid%4) keeps
// columns p*CW .. p*CW+CW-1 of row r in registers (CW = ceil(d/4) rounded up
// to a multiple of 4; columns >= d are zero).
//
// Sweep 1 is modified Gram–Schmidt, row by row.  fp32 leaves the rows
// orthogonal only to about kappa * 2^-24, so a second pass re-orthogonalises
// them; as the rows are then orthonormal up to that small error E, the pass
// is one classical step q_r - sum_{s<r} (q_s . q_r) q_s computed for all rows
// at once, which equals a second modified sweep up to O(E^2).  Finally row r
// is scaled by the length of its own Gaussian vector.
template <int CW>
__global__ void __launch_bounds__(kMaxD * kTPR) orf_block_kernel(uint64_t seed, int m, int d,
                                                                 float* __restrict__ omega) {
  extern __shared__ __align__(16) float orf_smem[];
  float* qbuf = orf_smem;                         // [2][kTPR * CW] unit row of the current step
  float* rows = orf_smem + 2 * kTPR * CW;         // [d][kTPR * CW] all rows after sweep 1
  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  const int r = tid / kTPR;
  const int p = tid % kTPR;
  const bool row_ok = r < d;
  constexpr int RW = kTPR * CW;                   // floats per stored row

  float g[CW];
  float len2 = 0.f;
#pragma unroll
  for (int k = 0; k < CW; ++k) {
    const int c = p * CW + k;
    g[k] = 0.f;
    if (c < d && row_ok) {
      const uint64_t idx = (((uint64_t)b * d + r) * d + c) * 2ull;
      g[k] = normal_from_word(splitmix_word(seed, idx));
      const float x = normal_from_word(splitmix_word(seed, idx + 1ull));
      len2 = fmaf(x, x, len2);
    }
  }
  const float len = sqrtf(group4_sum(len2));

  // ---- sweep 1: modified Gram–Schmidt.  Every thread executes every shuffle
  // (full-warp masks); only the values they carry depend on the thread's role.
  for (int i = 0; i < d; ++i) {
    float* q = qbuf + (i & 1) * RW;
    const bool norm_row = (r == i);
    float n2[4] = {0.f, 0.f, 0.f, 0.f};
    if (norm_row) {
#pragma unroll
      for (int k = 0; k < CW; ++k) n2[k & 3] = fmaf(g[k], g[k], n2[k & 3]);
    }
    const float nn = group4_sum((n2[0] + n2[1]) + (n2[2] + n2[3]));
    if (norm_row) {
      const float inv = rsqrtf(nn);
#pragma unroll
      for (int k = 0; k < CW; k += 4) {
        g[k] *= inv;
        g[k + 1] *= inv;
        g[k + 2] *= inv;
        g[k + 3] *= inv;
        *reinterpret_cast<float4*>(q + p * CW + k) = make_float4(g[k], g[k + 1], g[k + 2], g[k + 3]);
      }
    }
    __syncthreads();
    const bool upd = row_ok && r > i;
    float qv[CW];
    float dp[4] = {0.f, 0.f, 0.f, 0.f};
    if (upd) {
#pragma unroll
      for (int k = 0; k < CW; k += 4) {
        const float4 v = *reinterpret_cast<const float4*>(q + p * CW + k);
        qv[k] = v.x;
        qv[k + 1] = v.y;
        qv[k + 2] = v.z;
        qv[k + 3] = v.w;
      }
#pragma unroll
      for (int k = 0; k < CW; ++k) dp[k & 3] = fmaf(qv[k], g[k], dp[k & 3]);
    }
    const float dot = group4_sum((dp[0] + dp[1]) + (dp[2] + dp[3]));
    if (upd) {
#pragma unroll
      for (int k = 0; k < CW; ++k) g[k] = fmaf(-dot, qv[k], g[k]);
    }
  }

  // ---- sweep 2: one classical re-orthogonalisation step, all rows at once
  if (row_ok) {
#pragma unroll
    for (int k = 0; k < CW; k += 4)
      *reinterpret_cast<float4*>(rows + r * RW + p * CW + k) = make_float4(g[k], g[k + 1], g[k + 2], g[k + 3]);
  }
  __syncthreads();
  const int warp_last_row = min(d, (tid / 32 + 1) * (32 / kTPR)) - 1;   // largest row of this warp
  float corr[CW];
#pragma unroll
  for (int k = 0; k < CW; ++k) corr[k] = 0.f;
  for (int s_ = 0; s_ < warp_last_row; ++s_) {
    float qv[CW];
#pragma unroll
    for (int k = 0; k < CW; k += 4) {
      const float4 v = *reinterpret_cast<const float4*>(rows + s_ * RW + p * CW + k);
      qv[k] = v.x;
      qv[k + 1] = v.y;
      qv[k + 2] = v.z;
      qv[k + 3] = v.w;
    }
    float dp[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int k = 0; k < CW; ++k) dp[k & 3] = fmaf(qv[k], g[k], dp[k & 3]);
    const float c = (row_ok && s_ < r) ? group4_sum((dp[0] + dp[1]) + (dp[2] + dp[3])) : group4_sum(0.f);
#pragma unroll
    for (int k = 0; k < CW; ++k) corr[k] = fmaf(c, qv[k], corr[k]);
  }
  float n2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int k = 0; k < CW; ++k) {
    g[k] -= corr[k];
    n2[k & 3] = fmaf(g[k], g[k], n2[k & 3]);
  }
  const float inv = rsqrtf(group4_sum((n2[0] + n2[1]) + (n2[2] + n2[3])));
  const int row = b * d + r;
  if (row_ok && row < m) {
#pragma unroll
    for (int k = 0; k < CW; ++k) {
      const int c = p * CW + k;
      if (c < d) omega[(size_t)row * d + c] = g[k] * inv * len;
    }
  }
}

// Hadamard ORF block b: sqrt(d) (H D_1)(H D_2)(H D_3), H the normalised
// Walsh-Hadamard matrix, D_p = diag(+-1) with sign i of product p from the
// top bit of SplitMix64 word (b*3 + p)*d + i ("Rethinking Attention with
// Performers" summary, §A.2 and §B.3 name Hadamard ORFs; the construction is
// the plain reading).  X starts as the identity; X <- X (H D_p) applies the
// fast Walsh-Hadamard transform to every row of X, then the column signs.
// One CTA per block, X [d][d+1] in shared memory; d a power of two.
__global__ void __launch_bounds__(256) hadamard_block_kernel(uint64_t seed, int m, int d, float* __restrict__ omega) {
  extern __shared__ float X[];
  const int b = blockIdx.x;
  const int ld = d + 1;
  for (int e = threadIdx.x; e < d * d; e += blockDim.x) {
    const int r = e / d, c = e - r * d;
    X[r * ld + c] = (r == c) ? 1.f : 0.f;
  }
  __syncthreads();
  const float inv_sqrt_d = rsqrtf(static_cast<float>(d));
  for (int p = 0; p < 3; ++p) {
    for (int h = 1; h < d; h <<= 1) {
      // d rows x d/2 butterflies (i, i + h) with (i & h) == 0
      for (int e = threadIdx.x; e < d * (d / 2); e += blockDim.x) {
        const int r = e / (d / 2), k = e - r * (d / 2);
        const int i = (k / h) * 2 * h + (k % h);
        const float a = X[r * ld + i], c = X[r * ld + i + h];
        X[r * ld + i] = a + c;
        X[r * ld + i + h] = a - c;
      }
      __syncthreads();
    }
    for (int e = threadIdx.x; e < d * d; e += blockDim.x) {
      const int r = e / d, c = e - r * d;
      const uint64_t w = splitmix_word(seed, static_cast<uint64_t>(b * 3 + p) * d + c);
      const float sgn = (w >> 63) ? -1.f : 1.f;
      X[r * ld + c] *= sgn * inv_sqrt_d;
    }
    __syncthreads();
  }
  const float sqrt_d = sqrtf(static_cast<float>(d));
  for (int e = threadIdx.x; e < d * d; e += blockDim.x) {
    const int r = e / d, c = e - r * d;
    const int row = b * d + r;
    if (row < m) omega[(size_t)row * d + c] = sqrt_d * X[r * ld + c];
  }
}

// Givens ORF block b: sqrt(d) G_K ... G_2 G_1, G_r the rotation by theta_r
// in the plane of coordinates (i_r, j_r) ("Rethinking Attention with
// Performers" summary, §A.2 and §B.3 name Givens ORFs, with O(m log d)
// numbers; the construction is the plain reading), K = 3 d ceil(log2 d).
// Rotation r reads SplitMix64 words 2c and 2c + 1, c = b K + r: i =
// floor(hi32 d / 2^32), j' = floor(lo32 (d - 1) / 2^32), j = j' + [j' >= i]
// from the first; theta = 2 pi (k + 1/2) / 2^23, k its top 23 bits, from the
// second.  The CTA first draws all K rotations in parallel into shared
// memory; G_r M then changes rows i and j of M within each column, so thread
// t carries column t of the block through the K rotations on its own (every
// thread reads the same rotation: a broadcast), with no barrier until the
// rows are written.  Shared memory: rot [K] (i, j, cos, sin), X [d][d]
// (column t touched only by thread t).
struct GivensRot {
  int i, j;
  float c, s;
};

__global__ void __launch_bounds__(128) givens_block_kernel(uint64_t seed, int m, int d, int n_rot,
                                                           float* __restrict__ omega) {
  extern __shared__ float4 givens_smem[];
  GivensRot* rot = reinterpret_cast<GivensRot*>(givens_smem);
  float* X = reinterpret_cast<float*>(givens_smem + n_rot);
  const int b = blockIdx.x, t = threadIdx.x;
  const uint64_t c0 = static_cast<uint64_t>(b) * static_cast<uint64_t>(n_rot);
  for (int r = t; r < n_rot; r += blockDim.x) {
    const uint64_t c = (c0 + static_cast<uint64_t>(r)) * 2ull;
    const uint64_t w0 = splitmix_word(seed, c);
    const uint64_t w1 = splitmix_word(seed, c + 1ull);
    const int i = static_cast<int>(((w0 >> 32) * static_cast<uint64_t>(d)) >> 32);
    const int jp = static_cast<int>(((w0 & 0xFFFFFFFFull) * static_cast<uint64_t>(d - 1)) >> 32);
    // 2 u = (k + 1/2) / 2^22, exact in fp32
    const float two_u = (static_cast<float>(static_cast<uint32_t>(w1 >> 41)) + 0.5f) * (1.0f / 4194304.0f);
    GivensRot g;
    g.i = i;
    g.j = jp + (jp >= i ? 1 : 0);
    sincospif(two_u, &g.s, &g.c);
    rot[r] = g;
  }
  if (t < d)
    for (int r = 0; r < d; ++r) X[r * d + t] = (r == t) ? 1.f : 0.f;
  __syncthreads();
  if (t < d) {
    for (int r = 0; r < n_rot; ++r) {
      const GivensRot g = rot[r];
      const float a = X[g.i * d + t], e = X[g.j * d + t];
      X[g.i * d + t] = g.c * a - g.s * e;
      X[g.j * d + t] = g.s * a + g.c * e;
    }
  }
  __syncthreads();
  const float sqrt_d = sqrtf(static_cast<float>(d));
  if (t < d)
    for (int r = 0; r < d && b * d + r < m; ++r) omega[(size_t)(b * d + r) * d + t] = sqrt_d * X[r * d + t];
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
  if (orthogonal == 3) {
    const int ceil_log2 = 32 - __builtin_clz(static_cast<unsigned>(d - 1));   // d >= 2
    const int n_rot = 3 * d * ceil_log2;
    const size_t smem = (size_t)n_rot * sizeof(float4) + (size_t)d * d * sizeof(float);   // 107 KB at d = 128
    cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(givens_block_kernel), smem);
    if (e != cudaSuccess) return e;
    const int threads = ((d + 31) / 32) * 32;
    givens_block_kernel<<<(m + d - 1) / d, threads, smem, stream>>>(seed, m, d, n_rot, omega);
    return cudaGetLastError();
  }
  if (orthogonal == 2) {
    const size_t smem = (size_t)d * (d + 1) * sizeof(float);
    cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(hadamard_block_kernel), smem);
    if (e != cudaSuccess) return e;
    hadamard_block_kernel<<<(m + d - 1) / d, 256, smem, stream>>>(seed, m, d, omega);
    return cudaGetLastError();
  }
  if (orthogonal) {
    const int nb = (m + d - 1) / d;
    const int threads = ((d * kTPR + 31) / 32) * 32;
    const int cw = (d + kTPR - 1) / kTPR;
    // shared memory: two unit rows + all d rows of kTPR * CW floats
    auto smem_for = [&](int CW) { return (size_t)(2 + d) * kTPR * CW * sizeof(float); };
    cudaError_t e = cudaSuccess;
    if (cw <= 4) {
      orf_block_kernel<4><<<nb, threads, smem_for(4), stream>>>(seed, m, d, omega);
    } else if (cw <= 8) {
      orf_block_kernel<8><<<nb, threads, smem_for(8), stream>>>(seed, m, d, omega);
    } else if (cw <= 16) {
      orf_block_kernel<16><<<nb, threads, smem_for(16), stream>>>(seed, m, d, omega);
    } else {
      e = ensure_dynamic_smem(reinterpret_cast<const void*>(orf_block_kernel<32>), smem_for(32));
      if (e != cudaSuccess) return e;
      orf_block_kernel<32><<<nb, threads, smem_for(32), stream>>>(seed, m, d, omega);
    }
  } else {
    const int n = m * d;
    iid_kernel<<<(n + 255) / 256, 256, 0, stream>>>(seed, m, d, omega);
  }
  return cudaGetLastError();
}

}  // namespace favor
