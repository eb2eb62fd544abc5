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
#include "tc_ptx.cuh"

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
constexpr int kPanel = 32 / kTPR;       // rows per warp: one panel
constexpr int kPartPad = 4;             // floats after each part of a stored row
constexpr int kOrfCluster = 8;          // CTAs drawing one block's normals

// Layout of one block's rows in shared memory.  Row r, part p (its columns
// p*CW .. p*CW+CW-1) starts at r*RW + p*PS: with PS = CW + 4 the four parts
// of a row fall in different banks, so a warp-wide 16-byte read of one row
// (four distinct addresses) meets no bank conflict; unpadded, the four parts
// share their banks and the read takes four times the passes.  With CW <= 16 the rows being
// subtracted are held in registers between their dot products and their
// updates, and a second group of warps (helpers, one thread per Gram–Schmidt
// thread) derives the lengths and takes half of the re-orthogonalisation;
// at CW = 32 (d > 64) the registers of 512 threads allow neither, and the
// rows are read twice instead.
template <int CW>
struct OrfLayout {
  static constexpr int PS = CW + kPartPad;
  static constexpr int RW = kTPR * PS;
  static constexpr bool kHeld = CW <= 16;
  static constexpr int kMaxThreads = (kHeld ? 2 : 1) * kTPR * kTPR * CW;
};

__device__ __forceinline__ float group4_sum(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 1);
  v += __shfl_xor_sync(0xffffffffu, v, 2);
  return v;
}

// Partial dot product of this thread's CW columns with the same columns of a
// row in shared memory (four accumulators).
template <int CW>
__device__ __forceinline__ float dot_part(const float* __restrict__ row, const float (&g)[CW]) {
  float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int k = 0; k < CW; k += 4) {
    const float4 v = *reinterpret_cast<const float4*>(row + k);
    a[0] = fmaf(v.x, g[k], a[0]);
    a[1] = fmaf(v.y, g[k + 1], a[1]);
    a[2] = fmaf(v.z, g[k + 2], a[2]);
    a[3] = fmaf(v.w, g[k + 3], a[3]);
  }
  return (a[0] + a[1]) + (a[2] + a[3]);
}

// acc -= c * row (this thread's CW columns of a row in shared memory)
template <int CW>
__device__ __forceinline__ void axpy_part(float c, const float* __restrict__ row, float (&acc)[CW]) {
#pragma unroll
  for (int k = 0; k < CW; k += 4) {
    const float4 v = *reinterpret_cast<const float4*>(row + k);
    acc[k] = fmaf(-c, v.x, acc[k]);
    acc[k + 1] = fmaf(-c, v.y, acc[k + 1]);
    acc[k + 2] = fmaf(-c, v.z, acc[k + 2]);
    acc[k + 3] = fmaf(-c, v.w, acc[k + 3]);
  }
}

// Barrier `id` (1..15) over n threads, whole warps: bar.sync waits for all n,
// bar.arrive counts this warp and goes on.
__device__ __forceinline__ void named_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void named_arrive(int id, int n) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory");
}

template <int CW>
__device__ __forceinline__ void load_part(const float* __restrict__ row, float (&x)[CW]) {
#pragma unroll
  for (int k = 0; k < CW; k += 4) {
    const float4 v = *reinterpret_cast<const float4*>(row + k);
    x[k] = v.x;
    x[k + 1] = v.y;
    x[k + 2] = v.z;
    x[k + 3] = v.w;
  }
}

template <int CW>
__device__ __forceinline__ void store_part(float* __restrict__ row, const float (&x)[CW]) {
#pragma unroll
  for (int k = 0; k < CW; k += 4)
    *reinterpret_cast<float4*>(row + k) = make_float4(x[k], x[k + 1], x[k + 2], x[k + 3]);
}

// acc -= sum_j c_j q_j over N unit rows q_j (stride RW) with c_j = q_j . g,
// the N coefficients taken together; with `below` only rows s0 + j < r count.
// The rows are read once and held in registers.
template <int CW, int N>
__device__ __forceinline__ void subtract_held(const float* __restrict__ q, const float (&g)[CW], float (&acc)[CW],
                                              int s0, int r, bool below) {
  constexpr int RW = OrfLayout<CW>::RW;
  float qv[N][CW];
#pragma unroll
  for (int j = 0; j < N; ++j) load_part<CW>(q + j * RW, qv[j]);
  float c[N];
#pragma unroll
  for (int j = 0; j < N; ++j) {
    float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int k = 0; k < CW; ++k) a[k & 3] = fmaf(qv[j][k], g[k], a[k & 3]);
    c[j] = group4_sum((a[0] + a[1]) + (a[2] + a[3]));
  }
#pragma unroll
  for (int j = 0; j < N; ++j) {
    const float cj = (!below || s0 + j < r) ? c[j] : 0.f;
#pragma unroll
    for (int k = 0; k < CW; ++k) acc[k] = fmaf(-cj, qv[j][k], acc[k]);
  }
}

// One CTA per d x d block.  Gram–Schmidt thread (row r = t/4, part p = t%4)
// keeps columns p*CW .. p*CW+CW-1 of row r in registers (CW = ceil(d/4)
// rounded up to a multiple of 4; columns >= d are zero), so warp w holds rows
// 8w .. 8w+7, panel w.
//
// Sweep 1 is block modified Gram–Schmidt over the panels.  Panel w is
// orthogonalised inside warp w, row by row, with no block barrier: the
// pivot u_i reaches the warp through shared memory and every later row g
// loses (u_i . g / u_i . u_i) u_i, both dots taken from the same copy, so the
// pivot's own norm is off the dependent chain.  The panel's rows are then
// normalised and published, and after one barrier every later panel loses
// its components along them (the panel's coefficients taken together).
// fp32 leaves the rows orthogonal only to about kappa * 2^-24, so sweep 2
// re-orthogonalises them: as they are orthonormal up to that small error E,
// one classical step q_r - sum_{s<r} (q_s . q_r) q_s for all rows at once
// equals a second modified sweep up to O(E^2); its dots all use the same q_r,
// so four rows s are taken at a time.  Finally row r is scaled by the length
// of its own Gaussian vector and the block leaves through shared memory in
// row order.
//
// The normals are drawn by a cluster of 8 CTAs per block: CTA rho draws rows
// [rho d / 8, (rho + 1) d / 8) of the Gaussian block and of the length
// vectors into the first CTA's shared memory, and after one cluster barrier
// the first CTA alone goes on (the draws are 2 d^2 Box–Muller normals, the
// one part of the build that parallelises).
//
// Shared memory: rows [n_rows][RW], lengths [n_rows], and draws [n_rows][RW]:
// the length vectors, later the helpers' half of the corrections.  The draws
// fill only rows and columns below d; the loads of the Gaussian rows and of
// the length vectors replace the rest by zero, and every row stored from
// then on carries those zeros.
template <int CW>
__global__ void __launch_bounds__(OrfLayout<CW>::kMaxThreads) orf_block_kernel(uint64_t seed, int m, int d,
                                                                                float* __restrict__ omega) {
  using Lay = OrfLayout<CW>;
  constexpr int PS = Lay::PS;
  constexpr int RW = Lay::RW;
  extern __shared__ __align__(16) float orf_smem[];
  const int n_panels = (d + kPanel - 1) / kPanel;
  const int n_rows = n_panels * kPanel;
  const int gs_threads = n_rows * kTPR;           // whole warps
  float* const rows = orf_smem;
  float* const lens = rows + n_rows * RW;
  float* const draws = lens + n_rows;             // 32-byte aligned: n_rows is a multiple of 8
  float* const hcorr = draws;
  const int b = blockIdx.x / kOrfCluster;

  // ---- the normals: Gaussian entry (r, c) of block b from word 2 e, its
  // length-vector entry from word 2 e + 1, e = (b d + r) d + c
  {
    const int rank = static_cast<int>(tc::cluster_ctarank());
    const int r0 = rank * d / kOrfCluster, r1 = (rank + 1) * d / kOrfCluster;
    const uint32_t rows0 = tc::map_to_rank(tc::smem_addr(rows), 0);
    const uint32_t draws0 = tc::map_to_rank(tc::smem_addr(draws), 0);
    const int n_e = (r1 - r0) * d;
    for (int e = threadIdx.x; e < n_e; e += blockDim.x) {
      const int rr = r0 + e / d, c = e - (e / d) * d;
      const uint64_t idx = (((uint64_t)b * d + rr) * d + c) * 2ull;
      const uint32_t off = 4u * static_cast<uint32_t>(rr * RW + (c / CW) * PS + c % CW);
      tc::st_cluster_f32(rows0 + off, normal_from_word(splitmix_word(seed, idx)));
      tc::st_cluster_f32(draws0 + off, normal_from_word(splitmix_word(seed, idx + 1ull)));
    }
  }
  tc::cluster_sync();                             // the draws are in the first CTA
  if (tc::cluster_ctarank() != 0) return;            // nothing reads the other CTAs' memory

  // helper warp j serves Gram–Schmidt warp n_panels - 1 - j: the warps with
  // the most re-orthogonalisation work pair with the least loaded
  // sub-partitions (warp w runs on sub-partition w mod 4)
  const bool helper = Lay::kHeld && threadIdx.x >= gs_threads;   // warp-uniform
  const int t = helper ? (((n_panels - 1 - ((threadIdx.x - gs_threads) >> 5)) << 5) | (threadIdx.x & 31))
                       : threadIdx.x;
  const int warp = t >> 5;                        // panel of row r
  const int li = (t & 31) / kTPR;                 // row within the panel
  const int r = t / kTPR;
  const int p = t % kTPR;
  const bool row_ok = r < d;
  float* const my_part = rows + r * RW + p * PS;

  // Gaussian row r (Gram–Schmidt threads) and the length of row r's own
  // Gaussian vector (helpers, else the same threads); columns past d are zero
  float g[CW];
  float len = 0.f;
  load_part<CW>(my_part, g);
#pragma unroll
  for (int k = 0; k < CW; ++k)
    if (helper || !row_ok || p * CW + k >= d) g[k] = 0.f;
  if (!Lay::kHeld || helper) {
    float x[CW];
    load_part<CW>(draws + r * RW + p * PS, x);
    float len2 = 0.f;
#pragma unroll
    for (int k = 0; k < CW; ++k) len2 = fmaf(row_ok && p * CW + k < d ? x[k] : 0.f, x[k], len2);
    len = sqrtf(group4_sum(len2));
    if (Lay::kHeld && p == 0) lens[r] = len;
  }

  // ---- sweep 1: block modified Gram–Schmidt.  Branches on `helper`, `warp`
  // and the panel's row count are warp-uniform, so every shuffle has the
  // full warp.
  for (int k = 0; k < n_panels; ++k) {
    if (!helper && warp == k) {
      const int rows_k = min(kPanel, d - k * kPanel);
      float n2_own = 1.f;
      for (int i = 0; i < rows_k; ++i) {
        if (li == i) store_part<CW>(my_part, g);
        __syncwarp();
        const float* u = rows + (k * kPanel + i) * RW + p * PS;
        float dp[4] = {0.f, 0.f, 0.f, 0.f};
        float nn[4] = {0.f, 0.f, 0.f, 0.f};
        float uv[Lay::kHeld ? CW : 1];
#pragma unroll
        for (int kk = 0; kk < CW; kk += 4) {
          const float4 v = *reinterpret_cast<const float4*>(u + kk);
          if constexpr (Lay::kHeld) {
            uv[kk] = v.x;
            uv[kk + 1] = v.y;
            uv[kk + 2] = v.z;
            uv[kk + 3] = v.w;
          }
          dp[0] = fmaf(v.x, g[kk], dp[0]);
          dp[1] = fmaf(v.y, g[kk + 1], dp[1]);
          dp[2] = fmaf(v.z, g[kk + 2], dp[2]);
          dp[3] = fmaf(v.w, g[kk + 3], dp[3]);
          nn[0] = fmaf(v.x, v.x, nn[0]);
          nn[1] = fmaf(v.y, v.y, nn[1]);
          nn[2] = fmaf(v.z, v.z, nn[2]);
          nn[3] = fmaf(v.w, v.w, nn[3]);
        }
        float dot = (dp[0] + dp[1]) + (dp[2] + dp[3]);
        float n2 = (nn[0] + nn[1]) + (nn[2] + nn[3]);
        dot += __shfl_xor_sync(0xffffffffu, dot, 1);
        n2 += __shfl_xor_sync(0xffffffffu, n2, 1);
        dot += __shfl_xor_sync(0xffffffffu, dot, 2);
        n2 += __shfl_xor_sync(0xffffffffu, n2, 2);
        if (li == i) n2_own = n2;
        if (li > i) {
          const float cf = __fdividef(dot, n2);
          if constexpr (Lay::kHeld) {
#pragma unroll
            for (int kk = 0; kk < CW; ++kk) g[kk] = fmaf(-cf, uv[kk], g[kk]);
          } else {
            axpy_part<CW>(cf, u, g);
          }
        }
      }
      __syncwarp();                               // the last pivot is read before it is overwritten
      // rows >= d (only in the last panel) are zero and stay zero
      const float inv = row_ok ? rsqrtf(n2_own) : 0.f;
#pragma unroll
      for (int kk = 0; kk < CW; ++kk) g[kk] *= inv;
      store_part<CW>(my_part, g);
    }
    __syncthreads();
    if (!helper && warp > k) {
      // panel k is full here (only the last panel can be short).  Warp k + 1
      // pivots next, so the later warps leave it the shared-memory pipe: they
      // start once it has subtracted the panel (barrier 1).
      const int n_wait = 32 * (n_panels - k - 1);  // warps k + 1 .. n_panels - 1
      if (warp > k + 1) named_sync(1, n_wait);
      const float* q = rows + k * kPanel * RW + p * PS;
      if constexpr (Lay::kHeld) {
        subtract_held<CW, 4>(q, g, g, 0, 0, false);
        subtract_held<CW, 4>(q + 4 * RW, g, g, 0, 0, false);
      } else {
        // the rows are read again for the updates rather than held
        float c[kPanel];
#pragma unroll
        for (int j = 0; j < kPanel; ++j) c[j] = dot_part<CW>(q + j * RW, g);
#pragma unroll
        for (int j = 0; j < kPanel; ++j) c[j] = group4_sum(c[j]);
        __syncwarp();     // keeps the compiler from holding the rows in registers
#pragma unroll
        for (int j = 0; j < kPanel; ++j) axpy_part<CW>(c[j], q + j * RW, g);
      }
      if (warp == k + 1 && k + 2 < n_panels) named_arrive(1, n_wait);
    }
  }

  // ---- sweep 2: one classical re-orthogonalisation step, all rows at once
  // (the last barrier of sweep 1 published every row).  Rows s < r of this
  // warp lie below 8 (warp + 1): 2 (warp + 1) groups of four.
  float corr[CW];
#pragma unroll
  for (int k = 0; k < CW; ++k) corr[k] = 0.f;
  const int n_groups = 2 * (warp + 1);
  if constexpr (Lay::kHeld) {
    const int split = (n_groups + 1) / 2;         // the helper takes the upper groups
    if (helper) load_part<CW>(my_part, g);
    for (int j = helper ? split : 0; j < (helper ? n_groups : split); ++j)
      subtract_held<CW, 4>(rows + 4 * j * RW + p * PS, g, corr, 4 * j, r, true);
    if (helper) store_part<CW>(hcorr + r * RW + p * PS, corr);
    __syncthreads();
    if (!helper) {
      float h[CW];
      load_part<CW>(hcorr + r * RW + p * PS, h);
#pragma unroll
      for (int k = 0; k < CW; ++k) corr[k] += h[k];
      len = lens[r];
    }
  } else {
    for (int s0 = 0; s0 < 4 * n_groups; s0 += 4) {
      const float* q = rows + s0 * RW + p * PS;
      float c[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) c[j] = dot_part<CW>(q + j * RW, g);
#pragma unroll
      for (int j = 0; j < 4; ++j) c[j] = group4_sum(c[j]);
      __syncwarp();
#pragma unroll
      for (int j = 0; j < 4; ++j) axpy_part<CW>(s0 + j < r ? c[j] : 0.f, q + j * RW, corr);
    }
  }
  float sc = 0.f;
  if (!helper) {
    float n2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int k = 0; k < CW; ++k) {
      g[k] += corr[k];
      n2[k & 3] = fmaf(g[k], g[k], n2[k & 3]);
    }
    const float nrm2 = group4_sum((n2[0] + n2[1]) + (n2[2] + n2[3]));
    sc = row_ok ? rsqrtf(nrm2) * len : 0.f;
  }
  __syncthreads();                                // every row has been read
  if (!helper) {
#pragma unroll
    for (int k = 0; k < CW; ++k) g[k] *= sc;
    store_part<CW>(my_part, g);
  }
  __syncthreads();
  const int n_out = min(d, m - b * d);
  float* const dst = omega + (size_t)b * d * d;
  if ((d & 3) == 0 && (reinterpret_cast<uintptr_t>(omega) & 15) == 0) {
    // four columns at a time (CW is a multiple of 4, so they share a part)
    const int dq = d >> 2;
    for (int e = threadIdx.x; e < n_out * dq; e += blockDim.x) {
      const int row = e / dq, c = (e - row * dq) << 2;
      reinterpret_cast<float4*>(dst)[e] =
          *reinterpret_cast<const float4*>(rows + row * RW + (c / CW) * PS + (c % CW));
    }
  } else {
    for (int e = threadIdx.x; e < n_out * d; e += blockDim.x) {
      const int row = e / d, c = e - row * d;
      dst[e] = rows[row * RW + (c / CW) * PS + (c % CW)];
    }
  }
}

// Hadamard ORF block b: sqrt(d) (H D_1)(H D_2)(H D_3), H the normalised
// Walsh-Hadamard matrix, D_p = diag(+-1) with sign i of product p from the
// top bit of SplitMix64 word (b*3 + p)*d + i ("Rethinking Attention with
// Performers" summary, §A.2 and §B.3 name Hadamard ORFs; the construction is
// the plain reading).  Row r starts as e_r; X <- X (H D_p) applies the fast
// Walsh-Hadamard transform to the row (strides 1, 2, 4, ..: a + c, a - c),
// then the column signs and 1/sqrt(d).  Rows are independent, so one warp
// carries one row: element i in lane i % 32, slot i / 32 (E = max(1, d/32)
// slots); strides below 32 pair lanes by shuffles, larger strides pair slots
// of the same lane.  d is a power of two; for d < 32 lanes >= d idle.
template <int E>
__global__ void __launch_bounds__(256) hadamard_rows_kernel(uint64_t seed, int m, int d, float* __restrict__ omega) {
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);     // global row of Omega, warp-uniform
  if (row >= m) return;
  const int b = row / d, r = row - b * d;
  float x[E];
#pragma unroll
  for (int s = 0; s < E; ++s) x[s] = (s * 32 + lane == r) ? 1.f : 0.f;
  const float inv_sqrt_d = rsqrtf(static_cast<float>(d));
  for (int p = 0; p < 3; ++p) {
    for (int h = 1; h < d; h <<= 1) {
      if (h < 32) {
        const bool upper = (lane & h) != 0;
#pragma unroll
        for (int s = 0; s < E; ++s) {
          const float o = __shfl_xor_sync(0xffffffffu, x[s], h);
          x[s] = upper ? o - x[s] : x[s] + o;
        }
      } else {
        const int k = h >> 5;                                // slot stride
#pragma unroll
        for (int s = 0; s < E; ++s) {
          if ((s & k) == 0) {
            const float a = x[s], c = x[s + k];
            x[s] = a + c;
            x[s + k] = a - c;
          }
        }
      }
    }
#pragma unroll
    for (int s = 0; s < E; ++s) {
      const int c = s * 32 + lane;
      const uint64_t w = splitmix_word(seed, static_cast<uint64_t>(b * 3 + p) * d + c);
      const float sgn = (w >> 63) ? -1.f : 1.f;
      x[s] *= sgn * inv_sqrt_d;
    }
  }
  const float sqrt_d = sqrtf(static_cast<float>(d));
#pragma unroll
  for (int s = 0; s < E; ++s) {
    const int c = s * 32 + lane;
    if (c < d) omega[(size_t)row * d + c] = sqrt_d * x[s];
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
    const int grid = (m + 7) / 8;                            // one warp per row
    if (d <= 32) hadamard_rows_kernel<1><<<grid, 256, 0, stream>>>(seed, m, d, omega);
    else if (d <= 64) hadamard_rows_kernel<2><<<grid, 256, 0, stream>>>(seed, m, d, omega);
    else hadamard_rows_kernel<4><<<grid, 256, 0, stream>>>(seed, m, d, omega);
    return cudaGetLastError();
  }
  if (orthogonal) {
    const int nb = (m + d - 1) / d;
    const int n_rows = ((d + kPanel - 1) / kPanel) * kPanel;
    const int gs_threads = n_rows * kTPR;
    const int cw = (d + kTPR - 1) / kTPR;
    cudaError_t e = cudaSuccess;
    auto launch = [&](auto kernel, int CW, bool held) {
      const int RW = kTPR * (CW + kPartPad);
      const size_t smem = ((size_t)2 * n_rows * RW + n_rows) * sizeof(float);
      e = ensure_dynamic_smem(reinterpret_cast<const void*>(kernel), smem);
      if (e != cudaSuccess) return;
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(nb * kOrfCluster);
      cfg.blockDim = dim3(gs_threads * (held ? 2 : 1));
      cfg.dynamicSmemBytes = smem;
      cfg.stream = stream;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = kOrfCluster;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      e = cudaLaunchKernelEx(&cfg, kernel, seed, m, d, omega);
    };
    if (cw <= 4) {
      launch(orf_block_kernel<4>, 4, OrfLayout<4>::kHeld);
    } else if (cw <= 8) {
      launch(orf_block_kernel<8>, 8, OrfLayout<8>::kHeld);
    } else if (cw <= 16) {
      launch(orf_block_kernel<16>, 16, OrfLayout<16>::kHeld);
    } else {
      launch(orf_block_kernel<32>, 32, OrfLayout<32>::kHeld);
    }
    if (e != cudaSuccess) return e;
  } else {
    const int n = m * d;
    iid_kernel<<<(n + 255) / 256, 256, 0, stream>>>(seed, m, d, omega);
  }
  return cudaGetLastError();
}

}  // namespace favor
