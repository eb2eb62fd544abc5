// CUDA-core FAVOR+ kernels (fp32 arithmetic): the path for fp32 storage, for
// shapes the tensor-core kernels do not cover, for the 1 + elu feature map
// and for the backward of both passes.  Every product runs on per-thread
// register tiles (RegTile, rowdot_block, outer_acc, gram_acc below).
//
// Formulas: "Performer — Rethinking Attention with Performers" (digest),
// §Key equations: phi(x) = m^-1/2 exp(Omega x - |x|^2/2) and
// Attn^ = D^-1 phi(Q)(phi(K)^T V), D = diag(phi(Q) phi(K)^T 1); §Methods:
// causal prefix sum G_t = sum_{s<=t} phi(k_s) v_s^T.
//
// Stabilisers (exact rewrites, not approximations):
//  * key side: phi(k) is evaluated as exp(l - R) with one constant R for the
//    whole call, R = max_i |w_i|^2 / 2 - 40 (see prep.cu and key_reference);
//    since l = |w|^2/2 - |s k - w|^2/2 <= max_i |w_i|^2/2, every key feature
//    is <= e^40 and the shared factor exp(-R) cancels between numerator and
//    normaliser;
//  * query side: the per-row constant max_i(s w_i.q) is subtracted, and
//    |q|^2/2 and m^-1/2 are dropped -- per-query constants cancel ("From
//    Performer to Linear Attention", §Simple Derivation).
#include <type_traits>

#include "backward.cuh"
#include "common.cuh"

namespace favor {
namespace {

constexpr int kFB = 64;        // features per CTA (state kernel) / per block of Omega
constexpr int kTT = 32;        // tokens per tile
constexpr int kThreads = 256;

template <typename T>
__device__ __forceinline__ void load_rows(const T* __restrict__ src, int nt, int d, float* dst, int ld) {
  for (int e = threadIdx.x; e < kTT * d; e += kThreads) {
    const int t = e / d, c = e - t * d;
    dst[t * ld + c] = (t < nt) ? to_f32(src[(size_t)t * d + c]) : 0.f;
  }
}

__device__ __forceinline__ void load_omega_block(const float* __restrict__ omega, int f0, int nf, int d,
                                                 float* om) {
  const int ld = d + 1;
  for (int e = threadIdx.x; e < kFB * d; e += kThreads) {
    const int f = e / d, c = e - f * d;
    om[f * ld + c] = (f < nf) ? omega[(size_t)(f0 + f) * d + c] : 0.f;
  }
}

// rows [f0, f0 + nf) of a per-head [m][d+1] fp32 matrix into blk [kFB][d+1]
__device__ __forceinline__ void load_state_block(const float* __restrict__ src, int f0, int nf, int d, float* blk) {
  const int ld = d + 1;
  for (int e = threadIdx.x; e < nf * ld; e += kThreads) blk[e] = src[(size_t)f0 * ld + e];
}

__device__ __forceinline__ void row_norms(const float* xs, int d, float* kn) {
  if (threadIdx.x < kTT) {
    const float* row = xs + threadIdx.x * (d + 1);
    float acc = 0.f;
    for (int c = 0; c < d; ++c) acc = fmaf(row[c], row[c], acc);
    kn[threadIdx.x] = acc;
  }
}

// Register tiles of a TT x 64 block (TT = 32 or 16 rows; 64 = kFB columns)
// over 256 threads: thread (tg, fl) owns rows tg and tg + TT/2 and columns
// fl + k kLanes, kLanes = 16 (TT = 32) or 32 (TT = 16).  Per step of a
// reduction a warp reads two row values (broadcasts) and 64 / kLanes column
// values (kLanes distinct rows or columns, conflict-free for odd strides) for
// 2 x 64 / kLanes multiply-adds per thread, instead of two shared-memory
// loads per multiply-add.  Every output is still one sequential fmaf chain
// in the reduction order of the plain loop.
template <int TT>
struct RegTile {
  static_assert(TT == 32 || TT == 16, "tile rows");
  static constexpr int kLanes = TT == 32 ? 16 : 32;
  static constexpr int kCols = kFB / kLanes;
  static constexpr int kHalf = TT / 2;
  // column groups covering n <= kMaxD + 1 columns (outer products)
  static constexpr int kWide = (kMaxD + 1 + kLanes - 1) / kLanes;
  __device__ static int tg() { return threadIdx.x / kLanes; }
  __device__ static int fl() { return threadIdx.x % kLanes; }
  __device__ static int row(int i) { return tg() + i * kHalf; }
  __device__ static int col(int k) { return fl() + k * kLanes; }
};

// acc[i][k] = sum_{c < n} A[row_i][c] B[col_k][c] (rows of A and B length n,
// strides lda, ldb); B has kFB rows.
template <int TT>
__device__ __forceinline__ void rowdot_block(const float* A, int lda, const float* B, int ldb, int n,
                                             float (&acc)[2][RegTile<TT>::kCols]) {
  using RT = RegTile<TT>;
  const float* a0 = A + RT::tg() * lda;
  const float* a1 = a0 + RT::kHalf * lda;
  const float* b = B + RT::fl() * ldb;
#pragma unroll
  for (int k = 0; k < RT::kCols; ++k) acc[0][k] = acc[1][k] = 0.f;
#pragma unroll 4
  for (int c = 0; c < n; ++c) {
    const float x0 = a0[c], x1 = a1[c];
#pragma unroll
    for (int k = 0; k < RT::kCols; ++k) {
      const float w = b[k * RT::kLanes * ldb + c];
      acc[0][k] = fmaf(x0, w, acc[0][k]);
      acc[1][k] = fmaf(x1, w, acc[1][k]);
    }
  }
}

// acc[i][k] += sum_{f < nf} P[row_i][f] S[f][col_k] for columns col_k < J
// (P row stride ldp, S row stride lds); KC column groups cover J.
template <int TT, int KC>
__device__ __forceinline__ void outer_acc(const float* P, int ldp, const float* S, int lds, int nf, int J,
                                          float (&acc)[2][KC]) {
  using RT = RegTile<TT>;
  const float* p0 = P + RT::tg() * ldp;
  const float* p1 = p0 + RT::kHalf * ldp;
  const float* sc = S + RT::fl();
  const int kn = (J - RT::fl() + RT::kLanes - 1) / RT::kLanes;   // this thread's columns below J
  for (int f = 0; f < nf; ++f) {
    const float x0 = p0[f], x1 = p1[f];
    const float* sr = sc + f * lds;
#pragma unroll
    for (int k = 0; k < KC; ++k) {
      if (k < kn) {
        const float w = sr[k * RT::kLanes];
        acc[0][k] = fmaf(x0, w, acc[0][k]);
        acc[1][k] = fmaf(x1, w, acc[1][k]);
      }
    }
  }
}

// Sums over the tokens of a tile for a block of 64 features: acc[i][k] +=
// sum_{t < nt} X[t][fg + 16 i] Y[t][jl + 16 k] for columns jl + 16 k < J,
// thread (fg, jl) = (tid / 16, tid % 16).  Per token a warp reads 4 feature
// values (two addresses each) and KC column values (16 consecutive) for
// 4 KC multiply-adds per thread; each output is one fmaf chain in token order.
constexpr int kGramWide = (kMaxD + 1 + 15) / 16;
template <int KC>
__device__ __forceinline__ void gram_acc(const float* X, int ldx, const float* Y, int ldy, int nt, int J,
                                         float (&acc)[4][KC]) {
  const int fg = threadIdx.x / 16, jl = threadIdx.x % 16;
  const int kn = (J - jl + 15) / 16;   // this thread's columns below J
  for (int t = 0; t < nt; ++t) {
    const float* xr = X + t * ldx + fg;
    const float* yr = Y + t * ldy + jl;
    float x[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) x[i] = xr[16 * i];
#pragma unroll
    for (int k = 0; k < KC; ++k) {
      if (k < kn) {
        const float y = yr[16 * k];
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[i][k] = fmaf(x[i], y, acc[i][k]);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// State partials: for (split, feature block, head) the CTA sums
//   S_p[f, :] = sum_t exp(l_tf - R) [v_t ; 1],  l_tf = s w_f.k_t - s^2 |k_t|^2 / 2
// over its token range.
// ---------------------------------------------------------------------------
// 1 + elu(a): 1 + a for a >= 0, exp(a) below (a NaN stays a NaN)
__device__ __forceinline__ float elu1(float a) { return a < 0.f ? expf(a) : 1.f + a; }

// Key feature from its scaled projection a = s w.k: exp(a - s^2 |k|^2 / 2 - R)
// for the positive random features, relu(a) for Performer-ReLU ("y < 0 ? 0
// : y" keeps a NaN a NaN), 1 + elu(a) for the linear-attention map.
template <int FM>
__device__ __forceinline__ float key_feature(float a, float half_sq, float R) {
  if constexpr (FM == FAVOR_FM_PRF) return expf(a - half_sq - R);
  else if constexpr (FM == FAVOR_FM_ELU1) return elu1(a);
  else return a < 0.f ? 0.f : a;
}

template <typename T, int FM>
__global__ void __launch_bounds__(kThreads, 3) state_partial_kernel(
    const T* __restrict__ K, const T* __restrict__ V, const float* __restrict__ omega,
    const float* __restrict__ key_ref, int L, int d, int m, float scale, int chunk, int n_split,
    float* __restrict__ partS) {
  extern __shared__ float smem[];
  const int split = blockIdx.x, fb = blockIdx.y, bh = blockIdx.z;
  const int ld = d + 1;
  float* om = smem;                       // [kFB][ld]
  float* ks = om + kFB * ld;              // [kTT][ld]
  float* vs = ks + kTT * ld;              // [kTT][ld]
  float* ph = vs + kTT * ld;              // [kTT][kFB + 1]
  float* kn = ph + kTT * (kFB + 1);       // [kTT]

  const int f0 = fb * kFB, nf = min(kFB, m - f0);
  const int l0 = split * chunk, l1 = min(L, l0 + chunk);
  const T* Kh = K + (size_t)bh * L * d;
  const T* Vh = V + (size_t)bh * L * d;
  const float hs2 = 0.5f * scale * scale;
  float R, W_unused;
  key_reference(key_ref, m, &R, &W_unused);
  load_omega_block(omega, f0, nf, d, om);
  // the normaliser column: [v ; 1] (load_rows fills columns < d only)
  if (threadIdx.x < kTT) vs[threadIdx.x * ld + d] = 1.f;

  // thread owns features fg + 16 i (i < 4) and columns jl + 16 k
  using RT = RegTile<kTT>;
  float acc[4][kGramWide];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int k = 0; k < kGramWide; ++k) acc[i][k] = 0.f;
  for (int t0 = l0; t0 < l1; t0 += kTT) {
    const int nt = min(kTT, l1 - t0);
    __syncthreads();
    load_rows(Kh + (size_t)t0 * d, nt, d, ks, ld);
    load_rows(Vh + (size_t)t0 * d, nt, d, vs, ld);
    __syncthreads();
    row_norms(ks, d, kn);
    __syncthreads();
    {
      float a[2][RT::kCols];
      rowdot_block<kTT>(ks, ld, om, ld, d, a);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int t = RT::row(i);
#pragma unroll
        for (int k = 0; k < RT::kCols; ++k) {
          const int f = RT::col(k);
          ph[t * (kFB + 1) + f] = (t < nt && f < nf) ? key_feature<FM>(scale * a[i][k], hs2 * kn[t], R) : 0.f;
        }
      }
    }
    __syncthreads();
    gram_acc<kGramWide>(ph, kFB + 1, vs, ld, nt, ld, acc);
  }
  const int fg = threadIdx.x / 16, jl = threadIdx.x % 16;
  float* dst = partS + (((size_t)bh * n_split + split) * m + f0) * ld;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int f = fg + 16 * i;
    if (f < nf)
#pragma unroll
      for (int k = 0; k < kGramWide; ++k) {
        const int j = jl + 16 * k;
        if (j < ld) dst[(size_t)f * ld + j] = acc[i][k];
      }
  }
}

// Bidirectional: state[h] = sum over splits of S_p, in split order.  One
// thread per state element (grid: element blocks x heads), eight partials'
// loads in flight at a time.
__global__ void __launch_bounds__(kThreads) merge_kernel(const float* __restrict__ partS, int d, int m, int n_split,
                                                         float* __restrict__ state) {
  const int bh = blockIdx.y;
  const size_t per = (size_t)m * (d + 1);
  const size_t e = (size_t)blockIdx.x * kThreads + threadIdx.x;
  if (e >= per) return;
  const float* src = partS + (size_t)bh * n_split * per + e;
  float acc = 0.f;
  for (int p0 = 0; p0 < n_split; p0 += 8) {
    float v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = p0 + u < n_split ? src[(size_t)(p0 + u) * per] : 0.f;
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (p0 + u < n_split) acc += v[u];
  }
  state[(size_t)bh * per + e] = acc;
}

dim3 merge_grid(const Shape& s) {
  const size_t per = (size_t)s.m * (s.d + 1);
  return dim3(static_cast<unsigned>((per + kThreads - 1) / kThreads), static_cast<unsigned>(s.BH()));
}

// Query-side features of one tile: pq[t][i] = exp(s w_i.q_t - max_i s w_i.q_t)
// (all m features, exact row maximum), rows t >= nt set to 0.
template <int FM>
__device__ void query_features(const float* qs, int nt, int d, int m, float scale,
                               const float* __restrict__ omega, float* om, float* pq, float* rowmax) {
  using RT = RegTile<kTT>;
  const int ld = d + 1, ldq = m + 1;
  const int n_fb = (m + kFB - 1) / kFB;
  for (int fb = 0; fb < n_fb; ++fb) {
    const int f0 = fb * kFB, nf = min(kFB, m - f0);
    __syncthreads();
    load_omega_block(omega, f0, nf, d, om);
    __syncthreads();
    float a[2][RT::kCols];
    rowdot_block<kTT>(qs, ld, om, ld, d, a);
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int k = 0; k < RT::kCols; ++k)
        if (RT::col(k) < nf) pq[RT::row(i) * ldq + f0 + RT::col(k)] = scale * a[i][k];
  }
  __syncthreads();
  if constexpr (FM != FAVOR_FM_PRF) {
    // Performer-ReLU or 1 + elu of the scaled projection, no row constant
    for (int e = threadIdx.x; e < kTT * m; e += kThreads) {
      const int t = e / m, f = e - t * m;
      const float a = pq[t * ldq + f];
      pq[t * ldq + f] = (t < nt) ? key_feature<FM>(a, 0.f, 0.f) : 0.f;
    }
    __syncthreads();
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int t = warp; t < kTT; t += kThreads / 32) {
    float mx = -INFINITY;
    for (int f = lane; f < m; f += 32) mx = fmaxf(mx, pq[t * ldq + f]);
    mx = warp_max(mx);
    if (lane == 0) rowmax[t] = mx;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < kTT * m; e += kThreads) {
    const int t = e / m, f = e - t * m;
    pq[t * ldq + f] = (t < nt) ? expf(pq[t * ldq + f] - rowmax[t]) : 0.f;
  }
  __syncthreads();
}

// num[t][j] (j <= d) in smem -> O = num[:, :d] / num[:, d]; flags bad normalisers.
template <typename T>
__device__ __forceinline__ void store_output(const float* num, int nt, int d, T* __restrict__ Oh,
                                             int32_t* status) {
  const int ld = d + 1;
  for (int e = threadIdx.x; e < nt * d; e += kThreads) {
    const int t = e / d, j = e - t * d;
    const float den = num[t * ld + d];
    if (!(den > 0.f) || !isfinite(den)) report_status(status, FAVOR_ERR_NONFINITE);
    Oh[(size_t)t * d + j] = from_f32<T>(num[t * ld + j] / den);
  }
}

template <typename T, int FM>
__global__ void __launch_bounds__(kThreads) bidir_output_kernel(
    const T* __restrict__ Q, T* __restrict__ O, const float* __restrict__ omega,
    const float* __restrict__ state, int L, int d, int m, float scale, int32_t* status) {
  extern __shared__ float smem[];
  const int ld = d + 1, ldq = m + 1;
  const int bh = blockIdx.y;
  const int t0 = blockIdx.x * kTT;
  const int nt = min(kTT, L - t0);
  float* qs = smem;                   // [kTT][ld]
  float* om = qs + kTT * ld;          // [kFB][ld]
  float* st = om + kFB * ld;          // [kFB][ld]
  float* pq = st + kFB * ld;          // [kTT][ldq]
  float* rowmax = pq + kTT * ldq;     // [kTT]

  load_rows(Q + ((size_t)bh * L + t0) * d, nt, d, qs, ld);
  query_features<FM>(qs, nt, d, m, scale, omega, om, pq, rowmax);

  using RT = RegTile<kTT>;
  float acc[2][RT::kWide];
#pragma unroll
  for (int k = 0; k < RT::kWide; ++k) acc[0][k] = acc[1][k] = 0.f;
  const float* sh = state + (size_t)bh * m * ld;
  const int n_fb = (m + kFB - 1) / kFB;
  for (int fb = 0; fb < n_fb; ++fb) {
    const int f0 = fb * kFB, nf = min(kFB, m - f0);
    __syncthreads();
    for (int e = threadIdx.x; e < nf * ld; e += kThreads) st[e] = sh[(size_t)f0 * ld + e];
    __syncthreads();
    outer_acc<kTT, RT::kWide>(pq + f0, ldq, st, ld, nf, ld, acc);
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int k = 0; k < RT::kWide; ++k)
      if (RT::col(k) < ld) qs[RT::row(i) * ld + RT::col(k)] = acc[i][k];
  __syncthreads();
  store_output(qs, nt, d, O + ((size_t)bh * L + t0) * d, status);
}

// ---------------------------------------------------------------------------
// Causal output: CTA = one superchunk of one head.  G starts as the exclusive
// prefix of earlier superchunk states (sum in superchunk order);
// each tile adds the masked intra-tile term, the inter term phi(Q) G and then
// G += phi(K)^T [V | 1].  G lives in the workspace (fp32).
// ---------------------------------------------------------------------------
template <typename T, int FM>
__global__ void __launch_bounds__(kThreads) causal_output_kernel(
    const T* __restrict__ Q, const T* __restrict__ K, const T* __restrict__ V, T* __restrict__ O,
    const float* __restrict__ omega, const float* __restrict__ key_ref, const float* __restrict__ partS,
    float* __restrict__ Gws, int L, int d, int m, float scale, int chunk, int n_sc, int32_t* status) {
  extern __shared__ float smem[];
  const int ld = d + 1, ldq = m + 1;
  const int sc = blockIdx.x, bh = blockIdx.y;
  const int n_fb = (m + kFB - 1) / kFB;
  float* qs = smem;                   // [kTT][ld]
  float* ks = qs + kTT * ld;          // [kTT][ld]
  float* vs = ks + kTT * ld;          // [kTT][ld]
  float* om = vs + kTT * ld;          // [kFB][ld]
  float* pq = om + kFB * ld;          // [kTT][ldq]
  float* pk = pq + kTT * ldq;         // [kTT][ldq]
  float* A = pk + kTT * ldq;          // [kTT][kTT + 1]
  float* kn = A + kTT * (kTT + 1);    // [kTT]
  float* rowmax = kn + kTT;           // [kTT]

  float Rk, W_unused;
  key_reference(key_ref, m, &Rk, &W_unused);
  const size_t per = (size_t)m * ld;
  float* G = Gws + ((size_t)bh * n_sc + sc) * per;
  for (int e = threadIdx.x; e < m * ld; e += kThreads) {
    float acc = 0.f;
    for (int p = 0; p < sc; ++p) acc += partS[((size_t)bh * n_sc + p) * per + e];
    G[e] = acc;
  }

  const float hs2 = 0.5f * scale * scale;
  const int l0 = sc * chunk, l1 = min(L, l0 + chunk);
  const size_t hoff = (size_t)bh * L * d;
  using RT = RegTile<kTT>;
  // the normaliser column: [v ; 1] (load_rows fills columns < d only)
  if (threadIdx.x < kTT) vs[threadIdx.x * ld + d] = 1.f;

  for (int t0 = l0; t0 < l1; t0 += kTT) {
    const int nt = min(kTT, l1 - t0);
    __syncthreads();
    load_rows(Q + hoff + (size_t)t0 * d, nt, d, qs, ld);
    load_rows(K + hoff + (size_t)t0 * d, nt, d, ks, ld);
    load_rows(V + hoff + (size_t)t0 * d, nt, d, vs, ld);
    __syncthreads();
    row_norms(ks, d, kn);
    // key features with the common scale M_w
    for (int fb = 0; fb < n_fb; ++fb) {
      const int f0 = fb * kFB, nf = min(kFB, m - f0);
      __syncthreads();
      load_omega_block(omega, f0, nf, d, om);
      __syncthreads();
      float a[2][RT::kCols];
      rowdot_block<kTT>(ks, ld, om, ld, d, a);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int t = RT::row(i);
#pragma unroll
        for (int k = 0; k < RT::kCols; ++k) {
          const int f = RT::col(k);
          if (f < nf) pk[t * ldq + f0 + f] = (t < nt) ? key_feature<FM>(scale * a[i][k], hs2 * kn[t], Rk) : 0.f;
        }
      }
    }
    query_features<FM>(qs, nt, d, m, scale, omega, om, pq, rowmax);
    // intra-tile scores, lower triangle with the diagonal: thread (tg, sl)
    // owns rows tg, tg + 16 and columns sl, sl + 16 (2 x 2 per thread)
    {
      const int tg = threadIdx.x / 16, sl = threadIdx.x % 16;
      const float* q0 = pq + tg * ldq;
      const float* q1 = q0 + 16 * ldq;
      const float* k0 = pk + sl * ldq;
      const float* k1 = k0 + 16 * ldq;
      float a00 = 0.f, a01 = 0.f, a10 = 0.f, a11 = 0.f;
#pragma unroll 4
      for (int i = 0; i < m; ++i) {
        const float x0 = q0[i], x1 = q1[i], y0 = k0[i], y1 = k1[i];
        a00 = fmaf(x0, y0, a00);
        a01 = fmaf(x0, y1, a01);
        a10 = fmaf(x1, y0, a10);
        a11 = fmaf(x1, y1, a11);
      }
      const float av[2][2] = {{a00, a01}, {a10, a11}};
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int t = tg + 16 * i, s_ = sl + 16 * j;
          A[t * (kTT + 1) + s_] = (s_ <= t && t < nt) ? av[i][j] : 0.f;
        }
    }
    // inter (phi(Q) G, G staged block by block from the workspace) then intra
    // (masked A [V | 1])
    float acc[2][RT::kWide];
#pragma unroll
    for (int k = 0; k < RT::kWide; ++k) acc[0][k] = acc[1][k] = 0.f;
    for (int fb = 0; fb < n_fb; ++fb) {
      const int f0 = fb * kFB, nf = min(kFB, m - f0);
      __syncthreads();
      load_state_block(G, f0, nf, d, om);
      __syncthreads();
      outer_acc<kTT, RT::kWide>(pq + f0, ldq, om, ld, nf, ld, acc);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int t = RT::row(i);
      for (int s = 0; s <= t && s < nt; ++s) {
        const float a = A[t * (kTT + 1) + s];
        const float* vr = vs + s * ld;
#pragma unroll
        for (int k = 0; k < RT::kWide; ++k)
          if (RT::col(k) < ld) acc[i][k] = fmaf(a, vr[RT::col(k)], acc[i][k]);
      }
    }
    __syncthreads();   // all reads of qs (projections) and G done
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int k = 0; k < RT::kWide; ++k)
        if (RT::col(k) < ld) qs[RT::row(i) * ld + RT::col(k)] = acc[i][k];
    __syncthreads();
    store_output(qs, nt, d, O + hoff + (size_t)t0 * d, status);
    // G += phi(K)^T [V | 1], each element one fmaf chain from its old value
    {
      const int fg = threadIdx.x / 16, jl = threadIdx.x % 16;
      for (int fb = 0; fb < n_fb; ++fb) {
        const int f0 = fb * kFB, nf = min(kFB, m - f0);
        float g[4][kGramWide];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int k = 0; k < kGramWide; ++k) {
            const int f = fg + 16 * i, j = jl + 16 * k;
            g[i][k] = (f < nf && j < ld) ? G[(size_t)(f0 + f) * ld + j] : 0.f;
          }
        gram_acc<kGramWide>(pk + f0, ldq, vs, ld, nt, ld, g);
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int k = 0; k < kGramWide; ++k) {
            const int f = fg + 16 * i, j = jl + 16 * k;
            if (f < nf && j < ld) G[(size_t)(f0 + f) * ld + j] = g[i][k];
          }
      }
    }
  }
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

SimtPlan simt_plan(bool causal, const Shape& s) {
  SimtPlan p{};
  const int BH = s.BH();
  p.n_fb = (s.m + kFB - 1) / kFB;
  const int tiles = (s.L + kTT - 1) / kTT;
  const int target = 2 * sm_count();
  int want = causal ? (target + BH - 1) / BH : (target + BH * p.n_fb - 1) / (BH * p.n_fb);
  want = max(1, min(want, tiles));
  const int tiles_per = (tiles + want - 1) / want;
  p.chunk = tiles_per * kTT;
  p.n_split = (s.L + p.chunk - 1) / p.chunk;
  const size_t per = (size_t)s.m * (s.d + 1) * sizeof(float);
  size_t off = kWsHeader;
  p.off_partS = off;
  off = align256(off + (size_t)BH * p.n_split * per);
  p.off_state = off;
  off = align256(off + (size_t)BH * (causal ? p.n_split : 1) * per);
  p.bytes = off;
  return p;
}

static size_t state_smem(int d) {
  const int ld = d + 1;
  return sizeof(float) * ((size_t)kFB * ld + 2 * kTT * ld + kTT * (kFB + 1) + kTT);
}
static size_t bidir_out_smem(int d, int m) {
  const int ld = d + 1;
  return sizeof(float) * ((size_t)kTT * ld + 2 * kFB * ld + kTT * (m + 1) + kTT);
}
static size_t causal_out_smem(int d, int m) {
  const int ld = d + 1;
  return sizeof(float) * ((size_t)3 * kTT * ld + kFB * ld + 2 * kTT * (m + 1) + kTT * (kTT + 1) + 2 * kTT);
}

template <typename KernelT>
static cudaError_t set_smem(KernelT k, size_t bytes) {
  return ensure_dynamic_smem(reinterpret_cast<const void*>(k), bytes);
}

template <typename T, int FM>
static cudaError_t state_impl(const void* K, const void* V, const float* omega, float scale, const Shape& s,
                              const SimtPlan& p, char* ws, cudaStream_t stream) {
  float* key_ref = reinterpret_cast<float*>(ws);
  cudaError_t e = launch_prep(omega, s.m, s.d, key_ref, nullptr, nullptr, 0, stream);
  if (e != cudaSuccess) return e;
  const size_t smem = state_smem(s.d);
  auto kern = state_partial_kernel<T, FM>;
  e = set_smem(kern, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.n_split, p.n_fb, s.BH());
  kern<<<grid, kThreads, smem, stream>>>(static_cast<const T*>(K), static_cast<const T*>(V), omega, key_ref, s.L,
                                         s.d, s.m, scale, p.chunk, p.n_split,
                                         reinterpret_cast<float*>(ws + p.off_partS));
  return cudaGetLastError();
}

// (storage type, feature map) as template arguments of `f`
template <typename F>
static cudaError_t dispatch(bool bf16, int fm, F&& f) {
  using Prf = std::integral_constant<int, FAVOR_FM_PRF>;
  using Relu = std::integral_constant<int, FAVOR_FM_RELU>;
  using Elu1 = std::integral_constant<int, FAVOR_FM_ELU1>;
  if (bf16) {
    if (fm == FAVOR_FM_RELU) return f(__nv_bfloat16{}, Relu{});
    if (fm == FAVOR_FM_ELU1) return f(__nv_bfloat16{}, Elu1{});
    return f(__nv_bfloat16{}, Prf{});
  }
  if (fm == FAVOR_FM_RELU) return f(float{}, Relu{});
  if (fm == FAVOR_FM_ELU1) return f(float{}, Elu1{});
  return f(float{}, Prf{});
}

cudaError_t simt_bidir_state(const void* K, const void* V, const float* omega, float scale, const Shape& s,
                             bool bf16, void* ws, int32_t* st, cudaStream_t stream, int fm) {
  (void)st;
  const SimtPlan p = simt_plan(false, s);
  char* w = static_cast<char*>(ws);
  cudaError_t e = dispatch(bf16, fm, [&](auto t, auto f) {
    return state_impl<decltype(t), decltype(f)::value>(K, V, omega, scale, s, p, w, stream);
  });
  if (e != cudaSuccess) return e;
  merge_kernel<<<merge_grid(s), kThreads, 0, stream>>>(reinterpret_cast<float*>(w + p.off_partS), s.d, s.m, p.n_split,
                                                reinterpret_cast<float*>(w + p.off_state));
  return cudaGetLastError();
}

// The decode state layout [bh][j][f] (j <= d, f < m: feature index fastest)
// from the split partials, summed in split order.
// One thread per state element (grid: element blocks x heads), eight
// partials' loads in flight at a time.
__global__ void __launch_bounds__(kThreads) merge_transposed_kernel(const float* __restrict__ partS, int d, int m,
                                                                    int n_split, float* __restrict__ state) {
  const int bh = blockIdx.y;
  const int ld = d + 1;
  const size_t per = (size_t)m * ld;
  const size_t e = (size_t)blockIdx.x * kThreads + threadIdx.x;
  if (e >= per) return;
  const int j = static_cast<int>(e / m), f = static_cast<int>(e - (size_t)j * m);
  const float* src = partS + (size_t)bh * n_split * per + (size_t)f * ld + j;
  float acc = 0.f;
  for (int p0 = 0; p0 < n_split; p0 += 8) {
    float v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = p0 + u < n_split ? src[(size_t)(p0 + u) * per] : 0.f;
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (p0 + u < n_split) acc += v[u];
  }
  state[(size_t)bh * per + e] = acc;
}

// The summed state of a whole sequence into `state` in the decode layout
// [BH][d+1][m]: the same partials and fixed-order merge as the bidirectional
// state, written transposed to the caller's array.
cudaError_t simt_state_export(const void* K, const void* V, const float* omega, float scale, const Shape& s,
                              bool bf16, void* ws, float* state, cudaStream_t stream) {
  const SimtPlan p = simt_plan(false, s);
  char* w = static_cast<char*>(ws);
  cudaError_t e = bf16 ? state_impl<__nv_bfloat16, FAVOR_FM_PRF>(K, V, omega, scale, s, p, w, stream)
                       : state_impl<float, FAVOR_FM_PRF>(K, V, omega, scale, s, p, w, stream);
  if (e != cudaSuccess) return e;
  merge_transposed_kernel<<<merge_grid(s), kThreads, 0, stream>>>(reinterpret_cast<float*>(w + p.off_partS), s.d, s.m,
                                                            p.n_split, state);
  return cudaGetLastError();
}

template <typename T, int FM>
static cudaError_t bidir_out_impl(const void* Q, void* O, const float* omega, float scale, const Shape& s,
                                  const SimtPlan& p, char* ws, int32_t* st, cudaStream_t stream) {
  const size_t smem = bidir_out_smem(s.d, s.m);
  auto kern = bidir_output_kernel<T, FM>;
  cudaError_t e = set_smem(kern, smem);
  if (e != cudaSuccess) return e;
  dim3 grid((s.L + kTT - 1) / kTT, s.BH());
  kern<<<grid, kThreads, smem, stream>>>(static_cast<const T*>(Q), static_cast<T*>(O), omega,
                                         reinterpret_cast<const float*>(ws + p.off_state), s.L, s.d, s.m, scale,
                                         st);
  return cudaGetLastError();
}

cudaError_t simt_bidir_output(const void* Q, void* O, const float* omega, float scale, const Shape& s,
                              bool bf16, void* ws, int32_t* st, cudaStream_t stream, int fm) {
  const SimtPlan p = simt_plan(false, s);
  char* w = static_cast<char*>(ws);
  return dispatch(bf16, fm, [&](auto t, auto f) {
    return bidir_out_impl<decltype(t), decltype(f)::value>(Q, O, omega, scale, s, p, w, st, stream);
  });
}

cudaError_t simt_causal_state(const void* K, const void* V, const float* omega, float scale, const Shape& s,
                              bool bf16, void* ws, int32_t* st, cudaStream_t stream, int fm) {
  (void)st;
  const SimtPlan p = simt_plan(true, s);
  char* w = static_cast<char*>(ws);
  return dispatch(bf16, fm, [&](auto t, auto f) {
    return state_impl<decltype(t), decltype(f)::value>(K, V, omega, scale, s, p, w, stream);
  });
}

template <typename T, int FM>
static cudaError_t causal_out_impl(const void* Q, const void* K, const void* V, void* O, const float* omega,
                                   float scale, const Shape& s, const SimtPlan& p, char* ws, int32_t* st,
                                   cudaStream_t stream) {
  const size_t smem = causal_out_smem(s.d, s.m);
  auto kern = causal_output_kernel<T, FM>;
  cudaError_t e = set_smem(kern, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.n_split, s.BH());
  kern<<<grid, kThreads, smem, stream>>>(
      static_cast<const T*>(Q), static_cast<const T*>(K), static_cast<const T*>(V), static_cast<T*>(O), omega,
      reinterpret_cast<const float*>(ws), reinterpret_cast<const float*>(ws + p.off_partS),
      reinterpret_cast<float*>(ws + p.off_state), s.L, s.d, s.m, scale, p.chunk, p.n_split, st);
  return cudaGetLastError();
}

cudaError_t simt_causal_output(const void* Q, const void* K, const void* V, void* O, const float* omega,
                               float scale, const Shape& s, bool bf16, void* ws, int32_t* st,
                               cudaStream_t stream, int fm) {
  const SimtPlan p = simt_plan(true, s);
  char* w = static_cast<char*>(ws);
  return dispatch(bf16, fm, [&](auto t, auto f) {
    return causal_out_impl<decltype(t), decltype(f)::value>(Q, K, V, O, omega, scale, s, p, w, st, stream);
  });
}

// ===========================================================================
// Backward of the bidirectional pass (CUDA cores, fp32 arithmetic): the
// chain rule through the forward ("Performer" digest, §Key equations):
//   N = phi(Q) S,  D = phi(Q) z,  O = N / D;  dN^ = [dO / D | dD] with
//   dD = -(dO . N) / D^2;
//   dphi(Q) = S~ dN^,  dS~ = phi(Q)^T dN^,  dphi(K) = dS~ [V | 1]^T,
//   dV = phi(K) dS~[:, :d];
//   through the feature map, g = dphi phi (positive random features) or
//   dphi [s w.x > 0] (Performer-ReLU):  dx = s (sum_i g_i w_i - [prf] s x sum_i g_i).
// Key features use the per-call reference R and query features the bound
// s |q| max_i |w_i| - 20 in both passes that meet through dN^: every
// gradient is invariant to these constants, which cancel as in the forward.
// ===========================================================================
namespace {

constexpr int kBT = 32;   // tokens per backward tile

template <int TT, typename T>
__device__ __forceinline__ void load_tile(const T* __restrict__ src, int nt, int d, float* dst) {
  const int ld = d + 1;
  for (int e = threadIdx.x; e < TT * d; e += kThreads) {
    const int t = e / d, c = e - t * d;
    dst[t * ld + c] = (t < nt) ? to_f32(src[(size_t)t * d + c]) : 0.f;
  }
}

template <int TT>
__device__ __forceinline__ void tile_norms(const float* xs, int d, float* out) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int t = warp; t < TT; t += kThreads / 32) {
    float a = 0.f;
    for (int c = lane; c < d; c += 32) a = fmaf(xs[t * (d + 1) + c], xs[t * (d + 1) + c], a);
    a = warp_sum(a);
    if (lane == 0) out[t] = a;
  }
}

// feature from p = s w.x and the row constant c
template <int FM>
__device__ __forceinline__ float bwd_feature(float p, float c) {
  if constexpr (FM == FAVOR_FM_PRF) return expf(p - c);
  else return key_feature<FM>(p, 0.f, 0.f);
}


// Performer-ReLU's slope [w.x > 0] jumps at w.x = 0, so the backward takes
// that sign from the exact projection wherever the fp32 one is within its
// rounding bound: |fl(w.x) - w.x| <= d 2^-24 sum_c |w_c x_c| <= d 2^-24 |x| W
// (W = max_i |w_i|), with a factor 2 of margin.  The threshold per row is
// carried in the row constant, which the ReLU features do not use.
__device__ __forceinline__ float relu_sign_bound(float x_norm2, int d, float W) {
  return 2.0f * static_cast<float>(d) * 5.9604645e-8f * sqrtf(x_norm2) * W;
}

// w.x in fp64 (the products of two fp32 numbers are exact in fp64)
__device__ __forceinline__ float exact_dot(const float* x, const float* w, int d) {
  double a = 0.0;
  for (int c = 0; c < d; ++c) a = fma(static_cast<double>(x[c]), static_cast<double>(w[c]), a);
  return static_cast<float>(a);
}

// features of the tile rows xs against all m rows of Omega into P [TT][ldp];
// for Performer-ReLU rowc[t] is the sign bound of row t (relu_sign_bound)
template <int TT, int FM>
__device__ void tile_features(const float* xs, const float* rowc, int nt, int d, int m, float scale,
                              const float* __restrict__ omega, float* om, float* P, int ldp) {
  const int ld = d + 1;
  const int n_fb = (m + kFB - 1) / kFB;
  using RT = RegTile<TT>;
  for (int fb = 0; fb < n_fb; ++fb) {
    const int f0 = fb * kFB, nf = min(kFB, m - f0);
    __syncthreads();
    load_omega_block(omega, f0, nf, d, om);
    __syncthreads();
    float acc[2][RT::kCols];
    rowdot_block<TT>(xs, ld, om, ld, d, acc);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int t = RT::row(i);
#pragma unroll
      for (int k = 0; k < RT::kCols; ++k) {
        const int f = RT::col(k);
        float a = acc[i][k];
        if constexpr (FM == FAVOR_FM_RELU) {
          if (t < nt && f < nf && fabsf(a) <= rowc[t]) a = exact_dot(xs + t * ld, om + f * ld, d);
        }
        if (f < nf) P[t * ldp + f0 + f] = t < nt ? bwd_feature<FM>(scale * a, rowc[t]) : 0.f;
      }
    }
  }
  __syncthreads();
}

// g <- dphi * phi (prf), dphi [phi > 0] (relu) or dphi min(phi, 1) (1 + elu:
// its slope is 1 where phi = 1 + a >= 1 and exp(a) = phi below) in G;
// gsum[t] = sum_i g
template <int TT, int FM>
__device__ void tile_g(const float* P, float* G, int ldp, int m, float* gsum) {
  for (int e = threadIdx.x; e < TT * m; e += kThreads) {
    const int t = e / m, i = e - t * m;
    const float ph = P[t * ldp + i], dp = G[t * ldp + i];
    if constexpr (FM == FAVOR_FM_PRF) G[t * ldp + i] = dp * ph;
    else if constexpr (FM == FAVOR_FM_ELU1) G[t * ldp + i] = dp * fminf(ph, 1.f);
    else G[t * ldp + i] = ph > 0.f ? dp : 0.f;
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int t = warp; t < TT; t += kThreads / 32) {
    float a = 0.f;
    for (int i = lane; i < m; i += 32) a += G[t * ldp + i];
    a = warp_sum(a);
    if (lane == 0) gsum[t] = a;
  }
  __syncthreads();
}

// dx_t = s (sum_i g[t][i] w_i - [prf] s x_t sum_i g[t][i]) stored as T [nt][d]
template <int TT, typename T, int FM>
__device__ void tile_input_grad(const float* xs, const float* G, int ldp, const float* gsum, int nt, int d, int m,
                                float scale, const float* __restrict__ omega, float* om, T* __restrict__ out) {
  using RT = RegTile<TT>;
  const int ld = d + 1;
  float acc[2][RT::kWide];
#pragma unroll
  for (int k = 0; k < RT::kWide; ++k) acc[0][k] = acc[1][k] = 0.f;
  const int n_fb = (m + kFB - 1) / kFB;
  for (int fb = 0; fb < n_fb; ++fb) {
    const int f0 = fb * kFB, nf = min(kFB, m - f0);
    __syncthreads();
    load_omega_block(omega, f0, nf, d, om);
    __syncthreads();
    outer_acc<TT, RT::kWide>(G + f0, ldp, om, ld, nf, d, acc);
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int t = RT::row(i);
#pragma unroll
    for (int k = 0; k < RT::kWide; ++k) {
      const int c = RT::col(k);
      if (t < nt && c < d) {
        float gx = acc[i][k];
        if constexpr (FM == FAVOR_FM_PRF) gx -= scale * xs[t * ld + c] * gsum[t];
        out[(size_t)t * d + c] = from_f32<T>(scale * gx);
      }
    }
  }
}

// Query pass, one tile of kBT tokens of one head: phi(Q), N and D from S~,
// dN^ (also written to the workspace for the feature-block pass), dphi(Q)
// = S~ dN^ and dQ.
template <typename T, int FM>
__global__ void __launch_bounds__(kThreads, 2) bwd_query_kernel(
    const T* __restrict__ Q, const T* __restrict__ dO, T* __restrict__ dQ, const float* __restrict__ omega,
    const float* __restrict__ key_ref, const float* __restrict__ state, float* __restrict__ dnw, int L, int d, int m,
    float scale, int32_t* status) {
  extern __shared__ float smem[];
  const int ld = d + 1, ldp = m + 1;
  const int bh = blockIdx.y, t0 = blockIdx.x * kBT, nt = min(kBT, L - t0);
  float* xs = smem;                 // [kBT][ld] s-free q rows
  float* go = xs + kBT * ld;        // [kBT][ld] dO, then dN^
  float* nd = go + kBT * ld;        // [kBT][ld] N | D
  float* om = nd + kBT * ld;        // [kFB][ld] Omega block / S~ block
  float* P = om + kFB * ld;         // [kBT][ldp] phi(Q)
  float* G = P + kBT * ldp;         // [kBT][ldp] dphi(Q), then g
  float* rs = G + kBT * ldp;        // [kBT] squared norms, then row constants
  float* gsum = rs + kBT;           // [kBT]
  const size_t row0 = (size_t)bh * L + t0;
  load_tile<kBT>(Q + row0 * d, nt, d, xs);
  load_tile<kBT>(dO + row0 * d, nt, d, go);
  __syncthreads();
  tile_norms<kBT>(xs, d, rs);
  __syncthreads();
  float R, W;
  key_reference(key_ref, m, &R, &W);
  if (threadIdx.x < kBT)
    rs[threadIdx.x] = FM == FAVOR_FM_PRF    ? scale * sqrtf(rs[threadIdx.x]) * W - 20.0f
                      : FM == FAVOR_FM_RELU ? relu_sign_bound(rs[threadIdx.x], d, W)
                                            : 0.f;
  tile_features<kBT, FM>(xs, rs, nt, d, m, scale, omega, om, P, ldp);

  // N | D
  using RT = RegTile<kBT>;
  const float* Sh = state + (size_t)bh * m * ld;
  float acc[2][RT::kWide];
#pragma unroll
  for (int k = 0; k < RT::kWide; ++k) acc[0][k] = acc[1][k] = 0.f;
  const int n_fb = (m + kFB - 1) / kFB;
  for (int fb = 0; fb < n_fb; ++fb) {
    const int f0 = fb * kFB, nf = min(kFB, m - f0);
    __syncthreads();
    load_state_block(Sh, f0, nf, d, om);
    __syncthreads();
    outer_acc<kBT, RT::kWide>(P + f0, ldp, om, ld, nf, ld, acc);
  }
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int k = 0; k < RT::kWide; ++k)
      if (RT::col(k) < ld) nd[RT::row(i) * ld + RT::col(k)] = acc[i][k];
  __syncthreads();
  // dN^ = [dO / D | -(dO . N) / D^2], one warp per row
  {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int t = warp; t < kBT; t += kThreads / 32) {
      const float D = nd[t * ld + d];
      float a = 0.f;
      for (int j = lane; j < d; j += 32) a = fmaf(go[t * ld + j], nd[t * ld + j], a);
      a = warp_sum(a);
      const bool valid = t < nt;
      if (valid && lane == 0 && (!(D > 0.f) || !isfinite(D))) report_status(status, FAVOR_ERR_NONFINITE);
      const float inv = 1.0f / D;
      __syncwarp();
      for (int j = lane; j < d; j += 32) go[t * ld + j] = valid ? go[t * ld + j] * inv : 0.f;
      if (lane == 0) go[t * ld + d] = valid ? -a * inv * inv : 0.f;
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < nt * ld; e += kThreads) dnw[row0 * ld + e] = go[e];
  // dphi(Q) = S~ dN^
  for (int fb = 0; fb < n_fb; ++fb) {
    const int f0 = fb * kFB, nf = min(kFB, m - f0);
    __syncthreads();
    load_state_block(Sh, f0, nf, d, om);
    __syncthreads();
    float g[2][RT::kCols];
    rowdot_block<kBT>(go, ld, om, ld, ld, g);
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int k = 0; k < RT::kCols; ++k)
        if (RT::col(k) < nf) G[RT::row(i) * ldp + f0 + RT::col(k)] = g[i][k];
  }
  __syncthreads();
  tile_g<kBT, FM>(P, G, ldp, m, gsum);
  tile_input_grad<kBT, T, FM>(xs, G, ldp, gsum, nt, d, m, scale, omega, om, dQ + row0 * d);
}

// Feature-block pass: partial dS~ of a token split and a block of features,
// sum_t phi(q_t)_f dN^_t (the same query features as the query pass).
template <typename T, int FM>
__global__ void __launch_bounds__(kThreads) bwd_dstate_partial_kernel(
    const T* __restrict__ Q, const float* __restrict__ dnw, const float* __restrict__ omega,
    const float* __restrict__ key_ref, int L, int d, int m, float scale, int chunk, int n_split,
    float* __restrict__ dpart) {
  extern __shared__ float smem[];
  const int split = blockIdx.x, fb = blockIdx.y, bh = blockIdx.z;
  const int ld = d + 1;
  float* om = smem;                   // [kFB][ld]
  float* xs = om + kFB * ld;          // [kBT][ld]
  float* dn = xs + kBT * ld;          // [kBT][ld]
  float* ph = dn + kBT * ld;          // [kBT][kFB + 1]
  float* rs = ph + kBT * (kFB + 1);   // [kBT]
  const int f0 = fb * kFB, nf = min(kFB, m - f0);
  const int l0 = split * chunk, l1 = min(L, l0 + chunk);
  float R, W;
  key_reference(key_ref, m, &R, &W);
  load_omega_block(omega, f0, nf, d, om);
  using RT = RegTile<kBT>;
  float acc[4][kGramWide];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int k = 0; k < kGramWide; ++k) acc[i][k] = 0.f;
  for (int t0 = l0; t0 < l1; t0 += kBT) {
    const int nt = min(kBT, l1 - t0);
    const size_t row0 = (size_t)bh * L + t0;
    __syncthreads();
    load_tile<kBT>(Q + row0 * d, nt, d, xs);
    for (int e = threadIdx.x; e < kBT * ld; e += kThreads) dn[e] = e < nt * ld ? dnw[row0 * ld + e] : 0.f;
    __syncthreads();
    tile_norms<kBT>(xs, d, rs);
    __syncthreads();
    {
      float a[2][RT::kCols];
      rowdot_block<kBT>(xs, ld, om, ld, d, a);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int t = RT::row(i);
        const float c = FM == FAVOR_FM_PRF ? scale * sqrtf(rs[t]) * W - 20.0f : 0.f;
#pragma unroll
        for (int k = 0; k < RT::kCols; ++k) {
          const int f = RT::col(k);
          ph[t * (kFB + 1) + f] = (t < nt && f < nf) ? bwd_feature<FM>(scale * a[i][k], c) : 0.f;
        }
      }
    }
    __syncthreads();
    gram_acc<kGramWide>(ph, kFB + 1, dn, ld, nt, ld, acc);
  }
  const int fg = threadIdx.x / 16, jl = threadIdx.x % 16;
  float* dst = dpart + (((size_t)bh * n_split + split) * m + f0) * ld;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int f = fg + 16 * i;
    if (f < nf)
#pragma unroll
      for (int k = 0; k < kGramWide; ++k) {
        const int j = jl + 16 * k;
        if (j < ld) dst[(size_t)f * ld + j] = acc[i][k];
      }
  }
}

// Key pass, one tile of kBT tokens of one head: phi(K), dphi(K) = dS~ [V|1]^T,
// dV = phi(K) dS~[:, :d] and dK.
template <typename T, int FM>
__global__ void __launch_bounds__(kThreads, 2) bwd_key_kernel(
    const T* __restrict__ K, const T* __restrict__ V, T* __restrict__ dK, T* __restrict__ dV,
    const float* __restrict__ omega, const float* __restrict__ key_ref, const float* __restrict__ dstate, int L,
    int d, int m, float scale) {
  extern __shared__ float smem[];
  const int ld = d + 1, ldp = m + 1;
  const int bh = blockIdx.y, t0 = blockIdx.x * kBT, nt = min(kBT, L - t0);
  float* xs = smem;                 // [kBT][ld] k rows
  float* vs = xs + kBT * ld;        // [kBT][ld] v | 1
  float* om = vs + kBT * ld;        // [kFB][ld]
  float* P = om + kFB * ld;         // [kBT][ldp] phi(K)
  float* G = P + kBT * ldp;         // [kBT][ldp] dphi(K), then g
  float* rs = G + kBT * ldp;        // [kBT]
  float* gsum = rs + kBT;           // [kBT]
  const size_t row0 = (size_t)bh * L + t0;
  load_tile<kBT>(K + row0 * d, nt, d, xs);
  load_tile<kBT>(V + row0 * d, nt, d, vs);
  if (threadIdx.x < kBT) vs[threadIdx.x * ld + d] = threadIdx.x < nt ? 1.f : 0.f;
  __syncthreads();
  tile_norms<kBT>(xs, d, rs);
  __syncthreads();
  float R, W;
  key_reference(key_ref, m, &R, &W);
  if (threadIdx.x < kBT)
    rs[threadIdx.x] = FM == FAVOR_FM_PRF    ? 0.5f * scale * scale * rs[threadIdx.x] + R
                      : FM == FAVOR_FM_RELU ? relu_sign_bound(rs[threadIdx.x], d, W)
                                            : 0.f;
  tile_features<kBT, FM>(xs, rs, nt, d, m, scale, omega, om, P, ldp);

  using RT = RegTile<kBT>;
  const float* dS = dstate + (size_t)bh * m * ld;
  float accv[2][RT::kWide];
#pragma unroll
  for (int k = 0; k < RT::kWide; ++k) accv[0][k] = accv[1][k] = 0.f;
  const int n_fb = (m + kFB - 1) / kFB;
  for (int fb = 0; fb < n_fb; ++fb) {
    const int f0 = fb * kFB, nf = min(kFB, m - f0);
    __syncthreads();
    load_state_block(dS, f0, nf, d, om);
    __syncthreads();
    float g[2][RT::kCols];
    rowdot_block<kBT>(vs, ld, om, ld, ld, g);
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int k = 0; k < RT::kCols; ++k)
        if (RT::col(k) < nf) G[RT::row(i) * ldp + f0 + RT::col(k)] = g[i][k];
    outer_acc<kBT, RT::kWide>(P + f0, ldp, om, ld, nf, d, accv);
  }
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int k = 0; k < RT::kWide; ++k) {
      const int t = RT::row(i), j = RT::col(k);
      if (t < nt && j < d) dV[(row0 + t) * d + j] = from_f32<T>(accv[i][k]);
    }
  __syncthreads();
  tile_g<kBT, FM>(P, G, ldp, m, gsum);
  tile_input_grad<kBT, T, FM>(xs, G, ldp, gsum, nt, d, m, scale, omega, om, dK + row0 * d);
}

size_t bwd_tile_smem(int d, int m) {
  const int ld = d + 1, ldp = m + 1;
  return sizeof(float) * ((size_t)3 * kBT * ld + (size_t)kFB * ld + (size_t)2 * kBT * ldp + 2 * kBT);
}
size_t bwd_dstate_smem(int d) {
  const int ld = d + 1;
  return sizeof(float) * ((size_t)kFB * ld + (size_t)2 * kBT * ld + (size_t)kBT * (kFB + 1) + kBT);
}

// ---------------------------------------------------------------------------
// Causal backward: one CTA per (chunk of tokens, head), walking the chunk in
// tiles of kCT tokens.  Each walk starts from its chunk's exclusive prefix
// (query walk) or suffix (key walk) state, summed beforehand from per-chunk
// partials in chunk order.  With the prefix state G~_c = sum over earlier
// tiles of phi(k) [v ; 1]^T and, inside a tile, A = tril(phi(Q) phi(K)^T):
//   N^_t = phi(q_t)^T G~_c + sum_{s<=t} A_ts [v_s ; 1]   (N | D)
//   dphi(q_t) = G~_c dN^_t + sum_{s<=t} (dN^_t . [v_s ; 1]) phi(k_s)
// (forward walk), and with the suffix state H_c = sum over later tiles of
// phi(q) dN^T (reverse walk):
//   dphi(k_s) = H_c [v_s ; 1] + sum_{t>=s} (dN^_t . [v_s ; 1]) phi(q_t)
//   dV_s = H_c[:, :d]^T phi(k_s) + sum_{t>=s} A_ts dN_t
// ---------------------------------------------------------------------------
constexpr int kCT = 16;

// state[f][j] += sum_{t < nt} X[t][f] Y[t][j] for all m features and j < ld
// (a per-head [m][ld] state in global memory, each element owned by one
// thread), by blocks of 64 features.  X rows of stride ldx hold the m
// features (the block past m reads into the next row: discarded).
__device__ __forceinline__ void add_tile_gram(const float* X, int ldx, const float* Y, int ld, int nt, int m,
                                              float* __restrict__ state) {
  const int fg = threadIdx.x / 16, jl = threadIdx.x % 16;
  const int n_fb = (m + kFB - 1) / kFB;
  for (int fb = 0; fb < n_fb; ++fb) {
    const int f0 = fb * kFB, nf = min(kFB, m - f0);
    float g[4][kGramWide];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int k = 0; k < kGramWide; ++k) g[i][k] = 0.f;
    gram_acc<kGramWide>(X + f0, ldx, Y, ld, nt, ld, g);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int f = fg + 16 * i;
      if (f < nf)
#pragma unroll
        for (int k = 0; k < kGramWide; ++k) {
          const int j = jl + 16 * k;
          if (j < ld) state[(size_t)(f0 + f) * ld + j] += g[i][k];
        }
    }
  }
}

template <typename T, int FM>
__global__ void __launch_bounds__(kThreads) cbwd_query_kernel(
    const T* __restrict__ Q, const T* __restrict__ K, const T* __restrict__ V, const T* __restrict__ dO,
    T* __restrict__ dQ, const float* __restrict__ omega, const float* __restrict__ key_ref, float* __restrict__ gst,
    float* __restrict__ dnw, int L, int d, int m, float scale, int chunk, int n_chunk, int32_t* status) {
  extern __shared__ float smem[];
  const int ld = d + 1, ldp = m + 1;
  const int c = blockIdx.x, bh = blockIdx.y;
  const int l0 = c * chunk, l1 = min(L, l0 + chunk);
  float* xs = smem;                   // [kCT][ld] q
  float* ks = xs + kCT * ld;          // [kCT][ld] k
  float* vs = ks + kCT * ld;          // [kCT][ld] v | 1
  float* go = vs + kCT * ld;          // [kCT][ld] dO, then dN^
  float* nd = go + kCT * ld;          // [kCT][ld] N | D
  float* om = nd + kCT * ld;          // [kFB][ld]
  float* P = om + kFB * ld;           // [kCT][ldp] phi(Q)
  float* Pk = P + kCT * ldp;          // [kCT][ldp] phi(K)
  float* G = Pk + kCT * ldp;          // [kCT][ldp] dphi(Q), then g
  float* A = G + kCT * ldp;           // [kCT][kCT + 1]
  float* Bm = A + kCT * (kCT + 1);    // [kCT][kCT + 1]
  float* rq = Bm + kCT * (kCT + 1);   // [kCT]
  float* rk = rq + kCT;               // [kCT]
  float* gsum = rk + kCT;             // [kCT]
  float* Gh = gst + ((size_t)bh * n_chunk + c) * m * ld;   // the chunk's exclusive prefix state
  float R, W;
  key_reference(key_ref, m, &R, &W);
  const int n_fb = (m + kFB - 1) / kFB;
  using RT = RegTile<kCT>;
  for (int t0 = l0; t0 < l1; t0 += kCT) {
    const int nt = min(kCT, l1 - t0);
    const size_t row0 = (size_t)bh * L + t0;
    __syncthreads();
    load_tile<kCT>(Q + row0 * d, nt, d, xs);
    load_tile<kCT>(K + row0 * d, nt, d, ks);
    load_tile<kCT>(V + row0 * d, nt, d, vs);
    load_tile<kCT>(dO + row0 * d, nt, d, go);
    if (threadIdx.x < kCT) vs[threadIdx.x * ld + d] = threadIdx.x < nt ? 1.f : 0.f;
    __syncthreads();
    tile_norms<kCT>(xs, d, rq);
    tile_norms<kCT>(ks, d, rk);
    __syncthreads();
    if (threadIdx.x < kCT) {
      rq[threadIdx.x] = FM == FAVOR_FM_PRF    ? scale * sqrtf(rq[threadIdx.x]) * W - 20.0f
                        : FM == FAVOR_FM_RELU ? relu_sign_bound(rq[threadIdx.x], d, W)
                                              : 0.f;
      rk[threadIdx.x] = FM == FAVOR_FM_PRF    ? 0.5f * scale * scale * rk[threadIdx.x] + R
                        : FM == FAVOR_FM_RELU ? relu_sign_bound(rk[threadIdx.x], d, W)
                                              : 0.f;
    }
    tile_features<kCT, FM>(xs, rq, nt, d, m, scale, omega, om, P, ldp);
    tile_features<kCT, FM>(ks, rk, nt, d, m, scale, omega, om, Pk, ldp);
    for (int e = threadIdx.x; e < kCT * kCT; e += kThreads) {
      const int t = e / kCT, s_ = e - t * kCT;
      float a = 0.f;
      if (s_ <= t && t < nt)
        for (int i = 0; i < m; ++i) a = fmaf(P[t * ldp + i], Pk[s_ * ldp + i], a);
      A[t * (kCT + 1) + s_] = a;
    }
    // N | D: prefix state part, then the tile's own (masked) part
    float acc[2][RT::kWide];
#pragma unroll
    for (int k = 0; k < RT::kWide; ++k) acc[0][k] = acc[1][k] = 0.f;
    for (int fb = 0; fb < n_fb; ++fb) {
      const int f0 = fb * kFB, nf = min(kFB, m - f0);
      __syncthreads();
      load_state_block(Gh, f0, nf, d, om);
      __syncthreads();
      outer_acc<kCT, RT::kWide>(P + f0, ldp, om, ld, nf, ld, acc);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int t = RT::row(i);
#pragma unroll
      for (int k = 0; k < RT::kWide; ++k) {
        const int j = RT::col(k);
        if (j < ld) {
          float a = acc[i][k];
          for (int s_ = 0; s_ <= t; ++s_) a = fmaf(A[t * (kCT + 1) + s_], vs[s_ * ld + j], a);
          nd[t * ld + j] = a;
        }
      }
    }
    __syncthreads();
    {
      const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
      for (int t = warp; t < kCT; t += kThreads / 32) {
        const float D = nd[t * ld + d];
        float a = 0.f;
        for (int j = lane; j < d; j += 32) a = fmaf(go[t * ld + j], nd[t * ld + j], a);
        a = warp_sum(a);
        const bool valid = t < nt;
        if (valid && lane == 0 && (!(D > 0.f) || !isfinite(D))) report_status(status, FAVOR_ERR_NONFINITE);
        const float inv = 1.0f / D;
        __syncwarp();
        for (int j = lane; j < d; j += 32) go[t * ld + j] = valid ? go[t * ld + j] * inv : 0.f;
        if (lane == 0) go[t * ld + d] = valid ? -a * inv * inv : 0.f;
      }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < nt * ld; e += kThreads) dnw[row0 * ld + e] = go[e];
    for (int e = threadIdx.x; e < kCT * kCT; e += kThreads) {
      const int t = e / kCT, s_ = e - t * kCT;
      float a = 0.f;
      if (s_ <= t)
        for (int j = 0; j < ld; ++j) a = fmaf(vs[s_ * ld + j], go[t * ld + j], a);
      Bm[t * (kCT + 1) + s_] = a;
    }
    // dphi(Q) = G~ dN^ + sum_{s<=t} B_ts phi(k_s)
    for (int fb = 0; fb < n_fb; ++fb) {
      const int f0 = fb * kFB, nf = min(kFB, m - f0);
      __syncthreads();
      load_state_block(Gh, f0, nf, d, om);
      __syncthreads();
      float g[2][RT::kCols];
      rowdot_block<kCT>(go, ld, om, ld, ld, g);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int t = RT::row(i);
#pragma unroll
        for (int k = 0; k < RT::kCols; ++k) {
          const int f = RT::col(k);
          if (f < nf) {
            float a = g[i][k];
            for (int s_ = 0; s_ <= t; ++s_) a = fmaf(Bm[t * (kCT + 1) + s_], Pk[s_ * ldp + f0 + f], a);
            G[t * ldp + f0 + f] = a;
          }
        }
      }
    }
    __syncthreads();
    tile_g<kCT, FM>(P, G, ldp, m, gsum);
    tile_input_grad<kCT, T, FM>(xs, G, ldp, gsum, nt, d, m, scale, omega, om, dQ + row0 * d);
    // G~ += phi(K)^T [V | 1] of this tile (each element owned by one thread)
    add_tile_gram(Pk, ldp, vs, ld, nt, m, Gh);
  }
}

template <typename T, int FM>
__global__ void __launch_bounds__(kThreads) cbwd_key_kernel(
    const T* __restrict__ Q, const T* __restrict__ K, const T* __restrict__ V, T* __restrict__ dK,
    T* __restrict__ dV, const float* __restrict__ omega, const float* __restrict__ key_ref, float* __restrict__ hst,
    const float* __restrict__ dnw, int L, int d, int m, float scale, int chunk, int n_chunk) {
  extern __shared__ float smem[];
  const int ld = d + 1, ldp = m + 1;
  const int c = blockIdx.x, bh = blockIdx.y;
  const int l0 = c * chunk, l1 = min(L, l0 + chunk);
  float* xs = smem;                   // [kCT][ld] q
  float* ks = xs + kCT * ld;          // [kCT][ld] k
  float* vs = ks + kCT * ld;          // [kCT][ld] v | 1
  float* go = vs + kCT * ld;          // [kCT][ld] dN^
  float* nd = go + kCT * ld;          // unused here (same layout as the query kernel)
  float* om = nd + kCT * ld;          // [kFB][ld]
  float* P = om + kFB * ld;           // [kCT][ldp] phi(Q)
  float* Pk = P + kCT * ldp;          // [kCT][ldp] phi(K)
  float* G = Pk + kCT * ldp;          // [kCT][ldp] dphi(K), then g
  float* A = G + kCT * ldp;           // [kCT][kCT + 1]  A_st = phi(k_s).phi(q_t), t >= s
  float* Cm = A + kCT * (kCT + 1);    // [kCT][kCT + 1]  C_st = dN^_t . [v_s ; 1], t >= s
  float* rq = Cm + kCT * (kCT + 1);   // [kCT]
  float* rk = rq + kCT;               // [kCT]
  float* gsum = rk + kCT;             // [kCT]
  float* Hh = hst + ((size_t)bh * n_chunk + c) * m * ld;   // the chunk's exclusive suffix state
  float R, W;
  key_reference(key_ref, m, &R, &W);
  const int n_fb = (m + kFB - 1) / kFB;
  using RT = RegTile<kCT>;
  const int n_tiles = (l1 - l0 + kCT - 1) / kCT;
  for (int tile = n_tiles - 1; tile >= 0; --tile) {
    const int t0 = l0 + tile * kCT;
    const int nt = min(kCT, l1 - t0);
    const size_t row0 = (size_t)bh * L + t0;
    __syncthreads();
    load_tile<kCT>(Q + row0 * d, nt, d, xs);
    load_tile<kCT>(K + row0 * d, nt, d, ks);
    load_tile<kCT>(V + row0 * d, nt, d, vs);
    for (int e = threadIdx.x; e < kCT * ld; e += kThreads) go[e] = e < nt * ld ? dnw[row0 * ld + e] : 0.f;
    if (threadIdx.x < kCT) vs[threadIdx.x * ld + d] = threadIdx.x < nt ? 1.f : 0.f;
    __syncthreads();
    tile_norms<kCT>(xs, d, rq);
    tile_norms<kCT>(ks, d, rk);
    __syncthreads();
    if (threadIdx.x < kCT) {
      rq[threadIdx.x] = FM == FAVOR_FM_PRF    ? scale * sqrtf(rq[threadIdx.x]) * W - 20.0f
                        : FM == FAVOR_FM_RELU ? relu_sign_bound(rq[threadIdx.x], d, W)
                                              : 0.f;
      rk[threadIdx.x] = FM == FAVOR_FM_PRF    ? 0.5f * scale * scale * rk[threadIdx.x] + R
                        : FM == FAVOR_FM_RELU ? relu_sign_bound(rk[threadIdx.x], d, W)
                                              : 0.f;
    }
    tile_features<kCT, FM>(xs, rq, nt, d, m, scale, omega, om, P, ldp);
    tile_features<kCT, FM>(ks, rk, nt, d, m, scale, omega, om, Pk, ldp);
    for (int e = threadIdx.x; e < kCT * kCT; e += kThreads) {
      const int s_ = e / kCT, t = e - s_ * kCT;
      float a = 0.f, c = 0.f;
      if (t >= s_ && t < nt) {
        for (int i = 0; i < m; ++i) a = fmaf(Pk[s_ * ldp + i], P[t * ldp + i], a);
        for (int j = 0; j < ld; ++j) c = fmaf(go[t * ld + j], vs[s_ * ld + j], c);
      }
      A[s_ * (kCT + 1) + t] = a;
      Cm[s_ * (kCT + 1) + t] = c;
    }
    float accv[2][RT::kWide];
#pragma unroll
    for (int k = 0; k < RT::kWide; ++k) accv[0][k] = accv[1][k] = 0.f;
    for (int fb = 0; fb < n_fb; ++fb) {
      const int f0 = fb * kFB, nf = min(kFB, m - f0);
      __syncthreads();
      load_state_block(Hh, f0, nf, d, om);
      __syncthreads();
      float g[2][RT::kCols];
      rowdot_block<kCT>(vs, ld, om, ld, ld, g);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int s_ = RT::row(i);
#pragma unroll
        for (int k = 0; k < RT::kCols; ++k) {
          const int f = RT::col(k);
          if (f < nf) {
            float a = g[i][k];
            for (int t = s_; t < kCT; ++t) a = fmaf(Cm[s_ * (kCT + 1) + t], P[t * ldp + f0 + f], a);
            G[s_ * ldp + f0 + f] = a;
          }
        }
      }
      outer_acc<kCT, RT::kWide>(Pk + f0, ldp, om, ld, nf, d, accv);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int s_ = RT::row(i);
#pragma unroll
      for (int k = 0; k < RT::kWide; ++k) {
        const int j = RT::col(k);
        if (s_ < nt && j < d) {
          float a = accv[i][k];
          for (int t = s_; t < kCT; ++t) a = fmaf(A[s_ * (kCT + 1) + t], go[t * ld + j], a);
          dV[(row0 + s_) * d + j] = from_f32<T>(a);
        }
      }
    }
    __syncthreads();
    tile_g<kCT, FM>(Pk, G, ldp, m, gsum);
    tile_input_grad<kCT, T, FM>(ks, G, ldp, gsum, nt, d, m, scale, omega, om, dK + row0 * d);
    // H += phi(Q)^T dN^ of this tile
    add_tile_gram(P, ldp, go, ld, nt, m, Hh);
  }
}

// Chunk states of one head in place: exclusive prefix (reverse = false) or
// suffix (reverse = true) sums, in chunk order.
__global__ void __launch_bounds__(kThreads) chunk_scan_kernel(float* __restrict__ cst, int per, int n_chunk,
                                                              bool reverse) {
  const int e = blockIdx.x * kThreads + threadIdx.x, bh = blockIdx.y;
  if (e >= per) return;
  float* base = cst + (size_t)bh * n_chunk * per + e;
  float run = 0.f;
  // eight chunks' loads in flight before their stores (the scan is in place,
  // so the compiler would otherwise wait for each load behind the previous
  // store); the running sum keeps its order
  for (int i0 = 0; i0 < n_chunk; i0 += 8) {
    float x[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u;
      const int c = reverse ? n_chunk - 1 - i : i;
      x[u] = i < n_chunk ? base[(size_t)c * per] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = i0 + u;
      if (i >= n_chunk) break;
      const int c = reverse ? n_chunk - 1 - i : i;
      base[(size_t)c * per] = run;
      run += x[u];
    }
  }
}

size_t cbwd_smem(int d, int m) {
  const int ld = d + 1, ldp = m + 1;
  return sizeof(float) * ((size_t)5 * kCT * ld + (size_t)kFB * ld + (size_t)3 * kCT * ldp +
                          (size_t)2 * kCT * (kCT + 1) + 3 * kCT);
}

}  // namespace

BwdPlan bwd_plan(const Shape& s) {
  BwdPlan b{};
  b.fwd = simt_plan(false, s);
  const size_t ld = (size_t)s.d + 1, BH = (size_t)s.BH();
  size_t off = align256(b.fwd.bytes);
  b.off_dn = off;
  off = align256(off + BH * s.L * ld * sizeof(float));
  b.off_dpart = off;
  off = align256(off + BH * b.fwd.n_split * s.m * ld * sizeof(float));
  b.off_dstate = off;
  off = align256(off + BH * s.m * ld * sizeof(float));
  b.bytes = off;
  // causal chunks: about four waves of two CTAs per SM over the heads
  const int tiles = (s.L + kCT - 1) / kCT;
  int want = (8 * sm_count() + s.BH() - 1) / s.BH();
  want = max(1, min(want, tiles));
  b.c_chunk = max(1, (tiles + want - 1) / want) * kCT;
  b.c_n = (s.L + b.c_chunk - 1) / b.c_chunk;
  b.off_cstate = b.off_dpart;
  b.bytes = max(b.bytes, align256(b.off_cstate + BH * b.c_n * s.m * ld * sizeof(float)));
  return b;
}

cudaError_t simt_bwd_causal(const void* Q, const void* K, const void* V, const void* dO, void* dQ, void* dK,
                            void* dV, const float* omega, float scale, const Shape& s, bool bf16, void* ws, int32_t* st,
                            cudaStream_t stream, int fm) {
  const BwdPlan b = bwd_plan(s);
  char* w = static_cast<char*>(ws);
  float* key_ref = reinterpret_cast<float*>(w);
  cudaError_t e = launch_prep(omega, s.m, s.d, key_ref, nullptr, nullptr, 0, stream);
  if (e != cudaSuccess) return e;
  // per (head, chunk): chunk sums of phi(k) [v ; 1]^T -> exclusive prefixes
  // (query walks) -> chunk sums of phi(q) dN^T -> exclusive suffixes (key walks)
  float* cst = reinterpret_cast<float*>(w + b.off_cstate);
  float* dnw = reinterpret_cast<float*>(w + b.off_dn);
  const size_t sm = cbwd_smem(s.d, s.m), ssm = state_smem(s.d), dsm = bwd_dstate_smem(s.d);
  const int per = s.m * (s.d + 1);
  const dim3 walks(b.c_n, s.BH()), sums(b.c_n, b.fwd.n_fb, s.BH()), scan((per + kThreads - 1) / kThreads, s.BH());
  return dispatch(bf16, fm, [&](auto tag, auto f) {
    using T = decltype(tag);
    constexpr int FM = decltype(f)::value;
    cudaError_t r = set_smem(cbwd_query_kernel<T, FM>, sm);
    if (r == cudaSuccess) r = set_smem(cbwd_key_kernel<T, FM>, sm);
    if (r == cudaSuccess) r = set_smem(state_partial_kernel<T, FM>, ssm);
    if (r == cudaSuccess) r = set_smem(bwd_dstate_partial_kernel<T, FM>, dsm);
    if (r != cudaSuccess) return r;
    state_partial_kernel<T, FM><<<sums, kThreads, ssm, stream>>>(static_cast<const T*>(K), static_cast<const T*>(V),
                                                                 omega, key_ref, s.L, s.d, s.m, scale, b.c_chunk,
                                                                 b.c_n, cst);
    chunk_scan_kernel<<<scan, kThreads, 0, stream>>>(cst, per, b.c_n, false);
    cbwd_query_kernel<T, FM><<<walks, kThreads, sm, stream>>>(
        static_cast<const T*>(Q), static_cast<const T*>(K), static_cast<const T*>(V), static_cast<const T*>(dO),
        static_cast<T*>(dQ), omega, key_ref, cst, dnw, s.L, s.d, s.m, scale, b.c_chunk, b.c_n, st);
    bwd_dstate_partial_kernel<T, FM><<<sums, kThreads, dsm, stream>>>(
        static_cast<const T*>(Q), dnw, omega, key_ref, s.L, s.d, s.m, scale, b.c_chunk, b.c_n, cst);
    chunk_scan_kernel<<<scan, kThreads, 0, stream>>>(cst, per, b.c_n, true);
    cbwd_key_kernel<T, FM><<<walks, kThreads, sm, stream>>>(
        static_cast<const T*>(Q), static_cast<const T*>(K), static_cast<const T*>(V), static_cast<T*>(dK),
        static_cast<T*>(dV), omega, key_ref, cst, dnw, s.L, s.d, s.m, scale, b.c_chunk, b.c_n);
    return cudaGetLastError();
  });
}

cudaError_t simt_bwd_bidir(const void* Q, const void* K, const void* V, const void* dO, void* dQ, void* dK, void* dV,
                           const float* omega, float scale, const Shape& s, bool bf16, void* ws, int32_t* st,
                           cudaStream_t stream, int fm) {
  const BwdPlan b = bwd_plan(s);
  char* w = static_cast<char*>(ws);
  // S~ = [phi(K)^T V | phi(K)^T 1] (and the key reference in the header)
  cudaError_t e = simt_bidir_state(K, V, omega, scale, s, bf16, ws, st, stream, fm);
  if (e != cudaSuccess) return e;
  const float* key_ref = reinterpret_cast<const float*>(w);
  const float* state = reinterpret_cast<const float*>(w + b.fwd.off_state);
  float* dnw = reinterpret_cast<float*>(w + b.off_dn);
  float* dpart = reinterpret_cast<float*>(w + b.off_dpart);
  float* dstate = reinterpret_cast<float*>(w + b.off_dstate);
  const dim3 tiles((s.L + kBT - 1) / kBT, s.BH());
  const size_t tsm = bwd_tile_smem(s.d, s.m), dsm = bwd_dstate_smem(s.d);
  return dispatch(bf16, fm, [&](auto tag, auto f) {
    using T = decltype(tag);
    constexpr int FM = decltype(f)::value;
    cudaError_t r = set_smem(bwd_query_kernel<T, FM>, tsm);
    if (r == cudaSuccess) r = set_smem(bwd_key_kernel<T, FM>, tsm);
    if (r == cudaSuccess) r = set_smem(bwd_dstate_partial_kernel<T, FM>, dsm);
    if (r != cudaSuccess) return r;
    bwd_query_kernel<T, FM><<<tiles, kThreads, tsm, stream>>>(static_cast<const T*>(Q), static_cast<const T*>(dO),
                                                              static_cast<T*>(dQ), omega, key_ref, state, dnw, s.L,
                                                              s.d, s.m, scale, st);
    bwd_dstate_partial_kernel<T, FM><<<dim3(b.fwd.n_split, b.fwd.n_fb, s.BH()), kThreads, dsm, stream>>>(
        static_cast<const T*>(Q), dnw, omega, key_ref, s.L, s.d, s.m, scale, b.fwd.chunk, b.fwd.n_split, dpart);
    merge_kernel<<<merge_grid(s), kThreads, 0, stream>>>(dpart, s.d, s.m, b.fwd.n_split, dstate);
    bwd_key_kernel<T, FM><<<tiles, kThreads, tsm, stream>>>(static_cast<const T*>(K), static_cast<const T*>(V),
                                                            static_cast<T*>(dK), static_cast<T*>(dV), omega, key_ref,
                                                            dstate, s.L, s.d, s.m, scale);
    return cudaGetLastError();
  });
}

}  // namespace favor
