// Tensor-core (tcgen05) gradients of the bidirectional FAVOR+ pass, d = 64,
// m in {128, 256}, bf16 inputs and gradients.
//
// The forward ("Performer — Rethinking Attention with Performers" (digest),
// §Key equations): S = phi(K)^T V (m x d), z = phi(K)^T 1, N_t = phi(q_t)^T
// S, D_t = phi(q_t) . z, o_t = N_t / D_t.  The chain rule through it, for the
// loss sum_t dO_t . o_t, with delta_t = dO_t . o_t and Psi_t = phi(q_t) / D_t:
//   dphi(q_t) = (S dO_t - delta_t z) / D_t
//   dS = sum_t Psi_t dO_t^T,   dz = -sum_t Psi_t delta_t
//   dphi(k_s) = dS v_s + dz,   dv_s = dS^T phi(k_s)
// and through the feature map x -> phi(x), with g_i = dphi_i phi_i (positive
// random features: dphi_i/dx = phi_i (s w_i - s^2 x)), g_i = dphi_i [w_i.x > 0]
// (Performer-ReLU: s w_i [w_i.x > 0]) or g_i = dphi_i min(phi_i, 1) (1 + elu:
// slope 1 above 0 and e^a = phi below):
//   dx = s (sum_i g_i w_i - [prf] s x sum_i g_i).
// Every product is computed from the kernels' stabilised features: phi(q)
// carries the row's own constant (its largest exponent) and phi(k) the key
// reference R.  A per-row constant c scales phi by e^-c and dphi by e^c, so
// g_i and every gradient are unchanged ("From Performer to Linear
// Attention", §Simple Derivation: the constant cancels).  For a query
// sum_i g_i = phi . dphi = (N_t . dO_t - delta_t D_t) / D_t = 0, so the
// query gradient has no s x sum_i g_i term.
//
// Precision.  The key gradient of the softmax features is a difference of
// nearly equal sums for long keys (sum_i g_i w_i against s k sum_i g_i, and
// dS v_s against -dz), so it magnifies the rounding of what feeds dS and dz.
// Hence: D_t is summed in fp32 on the CUDA cores from the fp32 normaliser z
// of the forward state (not from its bf16 image); dO enters the dS product
// unrounded (the 1 / D_t rides in Psi); delta_t is carried as a bf16 pair
// (hi + lo) in two columns of the same operand; dS is handed to the key
// kernel as a pair of bf16 images (hi + lo) and dz in fp32.
//
// Two kernels after the forward's state stage (prep, state kernel: S, z as a
// bf16 image and z in fp32), each on one CTA per SM taking an even share of
// the (head, tile) list (a share may cross from one head into the next):
//   query kernel
//     P = Q Omega^T                    M = 128 tokens,   N = m,      K = d   fp16
//     N = phi(Q) S                     M = 128 tokens,   N = d,      K = m
//     [dS | dz] += Psi^T [dO | -delta] M = 128 features, N = d + 16, K = 128 tokens
//     T = dO S^T                       M = 128 tokens,   N = m,      K = d
//     dQ = s G Omega                   M = 128 tokens,   N = d,      K = m   fp16
//     each head's [dS | dz] part goes to the slot of the CTA's place among the
//     head's CTAs; a merge kernel adds the slots in order into the dS pair and dz
//   key kernel
//     P = K Omega^T,  dV = phi(K) dS_hi,  T = V (dS_hi + dS_lo)^T,  dK = s G Omega
// G = g rounded to bf16, then scaled per row by a power of two that puts
// its largest entry in [2^14, 2^15), in fp16 (the operand type of the fp16
// Omega image); the scale comes off exactly in the epilogue.
//
// Warp roles as in the forward kernels: warp 0 TMA, warp 1 MMA issue (one
// thread), warps 2-3 rewrite each Q or K tile as fp16 (and take the squared
// row norms), warps 4-11 two epilogue warpgroups (thread = one TMEM lane =
// one token; at m = 256 warpgroup w owns feature block w, at m = 128 the
// warpgroups split the block's columns).  One tile is in flight between the
// MMA steps and the epilogue steps; TMA loads run ahead.  Every wait is
// bounded; a wait that runs out raises the CTA's abort flag and records
// FAVOR_ERR_TIMEOUT.
#include <cuda_fp16.h>

#include <algorithm>

#include "tc.cuh"
#include "tc_util.cuh"

namespace favor {
namespace {

using namespace tc;

constexpr int kD = 64;
constexpr int kGN = kD + 16;                // rows of the forward state image; columns of [dS | dz]
constexpr int kTileBytes = kD * kBM * 2;    // one 128-token tile of Q, K, V, dO (one swizzle atom)
constexpr int kBwdThreads = 384;
// tensor-memory columns: P and then T at [0, m); the query kernel's N and
// then dQ at kNQCol, its [dS | dz] blocks at kDSCol + kGN b; the key
// kernel's dV at kDVCol and dK at kDKCol
constexpr uint32_t kNQCol = 256, kDSCol = 352, kDVCol = 256, kDKCol = 320;

struct GradParams {
  const float* key_ref;       // row-norm maxima of Omega (key_reference)
  const float* omega;         // fp32 Omega [m][d] (Performer-ReLU slope guard)
  const uint8_t* omega_img;   // fp16 Omega image [m rows][128 B]
  const uint8_t* state_img;   // query kernel: S (bf16 [m/64][d+16][128 B] per head)
  const float* zvec;          // query kernel: z; key kernel: dz (fp32 [m] per head)
  const uint8_t* ds_hi;       // key kernel: dS pair (bf16 [m/64][d][128 B] per head)
  const uint8_t* ds_lo;
  float* partS;               // query kernel: [dS | dz] partials [BH][m/128][parts][d+1][128], slot = the
                              // CTA's place among the head's CTAs
  int32_t* status;
  int L, m;
  int n_heads;                // B H: the CTAs split the (head, tile) list evenly
  int parts;                  // query kernel: partial slots per head
  float scale;
};


// power of two that brings a row's largest |g| into [2^14, 2^15) (1 for an
// all-zero row), and its inverse; both normal floats for every finite max
__device__ __forceinline__ void row_scale(float gmax, float* beta, float* inv_beta) {
  const int e = static_cast<int>((__float_as_uint(gmax) >> 23) & 0xFFu);
  int be = 268 - e;                           // 2^(14 - (e - 127)) as a biased exponent
  be = gmax > 0.f ? min(max(be, 1), 253) : 127;
  *beta = __uint_as_float(static_cast<uint32_t>(be) << 23);
  *inv_beta = __uint_as_float(static_cast<uint32_t>(254 - be) << 23);
}

// In place: x[j] = bf16x2(g_2j, g_2j+1) for j < 16 (g as fp32 bits)
__device__ __forceinline__ void pack_g_bf16(uint32_t (&x)[32]) {
#pragma unroll
  for (int j = 0; j < 16; ++j) x[j] = pack_bf16(__uint_as_float(x[2 * j]), __uint_as_float(x[2 * j + 1]));
}
// In place: bf16 pairs -> fp16 pairs times beta (16 words)
__device__ __forceinline__ void rescale_f16(uint32_t (&w)[16], float beta) {
#pragma unroll
  for (int j = 0; j < 16; ++j) w[j] = pack_f16_sat(__uint_as_float(w[j] << 16) * beta, __uint_as_float(w[j] & 0xFFFF0000u) * beta);
}

// Four 16-byte chunks (32 bf16 values) of row t of a swizzle atom, from
// logical chunk ch0
__device__ __forceinline__ void load_row32(const uint8_t* atom, int ch0, int t, uint32_t (&w)[16]) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint4 u = *reinterpret_cast<const uint4*>(atom + t * 128 + (((ch0 + c) ^ (t & 7)) << 4));
    w[4 * c] = u.x;
    w[4 * c + 1] = u.y;
    w[4 * c + 2] = u.z;
    w[4 * c + 3] = u.w;
  }
}
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Performer-ReLU slope guard.  The projection runs with Omega rounded to fp16,
// which moves w_i.x by at most 2^-11 sum_k |x_k w_ik| <= 2^-11 |x| max|w|;
// the slope [w_i.x > 0] is a step, so a feature whose fp16 projection lies
// within tau (twice that bound) of 0 takes its sign from w_i.x recomputed in
// fp32 from the fp32 Omega and the row (exact in the fp16 tile), and where
// that sum is itself within its rounding bound (2 d 2^-24 sum_k |x_k w_ik|)
// of 0, in fp64 (every product of a bf16 x and an fp32 w is exact there).
// x holds the raw projections of features f0 .. f0 + 31 of row t; such a
// feature becomes 0 or a positive value below tau / 256 (its true size is
// below tau either way).
__device__ __forceinline__ void relu_guard(uint32_t (&x)[32], int f0, float tau, const uint8_t* tile, int t,
                                           const float* __restrict__ omega) {
  uint32_t flag = 0;
#pragma unroll
  for (int j = 0; j < 32; ++j) flag |= (fabsf(__uint_as_float(x[j])) <= tau ? 1u : 0u) << j;
  uint32_t pos = 0, todo = flag;
  while (todo != 0u) {
    const int j = __ffs(todo) - 1;
    todo &= todo - 1u;
    const float4* w = reinterpret_cast<const float4*>(omega + (size_t)(f0 + j) * kD);
    float acc = 0.f, mag = 0.f;
#pragma unroll 2
    for (int c = 0; c < kD / 8; ++c) {
      const uint4 u = *reinterpret_cast<const uint4*>(tile + t * 128 + ((c ^ (t & 7)) << 4));
      const float4 a = __ldg(w + 2 * c), b = __ldg(w + 2 * c + 1);
      const uint32_t h[4] = {u.x, u.y, u.z, u.w};
      const float wv[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float x0 = __half2float(__ushort_as_half(static_cast<unsigned short>(h[k] & 0xFFFFu)));
        const float x1 = __half2float(__ushort_as_half(static_cast<unsigned short>(h[k] >> 16)));
        acc = fmaf(x0, wv[2 * k], acc);
        acc = fmaf(x1, wv[2 * k + 1], acc);
        mag = fmaf(fabsf(x0), fabsf(wv[2 * k]), mag);
        mag = fmaf(fabsf(x1), fabsf(wv[2 * k + 1]), mag);
      }
    }
    bool positive = acc > 0.f;
    if (fabsf(acc) <= mag * (2.0f * kD * 0x1p-24f)) {
      double acc64 = 0.0;
      for (int c = 0; c < kD / 8; ++c) {
        const uint4 u = *reinterpret_cast<const uint4*>(tile + t * 128 + ((c ^ (t & 7)) << 4));
        const float4 a = __ldg(w + 2 * c), b = __ldg(w + 2 * c + 1);
        const uint32_t h[4] = {u.x, u.y, u.z, u.w};
        const float wv[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          acc64 = fma((double)__half2float(__ushort_as_half(static_cast<unsigned short>(h[k] & 0xFFFFu))),
                      (double)wv[2 * k], acc64);
          acc64 = fma((double)__half2float(__ushort_as_half(static_cast<unsigned short>(h[k] >> 16))),
                      (double)wv[2 * k + 1], acc64);
        }
      }
      positive = acc64 > 0.0;
    }
    if (positive) pos |= 1u << j;
  }
#pragma unroll
  for (int j = 0; j < 32; ++j)
    if ((flag >> j) & 1u) x[j] = ((pos >> j) & 1u) ? __float_as_uint(fmaxf(__uint_as_float(x[j]), tau * 0x1p-8f)) : 0u;
}
// tau of the guard for a row of squared norm x2 (the second term covers the
// fp16 rounding of row entries below the fp16 normal range)
__device__ __forceinline__ float relu_tau(float x2, float wmax) { return wmax * (sqrtf(x2) * 0x1p-10f + 0x1p-21f); }

// Adds one head's first `count` fp32 [dS | dz] partials ([M/128][parts][D+1][128],
// feature fastest) in slot order: dS as a bf16 pair hi + lo (hi = bf16(x),
// lo = bf16(x - hi); images [M/64 atoms][D rows][128 B], 128-byte swizzle)
// and dz in fp32.  Items [e_begin, e_end) of the NFB (D + 1) 32 items =
// (block, row n, 4 features), by all `nthreads` threads.
template <int D, int M>
__device__ void merge_grad_state(const float* __restrict__ base, int parts, int count, uint8_t* __restrict__ hi,
                                 uint8_t* __restrict__ lo, float* __restrict__ dz, int e_begin, int e_end,
                                 int nthreads) {
  constexpr int NG = kFB / 4;
  constexpr int kBatch = 4;
  for (int e0 = e_begin + threadIdx.x; e0 < e_end; e0 += kBatch * nthreads) {
    float4 acc[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
    // the loads of up to kPartBatch slots in flight together, added in slot order
    constexpr int kPartBatch = 4;
    for (int p0 = 0; p0 < count; p0 += kPartBatch) {
      float4 v[kPartBatch][kBatch];
#pragma unroll
      for (int pp = 0; pp < kPartBatch; ++pp)
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          const int e = e0 + u * nthreads;
          const int g = e % NG, n = (e / NG) % (D + 1), b = e / (NG * (D + 1));
          const int p = p0 + pp;
          v[pp][u] = (e < e_end && p < count)
                         ? *reinterpret_cast<const float4*>(base + (((size_t)b * parts + p) * (D + 1) + n) * kFB + g * 4)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
      for (int pp = 0; pp < kPartBatch; ++pp) {
        if (p0 + pp >= count) break;
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          acc[u].x += v[pp][u].x;
          acc[u].y += v[pp][u].y;
          acc[u].z += v[pp][u].z;
          acc[u].w += v[pp][u].w;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int e = e0 + u * nthreads;
      if (e >= e_end) break;
      const int g = e % NG, n = (e / NG) % (D + 1), b = e / (NG * (D + 1));
      const int f = b * kFB + g * 4;
      if (n == D) {
        *reinterpret_cast<float4*>(dz + f) = acc[u];
        continue;
      }
      const float a[4] = {acc[u].x, acc[u].y, acc[u].z, acc[u].w};
      float h[4], l[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        h[k] = __bfloat162float(__float2bfloat16_rn(a[k]));
        l[k] = a[k] - h[k];
      }
      const int atom = f >> 6, cc = f & 63;
      const size_t off = ((size_t)atom * D + n) * 128 + (((cc >> 3) ^ (n & 7)) << 4) + (cc & 7) * 2;
      *reinterpret_cast<uint2*>(hi + off) = make_uint2(pack_bf16(h[0], h[1]), pack_bf16(h[2], h[3]));
      *reinterpret_cast<uint2*>(lo + off) = make_uint2(pack_bf16(l[0], l[1]), pack_bf16(l[2], l[3]));
    }
  }
}

// ---------------------------------------------------------------------------
// query kernel
// ---------------------------------------------------------------------------
struct GqCfg {
  static constexpr int NSQ = 2;
  static constexpr int kOmega = 0;                       // fp16 Omega image, up to 256 rows
  static constexpr int kState = kOmega + 256 * kD * 2;   // bf16 [S | z] image, up to 256 x kGN
  static constexpr int kZ = kState + 256 * kGN * 2;      // fp32 z [256]
  static constexpr int kQ = kZ + 1024;                   // [NSQ] Q tiles (fp16 after the rewrite)
  static constexpr int kDO = kQ + NSQ * kTileBytes;      // dO tile: columns 0-63 of [dO | -delta]
  static constexpr int kDl = kDO + kTileBytes;           // columns 64-127: -delta as (hi, lo); also stages dQ
  static constexpr int kPhi = kDl + kTileBytes;          // [m/128][2 atoms]: phi(Q), Psi, then G (fp16)
  static constexpr int kX = kPhi + 4 * kAtom;            // row exchange [4][2][128] floats
  static constexpr int kNorm = kX + 4 * 2 * kBM * 4;     // [NSQ][128] squared query norms
  static constexpr int kBars = kNorm + NSQ * kBM * 4;
  static constexpr int kSmem = kBars + 512 + 1024;
};
static_assert(GqCfg::kSmem <= 232448, "shared memory");
static_assert(GqCfg::kQ % 1024 == 0 && GqCfg::kPhi % 1024 == 0, "operand alignment");

template <int M, int FM>
__global__ void __launch_bounds__(kBwdThreads, 1) grad_query_kernel(const __grid_constant__ CUtensorMap mapQ,
                                                                    const __grid_constant__ CUtensorMap mapDO,
                                                                    const __grid_constant__ CUtensorMap mapDQ,
                                                                    GradParams prm) {
  using C = GqCfg;
  constexpr int NFB = M / kFB;
  constexpr int NSQ = C::NSQ;
  constexpr bool kGuard = FM == FAVOR_FM_RELU;   // the epilogue reads Q after the projection
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::kBars);
  uint64_t* q_full = bars;                // [NSQ] Q landed
  uint64_t* q_empty = q_full + NSQ;       // [NSQ] the projection (ReLU: the slope guard) has read it
  uint64_t* qn_full = q_empty + NSQ;      // [NSQ] Q rewritten as fp16, norms written
  uint64_t* d_full = qn_full + NSQ;       // dO landed
  uint64_t* d_empty = d_full + 1;         // the tile's dS and T products have read dO
  uint64_t* p_full = d_empty + 1;         // projection complete
  uint64_t* p_free = p_full + 1;          // projection copied out
  uint64_t* phi_full = p_free + 1;        // phi(Q) written
  uint64_t* n_full = phi_full + 1;        // N complete
  uint64_t* n_free = n_full + 1;          // N copied out
  uint64_t* dn_full = n_free + 1;         // -delta written, phi(Q) rescaled to Psi
  uint64_t* t_full = dn_full + 1;         // dS step and T complete
  uint64_t* t_free = t_full + 1;          // T copied out
  uint64_t* g_full = t_free + 1;          // G written
  uint64_t* dq_full = g_full + 1;         // dQ complete
  uint64_t* dq_free = dq_full + 1;        // dQ copied out
  uint64_t* setup_bar = dq_free + 1;
  uint64_t* done_bar = setup_bar + 1;
  uint64_t* img_full = done_bar + 1;      // phase k: the k-th head's S image and z landed
  uint64_t* img_free = img_full + 1;      // phase k: the k-th head's last tile no longer reads them
  uint64_t* ds_free = img_free + 1;       // phase k: the k-th head's [dS | dz] copied out of tensor memory
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ds_free + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* xch = reinterpret_cast<float*>(sm + C::kX);
  float* norm_s = reinterpret_cast<float*>(sm + C::kNorm);
  const float* z_s = reinterpret_cast<const float*>(sm + C::kZ);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // this CTA's tiles: the contiguous range [g0, g1) of the (head, tile) list,
  // which may cross from one head into the next; each head's [dS | dz] part
  // goes to the slot of this CTA's place among the head's CTAs
  const int nt = (prm.L + kBM - 1) / kBM;
  const long long total = (long long)prm.n_heads * nt;
  const int g0 = range_first(total, blockIdx.x, gridDim.x);
  const int g1 = range_first(total, blockIdx.x + 1, gridDim.x);
  const int n_tiles = g1 - g0;
  const int h0 = g0 / nt;
  const int n_heads = n_tiles > 0 ? (g1 - 1) / nt - h0 + 1 : 0;
  auto head_of = [&](int i) { return (g0 + i) / nt; };
  auto tile_of = [&](int i) { return (g0 + i) - head_of(i) * nt; };
  auto head_starts = [&](int i) { return i == 0 || head_of(i) != head_of(i - 1); };
  auto head_ends = [&](int i) { return i == n_tiles - 1 || head_of(i + 1) != head_of(i); };
  const WaitCtx wctx{abort_flag, prm.status};

  if (threadIdx.x == 0) {
    for (int i = 0; i < NSQ; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], kGuard ? kEpiWarps : 1);
      mbar_init(&qn_full[i], kNormWarps);
    }
    mbar_init(d_full, 1);
    mbar_init(d_empty, 1);
    mbar_init(p_full, 1);
    mbar_init(p_free, kEpiWarps);
    mbar_init(phi_full, kEpiWarps);
    mbar_init(n_full, 1);
    mbar_init(n_free, kEpiWarps);
    mbar_init(dn_full, kEpiWarps);
    mbar_init(t_full, 1);
    mbar_init(t_free, kEpiWarps);
    mbar_init(g_full, kEpiWarps);
    mbar_init(dq_full, 1);
    mbar_init(dq_free, kEpiWarps);
    mbar_init(setup_bar, 1);
    mbar_init(done_bar, 1);
    mbar_init(img_full, 1);
    mbar_init(img_free, kEpiWarps);
    mbar_init(ds_free, kEpiWarps);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      prefetch_tmap(&mapQ);
      prefetch_tmap(&mapDO);
      prefetch_tmap(&mapDQ);
      const uint32_t ob = M * kD * 2, sb = M * kGN * 2, zb = M * 4;
      mbar_arrive_expect_tx(setup_bar, ob);
      bulk_load(sm + C::kOmega, prm.omega_img, ob, setup_bar);
      // head k's S image and z go in once head k - 1's last tile is done with them
      auto load_head = [&](int k) {
        const size_t hh = (size_t)(h0 + k);
        mbar_arrive_expect_tx(img_full, sb + zb);
        bulk_load(sm + C::kState, prm.state_img + hh * sb, sb, img_full);
        bulk_load(sm + C::kZ, prm.zvec + hh * M, zb, img_full);
      };
      int ni = 0;
      if (n_heads > 0) load_head(ni++);
      // Q tile x goes to slot x % NSQ once tile x - NSQ's reader is done;
      // dO tile x once tile x - 1's products have read the dO slot
      Watchdog wd(wctx);
      int nq = 0, nd = 0;
      bool ok = true;
      while (ok && (nq < n_tiles || nd < n_tiles || ni < n_heads)) {
        bool progress = false;
        if (nq < n_tiles && (nq < NSQ || mbar_test_wait(smem_addr(&q_empty[nq % NSQ]), ((nq / NSQ) - 1) & 1))) {
          const int st = nq % NSQ;
          mbar_arrive_expect_tx(&q_full[st], kTileBytes);
          tma_load_3d(sm + C::kQ + st * kTileBytes, &mapQ, 0, tile_of(nq) * kBM, head_of(nq), &q_full[st]);
          ++nq;
          progress = true;
        }
        if (nd < nq && (nd == 0 || mbar_test_wait(smem_addr(d_empty), (nd - 1) & 1))) {
          mbar_arrive_expect_tx(d_full, kTileBytes);
          tma_load_3d(sm + C::kDO, &mapDO, 0, tile_of(nd) * kBM, head_of(nd), d_full);
          ++nd;
          progress = true;
        }
        if (ni < n_heads && mbar_test_wait(smem_addr(img_free), (ni - 1) & 1)) {
          load_head(ni++);
          progress = true;
        }
        if (progress) wd.progress();
        else ok = wd.idle();
      }
      for (int x = max(0, nq - NSQ); x < nq; ++x) mbar_wait(&q_full[x % NSQ], (x / NSQ) & 1, wctx);
      if (nd > 0) mbar_wait(d_full, (nd - 1) & 1, wctx);
      if (ni > 0) mbar_wait(img_full, (ni - 1) & 1, wctx);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t id_proj = idesc_f16(kBM, M, false, false);
      constexpr uint32_t id_n = idesc_bf16(kBM, kD, false, false);
      constexpr uint32_t id_ds = idesc_bf16(kFB, kGN, true, true);
      constexpr uint32_t id_t = idesc_bf16(kBM, M, false, true);
      constexpr uint32_t id_dq = idesc_f16(kBM, kD, false, true);
      const uint32_t omega_a = smem_addr(sm + C::kOmega);
      const uint32_t state_a = smem_addr(sm + C::kState);
      const uint32_t phi_a = smem_addr(sm + C::kPhi);
      const uint32_t do_a = smem_addr(sm + C::kDO);
      bool ok = mbar_wait(setup_bar, 0, wctx);
      // event-driven issue of the four MMA steps of each tile, each as soon
      // as its operands and its tensor-memory columns are ready
      Watchdog wd(wctx);
      int ia = 0, ib = 0, ic = 0, id = 0;
      while (ok && id < n_tiles) {
        bool progress = false;
        if (ia < n_tiles) {
          // P = Q Omega^T into [0, M) once the previous tile's T is out
          const int st = ia % NSQ;
          if (mbar_test_wait(smem_addr(&qn_full[st]), (ia / NSQ) & 1) &&
              (ia == 0 || mbar_test_wait(smem_addr(t_free), (ia - 1) & 1))) {
            tc_fence_after();
            const uint64_t a0 = sdesc(smem_addr(sm + C::kQ + st * kTileBytes), 16, 1024);
            const uint64_t b0 = sdesc(omega_a, 16, 1024);
#pragma unroll
            for (int k = 0; k < kD / 16; ++k)
              mma_bf16(tmem, dadd(a0, kstep_k(k, kAtom)), dadd(b0, kstep_k(k, M * 128)), id_proj, k > 0);
            mma_commit(p_full);
            if (!kGuard) mma_commit(&q_empty[st]);
            ++ia;
            progress = true;
          }
        }
        if (ib < ia && mbar_test_wait(smem_addr(phi_full), ib & 1) &&
            mbar_test_wait(smem_addr(img_full), (head_of(ib) - h0) & 1) &&
            (ib == 0 || mbar_test_wait(smem_addr(dq_free), (ib - 1) & 1))) {
          // N = phi(Q) S (the first d rows of the image)
          tc_fence_after();
          const uint64_t a0 = sdesc(phi_a, 16, 1024);
          const uint64_t b0 = sdesc(state_a, 16, 1024);
#pragma unroll
          for (int fb = 0; fb < NFB; ++fb)
#pragma unroll
            for (int kk = 0; kk < kFB / 16; ++kk)
              mma_bf16(tmem + kNQCol, dadd(a0, fb * 2 * kAtom + kstep_k(kk, kAtom)),
                       dadd(b0, fb * 2 * kGN * 128 + kstep_k(kk, kGN * 128)), id_n, (fb > 0) || (kk > 0));
          mma_commit(n_full);
          ++ib;
          progress = true;
        }
        // a head's first tile restarts the [dS | dz] accumulators once the
        // previous head's were copied out
        const bool fresh = ic < ib && head_starts(ic);
        if (ic < ib && mbar_test_wait(smem_addr(dn_full), ic & 1) && mbar_test_wait(smem_addr(p_free), ic & 1) &&
            (!fresh || ic == 0 || mbar_test_wait(smem_addr(ds_free), (head_of(ic) - h0 - 1) & 1))) {
          tc_fence_after();
          // [dS | dz]_b += Psi_b^T [dO | -delta] (both token-major: MN-major;
          // the -delta columns sit one tile after the dO tile)
          const uint64_t bd = sdesc(do_a, kTileBytes, 1024);
#pragma unroll
          for (int fb = 0; fb < NFB; ++fb) {
            const uint64_t a0 = sdesc(phi_a + fb * 2 * kAtom, kAtom, 1024);
#pragma unroll
            for (int k = 0; k < kBM / 16; ++k)
              mma_bf16(tmem + kDSCol + fb * kGN, dadd(a0, kstep_mn(k)), dadd(bd, kstep_mn(k)), id_ds,
                       !fresh || (k > 0));
          }
          // T = dO S^T into [0, M): the image's first d rows are the K dimension
          const uint64_t a1 = sdesc(do_a, 16, 1024);
          const uint64_t b1 = sdesc(state_a, kGN * 128, 1024);
#pragma unroll
          for (int k = 0; k < kD / 16; ++k)
            mma_bf16(tmem, dadd(a1, kstep_k(k, kAtom)), dadd(b1, kstep_mn(k)), id_t, k > 0);
          mma_commit(t_full);
          mma_commit(d_empty);
          ++ic;
          progress = true;
        }
        if (id < ic && mbar_test_wait(smem_addr(g_full), id & 1) && mbar_test_wait(smem_addr(n_free), id & 1)) {
          // dQ (scaled) = G Omega: the Omega image's rows are the K dimension
          tc_fence_after();
          const uint64_t a0 = sdesc(phi_a, 16, 1024);
          const uint64_t b0 = sdesc(omega_a, M * 128, 1024);
#pragma unroll
          for (int fb = 0; fb < NFB; ++fb)
#pragma unroll
            for (int kk = 0; kk < kFB / 16; ++kk)
              mma_bf16(tmem + kNQCol, dadd(a0, fb * 2 * kAtom + kstep_k(kk, kAtom)), dadd(b0, kstep_mn(fb * 8 + kk)),
                       id_dq, (fb > 0) || (kk > 0));
          mma_commit(dq_full);
          ++id;
          progress = true;
        }
        if (progress) wd.progress();
        else ok = wd.idle();
      }
      mma_commit(done_bar);
      mbar_wait(done_bar, 0, wctx);
    }
  } else if (warp < 2 + kNormWarps) {
    // Q rewritten as fp16 for the projection; squared norms for the guard
    for (int i = 0; i < n_tiles; ++i) {
      const int st = i % NSQ;
      if (!mbar_wait(&q_full[st], (i / NSQ) & 1, wctx)) break;
      uint8_t* qt = sm + C::kQ + st * kTileBytes;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int r = (warp - 2) * 64 + lane + 32 * j;
        norm_s[st * kBM + r] = tile_row_sq_to_f16<kD>(qt, r);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&qn_full[st]);
    }
  } else {
    const int wg = (warp - 4) >> 2;
    const int q = warp & 3;
    const int t = q * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    const int my_fb = (NFB == 2) ? wg : 0;
    constexpr int kChunks = (NFB == 2) ? 4 : 2;    // 32-column chunks of this thread's columns
    const int c0 = (NFB == 2) ? 0 : wg * 64;       // this thread's first column of block my_fb
    const int f_base = my_fb * kFB + c0;           // its first feature
    const float c1 = feature_c1<FM>(prm.scale);
    uint8_t* phi_blk = sm + C::kPhi + my_fb * 2 * kAtom;
    const uint32_t phi_blk_a = smem_addr(phi_blk);
    const uint32_t dl_a = smem_addr(sm + C::kDl);
    const uint8_t* dot = sm + C::kDO;
    float* xa = xch;                  // [2][128] row maxima of the projections
    float* xb = xch + 2 * kBM;        // [2][128] partial dO . N
    float* xc = xch + 4 * kBM;        // [2][128] partial max |g|
    float* xd = xch + 6 * kBM;        // [2][128] partial D
    float R_unused, W;
    key_reference(prm.key_ref, prm.m, &R_unused, &W);
    bool ok = true;
    for (int i = 0; i < n_tiles; ++i) {
      const int hi_t = head_of(i), ti = tile_of(i);
      const bool valid = ti * kBM + t < prm.L;
      if (ok) ok = mbar_wait(img_full, (hi_t - h0) & 1, wctx);   // this head's z
      const int qs = i % NSQ;
      // ---- phi(Q): the row's reference is its largest exponent; rows past
      // the sequence end get 0.  D = phi(Q) . z summed in fp32 alongside.
      if (ok) ok = mbar_wait(p_full, i & 1, wctx);
      tc_fence_after();
      float bias = valid ? 0.f : INFINITY;
      if constexpr (FM == FAVOR_FM_PRF) {
        float pm = -INFINITY;
#pragma unroll 1
        for (int ch = 0; ch < kChunks; ++ch) {
          uint32_t x[32];
          if (ok) {
            tmem_ld32(tmem + lane_off + f_base + 32 * ch, x);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) pm = fmaxf(pm, __uint_as_float(x[j]));
          }
        }
        xa[wg * kBM + t] = pm;
        named_bar(1, kEpiThreads);
        if (valid) bias = fmaxf(xa[t], xa[kBM + t]) * c1;
      }
      float dpart = 0.f;
#pragma unroll 1
      for (int ch = 0; ch < kChunks; ++ch) {
        uint32_t x[32];
        if (ok) {
          tmem_ld32(tmem + lane_off + f_base + 32 * ch, x);
          tmem_ld_wait();
        }
        if (ch == kChunks - 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(p_free);
        }
        if (ok) {
          if constexpr (kGuard)
            relu_guard(x, f_base + 32 * ch, relu_tau(norm_s[qs * kBM + t], W), sm + C::kQ + qs * kTileBytes, t,
                       prm.omega);
          feature_pack<FM>(x, c1, bias);
          const float4* zc = reinterpret_cast<const float4*>(z_s + f_base + 32 * ch);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float4 zz = zc[j];
            dpart = fmaf(bf_lo(x[2 * j]), zz.x, dpart);
            dpart = fmaf(bf_hi(x[2 * j]), zz.y, dpart);
            dpart = fmaf(bf_lo(x[2 * j + 1]), zz.z, dpart);
            dpart = fmaf(bf_hi(x[2 * j + 1]), zz.w, dpart);
          }
          store_row<16>(phi_blk_a, kAtom, t, c0 + 32 * ch, x);
        }
      }
      xd[wg * kBM + t] = dpart;
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(phi_full);
        if (kGuard) mbar_arrive(&q_empty[qs]);
      }

      // ---- delta = dO . N / D; the -delta columns; phi(Q) -> Psi = phi(Q) / D
      if (ok) ok = mbar_wait(n_full, i & 1, wctx);
      if (ok) ok = mbar_wait(d_full, i & 1, wctx);
      tc_fence_after();
      float part = 0.f;
#pragma unroll 1
      for (int hf = 0; hf < 2; ++hf) {
        // 16 of this thread's 32 columns of N and of dO
        uint32_t nv[16];
        if (ok) {
          tmem_ld16(tmem + lane_off + kNQCol + wg * 32 + 16 * hf, nv);
          tmem_ld_wait();
        }
        if (hf == 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(n_free);
        }
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int chunk = wg * 4 + 2 * hf + c;
          const uint4 u = *reinterpret_cast<const uint4*>(dot + t * 128 + ((chunk ^ (t & 7)) << 4));
          const uint32_t dw[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            part = fmaf(bf_lo(dw[j]), __uint_as_float(nv[8 * c + 2 * j]), part);
            part = fmaf(bf_hi(dw[j]), __uint_as_float(nv[8 * c + 2 * j + 1]), part);
          }
        }
      }
      xb[wg * kBM + t] = part;
      // the previous tile's dQ store has read its staging (the -delta tile)
      if (threadIdx.x == kEpiTid0 && i > 0) bulk_wait_read0();
      named_bar(1, kEpiThreads);
      const float den = xd[t] + xd[kBM + t];      // halves added in a fixed order
      if (ok && valid && (!(den > 0.f) || !isfinite(den))) report_status(prm.status, FAVOR_ERR_NONFINITE);
      const float inv = valid ? 1.0f / den : 0.f;
      const float delta = (xb[t] + xb[kBM + t]) * inv;
      if (wg == 1) {
        // columns 64-71 of row t: (-delta hi, -delta lo, 0, ...), 72-79: 0
        const float dh = __bfloat162float(__float2bfloat16_rn(delta));
        st_shared_v4(dl_a + t * 128 + ((t & 7) << 4), pack_bf16(-dh, -(delta - dh)), 0u, 0u, 0u);
        st_shared_v4(dl_a + t * 128 + ((1 ^ (t & 7)) << 4), 0u, 0u, 0u, 0u);
      }
#pragma unroll 1
      for (int ch = 0; ch < kChunks; ++ch) {
        const int col = c0 + 32 * ch;
        uint32_t w[16];
        load_row32(phi_blk + (col >> 6) * kAtom, (col & 63) >> 3, t, w);
#pragma unroll
        for (int j = 0; j < 16; ++j) w[j] = pack_bf16(bf_lo(w[j]) * inv, bf_hi(w[j]) * inv);
        store_row<16>(phi_blk_a, kAtom, t, col, w);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(dn_full);

      // ---- g = dphi * slope: dphi = (T - delta z) / D, phi = Psi D; G
      // (scaled per row, fp16) over Psi
      if (ok) ok = mbar_wait(t_full, i & 1, wctx);
      tc_fence_after();
      auto chunk_g = [&](int ch, uint32_t (&x)[32]) {
        const int col = c0 + 32 * ch;
        tmem_ld32(tmem + lane_off + f_base + 32 * ch, x);
        uint32_t w[16];
        load_row32(phi_blk + (col >> 6) * kAtom, (col & 63) >> 3, t, w);
        tmem_ld_wait();
        const float4* zc = reinterpret_cast<const float4*>(z_s + f_base + 32 * ch);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float4 zz = zc[j];
          const float zv[4] = {zz.x, zz.y, zz.z, zz.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int o = 4 * j + k;
            const float psi = (k & 1) ? bf_hi(w[o >> 1]) : bf_lo(w[o >> 1]);
            const float e = fmaf(-delta, zv[k], __uint_as_float(x[o]));   // dphi D
            float gv;
            if constexpr (FM == FAVOR_FM_PRF) gv = e * psi;
            else if constexpr (FM == FAVOR_FM_ELU1) gv = e * inv * fminf(psi * den, 1.f);
            else gv = psi > 0.f ? e * inv : 0.f;
            x[o] = __float_as_uint(gv);
          }
        }
      };
      // g (bf16) over Psi, then rescaled by the row's power of two to fp16
      float gmax = 0.f;
#pragma unroll 1
      for (int ch = 0; ch < kChunks; ++ch) {
        uint32_t g[32];
        if (ok) chunk_g(ch, g);
        if (ch == kChunks - 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(t_free);
        }
        if (ok) {
#pragma unroll
          for (int j = 0; j < 32; ++j) gmax = fmaxf(gmax, fabsf(__uint_as_float(g[j])));
          pack_g_bf16(g);
          store_row<16>(phi_blk_a, kAtom, t, c0 + 32 * ch, g);
        }
      }
      if (head_ends(i)) {
        // the head's S image and z: read by this tile's products (complete)
        // and by the pass above, for the last time
        __syncwarp();
        if (lane == 0) mbar_arrive(img_free);
      }
      xc[wg * kBM + t] = gmax;
      named_bar(1, kEpiThreads);
      float beta, inv_beta;
      row_scale(fmaxf(xc[t], xc[kBM + t]), &beta, &inv_beta);
#pragma unroll 1
      for (int ch = 0; ch < kChunks; ++ch) {
        const int col = c0 + 32 * ch;
        uint32_t w[16];
        load_row32(phi_blk + (col >> 6) * kAtom, (col & 63) >> 3, t, w);
        rescale_f16(w, beta);
        store_row<16>(phi_blk_a, kAtom, t, col, w);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(g_full);

      if (head_ends(i)) {
        // the head's [dS | dz] part (complete with this tile's products) to
        // its slot: lane f = feature f of a block; dz is the sum of the two
        // -delta columns.  Two blocks: warpgroup w reads block w; one block:
        // the warpgroups split the d columns.
        const int slot = (int)blockIdx.x - range_cta(total, (long long)hi_t * nt, gridDim.x);
        const int sfb = (NFB == 2) ? wg : 0;
        float* dst = prm.partS + ((((size_t)hi_t * NFB + sfb) * prm.parts + slot) * (kD + 1)) * kFB;
        const uint32_t s_col = tmem + lane_off + kDSCol + sfb * kGN;
#pragma unroll 1
        for (int cb = 0; cb < kD / 16; ++cb) {
          if (NFB == 1 && (cb >> 1) != wg) continue;
          uint32_t v[16];
          if (ok) {
            tmem_ld16(s_col + cb * 16, v);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j) dst[(size_t)(cb * 16 + j) * kFB + t] = __uint_as_float(v[j]);
          }
        }
        if (NFB == 2 || wg == 1) {
          uint32_t z[8];
          if (ok) {
            tmem_ld8(s_col + kD, z);
            tmem_ld_wait();
            dst[(size_t)kD * kFB + t] = __uint_as_float(z[0]) + __uint_as_float(z[1]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(ds_free);
      }

      // ---- dQ = s (G Omega) / beta, staged in the -delta tile (read by this
      // tile's dS product, complete once dQ is)
      if (ok) ok = mbar_wait(dq_full, i & 1, wctx);
      tc_fence_after();
      const float f = prm.scale * inv_beta;
#pragma unroll 1
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t v[16];
        if (ok) {
          tmem_ld16(tmem + lane_off + kNQCol + wg * 32 + 16 * hf, v);
          tmem_ld_wait();
        }
        if (hf == 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(dq_free);
        }
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int chunk = wg * 4 + 2 * hf + c;
          const int o = 8 * c;
          st_shared_v4(dl_a + t * 128 + ((chunk ^ (t & 7)) << 4),
                       pack_bf16(__uint_as_float(v[o]) * f, __uint_as_float(v[o + 1]) * f),
                       pack_bf16(__uint_as_float(v[o + 2]) * f, __uint_as_float(v[o + 3]) * f),
                       pack_bf16(__uint_as_float(v[o + 4]) * f, __uint_as_float(v[o + 5]) * f),
                       pack_bf16(__uint_as_float(v[o + 6]) * f, __uint_as_float(v[o + 7]) * f));
        }
      }
      fence_proxy_async_smem();
      named_bar(1, kEpiThreads);
      if (threadIdx.x == kEpiTid0 && ok && !*abort_flag) {
        tma_store_3d(&mapDQ, 0, ti * kBM, hi_t, sm + C::kDl);
        bulk_commit();
      }
    }
    if (threadIdx.x == kEpiTid0) bulk_wait0();
    mbar_wait(done_bar, 0, wctx);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// CTA (head, y): a 1 / kMergeSplit share of the head's items, its [dS | dz]
// parts (one per query-kernel CTA that covered the head, in CTA order) added
// into the dS pair and dz
constexpr int kMergeSplit = 8;
template <int M>
__global__ void __launch_bounds__(128) grad_merge_kernel(const float* __restrict__ partS, int parts, int nt,
                                                         int n_heads, int n_ctas, uint8_t* __restrict__ hi,
                                                         uint8_t* __restrict__ lo, float* __restrict__ dz) {
  constexpr int NFB = M / kFB;
  constexpr int kItems = NFB * (kD + 1) * (kFB / 4);
  constexpr int kShare = (kItems + kMergeSplit - 1) / kMergeSplit;
  const int h = blockIdx.x;
  const long long total = (long long)n_heads * nt;
  const int count = range_cta(total, (long long)(h + 1) * nt - 1, n_ctas) - range_cta(total, (long long)h * nt, n_ctas) + 1;
  merge_grad_state<kD, M>(partS + (size_t)h * NFB * parts * (kD + 1) * kFB, parts, count, hi + (size_t)h * M * kD * 2,
                          lo + (size_t)h * M * kD * 2, dz + (size_t)h * M, blockIdx.y * kShare,
                          min(kItems, (int)(blockIdx.y + 1) * kShare), blockDim.x);
}

// ---------------------------------------------------------------------------
// key kernel
// ---------------------------------------------------------------------------
struct GkCfg {
  // a K slot is released once dK has been stored from it (the epilogue reads
  // k there for the s k sum_i g_i term), the V slot once dV has
  static constexpr int NK = 2;
  static constexpr int kOmega = 0;                       // fp16 Omega image, up to 256 rows
  static constexpr int kHi = kOmega + 256 * kD * 2;      // bf16 dS pair, up to 256 x d each
  static constexpr int kLo = kHi + 256 * kD * 2;
  static constexpr int kZ = kLo + 256 * kD * 2;          // fp32 dz [256]
  static constexpr int kK = kZ + 1024;                   // [NK] K tiles (fp16 after the rewrite), then dK
  static constexpr int kV = kK + NK * kTileBytes;        // V tile, then dV
  static constexpr int kPhi = kV + kTileBytes;           // [m/128][2 atoms]: phi(K), then G (fp16)
  static constexpr int kNorm = kPhi + 4 * kAtom;         // [NK][128] squared key norms
  static constexpr int kX = kNorm + NK * kBM * 4;        // row exchange [2][2][128] floats
  static constexpr int kBars = kX + 2 * 2 * kBM * 4;
  static constexpr int kSmem = kBars + 512 + 1024;
};
static_assert(GkCfg::kSmem <= 232448, "shared memory");
static_assert(GkCfg::kK % 1024 == 0 && GkCfg::kPhi % 1024 == 0, "operand alignment");

template <int M, int FM>
__global__ void __launch_bounds__(kBwdThreads, 1) grad_key_kernel(const __grid_constant__ CUtensorMap mapK,
                                                                  const __grid_constant__ CUtensorMap mapV,
                                                                  const __grid_constant__ CUtensorMap mapDK,
                                                                  const __grid_constant__ CUtensorMap mapDV,
                                                                  GradParams prm) {
  using C = GkCfg;
  constexpr int NFB = M / kFB;
  constexpr int NK = C::NK;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::kBars);
  uint64_t* k_full = bars;                // [NK]
  uint64_t* k_empty = k_full + NK;        // [NK] dK stored from the slot
  uint64_t* kn_full = k_empty + NK;       // [NK] K in fp16, norms written
  uint64_t* v_full = kn_full + NK;
  uint64_t* v_empty = v_full + 1;         // dV stored from the slot
  uint64_t* p_full = v_empty + 1;
  uint64_t* p_free = p_full + 1;
  uint64_t* phi_full = p_free + 1;
  uint64_t* t_full = phi_full + 1;        // dV and T complete
  uint64_t* t_free = t_full + 1;          // T copied out
  uint64_t* dv_free = t_free + 1;         // dV copied out
  uint64_t* g_full = dv_free + 1;
  uint64_t* dk_full = g_full + 1;
  uint64_t* dk_free = dk_full + 1;
  uint64_t* setup_bar = dk_free + 1;
  uint64_t* done_bar = setup_bar + 1;
  uint64_t* img_full = done_bar + 1;      // phase k: the k-th head's dS pair and dz landed
  uint64_t* img_free = img_full + 1;      // phase k: the k-th head's last tile no longer reads them
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(img_free + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* norm_s = reinterpret_cast<float*>(sm + C::kNorm);
  float* xch = reinterpret_cast<float*>(sm + C::kX);
  const float* dz_s = reinterpret_cast<const float*>(sm + C::kZ);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // this CTA's tiles: the contiguous range [g0, g1) of the (head, tile) list,
  // which may cross from one head into the next
  const int nt = (prm.L + kBM - 1) / kBM;
  const long long total = (long long)prm.n_heads * nt;
  const int g0 = (int)(total * blockIdx.x / gridDim.x);
  const int g1 = (int)(total * (blockIdx.x + 1) / gridDim.x);
  const int n_tiles = g1 - g0;
  const int h0 = g0 / nt;
  const int n_heads = n_tiles > 0 ? (g1 - 1) / nt - h0 + 1 : 0;
  auto head_of = [&](int i) { return (g0 + i) / nt; };      // the CTA's i-th tile's head
  auto tile_of = [&](int i) { return (g0 + i) - head_of(i) * nt; };
  const WaitCtx wctx{abort_flag, prm.status};

  if (threadIdx.x == 0) {
    for (int i = 0; i < NK; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
      mbar_init(&kn_full[i], kNormWarps);
    }
    mbar_init(v_full, 1);
    mbar_init(v_empty, 1);
    mbar_init(p_full, 1);
    mbar_init(p_free, kEpiWarps);
    mbar_init(phi_full, kEpiWarps);
    mbar_init(t_full, 1);
    mbar_init(t_free, kEpiWarps);
    mbar_init(dv_free, kEpiWarps);
    mbar_init(g_full, kEpiWarps);
    mbar_init(dk_full, 1);
    mbar_init(dk_free, kEpiWarps);
    mbar_init(setup_bar, 1);
    mbar_init(done_bar, 1);
    mbar_init(img_full, 1);
    mbar_init(img_free, kEpiWarps);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      prefetch_tmap(&mapK);
      prefetch_tmap(&mapV);
      prefetch_tmap(&mapDK);
      prefetch_tmap(&mapDV);
      const uint32_t ob = M * kD * 2, hb = M * kD * 2, zb = M * 4;
      mbar_arrive_expect_tx(setup_bar, ob);
      bulk_load(sm + C::kOmega, prm.omega_img, ob, setup_bar);
      // head k's dS pair and dz go in once head k - 1's last tile is done with them
      auto load_head = [&](int k) {
        const size_t hh = (size_t)(h0 + k);
        mbar_arrive_expect_tx(img_full, 2 * hb + zb);
        bulk_load(sm + C::kHi, prm.ds_hi + hh * hb, hb, img_full);
        bulk_load(sm + C::kLo, prm.ds_lo + hh * hb, hb, img_full);
        bulk_load(sm + C::kZ, prm.zvec + hh * M, zb, img_full);
      };
      int ni = 0;
      if (n_heads > 0) load_head(ni++);
      Watchdog wd(wctx);
      int nk = 0, nv = 0;
      bool ok = true;
      while (ok && (nk < n_tiles || nv < n_tiles || ni < n_heads)) {
        bool progress = false;
        if (nk < n_tiles && (nk < NK || mbar_test_wait(smem_addr(&k_empty[nk % NK]), ((nk / NK) - 1) & 1))) {
          const int st = nk % NK;
          mbar_arrive_expect_tx(&k_full[st], kTileBytes);
          tma_load_3d(sm + C::kK + st * kTileBytes, &mapK, 0, tile_of(nk) * kBM, head_of(nk), &k_full[st]);
          ++nk;
          progress = true;
        }
        if (nv < nk && (nv == 0 || mbar_test_wait(smem_addr(v_empty), (nv - 1) & 1))) {
          mbar_arrive_expect_tx(v_full, kTileBytes);
          tma_load_3d(sm + C::kV, &mapV, 0, tile_of(nv) * kBM, head_of(nv), v_full);
          ++nv;
          progress = true;
        }
        if (ni < n_heads && mbar_test_wait(smem_addr(img_free), (ni - 1) & 1)) {
          load_head(ni++);
          progress = true;
        }
        if (progress) wd.progress();
        else ok = wd.idle();
      }
      for (int x = max(0, nk - NK); x < nk; ++x) mbar_wait(&k_full[x % NK], (x / NK) & 1, wctx);
      if (nv > 0) mbar_wait(v_full, (nv - 1) & 1, wctx);
      if (ni > 0) mbar_wait(img_full, (ni - 1) & 1, wctx);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t id_proj = idesc_f16(kBM, M, false, false);
      constexpr uint32_t id_dv = idesc_bf16(kBM, kD, false, false);
      constexpr uint32_t id_t = idesc_bf16(kBM, M, false, true);
      constexpr uint32_t id_dk = idesc_f16(kBM, kD, false, true);
      const uint32_t omega_a = smem_addr(sm + C::kOmega);
      const uint32_t hi_a = smem_addr(sm + C::kHi);
      const uint32_t lo_a = smem_addr(sm + C::kLo);
      const uint32_t phi_a = smem_addr(sm + C::kPhi);
      const uint32_t v_a = smem_addr(sm + C::kV);
      bool ok = mbar_wait(setup_bar, 0, wctx);
      Watchdog wd(wctx);
      int ia = 0, ic = 0, id = 0;
      while (ok && id < n_tiles) {
        bool progress = false;
        if (ia < n_tiles) {
          const int st = ia % NK;
          if (mbar_test_wait(smem_addr(&kn_full[st]), (ia / NK) & 1) &&
              (ia == 0 || mbar_test_wait(smem_addr(t_free), (ia - 1) & 1))) {
            tc_fence_after();
            const uint64_t a0 = sdesc(smem_addr(sm + C::kK + st * kTileBytes), 16, 1024);
            const uint64_t b0 = sdesc(omega_a, 16, 1024);
#pragma unroll
            for (int k = 0; k < kD / 16; ++k)
              mma_bf16(tmem, dadd(a0, kstep_k(k, kAtom)), dadd(b0, kstep_k(k, M * 128)), id_proj, k > 0);
            mma_commit(p_full);
            ++ia;
            progress = true;
          }
        }
        if (ic < ia && mbar_test_wait(smem_addr(phi_full), ic & 1) && mbar_test_wait(smem_addr(p_free), ic & 1) &&
            mbar_test_wait(smem_addr(v_full), ic & 1) &&
            mbar_test_wait(smem_addr(img_full), (head_of(ic) - h0) & 1) &&
            (ic == 0 || mbar_test_wait(smem_addr(dv_free), (ic - 1) & 1))) {
          tc_fence_after();
          // dV = phi(K) dS_hi (the image's features are the K dimension)
          const uint64_t a0 = sdesc(phi_a, 16, 1024);
          const uint64_t b0 = sdesc(hi_a, 16, 1024);
#pragma unroll
          for (int fb = 0; fb < NFB; ++fb)
#pragma unroll
            for (int kk = 0; kk < kFB / 16; ++kk)
              mma_bf16(tmem + kDVCol, dadd(a0, fb * 2 * kAtom + kstep_k(kk, kAtom)),
                       dadd(b0, fb * 2 * kD * 128 + kstep_k(kk, kD * 128)), id_dv, (fb > 0) || (kk > 0));
          // T = V (dS_hi + dS_lo)^T into [0, M) (the images' rows are the K dimension)
          const uint64_t av = sdesc(v_a, 16, 1024);
          const uint64_t bh0 = sdesc(hi_a, kD * 128, 1024);
          const uint64_t bl0 = sdesc(lo_a, kD * 128, 1024);
#pragma unroll
          for (int k = 0; k < kD / 16; ++k) mma_bf16(tmem, dadd(av, kstep_k(k, kAtom)), dadd(bh0, kstep_mn(k)), id_t, k > 0);
#pragma unroll
          for (int k = 0; k < kD / 16; ++k) mma_bf16(tmem, dadd(av, kstep_k(k, kAtom)), dadd(bl0, kstep_mn(k)), id_t, true);
          mma_commit(t_full);
          ++ic;
          progress = true;
        }
        if (id < ic && mbar_test_wait(smem_addr(g_full), id & 1) &&
            (id == 0 || mbar_test_wait(smem_addr(dk_free), (id - 1) & 1))) {
          // dK (scaled, without the s k sum g term) = G Omega
          tc_fence_after();
          const uint64_t a0 = sdesc(phi_a, 16, 1024);
          const uint64_t b0 = sdesc(omega_a, M * 128, 1024);
#pragma unroll
          for (int fb = 0; fb < NFB; ++fb)
#pragma unroll
            for (int kk = 0; kk < kFB / 16; ++kk)
              mma_bf16(tmem + kDKCol, dadd(a0, fb * 2 * kAtom + kstep_k(kk, kAtom)), dadd(b0, kstep_mn(fb * 8 + kk)),
                       id_dk, (fb > 0) || (kk > 0));
          mma_commit(dk_full);
          ++id;
          progress = true;
        }
        if (progress) wd.progress();
        else ok = wd.idle();
      }
      mma_commit(done_bar);
      mbar_wait(done_bar, 0, wctx);
    }
  } else if (warp < 2 + kNormWarps) {
    // squared norms of the K rows; K rewritten as fp16
    for (int i = 0; i < n_tiles; ++i) {
      const int ks = i % NK;
      if (!mbar_wait(&k_full[ks], (i / NK) & 1, wctx)) break;
      uint8_t* kt = sm + C::kK + ks * kTileBytes;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int r = (warp - 2) * 64 + lane + 32 * j;
        norm_s[ks * kBM + r] = tile_row_sq_to_f16<kD>(kt, r);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&kn_full[ks]);
    }
  } else {
    const int wg = (warp - 4) >> 2;
    const int q = warp & 3;
    const int t = q * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    const int my_fb = (NFB == 2) ? wg : 0;
    constexpr int kChunks = (NFB == 2) ? 4 : 2;    // 32-column chunks of this thread's columns
    const int c0 = (NFB == 2) ? 0 : wg * 64;
    const int f_base = my_fb * kFB + c0;
    float R, W;
    key_reference(prm.key_ref, prm.m, &R, &W);
    const float c1 = feature_c1<FM>(prm.scale);
    const float hs2 = 0.5f * prm.scale * prm.scale;
    uint8_t* phi_blk = sm + C::kPhi + my_fb * 2 * kAtom;
    const uint32_t phi_blk_a = smem_addr(phi_blk);
    const uint32_t vt = smem_addr(sm + C::kV);
    float* xa = xch;                  // [2][128] partial max |g|
    float* xb = xch + 2 * kBM;        // [2][128] partial sum g
    bool ok = mbar_wait(setup_bar, 0, wctx);   // dz is read from shared memory below
    for (int i = 0; i < n_tiles; ++i) {
      const int ks = i % NK;
      const int hi_t = head_of(i), ti = tile_of(i);
      const bool valid = ti * kBM + t < prm.L;
      const bool head_ends = i == n_tiles - 1 || head_of(i + 1) != hi_t;
      // ---- phi(K) = exp(s w.k - s^2 |k|^2 / 2 - R); rows past L get 0
      if (ok) ok = mbar_wait(&kn_full[ks], (i / NK) & 1, wctx);
      const float bias =
          !valid ? INFINITY : (FM == FAVOR_FM_PRF ? (hs2 * norm_s[ks * kBM + t] + R) * kLog2e : 0.f);
      if (ok) ok = mbar_wait(p_full, i & 1, wctx);
      tc_fence_after();
#pragma unroll 1
      for (int ch = 0; ch < kChunks; ++ch) {
        uint32_t x[32];
        if (ok) {
          tmem_ld32(tmem + lane_off + f_base + 32 * ch, x);
          tmem_ld_wait();
        }
        if (ch == kChunks - 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(p_free);
        }
        if (ok) {
          if constexpr (FM == FAVOR_FM_RELU)
            relu_guard(x, f_base + 32 * ch, relu_tau(norm_s[ks * kBM + t], W), sm + C::kK + ks * kTileBytes, t,
                       prm.omega);
          feature_pack<FM>(x, c1, bias);
          store_row<16>(phi_blk_a, kAtom, t, c0 + 32 * ch, x);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(phi_full);

      // ---- dV, staged over the V tile (read by T, complete with dV)
      if (ok) ok = mbar_wait(t_full, i & 1, wctx);
      tc_fence_after();
#pragma unroll 1
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t v[16];
        if (ok) {
          tmem_ld16(tmem + lane_off + kDVCol + wg * 32 + 16 * hf, v);
          tmem_ld_wait();
        }
        if (hf == 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(dv_free);
        }
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int chunk = wg * 4 + 2 * hf + c;
          const int o = 8 * c;
          st_shared_v4(vt + t * 128 + ((chunk ^ (t & 7)) << 4),
                       pack_bf16(__uint_as_float(v[o]), __uint_as_float(v[o + 1])),
                       pack_bf16(__uint_as_float(v[o + 2]), __uint_as_float(v[o + 3])),
                       pack_bf16(__uint_as_float(v[o + 4]), __uint_as_float(v[o + 5])),
                       pack_bf16(__uint_as_float(v[o + 6]), __uint_as_float(v[o + 7])));
        }
      }
      fence_proxy_async_smem();
      // ---- g = (T + dz) * slope(phi): row maximum and (prf) row sum
      if (ok) ok = mbar_wait(img_full, (hi_t - h0) & 1, wctx);   // this head's dz
      auto chunk_g = [&](int ch, uint32_t (&x)[32]) {
        const int col = c0 + 32 * ch;
        tmem_ld32(tmem + lane_off + f_base + 32 * ch, x);
        uint32_t w[16];
        load_row32(phi_blk + (col >> 6) * kAtom, (col & 63) >> 3, t, w);
        tmem_ld_wait();
        const float4* zc = reinterpret_cast<const float4*>(dz_s + f_base + 32 * ch);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float4 zz = zc[j];
          const float zv[4] = {zz.x, zz.y, zz.z, zz.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int o = 4 * j + k;
            const float ph = (k & 1) ? bf_hi(w[o >> 1]) : bf_lo(w[o >> 1]);
            const float dphi = __uint_as_float(x[o]) + zv[k];
            float gv;
            if constexpr (FM == FAVOR_FM_PRF) gv = dphi * ph;
            else if constexpr (FM == FAVOR_FM_ELU1) gv = dphi * fminf(ph, 1.f);
            else gv = ph > 0.f ? dphi : 0.f;
            x[o] = __float_as_uint(gv);
          }
        }
      };
      // g (bf16) over phi(K), then rescaled by the row's power of two to fp16
      float gmax = 0.f, gsum = 0.f;
#pragma unroll 1
      for (int ch = 0; ch < kChunks; ++ch) {
        uint32_t g[32];
        if (ok) chunk_g(ch, g);
        if (ch == kChunks - 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(t_free);
        }
        if (ok) {
          float s8[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) s8[j] = 0.f;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            gmax = fmaxf(gmax, fabsf(__uint_as_float(g[j])));
            s8[j & 7] += __uint_as_float(g[j]);
          }
          gsum += ((s8[0] + s8[1]) + (s8[2] + s8[3])) + ((s8[4] + s8[5]) + (s8[6] + s8[7]));
          pack_g_bf16(g);
          store_row<16>(phi_blk_a, kAtom, t, c0 + 32 * ch, g);
        }
      }
      if (head_ends) {
        // the head's dS pair and dz: read by this tile's products (complete)
        // and by the pass above, for the last time
        __syncwarp();
        if (lane == 0) mbar_arrive(img_free);
      }
      xa[wg * kBM + t] = gmax;
      xb[wg * kBM + t] = gsum;
      named_bar(1, kEpiThreads);
      if (threadIdx.x == kEpiTid0) {
        if (ok && !*abort_flag) {
          tma_store_3d(&mapDV, 0, ti * kBM, hi_t, sm + C::kV);
          bulk_commit();
        }
        // the V slot takes the next tile once the store has read it
        bulk_wait_read0();
        mbar_arrive(v_empty);
      }
      float beta, inv_beta;
      row_scale(fmaxf(xa[t], xa[kBM + t]), &beta, &inv_beta);
      const float gs = xb[t] + xb[kBM + t];
#pragma unroll 1
      for (int ch = 0; ch < kChunks; ++ch) {
        const int col = c0 + 32 * ch;
        uint32_t w[16];
        load_row32(phi_blk + (col >> 6) * kAtom, (col & 63) >> 3, t, w);
        rescale_f16(w, beta);
        store_row<16>(phi_blk_a, kAtom, t, col, w);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(g_full);

      // ---- dK = s ((G Omega) / beta - [prf] s k sum_i g_i), over the K tile
      if (ok) ok = mbar_wait(dk_full, i & 1, wctx);
      tc_fence_after();
      uint8_t* kt = sm + C::kK + ks * kTileBytes;
      const float f = prm.scale * inv_beta;
      const float fk = FM == FAVOR_FM_PRF ? prm.scale * prm.scale * gs : 0.f;
#pragma unroll 1
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t v[16];
        if (ok) {
          tmem_ld16(tmem + lane_off + kDKCol + wg * 32 + 16 * hf, v);
          tmem_ld_wait();
        }
        if (hf == 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(dk_free);
        }
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int chunk = wg * 4 + 2 * hf + c;
          uint8_t* p = kt + t * 128 + ((chunk ^ (t & 7)) << 4);
          const uint4 u = *reinterpret_cast<const uint4*>(p);
          const uint32_t w[4] = {u.x, u.y, u.z, u.w};
          uint32_t o[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float k0 = __half2float(__ushort_as_half(static_cast<unsigned short>(w[j] & 0xFFFFu)));
            const float k1 = __half2float(__ushort_as_half(static_cast<unsigned short>(w[j] >> 16)));
            const float a0 = __uint_as_float(v[8 * c + 2 * j]) * f - fk * k0;
            const float a1 = __uint_as_float(v[8 * c + 2 * j + 1]) * f - fk * k1;
            o[j] = pack_bf16(a0, a1);
          }
          st_shared_v4(smem_addr(p), o[0], o[1], o[2], o[3]);
        }
      }
      fence_proxy_async_smem();
      named_bar(1, kEpiThreads);
      if (threadIdx.x == kEpiTid0) {
        if (ok && !*abort_flag) {
          tma_store_3d(&mapDK, 0, ti * kBM, hi_t, kt);
          bulk_commit();
        }
        // the K slot is reused once the store has read it
        bulk_wait_read0();
        mbar_arrive(&k_empty[ks]);
      }
    }
    if (threadIdx.x == kEpiTid0) bulk_wait0();
    mbar_wait(done_bar, 0, wctx);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
struct GradLayout {
  TcLayout fwd;
  int ctas, parts;              // CTAs of each backward kernel; [dS | dz] slots per head
  size_t off_z, off_part, off_hi, off_lo, off_dz, bytes;
};

GradLayout grad_layout(const Shape& s) {
  GradLayout g{};
  const size_t BH = s.BH();
  const long long total = (long long)BH * ((s.L + kBM - 1) / kBM);
  g.fwd = tc_bidir_layout(s);
  // one CTA per SM (or per tile), each an even share of the (head, tile)
  // list; a head meets at most ceil(ctas / BH) + 1 of them
  g.ctas = (int)std::min<long long>(sm_count(), total);
  g.parts = (g.ctas + (int)BH - 1) / (int)BH + 1;
  g.off_z = align_up(g.fwd.bytes, 1024);                                  // fp32 z [BH][m]
  g.off_part = align_up(g.off_z + BH * s.m * 4, 1024);                    // fp32 [BH][m/128][parts][d+1][128]
  g.off_hi = align_up(g.off_part + BH * s.m * g.parts * (kD + 1) * 4, 1024);  // bf16 dS pair [BH][m/64][d][128 B]
  g.off_lo = align_up(g.off_hi + BH * s.m * kD * 2, 1024);
  g.off_dz = align_up(g.off_lo + BH * s.m * kD * 2, 1024);                // fp32 dz [BH][m]
  g.bytes = align_up(g.off_dz + BH * s.m * 4, 1024);
  return g;
}

template <int M, int FM>
cudaError_t launch_grad(const void* Q, const void* K, const void* V, const void* dO, void* dQ, void* dK, void* dV,
                        const float* omega, const Shape& s, float scale, char* ws, int32_t* status,
                        cudaStream_t stream) {
  const GradLayout g = grad_layout(s);
  CUtensorMap mq, mdo, mdq, mk, mv, mdk, mdv;
  if (!make_map(&mq, Q, s) || !make_map(&mdo, dO, s) || !make_map(&mdq, dQ, s) || !make_map(&mk, K, s) ||
      !make_map(&mv, V, s) || !make_map(&mdk, dK, s) || !make_map(&mdv, dV, s))
    return cudaErrorInvalidValue;
  uint8_t* hi = reinterpret_cast<uint8_t*>(ws + g.off_hi);
  uint8_t* lo = reinterpret_cast<uint8_t*>(ws + g.off_lo);
  float* dz = reinterpret_cast<float*>(ws + g.off_dz);
  float* part = reinterpret_cast<float*>(ws + g.off_part);
  GradParams a{};
  a.key_ref = reinterpret_cast<const float*>(ws);
  a.omega = omega;
  a.omega_img = reinterpret_cast<const uint8_t*>(ws + g.fwd.off_omega_img);
  a.state_img = reinterpret_cast<const uint8_t*>(ws + g.fwd.off_state_img);
  a.zvec = reinterpret_cast<const float*>(ws + g.off_z);
  a.partS = part;
  a.status = status;
  a.L = s.L;
  a.m = s.m;
  a.n_heads = s.BH();
  a.parts = g.parts;
  a.scale = scale;
  GradParams b{};
  b.key_ref = a.key_ref;
  b.omega = omega;
  b.omega_img = a.omega_img;
  b.zvec = dz;
  b.ds_hi = hi;
  b.ds_lo = lo;
  b.status = status;
  b.L = s.L;
  b.m = s.m;
  b.n_heads = s.BH();
  b.scale = scale;
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(grad_query_kernel<M, FM>), GqCfg::kSmem);
  if (e == cudaSuccess)
    e = ensure_dynamic_smem(reinterpret_cast<const void*>(grad_key_kernel<M, FM>), GkCfg::kSmem);
  if (e != cudaSuccess) return e;
  grad_query_kernel<M, FM><<<g.ctas, kBwdThreads, GqCfg::kSmem, stream>>>(mq, mdo, mdq, a);
  grad_merge_kernel<M><<<dim3(s.BH(), kMergeSplit), 128, 0, stream>>>(part, g.parts, (s.L + kBM - 1) / kBM, s.BH(),
                                                                      g.ctas, hi, lo, dz);
  grad_key_kernel<M, FM><<<g.ctas, kBwdThreads, GkCfg::kSmem, stream>>>(mk, mv, mdk, mdv, b);
  return cudaGetLastError();
}

template <int FM>
cudaError_t grad_fm(const void* Q, const void* K, const void* V, const void* dO, void* dQ, void* dK, void* dV,
                    const float* omega, const Shape& s, float scale, char* ws, int32_t* status, cudaStream_t stream) {
  return s.m == 256 ? launch_grad<256, FM>(Q, K, V, dO, dQ, dK, dV, omega, s, scale, ws, status, stream)
                    : launch_grad<128, FM>(Q, K, V, dO, dQ, dK, dV, omega, s, scale, ws, status, stream);
}

}  // namespace

bool tc_bwd_supported(bool causal, int d, int m, bool bf16) { return !causal && bf16 && d == kD && (m == 128 || m == 256); }

size_t tc_bwd_workspace_bytes(const Shape& s) { return grad_layout(s).bytes; }

cudaError_t tc_bwd_bidir(const void* Q, const void* K, const void* V, const void* dO, void* dQ, void* dK, void* dV,
                         const float* omega, float scale, const Shape& s, void* ws, int32_t* status,
                         cudaStream_t stream, int fm) {
  char* w = static_cast<char*>(ws);
  // prep (key reference, fp16 Omega image) and the
  // forward's state: the bf16 image of [S | z] and z in fp32
  cudaError_t e = tc_state(false, K, V, omega, scale, s, ws, status, stream, fm,
                           reinterpret_cast<float*>(w + grad_layout(s).off_z));
  if (e != cudaSuccess) return e;
  if (fm == FAVOR_FM_RELU) return grad_fm<FAVOR_FM_RELU>(Q, K, V, dO, dQ, dK, dV, omega, s, scale, w, status, stream);
  if (fm == FAVOR_FM_ELU1) return grad_fm<FAVOR_FM_ELU1>(Q, K, V, dO, dQ, dK, dV, omega, s, scale, w, status, stream);
  return grad_fm<FAVOR_FM_PRF>(Q, K, V, dO, dQ, dK, dV, omega, s, scale, w, status, stream);
}

}  // namespace favor
