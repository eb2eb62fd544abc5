// Tensor-core (tcgen05) FAVOR+ kernels for sm_103a: bf16 operands in shared
// memory (TMA, 128-byte swizzle), fp32 accumulators in tensor memory.
//
// "Performer — Rethinking Attention with Performers" (digest), §Key equations
// and the flowchart: phi(K)^T V and phi(K)^T 1 are formed first, then
// phi(Q) times each, then the row-wise divide.  The three contractions are
// dense GEMMs and run on the tensor cores:
//   projection   P   = X Omega^T           (M = 128 tokens, N = 128 features, K = d)
//   state        S~ += phi(K)^T [V | 1]    (M = 128 features, N = d + 16,   K = 128 tokens)
//   output       O   = phi(Q) S~           (M = 128 tokens,   N = d + 16,   K = m)
// The exponentials of the feature map run on the CUDA cores between them
// (TMEM -> registers -> bf16 in shared memory).
//
// Warp roles in both kernels (192 threads): warp 0 issues TMA loads, warp 1
// owns tensor memory and issues the MMAs (one elected thread), warps 2-5 are
// the epilogue (thread = one TMEM lane = one token or one feature).
#include <cudaTypedefs.h>

#include <mutex>

#include "tc.cuh"
#include "tc_ptx.cuh"

namespace favor {
namespace {

using namespace tc;

constexpr int kBM = 128;          // tokens per tile
constexpr int kFB = 128;          // features per state CTA
constexpr int kThreads = 192;
constexpr int kEpiThreads = 128;
constexpr uint32_t kTmemCols = 512;
constexpr int kAtom = 128 * 128;  // bytes of one [128 rows][128 B] swizzle block

// ---------------------------------------------------------------------------
// workspace layout of the tensor-core path
// ---------------------------------------------------------------------------
struct TcPlan {
  int n_fb, n_tiles, n_split, tiles_per_split;   // state kernel
  int out_tiles_per_cta, out_ctas;               // output kernel
  size_t off_omega_img, off_counters, off_partS, off_state_img, bytes;
};

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Splits of `tiles` tiles for each of `units` independent rows of CTAs: the
// fewest splits minimising waves x (tiles per CTA + per-CTA set-up, counted
// as kCtaOverheadTiles tiles).
constexpr int kCtaOverheadTiles = 3;
int pick_split(int units, int tiles, int sms) {
  int best = 1;
  long best_cost = -1;
  for (int s = 1; s <= tiles; ++s) {
    const long ctas = (long)units * s;
    const long waves = (ctas + sms - 1) / sms;
    const long cost = waves * ((tiles + s - 1) / s + kCtaOverheadTiles);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = s;
    }
  }
  return best;
}

TcPlan tc_plan(const Shape& s) {
  TcPlan p{};
  const int BH = s.BH();
  const int sms = 152;
  p.n_fb = s.m / kFB;
  p.n_tiles = (s.L + kBM - 1) / kBM;
  p.n_split = pick_split(BH * p.n_fb, p.n_tiles, sms);
  p.tiles_per_split = (p.n_tiles + p.n_split - 1) / p.n_split;
  p.n_split = (p.n_tiles + p.tiles_per_split - 1) / p.tiles_per_split;
  const int oc = pick_split(BH, p.n_tiles, sms);
  p.out_tiles_per_cta = (p.n_tiles + oc - 1) / oc;
  p.out_ctas = (p.n_tiles + p.out_tiles_per_cta - 1) / p.out_tiles_per_cta;
  size_t off = kWsHeader;
  off = align_up(off, 1024);
  p.off_omega_img = off;
  off = align_up(off + (size_t)s.m * s.d * 2, 1024);
  p.off_counters = off;
  off = align_up(off + (size_t)BH * p.n_fb * sizeof(uint32_t), 1024);
  p.off_partS = off;
  off = align_up(off + (size_t)BH * p.n_fb * p.n_split * (s.d + 1) * kFB * sizeof(float), 1024);
  p.off_state_img = off;
  off = align_up(off + (size_t)BH * s.m * (s.d + 16) * 2, 1024);
  p.bytes = off;
  return p;
}

// ---------------------------------------------------------------------------
// shared epilogue pieces
// ---------------------------------------------------------------------------

// Squared norm of row t of a [128][d] bf16 tile stored as 64-column swizzle
// blocks (TMA layout).
template <int D>
__device__ __forceinline__ float tile_row_sq(const uint8_t* tile, int t) {
  float acc = 0.f;
#pragma unroll
  for (int a = 0; a < D / 64; ++a) {
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint4 v = *reinterpret_cast<const uint4*>(tile + a * kAtom + t * 128 + ((c ^ (t & 7)) << 4));
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float lo = __uint_as_float(w[j] << 16);
        const float hi = __uint_as_float(w[j] & 0xFFFF0000u);
        acc = fmaf(lo, lo, acc);
        acc = fmaf(hi, hi, acc);
      }
    }
  }
  return acc;
}

// phi for 32 consecutive features of one row, written as bf16 into the
// swizzled [feature atom][128 rows][128 B] buffer: phi = 2^(p*c1 - b).
__device__ __forceinline__ void write_phi32(uint32_t phi_base, int t, int f0, const uint32_t (&p)[32], float c1,
                                            float b, bool valid) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t w[4];
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const float x0 = valid ? ex2(fmaf(__uint_as_float(p[8 * j + 2 * h]), c1, -b)) : 0.f;
      const float x1 = valid ? ex2(fmaf(__uint_as_float(p[8 * j + 2 * h + 1]), c1, -b)) : 0.f;
      w[h] = pack_bf16(x0, x1);
    }
    const int f = f0 + 8 * j;
    const int atom = f >> 6, chunk = (f & 63) >> 3;
    st_shared_v4(phi_base + atom * kAtom + t * 128 + ((chunk ^ (t & 7)) << 4), w[0], w[1], w[2], w[3]);
  }
}

// ---------------------------------------------------------------------------
// state kernel: one (L split, 128-feature block, head) per CTA
// ---------------------------------------------------------------------------
struct StateParams {
  const float* key_ref;
  const uint8_t* omega_img;
  float* partS;            // [BH][n_fb][n_split][d+1][128]
  uint32_t* counters;      // [BH][n_fb]
  uint8_t* state_img;      // [BH][m/64][d+16][128 B]
  int32_t* status;
  int L, m, n_split, tiles_per_split;
  float scale;
};

template <int D>
struct StateCfg {
  static constexpr int NS = (D == 64) ? 3 : 2;      // K/V stages
  static constexpr int NPHI = (D == 64) ? 2 : 1;    // phi buffers
  static constexpr int kTileBytes = D * kBM * 2;    // one K or V tile
  static constexpr int kOmega = 0;
  static constexpr int kOnes = kOmega + kFB * D * 2;
  static constexpr int kStages = kOnes + kAtom;
  static constexpr int kPhi = kStages + NS * 2 * kTileBytes;
  static constexpr int kBars = kPhi + NPHI * kAtom * 2;
  static constexpr int kSmem = kBars + 256 + 1024;  // + barriers/slots + alignment slack
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1) state_kernel(const __grid_constant__ CUtensorMap mapK,
                                                            const __grid_constant__ CUtensorMap mapV,
                                                            StateParams prm) {
  using C = StateCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::kBars);
  uint64_t* full = bars;                      // [NS]
  uint64_t* empty = full + C::NS;             // [NS]
  uint64_t* p_full = empty + C::NS;           // [2]
  uint64_t* p_free = p_full + 2;              // [2]
  uint64_t* phi_full = p_free + 2;            // [NPHI]
  uint64_t* phi_free = phi_full + C::NPHI;    // [NPHI]
  uint64_t* setup_bar = phi_free + C::NPHI;
  uint64_t* done_bar = setup_bar + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* is_last = const_cast<int*>(abort_flag) + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x, fb = blockIdx.y, bh = blockIdx.z;
  const int n_fb = gridDim.y;
  const int tile0 = split * prm.tiles_per_split;
  const int n_tiles_total = (prm.L + kBM - 1) / kBM;
  const int n_tiles = min(prm.tiles_per_split, n_tiles_total - tile0);
  const WaitCtx wctx{abort_flag, prm.status};

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&p_full[i], 1);
      mbar_init(&p_free[i], 4);
    }
    for (int i = 0; i < C::NPHI; ++i) {
      mbar_init(&phi_full[i], 4);
      mbar_init(&phi_free[i], 1);
    }
    mbar_init(setup_bar, 1);
    mbar_init(done_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (warp >= 2) {
    // all-ones block: the extra 16 columns of [V | 1]
    const uint32_t one2 = 0x3F803F80u;
    for (int e = threadIdx.x - 64; e < kAtom / 16; e += kEpiThreads)
      *reinterpret_cast<uint4*>(sm + C::kOnes + e * 16) = make_uint4(one2, one2, one2, one2);
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      prefetch_tmap(&mapK);
      prefetch_tmap(&mapV);
      mbar_arrive_expect_tx(setup_bar, kFB * D * 2);
      bulk_load(sm + C::kOmega, prm.omega_img + (size_t)fb * kFB * D * 2, kFB * D * 2, setup_bar);
      int last_issue[C::NS];
      for (int i = 0; i < C::NS; ++i) last_issue[i] = -1;
      for (int i = 0; i < n_tiles; ++i) {
        const int st = i % C::NS;
        if (i >= C::NS && !mbar_wait(&empty[st], ((i / C::NS) - 1) & 1, wctx)) break;
        mbar_arrive_expect_tx(&full[st], 2 * C::kTileBytes);
        uint8_t* kt = sm + C::kStages + st * 2 * C::kTileBytes;
        uint8_t* vt = kt + C::kTileBytes;
        const int row = (tile0 + i) * kBM;
#pragma unroll
        for (int a = 0; a < D / 64; ++a) {
          tma_load_3d(kt + a * kAtom, &mapK, a * 64, row, bh, &full[st]);
          tma_load_3d(vt + a * kAtom, &mapV, a * 64, row, bh, &full[st]);
        }
        last_issue[st] = i;
      }
      // drain: every issued load has landed before the CTA can exit
      for (int st = 0; st < C::NS; ++st)
        if (last_issue[st] >= 0) mbar_wait(&full[st], (last_issue[st] / C::NS) & 1, wctx);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t id_proj = idesc_bf16(kBM, kFB, false, false);
      const uint32_t id_state = idesc_bf16(kFB, D, true, true);
      const uint32_t id_ones = idesc_bf16(kFB, 16, true, true);
      const uint32_t s_tm = tmem + 256;           // S~: columns 256 .. 256+d+15
      const uint32_t omega_a = smem_addr(sm + C::kOmega);
      const uint32_t ones_a = smem_addr(sm + C::kOnes);
      bool ok = mbar_wait(setup_bar, 0, wctx);
      auto issue_state = [&](int j) -> bool {
        const int b = j % C::NPHI;
        if (!mbar_wait(&phi_full[b], (j / C::NPHI) & 1, wctx)) return false;
        tc_fence_after();
        const uint32_t phi_a = smem_addr(sm + C::kPhi + b * 2 * kAtom);
        const uint32_t v_a = smem_addr(sm + C::kStages + (j % C::NS) * 2 * C::kTileBytes + C::kTileBytes);
#pragma unroll
        for (int k = 0; k < kBM / 16; ++k) {
          const uint64_t ad = sdesc(phi_a + k * 2048, kAtom, 1024);
          const bool acc = (j > 0) || (k > 0);
          mma_bf16(s_tm, ad, sdesc(v_a + k * 2048, kAtom, 1024), id_state, acc);
          mma_bf16(s_tm + D, ad, sdesc(ones_a + k * 2048, kAtom, 1024), id_ones, acc);
        }
        mma_commit(&phi_free[b]);
        mma_commit(&empty[j % C::NS]);
        return true;
      };
      for (int i = 0; ok && i < n_tiles; ++i) {
        const int st = i % C::NS, pb = i & 1;
        if (!mbar_wait(&full[st], (i / C::NS) & 1, wctx)) { ok = false; break; }
        if (i >= 2 && !mbar_wait(&p_free[pb], ((i >> 1) - 1) & 1, wctx)) { ok = false; break; }
        tc_fence_after();
        const uint32_t k_a = smem_addr(sm + C::kStages + st * 2 * C::kTileBytes);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * kAtom + (k & 3) * 32;
          mma_bf16(tmem + pb * kFB, sdesc(k_a + off, 16, 1024), sdesc(omega_a + off, 16, 1024), id_proj, k > 0);
        }
        mma_commit(&p_full[pb]);
        if (i > 0 && !issue_state(i - 1)) { ok = false; break; }
      }
      if (ok && n_tiles > 0) issue_state(n_tiles - 1);
      mma_commit(done_bar);
      mbar_wait(done_bar, 0, wctx);
    }
  } else {
    // ---------------- epilogue: 128 threads, one TMEM lane each ----------------
    const int q = warp & 3;
    const int t = q * 32 + lane;                   // token row of P, feature row of S~
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    const float R = *prm.key_ref;
    const float c1 = prm.scale * kLog2e;
    const float hs2 = 0.5f * prm.scale * prm.scale;
    bool ok = true;
    for (int i = 0; ok && i < n_tiles; ++i) {
      const int st = i % C::NS, pb = i & 1, b = i % C::NPHI;
      if (!mbar_wait(&p_full[pb], (i >> 1) & 1, wctx)) { ok = false; break; }
      tc_fence_after();
      const uint8_t* kt = sm + C::kStages + st * 2 * C::kTileBytes;
      const float ksq = tile_row_sq<D>(kt, t);
      const float bias = (hs2 * ksq + R) * kLog2e;
      const bool valid = (tile0 + i) * kBM + t < prm.L;
      if (i >= C::NPHI && !mbar_wait(&phi_free[b], ((i / C::NPHI) - 1) & 1, wctx)) { ok = false; break; }
      const uint32_t phi_a = smem_addr(sm + C::kPhi + b * 2 * kAtom);
#pragma unroll
      for (int cb = 0; cb < kFB / 32; ++cb) {
        uint32_t p[32];
        tmem_ld32(tmem + lane_off + pb * kFB + cb * 32, p);
        tmem_ld_wait();
        write_phi32(phi_a, t, cb * 32, p, c1, bias, valid);
      }
      tc_fence_before();
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&p_free[pb]);
        mbar_arrive(&phi_full[b]);
      }
    }
    // final state: lane f holds feature f of this block
    const bool done = mbar_wait(done_bar, 0, wctx);
    tc_fence_after();
    float* dst = prm.partS + ((((size_t)bh * n_fb + fb) * prm.n_split + split) * (D + 1)) * kFB;
    if (done && !*abort_flag) {
#pragma unroll
      for (int cb = 0; cb < D / 32; ++cb) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_off + 256 + cb * 32, v);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) dst[(size_t)(cb * 32 + j) * kFB + t] = __uint_as_float(v[j]);
      }
      uint32_t z[16];
      tmem_ld16(tmem + lane_off + 256 + D, z);
      tmem_ld_wait();
      dst[(size_t)D * kFB + t] = __uint_as_float(z[0]);
    }
    tc_fence_before();
    // the last CTA of this (head, feature block) adds the splits in order
    named_bar(1, kEpiThreads);
    if (threadIdx.x == 64) {
      __threadfence();
      const uint32_t old = atomicAdd(&prm.counters[bh * n_fb + fb], 1u);
      *is_last = (old == (uint32_t)(prm.n_split - 1)) ? 1 : 0;
    }
    named_bar(1, kEpiThreads);
    if (*is_last) {
      __threadfence();
      const float* src = prm.partS + (((size_t)bh * n_fb + fb) * prm.n_split) * (D + 1) * kFB;
      uint8_t* img = prm.state_img + (size_t)bh * prm.m * (D + 16) * 2;
      const int f = fb * kFB + t;               // feature of this thread
      const int atom = f >> 6, cc = f & 63;
      for (int n = 0; n < D + 16; ++n) {
        float acc = 0.f;
        if (n <= D)
          for (int p = 0; p < prm.n_split; ++p) acc += src[((size_t)p * (D + 1) + n) * kFB + t];
        const size_t off = ((size_t)atom * (D + 16) + n) * 128 + (((cc >> 3) ^ (n & 7)) << 4) + (cc & 7) * 2;
        *reinterpret_cast<__nv_bfloat16*>(img + off) = __float2bfloat16_rn(acc);
      }
      if (threadIdx.x == 64) prm.counters[bh * n_fb + fb] = 0;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------------------
// output kernel: CTA = a run of 128-token tiles of one head; m <= 256
// ---------------------------------------------------------------------------
struct OutParams {
  const uint8_t* omega_img;
  const uint8_t* state_img;
  int32_t* status;
  int L, m, tiles_per_cta;
  float scale;
};

template <int D>
struct OutCfg {
  static constexpr int NSQ = 2;
  static constexpr int kTileBytes = D * kBM * 2;
  static constexpr int kOmegaMax = 256 * D * 2;
  static constexpr int kStateMax = 256 * (D + 16) * 2;
  static constexpr int kOmega = 0;
  static constexpr int kState = kOmega + kOmegaMax;
  static constexpr int kQ = kState + kStateMax;
  static constexpr int kPhi = kQ + NSQ * kTileBytes;
  static constexpr int kOut = kPhi + 4 * kAtom;      // 128 x 256 bf16
  static constexpr int kBars = kOut + kTileBytes;
  static constexpr int kSmem = kBars + 256 + 1024;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1) output_kernel(const __grid_constant__ CUtensorMap mapQ,
                                                             const __grid_constant__ CUtensorMap mapO,
                                                             OutParams prm) {
  using C = OutCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::kBars);
  uint64_t* q_full = bars;               // [NSQ]
  uint64_t* q_empty = q_full + C::NSQ;   // [NSQ]
  uint64_t* p_full = q_empty + C::NSQ;
  uint64_t* p_free = p_full + 1;
  uint64_t* phi_full = p_free + 1;
  uint64_t* phi_free = phi_full + 1;
  uint64_t* o_full = phi_free + 1;       // [2]
  uint64_t* o_free = o_full + 2;         // [2]
  uint64_t* setup_bar = o_free + 2;
  uint64_t* done_bar = setup_bar + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.y;
  const int n_tiles_total = (prm.L + kBM - 1) / kBM;
  const int tile0 = blockIdx.x * prm.tiles_per_cta;
  const int n_tiles = min(prm.tiles_per_cta, n_tiles_total - tile0);
  const int m = prm.m;
  const int n_fb = m / kFB;
  const WaitCtx wctx{abort_flag, prm.status};
  const uint32_t o_col[2] = {256u, 256u + 128u};   // O accumulators (d + 16 <= 128 columns each)

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NSQ; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);
    }
    mbar_init(p_full, 1);
    mbar_init(p_free, 4);
    mbar_init(phi_full, 4);
    mbar_init(phi_free, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&o_full[i], 1);
      mbar_init(&o_free[i], 4);
    }
    mbar_init(setup_bar, 1);
    mbar_init(done_bar, 1);
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
      prefetch_tmap(&mapO);
      const uint32_t ob = m * D * 2, sb = m * (D + 16) * 2;
      mbar_arrive_expect_tx(setup_bar, ob + sb);
      bulk_load(sm + C::kOmega, prm.omega_img, ob, setup_bar);
      bulk_load(sm + C::kState, prm.state_img + (size_t)bh * sb, sb, setup_bar);
      int last_issue[C::NSQ];
      for (int i = 0; i < C::NSQ; ++i) last_issue[i] = -1;
      for (int i = 0; i < n_tiles; ++i) {
        const int st = i % C::NSQ;
        if (i >= C::NSQ && !mbar_wait(&q_empty[st], ((i / C::NSQ) - 1) & 1, wctx)) break;
        mbar_arrive_expect_tx(&q_full[st], C::kTileBytes);
        uint8_t* qt = sm + C::kQ + st * C::kTileBytes;
#pragma unroll
        for (int a = 0; a < D / 64; ++a) tma_load_3d(qt + a * kAtom, &mapQ, a * 64, (tile0 + i) * kBM, bh, &q_full[st]);
        last_issue[st] = i;
      }
      for (int st = 0; st < C::NSQ; ++st)
        if (last_issue[st] >= 0) mbar_wait(&q_full[st], (last_issue[st] / C::NSQ) & 1, wctx);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t id_proj = idesc_bf16(kBM, kFB, false, false);
      const uint32_t id_out = idesc_bf16(kBM, D + 16, false, false);
      const uint32_t omega_a = smem_addr(sm + C::kOmega);
      const uint32_t state_a = smem_addr(sm + C::kState);
      const uint32_t phi_a = smem_addr(sm + C::kPhi);
      bool ok = mbar_wait(setup_bar, 0, wctx);
      for (int i = 0; ok && i < n_tiles; ++i) {
        const int st = i % C::NSQ, ob = i & 1;
        if (!mbar_wait(&q_full[st], (i / C::NSQ) & 1, wctx)) { ok = false; break; }
        if (i >= 1 && !mbar_wait(p_free, (i - 1) & 1, wctx)) { ok = false; break; }
        tc_fence_after();
        const uint32_t q_a = smem_addr(sm + C::kQ + st * C::kTileBytes);
        for (int f = 0; f < n_fb; ++f) {
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint32_t off = (k >> 2) * kAtom + (k & 3) * 32;
            mma_bf16(tmem + f * kFB, sdesc(q_a + off, 16, 1024),
                     sdesc(omega_a + f * kFB * D * 2 + off, 16, 1024), id_proj, k > 0);
          }
        }
        mma_commit(p_full);
        mma_commit(&q_empty[st]);
        if (!mbar_wait(phi_full, i & 1, wctx)) { ok = false; break; }
        if (i >= 2 && !mbar_wait(&o_free[ob], ((i >> 1) - 1) & 1, wctx)) { ok = false; break; }
        tc_fence_after();
        for (int kk = 0; kk < m / 16; ++kk) {
          const uint32_t pa = phi_a + (kk >> 2) * kAtom + (kk & 3) * 32;
          const uint32_t sa = state_a + (kk >> 2) * (D + 16) * 128 + (kk & 3) * 32;
          mma_bf16(tmem + o_col[ob], sdesc(pa, 16, 1024), sdesc(sa, 16, 1024), id_out, kk > 0);
        }
        mma_commit(&o_full[ob]);
        mma_commit(phi_free);
      }
      mma_commit(done_bar);
      mbar_wait(done_bar, 0, wctx);
    }
  } else {
    const int q = warp & 3;
    const int t = q * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    const float c1 = prm.scale * kLog2e;
    const uint32_t phi_a = smem_addr(sm + C::kPhi);
    const uint32_t out_a = smem_addr(sm + C::kOut);
    bool ok = true;
    // writes O of tile j (TMEM buffer j & 1) through the staging tile + TMA store
    auto store_out = [&](int j) {
      const int ob = j & 1;
      const bool have = mbar_wait(&o_full[ob], (j >> 1) & 1, wctx);
      tc_fence_after();
      float o[D];
      float den = 1.f;
      if (have) {
#pragma unroll
        for (int cb = 0; cb < D / 32; ++cb) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_off + o_col[ob] + cb * 32, v);
          tmem_ld_wait();
#pragma unroll
          for (int x = 0; x < 32; ++x) o[cb * 32 + x] = __uint_as_float(v[x]);
        }
        uint32_t z[16];
        tmem_ld16(tmem + lane_off + o_col[ob] + D, z);
        tmem_ld_wait();
        den = __uint_as_float(z[0]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&o_free[ob]);
      const int row = (tile0 + j) * kBM + t;
      if (row < prm.L && (!(den > 0.f) || !isfinite(den))) report_status(prm.status, FAVOR_ERR_NONFINITE);
      const float inv = 1.0f / den;
      if (threadIdx.x == 64 && j > 0) bulk_wait_read0();   // previous store has left the staging tile
      named_bar(1, kEpiThreads);
#pragma unroll
      for (int a = 0; a < D / 64; ++a) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const float* x = o + a * 64 + c * 8;
          st_shared_v4(out_a + a * kAtom + t * 128 + ((c ^ (t & 7)) << 4), pack_bf16(x[0] * inv, x[1] * inv),
                       pack_bf16(x[2] * inv, x[3] * inv), pack_bf16(x[4] * inv, x[5] * inv),
                       pack_bf16(x[6] * inv, x[7] * inv));
        }
      }
      fence_proxy_async_smem();
      named_bar(1, kEpiThreads);
      if (threadIdx.x == 64 && have && !*abort_flag) {
#pragma unroll
        for (int a = 0; a < D / 64; ++a) tma_store_3d(&mapO, a * 64, (tile0 + j) * kBM, bh, sm + C::kOut + a * kAtom);
        bulk_commit();
      }
    };
    for (int i = 0; i < n_tiles; ++i) {
      if (ok) ok = mbar_wait(p_full, i & 1, wctx);
      tc_fence_after();
      // pass 1: exact row maximum over all m features
      float mx = -INFINITY;
      if (ok) {
        for (int cb = 0; cb < m / 32; ++cb) {
          uint32_t p[32];
          tmem_ld32(tmem + lane_off + cb * 32, p);
          tmem_ld_wait();
#pragma unroll
          for (int x = 0; x < 32; ++x) mx = fmaxf(mx, __uint_as_float(p[x]));
        }
      }
      const float bias = mx * c1;
      if (ok && i >= 1) ok = mbar_wait(phi_free, (i - 1) & 1, wctx);
      if (ok) {
        for (int cb = 0; cb < m / 32; ++cb) {
          uint32_t p[32];
          tmem_ld32(tmem + lane_off + cb * 32, p);
          tmem_ld_wait();
          write_phi32(phi_a, t, cb * 32, p, c1, bias, true);
        }
      }
      tc_fence_before();
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(p_free);
        mbar_arrive(phi_full);
      }
      if (i >= 1) store_out(i - 1);
    }
    if (n_tiles >= 1) store_out(n_tiles - 1);
    if (threadIdx.x == 64) bulk_wait0();
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
PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// [BH, L, d] bf16 viewed as a 3-D tensor {d, L, BH}; box {64, 128, 1}; 128B swizzle.
bool make_map(CUtensorMap* map, const void* base, const Shape& s) {
  auto enc = get_encode();
  if (enc == nullptr) return false;
  cuuint64_t dims[3] = {(cuuint64_t)s.d, (cuuint64_t)s.L, (cuuint64_t)s.BH()};
  cuuint64_t strides[2] = {(cuuint64_t)s.d * 2, (cuuint64_t)s.L * s.d * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)kBM, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int D>
cudaError_t launch_state(const void* K, const void* V, const Shape& s, const TcPlan& p, float scale, char* ws,
                         int32_t* status, cudaStream_t stream) {
  CUtensorMap mk, mv;
  if (!make_map(&mk, K, s) || !make_map(&mv, V, s)) return cudaErrorInvalidValue;
  StateParams prm{};
  prm.key_ref = reinterpret_cast<const float*>(ws);
  prm.omega_img = reinterpret_cast<const uint8_t*>(ws + p.off_omega_img);
  prm.partS = reinterpret_cast<float*>(ws + p.off_partS);
  prm.counters = reinterpret_cast<uint32_t*>(ws + p.off_counters);
  prm.state_img = reinterpret_cast<uint8_t*>(ws + p.off_state_img);
  prm.status = status;
  prm.L = s.L;
  prm.m = s.m;
  prm.n_split = p.n_split;
  prm.tiles_per_split = p.tiles_per_split;
  prm.scale = scale;
  const size_t smem = StateCfg<D>::kSmem;
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(state_kernel<D>), smem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.n_split, p.n_fb, s.BH());
  state_kernel<D><<<grid, kThreads, smem, stream>>>(mk, mv, prm);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_output(const void* Q, void* O, const Shape& s, const TcPlan& p, float scale, char* ws,
                          int32_t* status, cudaStream_t stream) {
  CUtensorMap mq, mo;
  if (!make_map(&mq, Q, s) || !make_map(&mo, O, s)) return cudaErrorInvalidValue;
  OutParams prm{};
  prm.omega_img = reinterpret_cast<const uint8_t*>(ws + p.off_omega_img);
  prm.state_img = reinterpret_cast<const uint8_t*>(ws + p.off_state_img);
  prm.status = status;
  prm.L = s.L;
  prm.m = s.m;
  prm.tiles_per_cta = p.out_tiles_per_cta;
  prm.scale = scale;
  const size_t smem = OutCfg<D>::kSmem;
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(output_kernel<D>), smem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.out_ctas, s.BH());
  output_kernel<D><<<grid, kThreads, smem, stream>>>(mq, mo, prm);
  return cudaGetLastError();
}

}  // namespace

bool tc_supported(bool causal, int d, int m, bool bf16) {
  if (!bf16 || causal) return false;
  return d == 64 && (m == 128 || m == 256);
}

size_t tc_workspace_bytes(bool causal, const Shape& s) {
  (void)causal;
  return tc_plan(s).bytes;
}

cudaError_t tc_state(bool causal, const void* K, const void* V, const float* omega, float scale, const Shape& s,
                     void* ws, int32_t* status, cudaStream_t stream) {
  if (causal) return cudaErrorNotSupported;
  const TcPlan p = tc_plan(s);
  char* w = static_cast<char*>(ws);
  cudaError_t e = launch_prep(omega, s.m, s.d, reinterpret_cast<float*>(w),
                              reinterpret_cast<uint8_t*>(w + p.off_omega_img), stream);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(w + p.off_counters, 0, (size_t)s.BH() * p.n_fb * sizeof(uint32_t), stream);
  if (e != cudaSuccess) return e;
  return launch_state<64>(K, V, s, p, scale, w, status, stream);
}

cudaError_t tc_output(bool causal, const void* Q, const void* K, const void* V, void* O, const float* omega,
                      float scale, const Shape& s, void* ws, int32_t* status, cudaStream_t stream) {
  (void)K;
  (void)V;
  (void)omega;
  if (causal) return cudaErrorNotSupported;
  const TcPlan p = tc_plan(s);
  return launch_output<64>(Q, O, s, p, scale, static_cast<char*>(ws), status, stream);
}

}  // namespace favor
