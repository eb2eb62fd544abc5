// Tensor-core (tcgen05) bidirectional FAVOR+ for d = 128: one 128-feature
// block of Omega per CTA ("feature-sliced").
//
// "Performer — Rethinking Attention with Performers" (digest), §Key
// equations: phi(K)^T [V | 1] is formed first, then phi(Q) times it, then
// the row-wise divide.  At d = 128 one 128-token tile of Q, K or V is 32 KB
// and one 128-feature block of Omega another 32 KB, so a CTA cannot hold
// Omega, the state and a pipeline of tiles for m up to 512 (Omega alone is
// 128 KB, the bf16 state 144 KB at m = 512).  Each CTA therefore owns one
// feature block:
//
//   state kernel  grid (splits x blocks, heads): P = K Omega_b^T (fp16), the
//                 features exp(l - R) written over the consumed K tile, then
//                 S~_b += phi(K)_b^T [V | 1] (N = d + 16: the normaliser rides
//                 in a ones block stored right after each V tile).  The last
//                 CTA of (head, block) adds the splits in order into the bf16
//                 state image.
//   output kernel thread-block clusters of m / 128 CTAs, as many as can be
//                 resident, each an even share of the (head, tile) list; CTA
//                 r holds block r of Omega and of the head's state.
//                 Each computes phi(Q)_r with its own exact row maximum c_r
//                 and the partial output O_r = phi(Q)_r S~_r (numerator and
//                 normaliser).  The partials meet in distributed shared
//                 memory: CTA r finalises columns [r d/n, (r+1) d/n) as
//                   sum_j 2^(c_j - c) O_j / sum_j 2^(c_j - c) z_j,  c = max_j c_j
//                 summed in rank order ("From Performer to Linear Attention",
//                 §Simple Derivation: a per-query constant cancels, so each
//                 partial may carry its own).
//
// Warp roles as in the d = 64 kernels: warp 0 TMA, warp 1 MMA issue (one
// thread), warps 2-3 rewrite each input tile as fp16 (and take the squared
// key norms), warps 4-11 two epilogue warpgroups splitting a tile's columns.
// Every wait is bounded; a wait that runs out raises the CTA's abort flag and
// records FAVOR_ERR_TIMEOUT.
#include "tc.cuh"
#include "tc_util.cuh"

namespace favor {
namespace {

using namespace tc;

constexpr int kD = 128;                 // head dimension of this family
constexpr int kTile = kD * kBM * 2;     // one Q, K or V tile: two 64-column swizzle atoms
constexpr int kGN = kD + 16;            // columns of [V | 1] and of the state (normaliser at column kD)
constexpr int kThreads = 384;           // warps 0 TMA, 1 MMA, 2-3 fp16 rewrite, 4-11 epilogue

// ---------------------------------------------------------------------------
// workspace
// ---------------------------------------------------------------------------
struct FsPlan {
  int n_fb, n_tiles;
  int tiles_per_split, n_split;   // state partials: splits per (head, feature block)
  size_t off_omega_img, off_counters, off_partS, off_state_img, bytes;
};

FsPlan fs_plan(const Shape& s) {
  FsPlan p{};
  const int BH = s.BH();
  p.n_fb = s.m / kFB;
  p.n_tiles = (s.L + kBM - 1) / kBM;
  const int sp = pick_split(BH * p.n_fb, p.n_tiles, sm_count());
  p.tiles_per_split = (p.n_tiles + sp - 1) / sp;
  p.n_split = (p.n_tiles + p.tiles_per_split - 1) / p.tiles_per_split;
  size_t off = align_up(kWsHeader, 1024);
  p.off_omega_img = off;   // fp16 Omega [d/64 atoms][m rows][128 B], swizzled
  off = align_up(off + (size_t)s.m * s.d * 2, 1024);
  p.off_counters = off;    // [BH][n_fb] merge counters
  off = align_up(off + (size_t)BH * p.n_fb * sizeof(uint32_t), 1024);
  p.off_partS = off;       // fp32 [BH][n_fb][n_split][d+1][128]
  off = align_up(off + (size_t)BH * p.n_fb * p.n_split * (s.d + 1) * kFB * sizeof(float), 1024);
  p.off_state_img = off;   // bf16 [BH][m/64][d+16][128 B], normaliser in row d
  off = align_up(off + (size_t)BH * s.m * (s.d + 16) * 2, 1024);
  p.bytes = off;
  return p;
}

// Causal: superchunks of tiles_per_sc tiles, one cluster each; the key-state
// kernel writes the partials of every superchunk but the last in sub_per_sc
// sub-splits; the clusters exchange partial outputs in shared memory.
struct FsCausalPlan {
  int n_fb, n_tiles;
  int tiles_per_sc, n_sc, sub_per_sc, tiles_per_split, n_split;
  size_t off_omega_img, off_partS, off_pre, bytes;
};


FsCausalPlan fsc_plan(const Shape& s) {
  FsCausalPlan p{};
  const int BH = s.BH();
  const int sms = sm_count();
  p.n_fb = s.m / kFB;
  p.n_tiles = (s.L + kBM - 1) / kBM;
  const int sc = pick_split(BH, p.n_tiles, max(1, sms / p.n_fb));
  p.tiles_per_sc = (p.n_tiles + sc - 1) / sc;
  p.n_sc = (p.n_tiles + p.tiles_per_sc - 1) / p.tiles_per_sc;
  // sub-splits of each earlier superchunk (dividing it) for the state kernel
  int best_k = 1;
  long best_cost = -1;
  for (int k = 1; k <= p.tiles_per_sc; ++k) {
    if (p.tiles_per_sc % k) continue;
    const long ctas = (long)BH * p.n_fb * (p.n_sc - 1) * k;
    const long cost = ((ctas + sms - 1) / sms) * (p.tiles_per_sc / k + kCtaOverheadTiles);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best_k = k;
    }
  }
  p.sub_per_sc = best_k;
  p.tiles_per_split = p.tiles_per_sc / best_k;
  p.n_split = (p.n_sc - 1) * best_k;
  size_t off = align_up(kWsHeader, 1024);
  p.off_omega_img = off;
  off = align_up(off + (size_t)s.m * s.d * 2, 1024);
  p.off_partS = off;   // fp32 [BH][n_fb][max(n_split, 1)][d+1][128]
  off = align_up(off + (size_t)BH * p.n_fb * max(p.n_split, 1) * (s.d + 1) * kFB * sizeof(float), 1024);
  p.off_pre = off;     // fp32 [BH][n_fb][n_sc][d+1][128]: each superchunk's initial state
  off = align_up(off + (size_t)BH * p.n_fb * p.n_sc * (s.d + 1) * kFB * sizeof(float), 1024);
  p.bytes = off;
  return p;
}

// ---------------------------------------------------------------------------
// state kernel
// ---------------------------------------------------------------------------
struct FsStateParams {
  const float* key_ref;
  const uint8_t* omega_img;
  float* partS;
  uint32_t* counters;
  uint8_t* state_img;
  int32_t* status;
  int L, m, n_fb, n_split, tiles_per_split;
  int merge;                  // bidirectional: the last CTA of (head, block) merges the splits
  float scale;
};

struct FsStateCfg {
  static constexpr int NS = 2;                                  // pipeline stages
  static constexpr int kOmega = 0;                              // this block: [2 atoms][128 rows][128 B]
  static constexpr int kStage = kOmega + 2 * kAtom;
  static constexpr int kStageBytes = kTile + kTile + kAtom;     // K (then phi(K)), V, ones atom
  static constexpr int kNorm = kStage + NS * kStageBytes;       // [NS][128] squared key norms
  static constexpr int kBars = kNorm + NS * kBM * 4;
  static constexpr int kSmem = kBars + 256 + 1024;
};
static_assert(FsStateCfg::kSmem <= 232448, "shared memory");

template <int FM>
__global__ void __launch_bounds__(kThreads, 1) fs_state_kernel(const __grid_constant__ CUtensorMap mapK,
                                                               const __grid_constant__ CUtensorMap mapV,
                                                               FsStateParams prm) {
  using C = FsStateCfg;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::kBars);
  uint64_t* full = bars;                     // [NS] K and V landed
  uint64_t* empty = full + C::NS;            // [NS] stage consumed by the state MMA
  uint64_t* kn_full = empty + C::NS;         // [NS] K in fp16, norms written
  uint64_t* phi_full = kn_full + C::NS;      // [NS] phi(K) written over K
  uint64_t* p_full = phi_full + C::NS;       // [2] projection buffers
  uint64_t* p_free = p_full + 2;             // [2]
  uint64_t* setup_bar = p_free + 2;
  uint64_t* done_bar = setup_bar + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* is_last = const_cast<int*>(abort_flag) + 1;
  float* norm_s = reinterpret_cast<float*>(sm + C::kNorm);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int fb = blockIdx.x % prm.n_fb, split = blockIdx.x / prm.n_fb, bh = blockIdx.y;
  const int tile0 = split * prm.tiles_per_split;
  const int n_tiles_total = (prm.L + kBM - 1) / kBM;
  const int n_tiles = min(prm.tiles_per_split, n_tiles_total - tile0);
  const WaitCtx wctx{abort_flag, prm.status};
  constexpr uint32_t S_COL = 256;             // state accumulator; projections at columns 0 and 128
  auto stage = [&](int st) { return sm + C::kStage + st * C::kStageBytes; };

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
      mbar_init(&kn_full[i], kNormWarps);
      mbar_init(&phi_full[i], kEpiWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&p_full[i], 1);
      mbar_init(&p_free[i], kEpiWarps);
    }
    mbar_init(setup_bar, 1);
    mbar_init(done_bar, 1);
    *abort_flag = 0;
    *is_last = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (warp >= 4) {
    for (int st = 0; st < C::NS; ++st) fill_ones_atom(stage(st) + 2 * kTile, kEpiTid0, kEpiThreads);
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
      mbar_arrive_expect_tx(setup_bar, 2 * kAtom);
      for (int a = 0; a < 2; ++a)
        bulk_load(sm + C::kOmega + a * kAtom, prm.omega_img + ((size_t)a * prm.m + fb * kFB) * 128, kAtom,
                  setup_bar);
      int last_issue[C::NS];
      for (int i = 0; i < C::NS; ++i) last_issue[i] = -1;
      for (int i = 0; i < n_tiles; ++i) {
        const int st = i % C::NS;
        if (i >= C::NS && !mbar_wait(&empty[st], ((i / C::NS) - 1) & 1, wctx)) break;
        mbar_arrive_expect_tx(&full[st], 2 * kTile);
        const int row = (tile0 + i) * kBM;
        for (int a = 0; a < 2; ++a) {
          tma_load_3d(stage(st) + a * kAtom, &mapK, a * 64, row, bh, &full[st]);
          tma_load_3d(stage(st) + kTile + a * kAtom, &mapV, a * 64, row, bh, &full[st]);
        }
        last_issue[st] = i;
      }
      for (int st = 0; st < C::NS; ++st)
        if (last_issue[st] >= 0) mbar_wait(&full[st], (last_issue[st] / C::NS) & 1, wctx);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t id_proj = idesc_f16(kBM, kFB, false, false);
      constexpr uint32_t id_state = idesc_bf16(kFB, kGN, true, true);
      const uint32_t omega_a = smem_addr(sm + C::kOmega);
      bool ok = mbar_wait(setup_bar, 0, wctx);
      auto ready = [](uint64_t* bar, int parity) { return mbar_test_wait(smem_addr(bar), parity & 1); };
      // event-driven: the projection of tile pi (into buffer pi & 1) once K is
      // in fp16 and the buffer's previous tile was copied out; the state step
      // of tile si once its features are written; projections first
      Watchdog wd(wctx);
      int pi = 0, si = 0;
      while (ok && si < n_tiles) {
        bool progress = false;
        if (pi < n_tiles) {
          const int st = pi % C::NS, pb = pi & 1;
          if (ready(&kn_full[st], pi / C::NS) && (pi < 2 || ready(&p_free[pb], (pi >> 1) - 1))) {
            tc_fence_after();
            const uint64_t a0 = sdesc(smem_addr(stage(st)), 16, 1024);
            const uint64_t b0 = sdesc(omega_a, 16, 1024);
#pragma unroll
            for (int k = 0; k < kD / 16; ++k)
              mma_bf16(tmem + pb * kFB, dadd(a0, kstep_k(k, kAtom)), dadd(b0, kstep_k(k, kAtom)), id_proj, k > 0);
            mma_commit(&p_full[pb]);
            ++pi;
            progress = true;
          }
        }
        if (si < pi) {
          const int st = si % C::NS;
          if (ready(&phi_full[st], si / C::NS)) {
            tc_fence_after();
            // A = phi(K)^T: features contiguous (M-major), two 64-feature atoms;
            // B = [V | 1]: V's two atoms and the ones atom, kAtom apart
            const uint64_t a0 = sdesc(smem_addr(stage(st)), kAtom, 1024);
            const uint64_t b0 = sdesc(smem_addr(stage(st) + kTile), kAtom, 1024);
#pragma unroll
            for (int k = 0; k < kBM / 16; ++k)
              mma_bf16(tmem + S_COL, dadd(a0, kstep_mn(k)), dadd(b0, kstep_mn(k)), id_state, (si > 0) || (k > 0));
            mma_commit(&empty[st]);
            ++si;
            progress = true;
          }
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
      const int st = i % C::NS;
      if (!mbar_wait(&full[st], (i / C::NS) & 1, wctx)) break;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int r = (warp - 2) * 64 + lane + 32 * j;
        norm_s[st * kBM + r] = tile_row_sq_to_f16<kD>(stage(st), r);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&kn_full[st]);
    }
  } else {
    // ---------------- epilogue: warpgroup w takes columns 64w .. 64w + 63 ----------------
    const int wg = (warp - 4) >> 2;
    const int q = warp & 3;
    const int t = q * 32 + lane;                   // token row of P, feature row of S~
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    const int col0 = wg * 64;
    float R, W_unused;
    key_reference(prm.key_ref, prm.m, &R, &W_unused);
    const float c1 = feature_c1<FM>(prm.scale);
    const float hs2 = 0.5f * prm.scale * prm.scale;
    bool ok = true;
    for (int i = 0; ok && i < n_tiles; ++i) {
      const int st = i % C::NS, pb = i & 1;
      if (!mbar_wait(&kn_full[st], (i / C::NS) & 1, wctx)) { ok = false; break; }
      // rows past L get 2^-inf = 0
      const bool valid = (tile0 + i) * kBM + t < prm.L;
      const float bias = !valid ? INFINITY : (FM == FAVOR_FM_PRF ? (hs2 * norm_s[st * kBM + t] + R) * kLog2e : 0.f);
      if (!mbar_wait(&p_full[pb], (i >> 1) & 1, wctx)) { ok = false; break; }
      tc_fence_after();
      uint32_t x[64];
      tmem_ld64(tmem + lane_off + pb * kFB + col0, x);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_free[pb]);
      feature_pack<FM>(x, c1, bias);
      // the projection has read K: its tile takes phi(K) (feature atom = warpgroup)
      store_row<32>(smem_addr(stage(st)), kAtom, t, col0, x);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&phi_full[st]);
    }
    // final partial state: lane f = feature f; the warpgroups take alternate
    // 32-column groups, warpgroup 1 the normaliser column
    const bool done = mbar_wait(done_bar, 0, wctx);
    tc_fence_after();
    if (done && !*abort_flag) {
      float* dst = prm.partS + ((((size_t)bh * prm.n_fb + fb) * prm.n_split + split) * (kD + 1)) * kFB;
      const uint32_t s_col = tmem + lane_off + S_COL;
#pragma unroll
      for (int cb = 0; cb < kD / 32; ++cb) {
        if ((cb & 1) != wg) continue;
        uint32_t v[32];
        tmem_ld32(s_col + cb * 32, v);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) dst[(size_t)(cb * 32 + j) * kFB + t] = __uint_as_float(v[j]);
      }
      if (wg == 1) {
        uint32_t z[8];
        tmem_ld8(s_col + kD, z);
        tmem_ld_wait();
        dst[(size_t)kD * kFB + t] = __uint_as_float(z[0]);
      }
    }
    tc_fence_before();
    if (prm.merge) {
      named_bar(1, kEpiThreads);
      if (threadIdx.x == kEpiTid0) {
        __threadfence();
        const uint32_t old = atomicAdd(&prm.counters[bh * prm.n_fb + fb], 1u);
        *is_last = (old == (uint32_t)(prm.n_split - 1)) ? 1 : 0;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
  // the last CTA of (head, block) adds the splits' partials (fixed split
  // order) into the bf16 state image; item = (row n, 4 consecutive features)
  if (*is_last) {
    __threadfence();
    uint8_t* img = prm.state_img + (size_t)bh * prm.m * kGN * 2;
    constexpr int NG = kFB / 4;
    constexpr int kItems = kGN * NG;
    constexpr int kBatch = 6;
    const float* base = prm.partS + ((size_t)bh * prm.n_fb + fb) * prm.n_split * (kD + 1) * kFB;
    for (int e0 = threadIdx.x; e0 < kItems; e0 += kBatch * kThreads) {
      float4 acc[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int p = 0; p < prm.n_split; ++p) {
        float4 v[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          const int e = e0 + u * kThreads;
          const int g = e % NG, n = e / NG;
          v[u] = (e < kItems && n <= kD)
                     ? *reinterpret_cast<const float4*>(base + ((size_t)p * (kD + 1) + n) * kFB + g * 4)
                     : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          acc[u].x += v[u].x;
          acc[u].y += v[u].y;
          acc[u].z += v[u].z;
          acc[u].w += v[u].w;
        }
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int e = e0 + u * kThreads;
        if (e >= kItems) break;
        const int g = e % NG, n = e / NG;
        const int f = fb * kFB + g * 4;
        const int atom = f >> 6, cc = f & 63;
        const size_t off = ((size_t)atom * kGN + n) * 128 + (((cc >> 3) ^ (n & 7)) << 4) + (cc & 7) * 2;
        *reinterpret_cast<uint2*>(img + off) = make_uint2(pack_bf16(acc[u].x, acc[u].y), pack_bf16(acc[u].z, acc[u].w));
      }
    }
    if (threadIdx.x == 0) prm.counters[bh * prm.n_fb + fb] = 0;
  }
}

// ---------------------------------------------------------------------------
// output kernel: clusters of NC CTAs (NC = m / 128), each an even share of the
// (head, tile) list; CTA rank r owns feature block r and finalises output
// columns [r W, (r + 1) W), W = d / NC.
// ---------------------------------------------------------------------------
struct FsOutParams {
  const uint8_t* omega_img;
  const uint8_t* state_img;
  __nv_bfloat16* O;
  int32_t* status;
  int L, m;
  int n_heads;             // B H: the clusters split the (head, tile) list evenly
  float scale;
};

template <int NC>
struct FsOutCfg {
  static constexpr int W = kD / NC;                       // output columns finalised per CTA
  static constexpr int RB = 2 * W + 16;                   // landing row bytes: W bf16 numerators, fp32 normaliser and reference, pad
  static constexpr int kLandTile = (NC - 1) * kBM * RB;   // one tile's rows from the other CTAs
  static constexpr int NSQ = 2;                           // Q stages (Q, then phi(Q) in place)
  static constexpr int kOmega = 0;                        // [2 atoms][128 feature rows][128 B]
  static constexpr int kState = kOmega + 2 * kAtom;       // [2 atoms][kGN rows][128 B]
  static constexpr int kQ = kState + 2 * kGN * 128;
  static constexpr int kXmax = kQ + NSQ * kTile;          // [tile parity][warpgroup][128] row maxima
  static constexpr int kLand = kXmax + 2 * 2 * kBM * 4;   // [tile parity][NC - 1 sources][128][RB]
  static constexpr int kBars = kLand + 2 * kLandTile;
  static constexpr int kSmem = kBars + 256 + 1024;
};
static_assert(FsOutCfg<4>::kSmem <= 232448 && FsOutCfg<2>::kSmem <= 232448, "shared memory");
static_assert((2 * kGN * 128) % 1024 == 0 && (kGN * 128) % 1024 == 0, "operand alignment");

template <int NC, int FM>
__global__ void __launch_bounds__(kThreads, 1) fs_output_kernel(const __grid_constant__ CUtensorMap mapQ,
                                                                FsOutParams prm) {
  using C = FsOutCfg<NC>;
  constexpr int W = C::W;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::kBars);
  uint64_t* q_full = bars;                  // [2] Q landed
  uint64_t* q_empty = q_full + 2;           // [2] stage consumed (projection and output MMA)
  uint64_t* qn_full = q_empty + 2;          // [2] Q in fp16
  uint64_t* p_full = qn_full + 2;           // [2] projection buffers
  uint64_t* p_free = p_full + 2;            // [2]
  uint64_t* phi_full = p_free + 2;          // [2] phi(Q) written over Q
  uint64_t* o_full = phi_full + 2;
  uint64_t* o_free = o_full + 1;
  uint64_t* land_full = o_free + 1;         // [tile parity] the other CTAs' partials for my columns have landed
  uint64_t* land_free = land_full + 2;      // [tile parity][4] owner r has read my partial of that parity
  uint64_t* setup_bar = land_free + 8;
  uint64_t* done_bar = setup_bar + 1;
  uint64_t* img_full = done_bar + 1;        // phase k: the k-th head's state block landed
  uint64_t* img_free = img_full + 1;        // phase k: the k-th head's last output MMA is complete
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(img_free + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* xmax = reinterpret_cast<float*>(sm + C::kXmax);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = NC > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  // this cluster's tiles: the contiguous range [g0, g1) of the (head, tile)
  // list, which may cross from one head into the next (each CTA reloads its
  // block of the state)
  const int nt = (prm.L + kBM - 1) / kBM;
  const long long total = (long long)prm.n_heads * nt;
  const int n_cl = (int)gridDim.x / NC, cl = (int)blockIdx.x / NC;
  const int g0 = range_first(total, cl, n_cl);
  const int n_tiles = range_first(total, cl + 1, n_cl) - g0;
  const int h0 = g0 / nt;
  const int n_heads = n_tiles > 0 ? (g0 + n_tiles - 1) / nt - h0 + 1 : 0;
  auto head_of = [&](int i) { return (g0 + i) / nt; };
  auto tile_of = [&](int i) { return (g0 + i) - head_of(i) * nt; };
  const WaitCtx wctx{abort_flag, prm.status};
  constexpr uint32_t O_COL = 256;            // output accumulator; projections at columns 0 and 128
  auto qstage = [&](int st) { return sm + C::kQ + st * kTile; };

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);
      mbar_init(&qn_full[i], kNormWarps);
      mbar_init(&p_full[i], 1);
      mbar_init(&p_free[i], kEpiWarps);
      mbar_init(&phi_full[i], kEpiWarps);
    }
    mbar_init(o_full, 1);
    mbar_init(o_free, kEpiWarps);
    // the partials arrive by st.async, counted in bytes: one arrival per
    // phase (the expected byte count, posted here for tiles 0 and 1 and by
    // the finalising warpgroup for tile j + 2 once tile j is read)
    for (int i = 0; i < 2; ++i) mbar_init(&land_full[i], 1);
    for (int i = 0; i < 8; ++i) mbar_init(&land_free[i], 4);   // owner i % 4's finalising warps
    mbar_init(setup_bar, 1);
    mbar_init(done_bar, 1);
    mbar_init(img_full, 1);
    mbar_init(img_free, 1);
    *abort_flag = 0;
    fence_barrier_init();
    if (NC > 1)
      for (int i = 0; i < 2; ++i) mbar_arrive_expect_tx(&land_full[i], C::kLandTile);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (NC > 1) cluster_sync();   // every CTA's barriers exist before any remote arrival
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      prefetch_tmap(&mapQ);
      constexpr uint32_t sb = 2 * kGN * 128;
      mbar_arrive_expect_tx(setup_bar, 2 * kAtom);
      for (int a = 0; a < 2; ++a)
        bulk_load(sm + C::kOmega + a * kAtom, prm.omega_img + ((size_t)a * prm.m + rank * kFB) * 128, kAtom,
                  setup_bar);
      // head k's block of the state goes in once head k - 1's last output MMA is complete
      auto load_head = [&](int k) {
        mbar_arrive_expect_tx(img_full, sb);
        bulk_load(sm + C::kState, prm.state_img + ((size_t)(h0 + k) * (prm.m / 64) + 2 * rank) * kGN * 128, sb,
                  img_full);
      };
      int ni = 0;
      if (n_heads > 0) load_head(ni++);
      Watchdog wd(wctx);
      int nq = 0;
      bool ok = true;
      while (ok && (nq < n_tiles || ni < n_heads)) {
        bool progress = false;
        if (nq < n_tiles && (nq < 2 || mbar_test_wait(smem_addr(&q_empty[nq & 1]), ((nq >> 1) - 1) & 1))) {
          const int st = nq & 1;
          mbar_arrive_expect_tx(&q_full[st], kTile);
          for (int a = 0; a < 2; ++a)
            tma_load_3d(qstage(st) + a * kAtom, &mapQ, a * 64, tile_of(nq) * kBM, head_of(nq), &q_full[st]);
          ++nq;
          progress = true;
        }
        if (ni < n_heads && mbar_test_wait(smem_addr(img_free), (ni - 1) & 1)) {
          load_head(ni++);
          progress = true;
        }
        if (progress) wd.progress();
        else ok = wd.idle();
      }
      for (int x = max(0, nq - 2); x < nq; ++x) mbar_wait(&q_full[x & 1], (x >> 1) & 1, wctx);
      if (ni > 0) mbar_wait(img_full, (ni - 1) & 1, wctx);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t id_proj = idesc_f16(kBM, kFB, false, false);
      constexpr uint32_t id_out = idesc_bf16(kBM, kGN, false, false);
      const uint32_t omega_a = smem_addr(sm + C::kOmega), state_a = smem_addr(sm + C::kState);
      bool ok = mbar_wait(setup_bar, 0, wctx);
      auto ready = [](uint64_t* bar, int parity) { return mbar_test_wait(smem_addr(bar), parity & 1); };
      // event-driven: projection of tile pi into buffer pi & 1; the output
      // step of tile oi once its features are written and the previous
      // tile's output was copied out; projections first
      Watchdog wd(wctx);
      int pi = 0, oi = 0;
      while (ok && oi < n_tiles) {
        bool progress = false;
        if (pi < n_tiles) {
          const int st = pi & 1;
          if (ready(&qn_full[st], pi >> 1) && (pi < 2 || ready(&p_free[st], (pi >> 1) - 1))) {
            tc_fence_after();
            const uint64_t a0 = sdesc(smem_addr(qstage(st)), 16, 1024);
            const uint64_t b0 = sdesc(omega_a, 16, 1024);
#pragma unroll
            for (int k = 0; k < kD / 16; ++k)
              mma_bf16(tmem + st * kFB, dadd(a0, kstep_k(k, kAtom)), dadd(b0, kstep_k(k, kAtom)), id_proj, k > 0);
            mma_commit(&p_full[st]);
            ++pi;
            progress = true;
          }
        }
        if (oi < pi) {
          const int st = oi & 1;
          if (ready(&phi_full[st], oi >> 1) && ready(img_full, head_of(oi) - h0) &&
              (oi == 0 || ready(o_free, oi - 1))) {
            tc_fence_after();
            const uint64_t a0 = sdesc(smem_addr(qstage(st)), 16, 1024);
            const uint64_t b0 = sdesc(state_a, 16, 1024);
#pragma unroll
            for (int k = 0; k < kFB / 16; ++k)
              mma_bf16(tmem + O_COL, dadd(a0, kstep_k(k, kAtom)), dadd(b0, kstep_k(k, kGN * 128)), id_out, k > 0);
            mma_commit(o_full);
            mma_commit(&q_empty[st]);
            // the head's last tile: its state block may be replaced
            if (oi == n_tiles - 1 || head_of(oi + 1) != head_of(oi)) mma_commit(img_free);
            ++oi;
            progress = true;
          }
        }
        if (progress) wd.progress();
        else ok = wd.idle();
      }
      mma_commit(done_bar);
      mbar_wait(done_bar, 0, wctx);
    }
  } else if (warp < 2 + kNormWarps) {
    // Q rewritten as fp16 for the projection
    for (int i = 0; i < n_tiles; ++i) {
      const int st = i & 1;
      if (!mbar_wait(&q_full[st], (i >> 1) & 1, wctx)) break;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int r = (warp - 2) * 64 + lane + 32 * j;
        (void)tile_row_sq_to_f16<kD>(qstage(st), r);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&qn_full[st]);
    }
  } else {
    // ---------------- epilogue: warpgroup w takes columns 64w .. 64w + 63 ----------------
    const int wg = (warp - 4) >> 2;
    const int q = warp & 3;
    const int t = q * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    const int col0 = wg * 64;
    const float c1 = feature_c1<FM>(prm.scale);
    // the warpgroup holding my own output columns (NC > 1)
    const int wg_fin = (rank * W) / 64;
    bool ok = true;

    // phi(Q) of tile i over the stage's Q; returns this CTA's row reference
    // (log2 units)
    auto features = [&](int i) {
      const int st = i & 1;
      if (ok) ok = mbar_wait(&p_full[st], (i >> 1) & 1, wctx);
      tc_fence_after();
      uint32_t x[64];
      tmem_ld64(tmem + lane_off + st * kFB + col0, x);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_free[st]);
      float bias = 0.f;
      if constexpr (FM == FAVOR_FM_PRF) {
        float pm = -INFINITY;
#pragma unroll
        for (int j = 0; j < 64; ++j) pm = fmaxf(pm, __uint_as_float(x[j]));
        float* xm = xmax + (i & 1) * 2 * kBM;
        xm[wg * kBM + t] = pm;
        named_bar(2, kEpiThreads);
        bias = fmaxf(xm[t], xm[kBM + t]) * c1;
      }
      if (ok) {
        feature_pack<FM>(x, c1, bias);
        store_row<32>(smem_addr(qstage(st)), kAtom, t, col0, x);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&phi_full[st]);
      return bias;
    };

    // the output of tile j: partials of the other CTAs' columns sent to them,
    // my columns finalised from all partials
    auto output = [&](int j, float bias) {
      const bool have = ok && mbar_wait(o_full, j & 1, wctx);
      tc_fence_after();
      uint32_t v[64], z[8];
      tmem_ld32_at<0>(tmem + lane_off + O_COL + col0, v);
      tmem_ld32_at<32>(tmem + lane_off + O_COL + col0 + 32, v);
      tmem_ld8(tmem + lane_off + O_COL + kD, z);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(o_free);
      const float den_own = __uint_as_float(z[0]);
      const int row = tile_of(j) * kBM + t;
      const bool valid = row < prm.L;
      __nv_bfloat16* orow = prm.O + ((size_t)head_of(j) * prm.L + (valid ? row : 0)) * kD;
      if constexpr (NC == 1) {
        if (have && valid) {
          if (!(den_own > 0.f) || !isfinite(den_own)) report_status(prm.status, FAVOR_ERR_NONFINITE);
          const float inv = __fdividef(1.0f, den_own);
#pragma unroll
          for (int c = 0; c < 64; c += 8)
            *reinterpret_cast<uint4*>(orow + col0 + c) =
                make_uint4(pack_bf16(__uint_as_float(v[c]) * inv, __uint_as_float(v[c + 1]) * inv),
                           pack_bf16(__uint_as_float(v[c + 2]) * inv, __uint_as_float(v[c + 3]) * inv),
                           pack_bf16(__uint_as_float(v[c + 4]) * inv, __uint_as_float(v[c + 5]) * inv),
                           pack_bf16(__uint_as_float(v[c + 6]) * inv, __uint_as_float(v[c + 7]) * inv));
        }
      } else {
        // send: every slice of my columns owned by another CTA, into the
        // tile parity's landing rows once the owner has read the ones two
        // tiles back; bf16 numerators, fp32 normaliser and reference
        const int par = j & 1;
#pragma unroll
        for (int sl = 0; sl < 64 / W; ++sl) {
          const int owner = (col0 + sl * W) / W;
          if (owner == rank) continue;
          if (ok && j >= 2) ok = mbar_wait_cluster(&land_free[par * 4 + owner], ((j >> 1) - 1) & 1, wctx);
          const int slot = rank < owner ? rank : rank - 1;
          const uint32_t dst = map_to_rank(
              smem_addr(sm + C::kLand + par * C::kLandTile + ((size_t)slot * kBM + t) * C::RB), static_cast<uint32_t>(owner));
          const uint32_t mb = map_to_rank(smem_addr(&land_full[par]), static_cast<uint32_t>(owner));
          if (ok) {
#pragma unroll
            for (int c = 0; c < W; c += 8)
              st_async_v4(dst + c * 2, pack_bf16(__uint_as_float(v[sl * W + c]), __uint_as_float(v[sl * W + c + 1])),
                          pack_bf16(__uint_as_float(v[sl * W + c + 2]), __uint_as_float(v[sl * W + c + 3])),
                          pack_bf16(__uint_as_float(v[sl * W + c + 4]), __uint_as_float(v[sl * W + c + 5])),
                          pack_bf16(__uint_as_float(v[sl * W + c + 6]), __uint_as_float(v[sl * W + c + 7])), mb);
            st_async_v4(dst + W * 2, __float_as_uint(den_own), __float_as_uint(bias), 0u, 0u, mb);
          }
        }
        if (wg == wg_fin) {
          // finalise my columns: every partial rescaled to the largest
          // reference; mine first, then the others in rank order
          if (ok) ok = mbar_wait(&land_full[par], (j >> 1) & 1, wctx);
          const uint8_t* land = sm + C::kLand + par * C::kLandTile;
          float bmax = bias;
          for (int sl = 0; sl < NC - 1; ++sl)
            bmax = fmaxf(bmax, *reinterpret_cast<const float*>(land + ((size_t)sl * kBM + t) * C::RB + 2 * W + 4));
          const bool hi = (rank * W - col0) != 0;   // my slice is the upper half of this thread's 64 columns
          const float sc_own = ex2(bias - bmax);
          float acc[W];
#pragma unroll
          for (int c = 0; c < W; ++c) acc[c] = sc_own * __uint_as_float(W == 64 ? v[c] : (hi ? v[(32 + c) & 63] : v[c]));
          float den = sc_own * den_own;
          for (int sl = 0; sl < NC - 1; ++sl) {
            const uint8_t* lr = land + ((size_t)sl * kBM + t) * C::RB;
            const float2 dr = *reinterpret_cast<const float2*>(lr + 2 * W);   // normaliser, reference
            const float sc = ex2(dr.y - bmax);
#pragma unroll
            for (int c = 0; c < W; c += 8) {
              const uint4 p4 = *reinterpret_cast<const uint4*>(lr + c * 2);
              const uint32_t w4[4] = {p4.x, p4.y, p4.z, p4.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                acc[c + 2 * e] = fmaf(sc, __uint_as_float(w4[e] << 16), acc[c + 2 * e]);
                acc[c + 2 * e + 1] = fmaf(sc, __uint_as_float(w4[e] & 0xFFFF0000u), acc[c + 2 * e + 1]);
              }
            }
            den = fmaf(sc, dr.x, den);
          }
          // the rows are read: re-arm this parity for tile j + 2, then let
          // their writers send it
          if (threadIdx.x == kEpiTid0 + kBM * wg_fin && ok) mbar_arrive_expect_tx(&land_full[par], C::kLandTile);
          __syncwarp();
          if (lane == 0)
            for (int src = 0; src < NC; ++src)
              if (src != rank)
                mbar_arrive_remote(map_to_rank(smem_addr(&land_free[par * 4 + rank]), static_cast<uint32_t>(src)));
          if (have && valid) {
            if (!(den > 0.f) || !isfinite(den)) report_status(prm.status, FAVOR_ERR_NONFINITE);
            const float inv = __fdividef(1.0f, den);
#pragma unroll
            for (int c = 0; c < W; c += 8)
              *reinterpret_cast<uint4*>(orow + rank * W + c) =
                  make_uint4(pack_bf16(acc[c] * inv, acc[c + 1] * inv), pack_bf16(acc[c + 2] * inv, acc[c + 3] * inv),
                             pack_bf16(acc[c + 4] * inv, acc[c + 5] * inv), pack_bf16(acc[c + 6] * inv, acc[c + 7] * inv));
          }
        }
      }
    };

    float bias_prev = 0.f;
    for (int i = 0; i < n_tiles; ++i) {
      const float b = features(i);
      if (i >= 1) output(i - 1, bias_prev);
      bias_prev = b;
    }
    if (n_tiles >= 1) output(n_tiles - 1, bias_prev);
    mbar_wait(done_bar, 0, wctx);
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (NC > 1) cluster_sync();   // no CTA leaves while another may still write to it
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------------------
// causal initial states: pre[sc] = the sum, in split order, of the partial
// states of the sub-splits of superchunks 0 .. sc - 1 (block = (head,
// feature block, state row n), thread = feature; eight loads in flight)
// ---------------------------------------------------------------------------
// causal kernel: a cluster of NC CTAs (NC = m / 128) per superchunk of one
// head, walking its 128-token chunks; CTA rank r holds feature block r of
// Omega and the block's rows of the running state G_r (fp32, tensor memory,
// columns 0 .. d-1 = phi(k)^T v, column d = the normaliser sums).  G_r
// starts as the fixed-order sum of the earlier superchunks' partial states of
// its block.  Per chunk c ("Performer" digest, §Methods, causal bullet: the
// prefix sum G_t = sum_{s<=t} phi(k_s) v_s^T, read blockwise):
//   phi(K_c)_r, phi(Q_c)_r  from P = X Omega_r^T in the tile X     (exponentials: CUDA cores)
//   A   = phi(Q_c)_r phi(K_c)_r^T   (into X once the projections are out)
//   O   = phi(Q_c)_r G_s,r          (G_s = bf16 copy of G_r before this chunk)
//   G_r += phi(K_c)_r^T [V_c | 1]
//   O  += mask(A) [V_c | 1]         (keys after the query zeroed, diagonal kept)
// so O is CTA r's partial of the chunk's output with its own row reference
// (the block's row maximum).  The partials of the NC CTAs meet in an
// L2-resident exchange buffer of the workspace; CTA r finalises columns
// [r W, (r + 1) W), W = d / NC, rescaling each partial to the largest
// reference ("From Performer to Linear Attention", §Simple Derivation).
// ---------------------------------------------------------------------------
struct FsCausalParams {
  const float* key_ref;
  const uint8_t* omega_img;
  const float* pre;       // [BH][n_fb][n_sc][d+1][128] initial states
  __nv_bfloat16* O;
  int32_t* status;
  int L, m, n_fb, tiles_per_sc, n_sc;
  float scale;
};


template <int NC>
struct FsCausalCfg {
  static constexpr int W = kD / NC;                        // output columns finalised per CTA
  static constexpr int RB = 2 * W + 16;                    // landing row bytes: W bf16 numerators, fp32 normaliser and reference, pad
  static constexpr int kLandChunk = (NC - 1) * kBM * RB;   // one chunk's rows from the other CTAs
  static constexpr int NB = NC == 4 ? 1 : 2;               // landing buffers (chunks in flight) that fit
  static constexpr int kOmega = 0;                         // [2 atoms][128 feature rows][128 B]
  static constexpr int kK = kOmega + 2 * kAtom;            // K_c, then phi(K_c) over it
  static constexpr int kQ = kK + kTile;                    // Q_c, then phi(Q_c), then the masked scores over it
  static constexpr int kV = kQ + kTile;                    // V_c, then the ones atom
  static constexpr int kGs = kV + kTile + kAtom;           // [2 atoms][kGN rows][128 B]
  static constexpr int kNorm = kGs + 2 * kGN * 128;        // [128] squared key norms
  static constexpr int kXmax = kNorm + kBM * 4;            // [2][2][128] row maxima
  static constexpr int kLand = kXmax + 2 * 2 * kBM * 4;    // [NB][NC - 1 sources][128][RB]
  static constexpr int kBars = kLand + (NC > 1 ? NB * kLandChunk : 0);
  static constexpr int kSmem = kBars + 512 + 1024;
};
static_assert(FsCausalCfg<4>::kSmem <= 232448 && FsCausalCfg<2>::kSmem <= 232448, "shared memory");
static_assert(FsCausalCfg<4>::kGs % 1024 == 0 && FsCausalCfg<4>::kQ % 1024 == 0, "operand alignment");

template <int NC, int FM>
__global__ void __launch_bounds__(kThreads, 1) fs_causal_kernel(const __grid_constant__ CUtensorMap mapQ,
                                                                const __grid_constant__ CUtensorMap mapK,
                                                                const __grid_constant__ CUtensorMap mapV,
                                                                FsCausalParams prm) {
  using C = FsCausalCfg<NC>;
  constexpr int W = C::W;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* b = reinterpret_cast<uint64_t*>(sm + C::kBars);
  uint64_t *k_full = b + 0, *q_full = b + 1, *v_full = b + 2;        // TMA landed
  uint64_t *kn_full = b + 3, *qn_full = b + 4;                       // K, Q in fp16 (K norms written)
  uint64_t *k_free = b + 5, *q_free = b + 6, *v_free = b + 7;        // slots consumed by the MMAs
  uint64_t *pk_full = b + 8, *pq_full = b + 9, *a_full = b + 10;     // X holds P_K, P_Q, A
  uint64_t *x_free = b + 11;                                         // X copied out
  uint64_t *kphi_full = b + 12, *qphi_full = b + 13, *gs_full = b + 14;
  uint64_t *g_done = b + 15, *oin_done = b + 16;                     // G step, O = phi(Q) G_s step complete
  uint64_t *ma_full = b + 17, *ma_free = b + 18;
  uint64_t *o_full = b + 19, *o_free = b + 20;
  uint64_t *land_full = b + 21;                                      // [NB] the other CTAs' partials for my columns
  uint64_t *land_free = b + 23;                                      // [NB][4] owner r has read my partial
  uint64_t *setup_bar = b + 31, *done_bar = b + 32;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(b + 33);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* norms = reinterpret_cast<float*>(sm + C::kNorm);
  float* xmax = reinterpret_cast<float*>(sm + C::kXmax);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = NC > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  const int sc = blockIdx.x / NC, bh = blockIdx.y;
  const int n_tiles_total = (prm.L + kBM - 1) / kBM;
  const int tile0 = sc * prm.tiles_per_sc;
  const int n_chunks = min(prm.tiles_per_sc, n_tiles_total - tile0);
  const WaitCtx wctx{abort_flag, prm.status};
  // TMEM columns: X (projections, then the chunk scores A), O, G_r
  constexpr uint32_t X_COL = 0, O_COL = 128, G_COL = 128 + kGN;

  if (threadIdx.x == 0) {
    for (uint64_t* bar : {k_full, q_full, v_full, k_free, q_free, v_free, pk_full, pq_full, a_full}) mbar_init(bar, 1);
    mbar_init(kn_full, kNormWarps);
    mbar_init(qn_full, kNormWarps);
    mbar_init(x_free, kEpiWarps);
    mbar_init(kphi_full, kEpiWarps);
    mbar_init(qphi_full, kEpiWarps);
    mbar_init(gs_full, kEpiWarps);
    mbar_init(g_done, 1);
    mbar_init(oin_done, 1);
    mbar_init(ma_full, kEpiWarps);
    mbar_init(ma_free, 1);
    mbar_init(o_full, 1);
    mbar_init(o_free, kEpiWarps);
    // partials arrive by st.async, counted in bytes (one arrival per phase:
    // the expected byte count, posted here for the first NB chunks and by the
    // finalising warpgroup for chunk j + NB once chunk j is read)
    for (int i = 0; i < 2; ++i) mbar_init(&land_full[i], 1);
    for (int i = 0; i < 8; ++i) mbar_init(&land_free[i], 4);   // owner i % 4's finalising warps
    mbar_init(setup_bar, 1);
    mbar_init(done_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
    if (NC > 1)
      for (int i = 0; i < C::NB; ++i) mbar_arrive_expect_tx(&land_full[i], C::kLandChunk);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (warp >= 4) {
    fill_ones_atom(sm + C::kV + kTile, kEpiTid0, kEpiThreads);
    // G_s rows d + 8 .. d + 15 of both atoms stay zero (G's columns there are zero)
    for (int e = threadIdx.x - kEpiTid0; e < 2 * 8 * 8; e += kEpiThreads) {
      const int atom = e >> 6, row = kD + 8 + ((e >> 3) & 7);
      *reinterpret_cast<uint4*>(sm + C::kGs + atom * kGN * 128 + row * 128 + (e & 7) * 16) = make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (NC > 1) cluster_sync();   // every CTA's barriers exist before any remote arrival
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      prefetch_tmap(&mapQ);
      prefetch_tmap(&mapK);
      prefetch_tmap(&mapV);
      mbar_arrive_expect_tx(setup_bar, 2 * kAtom);
      for (int a = 0; a < 2; ++a)
        bulk_load(sm + C::kOmega + a * kAtom, prm.omega_img + ((size_t)a * prm.m + rank * kFB) * 128, kAtom,
                  setup_bar);
      // each slot takes chunk c + 1's tile once the MMAs are done with chunk c's
      bool ok = true;
      for (int c = 0; ok && c < n_chunks; ++c) {
        const int row = (tile0 + c) * kBM;
        uint64_t* fulls[3] = {k_full, q_full, v_full};
        uint64_t* frees[3] = {k_free, ma_free, v_free};   // the Q slot holds the masked scores until O += mask(A)[V|1]
        const CUtensorMap* maps[3] = {&mapK, &mapQ, &mapV};
        const int offs[3] = {C::kK, C::kQ, C::kV};
        for (int kind = 0; ok && kind < 3; ++kind) {
          if (c >= 1 && !mbar_wait(frees[kind], (c - 1) & 1, wctx)) { ok = false; break; }
          mbar_arrive_expect_tx(fulls[kind], kTile);
          for (int a = 0; a < 2; ++a)
            tma_load_3d(sm + offs[kind] + a * kAtom, maps[kind], a * 64, row, bh, fulls[kind]);
        }
      }
      // drain: the last loads have landed
      if (n_chunks >= 1) {
        mbar_wait(k_full, (n_chunks - 1) & 1, wctx);
        mbar_wait(q_full, (n_chunks - 1) & 1, wctx);
        mbar_wait(v_full, (n_chunks - 1) & 1, wctx);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t id_proj = idesc_f16(kBM, kFB, false, false);
      constexpr uint32_t id_a = idesc_bf16(kBM, kBM, false, false);
      constexpr uint32_t id_g = idesc_bf16(kFB, kGN, true, true);
      constexpr uint32_t id_o = idesc_bf16(kBM, kGN, false, false);
      constexpr uint32_t id_oi = idesc_bf16(kBM, kGN, false, true);
      const uint32_t om_a = smem_addr(sm + C::kOmega), k_a = smem_addr(sm + C::kK), q_a = smem_addr(sm + C::kQ);
      const uint32_t v_a = smem_addr(sm + C::kV), gs_a = smem_addr(sm + C::kGs), ma_a = smem_addr(sm + C::kQ);
      bool ok = mbar_wait(setup_bar, 0, wctx);
      auto ready = [](uint64_t* bar, int parity) { return mbar_test_wait(smem_addr(bar), parity & 1); };
      // Event-driven issue.  X is used in order P_K(c), P_Q(c), A(c), each
      // use once the epilogue copied the previous one out; G(c) once phi(K_c),
      // V_c and the copy G_s(c) are in place; O(c) once phi(Q_c) and G_s(c)
      // are in place and O(c - 1) was read; O += mask(A) [V|1] once the masked
      // tile is stored.  A slot is released once every MMA that reads it is
      // issued (a commit covers all earlier MMAs).
      Watchdog wd(wctx);
      int nx = 0, ng = 0, no = 0, noi = 0;
      const int n_x = 3 * n_chunks;
      while (ok && noi < n_chunks) {
        bool progress = false;
        if (nx < n_x) {
          const int c = nx / 3, kind = nx % 3;
          const bool x_ok = nx == 0 || ready(x_free, nx - 1);
          const bool in_ok = kind == 0 ? ready(kn_full, c) : kind == 1 ? ready(qn_full, c)
                                                          : (ready(kphi_full, c) && ready(qphi_full, c));
          if (x_ok && in_ok) {
            tc_fence_after();
            if (kind < 2) {
              const uint64_t a0 = sdesc(kind == 0 ? k_a : q_a, 16, 1024), b0 = sdesc(om_a, 16, 1024);
#pragma unroll
              for (int k = 0; k < kD / 16; ++k)
                mma_bf16(tmem + X_COL, dadd(a0, kstep_k(k, kAtom)), dadd(b0, kstep_k(k, kAtom)), id_proj, k > 0);
              mma_commit(kind == 0 ? pk_full : pq_full);
            } else {
              // A = phi(Q_c) phi(K_c)^T: both K-major over the features
              const uint64_t a0 = sdesc(q_a, 16, 1024), b0 = sdesc(k_a, 16, 1024);
#pragma unroll
              for (int k = 0; k < kFB / 16; ++k)
                mma_bf16(tmem + X_COL, dadd(a0, kstep_k(k, kAtom)), dadd(b0, kstep_k(k, kAtom)), id_a, k > 0);
              mma_commit(a_full);
              if (ng > c) mma_commit(k_free);    // G(c) issued too: phi(K_c)'s slot is done
            }
            ++nx;
            progress = true;
          }
        }
        if (ng < n_chunks && ng < (nx + 2) / 3) {
          const int c = ng;
          if (ready(kphi_full, c) && ready(v_full, c) && ready(gs_full, c)) {
            tc_fence_after();
            const uint64_t a0 = sdesc(k_a, kAtom, 1024), b0 = sdesc(v_a, kAtom, 1024);
#pragma unroll
            for (int k = 0; k < kBM / 16; ++k)
              mma_bf16(tmem + G_COL, dadd(a0, kstep_mn(k)), dadd(b0, kstep_mn(k)), id_g, true);
            mma_commit(g_done);
            if (nx > 3 * c + 2) mma_commit(k_free);   // A(c) issued too
            ++ng;
            progress = true;
          }
        }
        if (no < n_chunks && no < (nx + 1) / 3) {
          const int c = no;
          if (ready(qphi_full, c) && ready(gs_full, c) && (c == 0 || ready(o_free, c - 1))) {
            tc_fence_after();
            const uint64_t a0 = sdesc(q_a, 16, 1024), b0 = sdesc(gs_a, 16, 1024);
#pragma unroll
            for (int k = 0; k < kFB / 16; ++k)
              mma_bf16(tmem + O_COL, dadd(a0, kstep_k(k, kAtom)), dadd(b0, kstep_k(k, kGN * 128)), id_o, k > 0);
            mma_commit(oin_done);
            ++no;
            progress = true;
          }
        }
        if (noi < no && noi < ng && ready(ma_full, noi)) {
          tc_fence_after();
          const uint64_t a0 = sdesc(ma_a, 16, 1024), b0 = sdesc(v_a, kAtom, 1024);
#pragma unroll
          for (int k = 0; k < kBM / 16; ++k)
            mma_bf16(tmem + O_COL, dadd(a0, kstep_k(k, kAtom)), dadd(b0, kstep_mn(k)), id_oi, true);
          mma_commit(o_full);
          mma_commit(v_free);
          mma_commit(ma_free);
          ++noi;
          progress = true;
        }
        if (progress) wd.progress();
        else ok = wd.idle();
      }
      mma_commit(done_bar);
      mbar_wait(done_bar, 0, wctx);
    }
  } else if (warp < 2 + kNormWarps) {
    // squared row norms of K_c; K_c and Q_c rewritten as fp16
    for (int c = 0; c < n_chunks; ++c) {
      if (!mbar_wait(k_full, c & 1, wctx)) break;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int r = (warp - 2) * 64 + lane + 32 * j;
        norms[r] = tile_row_sq_to_f16<kD>(sm + C::kK, r);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(kn_full);
      if (!mbar_wait(q_full, c & 1, wctx)) break;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int r = (warp - 2) * 64 + lane + 32 * j;
        (void)tile_row_sq_to_f16<kD>(sm + C::kQ, r);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(qn_full);
    }
  } else {
    // ---------------- epilogue: warpgroup w takes columns 64w .. 64w + 63 ----------------
    const int wg = (warp - 4) >> 2;
    const int q = warp & 3;
    const int t = q * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    const int col0 = wg * 64;
    float R, W_unused;
    key_reference(prm.key_ref, prm.m, &R, &W_unused);
    const float c1 = feature_c1<FM>(prm.scale);
    const float hs2 = 0.5f * prm.scale * prm.scale;
    const uint32_t k_a = smem_addr(sm + C::kK), q_a = smem_addr(sm + C::kQ), ma_a = q_a;   // masked scores over phi(Q)
    const uint32_t gs_a = smem_addr(sm + C::kGs);
    const int wg_fin = (rank * W) / 64;   // the warpgroup holding my output columns (NC > 1)
    bool ok = true;

    // G_r = the superchunk's initial state (the earlier superchunks' partials
    // of block r, summed in order by the prefix kernel): warpgroup 0 columns
    // 0 .. 79, warpgroup 1 columns 80 .. 143 (zero past d)
    {
      const int n0 = wg ? 80 : 0;
      const int ng16 = wg ? 4 : 5;
      const float* src = prm.pre + (((size_t)bh * prm.n_fb + rank) * prm.n_sc + sc) * (kD + 1) * kFB;
      for (int g = 0; g < ng16; ++g) {
        uint32_t r[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int n = n0 + 16 * g + j;
          r[j] = __float_as_uint(n <= kD ? src[(size_t)n * kFB + t] : 0.f);
        }
        tmem_st16(tmem + lane_off + G_COL + n0 + 16 * g, r);
      }
      tmem_st_wait();
    }
    // the G_s copies read columns the other warpgroup stored
    tc_fence_before();
    named_bar(1, kEpiThreads);
    tc_fence_after();

    auto max64 = [](const uint32_t (&x)[64]) {
      float pm = -INFINITY;
#pragma unroll
      for (int j = 0; j < 64; ++j) pm = fmaxf(pm, __uint_as_float(x[j]));
      return pm;
    };
    // G_s <- bf16(G_r), rows n < d + 8 (the normaliser column d, then zeros):
    // per group of 8 columns a 16x256b load per half of this warp's 32
    // features gives each thread two adjacent n of one feature;
    // stmatrix.trans turns each 8x8 block (features x n) into rows n of 8
    // features, one swizzle chunk each.  Warpgroup 0 takes groups 0 .. 8.
    auto copy_gs = [&]() {
      constexpr int kGroups = kD / 8 + 1;
      const int g0 = wg ? (kGroups + 1) / 2 : 0, g1 = wg ? kGroups : (kGroups + 1) / 2;
      const int f0 = 32 * q + 8 * (lane >> 3);
      tmem_state_to_rows<3>(tmem, G_COL, q, lane, g0, g1, gs_a + (f0 >> 6) * (kGN * 128));
    };

    // the output of chunk j: my partial to the exchange, my columns finalised
    auto out = [&](int j, float bias) {
      const bool have = ok && mbar_wait(o_full, j & 1, wctx);
      tc_fence_after();
      uint32_t v[64], z[8];
      tmem_ld32_at<0>(tmem + lane_off + O_COL + col0, v);
      tmem_ld32_at<32>(tmem + lane_off + O_COL + col0 + 32, v);
      tmem_ld8(tmem + lane_off + O_COL + kD, z);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(o_free);
      const float den_own = __uint_as_float(z[0]);
      const int row = (tile0 + j) * kBM + t;
      const bool valid = row < prm.L;
      __nv_bfloat16* orow = prm.O + ((size_t)bh * prm.L + (valid ? row : 0)) * kD;
      if constexpr (NC == 1) {
        if (have && valid) {
          if (!(den_own > 0.f) || !isfinite(den_own)) report_status(prm.status, FAVOR_ERR_NONFINITE);
          const float inv = __fdividef(1.0f, den_own);
#pragma unroll
          for (int c = 0; c < 64; c += 8)
            *reinterpret_cast<uint4*>(orow + col0 + c) =
                make_uint4(pack_bf16(__uint_as_float(v[c]) * inv, __uint_as_float(v[c + 1]) * inv),
                           pack_bf16(__uint_as_float(v[c + 2]) * inv, __uint_as_float(v[c + 3]) * inv),
                           pack_bf16(__uint_as_float(v[c + 4]) * inv, __uint_as_float(v[c + 5]) * inv),
                           pack_bf16(__uint_as_float(v[c + 6]) * inv, __uint_as_float(v[c + 7]) * inv));
        }
      } else {
        // send: every slice of my columns owned by another CTA, into landing
        // buffer j % NB of the owner once it has read that buffer's previous
        // chunk; bf16 numerators, fp32 normaliser and reference, by st.async
        const int buf = j % C::NB;
#pragma unroll
        for (int sl = 0; sl < 64 / W; ++sl) {
          const int owner = (col0 + sl * W) / W;
          if (owner == rank) continue;
          if (ok && j >= C::NB) ok = mbar_wait_cluster(&land_free[buf * 4 + owner], ((j / C::NB) - 1) & 1, wctx);
          const int slot = rank < owner ? rank : rank - 1;
          const uint32_t dst = map_to_rank(
              smem_addr(sm + C::kLand + buf * C::kLandChunk + ((size_t)slot * kBM + t) * C::RB),
              static_cast<uint32_t>(owner));
          const uint32_t mb = map_to_rank(smem_addr(&land_full[buf]), static_cast<uint32_t>(owner));
          if (ok) {
#pragma unroll
            for (int c = 0; c < W; c += 8)
              st_async_v4(dst + c * 2, pack_bf16(__uint_as_float(v[sl * W + c]), __uint_as_float(v[sl * W + c + 1])),
                          pack_bf16(__uint_as_float(v[sl * W + c + 2]), __uint_as_float(v[sl * W + c + 3])),
                          pack_bf16(__uint_as_float(v[sl * W + c + 4]), __uint_as_float(v[sl * W + c + 5])),
                          pack_bf16(__uint_as_float(v[sl * W + c + 6]), __uint_as_float(v[sl * W + c + 7])), mb);
            st_async_v4(dst + W * 2, __float_as_uint(den_own), __float_as_uint(bias), 0u, 0u, mb);
          }
        }
        if (wg == wg_fin) {
          // my columns: every partial rescaled to the largest reference; mine
          // first, then the others in rank order
          if (ok) ok = mbar_wait(&land_full[buf], (j / C::NB) & 1, wctx);
          const uint8_t* land = sm + C::kLand + buf * C::kLandChunk;
          float bmax = bias;
          for (int sl = 0; sl < NC - 1; ++sl)
            bmax = fmaxf(bmax, *reinterpret_cast<const float*>(land + ((size_t)sl * kBM + t) * C::RB + 2 * W + 4));
          const bool hi = (rank * W - col0) != 0;
          const float sc_own = ex2(bias - bmax);
          float acc[W];
#pragma unroll
          for (int c = 0; c < W; ++c) acc[c] = sc_own * __uint_as_float(W == 64 ? v[c] : (hi ? v[(32 + c) & 63] : v[c]));
          float den = sc_own * den_own;
          for (int sl = 0; sl < NC - 1; ++sl) {
            const uint8_t* lr = land + ((size_t)sl * kBM + t) * C::RB;
            const float2 dr = *reinterpret_cast<const float2*>(lr + 2 * W);   // normaliser, reference
            const float sc = ex2(dr.y - bmax);
#pragma unroll
            for (int c = 0; c < W; c += 8) {
              const uint4 p4 = *reinterpret_cast<const uint4*>(lr + c * 2);
              const uint32_t w4[4] = {p4.x, p4.y, p4.z, p4.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                acc[c + 2 * e] = fmaf(sc, __uint_as_float(w4[e] << 16), acc[c + 2 * e]);
                acc[c + 2 * e + 1] = fmaf(sc, __uint_as_float(w4[e] & 0xFFFF0000u), acc[c + 2 * e + 1]);
              }
            }
            den = fmaf(sc, dr.x, den);
          }
          // read: re-arm the buffer for chunk j + NB, then let its writers send
          if (threadIdx.x == kEpiTid0 + kBM * wg_fin && ok) mbar_arrive_expect_tx(&land_full[buf], C::kLandChunk);
          __syncwarp();
          if (lane == 0)
            for (int src = 0; src < NC; ++src)
              if (src != rank)
                mbar_arrive_remote(map_to_rank(smem_addr(&land_free[buf * 4 + rank]), static_cast<uint32_t>(src)));
          if (have && valid) {
            if (!(den > 0.f) || !isfinite(den)) report_status(prm.status, FAVOR_ERR_NONFINITE);
            const float inv = __fdividef(1.0f, den);
#pragma unroll
            for (int c = 0; c < W; c += 8)
              *reinterpret_cast<uint4*>(orow + rank * W + c) =
                  make_uint4(pack_bf16(acc[c] * inv, acc[c + 1] * inv), pack_bf16(acc[c + 2] * inv, acc[c + 3] * inv),
                             pack_bf16(acc[c + 4] * inv, acc[c + 5] * inv), pack_bf16(acc[c + 6] * inv, acc[c + 7] * inv));
          }
        }
      }
    };

    // G_s(0): the initial state
    if (ok) copy_gs();
    tc_fence_before();
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(gs_full);
    float bias_prev = 0.f;
    for (int c = 0; c < n_chunks; ++c) {
      const bool valid = (tile0 + c) * kBM + t < prm.L;
      // ---- phi(K_c)_r over K_c ----
      if (ok) ok = mbar_wait(pk_full, c & 1, wctx);
      if (ok) ok = mbar_wait(kn_full, c & 1, wctx);
      tc_fence_after();
      {
        uint32_t x[64];
        tmem_ld64(tmem + lane_off + X_COL + col0, x);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(x_free);
        // rows past the sequence end: an infinite bias makes their features 0
        const float bias_k = !valid ? INFINITY : (FM == FAVOR_FM_PRF ? (hs2 * norms[t] + R) * kLog2e : 0.f);
        if (ok) {
          feature_pack<FM>(x, c1, bias_k);
          store_row<32>(k_a, kAtom, t, col0, x);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(kphi_full);
      }
      // the previous chunk's output, deferred so that its MMAs overlap
      if (c >= 1) out(c - 1, bias_prev);
      // ---- phi(Q_c)_r over Q_c, with the block's row maximum as reference ----
      if (ok) ok = mbar_wait(pq_full, c & 1, wctx);
      tc_fence_after();
      float bias_q = 0.f;
      {
        uint32_t x[64];
        tmem_ld64(tmem + lane_off + X_COL + col0, x);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(x_free);
        if constexpr (FM == FAVOR_FM_PRF) {
          float* xm = xmax + (c & 1) * 2 * kBM;
          xm[wg * kBM + t] = max64(x);
          named_bar(2, kEpiThreads);
          bias_q = fmaxf(xm[t], xm[kBM + t]) * c1;
        }
        if (ok) {
          feature_pack<FM>(x, c1, bias_q);
          store_row<32>(q_a, kAtom, t, col0, x);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(qphi_full);
      }
      bias_prev = bias_q;
      // ---- masked A -> bf16 ----
      if (ok) ok = mbar_wait(a_full, c & 1, wctx);
      tc_fence_after();
      {
        uint32_t a[64];
        tmem_ld64(tmem + lane_off + X_COL + col0, a);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(x_free);
        // the masked scores go over phi(Q_c): O(c) = phi(Q_c) G_s must have read it
        if (ok) ok = mbar_wait(oin_done, c & 1, wctx);
        if (ok) {
          // this warp's rows 32q .. 32q+31 against keys col0 .. col0+63:
          // entirely kept, entirely masked, or on the diagonal
          if (col0 + 63 <= 32 * q) {
#pragma unroll
            for (int j = 0; j < 32; ++j) a[j] = pack_bf16(__uint_as_float(a[2 * j]), __uint_as_float(a[2 * j + 1]));
          } else if (col0 > 32 * q + 31) {
#pragma unroll
            for (int j = 0; j < 32; ++j) a[j] = 0u;
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int f = col0 + 2 * j;
              a[j] = pack_bf16(f <= t ? __uint_as_float(a[2 * j]) : 0.f, f + 1 <= t ? __uint_as_float(a[2 * j + 1]) : 0.f);
            }
          }
          store_row<32>(ma_a, kAtom, t, col0, a);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(ma_full);
      }
      // ---- G_s(c + 1) = bf16(G_r) once G(c) and O(c) are done with it; it
      // overlaps the next chunk's key projection ----
      if (c + 1 < n_chunks) {
        if (ok) ok = mbar_wait(g_done, c & 1, wctx);
        if (ok) ok = mbar_wait(oin_done, c & 1, wctx);
        tc_fence_after();
        if (ok) copy_gs();
        tc_fence_before();
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(gs_full);
      }
    }
    if (n_chunks >= 1) out(n_chunks - 1, bias_prev);
    mbar_wait(done_bar, 0, wctx);
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (NC > 1) cluster_sync();   // no CTA leaves while another may still arrive on its barriers
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
// the key-state kernel's share of a workspace plan
struct FsStateLaunch {
  size_t off_omega_img, off_counters, off_partS, off_state_img;
  int n_fb, n_split, tiles_per_split, merge;
};

template <int FM>
cudaError_t launch_fs_state(const void* K, const void* V, const Shape& s, const FsStateLaunch& sl, float scale,
                            char* ws, int32_t* status, cudaStream_t stream) {
  if (sl.n_split < 1) return cudaSuccess;
  CUtensorMap mk, mv;
  if (!make_map(&mk, K, s) || !make_map(&mv, V, s)) return cudaErrorInvalidValue;
  FsStateParams prm{};
  prm.key_ref = reinterpret_cast<const float*>(ws);
  prm.omega_img = reinterpret_cast<const uint8_t*>(ws + sl.off_omega_img);
  prm.partS = reinterpret_cast<float*>(ws + sl.off_partS);
  prm.counters = reinterpret_cast<uint32_t*>(ws + sl.off_counters);
  prm.state_img = reinterpret_cast<uint8_t*>(ws + sl.off_state_img);
  prm.status = status;
  prm.L = s.L;
  prm.m = s.m;
  prm.n_fb = sl.n_fb;
  prm.n_split = sl.n_split;
  prm.tiles_per_split = sl.tiles_per_split;
  prm.merge = sl.merge;
  prm.scale = scale;
  const size_t smem = FsStateCfg::kSmem;
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(fs_state_kernel<FM>), smem);
  if (e != cudaSuccess) return e;
  dim3 grid(sl.n_split * sl.n_fb, s.BH());
  fs_state_kernel<FM><<<grid, kThreads, smem, stream>>>(mk, mv, prm);
  return cudaGetLastError();
}

// Clusters of NC CTAs that can be resident at once (cached per device and NC).
template <int NC, int FM>
int resident_clusters(size_t smem) {
  static std::mutex mu;
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return sm_count() / NC;
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] == 0) {
    int n = 0;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(NC * 64, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = NC;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, fs_output_kernel<NC, FM>, &cfg) != cudaSuccess || n < 1) {
      (void)cudaGetLastError();
      n = sm_count() / NC;
    }
    cached[dev] = n;
  }
  return cached[dev];
}

template <int NC, int FM>
cudaError_t launch_fs_output(const void* Q, void* O, const Shape& s, const FsPlan& p, float scale, char* ws,
                             int32_t* status, cudaStream_t stream) {
  CUtensorMap mq;
  if (!make_map(&mq, Q, s)) return cudaErrorInvalidValue;
  const size_t smem = FsOutCfg<NC>::kSmem;
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(fs_output_kernel<NC, FM>), smem);
  if (e != cudaSuccess) return e;
  // as many clusters as can be resident (or one per tile), each an even share
  // of the (head, tile) list
  const int n_cl = (int)std::min<long long>(resident_clusters<NC, FM>(smem), (long long)s.BH() * p.n_tiles);
  FsOutParams prm{};
  prm.omega_img = reinterpret_cast<const uint8_t*>(ws + p.off_omega_img);
  prm.state_img = reinterpret_cast<const uint8_t*>(ws + p.off_state_img);
  prm.O = static_cast<__nv_bfloat16*>(O);
  prm.status = status;
  prm.L = s.L;
  prm.m = s.m;
  prm.n_heads = s.BH();
  prm.scale = scale;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(n_cl * NC, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = NC;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = NC > 1 ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, fs_output_kernel<NC, FM>, mq, prm);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int FM>
cudaError_t fs_output_nc(const void* Q, void* O, const Shape& s, const FsPlan& p, float scale, char* ws,
                         int32_t* status, cudaStream_t stream) {
  switch (p.n_fb) {
    case 1: return launch_fs_output<1, FM>(Q, O, s, p, scale, ws, status, stream);
    case 2: return launch_fs_output<2, FM>(Q, O, s, p, scale, ws, status, stream);
    default: return launch_fs_output<4, FM>(Q, O, s, p, scale, ws, status, stream);
  }
}

template <int NC, int FM>
cudaError_t launch_fs_causal(const void* Q, const void* K, const void* V, void* O, const Shape& s,
                             const FsCausalPlan& p, float scale, char* ws, int32_t* status, cudaStream_t stream) {
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, Q, s) || !make_map(&mk, K, s) || !make_map(&mv, V, s)) return cudaErrorInvalidValue;
  const size_t smem = FsCausalCfg<NC>::kSmem;
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(fs_causal_kernel<NC, FM>), smem);
  if (e != cudaSuccess) return e;
  FsCausalParams prm{};
  prm.key_ref = reinterpret_cast<const float*>(ws);
  prm.omega_img = reinterpret_cast<const uint8_t*>(ws + p.off_omega_img);
  prm.pre = reinterpret_cast<const float*>(ws + p.off_pre);
  prm.O = static_cast<__nv_bfloat16*>(O);
  prm.status = status;
  prm.L = s.L;
  prm.m = s.m;
  prm.n_fb = p.n_fb;
  prm.tiles_per_sc = p.tiles_per_sc;
  prm.n_sc = p.n_sc;
  prm.scale = scale;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(p.n_sc * NC, s.BH(), 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = NC;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = NC > 1 ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, fs_causal_kernel<NC, FM>, mq, mk, mv, prm);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int FM>
cudaError_t fs_causal_nc(const void* Q, const void* K, const void* V, void* O, const Shape& s,
                         const FsCausalPlan& p, float scale, char* ws, int32_t* status, cudaStream_t stream) {
  switch (p.n_fb) {
    case 1: return launch_fs_causal<1, FM>(Q, K, V, O, s, p, scale, ws, status, stream);
    case 2: return launch_fs_causal<2, FM>(Q, K, V, O, s, p, scale, ws, status, stream);
    default: return launch_fs_causal<4, FM>(Q, K, V, O, s, p, scale, ws, status, stream);
  }
}

}  // namespace

bool fs_supported(bool causal, int d, int m, bool bf16) {
  (void)causal;
  return bf16 && d == kD && (m == 128 || m == 256 || m == 512);
}

size_t fs_workspace_bytes(bool causal, const Shape& s) { return causal ? fsc_plan(s).bytes : fs_plan(s).bytes; }

cudaError_t fs_state(bool causal, const void* K, const void* V, const float* omega, float scale, const Shape& s,
                     void* ws, int32_t* status, cudaStream_t stream, int fm) {
  char* w = static_cast<char*>(ws);
  FsStateLaunch sl{};
  size_t off_counters = 0;
  int n_counters = 0;
  if (causal) {
    const FsCausalPlan p = fsc_plan(s);
    sl = FsStateLaunch{p.off_omega_img, 0, p.off_partS, 0, p.n_fb, p.n_split, p.tiles_per_split, 0};
  } else {
    const FsPlan p = fs_plan(s);
    sl = FsStateLaunch{p.off_omega_img, p.off_counters, p.off_partS, p.off_state_img, p.n_fb, p.n_split,
                       p.tiles_per_split, 1};
    off_counters = p.off_counters;
    n_counters = s.BH() * p.n_fb;
  }
  // prep: key reference header, fp16 Omega image, zeroed merge counters
  cudaError_t e = launch_prep(omega, s.m, s.d, reinterpret_cast<float*>(w),
                              reinterpret_cast<uint8_t*>(w + sl.off_omega_img),
                              n_counters ? reinterpret_cast<uint32_t*>(w + off_counters) : nullptr, n_counters, stream);
  if (e != cudaSuccess) return e;
  e = fm == FAVOR_FM_RELU   ? launch_fs_state<FAVOR_FM_RELU>(K, V, s, sl, scale, w, status, stream)
      : fm == FAVOR_FM_ELU1 ? launch_fs_state<FAVOR_FM_ELU1>(K, V, s, sl, scale, w, status, stream)
                            : launch_fs_state<FAVOR_FM_PRF>(K, V, s, sl, scale, w, status, stream);
  if (e != cudaSuccess || !causal) return e;
  const FsCausalPlan p = fsc_plan(s);
  state_prefix_kernel<kD><<<dim3(p.n_fb * (kD + 1), s.BH()), kFB, 0, stream>>>(
      reinterpret_cast<const float*>(w + p.off_partS), reinterpret_cast<float*>(w + p.off_pre), p.n_fb, p.n_split,
      p.sub_per_sc, p.n_sc);
  return cudaGetLastError();
}

cudaError_t fs_output(bool causal, const void* Q, const void* K, const void* V, void* O, float scale, const Shape& s,
                      void* ws, int32_t* status, cudaStream_t stream, int fm) {
  char* w = static_cast<char*>(ws);
  if (causal) {
    const FsCausalPlan p = fsc_plan(s);
    if (fm == FAVOR_FM_RELU) return fs_causal_nc<FAVOR_FM_RELU>(Q, K, V, O, s, p, scale, w, status, stream);
    if (fm == FAVOR_FM_ELU1) return fs_causal_nc<FAVOR_FM_ELU1>(Q, K, V, O, s, p, scale, w, status, stream);
    return fs_causal_nc<FAVOR_FM_PRF>(Q, K, V, O, s, p, scale, w, status, stream);
  }
  const FsPlan p = fs_plan(s);
  if (fm == FAVOR_FM_RELU) return fs_output_nc<FAVOR_FM_RELU>(Q, O, s, p, scale, w, status, stream);
  if (fm == FAVOR_FM_ELU1) return fs_output_nc<FAVOR_FM_ELU1>(Q, O, s, p, scale, w, status, stream);
  return fs_output_nc<FAVOR_FM_PRF>(Q, O, s, p, scale, w, status, stream);
}

}  // namespace favor
