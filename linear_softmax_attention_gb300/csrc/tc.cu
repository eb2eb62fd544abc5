// Tensor-core (tcgen05) FAVOR+ kernels for sm_103a: operands in shared memory
// (TMA, 128-byte swizzle), fp32 accumulators in tensor memory.
//
// "Performer — Rethinking Attention with Performers" (digest), §Key equations
// and the flowchart: phi(K)^T V and phi(K)^T 1 are formed first, then
// phi(Q) times each, then the row-wise divide; §Methods, causal bullet: the
// prefix sum G_t = sum_{s<=t} phi(k_s) v_s^T.  The contractions are dense
// GEMMs and run on the tensor cores:
//   projection  P  = X Omega^T         M = 128 tokens,   N = m (or 128), K = d   (fp16 operands)
//   state       S~ += phi(K)^T [V|1]   M = 128 features, N = d + 16,     K = 128 tokens
//   output      O  = phi(Q) S~         M = 128 tokens,   N = d + 16,     K = m
//   causal      [A | O] += phi(Q_c) [phi(K_c)^T | G_s]  (one MMA, N = 128 + d + 16),
//               O += mask(A) [V_c | 1]
// The exponentials of the feature map run on the CUDA cores between them
// (TMEM -> registers -> bf16 in shared memory).
//
// Measured on GB300, one M = 128 MMA instruction costs about the same for
// every N up to 128 and about twice that at N = 256, so the kernels issue few,
// wide instructions: the projection covers all m features at once where the
// tensor memory allows, and the normaliser column rides in the same MMA as V
// (the descriptor's leading-byte offset points from the V tile to a constant
// block whose first column is 1).  The projection runs in fp16: a warp
// rewrites each K or Q tile in place as fp16 while it computes the squared
// row norms, and Omega is kept as an fp16 image, which carries Omega to 11
// significant bits (bf16 Omega alone costs ~2.5% in the output).
//
// Warp roles: warp 0 issues TMA loads, warp 1 owns tensor memory and issues
// MMAs (one thread), warps 2-3 compute the squared row norms of the K (and Q)
// tiles and convert them to fp16, and eight epilogue warps form two
// warpgroups that split the columns of each 128-row tile (thread = one TMEM
// lane = one token or one feature).  The state kernel has a thirteenth warp
// that issues its state MMAs, so that a tile's projection never waits behind
// them on one thread (issuing costs ~60 cycles per MMA).  Epilogues copy a
// tile out of tensor memory and release it before they compute on it, so
// that the next MMA into the same columns overlaps their arithmetic.
#include <cudaTypedefs.h>

#include <mutex>

#include "tc.cuh"
#include "tc_util.cuh"

namespace favor {
namespace {

using namespace tc;

// ---------------------------------------------------------------------------
// workspace layout of the tensor-core path
// ---------------------------------------------------------------------------
struct TcPlan {
  bool causal;
  int n_fb, n_tiles;
  int tiles_per_split, n_split;      // state partials (bidir: L splits; causal: sub-splits of all
                                     // superchunks but the last)
  int out_tiles_per_cta, out_ctas;   // causal: tiles per superchunk, superchunks
  int out_grid;                      // bidir output kernel: one CTA per SM (or tile), each an even
                                     // share of the (head, tile) list
  int sub_per_sc;                    // causal: state sub-splits per superchunk
  size_t off_omega_img, off_counters, off_partS, off_state_img, off_pre, bytes;
};

TcPlan tc_plan(bool causal, const Shape& s) {
  TcPlan p{};
  const int BH = s.BH();
  const int sms = sm_count();
  p.causal = causal;
  p.n_fb = s.m / kFB;
  p.n_tiles = (s.L + kBM - 1) / kBM;
  if (!causal) {
    const int sp = pick_split(BH, p.n_tiles, sms);
    p.tiles_per_split = (p.n_tiles + sp - 1) / sp;
    p.n_split = (p.n_tiles + p.tiles_per_split - 1) / p.tiles_per_split;
    p.out_grid = (int)std::min<long long>(sms, (long long)BH * p.n_tiles);
  } else {
    const int sc = pick_split(BH, p.n_tiles, sms);
    p.out_tiles_per_cta = (p.n_tiles + sc - 1) / sc;                          // tiles per superchunk
    p.out_ctas = (p.n_tiles + p.out_tiles_per_cta - 1) / p.out_tiles_per_cta;  // superchunks
    // the states of all superchunks but the last, each computed in k equal
    // sub-splits (k divides the superchunk) so that enough CTAs run
    const int tps = p.out_tiles_per_cta;
    int best_k = 1;
    long best_cost = -1;
    for (int k = 1; k <= tps; ++k) {
      if (tps % k) continue;
      const long ctas = (long)BH * (p.out_ctas - 1) * k;
      const long cost = ((ctas + sms - 1) / sms) * (tps / k + kCtaOverheadTiles);
      if (best_cost < 0 || cost < best_cost) {
        best_cost = cost;
        best_k = k;
      }
    }
    p.sub_per_sc = best_k;
    p.tiles_per_split = tps / best_k;
    p.n_split = (p.out_ctas - 1) * best_k;
  }
  size_t off = align_up(kWsHeader, 1024);
  p.off_omega_img = off;
  off = align_up(off + (size_t)s.m * s.d * 2, 1024);   // fp16 image of Omega
  p.off_counters = off;
  off = align_up(off + (size_t)BH * sizeof(uint32_t), 1024);
  p.off_partS = off;
  off = align_up(off + (size_t)BH * p.n_fb * max(p.n_split, 1) * (s.d + 1) * kFB * sizeof(float), 1024);
  p.off_state_img = off;
  if (!causal) off = align_up(off + (size_t)BH * s.m * (s.d + 16) * 2, 1024);
  p.off_pre = off;   // causal: fp32 [BH][n_fb][superchunks][d+1][128], each superchunk's initial state
  if (causal) off = align_up(off + (size_t)BH * p.n_fb * p.out_ctas * (s.d + 1) * kFB * sizeof(float), 1024);
  p.bytes = off;
  return p;
}


// Causal initial states: the last superchunk sums this many partials at most
// (its predecessors' sub-splits); up to kDirectPartials the scan kernel adds
// them itself, above that the prefix kernel forms every superchunk's sum once.
constexpr int kDirectPartials = 4;
inline bool causal_direct(const TcPlan& p) { return (p.out_ctas - 1) * p.sub_per_sc <= kDirectPartials; }

// ---------------------------------------------------------------------------
// state kernel: one (token split, head) per CTA, all m features.
// Bidirectional: the last CTA of a head adds the splits (fixed order) into
// the bf16 state image read by the output kernel.  Causal: the partial of
// each superchunk but the last is kept for the scan.
// ---------------------------------------------------------------------------
struct StateParams {
  const float* key_ref;
  const uint8_t* omega_img;
  float* partS;            // [BH][n_fb][n_split][d+1][128]
  uint32_t* counters;      // [BH]
  uint8_t* state_img;      // [BH][m/64][d+16][128 B]
  float* zvec;             // bidirectional, optional: [BH][m] fp32 normaliser row of the merged state
  int32_t* status;
  int L, m, n_split, tiles_per_split, merge;
  float scale;
};

constexpr int kStateThreads = 416;   // warps 0 TMA, 1 projection MMAs, 2-3 norms, 4-11 epilogue, 12 state MMAs
constexpr int kStateIssuer = 12;

template <int D>
struct StateCfg {
  // K and V have rings of their own: a K slot is released once the tile's
  // projections have read it, a V slot once the state MMA has; the squared
  // norms of a K tile live one slot longer than the tile (the epilogue reads
  // them after the projection has released the K slot)
  static constexpr int NK = 4, NV = 3, NN = NK + 1;
  static constexpr int kTileBytes = D * kBM * 2;   // one K or V tile
  static constexpr int kOmega = 0;                 // fp16 image, up to 256 x D
  static constexpr int kK = kOmega + 256 * D * 2;
  static constexpr int kV = kK + NK * kTileBytes;
  static constexpr int kOnes = kV + NV * kTileBytes;             // above every V tile
  static constexpr int kPhi = kOnes + kOnesBytes;                // [fb][2 atoms][128][128 B]
  static constexpr int kNorm = kPhi + 2 * 2 * kAtom;             // [NN][128]
  static constexpr int kBars = kNorm + NN * kBM * 4;
  static constexpr int kSmem = kBars + 512 + 1024;
};

template <int D, int M, int FM>
__global__ void __launch_bounds__(kStateThreads, 1) state_kernel(const __grid_constant__ CUtensorMap mapK,
                                                                 const __grid_constant__ CUtensorMap mapV,
                                                                 StateParams prm) {
  using C = StateCfg<D>;
  constexpr int NFB = M / kFB;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::kBars);
  uint64_t* k_full = bars;                    // [NK] K landed
  uint64_t* k_empty = k_full + C::NK;         // [NK] the tile's projections have read it
  uint64_t* v_full = k_empty + C::NK;         // [NV]
  uint64_t* v_empty = v_full + C::NV;         // [NV] the state MMA has read it
  uint64_t* kn_full = v_empty + C::NV;        // [NN] K in fp16, norms written
  uint64_t* p_full = kn_full + C::NN;         // [2] per feature block
  uint64_t* p_free = p_full + 2;              // [2]
  uint64_t* phi_full = p_free + 2;            // [2]
  uint64_t* phi_free = phi_full + 2;          // [2]
  uint64_t* setup_bar = phi_free + 2;
  uint64_t* done_bar = setup_bar + 1;         // [2]: every projection MMA, every state MMA complete
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done_bar + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* is_last = const_cast<int*>(abort_flag) + 1;
  float* norm_s = reinterpret_cast<float*>(sm + C::kNorm);   // [NN][128]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x, bh = blockIdx.y;
  const int tile0 = split * prm.tiles_per_split;
  const int n_tiles_total = (prm.L + kBM - 1) / kBM;
  const int n_tiles = min(prm.tiles_per_split, n_tiles_total - tile0);
  const WaitCtx wctx{abort_flag, prm.status};
  constexpr uint32_t S_COL = 256;              // S~ of block fb at S_COL + 128 fb; P at 0

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NK; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
    }
    for (int i = 0; i < C::NV; ++i) {
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    for (int i = 0; i < C::NN; ++i) mbar_init(&kn_full[i], kNormWarps);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&p_full[i], 1);
      mbar_init(&p_free[i], kEpiWarps / NFB);     // the warps that own block i
      mbar_init(&phi_full[i], kEpiWarps / NFB);
      mbar_init(&phi_free[i], 1);
    }
    mbar_init(setup_bar, 1);
    mbar_init(&done_bar[0], 1);
    mbar_init(&done_bar[1], 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (warp >= 4 && warp < kStateIssuer) {
    fill_ones_block(sm + C::kOnes, kEpiTid0, kEpiThreads);
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
      // the fp16 image of Omega comes from the preparation kernel, which may
      // still run (programmatic launch): the first K and V tiles load first
      if (n_tiles > 0) {
        mbar_arrive_expect_tx(&k_full[0], C::kTileBytes);
        mbar_arrive_expect_tx(&v_full[0], C::kTileBytes);
#pragma unroll
        for (int a = 0; a < D / 64; ++a) {
          tma_load_3d(sm + C::kK + a * kAtom, &mapK, a * 64, tile0 * kBM, bh, &k_full[0]);
          tma_load_3d(sm + C::kV + a * kAtom, &mapV, a * 64, tile0 * kBM, bh, &v_full[0]);
        }
      }
      griddep_wait();
      mbar_arrive_expect_tx(setup_bar, M * D * 2);
      bulk_load(sm + C::kOmega, prm.omega_img, M * D * 2, setup_bar);
      // K tile x goes to K slot x % NK once the projections of tile x - NK
      // have read it, V tile x to V slot x % NV once the state MMA of tile
      // x - NV has; K is issued ahead of V
      Watchdog wd(wctx);
      int nk = n_tiles > 0 ? 1 : 0, nv = nk;
      bool ok = true;
      while (ok && (nk < n_tiles || nv < n_tiles)) {
        bool progress = false;
        if (nk < n_tiles &&
            (nk < C::NK || mbar_test_wait(smem_addr(&k_empty[nk % C::NK]), ((nk / C::NK) - 1) & 1))) {
          const int st = nk % C::NK;
          mbar_arrive_expect_tx(&k_full[st], C::kTileBytes);
#pragma unroll
          for (int a = 0; a < D / 64; ++a)
            tma_load_3d(sm + C::kK + st * C::kTileBytes + a * kAtom, &mapK, a * 64, (tile0 + nk) * kBM, bh, &k_full[st]);
          ++nk;
          progress = true;
        }
        if (nv < nk && (nv < C::NV || mbar_test_wait(smem_addr(&v_empty[nv % C::NV]), ((nv / C::NV) - 1) & 1))) {
          const int st = nv % C::NV;
          mbar_arrive_expect_tx(&v_full[st], C::kTileBytes);
#pragma unroll
          for (int a = 0; a < D / 64; ++a)
            tma_load_3d(sm + C::kV + st * C::kTileBytes + a * kAtom, &mapV, a * 64, (tile0 + nv) * kBM, bh, &v_full[st]);
          ++nv;
          progress = true;
        }
        if (progress) wd.progress();
        else ok = wd.idle();
      }
      // drain: the last loads of each ring have landed
      for (int x = max(0, nk - C::NK); x < nk; ++x) mbar_wait(&k_full[x % C::NK], (x / C::NK) & 1, wctx);
      for (int x = max(0, nv - C::NV); x < nv; ++x) mbar_wait(&v_full[x % C::NV], (x / C::NV) & 1, wctx);
    }
  } else if (warp == 1 || warp == kStateIssuer) {
    // two issuers: warp 1 the projections, warp 12 the state MMAs, so that
    // a tile's projection is never queued behind the previous tile's state
    // MMAs on one thread (issuing costs ~60 cycles per MMA)
    if (lane == 0) {
      constexpr uint32_t id_proj_all = idesc_f16(kBM, M, false, false);
      constexpr uint32_t id_state = idesc_bf16(kFB, D + 16, true, true);
      const uint32_t omega_a = smem_addr(sm + C::kOmega);
      const uint32_t ones_a = smem_addr(sm + C::kOnes);
      const bool proj = warp == 1;
      bool ok = mbar_wait(setup_bar, 0, wctx);
      Watchdog wd(wctx);
      int pi = 0, si = 0, sf = 0;
      while (ok && (proj ? pi < n_tiles : si < n_tiles)) {
        bool progress = false;
        if (proj) {
          // one N = m projection covers every block (half the MMA
          // instructions of one per block); it waits until every block's
          // previous tile was copied out
          const int ks = pi % C::NK;
          const bool ready = mbar_test_wait(smem_addr(&kn_full[pi % C::NN]), (pi / C::NN) & 1) &&
                             (pi == 0 || (mbar_test_wait(smem_addr(&p_free[0]), (pi - 1) & 1) &&
                                          (NFB == 1 || mbar_test_wait(smem_addr(&p_free[1]), (pi - 1) & 1))));
          if (ready) {
            tc_fence_after();
            const uint64_t a0 = sdesc(smem_addr(sm + C::kK + ks * C::kTileBytes), 16, 1024);
            const uint64_t b0 = sdesc(omega_a, 16, 1024);
#pragma unroll
            for (int k = 0; k < D / 16; ++k)
              mma_bf16(tmem, dadd(a0, kstep_k(k, kAtom)), dadd(b0, kstep_k(k, M * 128)), id_proj_all, k > 0);
            for (int f = 0; f < NFB; ++f) mma_commit(&p_full[f]);
            mma_commit(&k_empty[ks]);
            ++pi;
            progress = true;
          }
        } else {
          const int vs = si % C::NV;
          const bool ready = mbar_test_wait(smem_addr(&phi_full[sf]), si & 1) &&
                             (sf > 0 || mbar_test_wait(smem_addr(&v_full[vs]), (si / C::NV) & 1));
          if (ready) {
            tc_fence_after();
            const uint32_t v_a = smem_addr(sm + C::kV + vs * C::kTileBytes);
            const uint64_t a0 = sdesc(smem_addr(sm + C::kPhi + sf * 2 * kAtom), kAtom, 1024);
            const uint64_t b0 = sdesc(v_a, ones_a - v_a, 1024);
#pragma unroll
            for (int k = 0; k < kBM / 16; ++k)
              mma_bf16(tmem + S_COL + sf * 128, dadd(a0, kstep_mn(k)), vones_k(b0, k), id_state, (si > 0) || (k > 0));
            mma_commit(&phi_free[sf]);
            if (sf == NFB - 1) mma_commit(&v_empty[vs]);
            if (++sf == NFB) { sf = 0; ++si; }
            progress = true;
          }
        }
        if (progress) wd.progress();
        else ok = wd.idle();
      }
      mma_commit(&done_bar[proj ? 0 : 1]);
      mbar_wait(&done_bar[proj ? 0 : 1], 0, wctx);
    }
  } else if (warp < 2 + kNormWarps) {
    // squared norms of the K rows; K rewritten as fp16
    for (int i = 0; i < n_tiles; ++i) {
      const int ks = i % C::NK, ns = i % C::NN;
      if (!mbar_wait(&k_full[ks], (i / C::NK) & 1, wctx)) break;
      uint8_t* kt = sm + C::kK + ks * C::kTileBytes;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int r = (warp - 2) * 64 + lane + 32 * j;
        norm_s[ns * kBM + r] = tile_row_sq_to_f16<D>(kt, r);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&kn_full[ns]);
    }
  } else if (warp < kStateIssuer) {
    // ---------------- epilogue: two warpgroups x 128 lanes ----------------
    const int wg = (warp - 4) >> 2;
    const int q = warp & 3;
    const int t = q * 32 + lane;                   // token row of P, feature row of S~
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    const int col0 = wg * 64;                      // this warpgroup's columns of each feature block
    float R, W_unused;
    griddep_wait();   // the key reference comes from the preparation kernel
    key_reference(prm.key_ref, prm.m, &R, &W_unused);
    const float c1 = feature_c1<FM>(prm.scale);
    const float hs2 = 0.5f * prm.scale * prm.scale;
    bool ok = true;
    // m = 256: warpgroup w owns feature block w (128 columns in two passes),
    // so the two warps of an SMSP work on different blocks and fall out of
    // step (one exponentiates while the other loads or stores).  m = 128:
    // the warpgroups split the block's columns.
    const int my_fb = (NFB == 2) ? wg : 0;
    constexpr int kPasses = (NFB == 2) ? 2 : 1;
    const int c0 = (NFB == 2) ? 0 : col0;
    const uint32_t phi_a = smem_addr(sm + C::kPhi + my_fb * 2 * kAtom);
    for (int i = 0; ok && i < n_tiles; ++i) {
      const int ns = i % C::NN;
      if (!mbar_wait(&kn_full[ns], (i / C::NN) & 1, wctx)) { ok = false; break; }
      // rows past L get 2^-inf = 0
      const bool valid = (tile0 + i) * kBM + t < prm.L;
      const float bias = !valid ? INFINITY : (FM == FAVOR_FM_PRF ? (hs2 * norm_s[ns * kBM + t] + R) * kLog2e : 0.f);
      if (!mbar_wait(&p_full[my_fb], i & 1, wctx)) { ok = false; break; }
      tc_fence_after();
#pragma unroll
      for (int ps = 0; ps < kPasses; ++ps) {
        uint32_t x[64];
        tmem_ld64(tmem + lane_off + my_fb * kFB + c0 + 64 * ps, x);
        tmem_ld_wait();
        if (ps == kPasses - 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&p_free[my_fb]);
        }
        feature_pack<FM>(x, c1, bias);
        if (ps == 0 && i >= 1 && !mbar_wait(&phi_free[my_fb], (i - 1) & 1, wctx)) { ok = false; break; }
        store_row<32>(phi_a, kAtom, t, c0 + 64 * ps, x);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&phi_full[my_fb]);
    }
    // final state: lane f holds feature f of a block.  Two blocks: warpgroup
    // w reads block w; one block: the warpgroups split the d columns.
    const bool done = mbar_wait(&done_bar[1], 0, wctx);
    tc_fence_after();
    if (done && !*abort_flag) {
      const int sfb = (NFB == 2) ? wg : 0;
      float* dst = prm.partS + ((((size_t)bh * NFB + sfb) * prm.n_split + split) * (D + 1)) * kFB;
      const uint32_t s_col = tmem + lane_off + S_COL + sfb * 128;
#pragma unroll
      for (int cb = 0; cb < D / 32; ++cb) {
        if (NFB == 1 && (cb & 1) != wg) continue;
        uint32_t v[32];
        tmem_ld32(s_col + cb * 32, v);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) dst[(size_t)(cb * 32 + j) * kFB + t] = __uint_as_float(v[j]);
      }
      if (NFB == 2 || wg == 1) {
        uint32_t z[8];
        tmem_ld8(s_col + D, z);
        tmem_ld_wait();
        dst[(size_t)D * kFB + t] = __uint_as_float(z[0]);
      }
    }
    tc_fence_before();
    if (prm.merge) {
      named_bar(1, kEpiThreads);
      if (threadIdx.x == kEpiTid0) {
        __threadfence();
        const uint32_t old = atomicAdd(&prm.counters[bh], 1u);
        *is_last = (old == (uint32_t)(prm.n_split - 1)) ? 1 : 0;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
  // the last CTA of a head adds the splits' partial states (fixed split order)
  // into the bf16 state image read by the output kernel
  if (prm.merge && *is_last) {
    __threadfence();
    merge_partials<D, M>(prm.partS + (size_t)bh * NFB * prm.n_split * (D + 1) * kFB, prm.n_split, prm.n_split,
                         prm.state_img + (size_t)bh * M * (D + 16) * 2, threadIdx.x, kStateThreads,
                         prm.zvec != nullptr ? prm.zvec + (size_t)bh * M : nullptr);
    if (threadIdx.x == 0) prm.counters[bh] = 0;
  }
}

// ---------------------------------------------------------------------------
// bidirectional output kernel: one CTA per SM, each an even share of the
// (head, tile) list (a share may cross into the next head: the S~ image is
// reloaded).
// Query row reference: the row's largest exponent max_i s w_i.q, read from
// the projection tile in tensor memory before any feature is formed ("From
// Performer to Linear Attention", §Simple Derivation: any per-query constant
// cancels), so the largest phi(q) of every row is exactly 1 whatever the
// norm of q.  Each warpgroup holds half of a row's projections (one feature
// block each at m = 256, half the columns at m = 128); the two halves meet
// in shared memory.
// ---------------------------------------------------------------------------
struct OutParams {
  const float* key_ref;    // row-norm maxima (key_reference)
  const uint8_t* omega_img;
  const uint8_t* state_img;
  int32_t* status;
  int L, m;
  int n_heads;             // B H: the CTAs split the (head, tile) list evenly
  float scale;
};

constexpr int kOutThreads = 384;   // warps 0 TMA, 1 MMA, 2-3 norms, 4-11 epilogue

template <int D>
struct OutCfg {
  static constexpr int NSQ = 4;
  static constexpr int kTileBytes = D * kBM * 2;
  static constexpr int kOmega = 0;                          // fp16 image, up to 256 x D
  static constexpr int kState = kOmega + 256 * D * 2;       // bf16 S~ image, up to 256 x (D + 16)
  static constexpr int kQ = kState + 256 * (D + 16) * 2;
  static constexpr int kPhi = kQ + NSQ * kTileBytes;        // [fb][2 atoms][128][128 B]
  static constexpr int kOut = kPhi + 4 * kAtom;             // output staging tile
  static constexpr int kXmax = kOut + kTileBytes;           // [tile parity][warpgroup][128] row maxima
  static constexpr int kBars = kXmax + 2 * 2 * kBM * 4;
  static constexpr int kSmem = kBars + 512 + 1024;
};

template <int D, int M, int FM>
__global__ void __launch_bounds__(kOutThreads, 1) output_kernel(const __grid_constant__ CUtensorMap mapQ,
                                                                const __grid_constant__ CUtensorMap mapO,
                                                                OutParams prm) {
  using C = OutCfg<D>;
  constexpr int NFB = M / kFB;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::kBars);
  uint64_t* q_full = bars;                  // [NSQ]
  uint64_t* q_empty = q_full + C::NSQ;      // [NSQ] the tile's last projection has read it
  uint64_t* qn_full = q_empty + C::NSQ;     // [NSQ] Q rewritten as fp16
  uint64_t* p_full = qn_full + C::NSQ;      // [2] per feature block
  uint64_t* p_free = p_full + 2;            // [2]
  uint64_t* phi_full = p_free + 2;          // [2]
  uint64_t* phi_free = phi_full + 2;        // [2]
  uint64_t* o_full = phi_free + 2;          // [2]
  uint64_t* o_free = o_full + 2;            // [2]
  uint64_t* setup_bar = o_free + 2;
  uint64_t* done_bar = setup_bar + 1;
  uint64_t* img_full = done_bar + 1;        // phase k: the k-th head's S~ image landed
  uint64_t* img_free = img_full + 1;        // phase k: the k-th head's last output MMA is complete
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(img_free + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* xmax = reinterpret_cast<float*>(sm + C::kXmax);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // this CTA's tiles: the contiguous range [g0, g1) of the (head, tile) list,
  // which may cross from one head into the next (the S~ image is reloaded)
  const int nt = (prm.L + kBM - 1) / kBM;
  const long long total = (long long)prm.n_heads * nt;
  const int g0 = range_first(total, blockIdx.x, gridDim.x);
  const int g1 = range_first(total, blockIdx.x + 1, gridDim.x);
  const int n_tiles = g1 - g0;
  const int h0 = g0 / nt;
  const int n_heads = n_tiles > 0 ? (g1 - 1) / nt - h0 + 1 : 0;
  auto head_of = [&](int i) { return (g0 + i) / nt; };
  auto tile_of = [&](int i) { return (g0 + i) - head_of(i) * nt; };
  const WaitCtx wctx{abort_flag, prm.status};
  const uint32_t o_col[2] = {256u, 384u};   // O accumulators (d + 16 columns each); P at 0

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NSQ; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);
      mbar_init(&qn_full[i], kNormWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&p_full[i], 1);
      mbar_init(&p_free[i], kEpiWarps / NFB);     // the warps that own block i
      mbar_init(&phi_full[i], kEpiWarps / NFB);
      mbar_init(&phi_free[i], 1);
      mbar_init(&o_full[i], 1);
      mbar_init(&o_free[i], kEpiWarps);
    }
    mbar_init(setup_bar, 1);
    mbar_init(done_bar, 1);
    mbar_init(img_full, 1);
    mbar_init(img_free, 1);
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
      const uint32_t ob = M * D * 2, sb = M * (D + 16) * 2;
      mbar_arrive_expect_tx(setup_bar, ob);
      bulk_load(sm + C::kOmega, prm.omega_img, ob, setup_bar);
      // head k's S~ image goes in once head k - 1's last output MMA is complete
      auto load_head = [&](int k) {
        mbar_arrive_expect_tx(img_full, sb);
        bulk_load(sm + C::kState, prm.state_img + (size_t)(h0 + k) * sb, sb, img_full);
      };
      int ni = 0;
      if (n_heads > 0) load_head(ni++);
      Watchdog wd(wctx);
      int nq = 0;
      bool ok = true;
      while (ok && (nq < n_tiles || ni < n_heads)) {
        bool progress = false;
        if (nq < n_tiles && (nq < C::NSQ || mbar_test_wait(smem_addr(&q_empty[nq % C::NSQ]), ((nq / C::NSQ) - 1) & 1))) {
          const int st = nq % C::NSQ;
          mbar_arrive_expect_tx(&q_full[st], C::kTileBytes);
          uint8_t* qt = sm + C::kQ + st * C::kTileBytes;
#pragma unroll
          for (int a = 0; a < D / 64; ++a)
            tma_load_3d(qt + a * kAtom, &mapQ, a * 64, tile_of(nq) * kBM, head_of(nq), &q_full[st]);
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
      for (int x = max(0, nq - C::NSQ); x < nq; ++x) mbar_wait(&q_full[x % C::NSQ], (x / C::NSQ) & 1, wctx);
      if (ni > 0) mbar_wait(img_full, (ni - 1) & 1, wctx);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t id_proj_all = idesc_f16(kBM, M, false, false);
      constexpr uint32_t id_out = idesc_bf16(kBM, D + 16, false, false);
      const uint32_t omega_a = smem_addr(sm + C::kOmega);
      const uint32_t state_a = smem_addr(sm + C::kState);
      bool ok = mbar_wait(setup_bar, 0, wctx);
      // event-driven issue: the next projection step (tile, block) and the
      // next output step (tile, block) are each issued as soon as their
      // inputs are ready, projections first
      Watchdog wd(wctx);
      int pi = 0, oi = 0, of = 0;
      while (ok && (pi < n_tiles || oi < n_tiles)) {
        bool progress = false;
        if (pi < n_tiles) {
          // one projection of N = m covers every block (see the state kernel)
          const int st = pi % C::NSQ;
          const bool ready = mbar_test_wait(smem_addr(&qn_full[st]), (pi / C::NSQ) & 1) &&
                             (pi == 0 || (mbar_test_wait(smem_addr(&p_free[0]), (pi - 1) & 1) &&
                                          (NFB == 1 || mbar_test_wait(smem_addr(&p_free[1]), (pi - 1) & 1))));
          if (ready) {
            tc_fence_after();
            const uint64_t a0 = sdesc(smem_addr(sm + C::kQ + st * C::kTileBytes), 16, 1024);
            const uint64_t b0 = sdesc(omega_a, 16, 1024);
#pragma unroll
            for (int k = 0; k < D / 16; ++k)
              mma_bf16(tmem, dadd(a0, kstep_k(k, kAtom)), dadd(b0, kstep_k(k, M * 128)), id_proj_all, k > 0);
            for (int f = 0; f < NFB; ++f) mma_commit(&p_full[f]);
            mma_commit(&q_empty[st]);
            ++pi;
            progress = true;
          }
        }
        if (oi < n_tiles) {
          const int ob = oi & 1;
          const bool ready = mbar_test_wait(smem_addr(&phi_full[of]), oi & 1) &&
                             mbar_test_wait(smem_addr(img_full), (head_of(oi) - h0) & 1) &&
                             (of > 0 || oi < 2 || mbar_test_wait(smem_addr(&o_free[ob]), ((oi >> 1) - 1) & 1));
          if (ready) {
            tc_fence_after();
            const uint64_t a0 = sdesc(smem_addr(sm + C::kPhi + of * 2 * kAtom), 16, 1024);
            const uint64_t b0 = sdesc(state_a + of * 2 * (D + 16) * 128, 16, 1024);
#pragma unroll
            for (int kk = 0; kk < kFB / 16; ++kk)
              mma_bf16(tmem + o_col[ob], dadd(a0, kstep_k(kk, kAtom)), dadd(b0, kstep_k(kk, (D + 16) * 128)), id_out,
                       (of > 0) || (kk > 0));
            mma_commit(&phi_free[of]);
            if (of == NFB - 1) {
              mma_commit(&o_full[ob]);
              // the head's last tile: its S~ image may be replaced
              if (oi == n_tiles - 1 || head_of(oi + 1) != head_of(oi)) mma_commit(img_free);
            }
            if (++of == NFB) { of = 0; ++oi; }
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
    // Q rewritten as fp16 for the projection (its norm is not needed: the
    // query reference comes from the projections themselves)
    for (int i = 0; i < n_tiles; ++i) {
      const int st = i % C::NSQ;
      if (!mbar_wait(&q_full[st], (i / C::NSQ) & 1, wctx)) break;
      uint8_t* qt = sm + C::kQ + st * C::kTileBytes;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int r = (warp - 2) * 64 + lane + 32 * j;
        (void)tile_row_sq_to_f16<D>(qt, r);
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
    const int col0 = wg * 64;                      // this warpgroup's columns of each feature block
    const float c1 = feature_c1<FM>(prm.scale);
    const uint32_t out_a = smem_addr(sm + C::kOut);
    bool ok = true;
    auto store_out = [&](int j) {
      const int ob = j & 1;
      const bool have = ok && mbar_wait(&o_full[ob], (j >> 1) & 1, wctx);
      tc_fence_after();
      uint32_t v[32], z[8];
      if (have) {
        tmem_ld32(tmem + lane_off + o_col[ob] + wg * 32, v);
        tmem_ld8(tmem + lane_off + o_col[ob] + D, z);
        tmem_ld_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&o_free[ob]);
      const float den = have ? __uint_as_float(z[0]) : 1.f;
      const int row = tile_of(j) * kBM + t;
      if (have && row < prm.L && (!(den > 0.f) || !isfinite(den))) report_status(prm.status, FAVOR_ERR_NONFINITE);
      const float inv = __fdividef(1.0f, den);
      if (threadIdx.x == kEpiTid0 && j > 0) bulk_wait_read0();   // previous store has left the staging tile
      named_bar(1, kEpiThreads);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int chunk = wg * 4 + c;
        const int o = c * 8;
        st_shared_v4(out_a + t * 128 + ((chunk ^ (t & 7)) << 4),
                     pack_bf16(__uint_as_float(v[o]) * inv, __uint_as_float(v[o + 1]) * inv),
                     pack_bf16(__uint_as_float(v[o + 2]) * inv, __uint_as_float(v[o + 3]) * inv),
                     pack_bf16(__uint_as_float(v[o + 4]) * inv, __uint_as_float(v[o + 5]) * inv),
                     pack_bf16(__uint_as_float(v[o + 6]) * inv, __uint_as_float(v[o + 7]) * inv));
      }
      fence_proxy_async_smem();
      named_bar(1, kEpiThreads);
      if (threadIdx.x == kEpiTid0 && have && !*abort_flag) {
        tma_store_3d(&mapO, 0, tile_of(j) * kBM, head_of(j), sm + C::kOut);
        bulk_commit();
      }
    };
    for (int i = 0; i < n_tiles; ++i) {
      const int my_fb = (NFB == 2) ? wg : 0;   // m = 256: warpgroup w owns feature block w
      if (ok) ok = mbar_wait(&p_full[my_fb], i & 1, wctx);
      // m = 256: two passes of 64 columns over the owned block; m = 128: the
      // warpgroups split the block's columns
      constexpr int kPasses = (NFB == 2) ? 2 : 1;
      const int c0 = (NFB == 2) ? 0 : col0;
      tc_fence_after();
      float bias = 0.f;
      if constexpr (FM == FAVOR_FM_PRF) {
        // the row's largest projection: this thread's columns, then the
        // other warpgroup's half through shared memory (parity-buffered by
        // tile, so a slot is rewritten only after both halves passed the
        // next tile's barrier)
        float pm = -INFINITY;
#pragma unroll
        for (int ps = 0; ps < kPasses; ++ps) {
          uint32_t x[64];
          if (ok) {
            tmem_ld64(tmem + lane_off + my_fb * kFB + c0 + 64 * ps, x);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 64; ++j) pm = fmaxf(pm, __uint_as_float(x[j]));
          }
        }
        float* xm = xmax + (i & 1) * 2 * kBM;
        xm[wg * kBM + t] = pm;
        named_bar(2, kEpiThreads);
        bias = fmaxf(xm[t], xm[kBM + t]) * c1;
      }
#pragma unroll
      for (int ps = 0; ps < kPasses; ++ps) {
        uint32_t x[64];
        if (ok) {
          tmem_ld64(tmem + lane_off + my_fb * kFB + c0 + 64 * ps, x);
          tmem_ld_wait();
        }
        if (ps == kPasses - 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&p_free[my_fb]);
        }
        if (ok) {
          feature_pack<FM>(x, c1, bias);
          if (ps == 0 && i >= 1) ok = mbar_wait(&phi_free[my_fb], (i - 1) & 1, wctx);
          if (ok) store_row<32>(smem_addr(sm + C::kPhi + my_fb * 2 * kAtom), kAtom, t, c0 + 64 * ps, x);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&phi_full[my_fb]);
      if (i >= 1) store_out(i - 1);
    }
    if (n_tiles >= 1) store_out(n_tiles - 1);
    if (threadIdx.x == kEpiTid0) bulk_wait0();
    mbar_wait(done_bar, 0, wctx);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------------------
// causal kernel: CTA = one superchunk of one head, walking 128-token chunks.
// G (m x (d+16), fp32) lives in tensor memory; it starts as the sum, in
// order, of the partial states of the sub-splits of the earlier superchunks.  Per chunk c and 128-feature block fb:
//   phi(K_c)_fb and G_s,fb <- bf16(G_fb), side by side in one operand;
//   phi(Q_c)_fb                                                   (CUDA cores)
//   G_fb += phi(K_c)_fb^T [V_c | 1];
//   [A | O] += phi(Q_c)_fb [phi(K_c)_fb^T | G_s,fb]              (tensor cores)
// then A's upper triangle is zeroed (diagonal kept), O += A [V_c | 1], and
// O is divided by its normaliser column.  The query row reference is the
// row's largest exponent max_i s w_i.q ("From Performer to Linear
// Attention", §Simple Derivation: a per-query constant cancels), so the
// largest phi(q) of each row is at least 1 at any input norm.  The tile X
// holds one feature block at a time, so the reference is block 0's row
// maximum c_0; a later block whose maximum c_b exceeds the reference by more
// than 20 nats (its features would pass e^20) moves the row's reference to
// c_b, and the row's accumulated A and O are first scaled by
// exp(c_ref - c_b) in tensor memory (the previous [A|O] step is complete by
// then: phi(Q) has a single buffer).
// ---------------------------------------------------------------------------
struct CausalParams {
  const float* key_ref;   // row-norm maxima (key_reference)
  const uint8_t* omega_img;
  const float* pre;       // [BH][n_fb][n_sc][d+1][128] initial states (superchunks > 0), or null:
  const float* partS;     // then [BH][n_fb][n_split][d+1][128] partials summed here
  int32_t* status;
  int L, m, n_sc, tiles_per_sc, n_split, sub_per_sc;
  float scale;
};

constexpr int kCausalThreads = 384;   // warps 0 TMA, 1 MMA, 2-3 norms, 4-11 epilogue

template <int D>
struct CausalCfg {
  static constexpr int kTileBytes = D * kBM * 2;
  static constexpr int kSlots = 4;                                  // ring of K, Q, V tiles
  static constexpr int kKGRows = kBM + D + 16;                      // phi(K) tokens, then G_s columns
  static constexpr int kKGAtom = kKGRows * 128;
  static constexpr int kOmega = 0;                                  // fp16 image, up to 256 x D
  static constexpr int kRing = kOmega + 256 * D * 2;                // tile x of the sequence K0 Q0 V0 K1 .. in slot x % 4
  static constexpr int kOnes = kRing + kSlots * kTileBytes;         // above every V tile
  static constexpr int kKG = kOnes + kOnesBytes;                    // [2 atoms][kKGRows][128 B]
  static constexpr int kPhiQ = kKG + 2 * kKGAtom;                   // [2 atoms][128][128 B]
  static constexpr int kMA = kPhiQ + 2 * kAtom;                     // masked A; also the output staging tile
  static constexpr int kNorm = kMA + 2 * kAtom;                     // [2 chunks][128] squared key norms
  static constexpr int kXmax = kNorm + 2 * kBM * 4;                 // [chunk parity][warpgroup][128] row maxima
  static constexpr int kBars = kXmax + 2 * 2 * kBM * 4;
  static constexpr int kSmem = kBars + 512 + 1024;
};
static_assert(CausalCfg<64>::kSmem <= 232448, "shared memory");
static_assert(StateCfg<64>::kSmem <= 232448, "shared memory");

template <int D, int M, int FM>
__global__ void __launch_bounds__(kCausalThreads, 1) causal_kernel(const __grid_constant__ CUtensorMap mapQ,
                                                                   const __grid_constant__ CUtensorMap mapK,
                                                                   const __grid_constant__ CUtensorMap mapV,
                                                                   const __grid_constant__ CUtensorMap mapO,
                                                                   CausalParams prm) {
  using C = CausalCfg<D>;
  constexpr int NFB = M / kFB;
  constexpr int GN = D + 16;                    // columns of G and of [V | 1]
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* b = reinterpret_cast<uint64_t*>(sm + C::kBars);
  uint64_t *slot_full = b + 0, *slot_free = b + 4;                   // [kSlots]
  uint64_t *kn_full = b + 8, *qn_full = b + 10;                      // [chunk parity]
  uint64_t *pk_full = b + 12, *pq_full = b + 13, *x_free = b + 14;
  uint64_t *kg_full = b + 15, *phiq_full = b + 16, *kg_free = b + 17, *phiq_free = b + 18;
  uint64_t *gdone = b + 19;                                          // [feature block]
  uint64_t *a_full = b + 21, *as_full = b + 22, *o_full = b + 23, *o_free = b + 24;
  uint64_t *setup_bar = b + 25, *done_bar = b + 26;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(b + 27);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* norms = reinterpret_cast<float*>(sm + C::kNorm);   // [c&1][128]
  float* xmax = reinterpret_cast<float*>(sm + C::kXmax);
  constexpr int XS = 2 * NFB;                   // uses of the projection tile X per chunk

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sc = blockIdx.x, bh = blockIdx.y;
  const int n_tiles_total = (prm.L + kBM - 1) / kBM;
  const int tile0 = sc * prm.tiles_per_sc;
  const int n_chunks = min(prm.tiles_per_sc, n_tiles_total - tile0);
  const WaitCtx wctx{abort_flag, prm.status};
  // TMEM columns: X (one projection block), A (chunk scores) and O side by
  // side, then G_fb at G_COL + fb * GN
  constexpr uint32_t X_COL = 0, A_COL = 128, O_COL = 256, G_COL = 336;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2 * C::kSlots; ++i) mbar_init(&b[i], 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&kn_full[i], kNormWarps);
      mbar_init(&qn_full[i], kNormWarps);
      mbar_init(&gdone[i], 1);
    }
    mbar_init(pk_full, 1);
    mbar_init(pq_full, 1);
    mbar_init(x_free, kEpiWarps);
    mbar_init(kg_full, kEpiWarps);
    mbar_init(phiq_full, kEpiWarps);
    mbar_init(kg_free, 1);
    mbar_init(phiq_free, 1);
    mbar_init(a_full, 1);
    mbar_init(as_full, kEpiWarps);
    mbar_init(o_full, 1);
    mbar_init(o_free, kEpiWarps);
    mbar_init(setup_bar, 1);
    mbar_init(done_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (warp >= 4) {
    fill_ones_block(sm + C::kOnes, kEpiTid0, kEpiThreads);
    // G_s rows D + 8 .. D + 15 of both atoms: zero for the whole kernel
    for (int e = threadIdx.x - kEpiTid0; e < 2 * 8 * 8; e += kEpiThreads) {
      const int atom = e >> 6, row = kBM + D + 8 + ((e >> 3) & 7);
      *reinterpret_cast<uint4*>(sm + C::kKG + atom * C::kKGAtom + row * 128 + (e & 7) * 16) = make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      prefetch_tmap(&mapQ);
      prefetch_tmap(&mapK);
      prefetch_tmap(&mapV);
      prefetch_tmap(&mapO);
      mbar_arrive_expect_tx(setup_bar, M * D * 2);
      bulk_load(sm + C::kOmega, prm.omega_img, M * D * 2, setup_bar);
      // tile x = 3c + (0: K, 1: Q, 2: V) of chunk c goes to slot x % 4 once
      // the tile four places earlier has been consumed
      const int n_x = 3 * n_chunks;
      for (int x = 0; x < n_x; ++x) {
        const int s_ = x % C::kSlots, c = x / 3, kind = x % 3;
        if (x >= C::kSlots && !mbar_wait(&slot_free[s_], ((x / C::kSlots) - 1) & 1, wctx)) break;
        mbar_arrive_expect_tx(&slot_full[s_], C::kTileBytes);
        const CUtensorMap* map = kind == 0 ? &mapK : (kind == 1 ? &mapQ : &mapV);
        for (int a = 0; a < D / 64; ++a)
          tma_load_3d(sm + C::kRing + s_ * C::kTileBytes + a * kAtom, map, a * 64, (tile0 + c) * kBM, bh,
                      &slot_full[s_]);
      }
      // drain: the last loads have landed
      for (int x = max(0, n_x - C::kSlots); x < n_x; ++x)
        mbar_wait(&slot_full[x % C::kSlots], (x / C::kSlots) & 1, wctx);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t id_proj = idesc_f16(kBM, kFB, false, false);
      constexpr uint32_t id_g = idesc_bf16(kFB, GN, true, true);
      constexpr uint32_t id_ao = idesc_bf16(kBM, kBM + GN, false, false);
      constexpr uint32_t id_oi = idesc_bf16(kBM, GN, false, true);
      const uint32_t om_a = smem_addr(sm + C::kOmega), ones_a = smem_addr(sm + C::kOnes);
      const uint32_t ring_a = smem_addr(sm + C::kRing);
      auto slot_of = [](int c, int kind) { return (3 * c + kind) % C::kSlots; };
      const uint32_t kg_a = smem_addr(sm + C::kKG), phiq_a = smem_addr(sm + C::kPhiQ);
      const uint32_t ma_a = smem_addr(sm + C::kMA);
      bool ok = mbar_wait(setup_bar, 0, wctx);
      auto ready = [](uint64_t* bar, int parity) { return mbar_test_wait(smem_addr(bar), parity & 1); };
      // Event-driven issue.  The projection tile X is used in a fixed order
      // per chunk c: P_K(c, fb), P_Q(c, fb) per block; each use waits until
      // the epilogue copied the previous one out.  G(u)
      // after phi(K)_u and G_s are in the KG slot; [A|O](u) after G(u) and
      // phi(Q)_u; O += mask(A) V after the chunk's last [A|O] and the masked
      // tile.  Each kind is probed only once its predecessor has been issued,
      // so no barrier can be two phases ahead.
      Watchdog wd(wctx);
      int nx = 0, npk = 0, npq = 0, ng = 0, nao = 0, noi = 0;
      const int n_x = n_chunks * XS;
      while (ok && noi < n_chunks) {
        bool progress = false;
        // a chunk's first use of X waits until the previous chunk's last
        // [A|O] is issued: queued ahead of it, it would delay the scores the
        // epilogue is waiting for
        if (nx < n_x) {
          const int c = nx / XS, r = nx % XS;
          const int fb = r >> 1;
          const bool is_k = (r & 1) == 0;
          const bool order_ok = r != 0 || nao >= c * NFB;
          const bool x_ok = nx == 0 || ready(x_free, (nx - 1) & 1);
          const bool in_ok = is_k ? ready(&kn_full[c & 1], c >> 1) : ready(&qn_full[c & 1], c >> 1);
          if (order_ok && x_ok && in_ok) {
            tc_fence_after();
            const uint64_t a0 = sdesc(ring_a + slot_of(c, is_k ? 0 : 1) * C::kTileBytes, 16, 1024);
            const uint64_t b0 = sdesc(om_a + fb * kFB * 128, 16, 1024);
#pragma unroll
            for (int k = 0; k < D / 16; ++k)
              mma_bf16(tmem + X_COL, dadd(a0, kstep_k(k, kAtom)), dadd(b0, kstep_k(k, M * 128)), id_proj, k > 0);
            if (is_k) {
              mma_commit(pk_full);
              if (fb == NFB - 1) mma_commit(&slot_free[slot_of(c, 0)]);
              ++npk;
            } else {
              mma_commit(pq_full);
              if (fb == NFB - 1) mma_commit(&slot_free[slot_of(c, 1)]);
              ++npq;
            }
            ++nx;
            progress = true;
          }
        }
        if (ng < npk) {
          const int c = ng / NFB, fb = ng % NFB;
          const int vs = slot_of(c, 2);
          if (ready(kg_full, ng) && (fb != 0 || ready(&slot_full[vs], (3 * c + 2) / C::kSlots))) {
            tc_fence_after();
            const uint32_t v_a = ring_a + vs * C::kTileBytes;
            const uint64_t a0 = sdesc(kg_a, C::kKGAtom, 1024), b0 = sdesc(v_a, ones_a - v_a, 1024);
#pragma unroll
            for (int k = 0; k < kBM / 16; ++k)
              mma_bf16(tmem + G_COL + fb * GN, dadd(a0, kstep_mn(k)), vones_k(b0, k), id_g, true);
            mma_commit(&gdone[fb]);
            ++ng;
            progress = true;
          }
        }
        if (nao < ng && nao < npq) {
          const int c = nao / NFB, fb = nao % NFB;
          if (ready(phiq_full, nao) && (fb != 0 || c == 0 || ready(o_free, c - 1))) {
            tc_fence_after();
            const uint64_t a0 = sdesc(phiq_a, 16, 1024), b0 = sdesc(kg_a, 16, 1024);
#pragma unroll
            for (int k = 0; k < kFB / 16; ++k)
              mma_bf16(tmem + A_COL, dadd(a0, kstep_k(k, kAtom)), dadd(b0, kstep_k(k, C::kKGAtom)), id_ao,
                       (fb > 0) || (k > 0));
            mma_commit(kg_free);
            mma_commit(phiq_free);
            if (fb == NFB - 1) mma_commit(a_full);
            ++nao;
            progress = true;
          }
        }
        if ((noi + 1) * NFB <= nao && ready(as_full, noi)) {
          tc_fence_after();
          const uint32_t v_a = ring_a + slot_of(noi, 2) * C::kTileBytes;
          const uint64_t a0 = sdesc(ma_a, 16, 1024), b0 = sdesc(v_a, ones_a - v_a, 1024);
#pragma unroll
          for (int k = 0; k < kBM / 16; ++k)
            mma_bf16(tmem + O_COL, dadd(a0, kstep_k(k, kAtom)), vones_k(b0, k), id_oi, true);
          mma_commit(o_full);
          mma_commit(&slot_free[slot_of(noi, 2)]);
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
    // squared row norms of K_c (double-buffered by chunk parity); K_c and
    // Q_c rewritten as fp16
    for (int c = 0; c < n_chunks; ++c) {
      float* nk = norms + (c & 1) * kBM;
      const int ks = (3 * c) % C::kSlots, qs = (3 * c + 1) % C::kSlots;
      if (!mbar_wait(&slot_full[ks], ((3 * c) / C::kSlots) & 1, wctx)) break;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int r = (warp - 2) * 64 + lane + 32 * j;
        nk[r] = tile_row_sq_to_f16<D>(sm + C::kRing + ks * C::kTileBytes, r);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&kn_full[c & 1]);
      if (!mbar_wait(&slot_full[qs], ((3 * c + 1) / C::kSlots) & 1, wctx)) break;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int r = (warp - 2) * 64 + lane + 32 * j;
        (void)tile_row_sq_to_f16<D>(sm + C::kRing + qs * C::kTileBytes, r);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&qn_full[c & 1]);
    }
  } else {
    // ---------------- epilogue ----------------
    const int wg = (warp - 4) >> 2;
    const int q = warp & 3;
    const int t = q * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    float R, W_unused;
    key_reference(prm.key_ref, prm.m, &R, &W_unused);
    const float c1 = feature_c1<FM>(prm.scale);
    const float hs2 = 0.5f * prm.scale * prm.scale;
    const uint32_t kg_a = smem_addr(sm + C::kKG), phiq_a = smem_addr(sm + C::kPhiQ);
    const uint32_t ma_a = smem_addr(sm + C::kMA);
    const int col0 = wg * 64;                 // this warpgroup's 64 of a block's 128 columns
    // G columns of this warpgroup: 0..47 or 48..GN-1
    constexpr int kG0 = 48;
    const int n0 = wg ? kG0 : 0;
    const int ng16 = wg ? (GN - kG0) / 16 : kG0 / 16;
    // G_s groups of 8 columns copied per chunk: n < D + 8 (the normaliser
    // column D and zeros), split between the two warpgroups
    constexpr int kGGroups = D / 8 + 1;
    const int g_first = wg ? (kGGroups + 1) / 2 : 0;
    const int g_end = wg ? kGGroups : (kGGroups + 1) / 2;
    // G_init: the superchunk's initial state, the fixed-order sum of the
    // earlier superchunks' partial states: formed by the prefix kernel when
    // the later superchunks have many, summed here in the same order (so to
    // the same bits) when every superchunk has at most a few; all of this
    // thread's loads of a partial in flight together
    for (int fb = 0; fb < NFB; ++fb) {
      constexpr int kMaxG = (kG0 > GN - kG0 ? kG0 : GN - kG0) / 16;
      float acc[kMaxG][16];
      if (prm.pre != nullptr) {
        const float* src = prm.pre + (((size_t)bh * NFB + fb) * prm.n_sc + sc) * (D + 1) * kFB;
#pragma unroll
        for (int g = 0; g < kMaxG; ++g)
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int n = n0 + 16 * g + j;
            acc[g][j] = (sc > 0 && g < ng16 && n <= D) ? src[(size_t)n * kFB + t] : 0.f;
          }
      } else {
#pragma unroll
        for (int g = 0; g < kMaxG; ++g)
#pragma unroll
          for (int j = 0; j < 16; ++j) acc[g][j] = 0.f;
        const float* src = prm.partS + ((size_t)bh * NFB + fb) * max(prm.n_split, 1) * (D + 1) * kFB;
        const int np = sc * prm.sub_per_sc;
        for (int p = 0; p < np; p += 2) {   // two partials' loads in flight, added in order
          float v[2][kMaxG][16];
#pragma unroll
          for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int g = 0; g < kMaxG; ++g)
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const int n = n0 + 16 * g + j;
                v[u][g][j] = (p + u < np && g < ng16 && n <= D) ? src[((size_t)(p + u) * (D + 1) + n) * kFB + t] : 0.f;
              }
#pragma unroll
          for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int g = 0; g < kMaxG; ++g)
#pragma unroll
              for (int j = 0; j < 16; ++j)
                if (p + u < np) acc[g][j] += v[u][g][j];
        }
      }
#pragma unroll
      for (int g = 0; g < kMaxG; ++g) {
        if (g >= ng16) break;
        uint32_t r[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) r[j] = __float_as_uint(acc[g][j]);
        tmem_st16(tmem + lane_off + G_COL + fb * GN + n0 + 16 * g, r);
      }
    }
    tmem_st_wait();
    // the G_s copies below read columns the other warpgroup stored
    tc_fence_before();
    named_bar(1, kEpiThreads);
    tc_fence_after();
    bool ok = true;
    auto out = [&](int j) {
      const bool have = ok && mbar_wait(o_full, j & 1, wctx);
      tc_fence_after();
      uint32_t v[32], z[8];
      tmem_ld32(tmem + lane_off + O_COL + wg * 32, v);
      tmem_ld8(tmem + lane_off + O_COL + D, z);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(o_free);
      const float den = have ? __uint_as_float(z[0]) : 1.f;
      if (have && (tile0 + j) * kBM + t < prm.L && (!(den > 0.f) || !isfinite(den)))
        report_status(prm.status, FAVOR_ERR_NONFINITE);
      const float inv = __fdividef(1.0f, den);
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        const int chunk = wg * 4 + cc;
        const int o = cc * 8;
        st_shared_v4(ma_a + t * 128 + ((chunk ^ (t & 7)) << 4),
                     pack_bf16(__uint_as_float(v[o]) * inv, __uint_as_float(v[o + 1]) * inv),
                     pack_bf16(__uint_as_float(v[o + 2]) * inv, __uint_as_float(v[o + 3]) * inv),
                     pack_bf16(__uint_as_float(v[o + 4]) * inv, __uint_as_float(v[o + 5]) * inv),
                     pack_bf16(__uint_as_float(v[o + 6]) * inv, __uint_as_float(v[o + 7]) * inv));
      }
      fence_proxy_async_smem();
      named_bar(1, kEpiThreads);
      if (threadIdx.x == kEpiTid0 && have && !*abort_flag) {
        tma_store_3d(&mapO, 0, (tile0 + j) * kBM, bh, sm + C::kMA);
        bulk_commit();
      }
    };
    // the row's largest query projection in block u, this thread's columns
    // and then the other warpgroup's half through shared memory (slots
    // parity-buffered by block step: a slot is rewritten only after both
    // halves passed the next exchange)
    auto row_max = [&](int u, float pm) {
      float* xm = xmax + (u & 1) * 2 * kBM;
      xm[wg * kBM + t] = pm;
      named_bar(2, kEpiThreads);
      return fmaxf(xm[t], xm[kBM + t]);
    };
    auto max64 = [](const uint32_t (&x)[64]) {
      float pm = -INFINITY;
#pragma unroll
      for (int j = 0; j < 64; ++j) pm = fmaxf(pm, __uint_as_float(x[j]));
      return pm;
    };
    // the row's reference (largest raw projection so far in log2 units, times c1)
    float bias_q = 0.f;
    // a later block may exceed the reference by this much before the row is
    // rescaled: its features stay below e^20
    const float kRescale = 20.0f * kLog2e;
    // this warpgroup's columns of A (col0 .. col0 + 63) and of O (32 of the
    // first 64 and 8 of the last 16; warpgroup 0's 8 hold the normaliser),
    // each access aligned to its width
    const uint32_t a_cols = tmem + lane_off + A_COL + col0;
    const uint32_t o_cols = tmem + lane_off + O_COL + wg * 32;
    const uint32_t o_tail = tmem + lane_off + O_COL + D + wg * 8;
    static_assert(GN - D == 16, "O tail");
    for (int c = 0; c < n_chunks; ++c) {
      const bool valid = (tile0 + c) * kBM + t < prm.L;
      const float* nk = norms + (c & 1) * kBM;
      for (int fb = 0; fb < NFB; ++fb) {
        const int u = c * NFB + fb;
        // ---- phi(K)_fb and G_s,fb ----
        if (ok) ok = mbar_wait(pk_full, u & 1, wctx);
        if (ok && fb == 0) ok = mbar_wait(&kn_full[c & 1], (c >> 1) & 1, wctx);
        // rows past the sequence end: an infinite bias makes their features 0
        const float bias_k = !valid ? INFINITY : (FM == FAVOR_FM_PRF ? (hs2 * nk[t] + R) * kLog2e : 0.f);
        tc_fence_after();
        {
          // loaded even after a failed wait (the kernel is then aborting and the
          // values are dropped): a conditional load keeps both paths' registers live
          uint32_t x[64];
          tmem_ld64(tmem + lane_off + X_COL + col0, x);
          tmem_ld_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(x_free);
          if (ok) feature_pack<FM>(x, c1, bias_k);
          if (ok && u >= 1) ok = mbar_wait(kg_free, (u - 1) & 1, wctx);
          if (ok && c >= 1) ok = mbar_wait(&gdone[fb], (c - 1) & 1, wctx);
          tc_fence_after();
          if (ok) store_row<32>(kg_a, C::kKGAtom, t, col0, x);
        }
        if (ok) {
          // G_s,fb rows 128 + n for n < D + 8 (rows D + 1 .. stay zero: G's
          // columns there are zero), three column groups' loads in flight
          const int f0 = 32 * q + 8 * (lane >> 3);
          tmem_state_to_rows<3>(tmem, G_COL + fb * GN, q, lane, g_first, g_end,
                                kg_a + (f0 >> 6) * C::kKGAtom + kBM * 128);
        }
        tc_fence_before();
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(kg_full);
        // the previous chunk's output, deferred so that its MMAs overlap
        if (fb == 0 && c >= 1) {
          out(c - 1);
        }
        // ---- phi(Q)_fb ----
        if (ok) ok = mbar_wait(pq_full, u & 1, wctx);
        tc_fence_after();
        {
          // loaded even after a failed wait (the kernel is then aborting and the
          // values are dropped): a conditional load keeps both paths' registers live
          uint32_t x[64];
          tmem_ld64(tmem + lane_off + X_COL + col0, x);
          tmem_ld_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(x_free);
          float shrink = 1.f;   // factor on the row's A and O so far (block > 0)
          if constexpr (FM == FAVOR_FM_PRF) {
            const float bm = row_max(u, max64(x)) * c1;
            if (fb == 0) {
              bias_q = bm;
            } else if (bm > bias_q + kRescale) {
              shrink = ex2(bias_q - bm);
              bias_q = bm;
            }
          }
          if (ok) feature_pack<FM>(x, c1, bias_q);
          // [A|O] of the previous block is complete once phi(Q)'s buffer is free
          if (ok && u >= 1) ok = mbar_wait(phiq_free, (u - 1) & 1, wctx);
          if (fb > 0 && __any_sync(0xffffffffu, shrink != 1.f)) {
            tc_fence_after();
            uint32_t r[32], z8[8];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              tmem_ld32(a_cols + 32 * h, r);
              tmem_ld_wait();
#pragma unroll
              for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * shrink);
              tmem_st32(a_cols + 32 * h, r);
            }
            tmem_ld32(o_cols, r);
            tmem_ld8(o_tail, z8);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * shrink);
#pragma unroll
            for (int j = 0; j < 8; ++j) z8[j] = __float_as_uint(__uint_as_float(z8[j]) * shrink);
            tmem_st32(o_cols, r);
            tmem_st8(o_tail, z8);
            tmem_st_wait();
            tc_fence_before();
          }
          if (ok) store_row<32>(phiq_a, kAtom, t, col0, x);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(phiq_full);
      }
      // ---- masked A -> bf16 (the staging tile of the previous store) ----
      if (ok) ok = mbar_wait(a_full, c & 1, wctx);
      tc_fence_after();
      {
        uint32_t a[64];
        tmem_ld64(tmem + lane_off + A_COL + col0, a);
        tmem_ld_wait();
        tc_fence_before();
        if (threadIdx.x == kEpiTid0 && c >= 1) bulk_wait_read0();
        named_bar(1, kEpiThreads);
        if (ok) {
          // this warp's rows 32q .. 32q+31 against columns col0 .. col0+63:
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
              a[j] = pack_bf16(f <= t ? __uint_as_float(a[2 * j]) : 0.f,
                               f + 1 <= t ? __uint_as_float(a[2 * j + 1]) : 0.f);
            }
          }
          store_row<32>(ma_a, kAtom, t, col0, a);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(as_full);
    }
    if (n_chunks >= 1) out(n_chunks - 1);
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
template <int D, int M, int FM>
cudaError_t launch_state(const void* K, const void* V, const Shape& s, const TcPlan& p, float scale, char* ws,
                         int32_t* status, cudaStream_t stream, float* zvec) {
  if (p.n_split < 1) return cudaSuccess;
  CUtensorMap mk, mv;
  if (!make_map(&mk, K, s) || !make_map(&mv, V, s)) return cudaErrorInvalidValue;
  StateParams prm{};
  prm.key_ref = reinterpret_cast<const float*>(ws);
  prm.omega_img = reinterpret_cast<const uint8_t*>(ws + p.off_omega_img);
  prm.partS = reinterpret_cast<float*>(ws + p.off_partS);
  prm.counters = reinterpret_cast<uint32_t*>(ws + p.off_counters);
  prm.state_img = reinterpret_cast<uint8_t*>(ws + p.off_state_img);
  prm.zvec = zvec;
  prm.status = status;
  prm.L = s.L;
  prm.m = s.m;
  prm.n_split = p.n_split;
  prm.tiles_per_split = p.tiles_per_split;
  prm.merge = p.causal ? 0 : 1;
  prm.scale = scale;
  const size_t smem = StateCfg<D>::kSmem;
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(state_kernel<D, M, FM>), smem);
  if (e != cudaSuccess) return e;
  // programmatic launch: the kernel's set-up and first tile loads overlap the
  // preparation kernel before it in the stream
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(p.n_split, s.BH());
  cfg.blockDim = dim3(kStateThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, state_kernel<D, M, FM>, mk, mv, prm);
}

template <int D, int M, int FM>
cudaError_t launch_output(const void* Q, void* O, const Shape& s, const TcPlan& p, float scale, char* ws,
                          int32_t* status, cudaStream_t stream) {
  CUtensorMap mq, mo;
  if (!make_map(&mq, Q, s) || !make_map(&mo, O, s)) return cudaErrorInvalidValue;
  OutParams prm{};
  prm.key_ref = reinterpret_cast<const float*>(ws);
  prm.omega_img = reinterpret_cast<const uint8_t*>(ws + p.off_omega_img);
  prm.state_img = reinterpret_cast<const uint8_t*>(ws + p.off_state_img);
  prm.status = status;
  prm.L = s.L;
  prm.m = s.m;
  prm.n_heads = s.BH();
  prm.scale = scale;
  const size_t smem = OutCfg<D>::kSmem;
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(output_kernel<D, M, FM>), smem);
  if (e != cudaSuccess) return e;
  // one CTA per SM (or per tile), each an even share of the (head, tile) list
  output_kernel<D, M, FM><<<p.out_grid, kOutThreads, smem, stream>>>(mq, mo, prm);
  return cudaGetLastError();
}

template <int D, int M, int FM>
cudaError_t launch_causal(const void* Q, const void* K, const void* V, void* O, const Shape& s, const TcPlan& p,
                          float scale, char* ws, int32_t* status, cudaStream_t stream) {
  CUtensorMap mq, mk, mv, mo;
  if (!make_map(&mq, Q, s) || !make_map(&mk, K, s) || !make_map(&mv, V, s) || !make_map(&mo, O, s))
    return cudaErrorInvalidValue;
  CausalParams prm{};
  prm.key_ref = reinterpret_cast<const float*>(ws);
  prm.omega_img = reinterpret_cast<const uint8_t*>(ws + p.off_omega_img);
  prm.pre = causal_direct(p) ? nullptr : reinterpret_cast<const float*>(ws + p.off_pre);
  prm.partS = reinterpret_cast<const float*>(ws + p.off_partS);
  prm.status = status;
  prm.L = s.L;
  prm.m = s.m;
  prm.n_sc = p.out_ctas;
  prm.tiles_per_sc = p.out_tiles_per_cta;
  prm.n_split = p.n_split;
  prm.sub_per_sc = p.sub_per_sc;
  prm.scale = scale;
  const size_t smem = CausalCfg<D>::kSmem;
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(causal_kernel<D, M, FM>), smem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.out_ctas, s.BH());
  causal_kernel<D, M, FM><<<grid, kCausalThreads, smem, stream>>>(mq, mk, mv, mo, prm);
  return cudaGetLastError();
}

}  // namespace

bool tc_supported(bool causal, int d, int m, bool bf16) {
  if (!bf16) return false;
  if (d == 64) return m == 128 || m == 256;
  return fs_supported(causal, d, m, bf16);
}

TcLayout tc_bidir_layout(const Shape& s) {
  const TcPlan p = tc_plan(false, s);
  TcLayout l{};
  l.off_omega_img = p.off_omega_img;
  l.off_counters = p.off_counters;
  l.off_partS = p.off_partS;
  l.off_state_img = p.off_state_img;
  l.bytes = p.bytes;
  return l;
}

size_t tc_workspace_bytes(bool causal, const Shape& s) {
  return s.d == 64 ? tc_plan(causal, s).bytes : fs_workspace_bytes(causal, s);
}

template <int FM>
cudaError_t tc_state_fm(bool causal, const void* K, const void* V, const float* omega, float scale, const Shape& s,
                        void* ws, int32_t* status, cudaStream_t stream, float* zvec) {
  const TcPlan p = tc_plan(causal, s);
  char* w = static_cast<char*>(ws);
  // prep also zeroes the bidirectional merge counters
  cudaError_t e = launch_prep(omega, s.m, s.d, reinterpret_cast<float*>(w),
                              reinterpret_cast<uint8_t*>(w + p.off_omega_img),
                              causal ? nullptr : reinterpret_cast<uint32_t*>(w + p.off_counters), causal ? 0 : s.BH(),
                              stream);
  if (e != cudaSuccess) return e;
  e = s.m == 256 ? launch_state<64, 256, FM>(K, V, s, p, scale, w, status, stream, zvec)
                 : launch_state<64, 128, FM>(K, V, s, p, scale, w, status, stream, zvec);
  if (e != cudaSuccess || !causal || p.n_split < 1 || causal_direct(p)) return e;
  state_prefix_kernel<64><<<dim3(p.n_fb * 65, s.BH()), kFB, 0, stream>>>(
      reinterpret_cast<const float*>(w + p.off_partS), reinterpret_cast<float*>(w + p.off_pre), p.n_fb, p.n_split,
      p.sub_per_sc, p.out_ctas);
  return cudaGetLastError();
}

template <int FM>
cudaError_t tc_output_fm(bool causal, const void* Q, const void* K, const void* V, void* O, const Shape& s,
                         float scale, void* ws, int32_t* status, cudaStream_t stream) {
  const TcPlan p = tc_plan(causal, s);
  char* w = static_cast<char*>(ws);
  if (causal)
    return s.m == 256 ? launch_causal<64, 256, FM>(Q, K, V, O, s, p, scale, w, status, stream)
                      : launch_causal<64, 128, FM>(Q, K, V, O, s, p, scale, w, status, stream);
  return s.m == 256 ? launch_output<64, 256, FM>(Q, O, s, p, scale, w, status, stream)
                    : launch_output<64, 128, FM>(Q, O, s, p, scale, w, status, stream);
}

cudaError_t tc_state(bool causal, const void* K, const void* V, const float* omega, float scale, const Shape& s,
                     void* ws, int32_t* status, cudaStream_t stream, int fm, float* zvec) {
  if (s.d != 64) return fs_state(causal, K, V, omega, scale, s, ws, status, stream, fm);
  if (fm == FAVOR_FM_RELU) return tc_state_fm<FAVOR_FM_RELU>(causal, K, V, omega, scale, s, ws, status, stream, zvec);
  if (fm == FAVOR_FM_ELU1) return tc_state_fm<FAVOR_FM_ELU1>(causal, K, V, omega, scale, s, ws, status, stream, zvec);
  return tc_state_fm<FAVOR_FM_PRF>(causal, K, V, omega, scale, s, ws, status, stream, zvec);
}

cudaError_t tc_output(bool causal, const void* Q, const void* K, const void* V, void* O, const float* omega,
                      float scale, const Shape& s, void* ws, int32_t* status, cudaStream_t stream, int fm) {
  (void)omega;
  if (s.d != 64) return fs_output(causal, Q, K, V, O, scale, s, ws, status, stream, fm);
  if (fm == FAVOR_FM_RELU) return tc_output_fm<FAVOR_FM_RELU>(causal, Q, K, V, O, s, scale, ws, status, stream);
  if (fm == FAVOR_FM_ELU1) return tc_output_fm<FAVOR_FM_ELU1>(causal, Q, K, V, O, s, scale, ws, status, stream);
  return tc_output_fm<FAVOR_FM_PRF>(causal, Q, K, V, O, s, scale, ws, status, stream);
}

}  // namespace favor
