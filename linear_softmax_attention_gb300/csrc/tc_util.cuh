// Pieces shared by the tensor-core (tcgen05) kernel files: tile constants,
// the fp16 rewrite of an input tile, TMEM loads, the feature-map epilogues,
// swizzled shared-memory stores, descriptor arithmetic, grid splitting and
// the TMA tensor map of a [B, H, L, d] bf16 tensor.
#pragma once

#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace favor {
namespace tc {

constexpr int kBM = 128;          // tokens per tile
constexpr int kFB = 128;          // features per block
constexpr uint32_t kTmemCols = 512;
constexpr int kAtom = 128 * 128;  // bytes of one [128 rows][128 B] swizzle block
constexpr int kEpiWarps = 8;
constexpr int kEpiThreads = 256;
constexpr int kEpiTid0 = 128;   // first epilogue thread (warps 4-11)
constexpr int kNormWarps = 2;

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Splits of `tiles` tiles for each of `units` independent rows of CTAs: the
// fewest splits minimising waves x (tiles per CTA + per-CTA set-up, counted
// as kCtaOverheadTiles tiles).
constexpr int kCtaOverheadTiles = 3;
inline int pick_split(int units, int tiles, int sms) {
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

// The CTAs of a grid of n_ctas split the list of B H x tiles (head, tile)
// pairs evenly: CTA c takes entries [range_first(c), range_first(c + 1)),
// which may cross from one head into the next.
__host__ __device__ __forceinline__ int range_first(long long total, int c, int n_ctas) {
  return (int)(total * c / n_ctas);
}
// the CTA holding list entry x
__host__ __device__ __forceinline__ int range_cta(long long total, long long x, int n_ctas) {
  return (int)(((x + 1) * n_ctas + total - 1) / total) - 1;
}

// ---------------------------------------------------------------------------
// shared device pieces
// ---------------------------------------------------------------------------

// Squared norm of row t of a [128][D] bf16 tile stored as 64-column swizzle
// blocks (TMA layout); the row is rewritten in place as fp16 (round to
// nearest, saturating at +-65504) for the projection MMA.  A key whose
// entries reach the fp16 limit has |s k|^2 / 2 so far above any projection
// that its feature is 0 in fp32 either way.
template <int D>
__device__ __forceinline__ float tile_row_sq_to_f16(uint8_t* tile, int t) {
  constexpr int NC = D / 8;                     // 16-byte chunks per row
  uint4 v[NC];
#pragma unroll
  for (int c = 0; c < NC; ++c)
    v[c] = *reinterpret_cast<const uint4*>(tile + (c >> 3) * kAtom + t * 128 + (((c & 7) ^ (t & 7)) << 4));
  // eight partial sums (one per element position of a 16-byte chunk) keep
  // the dependent chain of multiply-adds short
  float acc[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j] = 0.f;
#pragma unroll
  for (int c = 0; c < NC; ++c) {
    const uint32_t w[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float lo = __uint_as_float(w[j] << 16);
      const float hi = __uint_as_float(w[j] & 0xFFFF0000u);
      acc[2 * j] = fmaf(lo, lo, acc[2 * j]);
      acc[2 * j + 1] = fmaf(hi, hi, acc[2 * j + 1]);
      o[j] = pack_f16_sat(lo, hi);
    }
    v[c] = make_uint4(o[0], o[1], o[2], o[3]);
  }
#pragma unroll
  for (int c = 0; c < NC; ++c)
    *reinterpret_cast<uint4*>(tile + (c >> 3) * kAtom + t * 128 + (((c & 7) ^ (t & 7)) << 4)) = v[c];
  return ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
}

// tcgen05.ld 32x32b.x32 into r[OFF .. OFF+31]
template <int OFF, int N>
__device__ __forceinline__ void tmem_ld32_at(uint32_t taddr, uint32_t (&r)[N]) {
  static_assert(OFF + 32 <= N, "range");
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[OFF + 0]), "=r"(r[OFF + 1]), "=r"(r[OFF + 2]), "=r"(r[OFF + 3]), "=r"(r[OFF + 4]), "=r"(r[OFF + 5]),
        "=r"(r[OFF + 6]), "=r"(r[OFF + 7]), "=r"(r[OFF + 8]), "=r"(r[OFF + 9]), "=r"(r[OFF + 10]), "=r"(r[OFF + 11]),
        "=r"(r[OFF + 12]), "=r"(r[OFF + 13]), "=r"(r[OFF + 14]), "=r"(r[OFF + 15]), "=r"(r[OFF + 16]),
        "=r"(r[OFF + 17]), "=r"(r[OFF + 18]), "=r"(r[OFF + 19]), "=r"(r[OFF + 20]), "=r"(r[OFF + 21]),
        "=r"(r[OFF + 22]), "=r"(r[OFF + 23]), "=r"(r[OFF + 24]), "=r"(r[OFF + 25]), "=r"(r[OFF + 26]),
        "=r"(r[OFF + 27]), "=r"(r[OFF + 28]), "=r"(r[OFF + 29]), "=r"(r[OFF + 30]), "=r"(r[OFF + 31])
      : "r"(taddr));
}
// 64 consecutive columns into r[0 .. 63]
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&r)[64]) {
  tmem_ld32_at<0>(taddr, r);
  tmem_ld32_at<32>(taddr + 32, r);
}

// In place: x[j] = bf16x2(2^(x[2j] c1 - b), 2^(x[2j+1] c1 - b)) for j < N/2
// (zeros if !valid).
template <int N>
__device__ __forceinline__ void exp_pack(uint32_t (&x)[N], float c1, float b, bool valid) {
#pragma unroll
  for (int j = 0; j < N / 2; ++j) {
    const float y0 = valid ? ex2(fmaf(__uint_as_float(x[2 * j]), c1, -b)) : 0.f;
    const float y1 = valid ? ex2(fmaf(__uint_as_float(x[2 * j + 1]), c1, -b)) : 0.f;
    x[j] = pack_bf16(y0, y1);
  }
}

// Feature maps: positive random features (the softmax kernel),
// Performer-ReLU, relu(s w.x), or 1 + elu (below) ("Rethinking Attention with Performers"
// summary, §2 generalized kernelizable attention: other kernels by changing
// the feature-map function).  ReLU: b = 0 on valid rows and +inf past the
// sequence end (feature 0); "y < 0 ? 0 : y" keeps a NaN a NaN.
template <int N>
__device__ __forceinline__ void relu_pack(uint32_t (&x)[N], float c1, float b) {
#pragma unroll
  for (int j = 0; j < N / 2; ++j) {
    float y0 = fmaf(__uint_as_float(x[2 * j]), c1, -b);
    float y1 = fmaf(__uint_as_float(x[2 * j + 1]), c1, -b);
    y0 = y0 < 0.f ? 0.f : y0;
    y1 = y1 < 0.f ? 0.f : y1;
    x[j] = pack_bf16(y0, y1);
  }
}
// 1 + elu(a) of a = s w.x - b: 1 + a for a >= 0, e^a below ("From
// Performer to Linear Attention": the linear-attention feature map, here in
// the slot of f(w_i^T x)).  Past the sequence end b = +inf gives e^-inf = 0;
// a NaN fails a >= 0 and stays a NaN.
template <int N>
__device__ __forceinline__ void elu1_pack(uint32_t (&x)[N], float c1, float b) {
#pragma unroll
  for (int j = 0; j < N / 2; ++j) {
    const float a0 = fmaf(__uint_as_float(x[2 * j]), c1, -b);
    const float a1 = fmaf(__uint_as_float(x[2 * j + 1]), c1, -b);
    const float y0 = a0 >= 0.f ? 1.f + a0 : ex2(a0 * kLog2e);
    const float y1 = a1 >= 0.f ? 1.f + a1 : ex2(a1 * kLog2e);
    x[j] = pack_bf16(y0, y1);
  }
}
template <int FM, int N>
__device__ __forceinline__ void feature_pack(uint32_t (&x)[N], float c1, float b) {
  if constexpr (FM == FAVOR_FM_PRF) exp_pack<N>(x, c1, b, true);
  else if constexpr (FM == FAVOR_FM_ELU1) elu1_pack<N>(x, c1, b);
  else relu_pack<N>(x, c1, b);
}
// multiplier of the projection in the feature exponent / argument
template <int FM>
__device__ __forceinline__ float feature_c1(float scale) {
  return FM == FAVOR_FM_PRF ? scale * kLog2e : scale;
}

// Row t, columns col0 .. col0 + 2*NW - 1 (col0 a multiple of 8) of a tile of
// 64-column swizzle blocks `atom_stride` bytes apart, from NW packed words.
template <int NW, int N>
__device__ __forceinline__ void store_row(uint32_t base, int atom_stride, int t, int col0, const uint32_t (&x)[N]) {
#pragma unroll
  for (int c = 0; c < NW / 4; ++c) {
    const int col = col0 + 8 * c;
    const int atom = col >> 6, chunk = (col & 63) >> 3;
    st_shared_v4(base + atom * atom_stride + t * 128 + ((chunk ^ (t & 7)) << 4), x[4 * c], x[4 * c + 1],
                 x[4 * c + 2], x[4 * c + 3]);
  }
}

// Constant [16 rows][128 B] block, MN-major swizzled: element 0 of every
// row is 1, the rest 0.  Read as columns d .. d+15 of [V | 1] by every k-step
// (each MMA's leading-byte offset points back to it).
constexpr int kOnesBytes = 16 * 128;
__device__ __forceinline__ void fill_ones_block(uint8_t* p, int tid0, int nthreads) {
  for (int e = threadIdx.x - tid0; e < kOnesBytes / 16; e += nthreads) {
    const int row = e >> 3, logical = (e & 7) ^ (row & 7);
    *reinterpret_cast<uint4*>(p + e * 16) = make_uint4(logical == 0 ? 0x3F80u : 0u, 0u, 0u, 0u);
  }
}

// [128 rows][128 B] block whose row r reads, unswizzled, (1, 0, ..., 0): as
// the atom after a 64-column K-major tile, columns 64 .. 127 of [X | 1]
__device__ __forceinline__ void fill_ones_atom(uint8_t* p, int tid0, int nthreads) {
  for (int e = threadIdx.x - tid0; e < kAtom / 16; e += nthreads) {
    const int row = e >> 3, logical = (e & 7) ^ (row & 7);
    *reinterpret_cast<uint4*>(p + e * 16) = make_uint4(logical == 0 ? 0x3F80u : 0u, 0u, 0u, 0u);
  }
}

// Descriptor arithmetic.  A descriptor's start-address field holds bytes >> 4
// in its low bits, so a k-step is an add to the base descriptor built once
// per MMA group (rebuilding it per MMA costs the issuing thread ~40 issue
// slots, which halves the MMA rate when epilogue warps share its SMSP).
__device__ __forceinline__ uint64_t dadd(uint64_t d, uint32_t bytes) { return d + (bytes >> 4); }
// K-major SW128: k-step k (16 elements) within 64-element atoms `atom` bytes apart
__host__ __device__ constexpr uint32_t kstep_k(int k, int atom) { return (k >> 2) * atom + (k & 3) * 32; }
// MN-major SW128: k-step k is 16 rows of 128 B
__host__ __device__ constexpr uint32_t kstep_mn(int k) { return k * 2048; }
// [V | 1] at k-step k: start advances by 2048 k, the offset back to the ones
// block shrinks by the same amount
__device__ __forceinline__ uint64_t vones_k(uint64_t d0, int k) {
  return d0 + static_cast<uint64_t>(k * 128) - (static_cast<uint64_t>(k * 128) << 16);
}

// The causal state's bf16 copy: columns n = 8g .. 8g + 7 (groups g0 <= g <
// g1) of G in tensor memory (lane = feature; this warp's 32 features from
// lane 32q) into rows n of a K-major operand, 8 features per 16-byte swizzle
// chunk.  `rows` is the address of row 0 of the atom holding this thread's
// stmatrix features (32q + 8 (lane / 8) onward).  Per group a 16x256b load
// per half of the warp's features gives each thread two adjacent n of one
// feature; stmatrix.trans turns each 8x8 block (features x n) into rows n.
// KB groups' loads are in flight together (one wait per KB groups).
template <int KB>
__device__ __forceinline__ void tmem_state_to_rows(uint32_t tmem, uint32_t g_col, int q, int lane, int g0, int g1,
                                                   uint32_t rows) {
  const int kr = lane & 7;
  const int fch = ((32 * q + 8 * (lane >> 3)) & 63) >> 3;
#pragma unroll 1
  for (int gb = g0; gb < g1; gb += KB) {
    uint32_t lo[KB][4], hi[KB][4];
#pragma unroll
    for (int u = 0; u < KB; ++u) {
      const uint32_t col = g_col + 8 * min(gb + u, g1 - 1);   // a past-the-end group reloads the last one
      tmem_ld16x256(tmem + (static_cast<uint32_t>(32 * q) << 16) + col, lo[u]);
      tmem_ld16x256(tmem + (static_cast<uint32_t>(32 * q + 16) << 16) + col, hi[u]);
    }
    tmem_ld_wait();
#pragma unroll
    for (int u = 0; u < KB; ++u) {
      if (gb + u >= g1) break;
      const int n = 8 * (gb + u) + kr;
      stmatrix_x4_trans(rows + n * 128 + ((fch ^ (n & 7)) << 4),
                        pack_bf16(__uint_as_float(lo[u][0]), __uint_as_float(lo[u][1])),
                        pack_bf16(__uint_as_float(lo[u][2]), __uint_as_float(lo[u][3])),
                        pack_bf16(__uint_as_float(hi[u][0]), __uint_as_float(hi[u][1])),
                        pack_bf16(__uint_as_float(hi[u][2]), __uint_as_float(hi[u][3])));
    }
  }
}

// The fixed-order sum of one head's first `count` fp32 partial states
// ([M/128 blocks][stride][D + 1][128], feature fastest) as its bf16 state
// image ([M/64 atoms][D + 16 rows][128 B], 128-byte swizzle, the normaliser
// in row D, rows past it zero), by `nthreads` threads (this one is number
// `tid`) with eight items' loads in flight per partial.  Item = (block b,
// state row n, 4 consecutive features).  With `zvec` non-null, the
// normaliser row (n = D) also goes to zvec[0, M) in fp32.
template <int D, int M>
__device__ void merge_partials(const float* __restrict__ base, int stride, int count, uint8_t* __restrict__ img,
                               int tid, int nthreads, float* __restrict__ zvec = nullptr) {
  constexpr int NFB = M / kFB;
  constexpr int NG = kFB / 4;
  constexpr int kItems = NFB * (D + 16) * NG;
  constexpr int kBatch = 8;
  for (int e0 = tid; e0 < kItems; e0 += kBatch * nthreads) {
    float4 acc[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int p = 0; p < count; ++p) {
      float4 v[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int e = e0 + u * nthreads;
        const int g = e % NG, n = (e / NG) % (D + 16), b = e / (NG * (D + 16));
        v[u] = (e < kItems && n <= D)
                   ? *reinterpret_cast<const float4*>(base + (((size_t)b * stride + p) * (D + 1) + n) * kFB + g * 4)
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
      const int e = e0 + u * nthreads;
      if (e >= kItems) break;
      const int g = e % NG, n = (e / NG) % (D + 16), b = e / (NG * (D + 16));
      const int f = b * kFB + g * 4;
      const int atom = f >> 6, cc = f & 63;
      const size_t off = ((size_t)atom * (D + 16) + n) * 128 + (((cc >> 3) ^ (n & 7)) << 4) + (cc & 7) * 2;
      *reinterpret_cast<uint2*>(img + off) = make_uint2(pack_bf16(acc[u].x, acc[u].y), pack_bf16(acc[u].z, acc[u].w));
      if (zvec != nullptr && n == D) *reinterpret_cast<float4*>(zvec + f) = acc[u];
    }
  }
}

// Initial causal states of the superchunks of each (head, feature block):
// superchunk sc starts from the fixed-order sum of the partial states of the
// sub-splits of superchunks 0 .. sc - 1 (block = (head, feature block, state
// row n), thread = feature; eight loads in flight).  partS is
// [heads x blocks][n_split][D + 1][128], pre [heads x blocks][n_sc][D + 1][128].
template <int D>
__global__ void __launch_bounds__(kFB) state_prefix_kernel(const float* __restrict__ partS, float* __restrict__ pre,
                                                           int n_fb, int n_split, int sub_per_sc, int n_sc) {
  const int f = threadIdx.x;
  const int n = blockIdx.x % (D + 1), hb = blockIdx.y * n_fb + blockIdx.x / (D + 1);
  constexpr size_t kStride = (size_t)(D + 1) * kFB;
  const float* src = partS + (size_t)hb * max(n_split, 1) * kStride + (size_t)n * kFB + f;
  float* dst = pre + (size_t)hb * n_sc * kStride + (size_t)n * kFB + f;
  float acc = 0.f;
  for (int p0 = 0; p0 < n_split; p0 += 8) {
    float v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = (p0 + u < n_split) ? src[(size_t)(p0 + u) * kStride] : 0.f;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int p = p0 + u;
      if (p >= n_split) break;
      if (p % sub_per_sc == 0) dst[(size_t)(p / sub_per_sc) * kStride] = acc;
      acc += v[u];
    }
  }
  dst[(size_t)(n_sc - 1) * kStride] = acc;
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
inline PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
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
inline bool make_map(CUtensorMap* map, const void* base, const Shape& s) {
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

}  // namespace tc
}  // namespace favor
