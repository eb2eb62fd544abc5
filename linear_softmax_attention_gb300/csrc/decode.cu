// Incremental causal FAVOR+: one new token per (b, h), the prefix state
// carried between calls.
//
// "From Performer to Linear Attention" (Su), §Concentrating Attention: a
// causal linear attention is a unidirectional RNN.  "Performer — Rethinking
// Attention with Performers" (digest), §Methods, causal bullet: the state is
// the prefix sum G_t = sum_{s<=t} phi(k_s) v_s^T (with z_t = sum phi(k_s)
// beside it).  Per call and head:
//   state += phi(s k) [v ; 1]^T,  o = phi(s q)^T state[:, :d] / phi(s q)^T state[:, d]
// The state is fp32 [d+1][m] per head (column i = feature i, the last row
// the normaliser sums); its key features
// use the reference R = max_i |w_i|^2 / 2 - 40 of the sequence kernels, so a
// state from favor_decode_prefill continues here.  The query features use
// the query's largest exponent max_i s w_i.q, so the largest is exactly 1 at
// any norm of q: a per-query constant, it cancels in the ratio ("From
// Performer to Linear Attention", §Simple Derivation).
//
// One CTA per head.  Bound by the state's HBM traffic: m (d+1) fp32 read and
// written per head and token (133 KB at m = 256, d = 64); Omega (m x d fp32)
// is read by every CTA and stays in L2.  Where it fits (m (d + 4) floats up to
// 100 KB, so two CTAs share an SM) each CTA first copies Omega into shared
// memory with coalesced 16-byte asynchronous copies, rows padded to d + 4
// floats so that the row a thread reads sits in its own banks; read straight
// from L2, every lane's row is a separate line and the requests, not the
// bytes, set the time.
#include <type_traits>

#include "common.cuh"

namespace favor {
namespace {

constexpr int kDecThreads = 256;
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kCB = 16;                              // state columns per block of loads
constexpr size_t kStageOmegaMax = 100 * 1024;        // bytes of padded Omega copied into shared memory

// NF features per thread: 1 for m <= 256, 2 for m <= 512
template <typename T, int NF>
__global__ void __launch_bounds__(kDecThreads, 2) decode_step_kernel(const T* __restrict__ q, const T* __restrict__ k,
                                                                  const T* __restrict__ v, T* __restrict__ o,
                                                                  const float* __restrict__ omega, int d, int m,
                                                                  float scale, float* __restrict__ state,
                                                                  int32_t* __restrict__ status, int staged) {
  __shared__ float qs[kMaxD], ks[kMaxD], vs[kMaxD + 1];
  __shared__ float phq[kMaxM], phk[kMaxM];
  __shared__ float part[kDecWarps][kMaxD + 1];
  __shared__ float num[kMaxD + 1];
  __shared__ float wred[kDecWarps], qred[kDecWarps];
  __shared__ float sqn[1];
  extern __shared__ __align__(16) float om_s[];     // [m][d + 4] when staged
  const int bh = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ld = d + 1;
  const int ldw = d + 4;

  if (staged) {
    const int dq = d >> 2;
    for (int e = tid; e < m * dq; e += kDecThreads) {
      const int f = e / dq, j4 = e - f * dq;
      const uint32_t dst = static_cast<uint32_t>(__cvta_generic_to_shared(om_s + f * ldw + 4 * j4));
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(omega + 4 * (size_t)e) : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
  for (int j = tid; j < d; j += kDecThreads) {
    const size_t e = (size_t)bh * d + j;
    qs[j] = to_f32(q[e]);
    ks[j] = to_f32(k[e]);
    vs[j] = to_f32(v[e]);
  }
  if (tid == 0) vs[d] = 1.f;
  __syncthreads();
  if (warp == 0) {
    // |k|^2 for the key features' exponent
    float a = 0.f;
    for (int j = lane; j < d; j += 32) a = fmaf(ks[j], ks[j], a);
    a = warp_sum(a);
    if (lane == 0) sqn[0] = a;
  }

  // the first super-block of state columns is loaded before the
  // projections (it does not depend on them), so its HBM round trip overlaps
  // the Omega reads; every load of a super-block is in flight at once
  constexpr int NB = NF == 1 ? 5 : 1;              // 16-column blocks per super-block
  constexpr int SB = NB * kCB;
  float* st = state + (size_t)bh * ld * m;
  float g[SB][NF];
  auto load_sb = [&](int j0) {
#pragma unroll
    for (int c = 0; c < SB; ++c) {
      const int j = j0 + c;
#pragma unroll
      for (int i = 0; i < NF; ++i) {
        const int f = tid + i * kDecThreads;
        g[c][i] = (j < ld && f < m) ? st[(size_t)j * m + f] : 0.f;
      }
    }
  };
  load_sb(0);
  if (staged) asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();                                   // the copy of Omega is complete

  // w_f.q, w_f.k and |w_f|^2 for the features f = tid + 256 i of this thread
  float pq[NF], pk[NF];
  float w2max = 0.f, pqmax = -INFINITY;
#pragma unroll
  for (int i = 0; i < NF; ++i) {
    const int f = tid + i * kDecThreads;
    float dq = 0.f, dk = 0.f, w2 = 0.f;
    if (f < m) {
      const float* w = omega + (size_t)f * d;
      if (staged || (d & 3) == 0) {
        // rows are 16-byte aligned: 16-byte loads, a quarter of the requests
        const float4* w4 = staged ? reinterpret_cast<const float4*>(om_s + f * ldw) : reinterpret_cast<const float4*>(w);
        for (int j4 = 0; j4 < d / 4; ++j4) {
          const float4 x = staged ? w4[j4] : __ldg(w4 + j4);
          const int j = 4 * j4;
          dq = fmaf(x.x, qs[j], dq);
          dk = fmaf(x.x, ks[j], dk);
          w2 = fmaf(x.x, x.x, w2);
          dq = fmaf(x.y, qs[j + 1], dq);
          dk = fmaf(x.y, ks[j + 1], dk);
          w2 = fmaf(x.y, x.y, w2);
          dq = fmaf(x.z, qs[j + 2], dq);
          dk = fmaf(x.z, ks[j + 2], dk);
          w2 = fmaf(x.z, x.z, w2);
          dq = fmaf(x.w, qs[j + 3], dq);
          dk = fmaf(x.w, ks[j + 3], dk);
          w2 = fmaf(x.w, x.w, w2);
        }
      } else {
        for (int j = 0; j < d; ++j) {
          const float wj = __ldg(w + j);
          dq = fmaf(wj, qs[j], dq);
          dk = fmaf(wj, ks[j], dk);
          w2 = fmaf(wj, wj, w2);
        }
      }
      w2max = fmaxf(w2max, w2);
      pqmax = fmaxf(pqmax, dq);
    }
    pq[i] = dq;
    pk[i] = dk;
  }
  w2max = warp_max(w2max);
  pqmax = warp_max(pqmax);
  if (lane == 0) {
    wred[warp] = w2max;
    qred[warp] = pqmax;
  }
  __syncthreads();
  float w2 = wred[0], qmax = qred[0];
  for (int i = 1; i < kDecWarps; ++i) {
    w2 = fmaxf(w2, wred[i]);
    qmax = fmaxf(qmax, qred[i]);
  }
  const float R = 0.5f * w2 - kKeyHeadroom;
  const float bq = scale * qmax;
  const float hk = 0.5f * scale * scale * sqn[0];
#pragma unroll
  for (int i = 0; i < NF; ++i) {
    const int f = tid + i * kDecThreads;
    if (f < m) {
      phk[f] = expf(scale * pk[i] - hk - R);
      phq[f] = expf(scale * pq[i] - bq);
    }
  }
  __syncthreads();

  // state columns j (rows of the [d+1][m] layout): thread t owns features
  // t (and t + 256), so every access is a whole-warp coalesced 128-byte row
  // segment.  The column sums sum_f phi(q)_f g_jf are accumulated per
  // thread, reduced within each warp by a shuffle reduce-scatter over blocks
  // of 16 columns, then across warps in a fixed order.
  float fk[NF], fq[NF];
#pragma unroll
  for (int i = 0; i < NF; ++i) {
    const int f = tid + i * kDecThreads;
    fk[i] = f < m ? phk[f] : 0.f;
    fq[i] = f < m ? phq[f] : 0.f;
  }
  for (int j0 = 0; j0 < ld; j0 += SB) {
    if (j0 > 0) load_sb(j0);
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      const int jb = j0 + b * kCB;
      float p[kCB];
#pragma unroll
      for (int c = 0; c < kCB; ++c) {
        const int j = jb + c;
        float acc = 0.f;
        if (j < ld) {
          const float vj = vs[j];
#pragma unroll
          for (int i = 0; i < NF; ++i) {
            const int f = tid + i * kDecThreads;
            if (f < m) {
              const float gn = fmaf(fk[i], vj, g[b * kCB + c][i]);
              st[(size_t)j * m + f] = gn;
              acc = fmaf(fq[i], gn, acc);
            }
          }
        }
        p[c] = acc;
      }
      // reduce-scatter over lane bits 3..0: after the step of offset o each
      // lane keeps the half of its values whose index bit o matches its lane
      // bit; then the two 16-lane halves are added
#pragma unroll
      for (int o = kCB / 2; o >= 1; o >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int c = 0; c < o; ++c) {
          const float keep = up ? p[c + o] : p[c];
          const float send = up ? p[c] : p[c + o];
          p[c] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
      }
      p[0] += __shfl_xor_sync(0xffffffffu, p[0], kCB);
      // lane l (and l + 16) holds the warp's sum of column jb + (l & 15)
      if (lane < kCB && jb + lane < ld) part[warp][jb + lane] = p[0];
    }
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
  const size_t stage_bytes = (size_t)m * (d + 4) * sizeof(float);
  const bool staged = (d & 3) == 0 && (reinterpret_cast<uintptr_t>(omega) & 15) == 0 && stage_bytes <= kStageOmegaMax;
  cudaError_t err = cudaSuccess;
  auto go = [&](auto tag, auto nf) {
    using T = decltype(tag);
    constexpr int NF = decltype(nf)::value;
    const size_t smem = staged ? stage_bytes : 0;
    err = ensure_dynamic_smem(reinterpret_cast<const void*>(decode_step_kernel<T, NF>), smem);
    if (err != cudaSuccess) return;
    decode_step_kernel<T, NF><<<BH, kDecThreads, smem, stream>>>(static_cast<const T*>(q), static_cast<const T*>(k),
                                                                 static_cast<const T*>(v), static_cast<T*>(o), omega,
                                                                 d, m, scale, state, status, staged ? 1 : 0);
  };
  using One = std::integral_constant<int, 1>;
  using Two = std::integral_constant<int, 2>;
  if (bf16) {
    if (m <= kDecThreads) go(__nv_bfloat16{}, One{});
    else go(__nv_bfloat16{}, Two{});
  } else {
    if (m <= kDecThreads) go(float{}, One{});
    else go(float{}, Two{});
  }
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

}  // namespace favor
