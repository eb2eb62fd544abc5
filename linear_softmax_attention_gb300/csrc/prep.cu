// Per-call preparation shared by both kernel families.
//
// Key reference R.  For every key k and feature i the exponent of the positive
// random feature is  l = s w_i.k - s^2 |k|^2 / 2 = |w_i|^2/2 - |s k - w_i|^2/2,
// so l <= max_i |w_i|^2 / 2 for every input.  Evaluating phi(k) as exp(l - R)
// with R = max_i |w_i|^2/2 - kKeyHeadroom keeps every key feature <= e^40: no
// overflow for any input, and R is one constant for all keys, heads and
// partial sums, so partial states add without rescaling and no output row
// depends (even in rounding) on keys it does not attend to.  The factor
// exp(-R) is common to numerator and normaliser and cancels.
#include "common.cuh"

namespace favor {
namespace {

constexpr int kPrepThreads = 32 * kPrepRows;   // one warp per row of Omega

// Grid of ceil(m / 8) CTAs; the CTAs also zero `n_counters` merge counters.
// Warp w of CTA b handles row i = 8b + w: its
// squared norm (the CTA writes the largest of its 8 into header slot b) and,
// if `image` is non-null, its fp16 image (round to nearest, saturating) for
// the projection MMAs: layout [64-column atom][m rows][128 B], 16-byte chunk
// c of row r stored at chunk c ^ (r % 8) (the 128-byte swizzle).  fp16
// carries w to 11 significant bits; bf16 w alone costs ~2.5% in the output.
__global__ void __launch_bounds__(kPrepThreads) prep_kernel(const float* __restrict__ omega, int m, int d,
                                                            float* __restrict__ header,
                                                            uint8_t* __restrict__ image,
                                                            uint32_t* __restrict__ counters, int n_counters) {
  __shared__ float red[32];
  // the state kernel that follows may start now (it waits before reading the
  // header and the image)
  asm volatile("griddepcontrol.launch_dependents;");
  for (int i = blockIdx.x * kPrepThreads + threadIdx.x; i < n_counters; i += gridDim.x * kPrepThreads) counters[i] = 0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i = blockIdx.x * kPrepRows + warp;
  float n2 = -INFINITY;
  if (i < m) {
    const float* row = omega + (size_t)i * d;
    float acc = 0.f;
    for (int c = lane; c < d; c += 32) acc = fmaf(row[c], row[c], acc);
    n2 = warp_sum(acc);
    if (image != nullptr) {
      for (int c = 2 * lane; c < d; c += 64) {
        const float w0 = row[c];
        const float w1 = (c + 1 < d) ? row[c + 1] : 0.f;
        uint32_t h;
        asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(h) : "f"(w1), "f"(w0));
        const int atom = c >> 6, cc = c & 63;
        const int chunk = (cc >> 3) ^ (i & 7);
        const size_t off = ((size_t)atom * m + i) * 128 + chunk * 16 + (cc & 7) * 2;
        *reinterpret_cast<uint32_t*>(image + off) = h;
      }
    }
  }
  const float w2 = block_max(n2, red);
  if (threadIdx.x == 0) header[blockIdx.x] = w2;
}

}  // namespace

cudaError_t launch_prep(const float* omega, int m, int d, float* header, uint8_t* image, uint32_t* counters,
                        int n_counters, cudaStream_t stream) {
  prep_kernel<<<(m + kPrepRows - 1) / kPrepRows, kPrepThreads, 0, stream>>>(omega, m, d, header, image, counters,
                                                                             n_counters);
  return cudaGetLastError();
}

}  // namespace favor
