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

// Grid of ceil(m / 8) CTAs; warp w of CTA b handles row i = 8b + w: its
// squared norm (the CTA writes the largest of its 8 into header slot b) and,
// if `image` is non-null, its bf16 images: hi = bf16(w) at `image` and
// lo = bf16(w - hi) m*d*2 bytes later, so that hi + lo carries w to about 16
// significant bits (the projection is two accumulating MMAs; bf16 w alone
// costs ~2% in the output).  Layout of each image: [feature block of 128]
// [64-column atom][128 rows][128 B], 16-byte chunk c of row r stored at
// chunk c ^ (r % 8) (the 128-byte swizzle).
__global__ void __launch_bounds__(kPrepThreads) prep_kernel(const float* __restrict__ omega, int m, int d,
                                                            float* __restrict__ header,
                                                            uint8_t* __restrict__ image) {
  __shared__ float red[32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i = blockIdx.x * kPrepRows + warp;
  float n2 = -INFINITY;
  if (i < m) {
    const float* row = omega + (size_t)i * d;
    float acc = 0.f;
    for (int c = lane; c < d; c += 32) acc = fmaf(row[c], row[c], acc);
    n2 = warp_sum(acc);
    if (image != nullptr) {
      const int n_atoms = (d + 63) / 64;
      const int fb = i >> 7, r = i & 127;
      for (int c = 2 * lane; c < d; c += 64) {
        const float w0 = row[c];
        const float w1 = (c + 1 < d) ? row[c + 1] : 0.f;
        const __nv_bfloat162 hi = __floats2bfloat162_rn(w0, w1);
        const __nv_bfloat162 lo = __floats2bfloat162_rn(w0 - __low2float(hi), w1 - __high2float(hi));
        const int atom = c >> 6, cc = c & 63;
        const int chunk = (cc >> 3) ^ (r & 7);
        const size_t off = ((size_t)(fb * n_atoms + atom) * 128 + r) * 128 + chunk * 16 + (cc & 7) * 2;
        *reinterpret_cast<__nv_bfloat162*>(image + off) = hi;
        *reinterpret_cast<__nv_bfloat162*>(image + (size_t)m * d * 2 + off) = lo;
      }
    }
  }
  const float w2 = block_max(n2, red);
  if (threadIdx.x == 0) header[blockIdx.x] = w2;
}

}  // namespace

cudaError_t launch_prep(const float* omega, int m, int d, float* header, uint8_t* image, cudaStream_t stream) {
  prep_kernel<<<(m + kPrepRows - 1) / kPrepRows, kPrepThreads, 0, stream>>>(omega, m, d, header, image);
  return cudaGetLastError();
}

}  // namespace favor
