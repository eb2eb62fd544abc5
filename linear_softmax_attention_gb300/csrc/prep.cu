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

constexpr float kKeyHeadroom = 40.0f;
constexpr int kPrepThreads = 512;

// One CTA: thread i < m owns row i of Omega.  Writes R (natural-log units)
// and, if `image` is non-null, Omega in bf16 as the tensor-core B operand:
// [feature block of 128][64-column atom][128 rows][128 B], 16-byte chunk c of
// row r stored at chunk c ^ (r % 8) (the 128-byte swizzle).
__global__ void __launch_bounds__(kPrepThreads) prep_kernel(const float* __restrict__ omega, int m, int d,
                                                            float* __restrict__ key_ref,
                                                            uint8_t* __restrict__ image) {
  __shared__ float red[32];
  float n2 = -INFINITY;
  for (int i = threadIdx.x; i < m; i += kPrepThreads) {
    const float* row = omega + (size_t)i * d;
    float acc = 0.f;
    for (int c = 0; c < d; ++c) acc = fmaf(row[c], row[c], acc);
    n2 = fmaxf(n2, acc);
  }
  const float w2 = block_max(n2, red);
  if (threadIdx.x == 0) *key_ref = 0.5f * w2 - kKeyHeadroom;
  if (image != nullptr) {
    const int n_atoms = (d + 63) / 64;
    for (int e = threadIdx.x; e < m * d; e += kPrepThreads) {
      const int i = e / d, c = e - i * d;
      const int fb = i >> 7, r = i & 127, atom = c >> 6, cc = c & 63;
      const int chunk = (cc >> 3) ^ (r & 7);
      const size_t off = ((size_t)(fb * n_atoms + atom) * 128 + r) * 128 + chunk * 16 + (cc & 7) * 2;
      *reinterpret_cast<__nv_bfloat16*>(image + off) = __float2bfloat16_rn(omega[e]);
    }
  }
}

}  // namespace

cudaError_t launch_prep(const float* omega, int m, int d, float* key_ref, uint8_t* image, cudaStream_t stream) {
  prep_kernel<<<1, kPrepThreads, 0, stream>>>(omega, m, d, key_ref, image);
  return cudaGetLastError();
}

}  // namespace favor
