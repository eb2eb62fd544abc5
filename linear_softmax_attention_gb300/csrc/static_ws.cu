// Bidirectional FAVOR+ for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc where they run the attention: code
// embedded in a host framework that owns all device memory and forbids
// allocation on its request path, or latency-critical code for which an
// allocation (which can synchronise the device and takes the driver's
// allocation lock) is not acceptable at the point of use.  This entry point
// runs the same kernels as favor_fwd_bidir with the scratch memory in a
// fixed file-scope device array instead of a caller-provided workspace.
#include <mutex>

#include "common.cuh"

namespace {

constexpr size_t kStaticScratchBytes = size_t(16) << 20;   // 16 MiB on every device that loads the library

__device__ __align__(256) uint8_t g_favor_static_scratch[kStaticScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_ptr[64] = {};

// Device address of the array on the current device (resolved once per
// device; the array's name in host code is only a host-side handle).  The
// resolution is refused while `stream` is being captured into a graph:
// *capturing is set and nothing else happens.
cudaError_t scratch_address(void** out, cudaStream_t stream, bool* capturing) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) {
      (void)cudaGetLastError();
      *capturing = true;
      return cudaErrorStreamCaptureUnsupported;
    }
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_favor_static_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" favor_status favor_fwd_bidir_static(const void* Q, const void* K, const void* V, void* O, int B, int H,
                                               int L, int d, const float* omega, int m, favor_dtype dt,
                                               float qk_scale, int32_t* dev_status, void* stream) {
  const size_t need = favor_workspace_bytes(0, B, H, L, d, m, dt);
  if (need == 0)   // malformed or unsupported shape: report it as favor_fwd_bidir would
    return favor::run_call(false, 3, Q, K, V, O, B, H, L, d, omega, m, dt, qk_scale, nullptr, 0, dev_status, stream);
  if (need > kStaticScratchBytes) return FAVOR_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  bool capturing = false;
  if (scratch_address(&scratch, static_cast<cudaStream_t>(stream), &capturing) != cudaSuccess)
    return capturing ? FAVOR_ERR_INVALID_ARG : FAVOR_ERR_CUDA;
  return favor::run_call(false, 3, Q, K, V, O, B, H, L, d, omega, m, dt, qk_scale, scratch, kStaticScratchBytes,
                         dev_status, stream);
}

extern "C" size_t favor_static_scratch_bytes(void) { return kStaticScratchBytes; }
