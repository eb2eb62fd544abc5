// Tensor-core (tcgen05) FAVOR+ kernels.
#include "tc.cuh"

namespace favor {

bool tc_supported(bool, int, int, bool) { return false; }
size_t tc_workspace_bytes(bool, const Shape&) { return 0; }
cudaError_t tc_state(bool, const void*, const void*, const float*, float, const Shape&, void*, int32_t*,
                     cudaStream_t) {
  return cudaErrorNotSupported;
}
cudaError_t tc_output(bool, const void*, const void*, const void*, void*, const float*, float, const Shape&, void*,
                      int32_t*, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace favor
