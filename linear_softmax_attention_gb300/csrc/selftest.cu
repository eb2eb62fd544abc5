// Test hook of the bounded waits (no fault): two warps wait on mbarriers
// that nothing completes; the first wait gives up after the wait limit and
// raises the abort flag, the second then returns at once.
#include "favor_selftest.h"
#include "tc_ptx.cuh"

namespace favor {
namespace {

constexpr uint64_t kSecondStartNs = 500000000ull;   // warp 1 begins waiting 0.5 s in

__global__ void wait_timeout_kernel(int32_t* status, int32_t* returned, int64_t* times_ns) {
  __shared__ __align__(8) uint64_t bars[2];
  __shared__ volatile int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bars[0], 1);
    tc::mbar_init(&bars[1], 1);
    tc::fence_barrier_init();
    abort_flag = 0;
    times_ns[0] = static_cast<int64_t>(tc::global_timer());
  }
  __syncthreads();
  if (lane != 0) return;
  if (warp == 1) {
    const uint64_t t0 = tc::global_timer();
    while (tc::global_timer() - t0 < kSecondStartNs) {
    }
  }
  const tc::WaitCtx ctx{&abort_flag, status};
  const bool done = tc::mbar_wait(&bars[warp], 0u, ctx);   // phase 0 never completes
  returned[warp] = done ? 1 : 2;
  times_ns[1 + warp] = static_cast<int64_t>(tc::global_timer());
}

}  // namespace
}  // namespace favor

extern "C" favor_status favor_selftest_wait_timeout(int32_t* status, int32_t* returned, int64_t* times_ns,
                                                    void* stream) {
  if (status == nullptr || returned == nullptr || times_ns == nullptr) return FAVOR_ERR_INVALID_ARG;
  favor::wait_timeout_kernel<<<1, 64, 0, static_cast<cudaStream_t>(stream)>>>(status, returned, times_ns);
  return cudaGetLastError() == cudaSuccess ? FAVOR_OK : FAVOR_ERR_CUDA;
}
