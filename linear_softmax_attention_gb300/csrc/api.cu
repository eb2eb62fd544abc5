// C ABI entry points: argument checks, workspace planning and dispatch.
#include <algorithm>
#include <cmath>

#include "backward.cuh"
#include "common.cuh"
#include "tc.cuh"

#include <mutex>
#include <unordered_map>

using favor::Shape;

namespace favor {

cudaError_t ensure_dynamic_smem(const void* kernel, size_t bytes) {
  static std::mutex mu;
  static std::unordered_map<const void*, size_t> done[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  size_t& have = done[dev][kernel];
  if (have >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) have = bytes;
  return e;
}

// Streaming multiprocessors of the current device (cached per device); the
// workspace plans size their grids by it, so a workspace is planned for the
// device it is used on.
int sm_count() {
  static std::mutex mu;
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

}  // namespace favor

namespace {

constexpr int kVersion = FAVOR_API_VERSION;

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// [p, p + n) as bytes
struct Range {
  const void* p;
  size_t n;
};
bool overlaps(const Range& a, const Range& b) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.p), b0 = reinterpret_cast<uintptr_t>(b.p);
  return a0 < b0 + b.n && b0 < a0 + a.n;
}

favor_status shape_ok(int B, int H, int L, int d, int m, favor_dtype dt) {
  if (B < 1 || H < 1 || L < 1 || d < 1 || m < 1) return FAVOR_ERR_INVALID_ARG;
  if (dt != FAVOR_F32 && dt != FAVOR_BF16) return FAVOR_ERR_INVALID_ARG;
  if (d > favor::kMaxD || m > favor::kMaxM) return FAVOR_ERR_UNSUPPORTED;
  const long long bh = (long long)B * H;
  if (bh > 65535) return FAVOR_ERR_UNSUPPORTED;
  if (bh * L * (long long)d >= (1ll << 31)) return FAVOR_ERR_UNSUPPORTED;
  return FAVOR_OK;
}

bool use_tc(bool causal, int d, int m, favor_dtype dt) { return favor::tc_supported(causal, d, m, dt == FAVOR_BF16); }

// the tensor-core kernels carry every feature map (the map only changes
// their epilogue)
bool use_tc_fm(bool causal, int d, int m, favor_dtype dt, int fm) {
  (void)fm;
  return use_tc(causal, d, m, dt);
}

bool fm_ok(int fm) { return fm == FAVOR_FM_PRF || fm == FAVOR_FM_RELU || fm == FAVOR_FM_ELU1; }

size_t ws_bytes_for(bool causal, const Shape& s, favor_dtype dt, int fm = FAVOR_FM_PRF) {
  if (use_tc_fm(causal, s.d, s.m, dt, fm)) return favor::tc_workspace_bytes(causal, s);
  return favor::simt_plan(causal, s).bytes;
}

enum Stage { kState = 1, kOutput = 2, kBoth = 3 };

favor_status run(bool causal, int stage, const void* Q, const void* K, const void* V, void* O, int B, int H, int L,
                 int d, const float* omega, int m, favor_dtype dt, float qk_scale, void* workspace,
                 size_t ws_bytes, int32_t* dev_status, void* stream_, int fm = FAVOR_FM_PRF) {
  favor_status st = shape_ok(B, H, L, d, m, dt);
  if (st != FAVOR_OK) return st;
  if (!fm_ok(fm)) return FAVOR_ERR_INVALID_ARG;
  if (!std::isfinite(qk_scale) || !(qk_scale > 0.f)) return FAVOR_ERR_INVALID_ARG;
  const bool need_q = (stage & kOutput) != 0;
  const bool need_kv = (stage & kState) != 0 || causal;
  if (omega == nullptr || workspace == nullptr) return FAVOR_ERR_INVALID_ARG;
  if (need_q && (Q == nullptr || O == nullptr)) return FAVOR_ERR_INVALID_ARG;
  if (need_kv && (K == nullptr || V == nullptr)) return FAVOR_ERR_INVALID_ARG;
  for (const void* p : {Q, K, V, static_cast<const void*>(O), static_cast<const void*>(omega)})
    if (p != nullptr && !aligned(p, 16)) return FAVOR_ERR_INVALID_ARG;
  if (!aligned(workspace, 256)) return FAVOR_ERR_INVALID_ARG;
  if (need_q && (O == Q || O == K || O == V)) return FAVOR_ERR_INVALID_ARG;
  const Shape s{B, H, L, d, m};
  if (ws_bytes < ws_bytes_for(causal, s, dt, fm)) return FAVOR_ERR_INVALID_ARG;

  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  const bool bf16 = dt == FAVOR_BF16;
  cudaError_t e = cudaSuccess;
  if (use_tc_fm(causal, d, m, dt, fm)) {
    if (stage & kState) e = favor::tc_state(causal, K, V, omega, qk_scale, s, workspace, dev_status, stream, fm);
    if (e == cudaSuccess && (stage & kOutput))
      e = favor::tc_output(causal, Q, K, V, O, omega, qk_scale, s, workspace, dev_status, stream, fm);
  } else if (!causal) {
    if (stage & kState)
      e = favor::simt_bidir_state(K, V, omega, qk_scale, s, bf16, workspace, dev_status, stream, fm);
    if (e == cudaSuccess && (stage & kOutput))
      e = favor::simt_bidir_output(Q, O, omega, qk_scale, s, bf16, workspace, dev_status, stream, fm);
  } else {
    if (stage & kState)
      e = favor::simt_causal_state(K, V, omega, qk_scale, s, bf16, workspace, dev_status, stream, fm);
    if (e == cudaSuccess && (stage & kOutput))
      e = favor::simt_causal_output(Q, K, V, O, omega, qk_scale, s, bf16, workspace, dev_status, stream, fm);
  }
  return e == cudaSuccess ? FAVOR_OK : FAVOR_ERR_CUDA;
}

}  // namespace

namespace favor {
favor_status run_call(bool causal, int stage, const void* Q, const void* K, const void* V, void* O, int B, int H,
                      int L, int d, const float* omega, int m, favor_dtype dt, float qk_scale, void* workspace,
                      size_t ws_bytes, int32_t* dev_status, void* stream) {
  return run(causal, stage, Q, K, V, O, B, H, L, d, omega, m, dt, qk_scale, workspace, ws_bytes, dev_status, stream);
}
}  // namespace favor

namespace {
favor_status bwd_run(bool causal, const void* Q, const void* K, const void* V, const void* dO, void* dQ, void* dK,
                     void* dV, int B, int H, int L, int d, const float* omega, int m, favor_dtype dt, float qk_scale,
                     favor_feature_map fm, void* workspace, size_t ws_bytes, int32_t* dev_status, void* stream) {
  favor_status st = shape_ok(B, H, L, d, m, dt);
  if (st != FAVOR_OK) return st;
  if (!fm_ok(fm)) return FAVOR_ERR_INVALID_ARG;
  if (!std::isfinite(qk_scale) || !(qk_scale > 0.f)) return FAVOR_ERR_INVALID_ARG;
  const void* in[] = {Q, K, V, dO, static_cast<const void*>(omega)};
  const void* out[] = {dQ, dK, dV};
  for (const void* p : in)
    if (p == nullptr || !aligned(p, 16)) return FAVOR_ERR_INVALID_ARG;
  for (const void* p : out) {
    if (p == nullptr || !aligned(p, 16)) return FAVOR_ERR_INVALID_ARG;
    for (const void* q : in)
      if (p == q) return FAVOR_ERR_INVALID_ARG;
  }
  if (dQ == dK || dQ == dV || dK == dV) return FAVOR_ERR_INVALID_ARG;
  if (workspace == nullptr || !aligned(workspace, 256)) return FAVOR_ERR_INVALID_ARG;
  const Shape s{B, H, L, d, m};
  const bool bf16 = dt == FAVOR_BF16;
  cudaStream_t st_ = static_cast<cudaStream_t>(stream);
  if (favor::tc_bwd_supported(causal, d, m, bf16)) {
    if (ws_bytes < favor::tc_bwd_workspace_bytes(s)) return FAVOR_ERR_INVALID_ARG;
    const cudaError_t e = favor::tc_bwd_bidir(Q, K, V, dO, dQ, dK, dV, omega, qk_scale, s, workspace, dev_status,
                                              st_, static_cast<int>(fm));
    return e == cudaSuccess ? FAVOR_OK : FAVOR_ERR_CUDA;
  }
  if (ws_bytes < favor::bwd_plan(s).bytes) return FAVOR_ERR_INVALID_ARG;
  cudaError_t e = causal ? favor::simt_bwd_causal(Q, K, V, dO, dQ, dK, dV, omega, qk_scale, s, bf16, workspace,
                                                  dev_status, st_, static_cast<int>(fm))
                         : favor::simt_bwd_bidir(Q, K, V, dO, dQ, dK, dV, omega, qk_scale, s, bf16, workspace,
                                                 dev_status, st_, static_cast<int>(fm));
  return e == cudaSuccess ? FAVOR_OK : FAVOR_ERR_CUDA;
}
}  // namespace

extern "C" {

int favor_api_version(void) { return kVersion; }

const char* favor_status_string(favor_status s) {
  switch (s) {
    case FAVOR_OK: return "ok";
    case FAVOR_ERR_INVALID_ARG: return "invalid argument";
    case FAVOR_ERR_UNSUPPORTED: return "unsupported shape";
    case FAVOR_ERR_CUDA: return "CUDA error";
    case FAVOR_ERR_TIMEOUT: return "device wait timed out";
    case FAVOR_ERR_NONFINITE: return "non-finite or non-positive normaliser";
  }
  return "unknown status";
}

const char* favor_path_name(int causal, int d, int m, favor_dtype dt) {
  if (shape_ok(1, 1, 1, d, m, dt) != FAVOR_OK) return "unsupported";
  return use_tc(causal != 0, d, m, dt) ? "tcgen05" : "simt";
}

favor_status favor_build_orf(uint64_t seed, int m, int d, int orthogonal, float* omega, void* stream) {
  if (omega == nullptr || m < 1 || d < 1 || m > favor::kMaxM || d > favor::kMaxD) return FAVOR_ERR_INVALID_ARG;
  if (orthogonal < 0 || orthogonal > 3) return FAVOR_ERR_INVALID_ARG;
  if (orthogonal == 2 && (d & (d - 1)) != 0) return FAVOR_ERR_UNSUPPORTED;   // Hadamard: d a power of two
  if (orthogonal == 3 && d < 2) return FAVOR_ERR_UNSUPPORTED;                // Givens: a plane needs d >= 2
  cudaError_t e = favor::launch_build_orf(seed, m, d, orthogonal, omega, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FAVOR_OK : FAVOR_ERR_CUDA;
}

size_t favor_workspace_bytes(int causal, int B, int H, int L, int d, int m, favor_dtype dt) {
  if (shape_ok(B, H, L, d, m, dt) != FAVOR_OK) return 0;
  return ws_bytes_for(causal != 0, Shape{B, H, L, d, m}, dt);
}

size_t favor_workspace_bytes_fm(int causal, int B, int H, int L, int d, int m, favor_dtype dt,
                                favor_feature_map fm) {
  if (shape_ok(B, H, L, d, m, dt) != FAVOR_OK || !fm_ok(fm)) return 0;
  return ws_bytes_for(causal != 0, Shape{B, H, L, d, m}, dt, fm);
}

#define FAVOR_ARGS                                                                                      \
  const void *Q, const void *K, const void *V, void *O, int B, int H, int L, int d, const float *omega, \
      int m, favor_dtype dt, float qk_scale, void *workspace, size_t ws_bytes, int32_t *dev_status,     \
      void *stream
#define FAVOR_PASS Q, K, V, O, B, H, L, d, omega, m, dt, qk_scale, workspace, ws_bytes, dev_status, stream

favor_status favor_fwd_bidir(FAVOR_ARGS) { return run(false, kBoth, FAVOR_PASS); }
favor_status favor_fwd_causal(FAVOR_ARGS) { return run(true, kBoth, FAVOR_PASS); }
favor_status favor_bidir_state(FAVOR_ARGS) { return run(false, kState, FAVOR_PASS); }
favor_status favor_bidir_output(FAVOR_ARGS) { return run(false, kOutput, FAVOR_PASS); }
favor_status favor_causal_state(FAVOR_ARGS) { return run(true, kState, FAVOR_PASS); }
favor_status favor_causal_output(FAVOR_ARGS) { return run(true, kOutput, FAVOR_PASS); }

favor_status favor_fwd_bidir_fm(const void* Q, const void* K, const void* V, void* O, int B, int H, int L, int d,
                                const float* omega, int m, favor_dtype dt, float qk_scale, favor_feature_map fm,
                                void* workspace, size_t ws_bytes, int32_t* dev_status, void* stream) {
  return run(false, kBoth, FAVOR_PASS, static_cast<int>(fm));
}
favor_status favor_fwd_causal_fm(const void* Q, const void* K, const void* V, void* O, int B, int H, int L, int d,
                                 const float* omega, int m, favor_dtype dt, float qk_scale, favor_feature_map fm,
                                 void* workspace, size_t ws_bytes, int32_t* dev_status, void* stream) {
  return run(true, kBoth, FAVOR_PASS, static_cast<int>(fm));
}

size_t favor_bwd_workspace_bytes(int B, int H, int L, int d, int m, favor_dtype dt) {
  if (shape_ok(B, H, L, d, m, dt) != FAVOR_OK) return 0;
  const Shape s{B, H, L, d, m};
  // one size serves both passes: the bidirectional pass may take the
  // tensor-core kernels, the causal pass the CUDA-core ones
  size_t bytes = favor::bwd_plan(s).bytes;
  if (favor::tc_bwd_supported(false, d, m, dt == FAVOR_BF16)) bytes = std::max(bytes, favor::tc_bwd_workspace_bytes(s));
  return bytes;
}


favor_status favor_bwd_bidir(const void* Q, const void* K, const void* V, const void* dO, void* dQ, void* dK,
                             void* dV, int B, int H, int L, int d, const float* omega, int m, favor_dtype dt,
                             float qk_scale, favor_feature_map fm, void* workspace, size_t ws_bytes,
                             int32_t* dev_status, void* stream) {
  return bwd_run(false, Q, K, V, dO, dQ, dK, dV, B, H, L, d, omega, m, dt, qk_scale, fm, workspace, ws_bytes,
                 dev_status, stream);
}

favor_status favor_bwd_causal(const void* Q, const void* K, const void* V, const void* dO, void* dQ, void* dK,
                              void* dV, int B, int H, int L, int d, const float* omega, int m, favor_dtype dt,
                              float qk_scale, favor_feature_map fm, void* workspace, size_t ws_bytes,
                              int32_t* dev_status, void* stream) {
  return bwd_run(true, Q, K, V, dO, dQ, dK, dV, B, H, L, d, omega, m, dt, qk_scale, fm, workspace, ws_bytes,
                 dev_status, stream);
}

favor_status favor_decode_step(const void* q, const void* k, const void* v, void* o, int B, int H, int d,
                               const float* omega, int m, favor_dtype dt, float qk_scale, float* state,
                               int32_t* dev_status, void* stream) {
  favor_status st = shape_ok(B, H, 1, d, m, dt);
  if (st != FAVOR_OK) return st;
  if (!std::isfinite(qk_scale) || !(qk_scale > 0.f)) return FAVOR_ERR_INVALID_ARG;
  for (const void* p : {q, k, v, static_cast<const void*>(o), static_cast<const void*>(omega),
                        static_cast<const void*>(state)})
    if (p == nullptr || !aligned(p, 16)) return FAVOR_ERR_INVALID_ARG;
  // o and the state are written: neither may overlap anything else
  const size_t e_sz = dt == FAVOR_BF16 ? 2 : 4;
  const size_t tok_bytes = (size_t)B * H * d * e_sz;
  const size_t st_bytes = (size_t)B * H * (d + 1) * m * sizeof(float);
  const Range ro{o, tok_bytes}, rs{state, st_bytes};
  for (const void* in : {q, k, v}) {
    const Range r{in, tok_bytes};
    if (overlaps(ro, r) || overlaps(rs, r)) return FAVOR_ERR_INVALID_ARG;
  }
  if (overlaps(ro, rs)) return FAVOR_ERR_INVALID_ARG;
  cudaError_t e = favor::launch_decode_step(q, k, v, o, B * H, d, omega, m, dt == FAVOR_BF16, qk_scale, state,
                                            dev_status, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FAVOR_OK : FAVOR_ERR_CUDA;
}

size_t favor_decode_prefill_workspace_bytes(int B, int H, int L, int d, int m, favor_dtype dt) {
  if (shape_ok(B, H, L, d, m, dt) != FAVOR_OK) return 0;
  return favor::simt_plan(false, Shape{B, H, L, d, m}).bytes;
}

favor_status favor_decode_prefill(const void* K, const void* V, int B, int H, int L, int d, const float* omega,
                                  int m, favor_dtype dt, float qk_scale, float* state, void* workspace,
                                  size_t ws_bytes, int32_t* dev_status, void* stream) {
  (void)dev_status;
  favor_status st = shape_ok(B, H, L, d, m, dt);
  if (st != FAVOR_OK) return st;
  if (!std::isfinite(qk_scale) || !(qk_scale > 0.f)) return FAVOR_ERR_INVALID_ARG;
  for (const void* p : {K, V, static_cast<const void*>(omega), static_cast<const void*>(state)})
    if (p == nullptr || !aligned(p, 16)) return FAVOR_ERR_INVALID_ARG;
  if (workspace == nullptr || !aligned(workspace, 256)) return FAVOR_ERR_INVALID_ARG;
  const Shape s{B, H, L, d, m};
  if (ws_bytes < favor::simt_plan(false, s).bytes) return FAVOR_ERR_INVALID_ARG;
  cudaError_t e = favor::simt_state_export(K, V, omega, qk_scale, s, dt == FAVOR_BF16, workspace, state,
                                           static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FAVOR_OK : FAVOR_ERR_CUDA;
}

}  // extern "C"
