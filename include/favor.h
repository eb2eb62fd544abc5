/*
 * favor.h — C ABI of the FAVOR+ forward pass for one GB300 GPU (sm_103a).
 *
 * FAVOR+ ("Fast Attention Via positive Orthogonal Random features") replaces
 * softmax(QK^T)V by a product of random-feature matrices:
 *
 *   phi(x)       = m^{-1/2} exp(Omega x - ||x||^2 / 2)            (PRF map)
 *   bidirectional:  Attn^(Q,K,V) = D^{-1} phi(Q) (phi(K)^T V),
 *                   D = diag(phi(Q) (phi(K)^T 1_L))
 *   unidirectional: out_t = phi(q_t)^T G_t / phi(q_t)^T z_t,
 *                   G_t = sum_{s<=t} phi(k_s) v_s^T,  z_t = sum_{s<=t} phi(k_s)
 *
 * Sources: "Performer — Rethinking Attention with Performers" (blog digest),
 * §Key equations and §Methods (FAVOR+); "Rethinking Attention with
 * Performers" (arXiv:2009.14794v4 summary), §2 FAVOR+ mechanism and §A.2
 * unidirectional attention; "From Performer to Linear Attention" (Su), §Simple
 * Derivation.
 *
 * Conventions shared by every call:
 *  - Q, K, V, O: device pointers to contiguous [B, H, L, d] tensors, d
 *    fastest, all of dtype `dt`; 16-byte aligned.  O may not alias Q, K, V.
 *  - omega: device pointer to fp32 [m, d], row i = omega_i, shared by every
 *    (b, h) and by Q and K.
 *  - qk_scale: temperature s > 0; q and k enter the feature map as s*q and
 *    s*k (s = d^{-1/4} reproduces softmax(QK^T / sqrt(d))).  A non-positive
 *    or non-finite s is FAVOR_ERR_INVALID_ARG.
 *  - workspace: caller-owned device scratch of at least
 *    favor_workspace_bytes(...) bytes, 256-byte aligned; its contents between
 *    calls do not matter.  Calls that share a workspace must be ordered on
 *    one stream.
 *  - dev_status: optional device int32 (may be NULL).  Kernels store a
 *    non-zero favor_status there when they detect a bounded wait that ran out
 *    (FAVOR_ERR_TIMEOUT) or a non-finite / non-positive normaliser
 *    (FAVOR_ERR_NONFINITE); the library never clears it.  Read it after the
 *    stream has synchronised.
 *  - stream: a cudaStream_t passed as void* (NULL = legacy default stream).
 *  - The library never allocates, frees or synchronises; all launches are
 *    asynchronous on `stream`.  The return value reports argument checks
 *    (made before anything is launched) and launch errors.
 *  - Supported: 1 <= L, 1 <= d <= 128, 1 <= m <= 512, B*H >= 1,
 *    B*H*L*d < 2^31.  bf16 with d = 64 and m in {128, 256}, or with
 *    d = 128 and m in {128, 256, 512}, runs on the tcgen05 tensor-core
 *    kernels (favor_path_name reports which); every other supported shape
 *    runs on CUDA-core kernels with fp32 arithmetic.
 */
#ifndef FAVOR_H_
#define FAVOR_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FAVOR_API_VERSION 1

typedef enum favor_status {
  FAVOR_OK = 0,
  FAVOR_ERR_INVALID_ARG = 1,  /* a pointer, size or alignment is out of contract */
  FAVOR_ERR_UNSUPPORTED = 2,  /* well-formed but outside the supported shapes    */
  FAVOR_ERR_CUDA = 3,         /* a CUDA runtime/driver call or launch failed      */
  FAVOR_ERR_TIMEOUT = 4,      /* device only: a bounded wait gave up              */
  FAVOR_ERR_NONFINITE = 5     /* device only: non-finite or <= 0 normaliser       */
} favor_status;

typedef enum favor_dtype {
  FAVOR_F32 = 0,   /* fp32 storage, fp32 arithmetic                            */
  FAVOR_BF16 = 1   /* bf16 storage, bf16 tensor-core operands, fp32 accumulate */
} favor_dtype;

/*
 * Feature map phi of the *_fm calls.  FAVOR_FM_PRF: positive random
 * features, phi(x) = m^{-1/2} exp(Omega x - ||x||^2 / 2), the softmax kernel
 * (every call without the _fm suffix).  FAVOR_FM_RELU: Performer-ReLU,
 * phi(x) = m^{-1/2} relu(Omega x) elementwise ("Rethinking Attention with
 * Performers" summary, §2 generalized kernelizable attention: other kernels
 * by changing the feature-map function; §3 and §D.2 name Performer-ReLU; the
 * pages print no formula, this is the plain reading).  relu is positively
 * homogeneous, so qk_scale cancels in the ReLU outputs.  FAVOR_FM_ELU1:
 * phi(x) = m^{-1/2} (1 + elu(Omega x)), 1 + a for a >= 0 and exp(a) below
 * ("From Performer to Linear Attention", the linear-attention feature map it
 * compares against; the "Performer" digest names it as Linear Attention's),
 * in the same slot as ReLU; with Omega = I_d (m = d) it is linear attention
 * itself.  Every map takes the path of the plain call for its shape (the
 * tensor-core kernels where they apply, the CUDA-core kernels otherwise):
 * the map changes only the epilogue that forms the features.
 */
typedef enum favor_feature_map {
  FAVOR_FM_PRF = 0,
  FAVOR_FM_RELU = 1,
  FAVOR_FM_ELU1 = 2
} favor_feature_map;

/* Library version (FAVOR_API_VERSION of the build). */
int favor_api_version(void);

/* Static English text for a status code (never NULL). */
const char* favor_status_string(favor_status s);

/*
 * favor_build_orf — draw the projection Omega [m, d] (fp32, row-major) into
 * the caller's device buffer `omega`, on `stream`.
 *
 * orthogonal = 1 (ORF): ceil(m/d) independent d x d blocks; block b's rows
 * are the Gram–Schmidt orthonormalisation of a Gaussian matrix, and row r is
 * then scaled to the length of an independent N(0, I_d) vector (a chi_d
 * sample), so each row keeps the N(0, I_d) marginal ("Performer" digest,
 * §Methods ORF bullet and the block-wise rule for m > d; arXiv summary §A.2:
 * orthogonality with marginals preserved).  The first m stacked rows are
 * kept.  orthogonal = 0: iid N(0, 1) entries.  orthogonal = 2 (Hadamard
 * ORF, d a power of two): block b = sqrt(d) (H D_1)(H D_2)(H D_3), H the
 * normalised d x d Walsh-Hadamard matrix, D_p = diag(+-1) with sign i of
 * product p from the top bit of SplitMix64 word (b*3 + p)*d + i (1 -> -1);
 * exactly orthogonal blocks with rows of length sqrt(d), O(m) random numbers
 * (arXiv summary §A.2: Hadamard ORFs, a small bias that tends to zero as d
 * grows; §B.3: their O(m) space; no construction is printed, this is the
 * plain reading).  orthogonal = 3 (Givens ORF, d >= 2): block b = sqrt(d)
 * G_K ... G_2 G_1 with K = 3 d ceil(log2 d) plane rotations, (G x)_i =
 * cos(theta) x_i - sin(theta) x_j, (G x)_j = sin(theta) x_i + cos(theta) x_j;
 * rotation r of block b reads SplitMix64 words 2c and 2c + 1, c = b K + r:
 * i = floor(hi32 d / 2^32), j' = floor(lo32 (d - 1) / 2^32), j = j' +
 * [j' >= i] from the first, theta = 2 pi (bits[41..63] + 1/2) / 2^23 from
 * the second; exactly orthogonal blocks (determinant +1) with rows of length
 * sqrt(d), O(m log d) random numbers (arXiv summary §A.2 and §B.3: Givens
 * ORFs, a small bias, O(m log d) space; again the plain reading).
 *
 * Random numbers: SplitMix64 word i = mix(seed + (i+1)*0x9E3779B97F4A7C15);
 * one normal per word by Box–Muller, z = sqrt(-2 ln u1) cos(2 pi u2) with
 * u1 = (bits[41..63] + 1/2) / 2^23 and u2 = (bits[18..40] + 1/2) / 2^23.
 * Counter of Gaussian entry (r, c) of block b: ((b*d + r)*d + c)*2; of
 * component c of row r's length vector: the same + 1; iid entry (i, c):
 * (i*d + c)*2.  Arithmetic is fp32 (two Gram–Schmidt sweeps).
 *
 * Errors: FAVOR_ERR_INVALID_ARG if omega is NULL, m, d out of range
 * (1 <= d <= 128, 1 <= m <= 512) or orthogonal not 0, 1, 2 or 3;
 * FAVOR_ERR_UNSUPPORTED for orthogonal = 2 with d not a power of two and for
 * orthogonal = 3 with d = 1.
 */
favor_status favor_build_orf(uint64_t seed, int m, int d, int orthogonal,
                             float* omega, void* stream);

/*
 * favor_workspace_bytes — scratch bytes needed by favor_fwd_bidir (causal = 0)
 * or favor_fwd_causal (causal = 1) and by their stage calls for the given
 * shape.  Returns 0 for arguments outside the supported shapes.
 */
size_t favor_workspace_bytes(int causal, int B, int H, int L, int d, int m,
                             favor_dtype dt);

/*
 * favor_fwd_bidir — bidirectional FAVOR+:
 *   O = D^{-1} phi(s Q) (phi(s K)^T V),  D = diag(phi(s Q) phi(s K)^T 1_L)
 * ("Performer" digest, §Key equations, linear attention line; flowchart:
 * phi(K)^T V and phi(K)^T 1 first, then phi(Q) times each, then the
 * row-wise divide).  Equivalent to favor_bidir_state then favor_bidir_output.
 */
favor_status favor_fwd_bidir(const void* Q, const void* K, const void* V, void* O,
                             int B, int H, int L, int d,
                             const float* omega, int m, favor_dtype dt, float qk_scale,
                             void* workspace, size_t ws_bytes,
                             int32_t* dev_status, void* stream);

/*
 * favor_fwd_causal — unidirectional FAVOR+ (diagonal included):
 *   O_t = phi(s q_t)^T G_t / phi(s q_t)^T z_t,
 *   G_t = sum_{s<=t} phi(s k_s) v_s^T,  z_t = sum_{s<=t} phi(s k_s)
 * ("Performer" digest, §Methods causal bullet; arXiv summary §2 "lower
 * triangular part" and §A.2 prefix sums).  Equivalent to favor_causal_state
 * then favor_causal_output.
 */
favor_status favor_fwd_causal(const void* Q, const void* K, const void* V, void* O,
                              int B, int H, int L, int d,
                              const float* omega, int m, favor_dtype dt, float qk_scale,
                              void* workspace, size_t ws_bytes,
                              int32_t* dev_status, void* stream);

/*
 * favor_fwd_bidir_fm, favor_fwd_causal_fm — favor_fwd_bidir and
 * favor_fwd_causal with the feature map `fm` (favor_feature_map) in place of
 * the positive random features; same arguments.  Every map takes the same
 * path and workspace size as the plain call (favor_workspace_bytes_fm equals
 * favor_workspace_bytes for each map).
 * A row whose features are all zero (every s w_i.q <= 0 under ReLU) has a
 * zero normaliser: its output is NaN and dev_status gets
 * FAVOR_ERR_NONFINITE (1 + elu is positive: it never has one).  fm outside
 * the enum is FAVOR_ERR_INVALID_ARG.
 */
size_t favor_workspace_bytes_fm(int causal, int B, int H, int L, int d, int m,
                                favor_dtype dt, favor_feature_map fm);
favor_status favor_fwd_bidir_fm(const void* Q, const void* K, const void* V, void* O,
                                int B, int H, int L, int d,
                                const float* omega, int m, favor_dtype dt, float qk_scale,
                                favor_feature_map fm, void* workspace, size_t ws_bytes,
                                int32_t* dev_status, void* stream);
favor_status favor_fwd_causal_fm(const void* Q, const void* K, const void* V, void* O,
                                 int B, int H, int L, int d,
                                 const float* omega, int m, favor_dtype dt, float qk_scale,
                                 favor_feature_map fm, void* workspace, size_t ws_bytes,
                                 int32_t* dev_status, void* stream);

/*
 * Stage calls (same arguments as the full calls; pointers a stage does not
 * read may be NULL).  They let a caller time or reuse each half:
 *
 * favor_bidir_state  — reads K, V; writes phi(K)^T [V | 1] (stabilised, one
 *                      shared scale per head) into the workspace.
 * favor_bidir_output — reads Q and the workspace state; writes O.
 * favor_causal_state — reads K, V; writes one phi(K)^T [V | 1] per
 *                      superchunk of the sequence into the workspace.
 * favor_causal_output— reads Q, K, V and those superchunk states; writes O.
 *
 * A *_output call must follow the matching *_state call with the same shape,
 * omega, qk_scale and workspace on the same stream.
 */
favor_status favor_bidir_state(const void* Q, const void* K, const void* V, void* O,
                               int B, int H, int L, int d,
                               const float* omega, int m, favor_dtype dt, float qk_scale,
                               void* workspace, size_t ws_bytes,
                               int32_t* dev_status, void* stream);
favor_status favor_bidir_output(const void* Q, const void* K, const void* V, void* O,
                                int B, int H, int L, int d,
                                const float* omega, int m, favor_dtype dt, float qk_scale,
                                void* workspace, size_t ws_bytes,
                                int32_t* dev_status, void* stream);
favor_status favor_causal_state(const void* Q, const void* K, const void* V, void* O,
                                int B, int H, int L, int d,
                                const float* omega, int m, favor_dtype dt, float qk_scale,
                                void* workspace, size_t ws_bytes,
                                int32_t* dev_status, void* stream);
favor_status favor_causal_output(const void* Q, const void* K, const void* V, void* O,
                                 int B, int H, int L, int d,
                                 const float* omega, int m, favor_dtype dt, float qk_scale,
                                 void* workspace, size_t ws_bytes,
                                 int32_t* dev_status, void* stream);

/*
 * favor_fwd_bidir_static — favor_fwd_bidir without a caller workspace.  This
 * entry point has no counterpart in the paper; it exists for callers that
 * cannot allocate device memory where they call the attention (code inside a
 * host framework that owns all device memory and forbids allocation on its
 * request path, or latency-critical code that must not take the allocation
 * path, which can synchronise the device).
 *
 * The scratch memory is one file-scope device array of
 * favor_static_scratch_bytes() bytes (16 MiB) that every GPU which loads this
 * library holds until the process exits.  The first call on each device
 * resolves the array's device address (cudaGetSymbolAddress) for that device,
 * so make that first call with the device current and outside any stream
 * capture: a first call on a stream that is being captured returns
 * FAVOR_ERR_INVALID_ARG without launching anything.  The address is kept for
 * the life of the process; after cudaDeviceReset (or any other teardown of
 * the device's primary context) do not call this entry point again.  No call
 * allocates or frees memory.
 *
 * All calls share the one array and leave their intermediate results in it;
 * the kernels clear what must start at zero.  Calls whose execution overlaps
 * on the GPU (different streams, or different host threads on one device)
 * race on the array: order them on one stream.
 *
 * Arguments and results are those of favor_fwd_bidir.  Shapes whose scratch
 * need (favor_workspace_bytes(0, ...)) exceeds the array return
 * FAVOR_ERR_UNSUPPORTED without launching anything.
 */
favor_status favor_fwd_bidir_static(const void* Q, const void* K, const void* V, void* O,
                                    int B, int H, int L, int d,
                                    const float* omega, int m, favor_dtype dt, float qk_scale,
                                    int32_t* dev_status, void* stream);

/* Size in bytes of the fixed scratch array used by favor_fwd_bidir_static. */
size_t favor_static_scratch_bytes(void);

/*
 * favor_bwd_bidir — gradients of the bidirectional pass: given dO = dL/dO
 * for O = favor_fwd_bidir_fm(Q, K, V), writes dQ, dK, dV (contiguous
 * [B, H, L, d], dtype `dt`, not aliasing the inputs).  The chain rule
 * through the forward ("Performer" digest, §Key equations):
 *   N = phi(Q) S, D = phi(Q) z, O = N / D;  dN^ = [dO / D | -(dO . N) / D^2]
 *   dphi(Q) = S~ dN^,  dS~ = phi(Q)^T dN^,  dphi(K) = dS~ [V | 1]^T,
 *   dV = phi(K) dS~[:, :d],  dx = s (sum_i g_i w_i - [prf] s x sum_i g_i)
 * with g = dphi phi (positive random features), dphi [s w.x > 0] (ReLU) or
 * dphi min(phi, 1) (1 + elu); Omega is not differentiated (it is a fixed
 * random draw).  bf16 with d = 64 and m in {128, 256} runs on the tcgen05
 * tensor-core kernels (bf16/fp16 operands, fp32 accumulation; D from the
 * fp32 normaliser, dS~ carried as a bf16 hi + lo pair), every other
 * supported shape on the CUDA-core kernels in fp32; workspace of
 * favor_bwd_workspace_bytes(...) bytes.  A zero or non-finite normaliser is
 * reported in dev_status.
 */
favor_status favor_bwd_bidir(const void* Q, const void* K, const void* V, const void* dO,
                             void* dQ, void* dK, void* dV, int B, int H, int L, int d,
                             const float* omega, int m, favor_dtype dt, float qk_scale,
                             favor_feature_map fm, void* workspace, size_t ws_bytes,
                             int32_t* dev_status, void* stream);
/*
 * favor_bwd_causal — the same for the causal pass (O = favor_fwd_causal_fm):
 * with the prefix state G~_c of the tiles before tile c and the suffix state
 * H_c = sum over later tiles of phi(q) dN^T,
 *   dphi(q_t) = G~_c dN^_t + sum_{s<=t in the tile} (dN^_t . [v_s ; 1]) phi(k_s)
 *   dphi(k_s) = H_c [v_s ; 1] + sum_{t>=s in the tile} (dN^_t . [v_s ; 1]) phi(q_t)
 *   dV_s = H_c[:, :d]^T phi(k_s) + sum_{t>=s in the tile} (phi(k_s).phi(q_t)) dN_t
 * ("Performer" digest, §Methods causal bullet, differentiated).  One CTA per
 * head walks the sequence forward then backward (CUDA-core kernels, every
 * shape).  Same arguments and workspace size as favor_bwd_bidir.
 */
favor_status favor_bwd_causal(const void* Q, const void* K, const void* V, const void* dO,
                              void* dQ, void* dK, void* dV, int B, int H, int L, int d,
                              const float* omega, int m, favor_dtype dt, float qk_scale,
                              favor_feature_map fm, void* workspace, size_t ws_bytes,
                              int32_t* dev_status, void* stream);
/* Workspace bytes of favor_bwd_bidir and favor_bwd_causal. */
size_t favor_bwd_workspace_bytes(int B, int H, int L, int d, int m, favor_dtype dt);

/*
 * Incremental causal FAVOR+ (token-by-token decoding).  The unidirectional
 * form is a recurrence over the prefix sums of favor_fwd_causal: a causal
 * linear attention is a unidirectional RNN whose state is (G_t, z_t)
 * ("From Performer to Linear Attention", §Concentrating Attention; "Performer"
 * digest, §Methods causal bullet and its related-work note on the prefix-sum
 * RNN view; arXiv summary, attention preliminaries: unidirectional attention
 * for autoregressive generation).  These calls carry that state between
 * calls so that one new token per sequence costs O(m d) instead of a pass
 * over the prefix.
 *
 * State layout: `state` is a caller-owned device fp32 array
 * [B, H, d + 1, m] (contiguous, 16-byte aligned, feature index fastest):
 * element (j, i) of head (b, h) holds
 *   sum_{s<=t} exp(s w_i.k_s - s^2 |k_s|^2 / 2 - R) [v_s ; 1]_j
 * (row j = d: the normaliser sums) with R = max_i |w_i|^2 / 2 - 40, a
 * constant of omega alone that every call
 * recomputes (it cancels in the output; it keeps every feature <= e^40).
 * A zero-filled state is the empty prefix.  The state is only meaningful to
 * these calls with the same omega and qk_scale.
 *
 * favor_decode_step — for each (b, h), with q, k, v, o contiguous [B, H, d]
 * (one token per sequence and head, dtype `dt`, 16-byte aligned):
 *   state += phi(s k) [v ; 1]^T   (the new token is part of its own prefix)
 *   o = phi(s q)^T state[:, :d] / phi(s q)^T state[:, d]
 * which equals row t of favor_fwd_causal over the whole sequence, given the
 * state of tokens 0 .. t-1.  The state is read and written in place; the
 * byte ranges of o and of the state may not overlap one another or those of
 * q, k, v (FAVOR_ERR_INVALID_ARG).  A zero or non-finite normaliser is
 * reported in dev_status (FAVOR_ERR_NONFINITE).  Supported: 1 <= d <= 128,
 * 1 <= m <= 512, 1 <= B*H <= 65535, bf16 or fp32.
 *
 * favor_decode_prefill — state = sum over the L tokens of K, V ([B, H, L, d])
 * of phi(s k_t) [v_t ; 1]^T in the layout above (overwriting the state):
 * the state after a prompt, ready for favor_decode_step on token L.  Needs a
 * workspace of favor_decode_prefill_workspace_bytes(...) bytes.
 */
favor_status favor_decode_step(const void* q, const void* k, const void* v, void* o,
                               int B, int H, int d,
                               const float* omega, int m, favor_dtype dt, float qk_scale,
                               float* state, int32_t* dev_status, void* stream);
favor_status favor_decode_prefill(const void* K, const void* V, int B, int H, int L, int d,
                                  const float* omega, int m, favor_dtype dt, float qk_scale,
                                  float* state, void* workspace, size_t ws_bytes,
                                  int32_t* dev_status, void* stream);
size_t favor_decode_prefill_workspace_bytes(int B, int H, int L, int d, int m, favor_dtype dt);

/*
 * favor_path_name — which kernel family a call with these arguments uses:
 * "tcgen05" (bf16 tensor-core kernels), "simt" (CUDA-core fp32 kernels) or
 * "unsupported".  Static string, never NULL.
 */
const char* favor_path_name(int causal, int d, int m, favor_dtype dt);

#ifdef __cplusplus
}
#endif

#endif /* FAVOR_H_ */
