"""FAVOR+ attention forward pass on one GB300 — thin Python binding.

Every function here only marshals arguments (device pointers, sizes, the
current CUDA stream) into the C ABI of ``libfavor.so`` (``include/favor.h``);
all arithmetic runs in the library's CUDA kernels.  PyTorch provides device
memory and streams.  There is no fallback: if the library is missing or a
call fails, an exception is raised.
"""

from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "load", "lib_path", "FavorError", "F32", "BF16", "api_version", "path_name", "build_orf", "new_omega",
    "workspace_bytes", "new_workspace", "fwd_bidir", "fwd_causal", "bidir_state", "bidir_output",
    "causal_state", "causal_output", "status_string", "ENTRY_POINTS", "fwd_bidir_static", "static_scratch_bytes",
    "new_decode_state", "decode_step", "decode_prefill", "decode_prefill_workspace_bytes", "FEATURE_MAPS",
    "bwd_bidir", "bwd_causal", "bwd_workspace_bytes", "selftest_wait_timeout",
]

F32 = 0
BF16 = 1
_DT = {torch.float32: F32, torch.bfloat16: BF16}
FEATURE_MAPS = {"prf": 0, "relu": 1, "elu1": 2}      # favor_feature_map

ENTRY_POINTS = ("favor_fwd_bidir", "favor_fwd_causal", "favor_bidir_state", "favor_bidir_output",
                "favor_causal_state", "favor_causal_output")

_HERE = os.path.dirname(os.path.abspath(__file__))
_lib = None


class FavorError(RuntimeError):
    pass


def lib_path() -> str:
    return os.path.join(_HERE, "libfavor.so")


def load():
    """Load libfavor.so (built by ``linear_softmax_attention_gb300.build``)."""
    global _lib
    if _lib is not None:
        return _lib
    path = lib_path()
    if not os.path.exists(path):
        raise FavorError(f"{path} is missing: build it with `python -m linear_softmax_attention_gb300.build`")
    lib = ctypes.CDLL(path)
    c_int, c_size, c_vp, c_float = ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_float
    lib.favor_api_version.restype = c_int
    lib.favor_status_string.restype = ctypes.c_char_p
    lib.favor_status_string.argtypes = [c_int]
    lib.favor_path_name.restype = ctypes.c_char_p
    lib.favor_path_name.argtypes = [c_int, c_int, c_int, c_int]
    lib.favor_build_orf.restype = c_int
    lib.favor_build_orf.argtypes = [ctypes.c_uint64, c_int, c_int, c_int, c_vp, c_vp]
    lib.favor_workspace_bytes.restype = c_size
    lib.favor_workspace_bytes.argtypes = [c_int, c_int, c_int, c_int, c_int, c_int, c_int]
    lib.favor_workspace_bytes_fm.restype = c_size
    lib.favor_workspace_bytes_fm.argtypes = [c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_int]
    fwd_args = [c_vp, c_vp, c_vp, c_vp, c_int, c_int, c_int, c_int, c_vp, c_int, c_int, c_float, c_vp, c_size,
                c_vp, c_vp]
    for name in ENTRY_POINTS:
        fn = getattr(lib, name)
        fn.restype = c_int
        fn.argtypes = fwd_args
    lib.favor_fwd_bidir_static.restype = c_int
    lib.favor_fwd_bidir_static.argtypes = [c_vp, c_vp, c_vp, c_vp, c_int, c_int, c_int, c_int, c_vp, c_int, c_int,
                                           c_float, c_vp, c_vp]
    lib.favor_static_scratch_bytes.restype = c_size
    fm_args = fwd_args[:12] + [c_int] + fwd_args[12:]
    for name in ("favor_fwd_bidir_fm", "favor_fwd_causal_fm"):
        fn = getattr(lib, name)
        fn.restype = c_int
        fn.argtypes = fm_args
    lib.favor_bwd_bidir.restype = c_int
    lib.favor_bwd_bidir.argtypes = [c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_int, c_int, c_int, c_int, c_vp, c_int,
                                    c_int, c_float, c_int, c_vp, c_size, c_vp, c_vp]
    lib.favor_bwd_causal.restype = c_int
    lib.favor_bwd_causal.argtypes = lib.favor_bwd_bidir.argtypes
    lib.favor_bwd_workspace_bytes.restype = c_size
    lib.favor_bwd_workspace_bytes.argtypes = [c_int, c_int, c_int, c_int, c_int, c_int]
    lib.favor_selftest_wait_timeout.restype = c_int
    lib.favor_selftest_wait_timeout.argtypes = [c_vp, c_vp, c_vp, c_vp]
    lib.favor_decode_step.restype = c_int
    lib.favor_decode_step.argtypes = [c_vp, c_vp, c_vp, c_vp, c_int, c_int, c_int, c_vp, c_int, c_int, c_float,
                                      c_vp, c_vp, c_vp]
    lib.favor_decode_prefill.restype = c_int
    lib.favor_decode_prefill.argtypes = [c_vp, c_vp, c_int, c_int, c_int, c_int, c_vp, c_int, c_int, c_float, c_vp,
                                         c_vp, c_size, c_vp, c_vp]
    lib.favor_decode_prefill_workspace_bytes.restype = c_size
    lib.favor_decode_prefill_workspace_bytes.argtypes = [c_int, c_int, c_int, c_int, c_int, c_int]
    _lib = lib
    return lib


def api_version() -> int:
    return load().favor_api_version()


def status_string(code: int) -> str:
    return load().favor_status_string(code).decode()


def _check(code: int, what: str):
    if code != 0:
        raise FavorError(f"{what}: {status_string(code)} (status {code})")


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def path_name(causal: bool, d: int, m: int, dtype) -> str:
    return load().favor_path_name(int(causal), d, m, _DT[dtype]).decode()


def build_orf(seed: int, omega: torch.Tensor, orthogonal=True, stream=None) -> torch.Tensor:
    """Fill ``omega`` (fp32 [m, d] on the GPU) with the projection for ``seed``:
    orthogonal=True (Gaussian ORF), False (iid), "hadamard" (Hadamard ORF,
    d a power of two) or "givens" (Givens ORF, d >= 2)."""
    if omega.dtype != torch.float32 or not omega.is_cuda or not omega.is_contiguous() or omega.dim() != 2:
        raise FavorError("omega must be a contiguous fp32 CUDA tensor [m, d]")
    m, d = omega.shape
    kind = {"hadamard": 2, "givens": 3}.get(orthogonal, None) if isinstance(orthogonal, str) else int(bool(orthogonal))
    if kind is None:
        raise FavorError(f"unknown projection kind {orthogonal!r}")
    _check(load().favor_build_orf(ctypes.c_uint64(seed & 0xFFFFFFFFFFFFFFFF), m, d, kind,
                                  omega.data_ptr(), _stream_handle(stream)), "favor_build_orf")
    return omega


def new_omega(seed: int, m: int, d: int, orthogonal: bool = True, device="cuda") -> torch.Tensor:
    om = torch.empty((m, d), dtype=torch.float32, device=device)
    return build_orf(seed, om, orthogonal)


def workspace_bytes(causal: bool, B: int, H: int, L: int, d: int, m: int, dtype, feature_map=None) -> int:
    """Workspace bytes of fwd_bidir / fwd_causal for this shape and feature
    map (every map takes the plain call's path and size)."""
    if feature_map in (None, "prf"):
        n = load().favor_workspace_bytes(int(causal), B, H, L, d, m, _DT[dtype])
    else:
        if feature_map not in FEATURE_MAPS:
            raise FavorError(f"feature_map must be one of {sorted(FEATURE_MAPS)}")
        n = load().favor_workspace_bytes_fm(int(causal), B, H, L, d, m, _DT[dtype], FEATURE_MAPS[feature_map])
    if n == 0:
        raise FavorError(f"unsupported shape B={B} H={H} L={L} d={d} m={m} {dtype}")
    return n


def new_workspace(causal: bool, B: int, H: int, L: int, d: int, m: int, dtype, device="cuda",
                  feature_map=None) -> torch.Tensor:
    n = workspace_bytes(causal, B, H, L, d, m, dtype, feature_map)
    return torch.zeros(n, dtype=torch.uint8, device=device)


def _call(name: str, Q, K, V, O, omega, qk_scale, workspace, dev_status, stream, feature_map=None):
    ref = next(t for t in (Q, K, V, O) if t is not None)
    B, H, L, d = ref.shape
    m = omega.shape[0]
    dt = _DT[ref.dtype]
    for t in (Q, K, V, O):
        if t is not None and (not t.is_cuda or not t.is_contiguous() or t.dtype != ref.dtype
                              or tuple(t.shape) != (B, H, L, d)):
            raise FavorError(f"{name}: Q/K/V/O must be contiguous CUDA tensors of one dtype and shape [B,H,L,d]")
    if omega.dtype != torch.float32 or omega.shape[1] != d or not omega.is_contiguous():
        raise FavorError(f"{name}: omega must be contiguous fp32 [m, {d}]")
    ptr = (lambda t: t.data_ptr() if t is not None else None)
    head = (ptr(Q), ptr(K), ptr(V), ptr(O), B, H, L, d, omega.data_ptr(), m, dt, float(qk_scale))
    tail = (workspace.data_ptr(), workspace.numel() * workspace.element_size(), ptr(dev_status),
            _stream_handle(stream))
    if feature_map is None:
        code = getattr(load(), name)(*head, *tail)
    else:
        if feature_map not in FEATURE_MAPS:
            raise FavorError(f"{name}: feature_map must be one of {sorted(FEATURE_MAPS)}")
        name = name + "_fm"
        code = getattr(load(), name)(*head, FEATURE_MAPS[feature_map], *tail)
    _check(code, name)
    return O


def _out_like(x, O):
    return torch.empty_like(x) if O is None else O


def fwd_bidir(Q, K, V, omega, qk_scale, workspace, O=None, dev_status=None, stream=None, feature_map=None):
    """Bidirectional FAVOR+; returns O [B, H, L, d] (dtype of Q).  feature_map:
    None or "prf" (positive random features, the softmax kernel), "relu"
    (Performer-ReLU) or "elu1" (1 + elu, the linear-attention map)."""
    fm = None if feature_map in (None, "prf") else feature_map
    return _call("favor_fwd_bidir", Q, K, V, _out_like(Q, O), omega, qk_scale, workspace, dev_status, stream, fm)


def fwd_causal(Q, K, V, omega, qk_scale, workspace, O=None, dev_status=None, stream=None, feature_map=None):
    """Unidirectional (causal, prefix-sum) FAVOR+; returns O [B, H, L, d].
    feature_map as for fwd_bidir."""
    fm = None if feature_map in (None, "prf") else feature_map
    return _call("favor_fwd_causal", Q, K, V, _out_like(Q, O), omega, qk_scale, workspace, dev_status, stream, fm)


def bidir_state(K, V, omega, qk_scale, workspace, dev_status=None, stream=None):
    _call("favor_bidir_state", None, K, V, None, omega, qk_scale, workspace, dev_status, stream)


def bidir_output(Q, omega, qk_scale, workspace, O=None, dev_status=None, stream=None):
    return _call("favor_bidir_output", Q, None, None, _out_like(Q, O), omega, qk_scale, workspace, dev_status,
                 stream)


def causal_state(K, V, omega, qk_scale, workspace, dev_status=None, stream=None):
    _call("favor_causal_state", None, K, V, None, omega, qk_scale, workspace, dev_status, stream)


def causal_output(Q, K, V, omega, qk_scale, workspace, O=None, dev_status=None, stream=None):
    return _call("favor_causal_output", Q, K, V, _out_like(Q, O), omega, qk_scale, workspace, dev_status, stream)


def static_scratch_bytes() -> int:
    return load().favor_static_scratch_bytes()


def fwd_bidir_static(Q, K, V, omega, qk_scale, O=None, dev_status=None, stream=None):
    """Bidirectional FAVOR+ with the library's fixed device scratch (no
    workspace argument, nothing allocated by the library)."""
    O = torch.empty_like(Q) if O is None else O
    B, H, L, d = Q.shape
    for t in (Q, K, V, O):
        if not t.is_cuda or not t.is_contiguous() or t.dtype != Q.dtype or tuple(t.shape) != (B, H, L, d):
            raise FavorError("fwd_bidir_static: Q/K/V/O must be contiguous CUDA tensors of one dtype and shape")
    code = load().favor_fwd_bidir_static(Q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(), B, H, L, d,
                                         omega.data_ptr(), omega.shape[0], _DT[Q.dtype], float(qk_scale),
                                         dev_status.data_ptr() if dev_status is not None else None,
                                         _stream_handle(stream))
    _check(code, "favor_fwd_bidir_static")
    return O


def new_decode_state(B: int, H: int, m: int, d: int, device="cuda") -> torch.Tensor:
    """Zero decode state (the empty prefix): fp32 [B, H, d + 1, m]."""
    return torch.zeros((B, H, d + 1, m), dtype=torch.float32, device=device)


def decode_step(q, k, v, omega, qk_scale, state, o=None, dev_status=None, stream=None):
    """One causal step per (b, h): q, k, v [B, H, d]; adds this token to
    ``state`` (in place) and returns o [B, H, d], the token's causal output."""
    B, H, d = q.shape
    m = omega.shape[0]
    o = torch.empty_like(q) if o is None else o
    for t in (q, k, v, o):
        if not t.is_cuda or not t.is_contiguous() or t.dtype != q.dtype or tuple(t.shape) != (B, H, d):
            raise FavorError("decode_step: q/k/v/o must be contiguous CUDA tensors of one dtype and shape [B,H,d]")
    if (state.dtype != torch.float32 or not state.is_contiguous() or tuple(state.shape) != (B, H, d + 1, m)):
        raise FavorError(f"decode_step: state must be contiguous fp32 [B, H, {d + 1}, {m}]")
    if omega.dtype != torch.float32 or tuple(omega.shape) != (m, d) or not omega.is_contiguous():
        raise FavorError(f"decode_step: omega must be contiguous fp32 [m, {d}]")
    code = load().favor_decode_step(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), B, H, d,
                                    omega.data_ptr(), m, _DT[q.dtype], float(qk_scale), state.data_ptr(),
                                    dev_status.data_ptr() if dev_status is not None else None,
                                    _stream_handle(stream))
    _check(code, "favor_decode_step")
    return o


def decode_prefill_workspace_bytes(B: int, H: int, L: int, d: int, m: int, dtype) -> int:
    n = load().favor_decode_prefill_workspace_bytes(B, H, L, d, m, _DT[dtype])
    if n == 0:
        raise FavorError("unsupported shape")
    return n


def decode_prefill(K, V, omega, qk_scale, state, workspace=None, dev_status=None, stream=None):
    """state = the decode state after the L tokens of K, V [B, H, L, d]
    (overwritten); returns state."""
    B, H, L, d = K.shape
    m = omega.shape[0]
    for t in (K, V):
        if not t.is_cuda or not t.is_contiguous() or t.dtype != K.dtype or tuple(t.shape) != (B, H, L, d):
            raise FavorError("decode_prefill: K/V must be contiguous CUDA tensors of one dtype and shape [B,H,L,d]")
    if (state.dtype != torch.float32 or not state.is_contiguous() or tuple(state.shape) != (B, H, d + 1, m)):
        raise FavorError(f"decode_prefill: state must be contiguous fp32 [B, H, {d + 1}, {m}]")
    if workspace is None:
        n = decode_prefill_workspace_bytes(B, H, L, d, m, K.dtype)
        workspace = torch.empty(n, dtype=torch.uint8, device=K.device)
    code = load().favor_decode_prefill(K.data_ptr(), V.data_ptr(), B, H, L, d, omega.data_ptr(), m, _DT[K.dtype],
                                       float(qk_scale), state.data_ptr(), workspace.data_ptr(),
                                       workspace.numel() * workspace.element_size(),
                                       dev_status.data_ptr() if dev_status is not None else None,
                                       _stream_handle(stream))
    _check(code, "favor_decode_prefill")
    return state


def selftest_wait_timeout(stream=None, device="cuda"):
    """favor_selftest_wait_timeout: two device waits that run out (no fault).
    Returns (status, returned, times_ns) after synchronising: the device
    status (FAVOR_ERR_TIMEOUT expected), int32[2] with 2 for each wait that
    gave up, and int64[3] globaltimer stamps (start, warp 0 return, warp 1
    return)."""
    status = torch.zeros(1, dtype=torch.int32, device=device)
    returned = torch.zeros(2, dtype=torch.int32, device=device)
    times = torch.zeros(3, dtype=torch.int64, device=device)
    _check(load().favor_selftest_wait_timeout(status.data_ptr(), returned.data_ptr(), times.data_ptr(),
                                              _stream_handle(stream)), "favor_selftest_wait_timeout")
    torch.cuda.synchronize(device)
    return int(status.item()), returned.cpu().tolist(), times.cpu().tolist()


def bwd_workspace_bytes(B: int, H: int, L: int, d: int, m: int, dtype) -> int:
    n = load().favor_bwd_workspace_bytes(B, H, L, d, m, _DT[dtype])
    if n == 0:
        raise FavorError("unsupported shape")
    return n


def bwd_bidir(Q, K, V, dO, omega, qk_scale, workspace=None, feature_map="prf", dQ=None, dK=None, dV=None,
              dev_status=None, stream=None, causal=False):
    """Gradients (dQ, dK, dV) of the bidirectional (or, with causal=True, the
    causal) pass for the output gradient dO (all [B, H, L, d], one dtype)."""
    B, H, L, d = Q.shape
    m = omega.shape[0]
    dQ = torch.empty_like(Q) if dQ is None else dQ
    dK = torch.empty_like(K) if dK is None else dK
    dV = torch.empty_like(V) if dV is None else dV
    for t in (Q, K, V, dO, dQ, dK, dV):
        if not t.is_cuda or not t.is_contiguous() or t.dtype != Q.dtype or tuple(t.shape) != (B, H, L, d):
            raise FavorError("bwd_bidir: tensors must be contiguous CUDA tensors of one dtype and shape [B,H,L,d]")
    if omega.dtype != torch.float32 or tuple(omega.shape) != (m, d) or not omega.is_contiguous():
        raise FavorError(f"bwd_bidir: omega must be contiguous fp32 [m, {d}]")
    if feature_map not in FEATURE_MAPS:
        raise FavorError(f"bwd_bidir: feature_map must be one of {sorted(FEATURE_MAPS)}")
    if workspace is None:
        workspace = torch.empty(bwd_workspace_bytes(B, H, L, d, m, Q.dtype), dtype=torch.uint8, device=Q.device)
    name = "favor_bwd_causal" if causal else "favor_bwd_bidir"
    code = getattr(load(), name)(Q.data_ptr(), K.data_ptr(), V.data_ptr(), dO.data_ptr(), dQ.data_ptr(),
                                  dK.data_ptr(), dV.data_ptr(), B, H, L, d, omega.data_ptr(), m, _DT[Q.dtype],
                                  float(qk_scale), FEATURE_MAPS[feature_map], workspace.data_ptr(),
                                  workspace.numel() * workspace.element_size(),
                                  dev_status.data_ptr() if dev_status is not None else None, _stream_handle(stream))
    _check(code, name)
    return dQ, dK, dV


def bwd_causal(Q, K, V, dO, omega, qk_scale, workspace=None, feature_map="prf", dQ=None, dK=None, dV=None,
               dev_status=None, stream=None):
    """Gradients (dQ, dK, dV) of the causal pass."""
    return bwd_bidir(Q, K, V, dO, omega, qk_scale, workspace, feature_map, dQ, dK, dV, dev_status, stream,
                     causal=True)
