"""C-ABI checks that need no GPU: the library loads, exports every entry point
declared in include/*.h, and rejects bad arguments before launching."""

import ctypes
import os
import re

import pytest
import torch

import linear_softmax_attention_gb300 as favor

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = set()
    inc = os.path.join(ROOT, "include")
    for h in sorted(os.listdir(inc)):
        if h.endswith(".h"):
            text = re.sub(r"/\*.*?\*/", "", open(os.path.join(inc, h)).read(), flags=re.S)
            names.update(re.findall(r"\b(favor_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(favor.lib_path()):
        from linear_softmax_attention_gb300 import build
        build.build()
    return favor.load()


def test_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert len(names) >= 11
    assert "favor_selftest_wait_timeout" in names
    for n in names:
        assert hasattr(lib, n), n


def test_version_and_status_strings(lib):
    assert favor.api_version() == 1
    for code, text in [(0, "ok"), (1, "invalid argument"), (2, "unsupported shape"), (4, "device wait timed out")]:
        assert favor.status_string(code) == text


def test_workspace_sizes(lib):
    assert favor.workspace_bytes(False, 1, 1, 512, 64, 64, torch.float32) > 0
    assert favor.workspace_bytes(True, 4, 8, 8192, 64, 256, torch.bfloat16) > 0
    assert lib.favor_workspace_bytes(0, 1, 1, 0, 64, 64, 0) == 0          # L = 0
    assert lib.favor_workspace_bytes(0, 1, 1, 16, 129, 64, 0) == 0        # d too large
    assert lib.favor_workspace_bytes(0, 1, 1, 16, 64, 513, 0) == 0        # m too large
    assert lib.favor_workspace_bytes(0, 1, 1, 16, 64, 64, 7) == 0         # bad dtype


def test_path_names(lib):
    assert favor.path_name(False, 64, 64, torch.float32) == "simt"
    assert favor.path_name(False, 200, 64, torch.float32) == "unsupported"


def _call(lib, name, **kw):
    args = dict(Q=16, K=16, V=16, O=32, B=1, H=1, L=8, d=8, omega=48, m=8, dt=0, s=1.0, ws=256, nbytes=1 << 30,
                st=None, stream=None)
    args.update(kw)
    return getattr(lib, name)(args["Q"], args["K"], args["V"], args["O"], args["B"], args["H"], args["L"],
                              args["d"], args["omega"], args["m"], args["dt"], args["s"], args["ws"],
                              args["nbytes"], args["st"], args["stream"])


@pytest.mark.parametrize("name", favor.ENTRY_POINTS)
def test_bad_arguments_rejected_before_launch(lib, name):
    # every case fails the host-side checks, so nothing reaches the GPU
    assert _call(lib, name, omega=None) == 1
    assert _call(lib, name, ws=None) == 1
    assert _call(lib, name, L=0) == 1
    assert _call(lib, name, d=129) == 2
    assert _call(lib, name, m=600) == 2
    assert _call(lib, name, dt=3) == 1
    assert _call(lib, name, s=float("nan")) == 1
    assert _call(lib, name, s=0.0) == 1
    assert _call(lib, name, s=-0.5) == 1
    assert _call(lib, name, ws=8) == 1                 # workspace not 256-byte aligned
    assert _call(lib, name, nbytes=16) == 1            # workspace too small
    if "state" not in name:
        assert _call(lib, name, Q=None) == 1
        assert _call(lib, name, O=16) == 1             # O aliases Q
        assert _call(lib, name, Q=24) == 1             # misaligned
    if "bidir_output" not in name:
        assert _call(lib, name, K=None) == 1


def test_build_orf_rejects_bad_arguments(lib):
    assert lib.favor_build_orf(ctypes.c_uint64(0), 8, 8, 1, None, None) == 1
    assert lib.favor_build_orf(ctypes.c_uint64(0), 0, 8, 1, 16, None) == 1
    assert lib.favor_build_orf(ctypes.c_uint64(0), 8, 200, 1, 16, None) == 1
    assert lib.favor_build_orf(ctypes.c_uint64(0), 8, 8, 4, 16, None) == 1      # unknown kind
    assert lib.favor_build_orf(ctypes.c_uint64(0), 8, 8, -1, 16, None) == 1     # unknown kind
    assert lib.favor_build_orf(ctypes.c_uint64(0), 8, 1, 3, 16, None) == 2      # Givens needs d >= 2
    assert lib.favor_build_orf(ctypes.c_uint64(0), 8, 12, 2, 16, None) == 2     # Hadamard needs a power of two


def test_product_code_does_not_touch_the_oracle():
    pkg = os.path.join(ROOT, "linear_softmax_attention_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in text.lower(), f


def test_decode_rejects_bad_arguments_before_launch(lib):
    # favor_decode_step(q, k, v, o, B, H, d, omega, m, dt, s, state, status, stream)
    def step(**kw):
        # fake, never dereferenced addresses: q, k, v, o 32 bytes each, the state (d + 1) m 4 = 288
        a = dict(q=0x1000, k=0x2000, v=0x3000, o=0x4000, B=1, H=1, d=8, omega=0x5000, m=8, dt=0, s=1.0,
                 state=0x10000, st=None, stream=None)
        a.update(kw)
        return lib.favor_decode_step(a["q"], a["k"], a["v"], a["o"], a["B"], a["H"], a["d"], a["omega"], a["m"],
                                     a["dt"], a["s"], a["state"], a["st"], a["stream"])
    assert step(q=None) == 1
    assert step(state=None) == 1
    assert step(omega=None) == 1
    assert step(o=0x1000) == 1        # o aliases q
    assert step(o=0x10000) == 1       # o aliases the state
    assert step(o=0x1010) == 1        # o overlaps the end of q
    assert step(q=0x10000) == 1       # q aliases the state
    assert step(k=0x10010) == 1       # k inside the state
    assert step(v=0x10000 + 288 - 16) == 1    # v overlaps the end of the state
    assert step(q=0x1008) == 1        # misaligned
    assert step(d=129) == 2
    assert step(m=513) == 2
    assert step(B=0) == 1
    assert step(dt=5) == 1
    assert step(s=float("inf")) == 1

    def prefill(**kw):
        a = dict(K=16, V=16, B=1, H=1, L=8, d=8, omega=48, m=8, dt=0, s=1.0, state=64, ws=256, nbytes=1 << 30,
                 st=None, stream=None)
        a.update(kw)
        return lib.favor_decode_prefill(a["K"], a["V"], a["B"], a["H"], a["L"], a["d"], a["omega"], a["m"], a["dt"],
                                        a["s"], a["state"], a["ws"], a["nbytes"], a["st"], a["stream"])
    assert prefill(K=None) == 1
    assert prefill(state=None) == 1
    assert prefill(ws=None) == 1
    assert prefill(ws=8) == 1
    assert prefill(nbytes=16) == 1
    assert prefill(L=0) == 1
    assert prefill(m=600) == 2
    assert lib.favor_decode_prefill_workspace_bytes(2, 8, 300, 64, 256, 1) > 0
    assert lib.favor_decode_prefill_workspace_bytes(2, 8, 0, 64, 256, 1) == 0


@pytest.mark.parametrize("name", ["favor_fwd_bidir_fm", "favor_fwd_causal_fm"])
def test_feature_map_calls_reject_bad_arguments(lib, name):
    def call(fm=1, **kw):
        a = dict(Q=16, K=16, V=16, O=32, B=1, H=1, L=8, d=8, omega=48, m=8, dt=0, s=1.0, ws=256, nbytes=1 << 30,
                 st=None, stream=None)
        a.update(kw)
        return getattr(lib, name)(a["Q"], a["K"], a["V"], a["O"], a["B"], a["H"], a["L"], a["d"], a["omega"],
                                  a["m"], a["dt"], a["s"], fm, a["ws"], a["nbytes"], a["st"], a["stream"])
    assert call(fm=3) == 1             # not a favor_feature_map
    assert call(fm=-1) == 1
    assert call(omega=None) == 1
    assert call(L=0) == 1
    assert call(m=600) == 2
    assert call(nbytes=16) == 1


def test_feature_map_workspace_sizes(lib):
    for causal in (0, 1):
        # every feature map takes the plain call's path, hence its workspace
        for fm in (0, 1, 2):
            for dt in (0, 1):
                assert lib.favor_workspace_bytes_fm(causal, 2, 4, 1000, 64, 256, dt, fm) == \
                    lib.favor_workspace_bytes(causal, 2, 4, 1000, 64, 256, dt) > 0
        assert lib.favor_workspace_bytes_fm(causal, 2, 4, 1000, 64, 256, 1, 3) == 0
        assert lib.favor_workspace_bytes_fm(causal, 2, 4, 0, 64, 256, 1, 2) == 0


@pytest.mark.parametrize("name", ["favor_bwd_bidir", "favor_bwd_causal"])
def test_backward_rejects_bad_arguments_before_launch(lib, name):
    def call(**kw):
        a = dict(Q=16, K=32, V=48, dO=64, dQ=80, dK=96, dV=112, B=1, H=1, L=8, d=8, omega=128, m=8, dt=0, s=1.0,
                 fm=0, ws=256, nbytes=1 << 30, st=None, stream=None)
        a.update(kw)
        return getattr(lib, name)(a["Q"], a["K"], a["V"], a["dO"], a["dQ"], a["dK"], a["dV"], a["B"], a["H"],
                                  a["L"], a["d"], a["omega"], a["m"], a["dt"], a["s"], a["fm"], a["ws"],
                                  a["nbytes"], a["st"], a["stream"])
    assert call(dO=None) == 1
    assert call(dQ=None) == 1
    assert call(dQ=16) == 1            # dQ aliases Q
    assert call(dK=80) == 1            # dK aliases dQ
    assert call(fm=3) == 1
    assert call(ws=None) == 1
    assert call(nbytes=16) == 1
    assert call(s=0.0) == 1
    assert call(d=129) == 2
    assert lib.favor_bwd_workspace_bytes(2, 4, 1000, 64, 256, 1) > 0
    assert lib.favor_bwd_workspace_bytes(2, 4, 0, 64, 256, 1) == 0


def test_selftest_rejects_null_pointers(lib):
    assert lib.favor_selftest_wait_timeout(None, 16, 32, None) == 1
    assert lib.favor_selftest_wait_timeout(16, None, 32, None) == 1
    assert lib.favor_selftest_wait_timeout(16, 32, None, None) == 1
