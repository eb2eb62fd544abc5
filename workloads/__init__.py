"""Seeded synthetic inputs for the FAVOR+ forward pass.

This module only draws numbers and lays them out: it holds none of the
method's arithmetic, so both the CUDA library's tests/benchmark and the CPU
oracle can take their inputs from it.

Workloads (stand-ins for the pages' data: the Regular Transformer shape with
8 heads of d = 64, TrEMBL protein sequences of length 8192 over a 36-token
alphabet, ImageNet64 as a 12288-token pixel sequence, and a long-sequence
sweep; those datasets are not used):

  bidir-f32-B1H1L512-d64-m64       Q, K, V ~ N(0, 1), fp32
  bidir-bf16-B8H8L4096-d64-m256    Q, K, V ~ N(0, 1), bf16
  causal-bf16-B4H8L8192-d64-m256   tokens ~ U{0..35}; Q, K, V rows are the
                                   rows of independent N(0, 1) embedding
                                   tables [36, H*d] picked by the tokens
  causal-bf16-B2H8L12288-d64-m256  same with 256 pixel values; Omega is
                                   redrawn for every call (seed base + i)
  sweep-bf16-B1H16-d128            Q, K, V ~ N(0, 1), Q and K LayerNorm-ed
                                   over d (no affine, eps 1e-5) in fp32;
                                   m in {128, 256, 512}, L in {16K, 32K, 64K},
                                   bidirectional and causal

All draws use ``torch.Generator`` seeded with ``seed`` on the requested
device, in fp32, then cast to the storage dtype.  The temperature d**-0.25 is
not applied here: it is passed to the attention call as ``qk_scale``.
"""

from __future__ import annotations

from dataclasses import dataclass, replace

import torch

__all__ = ["Workload", "WORKLOADS", "SWEEP", "get", "make_qkv", "omega_seed_for_call"]


@dataclass(frozen=True)
class Workload:
    name: str
    mode: str            # "bidir" or "causal"
    dtype: str           # "f32" or "bf16"
    B: int
    H: int
    L: int
    d: int
    m: int
    inputs: str          # "normal", "tokens", "normal_ln"
    vocab: int = 0
    redraw_omega: bool = False
    seed: int = 0
    omega_seed: int = 0

    @property
    def qk_scale(self) -> float:
        return float(self.d) ** -0.25

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    w.name: w
    for w in [
        Workload("bidir-f32-B1H1L512-d64-m64", "bidir", "f32", 1, 1, 512, 64, 64, "normal"),
        Workload("bidir-bf16-B8H8L4096-d64-m256", "bidir", "bf16", 8, 8, 4096, 64, 256, "normal"),
        Workload("causal-bf16-B4H8L8192-d64-m256", "causal", "bf16", 4, 8, 8192, 64, 256, "tokens", vocab=36),
        Workload("causal-bf16-B2H8L12288-d64-m256", "causal", "bf16", 2, 8, 12288, 64, 256, "tokens",
                 vocab=256, redraw_omega=True),
    ]
}

SWEEP = {}
for _mode in ("bidir", "causal"):
    for _m in (128, 256, 512):
        for _L in (16384, 32768, 65536):
            _w = Workload(f"sweep-{_mode}-bf16-B1H16L{_L}-d128-m{_m}", _mode, "bf16", 1, 16, _L, 128, _m,
                          "normal_ln")
            SWEEP[_w.name] = _w


def get(name: str) -> Workload:
    if name in WORKLOADS:
        return WORKLOADS[name]
    return SWEEP[name]


def omega_seed_for_call(w: Workload, call_index: int) -> int:
    """Seed of Omega for call ``call_index`` (redrawn workloads add the index)."""
    return w.omega_seed + call_index if w.redraw_omega else w.omega_seed


def _layer_norm_lastdim(x: torch.Tensor, eps: float = 1e-5) -> torch.Tensor:
    mu = x.mean(dim=-1, keepdim=True)
    var = ((x - mu) ** 2).mean(dim=-1, keepdim=True)
    return (x - mu) / torch.sqrt(var + eps)


def make_qkv(w: Workload, seed: int | None = None, device="cpu", B: int | None = None,
             L: int | None = None, H: int | None = None):
    """Q, K, V of workload ``w`` as contiguous [B, H, L, d] tensors.

    ``B``, ``H`` and ``L`` override the workload's sizes (same recipe, smaller
    case).  Returns tensors in the workload's storage dtype on ``device``.
    """
    seed = w.seed if seed is None else seed
    B = w.B if B is None else B
    H = w.H if H is None else H
    L = w.L if L is None else L
    d = w.d
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    if w.inputs in ("normal", "normal_ln"):
        out = [torch.randn((B, H, L, d), generator=gen, device=device, dtype=torch.float32) for _ in range(3)]
        if w.inputs == "normal_ln":
            out[0] = _layer_norm_lastdim(out[0])
            out[1] = _layer_norm_lastdim(out[1])
    elif w.inputs == "tokens":
        tok = torch.randint(0, w.vocab, (B, L), generator=gen, device=device)
        out = []
        for _ in range(3):
            table = torch.randn((w.vocab, H * d), generator=gen, device=device, dtype=torch.float32)
            x = table[tok]                                   # [B, L, H*d]
            out.append(x.view(B, L, H, d).permute(0, 2, 1, 3).contiguous())
    else:
        raise ValueError(f"unknown input recipe {w.inputs!r}")
    return tuple(t.to(w.torch_dtype).contiguous() for t in out)
