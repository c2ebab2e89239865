"""Seeded synthetic inputs for decomposed relative-position attention.

This module only draws random tensors; it holds none of the method's
arithmetic, so both the CUDA path and the CPU oracle can be fed from it.

Workloads follow the DeepEncoder global-attention setting described on the
vLLM PR #55629 page (section "功能与动机", motivation: 64x64 global attention,
BF16) plus a small grid, a batched encoder, a ragged 40x40 grid, a wider
16-head encoder, the same encoder's windowed blocks (section 实现拆解 item 3
keeps them on SDPA): the 64x64 grid padded to 70x70 and cut into 25 windows
of 14x14, each window an independent attention problem, and the 64x64
encoder with head_dim 128 (section 风险与影响 names BLOCK_D = 64 as the
kernel's limit).  Each tensor is drawn as fp32 ``sigma * randn`` from one CPU
generator in the fixed order q, k, v, rel_pos_h, rel_pos_w and then
rounded-to-nearest to the workload dtype; the same rounded values go to the
GPU and to the oracle.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import torch

HEAD_DIM = 64


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    heads: int
    H: int
    W: int
    d: int = HEAD_DIM
    dtype: str = "bf16"          # "bf16" or "f16"
    sigma_q: float = 1.0
    sigma_k: float = 1.0
    sigma_v: float = 1.0
    sigma_table: float = 0.5
    scale: float = HEAD_DIM ** -0.5
    entry: str = "attention"     # which entry point the workload is quoted on
    windows: int = 1             # attention problems per image and head (windowed blocks)

    @property
    def BH(self) -> int:
        return self.B * self.windows * self.heads

    @property
    def N(self) -> int:
        return self.H * self.W

    @property
    def torch_dtype(self) -> torch.dtype:
        return {"bf16": torch.bfloat16, "f16": torch.float16}[self.dtype]

    def with_grid(self, H: int, W: int, B: int | None = None, heads: int | None = None) -> "Workload":
        return replace(self, H=H, W=W, B=self.B if B is None else B, heads=self.heads if heads is None else heads,
                       name=f"{self.name}-{H}x{W}")


# The workloads.  scale = head_dim**-0.5 (the SDPA default): 1/8 for head_dim
# 64; sigma is a standard deviation.
WORKLOADS: dict[str, Workload] = {
    "grid16": Workload("grid16", B=1, heads=2, H=16, W=16),
    "global64": Workload("global64", B=1, heads=12, H=64, W=64),
    "batched64": Workload("batched64", B=8, heads=12, H=64, W=64),
    "ragged40": Workload("ragged40", B=16, heads=12, H=40, W=40, dtype="f16", sigma_q=2.0, sigma_k=2.0,
                         sigma_v=1.0, sigma_table=1.0),
    "wide64": Workload("wide64", B=4, heads=16, H=64, W=64, entry="fused"),
    "window14": Workload("window14", B=1, heads=12, H=14, W=14, windows=25, entry="fused"),
    # the same 64x64 encoder with head_dim 128 (the pages' kernel fixes BLOCK_D = 64)
    "global64d128": Workload("global64d128", B=1, heads=12, H=64, W=64, d=128, scale=128 ** -0.5, entry="fused"),
}


def make_inputs(w: Workload, seed: int = 0) -> dict[str, torch.Tensor]:
    """Draw q, k, v ``[B*heads, H*W, d]`` and the tables ``[2H-1, d]``, ``[2W-1, d]`` on the CPU."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    shape = (w.BH, w.N, w.d)
    out = {}
    for name, sig, shp in (("q", w.sigma_q, shape), ("k", w.sigma_k, shape), ("v", w.sigma_v, shape),
                           ("rel_pos_h", w.sigma_table, (2 * w.H - 1, w.d)),
                           ("rel_pos_w", w.sigma_table, (2 * w.W - 1, w.d))):
        out[name] = (torch.randn(shp, generator=g, dtype=torch.float32) * sig).to(w.torch_dtype)
    return out


def to_f64(t: torch.Tensor):
    """Exact widening of a (rounded) tensor to a float64 NumPy array."""
    return t.detach().to("cpu", torch.float64).numpy()
