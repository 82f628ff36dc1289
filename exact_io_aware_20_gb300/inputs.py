"""Seeded synthetic inputs for the attention workloads.

This module holds no attention arithmetic: it only draws random tensors.  It
is the one module that both the GPU path's tests/benchmark and the CPU oracle
checks take their inputs from, so that both sides read the same bytes.

Recipe: a CPU ``torch.Generator`` seeded with ``seed``, ``torch.randn`` in
fp32, tensors drawn in the order Q, K, V, dO, multiplied by ``value_scale``
and then cast to the workload's 16-bit dtype.  Layout is [B, H, N, d] for Q and
dO and [B, Hkv, N, d] for K and V, d contiguous.
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    Hkv: int
    N: int
    d: int
    dtype: str          # "f16" or "bf16"
    causal: bool
    seed: int
    value_scale: float = 1.0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float16 if self.dtype == "f16" else torch.bfloat16

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    def flops_fwd(self) -> float:
        """4*B*H*N^2*d, halved under the causal mask (H counts query heads)."""
        f = 4.0 * self.B * self.H * self.N * self.N * self.d
        return f / 2 if self.causal else f

    def flops_bwd(self) -> float:
        return 2.5 * self.flops_fwd()


# The five workloads of the measurement plan.  Seeds are 1000 + index.
WORKLOADS = {
    "tiny": Workload("tiny", 1, 1, 1, 128, 64, "f16", False, 1001),
    "gpt_layer": Workload("gpt_layer", 8, 16, 16, 2048, 128, "bf16", False, 1002),
    "gpt_layer_causal": Workload("gpt_layer_causal", 8, 16, 16, 2048, 128, "bf16", True, 1002),
    "long_seq": Workload("long_seq", 1, 16, 16, 16384, 128, "bf16", True, 1003),
    "head256": Workload("head256", 4, 8, 8, 4096, 256, "f16", False, 1004, 0.5),
    "gqa8k": Workload("gqa8k", 2, 32, 8, 8192, 128, "bf16", True, 1005),
}


def make_inputs(w: Workload, device: str | torch.device = "cpu", Nk: int | None = None):
    """Q, K, V, dO for workload ``w`` (Nk overrides the key length if given)."""
    nk = w.N if Nk is None else Nk
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed)
    shapes = [(w.B, w.H, w.N, w.d), (w.B, w.Hkv, nk, w.d), (w.B, w.Hkv, nk, w.d),
              (w.B, w.H, w.N, w.d)]
    out = []
    for shp in shapes:
        t = torch.randn(shp, generator=g, dtype=torch.float32)
        if w.value_scale != 1.0:
            t = t * w.value_scale
        out.append(t.to(w.torch_dtype).to(device))
    return tuple(out)


def make_block_mask(heads: int, Nq: int, Nk: int, density: float, seed: int,
                    device: str | torch.device = "cpu") -> torch.Tensor:
    """Seeded random block mask for block-sparse attention: uint8
    [heads, ceil(Nq/128), ceil(Nk/128)], each 128 x 128 block kept (1) with
    probability ``density``."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    shape = (heads, -(-Nq // 128), -(-Nk // 128))
    return (torch.rand(shape, generator=g) < density).to(torch.uint8).to(device)
