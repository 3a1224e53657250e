"""Seeded synthetic workloads shared by the tests, the bench and the smoke check.

This module holds only shapes, seeds and random draws: none of the attention
arithmetic. Inputs are drawn in float32 from NumPy's PCG64 generator (its
stream is fixed across platforms and NumPy versions), scaled by sigma and
rounded to the working dtype (round-to-nearest-even) on the CPU, so every
consumer sees identical 16-bit values.

The five workloads follow the shapes the pages benchmark and describe:
a tiny MHA case; causal MHA with more keys than queries (bottom-right mask,
offset Sk - Sq = 256); and three D = 128 causal GQA prefill shapes with group
sizes 4, 2 and 8 ("NVIDIA闪存注意力实操" benchmark section: B=4, H=32, D=128,
causal; "MiniPaged-Qwen: Qwen3 Prefill FlashAttention" section 6: Hq=16,
Hkv=8, D=128).
"""

from __future__ import annotations

import dataclasses
import math

import numpy as np

__all__ = ["Workload", "WORKLOADS", "by_name", "draw_inputs", "draw_numpy", "draw_device"]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Sq: int
    Sk: int
    Hq: int
    Hkv: int
    D: int
    dtype: str          # "bf16" or "fp16"
    causal: bool
    sigma_qk: float     # std-dev of q and k entries
    sigma_v: float      # std-dev of v entries
    seed: int

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    def with_sizes(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = [
    Workload("tiny_mha_d64", 1, 128, 128, 2, 2, 64, "bf16", False, 1.0, 1.0, 1000),
    Workload("causal_mha_sq1280_sk1536", 1, 1280, 1536, 16, 16, 128, "fp16", True, 1.0, 1.0, 1001),
    Workload("causal_gqa4_b4_s4096", 4, 4096, 4096, 32, 8, 128, "bf16", True, 1.0, 1.0, 1002),
    Workload("causal_gqa2_b2_s8192_sigma2", 2, 8192, 8192, 16, 8, 128, "bf16", True, 2.0, 1.0, 1003),
    Workload("causal_gqa8_b1_s16384", 1, 16384, 16384, 32, 4, 128, "bf16", True, 1.0, 1.0, 1004),
]


def by_name(name: str) -> Workload:
    for w in WORKLOADS:
        if w.name == name:
            return w
    raise KeyError(name)


def draw_numpy(w: Workload):
    """float32 arrays q (B,Sq,Hq,D), k, v (B,Sk,Hkv,D), before dtype rounding.

    Draw order is q, then k, then v from one PCG64 stream seeded with
    ``w.seed``.
    """
    rng = np.random.Generator(np.random.PCG64(w.seed))
    q = rng.standard_normal((w.B, w.Sq, w.Hq, w.D), dtype=np.float32) * np.float32(w.sigma_qk)
    k = rng.standard_normal((w.B, w.Sk, w.Hkv, w.D), dtype=np.float32) * np.float32(w.sigma_qk)
    v = rng.standard_normal((w.B, w.Sk, w.Hkv, w.D), dtype=np.float32) * np.float32(w.sigma_v)
    return q, k, v


def draw_inputs(w: Workload):
    """CPU torch tensors q, k, v in the workload's dtype (RNE from float32)."""
    import torch

    dt = {"bf16": torch.bfloat16, "fp16": torch.float16}[w.dtype]
    return tuple(torch.from_numpy(a).to(dt) for a in draw_numpy(w))


def draw_device(shape, dtype: str, sigma: float, seed: int, device="cuda"):
    """A tensor too large to draw on the host (several GB): N(0, sigma^2)
    entries drawn directly in ``dtype`` ("bf16", "fp16" or "fp32") on ``device`` by torch's
    counter-based (Philox) generator seeded with ``seed``. A consumer that
    checks it on the host copies back the slices it reads."""
    import torch

    dt = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}[dtype]
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    t = torch.randn(shape, dtype=dt, device=device, generator=g)
    if sigma != 1.0:
        t.mul_(sigma)
    return t
