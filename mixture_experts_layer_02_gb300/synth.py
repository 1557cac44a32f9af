"""Seeded synthetic workloads for the MoE layer.

This module only draws random inputs and describes workload shapes; it holds
none of the layer's arithmetic.  Both the GPU path's callers and the oracle's
callers take their inputs from here, so both sides see the same bytes.

Workloads (shapes of the models the pages discuss, random-init weights):
  tiny        N=64,    D=128,  E=8,   K=2, D_ffn=256,   SiLU,   softmax over top-K
  mixtral     N=4096,  D=4096, E=8,   K=2, D_ffn=14336, SwiGLU, softmax over top-K
  dsv3        N=4096,  D=7168, E=256, K=8, D_ffn=2048,  SwiGLU, sigmoid + renormalise
  qwen3_N     N in {1,8,32,128,256}, D=2048, E=128, K=8, D_ffn=768, SwiGLU, softmax
  dsv3_zipf   N=16384, D=7168, E=256, K=8, D_ffn=2048,  SwiGLU, sigmoid + renormalise,
              router logits shifted per expert by ln p_e with p ~ Zipf(s=1.2)

Recipe: x ~ N(0,1); W_gate, W1, W3 ~ N(0, 1/D); W2 ~ N(0, 1/D_ffn); each drawn
in fp32 from torch's seeded generator on the target device, scaled in fp32,
then rounded to bf16 (round-to-nearest-even).  Every tensor has its own
generator seeded from (seed, tensor id), so a tensor does not depend on the
sizes of the others.  Tensor ids: x=0, W_gate=1, W1=2, W3=3, W2=4.
"""
from __future__ import annotations

import dataclasses
import math

import torch

SOFTMAX_TOPK = 0
SIGMOID_NORM = 1
ACT_SILU = 0
ACT_SWIGLU = 1


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    N: int
    D: int
    E: int
    K: int
    Dff: int
    act: int = ACT_SWIGLU
    mode: int = SOFTMAX_TOPK
    zipf_s: float = 0.0          # 0 = no router bias

    @property
    def rows(self) -> int:
        return self.N * self.K

    def with_tokens(self, N: int) -> "Workload":
        return dataclasses.replace(self, N=N, name=f"{self.name.split('@')[0]}@N{N}")

    def describe(self) -> dict:
        return dict(workload=self.name, N=self.N, D=self.D, E=self.E, K=self.K,
                    D_ffn=self.Dff, act="swiglu" if self.act == ACT_SWIGLU else "silu",
                    score="softmax_topk" if self.mode == SOFTMAX_TOPK else "sigmoid_norm",
                    router_bias=(f"zipf(s={self.zipf_s})" if self.zipf_s else None))


WORKLOADS = {
    "tiny": Workload("tiny", 64, 128, 8, 2, 256, ACT_SILU, SOFTMAX_TOPK),
    "mixtral": Workload("mixtral", 4096, 4096, 8, 2, 14336, ACT_SWIGLU, SOFTMAX_TOPK),
    "dsv3": Workload("dsv3", 4096, 7168, 256, 8, 2048, ACT_SWIGLU, SIGMOID_NORM),
    "dsv3_zipf": Workload("dsv3_zipf", 16384, 7168, 256, 8, 2048, ACT_SWIGLU, SIGMOID_NORM, 1.2),
}
# a smaller case of the mixtral kernels for profiler captures (1.4 GB of weights)
WORKLOADS["mixtral_small"] = Workload("mixtral_small", 2048, 4096, 4, 2, 14336, ACT_SWIGLU, SOFTMAX_TOPK)
# a smaller case of the DeepSeek-V3 kernels (64 experts, 5.6 GB of weights)
WORKLOADS["dsv3_small"] = Workload("dsv3_small", 1024, 7168, 64, 8, 2048, ACT_SWIGLU, SIGMOID_NORM)
# a smaller case of the skewed DeepSeek-V3 layer (64 experts with Zipf(1.2)
# routing bias: a few hot experts and a cold tail, 5.6 GB of weights)
WORKLOADS["dsv3_zipf_small"] = Workload("dsv3_zipf_small", 4096, 7168, 64, 8, 2048, ACT_SWIGLU, SIGMOID_NORM, 1.2)
for _n in (1, 8, 32, 128, 256):
    WORKLOADS[f"qwen3_N{_n}"] = Workload(f"qwen3_N{_n}", _n, 2048, 128, 8, 768,
                                         ACT_SWIGLU, SOFTMAX_TOPK)


def zipf_log_popularity(E: int, s: float) -> torch.Tensor:
    """ln p_i for p_i proportional to i^-s, i = 1..E, normalised to sum 1
    (fp64 on the CPU).  Expert e gets ln p_{e+1}, so expert 0 is the hottest."""
    i = torch.arange(1, E + 1, dtype=torch.float64)
    logp = -s * torch.log(i)
    return logp - torch.logsumexp(logp, 0)


def _gen(device, seed: int, tensor_id: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1_000_003 + tensor_id * 7919 + 12345) & 0x7FFF_FFFF_FFFF_FFFF)
    return g


def _normal_bf16(shape, scale: float, gen: torch.Generator, device) -> torch.Tensor:
    t = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if scale != 1.0:
        t.mul_(scale)
    return t.to(torch.bfloat16)


def _expert_stack(E, rows, cols, scale, gen, device) -> torch.Tensor:
    """[E, rows, cols] bf16, drawn one expert at a time (bounded fp32 temp)."""
    out = torch.empty((E, rows, cols), dtype=torch.bfloat16, device=device)
    for e in range(E):
        out[e] = _normal_bf16((rows, cols), scale, gen, device)
    return out


def make_inputs(wl: Workload, seed: int = 0, device="cpu") -> dict:
    """All inputs of one layer call: x, w_gate, bias (fp32 or None), w1, w3
    (None for SiLU), w2 -- bf16 tensors on ``device``."""
    dev = torch.device(device)
    x = _normal_bf16((wl.N, wl.D), 1.0, _gen(dev, seed, 0), dev)
    wg = _normal_bf16((wl.E, wl.D), 1.0 / math.sqrt(wl.D), _gen(dev, seed, 1), dev)
    w1 = _expert_stack(wl.E, wl.Dff, wl.D, 1.0 / math.sqrt(wl.D), _gen(dev, seed, 2), dev)
    w3 = (_expert_stack(wl.E, wl.Dff, wl.D, 1.0 / math.sqrt(wl.D), _gen(dev, seed, 3), dev)
          if wl.act == ACT_SWIGLU else None)
    w2 = _expert_stack(wl.E, wl.D, wl.Dff, 1.0 / math.sqrt(wl.Dff), _gen(dev, seed, 4), dev)
    bias = None
    if wl.zipf_s:
        bias = zipf_log_popularity(wl.E, wl.zipf_s).to(torch.float32).to(dev)
    return dict(x=x, w_gate=wg, bias=bias, w1=w1, w3=w3, w2=w2)


def make_tokens(wl: Workload, seed: int = 0, device="cpu", step: int = 0) -> torch.Tensor:
    """A fresh x [N,D] bf16 batch for step ``step`` (tensor id 100 + step)."""
    dev = torch.device(device)
    return _normal_bf16((wl.N, wl.D), 1.0, _gen(dev, seed, 100 + step), dev)


def bf16_bits(t: torch.Tensor):
    """Raw bf16 bits of a tensor as a numpy uint16 array (CPU copy)."""
    import numpy as np
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
