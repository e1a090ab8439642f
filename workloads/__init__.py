"""Seeded synthetic inputs for the routed top-k MoE experts forward.

This module only draws random numbers and rounds them to the storage dtypes.
It holds none of the method's arithmetic (no routing, no softmax, no matmul,
no quantisation), so both the CPU oracle and the CUDA path can take their
inputs from it without sharing any computation.

Workload shapes (the layer sizes of the benchmark cases):

* ``tiny``   - T=64,  H=128,  I=256,  E=8,   k=2
* ``qwen``   - Qwen1.5-MoE-A2.7B-shaped layer: H=2048, I=1408, E=60, k=4,
               T=4096 for prefill, T in {1, 8, 32, 128} for decode
* ``dsv3``   - DeepSeek-V3-shaped layer: H=7168, I=2048, E=256, k=8, T=8192,
               router logits skewed by a Zipf(s=1.1) expert bias
* ``dsv3_fp8`` - the DeepSeek-V3 shape with block-scaled e4m3 weights,
               T in {64, 16384}
* ``dsv3_e32`` - the DeepSeek-V3 width with 32 experts, uniform routing
               (profiling-sized)

Value recipe: hidden ~ N(0,1) rounded to bf16, expert weights ~ N(0, 0.02^2)
rounded to bf16, router logits ~ N(0,1) in fp32.  For the skewed workloads a
per-expert bias ``-s * ln(1 + pi(e))`` is added to every token's logits, where
``pi`` is a seeded permutation of the experts, so expert popularity follows a
Zipf(s) law that is not tied to the expert index.

Draw order from one ``torch.Generator`` seeded with ``seed`` on ``device``:
pi (skewed workloads only), logits, hidden, W_gate_up (expert by expert),
W_down (expert by expert).  The same (seed, device, shape) always gives the
same bytes; CPU and CUDA generators give different streams, so a test that
compares the two paths draws once and copies.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

__all__ = ["MoEShape", "SHAPES", "make_inputs", "shape_for"]


@dataclasses.dataclass(frozen=True)
class MoEShape:
    T: int
    H: int
    I: int
    E: int
    k: int
    zipf_s: Optional[float] = None

    def with_tokens(self, T: int) -> "MoEShape":
        return dataclasses.replace(self, T=T)


SHAPES = {
    "tiny": MoEShape(T=64, H=128, I=256, E=8, k=2),
    "qwen": MoEShape(T=4096, H=2048, I=1408, E=60, k=4),
    "dsv3": MoEShape(T=8192, H=7168, I=2048, E=256, k=8, zipf_s=1.1),
    "dsv3_fp8": MoEShape(T=16384, H=7168, I=2048, E=256, k=8, zipf_s=1.1),
    # DeepSeek-V3 width with 32 experts and uniform routing: a layer small
    # enough (1.4 GB of e4m3 weights) for detailed profiler captures
    "dsv3_e32": MoEShape(T=2048, H=7168, I=2048, E=32, k=8),
}


def shape_for(name: str, T: Optional[int] = None) -> MoEShape:
    s = SHAPES[name]
    return s if T is None else s.with_tokens(T)


def make_inputs(shape: MoEShape, seed: int = 0, device="cpu",
                weight_std: float = 0.02, logits_only: bool = False) -> dict:
    """Draw one workload.

    Returns a dict with ``logits`` (fp32 [T,E]), ``hidden`` (bf16 [T,H]),
    ``w_gate_up`` (bf16 [E,2I,H]; rows 0..I-1 gate, I..2I-1 up) and
    ``w_down`` (bf16 [E,H,I]), all on ``device``.
    """
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    T, H, I, E = shape.T, shape.H, shape.I, shape.E
    out = {}
    bias = None
    if shape.zipf_s is not None:
        perm = torch.randperm(E, generator=g, device=dev)
        ranks = (perm + 1).to(torch.float64)
        bias = (-shape.zipf_s * torch.log(ranks)).to(torch.float32)
    logits = torch.randn(T, E, generator=g, device=dev, dtype=torch.float32)
    if bias is not None:
        logits = logits + bias[None, :]
    out["logits"] = logits.contiguous()
    if logits_only:
        return out
    out["hidden"] = torch.randn(T, H, generator=g, device=dev,
                                dtype=torch.float32).to(torch.bfloat16)
    wgu = torch.empty(E, 2 * I, H, dtype=torch.bfloat16, device=dev)
    for e in range(E):
        wgu[e] = (torch.randn(2 * I, H, generator=g, device=dev,
                              dtype=torch.float32) * weight_std).to(torch.bfloat16)
    wd = torch.empty(E, H, I, dtype=torch.bfloat16, device=dev)
    for e in range(E):
        wd[e] = (torch.randn(H, I, generator=g, device=dev,
                             dtype=torch.float32) * weight_std).to(torch.bfloat16)
    out["w_gate_up"] = wgu
    out["w_down"] = wd
    return out


def zipf_bias_expected_share(E: int, s: float) -> list:
    """Zipf(s) share of each popularity rank (1-based) among E experts; used
    only to describe the skew of the synthetic logits in reports."""
    z = [1.0 / math.pow(r, s) for r in range(1, E + 1)]
    tot = sum(z)
    return [v / tot for v in z]
