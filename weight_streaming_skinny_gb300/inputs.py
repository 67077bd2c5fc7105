"""Seeded synthetic inputs for the decode linear layer.

This module only draws random numbers and lays them out in the storage formats
the library consumes.  It performs none of the layer's arithmetic (no products,
no sums, no dequantisation), so the CPU oracle and the CUDA path can both take
their inputs from here without sharing any of the method.

Distributions follow the decode workloads described in "Developing a custom
Qwen2.5 72B inference engine from scratch" (§1: Qwen2.5-72B, hidden size 8192,
80 decoder layers, ~152k vocabulary; §6.1: bf16 and weight-only FP8 decode
GEMV) and "9% faster GLM-5.3-Flash prefill with GPU-to-GPU IPC" (section
"TileLang: twice as fast, and no faster": 16-bit activations, FP8 weights with
one scale per 128x128 block, a ~6-token verify step):

* activations x[M, K]: N(0, 1) rounded to bf16;
* bf16 weights W[N, K]: N(0, 0.02) rounded to bf16;
* bias[N] (QKV projection only): N(0, 0.01) rounded to bf16;
* FP8 weights Wq[N, K]: N(0, 1), clamped to +-448, cast to OCP e4m3 (E4M3FN)
  with round-to-nearest-even by torch's cast;
* block scales S[ceil(N/128), ceil(K/128)]: fp32 lognormal, exp(ln 0.01 + 0.5 z).

Every tensor is drawn from its own ``torch.Generator`` seeded from
``seed_for(config_id, layer_idx, tensor)``, so any tensor can be regenerated on
its own, on the CPU or on a CUDA device (the two devices give different
streams; a test always hands both implementations the same bytes).
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

SEED_BASE = 20261202

# Qwen2.5-72B decoder-layer linear shapes (N, K) and whether the layer has a bias.
QWEN72B_HIDDEN = 8192
QWEN72B_LAYERS = 80
QWEN72B_SHAPES = {
    "qkv": (10240, 8192, True),
    "o": (8192, 8192, False),
    "gate_up": (59136, 8192, False),
    "down": (8192, 29568, False),
}
QWEN72B_LM_HEAD = (152064, 8192, False)

_TENSOR_SALT = {"x": 0, "w": 1, "bias": 2, "scales": 3}

DTYPE_BF16 = "bf16"
DTYPE_FP8_B128 = "fp8_b128"


def seed_for(config_id: int, layer_idx: int, tensor: str) -> int:
    """Seed of one tensor of one layer of one workload configuration."""
    return SEED_BASE + 1000 * config_id + layer_idx + 100_000_000 * _TENSOR_SALT[tensor]


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(seed)
    return g


def normal_bf16(shape, std: float, seed: int, device="cpu") -> torch.Tensor:
    """N(0, std^2) samples rounded (RNE) to bf16."""
    t = torch.randn(shape, generator=_gen(seed, device), device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(torch.bfloat16)


def fp8_e4m3_weights(shape, seed: int, device="cpu") -> torch.Tensor:
    """N(0,1) clamped to +-448 and cast to e4m3; returned as raw uint8 codes."""
    t = torch.randn(shape, generator=_gen(seed, device), device=device, dtype=torch.float32)
    t.clamp_(-448.0, 448.0)
    return t.to(torch.float8_e4m3fn).view(torch.uint8)


def block_scales(N: int, K: int, seed: int, device="cpu") -> torch.Tensor:
    """fp32 scales, one per 128x128 block: exp(ln(0.01) + 0.5 z)."""
    shape = ((N + 127) // 128, (K + 127) // 128)
    z = torch.randn(shape, generator=_gen(seed, device), device=device, dtype=torch.float32)
    return torch.exp(z * 0.5 + math.log(0.01))


@dataclass
class LayerInputs:
    """One decode linear: y[M,N] = x[M,K] . W[N,K]^T (+ bias)."""

    dtype: str
    M: int
    N: int
    K: int
    x: torch.Tensor            # bf16 [M, K]
    w: torch.Tensor            # bf16 [N, K] or uint8 e4m3 codes [N, K]
    scales: torch.Tensor | None  # fp32 [ceil(N/128), ceil(K/128)] (FP8 only)
    bias: torch.Tensor | None  # bf16 [N] or None

    @property
    def weight_bytes(self) -> int:
        if self.dtype == DTYPE_BF16:
            return 2 * self.N * self.K
        return self.N * self.K + 4 * ((self.N + 127) // 128) * ((self.K + 127) // 128)

    @property
    def algorithmic_bytes(self) -> int:
        """Weights (+ scales) + x + y + bias: every byte the layer must move once."""
        b = self.weight_bytes + 2 * self.M * self.K + 2 * self.M * self.N
        if self.bias is not None:
            b += 2 * self.N
        return b

    def to(self, device) -> "LayerInputs":
        mv = lambda t: None if t is None else t.to(device)  # noqa: E731
        return LayerInputs(self.dtype, self.M, self.N, self.K, mv(self.x), mv(self.w),
                           mv(self.scales), mv(self.bias))


def make_layer(dtype: str, M: int, N: int, K: int, *, bias: bool, config_id: int,
               layer_idx: int = 0, device="cpu", w_std: float = 0.02) -> LayerInputs:
    """Draw the inputs of one layer with the workload distributions above."""
    x = normal_bf16((M, K), 1.0, seed_for(config_id, layer_idx, "x"), device)
    b = normal_bf16((N,), 0.01, seed_for(config_id, layer_idx, "bias"), device) if bias else None
    if dtype == DTYPE_BF16:
        w = normal_bf16((N, K), w_std, seed_for(config_id, layer_idx, "w"), device)
        s = None
    elif dtype == DTYPE_FP8_B128:
        w = fp8_e4m3_weights((N, K), seed_for(config_id, layer_idx, "w"), device)
        s = block_scales(N, K, seed_for(config_id, layer_idx, "scales"), device)
    else:
        raise ValueError(f"unknown dtype {dtype!r}")
    return LayerInputs(dtype, M, N, K, x, w, s, b)


def bf16_bits(t: torch.Tensor):
    """Raw uint16 bit patterns of a bf16 tensor as a numpy array (CPU copy)."""
    import numpy as np
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


def u8_codes(t: torch.Tensor):
    """Raw uint8 codes of an e4m3 weight tensor as a numpy array (CPU copy)."""
    return t.detach().to("cpu").contiguous().view(torch.uint8).numpy()
