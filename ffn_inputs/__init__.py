"""Seeded synthetic inputs for the FP8 SwiGLU FFN block.

This module only draws random numbers and casts the draws to the block's
input dtype (bf16 bit patterns as ``uint16``).  It holds none of the block's
arithmetic: no normalisation, no quantisation, no matmul.  Both the CPU
oracle (tests) and the CUDA library (tests, bench) take their inputs from
here, so the two sides always see the same bits.

Workload shapes follow the Llama / Qwen FFN dimensions the pages train and
decode with ("llama_model.cpp", ``LLamaModel::_forward_block``: the FFN sees
``B*T`` tokens of width ``C`` and an intermediate width ``D``; the up
projection is ``[2*D, C]`` and the down projection ``[C, D]``, see
``fill_block_shapes``).  No trained weights or datasets exist here, so every
tensor is a seeded Gaussian:

* prefill: residual ``res`` and branch output ``x`` ~ N(0, 1), RMSNorm gain
  ~ 1 + N(0, 0.1), up/down weights ~ N(0, 0.02); drawn in fp32 in the order
  res, x, gain, W1, W2 and rounded to bf16 (the model dtype).  Configurations
  with outliers then draw two Bernoulli(0.001) masks (res, x) and multiply the
  selected fp32 draws by 20 before the bf16 rounding.
* decode: one token ``x`` ~ N(0, 1), gate|up weights ``[2H, C]`` (gate rows
  first) and down weights ``[C, H]`` ~ N(0, 0.02), drawn in that order, bf16.

Weights are returned in bf16; turning them into FP8 records (per-tensor
scale for prefill, per-row scale for decode) is the block's own arithmetic
and each side does it with its own quantiser.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class PrefillConfig:
    name: str
    B: int
    T: int
    C: int
    H: int
    eps: float
    outliers: bool = False
    seed: int = 0

    @property
    def N(self) -> int:
        return self.B * self.T

    @property
    def gemm_flop(self) -> int:
        # gate|up: 2*N*C*2H, down: 2*N*H*C
        return 2 * self.N * self.C * 2 * self.H + 2 * self.N * self.H * self.C


@dataclasses.dataclass(frozen=True)
class DecodeConfig:
    name: str
    C: int
    H: int
    seed: int = 0

    @property
    def weight_bytes(self) -> int:
        # FP8 weights (2H*C + C*H), fp32 row scales (2H + C), bf16 x and out.
        C, H = self.C, self.H
        return 2 * H * C + C * H + 4 * (2 * H + C) + 2 * C + 2 * C


PREFILL = {
    "tiny": PrefillConfig("tiny", B=2, T=32, C=256, H=768, eps=1e-5),
    "llama3.2-1b": PrefillConfig("llama3.2-1b", B=4, T=1024, C=2048, H=8192, eps=1e-5),
    "qwen2.5-7b": PrefillConfig("qwen2.5-7b", B=4, T=2048, C=3584, H=18944, eps=1e-6, outliers=True),
    "llama3-8b": PrefillConfig("llama3-8b", B=8, T=2048, C=4096, H=14336, eps=1e-5),
}

DECODE = {
    "llama3-8b-decode": DecodeConfig("llama3-8b-decode", C=4096, H=14336),
}


def _bf16_bits(t: torch.Tensor) -> np.ndarray:
    """fp32 tensor -> bf16 bit patterns (round to nearest even, torch's cast)."""
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def prefill_inputs(cfg: PrefillConfig, *, weights: bool = True) -> dict:
    """Draw res, x [N, C], gain [C] and (optionally) W1 [2H, C], W2 [C, H] as bf16 bits.

    ``weights=False`` skips the weight draws (the activations are drawn first,
    so they do not change); outlier masks are then drawn right after gain.
    """
    g = torch.Generator(device="cpu").manual_seed(cfg.seed)
    N, C, H = cfg.N, cfg.C, cfg.H
    res = torch.randn(N, C, generator=g, dtype=torch.float32)
    x = torch.randn(N, C, generator=g, dtype=torch.float32)
    gain = 1.0 + 0.1 * torch.randn(C, generator=g, dtype=torch.float32)
    out = {}
    if weights:
        w1 = 0.02 * torch.randn(2 * H, C, generator=g, dtype=torch.float32)
        w2 = 0.02 * torch.randn(C, H, generator=g, dtype=torch.float32)
        out["w1"] = _bf16_bits(w1)
        out["w2"] = _bf16_bits(w2)
        del w1, w2
    if cfg.outliers:
        m_res = torch.rand(N, C, generator=g) < 0.001
        m_x = torch.rand(N, C, generator=g) < 0.001
        res = torch.where(m_res, res * 20.0, res)
        x = torch.where(m_x, x * 20.0, x)
    out["res"] = _bf16_bits(res)
    out["x"] = _bf16_bits(x)
    out["gain"] = _bf16_bits(gain)
    out["eps"] = float(np.float32(cfg.eps))
    return out


def decode_inputs(cfg: DecodeConfig) -> dict:
    """Draw x [C], W_gate [H, C], W_up [H, C], W_down [C, H] as bf16 bits."""
    g = torch.Generator(device="cpu").manual_seed(cfg.seed)
    C, H = cfg.C, cfg.H
    x = torch.randn(C, generator=g, dtype=torch.float32)
    w_gu = 0.02 * torch.randn(2 * H, C, generator=g, dtype=torch.float32)
    w_d = 0.02 * torch.randn(C, H, generator=g, dtype=torch.float32)
    gu = _bf16_bits(w_gu)
    return {
        "x": _bf16_bits(x),
        "w_gate": np.ascontiguousarray(gu[:H]),
        "w_up": np.ascontiguousarray(gu[H:]),
        "w_down": _bf16_bits(w_d),
    }


def random_bf16(shape, seed: int, std: float = 1.0) -> np.ndarray:
    """Generic seeded N(0, std) bf16 tensor for shape sweeps and edge cases."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    return _bf16_bits(std * torch.randn(*shape, generator=g, dtype=torch.float32))


def random_codes(shape, seed: int) -> np.ndarray:
    """Seeded uniformly random FP8 E4M3 bit patterns, the two NaN codes excluded."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    c = torch.randint(0, 254, tuple(shape), generator=g, dtype=torch.int32).numpy()
    # map 0..253 onto the 254 finite codes (skip 0x7F and 0xFF)
    c = np.where(c >= 0x7F, c + 1, c)
    return c.astype(np.uint8)
