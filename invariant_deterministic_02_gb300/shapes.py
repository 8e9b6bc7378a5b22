"""Dimensions of the decoder layers and models the library is built and measured for.

Plain data: the model driver (``model.py``) reads these fields; the C ABI takes
them through ``bi_model_dims``.
"""
from __future__ import annotations

from dataclasses import dataclass


@dataclass
class LayerShape:
    d_model: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ffn_dim: int
    rms_eps: float = 1e-5
    rope_theta: float = 500000.0
    page_size: int = 16
    qk_norm: bool = False  # per-head RMSNorm of q and k before RoPE (Qwen3)

    @property
    def qkv_dim(self) -> int:
        return (self.n_q_heads + 2 * self.n_kv_heads) * self.head_dim


# Llama-3.1-8B-shaped and Qwen3-8B-shaped decoder layers
LLAMA31_8B_LAYER = LayerShape(4096, 32, 8, 128, 14336, 1e-5, 500000.0)
QWEN3_8B_LAYER = LayerShape(4096, 32, 8, 128, 12288, 1e-6, 1000000.0, qk_norm=True)
