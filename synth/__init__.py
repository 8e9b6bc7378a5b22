"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This module draws random numbers and lays them out; it holds none of the
method's arithmetic (no normalisation, no products, no softmax).  Every tensor
it returns lives on the CPU; callers copy it wherever they need it.  Values
destined for bf16 operands are drawn in fp32 and converted by torch's own
round-to-nearest-even conversion, so the CUDA path and the oracle start from
exactly the same bits.

Workload shapes follow the synthetic stand-ins for the pages' workloads:
random-init bf16 weights ~N(0, 0.02), activations ~N(0, 1), per-request KV
lengths uniform or log-uniform, physically shuffled KV pages of 16 tokens.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np
import torch

BF16 = torch.bfloat16
F32 = torch.float32


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed) & 0x7FFFFFFFFFFFFFFF)
    return g


def normal(shape, seed: int, std: float = 1.0, mean: float = 0.0, dtype=BF16) -> torch.Tensor:
    """Seeded N(mean, std^2) tensor, drawn in fp32 then converted to ``dtype``."""
    t = torch.randn(tuple(shape), generator=_gen(seed), dtype=F32)
    if std != 1.0:
        t.mul_(std)
    if mean != 0.0:
        t.add_(mean)
    return t.to(dtype)


def small_ints(shape, seed: int, lo: int = -8, hi: int = 8, dtype=BF16) -> torch.Tensor:
    """Seeded integers in [lo, hi] stored as ``dtype`` (exact in bf16 for |v| <= 256)."""
    t = torch.randint(lo, hi + 1, tuple(shape), generator=_gen(seed), dtype=torch.int64)
    return t.to(dtype)


def uniform_ints(n: int, lo: int, hi: int, seed: int) -> np.ndarray:
    """n seeded integers uniform on the closed range [lo, hi] (int32)."""
    rng = np.random.default_rng(seed)
    return rng.integers(lo, hi + 1, size=n, dtype=np.int64).astype(np.int32)


def loguniform_ints(n: int, lo: int, hi: int, seed: int) -> np.ndarray:
    """n seeded integers log-uniform on [lo, hi] (int32)."""
    rng = np.random.default_rng(seed)
    u = rng.uniform(math.log(lo), math.log(hi + 1), size=n)
    v = np.floor(np.exp(u)).astype(np.int64)
    return np.clip(v, lo, hi).astype(np.int32)


def token_ids(n: int, vocab: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return rng.integers(0, vocab, size=n, dtype=np.int64).astype(np.int32)


@dataclass
class PagedLayout:
    """Physical page assignment for a batch of requests.

    ``block_table[b][i]`` is the physical page holding tokens
    ``[i*page_size, (i+1)*page_size)`` of request ``b``; unused entries are -1.
    Pages are handed out in a seeded random order so that logically adjacent
    pages are physically scattered.
    """

    block_table: np.ndarray  # int32 [B][max_pages]
    num_pages: int
    page_size: int
    max_pages: int


def paged_layout(capacity_tokens, page_size: int, seed: int, spare_pages: int = 3,
                 max_pages: int | None = None) -> PagedLayout:
    caps = [int(c) for c in capacity_tokens]
    need = [(c + page_size - 1) // page_size for c in caps]
    mp = max(need) if need else 1
    if max_pages is not None:
        if max_pages < mp:
            raise ValueError("max_pages smaller than the longest request needs")
        mp = max_pages
    mp = max(mp, 1)
    total = sum(need) + spare_pages
    rng = np.random.default_rng(seed)
    perm = rng.permutation(total).astype(np.int32)
    bt = np.full((len(caps), mp), -1, dtype=np.int32)
    k = 0
    for b, n in enumerate(need):
        bt[b, :n] = perm[k:k + n]
        k += n
    return PagedLayout(bt, total, page_size, mp)


def linspace_control(rows: int, cols: int) -> torch.Tensor:
    """The linspace(-1000, 1000) matrix used as a split-sensitivity control, as bf16."""
    return torch.linspace(-1000.0, 1000.0, rows * cols, dtype=F32).reshape(rows, cols).to(BF16)


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


LLAMA31_8B_LAYER = LayerShape(4096, 32, 8, 128, 14336, 1e-5, 500000.0)
QWEN3_8B_LAYER = LayerShape(4096, 32, 8, 128, 12288, 1e-6, 1000000.0, qk_norm=True)
TINY_LAYER = LayerShape(256, 4, 2, 64, 512, 1e-5, 10000.0)
TINY_QK_LAYER = LayerShape(256, 4, 2, 64, 512, 1e-5, 10000.0, qk_norm=True)


def layer_weights(shape: LayerShape, seed: int, std: float = 0.02, gamma_std: float = 0.0):
    """Random-init bf16 weights of one pre-norm decoder layer (nn.Linear [out][in] layout).

    ``w_gate_up`` stacks the gate projection (rows 0..F-1) over the up projection
    (rows F..2F-1).  Norm weights are 1 (``gamma_std`` = 0) or ~N(1, gamma_std).
    """
    d, F, hd = shape.d_model, shape.ffn_dim, shape.head_dim
    qo = shape.n_q_heads * hd

    def gamma(s, n=d):
        if gamma_std == 0.0:
            return torch.ones(n, dtype=BF16)
        return normal((n,), s, std=gamma_std, mean=1.0)

    w = {
        "attn_norm": gamma(seed + 1),
        "w_qkv": normal((shape.qkv_dim, d), seed + 2, std=std),
        "w_o": normal((d, qo), seed + 3, std=std),
        "ffn_norm": gamma(seed + 4),
        "w_gate_up": normal((2 * F, d), seed + 5, std=std),
        "w_down": normal((d, F), seed + 6, std=std),
    }
    if shape.qk_norm:
        w["q_norm"] = gamma(seed + 7, hd)
        w["k_norm"] = gamma(seed + 8, hd)
    return w


def normal_device(shape, seed: int, std: float = 1.0, mean: float = 0.0, dtype=BF16, device="cuda") -> torch.Tensor:
    """Seeded N(mean, std^2) tensor drawn by torch's device generator (for full-size
    weights too large to draw on the host quickly)."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) & 0x7FFFFFFFFFFFFFFF)
    t = torch.randn(tuple(shape), generator=g, dtype=F32, device=device)
    if std != 1.0:
        t.mul_(std)
    if mean != 0.0:
        t.add_(mean)
    return t.to(dtype)


def fill_paged(k_cache: torch.Tensor, v_cache: torch.Tensor, block_row, K: torch.Tensor, V: torch.Tensor, start: int = 0):
    """Store K/V rows [L][Hkv][hd] of one request at positions start.. into paged caches
    [num_pages][Hkv][page_size][hd] following its block-table row (pure data movement)."""
    L = K.shape[0]
    ps = k_cache.shape[2]
    pos = torch.arange(start, start + L)
    row = torch.as_tensor(np.asarray(block_row), dtype=torch.int64)
    pages = row[pos // ps].to(k_cache.device)
    slots = (pos % ps).to(k_cache.device)
    k_cache[pages, :, slots, :] = K.to(k_cache.device, k_cache.dtype)
    v_cache[pages, :, slots, :] = V.to(v_cache.device, v_cache.dtype)
