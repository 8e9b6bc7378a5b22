"""Model driver over the C ABI: random-init weights, paged KV caches, batch descriptors.

Everything numeric runs in libbi's kernels through ``bi_model_forward``; this
module only owns device memory (via torch), hands out KV pages and builds the
batch descriptor (request -> query rows, first position, block-table row).
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass, field

import numpy as np
import torch

from . import (PROTECTED, Batch, LayerWeights, ModelDims, ModelWeights, PAGE_SIZE, bi_model_forward, bi_model_workspace,
               bi_rope_table, INVARIANT)
from .shapes import LLAMA31_8B_LAYER, QWEN3_8B_LAYER, LayerShape


@dataclass
class ModelShape:
    layer: LayerShape  # any object with LayerShape's fields
    n_layers: int
    vocab: int
    max_pos: int = 32768


QWEN3_8B = ModelShape(QWEN3_8B_LAYER, 36, 151936)
LLAMA31_8B = ModelShape(LLAMA31_8B_LAYER, 32, 128256)


def _normal(shape, seed: int, std: float, mean: float, device, on_host: bool) -> torch.Tensor:
    """Seeded N(mean, std^2) bf16 tensor for random-init weights, drawn in fp32 by
    torch's generator on the host or on the device."""
    gdev = "cpu" if on_host else device
    g = torch.Generator(device=gdev)
    g.manual_seed(int(seed) & 0x7FFFFFFFFFFFFFFF)
    t = torch.randn(tuple(shape), generator=g, dtype=torch.float32, device=gdev)
    if std != 1.0:
        t.mul_(std)
    if mean != 0.0:
        t.add_(mean)
    return t.to(torch.bfloat16).to(device)


@dataclass
class ForwardOut:
    logits: torch.Tensor  # [B][V] fp32
    top_v: torch.Tensor   # [B][k]
    top_i: torch.Tensor   # [B][k]


class PagePool:
    """Free list of physical KV pages; a request owns an ordered list of pages."""

    def __init__(self, num_pages: int, seed: int | None = None):
        order = np.arange(num_pages, dtype=np.int32)
        if seed is not None:
            order = np.random.default_rng(seed).permutation(num_pages).astype(np.int32)
        self.free = list(order[::-1])
        self.owned: dict[int, list[int]] = {}

    def ensure(self, req: int, tokens: int):
        pages = self.owned.setdefault(req, [])
        need = (tokens + PAGE_SIZE - 1) // PAGE_SIZE
        while len(pages) < need:
            if not self.free:
                raise MemoryError("KV page pool exhausted")
            pages.append(int(self.free.pop()))
        return pages

    def release(self, req: int):
        for p in reversed(self.owned.pop(req, [])):
            self.free.append(p)


class BiModel:
    def __init__(self, shape: ModelShape, weights: dict, num_pages: int, device="cuda", page_seed: int | None = None,
                 act_f32: bool = False):
        """act_f32: fp32 activations with the same bf16 weights and bf16 KV cache."""
        self.shape = shape
        self.device = device
        L = shape.layer
        self.w = weights
        self.dims = ModelDims(L.d_model, L.n_q_heads, L.n_kv_heads, L.head_dim, L.ffn_dim, shape.vocab, PAGE_SIZE,
                              shape.max_pos, L.rms_eps, 1 if act_f32 else 0)
        self.rope_cos = torch.empty((shape.max_pos, L.head_dim // 2), dtype=torch.float32, device=device)
        self.rope_sin = torch.empty_like(self.rope_cos)
        bi_rope_table(L.rope_theta, L.head_dim, shape.max_pos, self.rope_cos, self.rope_sin)
        self.num_pages = num_pages
        self.k_caches = [torch.zeros((num_pages, L.n_kv_heads, PAGE_SIZE, L.head_dim), dtype=torch.bfloat16,
                                     device=device) for _ in range(shape.n_layers)]
        self.v_caches = [torch.zeros_like(k) for k in self.k_caches]
        self.k_ptrs = (ctypes.c_void_p * max(1, shape.n_layers))(*[k.data_ptr() for k in self.k_caches])
        self.v_ptrs = (ctypes.c_void_p * max(1, shape.n_layers))(*[v.data_ptr() for v in self.v_caches])
        self._layer_structs = (LayerWeights * max(1, shape.n_layers))(*[
            LayerWeights(lw["attn_norm"].data_ptr(), lw["w_qkv"].data_ptr(), lw["w_o"].data_ptr(),
                         lw["ffn_norm"].data_ptr(), lw["w_gate_up"].data_ptr(), lw["w_down"].data_ptr(),
                         lw["q_norm"].data_ptr() if "q_norm" in lw else None,
                         lw["k_norm"].data_ptr() if "k_norm" in lw else None)
            for lw in weights["layers"]])
        self.mw = ModelWeights(weights["embed"].data_ptr(), self._layer_structs, shape.n_layers,
                               weights["final_norm"].data_ptr(), weights["lm_head"].data_ptr())
        self.pool = PagePool(num_pages, seed=page_seed)
        self.lengths: dict[int, int] = {}
        self._ws = None

    # ------------------------------------------------------------ construction
    @staticmethod
    def random_weights(shape: ModelShape, seed: int, device="cuda", std: float = 0.02, on_host: bool | None = None):
        """Random-init bf16 weights ~N(0, std^2) (the linear-layer [out][in] layout;
        w_gate_up stacks gate over up).  Small models draw on the host, large ones
        with the device's generator.  RMSNorm weights are 1, except the Qwen3 q/k head
        norms of large models, ~N(1, 0.1^2)."""
        L = shape.layer
        if on_host is None:
            on_host = L.d_model * L.ffn_dim * shape.n_layers < 64 * 1024 * 1024
        nrm = lambda dims, s, sd=std, mean=0.0: _normal(dims, s, sd, mean, device, on_host)
        ones = lambda n: torch.ones(n, dtype=torch.bfloat16, device=device)
        layers = []
        for i in range(shape.n_layers):
            s = seed + 100 * (i + 1)
            lw = {
                "attn_norm": ones(L.d_model),
                "w_qkv": nrm((L.qkv_dim, L.d_model), s + 2),
                "w_o": nrm((L.d_model, L.n_q_heads * L.head_dim), s + 3),
                "ffn_norm": ones(L.d_model),
                "w_gate_up": nrm((2 * L.ffn_dim, L.d_model), s + 5),
                "w_down": nrm((L.d_model, L.ffn_dim), s + 6),
            }
            if L.qk_norm:
                # small models: unit head norms; large ones: ~N(1, 0.1^2)
                lw["q_norm"] = ones(L.head_dim) if on_host else nrm((L.head_dim,), s + 7, 0.1, 1.0)
                lw["k_norm"] = ones(L.head_dim) if on_host else nrm((L.head_dim,), s + 8, 0.1, 1.0)
            layers.append(lw)
        embed = nrm((shape.vocab, L.d_model), seed + 1)
        head = nrm((shape.vocab, L.d_model), seed + 2)
        return {"embed": embed, "layers": layers, "final_norm": ones(L.d_model), "lm_head": head}

    @classmethod
    def random(cls, shape: ModelShape, seed: int, device="cuda", num_pages: int = 512, page_seed: int | None = 3,
               act_f32: bool = False):
        return cls(shape, cls.random_weights(shape, seed, device), num_pages, device, page_seed, act_f32)

    def host_weights(self):
        """float64 numpy copies of the weights (for the oracle on small models)."""
        f = lambda t: t.detach().cpu().double().numpy()
        return {"embed": f(self.w["embed"]), "final_norm": f(self.w["final_norm"]), "lm_head": f(self.w["lm_head"]),
                "layers": [{k: f(v) for k, v in lw.items()} for lw in self.w["layers"]]}

    # ------------------------------------------------------------ batches
    def make_batch(self, items, target_request: int = -1):
        """items: list of (request id, int32 token array).  Returns (Batch, keep-alive tensors, ids)."""
        B = len(items)
        counts = [len(t) for _, t in items]
        q_start = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
        pos0 = np.array([self.lengths.get(r, 0) for r, _ in items], dtype=np.int32)
        rows = [self.pool.ensure(r, int(p) + n) for (r, _), p, n in zip(items, pos0, counts)]
        max_pages = max(1, max(len(r) for r in rows))
        bt = np.full((B, max_pages), -1, dtype=np.int32)
        for b, r in enumerate(rows):
            bt[b, :len(r)] = r
        ids = np.concatenate([np.asarray(t, dtype=np.int32) for _, t in items])
        dev = lambda a: torch.from_numpy(a).to(self.device, non_blocking=False)
        keep = {"q_start": dev(q_start), "pos0": dev(pos0), "bt": dev(bt), "ids": dev(ids)}
        trow = int(q_start[target_request]) if target_request >= 0 else -1
        tcnt = counts[target_request] if target_request >= 0 else 0
        batch = Batch(B, int(q_start[-1]), max(counts), keep["q_start"].data_ptr(), keep["pos0"].data_ptr(),
                      keep["bt"].data_ptr(), max_pages, self.num_pages, target_request, trow, tcnt)
        return batch, keep

    def forward_batch(self, items, k: int = 20, mode=INVARIANT, target_request: int = -1) -> ForwardOut:
        batch, keep = self.make_batch(items, target_request)
        B = len(items)
        logits = torch.empty((B, self.shape.vocab), dtype=torch.float32, device=self.device)
        tv = torch.empty((B, k), dtype=torch.float32, device=self.device)
        ti = torch.empty((B, k), dtype=torch.int32, device=self.device)
        need = bi_model_workspace(self.dims, batch, mode)
        if self._ws is None or self._ws.numel() < need:
            self._ws = torch.empty(need, dtype=torch.uint8, device=self.device)
        bi_model_forward(self.dims, self.mw, self.rope_cos, self.rope_sin, keep["ids"], batch, self.k_ptrs,
                         self.v_ptrs, logits, k, tv, ti, mode=mode, workspace=self._ws, ws_bytes=need)
        for (r, t) in items:
            self.lengths[r] = self.lengths.get(r, 0) + len(t)
        torch.cuda.current_stream().synchronize()  # keep-alive tensors must outlive the launches
        return ForwardOut(logits, tv, ti)

    def install_history(self, req: int, length: int, seed: int):
        """Give request `req` a cached history of `length` tokens whose K/V (every
        layer) are seeded N(0, 1) bf16 values, as if it had been prefilled earlier."""
        if length <= 0:
            return
        pages = self.pool.ensure(req, length)
        L = self.shape.layer
        idx = torch.tensor(pages, dtype=torch.int64, device=self.device)
        n = len(pages)
        g = torch.Generator(device=self.device)
        for li in range(self.shape.n_layers):
            for ci, cache in enumerate((self.k_caches[li], self.v_caches[li])):
                g.manual_seed((seed * 1000003 + li * 2 + ci) & 0x7FFFFFFF)
                vals = torch.randn((n, L.n_kv_heads, PAGE_SIZE, L.head_dim), generator=g, device=self.device)
                cache[idx] = vals.to(torch.bfloat16)
        self.lengths[req] = length

    def pack_prefill(self, items, target, k: int = 20, tile_rows: int = 128, dummy="__pack_dummy__"):
        """BlockLock-Pack-style shared prefill of a protected request (zhaixingw.cn
        post on BlockLock, section on the two modes: terminal-anchored packing with
        an isolated dummy segment, then the protected request's KV state is taken
        out and it decodes alone).

        items: (request id, tokens) pairs, one of them `target`.  The target is
        packed last; a dummy request of filler tokens is inserted just before it
        so that the target's first token starts on a `tile_rows` boundary of the
        packed batch (its GEMM row tiles then hold no other request); the batch
        runs in PROTECTED mode with the target protected (the others take the
        FAST schedule); the dummy's pages are released afterwards.  The target's
        K/V stay in its own pages, ready for target-only decode.
        Returns (ForwardOut of the packed batch, the target's row)."""
        others = [(r, t) for r, t in items if r != target]
        tgt = [t for r, t in items if r == target]
        if len(tgt) != 1:
            raise ValueError("pack_prefill: target must appear once among the items")
        pad = (-sum(len(t) for _, t in others)) % tile_rows
        packed = list(others)
        if pad:
            packed.append((dummy, np.zeros(pad, dtype=np.int32)))
        packed.append((target, tgt[0]))
        out = self.forward_batch(packed, k=k, mode=PROTECTED, target_request=len(packed) - 1)
        if pad:
            self.release(dummy)
        return out, len(packed) - 1

    def copy_prefix(self, src: int, dst: int, tokens: int):
        """Prefix-cache hit: give request `dst` (which must hold no tokens yet) the
        first `tokens` cached positions of request `src`, by copying the K/V pages
        that hold them (every layer).  Later tokens of `dst` continue at position
        `tokens`; any part of a partly copied last page is overwritten then."""
        if self.lengths.get(dst, 0) or self.pool.owned.get(dst):
            raise ValueError("copy_prefix: destination request already holds tokens")
        if tokens <= 0 or tokens > self.lengths.get(src, 0):
            raise ValueError("copy_prefix: %d tokens of a %d-token request" % (tokens, self.lengths.get(src, 0)))
        n = (tokens + PAGE_SIZE - 1) // PAGE_SIZE
        s_idx = torch.tensor(self.pool.owned[src][:n], dtype=torch.int64, device=self.device)
        d_idx = torch.tensor(self.pool.ensure(dst, tokens), dtype=torch.int64, device=self.device)
        for caches in (self.k_caches, self.v_caches):
            for c in caches:
                c.index_copy_(0, d_idx, c.index_select(0, s_idx))
        self.lengths[dst] = tokens

    def reset(self):
        for r in list(self.lengths.keys()) + list(self.pool.owned.keys()):
            self.release(r)

    def release(self, req: int):
        self.pool.release(req)
        self.lengths.pop(req, None)
