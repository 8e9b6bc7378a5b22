"""Decoder layer through bi_layer_forward: oracle parity, prefill == decode, invariance, modes."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth
from tests.helpers import TOL_BF16, bits_equal, cuda, f64, max_rel_err

pytestmark = pytest.mark.gpu
bi = pytest.importorskip("invariant_deterministic_02_gb300")
PS = 16


class LayerRig:
    """One layer's weights, RoPE tables and a paged cache holding per-request histories."""

    def __init__(self, shape, seed, max_pos=8192, num_pages=4096, gamma_std=0.1, act_f32=False):
        self.shape = shape
        self.act_f32 = act_f32  # hidden states fp32 (fp32-activation layer) instead of bf16
        self.w_host = synth.layer_weights(shape, seed, std=0.02, gamma_std=gamma_std)
        self.w = {k: cuda(v) for k, v in self.w_host.items()}
        self.lw = bi.LayerWeights(*[self.w[k].data_ptr() for k in
                                    ("attn_norm", "w_qkv", "w_o", "ffn_norm", "w_gate_up", "w_down")],
                                  *[self.w[k].data_ptr() if k in self.w else None for k in ("q_norm", "k_norm")])
        self.dims = bi.ModelDims(shape.d_model, shape.n_q_heads, shape.n_kv_heads, shape.head_dim, shape.ffn_dim, 8,
                                 PS, max_pos, shape.rms_eps, 1 if act_f32 else 0)
        half = shape.head_dim // 2
        self.cos = torch.empty((max_pos, half), dtype=torch.float32, device="cuda")
        self.sin = torch.empty_like(self.cos)
        bi.bi_rope_table(shape.rope_theta, shape.head_dim, max_pos, self.cos, self.sin)
        self.num_pages = num_pages
        self.kc = torch.zeros((num_pages, shape.n_kv_heads, PS, shape.head_dim), dtype=torch.bfloat16, device="cuda")
        self.vc = torch.zeros_like(self.kc)
        self.free = list(np.random.default_rng(seed).permutation(num_pages))
        self.rows = {}  # request -> page list
        self.hist = {}  # request -> (K, V) float64 history in the oracle's view

    def add_request(self, req, hist_len, seed, capacity):
        need = (capacity + PS - 1) // PS
        self.rows[req] = [int(self.free.pop()) for _ in range(need)]
        K = synth.normal((hist_len, self.shape.n_kv_heads, self.shape.head_dim), seed)
        V = synth.normal((hist_len, self.shape.n_kv_heads, self.shape.head_dim), seed + 1)
        if hist_len:
            synth.fill_paged(self.kc, self.vc, self.rows[req], K, V)
        self.hist[req] = (f64(K), f64(V))

    def run(self, h, items, mode=bi.INVARIANT, target=-1):
        """items: list of (request, n_tokens, pos0).  h: [T][d] bf16, or fp32 with act_f32 (cuda), updated in place."""
        B = len(items)
        counts = [n for _, n, _ in items]
        qs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
        mp = max(len(self.rows[r]) for r, _, _ in items)
        bt = np.full((B, mp), -1, dtype=np.int32)
        for b, (r, _, _) in enumerate(items):
            bt[b, :len(self.rows[r])] = self.rows[r]
        keep = [cuda(torch.from_numpy(qs)), cuda(torch.tensor([p for _, _, p in items], dtype=torch.int32)),
                cuda(torch.from_numpy(bt))]
        tr = int(qs[target]) if target >= 0 else -1
        tc = counts[target] if target >= 0 else 0
        batch = bi.Batch(B, int(qs[-1]), max(counts), keep[0].data_ptr(), keep[1].data_ptr(), keep[2].data_ptr(), mp,
                         self.num_pages, target, tr, tc)
        bi.bi_layer_forward(self.dims, self.lw, self.cos, self.sin, h, batch, self.kc, self.vc, mode=mode)
        torch.cuda.synchronize()
        return h

    def oracle(self, h_in, items):
        kv = oracle.OracleKV(1, self.shape.n_kv_heads, self.shape.head_dim)
        for r, _, p0 in items:
            K, V = self.hist[r]
            kv.set(0, r, K[:p0], V[:p0])
        w = {k: f64(v) for k, v in self.w_host.items()}
        return oracle.layer_forward(f64(h_in), w, self.shape, kv, 0, [(r, n) for r, n, _ in items],
                                    [p for _, _, p in items], act32=self.act_f32)


@pytest.mark.parametrize("shape", [synth.TINY_LAYER, synth.TINY_QK_LAYER], ids=["plain", "qk_norm"])
def test_tiny_layer_prefill_then_decode_parity(shape):
    rig = LayerRig(shape, 3)
    rig.add_request(0, 0, 10, 64)
    rig.add_request(1, 0, 12, 64)
    h = synth.normal((42, 256), 5)
    items = [(0, 37, 0), (1, 5, 0)]
    out = rig.run(cuda(h), items)
    kv = oracle.OracleKV(1, 2, 64)
    w = {k: f64(v) for k, v in rig.w_host.items()}
    ref = oracle.layer_forward(f64(h), w, rig.shape, kv, 0, [(0, 37), (1, 5)], [0, 0])
    assert max_rel_err(f64(out), ref) <= TOL_BF16
    # one decode step for both, on top of the prefilled cache
    h2 = synth.normal((2, 256), 6)
    out2 = rig.run(cuda(h2), [(0, 1, 37), (1, 1, 5)])
    ref2 = oracle.layer_forward(f64(h2), w, rig.shape, kv, 0, [(0, 1), (1, 1)], [37, 5])
    assert max_rel_err(f64(out2), ref2) <= TOL_BF16


@pytest.mark.parametrize("B", [1, 4, 16, 64])
def test_llama8b_layer_decode_parity(B):
    shape = synth.LLAMA31_8B_LAYER
    rig = LayerRig(shape, 20 + B, num_pages=B * 260 + 8)
    lens = synth.uniform_ints(B, 128, 4096, 30 + B)
    for b in range(B):
        rig.add_request(b, int(lens[b]) - 1, 1000 + 2 * b, int(lens[b]))
    h = synth.normal((B, shape.d_model), 40 + B)
    items = [(b, 1, int(lens[b]) - 1) for b in range(B)]
    out = rig.run(cuda(h), items)
    ref = rig.oracle(h, items)
    assert max_rel_err(f64(out), ref) <= TOL_BF16


def test_llama8b_layer_target_bitwise_across_batches_and_modes():
    shape = synth.LLAMA31_8B_LAYER
    rig = LayerRig(shape, 7, num_pages=64 * 260 + 8)
    tlen = 2500
    rig.add_request("t", tlen - 1, 4321, tlen)
    ht = synth.normal((1, shape.d_model), 4322)
    ref = rig.run(cuda(ht), [("t", 1, tlen - 1)])
    refk = rig.run(cuda(ht), [("t", 1, tlen - 1)], mode=bi.INVARIANT_KSPLIT)
    lens = synth.uniform_ints(63, 128, 4096, 50)
    for b in range(63):
        rig.add_request(b, int(lens[b]) - 1, 2000 + 2 * b, int(lens[b]))
    for trial, B in enumerate([2, 5, 16, 64]):
        pos = (3 * trial + 1) % B
        others = [(b, 1, int(lens[b]) - 1) for b in range(B - 1)]
        items = others[:pos] + [("t", 1, tlen - 1)] + others[pos:]
        h = synth.normal((B, shape.d_model), 60 + trial)
        h[pos] = ht[0]
        out = rig.run(cuda(h), items)
        assert bits_equal(out[pos:pos + 1], ref), B
        hp = cuda(h)
        outp = rig.run(hp, items, mode=bi.PROTECTED, target=pos)
        assert bits_equal(outp[pos:pos + 1], ref), ("protected", B)
        outf = rig.run(cuda(h), items, mode=bi.FAST)
        refo = rig.oracle(h, items)
        assert max_rel_err(f64(outf), refo) <= TOL_BF16
        assert max_rel_err(f64(outp), refo) <= TOL_BF16
        outk = rig.run(cuda(h), items, mode=bi.INVARIANT_KSPLIT)
        assert bits_equal(outk[pos:pos + 1], refk), ("ksplit", B)
        assert max_rel_err(f64(outk), refo) <= TOL_BF16


@pytest.mark.parametrize("mode,shape", [(bi.INVARIANT, synth.LLAMA31_8B_LAYER),
                                        (bi.INVARIANT_KSPLIT, synth.LLAMA31_8B_LAYER),
                                        (bi.INVARIANT, synth.QWEN3_8B_LAYER)], ids=["llama", "llama-ksplit", "qwen3-qknorm"])
def test_layer_chunked_prefill_equals_token_by_token_decode(mode, shape):
    # INVARIANT_KSPLIT: prefill chunks of > 128 tokens merge the K parts inside a CTA,
    # decode runs them on separate CTAs; the bits must agree all the same.  The Qwen3
    # layer adds the per-head q/k RMSNorm before RoPE.
    L = 600
    h = synth.normal((L, shape.d_model), 70)
    outs = []
    for chunks in ([L], [256, 256, 88], [97] * 6 + [18], [1] * 40 + [L - 40]):
        rig = LayerRig(shape, 8, num_pages=64)
        rig.add_request(0, 0, 1, L)
        res = []
        p = 0
        for n in chunks:
            res.append(rig.run(cuda(h[p:p + n]), [(0, n, p)], mode=mode))
            p += n
        outs.append(torch.cat(res))
    for o in outs[1:]:
        assert bits_equal(o, outs[0])
    # token-by-token decode batched with a neighbour that prefills at the same time
    rig = LayerRig(shape, 8, num_pages=128)
    rig.add_request(0, 0, 1, L)
    rig.add_request(1, 0, 2, L)
    hn = synth.normal((L, shape.d_model), 71)
    res = []
    for p in range(L):
        x = torch.cat([h[p:p + 1], hn[p:p + 1]])
        res.append(rig.run(cuda(x), [(0, 1, p), (1, 1, p)], mode=mode)[0:1])
    assert bits_equal(torch.cat(res), outs[0])
