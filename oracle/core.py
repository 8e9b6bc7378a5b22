"""Float64 definitions of every step of the batch-invariant forward (test infrastructure only).

Citations name the page and the section the definition follows:
  [BI-notes]   "Batch-Invariant Kernel" reading notes (tom-jerr.github.io), sections RMSNorm / GEMM / Flash Attention
  [TML-digest] devpress.csdn digest of "Defeating Nondeterminism in LLM Inference", sections 2.3, 3.1-3.3
  [BlockLock]  zhaixingw.cn post on BlockLock, sections on greedy decoding and top-20 logits ("坑清单")
  [Book-19.7]  LLM full-stack book, section 19.7.4 (argmax tie-breaking)
"""
from __future__ import annotations

import math

import numpy as np

F64 = np.float64


# ---------------------------------------------------------------------------
# number formats
# ---------------------------------------------------------------------------
def round_bf16(x) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 value, ties to even.

    bfloat16 keeps 8 significant bits (1 implicit + 7 stored) and the float32
    exponent range; below 2**-126 the spacing is fixed at 2**-133.  Written from
    the format's definition: scale the value so the last kept bit is the unit,
    round half-to-even, scale back.  Overflow is not handled (inputs here are far
    below the bf16 maximum).
    """
    x = np.asarray(x, dtype=F64)
    m, e = np.frexp(x)  # x = m * 2**e, 0.5 <= |m| < 1
    q = np.maximum(e, -125) - 8  # exponent of the last kept bit
    return np.ldexp(np.rint(np.ldexp(x, -q)), q)


def round_f32(x) -> np.ndarray:
    """Round float64 values to the nearest float32 value (numpy's IEEE conversion)."""
    return np.asarray(x, dtype=F64).astype(np.float32).astype(F64)


# ---------------------------------------------------------------------------
# RMSNorm  [BI-notes, "RMSNorm", the formula; TML-digest §3.1]
# ---------------------------------------------------------------------------
def rmsnorm(x, gamma, eps: float) -> np.ndarray:
    """y_ij = x_ij / sqrt((1/d) * sum_j x_ij^2 + eps) * gamma_j, per row.

    eps sits inside the square root as in the notes' formula (the digest's
    code omits it; the formula is taken).
    """
    x = np.asarray(x, dtype=F64)
    g = np.asarray(gamma, dtype=F64)
    d = x.shape[-1]
    ms = np.sum(x * x, axis=-1, keepdims=True) / d
    return x / np.sqrt(ms + eps) * g


# ---------------------------------------------------------------------------
# GEMM  [TML-digest §3.2: C[i,j] = sum_k A[i,k] * B[k,j]]
# ---------------------------------------------------------------------------
def gemm(A, W) -> np.ndarray:
    """C = A @ W^T with W stored [N][K] (the linear-layer layout), float64.

    For bf16 inputs every product is exact in float64 and the K-sum carries
    53 bits, so this is the exact matrix product up to float64 rounding.
    """
    A = np.asarray(A, dtype=F64)
    W = np.asarray(W, dtype=F64)
    return A @ W.T


# ---------------------------------------------------------------------------
# Rotary position embedding (reading: the pages never spell out the layer;
# the standard rotate-half RoPE of Llama/Qwen-style decoders is taken)
# ---------------------------------------------------------------------------
def rope_inv_freq(head_dim: int, theta: float) -> np.ndarray:
    """f_i = theta ** (-2i / head_dim), i = 0 .. head_dim/2 - 1."""
    i = np.arange(head_dim // 2, dtype=F64)
    return np.power(F64(theta), -2.0 * i / head_dim)


def rope(x, pos, theta: float) -> np.ndarray:
    """Rotate pairs (i, i + hd/2) of the last axis by angle pos * f_i.

    ``x`` has shape [..., T, H, hd] with ``pos`` [T] (absolute token positions).
    out[i]        = x[i] cos(a_i) - x[i+hd/2] sin(a_i)
    out[i+hd/2]   = x[i+hd/2] cos(a_i) + x[i] sin(a_i)
    """
    x = np.asarray(x, dtype=F64)
    hd = x.shape[-1]
    half = hd // 2
    ang = np.asarray(pos, dtype=F64)[:, None] * rope_inv_freq(hd, theta)[None, :]  # [T][half]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    a, b = x[..., :half], x[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


# ---------------------------------------------------------------------------
# attention  [TML-digest §3.3; BI-notes "Flash Attention"]
# ---------------------------------------------------------------------------
def gather_pages(cache, block_row, length: int) -> np.ndarray:
    """Logical [length][Hkv][hd] view of one request in a paged cache [pages][Hkv][ps][hd]."""
    cache = np.asarray(cache, dtype=F64)
    ps = cache.shape[2]
    out = np.empty((length, cache.shape[1], cache.shape[3]), dtype=F64)
    for t in range(length):
        out[t] = cache[int(block_row[t // ps]), :, t % ps, :]
    return out


def attention(q, K, V, q_pos, scale: float) -> np.ndarray:
    """Causal grouped-query softmax attention for one request, float64.

    q: [Tq][Hq][hd]; K, V: [L][Hkv][hd] (absolute positions 0..L-1);
    q_pos: [Tq] absolute position of each query.  Query t attends to keys
    j <= q_pos[t].  Head h reads kv head h // (Hq/Hkv) (contiguous groups;
    reading: the pages do not name the grouping).  Scores are (q.k) * scale,
    softmax with the row maximum subtracted for range, output sum_j p_j v_j.
    """
    q = np.asarray(q, dtype=F64)
    K = np.asarray(K, dtype=F64)
    V = np.asarray(V, dtype=F64)
    Tq, Hq, hd = q.shape
    Hkv = K.shape[1]
    G = Hq // Hkv
    out = np.zeros((Tq, Hq, hd), dtype=F64)
    for t in range(Tq):
        n = int(q_pos[t]) + 1
        for h in range(Hq):
            g = h // G
            z = (K[:n, g, :] @ q[t, h, :]) * scale
            p = np.exp(z - z.max())
            p /= p.sum()
            out[t, h, :] = p @ V[:n, g, :]
    return out


def split_geometry(length: int, split: int = 256):
    """Fixed-size split-KV boundaries [TML-digest §3.3, the 500/1000-token example].

    Splits are [split*s, split*s + split) in absolute positions from 0.  Returns
    a list of (start, valid_tokens).  Reading: the digest's counts (245, 233)
    are inclusive of the last index; a KV of length L holds positions 0..L-1,
    so the last split of L=500 holds 244 tokens and that of L=1000 holds 232.
    """
    if length <= 0:
        return []
    n = (length + split - 1) // split
    return [(s * split, min(split, length - s * split)) for s in range(n)]


def split_partials(q_vec, K, V, q_pos: int, kv_group: int, scale: float, split: int = 256):
    """Per-split softmax state of one query head over each fixed split.

    For split s covering positions P_s = [split*s, split*s+split) ∩ [0, q_pos]:
      m_s = max_{j in P_s} z_j,  l_s = sum_{j in P_s} exp(z_j - m_s),
      o_s = sum_{j in P_s} exp(z_j - m_s) v_j,       z_j = (q.k_j) * scale.
    Returns arrays m [n], l [n], o [n][hd] (natural-exp domain).
    """
    q_vec = np.asarray(q_vec, dtype=F64)
    K = np.asarray(K, dtype=F64)[:, kv_group, :]
    V = np.asarray(V, dtype=F64)[:, kv_group, :]
    geo = split_geometry(q_pos + 1, split)
    m = np.empty(len(geo))
    l = np.empty(len(geo))
    o = np.empty((len(geo), V.shape[1]))
    for s, (a, n) in enumerate(geo):
        z = (K[a:a + n] @ q_vec) * scale
        m[s] = z.max()
        e = np.exp(z - m[s])
        l[s] = e.sum()
        o[s] = e @ V[a:a + n]
    return m, l, o


# ---------------------------------------------------------------------------
# pointwise ops [TML-digest §3: pointwise ops are batch-invariant as they stand]
# ---------------------------------------------------------------------------
def silu(x) -> np.ndarray:
    x = np.asarray(x, dtype=F64)
    return x / (1.0 + np.exp(-x))


def swiglu(g, u) -> np.ndarray:
    """silu(g) * u (SwiGLU gating of the feed-forward block)."""
    return silu(g) * np.asarray(u, dtype=F64)


# ---------------------------------------------------------------------------
# top-k / argmax [BlockLock post, "坑清单" items 2 and 5; Book-19.7.4 tie-breaking]
# ---------------------------------------------------------------------------
def topk(logits, k: int):
    """Per row: the k largest values, ordered by (value descending, index ascending).

    Reading: the pages show argmax flipping on near-ties but fix no rule; the
    lowest index wins a tie, which makes the selection a total order and its
    result unique.
    """
    L = np.asarray(logits, dtype=F64)
    if L.ndim == 1:
        L = L[None, :]
    rows, V = L.shape
    vals = np.empty((rows, k), dtype=F64)
    idx = np.empty((rows, k), dtype=np.int64)
    ar = np.arange(V)
    for r in range(rows):
        order = np.lexsort((ar, -L[r]))[:k]
        vals[r] = L[r, order]
        idx[r] = order
    return vals, idx


def argmax(logits) -> np.ndarray:
    """Greedy token: the largest logit, lowest index on ties."""
    return topk(logits, 1)[1][:, 0]


# ---------------------------------------------------------------------------
# decoder layer and model (reading: standard pre-norm Llama/Qwen-style layer;
# tensors are rounded to bf16 at the same boundaries as the CUDA path)
# ---------------------------------------------------------------------------
class OracleKV:
    """Contiguous per-request K/V history, float64 holding bf16-representable values."""

    def __init__(self, n_layers: int, n_kv_heads: int, head_dim: int):
        self.n_layers = n_layers
        self.hkv = n_kv_heads
        self.hd = head_dim
        self.k = {}  # (layer, request) -> [L][Hkv][hd]
        self.v = {}

    def length(self, layer: int, req: int) -> int:
        a = self.k.get((layer, req))
        return 0 if a is None else a.shape[0]

    def set(self, layer, req, K, V):
        self.k[(layer, req)] = np.asarray(K, dtype=F64)
        self.v[(layer, req)] = np.asarray(V, dtype=F64)

    def append(self, layer, req, k_new, v_new):
        empty = np.zeros((0, self.hkv, self.hd))
        self.k[(layer, req)] = np.concatenate([self.k.get((layer, req), empty), k_new], axis=0)
        self.v[(layer, req)] = np.concatenate([self.v.get((layer, req), empty), v_new], axis=0)


def _keep(x):
    """No rounding: the value is carried at (more than) fp32 precision."""
    return np.asarray(x, dtype=F64)


def layer_forward(h, w, shape, kv: OracleKV, layer: int, requests, pos0, act32: bool = False) -> np.ndarray:
    """One pre-norm decoder layer over a batch of requests.

    h: [T][d]; w: dict of float64 weights (see synth.layer_weights);
    requests: list of (request id, number of query tokens) in token order;
    pos0[i]: absolute position of request i's first query token, which must
    equal the request's current cache length (K/V of new tokens are appended
    to the cache before attention, so cached and new tokens are one sequence).

      x1 = R(rms(h, g1));      qkv = R(x1 Wqkv^T)
      [Qwen3 only, w has q_norm/k_norm: q, k = R(rms_head(q, gq)), R(rms_head(k, gk)),
       the RMSNorm of every head row of head_dim values]
      q = R(rope(q));  k = bf16(rope(k));  v = bf16(v);  append k, v to the cache
      att = R(attention(q, K, V));       h1 = R(h + att Wo^T)
      x2 = R(rms(h1, g2));     gu = R(x2 Wgu^T)
      a = R(silu(g) * u);      h2 = R(h1 + a Wd^T)

    R is the rounding of the activations between steps: bf16 by default.  With
    act32 -- the mixed-precision mitigation that the TML-digest names in section 2
    and again in section 6 (weights stay stored in 16 bits, activations are fp32)
    -- R is the identity: the oracle carries every activation exactly and the
    CUDA path carries it in fp32.  The KV cache holds bf16 in both cases (k and
    v are rounded when they are stored; reading: the cache is stored state, like
    the weights).
    """
    R = _keep if act32 else round_bf16
    h = np.asarray(h, dtype=F64)
    Hq, Hkv, hd = shape.n_q_heads, shape.n_kv_heads, shape.head_dim
    F = shape.ffn_dim
    x1 = R(rmsnorm(h, w["attn_norm"], shape.rms_eps))
    qkv = R(gemm(x1, w["w_qkv"]))
    T = h.shape[0]
    q = qkv[:, :Hq * hd].reshape(T, Hq, hd)
    k = qkv[:, Hq * hd:(Hq + Hkv) * hd].reshape(T, Hkv, hd)
    v = qkv[:, (Hq + Hkv) * hd:].reshape(T, Hkv, hd)
    if "q_norm" in w:
        q = R(rmsnorm(q, w["q_norm"], shape.rms_eps))  # per head row (last axis = head_dim)
        k = R(rmsnorm(k, w["k_norm"], shape.rms_eps))
    att = np.zeros((T, Hq, hd), dtype=F64)
    t0 = 0
    scale = 1.0 / math.sqrt(hd)
    for (req, nq), p0 in zip(requests, pos0):
        if kv.length(layer, req) != p0:
            raise ValueError("request %r: cache holds %d tokens, first query at %d"
                             % (req, kv.length(layer, req), p0))
        pos = np.arange(p0, p0 + nq)
        qr = R(rope(q[t0:t0 + nq], pos, shape.rope_theta))
        kr = round_bf16(rope(k[t0:t0 + nq], pos, shape.rope_theta))
        kv.append(layer, req, kr, round_bf16(v[t0:t0 + nq]))
        att[t0:t0 + nq] = attention(qr, kv.k[(layer, req)], kv.v[(layer, req)], pos, scale)
        t0 += nq
    att = R(att).reshape(T, Hq * hd)
    h1 = R(h + gemm(att, w["w_o"]))
    x2 = R(rmsnorm(h1, w["ffn_norm"], shape.rms_eps))
    gu = R(gemm(x2, w["w_gate_up"]))
    a = R(swiglu(gu[:, :F], gu[:, F:]))
    return R(h1 + gemm(a, w["w_down"]))


def model_forward(ids, emb, layers, final_norm, lm_head, shape, kv: OracleKV, requests, pos0, act32: bool = False):
    """Embedding gather -> decoder layers -> final RMSNorm -> lm-head logits.

    Returns float32-rounded logits [T][V] (the lm-head output is kept in fp32).
    act32: activations carried without rounding (see layer_forward).
    """
    h = np.asarray(emb, dtype=F64)[np.asarray(ids, dtype=np.int64)]
    for i, w in enumerate(layers):
        h = layer_forward(h, w, shape, kv, i, requests, pos0, act32=act32)
    xf = (_keep if act32 else round_bf16)(rmsnorm(h, final_norm, shape.rms_eps))
    return round_f32(gemm(xf, lm_head))
