"""Pins of the float64 oracle against things other than itself.

Each check is a closed form, a value printed on the pages (tests/golden), an
invariant of the mathematics, or a brute force written here independently of
the oracle (pure-Python loops over Python ints/floats).  Each is chosen so that
a plausible slip in the oracle (a dropped term, a wrong sign, axis or index, a
transposed operand, eps outside the root, a swapped RoPE pairing) fails it.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- bf16 rounding
def test_round_bf16_matches_torch_conversion():
    x = torch.randn(20000, generator=torch.Generator().manual_seed(3)) * 37.0
    x = torch.cat([x, torch.tensor([0.0, -0.0, 1e-39, -3e-40, 1.0, 255.5, 1e30])])
    ref = x.to(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.round_bf16(x.to(torch.float64).numpy())
    assert np.array_equal(ref, got)


def test_round_bf16_ties_to_even():
    # bf16 spacing at 1 is 2**-7.  1 + 2**-8 is a tie between 1 (even) and 1 + 2**-7 (odd).
    assert oracle.round_bf16(1.0 + 2.0 ** -8) == 1.0
    # 1 + 3*2**-8 is a tie between 1 + 2**-7 (odd) and 1 + 2**-6 (even).
    assert oracle.round_bf16(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6
    assert oracle.round_bf16(-(1.0 + 3 * 2.0 ** -8)) == -(1.0 + 2.0 ** -6)
    assert oracle.round_bf16(1.0 + 2.0 ** -8 + 2.0 ** -20) == 1.0 + 2.0 ** -7


# ---------------------------------------------------------------- RMSNorm
@pytest.mark.parametrize("c,eps,d", [(1.0, 1.0, 8), (2.5, 1e-5, 512), (-3.0, 0.25, 4096), (1e-3, 1e-5, 64)])
def test_rmsnorm_constant_row_closed_form(c, eps, d):
    # constant row c: mean square is c^2, so y_j = c / sqrt(c^2 + eps) * gamma_j
    gamma = np.linspace(0.5, 1.5, d)
    y = oracle.rmsnorm(np.full((1, d), c), gamma, eps)
    expect = np.array([c / math.sqrt(c * c + eps) * g for g in gamma])
    assert np.allclose(y[0], expect, rtol=1e-14, atol=0)


def test_rmsnorm_unit_rms_rows_independent():
    rng = np.random.default_rng(0)
    x = rng.normal(size=(6, 100)) * np.array([1e-3, 1, 10, 1e3, 0.5, 7])[:, None]
    y = oracle.rmsnorm(x, np.ones(100), 0.0)
    # gamma = 1, eps = 0: every output row has root-mean-square exactly 1
    for r in range(6):
        assert math.isclose(math.sqrt(sum(v * v for v in y[r]) / 100), 1.0, rel_tol=1e-13)
    # gamma = 1, eps > 0: mean square of the output is ms / (ms + eps)
    eps = 0.3
    y = oracle.rmsnorm(x, np.ones(100), eps)
    for r in range(6):
        ms = sum(v * v for v in x[r]) / 100
        assert math.isclose(sum(v * v for v in y[r]) / 100, ms / (ms + eps), rel_tol=1e-12)
    # each row depends on that row only
    y_all = oracle.rmsnorm(x, np.arange(100) / 50.0, 1e-5)
    for r in range(6):
        assert np.array_equal(y_all[r], oracle.rmsnorm(x[r:r + 1], np.arange(100) / 50.0, 1e-5)[0])


def test_rmsnorm_scale_invariant():
    rng = np.random.default_rng(1)
    x = rng.normal(size=(3, 64))
    g = rng.normal(size=64)
    assert np.allclose(oracle.rmsnorm(4.0 * x, g, 0.0), oracle.rmsnorm(x, g, 0.0), rtol=1e-14, atol=0)
    assert np.allclose(oracle.rmsnorm(-x, g, 0.0), -oracle.rmsnorm(x, g, 0.0), rtol=1e-14, atol=0)


# ---------------------------------------------------------------- GEMM
def _int_matmul_brute(A, W):
    M, K = len(A), len(A[0])
    N = len(W)
    return [[sum(A[i][k] * W[j][k] for k in range(K)) for j in range(N)] for i in range(M)]


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (3, 5, 7), (16, 9, 33), (2, 13, 512)])
def test_gemm_small_int_bruteforce_exact(M, N, K):
    A = synth.small_ints((M, K), seed=M * 100 + K)
    W = synth.small_ints((N, K), seed=N * 100 + K + 1)
    Ai = [[int(v) for v in row] for row in A.to(torch.int64).tolist()]
    Wi = [[int(v) for v in row] for row in W.to(torch.int64).tolist()]
    got = oracle.gemm(A.double().numpy(), W.double().numpy())
    assert got.shape == (M, N)
    assert got.tolist() == [[float(v) for v in row] for row in _int_matmul_brute(Ai, Wi)]


def test_gemm_one_hot_rows_select_columns():
    rng = np.random.default_rng(2)
    A = rng.normal(size=(4, 6))
    W = np.zeros((3, 6))
    W[0, 5] = 1.0
    W[1, 0] = 1.0
    W[2, 2] = -2.0
    C = oracle.gemm(A, W)
    assert np.array_equal(C[:, 0], A[:, 5])
    assert np.array_equal(C[:, 1], A[:, 0])
    assert np.array_equal(C[:, 2], -2.0 * A[:, 2])


# ---------------------------------------------------------------- RoPE
def test_rope_hand_example_rotate_half_pairing():
    # hd = 4, theta = 10000: f = [1, 0.01].  x = e0 at position 1 rotates within the pair (0, 2).
    x = np.array([[[1.0, 0.0, 0.0, 0.0]]])
    y = oracle.rope(x, [1], 10000.0)[0, 0]
    assert np.allclose(y, [math.cos(1.0), 0.0, math.sin(1.0), 0.0], atol=1e-15)
    x = np.array([[[0.0, 1.0, 0.0, 0.0]]])
    y = oracle.rope(x, [3], 10000.0)[0, 0]
    assert np.allclose(y, [0.0, math.cos(0.03), 0.0, math.sin(0.03)], atol=1e-15)
    x = np.array([[[0.0, 0.0, 1.0, 0.0]]])
    y = oracle.rope(x, [1], 10000.0)[0, 0]
    assert np.allclose(y, [-math.sin(1.0), 0.0, math.cos(1.0), 0.0], atol=1e-15)


def test_rope_position_zero_identity_and_norms():
    rng = np.random.default_rng(4)
    x = rng.normal(size=(5, 3, 64))
    assert np.array_equal(oracle.rope(x[:1], [0], 500000.0), x[:1])
    y = oracle.rope(x, np.array([0, 1, 17, 300, 32767]), 500000.0)
    n_in = x[..., :32] ** 2 + x[..., 32:] ** 2
    n_out = y[..., :32] ** 2 + y[..., 32:] ** 2
    assert np.allclose(n_in, n_out, rtol=1e-12)


def test_rope_relative_position_property():
    rng = np.random.default_rng(5)
    q = rng.normal(size=(1, 1, 128))
    k = rng.normal(size=(1, 1, 128))
    dots = []
    for m, n in [(10, 3), (110, 103), (5007, 5000)]:
        a = oracle.rope(q, [m], 1e6)[0, 0]
        b = oracle.rope(k, [n], 1e6)[0, 0]
        dots.append(float(a @ b))
    assert np.allclose(dots, dots[0], rtol=1e-9)


# ---------------------------------------------------------------- attention
def _attn_brute(q, K, V, n, scale):
    """Pure-Python softmax attention of one query vector over the first n keys."""
    z = [sum(qi * ki for qi, ki in zip(q, K[j])) * scale for j in range(n)]
    mx = max(z)
    e = [math.exp(v - mx) for v in z]
    s = sum(e)
    return [sum(e[j] * V[j][d] for j in range(n)) / s for d in range(len(V[0]))]


def test_attention_identical_keys_gives_mean_of_values():
    rng = np.random.default_rng(6)
    L, hd = 300, 64
    K = np.tile(rng.normal(size=(1, 1, hd)), (L, 1, 1))
    V = rng.normal(size=(L, 1, hd))
    q = rng.normal(size=(1, 4, hd))
    out = oracle.attention(q, K, V, [L - 1], 1 / 8)
    for h in range(4):
        assert np.allclose(out[0, h], V[:, 0].mean(axis=0), rtol=1e-12, atol=1e-14)


def test_attention_single_key_and_identical_values():
    rng = np.random.default_rng(7)
    K = rng.normal(size=(9, 2, 16))
    V = rng.normal(size=(9, 2, 16))
    q = rng.normal(size=(3, 4, 16))
    out = oracle.attention(q, K, V, [0, 0, 0], 0.25)
    for h in range(4):
        assert np.array_equal(out[:, h], np.repeat(V[0:1, h // 2], 3, axis=0))
    Vc = np.tile(V[:1], (9, 1, 1))
    out = oracle.attention(q, K, Vc, [8, 5, 2], 0.25)
    for h in range(4):
        assert np.allclose(out[:, h], np.repeat(Vc[0:1, h // 2], 3, axis=0), rtol=1e-13)


def test_attention_two_keys_closed_form_and_dominant_score():
    K = np.array([[[1.0, 0.0]], [[0.0, 1.0]]])
    V = np.array([[[2.0, -1.0]], [[5.0, 3.0]]])
    q = np.array([[[0.7, -0.4]]])
    s = 0.9
    p0 = 1.0 / (1.0 + math.exp((-0.4 - 0.7) * s))
    expect = [p0 * 2.0 + (1 - p0) * 5.0, p0 * -1.0 + (1 - p0) * 3.0]
    assert np.allclose(oracle.attention(q, K, V, [1], s)[0, 0], expect, rtol=1e-14)
    q = np.array([[[200.0, 0.0]]])
    assert np.allclose(oracle.attention(q, K, V, [1], 1.0)[0, 0], V[0, 0], rtol=0, atol=1e-80)


def test_attention_causal_and_gqa_grouping():
    rng = np.random.default_rng(8)
    L, Hkv, G, hd = 12, 3, 2, 8
    K = rng.normal(size=(L, Hkv, hd))
    V = rng.normal(size=(L, Hkv, hd))
    q = rng.normal(size=(L, Hkv * G, hd))
    pos = np.arange(L)
    out = oracle.attention(q, K, V, pos, 0.3)
    K2, V2 = K.copy(), V.copy()
    K2[7:] = rng.normal(size=K2[7:].shape)
    V2[7:] = 100.0
    out2 = oracle.attention(q, K2, V2, pos, 0.3)
    assert np.array_equal(out[:7], out2[:7])  # queries at positions < 7 never see keys >= 7
    assert not np.allclose(out[7:], out2[7:])
    # head h reads kv head h // G
    Vg = np.zeros((L, Hkv, hd))
    for g in range(Hkv):
        Vg[:, g, :] = g + 1.0
    outg = oracle.attention(q, K, Vg, pos, 0.3)
    for h in range(Hkv * G):
        assert np.allclose(outg[:, h], h // G + 1.0, rtol=1e-13)


def test_attention_bruteforce_tiny():
    rng = np.random.default_rng(9)
    for L in (1, 2, 5, 20):
        K = rng.normal(size=(L, 2, 6))
        V = rng.normal(size=(L, 2, 6))
        q = rng.normal(size=(L, 4, 6))
        pos = np.arange(L)
        out = oracle.attention(q, K, V, pos, 0.4)
        for t in range(L):
            for h in range(4):
                ref = _attn_brute(q[t, h].tolist(), K[:, h // 2].tolist(), V[:, h // 2].tolist(), t + 1, 0.4)
                assert np.allclose(out[t, h], ref, rtol=1e-12, atol=1e-14)


def test_gather_pages_follows_block_table():
    cache = np.arange(5 * 2 * 4 * 3, dtype=np.float64).reshape(5, 2, 4, 3)
    row = [3, 0, 4]
    got = oracle.gather_pages(cache, row, 10)
    for t in range(10):
        assert np.array_equal(got[t], cache[row[t // 4], :, t % 4, :])


# ---------------------------------------------------------------- split geometry / partials
def test_split_geometry_matches_page_examples():
    g = _golden("split_geometry.json")
    for case in g["fixed_split"]["cases"]:
        geo = oracle.split_geometry(case["kv_len"], g["fixed_split"]["split"])
        assert [a for a, _ in geo] == case["split_starts"]
        assert geo[-1][1] == case["last_valid"] == case["page_last_valid"] - 1
        qs = case["query_pos"] // g["fixed_split"]["split"]
        assert qs == case["query_split"]
    # the query at position 300 sees the same split 1 geometry in both contexts
    a = oracle.split_geometry(301, 256)
    assert a[1] == (256, 45)
    cv = g["cache_vs_new"]
    one_shot = [n for _, n in oracle.split_geometry(cv["cached"] + cv["new"], cv["block"])]
    assert one_shot == cv["one_shot_reduction_blocks"]
    assert one_shot != cv["separate_reduction_blocks"]
    assert sum(cv["separate_reduction_blocks"]) == cv["cached"] + cv["new"]


def _merge_exact(parts):
    """Log-sum-exp combination of (m, l, o) partials, pure Python."""
    M = max(m for m, _, _ in parts)
    den = sum(l * math.exp(m - M) for m, l, _ in parts)
    hd = len(parts[0][2])
    return [sum(o[d] * math.exp(m - M) for m, _, o in parts) / den for d in range(hd)]


def test_split_partials_recombine_to_attention():
    rng = np.random.default_rng(10)
    L, hd = 700, 16
    K = rng.normal(size=(L, 2, hd))
    V = rng.normal(size=(L, 2, hd))
    q = rng.normal(size=(hd,))
    for qp in (0, 255, 256, 511, 699):
        m, l, o = oracle.split_partials(q, K, V, qp, 1, 0.25)
        assert len(m) == qp // 256 + 1
        got = _merge_exact([(m[s], l[s], o[s].tolist()) for s in range(len(m))])
        ref = oracle.attention(q[None, None, :], K[:, 1:2], V[:, 1:2], [qp], 0.25)[0, 0]
        assert np.allclose(got, ref, rtol=1e-12, atol=1e-14)
        # each split state is the brute-force softmax numerator/denominator over its positions
        s = len(m) - 1
        lo = 256 * s
        z = [sum(a * b for a, b in zip(q.tolist(), K[j, 1].tolist())) * 0.25 for j in range(lo, qp + 1)]
        assert math.isclose(m[s], max(z), rel_tol=1e-13)
        assert math.isclose(l[s], sum(math.exp(v - max(z)) for v in z), rel_tol=1e-12)


# ---------------------------------------------------------------- pointwise
def test_silu_swiglu_identities():
    assert oracle.silu(0.0) == 0.0
    assert math.isclose(float(oracle.silu(1.0)), 1.0 / (1.0 + math.exp(-1.0)), rel_tol=1e-15)
    x = np.linspace(-20, 20, 401)
    assert np.allclose(oracle.silu(x) - oracle.silu(-x), x, rtol=1e-13, atol=1e-13)
    assert np.allclose(oracle.silu(np.array([40.0, 60.0])), [40.0, 60.0], rtol=1e-15)
    g = np.array([0.5, -2.0, 3.0])
    u = np.array([2.0, 0.5, -1.0])
    ref = [gi / (1 + math.exp(-gi)) * ui for gi, ui in zip(g, u)]
    assert np.allclose(oracle.swiglu(g, u), ref, rtol=1e-15)


# ---------------------------------------------------------------- top-k / argmax
def _topk_brute(row, k):
    """Repeated selection of the largest remaining value, lowest index on ties."""
    left = list(enumerate(row))
    out = []
    for _ in range(k):
        best = None
        for i, v in left:
            if best is None or v > best[1] or (v == best[1] and i < best[0]):
                best = (i, v)
        out.append(best)
        left.remove(best)
    return [v for _, v in out], [i for i, _ in out]


def test_topk_bruteforce_with_ties():
    rng = np.random.default_rng(11)
    rows = np.round(rng.normal(size=(5, 300)), 1)  # many exact ties
    vals, idx = oracle.topk(rows, 20)
    for r in range(5):
        bv, bi = _topk_brute(rows[r].tolist(), 20)
        assert vals[r].tolist() == bv
        assert idx[r].tolist() == bi


def test_argmax_tie_example_from_page():
    g = _golden("tie_logits.json")
    r1 = np.array(g["run1"], dtype=np.float32)
    r2 = np.array(g["run2"], dtype=np.float32)
    assert r1[0] == r1[1] and format(int(r1.view(np.uint32)[0]), "08x") == g["float32_bits"]
    got = [int(oracle.argmax(r1.astype(np.float64))[0]), int(oracle.argmax(r2.astype(np.float64))[0])]
    assert got == g["expected_argmax_lowest_index"]
    # with the values kept in float64 the pair is distinct and the flip the page describes appears
    assert [int(oracle.argmax(np.array(g["run1"]))[0]), int(oracle.argmax(np.array(g["run2"]))[0])] == g["page_claim_argmax"]


# ---------------------------------------------------------------- layer / model composition
def _tiny_weights(shape, seed, zero=()):
    w = {k: v.double().numpy() for k, v in synth.layer_weights(shape, seed, std=0.05, gamma_std=0.1).items()}
    for k in zero:
        w[k] = np.zeros_like(w[k])
    return w


@pytest.mark.parametrize("act32", [False, True])
def test_layer_zero_projections_is_identity(act32):
    shape = synth.TINY_LAYER
    w = _tiny_weights(shape, 1, zero=("w_o", "w_down"))
    h = synth.normal((5, shape.d_model), 3).double().numpy()
    if act32:
        h = h * (1 + 2.0 ** -12)  # not bf16-representable: an activation rounding would show
    kv = oracle.OracleKV(1, shape.n_kv_heads, shape.head_dim)
    out = oracle.layer_forward(h, w, shape, kv, 0, [(0, 5)], [0], act32=act32)
    assert np.array_equal(out, h)
    assert kv.length(0, 0) == 5
    # the cache holds bf16 values in both variants
    assert np.array_equal(oracle.round_bf16(kv.k[(0, 0)]), kv.k[(0, 0)])
    assert np.array_equal(oracle.round_bf16(kv.v[(0, 0)]), kv.v[(0, 0)])


@pytest.mark.parametrize("act32", [False, True])
def test_layer_prefill_equals_token_by_token_and_requests_independent(act32):
    shape = synth.TINY_LAYER
    w = _tiny_weights(shape, 2)
    h = synth.normal((7, shape.d_model), 4).double().numpy()
    kv1 = oracle.OracleKV(1, shape.n_kv_heads, shape.head_dim)
    full = oracle.layer_forward(h, w, shape, kv1, 0, [(0, 7)], [0], act32=act32)
    kv2 = oracle.OracleKV(1, shape.n_kv_heads, shape.head_dim)
    rows = [oracle.layer_forward(h[t:t + 1], w, shape, kv2, 0, [(0, 1)], [t], act32=act32) for t in range(7)]
    # With bf16 activations the roundings absorb the float64 matmul's own
    # batch-dependent summation order, so the rows agree exactly; with act32 they
    # agree to float64 rounding.
    tol = 1e-12 if act32 else 0
    assert np.allclose(np.concatenate(rows), full, rtol=tol, atol=tol)
    # a second request in the same batch does not change the first one's rows
    kv3 = oracle.OracleKV(1, shape.n_kv_heads, shape.head_dim)
    h2 = np.concatenate([h, synth.normal((3, shape.d_model), 5).double().numpy()])
    both = oracle.layer_forward(h2, w, shape, kv3, 0, [(0, 7), (1, 3)], [0, 0], act32=act32)
    assert np.allclose(both[:7], full, rtol=tol, atol=tol)


def test_layer_act32_single_token_by_hand():
    # fp32-activation variant: nothing is rounded between the steps except the
    # cached k and v (bf16).  One token at position 0 attends only to itself, so
    # its attention output is its own bf16-rounded v.
    shape = synth.TINY_LAYER
    w = _tiny_weights(shape, 3)
    d, hd, Hq, Hkv, F = shape.d_model, shape.head_dim, shape.n_q_heads, shape.n_kv_heads, shape.ffn_dim
    h = synth.normal((1, d), 6).double().numpy()
    kv = oracle.OracleKV(1, Hkv, hd)
    out = oracle.layer_forward(h, w, shape, kv, 0, [(0, 1)], [0], act32=True)
    x1 = h / np.sqrt(np.mean(h * h) + shape.rms_eps) * w["attn_norm"]
    v = oracle.round_bf16(x1 @ w["w_qkv"][(Hq + Hkv) * hd:].T).reshape(Hkv, hd)
    att = np.concatenate([v[hh // (Hq // Hkv)] for hh in range(Hq)])
    h1 = h[0] + att @ w["w_o"].T
    x2 = h1 / np.sqrt(np.mean(h1 * h1) + shape.rms_eps) * w["ffn_norm"]
    g, u = x2 @ w["w_gate_up"][:F].T, x2 @ w["w_gate_up"][F:].T
    h2 = h1 + (g / (1 + np.exp(-g)) * u) @ w["w_down"].T
    assert np.allclose(out[0], h2, rtol=1e-12, atol=1e-12)
    assert np.array_equal(kv.v[(0, 0)][0], v)
    # the bf16 variant differs (it rounds between the steps)
    kv2 = oracle.OracleKV(1, Hkv, hd)
    assert not np.array_equal(oracle.layer_forward(h, w, shape, kv2, 0, [(0, 1)], [0]), out)


def test_layer_attention_branch_single_token():
    # One token at position 0 attends only to itself, so the attention output is its own v.
    shape = synth.TINY_LAYER
    w = _tiny_weights(shape, 3, zero=("w_down",))
    d, hd, Hq, Hkv = shape.d_model, shape.head_dim, shape.n_q_heads, shape.n_kv_heads
    h = synth.normal((1, d), 6).double().numpy()
    kv = oracle.OracleKV(1, Hkv, hd)
    out = oracle.layer_forward(h, w, shape, kv, 0, [(0, 1)], [0])
    x1 = oracle.round_bf16(h / np.sqrt(np.mean(h * h) + shape.rms_eps) * w["attn_norm"])
    v = oracle.round_bf16(x1 @ w["w_qkv"][(Hq + Hkv) * hd:].T).reshape(Hkv, hd)
    att = np.concatenate([v[hh // (Hq // Hkv)] for hh in range(Hq)])
    assert np.allclose(out[0], oracle.round_bf16(h[0] + att @ w["w_o"].T), rtol=0, atol=0)


def test_layer_qk_norm_branch_by_hand():
    # Qwen3-shaped layers normalise every q head row and every k head row (head_dim values each) with their
    # own RMSNorm weights before RoPE (reading: the pages never describe the layer; the standard Qwen3 block
    # is taken).  A new token at position P attends to P cached keys and to itself; with w_down = 0 the layer
    # output is R(h + att Wo^T).  The computation below is written element by element from that reading.
    # Each plausible slip in the oracle's branch -- the norm after RoPE, q_norm and k_norm swapped, one norm
    # over all heads of a token -- moves the result by more than 5% of the attention term.
    shape = synth.TINY_QK_LAYER
    w = _tiny_weights(shape, 4, zero=("w_down",))
    d, hd, Hq, Hkv = shape.d_model, shape.head_dim, shape.n_q_heads, shape.n_kv_heads
    G, eps, P = Hq // Hkv, shape.rms_eps, 5
    # widely spread head-norm weights, so that mixing dims i and i + hd/2 (RoPE) before or after them shows
    w["q_norm"] = synth.normal((hd,), 12, std=0.5, mean=1.0).double().numpy()
    w["k_norm"] = synth.normal((hd,), 13, std=0.5, mean=1.0).double().numpy()
    h = synth.normal((1, d), 9).double().numpy()
    K0 = synth.normal((P, Hkv, hd), 10).double().numpy()
    V0 = synth.normal((P, Hkv, hd), 11).double().numpy()
    kv = oracle.OracleKV(1, Hkv, hd)
    kv.set(0, 0, K0, V0)
    out = oracle.layer_forward(h, w, shape, kv, 0, [(0, 1)], [P])[0]
    R = oracle.round_bf16  # pinned on its own above

    def norm_row(row, g):
        ms = sum(float(v) * float(v) for v in row) / len(row)
        r = 1.0 / math.sqrt(ms + eps)
        return np.array([float(v) * r * float(gi) for v, gi in zip(row, g)])

    def rot(vec, pos):
        half = hd // 2
        o = np.empty(hd)
        for i in range(half):
            ang = pos * shape.rope_theta ** (-2.0 * i / hd)
            c, s = math.cos(ang), math.sin(ang)
            o[i] = vec[i] * c - vec[i + half] * s
            o[i + half] = vec[i + half] * c + vec[i] * s
        return o

    def by_hand(variant):
        x1 = R(norm_row(h[0], w["attn_norm"]))
        qkv = R(x1 @ w["w_qkv"].T)
        q = qkv[:Hq * hd].reshape(Hq, hd)
        k = qkv[Hq * hd:(Hq + Hkv) * hd].reshape(Hkv, hd)
        v = R(qkv[(Hq + Hkv) * hd:].reshape(Hkv, hd))
        gq, gk = (w["k_norm"], w["q_norm"]) if variant == "swapped" else (w["q_norm"], w["k_norm"])
        if variant == "after_rope":
            qr = R(np.array([norm_row(rot(r, P), gq) for r in q]))
            kr = R(np.array([norm_row(rot(r, P), gk) for r in k]))
        else:
            if variant == "across_heads":
                qn = R(norm_row(q.ravel(), np.tile(gq, Hq))).reshape(Hq, hd)
                kn = R(norm_row(k.ravel(), np.tile(gk, Hkv))).reshape(Hkv, hd)
            else:
                qn = R(np.array([norm_row(r, gq) for r in q]))
                kn = R(np.array([norm_row(r, gk) for r in k]))
            qr = R(np.array([rot(r, P) for r in qn]))
            kr = R(np.array([rot(r, P) for r in kn]))
        att = np.empty((Hq, hd))
        for hh in range(Hq):
            g = hh // G
            keys = [K0[j, g] for j in range(P)] + [kr[g]]
            vals = [V0[j, g] for j in range(P)] + [v[g]]
            z = [sum(float(x) * float(y) for x, y in zip(qr[hh], key)) / math.sqrt(hd) for key in keys]
            e = [math.exp(t - max(z)) for t in z]
            att[hh] = sum(ej * vj for ej, vj in zip(e, vals)) / sum(e)
        return R(h[0] + R(att).ravel() @ w["w_o"].T)

    ref = by_hand("reading")
    term = np.max(np.abs(ref - h[0]))  # size of the attention term
    assert np.max(np.abs(out - ref)) <= 1e-3 * term
    assert np.array_equal(oracle.round_bf16(kv.k[(0, 0)][P]), kv.k[(0, 0)][P])  # the new key is cached as bf16
    for slip in ("after_rope", "swapped", "across_heads"):
        assert np.max(np.abs(by_hand(slip) - ref)) >= 2e-2 * term, slip


def test_model_without_layers_is_norm_then_head():
    shape = synth.TINY_LAYER
    V = 50
    emb = synth.normal((V, shape.d_model), 7).double().numpy()
    head = synth.normal((V, shape.d_model), 8, std=0.05).double().numpy()
    g = np.ones(shape.d_model)
    kv = oracle.OracleKV(0, shape.n_kv_heads, shape.head_dim)
    ids = [3, 49, 3]
    logits = oracle.model_forward(ids, emb, [], g, head, shape, kv, [(0, 3)], [0])
    assert np.array_equal(logits[0], logits[2])
    x = emb[49] / np.sqrt(np.mean(emb[49] ** 2) + shape.rms_eps)
    assert np.allclose(logits[1], oracle.round_bf16(x) @ head.T, rtol=1e-6)
    # fp32 activations: the normalised row is not rounded before the head
    l32 = oracle.model_forward(ids, emb, [], g, head, shape, kv, [(0, 3)], [0], act32=True)
    assert np.allclose(l32[1], x @ head.T, rtol=1e-6)
    assert not np.allclose(l32[1], oracle.round_bf16(x) @ head.T, rtol=1e-6, atol=0)


def test_three_bf16_terms_hold_an_fp32_value_exactly():
    # The reading behind the fp32-activation GEMM: an fp32 value a is the exact
    # sum of three bf16 values, hi = bf16(a), mid = bf16(a - hi),
    # lo = bf16(a - hi - mid), the differences taken in fp32 (exact there);
    # each bf16 x bf16 product is exact in fp32.  Checked over random values and
    # the binade edges of the range the activations use.
    rng = np.random.default_rng(0)
    a = np.concatenate([rng.standard_normal(200000) * 10.0 ** rng.integers(-30, 30, 200000),
                        np.float32(2.0) ** np.arange(-100, 100),
                        np.nextafter(np.float32(2.0) ** np.arange(-100, 100), np.float32(0)).astype(np.float64)])
    a = a.astype(np.float32)
    hi = oracle.round_bf16(a.astype(np.float64)).astype(np.float32)
    r1 = a - hi
    mid = oracle.round_bf16(r1.astype(np.float64)).astype(np.float32)
    r2 = r1 - mid
    lo = oracle.round_bf16(r2.astype(np.float64)).astype(np.float32)
    total = hi.astype(np.float64) + mid.astype(np.float64) + lo.astype(np.float64)
    # exact wherever the third term stays in bf16's normal range (|a| >= 2**-110);
    # below that the remainder is rounded to bf16's subnormal spacing 2**-133
    big = np.abs(a) >= 2.0 ** -110
    assert big.sum() > 0.99 * a.size
    assert np.array_equal(r2[big], lo[big])  # the third term is already a bf16 value
    assert np.array_equal(total[big], a[big].astype(np.float64))
    assert np.all(np.abs(total - a.astype(np.float64)) <= 2.0 ** -134)
    w = oracle.round_bf16(rng.standard_normal(hi.size)).astype(np.float32)
    for t in (hi, mid, lo):
        assert np.array_equal((t * w).astype(np.float64), t.astype(np.float64) * w.astype(np.float64))


def _sum_in_order(terms, dtype, order):
    """Sum terms [rows][K] along K in dtype, in one of three orders: "serial"
    (one running sum, k ascending), "pairwise" (a balanced tree: neighbours
    added level by level), or an int w (blocks of w consecutive terms summed
    serially, then the block sums added serially)."""
    t = np.asarray(terms, dtype=dtype)
    if order == "serial":
        acc = np.zeros(t.shape[0], dtype=dtype)
        for k in range(t.shape[1]):
            acc = (acc + t[:, k]).astype(dtype)
        return acc
    if order == "pairwise":
        while t.shape[1] > 1:
            if t.shape[1] % 2:
                t = np.concatenate([t, np.zeros((t.shape[0], 1), dtype=dtype)], axis=1)
            t = (t[:, 0::2] + t[:, 1::2]).astype(dtype)
        return t[:, 0]
    blocks = np.stack([_sum_in_order(t[:, k0:k0 + order], dtype, "serial")
                       for k0 in range(0, t.shape[1], order)], axis=1)
    return _sum_in_order(blocks, dtype, "serial")


def test_reduction_order_changes_fp32_sums_but_not_the_float64_oracle():
    # The mechanism behind the method (zhaixingw.cn BlockLock post, its float32 reproduction of the tiling
    # effect; devpress digest, section 2.1 on non-associative floating-point addition): one dot product
    # summed in different orders -- a running sum, a pairwise tree, blocks of the tile widths the GEMM uses
    # (32 .. 256 columns, 16-term instruction steps) -- rounds differently in fp32.  In float64 all the
    # orders agree to float64 rounding, which is why the oracle's sums can stand for the exact ones.
    rng = np.random.default_rng(11)
    K = 4096
    a = rng.standard_normal((16, K)).astype(np.float32)
    b = (rng.standard_normal((16, K)) * 0.02).astype(np.float32)
    terms = a.astype(np.float64) * b.astype(np.float64)  # every fp32 x fp32 product is exact in float64
    exact = np.array([oracle.gemm(a[r:r + 1].astype(np.float64), b[r:r + 1].astype(np.float64))[0, 0]
                      for r in range(a.shape[0])])
    scale = np.max(np.abs(exact))
    orders = ["serial", "pairwise", 16, 32, 64, 256]
    s32 = [_sum_in_order(terms.astype(np.float32), np.float32, o).astype(np.float64) for o in orders]
    s64 = [_sum_in_order(terms, np.float64, o) for o in orders]
    spread32 = max(np.max(np.abs(x - s32[0])) for x in s32[1:])
    spread64 = max(np.max(np.abs(x - s64[0])) for x in s64[1:])
    assert 0 < spread32 <= 1e-4 * scale  # fp32: a real, small difference between orders
    assert spread64 <= 1e-12 * scale  # float64: the order does not matter at any tolerance used
    for x in s64:
        assert np.max(np.abs(x - exact)) <= 1e-12 * scale
    # the orders really are different ones: a running sum and a tree disagree on some rows in fp32
    assert np.any(s32[0] != s32[1])
