"""fp32-activation variant (bf16 weights, fp32 activations, bf16 KV cache): the
GEMM over three bf16 planes of the fp32 activations, fp32 queries in attention,
the layer and the model; oracle parity and the same bitwise batch invariance as
the bf16 path."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.helpers import bits_equal, cuda, f64, max_rel_err
from tests.test_attention_gpu import Requests, random_kv
from tests.test_layer_gpu import LayerRig

pytestmark = pytest.mark.gpu
bi = pytest.importorskip("invariant_deterministic_02_gb300")
from invariant_deterministic_02_gb300.model import BiModel, ModelShape  # noqa: E402

F32 = torch.float32

# Tolerances of the fp32-activation path, against the float64 oracle:
# GEMM: the three plane products are exact; the tensor cores add each
#   instruction's products into the fp32 accumulator with an error of up to one
#   unit in the last place of the running sum (the measured maximum error grows
#   linearly with K, as truncation does), so after n = 3*ceil(K/16) instructions
#   the error is below n * 2^-23 of the sums' size: 9.2e-5 at K = 4096, 2.7e-4
#   at K = 12288 (measured maxima: 4.1e-5 and 1.2e-4).  Activations rounded to
#   bf16 first are off by ~2^-9 per element, several 1e-3 on C.


def tol_gemm32(K):
    return 3 * -(-K // 16) * 2.0 ** -23


# Attention: a score is an fp32 dot product of head_dim terms of size ~1 (sums
#   ~10), rounded to ~1e-5 absolute, which enters the softmax weights as a
#   relative error of that order.
TOL_ATTN32 = 1e-4
# Layer and model: the errors above, plus the K/V elements whose fp32 value lies
#   within fp32 noise of a bf16 rounding tie and so lands one bf16 step (2^-8
#   relative) away from the oracle's in the cache; after the O projection such
#   an element moves a layer output by ~1e-4 of its rms.
TOL_LAYER32 = 1e-3


def gemm32(A, W, R=None, mode=bi.INVARIANT, tr=-1, tc=0):
    C = torch.empty((A.shape[0], W.shape[0]), dtype=F32, device="cuda")
    bi.bi_gemm_f32a(A, W, C, residual=R, mode=mode, target_row=tr, target_count=tc)
    torch.cuda.synchronize()
    return C


# ---------------------------------------------------------------- GEMM with fp32 A
@pytest.mark.parametrize("M,K", [(1, 256), (70, 1024), (200, 512)])
def test_one_hot_weights_reproduce_fp32_activations_exactly(M, K):
    # C[:, j] = A[:, k_j]: every other product is an exact zero, so hi + mid + lo
    # must rebuild the fp32 value bit for bit (a dropped or misplaced plane shows).
    A = synth.normal((M, K), 7 + M, dtype=F32)
    assert not torch.equal(A, A.to(torch.bfloat16).to(F32))  # not bf16 values
    W = torch.zeros((64, K), dtype=torch.bfloat16)
    for j in range(64):
        W[j, (j * 7 + 3) % K] = 1.0
    C = gemm32(cuda(A), cuda(W))
    for j in range(64):
        assert bits_equal(C[:, j].cpu(), A[:, (j * 7 + 3) % K]), j


@pytest.mark.parametrize("M,N,K", [(3, 64, 256), (128, 136, 256), (300, 264, 256)])
def test_fixed_point_activations_exact(M, N, K):
    # A = integer + j/256 (12 significant bits: not bf16 values), W small integers:
    # every partial sum is a multiple of 2^-8 below 2^13, exact in fp32 in any order.
    ints = synth.small_ints((M, K), 30 + M, dtype=F32)
    frac = synth.small_ints((M, K), 31 + M, lo=0, hi=255, dtype=F32) / 256.0
    A = ints + frac
    W = synth.small_ints((N, K), 32 + N, lo=-3, hi=3)
    C = gemm32(cuda(A), cuda(W))
    assert np.array_equal(f64(C), oracle.gemm(f64(A), f64(W)))


@pytest.mark.parametrize("M,N,K", [(1, 512, 512), (64, 4096, 4096), (97, 1024, 4096), (300, 264, 520),
                                   (16, 4096, 12288)])
def test_random_parity_and_gain_over_bf16_activations(M, N, K):
    A = synth.normal((M, K), 40 + M, dtype=F32)
    W = synth.normal((N, K), 41 + N, std=0.02)
    exact = oracle.gemm(f64(A), f64(W))
    C = gemm32(cuda(A), cuda(W))
    err32 = max_rel_err(f64(C), exact)
    assert err32 <= tol_gemm32(K)
    # the same product with the activations rounded to bf16 first is far off
    Cb = torch.empty((M, N), dtype=F32, device="cuda")
    bi.bi_gemm(cuda(A).to(torch.bfloat16), cuda(W), Cb)
    torch.cuda.synchronize()
    assert max_rel_err(f64(Cb), exact) > 20 * err32


def test_fp32_residual_in_place():
    M, N, K = 70, 320, 640
    A = synth.normal((M, K), 51, dtype=F32)
    W = synth.normal((N, K), 52, std=0.02)
    R = synth.normal((M, N), 53, dtype=F32)
    C = gemm32(cuda(A), cuda(W), R=cuda(R))
    assert max_rel_err(f64(C), oracle.gemm(f64(A), f64(W)) + f64(R)) <= tol_gemm32(K)
    Rc = cuda(R)
    bi.bi_gemm_f32a(cuda(A), cuda(W), Rc, residual=Rc)
    torch.cuda.synchronize()
    assert bits_equal(Rc, C)


def test_row0_bitwise_across_M_and_modes():
    N, K = 4096, 4096
    W = synth.normal_device((N, K), 61, std=0.02)
    target = synth.normal((1, K), 62, dtype=F32)
    ref = refk = None
    for M in [1, 3, 16, 64, 97, 128, 129, 300, 1024]:
        A = synth.normal_device((M, K), 2000 + M, dtype=F32)
        A[0] = cuda(target)[0]
        row = gemm32(A, W)[0:1].clone()
        rowk = gemm32(A, W, mode=bi.INVARIANT_KSPLIT)[0:1].clone()
        if ref is None:
            ref, refk = row, rowk
        assert bits_equal(row, ref), "row 0 changed at M=%d" % M
        assert bits_equal(rowk, refk), "ksplit row 0 changed at M=%d" % M
        if M in (64, 300):
            # PROTECTED keeps the target row's bits, FAST stays within tolerance
            rowp = gemm32(A, W, mode=bi.PROTECTED, tr=0, tc=1)[0:1]
            assert bits_equal(rowp, ref), M
            Cf = gemm32(A, W, mode=bi.FAST)
            assert max_rel_err(f64(Cf[:4]), oracle.gemm(f64(A[:4]), f64(W))) <= tol_gemm32(K)
    assert max_rel_err(f64(ref), oracle.gemm(f64(target), f64(W))) <= tol_gemm32(K)
    assert max_rel_err(f64(refk), oracle.gemm(f64(target), f64(W))) <= tol_gemm32(K)


# ---------------------------------------------------------------- attention with fp32 q
def test_decode_fp32_query_parity():
    hq, hkv, hd = 32, 8, 128
    lens = synth.loguniform_ints(8, 64, 4096, 71)
    kvs = [random_kv(int(n), hkv, hd, 700 + 2 * b) for b, n in enumerate(lens)]
    req = Requests(kvs, hq, hkv, hd, seed=72)
    q = cuda(synth.normal((8, hq, hd), 73, dtype=F32))
    kl = cuda(torch.tensor(req.lens, dtype=torch.int32))
    out = torch.empty_like(q)
    bi.bi_decode_attention(q, req.kc, req.vc, req.bt, kl, req.dims, out)
    torch.cuda.synchronize()
    assert out.dtype == F32
    for b in range(8):
        K, V = req.kvs[b]
        ref = oracle.attention(f64(q[b:b + 1].cpu()), f64(K), f64(V), [req.lens[b] - 1], req.dims.scale)[0]
        assert max_rel_err(f64(out[b]), ref) <= TOL_ATTN32, b


def test_prefill_chunks_equal_decode_bitwise_fp32_query():
    hq, hkv, hd, L = 32, 8, 128, 1024
    K, V = random_kv(L, hkv, hd, 81)
    q = cuda(synth.normal((L, hq, hd), 82, dtype=F32))
    req = Requests([(K, V)], hq, hkv, hd, seed=81)

    def prefill(qc, c):
        out = torch.empty_like(qc)
        bi.bi_prefill_attention(qc, req.kc, req.vc, req.bt, cuda(torch.tensor([0, qc.shape[0]], dtype=torch.int32)),
                                cuda(torch.tensor([c], dtype=torch.int32)), req.dims, out)
        torch.cuda.synchronize()
        return out

    one = prefill(q, 0)
    chunks = torch.cat([prefill(q[c:c + 256], c) for c in range(0, L, 256)])
    assert bits_equal(one, chunks)
    for p in [0, 255, 256, 700, 1023]:
        out = torch.empty_like(q[p:p + 1])
        bi.bi_decode_attention(q[p:p + 1].contiguous(), req.kc, req.vc, req.bt,
                               cuda(torch.tensor([p + 1], dtype=torch.int32)), req.dims, out)
        torch.cuda.synchronize()
        assert bits_equal(out, one[p:p + 1]), p
        ref = oracle.attention(f64(q[p:p + 1].cpu()), f64(K), f64(V), [p], req.dims.scale)[0]
        assert max_rel_err(f64(one[p]), ref) <= TOL_ATTN32, p


# ---------------------------------------------------------------- layer
@pytest.mark.parametrize("shape", [synth.TINY_LAYER, synth.TINY_QK_LAYER], ids=["plain", "qk_norm"])
def test_tiny_layer_parity(shape):
    rig = LayerRig(shape, 3, act_f32=True)
    rig.add_request(0, 0, 10, 64)
    rig.add_request(1, 0, 12, 64)
    h = synth.normal((42, shape.d_model), 5, dtype=F32)
    items = [(0, 37, 0), (1, 5, 0)]
    out = rig.run(cuda(h), items)
    assert out.dtype == F32
    kv = oracle.OracleKV(1, shape.n_kv_heads, shape.head_dim)
    w = {k: f64(v) for k, v in rig.w_host.items()}
    ref = oracle.layer_forward(f64(h), w, shape, kv, 0, [(0, 37), (1, 5)], [0, 0], act32=True)
    assert max_rel_err(f64(out), ref) <= TOL_LAYER32
    h2 = synth.normal((2, shape.d_model), 6, dtype=F32)
    out2 = rig.run(cuda(h2), [(0, 1, 37), (1, 1, 5)])
    ref2 = oracle.layer_forward(f64(h2), w, shape, kv, 0, [(0, 1), (1, 1)], [37, 5], act32=True)
    assert max_rel_err(f64(out2), ref2) <= TOL_LAYER32


@pytest.mark.parametrize("B", [1, 16])
def test_qwen3_layer_decode_parity(B):
    shape = synth.QWEN3_8B_LAYER
    rig = LayerRig(shape, 90 + B, num_pages=B * 260 + 8, act_f32=True)
    lens = synth.uniform_ints(B, 128, 4096, 91 + B)
    for b in range(B):
        rig.add_request(b, int(lens[b]) - 1, 3000 + 2 * b, int(lens[b]))
    h = synth.normal((B, shape.d_model), 92 + B, dtype=F32)
    items = [(b, 1, int(lens[b]) - 1) for b in range(B)]
    out = rig.run(cuda(h), items)
    assert max_rel_err(f64(out), rig.oracle(h, items)) <= TOL_LAYER32


def test_layer_target_bitwise_across_batches_and_modes():
    shape = synth.LLAMA31_8B_LAYER
    rig = LayerRig(shape, 17, num_pages=32 * 260 + 8, act_f32=True)
    tlen = 1800
    rig.add_request("t", tlen - 1, 5321, tlen)
    ht = synth.normal((1, shape.d_model), 5322, dtype=F32)
    ref = rig.run(cuda(ht), [("t", 1, tlen - 1)])
    refk = rig.run(cuda(ht), [("t", 1, tlen - 1)], mode=bi.INVARIANT_KSPLIT)
    lens = synth.uniform_ints(31, 128, 4096, 150)
    for b in range(31):
        rig.add_request(b, int(lens[b]) - 1, 6000 + 2 * b, int(lens[b]))
    for trial, B in enumerate([2, 9, 32]):
        pos = (3 * trial + 1) % B
        others = [(b, 1, int(lens[b]) - 1) for b in range(B - 1)]
        items = others[:pos] + [("t", 1, tlen - 1)] + others[pos:]
        h = synth.normal((B, shape.d_model), 160 + trial, dtype=F32)
        h[pos] = ht[0]
        out = rig.run(cuda(h), items)
        assert bits_equal(out[pos:pos + 1], ref), B
        outp = rig.run(cuda(h), items, mode=bi.PROTECTED, target=pos)
        assert bits_equal(outp[pos:pos + 1], ref), ("protected", B)
        outk = rig.run(cuda(h), items, mode=bi.INVARIANT_KSPLIT)
        assert bits_equal(outk[pos:pos + 1], refk), ("ksplit", B)
        refo = rig.oracle(h, items)
        assert max_rel_err(f64(out), refo) <= TOL_LAYER32
        outf = rig.run(cuda(h), items, mode=bi.FAST)
        assert max_rel_err(f64(outf), refo) <= TOL_LAYER32


def test_qwen3_layer_chunked_prefill_equals_token_by_token_decode():
    shape = synth.QWEN3_8B_LAYER
    L = 300
    h = synth.normal((L, shape.d_model), 170, dtype=F32)
    outs = []
    for chunks in ([L], [129, 128, 43], [1] * 20 + [L - 20]):
        rig = LayerRig(shape, 18, num_pages=64, act_f32=True)
        rig.add_request(0, 0, 1, L)
        res, p = [], 0
        for n in chunks:
            res.append(rig.run(cuda(h[p:p + n]), [(0, n, p)]))
            p += n
        outs.append(torch.cat(res))
    for o in outs[1:]:
        assert bits_equal(o, outs[0])
    rig = LayerRig(shape, 18, num_pages=128, act_f32=True)
    rig.add_request(0, 0, 1, L)
    rig.add_request(1, 0, 2, L)
    hn = synth.normal((L, shape.d_model), 171, dtype=F32)
    res = []
    for p in range(L):
        x = torch.cat([h[p:p + 1], hn[p:p + 1]])
        res.append(rig.run(cuda(x), [(0, 1, p), (1, 1, p)])[0:1])
    assert bits_equal(torch.cat(res), outs[0])


# ---------------------------------------------------------------- model
def tiny_shape(layer=synth.TINY_QK_LAYER):
    return ModelShape(layer=layer, n_layers=2, vocab=512, max_pos=8448)  # decode neighbours reach 8000 + steps


def test_tiny_model_parity():
    shape = tiny_shape()
    m = BiModel.random(shape, seed=13, num_pages=256, act_f32=True)
    prompts = [synth.token_ids(n, shape.vocab, 190 + n) for n in (37, 5, 120)]
    out = m.forward_batch([(i, p) for i, p in enumerate(prompts)])
    w = m.host_weights()
    kv = oracle.OracleKV(shape.n_layers, shape.layer.n_kv_heads, shape.layer.head_dim)
    lens = [len(p) for p in prompts]
    logits = oracle.model_forward(np.concatenate(prompts), w["embed"], w["layers"], w["final_norm"], w["lm_head"],
                                  shape.layer, kv, [(i, n) for i, n in enumerate(lens)], [0, 0, 0], act32=True)
    last = np.cumsum(lens) - 1
    assert max_rel_err(out.logits.double().cpu().numpy(), logits[last]) <= TOL_LAYER32
    nxt = out.top_i[:, 0].cpu().numpy().astype(np.int32)
    out2 = m.forward_batch([(i, nxt[i:i + 1]) for i in range(3)])
    logits2 = oracle.model_forward(nxt, w["embed"], w["layers"], w["final_norm"], w["lm_head"], shape.layer, kv,
                                   [(i, 1) for i in range(3)], lens, act32=True)
    assert max_rel_err(out2.logits.double().cpu().numpy(), logits2) <= TOL_LAYER32
    tv, ti = oracle.topk(out2.logits.double().cpu().numpy(), 20)
    assert np.array_equal(out2.top_i.cpu().numpy(), ti)
    assert np.array_equal(out2.top_v.double().cpu().numpy(), tv)


def test_tiny_model_greedy_bit_exact_across_compositions():
    from tests.test_model_gpu import assert_same, greedy_run
    shape = tiny_shape()
    m = BiModel.random(shape, seed=14, num_pages=40000, page_seed=6, act_f32=True)
    prompt = synth.token_ids(64, shape.vocab, 4321)
    ref = greedy_run(m, prompt, 20, [64], 0, 0, 0, seed=2)
    for i, (chunks, nb, slot, dnb) in enumerate([([64], 3, 1, 5), ([7, 57], 2, 2, 63)]):
        assert_same(ref, greedy_run(m, prompt, 20, chunks, nb, slot, dnb, seed=20 + i), "composition %d" % i)
    assert_same(ref, greedy_run(m, prompt, 20, [40, 24], 3, 1, 7, seed=70, mode=bi.PROTECTED), "protected")
