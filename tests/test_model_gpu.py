"""Whole model through bi_model_forward: oracle parity on a tiny model, and the
target request's greedy tokens and top-20 logits bit-exact across every batch
composition tried (neighbour count and lengths, slot index, prefill chunking)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.helpers import max_rel_err

pytestmark = pytest.mark.gpu
bi = pytest.importorskip("invariant_deterministic_02_gb300")
from invariant_deterministic_02_gb300.model import QWEN3_8B, BiModel, ModelShape  # noqa: E402


def tiny_shape(layer=synth.TINY_LAYER):
    return ModelShape(layer=layer, n_layers=2, vocab=512, max_pos=8448)  # decode neighbours reach 8000 + steps


@pytest.mark.parametrize("layer", [synth.TINY_LAYER, synth.TINY_QK_LAYER], ids=["plain", "qk_norm"])
def test_tiny_model_prefill_and_decode_parity(layer):
    shape = tiny_shape(layer)
    m = BiModel.random(shape, seed=11, num_pages=256)
    prompts = [synth.token_ids(n, shape.vocab, 90 + n) for n in (37, 5, 120)]
    out = m.forward_batch([(i, p) for i, p in enumerate(prompts)])
    w = m.host_weights()
    kv = oracle.OracleKV(shape.n_layers, shape.layer.n_kv_heads, shape.layer.head_dim)
    lens = [len(p) for p in prompts]
    logits = oracle.model_forward(np.concatenate(prompts), w["embed"], w["layers"], w["final_norm"], w["lm_head"],
                                  shape.layer, kv, [(i, n) for i, n in enumerate(lens)], [0, 0, 0])
    last = np.cumsum(lens) - 1
    got = out.logits.double().cpu().numpy()
    assert max_rel_err(got, logits[last]) <= 2e-2
    nxt = out.top_i[:, 0].cpu().numpy().astype(np.int32)
    out2 = m.forward_batch([(i, nxt[i:i + 1]) for i in range(3)])
    logits2 = oracle.model_forward(nxt, w["embed"], w["layers"], w["final_norm"], w["lm_head"], shape.layer, kv,
                                   [(i, 1) for i in range(3)], lens)
    assert max_rel_err(out2.logits.double().cpu().numpy(), logits2) <= 2e-2
    # top-k of the GPU logits is exactly the oracle's selection on those same fp32 values
    tv, ti = oracle.topk(out2.logits.double().cpu().numpy(), 20)
    assert np.array_equal(out2.top_i.cpu().numpy(), ti)
    assert np.array_equal(out2.top_v.double().cpu().numpy(), tv)


def greedy_run(m: BiModel, prompt, steps, prefill_chunks, neighbours, target_slot, decode_neighbours, seed,
               mode=bi.INVARIANT):
    """Prefill the target prompt in the given chunks (each chunk batched with
    prefilling neighbours), then greedy-decode `steps` tokens batched with
    decode neighbours that carry random cached histories.  Returns the target's
    tokens and per-step top-20 (values, indices)."""
    m.reset()
    rng = np.random.default_rng(seed)
    V = m.shape.vocab
    T = "target"
    # prefill
    p = 0
    out = None
    for ci, n in enumerate(prefill_chunks):
        items = []
        for j in range(neighbours):
            r = ("pre", ci, j)
            L = int(rng.integers(100, 1200))
            items.append((r, synth.token_ids(L, V, seed * 31 + ci * 7 + j)))
        slot = min(target_slot, len(items))
        items.insert(slot, (T, prompt[p:p + n]))
        res = m.forward_batch(items, k=20, mode=mode, target_request=slot if mode == bi.PROTECTED else -1)
        out = (res, slot)
        for r, _ in items:
            if r != T:
                m.release(r)
        p += n
    res, slot = out
    tokens, tops = [], []
    tok = int(res.top_i[slot, 0])
    tokens.append(tok)
    tops.append((res.top_v[slot].cpu().numpy().view(np.uint32).copy(), res.top_i[slot].cpu().numpy().copy()))
    # decode
    hist = synth.uniform_ints(decode_neighbours, 100, 8000, seed + 5)
    nb_tok = {}
    for j in range(decode_neighbours):
        m.install_history(("dec", j), int(hist[j]), seed * 1000 + j)
        nb_tok[("dec", j)] = int(rng.integers(0, V))
    for s in range(steps - 1):
        items = [(("dec", j), np.array([nb_tok[("dec", j)]], dtype=np.int32)) for j in range(decode_neighbours)]
        slot = min(target_slot, len(items))
        items.insert(slot, (T, np.array([tok], dtype=np.int32)))
        res = m.forward_batch(items, k=20, mode=mode, target_request=slot if mode == bi.PROTECTED else -1)
        ti = res.top_i[:, 0].cpu().numpy()
        for b, (r, _) in enumerate(items):
            if r != T:
                nb_tok[r] = int(ti[b])
        tok = int(ti[slot])
        tokens.append(tok)
        tops.append((res.top_v[slot].cpu().numpy().view(np.uint32).copy(), res.top_i[slot].cpu().numpy().copy()))
    # every position, page and KV length the kernels met was in range
    assert bi.bi_device_error() == 0
    return tokens, tops


def assert_same(a, b, what):
    ta, pa = a
    tb, pb = b
    assert ta == tb, "%s: token sequences differ (first at %d)" % (
        what, next(i for i, (x, y) in enumerate(zip(ta, tb)) if x != y))
    for s, ((va, ia), (vb, ib)) in enumerate(zip(pa, pb)):
        assert np.array_equal(ia, ib) and np.array_equal(va, vb), "%s: top-20 differs at step %d" % (what, s)


def test_tiny_model_greedy_bit_exact_across_compositions():
    shape = tiny_shape()
    m = BiModel.random(shape, seed=12, num_pages=16384, page_seed=5)
    prompt = synth.token_ids(64, shape.vocab, 1234)
    ref = greedy_run(m, prompt, 30, [64], 0, 0, 0, seed=1)
    for i, (chunks, nb, slot, dnb) in enumerate([([64], 3, 1, 5), ([32, 32], 1, 0, 15), ([7, 57], 2, 2, 63),
                                                 ([1] * 4 + [60], 0, 0, 1)]):
        got = greedy_run(m, prompt, 30, chunks, nb, slot, dnb, seed=10 + i)
        assert_same(ref, got, "composition %d" % i)
    got = greedy_run(m, prompt, 30, [40, 24], 3, 1, 7, seed=50, mode=bi.PROTECTED)
    assert_same(ref, got, "protected")
    refk = greedy_run(m, prompt, 30, [64], 0, 0, 0, seed=1, mode=bi.INVARIANT_KSPLIT)
    got = greedy_run(m, prompt, 30, [7, 57], 2, 2, 63, seed=60, mode=bi.INVARIANT_KSPLIT)
    assert_same(refk, got, "ksplit")


def _oracle_steps(m, steps):
    """Oracle logits of one request computed alone: `steps` is a list of token
    arrays fed in order (a prefill, then decode tokens); returns the last-token
    logits of each step."""
    w = m.host_weights()
    sh = m.shape
    kv = oracle.OracleKV(sh.n_layers, sh.layer.n_kv_heads, sh.layer.head_dim)
    out, pos = [], 0
    for toks in steps:
        toks = np.asarray(toks, dtype=np.int32)
        lg = oracle.model_forward(toks, w["embed"], w["layers"], w["final_norm"], w["lm_head"], sh.layer, kv,
                                  [(0, len(toks))], [pos])
        out.append(lg[-1])
        pos += len(toks)
    return out


def test_blocklock_pack_target_bits_equal_invariant_alone():
    """BlockLock-Pack reading: the protected request is packed last behind a dummy
    segment that aligns it to a 128-row tile, the shared prefill runs PROTECTED
    (the neighbours FAST), then the target decodes alone.  Its tokens and top-20
    bits equal those of the target computed alone in INVARIANT mode, whatever the
    neighbours are, and its logits (packed prefill and the first decode step) agree
    with the oracle of the target computed alone (zhaixingw.cn BlockLock post, the
    Pack mode in "BlockLock 只锁住被保护的那条请求")."""
    shape = tiny_shape()
    m = BiModel.random(shape, seed=31, num_pages=4096, page_seed=11)
    V = shape.vocab
    prompt = synth.token_ids(90, V, 300)

    def decode_alone(req, first_tok, steps=12):
        toks, tops, logits = [first_tok], [], []
        for _ in range(steps):
            res = m.forward_batch([(req, np.array([toks[-1]], dtype=np.int32))], mode=bi.INVARIANT)
            toks.append(int(res.top_i[0, 0]))
            tops.append(res.top_v[0].cpu().numpy().view(np.uint32).copy())
            logits.append(res.logits[0].double().cpu().numpy())
        return toks, tops, logits

    res = m.forward_batch([("t", prompt)], mode=bi.INVARIANT)
    ref_first = (int(res.top_i[0, 0]), res.top_v[0].cpu().numpy().view(np.uint32).copy())
    ref = decode_alone("t", ref_first[0])
    orc = _oracle_steps(m, [prompt, [ref_first[0]]])
    m.reset()
    for trial, lens in enumerate([(37, 200), (5,), (130, 64, 300)]):
        items = [("n%d" % j, synth.token_ids(n, V, 400 + 10 * trial + j)) for j, n in enumerate(lens)]
        items.insert(trial % (len(items) + 1), ("t", prompt))
        out, row = m.pack_prefill(items, "t")
        assert out.top_i[row, 0].item() == ref_first[0]
        assert np.array_equal(out.top_v[row].cpu().numpy().view(np.uint32), ref_first[1])
        assert max_rel_err(out.logits[row].double().cpu().numpy(), orc[0]) <= 2e-2, trial
        for r, _ in items:
            if r != "t":
                m.release(r)
        got = decode_alone("t", ref_first[0])
        assert got[0] == ref[0], trial
        for a, b in zip(got[1], ref[1]):
            assert np.array_equal(a, b), trial
        assert max_rel_err(got[2][0], orc[1]) <= 2e-2, trial
        m.reset()


def test_prefix_kv_reuse_across_batches_bitwise():
    """A prompt's K/V computed inside one batch, reused by a new request in another
    batch composition (a prefix-cache hit), continues with exactly the bits of a
    request that computed everything alone, and its logits (suffix prefill and the
    first decode step) agree with the oracle of the request computed alone
    (zhaixingw.cn BlockLock post, the use cases in "batch 里换个邻居"; devpress
    digest section 3.3 on the KV cache)."""
    shape = tiny_shape()
    m = BiModel.random(shape, seed=21, num_pages=4096, page_seed=9)
    V = shape.vocab
    prompt = synth.token_ids(64, V, 77)
    suffix = synth.token_ids(20, V, 78)

    def continue_decode(req, first_items, steps=12):
        """Run `first_items` (req's suffix prefill, maybe with neighbours), then greedy
        decode req for `steps` tokens, batched with the decoding neighbour "nb" if it exists."""
        res = m.forward_batch(first_items)
        slot = [r for r, _ in first_items].index(req)
        toks, tops = [int(res.top_i[slot, 0])], [res.top_v[slot].cpu().numpy().view(np.uint32).copy()]
        logits = [res.logits[slot].double().cpu().numpy()]
        for _ in range(steps):
            items = [(req, np.array([toks[-1]], dtype=np.int32))]
            if "nb" in m.lengths:
                items.append(("nb", np.array([7], dtype=np.int32)))
            res = m.forward_batch(items)
            toks.append(int(res.top_i[0, 0]))
            tops.append(res.top_v[0].cpu().numpy().view(np.uint32).copy())
            logits.append(res.logits[0].double().cpu().numpy())
        return toks, tops, logits

    # reference: prompt and suffix prefilled by the request alone, then decode alone
    m.forward_batch([("ref", prompt)])
    ref = continue_decode("ref", [("ref", suffix)])
    m.reset()
    # the prompt is prefilled by request "src" inside a batch of three
    m.forward_batch([("a", synth.token_ids(300, V, 80)), ("src", prompt), ("b", synth.token_ids(17, V, 81))])
    m.release("a")
    m.release("b")
    # a new request reuses the prompt's 64 cached positions (4 pages) and prefills only the suffix,
    # in a batch with a decoding neighbour that has a long history
    m.install_history("nb", 1500, 82)
    m.copy_prefix("src", "dst", 64)
    got = continue_decode("dst", [("nb", np.array([5], dtype=np.int32)), ("dst", suffix)])
    assert got[0] == ref[0]
    for a, b in zip(got[1], ref[1]):
        assert np.array_equal(a, b)
    orc = _oracle_steps(m, [prompt, suffix, [ref[0][0]]])
    assert max_rel_err(got[2][0], orc[1]) <= 2e-2
    assert max_rel_err(got[2][1], orc[2]) <= 2e-2


@pytest.mark.slow
def test_qwen3_8b_greedy_200_tokens_bit_exact_across_compositions():
    """Full Qwen3-8B-shaped random-init model: a 512-token seeded prompt, greedy 200 tokens."""
    m = BiModel(QWEN3_8B, BiModel.random_weights(QWEN3_8B, seed=5), num_pages=36000, page_seed=9)
    prompt = synth.token_ids(512, QWEN3_8B.vocab, 1234)
    ref = greedy_run(m, prompt, 200, [512], 0, 0, 0, seed=1)
    trials = [([97] * 5 + [27], 3, 2, 7), ([512], 1, 1, 63), ([256, 256], 2, 0, 31)]
    for i, (chunks, nb, slot, dnb) in enumerate(trials):
        got = greedy_run(m, prompt, 200, chunks, nb, slot, dnb, seed=20 + i)
        assert_same(ref, got, "composition %d" % i)
