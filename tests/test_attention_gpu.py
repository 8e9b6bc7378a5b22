"""Paged split-KV attention: oracle parity, prefill == decode bitwise, batch invariance, modes."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.helpers import TOL_BF16, bits_equal, cuda, f64, max_rel_err

pytestmark = pytest.mark.gpu
bi = pytest.importorskip("invariant_deterministic_02_gb300")

PS = 16


class Requests:
    """A batch of requests whose K/V live in one physically shuffled paged cache."""

    def __init__(self, kvs, hq, hkv, hd, seed, max_pages=None, spare=3):
        self.kvs = kvs  # list of (K, V) [L][Hkv][hd] bf16 (cpu)
        self.lens = [k.shape[0] for k, _ in kvs]
        self.layout = synth.paged_layout(self.lens, PS, seed, spare_pages=spare, max_pages=max_pages)
        self.kc = torch.zeros((self.layout.num_pages, hkv, PS, hd), dtype=torch.bfloat16, device="cuda")
        self.vc = torch.zeros_like(self.kc)
        # fill unused slots with NaN bit patterns so that a masked-lane read would show
        self.kc.view(torch.int16).fill_(-1)
        self.vc.view(torch.int16).fill_(-1)
        for b, (K, V) in enumerate(kvs):
            synth.fill_paged(self.kc, self.vc, self.layout.block_table[b], K, V)
        self.bt = cuda(torch.from_numpy(self.layout.block_table))
        self.dims = bi.attn_dims(hq, hkv, hd, self.layout.max_pages, self.layout.num_pages)


def random_kv(L, hkv, hd, seed):
    return synth.normal((L, hkv, hd), seed), synth.normal((L, hkv, hd), seed + 1)


def decode(req: Requests, q, mode=bi.INVARIANT, target=-1, lens=None):
    lens = req.lens if lens is None else lens
    kl = cuda(torch.tensor(lens, dtype=torch.int32))
    out = torch.empty_like(q)
    bi.bi_decode_attention(q, req.kc, req.vc, req.bt, kl, req.dims, out, mode=mode, target_request=target)
    torch.cuda.synchronize()
    return out


def prefill(req: Requests, q, counts, pos0, mode=bi.INVARIANT, target=-1):
    qs = cuda(torch.tensor(np.concatenate([[0], np.cumsum(counts)]), dtype=torch.int32))
    p0 = cuda(torch.tensor(pos0, dtype=torch.int32))
    out = torch.empty_like(q)
    bi.bi_prefill_attention(q, req.kc, req.vc, req.bt, qs, p0, req.dims, out, mode=mode, target_request=target)
    torch.cuda.synchronize()
    return out


def oracle_decode(req, q, b):
    K, V = req.kvs[b]
    L = K.shape[0]
    return oracle.attention(f64(q[b:b + 1].cpu()), f64(K), f64(V), [L - 1], req.dims.scale)[0]


@pytest.mark.parametrize("B", [1, 2, 3, 8, 16])
def test_tiny_config_decode_parity_and_target_bits(B):
    hq = hkv = 4
    hd = 64
    target_kv = random_kv(300, hkv, hd, 1234)
    target_q = synth.normal((1, hq, hd), 1235)
    kvs = [target_kv] + [random_kv(300, hkv, hd, 50 * B + i) for i in range(B - 1)]
    req = Requests(kvs, hq, hkv, hd, seed=B)
    q = torch.cat([target_q, synth.normal((B - 1, hq, hd), 77 + B)]) if B > 1 else target_q
    out = decode(req, cuda(q))
    for b in range(B):
        assert max_rel_err(f64(out[b]), oracle.round_bf16(oracle_decode(req, q, b))) <= TOL_BF16
    alone = decode(Requests([target_kv], hq, hkv, hd, seed=999), cuda(target_q))
    assert bits_equal(out[0:1], alone)


LENS = [1, 15, 16, 17, 255, 256, 257, 300, 1000, 4096]


def test_gqa_decode_parity_lengths():
    hq, hkv, hd = 32, 8, 128
    kvs = [random_kv(L, hkv, hd, 10 + i) for i, L in enumerate(LENS)]
    req = Requests(kvs, hq, hkv, hd, seed=4)
    q = synth.normal((len(LENS), hq, hd), 99)
    out = decode(req, cuda(q))
    for b in range(len(LENS)):
        assert max_rel_err(f64(out[b]), oracle.round_bf16(oracle_decode(req, q, b))) <= TOL_BF16, LENS[b]


def test_identical_keys_give_mean_of_values():
    hq, hkv, hd, L = 32, 8, 128, 700
    K1 = synth.normal((1, hkv, hd), 5)
    K = K1.repeat(L, 1, 1)
    V = synth.normal((L, hkv, hd), 6)
    req = Requests([(K, V)], hq, hkv, hd, seed=5)
    out = decode(req, cuda(synth.normal((1, hq, hd), 7)))
    mean = f64(V).mean(axis=0)  # [Hkv][hd]
    for h in range(hq):
        assert max_rel_err(f64(out[0, h]), oracle.round_bf16(mean[h // 4])) <= TOL_BF16


def test_target_bitwise_across_batch_compositions():
    hq, hkv, hd = 32, 8, 128
    tkv = random_kv(2000, hkv, hd, 1234)
    tq = synth.normal((1, hq, hd), 1236)
    ref = None
    for trial, B in enumerate([1, 2, 4, 16, 64, 256]):
        lens = synth.loguniform_ints(B - 1, 64, 8000, 300 + trial).tolist()
        kvs = [random_kv(L, hkv, hd, 4000 + 7 * trial + i) for i, L in enumerate(lens)]
        pos = (trial * 5) % B
        kvs.insert(pos, tkv)
        q = synth.normal((B, hq, hd), 600 + trial)
        q[pos] = tq[0]
        req = Requests(kvs, hq, hkv, hd, seed=trial + 11)
        out = decode(req, cuda(q))
        if ref is None:
            ref = out[pos:pos + 1].clone()
            assert max_rel_err(f64(ref[0]), oracle.round_bf16(oracle_decode(req, q, pos))) <= TOL_BF16
        else:
            assert bits_equal(out[pos:pos + 1], ref), (B, pos)


def test_prefill_chunks_equal_decode_bitwise_2048():
    hq, hkv, hd, L = 32, 8, 128, 2048
    K, V = random_kv(L, hkv, hd, 21)
    q = cuda(synth.normal((L, hq, hd), 22))
    req = Requests([(K, V)], hq, hkv, hd, seed=21)
    one = prefill(req, q, [L], [0])
    chunks = torch.cat([prefill(req, q[c:c + 512], [512], [c]) for c in range(0, L, 512)])
    assert bits_equal(one, chunks)
    # all 2048 positions as one decode batch: request p is the sequence truncated at p
    bt = req.bt.repeat(L, 1)
    req_many = Requests.__new__(Requests)
    req_many.__dict__.update(req.__dict__)
    req_many.bt = bt.contiguous()
    dec = decode(req_many, q, lens=list(range(1, L + 1)))
    assert bits_equal(dec, one)
    # literal token-by-token decode on a sample of positions
    for p in [0, 1, 255, 256, 257, 511, 512, 1000, 1535, 2047]:
        d1 = decode(req, q[p:p + 1], lens=[p + 1])
        assert bits_equal(d1, one[p:p + 1]), p
    # parity on sampled positions
    for p in [0, 17, 255, 256, 700, 2047]:
        ref = oracle.attention(f64(q[p:p + 1].cpu()), f64(K), f64(V), [p], req.dims.scale)[0]
        assert max_rel_err(f64(one[p]), oracle.round_bf16(ref)) <= TOL_BF16


def test_prefill_multi_request_parity():
    hq, hkv, hd = 32, 8, 128
    # (cached tokens already in the cache, new tokens in this call)
    spec = [(0, 40), (300, 212), (1000, 1), (31, 300)]
    kvs = [random_kv(c + n, hkv, hd, 70 + i) for i, (c, n) in enumerate(spec)]
    req = Requests(kvs, hq, hkv, hd, seed=8)
    counts = [n for _, n in spec]
    q = synth.normal((sum(counts), hq, hd), 80)
    out = prefill(req, cuda(q), counts, [c for c, _ in spec])
    t0 = 0
    for b, (c, n) in enumerate(spec):
        K, V = kvs[b]
        ref = oracle.attention(f64(q[t0:t0 + n]), f64(K), f64(V), list(range(c, c + n)), req.dims.scale)
        assert max_rel_err(f64(out[t0:t0 + n]), oracle.round_bf16(ref)) <= TOL_BF16, b
        t0 += n


def test_cached_plus_new_example_invariant_vs_fast():
    # the cache/new example with the split size of this kernel: 300 cached + 212 new vs 512 at once
    hq, hkv, hd, L = 32, 8, 128, 512
    K, V = random_kv(L, hkv, hd, 90)
    q = cuda(synth.normal((L, hq, hd), 91))
    req = Requests([(K, V)], hq, hkv, hd, seed=9)
    one = prefill(req, q, [L], [0])
    two = torch.cat([prefill(req, q[:300], [300], [0]), prefill(req, q[300:], [212], [300])])
    assert bits_equal(one, two)
    f_one = prefill(req, q, [L], [0], mode=bi.FAST)
    f_two = torch.cat([prefill(req, q[:300], [300], [0], mode=bi.FAST),
                       prefill(req, q[300:], [212], [300], mode=bi.FAST)])
    assert not bits_equal(f_one, f_two), "separate cached/new reduction never changed a bit"
    for o in (f_one, f_two):
        for p in (299, 300, 511):
            ref = oracle.attention(f64(q[p:p + 1].cpu()), f64(K), f64(V), [p], req.dims.scale)[0]
            assert max_rel_err(f64(o[p]), oracle.round_bf16(ref)) <= TOL_BF16


def test_decode_fast_and_protected():
    hq, hkv, hd = 32, 8, 128
    lens = [3000, 5000, 700]
    kvs = [random_kv(L, hkv, hd, 100 + i) for i, L in enumerate(lens)]
    req = Requests(kvs, hq, hkv, hd, seed=10)
    q = cuda(synth.normal((3, hq, hd), 110))
    inv = decode(req, q)
    fast = decode(req, q, mode=bi.FAST)
    prot = decode(req, q, mode=bi.PROTECTED, target=1)
    assert bits_equal(prot[1:2], inv[1:2])
    assert not bits_equal(fast, inv)
    for b in range(3):
        ref = oracle.round_bf16(oracle_decode(req, q.cpu(), b))
        for o in (fast, prot):
            assert max_rel_err(f64(o[b]), ref) <= TOL_BF16


def test_empty_batch_and_bad_workspace():
    hq, hkv, hd = 32, 8, 128
    req = Requests([random_kv(20, hkv, hd, 1)], hq, hkv, hd, seed=1)
    q = cuda(synth.normal((1, hq, hd), 2))
    e = torch.empty((0, hq, hd), dtype=torch.bfloat16, device="cuda")
    bi.bi_decode_attention(e, req.kc, req.vc, req.bt, cuda(torch.zeros(0, dtype=torch.int32)), req.dims, e)
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(bi.BiError) as ei:
        bi.bi_decode_attention(q, req.kc, req.vc, req.bt, cuda(torch.tensor([20], dtype=torch.int32)), req.dims,
                               torch.empty_like(q), workspace=small)
    assert ei.value.status == bi.BI_ERR_WORKSPACE


def test_full_config_256_requests_up_to_32768_tokens():
    """Decode at the full size of the attention config: 256 requests whose KV lengths
    are log-uniform in [64, 32768], one of them forced to 32768 (128 splits: the whole
    merge tree), K/V drawn on the device.  Oracle parity on sampled requests, and the
    longest request's bits equal to decoding it alone."""
    hq, hkv, hd, B = 32, 8, 128, 256
    lens = synth.loguniform_ints(B, 64, 32768, 501).tolist()
    lens[17] = 32768
    layout = synth.paged_layout(lens, PS, 502)
    kc = torch.empty((layout.num_pages, hkv, PS, hd), dtype=torch.bfloat16, device="cuda")
    vc = torch.empty_like(kc)
    kc.view(torch.int16).fill_(-1)  # NaN patterns in unused slots: a masked-lane read would show
    vc.view(torch.int16).fill_(-1)

    def kv(b):
        return (synth.normal_device((lens[b], hkv, hd), 10000 + 2 * b),
                synth.normal_device((lens[b], hkv, hd), 10001 + 2 * b))

    for b in range(B):
        synth.fill_paged(kc, vc, layout.block_table[b], *kv(b))
    bt = cuda(torch.from_numpy(layout.block_table))
    dims = bi.attn_dims(hq, hkv, hd, layout.max_pages, layout.num_pages)
    q = synth.normal_device((B, hq, hd), 503)
    kl = cuda(torch.tensor(lens, dtype=torch.int32))
    out = torch.empty_like(q)
    bi.bi_decode_attention(q, kc, vc, bt, kl, dims, out)
    torch.cuda.synchronize()
    for b in sorted({17, int(np.argmin(lens)), 0, 100, 255}):
        K, V = kv(b)
        ref = oracle.attention(f64(q[b:b + 1]), f64(K), f64(V), [lens[b] - 1], dims.scale)[0]
        assert max_rel_err(f64(out[b]), oracle.round_bf16(ref)) <= TOL_BF16, (b, lens[b])
    one = torch.empty_like(q[17:18])
    bi.bi_decode_attention(q[17:18].contiguous(), kc, vc, bt[17:18].contiguous(), kl[17:18].contiguous(), dims, one)
    torch.cuda.synchronize()
    assert bits_equal(one, out[17:18])
