"""bi_decode_attention_noalloc: decode attention for callers that cannot allocate.

Such callers (a plugin living inside a framework whose allocator owns the GPU's
memory, a serving loop that may not call cudaMalloc) pass only inputs and
outputs; the library serves the scratch from its own fixed device array.  The
check: through the C ABI, two calls in a row give the same output as the
workspace-taking bi_decode_attention on the same inputs (bit for bit, which is
stricter than the bf16 tolerance the other tests use), and a batch too large for
the fixed scratch is refused with a clear error.  This file is collected last
so that a failure here does not hide the results of the other GPU tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
from tests.helpers import TOL_BF16, bits_equal, cuda, f64, max_rel_err

pytestmark = pytest.mark.gpu
bi = pytest.importorskip("invariant_deterministic_02_gb300")

PS = 16


def build_batch(lens, hq, hkv, hd, seed):
    layout = synth.paged_layout(lens, PS, seed)
    kc = torch.zeros((layout.num_pages, hkv, PS, hd), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    for b, L in enumerate(lens):
        synth.fill_paged(kc, vc, layout.block_table[b], synth.normal((L, hkv, hd), seed + 2 * b),
                         synth.normal((L, hkv, hd), seed + 2 * b + 1))
    q = cuda(synth.normal((len(lens), hq, hd), seed + 999))
    bt = cuda(torch.from_numpy(layout.block_table))
    kl = cuda(torch.tensor(lens, dtype=torch.int32))
    dims = bi.attn_dims(hq, hkv, hd, layout.max_pages, layout.num_pages)
    return q, kc, vc, bt, kl, dims


def call_noalloc(q, kc, vc, bt, kl, dims, out, mode=bi.INVARIANT, target=-1):
    # straight through the C entry point, no Python-side allocation
    st = bi.lib().bi_decode_attention_noalloc(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), bt.data_ptr(),
                                              kl.data_ptr(), q.shape[0], ctypes.byref(dims), out.data_ptr(), mode,
                                              target, torch.cuda.current_stream().cuda_stream)
    return st


@pytest.mark.parametrize("mode", [bi.INVARIANT, bi.FAST, bi.PROTECTED])
def test_noalloc_matches_workspace_path_on_two_calls(mode):
    lens = [1, 300, 2048, 4096, 17, 1000, 255, 257]
    q, kc, vc, bt, kl, dims = build_batch(lens, 32, 8, 128, 5)
    target = 3 if mode == bi.PROTECTED else -1
    ref = torch.empty_like(q)
    bi.bi_decode_attention(q, kc, vc, bt, kl, dims, ref, mode=mode, target_request=target)
    for call in range(2):
        out = torch.full_like(q, float("nan"))
        assert call_noalloc(q, kc, vc, bt, kl, dims, out, mode, target) == bi.BI_OK, \
            bi.lib().bi_last_error_message()
        torch.cuda.synchronize()
        assert max_rel_err(f64(out), f64(ref)) <= TOL_BF16
        assert bits_equal(out, ref), "call %d differs from bi_decode_attention" % call


def test_noalloc_refuses_batches_beyond_its_scratch():
    # 256 requests of up to 32768 tokens need far more than the fixed scratch
    hq, hkv, hd = 32, 8, 128
    q = torch.zeros((256, hq, hd), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((4, hkv, PS, hd), dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros((256, 2048), dtype=torch.int32, device="cuda")
    kl = torch.ones(256, dtype=torch.int32, device="cuda")
    dims = bi.attn_dims(hq, hkv, hd, 2048, 4)
    out = torch.empty_like(q)
    st = call_noalloc(q, kc, kc, bt, kl, dims, out)
    assert st == bi.BI_ERR_UNSUPPORTED
    msg = bi.lib().bi_last_error_message().decode()
    assert "scratch" in msg and "bi_decode_attention" in msg


def test_noalloc_fast_mode_at_decode_batch_64():
    # FAST plans about four work items per SM over the batch (a few splits per request at B = 64), so its
    # scratch fits easily; it is sized from the same split count the plan kernel uses
    lens = [int(v) for v in synth.uniform_ints(64, 128, 4096, 8)]
    q, kc, vc, bt, kl, dims = build_batch(lens, 32, 8, 128, 9)
    for mode, target in ((bi.FAST, -1), (bi.PROTECTED, 5)):
        ref = torch.empty_like(q)
        bi.bi_decode_attention(q, kc, vc, bt, kl, dims, ref, mode=mode, target_request=target)
        out = torch.full_like(q, float("nan"))
        assert call_noalloc(q, kc, vc, bt, kl, dims, out, mode, target) == bi.BI_OK, \
            bi.lib().bi_last_error_message()
        torch.cuda.synchronize()
        assert bits_equal(out, ref), mode


def test_noalloc_kv_len_beyond_block_table_is_clamped_and_reported():
    # a kv_len one past the block table's reach (max_pages * 16 + 1) is clamped by the plan kernel and
    # reported; no access leaves the caller's buffers or the scratch, and the next call is unaffected
    lens = [300, 100]
    q, kc, vc, bt, kl, dims = build_batch(lens, 32, 8, 128, 21)
    assert bi.bi_device_error() == 0
    bad = kl.clone()
    bad[0] = dims.max_pages * PS + 1
    out = torch.empty_like(q)
    assert call_noalloc(q, kc, vc, bt, bad, dims, out) == bi.BI_OK
    torch.cuda.synchronize()
    assert bi.bi_device_error() == 16
    ref = torch.empty_like(q)
    bi.bi_decode_attention(q, kc, vc, bt, kl, dims, ref)
    out2 = torch.full_like(q, float("nan"))
    assert call_noalloc(q, kc, vc, bt, kl, dims, out2) == bi.BI_OK
    torch.cuda.synchronize()
    assert bi.bi_device_error() == 0
    assert bits_equal(out2, ref)
