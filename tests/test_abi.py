"""The C ABI library builds, loads and exports every entry point include/bi.h declares (no GPU needed)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bi.h")


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bi_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def libpath():
    from invariant_deterministic_02_gb300.build import build_library
    return build_library()


def test_header_declares_the_boundary():
    syms = declared_symbols()
    for name in ["bi_rmsnorm", "bi_gemm", "bi_decode_attention", "bi_prefill_attention", "bi_layer_forward",
                 "bi_embed", "bi_topk", "bi_status_string", "bi_model_forward"]:
        assert name in syms


def test_library_exports_every_declared_symbol(libpath):
    out = subprocess.run(["nm", "-D", "--defined-only", libpath], capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT (bi_[a-z0-9_]+)$", out, flags=re.M))
    missing = [s for s in declared_symbols() if s not in exported]
    assert not missing, missing


def test_library_loads_and_answers_without_gpu(libpath):
    import invariant_deterministic_02_gb300 as bi
    l = bi.lib()
    for name in declared_symbols():
        assert hasattr(l, name)
    assert l.bi_status_string(0) == b"BI_OK"
    assert l.bi_status_string(3) == b"BI_ERR_WORKSPACE"
    assert l.bi_version() >= 100


def test_host_validation_rejects_bad_arguments_before_launch(libpath):
    # every check below fails on the host, so nothing reaches a GPU
    import invariant_deterministic_02_gb300 as bi
    l = bi.lib()
    assert l.bi_gemm(None, None, None, None, 4, 8, 7, bi.BI_BF16, 0, -1, 0, None, 0, None) == bi.BI_ERR_INVALID_ARG
    assert l.bi_gemm(None, None, None, None, 4, 12, 16, bi.BI_BF16, 0, -1, 0, None, 0, None) == bi.BI_ERR_UNSUPPORTED
    assert b"multiples of 8" in l.bi_last_error_message()
    assert l.bi_rmsnorm(None, None, None, 4, 12, bi.BI_BF16, 1e-5, 0, -1, 0, None, 0, None) == bi.BI_ERR_UNSUPPORTED
    assert l.bi_rmsnorm(None, None, None, 4, 16, bi.BI_BF16, 1e-5, 7, -1, 0, None, 0, None) == bi.BI_ERR_INVALID_ARG
    assert l.bi_rmsnorm(None, None, None, 4, 16, bi.BI_BF16, 1e-5, 2, 3, 5, None, 0, None) == bi.BI_ERR_INVALID_ARG
    d = bi.attn_dims(32, 8, 96, 4, 4)
    assert l.bi_decode_attention(None, None, None, None, None, 1, ctypes.byref(d), None, 0, -1, None, 0,
                                 None) == bi.BI_ERR_UNSUPPORTED
    d = bi.attn_dims(32, 4, 128, 4, 4)  # 8 query heads per kv head is not built
    assert l.bi_decode_attention(None, None, None, None, None, 1, ctypes.byref(d), None, 0, -1, None, 0,
                                 None) == bi.BI_ERR_UNSUPPORTED
    assert l.bi_topk(None, 2, 10, 40, None, None, None) == bi.BI_ERR_UNSUPPORTED
    # zero-size work is a no-op that succeeds without touching pointers
    assert l.bi_rmsnorm(None, None, None, 0, 16, bi.BI_BF16, 1e-5, 0, -1, 0, None, 0, None) == bi.BI_OK
    assert l.bi_gemm(None, None, None, None, 0, 8, 16, bi.BI_BF16, 0, -1, 0, None, 0, None) == bi.BI_OK


def test_ksplit_part_count_depends_on_weight_shape_only(libpath):
    # S = clamp(152 // ceil(N/256), 1, min(16, ceil(K/64) // 4)): a pure function of (N, K)
    import invariant_deterministic_02_gb300 as bi
    for (N, K), S in {(4096, 4096): 9, (6144, 4096): 6, (24576, 4096): 1, (151936, 4096): 1,
                      (4096, 12288): 9, (4096, 14336): 9, (256, 512): 2, (256, 64): 1, (512, 2048): 8,
                      (1032, 1000): 4, (40000, 512): 1}.items():
        assert bi.bi_gemm_ksplit(N, K) == S, (N, K)
    l = bi.lib()
    f = 4
    # decode-sized M: S partial planes of M x N fp32; larger M merges in the CTA and needs none
    assert l.bi_gemm_workspace(64, 4096, 4096, bi.INVARIANT_KSPLIT) == 9 * 64 * 4096 * f
    assert l.bi_gemm_workspace(128, 6144, 4096, bi.INVARIANT_KSPLIT) == 6 * 128 * 6144 * f
    assert l.bi_gemm_workspace(129, 4096, 4096, bi.INVARIANT_KSPLIT) == 0
    assert l.bi_gemm_workspace(64, 24576, 4096, bi.INVARIANT_KSPLIT) == 0
    assert l.bi_gemm_workspace(64, 4096, 4096, bi.INVARIANT) == 0
    # an out-of-range mode is rejected on the host
    assert l.bi_gemm(None, None, None, None, 4, 8, 16, bi.BI_BF16, 4, -1, 0, None, 0, None) == bi.BI_ERR_INVALID_ARG


def test_fp32_activation_entry_points_validate_and_size_on_the_host(libpath):
    import invariant_deterministic_02_gb300 as bi
    l = bi.lib()
    planes = lambda M, K: (3 * M * K * 2 + 255) // 256 * 256  # noqa: E731  three bf16 planes of A, 256-byte aligned
    assert l.bi_gemm_f32a_workspace(64, 4096, 4096, bi.INVARIANT) == planes(64, 4096)
    assert l.bi_gemm_f32a_workspace(64, 4096, 4096, bi.INVARIANT_KSPLIT) == planes(64, 4096) + 9 * 64 * 4096 * 4
    assert l.bi_gemm_f32a_workspace(0, 4096, 4096, bi.INVARIANT) == 0
    assert l.bi_gemm_f32a(None, None, None, None, 0, 8, 16, 0, -1, 0, None, 0, None) == bi.BI_OK
    assert l.bi_gemm_f32a(None, None, None, None, 4, 8, 7, 0, -1, 0, None, 0, None) == bi.BI_ERR_INVALID_ARG
    assert l.bi_gemm_f32a(None, None, None, None, 4, 8, 16, 9, -1, 0, None, 0, None) == bi.BI_ERR_INVALID_ARG
    assert l.bi_gemm_f32a(None, None, None, None, 4, 8, 16, 0, -1, 0, None, 0, None) == bi.BI_ERR_INVALID_ARG
    # act_f32 is a trailing field of both dims structs; zero keeps bf16 activations
    assert ctypes.sizeof(bi.AttnDims) == 8 * 4 and ctypes.sizeof(bi.ModelDims) == 10 * 4
    dims = [bi.ModelDims(256, 4, 2, 64, 512, 512, 16, 2048, 1e-5, a) for a in (0, 1, 2)]
    qs = (ctypes.c_int32 * 2)(0, 4)
    batch = bi.Batch(1, 4, 4, ctypes.addressof(qs), ctypes.addressof(qs), ctypes.addressof(qs), 1, 1, -1, 0, 0)
    w16, w32, bad = [l.bi_layer_workspace(ctypes.byref(d), ctypes.byref(batch), 0) for d in dims]
    assert w32 > w16 > 0 and bad == 0


def test_layer_and_model_entry_points_reject_bad_arguments_before_launch(libpath):
    # every failure below is found on the host before anything is launched, so no GPU is needed
    import invariant_deterministic_02_gb300 as bi
    l = bi.lib()
    qs = (ctypes.c_int32 * 2)(0, 4)
    batch = bi.Batch(1, 4, 4, ctypes.addressof(qs), ctypes.addressof(qs), ctypes.addressof(qs), 1, 1, -1, 0, 0)
    good = bi.ModelDims(256, 4, 2, 64, 512, 512, 16, 2048, 1e-5, 0)
    lw = bi.LayerWeights(*([None] * 8))
    dummy = ctypes.c_void_p(16)
    # act_f32 must be 0 or 1
    bad = bi.ModelDims(256, 4, 2, 64, 512, 512, 16, 2048, 1e-5, 3)
    assert l.bi_layer_forward(ctypes.byref(bad), ctypes.byref(lw), dummy, dummy, dummy, ctypes.byref(batch), dummy,
                              dummy, 0, dummy, 1 << 30, None) == bi.BI_ERR_INVALID_ARG
    assert b"act_f32" in l.bi_last_error_message()
    # page size other than 16, d_model not a multiple of 8
    for dims in (bi.ModelDims(256, 4, 2, 64, 512, 512, 8, 2048, 1e-5, 0),
                 bi.ModelDims(260, 4, 2, 64, 512, 512, 16, 2048, 1e-5, 0)):
        assert l.bi_layer_forward(ctypes.byref(dims), ctypes.byref(lw), dummy, dummy, dummy, ctypes.byref(batch),
                                  dummy, dummy, 0, dummy, 1 << 30, None) == bi.BI_ERR_UNSUPPORTED
    # a mode outside the enum, a null hidden state, a workspace smaller than the query
    assert l.bi_layer_forward(ctypes.byref(good), ctypes.byref(lw), dummy, dummy, dummy, ctypes.byref(batch), dummy,
                              dummy, 9, dummy, 1 << 30, None) == bi.BI_ERR_INVALID_ARG
    assert l.bi_layer_forward(ctypes.byref(good), ctypes.byref(lw), dummy, dummy, None, ctypes.byref(batch), dummy,
                              dummy, 0, dummy, 1 << 30, None) == bi.BI_ERR_INVALID_ARG
    need = l.bi_layer_workspace(ctypes.byref(good), ctypes.byref(batch), 0)
    assert need > 0
    assert l.bi_layer_forward(ctypes.byref(good), ctypes.byref(lw), dummy, dummy, dummy, ctypes.byref(batch), dummy,
                              dummy, 0, dummy, need - 1, None) == bi.BI_ERR_WORKSPACE
    # a batch whose protected request lies outside it
    bad_batch = bi.Batch(1, 4, 4, ctypes.addressof(qs), ctypes.addressof(qs), ctypes.addressof(qs), 1, 1, 3, 0, 1)
    assert l.bi_layer_workspace(ctypes.byref(good), ctypes.byref(bad_batch), 0) == 0
    # the model entry point: null model pointers, then a vocabulary that is not a multiple of 8
    args = (dummy, dummy, dummy, ctypes.byref(batch), None, None, dummy, 20, dummy, dummy, None, 0, dummy, 1 << 30,
            None)
    mw = bi.ModelWeights(None, None, 0, None, None)
    assert l.bi_model_forward(ctypes.byref(good), ctypes.byref(mw), *args) == bi.BI_ERR_INVALID_ARG
    mw = bi.ModelWeights(16, None, 0, 16, 16)  # no layers: only the embedding, final norm and head are named
    odd = bi.ModelDims(256, 4, 2, 64, 512, 500, 16, 2048, 1e-5, 0)
    assert l.bi_model_forward(ctypes.byref(odd), ctypes.byref(mw), *args) == bi.BI_ERR_UNSUPPORTED
    assert b"vocab" in l.bi_last_error_message()
