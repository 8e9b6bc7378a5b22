"""Gate|up GEMM + SwiGLU in one call: oracle parity, the same bits as the two separate
calls (fused epilogue and two-kernel path alike), and row invariance across M."""
import pytest
import torch

import oracle
import synth
from tests.helpers import TOL_BF16, bits_equal, cuda, f64, max_rel_err

pytestmark = pytest.mark.gpu
bi = pytest.importorskip("invariant_deterministic_02_gb300")


def fused(A, W, mode=bi.INVARIANT, tr=-1, tc=0):
    act = torch.empty((A.shape[0], W.shape[0] // 2), dtype=torch.bfloat16, device="cuda")
    bi.bi_gemm_swiglu(A, W, act, mode=mode, target_row=tr, target_count=tc)
    torch.cuda.synchronize()
    return act


def separate(A, W, mode=bi.INVARIANT, tr=-1, tc=0):
    gu = torch.empty((A.shape[0], W.shape[0]), dtype=torch.bfloat16, device="cuda")
    bi.bi_gemm(A, W, gu, mode=mode, target_row=tr, target_count=tc)
    act = torch.empty((A.shape[0], W.shape[0] // 2), dtype=torch.bfloat16, device="cuda")
    bi.bi_swiglu(gu, act)
    torch.cuda.synchronize()
    return act


# M <= 64 runs M = 64 instructions (lanes 16..31 take the upper columns), M <= 128 the
# full-height fused epilogue, larger M the two-kernel path; F values that leave a ragged
# last tile (F not a multiple of the tile's half width) are included.
SHAPES = [(1, 512, 512), (5, 200, 256), (33, 1000, 1024), (64, 12288, 4096), (97, 2056, 1024), (128, 776, 520),
          (200, 512, 1024), (300, 264, 72)]


@pytest.mark.parametrize("M,F,K", SHAPES)
def test_parity_with_oracle(M, F, K):
    A = synth.normal((M, K), 100 + M)
    W = synth.normal((2 * F, K), 101 + F, std=0.02)
    act = fused(cuda(A), cuda(W))
    gu = oracle.round_bf16(oracle.gemm(f64(A), f64(W)))
    ref = oracle.round_bf16(oracle.swiglu(gu[:, :F], gu[:, F:]))
    assert max_rel_err(f64(act), ref) <= TOL_BF16


@pytest.mark.parametrize("M,F,K", SHAPES)
@pytest.mark.parametrize("mode", [bi.INVARIANT, bi.FAST, bi.INVARIANT_KSPLIT], ids=["inv", "fast", "ksplit"])
def test_same_bits_as_gemm_then_swiglu(M, F, K, mode):
    A = cuda(synth.normal((M, K), 110 + M))
    W = cuda(synth.normal((2 * F, K), 111 + F, std=0.02))
    assert bits_equal(fused(A, W, mode), separate(A, W, mode))


def test_protected_target_same_bits():
    M, F, K = 100, 1024, 2048
    A = cuda(synth.normal((M, K), 120))
    W = cuda(synth.normal((2 * F, K), 121, std=0.02))
    assert bits_equal(fused(A, W, bi.PROTECTED, 40, 3), separate(A, W, bi.PROTECTED, 40, 3))


def test_row_invariant_across_batch_sizes():
    F, K = 12288, 4096
    W = cuda(synth.normal((2 * F, K), 130, std=0.02))
    A = synth.normal((300, K), 131)
    ref = fused(cuda(A[7:8]), W)
    for M in (8, 16, 64, 65, 128, 129, 300):
        assert bits_equal(fused(cuda(A[:M]), W)[7:8], ref), M


def test_empty_and_invalid():
    W = cuda(synth.normal((64, 64), 140))
    A = cuda(synth.normal((0, 64), 141))
    assert fused(A, W).shape == (0, 32)
    with pytest.raises(RuntimeError):
        bad = cuda(synth.normal((4, 64), 142))
        out = torch.empty((4, 30), dtype=torch.bfloat16, device="cuda")
        bi.bi_gemm_swiglu(bad, cuda(synth.normal((60, 64), 143)), out)  # F = 30 is not a multiple of 8
