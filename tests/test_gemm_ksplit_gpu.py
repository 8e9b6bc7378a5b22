"""INVARIANT_KSPLIT GEMM: the K-only split ("Batch-Invariant Kernel" notes, section GEMM).

The result is defined as ((0 + P_0) + P_1) + ... + P_{S-1} in fp32, P_s being the
INVARIANT accumulation over the k-tiles of part s, S = bi_gemm_ksplit(N, K).  For
M <= 128 the parts run on separate CTAs and a second pass adds them; for larger M
one CTA merges them in tensor memory.  These tests pin that definition against
INVARIANT sub-GEMMs, check bitwise invariance across M (which crosses both
paths), and parity with the float64 oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.helpers import TOL_BF16, bits_equal, cuda, f64, max_rel_err

pytestmark = pytest.mark.gpu
bi = pytest.importorskip("invariant_deterministic_02_gb300")


def gemm(A, W, out_dtype=torch.bfloat16, R=None, mode=bi.INVARIANT_KSPLIT):
    C = torch.empty((A.shape[0], W.shape[0]), dtype=out_dtype, device="cuda")
    bi.bi_gemm(A, W, C, residual=R, mode=mode)
    torch.cuda.synchronize()
    return C


def by_definition(A, W, R=None, out_dtype=torch.bfloat16):
    """Sum of the parts' INVARIANT fp32 GEMMs in part order, then residual, one rounding."""
    M, K = A.shape
    N = W.shape[0]
    S = bi.bi_gemm_ksplit(N, K)
    T = (K + 63) // 64
    acc = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    for s in range(S):
        k0, k1 = 64 * ((s * T) // S), min(K, 64 * (((s + 1) * T) // S))
        P = gemm(A[:, k0:k1].contiguous(), W[:, k0:k1].contiguous(), out_dtype=torch.float32, mode=bi.INVARIANT)
        acc = acc + P  # fp32, round to nearest: the order is the definition
    if out_dtype == torch.float32:
        return acc, S
    if R is not None:
        acc = acc + R.float()
    return acc.to(torch.bfloat16), S


@pytest.mark.parametrize("M", [1, 64, 128, 129, 300])
@pytest.mark.parametrize("N,K", [(256, 512), (512, 2048), (1032, 1000), (4096, 4096)])
def test_ksplit_equals_its_definition(M, N, K):
    A = synth.normal_device((M, K), 70 + M)
    W = synth.normal_device((N, K), 71 + N, std=0.02)
    R = synth.normal_device((M, N), 72)
    ref, S = by_definition(A, W, R)
    assert S > 1, "shape chosen to exercise the split"
    got = gemm(A, W, R=R)
    assert bits_equal(got, ref)
    ref32, _ = by_definition(A, W, out_dtype=torch.float32)
    assert bits_equal(gemm(A, W, out_dtype=torch.float32), ref32)


M_SWEEP = [1, 2, 3, 7, 16, 33, 64, 97, 128, 129, 256, 1023, 2048]


@pytest.mark.parametrize("N", [4096, 6144])
def test_ksplit_row0_bitwise_across_M(N):
    K = 4096
    W = synth.normal_device((N, K), 80 + N, std=0.02)
    target = cuda(synth.normal((1, K), 4321))
    ref = None
    for M in M_SWEEP:
        A = synth.normal_device((M, K), 2000 + M)
        A[0] = target[0]
        row = gemm(A, W)[0:1].clone()
        if ref is None:
            ref = row
        else:
            assert bits_equal(row, ref), "row 0 changed at M=%d" % M
    exact = oracle.round_bf16(f64(target) @ f64(W).T)
    assert max_rel_err(f64(ref), exact) <= TOL_BF16


@pytest.mark.parametrize("M,N,K", [(5, 4096, 4096), (64, 1032, 1000), (200, 512, 2048), (513, 640, 1536)])
def test_ksplit_parity_with_oracle(M, N, K):
    A = synth.normal((M, K), 90 + M)
    W = synth.normal((N, K), 91 + N, std=0.02)
    C = gemm(cuda(A), cuda(W))
    ref = oracle.round_bf16(oracle.gemm(f64(A), f64(W)))
    assert max_rel_err(f64(C), ref) <= TOL_BF16


@pytest.mark.parametrize("M", [64, 200])
def test_ksplit_single_part_is_invariant(M):
    N, K = 40000, 512  # 157 tiles of 256 columns: S = 1
    assert bi.bi_gemm_ksplit(N, K) == 1
    A = synth.normal_device((M, K), 95)
    W = synth.normal_device((N, K), 96, std=0.02)
    assert bits_equal(gemm(A, W), gemm(A, W, mode=bi.INVARIANT))


def test_ksplit_small_integers_exact():
    # every partial and every sum of partials is an integer below 2**24
    for M, N, K in [(3, 512, 2048), (150, 256, 1024)]:
        A = synth.small_ints((M, K), 13 + M)
        W = synth.small_ints((N, K), 14 + N)
        assert bi.bi_gemm_ksplit(N, K) > 1
        C = gemm(cuda(A), cuda(W), out_dtype=torch.float32)
        assert np.array_equal(f64(C), oracle.gemm(f64(A), f64(W)))
