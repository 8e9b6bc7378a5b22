"""tcgen05 GEMM: parity with the float64 oracle, bitwise invariance across M, modes."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.helpers import TOL_BF16, bits_equal, cuda, f64, max_rel_err

pytestmark = pytest.mark.gpu
bi = pytest.importorskip("invariant_deterministic_02_gb300")


def gemm(A, W, out_dtype=torch.bfloat16, R=None, mode=bi.INVARIANT, tr=-1, tc=0):
    C = torch.empty((A.shape[0], W.shape[0]), dtype=out_dtype, device="cuda")
    bi.bi_gemm(A, W, C, residual=R, mode=mode, target_row=tr, target_count=tc)
    torch.cuda.synchronize()
    return C


@pytest.mark.parametrize("M,N,K", [(1, 8, 16), (3, 64, 64), (128, 64, 128), (200, 136, 520), (17, 512, 1024),
                                   (300, 264, 72)])
def test_small_integers_exact(M, N, K):
    A = synth.small_ints((M, K), 11 + M)
    W = synth.small_ints((N, K), 12 + N)
    C = gemm(cuda(A), cuda(W), out_dtype=torch.float32)
    ref = oracle.gemm(f64(A), f64(W))
    assert np.array_equal(f64(C), ref)  # every partial sum is an integer below 2**24


def test_one_hot_weights_select_columns_exactly():
    M, K = 130, 256
    A = synth.normal((M, K), 3)
    W = torch.zeros((64, K), dtype=torch.bfloat16)
    for j in range(64):
        W[j, (j * 5) % K] = 1.0
    C = gemm(cuda(A), cuda(W))
    for j in range(64):
        assert bits_equal(C[:, j].cpu(), A[:, (j * 5) % K])


@pytest.mark.parametrize("M,N,K", [(1, 512, 512), (8, 512, 512), (16, 512, 512), (33, 512, 512), (64, 4096, 4096),
                                   (48, 1024, 12288), (97, 4096, 4096), (256, 1024, 4096), (513, 640, 1536)])
def test_random_parity_bf16(M, N, K):
    A = synth.normal((M, K), 20 + M)
    W = synth.normal((N, K), 21 + N, std=0.02)
    C = gemm(cuda(A), cuda(W))
    ref = oracle.round_bf16(oracle.gemm(f64(A), f64(W)))
    assert max_rel_err(f64(C), ref) <= TOL_BF16


def test_residual_and_fp32_output():
    M, N, K = 70, 320, 640
    A = synth.normal((M, K), 31)
    W = synth.normal((N, K), 32, std=0.02)
    R = synth.normal((M, N), 33)
    C = gemm(cuda(A), cuda(W), R=cuda(R))
    exact = oracle.gemm(f64(A), f64(W))
    assert max_rel_err(f64(C), oracle.round_bf16(exact + f64(R))) <= TOL_BF16
    C32 = gemm(cuda(A), cuda(W), out_dtype=torch.float32)
    assert np.max(np.abs(f64(C32) - exact)) <= 1e-5 * np.max(np.abs(exact)) * 4
    # in place: C aliases the residual
    Rc = cuda(R)
    bi.bi_gemm(cuda(A), cuda(W), Rc, residual=Rc)
    torch.cuda.synchronize()
    assert bits_equal(Rc, C)


M_SWEEP = [1, 2, 3, 4, 7, 8, 16, 32, 64, 97, 128, 256, 512, 1023, 1024, 2048, 4096]


@pytest.mark.parametrize("N", [4096, 14336, 151936])
def test_row0_bitwise_across_M_sweep(N):
    K = 4096
    W = synth.normal_device((N, K), 40 + N, std=0.02)
    target = synth.normal((1, K), 1234)
    ref = None
    for M in M_SWEEP:
        A = synth.normal_device((M, K), 1000 + M)
        A[0] = cuda(target)[0]
        C = gemm(A, W, out_dtype=torch.float32 if N == 151936 else torch.bfloat16)
        row = C[0:1].clone()
        if ref is None:
            ref = row
        else:
            assert bits_equal(row, ref), "row 0 changed at M=%d" % M
        del A, C
    # row 0 against the oracle on a sample of columns
    cols = torch.randperm(N, generator=torch.Generator().manual_seed(5))[:2048]
    Ws = f64(W[cols.to("cuda")])
    exact = f64(target) @ Ws.T
    got = f64(ref[0, cols.to("cuda")])
    if N != 151936:
        exact = oracle.round_bf16(exact)
    assert max_rel_err(got, exact) <= TOL_BF16


@pytest.mark.parametrize("N,K", [(4096, 4096), (6144, 4096), (4096, 12288)])
def test_every_row_bitwise_across_instruction_heights(N, K):
    # M <= 64 runs M = 64 instructions (16 accumulator rows per lane quarter), 64 < M <= 128 M = 128
    # instructions on one SM, larger M the SM-pair kernel: every row of the small product must come out
    # of all three with the same bits (a wrong row-to-lane map would move rows 16..63)
    W = synth.normal_device((N, K), 70 + N + K, std=0.02)
    big = synth.normal_device((300, K), 71)
    ref = gemm(big, W, out_dtype=torch.float32)
    for M in (17, 40, 64, 100, 128):
        C = gemm(big[:M].contiguous(), W, out_dtype=torch.float32)
        assert bits_equal(C, ref[:M]), "rows changed at M=%d" % M


def test_run_to_run_deterministic_2048():
    A = synth.normal_device((2048, 2048), 50)
    W = synth.normal_device((2048, 2048), 51, std=0.02)
    C1 = gemm(A, W, out_dtype=torch.float32)
    C2 = gemm(A, W, out_dtype=torch.float32)
    assert bits_equal(C1, C2)


def test_fast_split_k_positive_control_linspace():
    # the linspace(-1000, 1000) matrices of the matmul example: row 0 alone vs row 0 of the full batch
    B, D = 2048, 4096
    a = cuda(synth.linspace_control(B, D))
    b = cuda(synth.linspace_control(D, D))
    inv1 = gemm(a[:1], b, out_dtype=torch.float32)
    inv2 = gemm(a, b, out_dtype=torch.float32)[:1]
    assert bits_equal(inv1, inv2)
    fast1 = gemm(a[:1], b, out_dtype=torch.float32, mode=bi.FAST)
    fast2 = gemm(a, b, out_dtype=torch.float32, mode=bi.FAST)[:1]
    assert bits_equal(fast2, inv2)  # enough tiles: no split, same schedule
    assert not bits_equal(fast1, fast2), "split-K never changed row 0: the control is vacuous"
    exact = f64(a[:1].cpu()) @ f64(b.cpu()).T
    assert max_rel_err(f64(fast1), exact) <= 1e-3


def test_protected_target_tile_keeps_invariant_bits():
    M, N, K = 300, 512, 2048
    A = synth.normal((M, K), 60)
    W = cuda(synth.normal((N, K), 61, std=0.02))
    inv = gemm(cuda(A), W, out_dtype=torch.float32)
    fast = gemm(cuda(A), W, out_dtype=torch.float32, mode=bi.FAST)
    prot = gemm(cuda(A), W, out_dtype=torch.float32, mode=bi.PROTECTED, tr=140, tc=3)
    assert bits_equal(prot[128:256], inv[128:256])  # the tile holding rows 140..142 is never split
    assert not bits_equal(fast, inv)
    exact = oracle.gemm(f64(A), f64(W.cpu()))
    for C in (fast, prot):
        assert np.max(np.abs(f64(C) - exact)) <= 1e-4 * np.max(np.abs(exact))
    # target's bits independent of the batch it sits in
    A2 = synth.normal((40, K), 62)
    A2[7] = A[141]
    p2 = gemm(cuda(A2), W, out_dtype=torch.float32, mode=bi.PROTECTED, tr=7, tc=1)
    assert bits_equal(p2[7:8], inv[141:142])


@pytest.mark.parametrize("N,out_dtype", [(4096, torch.float32), (14336, torch.bfloat16)])
def test_multiwave_large_m_elementwise_parity(N, out_dtype):
    # M = 4096 spans several waves of the persistent tile loop, so CTAs reuse both tensor-memory
    # accumulators and flip every stage's phase many times; 64 sampled rows >= 128 (every column) are
    # compared with the float64 product
    M, K = 4096, 4096
    A = synth.normal_device((M, K), 70)
    W = synth.normal_device((N, K), 71, std=0.02)
    C = gemm(A, W, out_dtype=out_dtype)
    rows = torch.randperm(M - 128, generator=torch.Generator().manual_seed(72))[:63] + 128
    rows = torch.cat([rows, torch.tensor([M - 1])]).sort().values
    exact = oracle.gemm(f64(A[rows.to("cuda")]), f64(W))
    got = f64(C[rows.to("cuda")])
    if out_dtype == torch.bfloat16:
        assert max_rel_err(got, oracle.round_bf16(exact)) <= TOL_BF16
    else:
        assert np.max(np.abs(got - exact)) <= 1e-4 * np.max(np.abs(exact))


def test_bounded_wait_runs_out_and_the_next_call_is_clean():
    # The test hook drops the copies of one stage in CTA 0 and shortens every wait of that launch to
    # 100 ms: the wait for the missing stage runs out, the kernel stops all roles, drains and frees its
    # tensor memory, and reports a GEMM site code; the next launch is unaffected.
    M, N, K = 256, 1024, 2048
    A = cuda(synth.normal((M, K), 80))
    W = cuda(synth.normal((N, K), 81, std=0.02))
    bi.bi_device_error()  # start from clear error words
    ref = gemm(A, W, out_dtype=torch.float32)
    assert bi.bi_device_error() == 0
    bi.bi_debug_arm_gemm_stall(100_000_000)
    gemm(A, W, out_dtype=torch.float32)
    code = bi.bi_device_error()
    assert code in (1, 2, 3, 4), code
    again = gemm(A, W, out_dtype=torch.float32)
    assert bi.bi_device_error() == 0
    assert bits_equal(again, ref)


def test_device_error_word_clear_after_normal_runs():
    A = cuda(synth.normal((5, 64), 1))
    W = cuda(synth.normal((64, 64), 2))
    gemm(A, W)
    assert bi.bi_device_error() == 0
