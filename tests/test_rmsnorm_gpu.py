"""RMSNorm kernel: parity with the float64 oracle and bitwise batch invariance."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.helpers import TOL_BF16, TOL_F32, bits_equal, cuda, f64, max_rel_err

pytestmark = pytest.mark.gpu
bi = pytest.importorskip("invariant_deterministic_02_gb300")


def run(x, g, eps=1e-5, mode=bi.INVARIANT, tr=-1, tc=0):
    y = torch.empty_like(x)
    bi.bi_rmsnorm(x, g, y, eps, mode=mode, target_row=tr, target_count=tc)
    torch.cuda.synchronize()
    return y


@pytest.mark.parametrize("rows", [1, 2, 3, 8, 16])
def test_fp32_d512_parity(rows):
    x = synth.normal((rows, 512), 10 + rows, dtype=torch.float32)
    g = synth.normal((512,), 2, std=0.1, mean=1.0, dtype=torch.float32)
    y = run(cuda(x), cuda(g))
    ref = oracle.rmsnorm(f64(x), f64(g), 1e-5)
    assert max_rel_err(f64(y), ref) <= TOL_F32


@pytest.mark.parametrize("rows,d", [(1, 4096), (7, 4096), (300, 4096), (5, 8), (3, 16384), (33, 520)])
def test_bf16_parity(rows, d):
    x = synth.normal((rows, d), rows * 7 + d, dtype=torch.bfloat16)
    g = synth.normal((d,), 3, std=0.1, mean=1.0, dtype=torch.bfloat16)
    y = run(cuda(x), cuda(g))
    ref = oracle.round_bf16(oracle.rmsnorm(f64(x), f64(g), 1e-5))
    assert max_rel_err(f64(y), ref) <= TOL_BF16
    # and every output is one of the two bf16 neighbours of the exact value
    exact = oracle.rmsnorm(f64(x), f64(g), 1e-5)
    assert np.max(np.abs(f64(y) - exact) / np.maximum(np.abs(exact), 1e-30)) <= 2.0 ** -8 + 1e-6


def test_constant_rows_closed_form():
    d = 4096
    for c in (0.5, -3.0, 17.0):
        x = torch.full((4, d), c, dtype=torch.float32)
        g = torch.ones(d, dtype=torch.float32)
        y = f64(run(cuda(x), cuda(g), eps=1e-5))
        assert np.allclose(y, c / np.sqrt(c * c + 1e-5), rtol=2e-7, atol=0)


def test_target_row_bitwise_across_batch_compositions():
    d = 4096
    target = synth.normal((1, d), 1234, dtype=torch.bfloat16)
    g = cuda(synth.normal((d,), 5, std=0.1, mean=1.0, dtype=torch.bfloat16))
    ref = run(cuda(target), g)
    for trial, rows in enumerate([1, 2, 3, 64, 151, 152, 1000, 4097]):
        x = synth.normal((rows, d), 100 + trial, dtype=torch.bfloat16)
        pos = (trial * 37) % rows
        x[pos] = target[0]
        y = run(cuda(x), g)
        assert bits_equal(y[pos:pos + 1], ref), (rows, pos)
    # run to run
    assert bits_equal(run(cuda(target), g), ref)


def test_fast_mode_is_batch_dependent_and_protected_pins_target():
    d = 4096
    # fp32 rows: a changed reduction order shows in the output bits directly
    g = cuda(synth.normal((d,), 6, std=0.1, mean=1.0, dtype=torch.float32))
    diffs = 0
    for seed in range(8):
        t = synth.normal((1, d), 500 + seed, dtype=torch.float32)
        small = run(cuda(t), g, mode=bi.FAST)  # 1 row: split over many CTAs
        big_x = synth.normal((200, d), 600 + seed, dtype=torch.float32)
        big_x[0] = t[0]
        big = run(cuda(big_x), g, mode=bi.FAST)  # 200 rows: one CTA per row
        inv = run(cuda(t), g)
        assert bits_equal(big[0:1], inv)
        diffs += int(not bits_equal(small, big[0:1]))
        assert max_rel_err(f64(small), oracle.rmsnorm(f64(t), f64(g.cpu()), 1e-5)) <= TOL_F32
        # PROTECTED: the target row keeps the invariant bits inside a small (split) batch
        x = synth.normal((5, d), 700 + seed, dtype=torch.float32)
        x[2] = t[0]
        yp = run(cuda(x), g, mode=bi.PROTECTED, tr=2, tc=1)
        assert bits_equal(yp[2:3], inv)
        assert max_rel_err(f64(yp), oracle.rmsnorm(f64(x), f64(g.cpu()), 1e-5)) <= TOL_F32
    assert diffs > 0, "FAST mode never changed a row's bits: the negative control is vacuous"


def test_in_place_and_empty():
    x = cuda(synth.normal((9, 256), 8, dtype=torch.bfloat16))
    g = cuda(torch.ones(256, dtype=torch.bfloat16))
    ref = run(x.clone(), g)
    bi.bi_rmsnorm(x, g, x, 1e-5)
    torch.cuda.synchronize()
    assert bits_equal(x, ref)
    e = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    bi.bi_rmsnorm(e, g, e, 1e-5)
