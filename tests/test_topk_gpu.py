"""Deterministic top-k: exact agreement with the oracle's (value desc, index asc) order."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from tests.helpers import cuda

pytestmark = pytest.mark.gpu
bi = pytest.importorskip("invariant_deterministic_02_gb300")


def topk(logits, k):
    rows = logits.shape[0]
    tv = torch.empty((rows, k), dtype=torch.float32, device="cuda")
    ti = torch.empty((rows, k), dtype=torch.int32, device="cuda")
    bi.bi_topk(logits, k, tv, ti)
    torch.cuda.synchronize()
    return tv.cpu().numpy(), ti.cpu().numpy()


@pytest.mark.parametrize("k", [1, 5, 20, 32])
def test_topk_matches_oracle_with_ties(k):
    V = 151936
    x = synth.normal((6, V), 3, dtype=torch.float32)
    x = torch.round(x * 64) / 64  # many exact ties
    x[1, 1000:1040] = 9.0  # a tie block at the top
    x[2, :] = -1.0  # all equal
    x[3, V - 5:] = 50.0
    tv, ti = topk(cuda(x), k)
    ov, oi = oracle.topk(x.double().numpy(), k)
    assert np.array_equal(ti, oi)
    assert np.array_equal(tv.astype(np.float64), ov)
    assert list(ti[1][:min(k, 40)]) == list(range(1000, 1000 + min(k, 40)))
    assert list(ti[2]) == list(range(k))


def test_tie_example_from_page():
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "tie_logits.json")))
    x = torch.tensor([g["run1"], g["run2"]], dtype=torch.float32)
    _, ti = topk(cuda(x), 1)
    assert ti[:, 0].tolist() == g["expected_argmax_lowest_index"]


@pytest.mark.parametrize("V", [1, 7, 100, 513, 16385, 65536, 151935])
def test_topk_ragged_lengths(V):
    # lengths that leave warps without a segment, partial vector steps and (odd V) rows that
    # start off a 16-byte boundary, so the scalar tail path runs for whole rows
    k = min(20, V)
    x = synth.normal((5, V), 11, dtype=torch.float32)
    x = torch.round(x * 16) / 16
    x[4, :] = 0.5
    tv, ti = topk(cuda(x), k)
    ov, oi = oracle.topk(x.double().numpy(), k)
    assert np.array_equal(ti, oi)
    assert np.array_equal(tv.astype(np.float64), ov)
