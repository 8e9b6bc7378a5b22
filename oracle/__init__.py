"""Plain float64 CPU oracle for the batch-invariant transformer forward.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or link
anything in this package: only the test-suite, the smoke check and the bench's
CPU-baseline / reference arm use it.  It shares no code with the CUDA library
(no kernels, headers, tables, helpers or pre-/post-processing); the only thing
both sides consume is the seeded input data produced by ``synth``.

Every function here is the plain mathematical definition of one step, written
in float64 with numpy (library matmul/sort used as single steps, nothing
blocked, fused or reordered).  Split-KV partials and their merge tree are NOT
modelled: they only reorder an exact sum, so the oracle is the unsplit
softmax.  Where the pages leave a step open the reading taken is noted inline.

Pins (see tests/test_oracle_pins.py): every function is checked against
closed forms, worked examples printed on the pages, invariants and brute force
written independently of this module.
"""
from .core import (  # noqa: F401
    round_bf16,
    round_f32,
    rmsnorm,
    gemm,
    rope_inv_freq,
    rope,
    gather_pages,
    attention,
    silu,
    swiglu,
    topk,
    argmax,
    OracleKV,
    layer_forward,
    model_forward,
    split_geometry,
    split_partials,
)
