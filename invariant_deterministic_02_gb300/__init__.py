"""Python binding of libbi, the batch-invariant transformer forward for GB300 (sm_103a).

Argument marshalling only: every function below forwards to the C entry point
of the same name in ``libbi.so`` (declared in ``include/bi.h``), passing torch
tensors as raw device pointers and the current torch stream.  All computation
runs in the library's CUDA kernels; there is no Python or CPU fallback, and
importing a function whose library is missing raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libbi.so")

BI_OK = 0
BI_ERR_INVALID_ARG = 1
BI_ERR_UNSUPPORTED = 2
BI_ERR_WORKSPACE = 3
BI_ERR_CUDA = 4
BI_ERR_TIMEOUT = 5

INVARIANT = 0
FAST = 1
PROTECTED = 2
INVARIANT_KSPLIT = 3
MODES = {"invariant": INVARIANT, "fast": FAST, "protected": PROTECTED, "invariant_ksplit": INVARIANT_KSPLIT}

BI_F32 = 0
BI_BF16 = 1

SPLIT_TOKENS = 256
PAGE_SIZE = 16
TOPK_MAX = 32

EXPORTED = [
    "bi_status_string", "bi_last_error_message", "bi_version", "bi_num_sms", "bi_device_error",
    "bi_debug_arm_gemm_stall", "bi_fast_gemm_plan", "bi_fast_attention_plan",
    "bi_rmsnorm_workspace", "bi_rmsnorm", "bi_gemm_workspace", "bi_gemm_ksplit", "bi_gemm",
    "bi_gemm_f32a_workspace", "bi_gemm_f32a",
    "bi_decode_attention_workspace", "bi_decode_attention", "bi_decode_attention_noalloc",
    "bi_prefill_attention_workspace",
    "bi_prefill_attention", "bi_embed", "bi_rope_table", "bi_qkv_rope_store", "bi_swiglu", "bi_gemm_swiglu_workspace",
    "bi_gemm_swiglu", "bi_topk",
    "bi_layer_workspace", "bi_layer_forward", "bi_model_workspace", "bi_model_forward",
    "bi_profile_start", "bi_profile_stop", "bi_profile_read", "bi_profile_kernel_name", "bi_profile_kernel_count",
]


class BiError(RuntimeError):
    def __init__(self, status: int, fn: str, detail: str):
        self.status = status
        super().__init__("%s failed: %s: %s" % (fn, _status_name(status), detail))


def _status_name(st):
    return {0: "BI_OK", 1: "BI_ERR_INVALID_ARG", 2: "BI_ERR_UNSUPPORTED", 3: "BI_ERR_WORKSPACE",
            4: "BI_ERR_CUDA", 5: "BI_ERR_TIMEOUT"}.get(st, "BI_ERR_%d" % st)


# ------------------------------------------------------------------ C structs
class AttnDims(ctypes.Structure):
    _fields_ = [("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("max_pages", ctypes.c_int32), ("num_pages", ctypes.c_int32),
                ("scale", ctypes.c_float), ("act_f32", ctypes.c_int32)]


class LayerWeights(ctypes.Structure):
    _fields_ = [("attn_norm", ctypes.c_void_p), ("w_qkv", ctypes.c_void_p), ("w_o", ctypes.c_void_p),
                ("ffn_norm", ctypes.c_void_p), ("w_gate_up", ctypes.c_void_p), ("w_down", ctypes.c_void_p),
                ("q_norm", ctypes.c_void_p), ("k_norm", ctypes.c_void_p)]


class ModelDims(ctypes.Structure):
    _fields_ = [("d_model", ctypes.c_int32), ("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("ffn_dim", ctypes.c_int32), ("vocab", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("max_pos", ctypes.c_int32), ("rms_eps", ctypes.c_float),
                ("act_f32", ctypes.c_int32)]


class Batch(ctypes.Structure):
    _fields_ = [("num_requests", ctypes.c_int32), ("num_tokens", ctypes.c_int32), ("max_q_len", ctypes.c_int32),
                ("q_start", ctypes.c_void_p), ("pos0", ctypes.c_void_p), ("block_table", ctypes.c_void_p),
                ("max_pages", ctypes.c_int32), ("num_pages", ctypes.c_int32), ("target_request", ctypes.c_int32),
                ("target_row", ctypes.c_int32), ("target_count", ctypes.c_int32)]


class ModelWeights(ctypes.Structure):
    _fields_ = [("embed", ctypes.c_void_p), ("layers", ctypes.POINTER(LayerWeights)), ("num_layers", ctypes.c_int32),
                ("final_norm", ctypes.c_void_p), ("lm_head", ctypes.c_void_p)]


# ------------------------------------------------------------------ library loading
_lib = None


def _declare(lib):
    c_i32, c_i64, c_sz, c_f, c_d, vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float, \
        ctypes.c_double, ctypes.c_void_p
    P = ctypes.POINTER
    sig = {
        "bi_status_string": (ctypes.c_char_p, [c_i32]),
        "bi_last_error_message": (ctypes.c_char_p, []),
        "bi_version": (c_i32, []),
        "bi_num_sms": (c_i32, []),
        "bi_device_error": (c_i32, [P(c_i32), vp]),
        "bi_debug_arm_gemm_stall": (c_i32, [c_i64]),
        "bi_fast_gemm_plan": (c_i32, [c_i64, c_i64, c_i64, c_i32]),
        "bi_fast_attention_plan": (c_i32, [c_i32]),
        "bi_rmsnorm_workspace": (c_sz, [c_i64, c_i64, c_i32]),
        "bi_rmsnorm": (c_i32, [vp, vp, vp, c_i64, c_i64, c_i32, c_f, c_i32, c_i32, c_i32, vp, c_sz, vp]),
        "bi_gemm_workspace": (c_sz, [c_i64, c_i64, c_i64, c_i32]),
        "bi_gemm_ksplit": (c_i32, [c_i64, c_i64]),
        "bi_gemm": (c_i32, [vp, vp, vp, vp, c_i64, c_i64, c_i64, c_i32, c_i32, c_i32, c_i32, vp, c_sz, vp]),
        "bi_gemm_f32a_workspace": (c_sz, [c_i64, c_i64, c_i64, c_i32]),
        "bi_gemm_f32a": (c_i32, [vp, vp, vp, vp, c_i64, c_i64, c_i64, c_i32, c_i32, c_i32, vp, c_sz, vp]),
        "bi_decode_attention_workspace": (c_sz, [c_i32, P(AttnDims), c_i32]),
        "bi_decode_attention": (c_i32, [vp, vp, vp, vp, vp, c_i32, P(AttnDims), vp, c_i32, c_i32, vp, c_sz, vp]),
        "bi_decode_attention_noalloc": (c_i32, [vp, vp, vp, vp, vp, c_i32, P(AttnDims), vp, c_i32, c_i32, vp]),
        "bi_prefill_attention_workspace": (c_sz, [c_i32, c_i32, P(AttnDims), c_i32]),
        "bi_prefill_attention": (c_i32, [vp, vp, vp, vp, vp, vp, c_i32, c_i32, P(AttnDims), vp, c_i32, c_i32, vp,
                                         c_sz, vp]),
        "bi_embed": (c_i32, [vp, vp, vp, c_i64, c_i64, c_i64, vp]),
        "bi_rope_table": (c_i32, [c_d, c_i32, c_i32, vp, vp, vp]),
        "bi_qkv_rope_store": (c_i32, [vp, vp, vp, vp, vp, vp, c_i32, P(AttnDims), vp, vp, vp, vp]),
        "bi_swiglu": (c_i32, [vp, vp, c_i64, c_i64, vp]),
        "bi_gemm_swiglu_workspace": (c_sz, [c_i64, c_i64, c_i64, c_i32]),
        "bi_gemm_swiglu": (c_i32, [vp, vp, vp, c_i64, c_i64, c_i64, c_i32, c_i32, c_i32, vp, c_sz, vp]),
        "bi_topk": (c_i32, [vp, c_i64, c_i64, c_i32, vp, vp, vp]),
        "bi_layer_workspace": (c_sz, [P(ModelDims), P(Batch), c_i32]),
        "bi_layer_forward": (c_i32, [P(ModelDims), P(LayerWeights), vp, vp, vp, P(Batch), vp, vp, c_i32, vp, c_sz,
                                     vp]),
        "bi_model_workspace": (c_sz, [P(ModelDims), P(Batch), c_i32]),
        "bi_model_forward": (c_i32, [P(ModelDims), P(ModelWeights), vp, vp, vp, P(Batch), P(vp), P(vp), vp, c_i32,
                                     vp, vp, vp, c_i32, vp, c_sz, vp]),
        "bi_profile_start": (c_i32, [c_i32]),
        "bi_profile_stop": (c_i32, []),
        "bi_profile_read": (c_i32, [ctypes.c_char_p, P(c_i32), P(ctypes.c_double)]),
        "bi_profile_kernel_name": (ctypes.c_char_p, [c_i32]),
        "bi_profile_kernel_count": (c_i32, []),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args


def lib():
    """The loaded libbi.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libbi.so is missing at %s: build it with "
                               "`python -m invariant_deterministic_02_gb300.build`" % LIB_PATH)
        l = ctypes.CDLL(LIB_PATH)
        _declare(l)
        _lib = l
    return _lib


def _check(st: int, fn: str):
    if st != BI_OK:
        raise BiError(st, fn, lib().bi_last_error_message().decode(errors="replace"))


def _p(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _ws(nbytes: int, device, workspace):
    if nbytes == 0:
        return None, 0
    if workspace is not None:
        return workspace, workspace.numel() * workspace.element_size()
    return torch.empty(nbytes, dtype=torch.uint8, device=device), nbytes


def _mode(m):
    return MODES[m] if isinstance(m, str) else int(m)


# ------------------------------------------------------------------ wrappers
def bi_num_sms() -> int:
    return int(lib().bi_num_sms())


def bi_device_error(stream=None) -> int:
    """Synchronises, reads and clears the kernels' device error words: 0, or the
    site code of the first in-kernel wait that ran out (1-15) or of the first
    out-of-range KV length, block-table entry or position a kernel met (>= 16)."""
    code = ctypes.c_int32(0)
    st = lib().bi_device_error(ctypes.byref(code), _stream(stream))
    if st not in (BI_OK, BI_ERR_TIMEOUT, BI_ERR_INVALID_ARG) or (st != BI_OK and code.value == 0):
        _check(st, "bi_device_error")
    return int(code.value)


def bi_fast_gemm_plan(M: int, N: int, K: int, plan: int):
    """FAST-mode GEMMs of shape (M, N, K): 1 = INVARIANT's tile plan (no split-K), 0 = FAST's own rule."""
    _check(lib().bi_fast_gemm_plan(M, N, K, plan), "bi_fast_gemm_plan")


def bi_fast_attention_plan(plan: int):
    """FAST decode attention: 1 = the 256-token splits, 0 = the occupancy-chosen unit count."""
    _check(lib().bi_fast_attention_plan(plan), "bi_fast_attention_plan")


def bi_debug_arm_gemm_stall(wait_ns: int):
    """Test hook: the next bi_gemm of this thread drops one stage's copies and its
    waits give up after wait_ns (see include/bi.h)."""
    _check(lib().bi_debug_arm_gemm_stall(int(wait_ns)), "bi_debug_arm_gemm_stall")


def bi_rmsnorm(x, gamma, y, eps: float, mode=INVARIANT, target_row=-1, target_count=0, workspace=None,
               stream=None):
    rows, d = x.shape[0], x.shape[-1]
    dt = BI_BF16 if x.dtype == torch.bfloat16 else BI_F32
    m = _mode(mode)
    need = lib().bi_rmsnorm_workspace(rows, d, m)
    ws, nb = _ws(need, x.device, workspace)
    _check(lib().bi_rmsnorm(_p(x), _p(gamma), _p(y), rows, d, dt, eps, m, target_row, target_count, _p(ws), nb,
                            _stream(stream)), "bi_rmsnorm")
    return y


def bi_gemm_ksplit(N: int, K: int) -> int:
    """Part count of the INVARIANT_KSPLIT GEMM for an N x K weight."""
    return int(lib().bi_gemm_ksplit(N, K))


def bi_gemm(A, W, C, residual=None, mode=INVARIANT, target_row=-1, target_count=0, workspace=None, stream=None):
    M, K = A.shape
    N = W.shape[0]
    dt = BI_F32 if C.dtype == torch.float32 else BI_BF16
    m = _mode(mode)
    need = lib().bi_gemm_workspace(M, N, K, m)
    ws, nb = _ws(need, A.device, workspace)
    _check(lib().bi_gemm(_p(A), _p(W), _p(C), _p(residual), M, N, K, dt, m, target_row, target_count, _p(ws), nb,
                         _stream(stream)), "bi_gemm")
    return C


def bi_gemm_f32a(A, W, C, residual=None, mode=INVARIANT, target_row=-1, target_count=0, workspace=None,
                 stream=None):
    """fp32 A [M][K] times bf16 W [N][K] into fp32 C (+ fp32 residual)."""
    if A.dtype != torch.float32 or C.dtype != torch.float32 or W.dtype != torch.bfloat16 or \
            (residual is not None and residual.dtype != torch.float32):
        raise TypeError("bi_gemm_f32a: A, C (and residual) must be float32 and W bfloat16")
    M, K = A.shape
    N = W.shape[0]
    m = _mode(mode)
    need = lib().bi_gemm_f32a_workspace(M, N, K, m)
    ws, nb = _ws(need, A.device, workspace)
    _check(lib().bi_gemm_f32a(_p(A), _p(W), _p(C), _p(residual), M, N, K, m, target_row, target_count, _p(ws), nb,
                              _stream(stream)), "bi_gemm_f32a")
    return C


def attn_dims(num_q_heads, num_kv_heads, head_dim, max_pages, num_pages, scale=None) -> AttnDims:
    return AttnDims(num_q_heads, num_kv_heads, head_dim, PAGE_SIZE, max_pages, num_pages,
                    (1.0 / head_dim ** 0.5) if scale is None else scale, 0)


def _dims_for(dims: AttnDims, q) -> AttnDims:
    """A copy of dims whose act_f32 follows the dtype of q (fp32 q and out, or bf16)."""
    d = AttnDims.from_buffer_copy(dims)
    d.act_f32 = 1 if q.dtype == torch.float32 else 0
    return d


def bi_decode_attention(q, k_cache, v_cache, block_table, kv_lens, dims: AttnDims, out, mode=INVARIANT,
                        target_request=-1, workspace=None, stream=None):
    B = q.shape[0]
    m = _mode(mode)
    dims = _dims_for(dims, q)
    need = lib().bi_decode_attention_workspace(B, ctypes.byref(dims), m)
    ws, nb = _ws(need, q.device, workspace)
    _check(lib().bi_decode_attention(_p(q), _p(k_cache), _p(v_cache), _p(block_table), _p(kv_lens), B,
                                     ctypes.byref(dims), _p(out), m, target_request, _p(ws), nb, _stream(stream)),
           "bi_decode_attention")
    return out


def bi_decode_attention_noalloc(q, k_cache, v_cache, block_table, kv_lens, dims: AttnDims, out, mode=INVARIANT,
                                target_request=-1, stream=None):
    """bi_decode_attention without a workspace: the library serves the scratch from a
    fixed 16 MiB device array of its own (for callers that cannot allocate)."""
    dims = _dims_for(dims, q)
    _check(lib().bi_decode_attention_noalloc(_p(q), _p(k_cache), _p(v_cache), _p(block_table), _p(kv_lens),
                                             q.shape[0], ctypes.byref(dims), _p(out), _mode(mode), target_request,
                                             _stream(stream)), "bi_decode_attention_noalloc")
    return out


def bi_prefill_attention(q, k_cache, v_cache, block_table, q_start, q_pos0, dims: AttnDims, out, mode=INVARIANT,
                         target_request=-1, workspace=None, stream=None):
    T = q.shape[0]
    B = q_pos0.shape[0]
    m = _mode(mode)
    dims = _dims_for(dims, q)
    need = lib().bi_prefill_attention_workspace(B, T, ctypes.byref(dims), m)
    ws, nb = _ws(need, q.device, workspace)
    _check(lib().bi_prefill_attention(_p(q), _p(k_cache), _p(v_cache), _p(block_table), _p(q_start), _p(q_pos0), B,
                                      T, ctypes.byref(dims), _p(out), m, target_request, _p(ws), nb,
                                      _stream(stream)), "bi_prefill_attention")
    return out


def bi_embed(ids, table, out, stream=None):
    _check(lib().bi_embed(_p(ids), _p(table), _p(out), ids.shape[0], table.shape[1], table.shape[0],
                          _stream(stream)), "bi_embed")
    return out


def bi_rope_table(theta: float, head_dim: int, max_pos: int, cos_out, sin_out, stream=None):
    _check(lib().bi_rope_table(float(theta), head_dim, max_pos, _p(cos_out), _p(sin_out), _stream(stream)),
           "bi_rope_table")


def bi_qkv_rope_store(qkv, rope_cos, rope_sin, token_pos, token_req, block_table, dims: AttnDims, q_out, k_cache,
                      v_cache, stream=None):
    _check(lib().bi_qkv_rope_store(_p(qkv), _p(rope_cos), _p(rope_sin), _p(token_pos), _p(token_req),
                                   _p(block_table), qkv.shape[0], ctypes.byref(dims), _p(q_out), _p(k_cache),
                                   _p(v_cache), _stream(stream)), "bi_qkv_rope_store")


def bi_swiglu(gu, out, stream=None):
    T, F2 = gu.shape
    _check(lib().bi_swiglu(_p(gu), _p(out), T, F2 // 2, _stream(stream)), "bi_swiglu")
    return out


def bi_gemm_swiglu(A, W_gate_up, act, mode=INVARIANT, target_row=-1, target_count=0, workspace=None,
                   stream=None):
    """act [M][F] = SwiGLU of A [M][K] times W_gate_up [2F][K] (gate rows, then up rows), bf16."""
    M, K = A.shape
    F = W_gate_up.shape[0] // 2
    m = _mode(mode)
    need = lib().bi_gemm_swiglu_workspace(M, F, K, m)
    ws, nb = _ws(need, A.device, workspace)
    _check(lib().bi_gemm_swiglu(_p(A), _p(W_gate_up), _p(act), M, F, K, m, target_row, target_count, _p(ws), nb,
                                _stream(stream)), "bi_gemm_swiglu")
    return act


def bi_topk(logits, k: int, top_v, top_i, stream=None):
    rows, V = logits.shape
    _check(lib().bi_topk(_p(logits), rows, V, k, _p(top_v), _p(top_i), _stream(stream)), "bi_topk")
    return top_v, top_i


def bi_layer_workspace(dims: ModelDims, batch: Batch, mode=INVARIANT) -> int:
    return int(lib().bi_layer_workspace(ctypes.byref(dims), ctypes.byref(batch), _mode(mode)))


def bi_layer_forward(dims: ModelDims, weights: LayerWeights, rope_cos, rope_sin, hidden, batch: Batch, k_cache,
                     v_cache, mode=INVARIANT, workspace=None, stream=None):
    m = _mode(mode)
    need = lib().bi_layer_workspace(ctypes.byref(dims), ctypes.byref(batch), m)
    ws, nb = _ws(need, hidden.device, workspace)
    _check(lib().bi_layer_forward(ctypes.byref(dims), ctypes.byref(weights), _p(rope_cos), _p(rope_sin), _p(hidden),
                                  ctypes.byref(batch), _p(k_cache), _p(v_cache), m, _p(ws), nb, _stream(stream)),
           "bi_layer_forward")
    return hidden


def bi_model_workspace(dims: ModelDims, batch: Batch, mode=INVARIANT) -> int:
    return int(lib().bi_model_workspace(ctypes.byref(dims), ctypes.byref(batch), _mode(mode)))


def bi_model_forward(dims: ModelDims, weights: ModelWeights, rope_cos, rope_sin, ids, batch: Batch, k_ptrs, v_ptrs,
                     logits, k: int, top_v, top_i, greedy_ids=None, mode=INVARIANT, workspace=None, ws_bytes=None,
                     stream=None):
    """k_ptrs / v_ptrs: ctypes arrays (c_void_p * num_layers) of per-layer cache pointers."""
    m = _mode(mode)
    if workspace is None:
        need = lib().bi_model_workspace(ctypes.byref(dims), ctypes.byref(batch), m)
        workspace, ws_bytes = _ws(need, ids.device, None)
    elif ws_bytes is None:
        ws_bytes = workspace.numel() * workspace.element_size()
    _check(lib().bi_model_forward(ctypes.byref(dims), ctypes.byref(weights), _p(rope_cos), _p(rope_sin), _p(ids),
                                  ctypes.byref(batch), k_ptrs, v_ptrs, _p(logits), k, _p(top_v), _p(top_i),
                                  _p(greedy_ids), m, _p(workspace), ws_bytes, _stream(stream)), "bi_model_forward")


def bi_profile_start(max_launches: int):
    _check(lib().bi_profile_start(max_launches), "bi_profile_start")


def bi_profile_stop():
    _check(lib().bi_profile_stop(), "bi_profile_stop")


def bi_profile_read(kernel: str):
    """(launches, total milliseconds) of the kernel tag since bi_profile_start."""
    n = ctypes.c_int32(0)
    ms = ctypes.c_double(0.0)
    _check(lib().bi_profile_read(kernel.encode(), ctypes.byref(n), ctypes.byref(ms)), "bi_profile_read")
    return int(n.value), float(ms.value)


def bi_profile_kernels():
    l = lib()
    return [l.bi_profile_kernel_name(i).decode() for i in range(l.bi_profile_kernel_count())]
