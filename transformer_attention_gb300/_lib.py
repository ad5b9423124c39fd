"""ctypes binding of libgemma3attn.so: same names as the C ABI in include/gemma3_attn.h.

The functions here only marshal arguments (tensor -> device pointer, torch's
current CUDA stream -> cudaStream_t) and turn a non-zero status into an
exception.  All computation runs in the library's CUDA kernels; there is no
fallback: if the library is missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os

from .build import LIB

c_int, c_long, c_double, c_float, c_size_t, c_void_p = (
    ctypes.c_int, ctypes.c_long, ctypes.c_double, ctypes.c_float, ctypes.c_size_t, ctypes.c_void_p)

GEMMA3_OK = 0
GEMMA3_ERR_TIMEOUT = -5
GEMMA3_ERR_BAD_INPUT = -7
GEMMA3_LOCAL_SLIDING, GEMMA3_GLOBAL = 0, 1
GEMMA3_BF16, GEMMA3_F16, GEMMA3_F32 = 0, 1, 2
MODEL_SIZES = {"270M": 0, "1B": 1, "4B": 2, "12B": 3, "27B": 4}


class gemma3_attn_dims(ctypes.Structure):
    _fields_ = [("B", c_int), ("T", c_int), ("D", c_int), ("H", c_int), ("H_kv", c_int),
                ("d_h", c_int)]


class gemma3_block_weights(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in (
        "Wq", "Wkv", "Wo", "gamma_q", "gamma_k", "gamma_pre_attn", "gamma_post_attn",
        "gamma_pre_ffn", "gamma_post_ffn", "W_gating", "W_down")]


# name -> (restype, argtypes); mirrors include/gemma3_attn.h
SIGNATURES = {
    "gemma3_layer_attn_type": (c_int, [c_int, c_int]),
    "gemma3_layer_config": (c_int, [c_int, c_int, c_int, ctypes.POINTER(c_int),
                                    ctypes.POINTER(c_int), ctypes.POINTER(c_double),
                                    ctypes.POINTER(c_double)]),
    "gemma3_query_scale": (c_int, [c_int, c_int, c_int, c_int, ctypes.POINTER(c_float)]),
    "gemma3_attn_workspace_size": (c_int, [ctypes.POINTER(gemma3_attn_dims),
                                           ctypes.POINTER(c_size_t)]),
    "gemma3_attn_forward": (c_int, [ctypes.POINTER(gemma3_attn_dims), c_void_p, c_void_p, c_void_p,
                                    c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int,
                                    c_double, c_double, c_float, c_void_p, c_void_p, c_size_t,
                                    c_void_p]),
    "gemma3_attn_forward_noalloc": (c_int, [ctypes.POINTER(gemma3_attn_dims), c_void_p, c_void_p,
                                            c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                            c_void_p, c_int, c_int, c_double, c_double, c_float,
                                            c_void_p, c_void_p]),
    "gemma3_attn_noalloc_max_scratch": (c_size_t, []),
    "gemma3_block_attn_workspace_size": (c_int, [ctypes.POINTER(gemma3_attn_dims),
                                                 ctypes.POINTER(c_size_t)]),
    "gemma3_block_attn_forward": (c_int, [ctypes.POINTER(gemma3_attn_dims), c_void_p, c_int,
                                          c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                          c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int,
                                          c_int, c_double, c_double, c_float, c_void_p, c_size_t,
                                          c_void_p]),
    "gemma3_block_ffn_workspace_size": (c_int, [c_int, c_int, c_int, ctypes.POINTER(c_size_t)]),
    "gemma3_block_ffn_forward": (c_int, [c_int, c_int, c_int, c_void_p, c_void_p, c_void_p,
                                         c_void_p, c_void_p, c_void_p, c_void_p, c_size_t,
                                         c_void_p]),
    "gemma3_block_workspace_size": (c_int, [ctypes.POINTER(gemma3_attn_dims), c_int,
                                            ctypes.POINTER(c_size_t)]),
    "gemma3_block_forward": (c_int, [ctypes.POINTER(gemma3_attn_dims), c_int, c_void_p, c_int,
                                     c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                     c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                     c_void_p, c_void_p, c_int, c_int, c_double, c_double,
                                     c_float, c_void_p, c_size_t, c_void_p]),
    "gemma3_model_workspace_size": (c_int, [ctypes.POINTER(gemma3_attn_dims), c_int, c_int,
                                            ctypes.POINTER(c_size_t)]),
    "gemma3_model_forward": (c_int, [ctypes.POINTER(gemma3_attn_dims), c_int, c_int, c_int, c_int,
                                     c_void_p, c_void_p, c_void_p, c_void_p,
                                     ctypes.POINTER(gemma3_block_weights), c_void_p, c_void_p,
                                     c_void_p, c_size_t, c_void_p]),
    "gemma3_embed": (c_int, [c_void_p, c_void_p, c_int, c_int, c_int, c_float, c_void_p,
                             c_void_p]),
    "gemma3_attn_cached_workspace_size": (c_int, [ctypes.POINTER(gemma3_attn_dims), c_int,
                                                  ctypes.POINTER(c_size_t)]),
    "gemma3_attn_forward_cached": (c_int, [ctypes.POINTER(gemma3_attn_dims), c_int, c_int,
                                           c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                           c_void_p, c_void_p, c_void_p, c_int, c_int, c_double,
                                           c_double, c_float, c_void_p, c_void_p, c_void_p,
                                           c_void_p, c_void_p, c_size_t, c_void_p]),
    "gemma3_kv_cache_write": (c_int, [c_void_p, c_void_p, c_long, c_void_p, c_void_p, c_int,
                                      c_int, c_int, c_int, c_int, c_int, c_void_p, c_void_p,
                                      c_void_p, c_void_p]),
    "gemma3_cached_attention_workspace_size": (c_int, [c_int, c_int, c_int, c_int, c_int, c_int,
                                                       ctypes.POINTER(c_size_t)]),
    "gemma3_cached_attention": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                        c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int,
                                        c_int, c_int, c_int, c_int, c_void_p, c_size_t,
                                        c_void_p]),
    "gemma3_geglu": (c_int, [c_void_p, c_long, c_void_p, c_long, c_void_p, c_long, c_int, c_int,
                             c_int, c_int, c_void_p]),
    "gemma3_linear": (c_int, [c_void_p, c_long, c_void_p, c_long, c_void_p, c_long, c_int, c_int,
                              c_int, c_int, c_int, c_int, c_void_p, c_int, c_void_p]),
    "gemma3_qkv_proj_norm_rope": (c_int, [c_void_p, c_long, c_void_p, c_void_p, c_void_p,
                                          c_void_p, c_int, c_int, c_int, c_int, c_int, c_int,
                                          c_void_p, c_void_p, c_void_p, c_double, c_double,
                                          c_float, c_void_p, c_int, c_void_p]),
    "gemma3_linear_qk_norm_rope": (c_int, [c_void_p, c_long, c_void_p, c_long, c_void_p, c_long,
                                           c_int, c_int, c_int, c_int, c_void_p, c_void_p, c_int,
                                           c_int, c_double, c_double, c_float, c_void_p]),
    "gemma3_cast_bf16_f16": (c_int, [c_void_p, c_void_p, c_size_t, c_void_p]),
    "gemma3_qk_norm_rope": (c_int, [c_void_p, c_long, c_void_p, c_long, c_void_p, c_void_p,
                                    c_void_p, c_int, c_int, c_int, c_int, c_double, c_double,
                                    c_float, c_void_p]),
    "gemma3_flash_attention": (c_int, [c_void_p, c_void_p, c_void_p, c_long, c_void_p, c_int,
                                       c_void_p, c_int, c_int, c_int, c_int, c_int, c_int,
                                       c_void_p, c_void_p]),
    "gemma3_rmsnorm": (c_int, [c_void_p, c_int, c_void_p, c_void_p, c_int, c_int, c_int,
                               c_void_p, c_int, c_void_p]),
    "gemma3_postnorm_residual": (c_int, [c_void_p, c_void_p, c_int, c_void_p, c_void_p, c_int,
                                         c_int, c_void_p, c_int, c_void_p]),
    "gemma3_attn_check_status": (c_int, [c_void_p]),
    "gemma3_last_device_status": (c_int, []),
    "gemma3_set_gemm_tile_rows": (c_int, [c_int]),
    "gemma3_strerror": (ctypes.c_char_p, [c_int]),
    "gemma3_selftest_wait_timeout": (c_int, [ctypes.c_longlong, c_void_p]),
}

_lib = None


class Gemma3Error(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: status {status} ({strerror(status)})")


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise RuntimeError(
                f"{LIB} is missing: build it with transformer_attention_gb300.build.build() "
                "(nvcc, sm_103a); there is no CPU fallback")
        handle = ctypes.CDLL(LIB)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def strerror(status: int) -> str:
    return lib().gemma3_strerror(status).decode()


def _check(fn: str, status: int) -> int:
    if status < 0:
        raise Gemma3Error(fn, status)
    return status


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("tensor arguments must live on the GPU")
    return t.data_ptr()


def _stream(stream) -> int:
    import torch
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _dims(B, T, D, H, H_kv, d_h):
    return gemma3_attn_dims(B, T, D, H, H_kv, d_h)


# ---------------------------------------------------------------- same-name wrappers
def gemma3_layer_attn_type(layer: int, num_layers: int) -> int:
    return _check("gemma3_layer_attn_type", lib().gemma3_layer_attn_type(layer, num_layers))


def gemma3_layer_config(layer: int, num_layers: int, model_size: str):
    t, w, base, scale = c_int(), c_int(), c_double(), c_double()
    _check("gemma3_layer_config", lib().gemma3_layer_config(
        layer, num_layers, MODEL_SIZES[model_size], ctypes.byref(t), ctypes.byref(w),
        ctypes.byref(base), ctypes.byref(scale)))
    return t.value, w.value, base.value, scale.value


def gemma3_query_scale(model_size: str, D: int, H: int, d_h: int) -> float:
    a = c_float()
    _check("gemma3_query_scale",
           lib().gemma3_query_scale(MODEL_SIZES[model_size], D, H, d_h, ctypes.byref(a)))
    return a.value


def gemma3_attn_workspace_size(B, T, D, H, H_kv, d_h) -> int:
    n = c_size_t()
    d = _dims(B, T, D, H, H_kv, d_h)
    _check("gemma3_attn_workspace_size", lib().gemma3_attn_workspace_size(ctypes.byref(d),
                                                                          ctypes.byref(n)))
    return n.value


def gemma3_block_attn_workspace_size(B, T, D, H, H_kv, d_h) -> int:
    n = c_size_t()
    d = _dims(B, T, D, H, H_kv, d_h)
    _check("gemma3_block_attn_workspace_size",
           lib().gemma3_block_attn_workspace_size(ctypes.byref(d), ctypes.byref(n)))
    return n.value


def gemma3_attn_forward(dims, x, segment_pos, pad_lens, Wq, Wkv, Wo, gamma_q, gamma_k,
                        attn_type, window, rope_base, rope_scale, query_scale, out, workspace,
                        workspace_bytes, stream=None):
    d = _dims(*dims)
    return _check("gemma3_attn_forward", lib().gemma3_attn_forward(
        ctypes.byref(d), _ptr(x), _ptr(segment_pos), _ptr(pad_lens), _ptr(Wq), _ptr(Wkv),
        _ptr(Wo), _ptr(gamma_q), _ptr(gamma_k), attn_type, window, rope_base, rope_scale,
        query_scale, _ptr(out), _ptr(workspace), workspace_bytes, _stream(stream)))


def gemma3_attn_forward_noalloc(dims, x, segment_pos, pad_lens, Wq, Wkv, Wo, gamma_q, gamma_k,
                                attn_type, window, rope_base, rope_scale, query_scale, out,
                                stream=None):
    """gemma3_attn_forward without a workspace: for callers that cannot
    allocate device memory; uses the library's fixed per-device scratch."""
    d = _dims(*dims)
    return _check("gemma3_attn_forward_noalloc", lib().gemma3_attn_forward_noalloc(
        ctypes.byref(d), _ptr(x), _ptr(segment_pos), _ptr(pad_lens), _ptr(Wq), _ptr(Wkv),
        _ptr(Wo), _ptr(gamma_q), _ptr(gamma_k), attn_type, window, rope_base, rope_scale,
        query_scale, _ptr(out), _stream(stream)))


def gemma3_attn_noalloc_max_scratch() -> int:
    return lib().gemma3_attn_noalloc_max_scratch()


def gemma3_block_attn_forward(dims, x, x_dtype, y, segment_pos, pad_lens, Wq, Wkv, Wo, gamma_q,
                              gamma_k, gamma_pre, gamma_post, attn_type, window, rope_base,
                              rope_scale, query_scale, workspace, workspace_bytes, stream=None):
    d = _dims(*dims)
    return _check("gemma3_block_attn_forward", lib().gemma3_block_attn_forward(
        ctypes.byref(d), _ptr(x), x_dtype, _ptr(y), _ptr(segment_pos), _ptr(pad_lens), _ptr(Wq),
        _ptr(Wkv), _ptr(Wo), _ptr(gamma_q), _ptr(gamma_k), _ptr(gamma_pre), _ptr(gamma_post),
        attn_type, window, rope_base, rope_scale, query_scale, _ptr(workspace), workspace_bytes,
        _stream(stream)))


def gemma3_block_ffn_workspace_size(M, D, D_ff) -> int:
    n = c_size_t()
    _check("gemma3_block_ffn_workspace_size",
           lib().gemma3_block_ffn_workspace_size(M, D, D_ff, ctypes.byref(n)))
    return n.value


def gemma3_block_ffn_forward(M, D, D_ff, h, y, gamma_pre_ffn, gamma_post_ffn, W_gating, W_down,
                             workspace, workspace_bytes, stream=None):
    return _check("gemma3_block_ffn_forward", lib().gemma3_block_ffn_forward(
        M, D, D_ff, _ptr(h), _ptr(y), _ptr(gamma_pre_ffn), _ptr(gamma_post_ffn), _ptr(W_gating),
        _ptr(W_down), _ptr(workspace), workspace_bytes, _stream(stream)))


def gemma3_block_workspace_size(dims, D_ff) -> int:
    n = c_size_t()
    d = _dims(*dims)
    _check("gemma3_block_workspace_size",
           lib().gemma3_block_workspace_size(ctypes.byref(d), D_ff, ctypes.byref(n)))
    return n.value


def gemma3_block_forward(dims, D_ff, x, x_dtype, y, segment_pos, pad_lens, Wq, Wkv, Wo, gamma_q,
                         gamma_k, gamma_pre_attn, gamma_post_attn, gamma_pre_ffn, gamma_post_ffn,
                         W_gating, W_down, attn_type, window, rope_base, rope_scale, query_scale,
                         workspace, workspace_bytes, stream=None):
    d = _dims(*dims)
    return _check("gemma3_block_forward", lib().gemma3_block_forward(
        ctypes.byref(d), D_ff, _ptr(x), x_dtype, _ptr(y), _ptr(segment_pos), _ptr(pad_lens),
        _ptr(Wq), _ptr(Wkv), _ptr(Wo), _ptr(gamma_q), _ptr(gamma_k), _ptr(gamma_pre_attn),
        _ptr(gamma_post_attn), _ptr(gamma_pre_ffn), _ptr(gamma_post_ffn), _ptr(W_gating),
        _ptr(W_down), attn_type, window, rope_base, rope_scale, query_scale, _ptr(workspace),
        workspace_bytes, _stream(stream)))


def gemma3_model_workspace_size(dims, D_ff, V) -> int:
    n = c_size_t()
    d = _dims(*dims)
    _check("gemma3_model_workspace_size",
           lib().gemma3_model_workspace_size(ctypes.byref(d), D_ff, V, ctypes.byref(n)))
    return n.value


def gemma3_model_forward(dims, D_ff, V, num_layers, model_size, tokens, segment_pos, pad_lens, E,
                         layers, gamma_final, logits, workspace, workspace_bytes, stream=None):
    """``layers``: a sequence of dicts of device tensors keyed by the
    gemma3_block_weights field names; ``model_size``: "270M" .. "27B"."""
    d = _dims(*dims)
    arr = (gemma3_block_weights * max(1, num_layers))()
    for i, L in enumerate(layers):
        for name, _ in gemma3_block_weights._fields_:
            setattr(arr[i], name, _ptr(L[name]))
    return _check("gemma3_model_forward", lib().gemma3_model_forward(
        ctypes.byref(d), D_ff, V, num_layers, MODEL_SIZES[model_size], _ptr(tokens),
        _ptr(segment_pos), _ptr(pad_lens), _ptr(E), arr, _ptr(gamma_final), _ptr(logits),
        _ptr(workspace), workspace_bytes, _stream(stream)))


def gemma3_embed(tokens, E, V, D, M, scale, x, stream=None):
    return _check("gemma3_embed", lib().gemma3_embed(_ptr(tokens), _ptr(E), V, D, M, scale,
                                                     _ptr(x), _stream(stream)))


def gemma3_attn_cached_workspace_size(dims, S) -> int:
    n = c_size_t()
    d = _dims(*dims)
    _check("gemma3_attn_cached_workspace_size",
           lib().gemma3_attn_cached_workspace_size(ctypes.byref(d), S, ctypes.byref(n)))
    return n.value


def gemma3_attn_forward_cached(dims, S, end_index, x, segment_pos, pad_lens, Wq, Wkv, Wo,
                               gamma_q, gamma_k, attn_type, window, rope_base, rope_scale,
                               query_scale, K_cache, V_cache, pos_cache, out, workspace,
                               workspace_bytes, stream=None):
    d = _dims(*dims)
    return _check("gemma3_attn_forward_cached", lib().gemma3_attn_forward_cached(
        ctypes.byref(d), S, end_index, _ptr(x), _ptr(segment_pos), _ptr(pad_lens), _ptr(Wq),
        _ptr(Wkv), _ptr(Wo), _ptr(gamma_q), _ptr(gamma_k), attn_type, window, rope_base,
        rope_scale, query_scale, _ptr(K_cache), _ptr(V_cache), _ptr(pos_cache), _ptr(out),
        _ptr(workspace), workspace_bytes, _stream(stream)))


def gemma3_kv_cache_write(K_rows, V_rows, ld_rows, segment_pos, pad_lens, B, T, S, end_index,
                          H_kv, d_h, K_cache, V_cache, pos_cache, stream=None):
    return _check("gemma3_kv_cache_write", lib().gemma3_kv_cache_write(
        _ptr(K_rows), _ptr(V_rows), ld_rows, _ptr(segment_pos), _ptr(pad_lens), B, T, S,
        end_index, H_kv, d_h, _ptr(K_cache), _ptr(V_cache), _ptr(pos_cache), _stream(stream)))


def gemma3_cached_attention_workspace_size(B, T, S, H, H_kv, d_h) -> int:
    n = c_size_t()
    _check("gemma3_cached_attention_workspace_size", lib().gemma3_cached_attention_workspace_size(
        B, T, S, H, H_kv, d_h, ctypes.byref(n)))
    return n.value


def gemma3_cached_attention(Q, K_cache, V_cache, pos_cache, segment_pos, pad_lens, O, o_dtype, B,
                            T, S, end_index, H, H_kv, d_h, window, workspace, workspace_bytes,
                            stream=None):
    return _check("gemma3_cached_attention", lib().gemma3_cached_attention(
        _ptr(Q), _ptr(K_cache), _ptr(V_cache), _ptr(pos_cache), _ptr(segment_pos),
        _ptr(pad_lens), _ptr(O), o_dtype, B, T, S, end_index, H, H_kv, d_h, window,
        _ptr(workspace), workspace_bytes, _stream(stream)))


def gemma3_geglu(A, lda, W_gating, ldw, Z, ldz, M, D_ff, K, in_dtype, stream=None):
    return _check("gemma3_geglu", lib().gemma3_geglu(
        _ptr(A), lda, _ptr(W_gating), ldw, _ptr(Z), ldz, M, D_ff, K, in_dtype, _stream(stream)))


def gemma3_linear(A, lda, W, ldw, C, ldc, M, N, K, in_dtype, out_dtype, max_ctas=0,
                  stream=None, pad_lens=None, seg_T=0):
    return _check("gemma3_linear", lib().gemma3_linear(
        _ptr(A), lda, _ptr(W), ldw, _ptr(C), ldc, M, N, K, in_dtype, out_dtype, max_ctas,
        _ptr(pad_lens), seg_T, _stream(stream)))


def gemma3_qkv_proj_norm_rope(x, ldx, Wq, Wkv, Q, KV, M, D, H, H_kv, d_h, in_dtype, gamma_q,
                              gamma_k, pos, rope_base, rope_scale, query_scale, stream=None,
                              pad_lens=None, seg_T=0):
    return _check("gemma3_qkv_proj_norm_rope", lib().gemma3_qkv_proj_norm_rope(
        _ptr(x), ldx, _ptr(Wq), _ptr(Wkv), _ptr(Q), _ptr(KV), M, D, H, H_kv, d_h, in_dtype,
        _ptr(gamma_q), _ptr(gamma_k), _ptr(pos), rope_base, rope_scale, query_scale,
        _ptr(pad_lens), seg_T, _stream(stream)))


def gemma3_linear_qk_norm_rope(A, lda, W, ldw, C, ldc, M, N, K, in_dtype, gamma, pos, d_h, n_norm,
                               rope_base, rope_scale, scale, stream=None):
    return _check("gemma3_linear_qk_norm_rope", lib().gemma3_linear_qk_norm_rope(
        _ptr(A), lda, _ptr(W), ldw, _ptr(C), ldc, M, N, K, in_dtype, _ptr(gamma), _ptr(pos), d_h,
        n_norm, rope_base, rope_scale, scale, _stream(stream)))


def gemma3_cast_bf16_f16(src, dst, n, stream=None):
    return _check("gemma3_cast_bf16_f16", lib().gemma3_cast_bf16_f16(_ptr(src), _ptr(dst), n,
                                                                      _stream(stream)))


def gemma3_qk_norm_rope(Q, ldq, K, ldk, gamma_q, gamma_k, pos, M, H, H_kv, d_h, rope_base,
                        rope_scale, query_scale, stream=None):
    return _check("gemma3_qk_norm_rope", lib().gemma3_qk_norm_rope(
        _ptr(Q), ldq, _ptr(K), ldk, _ptr(gamma_q), _ptr(gamma_k), _ptr(pos), M, H, H_kv, d_h,
        rope_base, rope_scale, query_scale, _stream(stream)))


def gemma3_flash_attention(Q, K, V, ldkv, O, o_dtype, pad_lens, B, T, H, H_kv, d_h, window,
                           scratch=None, stream=None):
    """scratch: a 256-byte device tensor for the dynamic work order, or None
    for the fixed assignment."""
    return _check("gemma3_flash_attention", lib().gemma3_flash_attention(
        _ptr(Q), _ptr(K), _ptr(V), ldkv, _ptr(O), o_dtype, _ptr(pad_lens), B, T, H, H_kv, d_h,
        window, _ptr(scratch), _stream(stream)))


def gemma3_rmsnorm(x, x_dtype, gamma, u, u_dtype, M, D, stream=None, pad_lens=None, seg_T=0):
    return _check("gemma3_rmsnorm", lib().gemma3_rmsnorm(_ptr(x), x_dtype, _ptr(gamma), _ptr(u),
                                                         u_dtype, M, D, _ptr(pad_lens), seg_T,
                                                         _stream(stream)))


def gemma3_postnorm_residual(a, x, x_dtype, gamma, y, M, D, stream=None, pad_lens=None, seg_T=0):
    return _check("gemma3_postnorm_residual", lib().gemma3_postnorm_residual(
        _ptr(a), _ptr(x), x_dtype, _ptr(gamma), _ptr(y), M, D, _ptr(pad_lens), seg_T,
        _stream(stream)))


def gemma3_attn_check_status(stream=None) -> int:
    """Synchronises the stream and returns the library status (raises on error)."""
    return _check("gemma3_attn_check_status", lib().gemma3_attn_check_status(_stream(stream)))


def gemma3_last_device_status() -> int:
    return lib().gemma3_last_device_status()


def gemma3_set_gemm_tile_rows(rows: int) -> int:
    """Rows per projection-GEMM tile for later calls (0 chosen per call, 128
    or 256); returns the previous setting."""
    return _check("gemma3_set_gemm_tile_rows", lib().gemma3_set_gemm_tile_rows(rows))


def gemma3_selftest_wait_timeout(timeout_ns: int, stream=None) -> int:
    """Returns the raw status (GEMMA3_ERR_TIMEOUT expected); never raises on it."""
    return lib().gemma3_selftest_wait_timeout(timeout_ns, _stream(stream))
