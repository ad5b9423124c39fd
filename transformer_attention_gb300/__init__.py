"""Gemma 3 attention-block forward pass on one GB300 (sm_103a).

The compute lives in libgemma3attn.so (CUDA kernels behind the C ABI of
include/gemma3_attn.h).  ``_lib`` binds that ABI under the same names;
the helpers below only allocate outputs and workspaces with torch and call it.
"""
from __future__ import annotations

from ._lib import (  # noqa: F401  (re-exported C-ABI names)
    GEMMA3_BF16, GEMMA3_F16, GEMMA3_F32, GEMMA3_GLOBAL, GEMMA3_LOCAL_SLIDING, Gemma3Error,
    gemma3_attn_cached_workspace_size, gemma3_attn_check_status, gemma3_attn_forward,
    gemma3_attn_forward_cached, gemma3_attn_workspace_size, gemma3_cached_attention,
    gemma3_cached_attention_workspace_size, gemma3_kv_cache_write,
    gemma3_block_attn_forward, gemma3_block_attn_workspace_size, gemma3_block_ffn_forward,
    gemma3_block_ffn_workspace_size, gemma3_block_forward, gemma3_block_workspace_size,
    gemma3_cast_bf16_f16, gemma3_geglu,
    gemma3_flash_attention,
    gemma3_last_device_status, gemma3_layer_attn_type, gemma3_layer_config, gemma3_linear,
    gemma3_linear_qk_norm_rope, gemma3_qkv_proj_norm_rope, gemma3_embed, gemma3_model_forward, gemma3_model_workspace_size,
    GEMMA3_ERR_BAD_INPUT,
    gemma3_postnorm_residual, gemma3_qk_norm_rope, gemma3_query_scale, gemma3_rmsnorm,
    gemma3_selftest_wait_timeout, gemma3_set_gemm_tile_rows, lib)

__all__ = ["attention_forward", "attention_forward_cached", "block_attention_forward",
           "block_forward", "model_forward", "new_kv_cache", "linear", "lib"]


def _empty_ws(nbytes: int, device):
    import torch
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def attention_forward(x, segment_pos, pad_lens, Wq, Wkv, Wo, gamma_q, gamma_k, *, H, H_kv,
                      attn_type, window, rope_base, rope_scale, query_scale, out=None,
                      workspace=None, stream=None):
    """One attention layer: x [B,T,D] bf16 (CUDA) -> out [B,T,D] bf16.

    attn_type: GEMMA3_LOCAL_SLIDING or GEMMA3_GLOBAL.  pad_lens may be None.
    """
    import torch
    B, T, D = x.shape
    d_h = gamma_q.shape[0]
    dims = (B, T, D, H, H_kv, d_h)
    ws_bytes = gemma3_attn_workspace_size(*dims)
    if workspace is None:
        workspace = _empty_ws(ws_bytes, x.device)
    if out is None:
        out = torch.empty((B, T, D), dtype=torch.bfloat16, device=x.device)
    gemma3_attn_forward(dims, x, segment_pos, pad_lens, Wq, Wkv, Wo, gamma_q, gamma_k, attn_type,
                        window, rope_base, rope_scale, query_scale, out, workspace,
                        workspace.numel(), stream)
    return out


def new_kv_cache(B, S, H_kv, d_h, device):
    """An empty KV cache of S slots per row: (K_cache, V_cache) [B, S, H_kv,
    d_h] fp16 and pos_cache [B, S] int32, every stored position -1."""
    import torch
    K = torch.zeros((B, S, H_kv, d_h), dtype=torch.float16, device=device)
    V = torch.zeros_like(K)
    pos = torch.full((B, S), -1, dtype=torch.int32, device=device)
    return K, V, pos


def attention_forward_cached(x, segment_pos, pad_lens, cache, end_index, Wq, Wkv, Wo, gamma_q,
                             gamma_k, *, H, H_kv, attn_type, window, rope_base, rope_scale,
                             query_scale, out=None, workspace=None, stream=None):
    """One attention layer over x [B,T,D] bf16, new tokens written to slots
    [end_index, end_index + T) of ``cache`` = (K_cache, V_cache, pos_cache)
    from new_kv_cache (updated in place).  Returns out [B,T,D] bf16."""
    import torch
    B, T, D = x.shape
    d_h = gamma_q.shape[0]
    K_cache, V_cache, pos_cache = cache
    S = pos_cache.shape[1]
    dims = (B, T, D, H, H_kv, d_h)
    ws_bytes = gemma3_attn_cached_workspace_size(dims, S)
    if workspace is None:
        workspace = _empty_ws(ws_bytes, x.device)
    if out is None:
        out = torch.empty((B, T, D), dtype=torch.bfloat16, device=x.device)
    gemma3_attn_forward_cached(dims, S, end_index, x, segment_pos, pad_lens, Wq, Wkv, Wo,
                               gamma_q, gamma_k, attn_type, window, rope_base, rope_scale,
                               query_scale, K_cache, V_cache, pos_cache, out, workspace,
                               workspace.numel(), stream)
    return out


def block_attention_forward(x, segment_pos, pad_lens, Wq, Wkv, Wo, gamma_q, gamma_k, gamma_pre,
                            gamma_post, *, H, H_kv, attn_type, window, rope_base, rope_scale,
                            query_scale, y=None, workspace=None, stream=None):
    """y = x + RMSNorm_post(Attn(RMSNorm_pre(x))); x bf16 or fp32, y fp32 (may be x)."""
    import torch
    B, T, D = x.shape
    d_h = gamma_q.shape[0]
    dims = (B, T, D, H, H_kv, d_h)
    ws_bytes = gemma3_block_attn_workspace_size(*dims)
    if workspace is None:
        workspace = _empty_ws(ws_bytes, x.device)
    if y is None:
        y = torch.empty((B, T, D), dtype=torch.float32, device=x.device)
    x_dtype = GEMMA3_F32 if x.dtype == torch.float32 else GEMMA3_BF16
    gemma3_block_attn_forward(dims, x, x_dtype, y, segment_pos, pad_lens, Wq, Wkv, Wo, gamma_q,
                              gamma_k, gamma_pre, gamma_post, attn_type, window, rope_base,
                              rope_scale, query_scale, workspace, workspace.numel(), stream)
    return y


def block_forward(x, segment_pos, pad_lens, Wq, Wkv, Wo, gamma_q, gamma_k, gamma_pre_attn,
                  gamma_post_attn, gamma_pre_ffn, gamma_post_ffn, W_gating, W_down, *, H, H_kv,
                  attn_type, window, rope_base, rope_scale, query_scale, y=None,
                  workspace=None, stream=None):
    """The whole block: y = h + FFN sandwich(h), h = x + attention sandwich(x).
    x bf16 or fp32 [B,T,D]; y fp32 (may be x); W_gating [2,D_ff,D], W_down [D,D_ff]."""
    import torch
    B, T, D = x.shape
    d_h = gamma_q.shape[0]
    D_ff = W_gating.shape[1]
    dims = (B, T, D, H, H_kv, d_h)
    ws_bytes = gemma3_block_workspace_size(dims, D_ff)
    if workspace is None:
        workspace = _empty_ws(ws_bytes, x.device)
    if y is None:
        y = torch.empty((B, T, D), dtype=torch.float32, device=x.device)
    x_dtype = GEMMA3_F32 if x.dtype == torch.float32 else GEMMA3_BF16
    gemma3_block_forward(dims, D_ff, x, x_dtype, y, segment_pos, pad_lens, Wq, Wkv, Wo, gamma_q,
                         gamma_k, gamma_pre_attn, gamma_post_attn, gamma_pre_ffn, gamma_post_ffn,
                         W_gating, W_down, attn_type, window, rope_base, rope_scale, query_scale,
                         workspace, workspace.numel(), stream)
    return y


def model_forward(tokens, segment_pos, pad_lens, E, layers, gamma_final, *, H, H_kv, D_ff,
                  model_size, logits=None, workspace=None, stream=None):
    """The model: tokens [B,T] int32 -> logits [B,T,V] fp32 (read-out through
    E [V,D] bf16).  ``layers``: list of dicts of device tensors (Wq, Wkv, Wo,
    gamma_q, gamma_k, gamma_pre_attn, gamma_post_attn, gamma_pre_ffn,
    gamma_post_ffn, W_gating [2,D_ff,D], W_down [D,D_ff])."""
    import torch
    B, T = tokens.shape
    V, D = E.shape
    d_h = layers[0]["gamma_q"].shape[0] if layers else 256
    dims = (B, T, D, H, H_kv, d_h)
    ws_bytes = gemma3_model_workspace_size(dims, D_ff, V)
    if workspace is None:
        workspace = _empty_ws(ws_bytes, tokens.device)
    if logits is None:
        logits = torch.empty((B, T, V), dtype=torch.float32, device=tokens.device)
    gemma3_model_forward(dims, D_ff, V, len(layers), model_size, tokens, segment_pos, pad_lens,
                         E, layers, gamma_final, logits, workspace, workspace.numel(), stream)
    return logits


def linear(A, W, out_dtype=None, max_ctas=0, stream=None):
    """C = A @ W^T on the tcgen05 GEMM (A [M,K], W [N,K], both bf16 or both f16)."""
    import torch
    out_dtype = out_dtype or torch.bfloat16
    code = {torch.bfloat16: GEMMA3_BF16, torch.float16: GEMMA3_F16, torch.float32: GEMMA3_F32}
    if A.dtype != W.dtype or A.dtype not in (torch.bfloat16, torch.float16):
        raise ValueError("A and W must both be bf16 or both f16")
    M, K = A.shape
    N = W.shape[0]
    C = torch.empty((M, N), dtype=out_dtype, device=A.device)
    gemma3_linear(A, A.stride(0), W, W.stride(0), C, C.stride(0), M, N, K, code[A.dtype],
                  code[out_dtype], max_ctas, stream)
    return C
