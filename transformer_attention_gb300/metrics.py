"""Work accounting of the attention-layer forward pass (algorithmic FLOPs and
bytes per kernel launch), used by the benchmark's roofline figures.

FLOPs count only unmasked (t, s) pairs with t, s < valid: attention costs
2 * d_h flops per pair per head for Q K^T and as much again for P V; a GEMM
costs 2 * M * N * K.  Bytes are the minimum each memory-bound kernel must
move (every input read once, every output written once).
"""
from __future__ import annotations


def unmasked_pairs(valid: int, window: int) -> int:
    """Pairs t - W < s <= t (or s <= t when window == 0) with 0 <= s <= t < valid."""
    if valid <= 0:
        return 0
    if window <= 0 or window >= valid:
        return valid * (valid + 1) // 2
    # rows t < W see t + 1 keys, the rest see exactly W keys
    return window * (window + 1) // 2 + (valid - window) * window


def attention_flops(valids, H: int, d_h: int, window: int) -> float:
    return 4.0 * d_h * H * sum(unmasked_pairs(v, window) for v in valids)


def gemm_flops(M: int, N: int, K: int) -> float:
    return 2.0 * M * N * K


def layer_gemm_flops(M: int, D: int, H: int, H_kv: int, d_h: int) -> dict:
    return {
        "q_proj": gemm_flops(M, H * d_h, D),
        "kv_proj": gemm_flops(M, 2 * H_kv * d_h, D),
        "o_proj": gemm_flops(M, D, H * d_h),
    }


def prologue_bytes(M: int, H: int, H_kv: int, d_h: int) -> float:
    # fp16 read + fp16 write of every Q and K head vector, plus one int32 position
    return M * ((H + H_kv) * d_h * 2 * 2 + 4)


def rmsnorm_bytes(M: int, D: int, in_bytes: int) -> float:
    return M * D * (in_bytes + 2)


def postnorm_bytes(M: int, D: int, x_bytes: int) -> float:
    return M * D * (4 + x_bytes + 4)
