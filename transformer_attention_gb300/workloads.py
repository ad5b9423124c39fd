"""Seeded synthetic workloads for the Gemma 3 attention-block forward pass.

This module only *draws numbers*: shapes, seeds and value distributions of the
five synthetic workloads, and the random tensors that both the CUDA path and
the fp64 oracle consume.  It holds none of the method's arithmetic (no norm,
rotation, mask or softmax); the per-layer routing of the 6-layer stack is left
to the callers (the C-ABI routing helper on the GPU side, the oracle's own
routing on the checking side).

Every tensor is generated on the CPU from a torch.Generator seeded per
(tensor seed, row block), so a checker can regenerate any block of rows of a
multi-GB activation without drawing the rest.  Values are sampled in fp32 and
rounded to bf16 with round-to-nearest-even (torch's ``.to(torch.bfloat16)``).

Distribution notation: "N(0, 1/D)" and "gamma ~ N(0, 0.1)" read the second
argument as a variance (weight std D**-0.5, gamma std 0.1**0.5).
"""
from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import torch

ROW_BLOCK = 1024          # rows of x per independently seeded block

# Seeds of the individual input tensors (per layer: + 100 * layer).
SEED_X, SEED_WQ, SEED_WKV, SEED_WO, SEED_GQ, SEED_GK, SEED_PAD = 1, 2, 3, 4, 5, 6, 7
SEED_GPRE, SEED_GPOST = 8, 9
SEED_WGATE, SEED_WDOWN, SEED_GPRE_FFN, SEED_GPOST_FFN = 10, 11, 12, 13
SEED_KCACHE, SEED_VCACHE = 14, 15
SEED_TOKENS, SEED_EMBED, SEED_GFINAL = 16, 17, 18


@dataclass(frozen=True)
class Workload:
    """Shape and input recipe of one synthetic workload."""
    name: str
    B: int
    T: int
    D: int
    H: int
    H_kv: int
    d_h: int
    attn_type: str            # "local" | "global" | "stack" (routed per layer)
    window: int               # local window W (0 for a global layer)
    rope_base: float
    rope_scale: float
    query_scale: float
    model_size: str           # Gemma 3 size the shape follows
    pad: tuple = ("none",)    # ("none",) | ("pad_uniform", lo, hi) | ("valid_uniform", lo, hi)
    num_layers: int = 1
    d_ff: int = 0             # > 0: the workload is the whole block (attention + feed-forward)
    cache_len: int = 0        # > 0: T new tokens per row appended to a KV cache of this many slots
    vocab: int = 0            # > 0: the whole model (embedding, routed full blocks, read-out)
    description: str = field(default="", compare=False)

    @property
    def M(self) -> int:
        return self.B * self.T

    @property
    def G(self) -> int:
        return self.H // self.H_kv


WORKLOADS = {
    "tiny_local": Workload(
        "tiny_local", B=1, T=1024, D=1152, H=4, H_kv=1, d_h=256, attn_type="local",
        window=512, rope_base=1e4, rope_scale=1.0, query_scale=256 ** -0.5, model_size="1B",
        description="tiny local MQA layer: B1 T1024 D1152 H4/1 d256 W512"),
    "1b_global": Workload(
        "1b_global", B=4, T=8192, D=1152, H=4, H_kv=1, d_h=256, attn_type="global",
        window=0, rope_base=1e6, rope_scale=1.0, query_scale=256 ** -0.5, model_size="1B",
        pad=("pad_uniform", 0, 1024),
        description="1B-shaped global MQA layer: B4 T8192 D1152 H4/1 d256, pads U{0..1024}"),
    "4b_local": Workload(
        "4b_local", B=2, T=32768, D=2560, H=8, H_kv=4, d_h=256, attn_type="local",
        window=1024, rope_base=1e4, rope_scale=1.0, query_scale=256 ** -0.5, model_size="4B",
        description="4B-shaped local GQA layer: B2 T32768 D2560 H8/4 d256 W1024"),
    "27b_global": Workload(
        "27b_global", B=1, T=131072, D=5376, H=32, H_kv=16, d_h=128, attn_type="global",
        window=0, rope_base=1e6, rope_scale=8.0, query_scale=168 ** -0.5, model_size="27B",
        description="27B-shaped long-context global GQA layer: B1 T131072 D5376 H32/16 d128"),
    "12b_stack": Workload(
        "12b_stack", B=8, T=16384, D=3840, H=16, H_kv=8, d_h=256, attn_type="stack",
        window=1024, rope_base=0.0, rope_scale=0.0, query_scale=256 ** -0.5, model_size="12B",
        pad=("valid_uniform", 2048, 16384), num_layers=6,
        description="12B-shaped 6-layer routed attention stack: B8 T16384 D3840 H16/8 d256"),
    # The full-block row (attention sandwich + GeGLU feed-forward sandwich) on
    # the 4B-shaped local layer; the feed-forward width 4D follows the 4B size.
    "4b_block": Workload(
        "4b_block", B=2, T=32768, D=2560, H=8, H_kv=4, d_h=256, attn_type="local",
        window=1024, rope_base=1e4, rope_scale=1.0, query_scale=256 ** -0.5, model_size="4B",
        d_ff=10240,
        description="4B-shaped full block: local attention layer + GeGLU FFN (D_ff 10240)"),
}

# Decode steps with a KV cache (one new token per row) on the 4B-shaped local
# and the 27B-shaped global layer: the cache holds a prompt that fills every
# slot but the last, which the new token is written to.
WORKLOADS["4b_local_decode"] = Workload(
    "4b_local_decode", B=2, T=1, D=2560, H=8, H_kv=4, d_h=256, attn_type="local", window=1024,
    rope_base=1e4, rope_scale=1.0, query_scale=256 ** -0.5, model_size="4B", cache_len=32768,
    description="decode step, 4B-shaped local layer: B2, 1 new token after 32767 cached, W1024")
WORKLOADS["27b_global_decode"] = Workload(
    "27b_global_decode", B=1, T=1, D=5376, H=32, H_kv=16, d_h=128, attn_type="global", window=0,
    rope_base=1e6, rope_scale=8.0, query_scale=168 ** -0.5, model_size="27B", cache_len=131072,
    description="decode step, 27B-shaped global layer: B1, 1 new token after 131071 cached")

# The model around the blocks on the 1B sizes: embedding, one routing tile of
# six full blocks (the pages give no depth table) and the read-out through a
# synthetic 32768-row embedding table (the pages give no vocabulary size).
WORKLOADS["1b_model"] = Workload(
    "1b_model", B=2, T=4096, D=1152, H=4, H_kv=1, d_h=256, attn_type="stack", window=512,
    rope_base=0.0, rope_scale=0.0, query_scale=256 ** -0.5, model_size="1B", num_layers=6,
    d_ff=6 * 1152, vocab=32768,
    description="1B-shaped model: embed, 6 routed full blocks (D_ff 6912), tied read-out V32768")

ORDER = ["tiny_local", "1b_global", "4b_local", "27b_global", "12b_stack", "4b_block",
         "4b_local_decode", "27b_global_decode", "1b_model"]


def small(w: Workload, **kw) -> Workload:
    """A copy of ``w`` with some fields replaced (for reduced-size test cases)."""
    d = dict(w.__dict__)
    d.update(kw)
    return Workload(**d)


# ----------------------------------------------------------------------------
# random draws
# ----------------------------------------------------------------------------
def _gen(seed: int, block: int = 0) -> torch.Generator:
    return torch.Generator().manual_seed((seed << 24) + block)


def _normal_bf16(shape, std: float, seed: int, block: int = 0) -> torch.Tensor:
    g = _gen(seed, block)
    t = torch.randn(shape, generator=g, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(torch.bfloat16)


def x_rows(w: Workload, b: int, t0: int, t1: int, seed: int = SEED_X) -> torch.Tensor:
    """Rows [t0, t1) of batch row b of the activation x, bf16 [t1-t0, D]."""
    out = []
    blk0, blk1 = t0 // ROW_BLOCK, (t1 + ROW_BLOCK - 1) // ROW_BLOCK
    for blk in range(blk0, blk1):
        key = b * ((w.T + ROW_BLOCK - 1) // ROW_BLOCK) + blk
        rows = min(ROW_BLOCK, w.T - blk * ROW_BLOCK)
        full = _normal_bf16((rows, w.D), 1.0, seed, key)
        lo = max(t0 - blk * ROW_BLOCK, 0)
        hi = min(t1 - blk * ROW_BLOCK, rows)
        out.append(full[lo:hi])
    return torch.cat(out, 0)


def x_full(w: Workload, seed: int = SEED_X, threads: int = 16) -> torch.Tensor:
    """The whole activation x, bf16 [B, T, D] (blocks drawn in parallel)."""
    x = torch.empty((w.B, w.T, w.D), dtype=torch.bfloat16)
    nblk = (w.T + ROW_BLOCK - 1) // ROW_BLOCK

    def fill(job):
        b, blk = job
        t0 = blk * ROW_BLOCK
        t1 = min(t0 + ROW_BLOCK, w.T)
        x[b, t0:t1] = x_rows(w, b, t0, t1, seed)

    jobs = [(b, k) for b in range(w.B) for k in range(nblk)]
    with ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(fill, jobs))
    return x


def weights(w: Workload, layer: int = 0) -> dict:
    """Projection weights and QK-norm scales of one layer (bf16, CPU).

    Layouts (row-major): Wq [H*d_h, D] (row n = h*d_h + c), Wkv [2, H_kv*d_h, D]
    ([0] = K, [1] = V), Wo [D, H*d_h], gamma_q / gamma_k [d_h].
    """
    off = 100 * layer
    std_in = 1.0 / math.sqrt(w.D)
    return {
        "Wq": _normal_bf16((w.H * w.d_h, w.D), std_in, SEED_WQ + off),
        "Wkv": _normal_bf16((2, w.H_kv * w.d_h, w.D), std_in, SEED_WKV + off),
        "Wo": _normal_bf16((w.D, w.H * w.d_h), std_in, SEED_WO + off),
        "gamma_q": _normal_bf16((w.d_h,), math.sqrt(0.1), SEED_GQ + off),
        "gamma_k": _normal_bf16((w.d_h,), math.sqrt(0.1), SEED_GK + off),
    }


def block_norm_gammas(w: Workload, layer: int) -> dict:
    """Pre- and post-attention RMSNorm scales [D] of one stack layer (bf16)."""
    off = 100 * layer
    return {
        "gamma_pre": _normal_bf16((w.D,), math.sqrt(0.1), SEED_GPRE + off),
        "gamma_post": _normal_bf16((w.D,), math.sqrt(0.1), SEED_GPOST + off),
    }


def ffn_weights(w: Workload, layer: int = 0) -> dict:
    """Feed-forward weights of one block (bf16, CPU): W_gating [2, D_ff, D]
    ([0] gate, [1] up), W_down [D, D_ff] (the (D_ff, D) linear stored
    transposed), and the pre/post feed-forward RMSNorm scales [D]."""
    off = 100 * layer
    return {
        "W_gating": _normal_bf16((2, w.d_ff, w.D), 1.0 / math.sqrt(w.D), SEED_WGATE + off),
        "W_down": _normal_bf16((w.D, w.d_ff), 1.0 / math.sqrt(w.d_ff), SEED_WDOWN + off),
        "gamma_pre_ffn": _normal_bf16((w.D,), math.sqrt(0.1), SEED_GPRE_FFN + off),
        "gamma_post_ffn": _normal_bf16((w.D,), math.sqrt(0.1), SEED_GPOST_FFN + off),
    }


def tokens(w: Workload) -> torch.Tensor:
    """Token ids of a model workload, int32 [B, T], uniform over [0, vocab)."""
    g = _gen(SEED_TOKENS)
    return torch.randint(0, w.vocab, (w.B, w.T), generator=g, dtype=torch.int64).to(torch.int32)


def model_tables(w: Workload) -> dict:
    """The embedding table E [vocab, D] ~ N(0, 1/D) (so E * sqrt(D) has unit
    variance) and the final RMSNorm scale [D] ~ N(0, 0.1), bf16."""
    return {"E": _normal_bf16((w.vocab, w.D), 1.0 / math.sqrt(w.D), SEED_EMBED),
            "gamma_final": _normal_bf16((w.D,), math.sqrt(0.1), SEED_GFINAL)}


def pad_lens(w: Workload) -> torch.Tensor:
    """Trailing pad count per batch row, int32 [B] (valid length = T - pad)."""
    g = _gen(SEED_PAD)
    kind = w.pad[0]
    if kind == "none":
        return torch.zeros(w.B, dtype=torch.int32)
    lo, hi = w.pad[1], w.pad[2]
    draw = torch.randint(lo, hi + 1, (w.B,), generator=g, dtype=torch.int64)
    if kind == "pad_uniform":
        return draw.to(torch.int32)
    if kind == "valid_uniform":
        return (w.T - draw).to(torch.int32)
    raise ValueError(kind)


def segment_pos(w: Workload) -> torch.Tensor:
    """RoPE positions, int32 [B, T]: 0..T-1 in every batch row, or for a
    decode workload the positions after the cached prompt (end .. end+T-1)."""
    base = w.cache_len - w.T if w.cache_len > 0 else 0
    return (base + torch.arange(w.T, dtype=torch.int32)).repeat(w.B, 1)


def kv_cache(w: Workload, threads: int = 16):
    """The prompt's cache of a decode workload (CPU): K' and V [B, S, H_kv, d_h]
    fp16 drawn N(0, 1) (sampled in fp32, rounded to nearest even) in slots
    [0, S - T), and the stored positions [B, S] int32: 0 .. S-T-1 there and -1
    (empty) in the last T slots, which the new tokens are written to."""
    S, end = w.cache_len, w.cache_len - w.T
    K = torch.zeros((w.B, S, w.H_kv, w.d_h), dtype=torch.float16)
    V = torch.zeros_like(K)
    pos = torch.full((w.B, S), -1, dtype=torch.int32)
    pos[:, :end] = torch.arange(end, dtype=torch.int32)
    nblk = (end + ROW_BLOCK - 1) // ROW_BLOCK

    def fill(job):
        b, blk = job
        s0, s1 = blk * ROW_BLOCK, min((blk + 1) * ROW_BLOCK, end)
        key = b * nblk + blk
        for buf, seed in ((K, SEED_KCACHE), (V, SEED_VCACHE)):
            g = _gen(seed, key)
            buf[b, s0:s1] = torch.randn((s1 - s0, w.H_kv, w.d_h), generator=g,
                                        dtype=torch.float32).to(torch.float16)

    jobs = [(b, k) for b in range(w.B) for k in range(nblk)]
    with ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(fill, jobs))
    return K, V, pos


def valid_tokens(w: Workload) -> int:
    return int((w.T - pad_lens(w).to(torch.int64)).sum())
