"""fp64 CPU oracle of the Gemma 3 attention-block forward pass.

TEST INFRASTRUCTURE.  This module is the checker, not the product: only the
test suite, the smoke check and the benchmark's CPU-baseline leg may import
it.  It shares no code with the CUDA path (no kernels, headers, tables or
helpers); both only consume the same seeded inputs.

Every step is written out in float64 with plain PyTorch CPU tensor ops, in the
order the pages give, so it can be checked against them by eye.  Citations
name the page and the section on it:

  [AB] "Gemma 3 Attention Block"          (sections Overview, How it works)
  [FB] "Full Gemma 3 Block"               (How it works: Block.__call__ equations)
  [RT] "Global vs Local Layer Routing"    (How it works, Watch-outs)
  [QK] "QK-Norm"                          (How it works: RMSNorm equation, Watch-outs)
  [FB] last paragraph of How it works: the model around the blocks

Readings where the pages are silent (each also listed in the design notes):
  R1  RoPE: the pages name only a base frequency and a scale.  We use the
      frequencies base**(-2c/d_h) for c < d_h/2, rotate the pair
      (c, c + d_h/2) by angle (pos/scale)*freq_c, and divide the position by
      the scale (the routing page calls the scale a positional-interpolation
      factor).  The pairing and the frequency law are PARITY UNPINNED by the
      pages; the pins fix only properties every such rotation has.
  R2  Masks index the sequence axis t, s; segment_pos feeds RoPE only.
  R3  Padding is trailing: keys s >= T - pad_b are blocked.  Query rows
      t >= T - pad_b have no defined output; the oracle returns 0 there.
  R4  Window: a local layer keeps t - W < s <= t (sliding mask x causal).
  R5  gamma_q / gamma_k have shape [d_h], shared across heads and positions.
  R6  GQA: query head h reads kv head h // G (reshape to [H_kv, G]).
  R7  The query scale multiplies Q after RoPE, before the logits.
  R8  A cache slot that holds no token stores position -1 (EMPTY_SLOT); a
      fresh cache is all empty, and pad tokens are written as empty.
  R9  With a cache, the causal-and-padding mask is over slots (s <= the
      query's own slot, slot not empty) and the sliding mask compares stored
      positions with the query position.
  R10 The model's read-out multiplies by the embedding table itself (the
      page's last step reads the logits out through that table, in garbled
      words); the depth N and the vocabulary size V are parameters (the
      page's depth table is empty and it names no vocabulary size).
"""
from __future__ import annotations

import math

import torch

F64 = torch.float64

# [AB] How it works (Scores): value the blocked logits are filled with.
K_MASK = -2.3819763e38
# [QK] How it works: RMSNorm epsilon; [FB] How it works: same eps on block norms.
RMS_EPS = 1e-6

# [RT] How it works: the six-slot routing tile, local first.
LOCAL_SLIDING, GLOBAL = "LOCAL_SLIDING", "GLOBAL"
GEMMA3_ATTENTION_PATTERN = (LOCAL_SLIDING,) * 5 + (GLOBAL,)


# ----------------------------------------------------------------------------
# routing
# ----------------------------------------------------------------------------
def make_attention_layers_types(num_layers: int, pattern=GEMMA3_ATTENTION_PATTERN):
    """[RT] How it works: tile the pattern over the depth; a depth that is not a
    multiple of the tile length gets the prefix pattern[:N % len] appended (so
    leftover layers are local, never a stray global)."""
    reps, rem = divmod(num_layers, len(pattern))
    return tuple(pattern) * reps + tuple(pattern[:rem])


def layer_params(attn_type: str, model_size: str):
    """[RT] How it works (Transformer.setup mapping) and [AB] Overview/Routing:
    local layers: RoPE base 1e4, scale 1, window 1024 (512 on 270M/1B);
    global layers: base 1e6, scale 8 on 4B/12B/27B, 1 on 270M/1B (the small
    configs leave global_scale_factor at its default).
    Returns (rope_base, rope_scale, window); window 0 means "no window"."""
    small = model_size in ("270M", "1B")
    if attn_type == LOCAL_SLIDING:
        return 1e4, 1.0, (512 if small else 1024)
    if attn_type == GLOBAL:
        return 1e6, (1.0 if small else 8.0), 0
    raise ValueError(attn_type)


def query_pre_attn_scalar(model_size: str, D: int, H: int, d_h: int) -> float:
    """[AB] How it works (query scale case split): d_h**-1/2, except on 27B
    where it is (D/H)**-1/2."""
    if model_size == "27B":
        return (D / H) ** -0.5
    return d_h ** -0.5


# ----------------------------------------------------------------------------
# per-step definitions
# ----------------------------------------------------------------------------
def rms_norm(x: torch.Tensor, gamma: torch.Tensor, eps: float = RMS_EPS) -> torch.Tensor:
    """[QK] How it works, RMSNorm equation: x / sqrt(mean(x^2) + eps) * (1 + gamma),
    mean over the last axis only ([QK] How it works; [FB] How it works)."""
    x = x.to(F64)
    ms = (x * x).mean(dim=-1, keepdim=True)
    return x / torch.sqrt(ms + eps) * (1.0 + gamma.to(F64))


def rope(x: torch.Tensor, positions: torch.Tensor, base: float, scale: float) -> torch.Tensor:
    """Rotary embedding of x [..., T, n_heads, d_h] at integer positions [..., T].

    [AB] How it works (QK-norm, then RoPE, then scale) names the layer's base
    frequency and scale; the rotation itself is reading R1 (parity unpinned)."""
    x = x.to(F64)
    d_h = x.shape[-1]
    half = d_h // 2
    c = torch.arange(half, dtype=F64)
    freq = torch.pow(torch.tensor(base, dtype=F64), -2.0 * c / d_h)          # [half]
    angle = (positions.to(F64) / scale)[..., None] * freq                       # [..., T, half]
    cos = torch.cos(angle)[..., None, :]                                       # [..., T, 1, half]
    sin = torch.sin(angle)[..., None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return torch.cat([x1 * cos - x2 * sin, x2 * cos + x1 * sin], dim=-1)


def create_sliding_mask(t_idx: torch.Tensor, s_idx: torch.Tensor, window: int) -> torch.Tensor:
    """[AB] How it works, sliding-mask equation: M[t,s] = 1[s > t-W] * 1[s < t+W]."""
    t = t_idx[:, None]
    s = s_idx[None, :]
    return (s > t - window) & (s < t + window)


def causal_padding_mask(t_idx: torch.Tensor, s_idx: torch.Tensor, valid_len: int) -> torch.Tensor:
    """[AB] How it works (input attn_mask is causal and padding); readings R2, R3:
    keep s <= t and s < valid_len."""
    t = t_idx[:, None]
    s = s_idx[None, :]
    return (s <= t) & (s < valid_len)


def project(x: torch.Tensor, W: torch.Tensor) -> torch.Tensor:
    """[AB] How it works (Projections): y[..., n] = sum_d x[..., d] * W[n, d]."""
    return torch.matmul(x.to(F64), W.to(F64).transpose(0, 1))


# ----------------------------------------------------------------------------
# the attention layer
# ----------------------------------------------------------------------------
def normalised_rotated_qk(x_rows, positions, Wq, Wkv, gamma_q, gamma_k, *,
                          H, H_kv, d_h, rope_base, rope_scale):
    """Q and K of the given token rows after QK-norm and RoPE, before the query
    scale ([AB] How it works: projections, then QK-norm, then RoPE).
    x_rows [n, D], positions [n] -> (Q [n, H, d_h], K [n, H_kv, d_h]) in fp64."""
    Q = project(x_rows, Wq).reshape(-1, H, d_h)
    K = project(x_rows, Wkv[0]).reshape(-1, H_kv, d_h)
    Q = rms_norm(Q, gamma_q)                         # [QK] separate _query_norm
    K = rms_norm(K, gamma_k)                         # [QK] separate _key_norm
    Q = rope(Q, positions, rope_base, rope_scale)
    K = rope(K, positions, rope_base, rope_scale)
    return Q, K


def attend(Q, K, V, t_idx, s_idx, valid, attn_type, window):
    """Masked softmax attention of one batch row ([AB] How it works, Scores).

    Q [Tq, H, d_h] (query scale applied), K, V [S, H_kv, d_h] at key positions
    s_idx, query positions t_idx.  Q is reshaped to [Tq, H_kv, G, d_h] and
    contracted with K; blocked logits are K_MASK; softmax over s mixes V.
    Returns [Tq, H, d_h]."""
    # Mask: causal + padding; local layers also multiply in the sliding mask
    mask = causal_padding_mask(t_idx, s_idx, valid)
    if attn_type == LOCAL_SLIDING:
        mask = mask & create_sliding_mask(t_idx, s_idx, window)
    return attend_masked(Q, K, V, mask)


def attend_masked(Q, K, V, mask):
    """[AB] How it works, Scores: GQA logits, K_MASK where ``mask`` [Tq, S] is
    False, softmax over s, V mix.  Q [Tq, H, d_h], K, V [S, H_kv, d_h];
    returns [Tq, H, d_h]."""
    Tq, H, d_h = Q.shape
    H_kv = K.shape[1]
    G = H // H_kv
    Qg = Q.reshape(Tq, H_kv, G, d_h)
    logits = torch.einsum("tkgc,skc->tkgs", Qg, K)        # [Tq, H_kv, G, S]
    logits = torch.where(mask[:, None, None, :], logits, torch.tensor(K_MASK, dtype=F64))

    # Softmax over s, then mix V ([AB] Scores)
    probs = torch.softmax(logits, dim=-1)
    return torch.einsum("tkgs,skc->tkgc", probs, V).reshape(Tq, H, d_h)


def attention_layer(x, segment_pos, pad_lens, Wq, Wkv, Wo, gamma_q, gamma_k, *,
                    H, H_kv, d_h, attn_type, window, rope_base, rope_scale,
                    query_scale, rows=None):
    """Forward pass of one Gemma 3 attention layer, in float64.

    x [B,T,D], segment_pos [B,T] int, pad_lens [B] int or None, Wq [H*d_h, D],
    Wkv [2, H_kv*d_h, D], Wo [D, H*d_h], gamma_q/gamma_k [d_h];
    attn_type LOCAL_SLIDING | GLOBAL.

    ``rows`` (optional) is a list, per batch row, of query positions to compute;
    only the keys those queries can see are projected.  Every other key is
    blocked for every requested query, and a blocked logit contributes
    exp(K_MASK - max) == 0.0 exactly in fp64, so the sampled outputs equal the
    corresponding rows of the full computation.

    Returns out [B,T,D] (rows=None) or a list, per batch row, of [len(rows[b]), D].
    """
    B, T, D = x.shape
    if pad_lens is None:
        pad_lens = torch.zeros(B, dtype=torch.int64)
    outs = []
    for b in range(B):
        valid = T - int(pad_lens[b])
        t_req = torch.arange(T) if rows is None else torch.as_tensor(rows[b], dtype=torch.int64)
        if t_req.numel() == 0:
            outs.append(torch.zeros(0, D, dtype=F64))
            continue
        # Keys any requested query can see: s <= t (causal) and, on local
        # layers, s > t - W; the union over the requested rows.
        if rows is None:
            s_idx = torch.arange(T)
        else:
            seen = torch.zeros(T, dtype=torch.bool)
            for t in t_req.tolist():
                lo = max(0, t - window + 1) if attn_type == LOCAL_SLIDING else 0
                seen[lo:t + 1] = True
            s_idx = torch.nonzero(seen).flatten()

        # Projections ([AB] How it works, Projections)
        xq = x[b, t_req]                                   # [Tq, D]
        xs = x[b, s_idx]                                   # [S, D]
        Q = project(xq, Wq).reshape(-1, H, d_h)
        K = project(xs, Wkv[0]).reshape(-1, H_kv, d_h)
        V = project(xs, Wkv[1]).reshape(-1, H_kv, d_h)

        # QK-norm with separate scales for Q and K; V is not normalised
        # ([QK] How it works, Overview)
        Q = rms_norm(Q, gamma_q)
        K = rms_norm(K, gamma_k)

        # RoPE with the layer's base and scale ([AB] How it works)
        Q = rope(Q, segment_pos[b, t_req], rope_base, rope_scale)
        K = rope(K, segment_pos[b, s_idx], rope_base, rope_scale)

        # Query scale after RoPE ([QK] How it works; [AB] query-scale cases)
        Q = Q * query_scale

        enc = attend(Q, K, V, t_req, s_idx, valid, attn_type, window)
        out = project(enc.reshape(-1, H * d_h), Wo)        # [Tq, D] (attn_vec_einsum)

        # Reading R3: rows past the valid length have no output
        out[t_req >= valid] = 0.0
        outs.append(out)

    if rows is None:
        return torch.stack(outs, 0)
    return outs


# ----------------------------------------------------------------------------
# the KV-cache path
# ----------------------------------------------------------------------------
# Reading R8: stored position of a cache slot that holds no token (never
# written, or written by a pad token).  Every real position is >= 0.
EMPTY_SLOT = -1


def init_cache(B: int, S: int, H_kv: int, d_h: int) -> dict:
    """An empty left-aligned cache of S slots per batch row ([AB] How it works,
    Cache): K and V [B, S, H_kv, d_h] and the stored positions [B, S]."""
    return {"k": torch.zeros(B, S, H_kv, d_h, dtype=F64),
            "v": torch.zeros(B, S, H_kv, d_h, dtype=F64),
            "pos": torch.full((B, S), EMPTY_SLOT, dtype=torch.int64)}


def dynamic_update_slice(buf: torch.Tensor, update: torch.Tensor, start: int) -> torch.Tensor:
    """[AB] How it works, Cache: a copy of ``buf`` whose slots
    [start, start + update.shape[1]) along axis 1 are replaced by ``update``;
    every other slot keeps its value."""
    out = buf.clone()
    out[:, start:start + update.shape[1]] = update.to(out.dtype)
    return out


def cache_mask(q_slots, q_pos, slot_pos, attn_type, window):
    """Mask of one batch row's queries over its cache slots.

    q_slots [Tq] are the slots the queries were written to, q_pos [Tq] their
    positions, slot_pos [S] the stored positions.  Reading R9: the incoming
    causal-and-padding mask over the cache keeps s <= slot(t) and slots that
    hold a token (stored position >= 0); a local layer multiplies in the
    sliding mask of [AB] How it works evaluated on the stored positions, which
    is what the stored positions are kept for ([AB] How it works, Cache)."""
    s = torch.arange(slot_pos.shape[0])
    mask = (s[None, :] <= q_slots[:, None]) & (slot_pos[None, :] >= 0)
    if attn_type == LOCAL_SLIDING:
        mask = mask & create_sliding_mask(q_pos, slot_pos, window)
    return mask


def attention_layer_cached(x, segment_pos, pad_lens, cache, end_index, Wq, Wkv, Wo,
                           gamma_q, gamma_k, *, H, H_kv, d_h, attn_type, window,
                           rope_base, rope_scale, query_scale):
    """One attention layer over T new tokens per batch row with a KV cache.

    [AB] How it works: the new tokens' K (after QK-norm and RoPE) and V, and
    their positions, are written into the left-aligned cache at slot
    ``end_index`` with dynamic_update_slice; the queries then attend over every
    cache slot under ``cache_mask``.  Pad tokens (t >= T - pad_b, reading R3)
    are stored with position EMPTY_SLOT and get output 0.

    x [B,T,D], segment_pos [B,T], cache from ``init_cache`` (or a previous
    call).  Returns (out [B,T,D], the updated cache); the input cache is not
    modified.
    """
    B, T, D = x.shape
    S = cache["pos"].shape[1]
    if end_index < 0 or end_index + T > S:
        raise ValueError("cache overflow: end_index + T > S")
    if pad_lens is None:
        pad_lens = torch.zeros(B, dtype=torch.int64)
    t = torch.arange(T)
    is_pad = t[None, :] >= (T - torch.as_tensor(pad_lens, dtype=torch.int64))[:, None]   # [B, T]

    # Projections, QK-norm, RoPE, then the query scale ([AB] How it works)
    Q = project(x, Wq).reshape(B, T, H, d_h)
    K = project(x, Wkv[0]).reshape(B, T, H_kv, d_h)
    V = project(x, Wkv[1]).reshape(B, T, H_kv, d_h)
    Q = rms_norm(Q, gamma_q)
    K = rms_norm(K, gamma_k)
    Q = rope(Q, segment_pos, rope_base, rope_scale)
    K = rope(K, segment_pos, rope_base, rope_scale)
    Q = Q * query_scale

    # Cache write ([AB] How it works, Cache)
    stored_pos = torch.where(is_pad, torch.tensor(EMPTY_SLOT), segment_pos.to(torch.int64))
    new = {"k": dynamic_update_slice(cache["k"], K, end_index),
           "v": dynamic_update_slice(cache["v"], V, end_index),
           "pos": dynamic_update_slice(cache["pos"], stored_pos, end_index)}

    outs = []
    for b in range(B):
        mask = cache_mask(end_index + t, segment_pos[b].to(torch.int64), new["pos"][b],
                          attn_type, window)
        enc = attend_masked(Q[b], new["k"][b], new["v"][b], mask)
        out = project(enc.reshape(T, H * d_h), Wo)
        out[is_pad[b]] = 0.0
        outs.append(out)
    return torch.stack(outs, 0), new


def block_attention(x, gamma_pre, gamma_post, **layer_kwargs):
    """[FB] How it works, first three lines of Block.__call__:
    a = Attn(RMSNorm_pre(x)); a <- RMSNorm_post(a); h = x + a.
    x is the residual stream [B,T,D]; everything stays in fp64."""
    u = rms_norm(x, gamma_pre)
    a = attention_layer(u, **layer_kwargs)
    return x.to(F64) + rms_norm(a, gamma_post)


def attention_stack(x, layers, *, model_size, H, H_kv, d_h, segment_pos, pad_lens):
    """The routed attention stack: layer l has type P[l mod 6] ([RT] How it works)
    and the RoPE base/scale/window that type selects ([RT] Transformer.setup
    mapping); each layer is the block-attention sandwich of ``block_attention``.

    ``layers`` is a list of dicts with Wq, Wkv, Wo, gamma_q, gamma_k,
    gamma_pre, gamma_post.  Pad rows keep the residual unchanged: their
    attention output is 0 (reading R3) and RMSNorm(0) == 0.
    """
    B, T, D = x.shape
    types = make_attention_layers_types(len(layers))
    h = x.to(F64)
    for l, p in enumerate(layers):
        base, scale, window = layer_params(types[l], model_size)
        h = block_attention(
            h, p["gamma_pre"], p["gamma_post"], segment_pos=segment_pos,
            pad_lens=pad_lens, Wq=p["Wq"], Wkv=p["Wkv"], Wo=p["Wo"],
            gamma_q=p["gamma_q"], gamma_k=p["gamma_k"], H=H, H_kv=H_kv, d_h=d_h,
            attn_type=types[l], window=window, rope_base=base, rope_scale=scale,
            query_scale=query_pre_attn_scalar(model_size, D, H, d_h))
    return h


# ----------------------------------------------------------------------------
# the feed-forward half of the block
# ----------------------------------------------------------------------------
def ffn_hidden_dim(model_size: str, D: int) -> int:
    """[FB] How it works (MLP): hidden widths 2048 on 270M, 6D on 1B, and 4D on
    4B/12B/27B (hidden_dim = embed_dim * 8 // 2)."""
    if model_size == "270M":
        return 2048
    if model_size == "1B":
        return 6 * D
    return D * 8 // 2


def gelu_tanh(x: torch.Tensor) -> torch.Tensor:
    """[FB] How it works (MLP): the Flax default GELU, its tanh approximation:
    0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3)))."""
    x = x.to(F64)
    return 0.5 * x * (1.0 + torch.tanh(math.sqrt(2.0 / math.pi) * (x + 0.044715 * x ** 3)))


def feed_forward(u: torch.Tensor, W_gating: torch.Tensor, W_down: torch.Tensor) -> torch.Tensor:
    """[FB] How it works (MLP): the gating einsum '...F,NHF->...NH' with the
    weight stored as (2, D_ff, D) gives [..., 2, D_ff]; slice 0 is uW_g and
    slice 1 is uW_u; FFN(u) = (GELU(uW_g) * (uW_u)) W_d with W_d of shape
    (D_ff, D)."""
    gate_up = torch.einsum("...f,nhf->...nh", u.to(F64), W_gating.to(F64))
    z = gelu_tanh(gate_up[..., 0, :]) * gate_up[..., 1, :]
    return torch.matmul(z, W_down.to(F64))


def block_ffn(h, gamma_pre_ffn, gamma_post_ffn, W_gating, W_down):
    """[FB] How it works, last three lines of Block.__call__:
    m = FFN(RMSNorm_pre-ffn(h)); m <- RMSNorm_post-ffn(m); y = h + m.
    Rows are independent (pad rows too: the pages define no mask here)."""
    m = feed_forward(rms_norm(h, gamma_pre_ffn), W_gating, W_down)
    return h.to(F64) + rms_norm(m, gamma_post_ffn)


def full_block(x, gamma_pre_attn, gamma_post_attn, gamma_pre_ffn, gamma_post_ffn, W_gating,
               W_down, **layer_kwargs):
    """[FB] How it works, Block.__call__: the attention sandwich, then the
    feed-forward sandwich, on the residual stream (fp64)."""
    h = block_attention(x, gamma_pre_attn, gamma_post_attn, **layer_kwargs)
    return block_ffn(h, gamma_pre_ffn, gamma_post_ffn, W_gating, W_down)


# ----------------------------------------------------------------------------
# the model around the blocks
# ----------------------------------------------------------------------------
def embed(tokens: torch.Tensor, E: torch.Tensor) -> torch.Tensor:
    """[FB] How it works, last paragraph: the token's row of the embedding
    table times sqrt(D).  tokens [B, T] int, E [V, D] -> [B, T, D] fp64."""
    D = E.shape[1]
    return E.to(F64)[tokens.to(torch.int64)] * math.sqrt(D)


def tied_logits(h: torch.Tensor, E: torch.Tensor) -> torch.Tensor:
    """[FB] How it works, last paragraph: the read-out uses the embedding
    table, logits[..., v] = sum_d h[..., d] * E[v, d]; no final-logit
    soft-cap ([FB] Overview: none on any size)."""
    return torch.matmul(h.to(F64), E.to(F64).transpose(0, 1))


def model_forward(tokens, E, layers, gamma_final, *, model_size, H, H_kv, d_h, segment_pos,
                  pad_lens):
    """[FB] How it works, last paragraph: embed (times sqrt(D)), N blocks,
    final RMSNorm, read-out through the embedding table.  Block l has type
    P[l mod 6] and that type's RoPE base/scale/window ([RT] How it works).

    ``layers``: list of dicts with Wq, Wkv, Wo, gamma_q, gamma_k, gamma_pre,
    gamma_post, gamma_pre_ffn, gamma_post_ffn, W_gating (2, D_ff, D) and
    W_down (D_ff, D).  Returns logits [B, T, V] in fp64."""
    x = embed(tokens, E)
    D = E.shape[1]
    types = make_attention_layers_types(len(layers))
    alpha = query_pre_attn_scalar(model_size, D, H, d_h)
    for l, p in enumerate(layers):
        base, scale, window = layer_params(types[l], model_size)
        x = full_block(x, p["gamma_pre"], p["gamma_post"], p["gamma_pre_ffn"],
                       p["gamma_post_ffn"], p["W_gating"], p["W_down"], segment_pos=segment_pos,
                       pad_lens=pad_lens, Wq=p["Wq"], Wkv=p["Wkv"], Wo=p["Wo"],
                       gamma_q=p["gamma_q"], gamma_k=p["gamma_k"], H=H, H_kv=H_kv, d_h=d_h,
                       attn_type=types[l], window=window, rope_base=base, rope_scale=scale,
                       query_scale=alpha)
    return tied_logits(rms_norm(x, gamma_final), E)
