"""Pins of the fp64 oracle to facts the pages and the mathematics fix.

Every check here is independent of the oracle's own formulas: closed-form
special cases, invariants, values the pages print (tests/golden/), and a
brute-force scalar re-derivation of attention on tiny inputs written from the
pages' prose with plain Python loops.
"""
import json
import math
import os

import pytest
import torch

from oracle import gemma3_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
F64 = torch.float64


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ----------------------------------------------------------------------------
# brute force: scalar loops, written from the pages' prose
# ----------------------------------------------------------------------------
def _matvec(W, v):
    return [sum(W[n][d] * v[d] for d in range(len(v))) for n in range(len(W))]


def _rmsnorm_scalar(v, gamma, eps=1e-6):
    m = sum(a * a for a in v) / len(v)
    r = 1.0 / math.sqrt(m + eps)
    return [a * r * (1.0 + g) for a, g in zip(v, gamma)]


def _rope_scalar(v, pos, base, scale):
    # Reading R1: pair (c, c + d/2) rotated by (pos / scale) * base^(-2c/d).
    d = len(v)
    h = d // 2
    out = list(v)
    for c in range(h):
        a = (pos / scale) * base ** (-2.0 * c / d)
        out[c] = v[c] * math.cos(a) - v[c + h] * math.sin(a)
        out[c + h] = v[c + h] * math.cos(a) + v[c] * math.sin(a)
    return out


def brute_attention(x, pos, valid, Wq, Wk, Wv, Wo, gq, gk, H, Hkv, dh, local, W,
                    base, scale, alpha):
    """One batch row.  x: T lists of D floats.  Returns T lists of D floats.

    Keep key s for query t when s <= t, s < valid and (global, or t - W < s):
    the pages' causal-and-padding mask times the sliding mask.  Query head h
    reads kv head h // (H/Hkv).  Pad query rows return zeros (reading R3).
    """
    T, D = len(x), len(x[0])
    G = H // Hkv
    q = [_matvec(Wq, x[t]) for t in range(T)]
    k = [_matvec(Wk, x[t]) for t in range(T)]
    v = [_matvec(Wv, x[t]) for t in range(T)]
    qh = [[_rope_scalar(_rmsnorm_scalar(q[t][h * dh:(h + 1) * dh], gq), pos[t], base, scale)
           for h in range(H)] for t in range(T)]
    kh = [[_rope_scalar(_rmsnorm_scalar(k[t][j * dh:(j + 1) * dh], gk), pos[t], base, scale)
           for j in range(Hkv)] for t in range(T)]
    vh = [[v[t][j * dh:(j + 1) * dh] for j in range(Hkv)] for t in range(T)]
    out = []
    for t in range(T):
        if t >= valid:
            out.append([0.0] * D)
            continue
        enc = []
        for h in range(H):
            j = h // G
            allowed = [s for s in range(T)
                       if s <= t and s < valid and (not local or s > t - W)]
            logits = {s: alpha * sum(qh[t][h][c] * kh[s][j][c] for c in range(dh))
                      for s in allowed}
            mx = max(logits.values())
            e = {s: math.exp(logits[s] - mx) for s in allowed}
            z = sum(e.values())
            enc.extend(sum(e[s] / z * vh[s][j][c] for s in allowed) for c in range(dh))
        out.append(_matvec(Wo, enc))
    return out


def _rand(shape, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g, dtype=F64) * std)


def _case(T=12, D=8, H=4, Hkv=2, dh=4, seed=0, valid=None):
    x = _rand((1, T, D), seed)
    Wq = _rand((H * dh, D), seed + 1, D ** -0.5)
    Wkv = _rand((2, Hkv * dh, D), seed + 2, D ** -0.5)
    Wo = _rand((D, H * dh), seed + 3, D ** -0.5)
    gq = _rand((dh,), seed + 4, 0.3)
    gk = _rand((dh,), seed + 5, 0.3)
    pos = torch.arange(T).reshape(1, T)
    pad = torch.tensor([0 if valid is None else T - valid])
    return dict(x=x, segment_pos=pos, pad_lens=pad, Wq=Wq, Wkv=Wkv, Wo=Wo,
                gamma_q=gq, gamma_k=gk)


def _run_both(case, H, Hkv, dh, local, W, base=1e4, scale=1.0, alpha=0.5):
    T = case["x"].shape[1]
    valid = T - int(case["pad_lens"][0])
    got = O.attention_layer(
        **case, H=H, H_kv=Hkv, d_h=dh,
        attn_type=O.LOCAL_SLIDING if local else O.GLOBAL, window=W,
        rope_base=base, rope_scale=scale, query_scale=alpha)[0]
    ref = brute_attention(
        case["x"][0].tolist(), case["segment_pos"][0].tolist(), valid,
        case["Wq"].tolist(), case["Wkv"][0].tolist(), case["Wkv"][1].tolist(),
        case["Wo"].tolist(), case["gamma_q"].tolist(), case["gamma_k"].tolist(),
        H, Hkv, dh, local, W, base, scale, alpha)
    return got, torch.tensor(ref, dtype=F64)


# ----------------------------------------------------------------------------
# brute-force enumeration on T <= 16
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("local,W,valid,H,Hkv", [
    (False, 0, None, 4, 2),
    (False, 0, 9, 4, 1),
    (True, 1, None, 4, 2),
    (True, 3, None, 2, 2),
    (True, 5, 11, 4, 4),
    (True, 16, 7, 4, 1),
    (True, 4, 16, 4, 2),
])
def test_bruteforce_matches(local, W, valid, H, Hkv):
    T = 16 if valid in (None, 16) else 13
    case = _case(T=T, H=H, Hkv=Hkv, seed=10 * W + H, valid=valid)
    got, ref = _run_both(case, H, Hkv, 4, local, W, base=10.0, scale=2.0, alpha=0.7)
    assert torch.allclose(got, ref, rtol=1e-12, atol=1e-12), (got - ref).abs().max()


def test_mask_sets_enumerated():
    # The sliding mask times the causal mask keeps exactly t - W < s <= t.
    for T in (1, 2, 5, 16):
        for W in (1, 2, 3, 8, 20):
            idx = torch.arange(T)
            m = O.create_sliding_mask(idx, idx, W) & O.causal_padding_mask(idx, idx, T)
            for t in range(T):
                for s in range(T):
                    assert bool(m[t, s]) == (t - W < s <= t)


# ----------------------------------------------------------------------------
# projections: scalar loops
# ----------------------------------------------------------------------------
def test_projection_scalar_loops():
    x = _rand((3, 5), 1)
    W = _rand((7, 5), 2)
    got = O.project(x, W)
    for i in range(3):
        for n in range(7):
            ref = sum(float(x[i, d]) * float(W[n, d]) for d in range(5))
            assert abs(float(got[i, n]) - ref) < 1e-12


# ----------------------------------------------------------------------------
# RMSNorm closed forms ("QK-Norm", How it works and Watch-outs)
# ----------------------------------------------------------------------------
def test_rmsnorm_constant_vector_closed_form():
    for c in (0.5, -3.0, 1e-4):
        x = torch.full((6,), c, dtype=F64)
        y = O.rms_norm(x, torch.zeros(6, dtype=F64))
        assert torch.allclose(y, torch.full((6,), c / math.sqrt(c * c + 1e-6), dtype=F64),
                              rtol=1e-14, atol=0)


def test_rmsnorm_one_hot_closed_form():
    x = torch.zeros(8, dtype=F64)
    x[3] = 2.0
    g = torch.linspace(-0.5, 0.5, 8, dtype=F64)
    y = O.rms_norm(x, g)
    expect = 2.0 / math.sqrt(4.0 / 8 + 1e-6) * (1 + float(g[3]))
    assert abs(float(y[3]) - expect) < 1e-13
    assert float(y.abs().sum() - y[3].abs()) == 0.0


def test_rmsnorm_zero_gamma_is_identity_up_to_rms_and_unit_rms():
    x = _rand((5, 3, 64), 7, 3.0)
    y = O.rms_norm(x, torch.zeros(64, dtype=F64))
    m = (x * x).mean(-1)
    rms_y = (y * y).mean(-1).sqrt()
    # Every normalised head has RMS sqrt(m / (m + eps)) (1 up to eps).
    assert torch.allclose(rms_y, (m / (m + 1e-6)).sqrt(), rtol=1e-13, atol=0)
    assert torch.allclose(rms_y, torch.ones_like(rms_y), atol=1e-6)
    # gamma = 0: same direction as x (identity up to RMS scaling).
    ratio = y / x
    assert torch.allclose(ratio, ratio[..., :1].expand_as(ratio), rtol=1e-12)


def test_rmsnorm_last_axis_only():
    x = _rand((2, 3, 16), 3)
    g = _rand((16,), 4, 0.3)
    y = O.rms_norm(x, g)
    for i in range(2):
        for j in range(3):
            assert torch.allclose(O.rms_norm(x[i, j], g), y[i, j], rtol=1e-14, atol=0)


# ----------------------------------------------------------------------------
# RoPE invariants (the rotation law itself is a reading: parity unpinned)
# ----------------------------------------------------------------------------
def test_rope_pos0_identity_and_norm_preserving():
    x = _rand((1, 9, 3, 32), 11)
    pos = torch.arange(9).reshape(1, 9) * 1000
    y = O.rope(x, torch.zeros(1, 9, dtype=torch.int64), 1e4, 1.0)
    assert torch.equal(y, x)
    y = O.rope(x, pos, 1e6, 8.0)
    assert torch.allclose(y.norm(dim=-1), x.norm(dim=-1), rtol=1e-13)
    # pairs (c, c + d/2) keep their own norm: a rotation acts inside each pair
    h = 16
    pn_x = x[..., :h] ** 2 + x[..., h:] ** 2
    pn_y = y[..., :h] ** 2 + y[..., h:] ** 2
    assert torch.allclose(pn_x, pn_y, rtol=1e-12)


def test_rope_relative_position_logits_invariant():
    q = _rand((1, 6, 1, 16), 1)
    k = _rand((1, 6, 1, 16), 2)
    pos = torch.tensor([[0, 5, 17, 100, 4000, 131071]])
    for base, scale in ((1e4, 1.0), (1e6, 8.0)):
        ref = torch.einsum("btc,bsc->bts", O.rope(q, pos, base, scale)[:, :, 0],
                           O.rope(k, pos, base, scale)[:, :, 0])
        for shift in (1, 123, 77777):
            got = torch.einsum("btc,bsc->bts", O.rope(q, pos + shift, base, scale)[:, :, 0],
                               O.rope(k, pos + shift, base, scale)[:, :, 0])
            assert torch.allclose(got, ref, rtol=0, atol=1e-9 * ref.abs().max())


def test_rope_composition_and_scale_semantics():
    x = _rand((1, 4, 2, 8), 5)
    p1 = torch.tensor([[1, 2, 30, 400]])
    p2 = torch.tensor([[7, 0, 5, 123]])
    a = O.rope(O.rope(x, p1, 1e4, 1.0), p2, 1e4, 1.0)
    b = O.rope(x, p1 + p2, 1e4, 1.0)
    assert torch.allclose(a, b, atol=1e-12)
    # scale s at position s*p rotates like scale 1 at position p
    assert torch.allclose(O.rope(x, 8 * p1, 1e6, 8.0), O.rope(x, p1, 1e6, 1.0), atol=1e-12)


def test_rope_lowest_pair_turns_by_position():
    # The c = 0 pair has frequency base^0 = 1 under every base: angle = pos/scale.
    x = torch.zeros(1, 1, 1, 8, dtype=F64)
    x[..., 0] = 1.0
    for pos, scale in ((3, 1.0), (40, 8.0)):
        y = O.rope(x, torch.tensor([[pos]]), 1e4, scale)
        a = pos / scale
        assert abs(float(y[..., 0]) - math.cos(a)) < 1e-14
        assert abs(float(y[..., 4]) - math.sin(a)) < 1e-14


# ----------------------------------------------------------------------------
# attention-level invariants
# ----------------------------------------------------------------------------
def _layer(case, **kw):
    base = dict(H=4, H_kv=2, d_h=8, attn_type=O.GLOBAL, window=0, rope_base=1e4,
                rope_scale=1.0, query_scale=8 ** -0.5)
    base.update(kw)
    return O.attention_layer(**case, **base)


def test_local_with_window_ge_T_equals_global():
    case = _case(T=40, D=16, H=4, Hkv=2, dh=8, seed=3, valid=33)
    g = _layer(case)
    for W in (40, 41, 1000):
        l = _layer(case, attn_type=O.LOCAL_SLIDING, window=W)
        assert torch.equal(g, l)
    l = _layer(case, attn_type=O.LOCAL_SLIDING, window=20)
    assert not torch.allclose(g, l)


def test_gqa_equals_mha_with_replicated_kv_heads():
    H, Hkv, dh = 4, 2, 8
    case = _case(T=24, D=16, H=H, Hkv=Hkv, dh=dh, seed=4)
    gqa = _layer(case, H=H, H_kv=Hkv, d_h=dh)
    G = H // Hkv
    Wk, Wv = case["Wkv"][0].reshape(Hkv, dh, -1), case["Wkv"][1].reshape(Hkv, dh, -1)
    rep = lambda W: W.repeat_interleave(G, dim=0).reshape(H * dh, -1)
    mha_case = dict(case, Wkv=torch.stack([rep(Wk), rep(Wv)]))
    mha = _layer(mha_case, H=H, H_kv=H, d_h=dh)
    assert torch.allclose(gqa, mha, rtol=1e-12, atol=1e-14)


def test_softmax_weights_sum_to_one_constant_values():
    # Feature 0 of x is 1 on every row and only it feeds V, so V[s] = v for all s;
    # with weights summing to one each valid row's output is v @ Wo^T.
    case = _case(T=20, D=16, H=4, Hkv=2, dh=8, seed=6, valid=15)
    case["x"][..., 0] = 1.0
    Wv = torch.zeros(2 * 8, 16, dtype=F64)
    Wv[:, 0] = _rand((16,), 9)
    case["Wkv"] = torch.stack([case["Wkv"][0], Wv])
    for kw in (dict(), dict(attn_type=O.LOCAL_SLIDING, window=3)):
        out = _layer(case, **kw)[0]
        enc = Wv[:, 0].reshape(2, 8).repeat_interleave(2, dim=0).reshape(-1)
        expect = case["Wo"] @ enc
        assert torch.allclose(out[:15], expect.expand(15, -1), rtol=1e-12, atol=1e-14)
        assert torch.equal(out[15:], torch.zeros_like(out[15:]))


def test_logits_shift_invariance_end_to_end():
    case = _case(T=16, D=16, H=4, Hkv=1, dh=8, seed=8)
    a = _layer(case, H=4, H_kv=1, rope_base=1e6, rope_scale=8.0)
    shifted = dict(case, segment_pos=case["segment_pos"] + 100000)
    b = _layer(shifted, H=4, H_kv=1, rope_base=1e6, rope_scale=8.0)
    assert torch.allclose(a, b, rtol=0, atol=1e-9)


def test_sampled_rows_equal_full_rows():
    case = _case(T=48, D=16, H=4, Hkv=2, dh=8, seed=12, valid=40)
    for kw in (dict(), dict(attn_type=O.LOCAL_SLIDING, window=7)):
        full = _layer(case, **kw)[0]
        rows = [0, 6, 7, 20, 39, 40, 47]
        samp = _layer(case, rows=[rows], **kw)[0]
        assert torch.allclose(samp, full[rows], rtol=1e-12, atol=1e-14)


def test_k_mask_blocked_logits_are_exact_zero_weight():
    # A blocked logit K_MASK next to any finite logit has weight exp(K_MASK - m) == 0.
    l = torch.tensor([0.3, O.K_MASK, -5.0], dtype=F64)
    p = torch.softmax(l, 0)
    assert float(p[1]) == 0.0


# ----------------------------------------------------------------------------
# values the pages print
# ----------------------------------------------------------------------------
def test_constants_match_pages():
    c = _golden("constants.json")
    assert O.K_MASK == c["K_MASK"]["value"]
    assert O.RMS_EPS == c["rms_eps"]["value"]
    q27 = c["query_scale_27B"]
    assert O.query_pre_attn_scalar("27B", q27["D"], q27["H"], q27["d_h"]) == pytest.approx(
        q27["value"], rel=1e-15)
    assert O.query_pre_attn_scalar("27B", q27["D"], q27["H"], q27["d_h"]) != 128 ** -0.5
    qd = c["query_scale_default"]
    for size in ("1B", "4B", "12B"):
        assert O.query_pre_attn_scalar(size, 2560, 8, qd["d_h"]) == qd["value"]
    for size, kind, base, scale, window in c["layer_params"]["rows"]:
        assert O.layer_params(kind, size) == (base, scale, window)


def test_routing_golden_table():
    g = _golden("routing_types.json")["types"]
    for n, s in g.items():
        got = O.make_attention_layers_types(int(n))
        assert "".join("L" if t == O.LOCAL_SLIDING else "G" for t in got) == s


def test_routing_counts_and_first_local():
    for n in range(1, 64):
        t = O.make_attention_layers_types(n)
        assert len(t) == n and t[0] == O.LOCAL_SLIDING
        assert sum(x == O.GLOBAL for x in t) == n // 6
        assert all(x == O.LOCAL_SLIDING for x in t[n - n % 6:])
