"""Pins of the oracle's model wrapper ("Full Gemma 3 Block", How it works,
last paragraph: embed times sqrt(D), N blocks, final RMSNorm, read-out
through the embedding table), with the routing of "Global vs Local Layer
Routing".

Closed forms (embedding rows of +-1 entries; a scaled identity table through
a zero-layer model), scalar loops for the read-out, and the hand-written
routing table of tests/golden/ for the layer types inside the model; the
planted mistakes at the end each fail one of them.
"""
import json
import math
import os

import pytest
import torch

from oracle import gemma3_oracle as O

F64 = torch.float64
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g, dtype=F64) * std


def test_embedding_of_unit_entries_has_mean_square_d():
    # rows of +-1 entries: every embedded element is +-sqrt(D), so the mean
    # square over a row is exactly D and the signs are the table's
    V, D = 11, 48
    signs = torch.where(_rand((V, D), 1) > 0, 1.0, -1.0).to(F64)
    tokens = torch.tensor([[0, 5, 10, 5]])
    x = O.embed(tokens, signs)
    assert torch.allclose((x * x).mean(-1), torch.full((1, 4), float(D), dtype=F64),
                          rtol=1e-15, atol=0)
    assert torch.equal(torch.sign(x[0]), signs[tokens[0]])


def _zero_layer_closed_form(D, s, gamma, t):
    # E = s * I (V = D): x = sqrt(D) s e_t, mean(x^2) = s^2, so the final norm
    # gives sqrt(D) s / sqrt(s^2 + eps) (1 + gamma_t) e_t and the read-out
    # multiplies by s: logits = delta_{tv} sqrt(D) s^2 (1 + gamma_t) / sqrt(s^2 + eps).
    out = torch.zeros(D, dtype=F64)
    out[t] = math.sqrt(D) * s * s * (1.0 + float(gamma[t])) / math.sqrt(s * s + 1e-6)
    return out


@pytest.mark.parametrize("s", [0.05, 1.0, 3.0])
def test_zero_layer_model_closed_form(s):
    D = 32
    E = s * torch.eye(D, dtype=F64)
    gamma = _rand((D,), 2, 0.3)
    tokens = torch.tensor([[3, 0, 31]])
    logits = O.model_forward(tokens, E, [], gamma, model_size="1B", H=2, H_kv=1, d_h=16,
                             segment_pos=torch.arange(3)[None], pad_lens=None)
    for i, t in enumerate(tokens[0].tolist()):
        assert torch.allclose(logits[0, i], _zero_layer_closed_form(D, s, gamma, t),
                              rtol=1e-13, atol=1e-15)


def test_tied_read_out_scalar_loops():
    V, D = 7, 10
    E = _rand((V, D), 3)
    h = _rand((2, 3, D), 4)
    got = O.tied_logits(h, E)
    for b in range(2):
        for t in range(3):
            for v in range(V):
                ref = sum(float(h[b, t, d]) * float(E[v, d]) for d in range(D))
                assert abs(float(got[b, t, v]) - ref) < 1e-12


def _layers(n, D, H, H_kv, d_h, D_ff, seed):
    out = []
    for l in range(n):
        k = seed + 100 * l
        out.append(dict(
            Wq=_rand((H * d_h, D), k + 1, D ** -0.5), Wkv=_rand((2, H_kv * d_h, D), k + 2, D ** -0.5),
            Wo=_rand((D, H * d_h), k + 3, (H * d_h) ** -0.5), gamma_q=_rand((d_h,), k + 4, 0.3),
            gamma_k=_rand((d_h,), k + 5, 0.3), gamma_pre=_rand((D,), k + 6, 0.3),
            gamma_post=_rand((D,), k + 7, 0.3), gamma_pre_ffn=_rand((D,), k + 8, 0.3),
            gamma_post_ffn=_rand((D,), k + 9, 0.3),
            W_gating=_rand((2, D_ff, D), k + 10, D ** -0.5),
            W_down=_rand((D_ff, D), k + 11, D_ff ** -0.5)))
    return out


def test_model_layers_follow_the_golden_routing_table():
    # 7 blocks on the 1B-shaped sizes (window 512) with T = 530 > 512, so a
    # local and a global layer differ; the model must equal the chain whose
    # types are read from the hand-written table.
    with open(os.path.join(GOLDEN, "routing_types.json")) as f:
        types = json.load(f)["types"]["7"]
    V, D, H, H_kv, d_h, D_ff, T = 64, 16, 2, 1, 8, 32, 530
    E = _rand((V, D), 5, D ** -0.5)
    layers = _layers(7, D, H, H_kv, d_h, D_ff, 50)
    gf = _rand((D,), 6, 0.3)
    g = torch.Generator().manual_seed(7)
    tokens = torch.randint(0, V, (1, T), generator=g)
    pos = torch.arange(T)[None]
    got = O.model_forward(tokens, E, layers, gf, model_size="1B", H=H, H_kv=H_kv, d_h=d_h,
                          segment_pos=pos, pad_lens=None)
    x = O.embed(tokens, E)
    for l, p in enumerate(layers):
        local = types[l] == "L"
        x = O.full_block(x, p["gamma_pre"], p["gamma_post"], p["gamma_pre_ffn"],
                         p["gamma_post_ffn"], p["W_gating"], p["W_down"], segment_pos=pos,
                         pad_lens=None, Wq=p["Wq"], Wkv=p["Wkv"], Wo=p["Wo"],
                         gamma_q=p["gamma_q"], gamma_k=p["gamma_k"], H=H, H_kv=H_kv, d_h=d_h,
                         attn_type=O.LOCAL_SLIDING if local else O.GLOBAL,
                         window=512 if local else 0, rope_base=1e4 if local else 1e6,
                         rope_scale=1.0, query_scale=d_h ** -0.5)
    ref = O.tied_logits(O.rms_norm(x, gf), E)
    assert torch.allclose(got, ref, rtol=1e-12, atol=1e-12)
    # and the types matter here: all-global differs
    x2 = O.embed(tokens, E)
    for p in layers:
        x2 = O.full_block(x2, p["gamma_pre"], p["gamma_post"], p["gamma_pre_ffn"],
                          p["gamma_post_ffn"], p["W_gating"], p["W_down"], segment_pos=pos,
                          pad_lens=None, Wq=p["Wq"], Wkv=p["Wkv"], Wo=p["Wo"],
                          gamma_q=p["gamma_q"], gamma_k=p["gamma_k"], H=H, H_kv=H_kv,
                          d_h=d_h, attn_type=O.GLOBAL, window=0, rope_base=1e6,
                          rope_scale=1.0, query_scale=d_h ** -0.5)
    assert not torch.allclose(O.tied_logits(O.rms_norm(x2, gf), E), ref, rtol=1e-6, atol=1e-6)


def test_embedding_scale_reaches_the_residual_stream():
    # One block whose attention output projection is zero: h = x + RMSNorm(0)
    # = x, then y = x + RMSNorm_post(FFN(...)).  The post-norm term has the
    # same size whatever x's scale, so y / |x| depends on sqrt(D): compare the
    # model with the chain built on an explicitly scaled embedding.
    V, D, H, H_kv, d_h, D_ff, T = 32, 16, 2, 1, 8, 32, 5
    E = _rand((V, D), 8, D ** -0.5)
    layers = _layers(1, D, H, H_kv, d_h, D_ff, 90)
    layers[0]["Wo"] = torch.zeros_like(layers[0]["Wo"])
    gf = torch.zeros(D, dtype=F64)
    tokens = torch.tensor([[1, 2, 3, 4, 5]])
    pos = torch.arange(T)[None]
    got = O.model_forward(tokens, E, layers, gf, model_size="1B", H=H, H_kv=H_kv, d_h=d_h,
                          segment_pos=pos, pad_lens=None)
    p = layers[0]
    x = E[tokens] * math.sqrt(D)
    m = O.feed_forward(O.rms_norm(x, p["gamma_pre_ffn"]), p["W_gating"], p["W_down"])
    y = x + O.rms_norm(m, p["gamma_post_ffn"])
    ref = O.tied_logits(O.rms_norm(y, gf), E)
    assert torch.allclose(got, ref, rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------------------------
# planted mistakes (on the CPU, in the oracle)
# ----------------------------------------------------------------------------
def _fails(fn, *a):
    try:
        fn(*a)
    except AssertionError:
        return True
    return False


def test_missing_sqrt_d_is_caught(monkeypatch):
    monkeypatch.setattr(O, "embed", lambda tokens, E: E.to(F64)[tokens.to(torch.int64)])
    assert _fails(test_embedding_of_unit_entries_has_mean_square_d)
    assert _fails(test_embedding_scale_reaches_the_residual_stream)


def test_final_norm_without_one_plus_gamma_is_caught(monkeypatch):
    real = O.rms_norm

    def gamma_only(x, gamma, eps=1e-6):
        x = x.to(F64)
        return x / torch.sqrt((x * x).mean(-1, keepdim=True) + eps) * gamma.to(F64)

    monkeypatch.setattr(O, "rms_norm", gamma_only)
    assert _fails(test_zero_layer_model_closed_form, 1.0)
    monkeypatch.setattr(O, "rms_norm", real)


def test_routing_from_one_is_caught(monkeypatch):
    real = O.make_attention_layers_types
    monkeypatch.setattr(O, "make_attention_layers_types",
                        lambda n, pattern=O.GEMMA3_ATTENTION_PATTERN: real(n + 1)[1:])
    assert _fails(test_model_layers_follow_the_golden_routing_table)
