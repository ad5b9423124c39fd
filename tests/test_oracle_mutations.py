"""Planted mistakes in the oracle must be caught by its pins.

Each case swaps one function of the oracle (on the CPU, via monkeypatch) for a
plausible wrong variant -- most of them the pages' own "Watch-outs" -- and
checks that at least one pin test then fails.
"""
import pytest
import torch

from oracle import gemma3_oracle as O
from tests import test_oracle_pins as P

F64 = torch.float64


def _fails(fn, *a):
    try:
        fn(*a)
    except AssertionError:
        return True
    return False


def _t5_rms_norm(x, gamma, eps=1e-6):
    # "QK-Norm", Watch-outs: gamma * x_hat instead of (1 + gamma) * x_hat
    x = x.to(F64)
    return x / torch.sqrt((x * x).mean(-1, keepdim=True) + eps) * gamma.to(F64)


def _rms_norm_wrong_axis(x, gamma, eps=1e-6):
    x = x.to(F64)
    if x.dim() < 2:
        return x / torch.sqrt((x * x).mean() + eps) * (1 + gamma.to(F64))
    return x / torch.sqrt((x * x).mean(dim=(-1, -2), keepdim=True) + eps) * (1 + gamma.to(F64))


def test_t5_style_norm_is_caught(monkeypatch):
    monkeypatch.setattr(O, "rms_norm", _t5_rms_norm)
    assert _fails(P.test_rmsnorm_zero_gamma_is_identity_up_to_rms_and_unit_rms)
    assert _fails(P.test_bruteforce_matches, False, 0, None, 4, 2)


def test_norm_over_wrong_axis_is_caught(monkeypatch):
    monkeypatch.setattr(O, "rms_norm", _rms_norm_wrong_axis)
    assert _fails(P.test_rmsnorm_last_axis_only)


def test_rope_before_norm_is_caught(monkeypatch):
    # "QK-Norm", Watch-outs: norm before RoPE, not after.  The planted variant
    # defers each norm until after the rotation of the same tensor.
    real_norm, real_rope = O.rms_norm, O.rope
    pending = []

    def norm_later(x, gamma, eps=1e-6):
        pending.append(gamma)
        return x.to(F64)

    def rope_then_norm(x, positions, base, scale):
        return real_norm(real_rope(x, positions, base, scale), pending.pop(0))

    monkeypatch.setattr(O, "rms_norm", norm_later)
    monkeypatch.setattr(O, "rope", rope_then_norm)
    assert _fails(P.test_bruteforce_matches, False, 0, None, 4, 2)


def test_tied_qk_gamma_is_caught(monkeypatch):
    # "QK-Norm", Watch-outs: one RMSNorm reused for Q and K is a different model.
    real = O.attention_layer

    def tied(*a, **kw):
        if "gamma_k" in kw and "gamma_q" in kw:
            kw = dict(kw, gamma_k=kw["gamma_q"])
        return real(*a, **kw)

    monkeypatch.setattr(O, "attention_layer", tied)
    assert _fails(P.test_bruteforce_matches, True, 5, 11, 4, 4)


def test_missing_query_scale_is_caught(monkeypatch):
    # "QK-Norm", Watch-outs: QK-norm does not replace the query scale.
    real = O.attention_layer
    monkeypatch.setattr(O, "attention_layer", lambda *a, **kw: real(*a, **dict(kw, query_scale=1.0)))
    assert _fails(P.test_bruteforce_matches, False, 0, 9, 4, 1)


def test_wrong_gqa_head_map_is_caught(monkeypatch):
    # kv head h % H_kv instead of h // G
    real_einsum = torch.einsum

    def einsum(eq, *ops):
        if eq == "tkgc,skc->tkgs":
            q, k = ops
            Tq, Hkv, G, dh = q.shape
            qh = q.reshape(Tq, Hkv * G, dh)
            kk = k[:, torch.arange(Hkv * G) % Hkv]
            return real_einsum("thc,shc->ths", qh, kk).reshape(Tq, Hkv, G, -1)
        if eq == "tkgs,skc->tkgc":
            p, v = ops
            Tq, Hkv, G, S = p.shape
            vv = v[:, torch.arange(Hkv * G) % Hkv]
            return real_einsum("ths,shc->thc", p.reshape(Tq, Hkv * G, S), vv).reshape(Tq, Hkv, G, -1)
        return real_einsum(eq, *ops)

    monkeypatch.setattr(O.torch, "einsum", einsum)
    assert _fails(P.test_gqa_equals_mha_with_replicated_kv_heads)


def test_window_off_by_one_is_caught(monkeypatch):
    monkeypatch.setattr(O, "create_sliding_mask",
                        lambda t, s, W: (s[None, :] >= t[:, None] - W) & (s[None, :] < t[:, None] + W))
    assert _fails(P.test_mask_sets_enumerated)
    assert _fails(P.test_bruteforce_matches, True, 3, None, 2, 2)


def test_one_based_routing_is_caught(monkeypatch):
    # "Global vs Local Layer Routing", Watch-outs: a 1-based "every 6th layer is
    # global" rule inverts the stack.
    monkeypatch.setattr(O, "make_attention_layers_types",
                        lambda n, pattern=O.GEMMA3_ATTENTION_PATTERN:
                        tuple(O.GLOBAL if (l % 6) == 0 else O.LOCAL_SLIDING for l in range(n)))
    assert _fails(P.test_routing_golden_table)


def test_wrap_remainder_routing_is_caught(monkeypatch):
    # "Do not force an exact 5:1": a remainder that wraps to insert a global
    monkeypatch.setattr(O, "make_attention_layers_types",
                        lambda n, pattern=O.GEMMA3_ATTENTION_PATTERN:
                        tuple(pattern[l % 6] if l < n - 1 or n % 6 == 0 else O.GLOBAL
                              for l in range(n)))
    assert _fails(P.test_routing_golden_table)


def test_gemma2_defaults_are_caught(monkeypatch):
    # "Global vs Local Layer Routing", Watch-outs: Gemma 2's 4096 window and
    # one base for every layer are wrong defaults.
    monkeypatch.setattr(O, "layer_params", lambda kind, size: (1e4, 1.0, 4096))
    assert _fails(P.test_constants_match_pages)


def test_rope_without_scale_division_is_caught(monkeypatch):
    real = O.rope
    monkeypatch.setattr(O, "rope", lambda x, p, base, scale: real(x, p, base, 1.0))
    assert _fails(P.test_rope_composition_and_scale_semantics)


def test_causal_leak_is_caught(monkeypatch):
    monkeypatch.setattr(O, "causal_padding_mask",
                        lambda t, s, valid: (s[None, :] <= t[:, None] + 1) & (s[None, :] < valid))
    assert _fails(P.test_bruteforce_matches, False, 0, None, 4, 2)


def test_padding_ignored_is_caught(monkeypatch):
    monkeypatch.setattr(O, "causal_padding_mask",
                        lambda t, s, valid: (s[None, :] <= t[:, None]))
    real = O.attention_layer

    def no_zero(*a, **kw):
        kw = dict(kw)
        kw["pad_lens"] = torch.zeros_like(kw["pad_lens"])
        return real(*a, **kw)

    monkeypatch.setattr(O, "attention_layer", no_zero)
    assert _fails(P.test_bruteforce_matches, False, 0, 9, 4, 1)


# ---------------------------------------------------------------- feed-forward half
from tests import test_oracle_ffn_pins as PF  # noqa: E402


def test_gate_and_up_swapped_is_caught(monkeypatch):
    real = O.feed_forward
    monkeypatch.setattr(O, "feed_forward", lambda u, W, Wd: real(u, W.flip(0), Wd))
    assert _fails(PF.test_feed_forward_scalar_brute_force)


def test_exact_erf_gelu_is_caught(monkeypatch):
    # The page names the approximate tanh form, not the erf form.
    monkeypatch.setattr(O, "gelu_tanh",
                        lambda x: x.to(F64) * 0.5 * (1 + torch.special.erf(x.to(F64) / 2 ** 0.5)))
    assert _fails(PF.test_gelu_tanh_odd_part_is_identity) or _fails(
        PF.test_feed_forward_scalar_brute_force)
    assert _fails(PF.test_gelu_tanh_is_close_to_exact_gelu)


def test_gelu_on_up_slice_is_caught(monkeypatch):
    def wrong(u, W, Wd):
        gu = torch.einsum("...f,nhf->...nh", u.to(F64), W.to(F64))
        return torch.matmul(gu[..., 0, :] * O.gelu_tanh(gu[..., 1, :]), Wd.to(F64))
    monkeypatch.setattr(O, "feed_forward", wrong)
    assert _fails(PF.test_feed_forward_scalar_brute_force)


def test_missing_post_ffn_norm_is_caught(monkeypatch):
    monkeypatch.setattr(O, "block_ffn", lambda h, g1, g2, W, Wd: h.to(F64) + O.feed_forward(
        O.rms_norm(h, g1), W, Wd))
    assert _fails(PF.test_block_ffn_structural_zeros)


def test_hidden_width_8d_is_caught(monkeypatch):
    monkeypatch.setattr(O, "ffn_hidden_dim", lambda size, D: 8 * D)
    assert _fails(PF.test_hidden_dims_match_page)
