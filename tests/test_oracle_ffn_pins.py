"""Pins of the oracle's feed-forward half ("Full Gemma 3 Block", How it works:
the MLP paragraph and the last three lines of Block.__call__).

Independent of the oracle's formulas: properties of the tanh-form GELU,
closeness to the exact (erf) GELU, a scalar brute force of the gated
feed-forward written from the einsum string, structural zeros of the block,
and the hidden-width table the page prints.
"""
import json
import math
import os

import torch

from oracle import gemma3_oracle as O

F64 = torch.float64
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g, dtype=F64) * std


def test_gelu_tanh_odd_part_is_identity():
    # tanh is odd, so gelu(x) - gelu(-x) = x for the tanh form.
    x = torch.linspace(-8, 8, 1001, dtype=F64)
    assert torch.allclose(O.gelu_tanh(x) - O.gelu_tanh(-x), x, rtol=0, atol=1e-13)


def test_gelu_tanh_limits_and_zero():
    assert float(O.gelu_tanh(torch.tensor(0.0, dtype=F64))) == 0.0
    big = torch.tensor([30.0, 50.0], dtype=F64)
    assert torch.allclose(O.gelu_tanh(big), big, rtol=1e-15)
    assert torch.all(O.gelu_tanh(-big).abs() < 1e-30)


def test_gelu_tanh_is_close_to_exact_gelu():
    # The tanh form approximates x * Phi(x); on [-6, 6] the two differ by
    # well under 1e-3 but not by less than 1e-5 (it is not the erf form).
    x = torch.linspace(-6, 6, 2001, dtype=F64)
    exact = torch.tensor([v * 0.5 * (1 + math.erf(v / math.sqrt(2))) for v in x.tolist()],
                         dtype=F64)
    d = (O.gelu_tanh(x) - exact).abs().max()
    assert 1e-5 < float(d) < 1e-3


def _brute_ffn(u, Wg, Wd):
    """Scalar loops: gate/up[n][h] = sum_f u[f] * W[n][h][f] (the einsum
    '...F,NHF->...NH'); z[h] = gelu(gate[h]) * up[h] with the tanh form;
    out[d] = sum_h z[h] * Wd[h][d] (W_d of shape (D_ff, D))."""
    D = len(u)
    Dff = len(Wg[0])
    gu = [[sum(u[f] * Wg[n][h][f] for f in range(D)) for h in range(Dff)] for n in range(2)]
    z = []
    for h in range(Dff):
        g = gu[0][h]
        z.append(0.5 * g * (1 + math.tanh(math.sqrt(2 / math.pi) * (g + 0.044715 * g ** 3)))
                 * gu[1][h])
    return [sum(z[h] * Wd[h][d] for h in range(Dff)) for d in range(len(Wd[0]))]


def test_feed_forward_scalar_brute_force():
    D, Dff = 6, 10
    u = _rand((3, D), 1)
    Wg = _rand((2, Dff, D), 2, 0.5)
    Wd = _rand((Dff, D), 3, 0.3)
    got = O.feed_forward(u, Wg, Wd)
    for i in range(3):
        ref = _brute_ffn(u[i].tolist(), Wg.tolist(), Wd.tolist())
        assert torch.allclose(got[i], torch.tensor(ref, dtype=F64), rtol=1e-12, atol=1e-13)


def test_zero_up_slice_gives_zero_ffn():
    u = _rand((4, 8), 4)
    Wg = _rand((2, 12, 8), 5)
    Wg[1] = 0.0
    assert torch.equal(O.feed_forward(u, Wg, _rand((12, 8), 6)), torch.zeros(4, 8, dtype=F64))


def test_block_ffn_structural_zeros():
    h = _rand((2, 5, 8), 7)
    Wg = _rand((2, 12, 8), 8)
    g = _rand((8,), 9, 0.3)
    # W_d = 0: m = 0, RMSNorm(0) = 0, so y = h exactly.
    assert torch.equal(O.block_ffn(h, g, g, Wg, torch.zeros(12, 8, dtype=F64)), h)
    # post-ffn scale (1 + gamma) = 0: the sandwich adds nothing.
    assert torch.equal(O.block_ffn(h, g, -torch.ones(8, dtype=F64), Wg, _rand((12, 8), 10)), h)


def test_block_ffn_is_rowwise():
    h = _rand((1, 9, 8), 11)
    Wg, Wd = _rand((2, 16, 8), 12), _rand((16, 8), 13)
    g1, g2 = _rand((8,), 14, 0.3), _rand((8,), 15, 0.3)
    full = O.block_ffn(h, g1, g2, Wg, Wd)
    for t in range(9):
        assert torch.allclose(O.block_ffn(h[:, t:t + 1], g1, g2, Wg, Wd), full[:, t:t + 1],
                              rtol=1e-14, atol=0)


def test_hidden_dims_match_page():
    with open(os.path.join(GOLDEN, "ffn_hidden_dims.json")) as f:
        rows = json.load(f)["rows"]
    for size, D, Dff in rows:
        assert O.ffn_hidden_dim(size, D) == Dff
