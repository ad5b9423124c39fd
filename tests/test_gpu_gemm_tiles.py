"""The projection GEMM's 256-row tiles against its 128-row tiles.

A 256-row tile is two 128-row halves that share each staged W tile; the
halves' accumulators fill TMEM, so a tile's second half may start its MMAs
several k-steps after the first (the stages it needs are held until then).
Each half sums its k-steps in the same order as a 128-row tile, so every
output must equal the 128-row result bit for bit, whatever the shape: an
odd count of 128-row M tiles (a last unit with no second half), fewer
k-steps than stages, ragged M / N / K, a half-width last tile column,
persistent grids that turn the rings over many times, padded batch
segments, the GeGLU epilogue, and the whole layer and block entry points
that run these GEMMs.  The products are also compared with fp64.
"""
import pytest
import torch

from oracle import gemma3_oracle as O
from tests import helpers as Hh
from tests.helpers import rel_frob
from transformer_attention_gb300 import workloads as WL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from transformer_attention_gb300.build import build
    build()
    import transformer_attention_gb300 as G3
    G3.lib()
    torch.cuda.init()


def _with_rows(rows, fn):
    """fn() with the GEMM's rows per tile set to `rows`, restored after."""
    import transformer_attention_gb300 as G3
    prev = G3.gemma3_set_gemm_tile_rows(rows)
    try:
        out = fn()
        assert G3.gemma3_attn_check_status() == 0
        return out
    finally:
        G3.gemma3_set_gemm_tile_rows(prev)


def _randn(shape, seed, std=1.0, dtype=torch.bfloat16):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * std).to(dtype)


SHAPES = [
    (640, 512, 1152),     # 5 M tiles: the last unit's second half holds no rows
    (1024, 2048, 2560),   # long K: stages held for the second half, then caught up
    (389, 1096, 520),     # ragged M and K; a last tile column of 72 (half-width MMAs)
    (256, 256, 64),       # one k-step, fewer than the stages
    (384, 384, 128),      # two k-steps; 3 M tiles; N 1.5 tiles
    (5170, 2200, 1024),   # more units than SMs, 41 M tiles
    (130, 200, 72),       # one unit, two ragged halves
]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("out", ["bf16", "f32"])
@pytest.mark.parametrize("inp", ["bf16", "f16"])
def test_two_half_tiles_equal_one_half(M, N, K, out, inp):
    import transformer_attention_gb300 as G3
    dt = {"bf16": torch.bfloat16, "f32": torch.float32}[out]
    it = {"bf16": torch.bfloat16, "f16": torch.float16}[inp]
    A = _randn((M, K), 11, 1.0, it)
    W = _randn((N, K), 12, K ** -0.5, it)
    Ad, Wd = A.cuda(), W.cuda()
    C1 = _with_rows(128, lambda: G3.linear(Ad, Wd, out_dtype=dt))
    C2 = _with_rows(256, lambda: G3.linear(Ad, Wd, out_dtype=dt))
    assert torch.equal(C1.cpu(), C2.cpu())
    tol = {"bf16": 4e-3, "f32": 1e-5}[out]
    assert rel_frob(C2.cpu(), O.project(A, W)) <= tol


@pytest.mark.parametrize("max_ctas", [3, 1])
def test_two_half_tiles_small_grid(max_ctas):
    # 40 units of 256 x 256 walked by 3 CTAs, or by one: the three-stage ring
    # and the two halves' accumulator phases turn over many times per CTA
    import transformer_attention_gb300 as G3
    A = _randn((2048, 640), 13).cuda()
    W = _randn((2560, 640), 14, 640 ** -0.5).cuda()
    C1 = _with_rows(128, lambda: G3.linear(A, W, out_dtype=torch.float32))
    C2 = _with_rows(256, lambda: G3.linear(A, W, out_dtype=torch.float32, max_ctas=max_ctas))
    assert torch.equal(C1.cpu(), C2.cpu())


@pytest.mark.parametrize("pads", [[0, 200, 384, 100], [384, 0, 250], [300, 300, 300]])
@pytest.mark.parametrize("max_ctas", [0, 1])
def test_two_half_tiles_pad_only_tiles(pads, max_ctas):
    """Segments of 384 rows with trailing padding: the computed 128-row tiles
    pair up across segments (a unit's halves may come from different
    segments); pad-only tiles stay unwritten; every computed row equals the
    128-row tiles' result.  With one CTA, every unit goes through the same
    rings in turn."""
    import transformer_attention_gb300 as G3
    T = 384
    M, N, K = T * len(pads), 640, 512
    A = _randn((M, K), 15).cuda()
    W = _randn((N, K), 16, K ** -0.5).cuda()
    pl = torch.tensor(pads, dtype=torch.int32, device="cuda")

    def run():
        C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        G3.gemma3_linear(A, K, W, K, C, N, M, N, K, G3.GEMMA3_BF16, G3.GEMMA3_F32, max_ctas,
                         pad_lens=pl, seg_T=T)
        return C.cpu()

    C1, C2 = _with_rows(128, run), _with_rows(256, run)
    assert torch.equal(C1.isnan(), C2.isnan())
    assert torch.equal(torch.nan_to_num(C1), torch.nan_to_num(C2))
    for b, pad in enumerate(pads):
        kept = -(-(T - pad) // 128) * 128
        assert not bool(C2[b * T:b * T + kept].isnan().any())
        assert bool(C2[b * T + kept:(b + 1) * T].isnan().all())


@pytest.mark.parametrize("M,D_ff,K", [(640, 1024, 512), (389, 640, 1152), (2048, 2560, 640)])
def test_two_half_tiles_geglu(M, D_ff, K):
    import transformer_attention_gb300 as G3
    A = _randn((M, K), 17, 1.0, torch.float16).cuda()
    Wg = _randn((2 * D_ff, K), 18, K ** -0.5, torch.float16).cuda()

    def run():
        Z = torch.empty((M, D_ff), dtype=torch.float16, device="cuda")
        G3.gemma3_geglu(A, K, Wg, K, Z, D_ff, M, D_ff, K, G3.GEMMA3_F16)
        return Z.cpu()

    Z1, Z2 = _with_rows(128, run), _with_rows(256, run)
    assert torch.equal(Z1, Z2)
    ref = O.gelu_tanh(O.project(A.cpu(), Wg[:D_ff].cpu())) * O.project(A.cpu(), Wg[D_ff:].cpu())
    assert rel_frob(Z2, ref) <= 2e-3


LAYER = dict(B=3, T=512, D=256, H=4, H_kv=2, d_h=256, attn_type="local", window=100,
             pad=("pad_uniform", 200, 512))


def test_layer_forward_equal_across_tile_rows():
    """gemma3_attn_forward with padding that fills whole 128-row tiles: the
    output projection (zeros written to pad-only tiles) runs on either tile
    height with the same output bytes."""
    import transformer_attention_gb300 as G3
    w = WL.small(WL.WORKLOADS["tiny_local"], name="tile_rows_layer", **LAYER)
    inp = Hh.make_inputs(w)
    dev = Hh.to_dev(inp)
    need = G3.gemma3_attn_workspace_size(w.B, w.T, w.D, w.H, w.H_kv, w.d_h)

    def run():
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        out = torch.full((w.B, w.T, w.D), float("nan"), dtype=torch.bfloat16, device="cuda")
        G3.gemma3_attn_forward((w.B, w.T, w.D, w.H, w.H_kv, w.d_h), dev["x"],
                               dev["segment_pos"], dev["pad_lens"], dev["Wq"], dev["Wkv"],
                               dev["Wo"], dev["gamma_q"], dev["gamma_k"], Hh.abi_type(w),
                               w.window, w.rope_base, w.rope_scale, w.query_scale, out, ws, need)
        return out.cpu()

    y1, y2 = _with_rows(128, run), _with_rows(256, run)
    assert torch.equal(y1, y2)
    assert not bool(y2.isnan().any())
    ref = Hh.oracle_forward(w, inp)
    for b in range(w.B):
        valid = w.T - int(inp["pad_lens"][b])
        if valid > 0:
            Hh.assert_close(y2[b, :valid], ref[b, :valid], f"two-half layer b={b}")


def test_block_forward_equal_across_tile_rows():
    """gemma3_block_forward (O, GeGLU and down projections, fp32 outputs):
    the same result bytes on either tile height."""
    import transformer_attention_gb300 as G3
    w = WL.small(WL.WORKLOADS["4b_block"], name="tile_rows_block", B=2, T=640, D=512, H=4,
                 H_kv=2, d_h=256, window=128, d_ff=1024, pad=("pad_uniform", 0, 80))
    inp = Hh.make_inputs(w)
    inp.update(WL.block_norm_gammas(w, 0))
    inp.update(WL.ffn_weights(w))
    dev = Hh.to_dev(inp)
    dims = (w.B, w.T, w.D, w.H, w.H_kv, w.d_h)
    need = G3.gemma3_block_workspace_size(dims, w.d_ff)

    def run():
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        y = torch.empty((w.B, w.T, w.D), dtype=torch.float32, device="cuda")
        G3.gemma3_block_forward(dims, w.d_ff, dev["x"], G3.GEMMA3_BF16, y, dev["segment_pos"],
                                dev["pad_lens"], dev["Wq"], dev["Wkv"], dev["Wo"],
                                dev["gamma_q"], dev["gamma_k"], dev["gamma_pre"],
                                dev["gamma_post"], dev["gamma_pre_ffn"], dev["gamma_post_ffn"],
                                dev["W_gating"], dev["W_down"], Hh.abi_type(w), w.window,
                                w.rope_base, w.rope_scale, w.query_scale, ws, need)
        return y.cpu()

    y1, y2 = _with_rows(128, run), _with_rows(256, run)
    assert torch.equal(y1, y2)
    assert bool(torch.isfinite(y2).all())
