"""GPU parity of the feed-forward half and the whole Gemma 3 block against
the fp64 oracle ("Full Gemma 3 Block", How it works: Block.__call__ and the
MLP paragraph).

- the GeGLU gating projection (tcgen05 GEMM with the GELU * up epilogue);
- the feed-forward sandwich alone;
- the whole block at reduced sizes (local and global layers, padding), in full;
- the 4B-shaped full block at full size on the first rows of a batch row
  (attention is causal and the feed-forward row-wise, so those rows depend on
  nothing later).
"""
import pytest
import torch

from oracle import gemma3_oracle as O
from tests import helpers as Hh
from transformer_attention_gb300 import workloads as WL

pytestmark = pytest.mark.gpu

F64 = torch.float64


@pytest.fixture(scope="module", autouse=True)
def _built():
    from transformer_attention_gb300.build import build
    build()


def _randn(shape, seed, std=1.0, dtype=torch.bfloat16):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * std).to(dtype)


@pytest.mark.parametrize("M,D,D_ff", [(256, 512, 2048), (300, 640, 1000), (1024, 2560, 10240),
                                      # a wave of tiles, odd m-tile count, ragged D_ff
                                      (1100, 640, 2600)])
def test_geglu_gemm_matches_oracle(M, D, D_ff):
    import transformer_attention_gb300 as G3
    u = _randn((M, D), 1, 1.0, torch.float16)
    Wg = _randn((2, D_ff, D), 2, D ** -0.5, torch.float16)
    z = torch.empty((M, D_ff), dtype=torch.float16, device="cuda")
    G3.gemma3_geglu(u.cuda(), D, Wg.cuda(), D, z, D_ff, M, D_ff, D, G3.GEMMA3_F16)
    assert G3.gemma3_attn_check_status() == 0
    gu = torch.einsum("mf,nhf->mnh", u.to(F64), Wg.to(F64))
    ref = O.gelu_tanh(gu[:, 0]) * gu[:, 1]
    assert Hh.rel_frob(z.cpu(), ref) <= 2e-3
    assert Hh.max_abs(z.cpu(), ref) <= 2e-2


def test_block_ffn_matches_oracle():
    import transformer_attention_gb300 as G3
    M, D, D_ff = 777, 640, 2560
    w = WL.small(WL.WORKLOADS["4b_block"], D=D, d_ff=D_ff)
    p = WL.ffn_weights(w)
    h = _randn((M, D), 3, 2.0, torch.float32)
    ws = torch.empty(G3.gemma3_block_ffn_workspace_size(M, D, D_ff), dtype=torch.uint8,
                     device="cuda")
    y = torch.empty((M, D), dtype=torch.float32, device="cuda")
    dev = {k: v.cuda() for k, v in p.items()}
    G3.gemma3_block_ffn_forward(M, D, D_ff, h.cuda(), y, dev["gamma_pre_ffn"],
                                dev["gamma_post_ffn"], dev["W_gating"], dev["W_down"], ws,
                                ws.numel())
    assert G3.gemma3_attn_check_status() == 0
    ref = O.block_ffn(h, p["gamma_pre_ffn"], p["gamma_post_ffn"], p["W_gating"],
                      p["W_down"].transpose(0, 1))
    Hh.assert_close(y.cpu(), ref, "block ffn")


def _gpu_block(w, inp, ffn):
    import transformer_attention_gb300 as G3
    dev = Hh.to_dev(dict(inp, **ffn))
    y = G3.block_forward(dev["x"], dev["segment_pos"], dev["pad_lens"], dev["Wq"], dev["Wkv"],
                         dev["Wo"], dev["gamma_q"], dev["gamma_k"], dev["gamma_pre"],
                         dev["gamma_post"], dev["gamma_pre_ffn"], dev["gamma_post_ffn"],
                         dev["W_gating"], dev["W_down"], H=w.H, H_kv=w.H_kv,
                         attn_type=Hh.abi_type(w), window=w.window, rope_base=w.rope_base,
                         rope_scale=w.rope_scale, query_scale=w.query_scale)
    assert G3.gemma3_attn_check_status() == 0
    return y


def _oracle_block(w, inp, ffn, x=None, pad_lens=None, segment_pos=None):
    return O.full_block(
        inp["x"] if x is None else x, inp["gamma_pre"], inp["gamma_post"],
        ffn["gamma_pre_ffn"], ffn["gamma_post_ffn"], ffn["W_gating"],
        ffn["W_down"].transpose(0, 1),
        segment_pos=inp["segment_pos"] if segment_pos is None else segment_pos,
        pad_lens=inp["pad_lens"] if pad_lens is None else pad_lens, Wq=inp["Wq"],
        Wkv=inp["Wkv"], Wo=inp["Wo"], gamma_q=inp["gamma_q"], gamma_k=inp["gamma_k"], H=w.H,
        H_kv=w.H_kv, d_h=w.d_h, attn_type=Hh.oracle_type(w), window=w.window,
        rope_base=w.rope_base, rope_scale=w.rope_scale, query_scale=w.query_scale)


SMALL = [
    dict(B=2, T=700, D=512, H=4, H_kv=2, d_h=256, window=256, d_ff=2048,
         pad=("pad_uniform", 0, 200)),
    dict(B=1, T=600, D=384, H=4, H_kv=2, d_h=128, attn_type="global", window=0,
         rope_base=1e6, rope_scale=8.0, d_ff=1536),
]


@pytest.mark.parametrize("kw", SMALL, ids=["local-d256", "global-d128"])
def test_small_full_block(kw):
    w = WL.small(WL.WORKLOADS["4b_block"], name="block_small", **kw)
    inp = Hh.make_inputs(w)
    inp.update(WL.block_norm_gammas(w, 0))
    ffn = WL.ffn_weights(w)
    got = _gpu_block(w, inp, ffn).cpu()
    ref = _oracle_block(w, inp, ffn)
    for b in range(w.B):
        valid = w.T - int(inp["pad_lens"][b])
        Hh.assert_close(got[b, :valid], ref[b, :valid], f"full block b={b}")


@pytest.mark.slow
def test_full_size_4b_block_prefix():
    """The 4B-shaped block (B2 T32768) on the GPU; the oracle runs the first
    4096 tokens of each batch row (four 1024-token windows) through the
    whole block."""
    w = WL.WORKLOADS["4b_block"]
    inp = Hh.make_inputs(w)
    inp.update(WL.block_norm_gammas(w, 0))
    ffn = WL.ffn_weights(w)
    got = _gpu_block(w, inp, ffn)
    L = 4096
    for b in range(w.B):
        ref = _oracle_block(w, inp, ffn, x=inp["x"][b:b + 1, :L],
                            pad_lens=torch.zeros(1, dtype=torch.int64),
                            segment_pos=inp["segment_pos"][b:b + 1, :L])[0]
        Hh.assert_close(got[b, :L].cpu(), ref, f"4b block prefix b={b}")
