"""GPU parity of the model wrapper (gemma3_model_forward) against the fp64
oracle's model_forward: embedding times sqrt(D), routed full blocks, final
RMSNorm, read-out through the embedding table.

- a small model of 7 blocks (5 local, 1 global, 1 local) on 1B-style heads
  with a sequence longer than the local window and padded rows, all logits;
- the embedding stage alone, and its bounds check (a token id outside the
  table gives a zero row and GEMMA3_ERR_BAD_INPUT, raised by the kernel's own
  check, never an out-of-bounds read);
- the 1B-shaped model workload at full size in the benchmark's launch
  configuration, checked on a causal prefix of batch row 0 (rows before n do
  not depend on later tokens, so the oracle runs only those n tokens).
"""
import math

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
    import transformer_attention_gb300 as G3
    G3.lib()


def _layer_weights(w, l):
    p = dict(WL.weights(w, l), **WL.block_norm_gammas(w, l), **WL.ffn_weights(w, l))
    return p


def _gpu_layers(w):
    out = []
    for l in range(w.num_layers):
        p = _layer_weights(w, l)
        out.append({"Wq": p["Wq"].cuda(), "Wkv": p["Wkv"].cuda(), "Wo": p["Wo"].cuda(),
                    "gamma_q": p["gamma_q"].cuda(), "gamma_k": p["gamma_k"].cuda(),
                    "gamma_pre_attn": p["gamma_pre"].cuda(),
                    "gamma_post_attn": p["gamma_post"].cuda(),
                    "gamma_pre_ffn": p["gamma_pre_ffn"].cuda(),
                    "gamma_post_ffn": p["gamma_post_ffn"].cuda(),
                    "W_gating": p["W_gating"].cuda(), "W_down": p["W_down"].cuda()})
    return out


def _oracle_layers(w):
    out = []
    for l in range(w.num_layers):
        p = _layer_weights(w, l)
        p["W_down"] = p["W_down"].transpose(0, 1)   # the page's (D_ff, D) linear
        out.append(p)
    return out


def _gpu_model(w, tokens, pos, pad):
    import transformer_attention_gb300 as G3
    t = WL.model_tables(w)
    logits = G3.model_forward(tokens.cuda(), pos.cuda(), None if pad is None else pad.cuda(),
                              t["E"].cuda(), _gpu_layers(w), t["gamma_final"].cuda(), H=w.H,
                              H_kv=w.H_kv, D_ff=w.d_ff, model_size=w.model_size)
    assert G3.gemma3_attn_check_status() == 0
    return logits.cpu()


def test_small_model_all_logits():
    w = WL.small(WL.WORKLOADS["1b_model"], name="model_small", B=2, T=700, D=256, d_ff=768,
                 vocab=2048, num_layers=7, pad=("pad_uniform", 0, 60))
    tokens, pos, pad = WL.tokens(w), WL.segment_pos(w), WL.pad_lens(w)
    got = _gpu_model(w, tokens, pos, pad)
    t = WL.model_tables(w)
    ref = O.model_forward(tokens, t["E"], _oracle_layers(w), t["gamma_final"],
                          model_size=w.model_size, H=w.H, H_kv=w.H_kv, d_h=w.d_h,
                          segment_pos=pos, pad_lens=pad)
    for b in range(w.B):
        Hh.assert_close(got[b], ref[b], f"b={b}")


def test_embed_stage_and_bad_token():
    import transformer_attention_gb300 as G3
    V, D, M = 100, 264, 5
    E = torch.randn((V, D), generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    tok = torch.tensor([0, 99, 42, 7, 7], dtype=torch.int32)
    x = torch.empty((M, D), dtype=torch.float32, device="cuda")
    G3.gemma3_embed(tok.cuda(), E.cuda(), V, D, M, math.sqrt(D), x)
    assert G3.gemma3_attn_check_status() == 0
    ref = E.float()[tok.long()] * math.sqrt(D)
    assert torch.allclose(x.cpu(), ref, rtol=1e-6, atol=0)
    bad = torch.tensor([1, V, -1, 3, 4], dtype=torch.int32)
    G3.gemma3_embed(bad.cuda(), E.cuda(), V, D, M, math.sqrt(D), x)
    with pytest.raises(G3.Gemma3Error) as ei:
        G3.gemma3_attn_check_status()
    assert ei.value.status == G3.GEMMA3_ERR_BAD_INPUT
    out = x.cpu()
    assert torch.equal(out[1], torch.zeros(D)) and torch.equal(out[2], torch.zeros(D))
    assert torch.allclose(out[0], E.float()[1] * math.sqrt(D), rtol=1e-6, atol=0)


@pytest.mark.slow
def test_model_workload_full_size_prefix():
    """The 1B-shaped 6-block model (B2 T4096) on the GPU; the oracle runs batch
    row 0 in full (4096 tokens: eight 512-token local windows, the global
    layer over every key, all 32768 logits of every token)."""
    w = WL.WORKLOADS["1b_model"]
    tokens, pos = WL.tokens(w), WL.segment_pos(w)
    got = _gpu_model(w, tokens, pos, None)
    n = w.T
    t = WL.model_tables(w)
    ref = O.model_forward(tokens[:1, :n], t["E"], _oracle_layers(w), t["gamma_final"],
                          model_size=w.model_size, H=w.H, H_kv=w.H_kv, d_h=w.d_h,
                          segment_pos=pos[:1, :n], pad_lens=None)
    Hh.assert_close(got[0, :n], ref[0], "1b_model row 0 in full")
