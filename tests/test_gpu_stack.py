"""GPU parity of the routed block-attention stack against the fp64 oracle.

Each layer l is y = x + RMSNorm_post(Attn(RMSNorm_pre(x))) ("Full Gemma 3
Block", How it works) with the attention type P[l mod 6] and the RoPE base,
scale and window that type selects ("Global vs Local Layer Routing", How it
works).  The GPU side takes its per-layer parameters from the C-ABI routing
helper, the oracle from its own routing.
"""
import pytest
import torch

from oracle import gemma3_oracle as O
from tests import helpers as Hh
from transformer_attention_gb300 import workloads as WL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from transformer_attention_gb300.build import build
    build()


def _gpu_stack(w, x_cpu, pads):
    import transformer_attention_gb300 as G3
    x = x_cpu.cuda()
    pos = WL.segment_pos(w).cuda()
    pad = pads.cuda()
    y = torch.empty((w.B, w.T, w.D), dtype=torch.float32, device="cuda")
    src = x
    for l in range(w.num_layers):
        p = {k: v.cuda() for k, v in dict(WL.weights(w, l), **WL.block_norm_gammas(w, l)).items()}
        t, win, base, scale = G3.gemma3_layer_config(l, w.num_layers, w.model_size)
        G3.block_attention_forward(src, pos, pad, p["Wq"], p["Wkv"], p["Wo"], p["gamma_q"],
                                   p["gamma_k"], p["gamma_pre"], p["gamma_post"], H=w.H,
                                   H_kv=w.H_kv, attn_type=t, window=win, rope_base=base,
                                   rope_scale=scale, query_scale=w.query_scale, y=y)
        src = y
    assert G3.gemma3_attn_check_status() == 0
    return y


def _oracle_stack(w, x, pads, T):
    layers = [dict(WL.weights(w, l), **WL.block_norm_gammas(w, l)) for l in range(w.num_layers)]
    return O.attention_stack(x, layers, model_size=w.model_size, H=w.H, H_kv=w.H_kv, d_h=w.d_h,
                             segment_pos=torch.arange(T).repeat(x.shape[0], 1), pad_lens=pads)


def test_small_stack_full():
    w = WL.small(WL.WORKLOADS["12b_stack"], name="stack_small", B=2, T=1300, D=512, H=4,
                 H_kv=2, pad=("valid_uniform", 1100, 1300))
    x = WL.x_full(w)
    pads = WL.pad_lens(w)
    got = _gpu_stack(w, x, pads).cpu()
    ref = _oracle_stack(w, x, pads, w.T)
    for b in range(w.B):
        valid = w.T - int(pads[b])
        Hh.assert_close(got[b, :valid], ref[b, :valid], f"stack b={b}")
        # pad rows: attention output 0 and RMSNorm(0) = 0, so y = x exactly
        assert torch.equal(got[b, valid:], x[b, valid:].float())


@pytest.mark.slow
def test_full_size_stack_shortest_row_in_full():
    """Full 12B-shaped stack (B8 T16384, 6 layers) on the GPU; the oracle runs
    the batch row with the fewest valid tokens through all six layers over its
    whole valid length (the global layer l = 5 over every valid key), and the
    row's pad tail must pass the residual through unchanged."""
    w = WL.WORKLOADS["12b_stack"]
    x = WL.x_full(w)
    pads = WL.pad_lens(w)
    got = _gpu_stack(w, x, pads)
    valids = w.T - pads
    b = int(torch.argmin(valids))
    valid = int(valids[b])
    # pad keys are blocked for every valid query, so the valid rows of the
    # padded row equal the unpadded stack over its first `valid` tokens
    ref = _oracle_stack(w, x[b:b + 1, :valid], torch.zeros(1, dtype=torch.int64), valid)[0]
    Hh.assert_close(got[b, :valid].cpu(), ref, f"12b stack row b={b} (valid {valid}) in full")
    assert torch.equal(got[b, valid:].cpu(), x[b, valid:].float())


@pytest.mark.slow
def test_full_size_stack_prefix():
    """Full 12B-shaped stack (B8 T16384, 6 layers) on the GPU; the oracle runs
    the first L = 6144 tokens of the longest batch row through all six layers
    (the stack is causal, so those rows depend on nothing later): six local
    windows over the whole prefix and the global layer over 6144 keys."""
    w = WL.WORKLOADS["12b_stack"]
    x = WL.x_full(w)
    pads = WL.pad_lens(w)
    got = _gpu_stack(w, x, pads)
    L = 6144
    valids = w.T - pads
    b = int(torch.argmax(valids))
    ref = _oracle_stack(w, x[b:b + 1, :L], torch.zeros(1, dtype=torch.int64), L)[0]
    Hh.assert_close(got[b, :L].cpu(), ref, f"12b stack prefix b={b} (first {L} tokens)")
    valid = int(valids[b])
    if valid < w.T:
        assert torch.equal(got[b, valid:].cpu(), x[b, valid:].float())
