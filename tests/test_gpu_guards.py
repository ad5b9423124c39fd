"""Guard bytes around every buffer the entry points write.

compute-sanitizer is closed on the GPUs these tests run on, so out-of-range
writes are looked for this way: each output, cache and workspace sits in a
larger allocation whose bytes before and after it hold a pattern, the call
runs, and the pattern must be unchanged.  The workspace may be written only
in the bytes the size query asked for; a cache only in the new tokens'
slots; a strided output only in its rows' first N columns.  Inputs are checked to
be left as they were.  Covered: the linear (few-row and tiled, 128- and 256-row tiles), one layer
(local d_h = 256 and global d_h = 128, padded rows), the whole block, and a
decode step and a prompt chunk over a cache (local and global).
"""
import pytest
import torch

from tests import helpers as Hh
from transformer_attention_gb300 import workloads as WL

pytestmark = pytest.mark.gpu

GUARD = 1 << 16          # bytes of pattern on each side (keeps 256-byte alignment)
PATTERN = 0xA5


@pytest.fixture(scope="module", autouse=True)
def _built():
    from transformer_attention_gb300.build import build
    build()
    import transformer_attention_gb300 as G3
    G3.lib()


class Guarded:
    """`nbytes` of device memory between two GUARD-byte runs of PATTERN."""

    def __init__(self, nbytes, fill=None):
        self.n = nbytes
        self.buf = torch.full((2 * GUARD + nbytes,), PATTERN, dtype=torch.uint8, device="cuda")
        self.inner = self.buf[GUARD:GUARD + nbytes]
        if fill is not None:
            self.inner.copy_(fill.reshape(-1).view(torch.uint8))

    def view(self, dtype, shape):
        return self.inner.view(dtype).view(shape)

    def guards_intact(self):
        g = self.buf.cpu()
        return bool((g[:GUARD] == PATTERN).all()) and bool((g[GUARD + self.n:] == PATTERN).all())


def _inputs_dev(inp):
    dev = Hh.to_dev(inp)
    return dev, {k: v.clone() for k, v in dev.items() if isinstance(v, torch.Tensor)}


def _inputs_unchanged(dev, before):
    return all(torch.equal(dev[k], v) for k, v in before.items())


LAYERS = [
    dict(B=2, T=333, D=256, H=4, H_kv=1, d_h=256, attn_type="local", window=100,
         pad=("pad_uniform", 0, 120)),
    dict(B=2, T=260, D=384, H=4, H_kv=2, d_h=128, attn_type="global", window=0,
         rope_base=1e6, rope_scale=8.0, query_scale=168 ** -0.5, pad=("pad_uniform", 0, 100)),
    # padding that fills whole 128-row tiles (the projections write them as zeros)
    dict(B=3, T=512, D=256, H=4, H_kv=2, d_h=256, attn_type="local", window=100,
         pad=("pad_uniform", 200, 512)),
]


@pytest.mark.parametrize("kw", LAYERS, ids=["local-d256", "global-d128", "pad-tiles-d256"])
@pytest.mark.parametrize("rows", [0, 256])
def test_layer_writes_only_out_and_its_workspace(kw, rows):
    """(rows: the projection GEMM's tile height, chosen per call or forced
    to 256-row tiles for the output projection.)"""
    import transformer_attention_gb300 as G3
    w = WL.small(WL.WORKLOADS["tiny_local"], name="guard", **kw)
    inp = Hh.make_inputs(w)
    dev, before = _inputs_dev(inp)
    need = G3.gemma3_attn_workspace_size(w.B, w.T, w.D, w.H, w.H_kv, w.d_h)
    ws = Guarded(need)
    out = Guarded(w.B * w.T * w.D * 2)
    prev = G3.gemma3_set_gemm_tile_rows(rows)
    try:
        G3.gemma3_attn_forward((w.B, w.T, w.D, w.H, w.H_kv, w.d_h), dev["x"],
                               dev["segment_pos"], dev["pad_lens"], dev["Wq"], dev["Wkv"],
                               dev["Wo"], dev["gamma_q"], dev["gamma_k"], Hh.abi_type(w),
                               w.window, w.rope_base, w.rope_scale, w.query_scale, out.inner,
                               ws.inner, need)
        assert G3.gemma3_attn_check_status() == 0
    finally:
        G3.gemma3_set_gemm_tile_rows(prev)
    assert ws.guards_intact() and out.guards_intact()
    assert _inputs_unchanged(dev, before)
    # and the result is the layer's
    got = out.view(torch.bfloat16, (w.B, w.T, w.D)).cpu()
    ref = Hh.oracle_forward(w, inp)
    for b in range(w.B):
        valid = w.T - int(inp["pad_lens"][b])
        Hh.assert_close(got[b, :valid], ref[b, :valid], f"guarded layer {w.d_h} b={b}")


def test_block_writes_only_y_and_its_workspace():
    import transformer_attention_gb300 as G3
    w = WL.small(WL.WORKLOADS["4b_block"], name="guard_block", B=2, T=300, D=512, H=4, H_kv=2,
                 d_h=256, window=128, d_ff=1024, pad=("pad_uniform", 0, 80))
    inp = Hh.make_inputs(w)
    inp.update(WL.block_norm_gammas(w, 0))
    inp.update(WL.ffn_weights(w))
    dev, before = _inputs_dev(inp)
    dims = (w.B, w.T, w.D, w.H, w.H_kv, w.d_h)
    need = G3.gemma3_block_workspace_size(dims, w.d_ff)
    ws = Guarded(need)
    y = Guarded(w.B * w.T * w.D * 4)
    G3.gemma3_block_forward(dims, w.d_ff, dev["x"], G3.GEMMA3_BF16, y.inner, dev["segment_pos"],
                            dev["pad_lens"], dev["Wq"], dev["Wkv"], dev["Wo"], dev["gamma_q"],
                            dev["gamma_k"], dev["gamma_pre"], dev["gamma_post"],
                            dev["gamma_pre_ffn"], dev["gamma_post_ffn"], dev["W_gating"],
                            dev["W_down"], Hh.abi_type(w), w.window, w.rope_base, w.rope_scale,
                            w.query_scale, ws.inner, need)
    assert G3.gemma3_attn_check_status() == 0
    assert ws.guards_intact() and y.guards_intact()
    assert _inputs_unchanged(dev, before)
    assert bool(torch.isfinite(y.view(torch.float32, (w.B, w.T, w.D))).all())


@pytest.mark.parametrize("M", [2, 333, 1400])
@pytest.mark.parametrize("out_dtype", ["bf16", "f32"])
@pytest.mark.parametrize("rows", [0, 256])
def test_linear_writes_only_its_columns(M, out_dtype, rows):
    """C = A W^T into rows of stride ldc > N: the gap after each row's N
    columns and the bytes around C keep their pattern (few-row and tiled, on
    the chosen tile height and on 256-row tiles)."""
    import transformer_attention_gb300 as G3
    N, K, ldc = 1096, 512, 1104
    g = torch.Generator().manual_seed(11)
    A = torch.randn((M, K), generator=g).to(torch.bfloat16).cuda()
    W = (torch.randn((N, K), generator=g) / K ** 0.5).to(torch.bfloat16).cuda()
    dt, code = ((torch.bfloat16, G3.GEMMA3_BF16) if out_dtype == "bf16"
                else (torch.float32, G3.GEMMA3_F32))
    esz = torch.tensor([], dtype=dt).element_size()
    C = Guarded(M * ldc * esz)
    prev = G3.gemma3_set_gemm_tile_rows(rows)
    try:
        G3.gemma3_linear(A, K, W, K, C.inner, ldc, M, N, K, G3.GEMMA3_BF16, code)
        assert G3.gemma3_attn_check_status() == 0
    finally:
        G3.gemma3_set_gemm_tile_rows(prev)
    assert C.guards_intact()
    rows = C.inner.view(torch.uint8).view(M, ldc * esz).cpu()
    assert bool((rows[:, N * esz:] == PATTERN).all())
    got = C.view(dt, (M, ldc))[:, :N].float().cpu()
    ref = A.double().cpu() @ W.double().cpu().T
    assert (got.double() - ref).abs().max().item() < 2e-2 * (1 + ref.abs().max().item())


DECODES = {
    # one decode step on a local layer whose window is shorter than the cache
    "decode-local-d256": dict(B=2, T=1, cache_len=900, D=256, H=4, H_kv=2, d_h=256, window=300),
    # one decode step on a global d_h = 128 layer
    "decode-global-d128": dict(B=2, T=1, cache_len=900, D=256, H=4, H_kv=2, d_h=128,
                               attn_type="global", window=0, rope_base=1e6, rope_scale=8.0),
    # a 256-token prompt written at slot 0 of an empty cache (the flash branch)
    "prompt-global-d128": dict(B=2, T=256, cache_len=600, D=256, H=4, H_kv=2, d_h=128,
                               attn_type="global", window=0, rope_base=1e6, rope_scale=8.0),
}


@pytest.mark.parametrize("name", list(DECODES))
def test_cached_layer_writes_only_its_slots(name):
    import transformer_attention_gb300 as G3
    kw = DECODES[name]
    w = WL.small(WL.WORKLOADS["4b_local_decode"], name="guard_cached", **kw)
    S = w.cache_len
    if name.startswith("prompt"):
        end = 0
        K0 = torch.zeros((w.B, S, w.H_kv, w.d_h), dtype=torch.float16)
        V0, p0 = torch.zeros_like(K0), torch.full((w.B, S), -1, dtype=torch.int32)
        pos = torch.arange(w.T, dtype=torch.int32).repeat(w.B, 1)
    else:
        end = S - w.T
        K0, V0, p0 = WL.kv_cache(w)
        pos = WL.segment_pos(w)
    inp = Hh.make_inputs(w)
    inp["segment_pos"] = pos
    dev, before = _inputs_dev(inp)
    Kc, Vc = Guarded(K0.numel() * 2, K0), Guarded(V0.numel() * 2, V0)
    pc = Guarded(p0.numel() * 4, p0)
    dims = (w.B, w.T, w.D, w.H, w.H_kv, w.d_h)
    need = G3.gemma3_attn_cached_workspace_size(dims, S)
    ws = Guarded(need)
    out = Guarded(w.B * w.T * w.D * 2)
    G3.gemma3_attn_forward_cached(dims, S, end, dev["x"], dev["segment_pos"], None, dev["Wq"],
                                  dev["Wkv"], dev["Wo"], dev["gamma_q"], dev["gamma_k"],
                                  Hh.abi_type(w), w.window, w.rope_base, w.rope_scale,
                                  w.query_scale, Kc.inner, Vc.inner, pc.inner, out.inner,
                                  ws.inner, need)
    assert G3.gemma3_attn_check_status() == 0
    for g in (Kc, Vc, pc, ws, out):
        assert g.guards_intact()
    assert _inputs_unchanged(dev, before)
    # only the new tokens' slots [end, end + T) of the cache changed
    K = Kc.view(torch.float16, K0.shape).cpu()
    V = Vc.view(torch.float16, V0.shape).cpu()
    p = pc.view(torch.int32, p0.shape).cpu()
    new = slice(end, end + w.T)
    for got, ref in ((K, K0), (V, V0), (p, p0)):
        assert torch.equal(got[:, :end], ref[:, :end])
        assert torch.equal(got[:, end + w.T:], ref[:, end + w.T:])
    assert torch.equal(p[:, new], pos)
    assert bool(torch.isfinite(out.view(torch.bfloat16, (w.B, w.T, w.D)).float()).all())
