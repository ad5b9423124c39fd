"""End-to-end GPU parity of gemma3_attn_forward against the fp64 oracle.

- the tiny local workload (B1 T1024 D1152 H4/1 d256 W512) checked in full;
- reduced shapes with ragged tails, T < W, padding and G in {1, 2, 4},
  d_h in {128, 256}, checked in full; padding that fills whole 128-row
  tiles (all-padding rows included);
- the normalised and rotated Q/K of the forward's own stages (max abs 1e-2);
- the three single-layer workloads at full size, in the launch configuration
  the benchmark times, on sampled query rows across the whole sequence that
  the oracle computes one by one (rows past the valid length must be exactly
  zero).
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
    import transformer_attention_gb300 as G3
    G3.lib()


def _check_full(w, inp):
    dev = Hh.to_dev(inp)
    got = Hh.gpu_forward(w, dev).cpu()
    ref = Hh.oracle_forward(w, inp)
    for b in range(w.B):
        valid = w.T - int(inp["pad_lens"][b])
        if valid > 0:
            Hh.assert_close(got[b, :valid], ref[b, :valid], f"{w.name} b={b}")
        assert torch.equal(got[b, valid:], torch.zeros_like(got[b, valid:]))


def test_tiny_local_full():
    w = WL.WORKLOADS["tiny_local"]
    _check_full(w, Hh.make_inputs(w))


SMALL = [
    dict(B=2, T=333, D=256, H=4, H_kv=1, d_h=256, attn_type="local", window=100),
    dict(B=1, T=500, D=512, H=8, H_kv=4, d_h=256, attn_type="global", window=0),
    dict(B=2, T=260, D=384, H=4, H_kv=2, d_h=128, attn_type="global", window=0,
         rope_base=1e6, rope_scale=8.0, query_scale=168 ** -0.5, pad=("pad_uniform", 0, 100)),
    dict(B=1, T=200, D=256, H=2, H_kv=2, d_h=128, attn_type="local", window=1024),
    dict(B=3, T=129, D=1152, H=4, H_kv=1, d_h=256, attn_type="global", window=0,
         pad=("pad_uniform", 0, 129)),
    dict(B=1, T=1100, D=640, H=8, H_kv=2, d_h=128, attn_type="local", window=512),
]


@pytest.mark.parametrize("kw", SMALL, ids=lambda k: f"T{k['T']}-H{k['H']}/{k['H_kv']}-d{k['d_h']}-{k['attn_type']}")
def test_small_shapes_full(kw):
    base = WL.WORKLOADS["tiny_local"]
    w = WL.small(base, name="small", **kw)
    _check_full(w, Hh.make_inputs(w))


# T a multiple of 128 with trailing padding that fills whole 128-row tiles
# (the projections skip those tiles and write their rows as zeros): a full
# row, a row with its last two tiles padding, an all-padding row; d_h 128
# with a row of one valid token.
PAD_TILES = [
    (dict(B=3, T=512, D=256, H=4, H_kv=2, d_h=256, attn_type="local", window=100),
     [0, 300, 512]),
    (dict(B=2, T=384, D=384, H=4, H_kv=2, d_h=128, attn_type="global", window=0,
          rope_base=1e6, rope_scale=8.0, query_scale=168 ** -0.5), [130, 383]),
]


@pytest.mark.parametrize("kw,pads", PAD_TILES, ids=["d256-local", "d128-global"])
def test_pad_only_tiles(kw, pads):
    base = WL.WORKLOADS["tiny_local"]
    w = WL.small(base, name="pad_tiles", **kw)
    inp = Hh.make_inputs(w)
    inp["pad_lens"] = torch.tensor(pads, dtype=torch.int32)
    _check_full(w, inp)


def test_normalised_rotated_qk_of_the_forward_stages():
    """Q/K after the projection GEMM and the prologue, before the query scale,
    against the oracle's normalised and rotated Q/K (max abs <= 1e-2)."""
    import transformer_attention_gb300 as G3
    for name in ("tiny_local", "27b_global"):
        w = WL.WORKLOADS[name]
        T = 4096
        w = WL.small(w, T=T)
        rows_t = torch.tensor([0, 1, 2047, 4095])
        x = WL.x_full(w)
        inp = Hh.make_inputs(w, x=x)
        if name == "27b_global":
            inp["segment_pos"] = inp["segment_pos"] + 131072 - T   # far positions
        dev = Hh.to_dev(inp)
        M, HD, KVD = w.B * T, w.H * w.d_h, w.H_kv * w.d_h
        xq = dev["x"].reshape(M, w.D)
        Q = torch.empty((M, HD), dtype=torch.float16, device="cuda")
        KV = torch.empty((M, 2 * KVD), dtype=torch.float16, device="cuda")
        G3.gemma3_linear(xq, w.D, dev["Wq"], w.D, Q, HD, M, HD, w.D, G3.GEMMA3_BF16,
                         G3.GEMMA3_F16)
        G3.gemma3_linear(xq, w.D, dev["Wkv"], w.D, KV, 2 * KVD, M, 2 * KVD, w.D, G3.GEMMA3_BF16,
                         G3.GEMMA3_F16)
        G3.gemma3_qk_norm_rope(Q, HD, KV, 2 * KVD, dev["gamma_q"], dev["gamma_k"],
                               dev["segment_pos"], M, w.H, w.H_kv, w.d_h, w.rope_base,
                               w.rope_scale, w.query_scale)
        assert G3.gemma3_attn_check_status() == 0
        q_ref, k_ref = O.normalised_rotated_qk(
            x[0, rows_t], inp["segment_pos"][0, rows_t], inp["Wq"], inp["Wkv"], inp["gamma_q"],
            inp["gamma_k"], H=w.H, H_kv=w.H_kv, d_h=w.d_h, rope_base=w.rope_base,
            rope_scale=w.rope_scale)
        q_got = Q.cpu()[rows_t].reshape(-1, w.H, w.d_h).to(F64) / w.query_scale
        k_got = KV.cpu()[rows_t, :KVD].reshape(-1, w.H_kv, w.d_h).to(F64)
        assert Hh.max_abs(q_got, q_ref) <= Hh.QK_MAX_ABS, name
        assert Hh.max_abs(k_got, k_ref) <= Hh.QK_MAX_ABS, name


@pytest.mark.parametrize("name,limit,n_random", [
    ("1b_global", None, 24),
    ("4b_local", None, 24),
    pytest.param("27b_global", None, 12, marks=pytest.mark.slow),
])
def test_full_size_sampled_rows(name, limit, n_random):
    """Full-size workload on the GPU; sampled rows against the oracle, spread
    over the whole sequence (for the 131072-token global layer the oracle
    projects every key once: rows up to t = 131071 see the full causal
    prefix, so the long online-softmax reduction over ~1024 key tiles and the
    longest work items are checked)."""
    w = WL.WORKLOADS[name]
    inp = Hh.make_inputs(w)
    dev = Hh.to_dev(inp)
    got = Hh.gpu_forward(w, dev)
    del dev
    rows = []
    for b in range(w.B):
        valid = w.T - int(inp["pad_lens"][b])
        rows.append(Hh.sample_rows(w, valid, n_random, seed=100 + b, limit=limit))
    ref = Hh.oracle_forward(w, inp, rows=rows)
    for b in range(w.B):
        valid = w.T - int(inp["pad_lens"][b])
        r = torch.tensor(rows[b])
        g = got[b, r].cpu()
        keep = r < valid
        Hh.assert_close(g[keep], ref[b][keep], f"{name} b={b}")
        assert torch.equal(g[~keep], torch.zeros_like(g[~keep]))
        if valid < w.T:
            tail = got[b, valid:]
            assert bool((tail == 0).all()), "pad rows must be zero"
