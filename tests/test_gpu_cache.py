"""GPU parity of the KV-cache path against the fp64 oracle.

- the cache write: bit-exact slots and stored positions, other slots untouched;
- attention over a cache (the stage entry): decode (T = 1) and multi-token
  queries, d_h 128/256, G 1/2/4, global and local windows, caches with empty
  slots, position gaps and stale slots past the causal limit, ragged tails,
  one and many slot splits, against the oracle's cache mask + attention;
- whole layers through gemma3_attn_forward_cached: a padded prompt, decode
  steps and a chunk, call by call against the oracle's cached layer (which
  carries its own fp64 cache), including the flash-kernel prompt branch;
- the two decode workloads at full size (4B local, cache 32768; 27B global,
  cache 131072), in the benchmark's launch configuration, all output rows.
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


def _f16(shape, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g, dtype=torch.float32) * std).to(torch.float16)


# ---------------------------------------------------------------- cache write
def test_kv_cache_write_bit_exact():
    import transformer_attention_gb300 as G3
    B, T, S, end, H_kv, d_h = 3, 5, 40, 17, 2, 128
    KVD = H_kv * d_h
    ld = 2 * KVD + 64
    rows = _f16((B * T, ld), 1).cuda()
    seg = torch.randint(0, 1000, (B, T), generator=torch.Generator().manual_seed(2),
                        dtype=torch.int32).cuda()
    pad = torch.tensor([0, 2, 5], dtype=torch.int32).cuda()
    Kc0 = _f16((B, S, H_kv, d_h), 3)
    Vc0 = _f16((B, S, H_kv, d_h), 4)
    pc0 = torch.randint(-1, 50, (B, S), generator=torch.Generator().manual_seed(5),
                        dtype=torch.int32)
    Kc, Vc, pc = Kc0.cuda(), Vc0.cuda(), pc0.cuda()
    G3.gemma3_kv_cache_write(rows, rows[:, KVD:], ld, seg, pad, B, T, S, end, H_kv, d_h, Kc, Vc,
                             pc)
    torch.cuda.synchronize()
    Kc, Vc, pc, rows, seg = Kc.cpu(), Vc.cpu(), pc.cpu(), rows.cpu(), seg.cpu()
    keep = torch.ones(S, dtype=torch.bool)
    keep[end:end + T] = False
    assert torch.equal(Kc[:, keep], Kc0[:, keep]) and torch.equal(Vc[:, keep], Vc0[:, keep])
    assert torch.equal(pc[:, keep], pc0[:, keep])
    r = rows.reshape(B, T, ld)
    assert torch.equal(Kc[:, end:end + T].reshape(B, T, KVD), r[..., :KVD])
    assert torch.equal(Vc[:, end:end + T].reshape(B, T, KVD), r[..., KVD:2 * KVD])
    for b, p in enumerate([0, 2, 5]):
        want = seg[b].clone()
        want[T - p:] = -1
        assert torch.equal(pc[b, end:end + T], want)


# ---------------------------------------------------------------- attention stage
STAGE = [
    # B, T, S, end, H, H_kv, d_h, window, pads, layout
    (2, 1, 1000, 999, 4, 1, 256, 0, None, "plain"),
    (2, 1, 3000, 2500, 8, 4, 256, 64, None, "gaps"),
    (1, 1, 5000, 4999, 4, 2, 128, 0, None, "plain"),
    (2, 3, 700, 600, 2, 2, 128, 100, [0, 1], "gaps"),
    (3, 2, 300, 10, 4, 1, 256, 0, [0, 0, 1], "stale"),
    (2, 5, 100, 50, 4, 4, 256, 7, None, "stale"),
    (1, 1, 1, 0, 4, 2, 128, 0, None, "plain"),
    (2, 20, 200, 100, 4, 2, 256, 33, [0, 3], "gaps"),
    (1, 1, 40000, 39999, 8, 4, 256, 1024, None, "plain"),
]


def _stage_inputs(B, T, S, end, H, H_kv, d_h, pads, layout, seed):
    """Q' (scaled like d_h**-0.5 query rows), a cache, stored and query positions."""
    Q = _f16((B, T, H, d_h), seed, d_h ** -0.5)
    K = _f16((B, S, H_kv, d_h), seed + 1)
    V = _f16((B, S, H_kv, d_h), seed + 2)
    pad = torch.tensor(pads if pads else [0] * B, dtype=torch.int32)
    pos = torch.full((B, S), -1, dtype=torch.int32)
    seg = torch.zeros((B, T), dtype=torch.int32)
    for b in range(B):
        p = torch.arange(end + T, dtype=torch.int32)
        if layout == "gaps":
            # an empty stretch (a padded prompt) and a jump of positions
            e0, e1 = end // 3, end // 3 + max(1, end // 10)
            p[e1:] += 50
            p[e0:e1] = -1
            p[e1:] -= (e1 - e0)
        pos[b, :end + T] = p
        if layout == "stale":
            # slots past the new tokens hold positions from an older sequence
            pos[b, end + T:] = torch.arange(S - end - T, dtype=torch.int32)
        seg[b] = pos[b, end:end + T]
        v = T - int(pad[b])
        pos[b, end + v:end + T] = -1
    return Q, K, V, pos, seg, pad


@pytest.mark.parametrize("case", STAGE, ids=lambda c: "B{}T{}S{}e{}H{}/{}d{}W{}{}".format(
    *c[:8], "-pad" if c[8] else "") + "-" + c[9])
def test_cached_attention_stage(case):
    import transformer_attention_gb300 as G3
    B, T, S, end, H, H_kv, d_h, W, pads, layout = case
    Q, K, V, pos, seg, pad = _stage_inputs(B, T, S, end, H, H_kv, d_h, pads, layout, 10 + S)
    nbytes = G3.gemma3_cached_attention_workspace_size(B, T, S, H, H_kv, d_h)
    ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device="cuda")
    Od = torch.empty((B, T, H, d_h), dtype=torch.float16, device="cuda")
    G3.gemma3_cached_attention(Q.cuda(), K.cuda(), V.cuda(), pos.cuda(), seg.cuda(), pad.cuda(),
                               Od, G3.GEMMA3_F16, B, T, S, end, H, H_kv, d_h, W, ws, ws.numel())
    assert G3.gemma3_attn_check_status() == 0
    got = Od.cpu()
    kind = O.LOCAL_SLIDING if W > 0 else O.GLOBAL
    for b in range(B):
        v = T - int(pad[b])
        mask = O.cache_mask(end + torch.arange(T), seg[b].to(torch.int64),
                            pos[b].to(torch.int64), kind, W)
        ref = O.attend_masked(Q[b].to(F64), K[b].to(F64), V[b].to(F64), mask)
        if v > 0:
            Hh.assert_close(got[b, :v], ref[:v], f"b={b}")
        assert torch.equal(got[b, v:], torch.zeros_like(got[b, v:]))


# ---------------------------------------------------------------- whole layers
def _layer_case(**kw):
    base = WL.WORKLOADS["tiny_local"]
    return WL.small(base, name="cache_small", **kw)


LAYERS = [
    dict(B=2, T=64, D=256, H=4, H_kv=2, d_h=256, attn_type="local", window=24, T0=40,
         pads=[0, 5], S=96),
    dict(B=2, T=64, D=384, H=4, H_kv=1, d_h=128, attn_type="global", window=0, T0=40,
         pads=[3, 0], S=80, rope_base=1e6, rope_scale=8.0, query_scale=168 ** -0.5),
    dict(B=1, T=200, D=256, H=4, H_kv=2, d_h=128, attn_type="global", window=0, T0=160,
         pads=[7], S=200),
    dict(B=2, T=64, D=256, H=2, H_kv=2, d_h=256, attn_type="local", window=8, T0=30,
         pads=[0, 0], S=64),
]


@pytest.mark.parametrize("kw", LAYERS, ids=lambda k: f"d{k['d_h']}-H{k['H']}/{k['H_kv']}-"
                         f"{k['attn_type']}-T0{k['T0']}")
def test_forward_cached_prompt_decode_chunk(kw):
    """A padded prompt at slot 0, then 1-token decode steps, then a 3-token
    chunk and a padded 4-token chunk (these few-row calls write the cache
    from the QK-norm/RoPE kernel); every call's output against the oracle's
    cached layer."""
    import transformer_attention_gb300 as G3
    kw = dict(kw)
    T0, pads, S = kw.pop("T0"), kw.pop("pads"), kw.pop("S")
    w = _layer_case(**kw)
    p = WL.weights(w)
    x_all = WL.x_full(w)
    dev = {k: v.cuda() for k, v in p.items()}
    B, d_h = w.B, w.d_h
    cache = G3.new_kv_cache(B, S, w.H_kv, d_h, "cuda")
    ocache = O.init_cache(B, S, w.H_kv, d_h)
    kind_g = G3.GEMMA3_LOCAL_SLIDING if w.attn_type == "local" else G3.GEMMA3_GLOBAL
    kind_o = Hh.oracle_type(w)
    pad_t = torch.tensor(pads, dtype=torch.int32)
    valid = [T0 - q for q in pads]

    # calls: (x rows, positions [B, n], pad or None, end slot)
    calls = [(x_all[:, :T0], torch.arange(T0, dtype=torch.int32).repeat(B, 1), pad_t, 0)]
    end, used = T0, T0
    for i in range(4):
        calls.append((x_all[:, used:used + 1],
                      torch.tensor([[v + i] for v in valid], dtype=torch.int32), None, end))
        end, used = end + 1, used + 1
    n = 3
    calls.append((x_all[:, used:used + n],
                  torch.stack([torch.arange(v + 4, v + 4 + n, dtype=torch.int32) for v in valid]),
                  None, end))
    end, used = end + n, used + n
    n = 4
    calls.append((x_all[:, used:used + n],
                  torch.stack([torch.arange(v + 7, v + 7 + n, dtype=torch.int32) for v in valid]),
                  torch.tensor([1] + [0] * (B - 1), dtype=torch.int32), end))

    for xc, seg, pad, e in calls:
        got = G3.attention_forward_cached(
            xc.contiguous().cuda(), seg.cuda(), None if pad is None else pad.cuda(), cache, e,
            dev["Wq"], dev["Wkv"], dev["Wo"], dev["gamma_q"], dev["gamma_k"], H=w.H,
            H_kv=w.H_kv, attn_type=kind_g, window=w.window, rope_base=w.rope_base,
            rope_scale=w.rope_scale, query_scale=w.query_scale).cpu()
        assert G3.gemma3_attn_check_status() == 0
        ref, ocache = O.attention_layer_cached(
            xc, seg, pad, ocache, e, p["Wq"], p["Wkv"], p["Wo"], p["gamma_q"], p["gamma_k"],
            H=w.H, H_kv=w.H_kv, d_h=d_h, attn_type=kind_o, window=w.window,
            rope_base=w.rope_base, rope_scale=w.rope_scale, query_scale=w.query_scale)
        Tn = xc.shape[1]
        for b in range(B):
            v = Tn - (int(pad[b]) if pad is not None else 0)
            Hh.assert_close(got[b, :v], ref[b, :v], f"end={e} b={b}")
            assert torch.equal(got[b, v:], torch.zeros_like(got[b, v:]))
    assert torch.equal(cache[2].cpu().to(torch.int64), ocache["pos"])


# ---------------------------------------------------------------- one decode step
# Decode steps (one new token per row) at the edges of the cache path: more
# rows than the query-row blocks hold, pad rows, an empty cache, a long cache
# split over many CTAs.
STEP = [
    # most rows, a pad row, four query heads per kv head, window inside the cache
    dict(B=4, D=256, H=4, H_kv=1, d_h=256, attn_type="local", window=50, S=300, end=250,
         pads=[0, 1, 0, 0]),
    # the first token of an empty cache, one query head per kv head
    dict(B=3, D=384, H=4, H_kv=4, d_h=128, attn_type="global", window=0, S=130, end=0,
         pads=None, rope_base=1e6, rope_scale=8.0),
    # five rows, one of them padding
    dict(B=5, D=256, H=4, H_kv=2, d_h=256, attn_type="local", window=64, S=200, end=150,
         pads=[0, 0, 1, 0, 0]),
    # a long global cache over many splits, the last slot
    dict(B=1, D=512, H=4, H_kv=2, d_h=128, attn_type="global", window=0, S=3000, end=2999,
         pads=None, query_scale=168 ** -0.5),
]


@pytest.mark.parametrize("kw", STEP, ids=lambda k: f"B{k['B']}-d{k['d_h']}-H{k['H']}/{k['H_kv']}-"
                         f"{k['attn_type']}-end{k['end']}")
def test_decode_step_against_oracle(kw):
    """One decode step over a cache holding a prompt in slots [0, end): the
    output rows, the new slot's K', V and position, and that no other slot
    changed, against the oracle's cached layer."""
    import transformer_attention_gb300 as G3
    kw = dict(kw)
    S, end, pads = kw.pop("S"), kw.pop("end"), kw.pop("pads")
    w = _layer_case(T=1, **kw)
    B, d_h = w.B, w.d_h
    p = WL.weights(w)
    dev = {k: v.cuda() for k, v in p.items()}
    x = WL.x_full(w)
    K0 = _f16((B, S, w.H_kv, d_h), 71 + S)
    V0 = _f16((B, S, w.H_kv, d_h), 72 + S)
    pos0 = torch.full((B, S), -1, dtype=torch.int32)
    pos0[:, :end] = torch.arange(end, dtype=torch.int32)
    seg = torch.full((B, 1), end, dtype=torch.int32)
    pad = None if pads is None else torch.tensor(pads, dtype=torch.int32)
    cache = (K0.cuda(), V0.cuda(), pos0.cuda())
    kind_g = G3.GEMMA3_LOCAL_SLIDING if w.attn_type == "local" else G3.GEMMA3_GLOBAL
    got = G3.attention_forward_cached(
        x.cuda(), seg.cuda(), None if pad is None else pad.cuda(), cache, end, dev["Wq"],
        dev["Wkv"], dev["Wo"], dev["gamma_q"], dev["gamma_k"], H=w.H, H_kv=w.H_kv,
        attn_type=kind_g, window=w.window, rope_base=w.rope_base, rope_scale=w.rope_scale,
        query_scale=w.query_scale).cpu()
    assert G3.gemma3_attn_check_status() == 0
    ocache = {"k": K0.to(F64), "v": V0.to(F64), "pos": pos0.to(torch.int64)}
    ref, ocache = O.attention_layer_cached(
        x, seg, pad, ocache, end, p["Wq"], p["Wkv"], p["Wo"], p["gamma_q"], p["gamma_k"],
        H=w.H, H_kv=w.H_kv, d_h=d_h, attn_type=Hh.oracle_type(w), window=w.window,
        rope_base=w.rope_base, rope_scale=w.rope_scale, query_scale=w.query_scale)
    Kc, Vc, pc = (t.cpu() for t in cache)
    assert torch.equal(pc.to(torch.int64), ocache["pos"])
    others = torch.ones(S, dtype=torch.bool)
    others[end] = False
    assert torch.equal(Kc[:, others], K0[:, others]) and torch.equal(Vc[:, others], V0[:, others])
    for b in range(B):
        if pad is not None and int(pad[b]) > 0:
            assert torch.equal(got[b], torch.zeros_like(got[b]))
            continue
        Hh.assert_close(got[b], ref[b], f"decode step b={b}")
        # the new slot: K' normalised and rotated, V as projected (fp16 storage)
        assert (Kc[b, end].to(F64) - ocache["k"][b, end]).abs().max() <= Hh.QK_MAX_ABS
        assert (Vc[b, end].to(F64) - ocache["v"][b, end]).abs().max() <= Hh.QK_MAX_ABS


# ---------------------------------------------------------------- full size
@pytest.mark.parametrize("name", ["4b_local_decode", "27b_global_decode"])
def test_decode_workload_full_size(name):
    import transformer_attention_gb300 as G3
    w = WL.WORKLOADS[name]
    S, end = w.cache_len, w.cache_len - w.T
    K, V, pos = WL.kv_cache(w)
    p = WL.weights(w)
    x = WL.x_full(w)
    seg = WL.segment_pos(w)
    dev = {k: v.cuda() for k, v in p.items()}
    cache = (K.cuda(), V.cuda(), pos.cuda())
    kind = G3.GEMMA3_LOCAL_SLIDING if w.attn_type == "local" else G3.GEMMA3_GLOBAL
    got = G3.attention_forward_cached(
        x.cuda(), seg.cuda(), None, cache, end, dev["Wq"], dev["Wkv"], dev["Wo"],
        dev["gamma_q"], dev["gamma_k"], H=w.H, H_kv=w.H_kv, attn_type=kind, window=w.window,
        rope_base=w.rope_base, rope_scale=w.rope_scale, query_scale=w.query_scale).cpu()
    assert G3.gemma3_attn_check_status() == 0
    new_pos = cache[2].cpu()
    ocache = {"k": K.to(F64), "v": V.to(F64), "pos": pos.to(torch.int64)}
    del K, V
    ref, ocache = O.attention_layer_cached(
        x, seg, None, ocache, end, p["Wq"], p["Wkv"], p["Wo"], p["gamma_q"], p["gamma_k"],
        H=w.H, H_kv=w.H_kv, d_h=w.d_h, attn_type=Hh.oracle_type(w), window=w.window,
        rope_base=w.rope_base, rope_scale=w.rope_scale, query_scale=w.query_scale)
    Hh.assert_close(got, ref, name)
    assert torch.equal(new_pos.to(torch.int64), ocache["pos"])
