"""Pins of the oracle's KV-cache path.

The cached layer is checked against the scalar brute force of
tests/test_oracle_pins.py (plain loops written from the pages' prose, no
cache): a prompt written into an empty cache, the same prompt decoded one
token at a time, in chunks, a padded prompt followed by decode steps, and a
cache whose stored positions jump (the sliding window must follow the
positions, not the slots).  Planted mistakes at the end show each pin bites.
"""
import pytest
import torch

from oracle import gemma3_oracle as O
from tests.test_oracle_pins import brute_attention

F64 = torch.float64
H, HKV, DH, D = 4, 2, 8, 16
BASE, SCALE, ALPHA = 100.0, 2.0, 0.6


def _rand(shape, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g, dtype=F64) * std


def _weights(seed):
    return dict(Wq=_rand((H * DH, D), seed + 1, D ** -0.5),
                Wkv=_rand((2, HKV * DH, D), seed + 2, D ** -0.5),
                Wo=_rand((D, H * DH), seed + 3, D ** -0.5),
                gamma_q=_rand((DH,), seed + 4, 0.3), gamma_k=_rand((DH,), seed + 5, 0.3))


def _cached(x, pos, pad, cache, end, w, local, W):
    return O.attention_layer_cached(
        x, pos, pad, cache, end, **w, H=H, H_kv=HKV, d_h=DH,
        attn_type=O.LOCAL_SLIDING if local else O.GLOBAL, window=W,
        rope_base=BASE, rope_scale=SCALE, query_scale=ALPHA)


def _brute(x_rows, pos, w, local, W):
    """Brute force over one token sequence (no padding): row t sees rows s <= t."""
    T = len(x_rows)
    return torch.tensor(brute_attention(
        x_rows, pos, T, w["Wq"].tolist(), w["Wkv"][0].tolist(), w["Wkv"][1].tolist(),
        w["Wo"].tolist(), w["gamma_q"].tolist(), w["gamma_k"].tolist(), H, HKV, DH, local, W,
        BASE, SCALE, ALPHA), dtype=F64)


TOL = dict(rtol=1e-11, atol=1e-12)
MASKS = [(False, 0), (True, 1), (True, 4), (True, 30)]


@pytest.mark.parametrize("local,W", MASKS)
def test_prompt_into_empty_cache_equals_bruteforce(local, W):
    B, T, S = 2, 12, 16
    x = _rand((B, T, D), 20)
    pos = torch.arange(T).repeat(B, 1)
    pad = torch.tensor([0, 3])
    w = _weights(21)
    out, cache = _cached(x, pos, pad, O.init_cache(B, S, HKV, DH), 0, w, local, W)
    for b in range(B):
        v = T - int(pad[b])
        ref = _brute(x[b, :v].tolist(), list(range(v)), w, local, W)
        assert torch.allclose(out[b, :v], ref, **TOL), (out[b, :v] - ref).abs().max()
        assert torch.equal(out[b, v:], torch.zeros(T - v, D, dtype=F64))
        assert torch.equal(cache["pos"][b, v:], torch.full((S - v,), O.EMPTY_SLOT))


@pytest.mark.parametrize("local,W", MASKS)
def test_decode_one_token_at_a_time_equals_bruteforce(local, W):
    T, S = 11, 13
    x = _rand((1, T, D), 30)
    w = _weights(31)
    ref = _brute(x[0].tolist(), list(range(T)), w, local, W)
    cache = O.init_cache(1, S, HKV, DH)
    for t in range(T):
        out, cache = _cached(x[:, t:t + 1], torch.tensor([[t]]), None, cache, t, w, local, W)
        assert torch.allclose(out[0, 0], ref[t], **TOL), (t, (out[0, 0] - ref[t]).abs().max())


@pytest.mark.parametrize("local,W", MASKS)
def test_chunked_prefill_equals_single_call(local, W):
    B, T, S = 2, 12, 20
    x = _rand((B, T, D), 40)
    pos = torch.arange(T).repeat(B, 1)
    w = _weights(41)
    full, full_cache = _cached(x, pos, None, O.init_cache(B, S, HKV, DH), 0, w, local, W)
    cache, end, outs = O.init_cache(B, S, HKV, DH), 0, []
    for n in (3, 1, 5, 2, 1):
        o, cache = _cached(x[:, end:end + n], pos[:, end:end + n], None, cache, end, w, local, W)
        outs.append(o)
        end += n
    assert torch.allclose(torch.cat(outs, 1), full, **TOL)
    for k in ("k", "v", "pos"):
        assert torch.allclose(cache[k].to(F64), full_cache[k].to(F64), **TOL)


@pytest.mark.parametrize("local,W", MASKS)
def test_padded_prompt_then_decode_equals_bruteforce(local, W):
    # Row b holds valid_b prompt tokens and T0 - valid_b empty slots; decode
    # tokens then go to slots T0, T0+1, ... at positions valid_b, valid_b+1, ...
    B, T0, n_dec, S = 2, 8, 4, 14
    pad = torch.tensor([0, 3])
    xp = _rand((B, T0, D), 50)
    xd = _rand((B, n_dec, D), 51)
    w = _weights(52)
    pos = torch.arange(T0).repeat(B, 1)
    _, cache = _cached(xp, pos, pad, O.init_cache(B, S, HKV, DH), 0, w, local, W)
    for i in range(n_dec):
        valid = T0 - pad
        dpos = (valid + i).reshape(B, 1)
        out, cache = _cached(xd[:, i:i + 1], dpos, None, cache, T0 + i, w, local, W)
        for b in range(B):
            v = int(valid[b])
            seq = torch.cat([xp[b, :v], xd[b, :i + 1]]).tolist()
            ref = _brute(seq, list(range(v + i + 1)), w, local, W)[-1]
            assert torch.allclose(out[b, 0], ref, **TOL), (b, i)


@pytest.mark.parametrize("W", [1, 3, 4, 6, 8, 50])
def test_window_follows_stored_positions_across_a_gap(W):
    # Slots 0..5 hold positions 0..5, slots 6..11 positions 40..45; the query
    # at slot 12 has position 46.  It must see exactly the stored tokens with
    # position in (46 - W, 46], as a cache-free causal pass over those tokens.
    pos_all = list(range(6)) + list(range(40, 47))
    x = _rand((1, 13, D), 60)
    w = _weights(61)
    cache = O.init_cache(1, 16, HKV, DH)
    _, cache = _cached(x[:, :12], torch.tensor([pos_all[:12]]), None, cache, 0, w, False, 0)
    out, _ = _cached(x[:, 12:], torch.tensor([[46]]), None, cache, 12, w, True, W)
    keep = [i for i, p in enumerate(pos_all) if p > 46 - W]
    ref = _brute(x[0, keep].tolist(), [pos_all[i] for i in keep], w, False, 0)[-1]
    assert torch.allclose(out[0, 0], ref, **TOL)


def test_uniform_position_shift_leaves_outputs_unchanged():
    T, S = 9, 12
    x = _rand((1, T, D), 70)
    w = _weights(71)
    res = []
    for shift in (0, 100000):
        cache, outs = O.init_cache(1, S, HKV, DH), []
        for t in range(T):
            o, cache = _cached(x[:, t:t + 1], torch.tensor([[t + shift]]), None, cache, t, w,
                               True, 4)
            outs.append(o)
        res.append(torch.cat(outs, 1))
    assert torch.allclose(res[0], res[1], rtol=0, atol=1e-9)


def test_cache_write_touches_only_the_new_slots():
    B, T, S, end = 2, 3, 10, 4
    w = _weights(81)
    prev = {"k": _rand((B, S, HKV, DH), 82), "v": _rand((B, S, HKV, DH), 83),
            "pos": torch.randint(0, 100, (B, S), generator=torch.Generator().manual_seed(84))}
    snapshot = {k: v.clone() for k, v in prev.items()}
    x = _rand((B, T, D), 85)
    pos = torch.tensor([[7, 8, 9], [20, 21, 22]])
    pad = torch.tensor([0, 1])
    _, new = _cached(x, pos, pad, prev, end, w, True, 3)
    for k in prev:
        assert torch.equal(prev[k], snapshot[k])                        # input untouched
        keep = torch.ones(S, dtype=torch.bool)
        keep[end:end + T] = False
        assert torch.equal(new[k][:, keep], prev[k][:, keep])
    assert new["pos"][:, end:end + T].tolist() == [[7, 8, 9], [20, 21, O.EMPTY_SLOT]]
    _, Kref = O.normalised_rotated_qk(x.reshape(-1, D), pos.reshape(-1), w["Wq"], w["Wkv"],
                                      w["gamma_q"], w["gamma_k"], H=H, H_kv=HKV, d_h=DH,
                                      rope_base=BASE, rope_scale=SCALE)
    assert torch.allclose(new["k"][:, end:end + T], Kref.reshape(B, T, HKV, DH), **TOL)
    Vref = (x.reshape(-1, D) @ w["Wkv"][1].T).reshape(B, T, HKV, DH)
    assert torch.allclose(new["v"][:, end:end + T], Vref, **TOL)


def test_cache_overflow_is_rejected():
    w = _weights(91)
    with pytest.raises(ValueError):
        _cached(_rand((1, 3, D), 92), torch.tensor([[0, 1, 2]]), None,
                O.init_cache(1, 4, HKV, DH), 2, w, False, 0)


# ----------------------------------------------------------------------------
# planted mistakes (on the CPU, in the oracle) must fail a pin above
# ----------------------------------------------------------------------------
def _fails(fn, *a):
    try:
        fn(*a)
    except AssertionError:
        return True
    return False


def test_window_on_slots_instead_of_positions_is_caught(monkeypatch):
    def slot_window(q_slots, q_pos, slot_pos, attn_type, window):
        s = torch.arange(slot_pos.shape[0])
        m = (s[None, :] <= q_slots[:, None]) & (slot_pos[None, :] >= 0)
        if attn_type == O.LOCAL_SLIDING:
            m = m & O.create_sliding_mask(q_slots, s, window)
        return m

    monkeypatch.setattr(O, "cache_mask", slot_window)
    assert _fails(test_window_follows_stored_positions_across_a_gap, 8)
    assert _fails(test_padded_prompt_then_decode_equals_bruteforce, True, 4)


def test_empty_slots_left_visible_is_caught(monkeypatch):
    def no_empty_check(q_slots, q_pos, slot_pos, attn_type, window):
        s = torch.arange(slot_pos.shape[0])
        m = s[None, :] <= q_slots[:, None]
        if attn_type == O.LOCAL_SLIDING:
            m = m & O.create_sliding_mask(q_pos, slot_pos, window)
        return m

    monkeypatch.setattr(O, "cache_mask", no_empty_check)
    assert _fails(test_padded_prompt_then_decode_equals_bruteforce, False, 0)


def test_write_one_slot_late_is_caught(monkeypatch):
    real = O.dynamic_update_slice
    monkeypatch.setattr(O, "dynamic_update_slice", lambda buf, upd, start: real(buf, upd, start + 1))
    assert _fails(test_decode_one_token_at_a_time_equals_bruteforce, False, 0)


def test_causal_limit_dropped_is_caught(monkeypatch):
    def no_causal(q_slots, q_pos, slot_pos, attn_type, window):
        m = (slot_pos[None, :] >= 0).expand(q_slots.shape[0], -1)
        if attn_type == O.LOCAL_SLIDING:
            m = m & O.create_sliding_mask(q_pos, slot_pos, window)
        return m

    monkeypatch.setattr(O, "cache_mask", no_causal)
    assert _fails(test_prompt_into_empty_cache_equals_bruteforce, False, 0)
