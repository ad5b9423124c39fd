"""Shared helpers of the GPU parity tests: inputs, tolerances, error metrics."""
from __future__ import annotations

import torch

from oracle import gemma3_oracle as O
from transformer_attention_gb300 import workloads as WL

# Tolerances stated for this path: block output relative Frobenius error and
# max abs error; normalised+rotated Q/K max abs error.
REL_FROB = 5e-3
MAX_ABS = 2e-2
QK_MAX_ABS = 1e-2


def rel_frob(got: torch.Tensor, ref: torch.Tensor) -> float:
    got, ref = got.to(torch.float64), ref.to(torch.float64)
    return float((got - ref).norm() / ref.norm().clamp_min(1e-300))


def max_abs(got: torch.Tensor, ref: torch.Tensor) -> float:
    return float((got.to(torch.float64) - ref.to(torch.float64)).abs().max())


# Every assert_close records (what, GPU rel_frob, GPU max_abs, floor rel_frob,
# floor max_abs); the floor is the error of the oracle itself rounded to
# bf16 (round to nearest even), the least a bf16 output can show.  The
# conftest prints the table at the end of the run.
RESULTS: list = []


def bf16_floor(ref: torch.Tensor):
    ref64 = ref.to(torch.float64)
    r = ref64.to(torch.bfloat16)
    return rel_frob(r, ref64), max_abs(r, ref64)


def assert_close(got, ref, what=""):
    rf, ma = rel_frob(got, ref), max_abs(got, ref)
    frf, fma = bf16_floor(ref)
    RESULTS.append((what, rf, ma, frf, fma))
    assert rf <= REL_FROB and ma <= MAX_ABS, (
        f"{what}: rel_frob={rf:.3e} max_abs={ma:.3e} (bf16 floor {frf:.3e} / {fma:.3e})")
    return rf, ma


def oracle_type(w: WL.Workload):
    return O.LOCAL_SLIDING if w.attn_type == "local" else O.GLOBAL


def abi_type(w: WL.Workload):
    import transformer_attention_gb300 as G3
    return G3.GEMMA3_LOCAL_SLIDING if w.attn_type == "local" else G3.GEMMA3_GLOBAL


def make_inputs(w: WL.Workload, layer: int = 0, x=None):
    """CPU inputs of one layer of workload ``w`` (bf16 / int32)."""
    inp = dict(WL.weights(w, layer))
    inp["x"] = WL.x_full(w) if x is None else x
    inp["segment_pos"] = WL.segment_pos(w)
    inp["pad_lens"] = WL.pad_lens(w)
    return inp


def to_dev(inp: dict, device="cuda") -> dict:
    return {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def gpu_forward(w: WL.Workload, dev: dict):
    import transformer_attention_gb300 as G3
    out = G3.attention_forward(
        dev["x"], dev["segment_pos"], dev["pad_lens"], dev["Wq"], dev["Wkv"], dev["Wo"],
        dev["gamma_q"], dev["gamma_k"], H=w.H, H_kv=w.H_kv, attn_type=abi_type(w),
        window=w.window, rope_base=w.rope_base, rope_scale=w.rope_scale,
        query_scale=w.query_scale)
    assert G3.gemma3_attn_check_status() == 0
    return out


def oracle_forward(w: WL.Workload, inp: dict, rows=None):
    return O.attention_layer(
        inp["x"], inp["segment_pos"], inp["pad_lens"], inp["Wq"], inp["Wkv"], inp["Wo"],
        inp["gamma_q"], inp["gamma_k"], H=w.H, H_kv=w.H_kv, d_h=w.d_h,
        attn_type=oracle_type(w), window=w.window, rope_base=w.rope_base,
        rope_scale=w.rope_scale, query_scale=w.query_scale, rows=rows)


def sample_rows(w: WL.Workload, valid: int, n_random: int, seed: int, limit: int | None = None):
    """Query rows to check: boundary rows (first, window edges, tile edges,
    the middle, the last two valid, first pad) and seeded random rows, all
    < limit (if given)."""
    hi = valid if limit is None else min(valid, limit)
    rows = {0, 1, 63, 64, 127, 128, 129, hi // 2 - 1, hi // 2, hi - 2, hi - 1}
    if w.window:
        rows |= {w.window - 1, w.window, w.window + 1, w.window + 127}
    if valid < w.T and (limit is None or valid < limit):
        rows |= {valid, w.T - 1}
    g = torch.Generator().manual_seed(seed)
    rows |= set(torch.randint(0, hi, (n_random,), generator=g).tolist())
    lim = w.T if limit is None else min(w.T, limit)
    return sorted(r for r in rows if 0 <= r < lim)
