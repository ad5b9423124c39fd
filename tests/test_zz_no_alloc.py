"""The no-allocation forward entry point, called through the C ABI.

gemma3_attn_forward_noalloc serves callers that cannot give the library a
workspace (code that may not call cudaMalloc, or whose device memory belongs
to another framework's pool): it keeps the layer's intermediate rows in a
fixed scratch array inside the library instead.  Its output must match the
fp64 oracle within the layer tolerances and the workspace entry point's
output, on two calls in a row (the second call finds the first call's
leftovers in the shared scratch), and problems larger than the scratch must
be refused before anything runs.

This file is collected last so that a run stopping at its first failure has
already run every other test.
"""
import ctypes

import pytest
import torch

from tests import helpers as Hh
from transformer_attention_gb300 import workloads as WL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from transformer_attention_gb300.build import build
    build()
    from transformer_attention_gb300 import _lib as L
    return L


def _args(w, dev, L):
    t = L.GEMMA3_LOCAL_SLIDING if w.attn_type == "local" else L.GEMMA3_GLOBAL
    return (dev["x"].data_ptr(), dev["segment_pos"].data_ptr(), dev["pad_lens"].data_ptr(),
            dev["Wq"].data_ptr(), dev["Wkv"].data_ptr(), dev["Wo"].data_ptr(),
            dev["gamma_q"].data_ptr(), dev["gamma_k"].data_ptr(), t, w.window, w.rope_base,
            w.rope_scale, w.query_scale)


def test_noalloc_matches_workspace_entry_point_twice(lib):
    L = lib
    c = L.lib()
    w = WL.small(WL.WORKLOADS["tiny_local"], name="noalloc", B=2, T=640,
                 pad=("pad_uniform", 0, 200))
    dims = L.gemma3_attn_dims(w.B, w.T, w.D, w.H, w.H_kv, w.d_h)
    need = ctypes.c_size_t()
    assert c.gemma3_attn_workspace_size(ctypes.byref(dims), ctypes.byref(need)) == 0
    assert need.value <= c.gemma3_attn_noalloc_max_scratch()

    inp = Hh.make_inputs(w)
    dev = Hh.to_dev(inp)
    oracle = Hh.oracle_forward(w, inp)
    stream = torch.cuda.current_stream().cuda_stream
    ref = torch.empty((w.B, w.T, w.D), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(need.value, dtype=torch.uint8, device="cuda")
    rc = c.gemma3_attn_forward(ctypes.byref(dims), *_args(w, dev, L), ref.data_ptr(),
                               ws.data_ptr(), need.value, stream)
    assert rc == 0
    assert c.gemma3_attn_check_status(stream) == 0

    for call in range(2):
        out = torch.full((w.B, w.T, w.D), float("nan"), dtype=torch.bfloat16, device="cuda")
        rc = c.gemma3_attn_forward_noalloc(ctypes.byref(dims), *_args(w, dev, L),
                                           out.data_ptr(), stream)
        assert rc == 0, (call, rc)
        assert c.gemma3_attn_check_status(stream) == 0
        got, exp = out.cpu(), ref.cpu()
        for b in range(w.B):
            valid = w.T - int(dev["pad_lens"][b])
            Hh.assert_close(got[b, :valid], oracle[b, :valid],
                            f"no-alloc call {call} b={b} vs oracle")
            Hh.assert_close(got[b, :valid], exp[b, :valid], f"no-alloc call {call} b={b}")
            assert bool((got[b, valid:] == 0).all())


def test_noalloc_refuses_problems_larger_than_its_scratch(lib):
    L = lib
    c = L.lib()
    w = WL.WORKLOADS["tiny_local"]
    dev = Hh.to_dev(Hh.make_inputs(w))
    big = L.gemma3_attn_dims(64, 4096, w.D, w.H, w.H_kv, w.d_h)   # needs ~1.5 GiB
    out = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    rc = c.gemma3_attn_forward_noalloc(ctypes.byref(big), *_args(w, dev, L), out.data_ptr(),
                                       torch.cuda.current_stream().cuda_stream)
    assert rc == -6                       # GEMMA3_ERR_WORKSPACE, nothing launched
    assert c.gemma3_attn_check_status(torch.cuda.current_stream().cuda_stream) == 0
