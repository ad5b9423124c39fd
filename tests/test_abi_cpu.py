"""CPU-side checks of the C ABI: the library builds and loads without a GPU,
exports every function include/gemma3_attn.h declares, and its host logic
(routing, query scale, workspace sizes, argument validation) is right."""
import json
import os
import re

import pytest

from transformer_attention_gb300 import _lib as L
from transformer_attention_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gemma3_attn.h")


@pytest.fixture(scope="module")
def lib():
    build()
    return L.lib()


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(gemma3_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_abi():
    names = _declared_functions()
    for n in ("gemma3_attn_forward", "gemma3_layer_attn_type", "gemma3_layer_config",
              "gemma3_attn_workspace_size", "gemma3_attn_check_status", "gemma3_strerror"):
        assert n in names


def test_library_exports_every_declared_function(lib):
    names = _declared_functions()
    assert names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in gemma3_attn.h but not exported"
    assert set(names) == set(L.SIGNATURES), "binding and header disagree"


def _declared_arities():
    """Parameter count of every function the header declares."""
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    out = {}
    for m in re.finditer(r"\b(gemma3_[a-z0-9_]+)\s*\(([^;{]*?)\)\s*;", src):
        params = " ".join(m.group(2).split())
        out[m.group(1)] = 0 if params in ("", "void") else params.count(",") + 1
    return out


def test_binding_argument_counts_match_header():
    # a ctypes table entry with the wrong number of arguments would pass
    # every call's arguments shifted; compare it with the header's prototypes
    arity = _declared_arities()
    assert set(arity) == set(L.SIGNATURES)
    for name, (_, argtypes) in L.SIGNATURES.items():
        assert len(argtypes) == arity[name], (name, len(argtypes), arity[name])


def test_routing_matches_golden_table(lib):
    with open(os.path.join(ROOT, "tests", "golden", "routing_types.json")) as f:
        table = json.load(f)["types"]
    for n, types in table.items():
        got = "".join("G" if L.gemma3_layer_attn_type(l, int(n)) == L.GEMMA3_GLOBAL else "L"
                      for l in range(int(n)))
        assert got == types


def test_routing_rejects_bad_layers(lib):
    assert lib.gemma3_layer_attn_type(6, 6) < 0
    assert lib.gemma3_layer_attn_type(-1, 6) < 0
    assert lib.gemma3_layer_attn_type(0, 0) < 0


def test_layer_config_matches_golden(lib):
    with open(os.path.join(ROOT, "tests", "golden", "constants.json")) as f:
        rows = json.load(f)["layer_params"]["rows"]
    for size, kind, base, scale, window in rows:
        layer = 5 if kind == "GLOBAL" else 0
        t, w, b, s = L.gemma3_layer_config(layer, 6, size)
        assert t == (L.GEMMA3_GLOBAL if kind == "GLOBAL" else L.GEMMA3_LOCAL_SLIDING)
        assert (b, s, w) == (base, scale, window)


def test_query_scale(lib):
    with open(os.path.join(ROOT, "tests", "golden", "constants.json")) as f:
        c = json.load(f)
    q = c["query_scale_27B"]
    assert L.gemma3_query_scale("27B", q["D"], q["H"], q["d_h"]) == pytest.approx(q["value"], rel=1e-7)
    assert L.gemma3_query_scale("4B", 2560, 8, 256) == pytest.approx(0.0625, rel=1e-7)


def test_workspace_sizes(lib):
    n = L.gemma3_attn_workspace_size(2, 100, 1152, 8, 4, 256)
    assert n >= 2 * 100 * (8 + 2 * 4) * 256 * 2
    nb = L.gemma3_block_attn_workspace_size(2, 100, 1152, 8, 4, 256)
    assert nb >= n + 2 * 100 * 1152 * 6


@pytest.mark.parametrize("dims,code", [
    ((1, 16, 1152, 4, 1, 64), -3),     # d_h unsupported
    ((1, 16, 1152, 8, 1, 256), -3),    # G = 8 unsupported
    ((1, 16, 1152, 6, 4, 256), -1),    # H % H_kv != 0
    ((1, 16, 1150, 4, 1, 256), -1),    # D % 8 != 0
    ((0, 16, 1152, 4, 1, 256), -1),    # empty batch
])
def test_workspace_size_validation(lib, dims, code):
    import ctypes
    d = L.gemma3_attn_dims(*dims)
    n = ctypes.c_size_t()
    assert lib.gemma3_attn_workspace_size(ctypes.byref(d), ctypes.byref(n)) == code


def test_forward_rejects_null_pointers_before_any_launch(lib):
    import ctypes
    d = L.gemma3_attn_dims(1, 128, 1152, 4, 1, 256)
    rc = lib.gemma3_attn_forward(ctypes.byref(d), None, None, None, None, None, None, None, None,
                                 0, 512, 1e4, 1.0, 0.0625, None, None, 0, None)
    assert rc == -1
    assert L.strerror(rc) == "invalid argument"


def test_forward_rejects_bad_type_and_window(lib):
    import ctypes
    d = L.gemma3_attn_dims(1, 128, 1152, 4, 1, 256)
    p = 4096  # never dereferenced: validation fails first
    args = [ctypes.byref(d)] + [p] * 8
    assert lib.gemma3_attn_forward(*args, 7, 512, 1e4, 1.0, 0.0625, p, p, 1 << 30, None) == -1
    assert lib.gemma3_attn_forward(*args, 0, 0, 1e4, 1.0, 0.0625, p, p, 1 << 30, None) == -1
    assert lib.gemma3_attn_forward(*args, 1, 0, -1.0, 1.0, 0.0625, p, p, 1 << 30, None) == -1


def test_linear_rejects_misaligned(lib):
    assert lib.gemma3_linear(4096 + 2, 64, 4096, 64, 4096, 64, 16, 16, 64, 0, 0, 0, None, 0, None) == -2
    assert lib.gemma3_linear(4096, 60, 4096, 64, 4096, 64, 16, 16, 64, 0, 0, 0, None, 0, None) == -1
    assert lib.gemma3_linear(4096, 64, 4096, 64, 4096, 64, 16, 16, 64, 2, 0, 0, None, 0, None) == -1


def test_norms_reject_bad_pad_segments(lib):
    p = 4096
    assert lib.gemma3_rmsnorm(p, 0, p, p, 1, 16, 64, p, 0, None) == -1
    assert lib.gemma3_rmsnorm(p, 0, p, p, 1, 16, 64, p, 5, None) == -1
    assert lib.gemma3_postnorm_residual(p, p, 0, p, p, 16, 64, p, 0, None) == -1
    assert lib.gemma3_postnorm_residual(p, p, 0, p, p, 16, 64, p, 5, None) == -1


def test_linear_rejects_bad_pad_segments(lib):
    # pad_lens given: the segment length must be >= 1 and divide M
    args = (4096, 64, 4096, 64, 4096, 64, 16, 16, 64, 0, 0, 0, 4096)
    assert lib.gemma3_linear(*args, 0, None) == -1
    assert lib.gemma3_linear(*args, 5, None) == -1


def test_gemm_tile_rows_setting(lib):
    # a host-side setting: each call returns the previous value, others are refused
    assert lib.gemma3_set_gemm_tile_rows(256) == 0
    assert lib.gemma3_set_gemm_tile_rows(128) == 256
    assert lib.gemma3_set_gemm_tile_rows(0) == 128
    assert lib.gemma3_set_gemm_tile_rows(192) == -1
    assert lib.gemma3_set_gemm_tile_rows(0) == 0
