"""GPU parity of each stage kernel against the fp64 oracle's definition of it.

Stages: the tcgen05 projection GEMM, the fused QK-norm + RoPE + query-scale
prologue, and the flash-attention kernel, each fed the same seeded inputs as
the oracle, at sizes spanning several tiles and a ragged tail.
"""
import math

import pytest
import torch

from oracle import gemma3_oracle as O
from tests.helpers import QK_MAX_ABS, max_abs, rel_frob

pytestmark = pytest.mark.gpu

F64 = torch.float64


@pytest.fixture(scope="module", autouse=True)
def _built():
    from transformer_attention_gb300.build import build
    build()
    import transformer_attention_gb300 as G3
    G3.lib()
    torch.cuda.init()


def _randn(shape, seed, std=1.0, dtype=torch.bfloat16):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * std).to(dtype)


# ---------------------------------------------------------------- projection GEMM
@pytest.mark.parametrize("M,N,K", [(256, 512, 1152), (300, 1152, 4096), (1024, 2048, 2560),
                                   (130, 200, 72), (128, 256, 64), (4096, 1536, 1024),
                                   (1, 2048, 2560), (2, 5376, 4096), (3, 88, 72), (5, 1000, 1160),
                                   (8, 512, 1152), (16, 4096, 5376), (17, 296, 264),
                                   # M <= 16 (the few-row kernel: W on the MMA's 128-row
                                   # side, K split over a cluster): many rows, wide K
                                   (2, 20000, 1024), (4, 64, 16384), (2, 64, 40000),
                                   # a wave or more of tiles, 8+ wide: odd m-tile count,
                                   # ragged M / N / K
                                   (5170, 2200, 1024), (2000, 3000, 200),
                                   # a wave of tiles 5 wide (one CTA per tile)
                                   (5170, 1152, 1024),
                                   # a last tile column at most half full
                                   # (half-width MMAs): 1096 = 4 x 256 + 72
                                   (640, 1096, 512), (384, 96, 256)])
@pytest.mark.parametrize("out", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("inp", ["bf16", "f16"])
def test_linear_matches_fp64(M, N, K, out, inp):
    import transformer_attention_gb300 as G3
    dt = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}[out]
    it = {"bf16": torch.bfloat16, "f16": torch.float16}[inp]
    A = _randn((M, K), 1, 1.0, it)
    W = _randn((N, K), 2, K ** -0.5, it)
    C = G3.linear(A.cuda(), W.cuda(), out_dtype=dt)
    assert G3.gemma3_attn_check_status() == 0
    ref = O.project(A, W)
    tol = {"bf16": 4e-3, "f16": 1e-3, "f32": 1e-5}[out]
    assert rel_frob(C.cpu(), ref) <= tol


def test_cast_bf16_f16_is_exact_rounding():
    import transformer_attention_gb300 as G3
    src = _randn((4096,), 5, 3.0)
    dst = torch.empty(4096, dtype=torch.float16, device="cuda")
    G3.gemma3_cast_bf16_f16(src.cuda(), dst, 4096)
    assert G3.gemma3_attn_check_status() == 0
    assert torch.equal(dst.cpu(), src.float().to(torch.float16))


def test_linear_small_grid_many_tiles():
    # a 3-CTA persistent grid walking 48 tiles exercises the accumulator ring
    import transformer_attention_gb300 as G3
    A = _randn((1024, 640), 3)
    W = _randn((1536, 640), 4, 640 ** -0.5)
    C = G3.linear(A.cuda(), W.cuda(), out_dtype=torch.float32, max_ctas=3)
    assert G3.gemma3_attn_check_status() == 0
    assert rel_frob(C.cpu(), O.project(A, W)) <= 1e-5


@pytest.mark.parametrize("max_ctas", [4, 1])
def test_linear_wide_output_small_grid(max_ctas):
    # 160 tiles of a 10-tile-wide output walked by a persistent grid of 4
    # CTAs, or by one: the stage ring and the accumulator ring turn over
    # many times within each CTA
    import transformer_attention_gb300 as G3
    A = _randn((2048, 640), 6)
    W = _randn((2560, 640), 7, 640 ** -0.5)
    C = G3.linear(A.cuda(), W.cuda(), out_dtype=torch.float32, max_ctas=max_ctas)
    assert G3.gemma3_attn_check_status() == 0
    assert rel_frob(C.cpu(), O.project(A, W)) <= 1e-5


def test_linear_tile_sums_independent_of_launch_size():
    # every tile sums its k-steps in the same order whatever the grid: the
    # first 128 rows of a 160-tile launch equal a 10-tile launch of those rows
    # bit for bit
    import transformer_attention_gb300 as G3
    A = _randn((2048, 640), 8).cuda()
    W = _randn((2560, 640), 9, 640 ** -0.5).cuda()
    C_all = G3.linear(A, W, out_dtype=torch.float32)
    C_one = G3.linear(A[:128].contiguous(), W, out_dtype=torch.float32)
    assert G3.gemma3_attn_check_status() == 0
    assert torch.equal(C_all[:128].cpu(), C_one.cpu())


# ---------------------------------------------------------------- QK-norm + RoPE prologue
@pytest.mark.parametrize("d_h,H,H_kv,base,scale,alpha", [
    (256, 4, 1, 1e4, 1.0, 256 ** -0.5),
    (256, 8, 4, 1e6, 8.0, 256 ** -0.5),
    (128, 32, 16, 1e6, 8.0, 168 ** -0.5),
    (128, 4, 2, 1e4, 1.0, 128 ** -0.5),
])
@pytest.mark.parametrize("M", [777, 3])   # head vectors 8 steps per warp / 1 step per warp
def test_qk_norm_rope_matches_oracle(d_h, H, H_kv, base, scale, alpha, M):
    import transformer_attention_gb300 as G3
    Qr = _randn((M, H * d_h), 10, 1.0, torch.float16)
    KVr = _randn((M, 2 * H_kv * d_h), 11, 1.0, torch.float16)
    gq = _randn((d_h,), 12, 0.1 ** 0.5)
    gk = _randn((d_h,), 13, 0.1 ** 0.5)
    g = torch.Generator().manual_seed(14)
    pos = torch.cat([torch.arange(0, 300), torch.randint(0, 131072, (475,), generator=g),
                     torch.tensor([131071, 2 ** 20])]).to(torch.int32)[-M:].contiguous()
    Qd, KVd = Qr.cuda(), KVr.cuda()
    G3.gemma3_qk_norm_rope(Qd, H * d_h, KVd, 2 * H_kv * d_h, gq.cuda(), gk.cuda(), pos.cuda(),
                           M, H, H_kv, d_h, base, scale, alpha)
    assert G3.gemma3_attn_check_status() == 0
    Qo, KVo = Qd.cpu(), KVd.cpu()
    q_ref = O.rope(O.rms_norm(Qr.reshape(M, H, d_h), gq)[None], pos[None], base, scale)[0]
    k_ref = O.rope(O.rms_norm(KVr[:, :H_kv * d_h].reshape(M, H_kv, d_h), gk)[None], pos[None],
                   base, scale)[0]
    q_got = Qo.reshape(M, H, d_h).to(F64) / alpha
    k_got = KVo[:, :H_kv * d_h].reshape(M, H_kv, d_h)
    assert max_abs(q_got, q_ref) <= QK_MAX_ABS
    assert max_abs(k_got, k_ref) <= QK_MAX_ABS
    # V columns are untouched ("QK-Norm": values are left unnormalised)
    assert torch.equal(KVo[:, H_kv * d_h:], KVr[:, H_kv * d_h:])


# ---------------------------------------------------------------- fused projection + prologue
@pytest.mark.parametrize("M,D,d_h,H,H_kv,base,scale,alpha,inp", [
    (300, 1152, 256, 4, 1, 1e6, 1.0, 256 ** -0.5, "bf16"),
    (1000, 512, 256, 8, 4, 1e4, 1.0, 256 ** -0.5, "f16"),
    (257, 384, 128, 4, 2, 1e6, 8.0, 168 ** -0.5, "bf16"),
    (129, 256, 128, 32, 16, 1e6, 8.0, 168 ** -0.5, "bf16"),
    (17, 192, 128, 2, 2, 1e4, 1.0, 128 ** -0.5, "f16"),
])
def test_linear_qk_norm_rope_matches_oracle(M, D, d_h, H, H_kv, base, scale, alpha, inp):
    """The Q and KV projections with QK-norm, RoPE and the query scale in the
    GEMM epilogue against the oracle's normalised and rotated Q/K (before
    the query scale) and its plain V projection."""
    import transformer_attention_gb300 as G3
    it = {"bf16": torch.bfloat16, "f16": torch.float16}[inp]
    code = {"bf16": G3.GEMMA3_BF16, "f16": G3.GEMMA3_F16}[inp]
    HD, KVD = H * d_h, H_kv * d_h
    x = _randn((M, D), 20, 1.0, it)
    Wq = _randn((HD, D), 21, D ** -0.5, it)
    Wkv = _randn((2, KVD, D), 22, D ** -0.5, it)
    gq = _randn((d_h,), 23, 0.1 ** 0.5)
    gk = _randn((d_h,), 24, 0.1 ** 0.5)
    g = torch.Generator().manual_seed(25)
    pos = torch.randint(0, 131072, (M,), generator=g).to(torch.int32)
    pos[:3] = torch.tensor([0, 1, 131071], dtype=torch.int32)
    Qd = torch.empty((M, HD), dtype=torch.float16, device="cuda")
    KVd = torch.empty((M, 2 * KVD), dtype=torch.float16, device="cuda")
    xd, posd = x.cuda(), pos.cuda()
    G3.gemma3_linear_qk_norm_rope(xd, D, Wq.cuda(), D, Qd, HD, M, HD, D, code, gq.cuda(), posd,
                                  d_h, HD, base, scale, alpha)
    G3.gemma3_linear_qk_norm_rope(xd, D, Wkv.reshape(2 * KVD, D).cuda(), D, KVd, 2 * KVD, M,
                                  2 * KVD, D, code, gk.cuda(), posd, d_h, KVD, base, scale, 1.0)
    assert G3.gemma3_attn_check_status() == 0
    q_ref, k_ref = O.normalised_rotated_qk(x, pos, Wq, Wkv, gq, gk, H=H, H_kv=H_kv, d_h=d_h,
                                           rope_base=base, rope_scale=scale)
    q_got = Qd.cpu().reshape(M, H, d_h).to(F64) / alpha
    kv = KVd.cpu()
    assert max_abs(q_got, q_ref) <= QK_MAX_ABS
    assert max_abs(kv[:, :KVD].reshape(M, H_kv, d_h), k_ref) <= QK_MAX_ABS
    assert rel_frob(kv[:, KVD:], O.project(x, Wkv[1])) <= 1e-3


@pytest.mark.parametrize("M,D,d_h,H,H_kv,base,scale,alpha", [
    (300, 1152, 256, 4, 1, 1e6, 1.0, 256 ** -0.5),     # one launch, Q 4 tiles + K|V 2 tiles
    (777, 640, 128, 32, 16, 1e6, 8.0, 168 ** -0.5),    # one launch, two heads per tile
    (9, 256, 256, 8, 4, 1e4, 1.0, 256 ** -0.5),        # <= 16 rows: one two-projection
    (2, 512, 128, 4, 2, 1e6, 8.0, 168 ** -0.5),        # launch of the few-row kernel + prologue
    (16, 384, 128, 2, 2, 1e4, 1.0, 128 ** -0.5),
    (40, 256, 128, 2, 1, 1e4, 1.0, 128 ** -0.5),       # K|V width 256 is one tile, K 128
])
def test_qkv_proj_norm_rope_matches_oracle(M, D, d_h, H, H_kv, base, scale, alpha):
    """The whole first stage (both projections with the prologue) against the
    oracle's normalised and rotated Q/K and its V projection."""
    import transformer_attention_gb300 as G3
    HD, KVD = H * d_h, H_kv * d_h
    x = _randn((M, D), 40, 1.0)
    Wq = _randn((HD, D), 41, D ** -0.5)
    Wkv = _randn((2, KVD, D), 42, D ** -0.5)
    gq = _randn((d_h,), 43, 0.1 ** 0.5)
    gk = _randn((d_h,), 44, 0.1 ** 0.5)
    g = torch.Generator().manual_seed(45)
    pos = torch.randint(0, 131072, (M,), generator=g).to(torch.int32)
    Qd = torch.empty((M, HD), dtype=torch.float16, device="cuda")
    KVd = torch.empty((M, 2 * KVD), dtype=torch.float16, device="cuda")
    G3.gemma3_qkv_proj_norm_rope(x.cuda(), D, Wq.cuda(), Wkv.cuda(), Qd, KVd, M, D, H, H_kv, d_h,
                                 G3.GEMMA3_BF16, gq.cuda(), gk.cuda(), pos.cuda(), base, scale,
                                 alpha)
    assert G3.gemma3_attn_check_status() == 0
    q_ref, k_ref = O.normalised_rotated_qk(x, pos, Wq, Wkv, gq, gk, H=H, H_kv=H_kv, d_h=d_h,
                                           rope_base=base, rope_scale=scale)
    kv = KVd.cpu()
    assert max_abs(Qd.cpu().reshape(M, H, d_h).to(F64) / alpha, q_ref) <= QK_MAX_ABS
    assert max_abs(kv[:, :KVD].reshape(M, H_kv, d_h), k_ref) <= QK_MAX_ABS
    assert rel_frob(kv[:, KVD:], O.project(x, Wkv[1])) <= 1e-3


@pytest.mark.parametrize("out_dtype", ["bf16", "f32"])
def test_linear_pad_only_tiles(out_dtype):
    """Three segments of 384 rows with 0, 200 and 384 trailing pad rows: the
    rows of pad-only 128-row tiles are left unwritten, every other row equals
    the product without pad_lens bit for bit (the same tiles, the same k
    order)."""
    import transformer_attention_gb300 as G3
    T, pads = 384, [0, 200, 384]
    M, N, K = T * len(pads), 640, 512
    A = _randn((M, K), 60, 1.0).cuda()
    W = _randn((N, K), 61, K ** -0.5).cuda()
    dt, code = ((torch.bfloat16, G3.GEMMA3_BF16) if out_dtype == "bf16"
                else (torch.float32, G3.GEMMA3_F32))
    full = torch.empty((M, N), dtype=dt, device="cuda")
    part = torch.full((M, N), float("nan"), dtype=dt, device="cuda")
    G3.gemma3_linear(A, K, W, K, full, N, M, N, K, G3.GEMMA3_BF16, code)
    G3.gemma3_linear(A, K, W, K, part, N, M, N, K, G3.GEMMA3_BF16, code,
                     pad_lens=torch.tensor(pads, dtype=torch.int32, device="cuda"), seg_T=T)
    assert G3.gemma3_attn_check_status() == 0
    full, part = full.cpu(), part.cpu()
    for b, pad in enumerate(pads):
        kept = -(-(T - pad) // 128) * 128          # rows of the tiles holding a valid row
        rows = slice(b * T, b * T + kept)
        assert torch.equal(part[rows], full[rows])
        assert bool(torch.isnan(part[b * T + kept:(b + 1) * T]).all())


def test_qkv_proj_pad_only_tiles():
    """The fused Q|KV stage with pad_lens: in pad-only tiles V rows are zeros
    and Q', K' rows unwritten; the rest equal the call without pad_lens bit
    for bit."""
    import transformer_attention_gb300 as G3
    T, pads, D, d_h, H, H_kv = 256, [100, 256, 0], 256, 256, 2, 1
    M, HD, KVD = T * len(pads), H * d_h, H_kv * d_h
    x = _randn((M, D), 62, 1.0).cuda()
    Wq = _randn((HD, D), 63, D ** -0.5).cuda()
    Wkv = _randn((2, KVD, D), 64, D ** -0.5).cuda()
    gq = _randn((d_h,), 65, 0.1 ** 0.5).cuda()
    gk = _randn((d_h,), 66, 0.1 ** 0.5).cuda()
    pos = torch.arange(M, dtype=torch.int32, device="cuda") % T
    outs = []
    for pl in (None, torch.tensor(pads, dtype=torch.int32, device="cuda")):
        Qd = torch.full((M, HD), float("nan"), dtype=torch.float16, device="cuda")
        KVd = torch.full((M, 2 * KVD), float("nan"), dtype=torch.float16, device="cuda")
        G3.gemma3_qkv_proj_norm_rope(x, D, Wq, Wkv, Qd, KVd, M, D, H, H_kv, d_h, G3.GEMMA3_BF16,
                                     gq, gk, pos, 1e4, 1.0, d_h ** -0.5, pad_lens=pl,
                                     seg_T=T if pl is not None else 0)
        assert G3.gemma3_attn_check_status() == 0
        outs.append((Qd.cpu(), KVd.cpu()))
    for i, (full, part) in enumerate(zip(outs[0], outs[1])):
        for b, pad in enumerate(pads):
            kept = -(-(T - pad) // 128) * 128
            assert torch.equal(part[b * T:b * T + kept], full[b * T:b * T + kept])
            tail = part[b * T + kept:(b + 1) * T]
            if i == 0:      # Q'
                assert bool(torch.isnan(tail).all())
            else:           # K' unwritten, V zeros
                assert bool(torch.isnan(tail[:, :KVD]).all())
                assert torch.equal(tail[:, KVD:], torch.zeros_like(tail[:, KVD:]))


def test_linear_qk_norm_rope_rejects_unaligned_heads():
    import transformer_attention_gb300 as G3
    x = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((384, 64), dtype=torch.bfloat16, device="cuda")
    C = torch.empty((64, 384), dtype=torch.float16, device="cuda")
    g = torch.zeros(128, dtype=torch.bfloat16, device="cuda")
    pos = torch.zeros(64, dtype=torch.int32, device="cuda")
    with pytest.raises(G3.Gemma3Error):   # n_norm = 128 is not a whole 256-wide tile
        G3.gemma3_linear_qk_norm_rope(x, 64, W, 64, C, 384, 64, 384, 64, G3.GEMMA3_BF16, g, pos,
                                      128, 128, 1e4, 1.0, 1.0)


# ---------------------------------------------------------------- flash attention
ATTN_CASES = [
    # B, T, H, H_kv, d_h, window, pads
    (2, 300, 4, 1, 256, 100, [0, 37]),
    (1, 1024, 8, 4, 256, 0, [0]),
    (2, 513, 4, 2, 128, 0, [0, 200]),
    (1, 700, 2, 2, 128, 256, [0]),
    (1, 640, 8, 2, 128, 0, [5]),
    (1, 257, 2, 2, 256, 0, [0]),
    (1, 1, 4, 1, 256, 0, [0]),
    (3, 190, 4, 1, 256, 64, [0, 189, 190]),
    (1, 1500, 4, 1, 256, 512, [0]),
    # d_h = 128 runs two query tiles per CTA: a second tile past T, a second
    # tile all padding, an item all padding, windows with one and four heads
    (2, 333, 4, 2, 128, 0, [0, 150]),
    (1, 100, 2, 2, 128, 0, [0]),
    (1, 300, 4, 1, 128, 100, [0]),
    (3, 260, 2, 1, 128, 64, [0, 259, 260]),
    (1, 1100, 8, 4, 128, 300, [0]),
    # local layers with more (b, kv head) pairs than one L2 ordering group
    # holds: groups of 8 pairs (d_h = 256) and of 50 + a partial 14 (d_h =
    # 128), with a one-token row and an all-padding row
    (4, 1024, 32, 16, 256, 1000, [0, 100, 1023, 1024]),
    (2, 512, 64, 32, 128, 200, [0, 77]),
    # d_h = 256 local layers run KV tiles from each item's first visible key:
    # last tiles of 128 (one head per kv head), 16 (two, a padded row) and
    # 112 keys (four), tiles that run past T
    (1, 2000, 2, 2, 256, 1024, [0]),
    (2, 900, 8, 4, 256, 200, [0, 333]),
    (1, 700, 8, 2, 256, 80, [3]),
]


@pytest.mark.parametrize("B,T,H,H_kv,d_h,window,pads", ATTN_CASES)
@pytest.mark.parametrize("o_f16,sched", [(False, True), (True, True), (False, False)])
def test_flash_attention_matches_oracle(B, T, H, H_kv, d_h, window, pads, o_f16, sched):
    import transformer_attention_gb300 as G3
    G = H // H_kv
    alpha = d_h ** -0.5
    # Q' carries the query scale; |q|, |k| ~ RMS-normalised heads with (1 + gamma)
    Q = (_randn((B, T, H, d_h), 20, 1.3, torch.float32) * alpha).to(torch.float16)
    KV = _randn((B, T, 2 * H_kv * d_h), 21, 1.3, torch.float16)
    pad = torch.tensor(pads, dtype=torch.int32)
    Qd, KVd = Q.cuda(), KV.cuda()
    Od = torch.empty((B, T, H, d_h), dtype=torch.float16 if o_f16 else torch.bfloat16,
                     device="cuda")
    Od.fill_(float("nan"))
    # sched: the work counter (dynamic order) or none (fixed assignment)
    scratch = torch.full((256,), 0x5A, dtype=torch.uint8, device="cuda") if sched else None
    G3.gemma3_flash_attention(Qd, KVd, KVd[..., H_kv * d_h:], 2 * H_kv * d_h, Od,
                              G3.GEMMA3_F16 if o_f16 else G3.GEMMA3_BF16, pad.cuda(), B, T,
                              H, H_kv, d_h, window, scratch)
    assert G3.gemma3_attn_check_status() == 0
    got = Od.cpu().to(F64)
    kind = O.LOCAL_SLIDING if window > 0 else O.GLOBAL
    for b in range(B):
        valid = T - pads[b]
        K = KV[b, :, :H_kv * d_h].reshape(T, H_kv, d_h).to(F64)
        V = KV[b, :, H_kv * d_h:].reshape(T, H_kv, d_h).to(F64)
        idx = torch.arange(T)
        if valid > 0:
            ref = O.attend(Q[b, :valid].to(F64), K, V, idx[:valid], idx, valid, kind, window)
            assert rel_frob(got[b, :valid], ref) <= 5e-3, (b, rel_frob(got[b, :valid], ref))
            assert max_abs(got[b, :valid], ref) <= 2e-2
        assert torch.equal(got[b, valid:], torch.zeros_like(got[b, valid:]))
    _ = G  # G in {1,2,4} is covered by the cases above


def test_flash_attention_local_window_ge_T_equals_global():
    import transformer_attention_gb300 as G3
    B, T, H, H_kv, d_h = 1, 384, 4, 2, 256
    Q = (_randn((B, T, H, d_h), 30, 1.0, torch.float32) / 16).to(torch.float16).cuda()
    KV = _randn((B, T, 2 * H_kv * d_h), 31, 1.0, torch.float16).cuda()
    outs = []
    for window in (0, T, 5 * T):
        Od = torch.empty((B, T, H, d_h), dtype=torch.bfloat16, device="cuda")
        G3.gemma3_flash_attention(Q, KV, KV[..., H_kv * d_h:], 2 * H_kv * d_h, Od, G3.GEMMA3_BF16,
                                  None, B, T, H, H_kv, d_h, window)
        outs.append(Od.cpu())
    assert G3.gemma3_attn_check_status() == 0
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])


# ---------------------------------------------------------------- block norms
# Widths of every row-kernel variant: the register-resident ones (D <= 1024,
# 2048, 4096, 6144) and the two-pass one above; row counts not a multiple of
# the 4 or 8 rows per CTA.
NORM_CASES = [(37, 256), (13, 1152), (9, 3840), (7, 5376), (5, 8192)]


@pytest.mark.parametrize("M,D", NORM_CASES)
@pytest.mark.parametrize("x_t,u_t", [("f32", "f16"), ("bf16", "bf16")])
def test_rmsnorm_rows_matches_oracle(M, D, x_t, u_t):
    import transformer_attention_gb300 as G3
    xd = {"f32": torch.float32, "bf16": torch.bfloat16}[x_t]
    ud = {"f16": torch.float16, "bf16": torch.bfloat16}[u_t]
    x = _randn((M, D), 50, 3.0, xd)
    gamma = _randn((D,), 51, 0.1 ** 0.5)
    u = torch.empty((M, D), dtype=ud, device="cuda")
    G3.gemma3_rmsnorm(x.cuda(), G3.GEMMA3_F32 if x_t == "f32" else G3.GEMMA3_BF16, gamma.cuda(),
                      u, G3.GEMMA3_F16 if u_t == "f16" else G3.GEMMA3_BF16, M, D)
    assert G3.gemma3_attn_check_status() == 0
    ref = O.rms_norm(x, gamma)
    tol = {"f16": 1e-3, "bf16": 4e-3}[u_t]
    assert rel_frob(u.cpu(), ref) <= tol


@pytest.mark.parametrize("M,D", NORM_CASES)
@pytest.mark.parametrize("x_t", ["f32", "bf16"])
def test_postnorm_residual_matches_oracle(M, D, x_t):
    import transformer_attention_gb300 as G3
    xd = {"f32": torch.float32, "bf16": torch.bfloat16}[x_t]
    a = _randn((M, D), 52, 2.0, torch.float32)
    x = _randn((M, D), 53, 1.0, xd)
    gamma = _randn((D,), 54, 0.1 ** 0.5)
    y = torch.empty((M, D), dtype=torch.float32, device="cuda")
    G3.gemma3_postnorm_residual(a.cuda(), x.cuda(), G3.GEMMA3_F32 if x_t == "f32" else
                                G3.GEMMA3_BF16, gamma.cuda(), y, M, D)
    assert G3.gemma3_attn_check_status() == 0
    ref = x.to(F64) + O.rms_norm(a, gamma)
    assert rel_frob(y.cpu(), ref) <= 1e-6


PAD_NORM = [1152, 3840, 5376]   # the two-pass and both register-resident pre-norms


@pytest.mark.parametrize("D", PAD_NORM)
def test_rmsnorm_pad_tiles_untouched(D):
    """With pad_lens the pre-norm leaves the rows of pad-only 128-row tiles
    untouched and writes every other row as without pad_lens."""
    import transformer_attention_gb300 as G3
    T, pads = 384, [0, 200, 384]
    M = T * len(pads)
    x = _randn((M, D), 55, 3.0, torch.float32).cuda()
    gamma = _randn((D,), 56, 0.1 ** 0.5).cuda()
    full = torch.empty((M, D), dtype=torch.float16, device="cuda")
    part = torch.full((M, D), float("nan"), dtype=torch.float16, device="cuda")
    G3.gemma3_rmsnorm(x, G3.GEMMA3_F32, gamma, full, G3.GEMMA3_F16, M, D)
    G3.gemma3_rmsnorm(x, G3.GEMMA3_F32, gamma, part, G3.GEMMA3_F16, M, D,
                      pad_lens=torch.tensor(pads, dtype=torch.int32, device="cuda"), seg_T=T)
    assert G3.gemma3_attn_check_status() == 0
    full, part = full.cpu(), part.cpu()
    for b, pad in enumerate(pads):
        kept = -(-(T - pad) // 128) * 128
        assert torch.equal(part[b * T:b * T + kept], full[b * T:b * T + kept])
        assert bool(torch.isnan(part[b * T + kept:(b + 1) * T]).all())


@pytest.mark.parametrize("D", [1152, 3840])
@pytest.mark.parametrize("inplace", [True, False])
def test_postnorm_pad_rows_pass_through(D, inplace):
    """With pad_lens the pad rows get y = x exactly without a being read (a
    holds NaN there), in place and not; valid rows as without pad_lens."""
    import transformer_attention_gb300 as G3
    T, pads = 256, [0, 100, 256]
    M = T * len(pads)
    valid = torch.ones(M, dtype=torch.bool)
    for b, pad in enumerate(pads):
        valid[b * T + T - pad:(b + 1) * T] = False
    a = _randn((M, D), 57, 2.0, torch.float32)
    a_nan = a.clone()
    a_nan[~valid] = float("nan")
    gamma = _randn((D,), 58, 0.1 ** 0.5).cuda()
    pl = torch.tensor(pads, dtype=torch.int32, device="cuda")
    if inplace:
        x = _randn((M, D), 59, 1.0, torch.float32)
        y_ref = x.clone().cuda()
        y = x.clone().cuda()
        G3.gemma3_postnorm_residual(a.cuda(), y_ref, G3.GEMMA3_F32, gamma, y_ref, M, D)
        G3.gemma3_postnorm_residual(a_nan.cuda(), y, G3.GEMMA3_F32, gamma, y, M, D,
                                    pad_lens=pl, seg_T=T)
        x_f = x
    else:
        x = _randn((M, D), 59, 1.0, torch.bfloat16).cuda()
        y_ref = torch.empty((M, D), dtype=torch.float32, device="cuda")
        y = torch.full((M, D), float("nan"), dtype=torch.float32, device="cuda")
        G3.gemma3_postnorm_residual(a.cuda(), x, G3.GEMMA3_BF16, gamma, y_ref, M, D)
        G3.gemma3_postnorm_residual(a_nan.cuda(), x, G3.GEMMA3_BF16, gamma, y, M, D,
                                    pad_lens=pl, seg_T=T)
        x_f = x.cpu().float()
    assert G3.gemma3_attn_check_status() == 0
    y, y_ref = y.cpu(), y_ref.cpu()
    assert torch.equal(y[valid], y_ref[valid])
    assert torch.equal(y[~valid], x_f[~valid])
