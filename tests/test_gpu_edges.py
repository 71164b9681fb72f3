"""GPU vs oracle on edge shapes and paths: odd widths, single rows, unaligned
pointers (the element-wise path), both weight dtypes, optional residual and
residual gradient, in-place calls, empty inputs, out-of-range positions,
determinism of the weight gradient, workspace errors and canary bands."""

import numpy as np
import pytest
import torch

import oracle
import rmsnorm_fwd_bwd_03_gb300 as gb

from _checks import Guarded, check_dw, check_io, check_rstd, dx_scale, to64

pytestmark = pytest.mark.gpu

IO = {"f32": torch.float32, "bf16": torch.bfloat16}


@pytest.fixture(scope="module", autouse=True)
def _library():
    from rmsnorm_fwd_bwd_03_gb300._build import build_library
    build_library()
    gb.library()


def _randn(shape, dtype, seed, scale=1.0, offset=0):
    g = torch.Generator(device="cuda").manual_seed(seed)
    n = int(np.prod(shape))
    buf = torch.randn(n + offset, generator=g, device="cuda", dtype=torch.float32) * scale
    return buf.to(dtype)[offset:].view(shape)  # offset > 0 gives a pointer off 16-byte alignment


# ---------------------------------------------------------------------------
# RMSNorm
# ---------------------------------------------------------------------------

RMS_SHAPES = [(1, 1), (3, 13), (5, 8), (7, 896), (33, 1000), (2, 1024), (17, 4100), (6, 8192),
              (3, 16384), (2, 20000), (300, 64)]


@pytest.mark.parametrize("T,H", RMS_SHAPES)
@pytest.mark.parametrize("io,wt", [("f32", "f32"), ("bf16", "bf16"), ("bf16", "f32")])
@pytest.mark.parametrize("residual", [True, False])
@pytest.mark.parametrize("offset", [0, 1])
def test_rmsnorm_shapes(T, H, io, wt, residual, offset):
    dt, wdt = IO[io], IO[wt]
    eps = 1e-5
    x = _randn((T, H), dt, 1, offset=offset)
    r = _randn((T, H), dt, 2, offset=offset) if residual else None
    w = (1 + 0.1 * _randn((H,), torch.float32, 3)).to(wdt)
    dy = _randn((T, H), dt, 4, offset=offset)
    dres = _randn((T, H), dt, 5, offset=offset) if residual else None
    y, h, rstd = gb.rmsnorm_fwd(x, w, eps, r)
    dx, part, P = gb.rmsnorm_bwd(dy, h, w, rstd, dres)
    dw = gb.rmsnorm_dw_finalize(part, P)
    torch.cuda.synchronize()
    w64 = to64(w)
    y_ref, h_ref, rstd_ref = oracle.rmsnorm_fwd(to64(x), None if r is None else to64(r), w64, eps, io=io)
    if residual:
        assert np.array_equal(to64(h), h_ref)
    check_io(to64(y), y_ref, io, "y")
    check_rstd(to64(rstd), rstd_ref)
    dres64 = None if dres is None else to64(dres)
    dx_ref, dw_ref = oracle.rmsnorm_bwd(to64(dy), dres64, h_ref, w64, eps)
    check_io(to64(dx), dx_ref, io, "dx", scale=dx_scale(to64(dy), w64, rstd_ref, dres64))
    check_dw(to64(dw), dw_ref)


def test_rmsnorm_largest_row():
    # H = 2^24, the largest width the entry points accept: one block per row on the
    # element-wise kernels, a single partial row.
    T, H = 1, 1 << 24
    x = _randn((T, H), torch.bfloat16, 6)
    r = _randn((T, H), torch.bfloat16, 7)
    w = (1 + 0.1 * _randn((H,), torch.float32, 8))
    dy = _randn((T, H), torch.bfloat16, 9)
    y, h, rstd = gb.rmsnorm_fwd(x, w, 1e-5, r)
    dx, part, P = gb.rmsnorm_bwd(dy, h, w, rstd, None)
    dw = gb.rmsnorm_dw_finalize(part, P)
    torch.cuda.synchronize()
    w64 = to64(w)
    y_ref, h_ref, rstd_ref = oracle.rmsnorm_fwd(to64(x), to64(r), w64, 1e-5, io="bf16")
    assert np.array_equal(to64(h), h_ref)
    check_io(to64(y), y_ref, "bf16", "y")
    check_rstd(to64(rstd), rstd_ref)
    dx_ref, dw_ref = oracle.rmsnorm_bwd(to64(dy), None, h_ref, w64, 1e-5)
    check_io(to64(dx), dx_ref, "bf16", "dx")
    check_dw(to64(dw), dw_ref)


def test_rmsnorm_outlier_channels_and_large_eps():
    T, H = 64, 4096
    x = _randn((T, H), torch.bfloat16, 11)
    x[:, ::100] *= 50
    w = (1 + 0.1 * _randn((H,), torch.float32, 12)).to(torch.bfloat16)
    for eps in (0.0, 1e-6, 10.0):
        y, h, rstd = gb.rmsnorm_fwd(x, w, eps)
        y_ref, _, rstd_ref = oracle.rmsnorm_fwd(to64(x), None, to64(w), eps)
        check_io(to64(y), y_ref, "bf16", f"y eps={eps}")
        check_rstd(to64(rstd), rstd_ref)


def test_rmsnorm_guard_bands_and_inplace_residual():
    T, H = 37, 1024
    dt = torch.bfloat16
    x = _randn((T, H), dt, 21)
    r = _randn((T, H), dt, 22)
    w = (1 + 0.1 * _randn((H,), torch.float32, 23)).to(dt)
    gy, gr = Guarded((T, H), dt), Guarded((T,), torch.float32)
    x_copy = x.clone()
    # residual_out aliases x exactly (in-place residual stream)
    y, h, rstd = gb.rmsnorm_fwd(x, w, 1e-6, r, y=gy.tensor, residual_out=x, rstd=gr.tensor)
    torch.cuda.synchronize()
    assert gy.intact() and gr.intact()
    y_ref, h_ref, _ = oracle.rmsnorm_fwd(to64(x_copy), to64(r), to64(w), 1e-6, io="bf16")
    assert np.array_equal(to64(x), h_ref)
    check_io(to64(y), y_ref, "bf16", "y")
    dy = _randn((T, H), dt, 24)
    P = gb.rmsnorm_bwd_num_partials(T, H, dt)
    gdx, gp, gdw = Guarded((T, H), dt), Guarded((P, H), torch.float32), Guarded((H,), torch.float32)
    gb.rmsnorm_bwd(dy, h, w, rstd, None, dx=gdx.tensor, dw_partial=gp.tensor)
    gb.rmsnorm_dw_finalize(gp.tensor, P, dw=gdw.tensor)
    torch.cuda.synchronize()
    assert gdx.intact() and gp.intact() and gdw.intact()


@pytest.mark.parametrize("T,H,dt", [(16384, 1024, torch.bfloat16), (4099, 4096, torch.bfloat16),
                                    (1000, 896, torch.float32), (50, 13, torch.bfloat16)])
def test_rmsnorm_dw_bitwise_deterministic(T, H, dt):
    h = _randn((T, H), dt, 31)
    dy = _randn((T, H), dt, 32)
    w = (1 + 0.1 * _randn((H,), torch.float32, 33)).to(dt)
    rstd = torch.rsqrt(h.float().pow(2).mean(-1) + 1e-5)
    outs = []
    for stream in (torch.cuda.current_stream(), torch.cuda.Stream()):
        with torch.cuda.stream(stream):
            dx, part, P = gb.rmsnorm_bwd(dy, h, w, rstd)
            outs.append((dx.clone(), gb.rmsnorm_dw_finalize(part, P).clone()))
        torch.cuda.synchronize()
    assert torch.equal(outs[0][0], outs[1][0])
    assert torch.equal(outs[0][1].view(torch.int32), outs[1][1].view(torch.int32))


def test_rmsnorm_dw_accumulate():
    T, H = 100, 512
    dt = torch.bfloat16
    h = _randn((T, H), dt, 41)
    dy = _randn((T, H), dt, 42)
    w = torch.ones(H, dtype=dt, device="cuda")
    rstd = torch.rsqrt(h.float().pow(2).mean(-1) + 1e-5)
    _, part, P = gb.rmsnorm_bwd(dy, h, w, rstd)
    dw1 = gb.rmsnorm_dw_finalize(part, P)
    dw2 = gb.rmsnorm_dw_finalize(part, P, dw=dw1.clone(), accumulate=True)
    torch.cuda.synchronize()
    assert torch.allclose(dw2, 2 * dw1, rtol=1e-6, atol=0)


def test_rmsnorm_workspace_too_small_and_empty():
    T, H = 1000, 1024
    dt = torch.bfloat16
    lib = gb.library()
    P = gb.rmsnorm_bwd_num_partials(T, H, dt)
    assert P >= 1
    t = torch.zeros((T, H), dtype=dt, device="cuda")
    w = torch.ones(H, dtype=dt, device="cuda")
    rs = torch.ones(T, dtype=torch.float32, device="cuda")
    part = torch.zeros((P, H), dtype=torch.float32, device="cuda")
    st = lib.gbln_rmsnorm_bwd(t.data_ptr(), None, t.data_ptr(), w.data_ptr(), rs.data_ptr(), t.data_ptr(),
                              part.data_ptr(), P - 1, T, H, gb.BF16, gb.BF16, None)
    assert st == 3  # GBLN_ERR_WORKSPACE
    assert gb.rmsnorm_bwd_num_partials(0, H, dt) == 0
    x = torch.empty((0, H), dtype=dt, device="cuda")
    y, h, rstd = gb.rmsnorm_fwd(x, w, 1e-5, x)
    assert y.shape == (0, H) and rstd.shape == (0,)
    dw = gb.rmsnorm_dw_finalize(torch.empty((1, H), device="cuda"), 0)
    torch.cuda.synchronize()
    assert torch.equal(dw, torch.zeros(H, device="cuda"))


# ---------------------------------------------------------------------------
# RoPE
# ---------------------------------------------------------------------------

# (40, 8, 128) and (44, 8, 128) sit on either side of the warp kernel's limit of
# 12 head rows per lane for bf16 (48 and 52 heads); (20, 4, 128) and (21, 4, 128)
# for float32 (24 and 25 heads of 16 units).
@pytest.mark.parametrize("T,Hq,Hk,D", [(1, 1, 0, 2), (5, 3, 1, 6), (7, 14, 2, 64), (9, 4, 4, 128),
                                        (33, 2, 1, 256), (3, 1, 1, 18), (5, 40, 8, 128),
                                        (5, 44, 8, 128), (6, 20, 4, 128), (6, 21, 4, 128)])
@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("offset", [0, 1])
def test_rope_shapes(T, Hq, Hk, D, io, offset):
    dt = IO[io]
    theta = 10000.0
    q = _randn((T, Hq, D), dt, 51, offset=offset)
    k = _randn((T, Hk, D), dt, 52, offset=offset) if Hk else None
    pos = torch.as_tensor(np.random.default_rng(53).integers(0, 5000, size=T), dtype=torch.int32, device="cuda")
    table = gb.rope_table(5000, D, theta)
    qo, ko = gb.rope_fwd(q, k, pos, table)
    dqi, dki = gb.rope_bwd(q, k, pos, table)
    torch.cuda.synchronize()
    p = pos.cpu().numpy()
    check_io(to64(qo), oracle.rope_fwd(to64(q), p, theta), io, "q'")
    check_io(to64(dqi), oracle.rope_bwd(to64(q), p, theta), io, "dq")
    if Hk:
        check_io(to64(ko), oracle.rope_fwd(to64(k), p, theta), io, "k'")
        check_io(to64(dki), oracle.rope_bwd(to64(k), p, theta), io, "dk")


@pytest.mark.parametrize("D,offset", [(8192, 0), (1024, 1)])
def test_rope_largest_heads(D, offset):
    # The largest head sizes: D = 8192 on the bf16 vector path (512 units of 8
    # elements per head half), D = 1024 on the element-wise path (512 units).
    T, dt, theta = 3, torch.bfloat16, 10000.0
    q = _randn((T, 1, D), dt, 61, offset=offset)
    k = _randn((T, 1, D), dt, 62, offset=offset)
    pos = torch.tensor([0, 7, 4095], dtype=torch.int32, device="cuda")
    table = gb.rope_table(4096, D, theta)
    qo, ko = gb.rope_fwd(q, k, pos, table)
    torch.cuda.synchronize()
    p = pos.cpu().numpy()
    check_io(to64(qo), oracle.rope_fwd(to64(q), p, theta), "bf16", "q'")
    check_io(to64(ko), oracle.rope_fwd(to64(k), p, theta), "bf16", "k'")


def test_rope_head_size_beyond_the_kernels_is_unsupported():
    # one unit more than either path takes: 513 vector units (bf16, D = 8208) and
    # 513 element units (unaligned, D = 1026)
    lib = gb.library()
    s = torch.cuda.current_stream().cuda_stream
    pos = torch.zeros(1, dtype=torch.int32, device="cuda")
    for D, off in ((8208, 0), (1026, 1)):
        q = _randn((D + 8,), torch.bfloat16, 63)
        table = gb.rope_table(1, D, 10000.0)
        qp = q.data_ptr() + 2 * off
        st = lib.gbln_rope_fwd(qp, None, qp, None, pos.data_ptr(), table.data_ptr(), 1, 1, 1, 0, D,
                               gb.BF16, s)
        assert st == 2, (D, st)  # GBLN_ERR_UNSUPPORTED


def test_rope_table_values():
    D, theta, max_pos = 128, 500000.0, 16384
    table = gb.rope_table(max_pos, D, theta)
    torch.cuda.synchronize()
    tab = table.cpu().numpy().astype(np.float64)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * oracle.rope_inv_freq(D, theta)[None, :]
    # one rounding of the exact value to float32: within half an ulp (2^-24 relative, 2^-25 absolute near 1)
    assert np.max(np.abs(tab[..., 0] - np.cos(ang))) <= 2.0 ** -24
    assert np.max(np.abs(tab[..., 1] - np.sin(ang))) <= 2.0 ** -24
    assert np.array_equal(tab[0, :, 0], np.ones(D // 2)) and np.array_equal(tab[0, :, 1], np.zeros(D // 2))


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_rope_in_place_identity_and_out_of_range(io):
    dt = IO[io]
    T, Hq, Hk, D = 8, 4, 2, 128
    q = _randn((T, Hq, D), dt, 61)
    k = _randn((T, Hk, D), dt, 62)
    q0, k0 = q.clone(), k.clone()
    table = gb.rope_table(100, D, 1e6)
    zeros = torch.zeros(T, dtype=torch.int32, device="cuda")
    gb.rope_fwd(q, k, zeros, table, q_out=q, k_out=k)  # in place, position 0
    torch.cuda.synchronize()
    assert torch.equal(q, q0) and torch.equal(k, k0)
    assert gb.device_error() == 0
    pos = torch.as_tensor([0, 5, 99, 100, -1, 3, 2000, 7], dtype=torch.int32, device="cuda")
    qo, ko = gb.rope_fwd(q, k, pos, table)
    torch.cuda.synchronize()
    bad = [3, 4, 6]
    good = [0, 1, 2, 5, 7]
    assert torch.isnan(qo[bad].float()).all() and torch.isnan(ko[bad].float()).all()
    p = pos.cpu().numpy()[good]
    check_io(to64(qo[good]), oracle.rope_fwd(to64(q0[good]), p, 1e6), io, "q' valid rows")
    # the out-of-range positions are reported through the device error word
    assert gb.device_error(clear=True) == gb.ERR_BAD_POSITION
    assert gb.device_error() == 0
    # the register path (unaligned rows) reports them too
    qu = _randn((T * Hq * D + 1,), dt, 63)[1:].view(T, Hq, D)
    qo2, _ = gb.rope_fwd(qu, None, pos, table)
    torch.cuda.synchronize()
    assert torch.isnan(qo2[bad].float()).all()
    assert gb.device_error(clear=True) == gb.ERR_BAD_POSITION


# ---------------------------------------------------------------------------
# Positions of packed documents
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("lengths", [[1], [5], [1, 1, 1], [3, 1, 7, 2, 1], list(range(1, 60)),
                                     [8192] * 3 + [17]])
def test_positions(lengths):
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    T = int(cu[-1])
    pos = gb.positions_from_cu_seqlens(torch.as_tensor(cu, device="cuda"), T)
    torch.cuda.synchronize()
    assert np.array_equal(pos.cpu().numpy().astype(np.int64), oracle.positions_from_doc_lengths(lengths))


# ---------------------------------------------------------------------------
# SwiGLU
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("T,I", [(1, 1), (3, 13), (2, 8), (5, 4864), (7, 1000), (1, 100003)])
@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("offset", [0, 1])
def test_swiglu_shapes(T, I, io, offset):
    dt = IO[io]
    g = _randn((T, I), dt, 71, scale=3.0, offset=offset)
    u = _randn((T, I), dt, 72, offset=offset)
    d = _randn((T, I), dt, 73, offset=offset)
    out = gb.swiglu_fwd(g, u)
    dg, du = gb.swiglu_bwd(d, g, u)
    torch.cuda.synchronize()
    g64, u64, d64 = to64(g), to64(u), to64(d)
    check_io(to64(out), oracle.swiglu_fwd(g64, u64), io, "out")
    dg_ref, du_ref = oracle.swiglu_bwd(d64, g64, u64)
    check_io(to64(dg), dg_ref, io, "dgate")
    check_io(to64(du), du_ref, io, "dup")


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_swiglu_extremes_and_in_place(io):
    dt = IO[io]
    vals = torch.tensor([0.0, -0.0, 1.0, -1.0, 20.0, -20.0, 80.0, -80.0, 87.0, -87.0, 100.0, -100.0,
                         1e-20, -1e-20, 3.0, -3.0], dtype=dt, device="cuda").repeat(4, 1)
    u = torch.linspace(-2, 2, vals.numel(), device="cuda").view_as(vals).to(dt)
    d = torch.linspace(1, -1, vals.numel(), device="cuda").view_as(vals).to(dt)
    out = gb.swiglu_fwd(vals, u)
    g64, u64, d64 = to64(vals), to64(u), to64(d)
    dg_ref, du_ref = oracle.swiglu_bwd(d64, g64, u64)
    gi, ui = vals.clone(), u.clone()
    gb.swiglu_bwd(d, gi, ui, dgate=gi, dup=ui)  # in place
    torch.cuda.synchronize()
    check_io(to64(out), oracle.swiglu_fwd(g64, u64), io, "out")
    check_io(to64(gi), dg_ref, io, "dgate in place")
    check_io(to64(ui), du_ref, io, "dup in place")


def test_swiglu_guard_bands():
    T, I = 19, 3072
    dt = torch.bfloat16
    g = _randn((T, I), dt, 81)
    u = _randn((T, I), dt, 82)
    d = _randn((T, I), dt, 83)
    go, gdg, gdu = Guarded((T, I), dt), Guarded((T, I), dt), Guarded((T, I), dt)
    gb.swiglu_fwd(g, u, out=go.tensor)
    gb.swiglu_bwd(d, g, u, dgate=gdg.tensor, dup=gdu.tensor)
    torch.cuda.synchronize()
    assert go.intact() and gdg.intact() and gdu.intact()


# bf16 launch paths: warp kernel with one chunk (24 heads of 128) and two chunks
# of head rows per lane (40 heads), TMA-staged kernel with several rows per
# thread and token (72 heads of 128) and one row (24 heads of 96: a head row of
# six 16-byte units, which does not divide a warp), register kernel (unaligned).
ROPE_PATHS = [(16, 8, 128, 0), (32, 8, 128, 0), (64, 8, 128, 0), (16, 8, 96, 0), (3, 1, 130, 1)]


@pytest.mark.parametrize("Hq,Hk,D,offset", ROPE_PATHS)
def test_rope_guard_bands(Hq, Hk, D, offset):
    T, dt = 23, torch.bfloat16
    q = _randn((T, Hq, D), dt, 85, offset=offset)
    k = _randn((T, Hk, D), dt, 86, offset=offset)
    pos = torch.arange(T, dtype=torch.int32, device="cuda")
    table = gb.rope_table(T, D, 1e6)
    gq, gk = Guarded((T, Hq, D), dt), Guarded((T, Hk, D), dt)
    gb.rope_fwd(q, k, pos, table, q_out=gq.tensor, k_out=gk.tensor)
    gdq, gdk = Guarded((T, Hq, D), dt), Guarded((T, Hk, D), dt)
    gb.rope_bwd(q, k, pos, table, dq_in=gdq.tensor, dk_in=gdk.tensor)
    torch.cuda.synchronize()
    assert gq.intact() and gk.intact() and gdq.intact() and gdk.intact()
    check_io(to64(gq.tensor), oracle.rope_fwd(to64(q), pos.cpu().numpy(), 1e6), "bf16", "q' guarded")


def test_layernorm_and_mxfp8_guard_bands():
    T, H, dt = 21, 1024, torch.bfloat16
    x, r, dy = _randn((T, H), dt, 87), _randn((T, H), dt, 88), _randn((T, H), dt, 89)
    w = (1 + 0.1 * _randn((H,), torch.float32, 90)).to(dt)
    gy, gh, gdx = Guarded((T, H), dt), Guarded((T, H), dt), Guarded((T, H), dt)
    gm, gr = Guarded((T,), torch.float32), Guarded((T,), torch.float32)
    y, h, mean, rstd = gb.layernorm_fwd(x, w, 1e-5, r, None, y=gy.tensor, residual_out=gh.tensor,
                                        mean=gm.tensor, rstd=gr.tensor)
    dx, part, P = gb.layernorm_bwd(dy, h, w, mean, rstd, None, dx=gdx.tensor)
    lib = gb.library()
    gq, gs = Guarded((T, H), torch.uint8), Guarded((T, H // 32), torch.uint8)
    gh2, gr2 = Guarded((T, H), dt), Guarded((T,), torch.float32)
    st = lib.gbln_rmsnorm_fwd_mxfp8(x.data_ptr(), r.data_ptr(), w.data_ptr(), None, gq.tensor.data_ptr(),
                                    gs.tensor.data_ptr(), gh2.tensor.data_ptr(), gr2.tensor.data_ptr(), T, H,
                                    1e-5, gb.BF16, gb.BF16, torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    for g in (gy, gh, gdx, gm, gr, gq, gs, gh2, gr2):
        assert g.intact()


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("Hq,Hk", [(32, 8), (64, 8)])
def test_rope_out_of_range_with_cos_sin_in_registers(io, Hq, Hk):
    # Threads that rotate several head rows per token hold the token's cos/sin
    # in registers (the warp kernel at 40 heads; with bf16 at 72 heads the
    # staged kernel); a bad position must still give NaN rows and the error
    # bit, and the other tokens the exact rotation.
    dt = IO[io]
    T, D = 9, 128
    q = _randn((T, Hq, D), dt, 71)
    k = _randn((T, Hk, D), dt, 72)
    table = gb.rope_table(50, D, 1e6)
    pos = torch.as_tensor([0, 49, 50, 7, -3, 1, 2, 3, 4], dtype=torch.int32, device="cuda")
    assert gb.device_error() == 0
    qo, ko = gb.rope_fwd(q, k, pos, table)
    dq, dk = gb.rope_bwd(q, k, pos, table)
    torch.cuda.synchronize()
    bad, good = [2, 4], [0, 1, 3, 5, 6, 7, 8]
    for t in (qo, ko, dq, dk):
        assert torch.isnan(t[bad].float()).all()
    p = pos.cpu().numpy()[good]
    check_io(to64(qo[good]), oracle.rope_fwd(to64(q[good]), p, 1e6), io, "q' valid rows")
    check_io(to64(dk[good]), oracle.rope_bwd(to64(k[good]), p, 1e6), io, "dk valid rows")
    assert gb.device_error(clear=True) == gb.ERR_BAD_POSITION


def test_wait_timeout_is_reported_and_the_context_stays_usable():
    # A bounded wait that nothing will satisfy runs out (no fault, no hang): the
    # error word gets the timeout bit, and the next calls run normally.
    assert gb.device_error() == 0
    gb.selftest_wait_timeout(256)
    torch.cuda.synchronize()
    assert gb.device_error() == gb.ERR_WAIT_TIMEOUT
    assert gb.device_error(clear=True) == gb.ERR_WAIT_TIMEOUT
    assert gb.device_error() == 0
    T, Hq, Hk, D = 64, 16, 8, 128
    q = _randn((T, Hq, D), torch.bfloat16, 95)
    k = _randn((T, Hk, D), torch.bfloat16, 96)
    pos = torch.arange(T, dtype=torch.int32, device="cuda")
    table = gb.rope_table(T, D, 1e6)
    qo, ko = gb.rope_fwd(q, k, pos, table)
    torch.cuda.synchronize()
    assert gb.device_error() == 0
    check_io(to64(qo), oracle.rope_fwd(to64(q), pos.cpu().numpy(), 1e6), "bf16", "q' after timeout")


@pytest.mark.parametrize("Hq,Hk,D", [(64, 8, 128), (16, 8, 96)])
def test_device_error_word_is_clear_after_staged_kernels(Hq, Hk, D):
    # RoPE's staged path (72 heads of 128; 24 heads of 96) bounds its waits on
    # TMA copies; none may have given up.
    T = 4097
    q = _randn((T, Hq, D), torch.bfloat16, 91)
    k = _randn((T, Hk, D), torch.bfloat16, 92)
    pos = torch.arange(T, dtype=torch.int32, device="cuda") % 1000
    table = gb.rope_table(1000, D, 5e5)
    qo, ko = gb.rope_fwd(q, k, pos, table)
    torch.cuda.synchronize()
    assert gb.device_error() == 0
    p = pos.cpu().numpy()
    rows = [0, 1, 2047, 4095, 4096]
    check_io(to64(qo[rows]), oracle.rope_fwd(to64(q[rows]), p[rows], 5e5), "bf16", "q' staged")
    check_io(to64(ko[rows]), oracle.rope_fwd(to64(k[rows]), p[rows], 5e5), "bf16", "k' staged")
