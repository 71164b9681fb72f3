"""GPU vs oracle for LayerNorm with fused residual add: forward (y, h, mean,
rstd) and backward (dx, dW, dB), across widths, dtypes, alignment and the
optional residual / bias / residual-gradient inputs; dW|dB bitwise reproducible."""

import numpy as np
import pytest
import torch

import oracle
import rmsnorm_fwd_bwd_03_gb300 as gb

from _checks import check_dw, check_io, check_rstd, dx_scale, to64

pytestmark = pytest.mark.gpu

IO = {"f32": torch.float32, "bf16": torch.bfloat16}


@pytest.fixture(scope="module", autouse=True)
def _library():
    from rmsnorm_fwd_bwd_03_gb300._build import build_library
    build_library()
    gb.library()


def _randn(shape, dtype, seed, scale=1.0, shift=0.0, offset=0):
    g = torch.Generator(device="cuda").manual_seed(seed)
    n = int(np.prod(shape))
    buf = torch.randn(n + offset, generator=g, device="cuda") * scale + shift
    return buf.to(dtype)[offset:].view(shape)


@pytest.mark.parametrize("T,H", [(1, 1), (3, 13), (5, 8), (7, 896), (33, 1000), (2, 1024), (17, 4100),
                                 (6, 8192), (3, 16384), (2, 20000), (300, 64)])
@pytest.mark.parametrize("io,wt", [("f32", "f32"), ("bf16", "bf16"), ("bf16", "f32")])
@pytest.mark.parametrize("opts", ["res+bias", "plain", "res"])
@pytest.mark.parametrize("offset", [0, 1])
def test_layernorm_shapes(T, H, io, wt, opts, offset):
    dt, wdt = IO[io], IO[wt]
    eps = 1e-5
    residual = "res" in opts
    with_bias = "bias" in opts
    x = _randn((T, H), dt, 1, 2.0, 0.5, offset)
    r = _randn((T, H), dt, 2, offset=offset) if residual else None
    w = (1 + 0.1 * _randn((H,), torch.float32, 3)).to(wdt)
    b = _randn((H,), torch.float32, 4).to(wdt) if with_bias else None
    dy = _randn((T, H), dt, 5, offset=offset)
    dres = _randn((T, H), dt, 6, offset=offset) if residual else None
    y, h, mean, rstd = gb.layernorm_fwd(x, w, eps, r, b)
    dx, part, P = gb.layernorm_bwd(dy, h, w, mean, rstd, dres)
    dw, db = gb.layernorm_dwdb_finalize(part, P)
    torch.cuda.synchronize()
    w64 = to64(w)
    b64 = None if b is None else to64(b)
    y_ref, h_ref, mean_ref, rstd_ref = oracle.layernorm_fwd(to64(x), None if r is None else to64(r), w64, b64,
                                                            eps, io=io)
    if residual:
        assert np.array_equal(to64(h), h_ref)
    check_io(to64(y), y_ref, io, "y")
    check_rstd(to64(rstd), rstd_ref)
    assert np.allclose(to64(mean), mean_ref, rtol=1e-5, atol=1e-6 * np.max(np.abs(h_ref)))
    dres64 = None if dres is None else to64(dres)
    dx_ref, dw_ref, db_ref = oracle.layernorm_bwd(to64(dy), dres64, h_ref, w64, eps)
    check_io(to64(dx), dx_ref, io, "dx", scale=dx_scale(to64(dy), w64, rstd_ref, dres64, terms=3))
    if H > 1:
        check_dw(to64(dw), dw_ref, "dW")
    else:
        assert abs(to64(dw)[0]) <= 1e-3 * max(1.0, np.abs(to64(dy)).sum())
    check_dw(to64(db), db_ref, "dB")


def test_layernorm_largest_row():
    # H = 2^24, the largest accepted width: element-wise kernels with long
    # per-thread sums (compensated), one partial row.
    T, H = 1, 1 << 24
    dt = torch.bfloat16
    x = _randn((T, H), dt, 21, 2.0, 0.5)
    r = _randn((T, H), dt, 22)
    w = (1 + 0.1 * _randn((H,), torch.float32, 23))
    b = _randn((H,), torch.float32, 24)
    dy = _randn((T, H), dt, 25)
    y, h, mean, rstd = gb.layernorm_fwd(x, w, 1e-5, r, b)
    dx, part, P = gb.layernorm_bwd(dy, h, w, mean, rstd)
    dw, db = gb.layernorm_dwdb_finalize(part, P)
    torch.cuda.synchronize()
    y_ref, h_ref, mean_ref, rstd_ref = oracle.layernorm_fwd(to64(x), to64(r), to64(w), to64(b), 1e-5, io="bf16")
    assert np.array_equal(to64(h), h_ref)
    check_io(to64(y), y_ref, "bf16", "y")
    check_rstd(to64(rstd), rstd_ref)
    assert np.allclose(to64(mean), mean_ref, rtol=1e-5, atol=1e-6 * np.max(np.abs(h_ref)))
    dx_ref, dw_ref, db_ref = oracle.layernorm_bwd(to64(dy), None, h_ref, to64(w), 1e-5)
    check_io(to64(dx), dx_ref, "bf16", "dx")
    check_dw(to64(dw), dw_ref, "dW")
    check_dw(to64(db), db_ref, "dB")


@pytest.mark.parametrize("H", [1024, 4096])  # grouped row blocks; one block per row
def test_layernorm_llama_width_deterministic_and_accumulate(H):
    T = 4099
    dt = torch.bfloat16
    x = _randn((T, H), dt, 11)
    x[:, ::100] *= 50  # outlier channels
    r = _randn((T, H), dt, 12)
    w = (1 + 0.1 * _randn((H,), torch.float32, 13)).to(dt)
    b = _randn((H,), torch.float32, 14).to(dt)
    dy = _randn((T, H), dt, 15)
    y, h, mean, rstd = gb.layernorm_fwd(x, w, 1e-5, r, b)
    outs = []
    for _ in range(2):
        dx, part, P = gb.layernorm_bwd(dy, h, w, mean, rstd)
        dw, db = gb.layernorm_dwdb_finalize(part, P)
        outs.append((dx.clone(), dw.clone(), db.clone()))
    dw2, db2 = gb.layernorm_dwdb_finalize(part, P, dw=outs[0][1].clone(), db=outs[0][2].clone(), accumulate=True)
    torch.cuda.synchronize()
    assert all(torch.equal(a, b) for a, b in zip(outs[0], outs[1]))
    assert torch.allclose(dw2, 2 * outs[0][1], rtol=1e-6) and torch.allclose(db2, 2 * outs[0][2], rtol=1e-6)
    rows = torch.as_tensor(np.random.default_rng(0).choice(T, 512, replace=False), device="cuda")
    y_ref, h_ref, _, rstd_ref = oracle.layernorm_fwd(to64(x[rows]), to64(r[rows]), to64(w), to64(b), 1e-5,
                                                     io="bf16")
    check_io(to64(y[rows]), y_ref, "bf16", "y sampled")
    dx_ref, _, _ = oracle.layernorm_bwd(to64(dy[rows]), None, h_ref, to64(w), 1e-5)
    check_io(to64(outs[0][0][rows]), dx_ref, "bf16", "dx sampled")
    _, dw_ref, db_ref = oracle.layernorm_bwd(to64(dy), None, to64(h), to64(w), 1e-5)
    check_dw(to64(outs[0][1]), dw_ref, "dW")
    check_dw(to64(outs[0][2]), db_ref, "dB")
