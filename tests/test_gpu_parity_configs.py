"""GPU vs oracle parity on the five layer workloads, at full size.

The CUDA path is called through the C ABI (via the ctypes binding) on the same
full-size tensors and with the same entry points and launch shapes that
``bench.py`` times.  The float64 CPU oracle then checks:
  * the residual-stream output h bit-exactly on every row, and the weight
    gradient dW (a sum over every row) against the oracle's full sum;
  * y, rstd, dx, RoPE and SwiGLU outputs on every row of the two small
    workloads, and on a seeded sample of rows (plus the first and last row and
    every document start) of the three large ones;
  * positions of packed documents bit-exactly on every token.
Tolerances are those of ``_checks``.
"""

import numpy as np
import pytest
import torch

import oracle
import rmsnorm_fwd_bwd_03_gb300 as gb
from rmsnorm_fwd_bwd_03_gb300.workload import ORDER, WORKLOADS, make_inputs

from _checks import check_dw, check_io, check_rstd, dx_scale, sample_rows, to64

pytestmark = pytest.mark.gpu

FULL = {"qwen05b_tiny_f32", "qwen3_0p6b"}
SAMPLE_ROWS = 4096
CHUNK = 2048


@pytest.fixture(scope="module", autouse=True)
def _library():
    from rmsnorm_fwd_bwd_03_gb300._build import build_library
    build_library()
    gb.library()
    yield
    torch.cuda.empty_cache()


def _rows(wl):
    if wl.name in FULL:
        return np.arange(wl.T)
    extra = wl.cu_seqlens()[:-1] if wl.packed else ()
    return sample_rows(wl.T, SAMPLE_ROWS, extra=extra)


@pytest.mark.parametrize("name", ORDER)
def test_rmsnorm_fwd_bwd(name):
    wl = WORKLOADS[name]
    inp = make_inputs(wl, "cuda", parts=("rmsnorm",))
    x, r, w, dy, dres = inp["x"], inp["residual"], inp["weight"], inp["dy"], inp["dres"]
    y, h, rstd = gb.rmsnorm_fwd(x, w, wl.eps, r)
    dx, part, P = gb.rmsnorm_bwd(dy, h, w, rstd, dres)
    dw = gb.rmsnorm_dw_finalize(part, P)
    torch.cuda.synchronize()

    w64 = to64(w)
    # h bit-exact and dW over every row, streamed in chunks.
    dw_ref = np.zeros(wl.H)
    for t0 in range(0, wl.T, CHUNK):
        sl = slice(t0, t0 + CHUNK)
        _, h_ref, _ = oracle.rmsnorm_fwd(to64(x[sl]), to64(r[sl]), w64, wl.eps, io=wl.io)
        assert np.array_equal(to64(h[sl]), h_ref), f"h differs in rows {t0}..{t0 + CHUNK}"
        dw_ref += oracle.rmsnorm_dw(to64(dy[sl]), h_ref, wl.eps)
    check_dw(to64(dw), dw_ref)

    rows = torch.as_tensor(_rows(wl), device="cuda")
    x_s, r_s, dy_s, dres_s = (to64(t.index_select(0, rows)) for t in (x, r, dy, dres))
    y_ref, h_ref, rstd_ref = oracle.rmsnorm_fwd(x_s, r_s, w64, wl.eps, io=wl.io)
    check_io(to64(y.index_select(0, rows)), y_ref, wl.io, f"{name} y")
    check_rstd(to64(rstd.index_select(0, rows)), rstd_ref, f"{name} rstd")
    dx_ref, _ = oracle.rmsnorm_bwd(dy_s, dres_s, h_ref, w64, wl.eps)
    check_io(to64(dx.index_select(0, rows)), dx_ref, wl.io, f"{name} dx",
             scale=dx_scale(dy_s, w64, rstd_ref, dres_s))


@pytest.mark.parametrize("name", ORDER)
def test_rope_fwd_bwd(name):
    wl = WORKLOADS[name]
    inp = make_inputs(wl, "cuda", parts=("rope",))
    cu = inp["cu_seqlens"]
    pos = gb.positions_from_cu_seqlens(cu, wl.T)
    table = gb.rope_table(wl.max_pos(), wl.D, wl.theta)
    qo, ko = gb.rope_fwd(inp["q"], inp["k"], pos, table)
    dqi, dki = gb.rope_bwd(inp["dq"], inp["dk"], pos, table)
    torch.cuda.synchronize()

    pos_ref = oracle.positions_from_cu_seqlens(cu.cpu().numpy())
    assert np.array_equal(pos.cpu().numpy().astype(np.int64), pos_ref)

    rows_np = _rows(wl)
    rows = torch.as_tensor(rows_np, device="cuda")
    p_s = pos_ref[rows_np]
    for src, out, fn, what in ((inp["q"], qo, oracle.rope_fwd, "q'"), (inp["k"], ko, oracle.rope_fwd, "k'"),
                               (inp["dq"], dqi, oracle.rope_bwd, "dq"), (inp["dk"], dki, oracle.rope_bwd, "dk")):
        ref = fn(to64(src.index_select(0, rows)), p_s, wl.theta)
        check_io(to64(out.index_select(0, rows)), ref, wl.io, f"{name} {what}")


@pytest.mark.parametrize("name", ORDER)
def test_swiglu_fwd_bwd(name):
    wl = WORKLOADS[name]
    inp = make_inputs(wl, "cuda", parts=("swiglu",))
    g, u, d = inp["gate"], inp["up"], inp["dout"]
    out = gb.swiglu_fwd(g, u)
    dg, du = gb.swiglu_bwd(d, g, u)
    torch.cuda.synchronize()
    rows = torch.as_tensor(_rows(wl), device="cuda")
    g_s, u_s, d_s = (to64(t.index_select(0, rows)) for t in (g, u, d))
    check_io(to64(out.index_select(0, rows)), oracle.swiglu_fwd(g_s, u_s), wl.io, f"{name} out")
    dg_ref, du_ref = oracle.swiglu_bwd(d_s, g_s, u_s)
    check_io(to64(dg.index_select(0, rows)), dg_ref, wl.io, f"{name} dgate")
    check_io(to64(du.index_select(0, rows)), du_ref, wl.io, f"{name} dup")
