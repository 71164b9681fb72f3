"""The operators beyond the step at full workload sizes, in the launch
configuration `bench.py --next` times: the gated unit with every activation on
a packed [T, 2I] gate|up tensor (forward, and backward into a packed gradient),
the plain GeLU-tanh, RoPE rotated in place inside a packed QKV tensor and with
interleaved pairing, LayerNorm forward (residual + bias) and backward (dres;
dW and dB), and the MXFP8 outputs of the RMSNorm and SwiGLU forwards.

Seeded rows (plus the first and last) are compared with the oracle; the
LayerNorm dW and dB against the oracle's sums over every row, streamed in
chunks.  Tolerances are those of ``_checks``."""

import numpy as np
import pytest
import torch

import oracle
import rmsnorm_fwd_bwd_03_gb300 as gb
from rmsnorm_fwd_bwd_03_gb300.workload import WORKLOADS

from _checks import check_dw, check_io, check_mxfp8, check_rstd, sample_rows, to64

pytestmark = pytest.mark.gpu

ACTS = ["silu", "gelu_tanh", "gelu_erf", "relu"]
SAMPLE = 256
CHUNK = 4096


@pytest.fixture(scope="module", autouse=True)
def _library():
    from rmsnorm_fwd_bwd_03_gb300._build import build_library
    build_library()
    gb.library()


def _rnd(g, *shape):
    return torch.randn(shape, generator=g, device="cuda").to(torch.bfloat16)


def _sampled(t, rows):
    return t.index_select(0, rows)


@pytest.mark.parametrize("name", ["qwen3_0p6b", "llama3_8b", "llama70b_width"])
def test_gated_units_full_size(name):
    wl = WORKLOADS[name]
    T, I = wl.T, wl.I
    g = torch.Generator(device="cuda").manual_seed(0)
    packed, dout = _rnd(g, T, 2 * I), _rnd(g, T, I)
    gate, up = packed[:, :I], packed[:, I:]
    rows = torch.as_tensor(sample_rows(T, SAMPLE), device="cuda")
    g64, u64, d64 = (to64(_sampled(t, rows)) for t in (gate, up, dout))
    grad = torch.empty((T, 2 * I), dtype=torch.bfloat16, device="cuda")
    for act in ACTS:
        out = gb.glu_fwd(gate, up, act)
        gb.glu_bwd(dout, gate, up, act, dgate=grad[:, :I], dup=grad[:, I:])
        torch.cuda.synchronize()
        check_io(to64(_sampled(out, rows)), oracle.glu_fwd(act, g64, u64), "bf16", f"{name} {act} out")
        dg_ref, du_ref = oracle.glu_bwd(act, d64, g64, u64)
        gs = _sampled(grad, rows)
        check_io(to64(gs[:, :I]), dg_ref, "bf16", f"{name} {act} dgate")
        check_io(to64(gs[:, I:]), du_ref, "bf16", f"{name} {act} dup")
    # SwiGLU forward with only the MXFP8 copy of its output
    q, sc = gb.glu_fwd_mxfp8(gate, up, "silu")
    torch.cuda.synchronize()
    check_mxfp8(_sampled(q, rows), _sampled(sc, rows), oracle.glu_fwd("silu", g64, u64),
                f"{name} swiglu mxfp8")
    # plain GeLU-tanh over a [T, I] activation
    x, dy = _rnd(g, T, I), _rnd(g, T, I)
    y = gb.act_fwd(x, "gelu_tanh")
    dx = gb.act_bwd(dy, x, "gelu_tanh")
    torch.cuda.synchronize()
    x64 = to64(_sampled(x, rows))
    check_io(to64(_sampled(y, rows)), oracle.act("gelu_tanh", x64), "bf16", f"{name} gelu_tanh")
    check_io(to64(_sampled(dx, rows)), to64(_sampled(dy, rows)) * oracle.act_grad("gelu_tanh", x64), "bf16",
             f"{name} gelu_tanh grad")


@pytest.mark.parametrize("name", ["qwen3_0p6b", "llama3_8b", "llama70b_width"])
def test_rope_strided_and_interleaved_full_size(name):
    wl = WORKLOADS[name]
    T, Hq, Hk, D = wl.T, wl.Hq, wl.Hk, wl.D
    g = torch.Generator(device="cuda").manual_seed(1)
    cu = torch.as_tensor(wl.cu_seqlens(), dtype=torch.int32, device="cuda")
    pos = gb.positions_from_cu_seqlens(cu, T)
    table = gb.rope_table(wl.max_pos(), D, wl.theta)
    starts = wl.cu_seqlens()[:-1]
    rows = torch.as_tensor(sample_rows(T, SAMPLE, extra=starts), device="cuda")
    p = pos.cpu().numpy()[rows.cpu().numpy()]
    # Q and K rotated in place inside one packed [T, (Hq + 2 Hk) D] QKV tensor
    W = (Hq + 2 * Hk) * D
    qkv = _rnd(g, T, W)
    orig = to64(_sampled(qkv, rows))
    q, k = qkv[:, :Hq * D].view(T, Hq, D), qkv[:, Hq * D:(Hq + Hk) * D].view(T, Hk, D)
    gb.rope_fwd_ex(q, k, pos, table, q_out=q, k_out=k)
    torch.cuda.synchronize()
    now = to64(_sampled(qkv, rows))
    n = len(p)
    check_io(now[:, :Hq * D].reshape(n, Hq, D), oracle.rope_fwd(orig[:, :Hq * D].reshape(n, Hq, D), p, wl.theta),
             "bf16", f"{name} q in packed qkv")
    check_io(now[:, Hq * D:(Hq + Hk) * D].reshape(n, Hk, D),
             oracle.rope_fwd(orig[:, Hq * D:(Hq + Hk) * D].reshape(n, Hk, D), p, wl.theta), "bf16",
             f"{name} k in packed qkv")
    assert np.array_equal(now[:, (Hq + Hk) * D:], orig[:, (Hq + Hk) * D:]), "V changed"
    # interleaved pairing on separate Q and K
    q2, k2 = _rnd(g, T, Hq, D), _rnd(g, T, Hk, D)
    qo, ko = gb.rope_fwd_ex(q2, k2, pos, table, pairing="interleaved")
    torch.cuda.synchronize()
    check_io(to64(_sampled(qo, rows)), oracle.rope_fwd(to64(_sampled(q2, rows)), p, wl.theta, "interleaved"),
             "bf16", f"{name} q interleaved")
    check_io(to64(_sampled(ko, rows)), oracle.rope_fwd(to64(_sampled(k2, rows)), p, wl.theta, "interleaved"),
             "bf16", f"{name} k interleaved")


@pytest.mark.parametrize("name", ["qwen3_0p6b", "llama3_8b", "llama70b_width"])
def test_layernorm_and_mxfp8_rmsnorm_full_size(name):
    wl = WORKLOADS[name]
    T, H, eps = wl.T, wl.H, wl.eps
    g = torch.Generator(device="cuda").manual_seed(2)
    x, r, dy, dres = (_rnd(g, T, H) for _ in range(4))
    w = (1 + 0.1 * torch.randn(H, generator=g, device="cuda")).to(torch.bfloat16)
    b = _rnd(g, H)
    y, h, mean, rstd = gb.layernorm_fwd(x, w, eps, r, b)
    dx, part, P = gb.layernorm_bwd(dy, h, w, mean, rstd, dres)
    dw, db = gb.layernorm_dwdb_finalize(part, P)
    torch.cuda.synchronize()
    rows = torch.as_tensor(sample_rows(T, SAMPLE), device="cuda")
    w64, b64 = to64(w), to64(b)
    y_ref, h_ref, mean_ref, rstd_ref = oracle.layernorm_fwd(to64(_sampled(x, rows)), to64(_sampled(r, rows)), w64,
                                                            b64, eps, io="bf16")
    assert np.array_equal(to64(_sampled(h, rows)), h_ref), f"{name}: residual output differs"
    check_io(to64(_sampled(y, rows)), y_ref, "bf16", f"{name} layernorm y")
    check_rstd(to64(_sampled(rstd, rows)), rstd_ref, f"{name} layernorm rstd")
    assert np.allclose(to64(_sampled(mean, rows)), mean_ref, rtol=1e-5, atol=1e-6 * np.max(np.abs(h_ref)))
    dx_ref, _, _ = oracle.layernorm_bwd(to64(_sampled(dy, rows)), to64(_sampled(dres, rows)), h_ref, w64, eps)
    check_io(to64(_sampled(dx, rows)), dx_ref, "bf16", f"{name} layernorm dx")
    # dW and dB over every row, from the GPU's h (bit-exact against the oracle above)
    dw_ref, db_ref = np.zeros(H), np.zeros(H)
    for t0 in range(0, T, CHUNK):
        sl = slice(t0, t0 + CHUNK)
        _, dwc, dbc = oracle.layernorm_bwd(to64(dy[sl]), None, to64(h[sl]), w64, eps)
        dw_ref += dwc
        db_ref += dbc
    check_dw(to64(dw), dw_ref, f"{name} layernorm dW")
    check_dw(to64(db), db_ref, f"{name} layernorm dB")
    # RMSNorm forward writing y only as MXFP8 (residual add, h and rstd as usual)
    _, q8, sc8, h2, rstd2 = gb.rmsnorm_fwd_mxfp8(x, w, eps, r, want_y=False)
    torch.cuda.synchronize()
    codes, scales, y64, hh, _ = oracle.rmsnorm_fwd_mxfp8(to64(_sampled(x, rows)), to64(_sampled(r, rows)), w64,
                                                         eps, "bf16")
    assert np.array_equal(to64(_sampled(h2, rows)), hh)
    check_mxfp8(_sampled(q8, rows), _sampled(sc8, rows), y64, f"{name} rmsnorm mxfp8")
