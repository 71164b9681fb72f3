"""GPU vs oracle for the MXFP8 outputs (E4M3 codes with one E8M0 scale per 32
values of a row): the RMSNorm forward and the gated-unit forward that deliver
their result as the next GEMM's FP8 operand.  Codes and scales are compared
with ``_checks.check_mxfp8`` (identical wherever the float32 bound cannot move
a decision); the other outputs of the RMSNorm entry must be bit-identical to
those of ``gbln_rmsnorm_fwd``, which has its own parity tests."""

import numpy as np
import pytest
import torch

import oracle
import rmsnorm_fwd_bwd_03_gb300 as gb

from _checks import check_mxfp8, to64

pytestmark = pytest.mark.gpu

IO = {"f32": torch.float32, "bf16": torch.bfloat16}


@pytest.fixture(scope="module", autouse=True)
def _library():
    from rmsnorm_fwd_bwd_03_gb300._build import build_library
    build_library()
    gb.library()


def _randn(shape, dtype, seed, scale=1.0):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return (torch.randn(shape, generator=g, device="cuda") * scale).to(dtype)


def _weight(H, dtype, seed):
    return (1 + 0.1 * _randn((H,), torch.float32, seed)).to(dtype)


def _rms_case(T, H, io, wt, residual, want_y, x=None, r=None, w=None, seed=0):
    dt = IO[io]
    x = _randn((T, H), dt, seed + 1) if x is None else x
    r = (_randn((T, H), dt, seed + 2) if r is None else r) if residual else None
    w = _weight(H, IO[wt], seed + 3) if w is None else w
    eps = 1e-6
    y, q, sc, h, rstd = gb.rmsnorm_fwd_mxfp8(x, w, eps, r, want_y=want_y)
    y0, h0, rstd0 = gb.rmsnorm_fwd(x, w, eps, r)
    torch.cuda.synchronize()
    # everything but the MXFP8 copy is what the plain forward writes
    assert torch.equal(h, h0) and torch.equal(rstd, rstd0)
    if want_y:
        assert torch.equal(y, y0)
    else:
        assert y is None
    codes, scales, y64, _, _ = oracle.rmsnorm_fwd_mxfp8(to64(x), None if r is None else to64(r),
                                                        to64(w), eps, io)
    check_mxfp8(q, sc, y64, f"rmsnorm mxfp8 T={T} H={H} {io}/{wt}")
    return q, sc


# H: warp-per-row widths (32 .. 1024), CTA-per-row widths (2048 .. 8192 bf16),
# and a width beyond the register path (element-wise kernel).
@pytest.mark.parametrize("io,wt", [("bf16", "bf16"), ("bf16", "f32"), ("f32", "f32")])
@pytest.mark.parametrize("T,H", [(1, 32), (37, 64), (129, 896), (64, 1024), (9, 4096), (5, 8192), (3, 17408)])
@pytest.mark.parametrize("residual", [True, False])
def test_rmsnorm_fwd_mxfp8(io, wt, T, H, residual):
    _rms_case(T, H, io, wt, residual, want_y=(T % 2 == 1))


@pytest.mark.parametrize("io", ["bf16", "f32"])
def test_rmsnorm_fwd_mxfp8_unaligned(io):
    # x one element past a 16-byte boundary: the element-wise kernel
    dt = IO[io]
    T, H = 19, 96
    buf = _randn((T * H + 1,), dt, 7)
    x = buf[1:].view(T, H)
    _rms_case(T, H, io, io, False, want_y=True, x=x)


def test_rmsnorm_fwd_mxfp8_outliers_and_zero_rows():
    # 1% of the channels scaled x50 (the packed-document workload's recipe) and
    # two all-zero rows: blocks holding an outlier get a large scale, the rest a
    # small one; a zero block gets scale byte 0 and zero codes.
    T, H = 64, 4096
    x = _randn((T, H), torch.float32, 11)
    cols = torch.randperm(H, generator=torch.Generator().manual_seed(0))[: round(0.01 * H)]
    x[:, cols.cuda()] *= 50
    x[5] = 0
    x[40] = 0
    x = x.to(torch.bfloat16)
    q, sc = _rms_case(T, H, "bf16", "bf16", False, want_y=True, x=x)
    assert torch.all(sc[5] == 0) and torch.all(q[5] == 0)
    assert torch.all(sc[40] == 0) and torch.all(q[40] == 0)


def test_rmsnorm_fwd_mxfp8_saturates_top_of_block():
    # A block whose largest value has a significand above 1.75: value / 2^e > 448,
    # so it saturates to 448 (code 0x7e) while the scale stays floor(log2) - 8.
    H = 64
    x = torch.zeros((1, H), dtype=torch.float32, device="cuda")
    x[0, 3] = 1.9
    x[0, 40] = 1.0
    w = torch.ones(H, dtype=torch.float32, device="cuda")
    _, q, sc, _, rstd = gb.rmsnorm_fwd_mxfp8(x, w, 0.0, None, want_y=False)
    torch.cuda.synchronize()
    y3 = 1.9 * rstd[0].item()
    se = int(np.floor(np.log2(y3))) - 8
    assert sc[0, 0].item() == se + 127
    assert q[0, 3].item() == 0x7E


def _glu_check(act, io, g, u, q, sc, what):
    ref = oracle.glu_fwd(act, to64(g), to64(u))
    # GeLU-erf cancels for x << 0: 0.5 x (1 + erf(x / sqrt 2)) carries an absolute
    # float32 error of about |x u| * 2^-23 (erff is accurate to 2 ulp).  Emulated
    # in float32 on these inputs it stays below 2.1e-7 of the block maximum, so
    # an absolute term of 1e-6 of the block maximum covers it; with that window
    # a few percent of the (small) codes become two-way cases.
    if act == "gelu_erf":
        check_mxfp8(q, sc, ref, what, abs_rel=1e-6, max_ambiguous=0.05)
    else:
        check_mxfp8(q, sc, ref, what)


@pytest.mark.parametrize("act", ["silu", "gelu_tanh", "gelu_erf", "relu"])
@pytest.mark.parametrize("io", ["bf16", "f32"])
@pytest.mark.parametrize("T,I", [(1, 32), (37, 3072), (66, 14336)])
def test_glu_fwd_mxfp8_contiguous(act, io, T, I):
    dt = IO[io]
    g, u = _randn((T, I), dt, 21, 3.0), _randn((T, I), dt, 22)
    q, sc = gb.glu_fwd_mxfp8(g, u, act)
    torch.cuda.synchronize()
    _glu_check(act, io, g, u, q, sc, f"glu mxfp8 {act} {io} T={T} I={I}")


@pytest.mark.parametrize("io", ["bf16", "f32"])
@pytest.mark.parametrize("T,I", [(33, 3072), (5, 96), (9, 3584), (6, 2560)])
def test_glu_fwd_mxfp8_packed_halves(io, T, I):
    dt = IO[io]
    packed = _randn((T, 2 * I), dt, 23, 2.0)
    g, u = packed[:, :I], packed[:, I:]
    q, sc = gb.glu_fwd_mxfp8(g, u, "silu")
    torch.cuda.synchronize()
    _glu_check("silu", io, g, u, q, sc, f"glu mxfp8 packed {io}")


def test_glu_fwd_mxfp8_unaligned_rows():
    # row stride 2I + 1 elements: not a multiple of the vector width -> element-wise kernel
    T, I = 17, 64
    buf = _randn((T, 2 * I + 1), torch.bfloat16, 25)
    g, u = buf[:, :I], buf[:, I:2 * I]
    q, sc = gb.glu_fwd_mxfp8(g, u, "silu")
    torch.cuda.synchronize()
    _glu_check("silu", "bf16", g, u, q, sc, "glu mxfp8 unaligned")


def test_mxfp8_entries_reject_bad_widths_and_accept_empty():
    lib = gb.library()
    x = torch.zeros((2, 48), dtype=torch.bfloat16, device="cuda")
    w = torch.ones(48, dtype=torch.bfloat16, device="cuda")
    q = torch.empty((2, 48), dtype=torch.uint8, device="cuda")
    sc = torch.empty((2, 2), dtype=torch.uint8, device="cuda")
    rs = torch.empty(2, dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert lib.gbln_rmsnorm_fwd_mxfp8(x.data_ptr(), None, w.data_ptr(), None, q.data_ptr(), sc.data_ptr(),
                                      None, rs.data_ptr(), 2, 48, 1e-6, gb.BF16, gb.BF16, s) == 1
    assert lib.gbln_glu_fwd_mxfp8(x.data_ptr(), x.data_ptr(), q.data_ptr(), sc.data_ptr(), 2, 48, 48, 48,
                                  0, gb.BF16, s) == 1
    assert lib.gbln_rmsnorm_fwd_mxfp8(None, None, None, None, None, None, None, None, 0, 64, 1e-6,
                                      gb.BF16, gb.BF16, s) == 0
    assert lib.gbln_glu_fwd_mxfp8(None, None, None, None, 0, 64, 64, 64, 0, gb.BF16, s) == 0
    assert gb.device_error() == 0
