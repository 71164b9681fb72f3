"""GPU vs oracle for the gated units with every activation (SiLU, GeLU in tanh
and erf form, ReLU), in contiguous, packed-[T, 2I] and unaligned layouts, and
for the plain activations.  Tolerances are those of ``_checks``."""

import pytest
import torch

import oracle
import rmsnorm_fwd_bwd_03_gb300 as gb

from _checks import check_io, to64

pytestmark = pytest.mark.gpu

IO = {"f32": torch.float32, "bf16": torch.bfloat16}
ACTS = ["silu", "gelu_tanh", "gelu_erf", "relu"]


@pytest.fixture(scope="module", autouse=True)
def _library():
    from rmsnorm_fwd_bwd_03_gb300._build import build_library
    build_library()
    gb.library()


def _randn(shape, dtype, seed, scale=1.0):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return (torch.randn(shape, generator=g, device="cuda") * scale).to(dtype)


def _check_glu(act, io, g, u, d, out, dg, du):
    g64, u64, d64 = to64(g), to64(u), to64(d)
    check_io(to64(out), oracle.glu_fwd(act, g64, u64), io, f"{act} out")
    dg_ref, du_ref = oracle.glu_bwd(act, d64, g64, u64)
    check_io(to64(dg), dg_ref, io, f"{act} dgate")
    check_io(to64(du), du_ref, io, f"{act} dup")


@pytest.mark.parametrize("act", ACTS)
@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("T,I", [(1, 8), (37, 3072), (5, 13), (64, 14336)])
def test_glu_contiguous(act, io, T, I):
    dt = IO[io]
    g, u, d = _randn((T, I), dt, 1, 3.0), _randn((T, I), dt, 2), _randn((T, I), dt, 3)
    out = gb.glu_fwd(g, u, act)
    dg, du = gb.glu_bwd(d, g, u, act)
    torch.cuda.synchronize()
    _check_glu(act, io, g, u, d, out, dg, du)


@pytest.mark.parametrize("act", ACTS)
@pytest.mark.parametrize("io", ["f32", "bf16"])
# Row widths chosen so the row-strided kernels run with each of their block
# widths (bf16: 3072 -> 192 threads, 3584 -> 224, 2560 -> 160, 40 -> 128;
# f32: 3072 and 4864 -> 256).
@pytest.mark.parametrize("T,I", [(33, 3072), (3, 40), (129, 4864), (7, 13), (17, 3584), (11, 2560)])
def test_glu_packed_halves(act, io, T, I):
    # gate and up are the two halves of one [T, 2I] projection output; the
    # gradient is written back into one packed [T, 2I] tensor as well.
    dt = IO[io]
    packed = _randn((T, 2 * I), dt, 4, 2.0)
    g, u = packed[:, :I], packed[:, I:]
    d = _randn((T, I), dt, 5)
    out = gb.glu_fwd(g, u, act)
    grad = torch.empty((T, 2 * I), dtype=dt, device="cuda")
    dg, du = gb.glu_bwd(d, g, u, act, dgate=grad[:, :I], dup=grad[:, I:])
    torch.cuda.synchronize()
    _check_glu(act, io, g, u, d, out, grad[:, :I], grad[:, I:])
    # the plain SwiGLU entry point agrees on the same values (contiguous copies)
    if act == "silu":
        ref = gb.swiglu_fwd(g.contiguous(), u.contiguous())
        torch.cuda.synchronize()
        assert torch.equal(ref, out)


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_glu_unaligned_and_in_place(io):
    dt = IO[io]
    T, I = 9, 1000
    buf = _randn((T * I + 1,), dt, 6, 3.0)
    g = buf[1:].view(T, I)  # off 16-byte alignment: element-wise path
    u = _randn((T, I), dt, 7)
    d = _randn((T, I), dt, 8)
    g0, u0 = g.clone(), u.clone()
    out = gb.glu_fwd(g, u, "gelu_tanh")
    gb.glu_bwd(d, g, u, "gelu_tanh", dgate=g, dup=u)  # in place
    torch.cuda.synchronize()
    check_io(to64(out), oracle.glu_fwd("gelu_tanh", to64(g0), to64(u0)), io, "out")
    dg_ref, du_ref = oracle.glu_bwd("gelu_tanh", to64(d), to64(g0), to64(u0))
    check_io(to64(g), dg_ref, io, "dgate in place")
    check_io(to64(u), du_ref, io, "dup in place")


@pytest.mark.parametrize("act", ACTS)
@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("n", [1, 13, 4096, 1000003])
def test_plain_activation(act, io, n):
    dt = IO[io]
    x, dy = _randn((n,), dt, 9, 3.0), _randn((n,), dt, 10)
    y = gb.act_fwd(x, act)
    dx = gb.act_bwd(dy, x, act)
    torch.cuda.synchronize()
    x64 = to64(x)
    check_io(to64(y), oracle.act(act, x64), io, f"{act} y")
    check_io(to64(dx), to64(dy) * oracle.act_grad(act, x64), io, f"{act} dx")
