"""The autograd wrappers inside a PyTorch graph: a toy layer (residual add +
RMSNorm, RoPE on Q/K, SwiGLU) run forward, a loss with fixed upstream
gradients backpropagated, and every gradient compared with the oracle's
backward passes.  bf16 tolerances of ``_checks``."""

import numpy as np
import pytest
import torch

import oracle
import rmsnorm_fwd_bwd_03_gb300 as gb
from rmsnorm_fwd_bwd_03_gb300 import autograd as ga

from _checks import check_dw, check_io, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    from rmsnorm_fwd_bwd_03_gb300._build import build_library
    build_library()
    gb.library()


def _randn(shape, dtype, seed, scale=1.0):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return (torch.randn(shape, generator=g, device="cuda") * scale).to(dtype)


def test_autograd_rmsnorm_with_residual():
    T, H, dt, eps = 64, 1024, torch.bfloat16, 1e-6
    x = _randn((T, H), dt, 1).requires_grad_()
    r = _randn((T, H), dt, 2).requires_grad_()
    w = (1 + 0.1 * _randn((H,), torch.float32, 3)).to(dt).requires_grad_()
    dy, dh = _randn((T, H), dt, 4), _randn((T, H), dt, 5)
    y, h = ga.rms_norm(x, w, eps, r)
    torch.autograd.backward([y, h], [dy, dh])
    torch.cuda.synchronize()
    y_ref, h_ref, _ = oracle.rmsnorm_fwd(to64(x), to64(r), to64(w), eps, io="bf16")
    assert np.array_equal(to64(h), h_ref)
    check_io(to64(y), y_ref, "bf16", "y")
    dx_ref, dw_ref = oracle.rmsnorm_bwd(to64(dy), to64(dh), h_ref, to64(w), eps)
    check_io(to64(x.grad), dx_ref, "bf16", "x.grad")
    assert torch.equal(x.grad, r.grad)
    # the float32 weight gradient is handed back in the weight's dtype (bf16 here)
    assert w.grad.dtype == torch.bfloat16
    check_io(to64(w.grad), dw_ref, "bf16", "weight.grad")


def test_autograd_layer_chain():
    # h = x + r; y = RMSNorm(h); q, k = rotary(y-derived projections); out = swiglu(gate, up)
    # with plain torch matmuls between (the GEMMs are not this library's).
    T, H, Hq, Hk, D, I = 48, 256, 4, 2, 64, 384
    dt = torch.float32
    x = _randn((T, H), dt, 11).requires_grad_()
    w = (1 + 0.1 * _randn((H,), torch.float32, 12)).requires_grad_()
    wq = (_randn((H, Hq * D), dt, 13) / H ** 0.5).requires_grad_()
    wk = (_randn((H, Hk * D), dt, 14) / H ** 0.5).requires_grad_()
    wg = (_randn((H, I), dt, 15) / H ** 0.5).requires_grad_()
    wu = (_randn((H, I), dt, 16) / H ** 0.5).requires_grad_()
    pos = torch.arange(T, dtype=torch.int32, device="cuda") % 20
    table = gb.rope_table(20, D, 1e4)
    y = ga.rms_norm(x, w, 1e-5)
    seen = {}
    y.register_hook(lambda g: seen.__setitem__("dY", g.detach().clone()))  # what the backward receives
    q, k = ga.rotary((y @ wq).view(T, Hq, D), (y @ wk).view(T, Hk, D), pos, table)
    out = ga.swiglu(y @ wg, y @ wu)
    cq, ck, co = _randn((T, Hq, D), dt, 17), _randn((T, Hk, D), dt, 18), _randn((T, I), dt, 19)
    loss = (q * cq).sum() + (k * ck).sum() + (out * co).sum()
    loss.backward()
    torch.cuda.synchronize()

    # the same chain through the oracle, gradients by hand with its backward passes
    X, W = to64(x), to64(w)
    WQ, WK, WG, WU = to64(wq), to64(wk), to64(wg), to64(wu)
    p = pos.cpu().numpy()
    Y, _, _ = oracle.rmsnorm_fwd(X, None, W, 1e-5)
    G, U = Y @ WG, Y @ WU
    dG, dU = oracle.swiglu_bwd(to64(co), G, U)
    dQ = oracle.rope_bwd(to64(cq), p, 1e4).reshape(T, Hq * D)
    dK = oracle.rope_bwd(to64(ck), p, 1e4).reshape(T, Hk * D)
    dY = dQ @ WQ.T + dK @ WK.T + dG @ WG.T + dU @ WU.T
    dX, dW = oracle.rmsnorm_bwd(dY, None, X, W, 1e-5)
    # The float32 GEMMs between the operators round dY (they are torch's, not this
    # library's), so x.grad is held to the stated float32 bound against the
    # oracle's backward of the dY the wrapper actually received, and to the
    # weight-gradient bound against the float64 chain.
    dX_seen, _ = oracle.rmsnorm_bwd(to64(seen["dY"]), None, X, W, 1e-5)
    check_io(to64(x.grad), dX_seen, "f32", "x.grad")
    check_dw(to64(x.grad).ravel(), dX.ravel(), "x.grad (float64 chain)")
    check_dw(to64(w.grad), dW, "weight.grad")
    check_dw(to64(wg.grad), Y.T @ dG, "wg.grad")
    check_dw(to64(wq.grad), Y.T @ dQ, "wq.grad")
