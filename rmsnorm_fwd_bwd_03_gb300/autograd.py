"""torch.autograd.Function wrappers around the C-ABI calls, so the operators can
sit inside a PyTorch training graph.  Every forward and backward runs in
libgbln's kernels (through the functions of this package); nothing here
computes anything itself.

* ``rms_norm(x, weight, eps, residual=None)`` -> ``y`` or ``(y, h)``: RMSNorm with
  the fused residual add.  With a residual, ``h = x + residual`` (the
  residual-stream output) is returned as well, and its gradient enters the
  backward pass as ``dresidual_out``; x and residual get the same gradient.
  The weight gradient comes from the two-pass fixed-order reduction (float32,
  cast to the weight's dtype).
* ``rotary(q, k, positions, cos_sin)`` -> ``(q', k')``: RoPE on Q and K
  (rotate-half pairing); the backward pass is the inverse rotation.
* ``swiglu(gate, up)`` -> ``silu(gate) * up``.
"""

from __future__ import annotations

import torch

from . import (rmsnorm_bwd, rmsnorm_dw_finalize, rmsnorm_fwd, rope_bwd, rope_fwd, swiglu_bwd,
               swiglu_fwd)


def _c(t):
    return None if t is None else t.contiguous()


class _RMSNorm(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, residual, weight, eps):
        y, h, rstd = rmsnorm_fwd(x.contiguous(), weight.contiguous(), eps, _c(residual))
        ctx.save_for_backward(h, weight, rstd)
        ctx.has_residual = residual is not None
        if residual is None:
            return y
        return y, h

    @staticmethod
    def backward(ctx, dy, dh=None):
        h, weight, rstd = ctx.saved_tensors
        dx, part, P = rmsnorm_bwd(dy.contiguous(), h, weight, rstd, _c(dh))
        dw = rmsnorm_dw_finalize(part, P).to(weight.dtype)
        return dx, (dx if ctx.has_residual else None), dw, None


def rms_norm(x, weight, eps, residual=None):
    return _RMSNorm.apply(x, residual, weight, float(eps))


class _Rotary(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, positions, cos_sin):
        ctx.save_for_backward(positions, cos_sin)
        return rope_fwd(q.contiguous(), k.contiguous(), positions, cos_sin)

    @staticmethod
    def backward(ctx, dq, dk):
        positions, cos_sin = ctx.saved_tensors
        dqi, dki = rope_bwd(dq.contiguous(), dk.contiguous(), positions, cos_sin)
        return dqi, dki, None, None


def rotary(q, k, positions, cos_sin):
    return _Rotary.apply(q, k, positions, cos_sin)


class _SwiGLU(torch.autograd.Function):
    @staticmethod
    def forward(ctx, gate, up):
        gate, up = gate.contiguous(), up.contiguous()
        ctx.save_for_backward(gate, up)
        return swiglu_fwd(gate, up)

    @staticmethod
    def backward(ctx, dout):
        gate, up = ctx.saved_tensors
        return swiglu_bwd(dout.contiguous(), gate, up)


def swiglu(gate, up):
    return _SwiGLU.apply(gate, up)
