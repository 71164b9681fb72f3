"""CPU oracle for the layer operators RMSNorm, rotary position embedding and SwiGLU.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The CUDA library never calls it and it never calls the CUDA library:
the two share no code, no constants and no helpers.

Everything here is plain numpy in float64, single-threaded (no BLAS call is
made), written as the textbook definition of each operator, one step per line,
so that it can be read against the sources by eye.  The sources name the
operators and their hyper-parameters but do not print their formulas:

* "Fast-LLM: 高效大语言模型训练框架", §三 技术架构, table "Transformer Block 结构"
  (normalization is LayerNorm / RMSNorm; the mixer is attention with RoPE; the
  MLP is gated or not, with SiLU / GeLU / ReLU) and §三 "训练配置示例" (``rms_norm``
  with ``epsilon``, ``rotary: type: default, theta``, ``gated: true,
  activation: silu``).
* "LLaMA-Factory Kernels 系统", the kernel table (fused RMSNorm, SwiGLU and RoPE
  operators).
* "Kernels（自定义内核）" (transformers docs), §Liger (RMSNorm, RoPE and SwiGLU
  fused into single kernels, for training, so with backward passes).

Readings taken where the sources are silent (each is listed with its reason in
the design notes of the repository):

* RMSNorm: ``rstd = 1/sqrt(mean(h^2) + eps)`` (eps inside the root), no mean
  subtraction, no bias, the weight multiplies (not ``1 + w``).
* Fused residual: ``h = x + residual`` is rounded to the I/O precision first;
  the rounded ``h`` is both the residual-stream output and what is normalised.
* RoPE: rotate-half pairing ``(i, i + D/2)``; frequencies
  ``theta_i = theta ** (-2 i / D)``; angle ``pos * theta_i``; the same rotation
  for every head of a token, Q and K alike; backward is the inverse rotation.
* SwiGLU: ``out = silu(gate) * up`` with ``silu(g) = g / (1 + exp(-g))``;
  gate and up are two separate tensors.

Pins for every function live in ``tests/test_oracle_pins.py``.
"""

from __future__ import annotations

import math

import numpy as np

__all__ = [
    "round_to_bf16",
    "round_to_f32",
    "round_io",
    "rmsnorm_fwd",
    "rmsnorm_bwd",
    "rmsnorm_dw",
    "layernorm_fwd",
    "layernorm_bwd",
    "rope_inv_freq",
    "rope_fwd",
    "rope_bwd",
    "silu",
    "swiglu_fwd",
    "swiglu_bwd",
    "ACTIVATIONS",
    "act",
    "act_grad",
    "glu_fwd",
    "glu_bwd",
    "positions_from_doc_lengths",
    "positions_from_cu_seqlens",
    "E4M3_MAX",
    "round_to_e4m3",
    "e4m3_encode",
    "e4m3_decode",
    "mx_scale_exponent",
    "mxfp8_quantize",
    "mxfp8_dequantize",
    "rmsnorm_fwd_mxfp8",
    "glu_fwd_mxfp8",
]


# ---------------------------------------------------------------------------
# Rounding to the I/O precision
# ---------------------------------------------------------------------------

def round_to_bf16(a):
    """Round float64 values to the nearest bfloat16 value, ties to even.

    bfloat16 keeps 8 significant bits (1 implicit + 7 stored) with float32's
    exponent range.  Written from that definition: split ``a = m * 2**e`` with
    ``0.5 <= |m| < 1``, scale ``m`` to an integer part of 8 bits, round half to
    even, scale back.  Values below float32's normal range and overflow to
    infinity are outside what this oracle is used for (inputs are O(1)).
    """
    a = np.asarray(a, dtype=np.float64)
    m, e = np.frexp(a)
    return np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)


def round_to_f32(a):
    """Round float64 values to the nearest float32 value (ties to even)."""
    return np.asarray(a, dtype=np.float64).astype(np.float32).astype(np.float64)


def round_io(a, io):
    """Round to the I/O precision ``io`` in {"bf16", "f32", None}; None = keep float64."""
    if io is None:
        return np.asarray(a, dtype=np.float64)
    if io == "bf16":
        return round_to_bf16(a)
    if io == "f32":
        return round_to_f32(a)
    raise ValueError(f"unknown io precision {io!r}")


# ---------------------------------------------------------------------------
# RMSNorm with fused residual add
# ("Fast-LLM: 高效大语言模型训练框架", §三 Transformer Block 结构 and 训练配置示例)
# ---------------------------------------------------------------------------

def rmsnorm_fwd(x, residual, weight, eps, io=None):
    """RMSNorm forward over the last axis, with an optional residual add first.

    x, residual: [T, H] float64 (residual may be None); weight: [H].
    Returns ``(y, h, rstd)``:
      h    = round_io(x + residual)   the residual-stream output (x if no residual)
      rstd = 1 / sqrt(mean(h**2) + eps)   per row, [T]
      y    = weight * h * rstd        exact, before any output rounding
    """
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(weight, dtype=np.float64)
    if residual is None:
        h = x
    else:
        h = round_io(x + np.asarray(residual, dtype=np.float64), io)
    ms = np.mean(h * h, axis=-1)
    rstd = 1.0 / np.sqrt(ms + eps)
    y = w * h * rstd[..., None]
    return y, h, rstd


def rmsnorm_bwd(dy, dres, h, weight, eps):
    """RMSNorm backward: gradient of ``(y, h)`` back to the pre-add input.

    dy: [T, H] gradient of y; dres: [T, H] gradient arriving on the
    residual-stream output h (None = zero); h: [T, H] the normalised input;
    weight: [H].  rstd is recomputed from h.  With n = h * rstd and
    g = dy * weight, the chain rule through y = weight * n gives
      dh = rstd * (g - n * mean(g * n))       per row
      dx = dh + dres                          (= gradient of x and of residual)
      dW = sum over rows of dy * n            [H]
    Returns ``(dx, dW)``.
    """
    dy = np.asarray(dy, dtype=np.float64)
    h = np.asarray(h, dtype=np.float64)
    w = np.asarray(weight, dtype=np.float64)
    rstd = 1.0 / np.sqrt(np.mean(h * h, axis=-1) + eps)
    n = h * rstd[..., None]
    g = dy * w
    c = np.mean(g * n, axis=-1)
    dx = rstd[..., None] * (g - n * c[..., None])
    if dres is not None:
        dx = dx + np.asarray(dres, dtype=np.float64)
    dw = np.sum(dy * n, axis=0)
    return dx, dw


def rmsnorm_dw(dy, h, eps, rows_per_chunk=4096):
    """Weight gradient alone, ``sum_t dy_t * h_t * rstd_t``, streamed over row chunks.

    Same arithmetic as the dW of :func:`rmsnorm_bwd`, for inputs too large to
    hold in float64 at once (arrays may be float32 or bfloat16-valued float32).
    """
    T, H = dy.shape
    dw = np.zeros(H, dtype=np.float64)
    for t0 in range(0, T, rows_per_chunk):
        hb = np.asarray(h[t0:t0 + rows_per_chunk], dtype=np.float64)
        dyb = np.asarray(dy[t0:t0 + rows_per_chunk], dtype=np.float64)
        rstd = 1.0 / np.sqrt(np.mean(hb * hb, axis=-1) + eps)
        dw += np.sum(dyb * hb * rstd[:, None], axis=0)
    return dw


# ---------------------------------------------------------------------------
# LayerNorm with fused residual add ("Fast-LLM: 高效大语言模型训练框架", §三 Transformer
# Block 结构: normalization LayerNorm / RMSNorm).  Standard form: subtract the
# row mean, divide by sqrt(variance + eps) (biased variance), scale by the
# weight, add the bias.
# ---------------------------------------------------------------------------

def layernorm_fwd(x, residual, weight, bias, eps, io=None):
    """Returns ``(y, h, mean, rstd)``:
      h    = round_io(x + residual)            (x if no residual)
      mean = mean(h);  var = mean((h - mean)**2);  rstd = 1 / sqrt(var + eps)
      y    = weight * (h - mean) * rstd + bias  (bias None = 0), exact
    """
    x = np.asarray(x, dtype=np.float64)
    if residual is None:
        h = x
    else:
        h = round_io(x + np.asarray(residual, dtype=np.float64), io)
    mean = np.mean(h, axis=-1)
    c = h - mean[..., None]
    var = np.mean(c * c, axis=-1)
    rstd = 1.0 / np.sqrt(var + eps)
    y = np.asarray(weight, dtype=np.float64) * c * rstd[..., None]
    if bias is not None:
        y = y + np.asarray(bias, dtype=np.float64)
    return y, h, mean, rstd


def layernorm_bwd(dy, dres, h, weight, eps):
    """Gradients of :func:`layernorm_fwd`.  With n = (h - mean) * rstd, g = dy * weight:
      dh = rstd * (g - mean(g) - n * mean(g * n));  dx = dh + dres
      dW = sum over rows of dy * n;  dB = sum over rows of dy
    Returns ``(dx, dW, dB)``.
    """
    dy = np.asarray(dy, dtype=np.float64)
    h = np.asarray(h, dtype=np.float64)
    mean = np.mean(h, axis=-1)
    c = h - mean[..., None]
    rstd = 1.0 / np.sqrt(np.mean(c * c, axis=-1) + eps)
    n = c * rstd[..., None]
    g = dy * np.asarray(weight, dtype=np.float64)
    dx = rstd[..., None] * (g - np.mean(g, axis=-1)[..., None] - n * np.mean(g * n, axis=-1)[..., None])
    if dres is not None:
        dx = dx + np.asarray(dres, dtype=np.float64)
    return dx, np.sum(dy * n, axis=0), np.sum(dy, axis=0)


# ---------------------------------------------------------------------------
# Rotary position embedding on Q and K
# ("Fast-LLM: 高效大语言模型训练框架", §三 框架结构 (attention with RoPE) and
#  训练配置示例 (rotary type default, theta); "LLaMA-Factory Kernels 系统")
# ---------------------------------------------------------------------------

def rope_inv_freq(D, theta):
    """Per-pair frequencies ``theta ** (-2 i / D)`` for i = 0 .. D/2 - 1."""
    i = np.arange(D // 2, dtype=np.float64)
    return np.power(float(theta), -2.0 * i / D)


def _rope_rotate(x, positions, theta, sign, pairing="half"):
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[-1]
    half = D // 2
    freq = rope_inv_freq(D, theta)                                  # [D/2]
    angle = np.asarray(positions, dtype=np.float64)[:, None] * freq  # [T, D/2]
    cos = np.cos(angle)[:, None, :]                                 # [T, 1, D/2]
    sin = sign * np.sin(angle)[:, None, :]
    if pairing == "half":          # pair (i, i + D/2)
        x1 = x[..., :half]
        x2 = x[..., half:]
    elif pairing == "interleaved":  # pair (2i, 2i + 1)
        x1 = x[..., 0::2]
        x2 = x[..., 1::2]
    else:
        raise ValueError(pairing)
    y1 = x1 * cos - x2 * sin
    y2 = x2 * cos + x1 * sin
    out = np.empty_like(x)
    if pairing == "half":
        out[..., :half] = y1
        out[..., half:] = y2
    else:
        out[..., 0::2] = y1
        out[..., 1::2] = y2
    return out


def rope_fwd(x, positions, theta, pairing="half"):
    """Rotate every head of token t by angle ``positions[t] * theta_i`` on pair i.

    x: [T, heads, D] float64; positions: [T] integers.  ``pairing`` "half" pairs
    element i with i + D/2 (the default rotary type); "interleaved" pairs 2i
    with 2i + 1.  Returns the rotated array.  Q and K are each passed through this
    with the same positions.
    """
    return _rope_rotate(x, positions, theta, +1.0, pairing)


def rope_bwd(dout, positions, theta, pairing="half"):
    """Gradient of :func:`rope_fwd`: the transpose (= inverse) rotation, angle negated."""
    return _rope_rotate(dout, positions, theta, -1.0, pairing)


# ---------------------------------------------------------------------------
# SwiGLU  (gated MLP with SiLU: "Fast-LLM: 高效大语言模型训练框架", §三 支持的 MLP 变体
#  and 训练配置示例; "LLaMA-Factory Kernels 系统"; "Kernels（自定义内核）" §Liger)
# ---------------------------------------------------------------------------

def _sigmoid(g):
    return 1.0 / (1.0 + np.exp(-g))


def silu(g):
    """SiLU, ``g * sigmoid(g)``."""
    g = np.asarray(g, dtype=np.float64)
    return g * _sigmoid(g)


def swiglu_fwd(gate, up):
    """``out = silu(gate) * up`` elementwise."""
    gate = np.asarray(gate, dtype=np.float64)
    up = np.asarray(up, dtype=np.float64)
    return silu(gate) * up


def swiglu_bwd(dout, gate, up):
    """Gradients of :func:`swiglu_fwd`.

    With s = sigmoid(g): d silu/dg = s + g * s * (1 - s) = s * (1 + g * (1 - s)), so
      dgate = dout * up * s * (1 + g * (1 - s))
      dup   = dout * g * s
    Returns ``(dgate, dup)``.
    """
    dout = np.asarray(dout, dtype=np.float64)
    g = np.asarray(gate, dtype=np.float64)
    u = np.asarray(up, dtype=np.float64)
    s = _sigmoid(g)
    dgate = dout * u * s * (1.0 + g * (1.0 - s))
    dup = dout * g * s
    return dgate, dup


# ---------------------------------------------------------------------------
# Gated and plain MLP activations ("Fast-LLM: 高效大语言模型训练框架", §三 支持的 MLP
# 变体: dense MLP gated or not, with SiLU / GeLU / ReLU).  GeLU comes in its exact
# form x * Phi(x) (Phi the standard normal CDF, via erf) and in the common tanh
# approximation 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))).
# ---------------------------------------------------------------------------

ACTIVATIONS = ("silu", "gelu_tanh", "gelu_erf", "relu")

_SQRT_2_OVER_PI = math.sqrt(2.0 / math.pi)


def act(name, x):
    """Activation value f(x)."""
    x = np.asarray(x, dtype=np.float64)
    if name == "silu":
        return silu(x)
    if name == "gelu_tanh":
        return 0.5 * x * (1.0 + np.tanh(_SQRT_2_OVER_PI * (x + 0.044715 * x ** 3)))
    if name == "gelu_erf":
        return 0.5 * x * (1.0 + _erf(x / math.sqrt(2.0)))
    if name == "relu":
        return np.maximum(x, 0.0)
    raise ValueError(name)


def act_grad(name, x):
    """Derivative f'(x) (for ReLU: 1 where x > 0, else 0)."""
    x = np.asarray(x, dtype=np.float64)
    if name == "silu":
        s = _sigmoid(x)
        return s * (1.0 + x * (1.0 - s))
    if name == "gelu_tanh":
        z = _SQRT_2_OVER_PI * (x + 0.044715 * x ** 3)
        t = np.tanh(z)
        dz = _SQRT_2_OVER_PI * (1.0 + 3.0 * 0.044715 * x ** 2)
        return 0.5 * (1.0 + t) + 0.5 * x * (1.0 - t * t) * dz
    if name == "gelu_erf":
        pdf = np.exp(-0.5 * x * x) / math.sqrt(2.0 * math.pi)
        return 0.5 * (1.0 + _erf(x / math.sqrt(2.0))) + x * pdf
    if name == "relu":
        return (x > 0).astype(np.float64)
    raise ValueError(name)


def _erf(x):
    from scipy.special import erf  # library primitive for the normal CDF
    return erf(x)


def glu_fwd(name, gate, up):
    """Gated unit ``out = f(gate) * up`` (SwiGLU is f = SiLU)."""
    return act(name, gate) * np.asarray(up, dtype=np.float64)


def glu_bwd(name, dout, gate, up):
    """Gradients of :func:`glu_fwd`: ``dgate = dout * up * f'(gate)``, ``dup = dout * f(gate)``."""
    dout = np.asarray(dout, dtype=np.float64)
    return dout * np.asarray(up, dtype=np.float64) * act_grad(name, gate), dout * act(name, gate)


# ---------------------------------------------------------------------------
# Positions for packed documents ("Fast-LLM: 高效大语言模型训练框架", §三 训练配置示例:
#  micro_batch_size counted in tokens, maximum_document_length; §三 数据管道)
# ---------------------------------------------------------------------------

def positions_from_doc_lengths(lengths):
    """Position of each token inside its own document: 0, 1, ..., L-1 per document, concatenated."""
    parts = [np.arange(int(L), dtype=np.int64) for L in lengths]
    if not parts:
        return np.zeros(0, dtype=np.int64)
    return np.concatenate(parts)


def positions_from_cu_seqlens(cu_seqlens):
    """Same, from cumulative document boundaries ``cu_seqlens`` (cu[0] = 0, cu[-1] = T)."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    return positions_from_doc_lengths(cu[1:] - cu[:-1])


# ---------------------------------------------------------------------------
# MXFP8 output: the FP8 operand layout of the next projection GEMM
# ("Kernels（自定义内核）": fusing the producer of a tensor with its consumer's
#  input conversion saves a pass over HBM; the format itself is the OCP
#  Microscaling Formats (MX) v1.0 specification's MXFP8 with E4M3 elements:
#  blocks of 32 consecutive values share one power-of-two scale stored as an
#  E8M0 byte).  Blocks run along the last axis (the GEMM's reduction axis).
# ---------------------------------------------------------------------------

E4M3_MAX = 448.0        # largest finite E4M3 magnitude: 1.75 * 2**8
_E4M3_EMIN = -6         # exponent of the smallest normal, 2**-6
_E4M3_MBITS = 3         # stored mantissa bits
_E4M3_EMAX = 8          # exponent of the largest normal (the MX "emax_elem")
_E8M0_BIAS = 127
MX_BLOCK = 32


def round_to_e4m3(a):
    """Round float64 values to the nearest E4M3 value, ties to even, saturating.

    E4M3 (as used by MXFP8): 1 sign bit, 4 exponent bits with bias 7, 3 mantissa
    bits, no infinities.  Normal values are ``(1 + m/8) * 2**e`` for e in
    [-6, 8]; below 2**-6 the spacing is the subnormal quantum 2**-9.  Written from
    that definition: the spacing at |a| is ``2**(max(floor(log2|a|), -6) - 3)``;
    divide by it, round half to even, multiply back.  Magnitudes that round
    beyond 448 become 448 (saturation); NaN stays NaN.
    """
    a = np.asarray(a, dtype=np.float64)
    mag = np.abs(a)
    with np.errstate(divide="ignore", invalid="ignore"):
        _, e2 = np.frexp(mag)           # mag = f * 2**e2 with 0.5 <= f < 1
    e = np.maximum(e2 - 1, _E4M3_EMIN)  # floor(log2 mag) for mag > 0, clamped at the subnormal range
    quantum = np.ldexp(1.0, e - _E4M3_MBITS)
    r = np.rint(mag / quantum) * quantum
    r = np.where(mag == 0, 0.0, r)
    r = np.minimum(r, E4M3_MAX)
    return np.where(np.isnan(a), np.nan, np.copysign(r, a))


def e4m3_encode(v):
    """Bit pattern (uint8) of E4M3 values ``v`` (which must already be E4M3 values)."""
    v = np.asarray(v, dtype=np.float64)
    sign = np.signbit(v).astype(np.uint8) << 7
    mag = np.abs(v)
    _, e2 = np.frexp(mag)
    e = e2 - 1
    normal = mag >= 2.0 ** _E4M3_EMIN
    # normal: exponent field e + 7, mantissa (mag / 2**e - 1) * 8
    ef = np.where(normal, e + 7, 0)
    mf = np.where(normal, np.rint((np.ldexp(mag, -e) - 1.0) * 8.0),
                  np.rint(mag / 2.0 ** (_E4M3_EMIN - _E4M3_MBITS)))
    code = sign | (ef.astype(np.uint8) << 3) | mf.astype(np.uint8)
    return np.where(np.isnan(v), np.uint8(0x7F), code).astype(np.uint8)


def e4m3_decode(code):
    """E4M3 bit patterns (uint8) to float64: sign, exponent field E, mantissa M;
    E = 0 gives ``M * 2**-9``, otherwise ``(1 + M/8) * 2**(E - 7)``; 0x7F / 0xFF are NaN."""
    c = np.asarray(code, dtype=np.uint8).astype(np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    E = (c >> 3) & 0xF
    M = c & 0x7
    val = np.where(E == 0, M * 2.0 ** (_E4M3_EMIN - _E4M3_MBITS),
                   (1.0 + M / 8.0) * np.ldexp(1.0, E - 7))
    val = s * val
    return np.where((E == 15) & (M == 7), np.nan, val)


def mx_scale_exponent(amax):
    """Shared exponent of an MX block with largest magnitude ``amax``.

    The MX conversion takes ``floor(log2(amax)) - emax_elem`` (emax_elem = 8 for
    E4M3), so the block's largest value lands in E4M3's top binade; E8M0 holds
    exponents -127..127, and an all-zero block takes the smallest, -127.
    """
    amax = np.asarray(amax, dtype=np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        _, e2 = np.frexp(amax)
    se = np.where(amax > 0, (e2 - 1) - _E4M3_EMAX, -_E8M0_BIAS)
    return np.clip(se, -_E8M0_BIAS, _E8M0_BIAS).astype(np.int64)


def mxfp8_quantize(v, block=MX_BLOCK):
    """MXFP8 (E4M3) quantization of ``v`` [..., N] in blocks of ``block`` along the last axis.

    Returns ``(codes, scales)``: codes uint8 [..., N] (E4M3 bit patterns of
    ``round_to_e4m3(v / 2**se)``) and scales uint8 [..., N / block] (E8M0:
    ``se + 127``), with ``se = mx_scale_exponent(max |v| over the block)``.
    """
    v = np.asarray(v, dtype=np.float64)
    n = v.shape[-1]
    if n % block:
        raise ValueError("the last axis must be a multiple of the block size")
    vb = v.reshape(v.shape[:-1] + (n // block, block))
    se = mx_scale_exponent(np.max(np.abs(vb), axis=-1))
    q = round_to_e4m3(vb / np.ldexp(1.0, se)[..., None])
    return e4m3_encode(q).reshape(v.shape), (se + _E8M0_BIAS).astype(np.uint8)


def mxfp8_dequantize(codes, scales, block=MX_BLOCK):
    """Values of an MXFP8 tensor: ``e4m3_decode(code) * 2**(scale - 127)`` per block."""
    c = np.asarray(codes)
    n = c.shape[-1]
    vals = e4m3_decode(c).reshape(c.shape[:-1] + (n // block, block))
    se = np.asarray(scales, dtype=np.int64) - _E8M0_BIAS
    return (vals * np.ldexp(1.0, se)[..., None]).reshape(c.shape)


def rmsnorm_fwd_mxfp8(x, residual, weight, eps, io=None):
    """RMSNorm forward whose output y is also delivered as MXFP8 (blocks along H).

    Returns ``(codes, scales, y, h, rstd)``: ``y, h, rstd`` as :func:`rmsnorm_fwd`
    (y exact, before any rounding) and ``codes, scales = mxfp8_quantize(y)``.
    """
    y, h, rstd = rmsnorm_fwd(x, residual, weight, eps, io)
    codes, scales = mxfp8_quantize(y)
    return codes, scales, y, h, rstd


def glu_fwd_mxfp8(name, gate, up):
    """Gated unit forward delivered as MXFP8: ``mxfp8_quantize(act(gate) * up)``."""
    return mxfp8_quantize(glu_fwd(name, gate, up))
