"""Planted mistakes in the oracle are caught by its pins.

Each case is one plausible slip in the oracle's source: a dropped term, a wrong
sign, a swapped operand, a wrong index, axis or constant.  The test builds a copy
of the oracle with that single textual change, points the pin tests of
``test_oracle_pins.py`` at the copy, runs the pins of the operator concerned and
requires at least one of them to fail.  The real oracle is not touched, and
everything runs on the CPU.
"""

import inspect
import os
import types

import pytest

import test_oracle_pins as pins

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
with open(os.path.join(ROOT, "oracle", "__init__.py"), encoding="utf-8") as _f:
    ORACLE_SRC = _f.read()

RMS, LN, ROPE = ("rmsnorm",), ("layernorm",), ("rope",)
ACTS = ("swiglu", "gelu", "activation")
MX = ("e4m3", "mx", "rmsnorm_fwd_mxfp8", "glu_fwd_mxfp8")

# (case id, text in the oracle, replacement, prefixes of the pin tests to run)
MUTANTS = [
    # RMSNorm
    ("rms_eps_outside_root", "rstd = 1.0 / np.sqrt(ms + eps)", "rstd = 1.0 / np.sqrt(ms) + eps", RMS),
    ("rms_one_plus_weight", "y = w * h * rstd[..., None]", "y = (1.0 + w) * h * rstd[..., None]", RMS),
    ("rms_residual_not_rounded", "h = round_io(x + np.asarray(residual, dtype=np.float64), io)",
     "h = x + np.asarray(residual, dtype=np.float64)", RMS),
    ("rms_sum_not_mean", "ms = np.mean(h * h, axis=-1)", "ms = np.sum(h * h, axis=-1)", RMS),
    ("rms_bwd_projection_dropped", "dx = rstd[..., None] * (g - n * c[..., None])",
     "dx = rstd[..., None] * g", RMS),
    ("rms_bwd_residual_grad_dropped",
     "        dx = dx + np.asarray(dres, dtype=np.float64)\n    dw = np.sum(dy * n, axis=0)",
     "        pass\n    dw = np.sum(dy * n, axis=0)", RMS),
    ("rms_bwd_dw_not_normalised", "dw = np.sum(dy * n, axis=0)", "dw = np.sum(dy * h, axis=0)", RMS),
    ("rms_dw_chunks_not_normalised", "dw += np.sum(dyb * hb * rstd[:, None], axis=0)",
     "dw += np.sum(dyb * hb, axis=0)", RMS),
    # LayerNorm
    ("ln_unbiased_variance", "var = np.mean(c * c, axis=-1)",
     "var = np.sum(c * c, axis=-1) / max(c.shape[-1] - 1, 1)", LN),
    ("ln_mean_not_subtracted", "c = h - mean[..., None]\n    var", "c = h\n    var", LN),
    ("ln_bwd_mean_term_dropped", "(g - np.mean(g, axis=-1)[..., None] - n *", "(g - n *", LN),
    ("ln_bwd_db_wrong", "np.sum(dy * n, axis=0), np.sum(dy, axis=0)",
     "np.sum(dy * n, axis=0), np.sum(dy * n, axis=0)", LN),
    # RoPE
    ("rope_frequency_exponent", "-2.0 * i / D", "-1.0 * i / D", ROPE),
    ("rope_sign", "y1 = x1 * cos - x2 * sin", "y1 = x1 * cos + x2 * sin", ROPE),
    ("rope_half_pairs_adjacent", "        x1 = x[..., :half]\n        x2 = x[..., half:]",
     "        x1 = x[..., 0::2]\n        x2 = x[..., 1::2]", ROPE),
    ("rope_bwd_not_inverse", "return _rope_rotate(dout, positions, theta, -1.0, pairing)",
     "return _rope_rotate(dout, positions, theta, +1.0, pairing)", ROPE),
    ("rope_interleaved_outputs_swapped", "        out[..., 0::2] = y1\n        out[..., 1::2] = y2",
     "        out[..., 0::2] = y2\n        out[..., 1::2] = y1", ROPE),
    ("rope_position_off_by_one", "angle = np.asarray(positions, dtype=np.float64)[:, None] * freq",
     "angle = (np.asarray(positions, dtype=np.float64)[:, None] + 1.0) * freq", ROPE),
    # SwiGLU and the other activations
    ("sigmoid_sign", "return 1.0 / (1.0 + np.exp(-g))", "return 1.0 / (1.0 + np.exp(g))", ACTS),
    ("swiglu_operands_swapped", "return silu(gate) * up", "return silu(up) * gate", ACTS),
    ("swiglu_bwd_term_dropped", "dgate = dout * u * s * (1.0 + g * (1.0 - s))", "dgate = dout * u * s", ACTS),
    ("swiglu_bwd_dup_wrong", "dup = dout * g * s", "dup = dout * s", ACTS),
    ("gelu_tanh_constant", "0.044715 * x ** 3)))", "0.04715 * x ** 3)))", ACTS),
    ("gelu_erf_scale_dropped", "return 0.5 * x * (1.0 + _erf(x / math.sqrt(2.0)))",
     "return 0.5 * x * (1.0 + _erf(x))", ACTS),
    ("gelu_erf_grad_density_dropped", ") + x * pdf", ")", ACTS),
    ("glu_bwd_dup_uses_up", "dout * act(name, gate)\n", "dout * act(name, up)\n", ACTS),
    # positions, bf16 rounding
    ("positions_start_at_one", "np.arange(int(L), dtype=np.int64)", "np.arange(1, int(L) + 1, dtype=np.int64)",
     ("positions",)),
    ("bf16_seven_bits", "np.rint(np.ldexp(m, 8)), e - 8)", "np.rint(np.ldexp(m, 7)), e - 7)", ("bf16",)),
    ("bf16_truncation", "np.rint(np.ldexp(m, 8))", "np.trunc(np.ldexp(m, 8))", ("bf16",)),
    # MXFP8
    ("mx_exponent_offset_dropped", "(e2 - 1) - _E4M3_EMAX, -_E8M0_BIAS)", "(e2 - 1), -_E8M0_BIAS)", MX),
    ("mx_exponent_ceil", "(e2 - 1) - _E4M3_EMAX, -_E8M0_BIAS)", "(e2) - _E4M3_EMAX, -_E8M0_BIAS)", MX),
    ("e4m3_floor_not_rne", "r = np.rint(mag / quantum) * quantum", "r = np.floor(mag / quantum) * quantum", MX),
    ("e4m3_no_saturation", "r = np.minimum(r, E4M3_MAX)", "r = r", MX),
    ("e8m0_bias_126", "_E8M0_BIAS = 127", "_E8M0_BIAS = 126", MX),
    ("e4m3_subnormal_exponent", "_E4M3_EMIN = -6 ", "_E4M3_EMIN = -7 ", MX),
    ("e4m3_nan_code", "np.uint8(0x7F), code", "np.uint8(0x7E), code", MX),
    ("e4m3_decode_subnormal_scale", "E == 0, M * 2.0 ** (_E4M3_EMIN - _E4M3_MBITS)",
     "E == 0, M * 2.0 ** (_E4M3_EMIN - _E4M3_MBITS + 1)", MX),
    ("mx_dequantize_bias", "se = np.asarray(scales, dtype=np.int64) - _E8M0_BIAS",
     "se = np.asarray(scales, dtype=np.int64) - 126", MX),
    # more LayerNorm, activation, RoPE and rounding slips
    ("ln_residual_not_rounded",
     "        h = round_io(x + np.asarray(residual, dtype=np.float64), io)\n    mean = np.mean(h, axis=-1)",
     "        h = x + np.asarray(residual, dtype=np.float64)\n    mean = np.mean(h, axis=-1)", LN),
    ("ln_bias_dropped", "        y = y + np.asarray(bias, dtype=np.float64)\n    return y, h, mean, rstd",
     "        pass\n    return y, h, mean, rstd", LN),
    ("ln_bwd_eps_dropped", "rstd = 1.0 / np.sqrt(np.mean(c * c, axis=-1) + eps)\n    n = c",
     "rstd = 1.0 / np.sqrt(np.mean(c * c, axis=-1))\n    n = c", LN),
    ("rms_bwd_eps_dropped", "rstd = 1.0 / np.sqrt(np.mean(h * h, axis=-1) + eps)\n    n = h * rstd",
     "rstd = 1.0 / np.sqrt(np.mean(h * h, axis=-1))\n    n = h * rstd", RMS),
    ("relu_grad_at_zero", "return (x > 0).astype(np.float64)", "return (x >= 0).astype(np.float64)", ACTS),
    ("silu_as_sigmoid", "return g * _sigmoid(g)", "return _sigmoid(g)", ACTS),
    ("gelu_tanh_grad_factor", "3.0 * 0.044715 * x ** 2", "0.044715 * x ** 2", ACTS),
    ("glu_fwd_operands_swapped", "return act(name, gate) * np.asarray(up, dtype=np.float64)",
     "return act(name, up) * np.asarray(gate, dtype=np.float64)", ACTS),
    ("rope_theta_power_sign", "np.power(float(theta), -2.0 * i / D)", "np.power(float(theta), 2.0 * i / D)", ROPE),
    ("cu_seqlens_not_differenced", "cu[1:] - cu[:-1]", "cu[1:]", ("positions",)),
    ("round_io_f32_as_bf16", '    if io == "f32":\n        return round_to_f32(a)',
     '    if io == "f32":\n        return round_to_bf16(a)', ("round_io",)),
    ("rms_residual_ignored",
     "    if residual is None:\n        h = x\n    else:\n        h = round_io(x + np.asarray(residual, dtype=np.float64), io)\n    ms",
     "    h = x\n    ms", RMS),
    ("rms_bwd_sum_not_mean", "c = np.mean(g * n, axis=-1)", "c = np.sum(g * n, axis=-1)", RMS),
    ("rms_bwd_weight_dropped", "g = dy * w\n", "g = dy\n", RMS),
    ("rms_dw_chunks_eps_dropped", "rstd = 1.0 / np.sqrt(np.mean(hb * hb, axis=-1) + eps)",
     "rstd = 1.0 / np.sqrt(np.mean(hb * hb, axis=-1))", RMS),
    ("rms_dw_chunks_skip_last_row", "for t0 in range(0, T, rows_per_chunk):",
     "for t0 in range(0, T - 1, rows_per_chunk):", RMS),
    ("ln_weight_dropped", "y = np.asarray(weight, dtype=np.float64) * c * rstd[..., None]",
     "y = c * rstd[..., None]", LN),
    ("ln_bwd_residual_grad_dropped",
     "        dx = dx + np.asarray(dres, dtype=np.float64)\n    return dx, np.sum",
     "        pass\n    return dx, np.sum", LN),
    ("ln_bwd_weight_dropped", "g = dy * np.asarray(weight, dtype=np.float64)\n    dx", "g = dy\n    dx", LN),
    ("rope_cos_from_sin", "    cos = np.cos(angle)[:, None, :]", "    cos = np.sin(angle)[:, None, :]", ROPE),
    ("rope_second_sign", "y2 = x2 * cos + x1 * sin", "y2 = x2 * cos - x1 * sin", ROPE),
    ("rope_half_outputs_swapped", "        out[..., :half] = y1\n        out[..., half:] = y2",
     "        out[..., :half] = y2\n        out[..., half:] = y1", ROPE),
    ("rope_frequency_over_half", "return np.power(float(theta), -2.0 * i / D)",
     "return np.power(float(theta), -2.0 * i / (D // 2))", ROPE),
    ("swiglu_bwd_s_for_one_minus_s", "dgate = dout * u * s * (1.0 + g * (1.0 - s))",
     "dgate = dout * u * s * (1.0 + g * s)", ACTS),
    ("gelu_tanh_half_dropped", "return 0.5 * x * (1.0 + np.tanh(", "return x * (1.0 + np.tanh(", ACTS),
    ("gelu_tanh_root_dropped", "_SQRT_2_OVER_PI = math.sqrt(2.0 / math.pi)", "_SQRT_2_OVER_PI = 2.0 / math.pi", ACTS),
    ("gelu_erf_density_norm", "pdf = np.exp(-0.5 * x * x) / math.sqrt(2.0 * math.pi)",
     "pdf = np.exp(-0.5 * x * x) / math.sqrt(math.pi)", ACTS),
    ("glu_bwd_up_dropped", "return dout * np.asarray(up, dtype=np.float64) * act_grad(name, gate)",
     "return dout * act_grad(name, gate)", ACTS),
    ("e4m3_one_bit_too_many", "quantum = np.ldexp(1.0, e - _E4M3_MBITS)", "quantum = np.ldexp(1.0, e - _E4M3_MBITS - 1)", MX),
    ("e4m3_sign_lost", "np.copysign(r, a))", "r)", MX),
    ("e4m3_encode_exponent_bias", "ef = np.where(normal, e + 7, 0)", "ef = np.where(normal, e + 8, 0)", MX),
    ("mx_one_scale_per_tensor", "se = mx_scale_exponent(np.max(np.abs(vb), axis=-1))",
     "se = mx_scale_exponent(np.max(np.abs(vb)) + 0 * np.max(np.abs(vb), axis=-1))", MX),
    ("mx_scale_multiplied", "q = round_to_e4m3(vb / np.ldexp(1.0, se)[..., None])",
     "q = round_to_e4m3(vb * np.ldexp(1.0, se)[..., None])", MX),
    ("mx_zero_block_exponent", "-_E8M0_BIAS)\n    return np.clip", "0)\n    return np.clip", MX),
    ("bf16_exponent_off", "np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)", "np.ldexp(np.rint(np.ldexp(m, 8)), e - 9)", ("bf16",)),
    ("positions_of_no_documents", "        return np.zeros(0, dtype=np.int64)", "        return np.zeros(1, dtype=np.int64)",
     ("positions",)),
]


def _mutant(old, new):
    assert ORACLE_SRC.count(old) >= 1, f"mutation site not found: {old!r}"
    mod = types.ModuleType("oracle_mutant")
    exec(compile(ORACLE_SRC.replace(old, new, 1), "oracle_mutant", "exec"), mod.__dict__)
    return mod


def _pin_calls(prefixes):
    """(name, callable) for every pin test (and parametrization) whose name starts with test_<prefix>."""
    starts = tuple("test_" + p for p in prefixes)
    for name, fn in inspect.getmembers(pins, inspect.isfunction):
        if not name.startswith(starts):
            continue
        marks = [m for m in getattr(fn, "pytestmark", []) if m.name == "parametrize"]
        if not marks:
            yield name, fn
            continue
        assert len(marks) == 1, name
        argname, values = marks[0].args
        for v in values:
            yield f"{name}[{v}]", (lambda fn=fn, argname=argname, v=v: fn(**{argname: v}))


def _failures(monkeypatch, module, prefixes):
    monkeypatch.setattr(pins, "oracle", module)
    failed, ran = [], 0
    for name, call in _pin_calls(prefixes):
        ran += 1
        try:
            call()
        except Exception:  # an assertion, or arithmetic the pin cannot carry out
            failed.append(name)
    return failed, ran


@pytest.mark.parametrize("prefixes", sorted({m[3] for m in MUTANTS}))
def test_selected_pins_pass_on_the_real_oracle(monkeypatch, prefixes):
    import oracle
    failed, ran = _failures(monkeypatch, oracle, prefixes)
    assert ran > 0 and not failed, failed


@pytest.mark.filterwarnings("ignore::RuntimeWarning")  # a slip may divide by zero: that fails a pin too
@pytest.mark.parametrize("case,old,new,prefixes", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_fails_a_pin(monkeypatch, case, old, new, prefixes):
    failed, ran = _failures(monkeypatch, _mutant(old, new), prefixes)
    assert ran > 0
    assert failed, f"{case}: no pin among {ran} caught the planted mistake"
