"""The Python binding checks every tensor against the sizes it passes to the C ABI.

The entry points receive bare pointers, so a tensor smaller than the sizes passed
would be read or written out of bounds on the GPU.  These checks run before any
CUDA call or library call, so they are exercised here with CPU tensors: each bad
call must raise and name the offending argument.
"""

import pytest
import torch

import rmsnorm_fwd_bwd_03_gb300 as gb

T, H = 4, 64
bf, f32 = torch.bfloat16, torch.float32


def _t(*shape, dtype=bf):
    return torch.zeros(shape, dtype=dtype)


def test_rmsnorm_fwd_rejects_mismatched_tensors():
    x, w = _t(T, H), _t(H)
    with pytest.raises(ValueError, match="weight"):
        gb.rmsnorm_fwd(x, _t(H - 1), 1e-6)
    with pytest.raises(ValueError, match="residual"):
        gb.rmsnorm_fwd(x, w, 1e-6, _t(T, H, dtype=f32))
    with pytest.raises(ValueError, match="residual"):
        gb.rmsnorm_fwd(x, w, 1e-6, _t(T + 1, H))
    with pytest.raises(ValueError, match="y"):
        gb.rmsnorm_fwd(x, w, 1e-6, y=_t(T, H // 2))
    with pytest.raises(ValueError, match="residual_out"):
        gb.rmsnorm_fwd(x, w, 1e-6, _t(T, H), residual_out=_t(T, H, dtype=f32))
    with pytest.raises(TypeError, match="rstd"):
        gb.rmsnorm_fwd(x, w, 1e-6, rstd=_t(T))
    with pytest.raises(ValueError, match="rstd"):
        gb.rmsnorm_fwd(x, w, 1e-6, rstd=_t(T - 1, dtype=f32))
    with pytest.raises(ValueError, match="weight"):
        gb.rmsnorm_fwd_mxfp8(x, _t(2 * H), 1e-6)


def test_rmsnorm_bwd_and_finalize_reject_mismatched_tensors():
    dy, h, w, rstd = _t(T, H), _t(T, H), _t(H), _t(T, dtype=f32)
    with pytest.raises(ValueError, match="h"):
        gb.rmsnorm_bwd(dy, _t(T, H, dtype=f32), w, rstd)
    with pytest.raises(ValueError, match="dresidual_out"):
        gb.rmsnorm_bwd(dy, h, w, rstd, _t(T, H + 8))
    with pytest.raises(ValueError, match="dx"):
        gb.rmsnorm_bwd(dy, h, w, rstd, dx=_t(T - 1, H))
    with pytest.raises(ValueError, match="rstd"):
        gb.rmsnorm_bwd(dy, h, w, _t(2 * T, dtype=f32))
    with pytest.raises(ValueError, match="dw_partial"):
        gb.rmsnorm_bwd(dy, h, w, rstd, dw_partial=_t(8, H - 1, dtype=f32))
    with pytest.raises(ValueError, match="dw_partial"):
        gb.rmsnorm_bwd(dy, h, w, rstd, dw_partial=_t(8, H))  # bf16, not float32
    with pytest.raises(ValueError, match="dw_partial"):
        gb.rmsnorm_dw_finalize(_t(3, H, dtype=f32), 4)       # fewer rows than P
    with pytest.raises(ValueError, match="dw"):
        gb.rmsnorm_dw_finalize(_t(3, H, dtype=f32), 3, dw=_t(H - 1, dtype=f32))
    with pytest.raises(ValueError, match="dw"):
        gb.rmsnorm_bwd_noalloc(dy, h, w, rstd, dw=_t(H + 1, dtype=f32))


def test_layernorm_rejects_mismatched_tensors():
    x, w = _t(T, H), _t(H)
    with pytest.raises(ValueError, match="bias"):
        gb.layernorm_fwd(x, w, 1e-5, bias=_t(H, dtype=f32))
    with pytest.raises(ValueError, match="mean"):
        gb.layernorm_fwd(x, w, 1e-5, mean=_t(T + 1, dtype=f32))
    mean, rstd = _t(T, dtype=f32), _t(T, dtype=f32)
    with pytest.raises(ValueError, match="dwdb_partial"):
        gb.layernorm_bwd(x, x, w, mean, rstd, dwdb_partial=_t(8, H, dtype=f32))  # needs 2H columns
    with pytest.raises(ValueError, match="db"):
        gb.layernorm_dwdb_finalize(_t(2, 2 * H, dtype=f32), 2, db=_t(2 * H, dtype=f32))


def test_rope_rejects_mismatched_tensors():
    Hq, Hk, D = 4, 2, 16
    q, k = _t(T, Hq, D), _t(T, Hk, D)
    pos, table = torch.zeros(T, dtype=torch.int32), _t(32, D // 2, 2, dtype=f32)
    with pytest.raises(ValueError, match="q"):
        gb.rope_fwd(_t(T, Hq * D), k, pos, table)
    with pytest.raises(ValueError, match="k"):
        gb.rope_fwd(q, _t(T, Hk, D + 2), pos, table)
    with pytest.raises(TypeError, match="positions"):
        gb.rope_fwd(q, k, torch.zeros(T, dtype=torch.int64), table)
    with pytest.raises(ValueError, match="positions"):
        gb.rope_fwd(q, k, torch.zeros(T - 1, dtype=torch.int32), table)
    with pytest.raises(ValueError, match="cos_sin"):
        gb.rope_fwd(q, k, pos, _t(32, D, 2, dtype=f32))
    with pytest.raises(ValueError, match="cos_sin"):
        gb.rope_fwd(q, k, pos, _t(32, D // 2, 2))  # bf16 table
    with pytest.raises(ValueError, match="q_out"):
        gb.rope_fwd(q, k, pos, table, q_out=_t(T, Hq, D, dtype=f32))
    with pytest.raises(ValueError, match="k_out"):
        gb.rope_bwd(q, k, pos, table, dk_in=_t(T, Hk + 1, D))
    with pytest.raises(TypeError, match="cos_sin"):
        gb.rope_table(32, D, 1e4, out=_t(32, D // 2, 2))
    with pytest.raises(ValueError, match="positions"):
        gb.positions_from_cu_seqlens(torch.tensor([0, T], dtype=torch.int32), T, out=_t(T + 1, dtype=torch.int32))


def test_gated_units_reject_mismatched_tensors():
    I = 32
    g, u = _t(T, I), _t(T, I)
    with pytest.raises(ValueError, match="out"):
        gb.swiglu_fwd(g, u, out=_t(T, I // 2))
    with pytest.raises(ValueError, match="dup"):
        gb.swiglu_bwd(g, g, u, dup=_t(T, I, dtype=f32))
    with pytest.raises(ValueError, match="up"):
        gb.glu_fwd(g, _t(T, I + 1))
    with pytest.raises(ValueError, match="out"):
        gb.glu_fwd(g, u, "relu", out=_t(T + 1, I))
    with pytest.raises(ValueError, match="dgate"):
        gb.glu_bwd(g, g, u, "gelu_tanh", dgate=_t(T, I - 8))
    with pytest.raises(ValueError, match="up"):
        gb.glu_fwd_mxfp8(g, _t(T, I, dtype=f32))
    with pytest.raises(ValueError, match="out"):
        gb.act_fwd(_t(100), "silu", out=_t(99))
    with pytest.raises(ValueError, match="dy"):
        gb.act_bwd(_t(99), _t(100), "silu")


def test_missing_library_raises_instead_of_falling_back(monkeypatch, tmp_path):
    # There is no CPU implementation behind the binding: with the shared library
    # absent, a call that passes its argument checks raises.
    monkeypatch.setattr(gb, "_lib", None)
    monkeypatch.setattr(gb, "_LIB_PATH", str(tmp_path / "libgbln.so"))
    with pytest.raises(RuntimeError, match="libgbln.so not found"):
        gb.library()
    with pytest.raises(RuntimeError, match="no fallback"):
        gb.rmsnorm_bwd_num_partials(T, H)
    with pytest.raises(RuntimeError, match="no fallback"):
        gb.version()
