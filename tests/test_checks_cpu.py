"""The GPU parity checks are not vacuous: each accepts the oracle's own values
rounded as the kernels round them, and rejects an output that is off by a bit
more than its stated bound (CPU only; the inputs come from the oracle)."""

import numpy as np
import pytest
import torch

import oracle
from _checks import DX_TERM_SCALE_MAX_H, Guarded, check_dw, check_io, check_mxfp8, check_rstd, dx_scale


def _ref(shape=(8, 64), seed=0):
    rng = np.random.default_rng(seed)
    x, r = rng.normal(size=shape), rng.normal(size=shape)
    w = 1 + 0.1 * rng.normal(size=shape[-1])
    y, _, rstd = oracle.rmsnorm_fwd(x, r, w, 1e-6)
    return y, rstd


def test_check_io_bf16_bound():
    y, _ = _ref()
    check_io(oracle.round_to_bf16(y), y, "bf16", "rounded once")
    bad = y.copy()
    bad[3, 5] = y[3, 5] * 1.02 + np.sign(y[3, 5]) * 1e-3   # just past 1e-2 |ref| + 1e-3
    with pytest.raises(AssertionError, match="1 of 512"):
        check_io(bad, y, "bf16", "one element off")
    near0 = np.zeros((2, 4))
    with pytest.raises(AssertionError):
        check_io(near0 + 1.5e-3, near0, "bf16", "absolute floor")
    check_io(near0 + 0.9e-3, near0, "bf16", "inside the absolute floor")


def test_check_io_f32_bound_and_non_finite():
    y, _ = _ref()
    check_io(oracle.round_to_f32(y), y, "f32", "rounded once")
    bad = y.copy()
    bad.flat[100] += 2e-5 * np.max(np.abs(y))
    with pytest.raises(AssertionError, match="normwise"):
        check_io(bad, y, "f32", "one element off")
    nan = y.copy()
    nan[0, 0] = np.nan
    with pytest.raises(AssertionError, match="non-finite"):
        check_io(nan, y, "f32", "nan")
    with pytest.raises(AssertionError):
        check_io(y[:, :-1], y, "f32", "shape")


def test_check_dw_and_rstd_bounds():
    rng = np.random.default_rng(1)
    dw = rng.normal(size=256)
    noise = rng.normal(size=256)
    noise *= np.linalg.norm(dw) / np.linalg.norm(noise)
    check_dw(dw + 5e-4 * noise, dw)
    with pytest.raises(AssertionError, match="rel-L2"):
        check_dw(dw + 2e-3 * noise, dw)
    _, rstd = _ref()
    check_rstd(rstd * (1 + 5e-6), rstd)
    with pytest.raises(AssertionError, match="max rel err"):
        check_rstd(rstd * (1 + 2e-5), rstd)


def test_check_mxfp8_accepts_the_oracle_and_rejects_a_flipped_code_or_scale():
    y, _ = _ref((8, 128), seed=2)
    q, sc = oracle.mxfp8_quantize(y)
    check_mxfp8(torch.from_numpy(q), torch.from_numpy(sc), y, "oracle codes")
    # one code moved by one E4M3 step: the block maximum, away from any rounding midpoint
    # (asserted), so that no value within the 1e-5 window rounds to the moved code
    b = 3
    j = int(np.argmax(np.abs(y[1, 32 * b:32 * b + 32]))) + 32 * b
    t = y[1, j] / 2.0 ** (int(sc[1, b]) - 127)
    assert oracle.round_to_e4m3(t * (1 - 1e-5)) == oracle.round_to_e4m3(t * (1 + 1e-5))
    q2 = q.copy()
    q2[1, j] = q2[1, j] - 1 if (q2[1, j] & 0x7) else q2[1, j] + 1
    with pytest.raises(AssertionError, match="codes off"):
        check_mxfp8(torch.from_numpy(q2), torch.from_numpy(sc), y, "flipped code")
    sc2 = sc.copy()
    sc2[5, 2] += 1
    with pytest.raises(AssertionError, match="scale bytes off"):
        check_mxfp8(torch.from_numpy(q), torch.from_numpy(sc2), y, "scale off by one")
    with pytest.raises(AssertionError):
        check_mxfp8(torch.from_numpy(q[:, :96]), torch.from_numpy(sc[:, :3]), y, "shape")


def test_guarded_band_detects_a_write_outside_the_region():
    g = Guarded((4, 8), torch.float32, device="cpu")
    g.tensor.fill_(1.0)
    assert g.intact()
    g.raw[g.band + g.n] = 0.0   # one element past the end
    assert not g.intact()
    h = Guarded((16,), torch.bfloat16, device="cpu")
    h.raw[h.band - 1] = 2.0     # one element before the start
    assert not h.intact()


def test_f32_dx_uses_max_ref_beyond_sixteen_channels():
    # The largest-term normaliser is only offered for rows of at most 16
    # channels; at the workload widths dX is held to 1e-5 of max|dx_ref|.
    rng = np.random.default_rng(5)
    for H, term in ((1, True), (DX_TERM_SCALE_MAX_H, True), (DX_TERM_SCALE_MAX_H + 1, False), (896, False)):
        T = 7
        x, dy, dres = rng.normal(size=(T, H)), rng.normal(size=(T, H)), rng.normal(size=(T, H))
        w = 1 + 0.1 * rng.normal(size=H)
        _, h, rstd = oracle.rmsnorm_fwd(x, None, w, 1e-5)
        dx_ref, _ = oracle.rmsnorm_bwd(dy, dres, h, w, 1e-5)
        sc = dx_scale(dy, w, rstd, dres)
        assert (sc is not None) == term, (H, sc)
        if not term:
            bad = dx_ref.copy()
            bad.flat[3] += 1.5e-5 * np.max(np.abs(dx_ref))
            with pytest.raises(AssertionError, match="normwise"):
                check_io(bad, dx_ref, "f32", f"dx H={H}", scale=sc)
            ok = dx_ref.copy()
            ok.flat[3] += 0.9e-5 * np.max(np.abs(dx_ref))
            check_io(ok, dx_ref, "f32", f"dx H={H}", scale=sc)
    # LayerNorm's three terms at 16 channels, none beyond
    dy16 = rng.normal(size=(3, 16))
    assert dx_scale(dy16, np.ones(16), np.ones(3), terms=3) == pytest.approx(3 * np.max(np.abs(dy16)))
    assert dx_scale(rng.normal(size=(3, 17)), np.ones(17), np.ones(3), terms=3) is None
