"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test fixes the oracle to a closed form, an invariant, a hand-worked value
(``tests/golden/``), an independent library routine or a finite difference, so
that a dropped term, a wrong sign, a wrong pairing or a swapped operand in the
oracle fails at least one of them.  CPU only.
"""

import cmath
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    out = []
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                out.append([float(v) for v in line.split()])
    return out


# ---------------------------------------------------------------------------
# bf16 rounding
# ---------------------------------------------------------------------------

def test_bf16_rounding_hand_cases():
    for num, den, enum, eden in _rows("bf16_rounding.txt"):
        got = oracle.round_to_bf16(np.array([num / den]))[0]
        assert got == enum / eden, (num, den, got)


def test_bf16_rounding_matches_torch_conversion():
    # torch's float32 -> bfloat16 cast is an independent round-to-nearest-even.
    g = torch.Generator().manual_seed(1)
    v = torch.randn(200000, generator=g) * torch.exp(torch.randn(200000, generator=g) * 4)
    ref = v.to(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.round_to_bf16(v.to(torch.float64).numpy())
    assert np.array_equal(got, ref)


def test_bf16_sum_rounding_matches_torch_on_bf16_pairs():
    # h = round(x + r) from double equals torch's (fp32 add, then RNE to bf16):
    # float32 has more than 2*8+2 bits, so its intermediate rounding is innocuous.
    g = torch.Generator().manual_seed(2)
    x = (torch.randn(100000, generator=g) * 3).to(torch.bfloat16)
    r = (torch.randn(100000, generator=g) * torch.exp(torch.randn(100000, generator=g) * 3)).to(torch.bfloat16)
    ref = (x.float() + r.float()).to(torch.bfloat16).double().numpy()
    got = oracle.round_to_bf16(x.double().numpy() + r.double().numpy())
    assert np.array_equal(got, ref)


def test_round_io_matches_torch_casts():
    # round_io picks the I/O precision: torch's float32 and bfloat16 casts are
    # independent round-to-nearest-even implementations; None keeps float64.
    g = torch.Generator().manual_seed(4)
    v = (torch.randn(50000, generator=g, dtype=torch.float64) * 10)
    a = v.numpy()
    assert np.array_equal(oracle.round_io(a, "f32"), v.to(torch.float32).double().numpy())
    assert np.array_equal(oracle.round_io(a, "bf16"), v.to(torch.bfloat16).double().numpy())
    assert np.array_equal(oracle.round_io(a, None), a)
    assert not np.array_equal(oracle.round_io(a, "f32"), a)


# ---------------------------------------------------------------------------
# RMSNorm forward
# ---------------------------------------------------------------------------

def test_rmsnorm_single_channel_hand_values():
    for h, eps, w, y in _rows("rmsnorm_h1.txt"):
        got, _, _ = oracle.rmsnorm_fwd(np.array([[h]]), None, np.array([w]), eps)
        assert got[0, 0] == pytest.approx(y, rel=1e-15, abs=1e-15)


def test_rmsnorm_unit_rms_closed_form():
    rng = np.random.default_rng(0)
    x = rng.normal(size=(7, 33))
    r = rng.normal(size=(7, 33))
    w = 1 + 0.1 * rng.normal(size=33)
    for eps in (0.0, 1e-5, 0.3):
        y, h, rstd = oracle.rmsnorm_fwd(x, r, w, eps)
        ms = np.mean(h * h, axis=1)
        rms = np.sqrt(np.mean((y / w) ** 2, axis=1))
        assert np.allclose(rms, np.sqrt(ms / (ms + eps)), rtol=1e-13, atol=0)
        if eps == 0.0:
            assert np.allclose(rms, 1.0, rtol=1e-13)
        assert np.array_equal(h, x + r)  # io=None keeps the exact sum


def test_rmsnorm_scale_invariance_at_zero_eps():
    rng = np.random.default_rng(1)
    x = rng.normal(size=(5, 16))
    w = rng.normal(size=16)
    y1, _, _ = oracle.rmsnorm_fwd(x, None, w, 0.0)
    y2, _, _ = oracle.rmsnorm_fwd(37.5 * x, None, w, 0.0)
    assert np.allclose(y1, y2, rtol=1e-13, atol=1e-14)


def test_rmsnorm_residual_rounded_before_normalising():
    # With bf16 I/O the stored h is the bf16 sum, and y normalises that h.
    x = np.array([[1.0, 1.0]])
    r = np.array([[2.0 ** -8, 0.0]])  # 1 + 2^-8 is a tie: rounds to 1
    y, h, rstd = oracle.rmsnorm_fwd(x, r, np.ones(2), 0.0, io="bf16")
    assert np.array_equal(h, [[1.0, 1.0]])
    assert np.allclose(y, [[1.0, 1.0]], rtol=1e-15)
    assert rstd[0] == pytest.approx(1.0, rel=1e-15)


# ---------------------------------------------------------------------------
# RMSNorm backward
# ---------------------------------------------------------------------------

def _rms_loss(x, r, w, eps, dy, dres):
    y, h, _ = oracle.rmsnorm_fwd(x, r, w, eps)
    return float(np.sum(dy * y) + np.sum(dres * h))


@pytest.mark.parametrize("H", [1, 5, 8])
def test_rmsnorm_bwd_central_differences(H):
    rng = np.random.default_rng(10 + H)
    T, eps, d = 3, 1e-2, 1e-6
    x = rng.normal(size=(T, H))
    r = rng.normal(size=(T, H))
    w = 1 + 0.1 * rng.normal(size=H)
    dy = rng.normal(size=(T, H))
    dres = rng.normal(size=(T, H))
    _, h, _ = oracle.rmsnorm_fwd(x, r, w, eps)
    dx, dw = oracle.rmsnorm_bwd(dy, dres, h, w, eps)
    fd_x = np.zeros_like(x)
    for idx in np.ndindex(x.shape):
        xp = x.copy(); xp[idx] += d
        xm = x.copy(); xm[idx] -= d
        fd_x[idx] = (_rms_loss(xp, r, w, eps, dy, dres) - _rms_loss(xm, r, w, eps, dy, dres)) / (2 * d)
    fd_w = np.zeros_like(w)
    for j in range(H):
        wp = w.copy(); wp[j] += d
        wm = w.copy(); wm[j] -= d
        fd_w[j] = (_rms_loss(x, r, wp, eps, dy, dres) - _rms_loss(x, r, wm, eps, dy, dres)) / (2 * d)
    assert np.allclose(dx, fd_x, rtol=1e-7, atol=1e-8)
    assert np.allclose(dw, fd_w, rtol=1e-7, atol=1e-8)


def test_rmsnorm_bwd_orthogonality_closed_form():
    # sum_j dh_j h_j = rstd * sum(g h) * eps / (ms + eps); zero when eps = 0.
    rng = np.random.default_rng(3)
    h = rng.normal(size=(4, 12))
    w = rng.normal(size=12)
    dy = rng.normal(size=(4, 12))
    for eps in (0.0, 0.5):
        dh, _ = oracle.rmsnorm_bwd(dy, None, h, w, eps)
        ms = np.mean(h * h, axis=1)
        rstd = 1 / np.sqrt(ms + eps)
        lhs = np.sum(dh * h, axis=1)
        rhs = rstd * np.sum(dy * w * h, axis=1) * eps / (ms + eps)
        assert np.allclose(lhs, rhs, rtol=1e-10, atol=1e-12)


def test_rmsnorm_dw_brute_force_and_chunked():
    rng = np.random.default_rng(4)
    T, H, eps = 9, 6, 1e-5
    h = rng.normal(size=(T, H))
    dy = rng.normal(size=(T, H))
    w = rng.normal(size=H)
    _, dw = oracle.rmsnorm_bwd(dy, None, h, w, eps)
    brute = [0.0] * H
    for t in range(T):
        rstd = 1.0 / math.sqrt(sum(v * v for v in h[t]) / H + eps)
        for j in range(H):
            brute[j] += dy[t, j] * h[t, j] * rstd
    assert np.allclose(dw, brute, rtol=1e-13)
    assert np.allclose(oracle.rmsnorm_dw(dy, h, eps, rows_per_chunk=2), brute, rtol=1e-13)


def test_rmsnorm_dw_sum_of_shards_equals_full():
    # The weight gradient of a token-sharded batch is the sum of per-shard gradients.
    rng = np.random.default_rng(5)
    T, H, eps = 40, 10, 1e-6
    h = rng.normal(size=(T, H))
    dy = rng.normal(size=(T, H))
    full = oracle.rmsnorm_dw(dy, h, eps)
    cuts = [0, 7, 19, 33, 40]
    parts = sum(oracle.rmsnorm_dw(dy[a:b], h[a:b], eps) for a, b in zip(cuts[:-1], cuts[1:]))
    assert np.allclose(parts, full, rtol=1e-12)


# ---------------------------------------------------------------------------
# RoPE
# ---------------------------------------------------------------------------

def test_rope_hand_values_d4():
    for row in _rows("rope_d4.txt"):
        pos, x, y = row[0], np.array(row[1:5]), np.array(row[5:9])
        got = oracle.rope_fwd(x.reshape(1, 1, 4), np.array([pos]), 10000.0)
        assert np.allclose(got.reshape(4), y, rtol=0, atol=1e-15)


def test_rope_inv_freq_values():
    f = oracle.rope_inv_freq(8, 10000.0)
    assert np.allclose(f, [1.0, 0.1, 0.01, 0.001], rtol=1e-15)


def test_rope_equals_complex_multiplication():
    # Pair (i, i + D/2) as the complex number x_i + j x_{i+D/2}, turned by exp(j pos theta_i).
    rng = np.random.default_rng(6)
    T, Hh, D, theta = 5, 3, 8, 500000.0
    x = rng.normal(size=(T, Hh, D))
    pos = rng.integers(0, 20000, size=T)
    got = oracle.rope_fwd(x, pos, theta)
    for t in range(T):
        for hh in range(Hh):
            for i in range(D // 2):
                z = complex(x[t, hh, i], x[t, hh, i + D // 2])
                zr = z * cmath.exp(1j * pos[t] * theta ** (-2.0 * i / D))
                assert got[t, hh, i] == pytest.approx(zr.real, abs=1e-11)
                assert got[t, hh, i + D // 2] == pytest.approx(zr.imag, abs=1e-11)


def test_rope_position_zero_is_identity_and_norm_preserved():
    rng = np.random.default_rng(7)
    x = rng.normal(size=(6, 4, 64))
    assert np.array_equal(oracle.rope_fwd(x, np.zeros(6), 1e6), x)
    pos = np.array([1, 2, 255, 4095, 8191, 16383])
    y = oracle.rope_fwd(x, pos, 1e6)
    pair_in = x[..., :32] ** 2 + x[..., 32:] ** 2
    pair_out = y[..., :32] ** 2 + y[..., 32:] ** 2
    assert np.allclose(pair_in, pair_out, rtol=1e-12)


def test_rope_relative_position():
    rng = np.random.default_rng(8)
    D, theta = 16, 10000.0
    q = rng.normal(size=(1, 1, D))
    k = rng.normal(size=(1, 1, D))
    for m, n, s in [(5, 2, 100), (0, 9, 3000), (77, 77, 12)]:
        a = np.sum(oracle.rope_fwd(q, [m], theta) * oracle.rope_fwd(k, [n], theta))
        b = np.sum(oracle.rope_fwd(q, [m + s], theta) * oracle.rope_fwd(k, [n + s], theta))
        assert a == pytest.approx(b, rel=1e-10, abs=1e-12)


def test_rope_bwd_inverts_fwd_and_is_its_adjoint():
    rng = np.random.default_rng(9)
    x = rng.normal(size=(4, 3, 32))
    g = rng.normal(size=(4, 3, 32))
    pos = np.array([0, 3, 1000, 16000])
    y = oracle.rope_fwd(x, pos, 5e5)
    assert np.allclose(oracle.rope_bwd(y, pos, 5e5), x, rtol=1e-12, atol=1e-12)
    assert np.sum(y * g) == pytest.approx(np.sum(x * oracle.rope_bwd(g, pos, 5e5)), rel=1e-12)
    assert np.allclose(oracle.rope_bwd(x, pos, 5e5), oracle.rope_fwd(x, -pos, 5e5), atol=1e-13)


def test_rope_d2_is_plain_rotation_by_pos_radians():
    x = np.array([[[0.3, -1.7]]])
    for p in (1, 2, 7):
        y = oracle.rope_fwd(x, [p], 12345.0).reshape(2)
        c, s = math.cos(p), math.sin(p)
        assert y[0] == pytest.approx(0.3 * c + 1.7 * s, abs=1e-15)
        assert y[1] == pytest.approx(-1.7 * c + 0.3 * s, abs=1e-15)


# ---------------------------------------------------------------------------
# SwiGLU
# ---------------------------------------------------------------------------

def test_swiglu_hand_values():
    for g, u, out in _rows("silu.txt"):
        assert oracle.swiglu_fwd(np.array([g]), np.array([u]))[0] == pytest.approx(out, rel=1e-15, abs=1e-16)


def test_swiglu_special_cases():
    dout = np.array([1.5, -2.0])
    u = np.array([3.0, 0.25])
    g = np.zeros(2)
    dgate, dup = oracle.swiglu_bwd(dout, g, u)
    assert np.array_equal(oracle.swiglu_fwd(g, u), [0.0, 0.0])
    assert np.allclose(dgate, 0.5 * dout * u, rtol=1e-15)
    assert np.array_equal(dup, [0.0, 0.0])
    big = np.array([40.0])
    assert oracle.swiglu_fwd(big, np.array([2.0]))[0] == pytest.approx(80.0, rel=1e-15)
    assert oracle.swiglu_fwd(np.array([-40.0]), np.array([2.0]))[0] == pytest.approx(0.0, abs=1e-15)


def test_swiglu_scalar_brute_force():
    rng = np.random.default_rng(11)
    g = rng.normal(size=50) * 3
    u = rng.normal(size=50)
    dout = rng.normal(size=50)
    out = oracle.swiglu_fwd(g, u)
    dgate, dup = oracle.swiglu_bwd(dout, g, u)
    for i in range(50):
        e = math.exp(-g[i])
        assert out[i] == pytest.approx(g[i] / (1 + e) * u[i], rel=1e-14, abs=1e-300)
        # product rule on g / (1 + e^-g): (1 + e + g e) / (1 + e)^2
        assert dgate[i] == pytest.approx(dout[i] * u[i] * (1 + e + g[i] * e) / (1 + e) ** 2, rel=1e-12, abs=1e-300)
        assert dup[i] == pytest.approx(dout[i] * g[i] / (1 + e), rel=1e-14, abs=1e-300)


def test_swiglu_bwd_central_differences():
    rng = np.random.default_rng(12)
    g = rng.normal(size=20) * 2
    u = rng.normal(size=20)
    dout = rng.normal(size=20)
    dgate, dup = oracle.swiglu_bwd(dout, g, u)
    d = 1e-6
    for i in range(20):
        gp = g.copy(); gp[i] += d
        gm = g.copy(); gm[i] -= d
        fd = (np.sum(dout * oracle.swiglu_fwd(gp, u)) - np.sum(dout * oracle.swiglu_fwd(gm, u))) / (2 * d)
        assert dgate[i] == pytest.approx(fd, rel=1e-7, abs=1e-9)
        up_ = u.copy(); up_[i] += d
        um = u.copy(); um[i] -= d
        fd = (np.sum(dout * oracle.swiglu_fwd(g, up_)) - np.sum(dout * oracle.swiglu_fwd(g, um))) / (2 * d)
        assert dup[i] == pytest.approx(fd, rel=1e-7, abs=1e-9)


def test_rope_bwd_central_differences():
    rng = np.random.default_rng(13)
    x = rng.normal(size=(2, 2, 8))
    dout = rng.normal(size=(2, 2, 8))
    pos = np.array([3, 11])
    grad = oracle.rope_bwd(dout, pos, 100.0)
    d = 1e-6
    for idx in np.ndindex(x.shape):
        xp = x.copy(); xp[idx] += d
        xm = x.copy(); xm[idx] -= d
        fd = (np.sum(dout * oracle.rope_fwd(xp, pos, 100.0)) - np.sum(dout * oracle.rope_fwd(xm, pos, 100.0))) / (2 * d)
        assert grad[idx] == pytest.approx(fd, rel=1e-7, abs=1e-9)


# ---------------------------------------------------------------------------
# Positions of packed documents
# ---------------------------------------------------------------------------

def test_positions_brute_force():
    lengths = [3, 1, 5, 2]
    pos = oracle.positions_from_doc_lengths(lengths)
    expect = []
    for L in lengths:
        p = 0
        for _ in range(L):
            expect.append(p)
            p += 1
    assert pos.tolist() == expect
    cu = np.concatenate([[0], np.cumsum(lengths)])
    assert oracle.positions_from_cu_seqlens(cu).tolist() == expect
    for start in cu[:-1]:
        assert pos[start] == 0
    assert oracle.positions_from_doc_lengths([]).size == 0


# ---------------------------------------------------------------------------
# Gated / plain activations
# ---------------------------------------------------------------------------

def test_gelu_hand_values():
    for row in open(os.path.join(GOLDEN, "gelu.txt"), encoding="utf-8"):
        row = row.strip()
        if not row or row.startswith("#"):
            continue
        form, x, val, tol = row.split()
        name = "gelu_erf" if form == "erf" else "gelu_tanh"
        got = oracle.act(name, np.array([float(x)]))[0]
        assert got == pytest.approx(float(val), abs=float(tol) + 1e-300), (name, x, got)


def test_activation_identities():
    x = np.linspace(-6, 6, 241)
    # GeLU(x) - GeLU(-x) = x in both forms (Phi(x) + Phi(-x) = 1; tanh is odd)
    for name in ("gelu_erf", "gelu_tanh"):
        assert np.allclose(oracle.act(name, x) - oracle.act(name, -x), x, atol=1e-13)
    # the two GeLU forms agree to the known approximation error (< 1e-3 on this range)
    assert np.max(np.abs(oracle.act("gelu_erf", x) - oracle.act("gelu_tanh", x))) < 1e-3
    assert np.array_equal(oracle.act("relu", x), np.where(x > 0, x, 0.0))
    assert np.allclose(oracle.act("silu", x), x / (1 + np.exp(-x)), rtol=1e-14)
    # SwiGLU is the SiLU-gated unit
    u = np.cos(x)
    assert np.array_equal(oracle.glu_fwd("silu", x, u), oracle.swiglu_fwd(x, u))
    dg, du = oracle.glu_bwd("silu", np.sin(x), x, u)
    dg2, du2 = oracle.swiglu_bwd(np.sin(x), x, u)
    assert np.allclose(dg, dg2, rtol=1e-13, atol=1e-15) and np.allclose(du, du2, rtol=1e-13, atol=1e-15)


def test_activation_values_and_slopes_at_zero():
    # Every activation is 0 at 0.  The slopes there: 1/2 for SiLU and both GeLU
    # forms (sigma(0) = Phi(0) = 1/2); ReLU takes the subgradient 0.
    z = np.array([0.0])
    for name in ("silu", "gelu_tanh", "gelu_erf", "relu"):
        assert oracle.act(name, z)[0] == 0.0
    for name in ("silu", "gelu_tanh", "gelu_erf"):
        assert oracle.act_grad(name, z)[0] == 0.5
    assert oracle.act_grad("relu", z)[0] == 0.0
    assert oracle.act_grad("relu", np.array([1e-300]))[0] == 1.0


@pytest.mark.parametrize("name", ["silu", "gelu_tanh", "gelu_erf", "relu"])
def test_activation_grad_central_differences(name):
    x = np.array([-4.1, -2.3, -0.7, -0.05, 0.13, 0.9, 1.7, 3.2, 5.5])
    d = 1e-6
    fd = (oracle.act(name, x + d) - oracle.act(name, x - d)) / (2 * d)
    assert np.allclose(oracle.act_grad(name, x), fd, rtol=1e-7, atol=1e-9)
    g = np.array([0.4, -1.2, 2.5])
    u = np.array([1.5, -0.3, 0.8])
    dout = np.array([0.7, 2.0, -1.1])
    dgate, dup = oracle.glu_bwd(name, dout, g, u)
    for i in range(3):
        gp = g.copy(); gp[i] += d
        gm = g.copy(); gm[i] -= d
        fd = (np.sum(dout * oracle.glu_fwd(name, gp, u)) - np.sum(dout * oracle.glu_fwd(name, gm, u))) / (2 * d)
        assert dgate[i] == pytest.approx(fd, rel=1e-7, abs=1e-9)
        up_ = u.copy(); up_[i] += d
        um = u.copy(); um[i] -= d
        fd = (np.sum(dout * oracle.glu_fwd(name, g, up_)) - np.sum(dout * oracle.glu_fwd(name, g, um))) / (2 * d)
        assert dup[i] == pytest.approx(fd, rel=1e-7, abs=1e-9)


def test_rope_interleaved_is_a_permuted_rotate_half():
    # Interleaved pairing (2i, 2i+1) = rotate-half pairing after de-interleaving
    # the head (evens then odds) and re-interleaving the result.
    rng = np.random.default_rng(20)
    T, Hh, D = 4, 3, 16
    x = rng.normal(size=(T, Hh, D))
    pos = np.array([0, 7, 300, 9000])
    perm = np.concatenate([np.arange(0, D, 2), np.arange(1, D, 2)])
    inv = np.argsort(perm)
    via_half = oracle.rope_fwd(x[..., perm], pos, 1e4)[..., inv]
    assert np.allclose(oracle.rope_fwd(x, pos, 1e4, "interleaved"), via_half, rtol=1e-14, atol=1e-14)
    y = oracle.rope_fwd(x, pos, 1e4, "interleaved")
    assert np.allclose(oracle.rope_bwd(y, pos, 1e4, "interleaved"), x, atol=1e-12)


def test_rope_interleaved_equals_complex_multiplication():
    rng = np.random.default_rng(21)
    D, theta = 8, 500000.0
    x = rng.normal(size=(2, 1, D))
    pos = np.array([3, 12345])
    got = oracle.rope_fwd(x, pos, theta, "interleaved")
    for t in range(2):
        for i in range(D // 2):
            z = complex(x[t, 0, 2 * i], x[t, 0, 2 * i + 1]) * cmath.exp(1j * pos[t] * theta ** (-2.0 * i / D))
            assert got[t, 0, 2 * i] == pytest.approx(z.real, abs=1e-11)
            assert got[t, 0, 2 * i + 1] == pytest.approx(z.imag, abs=1e-11)
    # with two elements both pairings are the same rotation
    x2 = rng.normal(size=(3, 2, 2))
    p2 = np.array([1, 5, 9])
    assert np.array_equal(oracle.rope_fwd(x2, p2, 1e4, "interleaved"), oracle.rope_fwd(x2, p2, 1e4))


# ---------------------------------------------------------------------------
# LayerNorm
# ---------------------------------------------------------------------------

def test_layernorm_closed_forms():
    rng = np.random.default_rng(30)
    x = rng.normal(size=(6, 20)) * 3 + 5
    w = 1 + 0.1 * rng.normal(size=20)
    b = rng.normal(size=20)
    for eps in (0.0, 1e-5, 0.7):
        y, h, mean, rstd = oracle.layernorm_fwd(x, None, w, b, eps)
        n = (y - b) / w
        var = np.var(x, axis=1)
        assert np.allclose(np.mean(n, axis=1), 0.0, atol=1e-13)           # zero mean
        assert np.allclose(np.mean(n * n, axis=1), var / (var + eps), rtol=1e-12)  # unit variance at eps 0
        assert np.allclose(mean, np.mean(x, axis=1), rtol=1e-15)
    # shift invariance, and equality with RMSNorm on zero-mean rows
    y1, *_ = oracle.layernorm_fwd(x, None, w, b, 1e-5)
    y2, *_ = oracle.layernorm_fwd(x + 123.25, None, w, b, 1e-5)
    assert np.allclose(y1, y2, rtol=1e-10, atol=1e-10)
    z = x - np.mean(x, axis=1, keepdims=True)
    yl, *_ = oracle.layernorm_fwd(z, None, w, None, 1e-5)
    yr, _, _ = oracle.rmsnorm_fwd(z, None, w, 1e-5)
    assert np.allclose(yl, yr, rtol=1e-12, atol=1e-13)
    # one channel: the normalised value is 0, the output is the bias, dx = dres
    y, _, _, _ = oracle.layernorm_fwd(np.array([[3.0]]), None, np.array([2.0]), np.array([0.5]), 1e-5)
    assert y[0, 0] == 0.5
    dx, dw, db = oracle.layernorm_bwd(np.array([[1.5]]), np.array([[0.25]]), np.array([[3.0]]), np.array([2.0]), 1e-5)
    assert dx[0, 0] == pytest.approx(0.25, abs=1e-15) and dw[0] == 0.0 and db[0] == 1.5


def test_layernorm_residual_rounded_before_normalising():
    # As for RMSNorm: with bf16 I/O the stored h is the bf16 sum, and y normalises that h.
    x = np.array([[1.0, 3.0]])
    r = np.array([[2.0 ** -8, 0.0]])  # 1 + 2^-8 is a tie: rounds to 1
    y, h, mean, rstd = oracle.layernorm_fwd(x, r, np.ones(2), None, 0.0, io="bf16")
    assert np.array_equal(h, [[1.0, 3.0]])
    assert mean[0] == 2.0 and rstd[0] == 1.0
    assert np.array_equal(y, [[-1.0, 1.0]])


@pytest.mark.parametrize("H", [2, 5, 8])
def test_layernorm_bwd_central_differences(H):
    rng = np.random.default_rng(31 + H)
    T, eps, d = 3, 1e-2, 1e-6
    x = rng.normal(size=(T, H))
    r = rng.normal(size=(T, H))
    w = 1 + 0.1 * rng.normal(size=H)
    b = rng.normal(size=H)
    dy = rng.normal(size=(T, H))
    dres = rng.normal(size=(T, H))

    def loss(x, w, b):
        y, h, _, _ = oracle.layernorm_fwd(x, r, w, b, eps)
        return float(np.sum(dy * y) + np.sum(dres * h))

    _, h, _, _ = oracle.layernorm_fwd(x, r, w, b, eps)
    dx, dw, db = oracle.layernorm_bwd(dy, dres, h, w, eps)
    for arr, grad, which in ((x, dx, "x"), (w, dw, "w"), (b, db, "b")):
        for idx in np.ndindex(arr.shape):
            ap = arr.copy(); ap[idx] += d
            am = arr.copy(); am[idx] -= d
            args_p = {"x": x, "w": w, "b": b}; args_p[which] = ap
            args_m = {"x": x, "w": w, "b": b}; args_m[which] = am
            fd = (loss(args_p["x"], args_p["w"], args_p["b"]) - loss(args_m["x"], args_m["w"], args_m["b"])) / (2 * d)
            assert grad[idx] == pytest.approx(fd, rel=1e-6, abs=1e-8), (which, idx)


# ---------------------------------------------------------------------------
# MXFP8 (E4M3 elements, E8M0 block scales)
# ---------------------------------------------------------------------------

def _mx_golden():
    rounds, blocks = [], []
    with open(os.path.join(GOLDEN, "e4m3_mx.txt"), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            tag, *vals = line.split()
            (rounds if tag == "round" else blocks).append(vals)
    return rounds, blocks


def test_e4m3_hand_cases():
    rounds, _ = _mx_golden()
    assert len(rounds) >= 15
    for num, den, enum, eden, code in rounds:
        v = int(num) / int(den)
        got = oracle.round_to_e4m3(np.array([v]))[0]
        assert got == int(enum) / int(eden), (v, got)
        assert oracle.e4m3_encode(np.array([got]))[0] == int(code, 16), (v, got)


def test_mx_block_hand_cases():
    _, blocks = _mx_golden()
    for an, ad, vn, vd, se, sbyte, code0 in blocks:
        amax, v0 = int(an) / int(ad), int(vn) / int(vd)
        blk = np.zeros((1, 32))
        blk[0, 0] = v0
        blk[0, 17] = -amax  # the block maximum is a magnitude
        codes, scales = oracle.mxfp8_quantize(blk)
        assert oracle.mx_scale_exponent(np.array([amax]))[0] == int(se)
        assert scales[0, 0] == int(sbyte, 16)
        assert codes[0, 0] == int(code0, 16)


def test_e4m3_format_constants():
    vals = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    finite = vals[~np.isnan(vals)]
    assert np.isnan(vals).sum() == 2                    # 0x7f and 0xff only
    assert finite.max() == 448.0 and finite.min() == -448.0
    pos = finite[finite > 0]
    assert pos.min() == 2.0 ** -9                        # smallest subnormal
    assert np.sort(pos)[7] == 2.0 ** -6                  # 7 subnormals, then the smallest normal
    assert len(np.unique(finite)) == 253                 # +0 and -0 compare equal
    # every finite code decodes to a value that encodes back to the same code
    codes = np.arange(256, dtype=np.uint8)[~np.isnan(vals)]
    assert np.array_equal(oracle.e4m3_encode(oracle.e4m3_decode(codes)), codes)
    # NaN encodes to the all-ones exponent and mantissa (0x7f), which decodes to NaN
    with np.errstate(invalid="ignore"):  # the NaN's exponent and mantissa fields are computed, then replaced
        nan_code = oracle.e4m3_encode(np.array([np.nan]))[0]
    assert nan_code & 0x7F == 0x7F and np.isnan(oracle.e4m3_decode(np.array([nan_code]))[0])


def test_e4m3_rounding_matches_torch_cast_in_range():
    # torch's float8_e4m3fn cast (round to nearest even) is an independent
    # implementation; it does not saturate, so compare inside the finite range,
    # including every midpoint between neighbouring positive and negative values.
    rng = np.random.default_rng(41)
    v = rng.standard_normal(100_000) * np.exp(rng.uniform(-14, 6.5, 100_000))
    grid = np.sort(oracle.e4m3_decode(np.arange(256, dtype=np.uint8)))
    grid = grid[~np.isnan(grid)]
    mids = (grid[1:] + grid[:-1]) / 2
    v = np.concatenate([v, mids, grid])
    v = v[np.abs(v) <= 448.0]
    ref = torch.tensor(v, dtype=torch.float64).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.round_to_e4m3(v)
    assert np.array_equal(np.nan_to_num(got), np.nan_to_num(ref))


def test_e4m3_rounding_error_bound_and_saturation():
    rng = np.random.default_rng(43)
    v = rng.standard_normal(50_000) * np.exp(rng.uniform(-10, 6, 50_000))
    q = oracle.round_to_e4m3(v)
    mag = np.abs(v)
    # half a spacing: 2**(floor(log2|v|) - 4) in the normal range, 2**-10 below it
    e = np.floor(np.log2(np.maximum(mag, 2.0 ** -6)))
    half = np.ldexp(1.0, (e - 4).astype(int))
    inside = mag <= 448.0
    assert np.all(np.abs(q - v)[inside] <= half[inside])
    assert np.all(np.abs(q[~inside]) == 448.0)
    assert np.all(np.sign(q[q != 0]) == np.sign(v[q != 0]))


def test_mxfp8_block_structure():
    # Blocks run along the last axis: scaling one block changes only its own
    # scale byte (by the power of two) and leaves every code unchanged.
    rng = np.random.default_rng(47)
    v = rng.standard_normal((3, 96))
    c0, s0 = oracle.mxfp8_quantize(v)
    assert c0.shape == (3, 96) and s0.shape == (3, 3)
    w = v.copy()
    w[1, 32:64] *= 8.0
    c1, s1 = oracle.mxfp8_quantize(w)
    assert np.array_equal(c1, c0)
    assert s1[1, 1] == s0[1, 1] + 3
    s1[1, 1] = s0[1, 1]
    assert np.array_equal(s1, s0)
    # each block's largest magnitude lands in E4M3's top binade [256, 448]
    deq = oracle.mxfp8_dequantize(c0, s0)
    for t in range(3):
        for b in range(3):
            blk = v[t, 32 * b:32 * (b + 1)]
            k = int(np.argmax(np.abs(blk)))
            top = abs(oracle.e4m3_decode(c0[t, 32 * b + k]))
            assert 256.0 <= top <= 448.0
    # dequantized values are within half an E4M3 spacing (relative 2**-4) of the inputs,
    # unless saturated at the top of the range
    rel = np.abs(deq - v) / np.abs(v)
    sat = np.abs(oracle.e4m3_decode(c0)) == 448.0
    small = np.abs(oracle.e4m3_decode(c0)) < 2.0 ** -6
    assert np.all(rel[~sat & ~small] <= 2.0 ** -4)


def test_mxfp8_zero_block_and_scale_clamps():
    codes, scales = oracle.mxfp8_quantize(np.zeros((1, 32)))
    assert np.all(codes == 0) and scales[0, 0] == 0
    assert oracle.mx_scale_exponent(np.array([2.0 ** -140]))[0] == -127
    assert oracle.mx_scale_exponent(np.array([2.0 ** 140]))[0] == 127


def test_rmsnorm_fwd_mxfp8_is_quantized_rmsnorm():
    rng = np.random.default_rng(53)
    x = rng.standard_normal((4, 64))
    r = rng.standard_normal((4, 64))
    w = 1 + 0.1 * rng.standard_normal(64)
    codes, scales, y, h, rstd = oracle.rmsnorm_fwd_mxfp8(x, r, w, 1e-6, "bf16")
    y2, h2, rstd2 = oracle.rmsnorm_fwd(x, r, w, 1e-6, "bf16")
    assert np.array_equal(y, y2) and np.array_equal(h, h2) and np.array_equal(rstd, rstd2)
    c2, s2 = oracle.mxfp8_quantize(y2)
    assert np.array_equal(codes, c2) and np.array_equal(scales, s2)
    # y = w * h * rstd: with w == 1 and eps = 0 every row has unit RMS, so the
    # dequantized rows have RMS 1 to within the E4M3 relative error
    c3, s3, *_ = oracle.rmsnorm_fwd_mxfp8(x, None, np.ones(64), 0.0)
    deq = oracle.mxfp8_dequantize(c3, s3)
    assert np.allclose(np.sqrt(np.mean(deq ** 2, axis=1)), 1.0, rtol=2.0 ** -4)


def test_glu_fwd_mxfp8_is_quantized_glu():
    rng = np.random.default_rng(59)
    g = rng.standard_normal((2, 64))
    u = rng.standard_normal((2, 64))
    codes, scales = oracle.glu_fwd_mxfp8("silu", g, u)
    c2, s2 = oracle.mxfp8_quantize(g / (1 + np.exp(-g)) * u)
    assert np.array_equal(codes, c2) and np.array_equal(scales, s2)
