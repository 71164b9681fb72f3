"""Tolerances and sampling shared by the GPU parity tests.

Bounds (written here, used everywhere):
  * float32 I/O: normwise maximum relative error  max|gpu - ref| / max|ref| <= 1e-5
    (elementwise relative error is ill-posed where outputs cross zero); only the
    normalisation dX of rows of at most DX_TERM_SCALE_MAX_H (16) channels is
    normalised by its largest term instead (``dx_scale``);
  * bf16 I/O: elementwise |gpu - ref| <= 1e-2 * |ref| + 1e-3, against the float64
    oracle value before any rounding to bf16;
  * RMSNorm weight gradient (float32 [H]): ||gpu - ref||_2 / ||ref||_2 <= 1e-3;
  * the residual-stream output h and integer positions: bit-exact;
  * rstd (float32 in both I/O types): elementwise relative 1e-5.
"""

import numpy as np
import torch

F32_NORMWISE = 1e-5
BF16_REL = 1e-2
BF16_ABS = 1e-3
DW_REL_L2 = 1e-3
RSTD_REL = 1e-5


def to64(t: torch.Tensor) -> np.ndarray:
    """Exact float64 copy of a float32 / bf16 tensor (any device)."""
    return t.detach().float().cpu().numpy().astype(np.float64)


def check_io(got, ref, io: str, what: str, scale=None):
    """``scale`` (float32 only) replaces max|ref| as the normalisation, and only
    where the output is a difference of larger terms that cancel by construction:
    the normalisation backward passes of rows no wider than DX_TERM_SCALE_MAX_H
    (``dx_scale`` returns None beyond that, which keeps max|ref|).  At H = 1 the
    RMSNorm dX terms rstd*g and rstd*n*c cancel to O(eps), and no float32
    arithmetic meets 1e-5 of the cancelled value; from a few dozen channels on
    the terms no longer cancel systematically and the stated bound applies."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    if got.size == 0:
        return
    if io == "f32":
        if scale is None:
            scale = np.max(np.abs(ref))
        scale = max(float(scale), float(np.max(np.abs(ref))))
        err = np.max(np.abs(got - ref)) / (scale if scale > 0 else 1.0)
        assert err <= F32_NORMWISE, f"{what}: normwise max rel err {err:.3e} > {F32_NORMWISE}"
    else:
        err = np.abs(got - ref)
        bound = BF16_REL * np.abs(ref) + BF16_ABS
        bad = err > bound
        if bad.any():
            i = np.unravel_index(np.argmax(err - bound), err.shape)
            raise AssertionError(
                f"{what}: {int(bad.sum())} of {err.size} elements out of bound; worst at {i}: "
                f"got {got[i]!r} ref {ref[i]!r}")


# Widest row whose normalisation-backward dX may be normalised by its largest
# term instead of max|ref| (see check_io).
DX_TERM_SCALE_MAX_H = 16


def dx_scale(dy, w, rstd, dres=None, terms=1):
    """Largest term of a normalisation dX, for rows of at most DX_TERM_SCALE_MAX_H
    channels: terms * max over rows of rstd * |dy * w| (+ max|dres|); RMSNorm
    has one such term, LayerNorm three (g, its mean and n * mean(g n)).  None for
    wider rows, so that check_io normalises by max|ref| as stated."""
    dy = np.asarray(dy)
    if dy.ndim == 0 or dy.shape[-1] > DX_TERM_SCALE_MAX_H:
        return None
    s = terms * np.max(np.abs(dy * np.asarray(w)) * np.asarray(rstd)[..., None]) if dy.size else 0.0
    if dres is not None and np.size(dres):
        s += np.max(np.abs(dres))
    return s


def check_dw(got, ref, what="dW"):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert rel <= DW_REL_L2, f"{what}: rel-L2 {rel:.3e} > {DW_REL_L2}"


def check_rstd(got, ref, what="rstd"):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rel = np.max(np.abs(got - ref) / np.abs(ref)) if ref.size else 0.0
    assert rel <= RSTD_REL, f"{what}: max rel err {rel:.3e} > {RSTD_REL}"


def sample_rows(T: int, n: int, seed: int = 123, extra=()) -> np.ndarray:
    """Seeded sample of row indices plus the first and last rows and any `extra` rows."""
    rng = np.random.default_rng(seed)
    rows = set(rng.choice(T, size=min(n, T), replace=False).tolist()) if T else set()
    rows.update(int(r) for r in extra if 0 <= r < T)
    if T:
        rows.update([0, T - 1])
    return np.array(sorted(rows), dtype=np.int64)


class Guarded:
    """A CUDA buffer with canary bands before and after the usable region."""

    BAND = 4096  # bytes on each side

    def __init__(self, shape, dtype, device="cuda", fill=0xA5):
        n = int(np.prod(shape)) if len(shape) else 1
        esz = torch.empty((), dtype=dtype).element_size()
        band = self.BAND // esz
        self.raw = torch.empty(n + 2 * band, dtype=dtype, device=device)
        self.raw.view(torch.uint8).fill_(fill)
        self.band = band
        self.n = n
        self.fill = fill
        self.tensor = self.raw[band:band + n].view(shape)

    def intact(self) -> bool:
        b = self.raw.view(torch.uint8)
        esz = self.raw.element_size()
        head = b[: self.band * esz]
        tail = b[(self.band + self.n) * esz:]
        return bool((head == self.fill).all()) and bool((tail == self.fill).all())


# MXFP8 codes are integers decided by floating point.  The kernel decides them
# from its float32 result, the oracle from the exact one; the two differ by at
# most the float32 bound above: relative 1e-5 (plus, where an activation
# cancels, an absolute term relative to the block's largest magnitude:
# ``abs_rel``).
# Wherever moving the exact value by that much cannot change a decision, the
# code (and the scale) must be identical; where it can, the kernel's must lie
# between the two outcomes.
MX_REL = 1e-5


def check_mxfp8(q_gpu, sc_gpu, v64, what: str, rel: float = MX_REL, abs_rel: float = 0.0,
                max_ambiguous: float = 1e-3):
    import oracle
    q = q_gpu.cpu().numpy()
    sc = sc_gpu.cpu().numpy()
    v = np.asarray(v64, dtype=np.float64)
    T, N = v.shape
    assert q.shape == (T, N) and sc.shape == (T, N // 32), (what, q.shape, sc.shape)
    vb = v.reshape(T, N // 32, 32)
    amax = np.abs(vb).max(axis=-1)
    se_lo = oracle.mx_scale_exponent(amax * (1 - rel))
    se_hi = oracle.mx_scale_exponent(amax * (1 + rel))
    se = sc.astype(np.int64) - 127
    bad = (se != se_lo) & (se != se_hi)
    assert not bad.any(), f"{what}: {bad.sum()} scale bytes off, first at {np.argwhere(bad)[0]}"
    t = vb / np.ldexp(1.0, se)[..., None]                     # exact values in the kernel's scale
    win = rel * np.abs(t) + abs_rel * (amax / np.ldexp(1.0, se))[..., None]
    lo = oracle.round_to_e4m3(t - win)                         # rounding is monotone
    hi = oracle.round_to_e4m3(t + win)
    got = oracle.e4m3_decode(q.reshape(T, N // 32, 32))
    bad = ~((got >= lo) & (got <= hi))
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {bad.sum()} codes off; first at {i}: gpu {got[i]!r}, "
                             f"exact {t[i]!r} -> [{lo[i]!r}, {hi[i]!r}]")
    amb = int((lo != hi).sum())
    if lo.size >= 4096:  # too few codes say nothing about the rate
        assert amb <= max_ambiguous * lo.size, f"{what}: {amb} of {lo.size} codes sit on a decision boundary"
