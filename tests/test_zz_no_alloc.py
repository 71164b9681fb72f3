"""The allocation-free RMSNorm backward (gbln_rmsnorm_bwd_noalloc) against the
float64 oracle and against the workspace version (gbln_rmsnorm_bwd +
gbln_rmsnorm_dw_finalize).

It serves callers that cannot allocate device memory when they run the backward
pass, so it keeps its dW partial sums in a fixed array inside the library instead
of a workspace argument.  The checks: two calls in a row on different inputs (the
second must not see the first's leftovers in the shared array) give dx and dW
within the tolerances of the other GPU tests, against the oracle where it runs in
seconds and against the workspace version everywhere; and shapes whose usual
partial-row count would overflow the array (P * H > 4 Mi floats), where the
entry point lowers the count, down to one or two partial rows near the largest
accepted width.  This file sorts last so that a run that stops at the first
failure has already run every other test; it also passes alone in a fresh
process.
"""

import numpy as np
import pytest
import torch

import oracle
import rmsnorm_fwd_bwd_03_gb300 as gb

from _checks import check_dw, check_io, dx_scale, to64

pytestmark = pytest.mark.gpu

SCRATCH_FLOATS = 4 << 20  # the library's fixed array of dW partials
EPS = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _library():
    from rmsnorm_fwd_bwd_03_gb300._build import build_library
    build_library()
    gb.library()


def _inputs(T, H, dt, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    h = torch.randn((T, H), generator=g, device="cuda").to(dt)
    dy = torch.randn((T, H), generator=g, device="cuda").to(dt)
    dres = torch.randn((T, H), generator=g, device="cuda").to(dt)
    w = (1 + 0.1 * torch.randn((H,), generator=g, device="cuda")).to(dt)
    rstd = torch.rsqrt(h.float().pow(2).mean(-1) + EPS)
    return dy, h, w, rstd, dres


def _check_against_oracle(dx, dw, dy, h, w, dres, io, what):
    dy64, h64, w64, dres64 = to64(dy), to64(h), to64(w), to64(dres)
    dx_ref, dw_ref = oracle.rmsnorm_bwd(dy64, dres64, h64, w64, EPS)
    rstd_ref = 1.0 / np.sqrt(np.mean(h64 * h64, axis=-1) + EPS)
    check_io(to64(dx), dx_ref, io, f"dx vs oracle, {what}", scale=dx_scale(dy64, w64, rstd_ref, dres64))
    check_dw(to64(dw), dw_ref, f"dW vs oracle, {what}")


# (T, H, dtype, oracle?): the bench-sized shapes are checked against the
# workspace version only (the oracle would take minutes on them).
SHAPES = [(16384, 1024, torch.bfloat16, False), (2048, 8192, torch.bfloat16, False),
          (256, 896, torch.float32, True), (77, 13, torch.bfloat16, True)]


@pytest.mark.parametrize("T,H,dt,with_oracle", SHAPES)
def test_noalloc_matches_workspace_version_twice(T, H, dt, with_oracle):
    io = "f32" if dt == torch.float32 else "bf16"
    for seed in (1, 2):  # two calls in a row through the same internal array
        dy, h, w, rstd, dres = _inputs(T, H, dt, seed)
        dx_ref, part, P = gb.rmsnorm_bwd(dy, h, w, rstd, dres)
        dw_ref = gb.rmsnorm_dw_finalize(part, P)
        dx, dw = gb.rmsnorm_bwd_noalloc(dy, h, w, rstd, dres)
        torch.cuda.synchronize()
        assert P * H <= SCRATCH_FLOATS  # the usual partial count fits the array
        check_io(to64(dx), to64(dx_ref), io, f"dx seed {seed}")
        check_dw(to64(dw), to64(dw_ref), f"dW seed {seed}")
        # same kernels, same partial count and summation order: bitwise equal too
        assert torch.equal(dx, dx_ref) and torch.equal(dw, dw_ref), f"not bitwise equal, seed {seed}"
        if with_oracle:
            _check_against_oracle(dx, dw, dy, h, w, dres, io, f"seed {seed}")


# Shapes whose usual partial-row count P would not fit the array, so the entry
# point lowers it to SCRATCH_FLOATS // H: float32 rows of 2^16 (element-wise
# kernel, P from 160 to 64, 2.5 rows per block), bf16 rows of 2^15 (P from the
# full grid to 128), and widths near the 4 Mi limit with three rows, where P
# drops to 2 and to 1.
REDUCED = [(160, 1 << 16, torch.float32), (640, 1 << 15, torch.bfloat16),
           (3, 1 << 21, torch.bfloat16), (3, SCRATCH_FLOATS - 8, torch.bfloat16)]


@pytest.mark.parametrize("T,H,dt", REDUCED)
def test_noalloc_reduced_partials_match_oracle(T, H, dt):
    io = "f32" if dt == torch.float32 else "bf16"
    P_usual = gb.rmsnorm_bwd_num_partials(T, H, dt)
    assert P_usual * H > SCRATCH_FLOATS, "shape does not reach the reduced-partials branch"
    for seed in (3, 4):
        dy, h, w, rstd, dres = _inputs(T, H, dt, seed)
        dx, dw = gb.rmsnorm_bwd_noalloc(dy, h, w, rstd, dres)
        dx_ws, part, P = gb.rmsnorm_bwd(dy, h, w, rstd, dres)
        dw_ws = gb.rmsnorm_dw_finalize(part, P)
        torch.cuda.synchronize()
        # dx does not depend on how rows are split into partials
        assert torch.equal(dx, dx_ws), f"dx seed {seed}"
        check_dw(to64(dw), to64(dw_ws), f"dW vs workspace version, seed {seed}")
        _check_against_oracle(dx, dw, dy, h, w, dres, io, f"T={T} H={H} seed {seed}")


def test_noalloc_rejects_rows_wider_than_its_array():
    lib = gb.library()
    fake = 0x10000
    H = SCRATCH_FLOATS + 8
    st = lib.gbln_rmsnorm_bwd_noalloc(fake, None, fake, fake, fake, fake, fake, 4, H,
                                      gb.BF16, gb.BF16, None)
    assert st == 3  # GBLN_ERR_WORKSPACE, nothing launched
    assert "workspace" in gb.status_string(st)
