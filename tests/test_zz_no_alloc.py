"""The allocation-free RMSNorm backward (gbln_rmsnorm_bwd_noalloc) against the
workspace version (gbln_rmsnorm_bwd + gbln_rmsnorm_dw_finalize).

It serves callers that cannot allocate device memory when they run the backward
pass, so it keeps its dW partial sums in a fixed array inside the library instead
of a workspace argument.  The check: two calls in a row on different inputs (the
second must not see the first's leftovers in the shared array) give the same dx
and dW as the workspace version, within the tolerances of the other GPU tests.
This file sorts last so that a run that stops at the first failure has already
run every other test; it also passes alone in a fresh process.
"""

import pytest
import torch

import rmsnorm_fwd_bwd_03_gb300 as gb

from _checks import check_dw, check_io, to64

pytestmark = pytest.mark.gpu


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
    rstd = torch.rsqrt(h.float().pow(2).mean(-1) + 1e-5)
    return dy, h, w, rstd, dres


@pytest.mark.parametrize("T,H,dt", [(16384, 1024, torch.bfloat16), (2048, 8192, torch.bfloat16),
                                    (256, 896, torch.float32), (77, 13, torch.bfloat16)])
def test_noalloc_matches_workspace_version_twice(T, H, dt):
    io = "f32" if dt == torch.float32 else "bf16"
    for seed in (1, 2):  # two calls in a row through the same internal array
        dy, h, w, rstd, dres = _inputs(T, H, dt, seed)
        dx_ref, part, P = gb.rmsnorm_bwd(dy, h, w, rstd, dres)
        dw_ref = gb.rmsnorm_dw_finalize(part, P)
        dx, dw = gb.rmsnorm_bwd_noalloc(dy, h, w, rstd, dres)
        torch.cuda.synchronize()
        check_io(to64(dx), to64(dx_ref), io, f"dx seed {seed}")
        check_dw(to64(dw), to64(dw_ref), f"dW seed {seed}")


def test_noalloc_rejects_rows_wider_than_its_array():
    lib = gb.library()
    fake = 0x10000
    H = (4 << 20) + 8
    st = lib.gbln_rmsnorm_bwd_noalloc(fake, None, fake, fake, fake, fake, fake, 4, H,
                                      gb.BF16, gb.BF16, None)
    assert st == 3  # GBLN_ERR_WORKSPACE, nothing launched
    assert "workspace" in gb.status_string(st)
