"""GPU vs oracle for RoPE on strided rows (Q and K inside one packed QKV tensor,
in place) and with interleaved pairing, forward and backward."""

import numpy as np
import pytest
import torch

import oracle
import rmsnorm_fwd_bwd_03_gb300 as gb

from _checks import check_io, to64

pytestmark = pytest.mark.gpu

IO = {"f32": torch.float32, "bf16": torch.bfloat16}


@pytest.fixture(scope="module", autouse=True)
def _library():
    from rmsnorm_fwd_bwd_03_gb300._build import build_library
    build_library()
    gb.library()


def _randn(shape, dtype, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return torch.randn(shape, generator=g, device="cuda").to(dtype)


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("pairing", ["half", "interleaved"])
@pytest.mark.parametrize("T,Hq,Hk,D", [(300, 32, 8, 128), (17, 14, 2, 64), (5, 3, 1, 6), (9, 4, 0, 128)])
@pytest.mark.parametrize("bwd", [False, True])
def test_rope_packed_qkv_in_place(io, pairing, T, Hq, Hk, D, bwd):
    dt = IO[io]
    W = (Hq + 2 * Hk) * D
    qkv = _randn((T, W), dt, 1)
    orig = qkv.clone()
    q = qkv[:, :Hq * D].view(T, Hq, D)
    k = qkv[:, Hq * D:(Hq + Hk) * D].view(T, Hk, D) if Hk else None
    pos = torch.as_tensor(np.random.default_rng(2).integers(0, 4000, size=T), dtype=torch.int32, device="cuda")
    table = gb.rope_table(4000, D, 5e5)
    fn = gb.rope_bwd_ex if bwd else gb.rope_fwd_ex
    if bwd:
        fn(q, k, pos, table, dq_in=q, dk_in=k, pairing=pairing)
    else:
        fn(q, k, pos, table, q_out=q, k_out=k, pairing=pairing)
    torch.cuda.synchronize()
    ofn = oracle.rope_bwd if bwd else oracle.rope_fwd
    p = pos.cpu().numpy()
    o = to64(orig)
    check_io(to64(q), ofn(o[:, :Hq * D].reshape(T, Hq, D), p, 5e5, pairing), io, "q in packed")
    if Hk:
        check_io(to64(k), ofn(o[:, Hq * D:(Hq + Hk) * D].reshape(T, Hk, D), p, 5e5, pairing), io, "k in packed")
        assert torch.equal(qkv[:, (Hq + Hk) * D:], orig[:, (Hq + Hk) * D:])  # V untouched


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("offset", [0, 1])
@pytest.mark.parametrize("T,Hq,Hk,D", [(65, 16, 8, 128), (7, 2, 1, 18), (3, 1, 1, 2)])
def test_rope_interleaved_contiguous(io, offset, T, Hq, Hk, D):
    dt = IO[io]
    g = torch.Generator(device="cuda").manual_seed(3)
    buf = torch.randn(T * Hq * D + offset, generator=g, device="cuda").to(dt)
    q = buf[offset:].view(T, Hq, D)
    k = _randn((T, Hk, D), dt, 4)
    pos = torch.arange(T, dtype=torch.int32, device="cuda") * 37 % 3000
    table = gb.rope_table(3000, D, 1e4)
    qo, ko = gb.rope_fwd_ex(q, k, pos, table, pairing="interleaved")
    dq, dk = gb.rope_bwd_ex(q, k, pos, table, pairing="interleaved")
    torch.cuda.synchronize()
    p = pos.cpu().numpy()
    check_io(to64(qo), oracle.rope_fwd(to64(q), p, 1e4, "interleaved"), io, "q'")
    check_io(to64(ko), oracle.rope_fwd(to64(k), p, 1e4, "interleaved"), io, "k'")
    check_io(to64(dq), oracle.rope_bwd(to64(q), p, 1e4, "interleaved"), io, "dq")
    check_io(to64(dk), oracle.rope_bwd(to64(k), p, 1e4, "interleaved"), io, "dk")


def test_rope_ex_half_matches_plain_entry_point():
    T, Hq, Hk, D = 513, 32, 8, 128
    q = _randn((T, Hq, D), torch.bfloat16, 5)
    k = _randn((T, Hk, D), torch.bfloat16, 6)
    pos = torch.arange(T, dtype=torch.int32, device="cuda")
    table = gb.rope_table(T, D, 5e5)
    a = gb.rope_fwd(q, k, pos, table)
    b = gb.rope_fwd_ex(q, k, pos, table)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
