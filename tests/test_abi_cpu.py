"""Host-side checks of the C ABI that need no GPU: the library builds, loads and
exports every entry point declared in include/gbln.h, and every invalid argument
is rejected on the host with the documented status before any CUDA call (these
calls never reach the device, so they run without one)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

OK, INVALID, UNSUPPORTED = 0, 1, 2
F32, BF16 = 0, 1
FAKE = 0x10000  # never dereferenced: every call below returns before touching memory


@pytest.fixture(scope="module")
def lib():
    from rmsnorm_fwd_bwd_03_gb300._build import build_library
    import rmsnorm_fwd_bwd_03_gb300 as gb
    build_library()
    return gb.library()


def _declared():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            with open(os.path.join(ROOT, "include", f), encoding="utf-8") as fh:
                src = fh.read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names.update(re.findall(r"\b(gbln_[a-z0-9_]+)\s*\(", src))
    return names


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 12
    for n in sorted(names):
        assert hasattr(lib, n), f"{n} declared but not exported"
    raw = ctypes.CDLL(lib._name)
    for n in names:
        getattr(raw, n)


def test_status_strings_and_version(lib):
    for s in range(5):
        assert lib.gbln_status_string(s).decode().startswith("GBLN_")
    assert b"unknown" in lib.gbln_status_string(99)
    assert lib.gbln_version() >= 100


def _fwd(lib, x=FAKE, r=None, w=FAKE, y=FAKE, ho=None, rstd=FAKE, T=4, H=8, eps=1e-5, io=BF16, wt=BF16):
    return lib.gbln_rmsnorm_fwd(x, r, w, y, ho, rstd, T, H, eps, io, wt, None)


def test_rmsnorm_fwd_rejects(lib):
    assert _fwd(lib, x=None) == INVALID
    assert _fwd(lib, w=None) == INVALID
    assert _fwd(lib, y=None) == INVALID
    assert _fwd(lib, rstd=None) == INVALID
    assert _fwd(lib, r=FAKE, ho=None) == INVALID
    assert _fwd(lib, T=-1) == INVALID
    assert _fwd(lib, H=0) == INVALID
    assert _fwd(lib, H=(1 << 24) + 1) == INVALID
    assert _fwd(lib, eps=-1e-6) == INVALID
    assert _fwd(lib, eps=float("nan")) == INVALID
    assert _fwd(lib, eps=float("inf")) == INVALID
    assert _fwd(lib, io=7) == INVALID
    assert _fwd(lib, io=F32, wt=BF16) == UNSUPPORTED
    assert _fwd(lib, T=0) == OK  # nothing to do, nothing launched
    assert _fwd(lib, T=0, r=FAKE, ho=FAKE, io=BF16, wt=F32) == OK
    assert _fwd(lib, T=0, x=None, w=None, y=None, rstd=None) == OK  # empty tensors: null data


def test_rmsnorm_bwd_and_finalize_reject(lib):
    def bwd(dy=FAKE, dr=None, h=FAKE, w=FAKE, rs=FAKE, dx=FAKE, part=FAKE, P=10, T=4, H=8, io=BF16, wt=BF16):
        return lib.gbln_rmsnorm_bwd(dy, dr, h, w, rs, dx, part, P, T, H, io, wt, None)
    for kw in ({"dy": None}, {"h": None}, {"w": None}, {"rs": None}, {"dx": None}, {"part": None},
               {"T": -3}, {"H": 0}, {"P": -1}, {"io": 5}):
        assert bwd(**kw) == INVALID, kw
    assert bwd(io=F32, wt=BF16) == UNSUPPORTED
    assert bwd(T=0) == OK
    assert bwd(T=0, dy=None, h=None, part=None) == OK
    assert lib.gbln_rmsnorm_bwd_num_partials(-1, 8, BF16) == -1
    assert lib.gbln_rmsnorm_bwd_num_partials(4, 0, BF16) == -1
    assert lib.gbln_rmsnorm_bwd_num_partials(4, 8, 9) == -1
    assert lib.gbln_rmsnorm_bwd_num_partials(0, 8, BF16) == 0
    assert lib.gbln_rmsnorm_dw_finalize(FAKE, -1, 8, FAKE, 0, None) == INVALID
    assert lib.gbln_rmsnorm_dw_finalize(FAKE, 4, 0, FAKE, 0, None) == INVALID
    assert lib.gbln_rmsnorm_dw_finalize(FAKE, 4, 8, None, 0, None) == INVALID
    assert lib.gbln_rmsnorm_dw_finalize(None, 4, 8, FAKE, 0, None) == INVALID


def test_rope_rejects(lib):
    def rope(fn, q=FAKE, k=FAKE, qo=FAKE, ko=FAKE, pos=FAKE, cs=FAKE, mp=100, T=4, Hq=2, Hk=1, D=8, io=BF16):
        return getattr(lib, fn)(q, k, qo, ko, pos, cs, mp, T, Hq, Hk, D, io, None)
    for fn in ("gbln_rope_fwd", "gbln_rope_bwd"):
        for kw in ({"q": None}, {"qo": None}, {"k": None}, {"ko": None}, {"pos": None}, {"cs": None},
                   {"D": 7}, {"D": 0}, {"Hq": 0, "Hk": 0}, {"Hq": -1}, {"T": -1}, {"mp": -1},
                   {"cs": FAKE + 4}, {"io": 3}):
            assert rope(fn, **kw) == INVALID, (fn, kw)
        assert rope(fn, T=0) == OK
        assert rope(fn, T=0, k=None, ko=None, Hk=0) == OK
    assert lib.gbln_rope_table(None, 10, 8, 1e4, None) == INVALID
    assert lib.gbln_rope_table(FAKE, -1, 8, 1e4, None) == INVALID
    assert lib.gbln_rope_table(FAKE, 10, 7, 1e4, None) == INVALID
    assert lib.gbln_rope_table(FAKE, 10, 8, 0.0, None) == INVALID
    assert lib.gbln_rope_table(FAKE, 10, 8, float("nan"), None) == INVALID
    assert lib.gbln_rope_table(FAKE, 0, 8, 1e4, None) == OK


def test_rope_ex_rejects(lib):
    def ex(fn, ldq=64, ldk=16, ldqo=64, ldko=16, pairing=0, T=4, q=FAKE):
        return getattr(lib, fn)(q, FAKE, FAKE, FAKE, FAKE, FAKE, 100, T, 4, 1, 16, ldq, ldk, ldqo, ldko,
                                pairing, BF16, None)
    for fn in ("gbln_rope_fwd_ex", "gbln_rope_bwd_ex"):
        assert ex(fn, ldq=63) == INVALID
        assert ex(fn, ldk=15) == INVALID
        assert ex(fn, ldqo=10) == INVALID
        assert ex(fn, ldko=0) == INVALID
        assert ex(fn, pairing=2) == INVALID
        assert ex(fn, q=None) == INVALID
        assert ex(fn, T=0, q=None) == OK


def test_positions_rejects(lib):
    f = lib.gbln_positions_from_cu_seqlens
    assert f(FAKE, 2, None, 10, None) == INVALID
    assert f(FAKE, -1, FAKE, 10, None) == INVALID
    assert f(None, 2, FAKE, 10, None) == INVALID
    assert f(FAKE, 0, FAKE, 10, None) == INVALID
    assert f(FAKE, 2, FAKE, -1, None) == INVALID
    assert f(None, 0, FAKE, 0, None) == OK


def test_swiglu_rejects(lib):
    assert lib.gbln_swiglu_fwd(None, FAKE, FAKE, 4, 8, BF16, None) == INVALID
    assert lib.gbln_swiglu_fwd(FAKE, None, FAKE, 4, 8, BF16, None) == INVALID
    assert lib.gbln_swiglu_fwd(FAKE, FAKE, None, 4, 8, BF16, None) == INVALID
    assert lib.gbln_swiglu_fwd(FAKE, FAKE, FAKE, -1, 8, BF16, None) == INVALID
    assert lib.gbln_swiglu_fwd(FAKE, FAKE, FAKE, 4, 0, BF16, None) == INVALID
    assert lib.gbln_swiglu_fwd(FAKE, FAKE, FAKE, 1 << 40, 1 << 30, BF16, None) == INVALID
    assert lib.gbln_swiglu_fwd(FAKE, FAKE, FAKE, 4, 8, 2, None) == INVALID
    assert lib.gbln_swiglu_fwd(FAKE, FAKE, FAKE, 0, 8, BF16, None) == OK
    assert lib.gbln_swiglu_fwd(None, None, None, 0, 8, BF16, None) == OK
    for i in range(5):
        args = [FAKE] * 5
        args[i] = None
        assert lib.gbln_swiglu_bwd(*args, 4, 8, BF16, None) == INVALID
    assert lib.gbln_swiglu_bwd(FAKE, FAKE, FAKE, FAKE, FAKE, 0, 8, F32, None) == OK


def test_layernorm_rejects(lib):
    f = FAKE
    def fwd(x=f, r=None, w=f, b=None, y=f, ho=None, m=f, rs=f, T=4, H=8, eps=1e-5, io=BF16, wt=BF16):
        return lib.gbln_layernorm_fwd(x, r, w, b, y, ho, m, rs, T, H, eps, io, wt, None)
    for kw in ({"x": None}, {"w": None}, {"y": None}, {"m": None}, {"rs": None}, {"r": f},
               {"T": -1}, {"H": 0}, {"eps": -1.0}, {"eps": float("nan")}, {"io": 4}):
        assert fwd(**kw) == INVALID, kw
    assert fwd(io=F32, wt=BF16) == UNSUPPORTED
    assert fwd(T=0, x=None, w=None, y=None, m=None, rs=None) == OK
    def bwd(dy=f, h=f, w=f, m=f, rs=f, dx=f, part=f, P=10, T=4, H=8):
        return lib.gbln_layernorm_bwd(dy, None, h, w, m, rs, dx, part, P, T, H, BF16, BF16, None)
    for kw in ({"dy": None}, {"h": None}, {"m": None}, {"part": None}, {"P": -1}, {"H": -2}):
        assert bwd(**kw) == INVALID, kw
    assert bwd(T=0, dy=None) == OK
    assert lib.gbln_layernorm_bwd_num_partials(-1, 8, BF16) == -1
    assert lib.gbln_layernorm_bwd_num_partials(0, 8, BF16) == 0
    assert lib.gbln_layernorm_dwdb_finalize(f, 2, 8, f, None, 0, None) == INVALID
    assert lib.gbln_layernorm_dwdb_finalize(None, 2, 8, f, f, 0, None) == INVALID


def test_glu_and_act_reject(lib):
    f = FAKE
    assert lib.gbln_glu_fwd(f, f, f, 4, 8, 7, 8, 8, 0, BF16, None) == INVALID  # ld < I
    assert lib.gbln_glu_fwd(f, f, f, 4, 8, 8, 8, 8, 9, BF16, None) == INVALID  # bad act
    assert lib.gbln_glu_fwd(None, f, f, 4, 8, 8, 8, 8, 0, BF16, None) == INVALID
    assert lib.gbln_glu_fwd(f, f, f, 4, 0, 8, 8, 8, 0, BF16, None) == INVALID
    assert lib.gbln_glu_fwd(None, None, None, 0, 8, 8, 8, 8, 0, BF16, None) == OK
    assert lib.gbln_glu_bwd(f, f, f, f, f, 4, 8, 8, 8, 8, 8, 3, 0, BF16, None) == INVALID
    assert lib.gbln_glu_bwd(f, f, f, None, f, 4, 8, 8, 8, 8, 8, 8, 0, BF16, None) == INVALID
    assert lib.gbln_glu_bwd(None, None, None, None, None, 0, 8, 8, 8, 8, 8, 8, 3, F32, None) == OK
    assert lib.gbln_act_fwd(None, f, 4, 0, BF16, None) == INVALID
    assert lib.gbln_act_fwd(f, f, 4, 4, BF16, None) == INVALID
    assert lib.gbln_act_fwd(f, f, -1, 0, BF16, None) == INVALID
    assert lib.gbln_act_fwd(None, None, 0, 2, F32, None) == OK
    assert lib.gbln_act_bwd(f, None, f, 4, 0, BF16, None) == INVALID
    assert lib.gbln_act_bwd(None, None, None, 0, 1, BF16, None) == OK


def test_mxfp8_entries_reject(lib):
    f = FAKE
    # H / I not a multiple of the 32-value MX block
    assert lib.gbln_rmsnorm_fwd_mxfp8(f, None, f, None, f, f, None, f, 4, 48, 1e-6, BF16, BF16, None) == INVALID
    assert lib.gbln_glu_fwd_mxfp8(f, f, f, f, 4, 48, 48, 48, 0, BF16, None) == INVALID
    # null code / scale outputs; null x; residual without residual_out
    assert lib.gbln_rmsnorm_fwd_mxfp8(f, None, f, None, None, f, None, f, 4, 64, 1e-6, BF16, BF16, None) == INVALID
    assert lib.gbln_rmsnorm_fwd_mxfp8(f, None, f, None, f, None, None, f, 4, 64, 1e-6, BF16, BF16, None) == INVALID
    assert lib.gbln_rmsnorm_fwd_mxfp8(None, None, f, None, f, f, None, f, 4, 64, 1e-6, BF16, BF16, None) == INVALID
    assert lib.gbln_rmsnorm_fwd_mxfp8(f, f, f, None, f, f, None, f, 4, 64, 1e-6, BF16, BF16, None) == INVALID
    assert lib.gbln_rmsnorm_fwd_mxfp8(f, None, f, None, f, f, None, f, 4, 64, -1.0, BF16, BF16, None) == INVALID
    assert lib.gbln_rmsnorm_fwd_mxfp8(f, None, f, None, f, f, None, f, 4, 64, 1e-6, F32, BF16, None) == UNSUPPORTED
    assert lib.gbln_glu_fwd_mxfp8(f, f, None, f, 4, 64, 64, 64, 0, BF16, None) == INVALID
    assert lib.gbln_glu_fwd_mxfp8(f, f, f, f, 4, 64, 63, 64, 0, BF16, None) == INVALID  # ld < I
    assert lib.gbln_glu_fwd_mxfp8(f, f, f, f, 4, 64, 64, 64, 9, BF16, None) == INVALID  # bad act
    # T == 0 is a no-op before any pointer is examined
    assert lib.gbln_rmsnorm_fwd_mxfp8(None, None, None, None, None, None, None, None, 0, 64, 1e-6, BF16, BF16, None) == OK
    assert lib.gbln_glu_fwd_mxfp8(None, None, None, None, 0, 64, 64, 64, 0, BF16, None) == OK


def test_device_error_rejects_null(lib):
    assert lib.gbln_device_error(None, 0) == INVALID


def test_selftest_rejects_bad_poll_counts(lib):
    assert lib.gbln_selftest_wait_timeout(0, None) == INVALID
    assert lib.gbln_selftest_wait_timeout((1 << 22) + 1, None) == INVALID


def test_binding_refuses_cpu_tensors(lib):
    import torch
    import rmsnorm_fwd_bwd_03_gb300 as gb
    x = torch.zeros(2, 8)
    with pytest.raises(ValueError):
        gb.rmsnorm_fwd(x, torch.ones(8), 1e-5)
    with pytest.raises(ValueError):
        gb.swiglu_fwd(x, x)


def _cuda_include():
    import shutil
    for cand in ("/usr/local/cuda", os.path.dirname(os.path.dirname(shutil.which("nvcc") or "/x/x"))):
        if os.path.exists(os.path.join(cand, "include", "cuda_runtime_api.h")):
            return os.path.join(cand, "include")
    return None


@pytest.mark.parametrize("lang,std", [("c", "c99"), ("c", "c11"), ("c++", "c++11"), ("c++", "c++17")])
def test_header_compiles_cleanly(tmp_path, lang, std):
    # The header is usable from plain C and from C++ without warnings, and with
    # the CUDA runtime header included first (cudaStream_t and the stream handle
    # type agree) or not at all.
    import shutil
    import subprocess
    gcc = shutil.which("gcc" if lang == "c" else "g++")
    if gcc is None:
        pytest.skip("no host compiler")
    cuda_inc = _cuda_include()
    srcs = {"plain": '#include "gbln.h"\nint main(void) { return gbln_version() > 0 ? 0 : 1; }\n'}
    if cuda_inc:
        srcs["with_cuda"] = ('#include <cuda_runtime_api.h>\n#include "gbln.h"\n'
                             "int main(void) { cudaStream_t s = 0; return gbln_swiglu_fwd(0, 0, 0, 0, 1, GBLN_BF16, s); }\n")
    for tag, text in srcs.items():
        src = tmp_path / (f"{tag}.c" if lang == "c" else f"{tag}.cpp")
        src.write_text(text)
        cmd = [gcc, f"-std={std}", "-Wall", "-Wextra", "-Werror", "-pedantic", "-fsyntax-only",
               "-I", os.path.join(ROOT, "include"), str(src)]
        if tag == "with_cuda":
            cmd[1:1] = ["-isystem", cuda_inc]
        r = subprocess.run(cmd, capture_output=True, text=True)
        assert r.returncode == 0, f"{tag} {std}: {r.stderr}"


def test_c_client_links_against_the_library(lib, tmp_path):
    # The plain-C client program (run against the oracle by the GPU tests) links
    # against libgbln with every entry point it uses resolved.
    import shutil
    import subprocess
    from rmsnorm_fwd_bwd_03_gb300._build import LIBDIR
    gcc, cuda_inc = shutil.which("gcc"), _cuda_include()
    if gcc is None or cuda_inc is None:
        pytest.skip("no host compiler or CUDA headers")
    cuda = os.path.dirname(cuda_inc)
    lib64 = os.path.join(cuda, "lib64")
    if not os.path.isdir(lib64):
        lib64 = os.path.join(cuda, "targets", os.uname().machine + "-linux", "lib")
    exe = tmp_path / "gbln_client"
    cmd = [gcc, "-O1", "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), "-I", cuda_inc,
           os.path.join(ROOT, "tests", "c_client", "gbln_client.c"), "-o", str(exe),
           "-L", LIBDIR, "-lgbln", "-L", lib64, "-lcudart", "-Wl,--no-undefined"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    assert exe.exists()
