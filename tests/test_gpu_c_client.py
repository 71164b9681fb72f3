"""The C ABI used from plain C: tests/c_client/gbln_client.c is compiled with gcc
against include/gbln.h and libgbln.so, runs RMSNorm / RoPE / SwiGLU forward and
backward on its own device buffers, and its dumped inputs and outputs are
checked against the CPU oracle here."""

import os
import shutil
import struct
import subprocess

import numpy as np
import pytest

import oracle

from _checks import check_mxfp8, check_dw, check_io, check_rstd, dx_scale

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _cuda_home():
    for cand in ("/usr/local/cuda",):
        if os.path.exists(os.path.join(cand, "include", "cuda_runtime_api.h")):
            return cand
    nvcc = shutil.which("nvcc")
    return os.path.dirname(os.path.dirname(nvcc)) if nvcc else None


def _read(path):
    out = {}
    with open(path, "rb") as f:
        while True:
            hdr = f.read(4)
            if not hdr:
                break
            (n,) = struct.unpack("<I", hdr)
            name = f.read(n).decode()
            (cnt,) = struct.unpack("<I", f.read(4))
            out[name] = np.frombuffer(f.read(4 * cnt), dtype=np.float32).astype(np.float64)
    return out


def test_c_client_against_oracle(tmp_path):
    from rmsnorm_fwd_bwd_03_gb300._build import LIBDIR, build_library
    build_library()
    cuda = _cuda_home()
    assert cuda, "CUDA toolkit not found"
    exe = tmp_path / "gbln_client"
    lib64 = os.path.join(cuda, "lib64")
    if not os.path.isdir(lib64):
        lib64 = os.path.join(cuda, "targets", os.uname().machine + "-linux", "lib")
    cmd = ["gcc", "-O2", "-std=c11", "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
           os.path.join(ROOT, "tests", "c_client", "gbln_client.c"), "-o", str(exe),
           "-L", LIBDIR, "-lgbln", "-L", lib64, "-lcudart", f"-Wl,-rpath,{LIBDIR}", f"-Wl,-rpath,{lib64}"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    dump = tmp_path / "out.bin"
    r = subprocess.run([str(exe), str(dump)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    d = _read(dump)
    T, H, HQ, HK, D, I = 37, 96, 3, 1, 32, 200
    x, res, w = d["x"].reshape(T, H), d["residual"].reshape(T, H), d["weight"]
    y_ref, h_ref, rstd_ref = oracle.rmsnorm_fwd(x, res, w, 1e-5, io="f32")
    assert np.array_equal(d["h"].reshape(T, H), h_ref)
    check_io(d["y"].reshape(T, H), y_ref, "f32", "y")
    check_rstd(d["rstd"], rstd_ref)
    dy, dres = d["dy"].reshape(T, H), d["dres"].reshape(T, H)
    dx_ref, dw_ref = oracle.rmsnorm_bwd(dy, dres, h_ref, w, 1e-5)
    check_io(d["dx"].reshape(T, H), dx_ref, "f32", "dx", scale=dx_scale(dy, w, rstd_ref, dres))
    check_dw(d["dW"], dw_ref)
    pos = oracle.positions_from_doc_lengths([20, T - 20])
    assert np.array_equal(d["positions"], pos)
    for name, src, heads, fn in (("q_out", "q", HQ, oracle.rope_fwd), ("k_out", "k", HK, oracle.rope_fwd),
                                 ("dq_in", "q", HQ, oracle.rope_bwd), ("dk_in", "k", HK, oracle.rope_bwd)):
        ref = fn(d[src].reshape(T, heads, D), pos, 10000.0)
        check_io(d[name].reshape(T, heads, D), ref, "f32", name)
    g, u, do = d["gate"], d["up"], d["dout"]
    check_io(d["out"], oracle.swiglu_fwd(g, u), "f32", "swiglu out")
    dg_ref, du_ref = oracle.swiglu_bwd(do, g, u)
    check_io(d["dgate"], dg_ref, "f32", "dgate")
    check_io(d["dup"], du_ref, "f32", "dup")
    # LayerNorm with residual and bias, backward with dres
    ly_ref, lh_ref, lmean_ref, lrstd_ref = oracle.layernorm_fwd(x, res, w, d["bias"], 1e-5, io="f32")
    check_io(d["ln_y"].reshape(T, H), ly_ref, "f32", "ln y")
    check_rstd(d["ln_rstd"], lrstd_ref, "ln rstd")
    assert np.allclose(d["ln_mean"], lmean_ref, rtol=1e-5, atol=1e-6 * np.max(np.abs(lh_ref)))
    ldx_ref, ldw_ref, ldb_ref = oracle.layernorm_bwd(dy, dres, lh_ref, w, 1e-5)
    check_io(d["ln_dx"].reshape(T, H), ldx_ref, "f32", "ln dx", scale=dx_scale(dy, w, lrstd_ref, dres, terms=3))
    check_dw(d["ln_dW"], ldw_ref, "ln dW")
    check_dw(d["ln_dB"], ldb_ref, "ln dB")
    # MXFP8 RMSNorm forward: codes and scales of y
    import torch
    q8 = torch.from_numpy(d["y_e4m3"].astype(np.uint8).reshape(T, H))
    sc8 = torch.from_numpy(d["y_scale"].astype(np.uint8).reshape(T, H // 32))
    check_mxfp8(q8, sc8, y_ref, "c client y mxfp8")
