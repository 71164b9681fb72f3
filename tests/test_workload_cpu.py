"""Host-side checks of the synthetic workloads: shapes as the benchmarked layer
widths state them, the algorithmic byte counts the bench divides by, and the
seeded generators (document lengths, outlier channels, input tensors).  CPU only."""

import numpy as np
import torch

from rmsnorm_fwd_bwd_03_gb300.workload import (ORDER, WORKLOADS, lognormal_doc_lengths, make_inputs,
                                               outlier_channels, scaled)


def test_workload_shapes():
    w = WORKLOADS
    assert ORDER[0] == "qwen05b_tiny_f32" and len(ORDER) == 5 and set(ORDER) == set(w)
    t = w["qwen05b_tiny_f32"]
    assert (t.T, t.H, t.Hq, t.Hk, t.D, t.I, t.dtype, t.theta, t.eps) == (256, 896, 14, 2, 64, 4864, torch.float32, 1e6, 1e-6)
    q = w["qwen3_0p6b"]
    assert (q.T, q.H, q.Hq, q.Hk, q.D, q.I, q.seq_len, q.theta, q.eps) == (16384, 1024, 16, 8, 128, 3072, 2048, 1e6, 1e-6)
    l8 = w["llama3_8b"]
    assert (l8.T, l8.H, l8.Hq, l8.Hk, l8.D, l8.I, l8.seq_len, l8.theta, l8.eps) == (32768, 4096, 32, 8, 128, 14336, 8192, 5e5, 1e-5)
    p = w["llama3_8b_packed_outliers"]
    assert (p.T, p.H, p.Hq, p.Hk, p.I, p.packed, p.outlier_frac, p.outlier_scale) == (65536, 4096, 32, 8, 14336, True, 0.01, 50.0)
    l70 = w["llama70b_width"]
    assert (l70.T, l70.H, l70.Hq, l70.Hk, l70.D, l70.I, l70.seq_len) == (32768, 8192, 64, 8, 128, 28672, 16384)
    # "~1.9 GB per gate/up tensor" at 70B widths
    assert abs(l70.T * l70.I * 2 / 1e9 - 1.88) < 0.01
    assert all(w[n].residual for n in ORDER)


def test_algorithmic_bytes_qwen3():
    # each input read once, each output written once (bf16: 2 bytes)
    a = WORKLOADS["qwen3_0p6b"].algorithmic_bytes()
    T, H, I = 16384, 1024, 3072
    assert a["rmsnorm_fwd"] == 4 * T * H * 2 + H * 2 + 4 * T        # x, r in; y, h out; weight; rstd
    assert a["rmsnorm_bwd"] == 4 * T * H * 2 + H * 2 + 4 * T        # dy, dres, h in; dx out; weight; rstd
    assert a["rope_fwd"] == a["rope_bwd"] == 2 * T * 24 * 128 * 2 + 4 * T
    assert a["swiglu_fwd"] == 3 * T * I * 2 and a["swiglu_bwd"] == 5 * T * I * 2
    assert a["positions"] == 4 * T and a["rmsnorm_dw_finalize"] == 0
    total = sum(a.values())
    assert abs(total / 1e9 - 1.48) < 0.01                            # the step's 1.48 GB


def test_packed_document_lengths():
    lengths = lognormal_doc_lengths(65536, seed=0)
    assert sum(lengths) == 65536
    assert max(lengths) <= 8192 and min(lengths[:-1]) >= 32
    assert lognormal_doc_lengths(65536, seed=0) == lengths            # seeded
    assert lognormal_doc_lengths(65536, seed=1) != lengths
    many = lognormal_doc_lengths(2_000_000, seed=5)[:-1]
    assert 450 < np.median(many) < 580                               # median 512 (clipping barely moves it)
    wl = WORKLOADS["llama3_8b_packed_outliers"]
    cu = wl.cu_seqlens()
    assert cu[0] == 0 and cu[-1] == wl.T and np.all(np.diff(cu) > 0)
    assert wl.max_pos() == max(lengths)


def test_outlier_channels():
    ch = outlier_channels(4096, 0.01)
    assert len(ch) == 41 and len(set(ch.tolist())) == 41 and ch.min() >= 0 and ch.max() < 4096
    assert np.array_equal(outlier_channels(4096, 0.01), ch)


def test_make_inputs_cpu_seeded_and_shaped():
    wl = scaled(WORKLOADS["llama3_8b_packed_outliers"], 512)
    a = make_inputs(wl, "cpu", seed=0)
    b = make_inputs(wl, "cpu", seed=0)
    assert set(a) == {"x", "residual", "weight", "dy", "dres", "q", "k", "dq", "dk", "cu_seqlens", "gate", "up", "dout"}
    for k in a:
        assert torch.equal(a[k], b[k]), k
    assert a["x"].shape == (512, 4096) and a["x"].dtype == torch.bfloat16
    assert a["q"].shape == (512, 32, 128) and a["k"].shape == (512, 8, 128)
    assert a["gate"].shape == (512, 14336)
    assert int(a["cu_seqlens"][-1]) == 512
    # the outlier channels carry ~50x the spread of the others
    ch = outlier_channels(4096, 0.01)
    x = a["x"].float()
    ratio = x[:, ch].std() / x[:, np.setdiff1d(np.arange(4096), ch)].std()
    assert 40 < float(ratio) < 60
    w = a["weight"].float()
    assert abs(float(w.mean()) - 1.0) < 0.01 and 0.08 < float(w.std()) < 0.12
    c = make_inputs(wl, "cpu", seed=1)
    assert not torch.equal(a["x"], c["x"])
