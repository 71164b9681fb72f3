"""Every entry point of the step enqueues on the caller's stream only: the whole
step captured into a CUDA graph replays to the same bits as eager launches,
and running it on a non-default stream gives the same bits as on the default
stream (all kernels are deterministic)."""

import pytest
import torch

import rmsnorm_fwd_bwd_03_gb300 as gb
from rmsnorm_fwd_bwd_03_gb300.workload import WORKLOADS, make_inputs, scaled

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    from rmsnorm_fwd_bwd_03_gb300._build import build_library
    build_library()
    gb.library()


def _step(wl, inp, table, outs):
    """The eight calls of one fwd + bwd step into preallocated outputs."""
    T = wl.T
    gb.positions_from_cu_seqlens(inp["cu_seqlens"], T, out=outs["pos"])
    gb.rmsnorm_fwd(inp["x"], inp["weight"], wl.eps, inp["residual"], y=outs["y"], residual_out=outs["h"],
                   rstd=outs["rstd"])
    gb.rope_fwd(inp["q"], inp["k"], outs["pos"], table, q_out=outs["qo"], k_out=outs["ko"])
    gb.swiglu_fwd(inp["gate"], inp["up"], out=outs["out"])
    gb.swiglu_bwd(inp["dout"], inp["gate"], inp["up"], dgate=outs["dg"], dup=outs["du"])
    gb.rope_bwd(inp["dq"], inp["dk"], outs["pos"], table, dq_in=outs["dqi"], dk_in=outs["dki"])
    gb.rmsnorm_bwd(inp["dy"], outs["h"], inp["weight"], outs["rstd"], inp["dres"], dx=outs["dx"],
                   dw_partial=outs["part"])
    gb.rmsnorm_dw_finalize(outs["part"], outs["P"], dw=outs["dw"])


def _alloc(wl, inp):
    e = torch.empty_like
    P = gb.rmsnorm_bwd_num_partials(wl.T, wl.H, wl.dtype)
    return {"pos": torch.empty(wl.T, dtype=torch.int32, device="cuda"), "y": e(inp["x"]), "h": e(inp["x"]),
            "rstd": torch.empty(wl.T, device="cuda"), "qo": e(inp["q"]), "ko": e(inp["k"]), "out": e(inp["gate"]),
            "dg": e(inp["gate"]), "du": e(inp["up"]), "dqi": e(inp["dq"]), "dki": e(inp["dk"]), "dx": e(inp["x"]),
            "part": torch.empty(P, wl.H, device="cuda"), "P": P, "dw": torch.empty(wl.H, device="cuda")}


def _same(a, b):
    for key in a:
        if key == "P":
            continue
        assert torch.equal(a[key].view(torch.uint8), b[key].view(torch.uint8)), key


@pytest.mark.parametrize("name,T", [("qwen3_0p6b", 4096), ("llama3_8b_packed_outliers", 3000),
                                    ("qwen05b_tiny_f32", 256)])
def test_step_in_cuda_graph_matches_eager(name, T):
    wl = scaled(WORKLOADS[name], T)
    inp = make_inputs(wl, "cuda")
    table = gb.rope_table(wl.max_pos(), wl.D, wl.theta)
    eager = _alloc(wl, inp)
    _step(wl, inp, table, eager)  # first calls on this device do their one-time set-up here
    torch.cuda.synchronize()
    graphed = _alloc(wl, inp)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        _step(wl, inp, table, graphed)
    for _ in range(2):
        for key, t in graphed.items():
            if key != "P":
                t.zero_()
        g.replay()
        torch.cuda.synchronize()
        _same(eager, graphed)
    assert gb.device_error() == 0


def test_step_on_side_stream_matches_default_stream():
    wl = scaled(WORKLOADS["llama3_8b"], 2048)
    inp = make_inputs(wl, "cuda")
    table = gb.rope_table(wl.max_pos(), wl.D, wl.theta)
    a = _alloc(wl, inp)
    _step(wl, inp, table, a)
    torch.cuda.synchronize()
    b = _alloc(wl, inp)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        _step(wl, inp, table, b)
    side.synchronize()
    _same(a, b)
