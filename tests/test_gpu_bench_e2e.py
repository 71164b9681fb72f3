"""bench.py's end-to-end leg moves the right bytes: after the timed steps, the
host copy of the last step's outputs equals that step's device output arena and
both device input arenas equal the host input (checked by the leg itself on
sampled chunks, here on a workload small enough to compare whole), and the
figures it reports are consistent."""

import pytest
import torch

pytestmark = pytest.mark.gpu


def test_e2e_leg_reads_back_what_the_step_wrote():
    import bench
    from rmsnorm_fwd_bwd_03_gb300._build import build_library
    from rmsnorm_fwd_bwd_03_gb300.workload import WORKLOADS, scaled
    build_library()
    wl = scaled(WORKLOADS["llama3_8b_packed_outliers"], 1024)
    r = bench.e2e_pipelined(wl, torch.device("cuda", 0), steps=3, warmup=3, world=1, seed=0)
    assert r["readback_verified"] is True
    assert r["value"] > 0 and r["ms_per_step"] > 0 and r["steps"] == 3
    # the arenas hold every input and output of the step (x, residual, dy, dres in; out,
    # dgate, dup among the outputs)
    assert r["h2d_bytes_per_step"] >= wl.T * wl.H * 2 * 4 and r["d2h_bytes_per_step"] >= wl.T * wl.I * 2 * 3


def test_same_chunks_detects_a_changed_byte():
    import bench
    dev = torch.arange(64 << 20, dtype=torch.int64, device="cuda").to(torch.uint8)
    host = dev.cpu()
    assert bench._same_chunks(host, dev, chunks=4, chunk_bytes=1 << 20)
    host[0] ^= 1
    assert not bench._same_chunks(host, dev, chunks=4, chunk_bytes=1 << 20)
    host[0] ^= 1
    host[-1] ^= 1  # the last chunk ends at the buffer's end
    assert not bench._same_chunks(host, dev, chunks=4, chunk_bytes=1 << 20)
