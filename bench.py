#!/usr/bin/env python
"""Throughput of one fused-layer-operator step on GB300: RMSNorm / RoPE / SwiGLU, forward + backward.

One step = every operator of the path once over one batch of tokens, in training
order: positions of packed documents -> RMSNorm forward (fused residual add) ->
RoPE forward on Q and K -> SwiGLU forward -> SwiGLU backward -> RoPE backward ->
RMSNorm backward (dX and dW partials) -> dW finalize.  Eight launches of the
library's kernels, called through the C ABI with device pointers.

Prints one JSON line.  ``value`` is tokens per second over all ranks with inputs
resident in HBM; ``e2e`` is the same step through the same C ABI with the inputs
in pinned host memory and the outputs read back, copies inside the timed region.
L2 is flushed between timed steps (a 2x L2 write, then a 2x L2 read of another
buffer, so no step data and no dirty lines remain in it).  ``--impl reference`` times
the float64 CPU oracle on a bounded sample of the same workload instead.

Multi-GPU (torchrun): each rank runs its own replica on its own batch (weak
scaling, no data-path collective); timing is max over ranks.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "fwd+bwd tokens/s and achieved HBM GB/s (% of GB300 peak), RMSNorm/RoPE/SwiGLU"
DEFAULT_WORKLOAD = "llama3_8b_packed_outliers"
FALLBACK_HBM_GBS = 6800.0
OPS = ["positions", "rmsnorm_fwd", "rope_fwd", "swiglu_fwd", "swiglu_bwd", "rope_bwd",
       "rmsnorm_bwd", "rmsnorm_dw_finalize"]
KERNEL_SOURCE = {"positions": "rope.cu", "rmsnorm_fwd": "rmsnorm.cu", "rope_fwd": "rope.cu",
                 "swiglu_fwd": "glu.cu", "swiglu_bwd": "glu.cu", "rope_bwd": "rope.cu",
                 "rmsnorm_bwd": "rmsnorm.cu", "rmsnorm_dw_finalize": "rmsnorm.cu"}
# DRAM bytes (read + write) per launch from one ncu capture, keyed by workload and
# operator, with the sha256 of the kernel source they were taken on: a changed
# kernel reports null until it is captured again.  Summaries live under profiles/.
NCU_TRAFFIC = {
    # glu_bwd_vec on the packed Llama-3-8B workload: dram__bytes_read.sum + dram__bytes_write.sum
    # at the same widths with 8192 and 16384 tokens (one launch each, cold L2: 1118481152 and
    # 2292602112 bytes), extrapolated along that line to 65536 tokens (the full launch is
    # beyond the size rule for a counter capture; the traffic grows by 143,325 bytes per token)
    ("llama3_8b_packed_outliers", "swiglu_bwd"): {"bytes": 9337327872, "src_sha": "e75f3acc8277048b"},
    # glu_bwd_vec at Qwen3-0.6B widths, the full launch (one capture, cold L2: ~56 MB of the
    # writes are still in L2 when it ends)
    ("qwen3_0p6b", "swiglu_bwd"): {"bytes": 447497216, "src_sha": "e75f3acc8277048b"},
}


def _src_sha(op):
    """Hash of the code (comments and whitespace removed) of the op's source file
    and the shared header it includes: the DRAM traffic recorded for a kernel is
    reported only while that code is unchanged."""
    h = hashlib.sha256()
    for name in (KERNEL_SOURCE[op], "common.cuh"):
        with open(os.path.join(ROOT, "rmsnorm_fwd_bwd_03_gb300", "csrc", name), encoding="utf-8") as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)   # block comments
        text = re.sub(r"//[^\n]*", " ", text)                  # line comments
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def _measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"

    def find(obj):
        if isinstance(obj, dict):
            for k, v in obj.items():
                if "hbm" in k.lower() and isinstance(v, (int, float)):
                    return float(v)
            for v in obj.values():
                r = find(v)
                if r:
                    return r
        return None
    v = find(d)
    return (v, "measured") if v else (FALLBACK_HBM_GBS, "fallback")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.gpu = gpu_index

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = [r.split(",") for r in (self.out or "").strip().splitlines() if r.strip()]
        rows = [[c.strip() for c in r] for r in rows if len(r) >= 9]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        def num(s):
            try:
                return float(s)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for name, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": num(rows[0][2]), "reasons": sorted(reasons),
                "power_w_median": statistics.median([num(r[3]) for r in rows if num(r[3]) is not None] or [0]),
                "samples": len(rows)}


class L2Flush:
    """Between timed steps: write a buffer of twice the L2 size (evicts the step's
    data), then read a second one of the same size (evicts the dirty lines of the
    write, so the next step neither finds its data in L2 nor pays for writing
    back lines that are not its own)."""

    def __init__(self, device):
        l2 = torch.cuda.get_device_properties(device).L2_cache_size
        n = max(2 * l2, 256 << 20) // 4
        self.w = torch.empty(n, dtype=torch.float32, device=device)
        self.r = torch.ones(n, dtype=torch.float32, device=device)

    def __call__(self):
        self.w.zero_()
        self.r.sum()


# ---------------------------------------------------------------------------
# The step through the C ABI
# ---------------------------------------------------------------------------

def _arena(tensors: dict, device, fill: bool):
    """One contiguous device buffer holding every tensor (256-byte aligned views)."""
    offs, total = {}, 0
    for key, t in tensors.items():
        offs[key] = total
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    buf = torch.empty(max(total, 256), dtype=torch.uint8, device=device)
    views = {}
    for key, t in tensors.items():
        nb = t.numel() * t.element_size()
        v = buf[offs[key]:offs[key] + nb].view(t.dtype).view(t.shape)
        if fill:
            v.copy_(t)
        views[key] = v
    return buf, views


class Step:
    """Device buffers and the eight C-ABI calls of one fwd + bwd step.

    Inputs live in one contiguous device arena and outputs in another, so that
    the end-to-end leg moves each direction with a single copy per step."""

    def __init__(self, wl, device, seed):
        import rmsnorm_fwd_bwd_03_gb300 as gb
        from rmsnorm_fwd_bwd_03_gb300.workload import make_inputs
        self.gb = gb
        self.lib = gb.library()
        self.wl = wl
        T, H = wl.T, wl.H
        gen = make_inputs(wl, device, seed=seed)
        self.in_arena, self.inp = _arena(gen, device, fill=True)
        del gen
        i = self.inp
        meta = lambda shape, dt: torch.empty(shape, dtype=dt, device="meta")  # noqa: E731  (shape/dtype only)
        like = lambda t: meta(t.shape, t.dtype)  # noqa: E731
        spec = {
            "positions": meta((T,), torch.int32),
            "y": like(i["x"]), "h": like(i["x"]),
            "rstd": meta((T,), torch.float32),
            "q_out": like(i["q"]), "k_out": like(i["k"]),
            "out": like(i["gate"]), "dgate": like(i["gate"]), "dup": like(i["up"]),
            "dq_in": like(i["dq"]), "dk_in": like(i["dk"]),
            "dx": like(i["x"]), "dw": meta((H,), torch.float32),
        }
        self.out_arena, self.out = _arena(spec, device, fill=False)
        self.P = gb.rmsnorm_bwd_num_partials(T, H, wl.dtype)
        self.partial = torch.empty((self.P, H), dtype=torch.float32, device=device)
        self.max_pos = wl.max_pos()
        self.table = gb.rope_table(self.max_pos, wl.D, wl.theta, device=device)
        self.io = gb.BF16 if wl.dtype == torch.bfloat16 else gb.F32
        torch.cuda.synchronize()

    def calls(self, stream_handle):
        """The eight (name, fn, args) calls of a step on the given stream."""
        i, o, wl, L = self.inp, self.out, self.wl, self.lib
        p = lambda t: t.data_ptr()  # noqa: E731
        T, H = wl.T, wl.H
        s = stream_handle
        return [
            ("positions", L.gbln_positions_from_cu_seqlens,
             (p(i["cu_seqlens"]), i["cu_seqlens"].numel() - 1, p(o["positions"]), T, s)),
            ("rmsnorm_fwd", L.gbln_rmsnorm_fwd,
             (p(i["x"]), p(i["residual"]), p(i["weight"]), p(o["y"]), p(o["h"]), p(o["rstd"]),
              T, H, wl.eps, self.io, self.io, s)),
            ("rope_fwd", L.gbln_rope_fwd,
             (p(i["q"]), p(i["k"]), p(o["q_out"]), p(o["k_out"]), p(o["positions"]), p(self.table),
              self.max_pos, T, wl.Hq, wl.Hk, wl.D, self.io, s)),
            ("swiglu_fwd", L.gbln_swiglu_fwd, (p(i["gate"]), p(i["up"]), p(o["out"]), T, wl.I, self.io, s)),
            ("swiglu_bwd", L.gbln_swiglu_bwd,
             (p(i["dout"]), p(i["gate"]), p(i["up"]), p(o["dgate"]), p(o["dup"]), T, wl.I, self.io, s)),
            ("rope_bwd", L.gbln_rope_bwd,
             (p(i["dq"]), p(i["dk"]), p(o["dq_in"]), p(o["dk_in"]), p(o["positions"]), p(self.table),
              self.max_pos, T, wl.Hq, wl.Hk, wl.D, self.io, s)),
            ("rmsnorm_bwd", L.gbln_rmsnorm_bwd,
             (p(i["dy"]), p(i["dres"]), p(o["h"]), p(i["weight"]), p(o["rstd"]), p(o["dx"]),
              p(self.partial), self.P, T, H, self.io, self.io, s)),
            ("rmsnorm_dw_finalize", L.gbln_rmsnorm_dw_finalize,
             (p(self.partial), self.P, H, p(o["dw"]), 0, s)),
        ]


def _cudart():
    """The CUDA runtime library this process has loaded (torch's), else the
    first one on the library path."""
    import ctypes
    torch.cuda.init()
    cands = []
    try:
        with open("/proc/self/maps") as f:
            cands = sorted({ln.split()[-1] for ln in f if "libcudart.so" in ln})
    except OSError:
        pass
    for name in cands + ["libcudart.so.13", "libcudart.so"]:
        try:
            lib = ctypes.CDLL(name)
        except OSError:
            continue
        lib.cudaHostAlloc.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.c_size_t, ctypes.c_uint]
        lib.cudaHostAlloc.restype = ctypes.c_int
        lib.cudaFreeHost.argtypes = [ctypes.c_void_p]
        lib.cudaFreeHost.restype = ctypes.c_int
        return lib
    raise RuntimeError("bench.py: no CUDA runtime library found for page-locked host buffers")


def _host_available():
    """MemAvailable of this host in bytes (0 if unknown)."""
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except (OSError, ValueError, IndexError):
        pass
    return 0


class PinnedHostBuffer:
    """Page-locked host memory from cudaHostAlloc, viewed as a uint8 CPU tensor
    (allocated outside torch's caching host allocator, which rounds sizes up to
    a power of two and keeps the blocks)."""

    def __init__(self, nbytes):
        import ctypes
        self._rt = _cudart()
        self._ptr = ctypes.c_void_p()
        st = self._rt.cudaHostAlloc(ctypes.byref(self._ptr), ctypes.c_size_t(nbytes), 0)
        if st != 0 or not self._ptr.value:
            raise RuntimeError(f"cudaHostAlloc of {nbytes} bytes failed with error {st}")
        self.tensor = torch.frombuffer((ctypes.c_uint8 * nbytes).from_address(self._ptr.value),
                                       dtype=torch.uint8)

    def free(self):
        if self._ptr is not None and self._ptr.value:
            self.tensor = None
            self._rt.cudaFreeHost(self._ptr)
            self._ptr = None


def _same_chunks(host, dev, chunks=16, chunk_bytes=16 << 20):
    """Byte equality of a host and a device uint8 buffer of the same size on
    `chunks` evenly spaced chunks (the whole buffer when it is small)."""
    n = host.numel()
    if dev.numel() != n:
        return False
    if n <= chunks * chunk_bytes:
        return torch.equal(host, dev.cpu())
    step = (n - chunk_bytes) // (chunks - 1)
    return all(torch.equal(host[o:o + chunk_bytes], dev[o:o + chunk_bytes].cpu())
               for o in range(0, n - chunk_bytes + 1, step)[:chunks])


def e2e_pipelined(wl, device, steps, warmup, world, seed):
    """Throughput of the step with inputs in pinned host memory and every output
    read back: per step one host-to-device copy of the input arena, the eight
    C-ABI calls, and one device-to-host copy of the output arena.  Two device
    buffer sets and three streams overlap step i's kernels with step i+1's
    upload and step i-1's download; every step's copies are inside the timed
    region."""
    sets = [Step(wl, device, seed), Step(wl, device, seed)]
    nin, nout = sets[0].in_arena.numel(), sets[0].out_arena.numel()
    # A throwaway page-locked block of twice the buffers' size (within half of the
    # host's available memory, shared by the ranks) is taken first and released once
    # the buffers are in place.  Measured on GB300 (Grace host): after another
    # process had run on the host (the oracle's reference arm, the test suite), this
    # pipeline took 92-107 ms per step of 17.7 GB with the buffers allocated straight
    # away and 59 ms with the throwaway block first, the rate of a host where no
    # other process had run (58-60 ms either way there); single copies ran at full
    # speed in every case.
    spare_bytes = min(2 * (nin + nout), _host_available() // (2 * world) - (nin + nout))
    spare = PinnedHostBuffer(spare_bytes) if spare_bytes > 0 else None
    pin_in = PinnedHostBuffer(nin)
    # one host buffer for the results: the read-backs are ordered on one stream
    pin_out = PinnedHostBuffer(nout)
    if spare is not None:
        spare.free()
    host_in, host_out = pin_in.tensor, pin_out.tensor
    host_in.copy_(sets[0].in_arena)
    s_in, s_comp, s_out = (torch.cuda.Stream(device) for _ in range(3))
    calls = [st.calls(s_comp.cuda_stream) for st in sets]
    ev_in = [torch.cuda.Event() for _ in sets]
    ev_comp = [torch.cuda.Event() for _ in sets]
    ev_out = [torch.cuda.Event() for _ in sets]

    def run(n):
        for it in range(n):
            b = it % 2
            with torch.cuda.stream(s_in):
                if it >= 2:
                    s_in.wait_event(ev_comp[b])  # step it-2 has finished reading set b
                sets[b].in_arena.copy_(host_in, non_blocking=True)
                ev_in[b].record(s_in)
            with torch.cuda.stream(s_comp):
                s_comp.wait_event(ev_in[b])
                if it >= 2:
                    s_comp.wait_event(ev_out[b])  # step it-2's outputs have been read back
                run_calls(calls[b])
                ev_comp[b].record(s_comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_comp[b])
                host_out.copy_(sets[b].out_arena, non_blocking=True)
                ev_out[b].record(s_out)

    run(warmup)
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    run(steps)
    s_out.wait_stream(s_in)
    s_out.wait_stream(s_comp)
    e1.record(s_out)
    torch.cuda.synchronize()
    ms = reduce_max(e0.elapsed_time(e1), world)
    h2d, d2h = nin, nout
    # The copies moved the right bytes: sampled chunks of the last step's read-back
    # equal its device output arena, and both device input arenas equal the host's.
    last = (steps - 1) % 2
    verified = (_same_chunks(host_out, sets[last].out_arena) and
                all(_same_chunks(host_in, st.in_arena) for st in sets))
    del host_in, host_out
    pin_in.free()
    pin_out.free()
    return {"value": world * wl.T * steps / (ms * 1e-3), "unit": "tokens/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": steps,
            "ms_per_step": ms / steps, "readback_verified": bool(verified),
            "method": "one H2D copy of the input arena from page-locked host memory (cudaHostAlloc), "
                      "the 8 C-ABI calls and one D2H copy of the output arena per step; copies on "
                      "their own streams overlap the neighbouring steps' kernels (two device buffer "
                      "sets)"}


def run_calls(calls, events=None):
    if events is None:
        for name, fn, args in calls:
            st = fn(*args)
            if st != 0:
                raise RuntimeError(f"{name} failed with status {st}")
        return
    events[0].record()
    for k, (name, fn, args) in enumerate(calls):
        st = fn(*args)
        if st != 0:
            raise RuntimeError(f"{name} failed with status {st}")
        events[k + 1].record()


# ---------------------------------------------------------------------------
# CPU oracle timing
# ---------------------------------------------------------------------------

# The oracle's calls in step order: (operator, fn(wl, inp, state)).  Each runs on
# the float64 copies of a contiguous block of tokens; h comes from the forward.
def _oracle_ops():
    import oracle

    def rms_fwd(wl, inp, st):
        st["h"] = oracle.rmsnorm_fwd(inp["x"], inp["residual"], inp["weight"], wl.eps, io=wl.io)[1]

    return [
        ("positions", lambda wl, inp, st: st.__setitem__(
            "pos", oracle.positions_from_cu_seqlens(inp["cu_seqlens"]))),
        ("rmsnorm_fwd", rms_fwd),
        ("rope_fwd", lambda wl, inp, st: (oracle.rope_fwd(inp["q"], st["pos"], wl.theta),
                                          oracle.rope_fwd(inp["k"], st["pos"], wl.theta))),
        ("swiglu_fwd", lambda wl, inp, st: oracle.swiglu_fwd(inp["gate"], inp["up"])),
        ("swiglu_bwd", lambda wl, inp, st: oracle.swiglu_bwd(inp["dout"], inp["gate"], inp["up"])),
        ("rope_bwd", lambda wl, inp, st: (oracle.rope_bwd(inp["dq"], st["pos"], wl.theta),
                                          oracle.rope_bwd(inp["dk"], st["pos"], wl.theta))),
        # dX and the weight gradient summed over every row of the block
        ("rmsnorm_bwd", lambda wl, inp, st: oracle.rmsnorm_bwd(inp["dy"], inp["dres"], st["h"],
                                                               inp["weight"], wl.eps)),
    ]


def oracle_step(wl, inp, per_op=None):
    """One fwd + bwd pass of the oracle over the rows of ``inp`` (float64 numpy
    arrays); with ``per_op`` (a dict) each operator's seconds are added to it."""
    st = {}
    for name, fn in _oracle_ops():
        t0 = time.perf_counter()
        fn(wl, inp, st)
        if per_op is not None:
            per_op[name] = per_op.get(name, 0.0) + time.perf_counter() - t0


def oracle_sample_inputs(wl, rows):
    """The first ``rows`` tokens of a workload of the same widths and document law
    (seed 0), as float64 numpy arrays: a contiguous block of consecutive tokens."""
    from rmsnorm_fwd_bwd_03_gb300.workload import make_inputs, scaled
    small = scaled(wl, rows, "_sample")
    inp = make_inputs(small, "cpu", seed=0)
    out = {}
    for k, v in inp.items():
        if k == "cu_seqlens":
            out[k] = v.numpy().astype(np.int64)
        else:
            out[k] = v.float().numpy().astype(np.float64)
    return small, out


def host_cpu():
    """CPU model and logical core count of this host (lscpu, else /proc/cpuinfo)."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if not model:
        try:
            with open("/proc/cpuinfo") as f:
                for line in f:
                    if line.lower().startswith(("model name", "cpu model")):
                        model = line.split(":", 1)[1].strip()
                        break
        except OSError:
            pass
    return {"cpu_model": model or "unknown", "host_logical_cores": os.cpu_count()}


class PinnedToOneCore:
    """Restrict this process to one core of its allowed set while timing the
    single-threaded oracle (restored afterwards)."""

    def __enter__(self):
        self.saved = None
        self.core = None
        if hasattr(os, "sched_setaffinity"):
            try:
                self.saved = os.sched_getaffinity(0)
                self.core = min(self.saved)
                os.sched_setaffinity(0, {self.core})
            except OSError:
                self.saved = None
        return self

    def cores(self):
        return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else 1

    def __exit__(self, *exc):
        if self.saved is not None:
            os.sched_setaffinity(0, self.saved)


ORACLE_ROWS = 4096          # contiguous tokens per oracle pass (at most)
REFERENCE_ARM_BUDGET_S = 150.0  # the whole --impl reference run, warm-up included


def reference_rows(wl, passes, budget_s=REFERENCE_ARM_BUDGET_S, lo=256):
    """Tokens per reference-arm step: ORACLE_ROWS when ``passes`` passes of that many
    fit in ``budget_s`` seconds, else fewer (a multiple of ``lo``, at least ``lo``),
    from the measured cost of one calibration pass over ``lo`` tokens."""
    small, inp = oracle_sample_inputs(wl, min(lo, wl.T))
    with PinnedToOneCore():
        t0 = time.perf_counter()
        oracle_step(small, inp)
        per_row = (time.perf_counter() - t0) / small.T
    rows = int(budget_s / max(passes, 1) / max(per_row, 1e-9)) // lo * lo
    return max(lo, min(ORACLE_ROWS, rows, wl.T))


def time_oracle(wl, rows, budget_s, passes=None, warmup=0):
    """The float64 oracle over a contiguous block of ``rows`` tokens of the workload,
    pinned to one core: whole passes of all operators until ``budget_s`` seconds
    have run (or exactly ``passes`` passes), and each operator's share.  Tokens/s
    of the block stand for the whole workload (extrapolated: every operator is
    independent per token, so its cost is linear in the token count)."""
    rows = min(rows, wl.T)
    small, inp = oracle_sample_inputs(wl, rows)
    per_op = {}
    with PinnedToOneCore() as pin:
        for _ in range(warmup):
            oracle_step(small, inp)
        n, t0 = 0, time.perf_counter()
        while True:
            oracle_step(small, inp, per_op)
            n += 1
            el = time.perf_counter() - t0
            if (passes is not None and n >= passes) or (passes is None and el >= budget_s):
                break
        cores = pin.cores()
        core = pin.core
    ops = {k: {"tokens_per_s": round(n * rows / v, 1), "s_per_pass": round(v / n, 4)}
           for k, v in per_op.items()}
    info = host_cpu()
    label = "extrapolated" if rows < wl.T else "full workload"
    return {"value": n * rows / el, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} passes of all 8 operators (forward and backward) over a contiguous block "
                      f"of {rows} tokens of {wl.name} (same widths and document law, seed 0), float64 "
                      f"numpy, one thread pinned to core {core}, {el:.1f} s; tokens/s {label} to the "
                      f"{wl.T}-token workload",
            "rows": rows, "passes": n, "seconds": round(el, 3), "tokens_per_s_label": label,
            "pinned_core": core, **info, "per_operator": ops, "ms_per_pass": 1e3 * el / n}


# ---------------------------------------------------------------------------

def run_single_op(args, wl, device):
    """Time one operator of the step alone: W untimed launches, then K launches,
    each timed with CUDA events, L2 flushed in between.  One JSON line."""
    from rmsnorm_fwd_bwd_03_gb300.workload import scaled
    from rmsnorm_fwd_bwd_03_gb300._build import build_library
    build_library()
    if args.tokens:
        wl = scaled(wl, args.tokens, f"_T{args.tokens}")
    step = Step(wl, device, seed=0)
    stream = torch.cuda.current_stream(device)
    calls = step.calls(stream.cuda_stream)
    run_calls(calls)  # every output of the step exists (h, rstd, positions, partials)
    call = [c for c in calls if c[0] == args.op]
    flush = L2Flush(device)
    for _ in range(args.warmup):
        flush()
        run_calls(call)
    torch.cuda.synchronize()
    times = []
    for _ in range(args.steps):
        flush()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(call) + 1)]
        run_calls(call, ev)
        times.append(ev)
    torch.cuda.synchronize()
    ms = sum(e[0].elapsed_time(e[-1]) for e in times) / args.steps
    alg = wl.algorithmic_bytes()[args.op]
    peak, peak_kind = _measured_peak()
    gbs = alg / (ms * 1e-3) / 1e9 if ms > 0 else 0.0
    print(json.dumps({"op": args.op, "workload": wl.name, "tokens": wl.T, "launches": args.steps,
                      "ms_per_launch": ms, "alg_bytes": alg, "GB/s": round(gbs, 1),
                      "frac": round(gbs / peak, 4), "peak": peak, "peak_kind": f"of {peak_kind}",
                      "device_error_word": step.gb.device_error()}))


def run_next_ops(args, wl, device):
    """Time the operators beyond the step (gated units with other activations and
    packed layouts, plain activations, strided / interleaved RoPE, LayerNorm,
    MXFP8 outputs of the RMSNorm and SwiGLU forwards) at
    the workload's widths: K launches each, CUDA events around each launch, L2
    flushed in between.  One JSON line with per-operator time and GB/s."""
    import rmsnorm_fwd_bwd_03_gb300 as gb
    from rmsnorm_fwd_bwd_03_gb300._build import build_library
    from rmsnorm_fwd_bwd_03_gb300.workload import scaled
    build_library()
    lib = gb.library()
    if args.tokens:
        wl = scaled(wl, args.tokens, f"_T{args.tokens}")
    T, H, I, D, Hq, Hk = wl.T, wl.H, wl.I, wl.D, wl.Hq, wl.Hk
    dt = wl.dtype
    b = 2 if dt == torch.bfloat16 else 4
    io = gb.BF16 if dt == torch.bfloat16 else gb.F32
    s = torch.cuda.current_stream(device).cuda_stream
    g = torch.Generator(device=device)
    g.manual_seed(0)
    rnd = lambda *shape: torch.randn(shape, generator=g, device=device).to(dt)  # noqa: E731
    p = lambda t: t.data_ptr()  # noqa: E731
    ops = {}

    # gated units on a packed [T, 2I] gate|up tensor and a packed [T, 2I] gradient
    packed, dout = rnd(T, 2 * I), rnd(T, I)
    out, grad = torch.empty(T, I, dtype=dt, device=device), torch.empty(T, 2 * I, dtype=dt, device=device)
    for act in ("silu", "gelu_tanh", "gelu_erf", "relu"):
        a = gb.ACT[act]
        ops[f"glu_fwd_packed_{act}"] = (lib.gbln_glu_fwd, (p(packed), p(packed) + I * b, p(out), T, I, 2 * I, 2 * I, I, a, io, s), 3 * T * I * b)
        ops[f"glu_bwd_packed_{act}"] = (lib.gbln_glu_bwd, (p(dout), p(packed), p(packed) + I * b, p(grad), p(grad) + I * b, T, I, I, 2 * I, 2 * I, 2 * I, 2 * I, a, io, s), 5 * T * I * b)
    x, dy = rnd(T, I), rnd(T, I)
    y = torch.empty_like(x)
    ops["act_fwd_gelu_tanh"] = (lib.gbln_act_fwd, (p(x), p(y), T * I, gb.ACT["gelu_tanh"], io, s), 2 * T * I * b)
    ops["act_bwd_gelu_tanh"] = (lib.gbln_act_bwd, (p(dy), p(x), p(y), T * I, gb.ACT["gelu_tanh"], io, s), 3 * T * I * b)

    # RoPE: Q and K rotated in place inside one packed QKV tensor; interleaved pairing
    W = (Hq + 2 * Hk) * D
    qkv = rnd(T, W)
    pos = gb.positions_from_cu_seqlens(torch.as_tensor(wl.cu_seqlens(), dtype=torch.int32, device=device), T)
    table = gb.rope_table(wl.max_pos(), D, wl.theta, device=device)
    rope_bytes = 2 * T * (Hq + Hk) * D * b + 4 * T
    ops["rope_fwd_packed_qkv_in_place"] = (lib.gbln_rope_fwd_ex, (p(qkv), p(qkv) + Hq * D * b, p(qkv), p(qkv) + Hq * D * b, p(pos), p(table), table.shape[0], T, Hq, Hk, D, W, W, W, W, 0, io, s), rope_bytes)
    q, k = rnd(T, Hq, D), rnd(T, Hk, D)
    qo, ko = torch.empty_like(q), torch.empty_like(k)
    ops["rope_fwd_interleaved"] = (lib.gbln_rope_fwd_ex, (p(q), p(k), p(qo), p(ko), p(pos), p(table), table.shape[0], T, Hq, Hk, D, Hq * D, Hk * D, Hq * D, Hk * D, 1, io, s), rope_bytes)

    # LayerNorm with residual and bias
    xl, rl, dyl, drl = rnd(T, H), rnd(T, H), rnd(T, H), rnd(T, H)
    wgt, bias = (1 + 0.1 * torch.randn(H, generator=g, device=device)).to(dt), rnd(H)
    yl, hl = torch.empty_like(xl), torch.empty_like(xl)
    mean, rstd = torch.empty(T, device=device), torch.empty(T, device=device)
    dxl = torch.empty_like(xl)
    P = gb.layernorm_bwd_num_partials(T, H, dt)
    part = torch.empty(P, 2 * H, device=device)
    dwl, dbl = torch.empty(H, device=device), torch.empty(H, device=device)
    ops["layernorm_fwd"] = (lib.gbln_layernorm_fwd, (p(xl), p(rl), p(wgt), p(bias), p(yl), p(hl), p(mean), p(rstd), T, H, wl.eps, io, io, s), 4 * T * H * b + 8 * T + 2 * H * b)
    ops["layernorm_bwd"] = (lib.gbln_layernorm_bwd, (p(dyl), p(drl), p(hl), p(wgt), p(mean), p(rstd), p(dxl), p(part), P, T, H, io, io, s), 4 * T * H * b + 8 * T + H * b)
    ops["layernorm_dwdb_finalize"] = (lib.gbln_layernorm_dwdb_finalize, (p(part), P, H, p(dwl), p(dbl), 0, s), 0)

    # MXFP8 outputs for the next GEMM: RMSNorm (+ residual) writing h, rstd and
    # y as E4M3 codes + one scale byte per 32 values (with and without the io copy
    # of y), and the packed SwiGLU forward writing only the MXFP8 result.
    if H % 32 == 0 and I % 32 == 0:
        yq, ysc = torch.empty(T, H, dtype=torch.uint8, device=device), torch.empty(T, H // 32, dtype=torch.uint8, device=device)
        wr = (1 + 0.1 * torch.randn(H, generator=g, device=device)).to(dt)
        mx_rms = 2 * T * H * b + T * H * b + T * H + T * H // 32 + 4 * T + H * b
        ops["rmsnorm_fwd_mxfp8"] = (lib.gbln_rmsnorm_fwd_mxfp8, (p(xl), p(rl), p(wr), None, p(yq), p(ysc), p(hl), p(rstd), T, H, wl.eps, io, io, s), mx_rms)
        ops["rmsnorm_fwd_mxfp8_and_y"] = (lib.gbln_rmsnorm_fwd_mxfp8, (p(xl), p(rl), p(wr), p(yl), p(yq), p(ysc), p(hl), p(rstd), T, H, wl.eps, io, io, s), mx_rms + T * H * b)
        gq, gsc = torch.empty(T, I, dtype=torch.uint8, device=device), torch.empty(T, I // 32, dtype=torch.uint8, device=device)
        ops["swiglu_fwd_packed_mxfp8"] = (lib.gbln_glu_fwd_mxfp8, (p(packed), p(packed) + I * b, p(gq), p(gsc), T, I, 2 * I, 2 * I, gb.ACT["silu"], io, s), 2 * T * I * b + T * I + T * I // 32)

    flush = L2Flush(device)
    peak, peak_kind = _measured_peak()
    res = {}
    for name in ["layernorm_fwd", "layernorm_bwd", "layernorm_dwdb_finalize"] + [n for n in ops if not n.startswith("layernorm")]:
        fn, fargs, alg = ops[name]
        for _ in range(args.warmup):
            flush()
            st = fn(*fargs)
            if st != 0:
                raise RuntimeError(f"{name}: status {st}")
        torch.cuda.synchronize()
        evs = []
        for _ in range(args.steps):
            flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn(*fargs)
            e1.record()
            evs.append((e0, e1))
        torch.cuda.synchronize()
        ms = sum(a.elapsed_time(c) for a, c in evs) / args.steps
        gbs = alg / (ms * 1e-3) / 1e9 if alg else 0.0
        res[name] = {"ms": round(ms, 5), "alg_bytes": alg, "GB/s": round(gbs, 1), "frac": round(gbs / peak, 4)}
    err = gb.device_error()
    print(json.dumps({"next_ops": res, "workload": wl.name, "tokens": T, "launches_each": args.steps,
                      "peak": peak, "peak_kind": f"of {peak_kind}", "device_error_word": err}))


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def reduce_max(value, world):
    if world == 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["gbln", "reference"], default="gbln")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--eager", action="store_true",
                    help="time the step as eight eager launches instead of one CUDA graph replay")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="seconds of oracle passes for the cpu_baseline leg (at least one pass)")
    ap.add_argument("--oracle-rows", type=int, default=0,
                    help="contiguous tokens of the workload per oracle pass (default: 4096 for "
                         "cpu_baseline; for --impl reference at most 4096, fewer when the run's "
                         "passes would not fit in a few minutes)")
    ap.add_argument("--op", choices=OPS, default=None,
                    help="time one operator alone (also the program under ncu captures)")
    ap.add_argument("--tokens", type=int, default=0,
                    help="with --op / --next: use the workload's widths with this many tokens")
    ap.add_argument("--next", action="store_true",
                    help="time the operators beyond the step (other activations, packed layouts, "
                         "strided / interleaved RoPE, LayerNorm) at the workload's widths")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    from rmsnorm_fwd_bwd_03_gb300.workload import WORKLOADS
    wl = WORKLOADS[args.workload]
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")

    config = {"workload": wl.name, "description": wl.description, "tokens": wl.T, "hidden": wl.H,
              "heads_q": wl.Hq, "heads_kv": wl.Hk, "head_dim": wl.D, "intermediate": wl.I,
              "rope_theta": wl.theta, "eps": wl.eps, "fused_residual": wl.residual,
              "global_batch_tokens": wl.T * world, "parallelism": f"replicas x{world}",
              "l2": "flushed between timed steps: 2x L2 written, then 2x L2 of another buffer read "
                    "(no step data and no dirty lines left in L2)"}

    if args.impl == "reference":
        if rank != 0:
            return
        # each step: one pass of the oracle over a contiguous block of the workload
        rows = args.oracle_rows or reference_rows(wl, args.steps + args.warmup)
        cb = time_oracle(wl, rows, 0.0, passes=args.steps, warmup=args.warmup)
        value = cb["value"]
        cb["sample"] = "each step: " + cb["sample"]
        line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": cb["ms_per_pass"],
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "impl": "reference", "config": config,
                "cpu_baseline": cb,
                "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (the library has no CPU path)")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    from rmsnorm_fwd_bwd_03_gb300._build import build_library
    build_library()

    if args.op:
        return run_single_op(args, wl, device)
    if args.next:
        return run_next_ops(args, wl, device)

    step = Step(wl, device, seed=rank)
    stream = torch.cuda.current_stream(device)
    calls = step.calls(stream.cuda_stream)
    flush = L2Flush(device)

    nk = len(calls)
    for _ in range(args.warmup):
        flush()
        run_calls(calls)
    torch.cuda.synchronize()

    # The step as one CUDA graph of the eight C-ABI calls (captured once, replayed
    # per step): the launch path a training loop would use.
    graph = None
    if not args.eager:
        cap = torch.cuda.Stream(device)
        cap.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cap):
            run_calls(step.calls(torch.cuda.current_stream(device).cuda_stream))
        torch.cuda.synchronize()
        for _ in range(args.warmup):
            flush()
            graph.replay()
        torch.cuda.synchronize()

    # Timed region 1 (the headline): K steps, events around each step, L2 flushed between.
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_wall0 = time.perf_counter()
        for k in range(args.steps):
            flush()
            evs[k][0].record()
            if graph is not None:
                graph.replay()
            else:
                run_calls(calls)
            evs[k][1].record()
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall0
    barrier(world)
    total_ms = sum(a.elapsed_time(b) for a, b in evs)
    total_ms_max = reduce_max(total_ms, world)
    ms_per_step = total_ms_max / args.steps
    value = world * wl.T * args.steps / (total_ms_max * 1e-3)

    # Timed region 2 (per-kernel durations for the roofline): eager steps with an
    # event between consecutive kernels on the launching stream.  Each interval
    # also holds that launch's front-end overhead, so these durations are upper
    # bounds and the GB/s derived from them lower bounds.
    kb = max(3, min(args.steps, 200))
    kevs = [[torch.cuda.Event(enable_timing=True) for _ in range(nk + 1)] for _ in range(kb)]
    torch.cuda.synchronize()
    for k in range(kb):
        flush()
        run_calls(calls, kevs[k])
    torch.cuda.synchronize()
    per_op = {name: 0.0 for name, _, _ in calls}
    eager_ms = 0.0
    for k in range(kb):
        e = kevs[k]
        eager_ms += e[0].elapsed_time(e[nk])
        for j, (name, _, _) in enumerate(calls):
            per_op[name] += e[j].elapsed_time(e[j + 1])
    for name in per_op:
        per_op[name] = reduce_max(per_op[name], world)

    alg = wl.algorithmic_bytes()
    peak, peak_kind = _measured_peak()
    kernels = {}
    for name in per_op:
        ms = per_op[name] / kb
        gbs = alg[name] / (ms * 1e-3) / 1e9 if ms > 0 else 0.0
        kernels[name] = {"ms": round(ms, 5), "alg_bytes": alg[name], "GB/s": round(gbs, 1),
                         "frac_of_peak": round(gbs / peak, 4)}
    dom = max(per_op, key=per_op.get)
    dom_ms = per_op[dom] / kb
    achieved = alg[dom] / (dom_ms * 1e-3) / 1e9
    tr = NCU_TRAFFIC.get((wl.name, dom))
    traffic = tr["bytes"] if tr and tr.get("src_sha") == _src_sha(dom) else None
    step_bytes = sum(alg.values())
    roofline = {"kernel": dom, "bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                "peak_kind": f"of {peak_kind}", "unit": "GB/s", "frac": round(achieved / peak, 4),
                "traffic": traffic, "alg_bytes_per_launch": alg[dom],
                "frac_of_8TBps": round(achieved / 8000.0, 4)}

    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            # arithmetic type of the kernels (float32 everywhere); io_dtype is what they read and write
            "dtype": "f32", "io_dtype": "bf16" if wl.dtype == torch.bfloat16 else "f32", "data": "synthetic",
            "config": config,
            "achieved_hbm_gbs_step": round(step_bytes / (ms_per_step * 1e-3) / 1e9, 1),
            "frac_of_peak_step": round(step_bytes / (ms_per_step * 1e-3) / 1e9 / peak, 4),
            "roofline": roofline, "kernels": kernels,
            "gpu_launches": nk * args.steps,
            "launch": "eager C-ABI calls" if graph is None else "CUDA graph of the 8 C-ABI calls, one replay per step",
            "per_kernel_region": {"steps": kb, "launch": "eager, event between kernels",
                                  "ms_per_step": round(eager_ms / kb, 5), "gpu_launches": nk * kb},
            "wall_s_timed_region": round(t_wall, 3),
            "clocks": clk.summary()}

    if not args.no_e2e:
        del graph
        ksteps = max(3, min(args.steps, 50))
        line["e2e"] = e2e_pipelined(wl, device, ksteps, args.warmup, world, seed=rank)
        line["gpu_launches_e2e"] = nk * ksteps

    # Bit 1 is set by a kernel whose bounded wait on its own copies ran out.
    line["device_error_word"] = step.gb.device_error()
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = time_oracle(wl, args.oracle_rows or ORACLE_ROWS, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line))


if __name__ == "__main__":
    main()
