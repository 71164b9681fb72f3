"""Seeded synthetic inputs for the layer-operator workloads.

This module only draws random numbers and lays out shapes; it holds none of the
operators' arithmetic, so both the CUDA tests and the CPU oracle can take their
inputs from it.  Shapes follow the layer widths the sources discuss: a small
Qwen-0.5B-width fp32 case, Qwen3-0.6B, Llama-3-8B (also as packed documents of
lognormal length with outlier channels, after "Fast-LLM: 高效大语言模型训练框架",
§三 训练配置示例: micro-batches counted in tokens, maximum_document_length) and a
70B-width layer.  No dataset is involved: every tensor is N(0, 1) (the RMSNorm
weight is 1 + 0.1 N(0, 1)) drawn from torch's generator with a fixed seed, in a
fixed order, in float32 and then rounded to the I/O dtype.
"""

from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    description: str
    T: int                 # tokens (rows)
    H: int                 # hidden size
    eps: float
    residual: bool         # fused residual add in the RMSNorm
    Hq: int
    Hk: int
    D: int                 # head size
    theta: float
    I: int                 # SwiGLU intermediate size
    dtype: torch.dtype
    seq_len: int = 0       # equal-length sequences (0 = packed documents)
    packed: bool = False
    outlier_frac: float = 0.0
    outlier_scale: float = 1.0

    @property
    def io(self) -> str:
        return "f32" if self.dtype == torch.float32 else "bf16"

    def doc_lengths(self, seed: int = 0) -> list:
        if not self.packed:
            return [self.seq_len] * (self.T // self.seq_len)
        return lognormal_doc_lengths(self.T, seed=seed)

    def cu_seqlens(self, seed: int = 0) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.doc_lengths(seed))]).astype(np.int32)

    def max_pos(self, seed: int = 0) -> int:
        return int(max(self.doc_lengths(seed)))

    def algorithmic_bytes(self) -> dict:
        """Minimum HBM bytes per call of each operator (each input read once, each output written once)."""
        b = 2 if self.dtype == torch.bfloat16 else 4
        T, H, I = self.T, self.H, self.I
        rows = T * H * b
        heads = T * (self.Hq + self.Hk) * self.D * b
        return {
            "positions": 4 * T,
            "rmsnorm_fwd": (4 if self.residual else 2) * rows + H * b + 4 * T,
            "rope_fwd": 2 * heads + 4 * T,
            "swiglu_fwd": 3 * T * I * b,
            "swiglu_bwd": 5 * T * I * b,
            "rope_bwd": 2 * heads + 4 * T,
            "rmsnorm_bwd": (4 if self.residual else 3) * rows + H * b + 4 * T,
            "rmsnorm_dw_finalize": 0,  # workspace traffic only; no algorithmic bytes
        }


WORKLOADS = {
    "qwen05b_tiny_f32": Workload(
        "qwen05b_tiny_f32", "tiny fp32 layer ops: 1 seq x 256 tokens, hidden 896, Q 14 x 64, K 2 x 64, SwiGLU 4864",
        T=256, H=896, eps=1e-6, residual=True, Hq=14, Hk=2, D=64, theta=1e6, I=4864,
        dtype=torch.float32, seq_len=256),
    "qwen3_0p6b": Workload(
        "qwen3_0p6b", "Qwen3-0.6B-shaped bf16: 8 seqs x 2048 tokens, hidden 1024, Q 16 x 128, K 8 x 128, SwiGLU 3072",
        T=16384, H=1024, eps=1e-6, residual=True, Hq=16, Hk=8, D=128, theta=1e6, I=3072,
        dtype=torch.bfloat16, seq_len=2048),
    "llama3_8b": Workload(
        "llama3_8b", "Llama-3-8B-shaped bf16: 4 seqs x 8192 tokens, hidden 4096, Q 32 x 128, K 8 x 128, SwiGLU 14336",
        T=32768, H=4096, eps=1e-5, residual=True, Hq=32, Hk=8, D=128, theta=5e5, I=14336,
        dtype=torch.bfloat16, seq_len=8192),
    "llama3_8b_packed_outliers": Workload(
        "llama3_8b_packed_outliers", "packed variable-length bf16: 65536 tokens of lognormal documents, Llama-3-8B widths, 1% of x's channels x50",
        T=65536, H=4096, eps=1e-5, residual=True, Hq=32, Hk=8, D=128, theta=5e5, I=14336,
        dtype=torch.bfloat16, packed=True, outlier_frac=0.01, outlier_scale=50.0),
    "llama70b_width": Workload(
        "llama70b_width", "70B-width bf16: 2 seqs x 16384 tokens, hidden 8192, Q 64 x 128, K 8 x 128, SwiGLU 28672",
        T=32768, H=8192, eps=1e-5, residual=True, Hq=64, Hk=8, D=128, theta=5e5, I=28672,
        dtype=torch.bfloat16, seq_len=16384),
}

# Order of the configurations as the task lists them (index 0 = the small parity case).
ORDER = ["qwen05b_tiny_f32", "qwen3_0p6b", "llama3_8b", "llama3_8b_packed_outliers", "llama70b_width"]


def lognormal_doc_lengths(total: int, median: int = 512, sigma: float = 1.0, lo: int = 32,
                          hi: int = 8192, seed: int = 0) -> list:
    """Document lengths ln L ~ N(ln median, sigma), rounded, clipped to [lo, hi], drawn
    until they cover ``total`` tokens; the last one is cut to fit exactly."""
    rng = np.random.default_rng(seed)
    out, s = [], 0
    while s < total:
        L = int(np.clip(round(float(rng.lognormal(math.log(median), sigma))), lo, hi))
        L = min(L, total - s)
        out.append(L)
        s += L
    return out


def outlier_channels(H: int, frac: float, seed: int = 0) -> np.ndarray:
    """round(frac * H) channel indices chosen by a seeded permutation."""
    k = int(round(frac * H))
    return np.sort(np.random.default_rng(seed + 1).permutation(H)[:k])


def _randn(g, shape, device, dtype):
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(dtype)


def make_inputs(wl: Workload, device="cuda", seed: int = 0, parts=("rmsnorm", "rope", "swiglu")) -> dict:
    """All inputs of one fwd + bwd pass of the three operators, in a fixed draw order.

    Keys: x, residual, weight, dy, dres (RMSNorm); q, k, dq, dk, cu_seqlens (RoPE);
    gate, up, dout (SwiGLU).  Parts not requested are skipped but their draws are
    still consumed only when generated, so each part's tensors depend on the seed
    and on which parts come before it in the fixed order rms -> rope -> swiglu.
    """
    device = torch.device(device)
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    out = {}
    T, H = wl.T, wl.H
    if "rmsnorm" in parts:
        x = torch.randn((T, H), generator=g, device=device, dtype=torch.float32)
        if wl.outlier_frac > 0:
            ch = torch.as_tensor(outlier_channels(H, wl.outlier_frac, seed), device=device)
            x[:, ch] *= wl.outlier_scale
        out["x"] = x.to(wl.dtype)
        out["residual"] = _randn(g, (T, H), device, wl.dtype)
        w = torch.randn((H,), generator=g, device=device, dtype=torch.float32)
        out["weight"] = (1.0 + 0.1 * w).to(wl.dtype)
        out["dy"] = _randn(g, (T, H), device, wl.dtype)
        out["dres"] = _randn(g, (T, H), device, wl.dtype)
    if "rope" in parts:
        out["q"] = _randn(g, (T, wl.Hq, wl.D), device, wl.dtype)
        out["k"] = _randn(g, (T, wl.Hk, wl.D), device, wl.dtype)
        out["dq"] = _randn(g, (T, wl.Hq, wl.D), device, wl.dtype)
        out["dk"] = _randn(g, (T, wl.Hk, wl.D), device, wl.dtype)
        out["cu_seqlens"] = torch.as_tensor(wl.cu_seqlens(seed), dtype=torch.int32, device=device)
    if "swiglu" in parts:
        I = wl.I
        out["gate"] = _randn(g, (T, I), device, wl.dtype)
        out["up"] = _randn(g, (T, I), device, wl.dtype)
        out["dout"] = _randn(g, (T, I), device, wl.dtype)
    return out


def scaled(wl: Workload, T: int, name_suffix: str = "_small") -> Workload:
    """The same widths with fewer tokens (for quick parity runs); packed docs keep their law."""
    seq = min(wl.seq_len, T) if wl.seq_len else 0
    if seq and T % seq:
        seq = T
    return dataclasses.replace(wl, name=wl.name + name_suffix, T=T, seq_len=seq)
