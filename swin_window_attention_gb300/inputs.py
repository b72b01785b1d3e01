"""Seeded synthetic inputs and the workload table for Swin window attention.

This module holds no attention arithmetic: it only names the workloads (shapes, window
size, shift, head count, I/O dtype) and draws their random inputs on the CPU with a
seeded ``torch.Generator``, so the GPU path, the oracle and the bench all see the same
values on any machine.

Workloads follow the Swin stage pyramid the NVIDIA Swin talk describes (section 1: stages
of falling resolution and growing width) at the ImageNet-style 224 and 384 resolutions;
no dataset or trained weight is involved. Seeds: ``1000*config + 10*stage`` for qkv, +1
for the bias table, +2 for the upstream gradient.

Distributions: qkv and dO ~ N(0, 1); the bias table is normal with std 0.02 truncated
at +-0.04 (resampled outside). Activations are rounded to bf16 except in the fp32 tiny
workload.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    config: int
    stage: int
    B: int
    H: int
    W: int
    C: int
    nH: int
    M: int
    s: int
    dtype: str  # "bf16" or "fp32" activation I/O
    bwd: bool = False

    @property
    def hd(self) -> int:
        return self.C // self.nH

    @property
    def N(self) -> int:
        return self.M * self.M

    @property
    def nW(self) -> int:
        return (self.H // self.M) * (self.W // self.M)

    @property
    def tokens(self) -> int:
        return self.B * self.H * self.W

    @property
    def window_heads(self) -> int:
        return self.B * self.nW * self.nH

    @property
    def seed(self) -> int:
        return 1000 * self.config + 10 * self.stage

    def with_batch(self, B: int) -> "Workload":
        return Workload(self.name, self.config, self.stage, B, self.H, self.W, self.C,
                        self.nH, self.M, self.s, self.dtype, self.bwd)


def _w(name, config, stage, B, HW, C, nH, M, s, dtype="bf16", bwd=False):
    return Workload(name, config, stage, B, HW, HW, C, nH, M, s, dtype, bwd)


WORKLOADS = [
    _w("tiny", 1, 0, 1, 8, 64, 2, 4, 2, dtype="fp32"),
    _w("swin_t_s1_wmsa", 2, 0, 32, 56, 96, 3, 7, 0),
    _w("swin_t_s1_swmsa", 2, 1, 32, 56, 96, 3, 7, 3),
    _w("swin_l224_s1", 3, 1, 64, 56, 192, 6, 7, 3),
    _w("swin_l224_s2", 3, 2, 64, 28, 384, 12, 7, 3),
    _w("swin_l224_s3", 3, 3, 64, 14, 768, 24, 7, 3),
    _w("swin_l224_s4", 3, 4, 64, 7, 1536, 48, 7, 0),
    _w("swin_l384_s1", 4, 1, 16, 96, 192, 6, 12, 6),
    _w("swin_l384_s2", 4, 2, 16, 48, 384, 12, 12, 6),
    _w("swin_l384_s3", 4, 3, 16, 24, 768, 24, 12, 6),
    _w("swin_l384_s4", 4, 4, 16, 12, 1536, 48, 12, 0),
    _w("swin_b224_s1", 5, 1, 128, 56, 128, 4, 7, 3, bwd=True),
    _w("swin_b224_s2", 5, 2, 128, 28, 256, 8, 7, 3, bwd=True),
    _w("swin_b224_s3", 5, 3, 128, 14, 512, 16, 7, 3, bwd=True),
    _w("swin_b224_s4", 5, 4, 128, 7, 1024, 32, 7, 0, bwd=True),
]
BY_NAME = {w.name: w for w in WORKLOADS}


def by_config(config: int):
    return [w for w in WORKLOADS if w.config == config]


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def normal(shape, seed: int) -> torch.Tensor:
    """fp32 N(0,1) on the CPU."""
    return torch.randn(*shape, generator=_gen(seed), dtype=torch.float32)


def trunc_normal(shape, seed: int, std: float = 0.02, bound: float = 0.04) -> torch.Tensor:
    """fp32 normal(0, std^2) with every sample outside +-bound redrawn."""
    g = _gen(seed)
    x = torch.randn(*shape, generator=g, dtype=torch.float32) * std
    bad = x.abs() > bound
    while bool(bad.any()):
        n = int(bad.sum())
        x[bad] = torch.randn(n, generator=g, dtype=torch.float32) * std
        bad = x.abs() > bound
    return x


def _act(x: torch.Tensor, dtype: str) -> torch.Tensor:
    return x.to(torch.bfloat16) if dtype == "bf16" else x


def make_qkv(wl: Workload, seed_offset: int = 0) -> torch.Tensor:
    """[B,H,W,3C] activation (bf16, or fp32 for the fp32 workload), CPU."""
    return _act(normal((wl.B, wl.H, wl.W, 3 * wl.C), wl.seed + seed_offset), wl.dtype)


def make_table(wl: Workload) -> torch.Tensor:
    """[(2M-1)^2, nH] fp32 relative-position bias table, CPU."""
    return trunc_normal(((2 * wl.M - 1) ** 2, wl.nH), wl.seed + 1)


def make_dout(wl: Workload) -> torch.Tensor:
    """[B,H,W,C] upstream gradient, same dtype as the activation, CPU."""
    return _act(normal((wl.B, wl.H, wl.W, wl.C), wl.seed + 2), wl.dtype)


def make_producer(wl: Workload):
    """Inputs of the producer step in front of the attention (LayerNorm over C, then the
    qkv projection), CPU: x [B,H,W,C] bf16 ~ N(0,1); gamma = 1 + 0.1 N(0,1) and
    beta = 0.1 N(0,1), fp32 [C]; W [3C, C] bf16, trunc-normal (std 0.02, +-0.04); b fp32
    [3C] = 0.02 N(0,1). Seeds: the workload's seed + 3, 4, 5, 6."""
    C = wl.C
    x = normal((wl.B, wl.H, wl.W, C), wl.seed + 3).to(torch.bfloat16)
    gb = normal((2, C), wl.seed + 4)
    gamma = 1.0 + 0.1 * gb[0]
    beta = 0.1 * gb[1]
    w = trunc_normal((3 * C, C), wl.seed + 5).to(torch.bfloat16)
    b = 0.02 * normal((3 * C,), wl.seed + 6)
    return x, gamma.contiguous(), beta.contiguous(), w, b


def make_consumer(wl: Workload):
    """Inputs of the consumer step after the attention (the output projection, then bias
    and residual), CPU: o [B,H,W,C] bf16 ~ N(0, 0.5^2) (the attention output, an average of
    N(0,1) values); Wp [C, C] bf16, trunc-normal (std 0.02, +-0.04); bp fp32 [C] =
    0.02 N(0,1); the residual (the block input) [B,H,W,C] bf16 ~ N(0,1). Seeds: the
    workload's seed + 7, 8, 9, 10."""
    C = wl.C
    o = (0.5 * normal((wl.B, wl.H, wl.W, C), wl.seed + 7)).to(torch.bfloat16)
    wp = trunc_normal((C, C), wl.seed + 8).to(torch.bfloat16)
    bp = 0.02 * normal((C,), wl.seed + 9)
    r = normal((wl.B, wl.H, wl.W, C), wl.seed + 10).to(torch.bfloat16)
    return o, wp, bp.contiguous(), r


FP8_MAX = 448.0  # the largest finite OCP FP8 E4M3 value


def make_qkv_fp8(wl: Workload):
    """The workload's qkv (the same seeded N(0,1) draw as make_qkv) encoded as OCP FP8
    E4M3 with one scale per tensor (q, k, v): scale = max|x| / 448, x8 = round(x / scale)
    to E4M3 (torch's round-to-nearest-even cast), CPU. Returns (qkv8 [B,H,W,3C]
    torch.float8_e4m3fn, (scale_q, scale_k, scale_v))."""
    x = normal((wl.B, wl.H, wl.W, 3 * wl.C), wl.seed)
    parts, scales = [], []
    for t in range(3):
        xt = x[..., t * wl.C:(t + 1) * wl.C]
        sc = float(xt.abs().max()) / FP8_MAX
        parts.append((xt / sc).to(torch.float8_e4m3fn))
        scales.append(sc)
    return torch.cat(parts, dim=-1), tuple(scales)


def fp8_decoded_f64(qkv8: torch.Tensor, scales, C: int):
    """Exact float64 numpy values of scale_t * x8 for each tensor t of an E4M3 qkv."""
    x = qkv8.to(torch.float64)
    for t in range(3):
        x[..., t * C:(t + 1) * C] *= scales[t]
    return x.numpy()


def act_f64(x: torch.Tensor):
    """Exact float64 numpy copy of the values the GPU path sees: bf16 inputs are widened
    as they are; fp32 inputs are first rounded to bf16 (round-to-nearest-even), which
    is what the library does on load for fp32 I/O."""
    if x.dtype == torch.float32:
        x = x.to(torch.bfloat16)
    return x.to(torch.float64).numpy()
