"""Seeded synthetic inputs for the dense product D = A @ B^T.

This module only draws random matrices (torch CPU generators, fixed seeds) and
lays them out; it holds none of the product's arithmetic.  Both the CUDA path
and the CPU oracle consume the exact bytes it returns.

Workloads (shapes, element types, value distributions and seeds):

=================  ================================  ==========================  ======
name               shape / types                     values                      seed
=================  ================================  ==========================  ======
single_cta         1 x (128x64 . (64x64)^T), f16     U[-1,1]; ints {-3..3}       1 / 2
                   -> f32
square4096_bf16    4096^3, bf16 TN -> bf16           N(0,1)/sqrt(K)              3
square8192_bf16    8192^3, bf16 TN -> f32            U[-1,1]                     4
batched256_f16     512 x 256^3, f16 TN -> f16        N(0,1)                      5
fp8_block8192      8192^3, e4m3 TN, fp32 scales per  pre-quantisation N(0,1),    6
                   1x128 (A) / 128x128 (B) -> bf16   scale = block absmax / 448
=================  ================================  ==========================  ======

The single-CTA example is the TVM TIRx "Blackwell Tensor Cores" walk-through
(Out = A @ B.T with A 128x64 and B 64x64, fp16 in, fp32 out).  The fp8 recipe
follows "Hopper and Blackwell GEMM", concept "FP8 and FP4, with block scaling":
every block of a row of A (1x128) and of B (128x128) carries its own fp32
scale; 448 is the largest finite E4M3 value.  An all-zero block gets scale 1.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import torch

E4M3_MAX = 448.0

TORCH_DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32,
                "tf32": torch.float32, "e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}
FP8_MAX = {"e4m3": 448.0, "e5m2": 57344.0}


@dataclass
class Workload:
    name: str
    M: int
    N: int
    K: int
    batch: int
    dtype_in: str           # "f16" | "bf16" | "e4m3"
    dtype_out: str          # "f32" | "bf16" | "f16"
    dist: str               # "uniform" | "normal" | "normal_sqrtk" | "ints"
    seed: int
    block_scaled: bool = False
    extra: dict = field(default_factory=dict)

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K * self.batch


WORKLOADS = {
    "single_cta": Workload("single_cta", 128, 64, 64, 1, "f16", "f32", "uniform", 1),
    "single_cta_ints": Workload("single_cta_ints", 128, 64, 64, 1, "f16", "f32", "ints", 2),
    "square4096_bf16": Workload("square4096_bf16", 4096, 4096, 4096, 1, "bf16", "bf16", "normal_sqrtk", 3),
    "square8192_bf16": Workload("square8192_bf16", 8192, 8192, 8192, 1, "bf16", "f32", "uniform", 4),
    "batched256_f16": Workload("batched256_f16", 256, 256, 256, 512, "f16", "f16", "normal", 5),
    "fp8_block8192": Workload("fp8_block8192", 8192, 8192, 8192, 1, "e4m3", "bf16", "normal", 6,
                              block_scaled=True),
}


def _draw(shape, dist: str, gen: torch.Generator, K: int) -> torch.Tensor:
    if dist == "uniform":
        return torch.rand(shape, generator=gen, dtype=torch.float32) * 2.0 - 1.0
    if dist == "normal":
        return torch.randn(shape, generator=gen, dtype=torch.float32)
    if dist == "normal_sqrtk":
        return torch.randn(shape, generator=gen, dtype=torch.float32) / float(K) ** 0.5
    if dist == "ints":
        return torch.randint(-3, 4, shape, generator=gen).to(torch.float32)
    raise ValueError(dist)


def block_quantize_e4m3(x: torch.Tensor, block_rows: int, block_cols: int = 128, fmt: str = "e4m3"):
    """Quantise a 2-D fp32 matrix to an 8-bit format with one fp32 scale per block.

    scale = absmax(block) / max_finite (448 for E4M3, 57344 for E5M2; 1 for an
    all-zero block), q = fmt(x / scale) using torch's round-to-nearest cast.
    Returns (q, scales) with scales of shape (ceil(R/block_rows), ceil(C/block_cols)).
    """
    fmax = FP8_MAX[fmt]
    R, C = x.shape
    rb = (R + block_rows - 1) // block_rows
    cb = (C + block_cols - 1) // block_cols
    pad = torch.zeros(rb * block_rows, cb * block_cols, dtype=torch.float32)
    pad[:R, :C] = x
    blocks = pad.view(rb, block_rows, cb, block_cols)
    amax = blocks.abs().amax(dim=(1, 3))
    scale = torch.where(amax > 0, amax / fmax, torch.ones_like(amax))
    scaled = blocks / scale[:, None, :, None]
    q = scaled.clamp(-fmax, fmax).to(TORCH_DTYPES[fmt])
    q = q.view(rb * block_rows, cb * block_cols)[:R, :C].contiguous()
    return q, scale.contiguous()


@dataclass
class Problem:
    """Host (CPU) tensors of one problem; A is [batch][M][K], B is [batch][N][K]."""
    wl: Workload
    A: torch.Tensor
    B: torch.Tensor
    scale_a: Optional[torch.Tensor] = None   # [M][ceil(K/128)] fp32
    scale_b: Optional[torch.Tensor] = None   # [ceil(N/128)][ceil(K/128)] fp32


def make(wl: Workload | str, *, seed: Optional[int] = None, dist: Optional[str] = None,
         M: Optional[int] = None, N: Optional[int] = None, K: Optional[int] = None,
         batch: Optional[int] = None, dtype_in: Optional[str] = None,
         dtype_b: Optional[str] = None) -> Problem:
    """Draw the inputs of a workload (optionally at another size, seed, value mix or
    input type; dtype_b sets B's type separately for 8-bit pairings)."""
    if isinstance(wl, str):
        wl = WORKLOADS[wl]
    wl = Workload(wl.name, M or wl.M, N or wl.N, K or wl.K, batch or wl.batch, dtype_in or wl.dtype_in,
                  wl.dtype_out, dist or wl.dist, wl.seed if seed is None else seed, wl.block_scaled)
    wl.extra["dtype_b"] = dtype_b or wl.dtype_in
    gen = torch.Generator().manual_seed(wl.seed)
    shape_a = (wl.batch, wl.M, wl.K) if wl.batch > 1 else (wl.M, wl.K)
    shape_b = (wl.batch, wl.N, wl.K) if wl.batch > 1 else (wl.N, wl.K)
    xa = _draw(shape_a, wl.dist, gen, wl.K)
    xb = _draw(shape_b, wl.dist, gen, wl.K)
    if not wl.block_scaled:
        t = TORCH_DTYPES[wl.dtype_in]
        return Problem(wl, xa.to(t).contiguous(), xb.to(TORCH_DTYPES[wl.extra["dtype_b"]]).contiguous())
    if wl.batch != 1:
        raise ValueError("block-scaled workloads are single problems")
    if wl.dist == "ints":
        # exact variant: small integers and scales in {1/2, 1, 2}, so every block
        # product, every scaled partial and every running sum is exact in fp32
        kb = (wl.K + 127) // 128
        qa = xa.to(TORCH_DTYPES[wl.dtype_in])
        qb = xb.to(TORCH_DTYPES[wl.extra["dtype_b"]])
        sa = torch.pow(2.0, torch.randint(-1, 2, (wl.M, kb), generator=gen).float())
        sb = torch.pow(2.0, torch.randint(-1, 2, ((wl.N + 127) // 128, kb), generator=gen).float())
        return Problem(wl, qa.contiguous(), qb.contiguous(), sa.contiguous(), sb.contiguous())
    qa, sa = block_quantize_e4m3(xa, 1, 128, wl.dtype_in)
    qb, sb = block_quantize_e4m3(xb, 128, 128, wl.extra["dtype_b"])
    return Problem(wl, qa, qb, sa, sb)


def sample_rows(M: int, batch: int = 1, n_random: int = 64, seed: int = 0, tile_m: int = 128):
    """Flat row indices b*M+m to check at full size: seeded random rows plus the
    first and last row of every tile edge (tile_m), in every batch sampled."""
    gen = torch.Generator().manual_seed(seed)
    rows = set(torch.randint(0, M * batch, (n_random,), generator=gen).tolist())
    for b in ({0, batch - 1} if batch > 1 else {0}):
        for m0 in range(0, M, tile_m):
            rows.add(b * M + m0)
            rows.add(b * M + min(m0 + tile_m, M) - 1)
    return sorted(rows)
