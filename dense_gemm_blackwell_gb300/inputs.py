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
mxfp8_8192         8192^3, e4m3 TN, E8M0 scale per   pre-quantisation N(0,1),    7
                   32 K elements (MXFP8) -> bf16     OCP shared exponent
mxfp4_8192         8192^3, e2m1 TN (packed), E8M0    pre-quantisation N(0,1),    8
                   per 32 (MXFP4) -> bf16            OCP shared exponent
nvfp4_8192         8192^3, e2m1 TN (packed), E4M3    pre-quantisation N(0,1),    9
                   per 16 + fp32 per tensor -> bf16  two-level scale
=================  ================================  ==========================  ======

The single-CTA example is the TVM TIRx "Blackwell Tensor Cores" walk-through
(Out = A @ B.T with A 128x64 and B 64x64, fp16 in, fp32 out).  The fp8 recipe
follows "Hopper and Blackwell GEMM", concept "FP8 and FP4, with block scaling":
every block of a row of A (1x128) and of B (128x128) carries its own fp32
scale; 448 is the largest finite E4M3 value.  An all-zero block gets scale 1.

The hardware block-scaled formats follow the same page's table (MXFP8: 32
elements per E8M0 scale; MXFP4: E2M1 elements, 32 per E8M0 scale; NVFP4: E2M1
elements, 16 per E4M3 scale plus one fp32 scale per tensor).  MX scales are the
OCP shared exponent of each block, floor(log2(absmax)) minus the element
format's largest exponent (8 for E4M3, 2 for E2M1), elements saturated to the
format's range.  NVFP4 uses a tensor scale absmax / (448 * 6), block scales
E4M3(block absmax / (6 * tensor scale)), then E2M1 of x / (block * tensor
scale).  Scale bytes are handed over in the tiled layout the library and the
oracle both document (512-byte tiles of 128 rows x 4 scales; see
pack_scales_tiled).  E2M1 operands are packed two per byte, element 2i in the
low nibble of byte i.
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
    "mxfp8_8192": Workload("mxfp8_8192", 8192, 8192, 8192, 1, "e4m3", "bf16", "normal", 7,
                           extra={"scale_mode": "mx"}),
    "mxfp4_8192": Workload("mxfp4_8192", 8192, 8192, 8192, 1, "e2m1", "bf16", "normal", 8,
                           extra={"scale_mode": "mx"}),
    "nvfp4_8192": Workload("nvfp4_8192", 8192, 8192, 8192, 1, "e2m1", "bf16", "normal", 9,
                           extra={"scale_mode": "nv"}),
}

# E2M1 magnitudes in code order (codes 0..7; bit 3 is the sign): the OCP MX
# 4-bit element format, 2 exponent bits with bias 1 and 1 mantissa bit
E2M1_GRID = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)
MX_EMAX = {"e4m3": 8, "e5m2": 15, "e2m1": 2}     # exponent of each element format's largest value


def e2m1_codes(x: torch.Tensor) -> torch.Tensor:
    """Round fp32 values to the nearest E2M1 value (ties to the even code, beyond
    6 saturated); returns the 4-bit codes as uint8.  The values are spaced 0.5
    below 2, 1 in [2, 4) and 2 in [4, 6], and codes count along them, so
    round-half-to-even within each binade picks the nearest code and, at a
    tie, the even one."""
    a = x.abs().clamp(max=6.0)
    idx = torch.where(a < 2.0, torch.round(a * 2.0),
                      torch.where(a < 4.0, 4.0 + torch.round(a - 2.0), 6.0 + torch.round((a - 4.0) * 0.5)))
    idx = idx.to(torch.int64)
    sign = ((x < 0) & (idx > 0)).to(torch.int64)
    return (idx | (sign << 3)).to(torch.uint8)


def pack_e2m1(codes: torch.Tensor) -> torch.Tensor:
    """[..., K] 4-bit codes -> [..., K/2] bytes, element 2i in the low nibble."""
    c = codes.to(torch.uint8)
    return (c[..., 0::2] | (c[..., 1::2] << 4)).contiguous()


def pack_scales_tiled(codes: torch.Tensor, fill: int = 127) -> torch.Tensor:
    """Scale bytes [..., R, KB] (row-major) -> the tiled layout: 512-byte tiles of
    128 rows x 4 scale columns, tile (r // 128, kb // 4) at tile index
    (r // 128) * ceil(KB / 4) + kb // 4, and inside a tile at byte
    (r % 32) * 16 + ((r // 32) % 4) * 4 + kb % 4.  Entries past R or KB hold
    `fill`.  Leading (batch) dimensions are kept; returns [..., bytes] uint8."""
    *lead, R, KB = codes.shape
    RB, KQ = (R + 127) // 128, (KB + 3) // 4
    pad = torch.full((*lead, RB * 128, KQ * 4), fill, dtype=torch.uint8)
    pad[..., :R, :KB] = codes.to(torch.uint8)
    # r = rb*128 + g*32 + l, kb = q*4 + j  ->  [rb][q][l][g][j]
    t = pad.reshape(*lead, RB, 4, 32, KQ, 4)                  # [rb][g][l][q][j]
    n = len(lead)
    t = t.permute(*range(n), n + 0, n + 3, n + 2, n + 1, n + 4)   # [rb][q][l][g][j]
    return t.contiguous().reshape(*lead, RB * KQ * 512)


def _mx_quantize(x: torch.Tensor, fmt: str):
    """OCP MX quantisation of [R, K] along K in blocks of 32: (element codes or
    float8 tensor, E8M0 scale codes [R, ceil(K/32)])."""
    R, K = x.shape
    KB = (K + 31) // 32
    pad = torch.zeros(R, KB * 32, dtype=torch.float32)
    pad[:, :K] = x
    blocks = pad.view(R, KB, 32)
    amax = blocks.abs().amax(dim=2)
    e = torch.floor(torch.log2(torch.where(amax > 0, amax, torch.ones_like(amax)))) - MX_EMAX[fmt]
    e = torch.where(amax > 0, e, torch.zeros_like(e)).clamp(-127, 127)
    scaled = (blocks / torch.pow(2.0, e)[:, :, None]).view(R, KB * 32)[:, :K]
    codes = (e + 127).to(torch.uint8)
    if fmt == "e2m1":
        return e2m1_codes(scaled), codes
    q = scaled.clamp(-FP8_MAX[fmt], FP8_MAX[fmt]).to(TORCH_DTYPES[fmt])
    return q.contiguous(), codes


def _nv_quantize(x: torch.Tensor, tensor_scale: float):
    """NVFP4 quantisation of [R, K] along K in blocks of 16: (E2M1 codes, E4M3
    block-scale codes [R, ceil(K/16)])."""
    R, K = x.shape
    KB = (K + 15) // 16
    pad = torch.zeros(R, KB * 16, dtype=torch.float32)
    pad[:, :K] = x
    blocks = pad.view(R, KB, 16)
    amax = blocks.abs().amax(dim=2)
    s = (amax / (6.0 * tensor_scale)).clamp(max=448.0).to(torch.float8_e4m3fn)
    sv = s.float()
    denom = torch.where(sv > 0, sv * tensor_scale, torch.ones_like(sv))
    scaled = (blocks / denom[:, :, None]).view(R, KB * 16)[:, :K]
    scaled = torch.where(sv.repeat_interleave(16, dim=1)[:, :K] > 0, scaled, torch.zeros_like(scaled))
    return e2m1_codes(scaled), s.view(torch.uint8)


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
    scale_a: Optional[torch.Tensor] = None   # [M][ceil(K/128)] fp32; MX / NV: tiled scale bytes
    scale_b: Optional[torch.Tensor] = None   # [ceil(N/128)][ceil(K/128)] fp32; MX / NV: tiled scale bytes
    tensor_scales: tuple = (1.0, 1.0)        # NV: one fp32 scale per tensor (A, B)
    scale_rows_a: Optional[torch.Tensor] = None   # MX / NV: the scale codes row-major [M][KB]
    scale_rows_b: Optional[torch.Tensor] = None   # MX / NV: [N][KB]


def make(wl: Workload | str, *, seed: Optional[int] = None, dist: Optional[str] = None,
         M: Optional[int] = None, N: Optional[int] = None, K: Optional[int] = None,
         batch: Optional[int] = None, dtype_in: Optional[str] = None,
         dtype_b: Optional[str] = None) -> Problem:
    """Draw the inputs of a workload (optionally at another size, seed, value mix or
    input type; dtype_b sets B's type separately for 8-bit pairings)."""
    if isinstance(wl, str):
        wl = WORKLOADS[wl]
    wl = Workload(wl.name, M or wl.M, N or wl.N, K or wl.K, batch or wl.batch, dtype_in or wl.dtype_in,
                  wl.dtype_out, dist or wl.dist, wl.seed if seed is None else seed, wl.block_scaled,
                  dict(wl.extra))
    wl.extra["dtype_b"] = dtype_b or wl.dtype_in
    if wl.extra.get("scale_mode") in ("mx", "nv"):
        return _make_hw_scaled(wl)
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


def _make_hw_scaled(wl: Workload) -> Problem:
    """MX / NVFP4 operands: element codes (E2M1 packed two per byte), tiled
    scale bytes, and the per-tensor scales of NVFP4."""
    mode = wl.extra["scale_mode"]
    if wl.batch != 1:
        raise ValueError("block-scaled workloads are single problems")
    if mode == "nv" and wl.dtype_in != "e2m1":
        raise ValueError("NVFP4 takes E2M1 elements")
    gen = torch.Generator().manual_seed(wl.seed)
    V = 32 if mode == "mx" else 16
    KB = (wl.K + V - 1) // V
    fmt_a, fmt_b = wl.dtype_in, wl.extra["dtype_b"]
    tensor_scales = (1.0, 1.0)

    def elements(R, fmt):
        if fmt == "e2m1":
            return torch.randint(0, 16, (R, wl.K), generator=gen).to(torch.uint8)
        return torch.randint(-3, 4, (R, wl.K), generator=gen).float().to(TORCH_DTYPES[fmt])

    if wl.dist == "ints":
        # exact variant: every product, scale and partial sum stays a small
        # dyadic number well inside fp32's 24 significant bits
        qa, qb = elements(wl.M, fmt_a), elements(wl.N, fmt_b)
        if mode == "mx":
            lo = 126 if fmt_a != "e2m1" else 127
            sa = torch.randint(lo, 129, (wl.M, KB), generator=gen).to(torch.uint8)
            sb = torch.randint(lo, 129, (wl.N, KB), generator=gen).to(torch.uint8)
        else:
            choice = torch.tensor([0x38, 0x40], dtype=torch.uint8)    # E4M3 1.0 and 2.0
            sa = choice[torch.randint(0, 2, (wl.M, KB), generator=gen)]
            sb = choice[torch.randint(0, 2, (wl.N, KB), generator=gen)]
            tensor_scales = (2.0, 0.5)
    else:
        xa = _draw((wl.M, wl.K), wl.dist, gen, wl.K)
        xb = _draw((wl.N, wl.K), wl.dist, gen, wl.K)
        if mode == "mx":
            qa, sa = _mx_quantize(xa, fmt_a)
            qb, sb = _mx_quantize(xb, fmt_b)
        else:
            ta = float(xa.abs().max()) / (448.0 * 6.0)
            tb = float(xb.abs().max()) / (448.0 * 6.0)
            tensor_scales = (ta, tb)
            qa, sa = _nv_quantize(xa, ta)
            qb, sb = _nv_quantize(xb, tb)
    if fmt_a == "e2m1":
        qa = pack_e2m1(qa)
    if fmt_b == "e2m1":
        qb = pack_e2m1(qb)
    # padding scale entries hold a random finite code: the product must not depend on them
    fill = int(torch.randint(100, 130, (1,), generator=gen))
    return Problem(wl, qa.contiguous(), qb.contiguous(), pack_scales_tiled(sa, fill), pack_scales_tiled(sb, fill),
                   tensor_scales, sa, sb)

