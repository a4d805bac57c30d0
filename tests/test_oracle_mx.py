"""Pins of the oracle's hardware block-scaled products (MXFP8, MXFP4, NVFP4).

"Hopper and Blackwell GEMM", concept "FP8 and FP4, with block scaling": every
row of A and of B is cut into blocks along K, and each block's values are
multiplied by that block's scale (MXFP8: 32 elements per E8M0 scale; MXFP4:
E2M1 elements, 32 per E8M0; NVFP4: E2M1, 16 per E4M3 scale plus one fp32
scale per tensor).  The oracle reads scales from the tiled layout (512-byte
tiles of 128 rows x 4 scales, lane = row mod 32, column = row / 32, "TMEM --
the accumulator's new home", section "Block-scaled MMA").

Each pin checks the oracle against something other than itself: torch's own
E8M0 decoder, the OCP value table of E2M1, numpy fp64 products of values
dequantised from the row-major scale arrays (which never go through the tiled
layout), exact block decompositions, and the locality of one scale.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from dense_gemm_blackwell_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_e8m0_decodes_every_code_like_torch():
    codes = np.arange(256, dtype=np.uint32)
    ours = oracle.decode("e8m0", codes)
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).double().numpy()
    assert np.isnan(ours[255]) and np.isnan(ref[255])
    assert np.array_equal(ours[:255], ref[:255])
    assert ours[127] == 1.0 and ours[0] == 2.0 ** -127 and ours[254] == 2.0 ** 127


def test_e2m1_decodes_the_ocp_table():
    table = json.load(open(os.path.join(GOLDEN, "e2m1_values.json")))["codes_0_to_15"]
    got = oracle.decode("e2m1", np.arange(16, dtype=np.uint32))
    assert np.array_equal(got, np.array(table)) and not np.isnan(got).any()
    assert np.array_equal(np.signbit(got), np.arange(16) >= 8)


def test_e2m1_values_are_exact_in_e4m3_and_round_trip():
    """Every E2M1 value is an E4M3 value (so the e4m3 decoder, pinned against
    torch, recovers it), and RNE encoding of each value gives back its code."""
    vals = oracle.decode("e2m1", np.arange(16, dtype=np.uint32))
    assert np.array_equal(oracle.decode("e4m3", oracle.encode("e4m3", vals)), vals)
    assert np.array_equal(oracle.encode("e2m1", vals[:8]), np.arange(8))
    # ties between neighbours go to the even code; beyond 6 saturates
    mids = [(0.25, 0.0), (0.75, 1.0), (1.25, 1.0), (1.75, 2.0), (2.5, 2.0), (3.5, 4.0), (5.0, 4.0), (9.0, 6.0)]
    for x, want in mids:
        assert oracle.round_to("e2m1", np.array([x]))[0] == want, x


def _dequant(codes, fmt):
    if fmt == "e2m1":
        return oracle.decode("e2m1", codes.numpy().astype(np.uint32))
    return codes.float().double().numpy()


def _unpack_e2m1(packed):
    b = packed.numpy()
    out = np.empty(b.shape[:-1] + (2 * b.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = b & 0xF
    out[..., 1::2] = b >> 4
    return torch.from_numpy(out)


def _numpy_reference(prob):
    """fp64 numpy product of dequantised values, scales from the row-major arrays."""
    wl = prob.wl
    mode = wl.extra["scale_mode"]
    V = 32 if mode == "mx" else 16
    fa, fb = wl.dtype_in, wl.extra["dtype_b"]
    qa = _unpack_e2m1(prob.A) if fa == "e2m1" else prob.A
    qb = _unpack_e2m1(prob.B) if fb == "e2m1" else prob.B
    if mode == "mx":
        sa = torch.pow(2.0, prob.scale_rows_a.double() - 127).numpy()
        sb = torch.pow(2.0, prob.scale_rows_b.double() - 127).numpy()
    else:
        sa = prob.scale_rows_a.view(torch.float8_e4m3fn).double().numpy() * prob.tensor_scales[0]
        sb = prob.scale_rows_b.view(torch.float8_e4m3fn).double().numpy() * prob.tensor_scales[1]
    a = _dequant(qa, fa) * np.repeat(sa, V, axis=1)[:, :wl.K]
    b = _dequant(qb, fb) * np.repeat(sb, V, axis=1)[:, :wl.K]
    return a @ b.T, np.abs(a) @ np.abs(b).T


def _oracle(prob, rows=None, **over):
    wl = prob.wl
    kw = dict(M=wl.M, N=wl.N, K=wl.K, dtype_a=wl.dtype_in, dtype_b=wl.extra["dtype_b"],
              scale_a=prob.scale_a, scale_b=prob.scale_b, scale_mode=wl.extra["scale_mode"],
              tensor_scales=prob.tensor_scales, rows=rows)
    kw.update(over)
    return oracle.gemm_rows(prob.A, prob.B, **kw)


CASES = [("mxfp8_8192", None), ("mxfp8_8192", "e5m2"), ("mxfp4_8192", None), ("nvfp4_8192", None)]


@pytest.mark.parametrize("name,dtype_b", CASES)
@pytest.mark.parametrize("dist", ["normal", "ints"])
def test_block_scaled_product_matches_numpy_dequantised(name, dtype_b, dist):
    """Ragged M, N and K (partial scale blocks and partial 128-row tiles)."""
    K = 200 if "fp8" in name else 208
    prob = inputs.make(name, M=150, N=131, K=K, dist=dist, seed=41, dtype_b=dtype_b)
    d, s = _oracle(prob)
    ref, sref = _numpy_reference(prob)
    scale = np.maximum(sref, 1e-300)
    assert np.max(np.abs(d[0] - ref) / scale) < 1e-13
    assert np.allclose(s[0], sref, rtol=1e-13, atol=0)
    if dist == "ints":
        assert np.array_equal(d[0], ref)    # small dyadic values: every sum is exact


@pytest.mark.parametrize("name", ["mxfp8_8192", "mxfp4_8192", "nvfp4_8192"])
def test_one_scale_changes_only_its_block(name):
    """Doubling the scale of block (m, kb) of A adds exactly that block's
    contribution to row m and leaves every other row unchanged."""
    prob = inputs.make(name, M=160, N=40, K=256, dist="ints", seed=42)
    wl = prob.wl
    mode = wl.extra["scale_mode"]
    V = 32 if mode == "mx" else 16
    d0, _ = _oracle(prob)
    m, kb = 137, 3
    rows = prob.scale_rows_a.clone()
    if mode == "mx":
        rows[m, kb] += 1                                   # E8M0: one more power of two
    else:
        rows[m, kb] = 0x40 if rows[m, kb] == 0x38 else 0x48   # E4M3 1.0 -> 2.0, 2.0 -> 4.0
    fill = int(prob.scale_a[-1])
    d1, _ = _oracle(prob, scale_a=inputs.pack_scales_tiled(rows, fill))
    changed = np.nonzero((d1[0] != d0[0]).any(axis=1))[0]
    assert set(changed.tolist()) <= {m}
    # the difference is the block product at the old scale (the new one is twice it)
    one_packed = inputs.pack_scales_tiled(prob.scale_rows_a, fill)
    qa = _unpack_e2m1(prob.A) if wl.dtype_in == "e2m1" else prob.A
    keep = torch.zeros(wl.K, dtype=torch.bool)
    keep[kb * V:(kb + 1) * V] = True
    if wl.dtype_in == "e2m1":
        qa = torch.where(keep, qa, torch.zeros_like(qa))
        A_block = inputs.pack_e2m1(qa)
    else:
        qa = torch.where(keep, qa.float(), torch.zeros(1)).to(prob.A.dtype)
        A_block = qa
    dblk, _ = oracle.gemm_rows(A_block, prob.B, M=wl.M, N=wl.N, K=wl.K, dtype_a=wl.dtype_in,
                               dtype_b=wl.extra["dtype_b"], scale_a=one_packed, scale_b=prob.scale_b,
                               scale_mode=mode, tensor_scales=prob.tensor_scales, rows=[m])
    assert np.array_equal(d1[0][m] - d0[0][m], dblk[0])


@pytest.mark.parametrize("name", ["mxfp8_8192", "mxfp4_8192", "nvfp4_8192"])
def test_product_is_the_sum_of_scaled_block_products(name):
    """D = sum over K blocks of (block product of the codes) * sA * sB, exactly."""
    prob = inputs.make(name, M=40, N=24, K=128, dist="ints", seed=43)
    wl = prob.wl
    mode = wl.extra["scale_mode"]
    V = 32 if mode == "mx" else 16
    d, _ = _oracle(prob)
    qa = _unpack_e2m1(prob.A) if wl.dtype_in == "e2m1" else prob.A
    qb = _unpack_e2m1(prob.B) if wl.extra["dtype_b"] == "e2m1" else prob.B
    a, b = _dequant(qa, wl.dtype_in), _dequant(qb, wl.extra["dtype_b"])
    if mode == "mx":
        sa, sb = 2.0 ** (prob.scale_rows_a.double().numpy() - 127), 2.0 ** (prob.scale_rows_b.double().numpy() - 127)
    else:
        sa = prob.scale_rows_a.view(torch.float8_e4m3fn).double().numpy()
        sb = prob.scale_rows_b.view(torch.float8_e4m3fn).double().numpy()
    total = np.zeros((wl.M, wl.N))
    for kb in range(wl.K // V):
        blk = a[:, kb * V:(kb + 1) * V] @ b[:, kb * V:(kb + 1) * V].T
        total += blk * sa[:, kb][:, None] * sb[:, kb][None, :]
    total *= prob.tensor_scales[0] * prob.tensor_scales[1]
    assert np.array_equal(d[0], total)


def test_batched_scales_follow_each_entry():
    """Two batch entries, packed one after the other (A: 2 row tiles of
    scales, B: 3): each entry's product equals the single-problem oracle,
    which the numpy pins above fix."""
    probs = [inputs.make("mxfp8_8192", M=150, N=300, K=96, dist="ints", seed=s) for s in (44, 45)]
    A = torch.stack([p.A for p in probs])
    B = torch.stack([p.B for p in probs])
    sa = torch.cat([p.scale_a for p in probs])
    sb = torch.cat([p.scale_b for p in probs])
    d, _ = oracle.gemm_rows(A, B, M=150, N=300, K=96, batch=2, dtype_a="e4m3", dtype_b="e4m3",
                            scale_a=sa, scale_b=sb, scale_mode="mx")
    for i, p in enumerate(probs):
        assert np.array_equal(d[i], _oracle(p)[0][0])
        assert np.array_equal(d[i], _numpy_reference(p)[0])


def test_tiled_layout_offsets():
    """The packer puts (r, kb) where the documented formula says, and the
    oracle reads every (r, kb) from there: a scale array whose entries are all
    distinct powers of two is recovered row by row through unit products."""
    R, KB = 300, 7
    codes = torch.arange(R * KB, dtype=torch.int64).reshape(R, KB) % 200 + 20
    packed = inputs.pack_scales_tiled(codes.to(torch.uint8), fill=0).numpy()
    KQ = (KB + 3) // 4
    for r in (0, 31, 32, 127, 128, 131, 299):
        for kb in range(KB):
            off = ((r // 128) * KQ + kb // 4) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + kb % 4
            assert packed[off] == codes[r, kb]
    # unit elements (e4m3 1.0), B a single row of ones with unit scales: D[m][0] = sum_kb 32 * 2^(e-127)
    K = KB * 32
    A = torch.ones(R, K).to(torch.float8_e4m3fn)
    B = torch.ones(1, K).to(torch.float8_e4m3fn)
    sb = inputs.pack_scales_tiled(torch.full((1, KB), 127, dtype=torch.uint8))
    d, _ = oracle.gemm_rows(A, B, M=R, N=1, K=K, dtype_a="e4m3", dtype_b="e4m3",
                            scale_a=torch.from_numpy(packed), scale_b=sb, scale_mode="mx")
    want = (32.0 * 2.0 ** (codes.double() - 127)).sum(dim=1).numpy()
    assert np.array_equal(d[0][:, 0], want)
