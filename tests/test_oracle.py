"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test ties the oracle to something other than itself: the format
definitions (checked against torch's independent casts), exact integer
arithmetic, numpy/BLAS products, closed forms, identity and permutation
matrices, brute force with an exactly rounded sum (math.fsum) on tiny shapes,
the worked examples of the pages, and invariants of block scaling.  A dropped
term, a wrong sign or index, or a transposed operand fails at least one.
"""
import math

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def codes16(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def codes8(t):
    return t.contiguous().view(torch.uint8).numpy()


# ---------------------------------------------------------------- codecs

@pytest.mark.parametrize("name,tdt", [("f16", torch.float16), ("bf16", torch.bfloat16)])
def test_decode_every_16bit_code_matches_torch(name, tdt):
    codes = np.arange(65536, dtype=np.uint32)
    mine = oracle.decode(name, codes)
    ref = torch.from_numpy(codes.astype(np.uint16).view(np.int16)).view(tdt).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], ref[~nan])
    # signed zeros keep their sign
    assert np.array_equal(np.signbit(mine[~nan]), np.signbit(ref[~nan]))


def test_decode_every_e4m3_code_matches_torch_and_ocp():
    codes = np.arange(256, dtype=np.uint32)
    mine = oracle.decode("e4m3", codes)
    ref = torch.from_numpy(codes.astype(np.uint8)).view(torch.float8_e4m3fn).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], ref[~nan])
    # OCP E4M3: only S.1111.111 is NaN, no infinities, largest finite 448, smallest subnormal 2^-9
    assert nan.sum() == 2 and np.isnan(mine[0x7F]) and np.isnan(mine[0xFF])
    assert mine[0x7E] == 448.0 and mine[0xFE] == -448.0
    assert mine[0x01] == 2.0 ** -9
    assert np.nanmax(np.abs(mine)) == 448.0


def _tie_values(name, n, seed):
    """Values exactly halfway between adjacent representable numbers (fp32-exact)."""
    rng = np.random.default_rng(seed)
    if name == "bf16":
        c = rng.integers(0, 0x7F00, n).astype(np.uint32)
        lo = oracle.decode("bf16", c)
        hi = oracle.decode("bf16", c + 1)
    else:
        c = rng.integers(0, 0x7BFF, n).astype(np.uint32)
        lo = oracle.decode("f16", c)
        hi = oracle.decode("f16", c + 1)
    mid = (lo + hi) / 2
    sign = np.where(rng.random(n) < 0.5, -1.0, 1.0)
    return (mid * sign).astype(np.float32)


@pytest.mark.parametrize("name,tdt", [("f16", torch.float16), ("bf16", torch.bfloat16)])
def test_round_to_16bit_matches_torch_rne(name, tdt):
    rng = np.random.default_rng(11)
    vals = np.concatenate([
        (rng.standard_normal(20000) * 10.0 ** rng.integers(-8, 6, 20000)).astype(np.float32),
        _tie_values(name, 20000, 12),
        np.array([0.0, -0.0, 65504.0, 65519.0, 65520.0, 1e-8, -1e-8, 6.0e-8, 3.0e38, -3.0e38],
                 dtype=np.float32),
    ])
    mine = oracle.round_to(name, vals.astype(np.float64))
    ref = torch.from_numpy(vals).to(tdt).double().numpy()
    assert np.array_equal(mine, ref)
    enc = oracle.encode(name, vals.astype(np.float64))
    assert np.array_equal(enc.astype(np.uint16), codes16(torch.from_numpy(vals).to(tdt)))


def test_round_to_f32_matches_numpy_cast():
    rng = np.random.default_rng(13)
    x = rng.standard_normal(50000) * 10.0 ** rng.integers(-40, 38, 50000)
    # exact fp32 ties: an fp32 value plus half its spacing
    f = rng.standard_normal(5000).astype(np.float32)
    ties = f.astype(np.float64) + np.spacing(np.abs(f)).astype(np.float64) / 2
    x = np.concatenate([x, ties])
    assert np.array_equal(oracle.round_to("f32", x), x.astype(np.float32).astype(np.float64))


def test_e4m3_encode_rne_and_saturation():
    rng = np.random.default_rng(14)
    x = (rng.standard_normal(20000) * 10.0 ** rng.integers(-3, 3, 20000)).astype(np.float32)
    x = np.clip(x, -448.0, 448.0)
    ref = codes8(torch.from_numpy(x).to(torch.float8_e4m3fn))
    mine = oracle.encode("e4m3", x.astype(np.float64)).astype(np.uint8)
    # +-0 both encode to a zero code; compare magnitudes of zeros loosely
    nz = x != 0
    assert np.array_equal(mine[nz], ref[nz])
    # saturating: beyond the largest finite value stays at +-448
    assert oracle.encode("e4m3", [449.0, 1e6, -1e6, np.inf])[:4].tolist() == [0x7E, 0x7E, 0xFE, 0x7E]


@pytest.mark.parametrize("name,bits", [("f16", 16), ("bf16", 16), ("e4m3", 8)])
def test_encode_inverts_decode(name, bits):
    codes = np.arange(1 << bits, dtype=np.uint32)
    vals = oracle.decode(name, codes)
    ok = ~np.isnan(vals)
    assert np.array_equal(oracle.encode(name, vals[ok]), codes[ok])


# ---------------------------------------------------------------- GEMM pins

def run(A, B, dtype, **kw):
    M, K = A.shape[-2], A.shape[-1]
    N = B.shape[-2]
    batch = A.shape[0] if A.dim() == 3 else 1
    return oracle.gemm(A, B, M=M, N=N, K=K, batch=batch, dtype_a=dtype, dtype_b=dtype, **kw)


def test_single_cta_example_integers_exact():
    """TVM TIRx "Blackwell Tensor Cores": Out = A @ B.T, A 128x64, B 64x64 fp16.
    Integer entries make every sum exact, so the oracle must equal int64 numpy."""
    g = torch.Generator().manual_seed(2)
    a = torch.randint(-3, 4, (128, 64), generator=g)
    b = torch.randint(-3, 4, (64, 64), generator=g)
    d, s = run(a.half(), b.half(), "f16")
    ref = a.numpy().astype(np.int64) @ b.numpy().astype(np.int64).T
    assert np.array_equal(d[0], ref.astype(np.float64))
    assert np.array_equal(s[0], np.abs(a.numpy()).astype(np.int64) @ np.abs(b.numpy()).astype(np.int64).T)


def test_single_cta_example_float_matches_page_check():
    """The page's own check: assert_close(out, a.float() @ b.float().T, rtol=atol=2e-4),
    applied to the oracle (rounded to the fp32 output), plus numpy fp64 to 1e-12."""
    g = torch.Generator().manual_seed(1)
    a = (torch.rand(128, 64, generator=g) * 2 - 1).half()
    b = (torch.rand(64, 64, generator=g) * 2 - 1).half()
    d, s = run(a, b, "f16")
    out = torch.from_numpy(oracle.round_to("f32", d[0]).astype(np.float32))
    torch.testing.assert_close(out, a.float() @ b.float().T, rtol=2e-4, atol=2e-4)
    ref64 = a.double().numpy() @ b.double().numpy().T
    assert np.max(np.abs(d[0] - ref64) / s[0]) < 1e-12


def test_mma_m16n8k16_fragment_example():
    """TVM TIRx "mma.sync", example "a 16x8 result with two K16 issues".

    Inputs regenerated with the page's recipe (default_rng(0), quarter integers).
    Products of quarter integers summed over 32 terms are exact in fp32, so the
    oracle must equal numpy fp32 a @ b.T bit for bit.  A CPU model of the warp
    instruction -- words packed as on the page, gathered into lanes with the
    page's ownership formulas, two K16 issues, D scattered by its formula --
    must give the same 16x8 result, and each map must own every element once.
    """
    rng = np.random.default_rng(0)
    a = (rng.integers(-4, 5, (16, 32)) / 4).astype("float16")
    b = (rng.integers(-4, 5, (8, 32)) / 4).astype("float16")
    d, _ = run(torch.from_numpy(a), torch.from_numpy(b), "f16")
    ref32 = a.astype("float32") @ b.astype("float32").T
    assert np.array_equal(d[0].astype(np.float32), ref32)
    assert np.array_equal(d[0], ref32.astype(np.float64))

    ap = np.ascontiguousarray(a.reshape(1, 16, 2, 16).transpose(0, 2, 1, 3)).view("uint32")
    bp = np.ascontiguousarray(b.reshape(1, 8, 2, 16).transpose(0, 2, 1, 3)).view("uint32")
    assert ap.shape == (1, 2, 16, 8) and bp.shape == (1, 2, 8, 8)

    def unpack(word):
        h = np.array([word], dtype=np.uint32).view(np.float16)
        return float(h[0]), float(h[1])

    dregs = np.zeros((32, 4), dtype=np.float32)
    for kk in range(2):
        a_tile = np.full((16, 16), np.nan)
        b_tile = np.full((8, 16), np.nan)
        owned_a = np.zeros((16, 8), int)
        owned_b = np.zeros((8, 8), int)
        for lane in range(32):
            for r in range(4):
                row, wc = lane // 4 + 8 * (r % 2), lane % 4 + 4 * (r // 2)
                owned_a[row, wc] += 1
                a_tile[row, 2 * wc], a_tile[row, 2 * wc + 1] = unpack(ap[0, kk, row, wc])
            for r in range(2):
                row, wc = lane // 4, lane % 4 + 4 * r
                owned_b[row, wc] += 1
                b_tile[row, 2 * wc], b_tile[row, 2 * wc + 1] = unpack(bp[0, kk, row, wc])
        assert (owned_a == 1).all() and (owned_b == 1).all()
        # one m16n8k16 issue: D = A . B^T + C, C = previous D (0 on the first issue)
        prod = (a_tile.astype(np.float32) @ b_tile.astype(np.float32).T).astype(np.float32)
        owned_d = np.zeros((16, 8), int)
        for lane in range(32):
            for r in range(4):
                i, j = lane // 4 + 8 * (r // 2), 2 * (lane % 4) + r % 2
                owned_d[i, j] += 1
                dregs[lane, r] = dregs[lane, r] + prod[i, j]
        assert (owned_d == 1).all()
    out = np.zeros((16, 8), dtype=np.float32)
    for lane in range(32):
        for r in range(4):
            out[lane // 4 + 8 * (r // 2), 2 * (lane % 4) + r % 2] = dregs[lane, r]
    assert np.array_equal(out, d[0].astype(np.float32))


@pytest.mark.parametrize("dtype,tdt", [("bf16", torch.bfloat16), ("f16", torch.float16), ("e4m3", torch.float8_e4m3fn)])
def test_identity_and_permutation(dtype, tdt):
    g = torch.Generator().manual_seed(7)
    M, K = 37, 48
    a = (torch.randint(-8, 9, (M, K), generator=g) / 4).to(tdt)
    eye = torch.eye(K).to(tdt)
    d, _ = run(a, eye, dtype)                      # B = I  ->  D = A
    assert np.array_equal(d[0], a.double().numpy())
    perm = torch.randperm(K, generator=g)
    P = torch.eye(K)[perm].to(tdt)                  # B = P  ->  D[:, n] = A[:, perm[n]]
    d, _ = run(a, P, dtype)
    assert np.array_equal(d[0], a.double().numpy()[:, perm.numpy()])
    Nb = 29
    bm = (torch.randint(-8, 9, (Nb, K), generator=g) / 4).to(tdt)
    d, _ = run(torch.eye(K).to(tdt), bm, dtype)    # A = I  ->  D = B^T
    assert np.array_equal(d[0], bm.double().numpy().T)


def test_closed_forms():
    K = 1000
    ones_a = torch.ones(5, K, dtype=torch.float16)
    ramp = torch.arange(1, 8, dtype=torch.float32)[:, None].expand(7, K).half()
    d, s = run(ones_a, ramp, "f16")                # D[m,n] = K (n+1)
    assert np.array_equal(d[0], np.tile(K * np.arange(1, 8, dtype=np.float64), (5, 1)))
    k = torch.arange(K, dtype=torch.float32) % 64   # D = sum_k (k mod 64)^2, exact in fp16 inputs
    v = k.half()[None, :]
    d, s = run(v, v, "f16")
    assert d[0, 0, 0] == float((k.double() ** 2).sum())
    neg = -v
    d, s = run(v, neg, "f16")                        # sign: D = -S
    assert d[0, 0, 0] == -s[0, 0, 0]


def _fsum_reference(a64, b64):
    """Exactly rounded D and S by math.fsum over exact fp64 products."""
    M, K = a64.shape
    N = b64.shape[0]
    d = np.empty((M, N))
    s = np.empty((M, N))
    for m in range(M):
        for n in range(N):
            p = a64[m] * b64[n]
            d[m, n] = math.fsum(p)
            s[m, n] = math.fsum(np.abs(p))
    return d, s


@pytest.mark.parametrize("dtype,tdt", [("bf16", torch.bfloat16), ("f16", torch.float16), ("e4m3", torch.float8_e4m3fn)])
def test_brute_force_tiny_shapes(dtype, tdt):
    """All M, N, K in a set spanning 1..17, against fsum of exact products, within
    the fp64 ascending-sum bound (K-1) 2^-53 S (+ half an ulp for fsum's rounding)."""
    g = torch.Generator().manual_seed(21)
    sizes = [1, 2, 3, 5, 8, 13, 16, 17]
    for M in sizes:
        for N in sizes:
            for K in sizes:
                a = (torch.rand(M, K, generator=g) * 4 - 2).to(tdt)
                b = (torch.rand(N, K, generator=g) * 4 - 2).to(tdt)
                d, s = run(a, b, dtype)
                rd, rs = _fsum_reference(a.double().numpy(), b.double().numpy())
                bound = (K - 1) * 2.0 ** -53 * rs + np.spacing(np.abs(rd))
                assert (np.abs(d[0] - rd) <= bound).all(), (M, N, K)
                assert np.allclose(s[0], rs, rtol=K * 2.0 ** -52, atol=0)


def test_layouts_strides_batches_and_majorness():
    """Padded leading dims, batch strides and MN-major operands address the same
    logical matrices: results equal the packed K-major case bit for bit, and the
    fsum brute force within the fp64 bound.  Non-square shapes catch a transpose."""
    g = torch.Generator().manual_seed(31)
    batch, M, N, K = 3, 11, 7, 19
    a = (torch.rand(batch, M, K, generator=g) * 2 - 1).bfloat16()
    b = (torch.rand(batch, N, K, generator=g) * 2 - 1).bfloat16()
    d0, s0 = run(a, b, "bf16")
    for m_ in range(batch):
        rd, _ = _fsum_reference(a[m_].double().numpy(), b[m_].double().numpy())
        assert (np.abs(d0[m_] - rd) <= (K - 1) * 2.0 ** -53 * s0[m_] + np.spacing(np.abs(rd))).all()
    # padded rows and padded batch stride
    lda, ldb, sa, sb = K + 5, K + 3, (M + 2) * (K + 5), (N + 1) * (K + 3)
    abuf = torch.zeros(batch * sa, dtype=torch.bfloat16)
    bbuf = torch.zeros(batch * sb, dtype=torch.bfloat16)
    for i in range(batch):
        abuf[i * sa:i * sa + M * lda].view(M, lda)[:, :K] = a[i]
        bbuf[i * sb:i * sb + N * ldb].view(N, ldb)[:, :K] = b[i]
    d1, _ = oracle.gemm(abuf, bbuf, M=M, N=N, K=K, batch=batch, dtype_a="bf16", dtype_b="bf16",
                        lda=lda, ldb=ldb, stride_a=sa, stride_b=sb)
    assert np.array_equal(d0, d1)
    # MN-major: A stored as [K][M], B as [K][N]
    at = a.transpose(1, 2).contiguous()
    bt = b.transpose(1, 2).contiguous()
    d2, _ = oracle.gemm(at, bt, M=M, N=N, K=K, batch=batch, dtype_a="bf16", dtype_b="bf16",
                        major_a="mn", major_b="mn")
    assert np.array_equal(d0, d2)
    # selected rows equal the corresponding rows of the full product
    rows = [0, M + 3, 2 * M + M - 1]
    dr, _ = oracle.gemm_rows(a, b, M=M, N=N, K=K, batch=batch, dtype_a="bf16", dtype_b="bf16", rows=rows)
    assert np.array_equal(dr, d0.reshape(batch * M, N)[rows])


def test_block_scaling_decomposes_into_scaled_block_products():
    """Block scaling ("Hopper and Blackwell GEMM", FP8 and FP4 with block scaling):
    each 128-deep block of the product is the unscaled block product times
    sA[m][kb] * sB[n/128][kb].  Checked against the unscaled oracle (pinned
    above) on K-slices, exactly (integer codes, power-of-two scales), with
    N and K spanning several 128-blocks and a ragged tail."""
    g = torch.Generator().manual_seed(41)
    M, N, K = 5, 300, 290
    kb = (K + 127) // 128
    qa = torch.randint(-3, 4, (M, K), generator=g).float().to(torch.float8_e4m3fn)
    qb = torch.randint(-3, 4, (N, K), generator=g).float().to(torch.float8_e4m3fn)
    sa = torch.pow(2.0, torch.randint(-4, 5, (M, kb), generator=g).float())
    sb = torch.pow(2.0, torch.randint(-4, 5, ((N + 127) // 128, kb), generator=g).float())
    d, s = oracle.gemm(qa, qb, M=M, N=N, K=K, dtype_a="e4m3", dtype_b="e4m3",
                       scale_a=sa.numpy(), scale_b=sb.numpy())
    expect = np.zeros((M, N))
    for j in range(kb):
        k0, k1 = 128 * j, min(K, 128 * j + 128)
        part, _ = oracle.gemm(qa[:, k0:k1].contiguous(), qb[:, k0:k1].contiguous(), M=M, N=N,
                              K=k1 - k0, dtype_a="e4m3", dtype_b="e4m3")
        col_scale = sb[np.arange(N) // 128, j].double().numpy()
        expect += part[0] * sa[:, j].double().numpy()[:, None] * col_scale[None, :]
    assert np.array_equal(d[0], expect)
    # unit scales reduce to the unscaled product
    d1, _ = oracle.gemm(qa, qb, M=M, N=N, K=K, dtype_a="e4m3", dtype_b="e4m3",
                        scale_a=np.ones((M, kb), np.float32), scale_b=np.ones(((N + 127) // 128, kb), np.float32))
    d0, _ = oracle.gemm(qa, qb, M=M, N=N, K=K, dtype_a="e4m3", dtype_b="e4m3")
    assert np.array_equal(d1, d0)
    # locality: doubling one scale of A touches one row; one scale of B one 128-column block
    sa2 = sa.clone(); sa2[3, 1] *= 2
    d2, _ = oracle.gemm(qa, qb, M=M, N=N, K=K, dtype_a="e4m3", dtype_b="e4m3", scale_a=sa2.numpy(), scale_b=sb.numpy())
    changed_rows = np.where((d2[0] != d[0]).any(axis=1))[0]
    assert set(changed_rows.tolist()) <= {3}
    sb2 = sb.clone(); sb2[2, 0] *= 2
    d3, _ = oracle.gemm(qa, qb, M=M, N=N, K=K, dtype_a="e4m3", dtype_b="e4m3", scale_a=sa.numpy(), scale_b=sb2.numpy())
    changed_cols = np.where((d3[0] != d[0]).any(axis=0))[0]
    assert changed_cols.size > 0 and changed_cols.min() >= 256 and changed_cols.max() < 300


def test_zero_sized_and_k_zero():
    a = torch.zeros(0, 8, dtype=torch.float16)
    b = torch.zeros(4, 8, dtype=torch.float16)
    d, s = run(a, b, "f16")
    assert d.shape == (1, 0, 4)
    d, s = oracle.gemm(torch.zeros(3, 0, dtype=torch.float16), torch.zeros(4, 0, dtype=torch.float16),
                       M=3, N=4, K=0, dtype_a="f16", dtype_b="f16")
    assert (d == 0).all() and (s == 0).all()


def test_decode_every_e5m2_code_matches_torch_and_ocp():
    codes = np.arange(256, dtype=np.uint32)
    mine = oracle.decode("e5m2", codes)
    ref = torch.from_numpy(codes.astype(np.uint8)).view(torch.float8_e5m2).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], ref[~nan])
    # OCP E5M2: IEEE-style infinities, largest finite 57344, smallest subnormal 2^-16
    assert mine[0x7C] == np.inf and mine[0xFC] == -np.inf
    assert mine[0x7B] == 57344.0 and mine[0x01] == 2.0 ** -16
    assert oracle.encode("e5m2", [57344.0, 1.5])[:2].tolist() == [0x7B, 0x3E]


def test_fp32_inputs_decode_exactly():
    """32-bit input codes (tf32 products are checked against the exact fp32 values)."""
    g = torch.Generator().manual_seed(61)
    a = torch.randn(9, 40, generator=g)
    b = torch.randn(7, 40, generator=g)
    d, s = oracle.gemm(a.numpy(), b.numpy(), M=9, N=7, K=40, dtype_a="f32", dtype_b="f32")
    rd, rs = _fsum_reference(a.double().numpy(), b.double().numpy())
    assert (np.abs(d[0] - rd) <= 39 * 2.0 ** -53 * rs + np.spacing(np.abs(rd))).all()


def test_mixed_fp8_formats():
    g = torch.Generator().manual_seed(62)
    qa = torch.randint(-3, 4, (6, 130), generator=g).float()
    qb = torch.randint(-3, 4, (5, 130), generator=g).float()
    d, _ = oracle.gemm(qa.to(torch.float8_e4m3fn), qb.to(torch.float8_e5m2), M=6, N=5, K=130,
                       dtype_a="e4m3", dtype_b="e5m2")
    assert np.array_equal(d[0], qa.double().numpy() @ qb.double().numpy().T)
