"""Planner gates of the hardware block-scaled path (host only, no GPU)."""
import pytest

import dense_gemm_blackwell_gb300 as dg

GB300 = dg.GemmDeviceProps(152, 232448, 10, 3)


@pytest.fixture(scope="module", autouse=True)
def built():
    dg.build()


def plan(M, N, K, a, b=None, mode=dg.GEMM_SCALE_MX_E8M0_32, **kw):
    d = dg.make_desc(M, N, K, dtype_a=a, dtype_b=b, dtype_d=dg.GEMM_BF16, scale_mode=mode, **kw)
    return dg.gemm_plan_query(d, GB300)


@pytest.mark.parametrize("a,b,mode,tile_k,stages", [
    (dg.GEMM_E4M3, dg.GEMM_E4M3, dg.GEMM_SCALE_MX_E8M0_32, 128, 5),
    (dg.GEMM_E5M2, dg.GEMM_E4M3, dg.GEMM_SCALE_MX_E8M0_32, 128, 5),
    (dg.GEMM_E2M1, dg.GEMM_E2M1, dg.GEMM_SCALE_MX_E8M0_32, 256, 5),
    (dg.GEMM_E2M1, dg.GEMM_E2M1, dg.GEMM_SCALE_NV_E4M3_16, 256, 5),
])
def test_square_8192_plans_pairs_of_256_wide_tiles(a, b, mode, tile_k, stages):
    st, info = plan(8192, 8192, 8192, a, b, mode)
    assert st == dg.GEMM_OK
    assert (info.kernel, info.cta_group, info.tile_m, info.tile_n, info.tile_k) == (dg.GEMM_KERNEL_MX, 2, 256, 256,
                                                                                   tile_k)
    assert info.stages == stages and info.tmem_stages == 1 and info.tmem_cols == 512
    assert info.smem_bytes <= GB300.smem_optin_bytes and info.block_threads == 384
    assert info.num_tiles == 32 * 32 and info.grid == 152


def test_tensor_memory_bounds_the_nvfp4_ring():
    """NVFP4 stages hold 4 scale slabs per row block (48 columns with B's two):
    at most 5 stages beside the 256-column accumulator."""
    st, info = plan(4096, 4096, 4096, dg.GEMM_E2M1, dg.GEMM_E2M1, dg.GEMM_SCALE_NV_E4M3_16, stages=6)
    assert st == dg.GEMM_ERR_UNSUPPORTED
    st, info = plan(4096, 4096, 4096, dg.GEMM_E2M1, dg.GEMM_E2M1, dg.GEMM_SCALE_NV_E4M3_16,
                    flags=dg.GEMM_FLAG_CTA_GROUP_1)
    assert st == dg.GEMM_OK and info.cta_group == 1 and info.stages == 3   # 32 KB of B per stage


@pytest.mark.parametrize("kw,want", [
    (dict(a=dg.GEMM_E2M1, b=dg.GEMM_E2M1, mode=dg.GEMM_SCALE_NONE), dg.GEMM_ERR_UNSUPPORTED),
    (dict(a=dg.GEMM_E4M3, b=dg.GEMM_E4M3, mode=dg.GEMM_SCALE_NV_E4M3_16), dg.GEMM_ERR_UNSUPPORTED),
    (dict(a=dg.GEMM_E4M3, b=dg.GEMM_E2M1, mode=dg.GEMM_SCALE_MX_E8M0_32), dg.GEMM_ERR_UNSUPPORTED),
    (dict(a=dg.GEMM_BF16, b=dg.GEMM_BF16, mode=dg.GEMM_SCALE_MX_E8M0_32), dg.GEMM_ERR_UNSUPPORTED),
    (dict(a=dg.GEMM_E2M1, b=dg.GEMM_E2M1, mode=dg.GEMM_SCALE_MX_E8M0_32, major_b=dg.GEMM_MN_MAJOR),
     dg.GEMM_ERR_UNSUPPORTED),
    (dict(a=dg.GEMM_E4M3, b=dg.GEMM_E4M3, mode=dg.GEMM_SCALE_MX_E8M0_32, tile_n=128), dg.GEMM_ERR_UNSUPPORTED),
    (dict(a=dg.GEMM_E4M3, b=dg.GEMM_E4M3, mode=dg.GEMM_SCALE_MX_E8M0_32, ld_sa=4), dg.GEMM_ERR_INVALID_ARG),
])
def test_unsupported_requests_fail_explicitly(kw, want):
    a, b, mode = kw.pop("a"), kw.pop("b"), kw.pop("mode")
    st, _ = plan(1024, 1024, 1024, a, b, mode, **kw)
    assert st == want


def test_odd_k_of_packed_fp4_is_refused():
    assert plan(256, 256, 255, dg.GEMM_E2M1, dg.GEMM_E2M1)[0] == dg.GEMM_ERR_UNSUPPORTED
    assert plan(256, 256, 0, dg.GEMM_E2M1, dg.GEMM_E2M1)[1].kernel == dg.GEMM_KERNEL_ZERO_FILL


def test_work_units_cover_every_tile_once():
    d = dg.make_desc(1000, 1300, 512, dtype_a=dg.GEMM_E4M3, dtype_d=dg.GEMM_BF16,
                     scale_mode=dg.GEMM_SCALE_MX_E8M0_32, max_ctas=12)
    st, info = dg.gemm_plan_query(d, GB300)
    assert st == dg.GEMM_OK and info.kernel == dg.GEMM_KERNEL_MX
    seen = []
    for c in range(info.grid // info.cta_group):
        i = 0
        while True:
            st, u = dg.gemm_plan_work_unit(d, info, c, i)
            assert st == dg.GEMM_OK
            if u.tile < 0:
                break
            assert (u.k_block_begin, u.k_block_end, u.role) == (0, 4, 0)
            seen.append(u.tile)
            i += 1
    assert sorted(seen) == list(range(info.num_tiles))


def test_mn_major_mxfp8_is_planned():
    """8-bit MX operands may be MN-major (packed E2M1 may not)."""
    for ma, mb in [(dg.GEMM_MN_MAJOR, dg.GEMM_K_MAJOR), (dg.GEMM_K_MAJOR, dg.GEMM_MN_MAJOR),
                   (dg.GEMM_MN_MAJOR, dg.GEMM_MN_MAJOR)]:
        st, info = plan(4096, 4096, 4096, dg.GEMM_E4M3, major_a=ma, major_b=mb)
        assert st == dg.GEMM_OK and info.kernel == dg.GEMM_KERNEL_MX

