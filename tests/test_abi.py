"""Host-side tests of the C ABI (no GPU): the library loads and exports every
function include/gemm.h declares, and the planner's decisions match the
numbers the pages print and the documented error behaviour."""
import ctypes
import json
import os

import pytest

import dense_gemm_blackwell_gb300 as dg

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_numbers.json")))

B200 = dg.GemmDeviceProps(sm_count=148, smem_optin_bytes=232448, cc_major=10, cc_minor=0)
GB300 = dg.GemmDeviceProps(sm_count=152, smem_optin_bytes=232448, cc_major=10, cc_minor=3)


@pytest.fixture(scope="module", autouse=True)
def built():
    dg.build()


def test_library_exports_every_declared_function():
    names = dg.header_functions()
    assert {"gemm_plan_create", "gemm_run", "gemm_plan_destroy", "gemm_sync_status",
            "gemm_status_string", "gemm_plan_query", "gemm_run_host"} <= set(names)
    raw = ctypes.CDLL(dg._LIB_PATH)
    for n in names:
        assert hasattr(raw, n), n


def test_status_strings_and_version():
    for code, name in [(0, "GEMM_OK"), (1, "GEMM_ERR_INVALID_ARG"), (2, "GEMM_ERR_UNSUPPORTED"),
                       (3, "GEMM_ERR_ALIGNMENT"), (4, "GEMM_ERR_CUDA"), (5, "GEMM_ERR_TIMEOUT"),
                       (6, "GEMM_ERR_NO_DEVICE"), (7, "GEMM_ERR_RESOURCES")]:
        assert dg.gemm_status_string(code) == name
    assert dg.gemm_status_string(99) == "GEMM_ERR_UNKNOWN"
    assert dg.gemm_version() >= 10000


def query(props=GB300, **kw):
    M, N, K = kw.pop("M"), kw.pop("N"), kw.pop("K")
    s, info = dg.gemm_plan_query(dg.make_desc(M, N, K, **kw), props)
    return s, info


def test_pipeline_budget_matches_cublasdx_card():
    """128x256x64 bf16 at depth 4 with two TMEM stages: 48 KiB per stage and
    196,708 B of stages + barriers + TMEM handle."""
    s, info = query(props=B200, M=4096, N=4096, K=4096, dtype_a=dg.GEMM_BF16, dtype_d=dg.GEMM_BF16,
                    flags=dg.GEMM_FLAG_CTA_GROUP_1, tile_n=256, stages=4)
    assert s == dg.GEMM_OK
    assert info.stage_bytes == GOLDEN["stage_bytes_128x256x64_bf16"]["value"]
    assert info.pipeline_bytes == GOLDEN["pipeline_bytes_depth4_128x256x64_bf16"]["value"]
    assert info.tmem_stages == GOLDEN["tmem_stages_128x256_f32"]["value"]
    assert info.tmem_cols == GOLDEN["tmem_total_columns"]["value"]
    assert info.smem_bytes <= GOLDEN["smem_optin_bytes_b200"]["value"]


def test_four_stages_fit_for_128x256_bf16():
    s, info = query(props=B200, M=4096, N=4096, K=4096, dtype_a=dg.GEMM_BF16, dtype_d=dg.GEMM_BF16,
                    flags=dg.GEMM_FLAG_CTA_GROUP_1, tile_n=256)
    assert s == dg.GEMM_OK
    assert info.stages == GOLDEN["stages_fit_128x256x64_bf16_228KB"]["value"]
    # one more stage does not fit the opt-in limit
    s, _ = query(props=B200, M=4096, N=4096, K=4096, dtype_a=dg.GEMM_BF16, dtype_d=dg.GEMM_BF16,
                 flags=dg.GEMM_FLAG_CTA_GROUP_1, tile_n=256, stages=5)
    assert s == dg.GEMM_ERR_RESOURCES


def test_single_cta_example_plan():
    """The single-CTA walk-through: 128x64 . (64x64)^T fp16 -> fp32, 64 TMEM columns."""
    s, info = query(M=128, N=64, K=64, dtype_a=dg.GEMM_F16, dtype_d=dg.GEMM_F32)
    assert s == dg.GEMM_OK
    assert info.kernel == dg.GEMM_KERNEL_SINGLE_CTA
    assert info.tmem_cols == GOLDEN["tmem_columns_128x64_f32"]["value"]
    assert info.block_threads == 128 and info.grid == 1


def test_headline_plan_is_pair_tiles():
    s, info = query(M=8192, N=8192, K=8192, dtype_a=dg.GEMM_BF16, dtype_d=dg.GEMM_F32)
    assert s == dg.GEMM_OK
    assert info.kernel == dg.GEMM_KERNEL_PERSISTENT
    # 512-wide pair tiles (two N = 256 MMAs per K step, one 512-column
    # accumulator), four ring stages of one 128-byte K atom (64 bf16)
    assert (info.cta_group, info.tile_m, info.tile_n, info.tile_k) == (2, 256, 512, 64)
    assert info.stages == 4 and info.stage_bytes == 128 * 128 + 256 * 128
    assert info.tmem_stages == 1 and info.tmem_cols == 512
    assert info.num_tiles == 32 * 16
    assert info.stream_k_tiles == 0      # 512 tiles over 76 pairs: the last wave is 74 % full
    assert info.grid == 152 and info.grid % 2 == 0
    assert info.tmem_cols <= 512 and info.tmem_stages * info.tile_n <= 512
    assert info.smem_bytes <= GB300.smem_optin_bytes


def test_stage_depth_flags():
    base = dict(M=8192, N=8192, K=8192, dtype_a=dg.GEMM_BF16, dtype_d=dg.GEMM_F32, tile_n=256)
    s, info = query(**base)
    assert s == dg.GEMM_OK and info.tile_k == 128 and info.stages == 3
    s, info = query(flags=dg.GEMM_FLAG_STAGE_K1, **base)
    assert s == dg.GEMM_OK and info.tile_k == 64 and info.stages == 6
    s, info = query(flags=dg.GEMM_FLAG_STAGE_K1 | dg.GEMM_FLAG_STAGE_K2, **base)
    assert s == dg.GEMM_ERR_INVALID_ARG
    # MN-major operands keep one atom per stage; asking for two is refused
    s, info = query(major_a=dg.GEMM_MN_MAJOR, **base)
    assert s == dg.GEMM_OK and info.tile_k == 64
    s, info = query(major_a=dg.GEMM_MN_MAJOR, flags=dg.GEMM_FLAG_STAGE_K2, **base)
    assert s == dg.GEMM_ERR_UNSUPPORTED
    # K within one atom: one atom per stage
    s, info = query(M=1024, N=1024, K=64, dtype_a=dg.GEMM_BF16, dtype_d=dg.GEMM_F32, flags=dg.GEMM_FLAG_NO_SINGLE_CTA)
    assert s == dg.GEMM_OK and info.tile_k == 64
    # tf32: 32 elements per atom
    s, info = query(M=4096, N=4096, K=4096, dtype_a=dg.GEMM_TF32, dtype_d=dg.GEMM_F32, tile_n=256)
    assert s == dg.GEMM_OK and info.tile_k == 64
    # 512-wide tiles keep one atom per stage; two are refused
    s, info = query(M=4096, N=4096, K=4096, dtype_a=dg.GEMM_BF16, dtype_d=dg.GEMM_F32, tile_n=512,
                    flags=dg.GEMM_FLAG_STAGE_K2)
    assert s == dg.GEMM_ERR_UNSUPPORTED


def test_batched_plan():
    s, info = query(M=256, N=256, K=256, batch=512, dtype_a=dg.GEMM_F16, dtype_d=dg.GEMM_F16)
    assert s == dg.GEMM_OK and info.kernel == dg.GEMM_KERNEL_PERSISTENT
    assert info.cta_group == 1 and info.tile_n == 256   # short K: single-SM tiles
    assert info.num_tiles == 512 * (256 // info.tile_m) * (256 // info.tile_n)


@pytest.mark.parametrize("kw,status", [
    (dict(M=-1, N=8, K=8), dg.GEMM_ERR_INVALID_ARG),
    (dict(M=8, N=8, K=8, dtype_a=7), dg.GEMM_ERR_INVALID_ARG),
    (dict(M=8, N=8, K=8, lda=4), dg.GEMM_ERR_INVALID_ARG),
    (dict(M=8, N=8, K=8, ldd=4), dg.GEMM_ERR_INVALID_ARG),
    (dict(M=8, N=8, K=8, dtype_a=dg.GEMM_F16, dtype_b=dg.GEMM_BF16), dg.GEMM_ERR_UNSUPPORTED),
    (dict(M=8, N=8, K=8, dtype_d=dg.GEMM_E4M3), dg.GEMM_ERR_UNSUPPORTED),
    (dict(M=8, N=8, K=8, scale_mode=dg.GEMM_SCALE_BLOCK_1x128_128x128), dg.GEMM_ERR_UNSUPPORTED),
    (dict(M=1024, N=1024, K=1024, tile_n=200), dg.GEMM_ERR_UNSUPPORTED),
    (dict(M=1024, N=1024, K=1024, tile_n=272), dg.GEMM_ERR_UNSUPPORTED),
    (dict(M=1024, N=1024, K=1024, stages=1), dg.GEMM_ERR_UNSUPPORTED),
    (dict(M=1024, N=1024, K=1024, stages=12, flags=dg.GEMM_FLAG_CTA_GROUP_1, tile_n=256), dg.GEMM_ERR_RESOURCES),
    (dict(M=1024, N=1024, K=1024, flags=dg.GEMM_FLAG_CTA_GROUP_1 | dg.GEMM_FLAG_CTA_GROUP_2), dg.GEMM_ERR_INVALID_ARG),
    (dict(M=4096, N=4096, K=4096, flags=dg.GEMM_FLAG_SINGLE_CTA), dg.GEMM_ERR_UNSUPPORTED),
])
def test_planner_rejects(kw, status):
    s, _ = query(**kw)
    assert s == status


def test_degenerate_sizes_plan():
    s, info = query(M=64, N=64, K=0)
    assert s == dg.GEMM_OK and info.kernel == dg.GEMM_KERNEL_ZERO_FILL
    s, info = query(M=0, N=64, K=64)
    assert s == dg.GEMM_OK and info.kernel == 0


def test_mn_major_plans():
    s, info = query(M=100, N=72, K=40, major_a=dg.GEMM_MN_MAJOR, major_b=dg.GEMM_MN_MAJOR)
    assert s == dg.GEMM_OK and info.kernel == dg.GEMM_KERNEL_SINGLE_CTA
    s, info = query(M=1000, N=72, K=40, major_b=dg.GEMM_MN_MAJOR)
    assert s == dg.GEMM_OK and info.kernel == dg.GEMM_KERNEL_PERSISTENT
    s, info = query(M=8192, N=8192, K=8192, major_a=dg.GEMM_MN_MAJOR, major_b=dg.GEMM_MN_MAJOR)
    assert s == dg.GEMM_OK and info.cta_group == 2
    # MN-major B is loaded in 64-column boxes: a pair's half tile must be a multiple of 64
    s, _ = query(M=8192, N=8192, K=8192, major_b=dg.GEMM_MN_MAJOR, flags=dg.GEMM_FLAG_CTA_GROUP_2, tile_n=192)
    assert s == dg.GEMM_ERR_UNSUPPORTED
    # tf32 needs K-major operands
    s, _ = query(M=4096, N=4096, K=4096, dtype_a=dg.GEMM_TF32, major_a=dg.GEMM_MN_MAJOR)
    assert s == dg.GEMM_ERR_UNSUPPORTED
    # block-scaled fp8: MN-major operands in 128-element boxes; a CTA's B rows
    # must be a whole number of boxes (a 128-wide pair tile gives each CTA 64)
    fp8 = dict(M=4096, N=4096, K=4096, dtype_a=dg.GEMM_E4M3, scale_mode=dg.GEMM_SCALE_BLOCK_1x128_128x128)
    for kw in (dict(major_a=dg.GEMM_MN_MAJOR), dict(major_b=dg.GEMM_MN_MAJOR),
               dict(major_a=dg.GEMM_MN_MAJOR, major_b=dg.GEMM_MN_MAJOR, flags=dg.GEMM_FLAG_CTA_GROUP_2, tile_n=256)):
        s, info = query(**fp8, **kw)
        assert s == dg.GEMM_OK and info.kernel == dg.GEMM_KERNEL_FP8_BLOCK, kw
    s, _ = query(**fp8, major_b=dg.GEMM_MN_MAJOR, flags=dg.GEMM_FLAG_CTA_GROUP_2, tile_n=128)
    assert s == dg.GEMM_ERR_UNSUPPORTED


def test_plan_create_without_device_fails_cleanly():
    try:
        import torch
        if torch.cuda.is_available():
            pytest.skip("a GPU is present")
    except ImportError:
        pass
    h = ctypes.c_void_p()
    s = dg.lib().gemm_plan_create(ctypes.byref(h), ctypes.byref(dg.make_desc(128, 64, 64)))
    assert s in (dg.GEMM_ERR_NO_DEVICE, dg.GEMM_ERR_CUDA)
    assert not h.value
    assert dg.gemm_plan_destroy(None) == dg.GEMM_OK


def test_fp8_block_plan():
    s, info = query(M=8192, N=8192, K=8192, dtype_a=dg.GEMM_E4M3, dtype_d=dg.GEMM_BF16,
                    scale_mode=dg.GEMM_SCALE_BLOCK_1x128_128x128)
    assert s == dg.GEMM_OK
    assert info.kernel == dg.GEMM_KERNEL_FP8_BLOCK
    # SM pairs on 256x256 tiles when there are pair tiles for half the SMs
    assert (info.cta_group, info.tile_m, info.tile_n, info.tile_k) == (2, 256, 256, 128)
    assert info.block_threads == 384 and info.tmem_cols == 512
    assert info.smem_bytes <= GB300.smem_optin_bytes and info.stages >= 4
    s, info = query(M=128, N=8192, K=8192, dtype_a=dg.GEMM_E4M3, dtype_d=dg.GEMM_BF16,
                    scale_mode=dg.GEMM_SCALE_BLOCK_1x128_128x128)
    assert s == dg.GEMM_OK and (info.cta_group, info.tile_m, info.tile_n) == (1, 128, 256)
    # e4m3 requires block scales; 16-bit inputs refuse them
    s, _ = query(M=1024, N=1024, K=1024, dtype_a=dg.GEMM_E4M3)
    assert s == dg.GEMM_ERR_UNSUPPORTED
    # tiles are 128 or 256 wide (4 or 2 TMEM partials); other widths are refused
    s, info = query(M=1024, N=1024, K=1024, dtype_a=dg.GEMM_E4M3, scale_mode=dg.GEMM_SCALE_BLOCK_1x128_128x128,
                    tile_n=128)
    assert s == dg.GEMM_OK and info.tmem_stages == 4
    s, _ = query(M=1024, N=1024, K=1024, dtype_a=dg.GEMM_E4M3, scale_mode=dg.GEMM_SCALE_BLOCK_1x128_128x128,
                 tile_n=192)
    assert s == dg.GEMM_ERR_UNSUPPORTED


def test_stream_k_plan():
    """Tiles that do not fill whole waves: the last wave plus one full wave are
    split along K (stream-K), one fp32 partial slot per cluster."""
    for kw in (dict(M=8192, N=8192, K=8192, tile_n=256),      # 1024 tiles over 76 pairs
               dict(M=2048, N=5120, K=4096)):                 # 80 512-wide tiles: the last wave holds 4
        s, info = query(dtype_a=dg.GEMM_BF16, dtype_d=dg.GEMM_F32, **kw)
        assert s == dg.GEMM_OK
        clusters = info.grid // info.cta_group
        assert info.num_tiles % clusters != 0
        assert info.stream_k_tiles == clusters + info.num_tiles % clusters, kw
        assert info.workspace_bytes >= clusters * info.cta_group * 128 * info.tile_n * 4
    # 512-wide tiles with a last wave at least half full stay data-parallel
    s, info = query(M=8192, N=8192, K=8192, dtype_a=dg.GEMM_BF16, dtype_d=dg.GEMM_F32)
    assert s == dg.GEMM_OK and info.tile_n == 512 and info.stream_k_tiles == 0
    # whole waves, short K (under 48 K atoms), or the flag: data-parallel only, no workspace
    for kw in (dict(M=256 * 76, N=256, K=8192), dict(M=256, N=256, K=256, batch=512),
               dict(M=8192, N=8192, K=2048, tile_n=256),
               dict(M=8192, N=8192, K=8192, flags=dg.GEMM_FLAG_NO_STREAM_K)):
        s, info = query(dtype_a=dg.GEMM_BF16, dtype_d=dg.GEMM_F32, **kw)
        assert s == dg.GEMM_OK and info.stream_k_tiles == 0 and info.workspace_bytes == 0, kw


def test_variant_dtype_plans():
    s, info = query(M=8192, N=8192, K=8192, dtype_a=dg.GEMM_TF32, dtype_d=dg.GEMM_F32)
    # 512-wide pair tiles, one 32-element atom per stage
    assert s == dg.GEMM_OK and info.kernel == dg.GEMM_KERNEL_PERSISTENT and (info.tile_n, info.tile_k) == (512, 32)
    s, info = query(M=4096, N=4096, K=4096, dtype_a=dg.GEMM_E4M3, dtype_b=dg.GEMM_E5M2, dtype_d=dg.GEMM_BF16,
                    scale_mode=dg.GEMM_SCALE_BLOCK_1x128_128x128)
    assert s == dg.GEMM_OK and info.kernel == dg.GEMM_KERNEL_FP8_BLOCK
    # tf32 is never handled by the thread-staged single-CTA kernel; 16/8-bit mixes are refused
    s, info = query(M=64, N=64, K=64, dtype_a=dg.GEMM_TF32, dtype_d=dg.GEMM_F32)
    assert s == dg.GEMM_OK and info.kernel == dg.GEMM_KERNEL_PERSISTENT
    s, _ = query(M=64, N=64, K=64, dtype_a=dg.GEMM_BF16, dtype_b=dg.GEMM_E4M3)
    assert s == dg.GEMM_ERR_UNSUPPORTED


def test_fp16_accumulation_plans():
    """fp16 accumulation: f16 inputs only, persistent kernel, data-parallel tiles."""
    f = dg.GEMM_FLAG_ACCUM_F16
    s, info = query(M=8192, N=8192, K=8192, dtype_a=dg.GEMM_F16, dtype_d=dg.GEMM_F16, flags=f)
    assert s == dg.GEMM_OK and info.kernel == dg.GEMM_KERNEL_PERSISTENT and info.stream_k_tiles == 0
    s, info = query(M=128, N=64, K=64, dtype_a=dg.GEMM_F16, dtype_d=dg.GEMM_F32, flags=f)   # single-CTA size
    assert s == dg.GEMM_OK and info.kernel == dg.GEMM_KERNEL_PERSISTENT
    for kw in (dict(dtype_a=dg.GEMM_BF16), dict(dtype_a=dg.GEMM_TF32),
               dict(dtype_a=dg.GEMM_F16, flags=f | dg.GEMM_FLAG_SINGLE_CTA)):
        kw.setdefault("flags", f)
        s, _ = query(M=1024, N=1024, K=1024, dtype_d=dg.GEMM_F32, **kw)
        assert s == dg.GEMM_ERR_UNSUPPORTED, kw
