"""Python binding of the GB300 dense GEMM library (D = A @ B^T, fp32 accumulation).

Argument marshalling only: every step of the product runs in the CUDA library
``libdgb_gemm.so`` (built by :func:`build`).  The functions keep the names of
the C ABI in ``include/gemm.h``; :class:`Plan` and :func:`matmul` wrap them for
torch CUDA tensors and the current torch stream.  There is no fallback: if the
library is missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

from ._build import LIB as _LIB_PATH, build as _build

__all__ = [
    "build", "lib", "GemmError", "GemmDesc", "GemmPlanInfo", "GemmDeviceProps", "GemmDeviceError",
    "gemm_plan_query", "gemm_plan_create", "gemm_plan_info", "gemm_run", "gemm_run_mx", "gemm_run_host",
    "gemm_run_noalloc",
    "gemm_sync_status", "gemm_plan_destroy", "gemm_status_string", "gemm_last_cuda_error",
    "gemm_version", "gemm_schedule_model", "gemm_schedule_choose", "gemm_plan_work_unit", "GemmWorkUnit", "Plan",
    "GemmMachine", "gemm_plan_schedule", "gemm_machine_gb300",
    "matmul", "header_functions",
]

# ---------------------------------------------------------------- constants (include/gemm.h)
GEMM_OK, GEMM_ERR_INVALID_ARG, GEMM_ERR_UNSUPPORTED, GEMM_ERR_ALIGNMENT = 0, 1, 2, 3
GEMM_ERR_CUDA, GEMM_ERR_TIMEOUT, GEMM_ERR_NO_DEVICE, GEMM_ERR_RESOURCES = 4, 5, 6, 7
GEMM_F16, GEMM_BF16, GEMM_E4M3, GEMM_F32, GEMM_E5M2, GEMM_TF32, GEMM_E2M1 = 0, 1, 2, 3, 4, 5, 6
GEMM_K_MAJOR, GEMM_MN_MAJOR = 0, 1
GEMM_SCALE_NONE, GEMM_SCALE_BLOCK_1x128_128x128, GEMM_SCALE_MX_E8M0_32, GEMM_SCALE_NV_E4M3_16 = 0, 1, 2, 3
GEMM_KERNEL_SINGLE_CTA, GEMM_KERNEL_PERSISTENT, GEMM_KERNEL_FP8_BLOCK, GEMM_KERNEL_ZERO_FILL = 1, 2, 3, 4
GEMM_KERNEL_MX = 5
GEMM_FLAG_CTA_GROUP_1 = 1 << 0
GEMM_FLAG_CTA_GROUP_2 = 1 << 1
GEMM_FLAG_NO_SINGLE_CTA = 1 << 2
GEMM_FLAG_SINGLE_CTA = 1 << 3
GEMM_FLAG_NO_L2_HINTS = 1 << 4
GEMM_FLAG_NO_STREAM_K = 1 << 5
GEMM_FLAG_EPILOGUE_DIRECT = 1 << 6
GEMM_FLAG_EPILOGUE_TMA = 1 << 7
GEMM_FLAG_STAGE_K1 = 1 << 8
GEMM_FLAG_STAGE_K2 = 1 << 9
GEMM_FLAG_ACCUM_F16 = 1 << 10
GEMM_FLAG_TEST_DROP_LOAD = 1 << 30

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "gemm.h")


class GemmDesc(ctypes.Structure):
    _fields_ = [
        ("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64), ("batch", ctypes.c_int64),
        ("dtype_a", ctypes.c_int32), ("dtype_b", ctypes.c_int32), ("dtype_d", ctypes.c_int32),
        ("major_a", ctypes.c_int32), ("major_b", ctypes.c_int32), ("scale_mode", ctypes.c_int32),
        ("lda", ctypes.c_int64), ("ldb", ctypes.c_int64), ("ldd", ctypes.c_int64),
        ("stride_a", ctypes.c_int64), ("stride_b", ctypes.c_int64), ("stride_d", ctypes.c_int64),
        ("ld_sa", ctypes.c_int64), ("ld_sb", ctypes.c_int64),
        ("stride_sa", ctypes.c_int64), ("stride_sb", ctypes.c_int64),
        ("flags", ctypes.c_uint32), ("tile_n", ctypes.c_int32), ("stages", ctypes.c_int32),
        ("max_ctas", ctypes.c_int32), ("wait_timeout_ns", ctypes.c_uint64),
        ("raster_group", ctypes.c_int32), ("reserved0", ctypes.c_int32),
    ]


class GemmPlanInfo(ctypes.Structure):
    _fields_ = [
        ("kernel", ctypes.c_int32), ("cta_group", ctypes.c_int32), ("tile_m", ctypes.c_int32),
        ("tile_n", ctypes.c_int32), ("tile_k", ctypes.c_int32), ("stages", ctypes.c_int32),
        ("tmem_stages", ctypes.c_int32), ("tmem_cols", ctypes.c_int32), ("grid", ctypes.c_int32),
        ("block_threads", ctypes.c_int32), ("num_tiles", ctypes.c_int64), ("stage_bytes", ctypes.c_int64),
        ("pipeline_bytes", ctypes.c_int64), ("smem_bytes", ctypes.c_int64),
        ("stream_k_tiles", ctypes.c_int32), ("epilogue", ctypes.c_int32), ("workspace_bytes", ctypes.c_int64),
    ]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


class GemmWorkUnit(ctypes.Structure):
    _fields_ = [("tile", ctypes.c_int32), ("batch", ctypes.c_int32), ("m_block", ctypes.c_int32),
                ("n_block", ctypes.c_int32), ("k_block_begin", ctypes.c_int32), ("k_block_end", ctypes.c_int32),
                ("role", ctypes.c_int32), ("slot", ctypes.c_int32),
                ("slot_first", ctypes.c_int32)]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


class GemmDeviceProps(ctypes.Structure):
    _fields_ = [("sm_count", ctypes.c_int32), ("smem_optin_bytes", ctypes.c_int32),
                ("cc_major", ctypes.c_int32), ("cc_minor", ctypes.c_int32)]


class GemmSchedParams(ctypes.Structure):
    _fields_ = [("tiles", ctypes.c_int32), ("k_slices", ctypes.c_int32), ("stages", ctypes.c_int32),
                ("accumulators", ctypes.c_int32), ("t_issue", ctypes.c_double), ("t_load", ctypes.c_double),
                ("t_mma", ctypes.c_double), ("t_epi", ctypes.c_double)]


class GemmSchedResult(ctypes.Structure):
    _fields_ = [("run_length", ctypes.c_double), ("tensor_busy", ctypes.c_double),
                ("steady_period", ctypes.c_double), ("stages_needed", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class GemmMachine(ctypes.Structure):
    _fields_ = [("mma_flops_per_cycle", ctypes.c_double), ("stage_fixed_cycles", ctypes.c_double),
                ("ingest_bytes_per_cycle", ctypes.c_double), ("load_latency_cycles", ctypes.c_double),
                ("tmem_read_bytes_per_cycle", ctypes.c_double), ("handback_cycles", ctypes.c_double)]


class GemmDeviceError(ctypes.Structure):
    _fields_ = [("code", ctypes.c_uint32), ("role", ctypes.c_uint32), ("stage", ctypes.c_uint32),
                ("tile", ctypes.c_uint32), ("block", ctypes.c_uint32), ("reserved", ctypes.c_uint32 * 3)]


class GemmError(RuntimeError):
    def __init__(self, status, where=""):
        self.status = int(status)
        msg = gemm_status_string(status) if _lib is not None else str(status)
        if self.status == GEMM_ERR_CUDA and _lib is not None:
            msg += " (cudaError %d)" % gemm_last_cuda_error()
        super().__init__("%s: %s" % (where, msg) if where else msg)


_lock = threading.Lock()
_lib = None


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the CUDA library in-tree (nvcc, sm_103a)."""
    return _build(force=force, verbose=verbose)


def lib():
    """The loaded CUDA library; raises if it has not been built."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(_LIB_PATH):
                    raise RuntimeError("CUDA library %s is missing: call dense_gemm_blackwell_gb300.build()"
                                       % _LIB_PATH)
                L = ctypes.CDLL(_LIB_PATH)
                vp, st = ctypes.c_void_p, ctypes.c_int
                L.gemm_plan_query.argtypes = [ctypes.POINTER(GemmDesc), ctypes.POINTER(GemmDeviceProps),
                                              ctypes.POINTER(GemmPlanInfo)]
                L.gemm_plan_query.restype = st
                L.gemm_plan_create.argtypes = [ctypes.POINTER(vp), ctypes.POINTER(GemmDesc)]
                L.gemm_plan_create.restype = st
                L.gemm_plan_info.argtypes = [vp, ctypes.POINTER(GemmPlanInfo)]
                L.gemm_plan_info.restype = st
                L.gemm_plan_work_unit.argtypes = [ctypes.POINTER(GemmDesc), ctypes.POINTER(GemmPlanInfo),
                                                  ctypes.c_int32, ctypes.c_int32, ctypes.POINTER(GemmWorkUnit)]
                L.gemm_plan_work_unit.restype = st
                L.gemm_run.argtypes = [vp, vp, vp, vp, vp, vp, vp]
                L.gemm_run.restype = st
                L.gemm_run_mx.argtypes = [vp] * 8
                L.gemm_run_mx.restype = st
                L.gemm_run_host.argtypes = [vp] * 12
                L.gemm_run_host.restype = st
                L.gemm_run_noalloc.argtypes = [ctypes.POINTER(GemmDesc), vp, vp, vp, vp, vp, vp,
                                               ctypes.POINTER(GemmDeviceError)]
                L.gemm_run_noalloc.restype = st
                L.gemm_sync_status.argtypes = [vp, vp, ctypes.POINTER(GemmDeviceError)]
                L.gemm_sync_status.restype = st
                L.gemm_plan_destroy.argtypes = [vp]
                L.gemm_plan_destroy.restype = st
                L.gemm_status_string.argtypes = [st]
                L.gemm_status_string.restype = ctypes.c_char_p
                L.gemm_last_cuda_error.restype = st
                L.gemm_schedule_model.argtypes = [ctypes.POINTER(GemmSchedParams), ctypes.POINTER(GemmSchedResult)]
                L.gemm_schedule_model.restype = st
                L.gemm_schedule_choose.argtypes = [ctypes.POINTER(GemmSchedParams), ctypes.c_int32, ctypes.c_int32,
                                                   ctypes.c_double, ctypes.POINTER(ctypes.c_int32),
                                                   ctypes.POINTER(ctypes.c_int32)]
                L.gemm_schedule_choose.restype = st
                L.gemm_plan_schedule.argtypes = [ctypes.POINTER(GemmDesc), ctypes.POINTER(GemmPlanInfo),
                                                 ctypes.POINTER(GemmDeviceProps), ctypes.POINTER(GemmMachine),
                                                 ctypes.POINTER(GemmSchedParams), ctypes.POINTER(GemmSchedResult),
                                                 ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32)]
                L.gemm_plan_schedule.restype = st
                L.gemm_machine_gb300.argtypes = [ctypes.POINTER(GemmMachine)]
                L.gemm_machine_gb300.restype = st
                L.gemm_version.restype = st
                _lib = L
    return _lib


def header_functions():
    """Names of the functions include/gemm.h declares."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(gemm_\w+)\s*\(", text, re.M)))


# ---------------------------------------------------------------- C ABI, same names

def gemm_plan_query(desc: GemmDesc, props: GemmDeviceProps):
    info = GemmPlanInfo()
    s = lib().gemm_plan_query(ctypes.byref(desc), ctypes.byref(props), ctypes.byref(info))
    return s, info


def gemm_plan_create(desc: GemmDesc):
    h = ctypes.c_void_p()
    s = lib().gemm_plan_create(ctypes.byref(h), ctypes.byref(desc))
    if s != GEMM_OK:
        raise GemmError(s, "gemm_plan_create")
    return h


def gemm_plan_info(plan) -> GemmPlanInfo:
    info = GemmPlanInfo()
    s = lib().gemm_plan_info(plan, ctypes.byref(info))
    if s != GEMM_OK:
        raise GemmError(s, "gemm_plan_info")
    return info


def gemm_plan_work_unit(desc: GemmDesc, info: GemmPlanInfo, cluster: int, index: int):
    """(status, GemmWorkUnit): the index-th unit of a cluster of a persistent plan; tile -1 past its last."""
    u = GemmWorkUnit()
    s = lib().gemm_plan_work_unit(ctypes.byref(desc), ctypes.byref(info), cluster, index, ctypes.byref(u))
    return s, u


def gemm_run(plan, A, B, D, scale_a=None, scale_b=None, stream=None) -> int:
    return lib().gemm_run(plan, A, B, D, scale_a, scale_b, stream)


def gemm_run_mx(plan, A, B, D, sf_a, sf_b, tensor_scales=None, stream=None) -> int:
    """Hardware block-scaled product (MX / NVFP4 plans); pointers are device addresses."""
    return lib().gemm_run_mx(plan, A, B, D, sf_a, sf_b, tensor_scales, stream)


def gemm_run_host(plan, hA, hB, hD, hsa, hsb, dA, dB, dD, dsa, dsb, stream=None) -> int:
    return lib().gemm_run_host(plan, hA, hB, hD, hsa, hsb, dA, dB, dD, dsa, dsb, stream)


def gemm_run_noalloc(desc: GemmDesc, A, B, D, scale_a=None, scale_b=None, stream=None, status_out=None) -> int:
    """Allocation-free product (see include/gemm.h); status_out: a GemmDeviceError or None."""
    ref = ctypes.byref(status_out) if status_out is not None else None
    return lib().gemm_run_noalloc(ctypes.byref(desc), A, B, D, scale_a, scale_b, stream, ref)


def gemm_sync_status(plan, stream=None):
    rec = GemmDeviceError()
    s = lib().gemm_sync_status(plan, stream, ctypes.byref(rec))
    return s, rec


def gemm_plan_destroy(plan) -> int:
    return lib().gemm_plan_destroy(plan)


def gemm_status_string(status) -> str:
    return lib().gemm_status_string(int(status)).decode()


def gemm_schedule_model(tiles, k_slices, stages, accumulators, t_issue, t_load, t_mma, t_epi):
    """Evaluate the pipeline schedule model; returns (status, GemmSchedResult)."""
    p = GemmSchedParams(tiles, k_slices, stages, accumulators, t_issue, t_load, t_mma, t_epi)
    r = GemmSchedResult()
    return lib().gemm_schedule_model(ctypes.byref(p), ctypes.byref(r)), r


def gemm_schedule_choose(tiles, k_slices, t_issue, t_load, t_mma, t_epi, max_stages, max_accumulators,
                         tolerance=0.0):
    """Fewest accumulators, then stages, within `tolerance` of the deepest pipeline: (status, S, A)."""
    p = GemmSchedParams(tiles, k_slices, 1, 1, t_issue, t_load, t_mma, t_epi)
    s, a = ctypes.c_int32(), ctypes.c_int32()
    st = lib().gemm_schedule_choose(ctypes.byref(p), max_stages, max_accumulators, tolerance,
                                    ctypes.byref(s), ctypes.byref(a))
    return st, s.value, a.value


def gemm_plan_schedule(desc: GemmDesc, info: GemmPlanInfo, props: GemmDeviceProps, machine=None):
    """The schedule model of a planned problem: (status, GemmSchedParams, GemmSchedResult, S, A), S and A
    being the model's choice within the plan's limits; machine None = the measured GB300 figures."""
    p, r = GemmSchedParams(), GemmSchedResult()
    s, a = ctypes.c_int32(), ctypes.c_int32()
    st = lib().gemm_plan_schedule(ctypes.byref(desc), ctypes.byref(info), ctypes.byref(props),
                                  ctypes.byref(machine) if machine is not None else None,
                                  ctypes.byref(p), ctypes.byref(r), ctypes.byref(s), ctypes.byref(a))
    return st, p, r, s.value, a.value


def gemm_machine_gb300() -> GemmMachine:
    m = GemmMachine()
    st = lib().gemm_machine_gb300(ctypes.byref(m))
    if st != GEMM_OK:
        raise GemmError(st, "gemm_machine_gb300")
    return m


def gemm_last_cuda_error() -> int:
    return lib().gemm_last_cuda_error()


def gemm_version() -> int:
    return lib().gemm_version()


# ---------------------------------------------------------------- torch convenience

def _dtype_code(t):
    import torch
    codes = {torch.float16: GEMM_F16, torch.bfloat16: GEMM_BF16, torch.float32: GEMM_F32,
             torch.float8_e4m3fn: GEMM_E4M3, torch.float8_e5m2: GEMM_E5M2}
    if t not in codes:
        raise TypeError("unsupported dtype %s" % t)
    return codes[t]


def _torch_dtype(code):
    import torch
    return {GEMM_F16: torch.float16, GEMM_BF16: torch.bfloat16, GEMM_F32: torch.float32,
            GEMM_E4M3: torch.float8_e4m3fn, GEMM_E5M2: torch.float8_e5m2}[code]


def make_desc(M, N, K, *, batch=1, dtype_a=GEMM_BF16, dtype_b=None, dtype_d=GEMM_F32,
              major_a=GEMM_K_MAJOR, major_b=GEMM_K_MAJOR, scale_mode=GEMM_SCALE_NONE,
              lda=0, ldb=0, ldd=0, stride_a=0, stride_b=0, stride_d=0, ld_sa=0, ld_sb=0,
              stride_sa=0, stride_sb=0, flags=0, tile_n=0, stages=0, max_ctas=0, wait_timeout_ns=0,
              raster_group=0) -> GemmDesc:
    d = GemmDesc()
    d.M, d.N, d.K, d.batch = M, N, K, batch
    d.dtype_a = dtype_a
    d.dtype_b = dtype_a if dtype_b is None else dtype_b
    d.dtype_d = dtype_d
    d.major_a, d.major_b, d.scale_mode = major_a, major_b, scale_mode
    d.lda, d.ldb, d.ldd = lda, ldb, ldd
    d.stride_a, d.stride_b, d.stride_d = stride_a, stride_b, stride_d
    d.ld_sa, d.ld_sb, d.stride_sa, d.stride_sb = ld_sa, ld_sb, stride_sa, stride_sb
    d.flags, d.tile_n, d.stages, d.max_ctas = flags, tile_n, stages, max_ctas
    d.wait_timeout_ns = wait_timeout_ns
    d.raster_group = raster_group
    return d


def current_stream_handle():
    """cudaStream_t of torch's current stream on the current device.  Uses the
    raw-handle query when this torch has it (torch.cuda.current_stream() builds
    a Stream object, about 3 us per call)."""
    import torch
    raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
    if raw is not None:
        return raw(torch._C._cuda_getDevice())
    return torch.cuda.current_stream().cuda_stream


class Plan:
    """A created plan (owns the C handle); use as a context manager or call close()."""

    def __init__(self, desc: GemmDesc):
        self.desc = desc
        self.handle = gemm_plan_create(desc)
        self.info = gemm_plan_info(self.handle)

    def run(self, A, B, D, scale_a=None, scale_b=None, stream=None):
        """Enqueue on `stream` (default: torch's current stream); tensors are torch CUDA tensors."""
        if stream is None:
            stream = current_stream_handle()
        s = lib().gemm_run(self.handle, A.data_ptr(), B.data_ptr(), D.data_ptr(),
                           None if scale_a is None else scale_a.data_ptr(),
                           None if scale_b is None else scale_b.data_ptr(), stream)
        if s != GEMM_OK:
            raise GemmError(s, "gemm_run")

    def run_mx(self, A, B, D, sf_a, sf_b, tensor_scales=None, stream=None):
        """Enqueue an MX / NVFP4 product: sf_a, sf_b are the tiled scale bytes and
        tensor_scales (NVFP4 only) a 2-element fp32 tensor, all torch CUDA tensors."""
        if stream is None:
            stream = current_stream_handle()
        s = lib().gemm_run_mx(self.handle, A.data_ptr(), B.data_ptr(), D.data_ptr(), sf_a.data_ptr(),
                              sf_b.data_ptr(), None if tensor_scales is None else tensor_scales.data_ptr(), stream)
        if s != GEMM_OK:
            raise GemmError(s, "gemm_run_mx")

    def run_host(self, hA, hB, hD, dA, dB, dD, hsa=None, hsb=None, dsa=None, dsb=None, stream=None):
        if stream is None:
            stream = current_stream_handle()
        ptr = lambda t: None if t is None else t.data_ptr()  # noqa: E731
        s = gemm_run_host(self.handle, ptr(hA), ptr(hB), ptr(hD), ptr(hsa), ptr(hsb), ptr(dA), ptr(dB),
                          ptr(dD), ptr(dsa), ptr(dsb), stream)
        if s != GEMM_OK:
            raise GemmError(s, "gemm_run_host")

    def sync_status(self, stream=None):
        if stream is None:
            stream = current_stream_handle()
        return gemm_sync_status(self.handle, stream)

    def close(self):
        if self.handle is not None:
            gemm_plan_destroy(self.handle)
            self.handle = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


_plan_cache = {}


def matmul(a, b, *, out=None, out_dtype=None, scale_a=None, scale_b=None, flags=0, tile_n=0, stages=0):
    """D = a @ b^T for torch CUDA tensors.

    a: [M, K] or [batch, M, K] (last dim contiguous), b: [N, K] or [batch, N, K];
    e4m3 inputs need scale_a [M, ceil(K/128)] and scale_b [ceil(N/128), ceil(K/128)] fp32.
    Returns D [M, N] / [batch, M, N] in out_dtype (default fp32).
    """
    import torch
    batched = a.dim() == 3
    if batched:
        batch, M, K = a.shape
        N = b.shape[1]
    else:
        batch, (M, K), N = 1, a.shape, b.shape[0]
    if a.stride(-1) != 1 or b.stride(-1) != 1:
        raise ValueError("inputs must be K-contiguous")
    code_d = _dtype_code(out_dtype or (out.dtype if out is not None else torch.float32))
    if out is None:
        shape = (batch, M, N) if batched else (M, N)
        out = torch.empty(shape, dtype=_torch_dtype(code_d), device=a.device)
    da = _dtype_code(a.dtype)
    db = _dtype_code(b.dtype)
    if da == GEMM_F32:   # fp32 inputs are multiplied at tf32 precision
        da = db = GEMM_TF32
    desc = make_desc(M, N, K, batch=batch, dtype_a=da, dtype_b=db, dtype_d=code_d,
                     scale_mode=GEMM_SCALE_BLOCK_1x128_128x128 if da in (GEMM_E4M3, GEMM_E5M2) else GEMM_SCALE_NONE,
                     lda=a.stride(-2), ldb=b.stride(-2), ldd=out.stride(-2),
                     stride_a=a.stride(0) if batched else 0, stride_b=b.stride(0) if batched else 0,
                     stride_d=out.stride(0) if batched else 0, flags=flags, tile_n=tile_n, stages=stages)
    key = (a.device.index, bytes(desc))
    plan = _plan_cache.get(key)
    if plan is None:
        plan = _plan_cache[key] = Plan(desc)
    plan.run(a, b, out, scale_a, scale_b)
    return out
