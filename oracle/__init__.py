"""CPU oracle for the dense product D = A @ B^T (fp64 accumulation).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` leg of ``bench.py`` may import this package.  The CUDA library
and its Python binding never import it, and it imports nothing from them.

The arithmetic lives in ``oracle.c`` (plain C, compiled here with gcc and
OpenMP, ``-ffp-contract=off`` so x86 and Arm hosts give identical sums).  This
module only marshals numpy arrays.  See the header of ``oracle.c`` for the
definition it follows and the passages of the pages it cites.

parity pins: every function here is pinned by ``tests/test_oracle.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

# element type codes of oracle.c
F16, BF16, E4M3, F32, E5M2, E2M1, E8M0 = 0, 1, 2, 3, 4, 5, 6
_NAMES = {"f16": F16, "float16": F16, "bf16": BF16, "bfloat16": BF16,
          "e4m3": E4M3, "float8_e4m3fn": E4M3, "f32": F32, "float32": F32,
          "e5m2": E5M2, "float8_e5m2": E5M2, "e2m1": E2M1, "e8m0": E8M0}
_BYTES = {F16: 2, BF16: 2, E4M3: 1, F32: 4, E5M2: 1, E2M1: 1, E8M0: 1}
# scale kinds of oracle.c (orc_problem.scaled)
_SCALE_KINDS = {None: 0, "fp32_block": 1, "mx": 2, "nv": 3}


def dtype_code(name) -> int:
    if isinstance(name, int):
        return name
    return _NAMES[str(name)]


class _Problem(ctypes.Structure):
    _fields_ = [
        ("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64), ("batch", ctypes.c_int64),
        ("dtype_a", ctypes.c_int32), ("dtype_b", ctypes.c_int32),
        ("major_a", ctypes.c_int32), ("major_b", ctypes.c_int32),
        ("lda", ctypes.c_int64), ("ldb", ctypes.c_int64),
        ("stride_a", ctypes.c_int64), ("stride_b", ctypes.c_int64),
        ("scaled", ctypes.c_int32), ("pad_", ctypes.c_int32),
        ("ld_sa", ctypes.c_int64), ("ld_sb", ctypes.c_int64),
        ("stride_sa", ctypes.c_int64), ("stride_sb", ctypes.c_int64),
        ("tensor_scale_a", ctypes.c_double), ("tensor_scale_b", ctypes.c_double),
    ]


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, OpenMP)."""
    with _lock:
        stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
        if force or stale:
            tmp = _LIB + ".tmp.%d" % os.getpid()
            cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
                   "-Wall", "-o", tmp, _SRC, "-lm"]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        lib.orc_decode.restype = ctypes.c_double
        lib.orc_decode.argtypes = [ctypes.c_int, ctypes.c_uint32]
        lib.orc_round.restype = ctypes.c_double
        lib.orc_round.argtypes = [ctypes.c_int, ctypes.c_double]
        lib.orc_encode.restype = ctypes.c_uint32
        lib.orc_encode.argtypes = [ctypes.c_int, ctypes.c_double]
        for name in ("orc_decode_array", "orc_round_array", "orc_encode_array"):
            getattr(lib, name).restype = None
        lib.orc_gemm_rows.restype = ctypes.c_int
        lib.orc_num_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def _ptr(a):
    return ctypes.c_void_p(a.ctypes.data) if a is not None else ctypes.c_void_p(0)


def decode(dtype, codes) -> np.ndarray:
    """Exact real values (fp64) of an array of element codes."""
    lib = _load()
    c = np.ascontiguousarray(np.asarray(codes).astype(np.uint32))
    out = np.empty(c.shape, dtype=np.float64)
    lib.orc_decode_array(ctypes.c_int(dtype_code(dtype)), _ptr(c), ctypes.c_int64(c.size), _ptr(out))
    return out


def round_to(dtype, x) -> np.ndarray:
    """Round-to-nearest-even of fp64 values to the format, returned as fp64."""
    lib = _load()
    v = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    out = np.empty(v.shape, dtype=np.float64)
    lib.orc_round_array(ctypes.c_int(dtype_code(dtype)), _ptr(v), ctypes.c_int64(v.size), _ptr(out))
    return out


def encode(dtype, x) -> np.ndarray:
    """Bit patterns (uint32) of round-to-nearest-even encodings of fp64 values."""
    lib = _load()
    v = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    out = np.empty(v.shape, dtype=np.uint32)
    lib.orc_encode_array(ctypes.c_int(dtype_code(dtype)), _ptr(v), ctypes.c_int64(v.size), _ptr(out))
    return out


def num_threads() -> int:
    return int(_load().orc_num_threads())


def _raw(x, dtype):
    """Element codes as a flat contiguous numpy array of the right width."""
    if hasattr(x, "detach"):  # a torch CPU tensor: view its bytes, no torch arithmetic
        import torch
        t = x.detach().contiguous()
        width = {1: torch.uint8, 2: torch.int16, 4: torch.int32}[t.element_size()]
        x = t.view(width).numpy()
    a = np.ascontiguousarray(x).reshape(-1)
    want = {1: np.uint8, 2: np.uint16, 4: np.uint32}[_BYTES[dtype_code(dtype)]]
    if a.dtype.itemsize != np.dtype(want).itemsize:
        raise ValueError("element width does not match dtype %r" % (dtype,))
    return a.view(want)


def gemm_rows(A, B, *, M, N, K, dtype_a, dtype_b, batch=1, major_a="k", major_b="k",
              lda=None, ldb=None, stride_a=None, stride_b=None,
              scale_a=None, scale_b=None, ld_sa=None, ld_sb=None, stride_sa=0, stride_sb=0,
              scale_mode=None, tensor_scales=(1.0, 1.0), rows=None):
    """Reference rows of D and of S = sum |a*b|.

    ``A``/``B`` hold raw element codes (numpy arrays or torch CPU tensors) laid
    out as described in ``oracle.c``; 4-bit E2M1 operands are bytes holding
    two elements each (``lda``/``ldb``/strides still count elements).
    ``scale_mode``: None (no scales, or fp32 block scales when ``scale_a`` is
    given), "mx" (E8M0 per 32) or "nv" (E4M3 per 16 times ``tensor_scales``);
    MX/NV scales are the tiled scale bytes, ``stride_sa``/``stride_sb`` the
    bytes between batch entries (0 = packed).  ``rows`` is a list of flat row
    indices ``b*M + m`` (``None`` = all rows).  Returns ``(D_ref, S)`` as
    float64 arrays of shape ``(len(rows), N)`` (or ``(batch, M, N)``).
    """
    lib = _load()
    ka = major_a in ("k", 0)
    kb = major_b in ("k", 0)
    p = _Problem()
    p.M, p.N, p.K, p.batch = M, N, K, batch
    p.dtype_a, p.dtype_b = dtype_code(dtype_a), dtype_code(dtype_b)
    p.major_a, p.major_b = (0 if ka else 1), (0 if kb else 1)
    p.lda = lda if lda is not None else (K if ka else M)
    p.ldb = ldb if ldb is not None else (K if kb else N)
    p.stride_a = stride_a if stride_a is not None else M * K
    p.stride_b = stride_b if stride_b is not None else N * K
    a = _raw(A, dtype_a)
    b = _raw(B, dtype_b)
    sa = sb = None
    p.scaled = 0
    p.tensor_scale_a, p.tensor_scale_b = float(tensor_scales[0]), float(tensor_scales[1])
    if scale_mode in ("mx", "nv"):
        p.scaled = _SCALE_KINDS[scale_mode]
        sa = _raw(scale_a, "e8m0")
        sb = _raw(scale_b, "e8m0")
        p.stride_sa, p.stride_sb = stride_sa, stride_sb
    elif scale_a is not None or scale_b is not None:
        p.scaled = 1
        sa = np.ascontiguousarray(np.asarray(scale_a, dtype=np.float32)).reshape(-1)
        sb = np.ascontiguousarray(np.asarray(scale_b, dtype=np.float32)).reshape(-1)
        kblocks = (K + 127) // 128
        p.ld_sa = ld_sa if ld_sa is not None else kblocks
        p.ld_sb = ld_sb if ld_sb is not None else kblocks
        p.stride_sa, p.stride_sb = stride_sa, stride_sb
    if rows is None:
        nrows = batch * M
        rows_arr = None
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        nrows = rows_arr.size
    d = np.empty((nrows, N), dtype=np.float64)
    s = np.empty((nrows, N), dtype=np.float64)
    rc = lib.orc_gemm_rows(ctypes.byref(p), _ptr(a), _ptr(b), _ptr(sa), _ptr(sb),
                           ctypes.c_int64(nrows), _ptr(rows_arr), _ptr(d), _ptr(s))
    if rc != 0:
        raise ValueError("oracle rejected the problem")
    if rows is None:
        return d.reshape(batch, M, N), s.reshape(batch, M, N)
    return d, s


def gemm(A, B, **kw):
    """Full reference product; same arguments as :func:`gemm_rows` without ``rows``."""
    kw.pop("rows", None)
    return gemm_rows(A, B, rows=None, **kw)
