"""CPU oracle for the pipelined GEMM -- TEST INFRASTRUCTURE, not product code.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its
``cpu_baseline`` leg and its ``--impl reference`` arm) may import this package.
It shares no code with the CUDA path in ``stage_software_pipelining_gb300``
and imports nothing from it.

The arithmetic lives in ``gemm_oracle.c``: the plain fp64 i-k-j triple loop of
``C = alpha*A*B + beta*C0`` together with ``Abs = |A|*|B|`` (the bound matrix
used by the tolerances).  The problem statement it follows is the one of
"CUTLASS-CuTe 初步(6)", section 2 "Thread Block Tile" (C += A*B, accumulated
over the K tiles) and of "Software Pipelining and Double Buffering", section
"Double buffering with shared memory" (acc += As*Bs over k, then C = acc).

This module only marshals arguments: it hands the raw input bits (fp32, fp16
or bf16 storage) and their strides to the C code, which decodes them exactly
to fp64 itself.

Every function here is pinned by ``tests/test_oracle.py`` against hand-worked
fixtures, identities, closed forms, exact rational arithmetic and library
routines; no function is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

T_F32, T_F16, T_BF16 = 0, 1, 2

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``gemm_oracle.c`` into ``liboracle.so`` (gcc, OpenMP) if stale."""
    with _lock:
        stale = (not os.path.exists(_LIB_PATH)
                 or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
        if force or stale:
            tmp = _LIB_PATH + f".tmp{os.getpid()}"
            cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-shared", "-fPIC",
                   "-o", tmp, _SRC, "-lm"]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _open(path: str):
    lib = ctypes.CDLL(path)
    i64, p, i32, f64 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int, ctypes.c_double
    common = [i64, i64, i64, p, i64, i32, p, i64, i32, i32, p, i64, i32, f64, f64]
    lib.oracle_gemm_rows.argtypes = common + [p, i64, p, i64, i64, i64, i32]
    lib.oracle_gemm_rows.restype = i32
    lib.oracle_gemm_entries.argtypes = common + [p, p, i64, p, p, i32]
    lib.oracle_gemm_entries.restype = i32
    lib.oracle_decode_f16.argtypes = [ctypes.c_uint16]
    lib.oracle_decode_f16.restype = f64
    lib.oracle_decode_bf16.argtypes = [ctypes.c_uint16]
    lib.oracle_decode_bf16.restype = f64
    lib.oracle_decode_f32.argtypes = [ctypes.c_uint32]
    lib.oracle_decode_f32.restype = f64
    lib.oracle_max_threads.argtypes = []
    lib.oracle_max_threads.restype = i32
    lib.oracle_copy_bytes.argtypes = [p, p, i64]
    lib.oracle_copy_bytes.restype = i32
    return lib


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = _open(_LIB_PATH)
    return _lib


class using_library:
    """Context manager: route this module's calls to another build of the
    oracle source (the tests use it to check that the pins reject copies of
    the oracle with a planted mistake)."""

    def __init__(self, path: str):
        self.path = path

    def __enter__(self):
        global _lib
        self.saved = _load()
        _lib = _open(self.path)
        return self

    def __exit__(self, *exc):
        global _lib
        _lib = self.saved
        return False


class _Operand:
    """A 2-D operand as raw storage: pointer, format code, strides (elements)."""

    def __init__(self, x, name):
        arr, code = _raw_view(x)
        if arr.ndim != 2:
            raise ValueError(f"{name} must be 2-D")
        item = arr.itemsize
        s0, s1 = arr.strides[0] // item, arr.strides[1] // item
        if arr.size == 0:            # empty arrays report zero strides
            s0, s1 = max(arr.shape[1], 1), 1
        self.keep = arr
        self.ptr = arr.ctypes.data
        self.code = code
        self.rows, self.cols = arr.shape
        self.s0, self.s1 = s0, s1


def _raw_view(x):
    """(numpy array of the storage bits or values, format code) for x."""
    try:
        import torch  # plain CPU tensors are accepted as inputs
        if isinstance(x, torch.Tensor):
            if x.device.type != "cpu":
                raise ValueError("the oracle takes host (CPU) tensors only")
            if x.dtype == torch.bfloat16:
                return x.view(torch.int16).numpy().view(np.uint16), T_BF16
            if x.dtype == torch.float16:
                return x.view(torch.int16).numpy().view(np.uint16), T_F16
            if x.dtype == torch.float32:
                return x.numpy(), T_F32
            raise ValueError(f"unsupported dtype {x.dtype}")
    except ImportError:
        pass
    x = np.asarray(x)
    if x.dtype == np.float32:
        return x, T_F32
    if x.dtype == np.float16:
        return x.view(np.uint16), T_F16
    raise ValueError(f"unsupported dtype {x.dtype}; bf16 must come as a torch tensor")


def _row_major_ld(op: _Operand, name: str) -> int:
    if op.rows > 1 and op.cols > 1 and op.s1 != 1:
        raise ValueError(f"{name} must be row-major (unit column stride)")
    return max(op.s0, op.cols, 1) if op.rows > 1 else max(op.cols, 1)


def _b_layout(op: _Operand):
    """(ldb, b_col_major) for B viewed as K x N."""
    K, N = op.rows, op.cols
    if op.s1 == 1 or N <= 1 and op.s0 != 1:
        ld = op.s0 if K > 1 else max(N, 1)
        return max(ld, N, 1), 0
    if op.s0 == 1:
        ld = op.s1 if N > 1 else max(K, 1)
        return max(ld, K, 1), 1
    raise ValueError("B must be row-major or column-major")


def _prepare(A, B, C0, beta):
    a = _Operand(A, "A")
    b = _Operand(B, "B")
    M, K = a.rows, a.cols
    if b.rows != K:
        raise ValueError(f"inner dimensions differ: A is {M}x{K}, B is {b.rows}x{b.cols}")
    N = b.cols
    lda = _row_major_ld(a, "A")
    ldb, bcm = _b_layout(b)
    if beta != 0.0:
        if C0 is None:
            raise ValueError("beta != 0 needs C0")
        c = _Operand(C0, "C0")
        if (c.rows, c.cols) != (M, N):
            raise ValueError("C0 must be M x N")
        ldc0 = _row_major_ld(c, "C0")
        cptr, ccode = c.ptr, c.code
    else:
        c, cptr, ccode, ldc0 = None, None, T_F32, max(N, 1)
    return a, b, c, M, N, K, lda, ldb, bcm, cptr, ccode, ldc0


def gemm(A, B, C0=None, alpha: float = 1.0, beta: float = 0.0, *, rows=None,
         nthreads: int = 0, with_abs: bool = True):
    """fp64 ``alpha*A@B + beta*C0`` and ``|A|@|B|`` on the host.

    A: M x K row-major; B: K x N row-major or column-major (a transposed view);
    C0: M x N row-major, not read when beta == 0.  ``rows=(r0, r1)`` computes
    only rows r0..r1-1 and returns arrays of shape (r1-r0, N).
    Returns (C, Abs) as float64 numpy arrays (Abs is None if not requested).
    """
    lib = _load()
    a, b, c, M, N, K, lda, ldb, bcm, cptr, ccode, ldc0 = _prepare(A, B, C0, beta)
    r0, r1 = (0, M) if rows is None else rows
    if not (0 <= r0 <= r1 <= M):
        raise ValueError("bad row range")
    out = np.zeros((r1 - r0, N), dtype=np.float64)
    absm = np.zeros_like(out) if with_abs else None
    ld = max(N, 1)
    base = out.ctypes.data
    abase = absm.ctypes.data if with_abs else None
    st = lib.oracle_gemm_rows(M, N, K, a.ptr, lda, a.code, b.ptr, ldb, b.code, bcm,
                              cptr, ldc0, ccode, float(alpha), float(beta),
                              base, ld, abase, ld, r0, r1, int(nthreads))
    if st != 0:
        raise RuntimeError(f"oracle_gemm_rows failed with status {st}")
    return out, absm


def gemm_entries(A, B, C0=None, alpha: float = 1.0, beta: float = 0.0, *, rows, cols,
                 nthreads: int = 0):
    """fp64 entries C[rows[t], cols[t]] and Abs[rows[t], cols[t]]."""
    lib = _load()
    a, b, c, M, N, K, lda, ldb, bcm, cptr, ccode, ldc0 = _prepare(A, B, C0, beta)
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    cc = np.ascontiguousarray(np.asarray(cols, dtype=np.int64))
    if r.shape != cc.shape or r.ndim != 1:
        raise ValueError("rows and cols must be 1-D and the same length")
    out = np.zeros(r.shape[0], dtype=np.float64)
    absv = np.zeros_like(out)
    st = lib.oracle_gemm_entries(M, N, K, a.ptr, lda, a.code, b.ptr, ldb, b.code, bcm,
                                 cptr, ldc0, ccode, float(alpha), float(beta),
                                 r.ctypes.data, cc.ctypes.data, r.shape[0],
                                 out.ctypes.data, absv.ctypes.data, int(nthreads))
    if st != 0:
        raise RuntimeError(f"oracle_gemm_entries failed with status {st}")
    return out, absv


def copy_bytes(src: np.ndarray) -> np.ndarray:
    """The streaming copy's result: a byte-for-byte copy of src (uint8)."""
    src = np.ascontiguousarray(np.asarray(src, dtype=np.uint8))
    out = np.empty_like(src)
    st = _load().oracle_copy_bytes(out.ctypes.data, src.ctypes.data, src.size)
    if st != 0:
        raise RuntimeError(f"oracle_copy_bytes failed with status {st}")
    return out


def decode_f16(bits: int) -> float:
    return _load().oracle_decode_f16(int(bits) & 0xFFFF)


def decode_bf16(bits: int) -> float:
    return _load().oracle_decode_bf16(int(bits) & 0xFFFF)


def decode_f32(bits: int) -> float:
    return _load().oracle_decode_f32(int(bits) & 0xFFFFFFFF)


def max_threads() -> int:
    return int(_load().oracle_max_threads())
