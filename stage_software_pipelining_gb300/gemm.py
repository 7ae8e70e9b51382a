"""ctypes binding over libgemm.so's C ABI (include/gemm.h).

Argument marshalling only: tensors become (pointer, leading dimension) pairs
and a dtype code; all arithmetic runs in the CUDA kernels of libgemm.so.
If the library is missing the first call raises: there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from .workloads import GEMM_BF16_BF16, GEMM_BF16_F32, GEMM_F16_F32, GEMM_F32

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libgemm.so")

GEMM_OK = 0
GEMM_ERR_ARG = -1
GEMM_ERR_UNSUPPORTED = -2
GEMM_ERR_ALIGN = -3
GEMM_ERR_LAUNCH = -4
GEMM_ERR_TIMEOUT = -5
GEMM_ERR_CUDA = -6
GEMM_ERR_SCRATCH = -7

# Tensor-core tiles (gemm_tile_t)
TILE_AUTO = 0
TILE_128x128 = 128
TILE_128x256 = 256
TILE_256x256_2SM = 512
TILE_256x512_2SM = 1024

# Deepest ring each tensor-core tile has shared memory for (gemm_max_stages);
# every stage is a K slice of 64.
TILE_MAX_STAGES = {TILE_128x128: 6, TILE_128x256: 4, TILE_256x256_2SM: 6, TILE_256x512_2SM: 4}
TC_MAX_STAGES = 6

# SIMT register-fragment schemes (gemm_simt_fragments_t), passed as `tile` for fp32
SIMT_FRAGMENTS_DOUBLE = 0
SIMT_FRAGMENTS_SINGLE = 1

# Every extern "C" symbol include/gemm.h declares.
EXPORTS = ("gemm", "gemm_ex", "gemm_checked", "gemm_host", "gemm_host_release",
           "gemm_status_string", "gemm_max_stages", "gemm_plan", "gemm_debug_set",
           "gemm_resolve_tile",
           "pipelined_copy", "gemm_schedule_set", "gemm_noalloc", "mma_rate",
           "gemm_clock_log", "mma_rate_pair")

_lock = threading.Lock()
_lib = None


class GemmError(RuntimeError):
    def __init__(self, status: int, what: str = "gemm"):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


def load_library(path: str = LIB_PATH):
    """Load libgemm.so and declare its signatures.  Raises if it is missing."""
    global _lib
    with _lock:
        if _lib is not None and path == LIB_PATH:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it first (python -c 'import __graft_entry__ as g; "
                "g.build()'); there is no CPU fallback")
        lib = ctypes.CDLL(path)
        i64, p, i32, f32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        base = [i64, i64, i64, p, i64, p, i64, p, i64, f32, f32, i32, i32]
        lib.gemm.argtypes = base + [p]
        lib.gemm_ex.argtypes = base + [i32, i32, p]
        lib.gemm_checked.argtypes = base + [i32, i32, p]
        lib.gemm_host.argtypes = base + [i32, i32, p]
        lib.gemm_noalloc.argtypes = base + [i32, i32, p]
        lib.gemm_noalloc.restype = i32
        for name in ("gemm", "gemm_ex", "gemm_checked", "gemm_host", "gemm_host_release",
                     "gemm_max_stages", "gemm_plan", "gemm_debug_set"):
            getattr(lib, name).restype = i32
        lib.gemm_host_release.argtypes = []
        lib.gemm_status_string.argtypes = [i32]
        lib.gemm_status_string.restype = ctypes.c_char_p
        lib.gemm_max_stages.argtypes = [i32, i32]
        lib.gemm_debug_set.argtypes = [i64, i32]
        lib.gemm_plan.argtypes = [i64, i64, i64, i32, i32, i32, i32, p, p, p]
        lib.gemm_resolve_tile.argtypes = [i64, i64, i64, i32, i32, i32]
        lib.gemm_resolve_tile.restype = i32
        lib.pipelined_copy.argtypes = [p, p, i64, i32, p]
        lib.pipelined_copy.restype = i32
        lib.gemm_schedule_set.argtypes = [i32]
        lib.gemm_schedule_set.restype = i32
        lib.mma_rate.argtypes = [i32, i32, p, p]
        lib.mma_rate.restype = i32
        lib.mma_rate_pair.argtypes = [i32, i32, p, p]
        lib.mma_rate_pair.restype = i32
        lib.gemm_clock_log.argtypes = [p]
        lib.gemm_clock_log.restype = i32
        if path == LIB_PATH:
            _lib = lib
        return lib


def status_string(status: int) -> str:
    try:
        return load_library().gemm_status_string(int(status)).decode()
    except RuntimeError:
        return f"status {status}"


_DTYPE_CODES = {(torch.float32, torch.float32): GEMM_F32,
                (torch.float16, torch.float32): GEMM_F16_F32,
                (torch.bfloat16, torch.float32): GEMM_BF16_F32,
                (torch.bfloat16, torch.bfloat16): GEMM_BF16_BF16}


def dtype_code(a_dtype: torch.dtype, c_dtype: torch.dtype) -> int:
    try:
        return _DTYPE_CODES[(a_dtype, c_dtype)]
    except KeyError:
        raise ValueError(f"unsupported type pair {a_dtype} -> {c_dtype}") from None


def _row_ld(t: torch.Tensor, name: str) -> int:
    if t.dim() != 2:
        raise ValueError(f"{name} must be 2-D")
    r, c = t.shape
    if r > 1 and c > 1 and t.stride(1) != 1:
        raise ValueError(f"{name} must be row-major (unit column stride)")
    return max(t.stride(0), c, 1) if r > 1 else max(c, 1)


def _b_ld(B: torch.Tensor):
    """(ldb, b_col_major) for B as a K x N matrix."""
    if B.dim() != 2:
        raise ValueError("B must be 2-D")
    K, N = B.shape
    if B.numel() == 0 or B.stride(1) == 1 and (K <= 1 or B.stride(0) >= N):
        return (max(B.stride(0), N, 1) if K > 1 else max(N, 1)), 0
    if B.stride(0) == 1:
        return (max(B.stride(1), K, 1) if N > 1 else max(K, 1)), 1
    raise ValueError("B must be row-major or column-major")


def _args(A, B, C):
    if A.dim() != 2 or B.dim() != 2 or C.dim() != 2:
        raise ValueError("A, B and C must be 2-D")
    M, K = A.shape
    K2, N = B.shape
    if K2 != K or tuple(C.shape) != (M, N):
        raise ValueError(f"shape mismatch: A {tuple(A.shape)}, B {tuple(B.shape)}, "
                         f"C {tuple(C.shape)}")
    if A.dtype != B.dtype:
        raise ValueError("A and B must have the same dtype")
    lda = _row_ld(A, "A")
    ldb, bcm = _b_ld(B)
    ldc = _row_ld(C, "C")
    return M, N, K, lda, ldb, bcm, ldc, dtype_code(A.dtype, C.dtype)


def default_stages(dtype: int, tile: int | None = None) -> int:
    """Ring depth used when a call passes none: 2 on the SIMT path; on the
    tensor-core path the deepest ring the (resolved) tile has room for, which
    is also its fastest (4 when no tile is given: valid for every tile)."""
    if dtype == GEMM_F32:
        return 2
    return TILE_MAX_STAGES.get(tile, 4)


def _stages_for(stages, code: int, M: int, N: int, K: int, tile: int) -> int:
    if stages is not None:
        return int(stages)
    if code == GEMM_F32:
        return default_stages(code)
    # The tile a 4-stage ring resolves to (every tile holds 4), then its deepest ring.
    return default_stages(code, resolve_tile(M, N, K, code, tile, stages=4))


def gemm(A: torch.Tensor, B: torch.Tensor, C: torch.Tensor, alpha: float = 1.0,
         beta: float = 0.0, stages: int | None = None, tile: int = TILE_AUTO,
         stream: torch.cuda.Stream | None = None, checked: bool = False) -> torch.Tensor:
    """C = alpha*A@B + beta*C in place on the GPU (libgemm.so gemm_ex / gemm_checked).

    A: M x K row-major; B: K x N row-major, or column-major as a transposed
    view of an N x K tensor; C: M x N row-major, fp32 (or bf16 for bf16 inputs).
    tile: a TILE_* code for the tensor-core path; a SIMT_FRAGMENTS_* code on the
    fp32 SIMT path.
    Raises GemmError on a non-OK status.  Returns C.
    """
    if not (A.is_cuda and B.is_cuda and C.is_cuda):
        raise ValueError("A, B and C must be CUDA tensors (use gemm_host for host buffers)")
    M, N, K, lda, ldb, bcm, ldc, code = _args(A, B, C)
    dev = C.device.index
    if stages is None and dev != torch.cuda.current_device():
        with torch.cuda.device(dev):
            st = _stages_for(stages, code, M, N, K, tile)
    else:
        st = _stages_for(stages, code, M, N, K, tile)
    s = (stream or torch.cuda.current_stream(dev)).cuda_stream
    lib = _lib or load_library()
    fn = lib.gemm_checked if checked else lib.gemm_ex
    args = (M, N, K, A.data_ptr(), lda, B.data_ptr(), ldb, C.data_ptr(), ldc,
            float(alpha), float(beta), code, st, bcm, int(tile), s)
    if dev == torch.cuda.current_device():
        status = fn(*args)
    else:
        with torch.cuda.device(dev):
            status = fn(*args)
    if status != GEMM_OK:
        raise GemmError(status, "gemm_checked" if checked else "gemm_ex")
    return C


def gemm_host(A: torch.Tensor, B: torch.Tensor, C: torch.Tensor, alpha: float = 1.0,
              beta: float = 0.0, stages: int | None = None, tile: int = TILE_AUTO,
              stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """The same operation on HOST tensors (libgemm.so gemm_host): copies in,
    computes on the current device, copies C back, synchronises."""
    for t, n in ((A, "A"), (B, "B"), (C, "C")):
        if t.device.type != "cpu":
            raise ValueError(f"{n} must be a host tensor")
    M, N, K, lda, ldb, bcm, ldc, code = _args(A, B, C)
    st = _stages_for(stages, code, M, N, K, tile)
    s = (stream or torch.cuda.current_stream()).cuda_stream
    status = load_library().gemm_host(M, N, K, A.data_ptr(), lda, B.data_ptr(), ldb,
                                      C.data_ptr(), ldc, float(alpha), float(beta), code, st,
                                      bcm, int(tile), s)
    if status != GEMM_OK:
        raise GemmError(status, "gemm_host")
    return C


def raw_call(name: str, *args) -> int:
    """Call an entry point with raw arguments (tests of the argument checks)."""
    return int(getattr(load_library(), name)(*args))


def max_stages(dtype: int, tile: int = TILE_AUTO) -> int:
    return int(load_library().gemm_max_stages(int(dtype), int(tile)))


def resolve_tile(M: int, N: int, K: int, dtype: int, tile: int = TILE_AUTO,
                 stages: int = 4) -> int:
    """The TILE_* code gemm uses for these sizes and this ring depth on the
    current device."""
    t = int(load_library().gemm_resolve_tile(M, N, K, int(dtype), int(tile), int(stages)))
    if t < 0:
        raise GemmError(t, "gemm_resolve_tile")
    return t


def plan(M: int, N: int, K: int, dtype: int, stages: int, b_col_major: bool = False,
         tile: int = TILE_AUTO) -> dict:
    """Launch geometry of a call (libgemm.so gemm_plan); needs a CUDA device."""
    grid, cluster, smem = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    st = load_library().gemm_plan(M, N, K, dtype, stages, int(b_col_major), tile,
                                  ctypes.byref(grid), ctypes.byref(cluster), ctypes.byref(smem))
    if st != GEMM_OK:
        raise GemmError(st, "gemm_plan")
    return {"grid": grid.value, "cluster": cluster.value, "smem_bytes": smem.value}


def pipelined_copy(dst: torch.Tensor, src: torch.Tensor, stages: int = 2,
                   stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """dst[:] = src[:] byte for byte (libgemm.so pipelined_copy); both CUDA
    tensors, contiguous, the same number of bytes (a multiple of 16)."""
    if dst.device.type != "cuda" or src.device.type != "cuda":
        raise ValueError("pipelined_copy takes CUDA tensors")
    if not dst.is_contiguous() or not src.is_contiguous():
        raise ValueError("pipelined_copy takes contiguous tensors")
    n = src.numel() * src.element_size()
    if dst.numel() * dst.element_size() != n:
        raise ValueError("dst and src differ in size")
    s = (stream or torch.cuda.current_stream(dst.device)).cuda_stream
    with torch.cuda.device(dst.device):
        st = load_library().pipelined_copy(dst.data_ptr(), src.data_ptr(), n, int(stages), s)
    if st != GEMM_OK:
        raise GemmError(st, "pipelined_copy")
    return dst


# FLOPs of one tcgen05.mma of the rate probe: M = 128, N = 256, K = 16.
MMA_RATE_FLOPS = 2 * 128 * 256 * 16


def mma_rate(n_mma: int = 8192, ctas: int | None = None, device: int | None = None,
             pair: bool = False) -> dict:
    """Dense bf16 tensor-pipe rate in FLOP per SM per clock (libgemm.so
    mma_rate): `ctas` CTAs (default: one per SM) each issue n_mma
    back-to-back 128 x 256 x 16 MMAs and count SM clocks.  With pair=True
    (mma_rate_pair) ctas/2 CTA pairs each issue n_mma 256 x 256 x 16
    cta_group::2 MMAs, the same FLOP per SM per instruction.  Synchronous."""
    dev = torch.cuda.current_device() if device is None else int(device)
    if ctas is None:
        ctas = torch.cuda.get_device_properties(dev).multi_processor_count
    units = int(ctas) // 2 if pair else int(ctas)
    cycles = (ctypes.c_longlong * units)()
    ms = ctypes.c_float()
    fn = load_library().mma_rate_pair if pair else load_library().mma_rate
    with torch.cuda.device(dev):
        st = fn(int(n_mma), units, cycles, ctypes.byref(ms))
    if st != GEMM_OK:
        raise GemmError(st, "mma_rate_pair" if pair else "mma_rate")
    cyc = sorted(int(c) for c in cycles)
    flops = n_mma * MMA_RATE_FLOPS
    ctas = 2 * units if pair else units
    return {"n_mma": int(n_mma), "ctas": int(ctas), "pair": bool(pair),
            "cycles_min": cyc[0], "cycles_median": cyc[len(cyc) // 2], "cycles_max": cyc[-1],
            "flop_per_clk_per_sm": flops / cyc[len(cyc) // 2],
            "elapsed_ms": ms.value,
            "tflops": flops * ctas / (ms.value * 1e-3) / 1e12}


def clock_log(buf: torch.Tensor | None) -> None:
    """Measurement hook (libgemm.so gemm_clock_log): with `buf` (two zeroed
    int64 on the GPU), CTA 0 of every later tensor-core launch adds its SM
    clock ticks to buf[0] and its nanoseconds to buf[1]; None turns it off."""
    if buf is not None and (buf.device.type != "cuda" or buf.dtype != torch.int64
                            or buf.numel() < 2 or not buf.is_contiguous()):
        raise ValueError("clock_log takes two contiguous int64 on the GPU")
    load_library().gemm_clock_log(None if buf is None else buf.data_ptr())


SCHEDULE_AUTO, SCHEDULE_FULL_TILES, SCHEDULE_STREAM_K = 0, 1, 2


def schedule_set(schedule: int) -> None:
    """Tile schedule of the tensor-core kernel (libgemm.so gemm_schedule_set)."""
    st = load_library().gemm_schedule_set(int(schedule))
    if st != GEMM_OK:
        raise GemmError(st, "gemm_schedule_set")


def debug_set(wait_limit_ns: int = 0, withhold_arrive: int = -1) -> None:
    load_library().gemm_debug_set(int(wait_limit_ns), int(withhold_arrive))
