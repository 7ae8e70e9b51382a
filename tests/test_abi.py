"""The C-ABI library (no GPU needed): it builds, loads, exports every symbol
include/gemm.h declares, and its host-side argument checks answer before any
CUDA call is made.  No test here launches a kernel."""
import ctypes
import os
import re
import subprocess

import pytest

from stage_software_pipelining_gb300 import build as gemm_build
from stage_software_pipelining_gb300 import gemm as G
from stage_software_pipelining_gb300.workloads import (GEMM_BF16_BF16, GEMM_BF16_F32,
                                                       GEMM_F16_F32, GEMM_F32)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gemm.h")

# Fake device addresses: the checks below reject the call before any pointer
# is used, so these are never dereferenced.
P = 0x7F0000000000
NULL = None


@pytest.fixture(scope="module")
def lib():
    gemm_build.build()
    return G.load_library()


def declared_functions():
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:int|const char\s*\*)\s*(\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_binding_exports():
    assert declared_functions() == sorted(G.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", G.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    for name in declared_functions():
        assert name in exported, name


def gemm_ex(lib, M, N, K, A=P, lda=None, B=P, ldb=None, C=P, ldc=None, alpha=1.0, beta=0.0,
            dtype=GEMM_BF16_F32, stages=3, bcm=0, tile=0):
    lda = K if lda is None else lda
    ldb = (K if bcm else N) if ldb is None else ldb
    ldc = N if ldc is None else ldc
    return lib.gemm_ex(M, N, K, A, lda, B, ldb, C, ldc, alpha, beta, dtype, stages, bcm, tile,
                       None)


def test_negative_sizes_rejected(lib):
    assert gemm_ex(lib, -1, 8, 8) == G.GEMM_ERR_ARG
    assert gemm_ex(lib, 8, -1, 8) == G.GEMM_ERR_ARG
    assert gemm_ex(lib, 8, 8, -1) == G.GEMM_ERR_ARG


def test_bad_dtype_and_stages(lib):
    assert gemm_ex(lib, 8, 8, 8, dtype=7) == G.GEMM_ERR_ARG
    assert gemm_ex(lib, 8, 8, 8, dtype=-1) == G.GEMM_ERR_ARG
    assert gemm_ex(lib, 8, 8, 8, stages=0) == G.GEMM_ERR_ARG
    assert gemm_ex(lib, 8, 8, 8, stages=7) == G.GEMM_ERR_ARG
    assert gemm_ex(lib, 8, 8, 8, dtype=GEMM_F32, stages=5) == G.GEMM_ERR_ARG
    # every stage is a K slice of 64: shared memory holds 6 stages for the
    # 128 x 128 and 256 x 256 pair tiles and 4 for the 128 x 256 and 256 x 512
    # tiles; 1..6 is the valid range, a deeper ring than an explicit tile
    # holds is a valid request the library does not implement
    for bad in (0, 7, 8, -1):
        for t in (0, G.TILE_128x128, G.TILE_256x256_2SM):
            assert gemm_ex(lib, 8, 512, 8, stages=bad, tile=t) == G.GEMM_ERR_ARG
    for s in (5, 6):
        assert gemm_ex(lib, 8, 512, 8, stages=s, tile=G.TILE_128x256) == G.GEMM_ERR_UNSUPPORTED
        assert gemm_ex(lib, 8, 512, 8, stages=s, tile=G.TILE_256x512_2SM) == \
            G.GEMM_ERR_UNSUPPORTED
    assert gemm_ex(lib, 8, 8, 8, tile=192) == G.GEMM_ERR_ARG
    assert gemm_ex(lib, 8, 8, 8, tile=2048) == G.GEMM_ERR_ARG
    assert gemm_ex(lib, 8, 8, 8, dtype=GEMM_F32, stages=2, tile=128) == G.GEMM_ERR_ARG
    assert gemm_ex(lib, 8, 8, 8, dtype=GEMM_F32, stages=2, tile=2) == G.GEMM_ERR_ARG
    assert gemm_ex(lib, 8, 8, 8, bcm=2) == G.GEMM_ERR_ARG


def test_leading_dimensions_too_small(lib):
    assert gemm_ex(lib, 8, 16, 24, lda=16) == G.GEMM_ERR_ARG
    assert gemm_ex(lib, 8, 16, 24, ldb=8) == G.GEMM_ERR_ARG
    assert gemm_ex(lib, 8, 16, 24, ldb=16, bcm=1) == G.GEMM_ERR_ARG
    assert gemm_ex(lib, 8, 16, 24, ldc=8) == G.GEMM_ERR_ARG


def test_null_pointers(lib):
    assert gemm_ex(lib, 8, 16, 24, A=NULL) == G.GEMM_ERR_ARG
    assert gemm_ex(lib, 8, 16, 24, B=NULL) == G.GEMM_ERR_ARG
    assert gemm_ex(lib, 8, 16, 24, C=NULL) == G.GEMM_ERR_ARG


def test_alignment_rules(lib):
    assert gemm_ex(lib, 8, 16, 24, A=P + 2) == G.GEMM_ERR_ALIGN
    assert gemm_ex(lib, 8, 16, 24, B=P + 8) == G.GEMM_ERR_ALIGN
    assert gemm_ex(lib, 8, 16, 24, C=P + 4) == G.GEMM_ERR_ALIGN
    # 16-bit inputs: lda must be a multiple of 8 elements (16 bytes)
    assert gemm_ex(lib, 8, 16, 20, lda=20) == G.GEMM_ERR_ALIGN
    assert gemm_ex(lib, 8, 16, 24, lda=28) == G.GEMM_ERR_ALIGN
    # fp32 output: ldc a multiple of 4
    assert gemm_ex(lib, 8, 18, 24, ldc=18) == G.GEMM_ERR_ALIGN
    # bf16 output: ldc a multiple of 8
    assert gemm_ex(lib, 8, 20, 24, ldc=20, dtype=GEMM_BF16_BF16) == G.GEMM_ERR_ALIGN
    # fp32 SIMT: lda a multiple of 4
    assert gemm_ex(lib, 8, 16, 6, lda=6, dtype=GEMM_F32, stages=2) == G.GEMM_ERR_ALIGN


def test_column_major_b_only_on_tensor_cores(lib):
    assert gemm_ex(lib, 8, 16, 24, dtype=GEMM_F32, stages=2, bcm=1) == G.GEMM_ERR_UNSUPPORTED


def test_oversized_dimensions(lib):
    big = 2**31
    assert gemm_ex(lib, big, 16, 16, lda=16) == G.GEMM_ERR_UNSUPPORTED


def test_empty_output_is_a_noop(lib):
    # M == 0 or N == 0 returns before touching CUDA, even with fake pointers
    assert gemm_ex(lib, 0, 16, 24) == G.GEMM_OK
    assert gemm_ex(lib, 8, 0, 24) == G.GEMM_OK
    assert lib.gemm(0, 0, 0, NULL, 1, NULL, 1, NULL, 1, 1.0, 0.0, GEMM_F16_F32, 2, None) == 0


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5, -6, -7):
        s = lib.gemm_status_string(code).decode()
        assert s.startswith("GEMM_")
    assert "unknown" in lib.gemm_status_string(42).decode()


def test_resolve_tile_without_a_device(lib):
    """Explicit tiles come back unchanged; SIMT types and bad codes are
    refused; on a host without a GPU the automatic choice is the pair tile
    for large M and N and the one-CTA tiles for a single 128-row/column."""
    rt = lib.gemm_resolve_tile
    for t in (G.TILE_128x128, G.TILE_128x256, G.TILE_256x256_2SM, G.TILE_256x512_2SM):
        assert rt(4096, 4096, 4096, GEMM_BF16_F32, t, 4) == t
    # long K takes the 512-wide pair tile, shorter K the 256-wide one
    assert rt(4096, 4096, 8192, GEMM_BF16_F32, 0, 4) == G.TILE_256x512_2SM
    assert rt(4096, 4096, 4096, GEMM_BF16_F32, 0, 4) == G.TILE_256x256_2SM
    assert rt(8, 8, 8, GEMM_F32, 0, 2) == G.GEMM_ERR_ARG
    assert rt(8, 8, 8, GEMM_BF16_F32, 192, 2) == G.GEMM_ERR_ARG
    assert rt(-1, 8, 8, GEMM_BF16_F32, 0, 2) == G.GEMM_ERR_ARG
    assert rt(100, 4096, 64, GEMM_BF16_F32, 0, 4) == G.TILE_128x256
    assert rt(4096, 100, 64, GEMM_BF16_F32, 0, 4) == G.TILE_128x128
    # a ring deeper than the automatic tile holds takes the tile of the same
    # rows per SM that holds six stages; explicit tiles never change
    assert rt(4096, 4096, 8192, GEMM_BF16_F32, 0, 5) == G.TILE_256x256_2SM
    assert rt(4096, 4096, 8192, GEMM_BF16_F32, 0, 6) == G.TILE_256x256_2SM
    assert rt(100, 4096, 64, GEMM_BF16_F32, 0, 6) == G.TILE_128x128
    assert rt(4096, 4096, 8192, GEMM_BF16_F32, G.TILE_256x512_2SM, 6) == G.TILE_256x512_2SM
    for bad in (0, 7):
        assert rt(4096, 4096, 4096, GEMM_BF16_F32, 0, bad) == G.GEMM_ERR_ARG


def test_max_stages(lib):
    assert lib.gemm_max_stages(GEMM_F32, 0) == 4
    assert lib.gemm_max_stages(GEMM_F32, 1) == 4      # single register fragment set
    assert lib.gemm_max_stages(GEMM_BF16_F32, G.TILE_128x256) == 4
    assert lib.gemm_max_stages(GEMM_BF16_F32, G.TILE_128x128) == 6
    assert lib.gemm_max_stages(GEMM_BF16_BF16, G.TILE_256x256_2SM) == 6
    assert lib.gemm_max_stages(GEMM_BF16_F32, G.TILE_256x512_2SM) == 4
    assert lib.gemm_max_stages(GEMM_F16_F32, 0) == 6
    assert lib.gemm_max_stages(GEMM_F32, 128) == G.GEMM_ERR_ARG
    assert lib.gemm_max_stages(9, 0) == G.GEMM_ERR_ARG


def test_host_entry_validates_first(lib):
    assert lib.gemm_host(-1, 8, 8, P, 8, P, 8, P, 8, 1.0, 0.0, GEMM_BF16_F32, 3, 0, 0,
                         None) == G.GEMM_ERR_ARG
    assert lib.gemm_host(0, 8, 8, P, 8, P, 8, P, 8, 1.0, 0.0, GEMM_BF16_F32, 3, 0, 0,
                         None) == G.GEMM_OK


def test_python_binding_marshalling():
    import torch
    A = torch.zeros(8, 24, dtype=torch.bfloat16)
    Bt = torch.zeros(16, 24, dtype=torch.bfloat16)
    C = torch.zeros(8, 16)
    assert G._args(A, Bt.t(), C)[5] == 1          # column-major B detected
    assert G._args(A, Bt.t().contiguous(), C)[5] == 0
    M, N, K, lda, ldb, bcm, ldc, code = G._args(A, Bt.t(), C)
    assert (M, N, K, lda, ldb, ldc, code) == (8, 16, 24, 24, 24, 16, GEMM_BF16_F32)
    with pytest.raises(ValueError):
        G._args(A, torch.zeros(23, 16, dtype=torch.bfloat16), C)
    with pytest.raises(ValueError):
        G.dtype_code(torch.float16, torch.float16)
    with pytest.raises(ValueError):
        G.gemm(A, Bt.t(), C)                      # host tensors on the device entry


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        G.load_library(str(tmp_path / "libgemm.so"))


def test_ctypes_signatures_cover_exports(lib):
    for name in G.EXPORTS:
        fn = getattr(lib, name)
        assert fn.restype in (ctypes.c_int, ctypes.c_char_p), name


def test_pipelined_copy_argument_checks(lib):
    c = lib.pipelined_copy
    assert c(P, P + 4096, 0, 2, None) == G.GEMM_OK          # empty: nothing touched
    assert c(P, P + 4096, -16, 2, None) == G.GEMM_ERR_ARG
    assert c(P, P + 4096, 64, 0, None) == G.GEMM_ERR_ARG
    assert c(P, P + 4096, 64, 9, None) == G.GEMM_ERR_ARG
    assert c(None, P, 64, 2, None) == G.GEMM_ERR_ARG
    assert c(P, P + 32, 64, 2, None) == G.GEMM_ERR_ARG       # overlapping ranges
    assert c(P + 8, P + 4096, 64, 2, None) == G.GEMM_ERR_ALIGN
    assert c(P, P + 4096, 40, 2, None) == G.GEMM_ERR_ALIGN   # not a multiple of 16


def test_schedule_hook(lib):
    assert lib.gemm_schedule_set(-1) == G.GEMM_ERR_ARG
    assert lib.gemm_schedule_set(3) == G.GEMM_ERR_ARG
    for v in (1, 2, 0):
        assert lib.gemm_schedule_set(v) == G.GEMM_OK


def test_noalloc_entry_validates_on_the_host(lib):
    na = lib.gemm_noalloc
    # the same argument checks as gemm_ex, answered before any CUDA call
    assert na(-1, 8, 8, P, 8, P, 8, P, 8, 1.0, 0.0, GEMM_BF16_F32, 3, 0, 0, None) == G.GEMM_ERR_ARG
    assert na(8, 16, 24, P + 2, 24, P, 16, P, 16, 1.0, 0.0, GEMM_BF16_F32, 3, 0, 0,
              None) == G.GEMM_ERR_ALIGN
    # the SIMT path has no scratch, so no allocation-free variant
    assert na(8, 16, 24, P, 24, P, 16, P, 16, 1.0, 0.0, GEMM_F32, 2, 0, 0,
              None) == G.GEMM_ERR_UNSUPPORTED
    assert na(0, 16, 24, P, 24, P, 16, P, 16, 1.0, 0.0, GEMM_BF16_F32, 3, 0, 0, None) == G.GEMM_OK
    # the 256 x 512 tile by name: its partials do not fit the fixed array, so
    # it is refused for every shape (also one that would need no partials)
    for M, N, K in ((0, 16, 24), (8192, 8192, 8192), (4864, 2048, 8192), (300, 520, 200)):
        assert na(M, N, K, P, max(K, 8), P, max(N, 8), P, max(N, 8), 1.0, 0.0, GEMM_BF16_F32, 4,
                  0, G.TILE_256x512_2SM, None) == G.GEMM_ERR_SCRATCH
    # stages 5 and 6 are valid on the noalloc path too (the automatic tile
    # then holds them); 7 is not
    assert na(8, 16, 24, P, 24, P, 16, P, 16, 1.0, 0.0, GEMM_BF16_F32, 7, 0, 0,
              None) == G.GEMM_ERR_ARG
    assert na(8, 16, 24, P, 24, P, 16, P, 16, 1.0, 0.0, GEMM_BF16_F32, 6, 0, G.TILE_128x256,
              None) == G.GEMM_ERR_UNSUPPORTED
    assert "fixed array" in lib.gemm_status_string(G.GEMM_ERR_SCRATCH).decode()


def test_mma_rate_argument_checks(lib):
    cyc = (ctypes.c_longlong * 4)()
    ms = ctypes.c_float()
    # answered before any CUDA call
    assert lib.mma_rate(0, 4, cyc, ctypes.byref(ms)) == G.GEMM_ERR_ARG
    assert lib.mma_rate((1 << 20) + 1, 4, cyc, ctypes.byref(ms)) == G.GEMM_ERR_ARG
    assert lib.mma_rate(16, 0, cyc, ctypes.byref(ms)) == G.GEMM_ERR_ARG
    assert lib.mma_rate(16, 4, None, ctypes.byref(ms)) == G.GEMM_ERR_ARG
    assert lib.mma_rate(16, 4, cyc, None) == G.GEMM_ERR_ARG


def test_default_stages_follow_the_tile():
    # the deepest ring each tile has room for; 4 (valid everywhere) without one
    assert G.default_stages(GEMM_F32) == 2
    assert G.default_stages(GEMM_BF16_F32) == 4
    assert G.default_stages(GEMM_BF16_F32, G.TILE_128x128) == 6
    assert G.default_stages(GEMM_BF16_F32, G.TILE_128x256) == 4
    assert G.default_stages(GEMM_BF16_F32, G.TILE_256x256_2SM) == 6
    assert G.default_stages(GEMM_BF16_F32, G.TILE_256x512_2SM) == 4


def test_mma_rate_pair_argument_checks(lib):
    cyc = (ctypes.c_longlong * 4)()
    ms = ctypes.c_float()
    assert lib.mma_rate_pair(0, 2, cyc, ctypes.byref(ms)) == G.GEMM_ERR_ARG
    assert lib.mma_rate_pair((1 << 20) + 1, 2, cyc, ctypes.byref(ms)) == G.GEMM_ERR_ARG
    assert lib.mma_rate_pair(16, 0, cyc, ctypes.byref(ms)) == G.GEMM_ERR_ARG
    assert lib.mma_rate_pair(16, 2, None, ctypes.byref(ms)) == G.GEMM_ERR_ARG
    assert lib.mma_rate_pair(16, 2, cyc, None) == G.GEMM_ERR_ARG


def test_binding_constants_match_the_header():
    """Every enum value include/gemm.h declares is the value the Python side
    passes: status codes, tensor-core tiles, SIMT fragment schemes, dtypes,
    and each tile's stage limit as gemm_max_stages reports it."""
    import re
    from stage_software_pipelining_gb300 import workloads as W
    text = open(HEADER).read()
    declared = {name: int(val) for name, val in
                re.findall(r"\b(GEMM_[A-Z0-9_x]+)\s*=\s*(-?\d+)", text)}
    expect = {
        "GEMM_OK": G.GEMM_OK, "GEMM_ERR_ARG": G.GEMM_ERR_ARG,
        "GEMM_ERR_UNSUPPORTED": G.GEMM_ERR_UNSUPPORTED, "GEMM_ERR_ALIGN": G.GEMM_ERR_ALIGN,
        "GEMM_ERR_LAUNCH": G.GEMM_ERR_LAUNCH, "GEMM_ERR_TIMEOUT": G.GEMM_ERR_TIMEOUT,
        "GEMM_ERR_CUDA": G.GEMM_ERR_CUDA, "GEMM_ERR_SCRATCH": G.GEMM_ERR_SCRATCH,
        "GEMM_TILE_AUTO": G.TILE_AUTO, "GEMM_TILE_128x128": G.TILE_128x128,
        "GEMM_TILE_128x256": G.TILE_128x256, "GEMM_TILE_256x256_2SM": G.TILE_256x256_2SM,
        "GEMM_TILE_256x512_2SM": G.TILE_256x512_2SM,
        "GEMM_SIMT_FRAGMENTS_DOUBLE": G.SIMT_FRAGMENTS_DOUBLE,
        "GEMM_SIMT_FRAGMENTS_SINGLE": G.SIMT_FRAGMENTS_SINGLE,
        "GEMM_F32": W.GEMM_F32, "GEMM_F16_F32": W.GEMM_F16_F32,
        "GEMM_BF16_F32": W.GEMM_BF16_F32, "GEMM_BF16_BF16": W.GEMM_BF16_BF16,
    }
    assert declared == expect
    lib = G.load_library()
    for tile, stages in G.TILE_MAX_STAGES.items():
        assert lib.gemm_max_stages(W.GEMM_BF16_F32, tile) == stages
